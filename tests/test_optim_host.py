"""Host logic of the optimizer wrapper (no GPU): the parameter
classification follows the oracle's tagging rule, and the flattening of
higher-rank parameters gives the shapes and update scale the printed Muon
class uses."""
import pytest
import torch

import oracle
from newton_schulz_orthogonalized_muon_gb300 import optim

NAMES = ["model.embed_tokens.weight", "lm_head.weight", "layers.0.attn.q_proj.weight", "layers.0.mlp.down_proj.bias",
         "layers.0.input_layernorm.weight", "h.3.attn.c_attn.weight", "conv.weight", "Embedding.table", "LM_HEAD.w",
         "wpe.weight"]


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("ndim", [1, 2, 3, 4])
def test_tagging_matches_the_oracle(name, ndim):
    assert optim.takes_muon(name, ndim) == oracle.is_muon_param(name, ndim)


def test_split_params_keeps_order_and_flattens_higher_rank():
    params = [("embed_tokens.weight", torch.zeros(10, 4)), ("a.weight", torch.zeros(8, 12)),
              ("a.bias", torch.zeros(12)), ("conv.weight", torch.zeros(16, 3, 5, 5)),
              ("frozen.weight", torch.zeros(4, 4, requires_grad=False)), ("b.weight", torch.zeros(6, 9, 2))]
    for _, p in params[:4] + params[5:]:
        p.requires_grad_(True)
    muon, adamw = optim.split_params(params)
    assert [e.name for e in muon] == ["a.weight"]
    assert [n for n, _ in adamw] == ["embed_tokens.weight", "a.bias", "conv.weight", "b.weight"]
    muon, adamw = optim.split_params(params, higher_rank=True)
    assert [(e.name, e.rows, e.cols, e.scale_dim) for e in muon] == [
        ("a.weight", 8, 12, 0), ("conv.weight", 16, 75, 16), ("b.weight", 6, 18, 9)]
    assert [n for n, _ in adamw] == ["embed_tokens.weight", "a.bias"]
    # the scale the library applies through scale_dim equals the oracle's p.shape[:2] rule
    for e in muon:
        sd = e.scale_dim or max(e.rows, e.cols)
        assert 0.2 * sd ** 0.5 == pytest.approx(oracle.update_scale(e.param.shape))
