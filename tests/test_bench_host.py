"""Host-side logic of bench.py (no GPU): the pipelined end-to-end loop's
slicing of a step into muon_step calls, and the pair-kernel rule that
labels the roofline kernel."""
import pytest

import bench
from newton_schulz_orthogonalized_muon_gb300 import flops
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl


def _bytes(specs, esz=2):
    return [s.shape[0] * s.shape[1] * esz for s in specs]


@pytest.mark.parametrize("name", ["llama3-8b", "moonlight-moe", "gpt2-small"])
def test_e2e_slices_cover_every_parameter_once_in_group_order(name):
    specs = bench.weight_set(name, None).muon
    nb = _bytes(specs)
    order = bench.e2e_slices(specs, nb)
    flat = [i for sl in order for i in sl]
    assert sorted(flat) == list(range(len(specs)))
    dims = [flops.ns_dims(specs[sl[0]].shape[0], specs[sl[0]].shape[1], specs[sl[0]].split_heads) for sl in order]
    for sl, d in zip(order, dims):
        # one same-shape group per call, at most the byte limit unless a
        # single matrix is larger
        assert all(flops.ns_dims(specs[i].shape[0], specs[i].shape[1], specs[i].split_heads) == d for i in sl)
        assert len(sl) == 1 or sum(nb[i] for i in sl) <= bench.E2E_SLICE_BYTES
    assert dims == sorted(dims)                      # the library's group order


def test_e2e_slices_cut_only_at_the_limit():
    specs = [wl.ParamSpec(f"p{i}", (64, 128)) for i in range(10)]
    nb = _bytes(specs)                               # 16 KiB each
    order = bench.e2e_slices(specs, nb, limit=3 * nb[0])
    assert [len(sl) for sl in order] == [3, 3, 3, 1]
    order = bench.e2e_slices(specs, nb, limit=nb[0] // 2)   # smaller than one matrix
    assert [len(sl) for sl in order] == [1] * 10


def test_e2e_slices_keep_transposed_partners_in_their_group():
    # 2048 x 1408 is the transpose of 1408 x 2048: one group, as in the library
    specs = [wl.ParamSpec("up", (1408, 2048)), wl.ParamSpec("down", (2048, 1408)),
             wl.ParamSpec("q", (2048, 2048), split_heads=16)]
    order = bench.e2e_slices(specs, _bytes(specs))
    assert order == [[2], [0, 1]]                    # (128, 2048) sorts before (1408, 2048)


@pytest.mark.parametrize("m,kernel,pair", [
    (4096, "update", True), (4096, "syrk", True), (1408, "syrk", True), (1408, "update", False),
    (1408, "final", False), (2176, "update", True), (768, "update", False), (768, "syrk", False),
    (256, "update", True), (256, "syrk", True), (640, "syrk", False), (128, "syrk", False)])
def test_pair_rule_matches_the_library(m, kernel, pair, monkeypatch):
    monkeypatch.delenv("MUON_TC_PAIR", raising=False)
    monkeypatch.delenv("MUON_TC_PAIR_MIN_M", raising=False)
    assert bench.uses_pairs(m, kernel) is pair


@pytest.mark.parametrize("m,kernel,pair", [
    (4096, "syrk", True), (4096, "poly", True), (4096, "update", True), (4096, "final", True),
    (1408, "update", True), (1408, "final", False), (640, "update", False)])
def test_gram_pair_rule_matches_the_library(m, kernel, pair, monkeypatch):
    # the Gram method runs R0, P and its m x m products on pairs by the
    # symmetric-product rule, and O = Q X0 by the UPDATE rule
    monkeypatch.delenv("MUON_TC_PAIR", raising=False)
    monkeypatch.delenv("MUON_TC_PAIR_MIN_M", raising=False)
    assert bench.uses_pairs(m, kernel, "gram") is pair


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("m,n,steps", [(4096, 14336, 5), (1024, 4096, 5), (256, 512, 3), (128, 2048, 1)])
def test_per_class_flops_add_up_to_the_method_total(method, m, n, steps):
    # the bench's per-kernel rows (launches x flops per launch) sum to the
    # method's own total, so the headline and the rows use one flop model
    launches = flops.kernel_launches(method, steps)
    per = flops.kernel_flops(method, m, n)
    total = sum(launches[k] * per[k] for k in launches)
    assert total == pytest.approx(flops.ns_flops(method, m, n, steps), rel=1e-12)
    assert bench.kernel_mode(method, "final") in ("FINAL_T", "G_FINAL_T")


def test_gram_flops_are_below_standard_only_for_wide_matrices():
    # R0 and O = Q X0 carry the n-dependent work (3 m^2 n), the iteration
    # (5 + 3 * 4) m^2 (m + 1): fewer flops than the standard method once
    # n / m is large enough
    assert flops.ns_flops("gram", 256, 16384) < 0.3 * flops.ns_flops("standard", 256, 16384)
    assert flops.ns_flops("gram", 4096, 4096) > flops.ns_flops("standard", 4096, 4096)


def test_e2e_last_slice_is_small():
    # the step's last read-back is not overlapped: the last group ends with a
    # slice of at most E2E_LAST_SLICE_BYTES (two 117 MB Llama matrices)
    specs = bench.weight_set("llama3-8b", None).muon
    nb = _bytes(specs)
    order = bench.e2e_slices(specs, nb)
    assert sum(nb[i] for i in order[-1]) <= bench.E2E_LAST_SLICE_BYTES
    assert len(order[-1]) >= 1
    assert sorted(i for sl in order for i in sl) == list(range(len(specs)))
    # a last group smaller than the limit is not cut
    small = [wl.ParamSpec(f"p{i}", (64, 128)) for i in range(10)]
    assert bench.e2e_slices(small, _bytes(small)) == [list(range(10))]


def test_e2e_subset_takes_the_same_fraction_of_every_group():
    # the bounded e2e keeps the first matrices of each same-shape group
    specs = ([wl.ParamSpec(f"a{i}", (1024, 4096)) for i in range(8)] +
             [wl.ParamSpec(f"b{i}", (4096, 1024)) for i in range(4)] +     # transposed: same group as a
             [wl.ParamSpec(f"c{i}", (512, 512)) for i in range(10)])
    keep = bench.e2e_subset(specs, _bytes(specs), 0.5)
    assert keep == sorted([0, 1, 2, 3, 4, 5] + list(range(12, 17)))
    assert bench.e2e_subset(specs, _bytes(specs), 0.01) == [0, 12]        # at least one per group
    assert bench.e2e_subset(specs, _bytes(specs), 1.0) == list(range(len(specs)))

