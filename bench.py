#!/usr/bin/env python
"""Benchmark of the GB300 Muon step.

One step = one full Muon step (momentum/Nesterov, Frobenius normalisation,
5 quintic Newton-Schulz iterations, decoupled update) over every hidden 2-D
matrix of a Llama-3-8B-shaped weight set (32 layers; q, o 4096x4096;
k, v 1024x4096; gate, up 14336x4096; down 4096x14336; bf16 params and
grads, fp32 momentum), synthetic seeded inputs resident in HBM.

Prints one JSON line.  `value` is the Newton-Schulz throughput in TFLOP/s
(algorithmic flops: symmetric products on one triangle) of the whole step;
`ms_per_step` is the step time.  With torchrun (N > 1) the matrices of N
copies of the set are dealt to the ranks by size-sorted ping-pong ownership
(weak scaling, no collective inside the step).

After the headline's timed regions, the default run also times the other
configurations compactly and reports them under "other_configs" (one GPU,
--workload llama3-8b only; --no-other-configs skips them): the Gram method
on the same Llama inputs, GPT-2-small in bf16 and in fp32, the single fp32
256x512 matrix, and the Moonlight-like MoE set, each with its own clocks.

--impl reference times the fp64 CPU oracle (the reference arm) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon step ms & Newton-Schulz TFLOP/s (bf16, % tensor peak) on 1 GB300"
UNIT = "TFLOP/s"
LR, WD, MU = 0.02, 0.1, 0.95
NS_STEPS = 5
E2E_SLICE_BYTES = 2 << 30      # parameters per muon_step call of the pipelined e2e loop
E2E_LAST_SLICE_BYTES = 256 << 20   # ... and in its last call, whose read-back is not overlapped
F32_TC_MAX_M = int(os.environ.get("MUON_F32_TC_MAX_M", "2048"))   # the library's fp32 tensor-core rule


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["llama3-8b", "gpt2-small", "moonlight-moe", "single-fp32", "wide"],
                    default="llama3-8b",
                    help="wide: the standard-vs-gram sweep over 64 Gaussian m x n matrices per shape; single-fp32: "
                         "one fp32 256x512 matrix")
    ap.add_argument("--param-dtype", choices=["bf16", "fp32"], default=None,
                    help="parameter and gradient dtype (default bf16; fp32 for single-fp32): fp32 runs the fp32 path")
    ap.add_argument("--ns-method", choices=["standard", "gram"], default="standard")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (parity runs only)")
    ap.add_argument("--workspace-gb", type=float, default=64.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adamw", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the compact timing of the other configurations after the headline")
    ap.add_argument("--cpu-baseline-plan", action="store_true",
                    help="time the fp64 oracle over all five configurations on the host cores and exit")
    return ap.parse_args(argv)


def weight_set(name, layers=None):
    from newton_schulz_orthogonalized_muon_gb300 import workloads as wl
    if name == "single-fp32":
        return wl.single_matrix_256x512()
    if name == "llama3-8b":
        return wl.llama3_8b(layers or 32)
    if name == "gpt2-small":
        return wl.gpt2_small(layers or 12)
    return wl.moonlight_moe(layers or 27)


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured (MEASURED_PEAKS.json)"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ workload

def make_inputs(specs, device, seed, batch=32, dtype=None, rank=64):
    """Seeded synthetic tensors on the device: W ~ N(0, 0.02), G low-rank
    (rank 64, orthonormal factors from QR of Gaussians, sigma_i = 0.5**(i/8))
    + 1e-3 N(0,1) noise, both bf16 (or `dtype`), M = 0 fp32.  Same-shape
    matrices are drawn in batches from one seeded torch.Generator per shape."""
    import torch
    dtype = dtype or torch.bfloat16
    from newton_schulz_orthogonalized_muon_gb300 import workloads as wl
    W, G, M = [None] * len(specs), [None] * len(specs), [None] * len(specs)
    by_shape = {}
    for i, s in enumerate(specs):
        by_shape.setdefault(tuple(s.shape), []).append(i)
    gen = torch.Generator(device=device)
    for k, (shape, idx) in enumerate(sorted(by_shape.items())):
        gen.manual_seed(wl.matrix_seed(seed, k))
        rows, cols = shape
        r = min(rank, rows, cols)
        sigma = 0.5 ** (torch.arange(r, device=device, dtype=torch.float32) / 8.0)
        for c0 in range(0, len(idx), batch):
            part = idx[c0:c0 + batch]
            nb = len(part)
            U, _ = torch.linalg.qr(torch.randn(nb, rows, r, generator=gen, device=device))
            V, _ = torch.linalg.qr(torch.randn(nb, cols, r, generator=gen, device=device))
            g = torch.bmm(U * sigma, V.transpose(1, 2))
            g.add_(torch.randn(nb, rows, cols, generator=gen, device=device), alpha=1e-3)
            w = torch.randn(nb, rows, cols, generator=gen, device=device).mul_(0.02)
            for j, i in enumerate(part):
                G[i] = g[j].to(dtype)
                W[i] = w[j].to(dtype)
                M[i] = torch.zeros(shape, dtype=torch.float32, device=device)
            del U, V, g, w
    return W, G, M


def owned_specs(ws, world, rank):
    from newton_schulz_orthogonalized_muon_gb300 import partition
    from newton_schulz_orthogonalized_muon_gb300.workloads import ParamSpec
    specs = [ParamSpec(f"replica{r}.{p.name}", p.shape, p.split_heads) for r in range(world) for p in ws.muon]
    sizes = [p.shape[0] * p.shape[1] for p in specs]
    mine = partition.owned(sizes, world, rank)
    return [specs[i] for i in mine], mine


# ------------------------------------------------------------ oracle arm

SAMPLE_SHAPE = (1024, 4096)
SAMPLE_TEXT = "one Muon step of one k_proj-shaped 1024x4096 matrix (fp64 numpy oracle)"


def oracle_sample_step(_cache={}):
    """One Muon step of one k_proj-shaped 1024x4096 matrix of the set in the
    fp64 oracle on the host cores.  Returns (seconds, algorithmic NS flops)."""
    import numpy as np
    import oracle
    from newton_schulz_orthogonalized_muon_gb300 import flops, workloads as wl
    if "in" not in _cache:
        _cache["in"] = (wl.weight(1, SAMPLE_SHAPE).astype(np.float64),
                        wl.lowrank_grad(2, SAMPLE_SHAPE[0], SAMPLE_SHAPE[1], 64).astype(np.float64))
    W, G = _cache["in"]
    M = np.zeros(SAMPLE_SHAPE)
    t0 = time.perf_counter()
    oracle.muon_step(W, G, M, lr=LR, wd=WD, mu=MU, nesterov=True)
    return time.perf_counter() - t0, flops.ns_flops_standard(SAMPLE_SHAPE[0], SAMPLE_SHAPE[1], NS_STEPS)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (x86 'model name', else lscpu's), and its
    logical core count."""
    name = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if name is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.startswith(("Model name", "Vendor ID")):
                    name = (name + " / " if name else "") + line.split(":", 1)[1].strip()
        except Exception:
            pass
    return {"model": name or "unknown", "logical_cores": os.cpu_count()}


def oracle_matrix_seconds(shape, split_heads=1, method="standard", seed=0):
    """Seconds of one fp64 oracle Muon step of one parameter of this shape
    (seeded low-rank gradient, zero momentum) on the host cores."""
    import numpy as np
    import oracle
    from newton_schulz_orthogonalized_muon_gb300 import workloads as wl
    W = wl.weight(seed + 1, shape).astype(np.float64)
    G = wl.lowrank_grad(seed + 2, shape[0], shape[1], 64).astype(np.float64)
    M = np.zeros(shape)
    t0 = time.perf_counter()
    oracle.muon_step(W, G, M, lr=LR, wd=WD, mu=MU, nesterov=True, split_heads=split_heads, method=method)
    return time.perf_counter() - t0


def set_groups(specs):
    """{(shape, split_heads): count} of a parameter list."""
    groups = {}
    for s_ in specs:
        key = (tuple(s_.shape), s_.split_heads)
        groups[key] = groups.get(key, 0) + 1
    return groups


def cpu_baseline(specs, method="standard"):
    """The fp64 oracle on the host cores over a bounded sample of the set:
    one parameter of every distinct (shape, split) of the set, each timed
    once; the step time of the whole set is extrapolated by the number of
    parameters of each shape (each shape's oracle time scales with its
    count), and the value is the set's NS flops over that time."""
    from newton_schulz_orthogonalized_muon_gb300 import flops
    rows, step_s, step_f, sample_s = [], 0.0, 0.0, 0.0
    for (shape, split), count in sorted(set_groups(specs).items()):
        t = oracle_matrix_seconds(shape, split, method)
        m, n = flops.ns_dims(shape[0], shape[1], split)
        f = split * flops.ns_flops(method, m, n, NS_STEPS)
        rows.append({"shape": list(shape), "split_heads": split, "count": count, "seconds_one": round(t, 3)})
        step_s += count * t
        step_f += count * f
        sample_s += t
    return {"value": step_f / step_s / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"one parameter of each of the set's {len(rows)} distinct shapes, timed once each "
                      f"({sample_s:.1f} s); the full step extrapolated by shape counts to {step_s:.0f} s",
            "extrapolated_step_s": step_s, "sample_seconds": round(sample_s, 2), "per_shape": rows,
            "cpu": cpu_model(), "ns_method": method}


def cpu_baseline_plan():
    """The fp64 oracle on the host cores over the five configurations:
    the single 256x512 fp32 matrix, the GPT-2-small set (three steps) and
    the wide sweep's m <= 1024 shapes (both methods) in full; the sweep's
    m = 2048 shapes on 4 of 64 matrices and the Llama-3-8B and Moonlight-MoE
    sets on one layer, extrapolated by matrix count (labelled)."""
    from newton_schulz_orthogonalized_muon_gb300 import flops, workloads as wl
    out = {"cpu": cpu_model(), "blas_threads": blas_threads(), "rows": []}

    def add(name, specs, reps, scale, method="standard", note="full"):
        t = 0.0
        for _ in range(reps):
            for i, s_ in enumerate(specs):
                t += oracle_matrix_seconds(s_.shape, s_.split_heads, method, seed=i)
        f = reps * sum(s_.split_heads * flops.ns_flops(method, *flops.ns_dims(s_.shape[0], s_.shape[1], s_.split_heads),
                                                       NS_STEPS) for s_ in specs)
        out["rows"].append({"config": name, "method": method, "timed_s": round(t, 2), "timed_tflops": f / t / 1e12,
                            "step_s": t * scale / reps, "timing": note})
        print(json.dumps(out["rows"][-1]), flush=True)

    add("single fp32 256x512", wl.single_matrix_256x512().muon, 1, 1)
    add("gpt2-small (3 steps)", wl.gpt2_small().muon, 3, 1, note="full, step_s per step")
    for m, n in wl.WIDE_SWEEP:
        for method in ("standard", "gram"):
            spec = [wl.ParamSpec(f"w{m}x{n}", (m, n))]
            if m <= 1024:
                add(f"wide {m}x{n} x{wl.WIDE_BATCH}", spec * wl.WIDE_BATCH, 1, 1, method)
            else:
                add(f"wide {m}x{n} x{wl.WIDE_BATCH}", spec * 4, 1, wl.WIDE_BATCH / 4, method,
                    note=f"4 of {wl.WIDE_BATCH} matrices timed, extrapolated x{wl.WIDE_BATCH // 4}")
    for method in ("standard", "gram"):
        add("llama3-8b", wl.llama3_8b(1).muon, 1, 32, method, note="one layer timed, extrapolated x32")
    add("moonlight-moe", wl.moonlight_moe(1).muon, 1, 27, note="one layer timed, extrapolated x27")
    print(json.dumps(out), flush=True)
    return 0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample_step()
    t_sum, f_sum = 0.0, 0.0
    for _ in range(args.steps):
        t, f = oracle_sample_step()
        t_sum += t
        f_sum += f
    value = f_sum / t_sum / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_sum / max(args.steps, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": "llama3-8b (bounded CPU sample: one k_proj-shaped 1024x4096 matrix per step)",
                      "ns_method": "standard", "ns_steps": NS_STEPS},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                            "sample": SAMPLE_TEXT + " per step"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import flops

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    ws = weight_set(args.workload, args.layers)
    specs, _ = owned_specs(ws, world, rank)
    fp32 = param_dtype(args) == "fp32"
    W, G, M = make_inputs(specs, dev, args.seed + 7919 * rank, dtype=torch.float32 if fp32 else torch.bfloat16,
                          rank=ws.grad_rank)
    split = [s.split_heads for s in specs]
    h = pkg.default_handle(local)
    h.set_workspace_limit(int(args.workspace_gb * (1 << 30)))
    stream = torch.cuda.current_stream()

    def step(grads=None):
        pkg.muon_step(W, grads or G, M, lr=LR, wd=WD, mu=MU, nesterov=True, ns_method=args.ns_method,
                      ns_steps=NS_STEPS, split_heads=split, handle=h)

    for _ in range(args.warmup):
        step()
    barrier()
    if h.check() != 0:
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    # timed region 1 (the headline): the steps alone
    launches0 = h.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    launches = h.launch_count() - launches0
    # timed region 2: the same number of steps with a CUDA event pair around
    # every launch on the launching stream (per-kernel times for the rows and
    # the roofline; the events cost time between small launches)
    h.set_profiling(True)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e2.record(stream)
    for _ in range(args.steps):
        step()
    e3.record(stream)
    barrier()
    ms_profiled = e2.elapsed_time(e3) / max(args.steps, 1)
    records = h.profile_records()
    h.set_profiling(False)
    clk = clocks.stop()
    status = h.check()
    if status != 0:
        raise RuntimeError(f"device error during the timed region: status {status}")

    method = args.ns_method
    alg, dense = flops.set_flops(specs, NS_STEPS, method)
    alg_std, _ = flops.set_flops(specs, NS_STEPS, "standard")
    if world > 1:
        t = torch.tensor([ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
        f = torch.tensor([alg, dense, alg_std], device=dev, dtype=torch.float64)
        dist.all_reduce(f, op=dist.ReduceOp.SUM)
        alg_all, dense_all, alg_std_all = float(f[0]), float(f[1]), float(f[2])
    else:
        ms_max, alg_all, dense_all, alg_std_all = ms, alg, dense, alg_std
    # the method's own algorithmic flops (standard: symmetric products on one
    # triangle; gram: R0, the m x m iteration and O = Q X0)
    value = alg_all / (ms_max / 1e3) / 1e12

    # ---- per kernel class and per (class, same-shape group), timed live above
    peaks, peak_src = load_peaks()
    groups = {}
    for s_ in specs:
        mn = flops.ns_dims(s_.shape[0], s_.shape[1], s_.split_heads)
        groups[mn] = groups.get(mn, 0) + s_.split_heads
    group_list = sorted(groups.items())            # the library's group order: ascending (m, n)
    iters = flops.kernel_launches(method, NS_STEPS)
    kernel_rows, per_group = {}, {}
    for k, tag, kms in records:
        row = kernel_rows.setdefault(k, {"ms_per_step": 0.0, "launches_per_step": 0.0})
        row["ms_per_step"] += kms / args.steps
        row["launches_per_step"] += 1.0 / args.steps
        if k in iters and 0 <= tag < len(group_list):
            key = (k, tag)
            e = per_group.setdefault(key, [0.0, 0])
            e[0] += kms
            e[1] += 1
    class_flops = {k: 0.0 for k in iters}
    group_rows = []
    for (k, tag), (kms, cnt) in sorted(per_group.items(), key=lambda x: -x[1][0]):
        (m, n), count = group_list[tag]
        kf = flops.kernel_flops(method, m, n)[k]
        fl = count * iters[k] * args.steps * kf
        class_flops[k] += fl
        row = {"kernel": k, "mode": kernel_mode(method, k, fp32), "group": f"{m}x{n}", "matrices": count, "launches": cnt,
               "ms_per_launch": kms / cnt, "flops_per_launch": fl / cnt, "tflops": fl / (kms / 1e3) / 1e12}
        if method == "gram" and not fp32:
            # tensor-core work: bf16x3 m x m products, two-plane final product
            row["mma_tflops"] = row["tflops"] * flops.kernel_mma_factor_gram()[k]
        elif fp32 and method == "standard" and m <= F32_TC_MAX_M:
            # three-plane operands: six bf16 MMAs per product
            row["mma_tflops"] = row["tflops"] * 6.0
        group_rows.append(row)
    for k, row in kernel_rows.items():
        if k in class_flops and row["ms_per_step"] > 0:
            row["tflops"] = class_flops[k] / (row["ms_per_step"] * args.steps / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    roofline = None
    if group_rows:
        top = group_rows[0]          # the (class, group) with the most time
        traffic = None
        tpath = os.path.join(ROOT, "profiles", "traffic.json")
        if os.path.exists(tpath):
            try:
                entry = json.load(open(tpath)).get(ws.name, {}).get(f"{top['mode']}@{top['group']}")
                if entry and entry.get("kernel_source_hash") == kernel_source_hash():
                    # per-matrix traffic (each matrix's tiles touch only that
                    # matrix) times this launch's matrices
                    traffic = entry["bytes_per_launch"] * top["matrices"] / entry.get("matrices", top["matrices"])
            except Exception:
                traffic = None
        m_top = int(top["group"].split("x")[0])
        if fp32:
            # the fp32 path's standard method runs on the tensor cores up to m = 2048
            kname = "ns_gemm_tc_kernel" if (method == "standard" and m_top <= F32_TC_MAX_M) else "ns_gemm_simt_kernel"
        else:
            kname = "ns_gemm_pair_kernel" if uses_pairs(m_top, top["kernel"], method) else "ns_gemm_tc_kernel"
        roofline = {"bound": "tensor", "kernel": f"{kname}<{top['mode']}> on the {top['group']} group "
                                                  f"({top['matrices']} matrices)",
                    "achieved": top["tflops"], "peak": peak, "unit": "TFLOP/s", "frac": top["tflops"] / peak,
                    "traffic": traffic, "flops_per_launch": top["flops_per_launch"],
                    "ms_per_launch": top["ms_per_launch"], "peak_source": f"bf16_tflops_sustained, {peak_src}",
                    "flops_model": "algorithmic" if method == "standard" and not fp32 else
                                   "algorithmic (one product per plane-split product; mma_tflops counts every MMA)"}
        if "mma_tflops" in top:
            roofline["mma_tflops"] = top["mma_tflops"]
    hbm = None
    if "prepare" in kernel_rows:
        nb = sum(flops.prepare_bytes(s.shape[0] * s.shape[1]) for s in specs)
        gbs = nb / (kernel_rows["prepare"]["ms_per_step"] / 1e3) / 1e9
        hbm = {"bound": "hbm", "kernel": "muon_prepare_kernel", "achieved": gbs, "peak": peaks["hbm_gbs"],
               "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "bytes_per_step": nb}
        # per same-shape group (the transposed parameters' groups write X through shared memory)
        pg = {}
        for k, tag, kms in records:
            if k == "prepare" and 0 <= tag < len(group_list):
                pg[tag] = pg.get(tag, 0.0) + kms
        rows = []
        for tag, kms in sorted(pg.items()):
            (m, n), count = group_list[tag]
            gb = flops.prepare_bytes(count * m * n)
            g_gbs = gb / (kms / args.steps / 1e3) / 1e9
            rows.append({"group": f"{m}x{n}", "matrices": count, "ms_per_step": kms / args.steps, "achieved": g_gbs,
                         "frac": g_gbs / peaks["hbm_gbs"]})
        if rows:
            hbm["groups"] = rows

    # ---- AdamW fallback over the set's AdamW parameters (embeddings, norms)
    adamw = None
    if not args.no_adamw and ws.adamw:
        adamw = run_adamw(args, ws, dev, stream, h, peaks)

    # ---- end to end through the public API: pinned host grads in, params out
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e_bounded(args, W, G, M, specs, split, h, dev, stream, alg_all, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(specs, method)

    # ---- the other configurations, after the headline's timed regions (one
    # GPU, default workload only): the Gram method on the same inputs, then
    # the small sets and the MoE set on fresh inputs
    others = None
    if world == 1 and not args.no_other_configs and args.workload == "llama3-8b" and args.layers is None \
            and method == "standard" and not fp32:
        others = {"llama3-8b gram": time_config(h, W, G, M, specs, "gram", args, peaks)}
        del W, G, M
        torch.cuda.empty_cache()
        others.update(other_configs(args, h, dev, peaks))

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f32" if fp32 else "bf16", "data": "synthetic",
               "config": {"workload": ws.name, "ns_method": args.ns_method, "ns_steps": NS_STEPS,
                          "muon_params_per_gpu": sum(s.shape[0] * s.shape[1] for s in specs),
                          "matrices_per_gpu": len(specs), "l2": "inputs larger than L2 (no flush needed)",
                          "lr": LR, "wd": WD, "mu": MU, "nesterov": True,
                          "param_dtype": param_dtype(args),
                          "ns_path": ("fp32 on the tensor cores: three-plane bf16 operands, six MMAs per product"
                                      if fp32 and method == "standard" else
                                      "fp32 on the CUDA cores" if fp32 else "bf16 tensor cores"),
                          "parallelism": f"layer-wise ownership x{world}" if world > 1 else "single GPU"},
               "step_ms": ms_max, "ms_per_step_with_launch_events": ms_profiled,
               "ns_tflops_dense_convention": dense_all / (ms_max / 1e3) / 1e12,
               "ns_flops_model": "standard algorithmic" if method == "standard" else "gram algorithmic",
               "ns_tflops_standard_equivalent": alg_std_all / (ms_max / 1e3) / 1e12,
               "ns_frac_of_peak": value / peak, "roofline": roofline, "roofline_hbm": hbm,
               "kernels": kernel_rows, "kernel_groups": group_rows, "gpu_launches": launches, "clocks": clk, "e2e": e2e, "adamw": adamw,
               "cpu_baseline": cpu, "other_configs": others}
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_config(h, W, G, M, specs, method, args, peaks, steps=3, warmup=3):
    """Compact timing of one configuration on given device tensors: warm-up,
    then `steps` steps bracketed by CUDA events (no per-launch events), then
    the same number of steps with per-launch events for the per-class rates.
    Returns step ms, the method's algorithmic NS TFLOP/s, its fraction of the
    measured sustained peak, per-class ms and TFLOP/s, and the clocks."""
    import torch
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import flops
    split = [s_.split_heads for s_ in specs]
    fp32 = W[0].dtype == torch.float32

    def step():
        pkg.muon_step(W, G, M, lr=LR, wd=WD, mu=MU, nesterov=True, ns_method=method, ns_steps=NS_STEPS,
                      split_heads=split, handle=h)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h.set_profiling(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    prof = h.profile()
    h.set_profiling(False)
    clk = clocks.stop()
    if h.check() != 0:
        raise RuntimeError(f"device error while timing the {method} configuration")
    alg, _ = flops.set_flops(specs, NS_STEPS, method)
    classes = {}
    per_class = {k: 0.0 for k in ("syrk", "poly", "update", "final")}
    it = flops.kernel_launches(method, NS_STEPS)
    for s_ in specs:
        m, n = flops.ns_dims(s_.shape[0], s_.shape[1], s_.split_heads)
        kf = flops.kernel_flops(method, m, n)
        for k in per_class:
            per_class[k] += s_.split_heads * it[k] * kf[k]
    for k, (kms, cnt) in prof.items():
        if cnt:
            row = {"ms_per_step": kms / steps}
            if k in per_class and kms > 0:
                row["tflops"] = per_class[k] / (kms / steps / 1e3) / 1e12
            classes[k] = row
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    value = alg / (ms / 1e3) / 1e12
    return {"ms_per_step": ms, "value": value, "unit": UNIT, "ns_frac_of_sustained_peak": value / peak,
            "ns_method": method, "dtype": "f32" if fp32 else "bf16", "steps": steps, "warmup": warmup,
            "kernels": classes, "clocks": clk}


def other_configs(args, h, dev, peaks):
    """The small sets (GPT-2-small in bf16 and fp32, the single fp32 256x512
    matrix) and the Moonlight-like MoE set, each on fresh seeded inputs,
    timed compactly after the headline."""
    import torch
    out = {}
    for name, wname, dtype in (("gpt2-small", "gpt2-small", torch.bfloat16),
                               ("gpt2-small fp32", "gpt2-small", torch.float32),
                               ("single fp32 256x512", "single-fp32", torch.float32),
                               ("moonlight-moe", "moonlight-moe", torch.bfloat16)):
        ws = weight_set(wname)
        specs = list(ws.muon)
        W, G, M = make_inputs(specs, dev, args.seed, dtype=dtype, rank=ws.grad_rank)
        out[name] = time_config(h, W, G, M, specs, "standard", args, peaks, steps=3 if wname == "moonlight-moe" else 10)
        del W, G, M
        torch.cuda.empty_cache()
    return out


def run_adamw(args, ws, dev, stream, h, peaks):
    """Time adamw_step over the weight set's AdamW parameters (bf16 params and
    grads, fp32 moments), HBM-bound: 22 algorithmic bytes per element."""
    import torch
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import flops
    gen = torch.Generator(device=dev)
    gen.manual_seed(12345)
    P = [torch.randn(s.shape, generator=gen, device=dev).mul_(0.02).to(torch.bfloat16) for s in ws.adamw]
    G = [torch.randn(s.shape, generator=gen, device=dev).mul_(1e-3).to(torch.bfloat16) for s in ws.adamw]
    Mm = [torch.zeros(s.shape, device=dev) for s in ws.adamw]
    V = [torch.zeros(s.shape, device=dev) for s in ws.adamw]
    kw = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, handle=h)
    for t in range(1, 4):
        pkg.adamw_step(P, G, Mm, V, step=t, **kw)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(args.steps, 3)
    e0.record(stream)
    for t in range(4, 4 + steps):
        pkg.adamw_step(P, G, Mm, V, step=t, **kw)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    numel = sum(p.numel() for p in P)
    nb = flops.adamw_bytes(numel, 2, 2)
    gbs = nb / (ms / 1e3) / 1e9
    out = {"kernel": "adamw_kernel", "tensors": len(P), "numel": numel, "ms_per_step": ms, "bytes_per_step": nb,
           "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}
    del P, G, Mm, V
    torch.cuda.empty_cache()
    return out


def e2e_slices(specs, param_bytes, limit=None, last_limit=None):
    """The muon_step calls of one pipelined e2e step: parameter indices grouped
    by the library's same-shape groups (NS dims after the transpose and
    Muon-Split rules, in ascending (m, n) order, the library's own order),
    each group cut into consecutive slices of at most `limit` bytes of
    parameters (at least one matrix per slice).  The step's read-back of the
    last slice is the one copy not overlapped with compute, so the last
    group ends with a slice of at most `last_limit` bytes."""
    from newton_schulz_orthogonalized_muon_gb300 import flops
    limit = E2E_SLICE_BYTES if limit is None else limit
    last_limit = E2E_LAST_SLICE_BYTES if last_limit is None else last_limit
    by_group = {}
    for i, s_ in enumerate(specs):
        by_group.setdefault(flops.ns_dims(s_.shape[0], s_.shape[1], s_.split_heads), []).append(i)
    order = []
    keys = sorted(by_group)
    for key in keys:
        members = by_group[key]
        tail = []
        if key == keys[-1] and sum(param_bytes[i] for i in members) > last_limit:
            # the final slice: matrices from the group's end, up to last_limit bytes (at least one)
            nbytes = 0
            while members and (not tail or nbytes + param_bytes[members[-1]] <= last_limit) \
                    and len(tail) < len(by_group[key]) - 1:
                nbytes += param_bytes[members[-1]]
                tail.insert(0, members[-1])
                members = members[:-1]
        cur, nbytes = [], 0
        for i in members:
            if cur and nbytes + param_bytes[i] > limit:
                order.append(cur)
                cur, nbytes = [], 0
            cur.append(i)
            nbytes += param_bytes[i]
        if cur:
            order.append(cur)
        if tail:
            order.append(tail)
    return order


def host_link(dev, stream):
    """This machine's host link as the e2e loop meets it: one 1 GiB copy each
    way between a pinned buffer and the device (best of three), and where the
    GPU sits (its PCI address, NUMA node and local CPUs from sysfs) against
    the CPUs this process may run on.  Host-to-device rates measured 33 GB/s
    on some machines and 210 GB/s on others for the same program."""
    import subprocess
    import torch
    out = {}
    n = 1 << 29
    hb = torch.ones(n, dtype=torch.bfloat16, pin_memory=True)
    db = torch.empty(n, dtype=torch.bfloat16, device=dev)
    for name, fn in (("h2d_gbs_1gib", lambda: db.copy_(hb, non_blocking=True)),
                     ("d2h_gbs_1gib", lambda: hb.copy_(db, non_blocking=True))):
        best = 0.0
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            best = max(best, 2 * n / (a.elapsed_time(b) / 1e3) / 1e9)
        out[name] = best
    del hb, db
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={dev.index or 0}", "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20).stdout.strip()
        out["gpu_pci"] = bus
        sysdir = "/sys/bus/pci/devices/" + bus.lower()[-12:]
        for key, fname in (("gpu_numa_node", "numa_node"), ("gpu_local_cpus", "local_cpulist")):
            if os.path.exists(os.path.join(sysdir, fname)):
                out[key] = open(os.path.join(sysdir, fname)).read().strip()
    except Exception:
        pass
    try:
        out["process_cpus"] = len(os.sched_getaffinity(0))
    except Exception:
        pass
    return out


def host_memory_bytes():
    """Physical memory of this machine (Linux), or None."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemTotal:"):
                return int(line.split()[1]) * 1024
    except Exception:
        pass
    return None


def e2e_subset(specs, param_bytes, frac):
    """Indices of the first ceil-down fraction `frac` (at least one) of each
    same-shape group's matrices, in the library's group order."""
    keep = []
    for idx in e2e_slices(specs, param_bytes, limit=1 << 62, last_limit=1 << 62):
        keep += idx[:max(1, int(len(idx) * frac))]
    return sorted(keep)


def run_e2e_bounded(args, W, G, M, specs, split, h, dev, stream, alg_all, world):
    """run_e2e over the whole set when its host buffers (gradients in,
    parameters out: twice the set's gradient bytes per rank) fit in half of
    the machine's memory shared by the ranks on it; otherwise over the first
    matrices of each same-shape group, the same fraction of every group, with
    the flop count of that subset summed over the ranks, and the fraction in
    the result (several ranks of a large set on one machine)."""
    import torch
    need = 2 * sum(g.numel() * g.element_size() for g in G) + (1 << 30)
    local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    mem = host_memory_bytes()
    if mem is None or need <= 0.5 * mem / max(local, 1):
        return run_e2e(args, W, G, M, specs, split, h, dev, stream, alg_all, world)
    frac = 0.5 * mem / max(local, 1) / need
    keep = e2e_subset(specs, [w.numel() * w.element_size() for w in W], frac)
    from newton_schulz_orthogonalized_muon_gb300 import flops
    sub = [specs[i] for i in keep]
    alg, _ = flops.set_flops(sub, NS_STEPS, args.ns_method)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([alg], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        alg = float(t.item())
    out = run_e2e(args, [W[i] for i in keep], [G[i] for i in keep], [M[i] for i in keep], sub,
                  [split[i] for i in keep], h, dev, stream, alg, world)
    out["subset"] = {"matrices_per_rank": len(keep), "of": len(specs), "reason":
                     f"host memory: {need / 1e9:.0f} GB of buffers per rank against {mem / 1e9:.0f} GB shared by "
                     f"{local} ranks"}
    return out


class HostBuffer:
    """Page-locked host memory for the e2e buffers: an anonymous mapping
    advised for transparent huge pages (madvise MADV_HUGEPAGE), touched by the
    CPU and registered with cudaHostRegister, so the copy engine walks 2 MiB
    pages; torch's pinned allocator (the system's base pages) if any step
    fails.  Some machines moved 14 GB from base-page pinned memory at 32-43 GB/s
    while a 1 GiB buffer ran at 211 GB/s."""

    def __init__(self, numel, dtype):
        import ctypes
        import mmap
        import torch
        self.addr = None
        nbytes = max(int(numel) * torch.empty((), dtype=dtype).element_size(), 1)
        try:
            libc = ctypes.CDLL("libc.so.6", use_errno=True)
            buf = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            addr = ctypes.addressof(ctypes.c_char.from_buffer(buf))
            libc.madvise(ctypes.c_void_p(addr), ctypes.c_size_t(nbytes), 14)     # MADV_HUGEPAGE
            t = torch.frombuffer(buf, dtype=dtype, count=int(numel))
            t.zero_()
            rc = torch.cuda.cudart().cudaHostRegister(addr, nbytes, 0)
            if int(getattr(rc, "value", rc)) != 0 or not t.is_pinned():
                raise RuntimeError("cudaHostRegister failed")
            self.buf, self.addr, self.tensor, self.kind = buf, addr, t, "huge-page mapping, cudaHostRegister"
        except Exception:
            self.tensor = torch.empty(int(numel), dtype=dtype, pin_memory=True)
            self.kind = "torch pinned memory"

    def release(self):
        import torch
        if self.addr is not None:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaHostUnregister(self.addr)
            self.addr = None
        self.tensor = None


def run_e2e(args, W, G, M, specs, split, h, dev, stream, alg_all, world):
    """Same step through the public API with host buffers: every step copies
    its gradients host->device from pinned memory and reads the updated
    parameters back device->host.

    "pipelined" (the reported value): the step is issued as several
    muon_step calls, one per slice of at most E2E_SLICE_BYTES of parameters
    within a same-shape group, groups in the library's order (ascending
    (m, n)); the gradients of step k+1 are copied in on one side stream, one
    copy per slice, while step k computes (a call waits for its own slice's
    gradients only), and each slice's parameters are read back on another
    side stream as soon as that slice's call has finished, while the later
    slices compute.  Step k+1's call for a slice waits for the read-back of
    the same slice from step k (it overwrites those parameters), so no device
    snapshot is needed and only the last slice's read-back is exposed.  Every
    step's copies are inside the timed region.  "serial": copy in, step, copy
    out, one after the other on one stream."""
    import torch
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    # one contiguous pinned allocation per direction, viewed per tensor: many
    # separate pinned blocks measured far slower on their first copy after a
    # pause (27-81 GB/s against ~210 GB/s for one large buffer)
    host_bufs = []

    def pinned_views(like):
        hb = HostBuffer(sum(t.numel() for t in like), like[0].dtype)
        host_bufs.append(hb)
        flat = hb.tensor
        views, off = [], 0
        for t in like:
            views.append(flat[off:off + t.numel()].view(t.shape))
            off += t.numel()
        return views
    link = host_link(dev, stream)
    # the gradients: one pinned host buffer and two device buffers, each laid
    # out in the calls' slice order, so that a step's host-to-device transfer
    # is one copy (per-tensor copies of the same bytes ran at 33-43 GB/s on
    # machines whose link moved a 1 GiB buffer at 211 GB/s)
    order = e2e_slices(specs, [w.numel() * w.element_size() for w in W])
    seq = [i for idx in order for i in idx]
    total = sum(G[i].numel() for i in seq)
    ghb = HostBuffer(total, G[0].dtype)
    host_bufs.append(ghb)
    gh_flat = ghb.tensor
    gd_flat = [torch.empty(total, dtype=G[0].dtype, device=dev) for _ in range(2)]
    Gh, Gd = [None] * len(G), [[None] * len(G), [None] * len(G)]
    off = 0
    for i in seq:
        n = G[i].numel()
        Gh[i] = gh_flat[off:off + n].view(G[i].shape)
        for q in range(2):
            Gd[q][i] = gd_flat[q][off:off + n].view(G[i].shape)
        off += n
    for i in seq:
        Gh[i].copy_(G[i])
    Wh = pinned_views(W)
    torch.cuda.synchronize()
    h2d = sum(g.numel() * g.element_size() for g in G)
    d2h = sum(w.numel() * w.element_size() for w in W)
    steps = max(1, args.steps)

    # element range of each slice in the flat layout
    bounds, off = [], 0
    for idx in order:
        n = sum(G[i].numel() for i in idx)
        bounds.append((off, off + n))
        off += n

    def copy_in(q, gi=None):
        if gi is None:
            gd_flat[q].copy_(gh_flat, non_blocking=True)
        else:
            a, b = bounds[gi]
            gd_flat[q][a:b].copy_(gh_flat[a:b], non_blocking=True)

    # diagnostic: the same bytes as one copy per tensor, once, outside the timed loops
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record(stream)
    for i in seq:
        Gd[1][i].copy_(Gh[i], non_blocking=True)
    b_.record(stream)
    torch.cuda.synchronize()
    link["h2d_gbs_per_tensor_copies"] = h2d / (a_.elapsed_time(b_) / 1e3) / 1e9

    def step(grads):
        pkg.muon_step(W, grads, M, lr=LR, wd=WD, mu=MU, nesterov=True, ns_method=args.ns_method, ns_steps=NS_STEPS,
                      split_heads=split, handle=h)

    # serial
    # events around the copies of the serial variant: the host-link rates the
    # e2e figure is bounded by (they differ from machine to machine)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]

    def serial_one(marks=None):
        if marks:
            marks[0].record(stream)
        copy_in(0)
        if marks:
            marks[1].record(stream)
        step(Gd[0])
        if marks:
            marks[2].record(stream)
        for wh, wd in zip(Wh, W):
            wh.copy_(wd, non_blocking=True)
        if marks:
            marks[3].record(stream)

    serial_one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        serial_one(ev[k])
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / steps
    h2d_ms = sum(m[0].elapsed_time(m[1]) for m in ev) / steps
    d2h_ms = sum(m[2].elapsed_time(m[3]) for m in ev) / steps

    # pipelined: two device gradient buffers; calls per slice of a same-shape group
    gbuf = Gd
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # per buffer and slice: that slice's gradients have arrived, so a step's
    # first call waits for its own slice only
    in_done = [[torch.cuda.Event() for _ in order] for _ in range(2)]
    group_done = [torch.cuda.Event() for _ in order]
    out_done = [torch.cuda.Event() for _ in order]
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    with torch.cuda.stream(s_in):
        for gi in range(len(order)):
            copy_in(0, gi)
            in_done[0][gi].record(s_in)
    for k in range(steps):
        cur = gbuf[k % 2]
        if k + 1 < steps:                               # next step's gradients, overlapped
            with torch.cuda.stream(s_in):
                if k >= 1:
                    s_in.wait_event(step_done_prev)     # the buffer was read by step k-1
                for gi in range(len(order)):
                    copy_in((k + 1) % 2, gi)
                    in_done[(k + 1) % 2][gi].record(s_in)
        for gi, idx in enumerate(order):
            stream.wait_event(in_done[k % 2][gi])       # this slice's gradients are in
            if k >= 1:
                stream.wait_event(out_done[gi])         # step k-1's parameters of this group are read back
            pkg.muon_step([W[i] for i in idx], [cur[i] for i in idx], [M[i] for i in idx], lr=LR, wd=WD, mu=MU,
                          nesterov=True, ns_method=args.ns_method, ns_steps=NS_STEPS,
                          split_heads=[split[i] for i in idx], handle=h)
            group_done[gi].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(group_done[gi])
                for i in idx:
                    Wh[i].copy_(W[i], non_blocking=True)
                out_done[gi].record(s_out)
        step_done_prev = torch.cuda.Event()
        step_done_prev.record(stream)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_clk = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms, serial_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, serial_ms = float(t[0]), float(t[1])
    # this rank's host-link rates (serial copies), then the whole job's bytes
    h2d_gbs, d2h_gbs = h2d / (h2d_ms / 1e3) / 1e9, d2h / (d2h_ms / 1e3) / 1e9
    if world > 1:
        nbytes = torch.tensor([h2d, d2h], device=dev, dtype=torch.float64)
        dist.all_reduce(nbytes, op=dist.ReduceOp.SUM)
        h2d, d2h = int(nbytes[0]), int(nbytes[1])
    kinds = sorted({hb.kind for hb in host_bufs})
    del gd_flat, Gd, gbuf, Gh, Wh, gh_flat
    for hb in host_bufs:
        hb.release()
    torch.cuda.empty_cache()
    return {"value": alg_all / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "mode": f"pipelined (copies overlapped with compute; {len(order)} calls per step, one per slice of at most "
                    f"{E2E_SLICE_BYTES >> 30} GiB of parameters of one same-shape group; the gradients in one "
                    f"host-to-device copy per slice, the parameters read back per tensor)",
            "serial_ms_per_step": serial_ms, "serial_value": alg_all / (serial_ms / 1e3) / 1e12,
            "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "host_link": link, "host_buffers": kinds, "clocks": e2e_clk}


def param_dtype(args):
    return args.param_dtype or ("fp32" if args.workload == "single-fp32" else "bf16")


def kernel_mode(method, kernel_class, fp32=False):
    """The kernel mode behind a reported kernel class (bf16 parameters, whose
    last product writes through tensor maps)."""
    if fp32:
        if method == "gram":
            return {"syrk": "G_R0", "poly": "G_P", "update": "G_PROD", "final": "G_FINAL"}[kernel_class]
        return {"syrk": "F_SYRK", "poly": "F_POLY", "update": "F_UPDATE", "final": "F_FINAL"}[kernel_class]
    if method == "gram":
        return {"syrk": "G_R0", "poly": "G_P", "update": "G_PROD", "final": "G_FINAL_T"}[kernel_class]
    return {"syrk": "SYRK", "poly": "POLY", "update": "UPDATE", "final": "FINAL_T"}[kernel_class]


def uses_pairs(m, kernel_class, method="standard"):
    """The library's rule for which products run on the CTA-pair kernels.
    A group uses pairs when m >= MUON_TC_PAIR_MIN_M (1024 by default) or
    m = 256.  Standard method: its symmetric products then; UPDATE / FINAL
    when, in addition, m is a multiple of 256 or m >= 2048.  Gram method: its
    symmetric products (R0, P, the m x m products), and O = Q X0 into bf16
    destinations by the UPDATE rule.  None with MUON_TC_PAIR=0, symmetric
    products only with MUON_TC_PAIR=sym."""
    env = os.environ.get("MUON_TC_PAIR")
    if env == "0" or m < 256:
        return False
    try:
        min_m = int(os.environ.get("MUON_TC_PAIR_MIN_M", "1024"))
    except ValueError:
        min_m = 1024
    if not (m >= min_m or m == 256):
        return False
    if (method == "standard" and kernel_class in ("update", "final")) or (method == "gram" and kernel_class == "final"):
        return env != "sym" and (m % 256 == 0 or m >= 2048)
    return True


def kernel_source_hash():
    import hashlib
    hsh = hashlib.sha256()
    for f in ("kernels_tc.cu", "kernels_tc2.cu", "tc_common.cuh", "common.cuh", "internal.h"):
        hsh.update(open(os.path.join(ROOT, "newton_schulz_orthogonalized_muon_gb300", "csrc", f), "rb").read())
    return hsh.hexdigest()[:16]


def run_wide(args):
    """Standard vs Gram Newton-Schulz on batches of 64 Gaussian bf16 matrices
    per (m, n); time per batch and relative error of one sampled matrix
    against the fp64 oracle (= the SVD closed form)."""
    import numpy as np
    import torch
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import flops, workloads as wl
    import oracle
    torch.cuda.set_device(0)
    h = pkg.default_handle(0)
    h.set_workspace_limit(int(args.workspace_gb * (1 << 30)))
    rows = []
    for m, n in wl.WIDE_SWEEP:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(wl.matrix_seed(7, m * 100000 + n))
        X = torch.randn(wl.WIDE_BATCH, m, n, generator=gen, device="cuda").to(torch.bfloat16)
        ref = oracle.newton_schulz(X[0].double().cpu().numpy())
        row = {"m": m, "n": n, "batch": wl.WIDE_BATCH}
        for method in ("standard", "gram"):
            Y = X.clone()
            for _ in range(max(args.warmup, 1)):
                Y.copy_(X)
                pkg.muon_orthogonalize(Y, ns_method=method, handle=h)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ms = 0.0
            for _ in range(args.steps):
                Y.copy_(X)
                e0.record()
                pkg.muon_orthogonalize(Y, ns_method=method, handle=h)
                e1.record()
                torch.cuda.synchronize()
                ms += e0.elapsed_time(e1)
            ms /= args.steps
            got = Y[0].double().cpu().numpy()
            f = flops.ns_flops_standard(m, n) if method == "standard" else flops.ns_flops_gram(m, n)
            row[method] = {"ms": ms, "tflops_algorithmic": wl.WIDE_BATCH * f / (ms / 1e3) / 1e12,
                           "rel_err_vs_fp64": float(np.linalg.norm(got - ref) / np.linalg.norm(ref))}
            del Y
        row["gram_speedup"] = row["standard"]["ms"] / row["gram"]["ms"]
        rows.append(row)
        del X
        torch.cuda.empty_cache()
    if h.check() != 0:
        raise RuntimeError("device error during the sweep")
    print(json.dumps({"workload": "wide-sweep", "unit": "ms per batch of 64", "rows": rows}), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_plan:
        return cpu_baseline_plan()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "wide":
        return run_wide(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
