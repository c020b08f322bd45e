"""ctypes binding of libmuon_gb300.so (argument marshalling only).

Every entry point mirrors the C ABI in include/muon.h: it checks that the
torch tensors it is given are CUDA, contiguous and of a supported dtype,
passes their device pointers and the current CUDA stream, and raises
MuonError on a non-OK status.  All arithmetic runs in the library's kernels;
if the library is missing this module raises instead of computing anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB_PATH

MUON_F32, MUON_BF16 = 0, 1
MUON_NS_STANDARD, MUON_NS_GRAM, MUON_NS_AUTO = 0, 1, 2
MUON_SCALE_RMS, MUON_SCALE_MUP = 0, 1
QUINTIC = (3.4445, -4.7750, 2.0315)

_STATUS = {0: "MUON_OK", 1: "MUON_ERR_INVALID_ARG", 2: "MUON_ERR_UNSUPPORTED", 3: "MUON_ERR_WORKSPACE",
           4: "MUON_ERR_CUDA", 5: "MUON_ERR_NONFINITE", 6: "MUON_ERR_TIMEOUT"}

EXPORTS = ("muon_handle_create", "muon_handle_destroy", "muon_handle_set_workspace_limit",
           "muon_handle_set_timeout_ns", "muon_handle_check", "muon_orthogonalize", "muon_step",
           "adamw_step", "muon_selftest_timeout", "muon_status_string", "muon_last_error", "muon_version",
           "muon_handle_set_profiling", "muon_handle_profile", "muon_handle_launch_count",
           "muon_orthogonalize_noalloc", "muon_handle_profile_records", "muon_step_ex", "muon_workspace_size",
           "muon_noalloc_check", "muon_noalloc_set_timeout_ns")
KERNEL_CLASSES = ("prepare", "norm", "syrk", "poly", "update", "final", "apply", "adamw")


class MuonError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        self.name = _STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}: {detail}" if detail else self.name)


class MuonParamC(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("momentum", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("param_dtype", ctypes.c_int32),
                ("grad_dtype", ctypes.c_int32), ("split_heads", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("scale_dim", ctypes.c_int64)]


class MuonStepOptionsC(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("mu", ctypes.c_float), ("nesterov", ctypes.c_int32),
                ("ns_method", ctypes.c_int32), ("ns_steps", ctypes.c_int32),
                ("coeffs", ctypes.POINTER(ctypes.c_float)), ("ns_dtype", ctypes.c_int32),
                ("scale_mode", ctypes.c_int32), ("update_rms", ctypes.c_float), ("extra_scale", ctypes.c_float),
                ("coeffs_per_step", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load (once) and type the shared library; raise if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint64
        fptr = ctypes.POINTER(ctypes.c_float)
        sig = {
            "muon_handle_create": (i32, [ctypes.POINTER(vp), ctypes.c_int]),
            "muon_handle_destroy": (i32, [vp]),
            "muon_handle_set_workspace_limit": (i32, [vp, ctypes.c_size_t]),
            "muon_handle_set_timeout_ns": (i32, [vp, u64]),
            "muon_handle_check": (i32, [vp, vp]),
            "muon_orthogonalize": (i32, [vp, vp, i32, i64, i64, i64, i32, fptr, i32, vp]),
            "muon_step": (i32, [vp, ctypes.POINTER(MuonParamC), i32, f32, f32, f32, i32, i32, i32, fptr, f32,
                                i32, vp]),
            "adamw_step": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                 ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32), i32, i64, f32, f32, f32, f32, f32, vp]),
            "muon_selftest_timeout": (i32, [vp, u64, vp]),
            "muon_status_string": (ctypes.c_char_p, [i32]),
            "muon_last_error": (ctypes.c_char_p, [vp]),
            "muon_version": (i32, []),
            "muon_handle_set_profiling": (i32, [vp, i32]),
            "muon_handle_profile": (i32, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64), i32]),
            "muon_handle_launch_count": (i32, [vp, ctypes.POINTER(u64)]),
            "muon_orthogonalize_noalloc": (i32, [vp, i32, i64, i64, i32, fptr, vp]),
            "muon_noalloc_check": (i32, [vp]),
            "muon_noalloc_set_timeout_ns": (i32, [u64]),
            "muon_handle_profile_records": (i32, [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), fptr, i32,
                                                  ctypes.POINTER(i32)]),
            "muon_step_ex": (i32, [vp, ctypes.POINTER(MuonParamC), i32, ctypes.POINTER(MuonStepOptionsC), vp]),
            "muon_workspace_size": (i32, [vp, ctypes.POINTER(MuonParamC), i32, i32, i32, i32, ctypes.POINTER(u64)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MUON_F32
    if t.dtype == torch.bfloat16:
        return MUON_BF16
    raise ValueError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _need_cuda(t: torch.Tensor, what: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _coeffs(coeffs):
    c = QUINTIC if coeffs is None else tuple(float(x) for x in coeffs)
    if len(c) != 3:
        raise ValueError("coeffs must hold (a, b, c)")
    return (ctypes.c_float * 3)(*c)


def _method(ns_method) -> int:
    if ns_method in ("standard", MUON_NS_STANDARD):
        return MUON_NS_STANDARD
    if ns_method in ("gram", MUON_NS_GRAM):
        return MUON_NS_GRAM
    if ns_method in ("auto", MUON_NS_AUTO):
        return MUON_NS_AUTO
    raise ValueError(f"unknown ns_method {ns_method!r}")


class MuonHandle:
    """Owns the library's device workspace and error word on one GPU."""

    def __init__(self, device: int | None = None):
        self._lib = load_library()
        self.device = torch.cuda.current_device() if device is None else int(device)
        h = ctypes.c_void_p()
        st = self._lib.muon_handle_create(ctypes.byref(h), self.device)
        if st != 0:
            raise MuonError(st, "muon_handle_create")
        self._h = h

    def _raise(self, st: int, what: str):
        if st != 0:
            detail = self._lib.muon_last_error(self._h)
            raise MuonError(st, f"{what}: {detail.decode() if detail else ''}")

    @property
    def ptr(self):
        return self._h

    def set_workspace_limit(self, nbytes: int):
        self._raise(self._lib.muon_handle_set_workspace_limit(self._h, int(nbytes)), "set_workspace_limit")

    def set_timeout_ns(self, ns: int):
        self._raise(self._lib.muon_handle_set_timeout_ns(self._h, int(ns)), "set_timeout_ns")

    def check(self, stream=None) -> int:
        """Synchronise the stream and return the device error status (0 = OK)."""
        return int(self._lib.muon_handle_check(self._h, ctypes.c_void_p(_stream_ptr(stream))))

    def set_profiling(self, enable: bool):
        self._raise(self._lib.muon_handle_set_profiling(self._h, 1 if enable else 0), "set_profiling")

    def profile(self) -> dict:
        """Per kernel class: (total ms, launches) since profiling was enabled or last read."""
        n = len(KERNEL_CLASSES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        self._raise(self._lib.muon_handle_profile(self._h, ms, cnt, n), "profile")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_CLASSES)}

    def profile_records(self, capacity: int = 1 << 16):
        """[(kernel class, group tag, ms)] per recorded launch, then clear."""
        cls = (ctypes.c_int32 * capacity)()
        tag = (ctypes.c_int32 * capacity)()
        ms = (ctypes.c_float * capacity)()
        n = ctypes.c_int32()
        self._raise(self._lib.muon_handle_profile_records(self._h, cls, tag, ms, capacity, ctypes.byref(n)),
                    "profile_records")
        return [(KERNEL_CLASSES[cls[i]], int(tag[i]), float(ms[i])) for i in range(min(n.value, capacity))]

    def launch_count(self) -> int:
        c = ctypes.c_uint64()
        self._raise(self._lib.muon_handle_launch_count(self._h, ctypes.byref(c)), "launch_count")
        return int(c.value)

    def close(self):
        if getattr(self, "_h", None) is not None:
            self._lib.muon_handle_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_handles: dict[int, MuonHandle] = {}


def default_handle(device: int | None = None) -> MuonHandle:
    dev = torch.cuda.current_device() if device is None else int(device)
    if dev not in _handles:
        _handles[dev] = MuonHandle(dev)
    return _handles[dev]


def muon_orthogonalize(X: torch.Tensor, steps: int = 5, coeffs=None, ns_method="standard",
                       handle: MuonHandle | None = None, stream=None) -> torch.Tensor:
    """In-place Newton-Schulz orthogonalisation of X ([m, n] or [batch, m, n])."""
    _need_cuda(X, "X")
    if X.dim() not in (2, 3):
        raise ValueError("X must be 2-D or 3-D")
    batch, m, n = (1, *X.shape) if X.dim() == 2 else tuple(X.shape)
    h = handle or default_handle(X.device.index)
    st = h._lib.muon_orthogonalize(h.ptr, ctypes.c_void_p(X.data_ptr()), _dtype_code(X), batch, m, n, int(steps),
                                   _coeffs(coeffs), _method(ns_method), ctypes.c_void_p(_stream_ptr(stream)))
    h._raise(st, "muon_orthogonalize")
    return X


def muon_orthogonalize_noalloc(X: torch.Tensor, steps: int = 5, coeffs=None, stream=None) -> torch.Tensor:
    """In-place orthogonalisation of one 2-D matrix without any device
    allocation (static scratch inside the library; see include/muon.h for
    the size limits and the sharing rules)."""
    _need_cuda(X, "X")
    if X.dim() != 2:
        raise ValueError("X must be 2-D")
    lib = load_library()
    with torch.cuda.device(X.device):
        st = lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), _dtype_code(X), X.shape[0], X.shape[1],
                                            int(steps), _coeffs(coeffs), ctypes.c_void_p(_stream_ptr(stream)))
    if st != 0:
        raise MuonError(st, "muon_orthogonalize_noalloc")
    return X


def noalloc_check(device=None, stream=None) -> int:
    """Synchronise the stream and return (then clear) the device error status
    of the allocation-free calls on this device (0 = OK, 5 = non-finite
    norm, 6 = a bounded wait ran out)."""
    lib = load_library()
    dev = torch.cuda.current_device() if device is None else int(device)
    with torch.cuda.device(dev):
        return int(lib.muon_noalloc_check(ctypes.c_void_p(_stream_ptr(stream))))


def muon_step(params, grads, momenta, *, lr: float, wd: float, mu: float = 0.95, nesterov: bool = True,
              ns_method="standard", ns_steps: int = 5, coeffs=None, update_rms: float = 0.2, ns_dtype=None,
              split_heads=None, scale_dims=None, scale_mode="rms", extra_scale: float = 1.0,
              handle: MuonHandle | None = None, stream=None):
    """One Muon step over lists of 2-D params (updated in place), grads and
    fp32 momentum buffers (updated in place).  scale_mode "rms":
    update_rms * sqrt(max(A, B)); "mup": sqrt(rows / cols); either times
    extra_scale (muon_step_ex).  coeffs: one (a, b, c), or a list of
    ns_steps triples (a per-step schedule)."""
    n = len(params)
    if len(grads) != n or len(momenta) != n:
        raise ValueError("params, grads and momenta must have the same length")
    split_heads = [1] * n if split_heads is None else list(split_heads)
    scale_dims = [0] * n if scale_dims is None else list(scale_dims)
    arr = (MuonParamC * max(n, 1))()
    for i, (p, g, mbuf) in enumerate(zip(params, grads, momenta)):
        _need_cuda(p, f"params[{i}]")
        _need_cuda(g, f"grads[{i}]")
        _need_cuda(mbuf, f"momenta[{i}]")
        if p.dim() != 2 or g.shape != p.shape or mbuf.shape != p.shape:
            raise ValueError(f"params[{i}]: param, grad and momentum must be 2-D of one shape")
        if mbuf.dtype != torch.float32:
            raise ValueError(f"momenta[{i}] must be float32")
        arr[i] = MuonParamC(p.data_ptr(), g.data_ptr(), mbuf.data_ptr(), p.shape[0], p.shape[1], _dtype_code(p),
                            _dtype_code(g), int(split_heads[i]), 0, int(scale_dims[i]))
    if ns_dtype is None:
        ns_dtype = MUON_BF16 if all(p.dtype == torch.bfloat16 for p in params) else MUON_F32
    elif isinstance(ns_dtype, torch.dtype):
        ns_dtype = MUON_BF16 if ns_dtype == torch.bfloat16 else MUON_F32
    modes = {"rms": MUON_SCALE_RMS, "mup": MUON_SCALE_MUP}
    if scale_mode not in modes:
        raise ValueError(f"scale_mode must be one of {tuple(modes)}")
    per_step = coeffs is not None and len(coeffs) > 0 and hasattr(coeffs[0], "__len__")
    if per_step:
        # a schedule: one (a, b, c) per Newton-Schulz step
        if len(coeffs) != int(ns_steps) or any(len(c) != 3 for c in coeffs):
            raise ValueError("a coefficient schedule needs one (a, b, c) per step")
        cf = (ctypes.c_float * (3 * len(coeffs)))(*[float(x) for c in coeffs for x in c])
    else:
        cf = _coeffs(coeffs)
    opts = MuonStepOptionsC(float(lr), float(wd), float(mu), 1 if nesterov else 0, _method(ns_method), int(ns_steps),
                            ctypes.cast(cf, ctypes.POINTER(ctypes.c_float)), int(ns_dtype), modes[scale_mode],
                            float(update_rms), float(extra_scale), 1 if per_step else 0)
    dev = params[0].device.index if n else None
    h = handle or default_handle(dev)
    st = h._lib.muon_step_ex(h.ptr, arr, n, ctypes.byref(opts), ctypes.c_void_p(_stream_ptr(stream)))
    h._raise(st, "muon_step_ex")


def workspace_size(shapes, *, ns_method="standard", ns_steps: int = 5, ns_dtype=torch.bfloat16, split_heads=None,
                   handle: MuonHandle | None = None, device=None) -> int:
    """Device workspace bytes muon_step would need for parameters of these
    (rows, cols) shapes on this handle (its workspace limit decides the
    chunking); nothing is enqueued."""
    n = len(shapes)
    split_heads = [1] * n if split_heads is None else list(split_heads)
    code = MUON_BF16 if ns_dtype in (torch.bfloat16, MUON_BF16) else MUON_F32
    arr = (MuonParamC * max(n, 1))()
    for i, (r, c) in enumerate(shapes):
        arr[i] = MuonParamC(None, None, None, int(r), int(c), code, code, int(split_heads[i]), 0, 0)
    h = handle or default_handle(device)
    out = ctypes.c_uint64(0)
    st = h._lib.muon_workspace_size(h.ptr, arr, n, _method(ns_method), int(ns_steps), int(code), ctypes.byref(out))
    h._raise(st, "muon_workspace_size")
    return int(out.value)


def adamw_step(params, grads, exp_avgs, exp_avg_sqs, *, step: int, lr: float, beta1: float, beta2: float,
               eps: float, wd: float, handle: MuonHandle | None = None, stream=None):
    """Fused AdamW over lists of tensors (params, exp_avg, exp_avg_sq updated in place)."""
    n = len(params)
    if not (len(grads) == len(exp_avgs) == len(exp_avg_sqs) == n):
        raise ValueError("all lists must have the same length")
    P = (ctypes.c_void_p * max(n, 1))()
    G = (ctypes.c_void_p * max(n, 1))()
    Mm = (ctypes.c_void_p * max(n, 1))()
    V = (ctypes.c_void_p * max(n, 1))()
    N = (ctypes.c_int64 * max(n, 1))()
    PD = (ctypes.c_int32 * max(n, 1))()
    GD = (ctypes.c_int32 * max(n, 1))()
    for i in range(n):
        for t, w in ((params[i], "params"), (grads[i], "grads"), (exp_avgs[i], "exp_avgs"),
                     (exp_avg_sqs[i], "exp_avg_sqs")):
            _need_cuda(t, f"{w}[{i}]")
            if t.numel() != params[i].numel():
                raise ValueError(f"{w}[{i}] has the wrong size")
        if exp_avgs[i].dtype != torch.float32 or exp_avg_sqs[i].dtype != torch.float32:
            raise ValueError("AdamW moments must be float32")
        P[i], G[i] = params[i].data_ptr(), grads[i].data_ptr()
        Mm[i], V[i] = exp_avgs[i].data_ptr(), exp_avg_sqs[i].data_ptr()
        N[i], PD[i], GD[i] = params[i].numel(), _dtype_code(params[i]), _dtype_code(grads[i])
    dev = params[0].device.index if n else None
    h = handle or default_handle(dev)
    st = h._lib.adamw_step(h.ptr, P, G, Mm, V, N, PD, GD, n, int(step), float(lr), float(beta1), float(beta2),
                           float(eps), float(wd), ctypes.c_void_p(_stream_ptr(stream)))
    h._raise(st, "adamw_step")


def selftest_timeout(timeout_ns: int = 1_000_000, handle: MuonHandle | None = None, stream=None) -> int:
    """Run the bounded-wait self-test and return the status of the following check."""
    h = handle or default_handle()
    h._raise(h._lib.muon_selftest_timeout(h.ptr, int(timeout_ns), ctypes.c_void_p(_stream_ptr(stream))),
             "muon_selftest_timeout")
    return h.check(stream)

