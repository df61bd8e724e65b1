"""Thin Python binding of libmuon.so, the GB300 (sm_103a) Muon optimizer step.

Every function here has the name of the C entry point it calls (include/muon.h)
and only marshals arguments: torch tensors become device pointers and
``cudaStream_t`` handles; every step of the method runs in the library's
kernels.  PyTorch provides device memory (the workspace, the caller's tensors)
and streams.  There is no fallback: libmuon.so is loaded on first use and a
missing library raises ImportError there.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmuon.so")
# the same library with the device range checks of the debug build (use_debug_library)
LIB_PATH_DEBUG = os.path.join(_HERE, "libmuon_debug.so")

# status codes, dtypes and enums of include/muon.h
MUON_OK = 0
MUON_WARN_NONFINITE = 1
MUON_ERR_INVALID = -1
MUON_ERR_NOT_PINNED = -2
MUON_ERR_NO_WORKSPACE = -3
MUON_ERR_CUDA = -4
MUON_ERR_TIMEOUT = -5
MUON_ERR_UNSUPPORTED = -6
MUON_ERR_DEVICE = -7
MUON_DTYPE_F32 = 0
MUON_DTYPE_BF16 = 1
MUON_NS_BF16 = 0
MUON_NS_TF32X3 = 1
MUON_MOMENTUM_EMA = 0
MUON_MOMENTUM_SGD = 1
MUON_NS_KERNEL_AUTO = 0
MUON_NS_KERNEL_GEMM = 1
MUON_NS_METHOD_STANDARD = 0
MUON_NS_METHOD_GRAM = 1
MUON_MAX_NS_STEPS = 16


class muon_shape(ctypes.Structure):
    _fields_ = [("rows", c_int64), ("cols", c_int64), ("count", c_int64), ("stride_elems", c_int64)]


class muon_config(ctypes.Structure):
    _fields_ = [("ns_a", c_float), ("ns_b", c_float), ("ns_c", c_float), ("eps", c_float),
                ("ns_precision", c_int32), ("momentum_form", c_int32), ("grad_dtype", c_int32),
                ("param_dtype", c_int32), ("max_inflight", c_int32), ("skip_nonfinite", c_int32),
                ("timing", c_int32), ("offload", c_int32), ("ns_kernel", c_int32),
                ("offload_zero_copy", c_int32), ("ns_momentum_fused", c_int32), ("ns_method", c_int32),
                ("reserved", c_int32 * 2)]


class muon_plan_info(ctypes.Structure):
    _fields_ = [("n_tensors", c_int64), ("n_matrices", c_int64), ("n_groups", c_int64),
                ("n_buckets", c_int64), ("max_bucket_matrices", c_int64),
                ("max_bucket_bytes", c_int64), ("workspace_bytes", c_size_t)]


class muon_bucket_info(ctypes.Structure):
    _fields_ = [("n_matrices", c_int64), ("bytes", c_int64), ("n_groups", c_int64),
                ("m", c_int64), ("n", c_int64), ("ns_single_kernel", c_int64),
                ("momentum_in_ns_kernel", c_int64)]


class muon_bucket_stats(ctypes.Structure):
    _fields_ = [("n_matrices", c_int64), ("n_groups", c_int64), ("m", c_int64), ("n", c_int64),
                ("bytes", c_int64), ("ns_workspace_bytes", c_int64), ("prep_ms", ctypes.c_double),
                ("ns_ms", ctypes.c_double), ("apply_ms", ctypes.c_double), ("h2d_ms", ctypes.c_double),
                ("d2h_ms", ctypes.c_double), ("h2d_bytes", c_int64), ("d2h_bytes", c_int64)]


class muon_stats(ctypes.Structure):
    _fields_ = [("prep_ms", ctypes.c_double), ("ns_ms", ctypes.c_double), ("apply_ms", ctypes.c_double),
                ("h2d_ms", ctypes.c_double), ("d2h_ms", ctypes.c_double), ("step_ms", ctypes.c_double),
                ("h2d_bytes", c_int64), ("d2h_bytes", c_int64), ("n_buckets", c_int64)]


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} not found at {path}; run __graft_entry__.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P = c_void_p
    sig = {
        "muon_config_default": (None, [POINTER(muon_config)]),
        "muon_plan": (c_int32, [POINTER(muon_shape), c_int32, POINTER(c_int32), c_int64,
                                POINTER(muon_config), POINTER(P)]),
        "muon_plan_workspace_bytes": (c_int32, [P, POINTER(c_size_t)]),
        "muon_plan_bind_workspace": (c_int32, [P, P, c_size_t]),
        "muon_step": (c_int32, [P, POINTER(P), POINTER(P), POINTER(P), c_int64, c_float, c_float,
                                c_int32, c_float, c_int32, P]),
        "muon_offload_step": (c_int32, [P, POINTER(P), POINTER(P), POINTER(P), c_int64, c_float,
                                        c_int32, c_int32, P, P, c_int64]),
        "muon_sync": (c_int32, [P, P, POINTER(c_int64)]),
        "muon_selftest_wait_timeout": (c_int32, [P, c_int64, P]),
        "muon_get_plan_info": (c_int32, [P, POINTER(muon_plan_info)]),
        "muon_get_bucket_info": (c_int32, [P, c_int64, POINTER(muon_bucket_info)]),
        "muon_set_ns_schedule": (c_int32, [P, POINTER(c_float), c_int32]),
        "muon_polar_express_coefficients": (c_int32, [c_int32, ctypes.c_double, ctypes.c_double,
                                                      POINTER(c_float), POINTER(ctypes.c_double)]),
        "muon_get_stats": (c_int32, [P, POINTER(muon_stats)]),
        "muon_last_error": (c_char_p, []),
        "muon_status_string": (c_char_p, [c_int32]),
        "muon_plan_destroy": (None, [P]),
        "muon_step_noalloc": (c_int32, [P, POINTER(P), POINTER(P), POINTER(P), c_int64, c_float, c_float,
                                        c_int32, c_float, c_int32, P]),
        "muon_noalloc_scratch_bytes": (c_size_t, []),
        "muon_inject_copy_failure": (c_int32, [P, c_int64]),
        "muon_get_bucket_stats": (c_int32, [P, c_int64, POINTER(muon_bucket_stats)]),
        "muon_get_input_norms": (c_int32, [P, POINTER(c_float), c_int64, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


_LIB_DEBUG = False


def use_debug_library(on: bool = True) -> None:
    """Route every later call to libmuon_debug.so (device range checks that record
    MUON_ERR_DEVICE instead of touching memory out of range) or back to libmuon.so.
    A plan belongs to the library that made it: switch only when no plan is alive."""
    global _LIB, _LIB_DEBUG
    _LIB = _load(LIB_PATH_DEBUG if on else LIB_PATH)
    _LIB_DEBUG = bool(on)


def using_debug_library() -> bool:
    return _LIB is not None and _LIB_DEBUG


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib().muon_last_error().decode() or _lib().muon_status_string(status).decode()
        super().__init__(f"{where}: {_lib().muon_status_string(status).decode()} ({status}): {msg}")


def _check(status: int, where: str) -> int:
    if status < 0:
        raise MuonError(status, where)
    return status


def muon_config_default(**overrides) -> muon_config:
    """The library's default configuration, with fields overridden by keyword."""
    cfg = muon_config()
    _lib().muon_config_default(byref(cfg))
    for k, v in overrides.items():
        if not hasattr(cfg, k):
            raise AttributeError(f"muon_config has no field {k!r}")
        setattr(cfg, k, v)
    return cfg


class Plan:
    """Owner of a muon_plan_t* (destroyed with the object) and its bound workspace."""

    def __init__(self, handle: int, n_tensors: int):
        self.handle = c_void_p(handle)
        self.n_tensors = n_tensors
        self.workspace = None

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            _lib().muon_plan_destroy(h)
            self.handle = c_void_p(0)


def _stream_ptr(stream) -> c_void_p:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return c_void_p(int(getattr(stream, "cuda_stream", stream)))


def _ptrs(tensors) -> ctypes.Array:
    arr = (c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = c_void_p(t.data_ptr() if hasattr(t, "data_ptr") else int(t))
    return arr


def muon_plan(shapes: Sequence[Sequence[int]], groups: Optional[Sequence[int]] = None,
              bucket_cap_bytes: int = 512 << 20, config: Optional[muon_config] = None) -> Plan:
    """shapes: (rows, cols[, count[, stride_elems]]) per tensor."""
    n = len(shapes)
    arr = (muon_shape * max(n, 1))()
    for i, s in enumerate(shapes):
        s = tuple(int(v) for v in s) + (1, 0)[len(s) - 2:] if len(s) < 4 else tuple(int(v) for v in s)
        arr[i] = muon_shape(s[0], s[1], s[2], s[3])
    g = None
    if groups is not None:
        g = (c_int32 * n)(*[int(v) for v in groups])
    out = c_void_p()
    _check(_lib().muon_plan(arr, n, g, int(bucket_cap_bytes), byref(config) if config is not None else None,
                         byref(out)), "muon_plan")
    return Plan(out.value, n)


def muon_plan_workspace_bytes(plan: Plan) -> int:
    v = c_size_t()
    _check(_lib().muon_plan_workspace_bytes(plan.handle, byref(v)), "muon_plan_workspace_bytes")
    return v.value


def muon_plan_bind_workspace(plan: Plan, workspace) -> None:
    """workspace: a torch uint8 CUDA tensor of at least muon_plan_workspace_bytes bytes."""
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib().muon_plan_bind_workspace(plan.handle, c_void_p(workspace.data_ptr()), nbytes),
           "muon_plan_bind_workspace")
    plan.workspace = workspace


def muon_step(plan: Plan, params, grads, momentum, lr: float, mu: float, nesterov: bool, wd: float,
              ns_steps: int = 5, stream=None) -> None:
    n = len(params)
    _check(_lib().muon_step(plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum), n, float(lr),
                         float(mu), int(bool(nesterov)), float(wd), int(ns_steps), _stream_ptr(stream)),
           "muon_step")


def muon_step_noalloc(plan: Plan, params, grads, momentum, lr: float, mu: float, nesterov: bool,
                      wd: float, ns_steps: int = 5, stream=None) -> None:
    """muon_step without a caller-bound workspace, for callers that cannot allocate
    device memory: the step runs in the library's static device scratch."""
    n = len(params)
    _check(_lib().muon_step_noalloc(plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum), n,
                                    float(lr), float(mu), int(bool(nesterov)), float(wd), int(ns_steps),
                                    _stream_ptr(stream)),
           "muon_step_noalloc")


def muon_inject_copy_failure(plan: Plan, nth: int) -> None:
    """The nth host-link copy of the plan's next offload step reports a failure
    (MUON_ERR_CUDA) instead of being enqueued; -1 clears it."""
    _check(_lib().muon_inject_copy_failure(plan.handle, int(nth)), "muon_inject_copy_failure")


def muon_noalloc_scratch_bytes() -> int:
    return int(_lib().muon_noalloc_scratch_bytes())


def muon_offload_step(plan: Plan, h_grads, h_momentum, h_update_out, mu: float, nesterov: bool,
                      ns_steps: int = 5, compute=None, copy=None, timeout_ms: int = 600_000) -> None:
    n = len(h_grads)
    _check(_lib().muon_offload_step(plan.handle, _ptrs(h_grads), _ptrs(h_momentum), _ptrs(h_update_out), n,
                                 float(mu), int(bool(nesterov)), int(ns_steps), _stream_ptr(compute),
                                 c_void_p(int(getattr(copy, "cuda_stream", copy))) if copy is not None
                                 else c_void_p(0), int(timeout_ms)),
           "muon_offload_step")


def muon_sync(plan: Plan, stream=None):
    """Returns (status, n_nonfinite); raises on errors (a device wait that ran out)."""
    nf = c_int64()
    st = _check(_lib().muon_sync(plan.handle, _stream_ptr(stream), byref(nf)), "muon_sync")
    return st, nf.value


def muon_selftest_wait_timeout(plan: Plan, limit_us: int, stream=None) -> None:
    """Enqueue the failure-path self-test: a one-CTA kernel whose bounded wait runs
    out after limit_us; the next muon_sync reports it (MUON_ERR_DEVICE)."""
    _check(_lib().muon_selftest_wait_timeout(plan.handle, int(limit_us), _stream_ptr(stream)),
           "muon_selftest_wait_timeout")


def muon_get_plan_info(plan: Plan) -> muon_plan_info:
    info = muon_plan_info()
    _check(_lib().muon_get_plan_info(plan.handle, byref(info)), "muon_get_plan_info")
    return info


def muon_get_bucket_info(plan: Plan, b: int) -> muon_bucket_info:
    info = muon_bucket_info()
    _check(_lib().muon_get_bucket_info(plan.handle, int(b), byref(info)), "muon_get_bucket_info")
    return info


def muon_set_ns_schedule(plan: Plan, coeffs) -> None:
    """Per-iteration (a, b, c) triples for later steps of the plan; [] restores the
    configuration's coefficients for every iteration."""
    flat = [float(v) for t in coeffs for v in t]
    n = len(flat) // 3
    if n * 3 != len(flat):
        raise ValueError("coefficients are (a, b, c) triples")
    arr = (c_float * max(len(flat), 1))(*flat)
    _check(_lib().muon_set_ns_schedule(plan.handle, arr if n else None, n), "muon_set_ns_schedule")


def muon_polar_express_coefficients(n_iters: int, lower: float = 1e-3, safety: float = 1.0):
    """(coefficient triples, per-iteration error bounds) of the minimax schedule,
    computed by the library on the host."""
    out = (c_float * (3 * int(n_iters)))()
    err = (ctypes.c_double * int(n_iters))()
    _check(_lib().muon_polar_express_coefficients(int(n_iters), float(lower), float(safety), out, err),
           "muon_polar_express_coefficients")
    return [tuple(out[3 * k:3 * k + 3]) for k in range(int(n_iters))], list(err)


def muon_get_stats(plan: Plan) -> muon_stats:
    st = muon_stats()
    _check(_lib().muon_get_stats(plan.handle, byref(st)), "muon_get_stats")
    return st


def muon_get_bucket_stats(plan: Plan, b: int) -> muon_bucket_stats:
    st = muon_bucket_stats()
    _check(_lib().muon_get_bucket_stats(plan.handle, int(b), byref(st)), "muon_get_bucket_stats")
    return st


def muon_get_input_norms(plan: Plan, stream=None):
    """||V||_F of every matrix's Newton-Schulz input in the last step, tensor order."""
    n = int(muon_get_plan_info(plan).n_matrices)
    out = (c_float * n)()
    _check(_lib().muon_get_input_norms(plan.handle, out, n, _stream_ptr(stream)), "muon_get_input_norms")
    return list(out)


def muon_status_string(status: int) -> str:
    return _lib().muon_status_string(int(status)).decode()


def allocate_workspace(plan: Plan, device=None):
    """torch-allocated workspace (256-byte aligned), bound to the plan."""
    import torch
    nbytes = muon_plan_workspace_bytes(plan)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")
    muon_plan_bind_workspace(plan, ws)
    return ws
