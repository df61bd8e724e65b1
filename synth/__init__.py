"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the Muon method.  It only turns
(seed, stream, step, element index) into numbers:

* Philox-4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw,
  "Parallel random numbers: as easy as 1, 2, 3" (SC'11), written from its
  published definition (round function, multipliers, Weyl key schedule).
* A Box-Muller normal deviate whose logarithm and cosine are evaluated with
  only IEEE-754 single-precision +, -, *, / and sqrt, in a fixed order, so that
  the numpy version here and the CUDA version in ``synth/csrc/synth.cu`` produce
  bit-identical values (the CUDA file is compiled without FMA contraction and
  uses the explicitly rounded intrinsics).
* Round-to-nearest-even conversion of fp32 to bfloat16 (returned as uint16 bits).

Element ``e`` of a tensor uses Philox block ``e // 2`` with
counter = (block lo32, block hi32, step, 0) and key = (seed, stream); even
elements take outputs (x0, x1) as (u1, u2), odd elements (x2, x3).
"""
from __future__ import annotations

import numpy as np

SEED = 0x4D756F6E  # "Muon"

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# dtype codes shared with the C-ABI headers (plain integers, no arithmetic).
F32 = 0
BF16 = 1

# Roles, so that every tensor of a workload draws from its own stream.
ROLE_W, ROLE_M, ROLE_G = 0, 1, 2


def stream_id(tensor_index: int, role: int) -> int:
    """Philox key word 1 for tensor ``tensor_index`` in role W/M/G."""
    return (int(tensor_index) * 8 + int(role)) & 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox-4x32 with 10 rounds on arrays of uint32 counters and a scalar key.

    Each round multiplies counter words 0 and 2 by the two Philox multipliers
    (64-bit products split into hi/lo halves), then permutes and xors with the
    key; the key is bumped by the Weyl constants between rounds.
    """
    c0 = np.asarray(c0).astype(np.uint64, copy=False)
    c1 = np.asarray(c1).astype(np.uint64, copy=False)
    c2 = np.asarray(c2).astype(np.uint64, copy=False)
    c3 = np.asarray(c3).astype(np.uint64, copy=False)
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    for r in range(10):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & 0xFFFFFFFF
            k1 = (k1 + PHILOX_W1) & 0xFFFFFFFF
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
    return (c0.astype(np.uint32), c1.astype(np.uint32),
            c2.astype(np.uint32), c3.astype(np.uint32))


def _f32(x):
    return np.float32(x)


# fp32 constants of the deterministic log/cos (shared by value with synth.cu).
_SQRT2 = _f32(1.41421356237)
_LN2 = _f32(0.693147180560)
_INV = [_f32(1.0 / k) for k in (3, 5, 7, 9, 11)]
_TWO_PI = _f32(6.28318530718)
_COS_K = [_f32(v) for v in (-1.0 / 2, 1.0 / 24, -1.0 / 720, 1.0 / 40320,
                            -1.0 / 3628800, 1.0 / 479001600,
                            -1.0 / 87178291200)]


def _ln32(u):
    """Natural log of fp32 u in (0, 1): exponent split + atanh series."""
    u = np.asarray(u, dtype=np.float32)
    bits = u.view(np.uint32)
    e = (bits >> np.uint32(23)).astype(np.int32) - 127
    f = ((bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    big = f > _SQRT2
    f = np.where(big, f * _f32(0.5), f).astype(np.float32)
    e = np.where(big, e + 1, e)
    one = _f32(1.0)
    t = ((f - one) / (f + one)).astype(np.float32)
    t2 = (t * t).astype(np.float32)
    p = _INV[4]
    p = p * t2 + _INV[3]
    p = (p * t2).astype(np.float32) + _INV[2]
    p = (p * t2).astype(np.float32) + _INV[1]
    p = (p * t2).astype(np.float32) + _INV[0]
    p = (p * t2).astype(np.float32) + one
    lnf = ((t * p).astype(np.float32) * _f32(2.0)).astype(np.float32)
    return ((e.astype(np.float32) * _LN2).astype(np.float32) + lnf).astype(np.float32)


def _cos2pi32(u):
    """cos(2*pi*u) for fp32 u in (0, 1), by symmetry reduction + Taylor series."""
    u = np.asarray(u, dtype=np.float32)
    v = (u - _f32(0.5)).astype(np.float32)          # exact
    w = np.abs(v)
    far = w > _f32(0.25)
    w = np.where(far, _f32(0.5) - w, w).astype(np.float32)  # exact
    sign = np.where(far, _f32(1.0), _f32(-1.0)).astype(np.float32)
    x = (w * _TWO_PI).astype(np.float32)
    y = (x * x).astype(np.float32)
    c = _COS_K[6]
    for k in (5, 4, 3, 2, 1, 0):
        c = ((c * y).astype(np.float32) + _COS_K[k]).astype(np.float32)
    c = ((c * y).astype(np.float32) + _f32(1.0)).astype(np.float32)
    return (sign * c).astype(np.float32)


def _unit(x):
    """uint32 -> fp32 in (0,1): ((x >> 8) + 0.5) * 2^-24, exact."""
    x = np.asarray(x, dtype=np.uint32)
    return (((x >> np.uint32(8)).astype(np.float32) + _f32(0.5))
            * _f32(2.0 ** -24)).astype(np.float32)


def _normal_blocks(seed: int, stream: int, step: int, b0: int, nb: int,
                   sigma: np.float32) -> np.ndarray:
    """2*nb deviates for Philox blocks [b0, b0+nb), interleaved (even, odd)."""
    block = np.arange(b0, b0 + nb, dtype=np.uint64)
    lo = block & _MASK32
    hi = block >> np.uint64(32)
    x0, x1, x2, x3 = philox4x32_10(lo, hi, np.full(nb, step & 0xFFFFFFFF, np.uint64),
                                   np.zeros(nb, np.uint64), seed, stream)
    out = np.empty((nb, 2), dtype=np.float32)
    for col, (ua, ub) in enumerate(((x0, x1), (x2, x3))):
        r = np.sqrt((_ln32(_unit(ua)) * _f32(-2.0)).astype(np.float32)).astype(np.float32)
        z = (r * _cos2pi32(_unit(ub))).astype(np.float32)
        out[:, col] = (z * sigma).astype(np.float32)
    return out.reshape(-1)


_CHUNK_BLOCKS = 1 << 15


def normal_f32(seed: int, stream: int, step: int, start: int, count: int,
               sigma: float = 1.0, threads: int | None = None) -> np.ndarray:
    """Standard-normal deviates for elements [start, start+count), times sigma (fp32).

    Work is split into cache-sized chunks of Philox blocks; chunks run on a
    thread pool (numpy releases the GIL), which changes no value.
    """
    if count <= 0:
        return np.zeros(0, dtype=np.float32)
    sig = _f32(sigma)
    b_first = start >> 1
    b_last = (start + count - 1) >> 1
    nb_total = b_last - b_first + 1
    chunks = [(b, min(_CHUNK_BLOCKS, b_first + nb_total - b))
              for b in range(b_first, b_first + nb_total, _CHUNK_BLOCKS)]
    if len(chunks) == 1:
        parts = [_normal_blocks(seed, stream, step, chunks[0][0], chunks[0][1], sig)]
    else:
        import os
        from concurrent.futures import ThreadPoolExecutor
        nt = threads or max(1, min(len(chunks), len(os.sched_getaffinity(0))))
        with ThreadPoolExecutor(max_workers=nt) as ex:
            parts = list(ex.map(lambda c: _normal_blocks(seed, stream, step, c[0], c[1], sig),
                                chunks))
    z = np.concatenate(parts)
    off = start - 2 * b_first
    return z[off:off + count]


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 to bfloat16, nearest-even, returned as uint16 bit patterns."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(nan, np.uint64(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to fp32 exactly."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def tensor(seed: int, stream: int, step: int, shape, sigma: float, dtype: int,
           start: int = 0) -> np.ndarray:
    """A tensor of N(0, sigma^2) values: fp32 array, or uint16 bf16 bits."""
    count = int(np.prod(shape)) if len(shape) else 1
    z = normal_f32(seed, stream, step, start, count, sigma).reshape(shape)
    if dtype == BF16:
        return f32_to_bf16_bits(z)
    if dtype == F32:
        return z
    raise ValueError(f"unknown dtype code {dtype}")


def as_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of an fp32 array or bf16 bit array to fp64."""
    if dtype == BF16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# device fill (libmuonsynth.so, the CUDA twin of normal_f32 / f32_to_bf16_bits)
# ---------------------------------------------------------------------------
_LIB = None


def _cuda_lib():
    global _LIB
    if _LIB is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmuonsynth.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing; build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.synth_fill_normal.restype = ctypes.c_int
        lib.synth_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint32,
                                          ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float, ctypes.c_int32,
                                          ctypes.c_void_p]
        lib.synth_philox.restype = ctypes.c_int
        lib.synth_philox.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_void_p]
        _LIB = lib
    return _LIB


def fill_normal_cuda(t, seed: int, stream: int, step: int, sigma: float, start: int = 0,
                     cuda_stream=None) -> None:
    """Fill a contiguous torch CUDA tensor (float32 or bfloat16) with elements
    [start, start + t.numel()) of the seeded tensor, bit-identical to ``tensor``."""
    import ctypes
    import torch
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("need a contiguous CUDA tensor")
    if t.dtype == torch.float32:
        code = F32
    elif t.dtype == torch.bfloat16:
        code = BF16
    else:
        raise ValueError(f"unsupported dtype {t.dtype}")
    s = cuda_stream if cuda_stream is not None else torch.cuda.current_stream()
    rc = _cuda_lib().synth_fill_normal(ctypes.c_void_p(t.data_ptr()), int(start), int(t.numel()),
                                       int(seed) & 0xFFFFFFFF, int(stream) & 0xFFFFFFFF,
                                       int(step) & 0xFFFFFFFF, float(sigma), code,
                                       ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal failed with CUDA error {rc}")


def philox_cuda(ctr, key):
    """Raw Philox-4x32-10 on the device: ctr (n,4) and key (n,2) uint32 numpy arrays."""
    import ctypes
    import torch
    n = ctr.shape[0]
    c = torch.from_numpy(np.ascontiguousarray(ctr, dtype=np.uint32).view(np.int32)).cuda()
    k = torch.from_numpy(np.ascontiguousarray(key, dtype=np.uint32).view(np.int32)).cuda()
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    rc = _cuda_lib().synth_philox(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(c.data_ptr()),
                                  ctypes.c_void_p(k.data_ptr()), n,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_philox failed with CUDA error {rc}")
    return out.cpu().numpy().view(np.uint32)
