"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds none of the attention arithmetic: it only turns
(seed, stream, flat index) into a bf16 value.  Both the CPU oracle tests and
the GPU path draw their inputs from here, so the two sides see bit-identical
operands.

Generator, defined once and implemented twice (numpy here, CUDA in
``synth.cu`` with the same steps):

* key      = splitmix64((seed << 32) | stream)
* r_c      = splitmix64(key + c * GAMMA)           (64-bit wrap-around)
* value i draws r_{2i} and r_{2i+1}:
  u1 = ((r_{2i} >> 11) + 1) 2^-53 in (0, 1],  u2 = (r_{2i+1} >> 11) 2^-53 in [0, 1)
* z_i      = sqrt(-2 ln u1) cos(2 pi u2)        (Box and Muller, 1958: an
             exact standard normal variate for exact uniforms; |z| < 8.6)
  with ln and cos evaluated by power series in plain IEEE double operations
  (add, multiply, divide, square root; no fused multiply-add), so the two
  copies round identically step for step:
    ln u1   = e ln 2 + 2 atanh(s): u1 = m 2^e with m in [sqrt(1/2), sqrt(2)),
              s = (m - 1) / (m + 1), atanh(s) = s sum_k s^(2k) / (2k + 1)
    cos 2 pi u2 by quarter turns: q = floor(4 u2), phi = (pi/2)(4 u2 - q),
              cos phi = sum_k (-1)^k phi^(2k) / (2k)!,
              sin phi = phi sum_k (-1)^k phi^(2k) / (2k + 1)!, k = 0..11
* value    = bf16_rne(float32_rne(mean + std * z_i))  (double arithmetic, no FMA)

splitmix64 is the mixing function of Steele, Lea and Flood (2014),
"Fast splittable pseudorandom number generators".

Streams (one per tensor, fixed order) are listed in ``STREAMS``.  Indices are
flat row-major positions in the full tensor, so any slice of a large tensor
(one batch row of a 15 GB input, say) can be drawn on its own.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
# Series coefficients as exact hex doubles (the same literals are in synth.cu):
# 1 / (2k + 1), (-1)^k / (2k)!, (-1)^k / (2k + 1)! for k = 0..11.
_ATANH = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "0x1.5555555555555p-2", "0x1.999999999999ap-3", "0x1.2492492492492p-3",
    "0x1.c71c71c71c71cp-4", "0x1.745d1745d1746p-4", "0x1.3b13b13b13b14p-4", "0x1.1111111111111p-4",
    "0x1.e1e1e1e1e1e1ep-5", "0x1.af286bca1af28p-5", "0x1.8618618618618p-5", "0x1.642c8590b2164p-5")]
_COS = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.0000000000000p-1", "0x1.5555555555555p-5", "-0x1.6c16c16c16c17p-10",
    "0x1.a01a01a01a01ap-16", "-0x1.27e4fb7789f5cp-22", "0x1.1eed8eff8d898p-29", "-0x1.93974a8c07c9dp-37",
    "0x1.ae7f3e733b81fp-45", "-0x1.6827863b97d97p-53", "0x1.e542ba4020225p-62", "-0x1.0ce396db7f853p-70")]
_SIN = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.5555555555555p-3", "0x1.1111111111111p-7", "-0x1.a01a01a01a01ap-13",
    "0x1.71de3a556c734p-19", "-0x1.ae64567f544e4p-26", "0x1.6124613a86d09p-33", "-0x1.ae7f3e733b81fp-41",
    "0x1.952c77030ad4ap-49", "-0x1.2f49b46814157p-57", "0x1.71b8ef6dcf572p-66", "-0x1.761b41316381ap-75")]
_LN2 = float.fromhex("0x1.62e42fefa39efp-1")
_HALF_PI = float.fromhex("0x1.921fb54442d18p+0")
_SQRT_HALF = float.fromhex("0x1.6a09e667f3bcdp-1")

STREAMS = {
    "x": 0,            # prefill input hidden states
    "w_in_norm": 1,    # input RMSNorm gain
    "w_q_a": 2,
    "w_q_a_norm": 3,
    "w_q_b": 4,
    "w_kv_a": 5,
    "w_kv_a_norm": 6,
    "w_kv_b": 7,
    "w_o": 8,
    "cache_x": 9,      # hidden states whose projections fill a decode cache
    "new_x": 10,       # the new token's hidden state in decode
    "w_post_norm": 11,  # the block's post-attention RMSNorm gain
    "w_1": 12,         # SwiGLU MLP gate projection
    "w_3": 13,         # SwiGLU MLP up projection
    "w_2": 14,         # SwiGLU MLP down projection
    "ffn_x": 15,       # hidden states fed to the MLP half on its own
}

# Distributions of the synthetic workload: (mean, std)
WEIGHT_DIST = (0.0, 0.02)
GAIN_DIST = (1.0, 0.1)
X_DIST = (0.0, 1.0)

# The eight weight tensors of one MLA sublayer (nn.Linear [out, in]) and the
# distribution each is drawn from.
WEIGHT_SPECS = {
    "w_in_norm": ((7168,), GAIN_DIST),
    "w_q_a": ((1536, 7168), WEIGHT_DIST),
    "w_q_a_norm": ((1536,), GAIN_DIST),
    "w_q_b": ((12288, 1536), WEIGHT_DIST),
    "w_kv_a": ((576, 7168), WEIGHT_DIST),
    "w_kv_a_norm": ((512,), GAIN_DIST),
    "w_kv_b": ((16384, 512), WEIGHT_DIST),
    "w_o": ((7168, 8192), WEIGHT_DIST),
}


# The four tensors of the block's MLP half: post-attention RMSNorm gain and
# the three bias-free SwiGLU matrices (intermediate width 18,432).
FFN_WEIGHT_SPECS = {
    "w_post_norm": ((7168,), GAIN_DIST),
    "w_1": ((18432, 7168), WEIGHT_DIST),
    "w_3": ((18432, 7168), WEIGHT_DIST),
    "w_2": ((7168, 18432), WEIGHT_DIST),
}


def ffn_weight_bits(seed: int = 0) -> dict:
    """bf16 bits of the MLP-half weights (about 396 M values)."""
    return {n: tensor_bits(seed, n, shape, dist) for n, (shape, dist) in FFN_WEIGHT_SPECS.items()}


def ffn_weights_cuda(seed: int = 0, device="cuda") -> dict:
    return {n: tensor_cuda(seed, n, shape, dist, device) for n, (shape, dist) in FFN_WEIGHT_SPECS.items()}


def weight_bits(seed: int = 0) -> dict:
    """bf16 bits of all weights (about 101 M values; a few seconds)."""
    return {n: tensor_bits(seed, n, shape, dist) for n, (shape, dist) in WEIGHT_SPECS.items()}


def weights_cuda(seed: int = 0, device="cuda") -> dict:
    """The same weights drawn directly on the GPU (bit-identical)."""
    return {n: tensor_cuda(seed, n, shape, dist, device) for n, (shape, dist) in WEIGHT_SPECS.items()}


def _splitmix64(x: np.ndarray) -> np.ndarray:
    x = x + np.uint64(GAMMA)
    x = (x ^ (x >> np.uint64(30))) * np.uint64(_M1)
    x = (x ^ (x >> np.uint64(27))) * np.uint64(_M2)
    return x ^ (x >> np.uint64(31))


def _splitmix64_inplace(x: np.ndarray, t: np.ndarray) -> None:
    """x <- splitmix64(x) (t: scratch of the same shape)."""
    x += np.uint64(GAMMA)
    for shift, mul in ((30, _M1), (27, _M2)):
        np.right_shift(x, np.uint64(shift), out=t)
        x ^= t
        x *= np.uint64(mul)
    np.right_shift(x, np.uint64(31), out=t)
    x ^= t


def stream_key(seed: int, stream: int) -> int:
    v = np.array([((seed & 0xFFFFFFFF) << 32) | (stream & 0xFFFFFFFF)], dtype=np.uint64)
    return int(_splitmix64(v)[0])


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


def _horner(x: np.ndarray, coef, out: np.ndarray) -> np.ndarray:
    """out <- sum_k coef[k] x^k, Horner's rule from the highest term
    (p = c_K; p = p x + c_k), one rounding per operation."""
    np.multiply(x, coef[-1], out=out)
    out += coef[-2]
    for c in reversed(coef[:-2]):
        out *= x
        out += c
    return out


def normal_bf16_bits(seed: int, stream: int, start: int, count: int,
                     mean: float, std: float, chunk: int = 1 << 16) -> np.ndarray:
    """bf16 bit patterns of values start .. start+count-1 of one stream
    (worked in cache-sized chunks with in-place operations)."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(count, dtype=np.uint16)
    m0 = min(chunk, count)
    if m0 == 0:
        return out
    ramp = np.arange(m0, dtype=np.int64).view(np.uint64)
    c2, r1, r2, t = (np.empty(m0, dtype=np.uint64) for _ in range(4))
    m, e, s, p, q, x, ps = (np.empty(m0, dtype=np.float64) for _ in range(7))
    mask = np.empty(m0, dtype=bool)
    f = np.empty(m0, dtype=np.float32)
    u = f.view(np.uint32)
    b = np.empty(m0, dtype=np.uint32)
    for c0 in range(0, count, chunk):
        n = min(chunk, count - c0)
        c2_, r1_, r2_, t_ = c2[:n], r1[:n], r2[:n], t[:n]
        m_, e_, s_, p_, q_, x_, ps_, k_ = m[:n], e[:n], s[:n], p[:n], q[:n], x[:n], ps[:n], mask[:n]
        np.add(ramp[:n], np.uint64(start + c0), out=c2_)
        c2_ *= np.uint64(2)                          # counter of value i's first draw
        for j, r_ in ((0, r1_), (1, r2_)):
            np.add(c2_, np.uint64(j), out=r_)
            r_ *= np.uint64(GAMMA)
            r_ += key
            _splitmix64_inplace(r_, t_)
            r_ >>= np.uint64(11)                     # 53 random bits
        # u1 = (r1 + 1) 2^-53 in (0, 1]; its exponent e and mantissa m in [1/2, 1)
        r1_ += np.uint64(1)
        np.copyto(m_, r1_, casting="unsafe")         # exact (< 2^53 + 1)
        m_ *= 2.0 ** -53
        mb = m_.view(np.uint64)
        np.right_shift(mb, np.uint64(52), out=t_)
        np.copyto(e_, t_, casting="unsafe")
        e_ -= 1022.0
        mb &= np.uint64(0x000FFFFFFFFFFFFF)
        mb |= np.uint64(1022 << 52)
        np.less(m_, _SQRT_HALF, out=k_)              # m in [sqrt(1/2), sqrt(2))
        np.multiply(m_, 2.0, out=m_, where=k_)
        np.subtract(e_, 1.0, out=e_, where=k_)
        # ln u1 = e ln 2 + 2 s sum_k s^2k / (2k + 1),  s = (m - 1) / (m + 1)
        np.add(m_, 1.0, out=p_)
        m_ -= 1.0
        np.divide(m_, p_, out=s_)
        np.multiply(s_, s_, out=x_)
        _horner(x_, _ATANH, p_)
        s_ *= p_
        s_ *= 2.0
        e_ *= _LN2
        e_ += s_                                     # ln u1
        e_ *= -2.0
        np.sqrt(e_, out=e_)                          # R = sqrt(-2 ln u1)
        # cos(2 pi u2) by quarter turns
        np.copyto(m_, r2_, casting="unsafe")
        m_ *= 2.0 ** -51                             # 4 u2, exact
        np.floor(m_, out=q_)
        m_ -= q_                                     # exact
        m_ *= _HALF_PI                               # phi
        np.multiply(m_, m_, out=x_)
        _horner(x_, _COS, p_)                        # cos phi
        _horner(x_, _SIN, ps_)
        ps_ *= m_                                    # sin phi
        np.negative(ps_, out=ps_, where=(q_ == 1.0))
        np.negative(p_, out=p_, where=(q_ == 2.0))
        np.copyto(p_, ps_, where=((q_ == 1.0) | (q_ == 3.0)))
        e_ *= p_                                     # z = R cos(2 pi u2)
        e_ *= std                                    # one rounding
        e_ += mean                                   # one rounding
        np.copyto(f[:n], e_, casting="same_kind")    # float32, round to nearest even
        u_, b_ = u[:n], b[:n]
        np.right_shift(u_, np.uint32(16), out=b_)    # bf16, round to nearest even
        b_ &= np.uint32(1)
        b_ += np.uint32(0x7FFF)
        b_ += u_
        b_ >>= np.uint32(16)
        np.copyto(out[c0:c0 + n], b_, casting="unsafe")
    return out


def tensor_bits(seed: int, name: str, shape, dist, rows=None) -> np.ndarray:
    """bf16 bits of a whole tensor, or of the given leading-dim rows of it.

    ``shape`` is the full tensor shape; ``rows`` (iterable of ints) selects
    flat indices along the first axis, so a slice of a huge tensor is drawn
    without drawing the rest.
    """
    shape = tuple(int(s) for s in shape)
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    mean, std = dist
    if rows is None:
        return normal_bf16_bits(seed, STREAMS[name], 0, int(np.prod(shape)), mean, std).reshape(shape)
    if isinstance(rows, range) and rows.step == 1:  # a contiguous block: one draw
        n = max(0, len(rows))
        return normal_bf16_bits(seed, STREAMS[name], rows.start * inner, n * inner, mean, std).reshape(
            (n,) + shape[1:])
    rows = list(rows)
    out = np.empty((len(rows),) + shape[1:], dtype=np.uint16)
    for i, r in enumerate(rows):
        out[i] = normal_bf16_bits(seed, STREAMS[name], r * inner, inner, mean, std).reshape(shape[1:])
    return out


# ---------------------------------------------------------------------------
# Same generator on the GPU (large tensors).  The library is built from
# synth.cu next to this file; it holds only the generator above.
# ---------------------------------------------------------------------------
_HERE = os.path.dirname(os.path.abspath(__file__))
SYNTH_SO = os.path.join(_HERE, "libmlasynth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(SYNTH_SO):
            raise RuntimeError(f"{SYNTH_SO} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(SYNTH_SO)
        lib.synth_normal_bf16.restype = ctypes.c_int
        lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32,
                                          ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_void_p]
        _lib = lib
    return _lib


def fill_normal_bf16_cuda(ptr: int, count: int, seed: int, stream: int, start: int,
                          mean: float, std: float, cuda_stream: int = 0) -> None:
    """Fill ``count`` bf16 values at device address ``ptr`` with values
    start .. start+count-1 of the stream (bit-identical to ``normal_bf16_bits``)."""
    rc = _load().synth_normal_bf16(ctypes.c_void_p(ptr), count, seed, stream, start,
                                   mean, std, ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed with CUDA error {rc}")


def tensor_cuda(seed: int, name: str, shape, dist, device="cuda", row_offset: int = 0):
    """A torch bf16 tensor on the GPU holding the stream's values.

    ``row_offset`` shifts the flat start by that many leading-dim rows of
    ``shape`` (a slice of a larger tensor of the same inner shape).
    """
    import torch
    shape = tuple(int(s) for s in shape)
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    mean, std = dist
    fill_normal_bf16_cuda(t.data_ptr(), t.numel(), seed, STREAMS[name], row_offset * inner,
                          mean, std, torch.cuda.current_stream().cuda_stream)
    return t
