"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds none of the attention arithmetic: it only turns
(seed, stream, flat index) into a bf16 value.  Both the CPU oracle tests and
the GPU path draw their inputs from here, so the two sides see bit-identical
operands.

Generator, defined once and implemented twice (numpy here, CUDA in
``synth.cu`` with the same steps):

* key      = splitmix64((seed << 32) | stream)
* r_i      = splitmix64(key + i * GAMMA)           (64-bit wrap-around)
* z_i      = (k0 + k1 + k2 + k3 - 131070) * sqrt(3) / 65536
             where k0..k3 are the four 16-bit fields of r_i.  This is the
             Irwin-Hall sum of four uniforms on (0, 1), centred and scaled to
             unit variance; every step is exact or a single IEEE rounding, so
             CPU and GPU agree bit for bit (no transcendental function).
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
# sqrt(3)/65536 as an exact double (sqrt is correctly rounded, /2^16 exact)
_ZSCALE = float.fromhex("0x1.bb67ae8584caap-16")

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


def normal_bf16_bits(seed: int, stream: int, start: int, count: int,
                     mean: float, std: float, chunk: int = 1 << 24) -> np.ndarray:
    """bf16 bit patterns of values start .. start+count-1 of one stream."""
    key = np.uint64(stream_key(seed, stream))
    out = np.empty(count, dtype=np.uint16)
    for c0 in range(0, count, chunk):
        n = min(chunk, count - c0)
        idx = np.arange(start + c0, start + c0 + n, dtype=np.uint64)
        r = _splitmix64(key + idx * np.uint64(GAMMA))
        ks = ((r & np.uint64(0xFFFF)) + ((r >> np.uint64(16)) & np.uint64(0xFFFF))
              + ((r >> np.uint64(32)) & np.uint64(0xFFFF)) + (r >> np.uint64(48)))
        z = (ks.astype(np.int64) - 131070).astype(np.float64) * _ZSCALE
        v = z * std          # one rounding
        v = v + mean         # one rounding
        out[c0:c0 + n] = f32_to_bf16_bits(v.astype(np.float32))
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
