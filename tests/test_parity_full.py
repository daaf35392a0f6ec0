"""Parity at the full benchmark sizes, in the launch configuration bench.py
times, on sampled outputs the oracle can compute one by one.

* prefill B=1, T=2048 and prefill B=8, T=4096 (both caches written): the
  GPU runs the whole batch; the oracle projects keys/values for every token
  of the sampled sequences and queries only at sampled positions.
* chunked prefill B=1, T=2048 after P0=2048 cached positions (oracle-built
  caches, rebuilt and latent forms), sampled query rows.
* decode B=64, P=1000 (rebuilt cache) and latent decode B=128, P=8192: the
  GPU fills every cache with its own cache-only prefill of the seeded
  'cache_x' tokens (checked against the oracle's caches for the sampled
  sequences), then the sampled sequences' cache rows are replaced by the
  oracle's bf16 caches so both sides decode from identical inputs.
* the absorbed chunk B=32, T=4 after P0=8188 latent positions (the bench's
  size), caches as for the decodes, sampled sequences.
Tolerance as in test_parity_small (max abs <= 2e-2, rel. Frobenius <= 1e-2;
cache entries one bf16 ulp more, the bf16 output half an ulp more).
"""
import numpy as np
import pytest

import synth
from oracle import mla_oracle as om
import mla_gb300 as m
from mla_testlib import (bits_to_cuda, cuda_to_f64, cuda_weights, f64_to_bits, oracle_weights, parity, parity_cache,
                         parity_out)

pytestmark = pytest.mark.gpu

D = 7168


@pytest.fixture(scope="module")
def W(gpu_available):
    wt = cuda_weights(0)
    return wt, m.make_weights(wt), oracle_weights(0)


def _prefill_case(W, B, T, b_samples, t_samples, with_cache):
    import torch
    x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST)
    out = torch.empty_like(x)
    delta = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    caches = (None,) * 4
    if with_cache:
        caches = (torch.zeros((B, 64, T, 192), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros((B, 64, T, 128), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros((B, T, 512), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros((B, T, 64), dtype=torch.bfloat16, device="cuda"))
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill(W[1], x, out, ws, *caches, T if with_cache else 0, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    for b in b_samples:
        xb = synth.bf16_bits_to_f64(synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST, rows=[b]))
        ref = om.prefill(W[2], xb, query_rows=t_samples)
        parity_out(cuda_to_f64(out[b, t_samples]), ref["out"][0], f"out b={b}")
        parity(cuda_to_f64(delta[b, t_samples]), ref["delta"][0], f"delta b={b}")
        if with_cache:
            kc, vc, ckv, kpe = caches
            parity_cache(cuda_to_f64(kc[b][:, t_samples]), ref["K"][0][:, t_samples], f"K cache b={b}")
            parity_cache(cuda_to_f64(vc[b][:, t_samples]), ref["V"][0][:, t_samples], f"V cache b={b}")
            parity_cache(cuda_to_f64(ckv[b]), ref["ckv"][0], f"latent cache b={b}")
            parity_cache(cuda_to_f64(kpe[b]), ref["kpe"][0], f"rotary-key cache b={b}")


def test_prefill_b1_t2048(W):
    _prefill_case(W, 1, 2048, [0], [0, 1, 127, 128, 1000, 2046, 2047], with_cache=False)


def test_prefill_b8_t4096_with_caches(W):
    _prefill_case(W, 8, 4096, [0, 5], [0, 129, 2048, 4095], with_cache=True)


def test_prefill_chunk_b1_p2048_t2048(W):
    """Chunked prefill of 2048 tokens after 2048 cached positions (the
    bench's chunk workload): the caches hold the oracle's bf16 rows of the
    seeded 'cache_x' tokens; sampled query rows on both sides."""
    import torch
    B, P0, T = 1, 2048, 2048
    cap = P0 + T
    xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P0, D), synth.X_DIST))
    c = om.cache_from_tokens(W[2], xc)
    Kb, Vb = f64_to_bits(c["K"]), f64_to_bits(c["V"])
    kc = torch.zeros((B, 64, cap, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, cap, 128), dtype=torch.bfloat16, device="cuda")
    kc[:, :, :P0].copy_(bits_to_cuda(Kb))
    vc[:, :, :P0].copy_(bits_to_cuda(Vb))
    x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST)
    out = torch.empty_like(x)
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill_chunk(W[1], x, P0, out, kc, vc, ws)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    rows = [0, 1, 127, 128, 1000, 2046, 2047]
    xb = synth.bf16_bits_to_f64(synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST))
    ref = om.prefill_with_past(W[2], xb, synth.bf16_bits_to_f64(Kb), synth.bf16_bits_to_f64(Vb),
                               query_rows=rows)
    parity_out(cuda_to_f64(out[0, rows]), ref["out"][0], "chunk out")
    parity_cache(cuda_to_f64(kc[0][:, [P0 + r for r in rows]]), ref["K"][0][:, rows], "chunk K rows")
    parity_cache(cuda_to_f64(vc[0][:, [P0 + r for r in rows]]), ref["V"][0][:, rows], "chunk V rows")


def test_prefill_chunk_latent_b1_p2048_t2048(W):
    """The same chunk against the latent cache (the bench's latent chunk
    workload): the oracle's bf16 latent rows of the seeded 'cache_x' tokens
    on both sides, sampled query rows."""
    import torch
    B, P0, T = 1, 2048, 2048
    cap = P0 + T
    xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P0, D), synth.X_DIST))
    c = om.cache_from_tokens(W[2], xc)
    Cb, Rb = f64_to_bits(c["ckv"]), f64_to_bits(c["kpe"])
    ckv = torch.zeros((B, cap, 512), dtype=torch.bfloat16, device="cuda")
    kpe = torch.zeros((B, cap, 64), dtype=torch.bfloat16, device="cuda")
    ckv[:, :P0].copy_(bits_to_cuda(Cb))
    kpe[:, :P0].copy_(bits_to_cuda(Rb))
    x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST)
    out = torch.empty_like(x)
    ws = m.alloc_workspace(m.MODE_CHUNK_LATENT, B, T, cap=cap)
    m.mla_prefill_chunk_latent(W[1], x, P0, out, ckv, kpe, ws)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    rows = [0, 1, 127, 128, 1000, 2046, 2047]
    xb = synth.bf16_bits_to_f64(synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST))
    ref = om.prefill_with_past_latent(W[2], xb, synth.bf16_bits_to_f64(Cb), synth.bf16_bits_to_f64(Rb),
                                      query_rows=rows)
    parity_out(cuda_to_f64(out[0, rows]), ref["out"][0], "latent chunk out")
    parity_cache(cuda_to_f64(ckv[0, [P0 + r for r in rows]]), ref["ckv"][0][rows], "latent chunk rows")


def _fill_caches(W, B, P, cap, rebuilt):
    """The library's own cache-only prefill over the seeded 'cache_x' tokens."""
    import torch
    if rebuilt:
        c1 = torch.zeros((B, 64, cap, 192), dtype=torch.bfloat16, device="cuda")
        c2 = torch.zeros((B, 64, cap, 128), dtype=torch.bfloat16, device="cuda")
    else:
        c1 = torch.zeros((B, cap, 512), dtype=torch.bfloat16, device="cuda")
        c2 = torch.zeros((B, cap, 64), dtype=torch.bfloat16, device="cuda")
    bs = max(1, min(B, (1 << 17) // P))
    ws = m.alloc_workspace(m.MODE_PREFILL, bs, P)
    for b0 in range(0, B, bs):
        nb = min(bs, B - b0)
        xc = synth.tensor_cuda(0, "cache_x", (nb, P, D), synth.X_DIST, row_offset=b0)
        if rebuilt:
            m.mla_prefill(W[1], xc, None, ws, c1[b0:b0 + nb], c2[b0:b0 + nb], None, None, cap)
        else:
            m.mla_prefill(W[1], xc, None, ws, None, None, c1[b0:b0 + nb], c2[b0:b0 + nb], cap)
    torch.cuda.synchronize()
    return c1, c2


def test_decode_b64_p1000(W):
    import torch
    B, P = 64, 1000
    cap = P + 1
    kc, vc = _fill_caches(W, B, P, cap, rebuilt=True)
    samples = [0, 37, 63]
    refs = {}
    for b in samples:
        xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P, D), synth.X_DIST, rows=[b]))
        c = om.cache_from_tokens(W[2], xc)
        # the GPU-built cache rows of this sequence match the oracle's
        pos = [0, 1, 500, 999]
        parity_cache(cuda_to_f64(kc[b][:, pos]), c["K"][0][:, pos], f"GPU-filled K cache b={b}")
        parity_cache(cuda_to_f64(vc[b][:, pos]), c["V"][0][:, pos], f"GPU-filled V cache b={b}")
        Kb, Vb = f64_to_bits(c["K"][0]), f64_to_bits(c["V"][0])
        kc[b, :, :P].copy_(bits_to_cuda(Kb))
        vc[b, :, :P].copy_(bits_to_cuda(Vb))
        refs[b] = (synth.bf16_bits_to_f64(Kb)[None], synth.bf16_bits_to_f64(Vb)[None])
    x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST)
    out = torch.empty_like(x)
    delta = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE, B, P)
    m.mla_decode(W[1], x, P, kc, vc, out, ws, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    xn = synth.bf16_bits_to_f64(synth.tensor_bits(0, "new_x", (B, D), synth.X_DIST))
    for b in samples:
        ref = om.decode(W[2], xn[b:b + 1], *refs[b])
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"decode out b={b}")
        parity(cuda_to_f64(delta[b:b + 1]), ref["delta"], f"decode delta b={b}")
        parity_cache(cuda_to_f64(kc[b:b + 1, :, P]), ref["k_new"], f"new K row b={b}")
        parity_cache(cuda_to_f64(vc[b:b + 1, :, P]), ref["v_new"], f"new V row b={b}")


def test_decode_latent_b128_p8192(W):
    import torch
    B, P = 128, 8192
    cap = P + 1
    ckv, kpe = _fill_caches(W, B, P, cap, rebuilt=False)
    samples = [0, 127]
    refs = {}
    for b in samples:
        xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P, D), synth.X_DIST, rows=[b]))
        c = om.cache_from_tokens(W[2], xc)
        parity_cache(cuda_to_f64(ckv[b, :P]), c["ckv"][0], f"GPU-filled latent cache b={b}")
        parity_cache(cuda_to_f64(kpe[b, :P]), c["kpe"][0], f"GPU-filled rotary-key cache b={b}")
        Cb, Rb = f64_to_bits(c["ckv"][0]), f64_to_bits(c["kpe"][0])
        ckv[b, :P].copy_(bits_to_cuda(Cb))
        kpe[b, :P].copy_(bits_to_cuda(Rb))
        refs[b] = (synth.bf16_bits_to_f64(Cb)[None], synth.bf16_bits_to_f64(Rb)[None])
    x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST)
    out = torch.empty_like(x)
    delta = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W[1], x, P, ckv, kpe, out, ws, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    xn = synth.bf16_bits_to_f64(synth.tensor_bits(0, "new_x", (B, D), synth.X_DIST))
    for b in samples:
        ref = om.decode_latent(W[2], xn[b:b + 1], *refs[b])
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"latent decode out b={b}")
        parity(cuda_to_f64(delta[b:b + 1]), ref["delta"], f"latent decode delta b={b}")
        parity_cache(cuda_to_f64(ckv[b:b + 1, P]), ref["ckv_new"], f"new latent row b={b}")
        parity_cache(cuda_to_f64(kpe[b:b + 1, P]), ref["kpe_new"], f"new rotary-key row b={b}")


def test_prefill_chunk_absorbed_b32_p8188_t4(W):
    """The absorbed chunk at the bench's size: 32 sequences, 4 new tokens
    after 8188 latent-cache positions.  The GPU prefill fills every cache
    (checked against the oracle for the sampled sequences, whose rows are
    then replaced by the oracle's bits); sampled sequences' outputs and new
    cache rows against the oracle's latent chunk."""
    import torch
    B, P0, T = 32, 8188, 4
    cap = P0 + T
    ckv, kpe = _fill_caches(W, B, P0, cap, rebuilt=False)
    samples = [0, 31]
    refs = {}
    for b in samples:
        xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P0, D), synth.X_DIST, rows=[b]))
        c = om.cache_from_tokens(W[2], xc)
        parity_cache(cuda_to_f64(ckv[b, :P0]), c["ckv"][0], f"GPU-filled latent cache b={b}")
        Cb, Rb = f64_to_bits(c["ckv"][0]), f64_to_bits(c["kpe"][0])
        ckv[b, :P0].copy_(bits_to_cuda(Cb))
        kpe[b, :P0].copy_(bits_to_cuda(Rb))
        refs[b] = (synth.bf16_bits_to_f64(Cb)[None], synth.bf16_bits_to_f64(Rb)[None])
    x = synth.tensor_cuda(0, "x", (B, T, D), synth.X_DIST)
    out = torch.empty_like(x)
    ws = m.alloc_workspace(m.MODE_CHUNK_ABSORBED, B, T, cap=cap)
    m.mla_prefill_chunk_absorbed(W[1], x, P0, out, ckv, kpe, ws)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    xb = synth.bf16_bits_to_f64(synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST))
    for b in samples:
        ref = om.prefill_with_past_latent(W[2], xb[b:b + 1], *refs[b])
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"absorbed chunk out b={b}")
        parity_cache(cuda_to_f64(ckv[b:b + 1, P0:]), ref["ckv"], f"absorbed chunk latent rows b={b}")
        parity_cache(cuda_to_f64(kpe[b:b + 1, P0:]), ref["kpe"], f"absorbed chunk rotary-key rows b={b}")


def test_decode_latent_varlen_b128_pmax8192(W):
    """The bench's ragged latent decode: 128 sequences with seeded lengths
    in [1, 8192] (the first 8192, the second 1), caches of 8192 positions
    filled by the library's cache-only prefill (rows beyond a sequence's
    length must be ignored); sampled sequences' rows replaced by the
    oracle's bf16 latent rows."""
    import torch
    B, P_max = 128, 8192
    cap = P_max + 1
    lengths = varlen_lengths(B, P_max)
    ckv, kpe = _fill_caches(W, B, P_max, cap, rebuilt=False)
    samples = [0, 1, 77]
    refs = {}
    for b in samples:
        Pb = lengths[b]
        xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P_max, D), synth.X_DIST, rows=[b]))
        c = om.cache_from_tokens(W[2], xc[:, :max(Pb, 1)])
        Cb, Rb = f64_to_bits(c["ckv"][0][:Pb]), f64_to_bits(c["kpe"][0][:Pb])
        ckv[b, :Pb].copy_(bits_to_cuda(Cb))
        kpe[b, :Pb].copy_(bits_to_cuda(Rb))
        refs[b] = (synth.bf16_bits_to_f64(Cb)[None], synth.bf16_bits_to_f64(Rb)[None])
    x = synth.tensor_cuda(0, "new_x", (B, D), synth.X_DIST)
    out = torch.empty_like(x)
    P = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P_max)
    m.mla_decode_latent_varlen(W[1], x, P, P_max, ckv, kpe, out, ws)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    xn = synth.bf16_bits_to_f64(synth.tensor_bits(0, "new_x", (B, D), synth.X_DIST))
    for b in samples:
        ref = om.decode_latent(W[2], xn[b:b + 1], *refs[b])
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"ragged latent decode out b={b} (P={lengths[b]})")
        parity_cache(cuda_to_f64(ckv[b:b + 1, lengths[b]]), ref["ckv_new"], f"new latent row b={b}")


def varlen_lengths(B, P_max):
    """Seeded per-sequence positions in [1, P_max]: the first sequence at
    P_max, the second at 1, the rest uniform."""
    lengths = [int(v) for v in np.random.default_rng(7).integers(1, P_max + 1, size=B)]
    lengths[0], lengths[1] = P_max, 1
    return lengths
