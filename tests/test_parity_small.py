"""CUDA path vs the CPU oracle at sizes the oracle finishes in seconds.

Full Kimi K2 dimensions (d = 7168, 64 heads, ...); seeded synthetic inputs
from ``synth`` on both sides; tolerance max abs <= 2e-2 and relative
Frobenius <= 1e-2 on out, Delta_attn (o_proj output before the residual)
and every cache the call writes, plus the rounding of bf16 storage (half a
unit in the last place for out, one for cache entries).  Shapes span several GEMM tiles (128 rows)
and attention tiles with ragged tails, plus the degenerate cases T = 1,
P = 0 and out aliasing x.
"""
import numpy as np
import pytest

import synth
from oracle import mla_oracle as om
import mla_gb300 as m
from mla_testlib import (bits_to_cuda, cuda_to_f64, cuda_weights, f64_to_bits, oracle_weights, parity,
                         parity_cache, parity_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def W(gpu_available):
    wt = cuda_weights(0)
    return wt, m.make_weights(wt), oracle_weights(0)


def run_prefill(W, B, T, with_cache=True, cap=None, inplace=False):
    import torch
    wt, ws_struct, _ = W
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = x.clone() if inplace else torch.empty_like(x)
    cap = cap or T
    kc = torch.zeros((B, 64, cap, 192), dtype=torch.bfloat16, device="cuda") if with_cache else None
    vc = torch.zeros((B, 64, cap, 128), dtype=torch.bfloat16, device="cuda") if with_cache else None
    ckv = torch.zeros((B, cap, 512), dtype=torch.bfloat16, device="cuda") if with_cache else None
    kpe = torch.zeros((B, cap, 64), dtype=torch.bfloat16, device="cuda") if with_cache else None
    delta = torch.empty((B, T, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_PREFILL, B, T)
    params = m.make_params(delta_out=delta)
    m.mla_prefill(ws_struct, out if inplace else x, out, wsp, kc, vc, ckv, kpe, cap if with_cache else 0, params)
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    return synth.bf16_bits_to_f64(xb), out, delta, kc, vc, ckv, kpe


@pytest.mark.parametrize("B,T", [(1, 16), (2, 300), (1, 1), (3, 129)])
def test_prefill_parity(W, B, T):
    x64, out, delta, kc, vc, ckv, kpe = run_prefill(W, B, T)
    ref = om.prefill(W[2], x64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc), ref["K"], "K cache")
    parity_cache(cuda_to_f64(vc), ref["V"], "V cache")
    parity_cache(cuda_to_f64(ckv), ref["ckv"], "latent cache")
    parity_cache(cuda_to_f64(kpe), ref["kpe"], "rotary-key cache")


def test_prefill_in_place_and_no_cache(W):
    B, T = 1, 70
    x64, out, delta, *_ = run_prefill(W, B, T, with_cache=False, inplace=True)
    ref = om.prefill(W[2], x64)
    parity_out(cuda_to_f64(out), ref["out"], "out (in place)")
    parity(cuda_to_f64(delta), ref["delta"], "delta")


def test_prefill_cache_capacity_larger_than_T(W):
    import torch
    B, T, cap = 2, 40, 100
    x64, out, delta, kc, vc, ckv, kpe = run_prefill(W, B, T, cap=cap)
    ref = om.prefill(W[2], x64)
    parity_cache(cuda_to_f64(kc[:, :, :T]), ref["K"], "K cache")
    parity_cache(cuda_to_f64(ckv[:, :T]), ref["ckv"], "latent cache")
    assert torch.count_nonzero(kc[:, :, T:]).item() == 0
    assert torch.count_nonzero(ckv[:, T:]).item() == 0


def make_caches(W, B, P, cap):
    """Caches of positions 0..P-1 built by the oracle from seeded tokens and
    rounded to bf16 storage; identical bits go to both sides."""
    import torch
    wo = W[2]
    xc = synth.bf16_bits_to_f64(synth.tensor_bits(0, "cache_x", (B, P, 7168), synth.X_DIST)) if P else None
    Kb = np.zeros((B, 64, cap, 192), np.uint16)
    Vb = np.zeros((B, 64, cap, 128), np.uint16)
    Cb = np.zeros((B, cap, 512), np.uint16)
    Rb = np.zeros((B, cap, 64), np.uint16)
    if P:
        c = om.cache_from_tokens(wo, xc)
        Kb[:, :, :P] = f64_to_bits(c["K"])
        Vb[:, :, :P] = f64_to_bits(c["V"])
        Cb[:, :P] = f64_to_bits(c["ckv"])
        Rb[:, :P] = f64_to_bits(c["kpe"])
    f = synth.bf16_bits_to_f64
    return (Kb, Vb, Cb, Rb), (f(Kb[:, :, :P]), f(Vb[:, :, :P]), f(Cb[:, :P]), f(Rb[:, :P]))


@pytest.mark.parametrize("B,P", [(3, 37), (2, 0), (1, 300), (5, 1)])
def test_decode_parity(W, B, P):
    import torch
    cap = P + 3
    (Kb, Vb, _, _), (K64, V64, _, _) = make_caches(W, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE, B, P)
    m.mla_decode(W[1], x, P, kc, vc, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.decode(W[2], synth.bf16_bits_to_f64(xb), K64, V64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P]), ref["k_new"], "new K row")
    parity_cache(cuda_to_f64(vc[:, :, P]), ref["v_new"], "new V row")
    # positions other than P are untouched
    assert np.array_equal(kc[:, :, :P].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), Kb[:, :, :P])


@pytest.mark.parametrize("B,P", [(3, 37), (2, 0), (1, 300), (4, 129)])
def test_decode_latent_parity(W, B, P):
    import torch
    cap = P + 2
    (_, _, Cb, Rb), (_, _, C64, R64) = make_caches(W, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W[1], x, P, ckv, kpe, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.decode_latent(W[2], synth.bf16_bits_to_f64(xb), C64, R64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(ckv[:, P]), ref["ckv_new"], "new latent row")
    parity_cache(cuda_to_f64(kpe[:, P]), ref["kpe_new"], "new rotary-key row")


def test_decode_latent_many_sequences(W):
    """B=500, P=70 (two 64-key tiles per sequence): each CTA's range of tiles
    covers the end of one sequence, whole sequences and the start of another,
    so the direct writes and the merged partials are both exercised.  The
    caches hold seeded bf16 values; the oracle runs on sampled sequences."""
    import torch
    B, P = 500, 70
    cap = P + 1
    Cb = synth.tensor_bits(0, "cache_x", (B, cap, 512), (0.0, 1.0))
    Rb = synth.tensor_bits(1, "cache_x", (B, cap, 64), (0.0, 1.7))
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    wsp = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W[1], x, P, ckv, kpe, out, wsp)
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    f = synth.bf16_bits_to_f64
    for b in [0, 1, 2, 3, 4, 131, 132, 133, 250, 251, 497, 498, 499]:
        ref = om.decode_latent(W[2], f(xb[b:b + 1]), f(Cb[b:b + 1, :P]), f(Rb[b:b + 1, :P]))
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"out b={b}")


@pytest.mark.parametrize("B,P0,T", [(2, 100, 37), (1, 128, 256), (1, 200, 300), (2, 0, 40), (3, 5, 1)])
def test_prefill_chunk_parity(W, B, P0, T):
    """Chunk of T tokens after P0 cached positions (oracle-built bf16 caches
    on both sides): past % 128 != 0 puts the offset diagonal across two key
    tiles; P0 = 0 is the plain prefill; T = 1 is a one-token chunk."""
    import torch
    cap = P0 + T + 3
    (Kb, Vb, Cb, Rb), (K64, V64, _, _) = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc, ckv, kpe = (bits_to_cuda(t) for t in (Kb, Vb, Cb, Rb))
    out = torch.empty_like(x)
    delta = torch.empty((B, T, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill_chunk(W[1], x, P0, out, kc, vc, wsp, ckv, kpe, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.prefill_with_past(W[2], synth.bf16_bits_to_f64(xb), K64, V64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P0:P0 + T]), ref["K"], "new K rows")
    parity_cache(cuda_to_f64(vc[:, :, P0:P0 + T]), ref["V"], "new V rows")
    parity_cache(cuda_to_f64(ckv[:, P0:P0 + T]), ref["ckv"], "new latent rows")
    parity_cache(cuda_to_f64(kpe[:, P0:P0 + T]), ref["kpe"], "new rotary-key rows")
    # rows before P0 and after P0 + T are untouched
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(kc[:, :, :P0]), Kb[:, :, :P0])
    assert np.array_equal(bits(vc[:, :, :P0]), Vb[:, :, :P0])
    assert np.array_equal(bits(ckv[:, :P0]), Cb[:, :P0])
    assert torch.count_nonzero(kc[:, :, P0 + T:]).item() == 0
    assert torch.count_nonzero(ckv[:, P0 + T:]).item() == 0


def test_prefill_in_two_chunks_equals_whole_prefill(W):
    """GPU prefill of the first T1 tokens, then a GPU chunk of the next T2
    from the caches it wrote: every output row matches the oracle's prefill
    of all T1 + T2 tokens."""
    import torch
    B, T1, T2 = 2, 70, 90
    T = T1 + T2
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc = torch.zeros((B, 64, T, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, T, 128), dtype=torch.bfloat16, device="cuda")
    x1, x2 = x[:, :T1].contiguous(), x[:, T1:].contiguous()
    o1, o2 = torch.empty_like(x1), torch.empty_like(x2)
    m.mla_prefill(W[1], x1, o1, m.alloc_workspace(m.MODE_PREFILL, B, T1), kc, vc, None, None, T)
    m.mla_prefill_chunk(W[1], x2, T1, o2, kc, vc, m.alloc_workspace(m.MODE_PREFILL, B, T2))
    torch.cuda.synchronize()
    ref = om.prefill(W[2], synth.bf16_bits_to_f64(xb))
    parity_out(cuda_to_f64(torch.cat([o1, o2], dim=1)), ref["out"], "two chunks")
    parity_cache(cuda_to_f64(kc), ref["K"], "K cache")


@pytest.mark.parametrize("B,P0,T", [(2, 100, 37), (1, 128, 256), (2, 0, 40), (1, 300, 1)])
def test_prefill_chunk_latent_parity(W, B, P0, T):
    """Chunk against the latent cache (oracle-built bf16 latent rows on both
    sides): the past keys and values are rebuilt from the cache."""
    import torch
    cap = P0 + T + 5
    (_, _, Cb, Rb), (_, _, C64, R64) = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    delta = torch.empty((B, T, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_CHUNK_LATENT, B, T, cap=cap)
    m.mla_prefill_chunk_latent(W[1], x, P0, out, ckv, kpe, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.prefill_with_past_latent(W[2], synth.bf16_bits_to_f64(xb), C64, R64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(ckv[:, P0:P0 + T]), ref["ckv"], "new latent rows")
    parity_cache(cuda_to_f64(kpe[:, P0:P0 + T]), ref["kpe"], "new rotary-key rows")
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(ckv[:, :P0]), Cb[:, :P0])
    assert np.array_equal(bits(kpe[:, :P0]), Rb[:, :P0])
    assert torch.count_nonzero(ckv[:, P0 + T:]).item() == 0


@pytest.mark.parametrize("B,P0,T", [(2, 100, 3), (1, 128, 1), (2, 0, 40), (3, 300, 5), (1, 63, 130)])
def test_prefill_chunk_absorbed_parity(W, B, P0, T):
    """The absorbed form of the latent chunk (W_UK into the query, W_UV
    after the attention, the cache never expanded) against the same oracle
    as the rebuilt form: the two compute the same values.  Rows past the
    chunk hold noise that must not be read."""
    import torch
    cap = P0 + T + 70
    (_, _, Cb, Rb), (_, _, C64, R64) = make_caches(W, B, P0, cap)
    noise = synth.tensor_bits(3, "cache_x", (B, cap, 576), (0.0, 4.0))
    Cb[:, P0 + T:] = noise[:, P0 + T:, :512]
    Rb[:, P0 + T:] = noise[:, P0 + T:, 512:]
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    delta = torch.empty((B, T, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_CHUNK_ABSORBED, B, T, cap=cap)
    m.mla_prefill_chunk_absorbed(W[1], x, P0, out, ckv, kpe, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.prefill_with_past_latent(W[2], synth.bf16_bits_to_f64(xb), C64[:, :P0], R64[:, :P0])
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(ckv[:, P0:P0 + T]), ref["ckv"], "new latent rows")
    parity_cache(cuda_to_f64(kpe[:, P0:P0 + T]), ref["kpe"], "new rotary-key rows")
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(ckv[:, :P0]), Cb[:, :P0])
    assert np.array_equal(bits(ckv[:, P0 + T:]), Cb[:, P0 + T:])


def test_prefill_chunk_absorbed_matches_rebuilt_form(W):
    """Same chunk through both latent-cache forms on the GPU: outputs and the
    cache rows written agree to rounding (the absorbed form's A-projection
    runs split-K, the rebuilt form's does not, so the fp32 sums are added in
    a different order)."""
    import torch
    B, P0, T = 2, 200, 4
    cap = P0 + T
    (_, _, Cb, Rb), _ = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    c1, r1 = bits_to_cuda(Cb), bits_to_cuda(Rb)
    c2, r2 = c1.clone(), r1.clone()
    o1, o2 = torch.empty_like(x), torch.empty_like(x)
    m.mla_prefill_chunk_latent(W[1], x, P0, o1, c1, r1, m.alloc_workspace(m.MODE_CHUNK_LATENT, B, T, cap=cap))
    m.mla_prefill_chunk_absorbed(W[1], x, P0, o2, c2, r2, m.alloc_workspace(m.MODE_CHUNK_ABSORBED, B, T, cap=cap))
    torch.cuda.synchronize()
    parity_cache(cuda_to_f64(c2), cuda_to_f64(c1), "latent rows")
    parity_cache(cuda_to_f64(r2), cuda_to_f64(r1), "rotary-key rows")
    parity_out(cuda_to_f64(o2), cuda_to_f64(o1), "absorbed against rebuilt")


def test_latent_prefill_then_latent_chunk_equals_whole_prefill(W):
    """GPU prefill writes the latent cache of the first T1 tokens, a GPU
    latent chunk runs the next T2: every output row matches the oracle's
    prefill of all T1 + T2 tokens."""
    import torch
    B, T1, T2 = 2, 70, 90
    T = T1 + T2
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv = torch.zeros((B, T, 512), dtype=torch.bfloat16, device="cuda")
    kpe = torch.zeros((B, T, 64), dtype=torch.bfloat16, device="cuda")
    x1, x2 = x[:, :T1].contiguous(), x[:, T1:].contiguous()
    o1, o2 = torch.empty_like(x1), torch.empty_like(x2)
    m.mla_prefill(W[1], x1, o1, m.alloc_workspace(m.MODE_PREFILL, B, T1), None, None, ckv, kpe, T)
    m.mla_prefill_chunk_latent(W[1], x2, T1, o2, ckv, kpe, m.alloc_workspace(m.MODE_CHUNK_LATENT, B, T2, cap=T))
    torch.cuda.synchronize()
    ref = om.prefill(W[2], synth.bf16_bits_to_f64(xb))
    parity_out(cuda_to_f64(torch.cat([o1, o2], dim=1)), ref["out"], "two chunks, latent cache")
    parity_cache(cuda_to_f64(ckv), ref["ckv"], "latent cache")


def test_prefill_chunk_rejects_bad_arguments(W):
    import torch
    B, T, P0 = 1, 8, 10
    x = torch.zeros((B, T, 7168), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    kc = torch.zeros((B, 64, P0 + T, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, P0 + T, 128), dtype=torch.bfloat16, device="cuda")
    wsp = m.alloc_workspace(m.MODE_PREFILL, B, T)
    for bad_p0 in (-1, P0 + 1):  # negative, or P0 + T beyond the cache capacity
        with pytest.raises(m.MlaError):
            m.mla_prefill_chunk(W[1], x, bad_p0, out, kc, vc, wsp)
    with pytest.raises(m.MlaError):
        m.mla_prefill_chunk(W[1], x, P0, None, kc, vc, wsp)


LENGTHS = [0, 37, 300, 1, 129]  # a ragged batch: P_b per sequence (P_max = 300)


def _ragged_caches(W, lengths, cap):
    """Oracle caches of P_max seeded tokens per sequence, with rows at or
    beyond each sequence's own length overwritten by noise (they must not
    be read)."""
    B, P_max = len(lengths), max(lengths)
    (Kb, Vb, Cb, Rb), _ = make_caches(W, B, P_max, cap)
    noise = synth.tensor_bits(3, "cache_x", (B, cap, 640), (0.0, 4.0))
    for b, P in enumerate(lengths):
        Kb[b, :, P:] = noise[b, None, P:, :192]
        Vb[b, :, P:] = noise[b, None, P:, 192:320]
        Cb[b, P:] = noise[b, P:, :512]
        Rb[b, P:] = noise[b, P:, 512:576]
    return Kb, Vb, Cb, Rb


def test_decode_varlen_parity(W):
    import torch
    B, P_max = len(LENGTHS), max(LENGTHS)
    cap = P_max + 2
    Kb, Vb, _, _ = _ragged_caches(W, LENGTHS, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    P = torch.tensor(LENGTHS, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE, B, P_max)
    m.mla_decode_varlen(W[1], x, P, P_max, kc, vc, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    f = synth.bf16_bits_to_f64
    ref = om.decode_varlen(W[2], f(xb), f(Kb), f(Vb), LENGTHS)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    kn, vn = bits(kc), bits(vc)
    for b, Pb in enumerate(LENGTHS):
        parity_cache(cuda_to_f64(kc[b:b + 1, :, Pb]), ref["k_new"][b:b + 1], f"new K row b={b}")
        parity_cache(cuda_to_f64(vc[b:b + 1, :, Pb]), ref["v_new"][b:b + 1], f"new V row b={b}")
        # every other row untouched
        assert np.array_equal(np.delete(kn[b], Pb, axis=1), np.delete(Kb[b], Pb, axis=1))
        assert np.array_equal(np.delete(vn[b], Pb, axis=1), np.delete(Vb[b], Pb, axis=1))


def test_decode_latent_varlen_parity(W):
    import torch
    B, P_max = len(LENGTHS), max(LENGTHS)
    cap = P_max + 2
    _, _, Cb, Rb = _ragged_caches(W, LENGTHS, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    P = torch.tensor(LENGTHS, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P_max)
    m.mla_decode_latent_varlen(W[1], x, P, P_max, ckv, kpe, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    f = synth.bf16_bits_to_f64
    ref = om.decode_latent_varlen(W[2], f(xb), f(Cb), f(Rb), LENGTHS)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    cn = bits(ckv)
    for b, Pb in enumerate(LENGTHS):
        parity_cache(cuda_to_f64(ckv[b:b + 1, Pb]), ref["ckv_new"][b:b + 1], f"new latent row b={b}")
        parity_cache(cuda_to_f64(kpe[b:b + 1, Pb]), ref["kpe_new"][b:b + 1], f"new rotary-key row b={b}")
        assert np.array_equal(np.delete(cn[b], Pb, axis=0), np.delete(Cb[b], Pb, axis=0))


def test_decode_latent_varlen_many_short_sequences(W):
    """B=300 sequences of 1 to 200 keys: most CTAs' ranges hold several
    whole sequences, some sequences are cut between CTAs."""
    import torch
    B = 300
    rng = np.random.default_rng(11)
    lengths = [int(v) for v in rng.integers(0, 200, size=B)]
    P_max = max(lengths)
    cap = P_max + 1
    Cb = synth.tensor_bits(0, "cache_x", (B, cap, 512), (0.0, 1.0))
    Rb = synth.tensor_bits(1, "cache_x", (B, cap, 64), (0.0, 1.7))
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    P = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    wsp = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P_max)
    m.mla_decode_latent_varlen(W[1], x, P, P_max, ckv, kpe, out, wsp)
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    f = synth.bf16_bits_to_f64
    for b in [0, 1, 2, 57, 150, 151, 298, 299]:
        Pb = lengths[b]
        ref = om.decode_latent(W[2], f(xb[b:b + 1]), f(Cb[b:b + 1, :Pb]), f(Rb[b:b + 1, :Pb]))
        parity_out(cuda_to_f64(out[b:b + 1]), ref["out"], f"out b={b} (P={Pb})")


def test_decode_varlen_out_of_range_length_is_reported(W):
    """A per-sequence position beyond P_max (or negative) cannot be checked
    on the host: the kernels clamp it, touch nothing outside the caches, and
    the device status reports the bad argument."""
    import torch
    B, P_max = 2, 20
    cap = P_max + 1
    kc = torch.zeros((B, 64, cap, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, cap, 128), dtype=torch.bfloat16, device="cuda")
    x = synth.tensor_cuda(0, "new_x", (B, 7168), synth.X_DIST)
    out = torch.empty_like(x)
    for bad in ([5, P_max + 7], [-3, 4]):
        P = torch.tensor(bad, dtype=torch.int32, device="cuda")
        wsp = m.alloc_workspace(m.MODE_DECODE, B, P_max)
        m.mla_decode_varlen(W[1], x, P, P_max, kc, vc, out, wsp)
        torch.cuda.synchronize()
        assert m.mla_device_status(wsp) == -1  # MLA_ERR_INVALID_ARG


def test_prefill_then_decode_chain(W):
    """GPU prefill of T-1 tokens fills the caches; GPU decode of token T-1
    must match the oracle's prefill row T-1 (both cache forms)."""
    import torch
    B, T = 2, 50
    xb = synth.tensor_bits(0, "x", (B, T, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    cap = T
    kc = torch.zeros((B, 64, cap, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, cap, 128), dtype=torch.bfloat16, device="cuda")
    ckv = torch.zeros((B, cap, 512), dtype=torch.bfloat16, device="cuda")
    kpe = torch.zeros((B, cap, 64), dtype=torch.bfloat16, device="cuda")
    xp = x[:, :T - 1].contiguous()
    outp = torch.empty_like(xp)
    m.mla_prefill(W[1], xp, outp, m.alloc_workspace(m.MODE_PREFILL, B, T - 1), kc, vc, ckv, kpe, cap)
    xn = x[:, T - 1].contiguous()
    o1 = torch.empty_like(xn)
    o2 = torch.empty_like(xn)
    m.mla_decode(W[1], xn, T - 1, kc, vc, o1, m.alloc_workspace(m.MODE_DECODE, B, T - 1))
    m.mla_decode_latent(W[1], xn, T - 1, ckv, kpe, o2, m.alloc_workspace(m.MODE_DECODE_LATENT, B, T - 1))
    torch.cuda.synchronize()
    ref = om.prefill(W[2], synth.bf16_bits_to_f64(xb), query_rows=[T - 1])["out"][:, 0]
    parity_out(cuda_to_f64(o1), ref, "decode after prefill")
    parity_out(cuda_to_f64(o2), ref, "latent decode after prefill")
