"""Edge cases of the CUDA path against the oracle: the online softmax's
rescale branch, non-default parameters, and guard bands around every buffer.

* Rescale branch.  The prefill, chunk and latent-decode attention kernels
  keep a running row maximum and rescale the accumulated output only when a
  row's maximum grows by more than 8 (log2 units) over a later key tile.  On
  the default workload the log2-scaled scores have a spread of about 1.2, so
  after the first tile the maximum never grows that far.  Here the scores
  are made larger -- softmax_scale 0.5 and 1.0 (7x and 14x the default
  1/sqrt(192)), or W_q_b scaled by 8 at the default scale -- and each test
  first checks on the oracle's own scores that its inputs do cross the
  threshold after the first tile ("Mix and project" page, code excerpt:
  scores times softmax_scale, mask, float32 softmax, P.V).  Larger scores
  make the softmax peaked and Delta about 20 times larger (RMS 0.75 against
  0.04 at scale 1.0), and with it every bf16 storage error: storing Q, K, V
  in bf16 alone moves Delta by about 0.02 there.  These tests therefore take
  the oracle's bf16-storage reading (``bf16_storage=True``: the activations
  each step hands on, the probabilities and the attention output stored in
  bf16, as the page's module runs) as the reference, at the stated bound.
* Parameters away from the defaults: eps = 0.25 for all three RMSNorms and
  RoPE base 500, for prefill, chunk and both decode forms.
* Guard bands.  Outputs, caches, Delta and the workspace sit inside larger
  buffers filled with a sentinel byte; after the call every byte outside
  the region the call may write is still the sentinel, including the cache
  rows past the ones the call writes (cache capacity above the written
  length), for ragged sizes T in {3, 17, 129} and P in {1, 127}.

Tolerance as everywhere: max abs <= 2e-2 and relative Frobenius <= 1e-2 on
Delta; half a bf16 unit in the last place more for out, one for cache
entries.
"""
import numpy as np
import pytest

import synth
from oracle import mla_oracle as om
import mla_gb300 as m
from mla_testlib import (bits_to_cuda, cuda_to_f64, cuda_weights, oracle_weights, parity, parity_cache, parity_out,
                         weight_bits)
from test_parity_small import make_caches

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
D = 7168
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def W(gpu_available):
    wt = cuda_weights(0)
    return wt, m.make_weights(wt), oracle_weights(0)


@pytest.fixture(scope="module")
def W8(gpu_available):
    """The same weights with W_q_b multiplied by 8 (exact in bf16): every
    query, hence every score, is 8 times larger."""
    bits = dict(weight_bits(0))
    wq = synth.bf16_bits_to_f64(bits["w_q_b"]) * 8.0
    bits["w_q_b"] = synth.f32_to_bf16_bits(wq.astype(np.float32))
    wt = {n: bits_to_cuda(b) for n, b in bits.items()}
    wo = dict(oracle_weights(0))
    wo["w_q_b"] = wq
    return wt, m.make_weights(wt), wo


def u16(t):
    return t.detach().contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)


def torch_int16():
    import torch
    return torch.int16


# ---------------------------------------------------------------------------
# the rescale branch
# ---------------------------------------------------------------------------
def assert_crosses(g, what):
    """Enough rows of the input raise their running maximum by more than 8
    (log2 units) over a key tile after the first (a lower bound of the rows
    on which the kernel rescales: its stored maximum lags the true running
    maximum by up to 8)."""
    n = int(np.count_nonzero(g > 8.0))
    assert n >= min(20, g.size // 8) and n >= 0.005 * g.size, \
        f"{what}: only {n} of {g.size} rows cross the rescale threshold"


def max_growth_log2(scores_log2, tile, first_pos=0):
    """Per query row (last axis = keys in order): the largest increase of
    the running maximum over a key tile after the first, in log2 units.
    Key tiles start at multiples of `tile` counted from key 0; first_pos
    masks nothing (callers pass -inf for masked keys)."""
    nk = scores_log2.shape[-1]
    run = np.max(scores_log2[..., :min(tile, nk)], axis=-1)
    best = np.zeros_like(run)
    for k0 in range(tile, nk, tile):
        mx = np.max(scores_log2[..., k0:k0 + tile], axis=-1)
        best = np.maximum(best, mx - run)
        run = np.maximum(run, mx)
    return best


def prefill_scores_log2(Wo, x64, scale, P0=0, K_past=None):
    """Oracle scores in log2 units [B, H, T, P0 + T] (masked keys -inf) for
    checking that an input crosses the rescale threshold."""
    B, T, _ = x64.shape
    pos = P0 + np.arange(T)
    t = om.project_tokens(Wo, x64, pos[None, :], om.KIMI_K2, om.DEFAULT_EPS, om.DEFAULT_ROPE_BASE)
    Q = t["Q"].transpose(0, 2, 1, 3)   # [B, H, T, 192]
    K = t["K"].transpose(0, 2, 1, 3)
    if K_past is not None:
        K = np.concatenate([K_past, K], axis=2)
    s = np.einsum("bhqd,bhkd->bhqk", Q, K) * scale * LOG2E
    keys = np.arange(P0 + T)
    return np.where(keys[None, None, None, :] <= pos[None, None, :, None], s, -np.inf)


def run_prefill(Wt, B, T, params_kw, seed=0, name="x"):
    import torch
    xb = synth.tensor_bits(seed, name, (B, T, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = torch.empty_like(x)
    kc = torch.zeros((B, 64, T, 192), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, 64, T, 128), dtype=torch.bfloat16, device="cuda")
    ckv = torch.zeros((B, T, 512), dtype=torch.bfloat16, device="cuda")
    kpe = torch.zeros((B, T, 64), dtype=torch.bfloat16, device="cuda")
    delta = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill(Wt[1], x, out, ws, kc, vc, ckv, kpe, T, m.make_params(delta_out=delta, **params_kw))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    return synth.bf16_bits_to_f64(xb), out, delta, (kc, vc, ckv, kpe)


def check_prefill(Wo, x64, out, delta, caches, eps=om.DEFAULT_EPS, base=om.DEFAULT_ROPE_BASE, scale=None,
                  bf16_storage=False):
    ref = om.prefill(Wo, x64, eps=eps, base=base, scale=scale, bf16_storage=bf16_storage)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    for t, k in zip(caches, ("K", "V", "ckv", "kpe")):
        parity_cache(cuda_to_f64(t), ref[k], f"{k} cache")


@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_prefill_rescale_branch_large_scale(W, scale):
    B, T = 1, 300   # three 128-key tiles, a ragged last one
    x64, out, delta, caches = run_prefill(W, B, T, {"softmax_scale": scale})
    assert_crosses(max_growth_log2(prefill_scores_log2(W[2], x64, scale), 128), f"prefill scale {scale}")
    check_prefill(W[2], x64, out, delta, caches, scale=scale, bf16_storage=True)


def test_prefill_rescale_branch_scaled_queries(W8):
    B, T = 2, 300
    x64, out, delta, caches = run_prefill(W8, B, T, {})
    assert_crosses(max_growth_log2(prefill_scores_log2(W8[2], x64, om.default_scale()), 128), "prefill W_q_b x 8")
    check_prefill(W8[2], x64, out, delta, caches, bf16_storage=True)


@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_prefill_chunk_rescale_branch(W, scale):
    """A chunk of 300 tokens after 200 cached positions: the query tiles walk
    key tiles across the cached part and the chunk's own keys, and the
    offset diagonal crosses two tiles."""
    import torch
    B, P0, T = 1, 200, 300
    cap = P0 + T
    (Kb, Vb, Cb, Rb), (K64, V64, _, _) = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out = torch.empty_like(x)
    delta = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill_chunk(W[1], x, P0, out, kc, vc, ws, params=m.make_params(delta_out=delta, softmax_scale=scale))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    x64 = synth.bf16_bits_to_f64(xb)
    assert_crosses(max_growth_log2(prefill_scores_log2(W[2], x64, scale, P0, K64), 128), f"chunk scale {scale}")
    ref = om.prefill_with_past(W[2], x64, K64, V64, scale=scale, bf16_storage=True)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P0:]), ref["K"], "new K rows")
    parity_cache(cuda_to_f64(vc[:, :, P0:]), ref["V"], "new V rows")


def seeded_latent_caches(B, P, cap, seed):
    """Latent caches of seeded values: c^KV-hat ~ N(0, 1) (the normalised
    latent has unit RMS times its gain) and k^R ~ N(0, 1.7) (an unnormalised
    rotary key of the synthetic workload)."""
    Cb = synth.tensor_bits(seed, "cache_x", (B, cap, 512), (0.0, 1.0))
    Rb = synth.tensor_bits(seed + 1, "cache_x", (B, cap, 64), (0.0, 1.7))
    return Cb, Rb


def latent_scores_log2(Wo, x_new64, C64, R64, P, scale):
    """Oracle scores of the new tokens against the rebuilt keys, log2 units [B, H, P + 1]."""
    t = om.project_tokens(Wo, x_new64, np.full((x_new64.shape[0],), P), om.KIMI_K2, om.DEFAULT_EPS,
                          om.DEFAULT_ROPE_BASE)
    K, _ = om.rebuild_kv(Wo, C64, R64)
    Kn = np.concatenate([K, t["K"][:, :, None]], axis=2)   # [B, H, P + 1, 192]
    return np.einsum("bhd,bhkd->bhk", t["Q"], Kn) * scale * LOG2E


@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_decode_latent_rescale_branch(W, scale):
    """32 sequences of 2048 keys: 32 tiles of 64 keys each, cut into one
    range per SM (about 7 tiles each), so the branch runs inside the
    persistent CTAs' online softmax and the merge combines partials of
    sequences cut between CTAs.  The oracle (rebuild then attend) runs on
    sampled sequences."""
    import torch
    B, P = 32, 2047
    cap = P + 1
    Cb, Rb = seeded_latent_caches(B, P, cap, 40)
    xb = synth.tensor_bits(4, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    delta = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W[1], x, P, ckv, kpe, out, ws, m.make_params(delta_out=delta, softmax_scale=scale))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    f = synth.bf16_bits_to_f64
    for b in [0, 5, 17, 31]:
        sl = slice(b, b + 1)
        C64, R64 = f(Cb[sl, :P]), f(Rb[sl, :P])
        if b == 0:
            assert_crosses(max_growth_log2(latent_scores_log2(W[2], f(xb[sl]), C64, R64, P, scale), 64),
                           f"latent decode scale {scale}")
        ref = om.decode_latent_absorbed(W[2], f(xb[sl]), C64, R64, scale=scale, bf16_storage=True)
        parity(cuda_to_f64(delta[sl]), ref["delta"], f"delta b={b}")
        parity_out(cuda_to_f64(out[sl]), ref["out"], f"out b={b}")
        parity_cache(cuda_to_f64(ckv[sl, P]), ref["ckv_new"], f"new latent row b={b}")


def test_decode_latent_rescale_branch_scaled_queries(W8):
    import torch
    B, P = 4, 1000
    cap = P + 1
    Cb, Rb = seeded_latent_caches(B, P, cap, 41)
    xb = synth.tensor_bits(5, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = torch.empty_like(x)
    delta = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W8[1], x, P, bits_to_cuda(Cb), bits_to_cuda(Rb), out, ws, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    f = synth.bf16_bits_to_f64
    ref = om.decode_latent_absorbed(W8[2], f(xb), f(Cb[:, :P]), f(Rb[:, :P]), bf16_storage=True)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")


@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_decode_rebuilt_large_scale_split_combine(W, scale):
    """Rebuilt-cache decode, B=4 P=1000 (the split-KV path: several splits
    per (sequence, head) merged by the log-sum-exp combine), on seeded
    caches (K ~ N(0, 1), V ~ N(0, 0.5)).  This kernel rescales on every
    key chunk (no threshold); the large scale checks its combine of
    partials whose maxima differ widely."""
    import torch
    B, P = 4, 1000
    cap = P + 1
    Kb = synth.tensor_bits(42, "cache_x", (B, 64, cap, 192), (0.0, 1.0))
    Vb = synth.tensor_bits(43, "cache_x", (B, 64, cap, 128), (0.0, 0.5))
    xb = synth.tensor_bits(6, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out = torch.empty_like(x)
    delta = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_DECODE, B, P)
    m.mla_decode(W[1], x, P, kc, vc, out, ws, m.make_params(delta_out=delta, softmax_scale=scale))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws) == 0
    f = synth.bf16_bits_to_f64
    ref = om.decode(W[2], f(xb), f(Kb[:, :, :P]), f(Vb[:, :, :P]), scale=scale, bf16_storage=True)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P]), ref["k_new"], "new K row")


# ---------------------------------------------------------------------------
# parameters away from the defaults
# ---------------------------------------------------------------------------
EPS, BASE = 0.25, 500.0


def test_prefill_nondefault_eps_and_rope_base(W):
    x64, out, delta, caches = run_prefill(W, 2, 129, {"eps": EPS, "rope_base": BASE})
    check_prefill(W[2], x64, out, delta, caches, eps=EPS, base=BASE)
    # the parameters matter: the default-parameter oracle is far off
    ref0 = om.prefill(W[2], x64)
    assert np.max(np.abs(cuda_to_f64(delta) - ref0["delta"])) > 0.1


def test_prefill_chunk_nondefault_eps_and_rope_base(W):
    import torch
    B, P0, T = 2, 700, 40   # positions up to 739: rotary angles of several turns at base 500
    cap = P0 + T
    (Kb, Vb, _, _), (K64, V64, _, _) = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out = torch.empty_like(x)
    delta = torch.empty((B, T, D), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill_chunk(W[1], x, P0, out, kc, vc, ws, params=m.make_params(delta_out=delta, eps=EPS, rope_base=BASE))
    torch.cuda.synchronize()
    ref = om.prefill_with_past(W[2], synth.bf16_bits_to_f64(xb), K64, V64, eps=EPS, base=BASE)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P0:]), ref["K"], "new K rows")


def test_decode_both_forms_nondefault_eps_and_rope_base(W):
    import torch
    B, P = 3, 900
    cap = P + 1
    Cb, Rb = seeded_latent_caches(B, P, cap, 44)
    Kb = synth.tensor_bits(45, "cache_x", (B, 64, cap, 192), (0.0, 1.0))
    Vb = synth.tensor_bits(46, "cache_x", (B, 64, cap, 128), (0.0, 0.5))
    xb = synth.tensor_bits(7, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    f = synth.bf16_bits_to_f64
    prm = dict(eps=EPS, rope_base=BASE)
    # rebuilt cache
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out, delta = torch.empty_like(x), torch.empty((B, D), dtype=torch.float32, device="cuda")
    m.mla_decode(W[1], x, P, kc, vc, out, m.alloc_workspace(m.MODE_DECODE, B, P), m.make_params(delta_out=delta, **prm))
    torch.cuda.synchronize()
    ref = om.decode(W[2], f(xb), f(Kb[:, :, :P]), f(Vb[:, :, :P]), eps=EPS, base=BASE)
    parity(cuda_to_f64(delta), ref["delta"], "rebuilt delta")
    parity_cache(cuda_to_f64(kc[:, :, P]), ref["k_new"], "rebuilt new K row")
    # latent cache
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out, delta = torch.empty_like(x), torch.empty((B, D), dtype=torch.float32, device="cuda")
    m.mla_decode_latent(W[1], x, P, ckv, kpe, out, m.alloc_workspace(m.MODE_DECODE_LATENT, B, P),
                        m.make_params(delta_out=delta, **prm))
    torch.cuda.synchronize()
    ref = om.decode_latent(W[2], f(xb), f(Cb[:, :P]), f(Rb[:, :P]), eps=EPS, base=BASE)
    parity(cuda_to_f64(delta), ref["delta"], "latent delta")
    parity_out(cuda_to_f64(out), ref["out"], "latent out")
    parity_cache(cuda_to_f64(kpe[:, P]), ref["kpe_new"], "latent new rotary-key row")


# ---------------------------------------------------------------------------
# guard bands
# ---------------------------------------------------------------------------
GUARD = 4096   # bytes on each side (a multiple of 256, so the inner region keeps its alignment)


class Guarded:
    """A tensor of `shape` / `dtype` inside a byte buffer of sentinel bytes
    with GUARD bytes before and after it.  fill = None leaves the tensor's
    own bytes at the sentinel too."""

    def __init__(self, shape, dtype, fill=None):
        import torch
        self.shape, self.dtype = tuple(shape), dtype
        self.nbytes = int(np.prod(self.shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(self.shape)
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:GUARD] == SENTINEL) and np.all(b[GUARD + self.nbytes:] == SENTINEL))


def guarded_workspace(mode, B, t_or_p, cap=0):
    import torch
    g = Guarded((m.workspace_size(mode, B, t_or_p, cap),), torch.uint8)
    return g


def sentinel_rows(t, axis, start):
    """The cache rows from `start` on along `axis` still hold the sentinel bytes."""
    import torch
    idx = [slice(None)] * t.dim()
    idx[axis] = slice(start, None)
    rows = t[tuple(idx)].contiguous().view(torch.uint8)
    return bool(torch.all(rows == SENTINEL).item())


@pytest.mark.parametrize("B,T", [(1, 3), (2, 17), (1, 129)])
def test_prefill_guard_bands(W, B, T):
    import torch
    cap = T + 2
    xb = synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST)
    x = Guarded((B, T, D), torch.bfloat16, bits_to_cuda(xb))
    out = Guarded((B, T, D), torch.bfloat16)
    delta = Guarded((B, T, D), torch.float32)
    kc = Guarded((B, 64, cap, 192), torch.bfloat16)
    vc = Guarded((B, 64, cap, 128), torch.bfloat16)
    ckv = Guarded((B, cap, 512), torch.bfloat16)
    kpe = Guarded((B, cap, 64), torch.bfloat16)
    ws = guarded_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill(W[1], x.t, out.t, ws.t, kc.t, vc.t, ckv.t, kpe.t, cap, m.make_params(delta_out=delta.t))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws.t) == 0
    for g, name in [(x, "x"), (out, "out"), (delta, "delta"), (kc, "K"), (vc, "V"), (ckv, "latent"),
                    (kpe, "rotary key"), (ws, "workspace")]:
        assert g.guards_intact(), f"{name}: bytes outside the buffer changed"
    assert np.array_equal(u16(x.t), xb), "x changed"
    for g, ax, name in [(kc, 2, "K"), (vc, 2, "V"), (ckv, 1, "latent"), (kpe, 1, "rotary key")]:
        assert sentinel_rows(g.t, ax, T), f"{name}: rows at or past T written"
    ref = om.prefill(W[2], synth.bf16_bits_to_f64(xb))
    parity(cuda_to_f64(delta.t), ref["delta"], "delta")
    parity_out(cuda_to_f64(out.t), ref["out"], "out")
    parity_cache(cuda_to_f64(kc.t[:, :, :T]), ref["K"], "K cache")
    parity_cache(cuda_to_f64(ckv.t[:, :T]), ref["ckv"], "latent cache")


@pytest.mark.parametrize("B,P0,T", [(1, 5, 3), (2, 127, 17)])
def test_prefill_chunk_guard_bands(W, B, P0, T):
    import torch
    cap = P0 + T + 2
    (Kb, Vb, Cb, Rb), (K64, V64, _, _) = make_caches(W, B, P0, cap)
    xb = synth.tensor_bits(0, "x", (B, T, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = Guarded((B, T, D), torch.bfloat16)
    kc = Guarded((B, 64, cap, 192), torch.bfloat16)
    vc = Guarded((B, 64, cap, 128), torch.bfloat16)
    kc.t[:, :, :P0] = bits_to_cuda(Kb[:, :, :P0])
    vc.t[:, :, :P0] = bits_to_cuda(Vb[:, :, :P0])
    ws = guarded_workspace(m.MODE_PREFILL, B, T)
    m.mla_prefill_chunk(W[1], x, P0, out.t, kc.t, vc.t, ws.t)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws.t) == 0
    for g, name in [(out, "out"), (kc, "K"), (vc, "V"), (ws, "workspace")]:
        assert g.guards_intact(), f"{name}: bytes outside the buffer changed"
    assert sentinel_rows(kc.t, 2, P0 + T) and sentinel_rows(vc.t, 2, P0 + T), "rows past P0 + T written"
    ref = om.prefill_with_past(W[2], synth.bf16_bits_to_f64(xb), K64, V64)
    parity_out(cuda_to_f64(out.t), ref["out"], "out")
    parity_cache(cuda_to_f64(kc.t[:, :, P0:P0 + T]), ref["K"], "new K rows")


@pytest.mark.parametrize("B,P", [(3, 1), (2, 127)])
def test_decode_guard_bands(W, B, P):
    import torch
    cap = P + 3
    (Kb, Vb, _, _), (K64, V64, _, _) = make_caches(W, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = Guarded((B, D), torch.bfloat16)
    delta = Guarded((B, D), torch.float32)
    kc = Guarded((B, 64, cap, 192), torch.bfloat16)
    vc = Guarded((B, 64, cap, 128), torch.bfloat16)
    kc.t[:, :, :P] = bits_to_cuda(Kb[:, :, :P])
    vc.t[:, :, :P] = bits_to_cuda(Vb[:, :, :P])
    ws = guarded_workspace(m.MODE_DECODE, B, P)
    m.mla_decode(W[1], x, P, kc.t, vc.t, out.t, ws.t, m.make_params(delta_out=delta.t))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws.t) == 0
    for g, name in [(out, "out"), (delta, "delta"), (kc, "K"), (vc, "V"), (ws, "workspace")]:
        assert g.guards_intact(), f"{name}: bytes outside the buffer changed"
    assert sentinel_rows(kc.t, 2, P + 1) and sentinel_rows(vc.t, 2, P + 1), "rows past P written"
    ref = om.decode(W[2], synth.bf16_bits_to_f64(xb), K64, V64)
    parity(cuda_to_f64(delta.t), ref["delta"], "delta")
    parity_cache(cuda_to_f64(kc.t[:, :, P]), ref["k_new"], "new K row")


@pytest.mark.parametrize("B,P", [(3, 1), (2, 127)])
def test_decode_latent_guard_bands(W, B, P):
    import torch
    cap = P + 3
    (_, _, Cb, Rb), (_, _, C64, R64) = make_caches(W, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, D), synth.X_DIST)
    x = bits_to_cuda(xb)
    out = Guarded((B, D), torch.bfloat16)
    ckv = Guarded((B, cap, 512), torch.bfloat16)
    kpe = Guarded((B, cap, 64), torch.bfloat16)
    ckv.t[:, :P] = bits_to_cuda(Cb[:, :P])
    kpe.t[:, :P] = bits_to_cuda(Rb[:, :P])
    ws = guarded_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent(W[1], x, P, ckv.t, kpe.t, out.t, ws.t)
    torch.cuda.synchronize()
    assert m.mla_device_status(ws.t) == 0
    for g, name in [(out, "out"), (ckv, "latent"), (kpe, "rotary key"), (ws, "workspace")]:
        assert g.guards_intact(), f"{name}: bytes outside the buffer changed"
    assert sentinel_rows(ckv.t, 1, P + 1) and sentinel_rows(kpe.t, 1, P + 1), "rows past P written"
    ref = om.decode_latent(W[2], synth.bf16_bits_to_f64(xb), C64, R64)
    parity_out(cuda_to_f64(out.t), ref["out"], "out")
    parity_cache(cuda_to_f64(ckv.t[:, P]), ref["ckv_new"], "new latent row")


@pytest.mark.parametrize("n", [3, 17, 129])
def test_ffn_guard_bands(gpu_available, n):
    import torch
    from mla_testlib import cuda_ffn_weights
    WF = m.make_ffn_weights(cuda_ffn_weights(0))
    x = synth.tensor_cuda(0, "ffn_x", (n, D), synth.X_DIST)
    out = Guarded((n, D), torch.bfloat16)
    delta = Guarded((n, D), torch.float32)
    ws = guarded_workspace(m.MODE_FFN, 1, n)
    m.mla_ffn(WF, x, out.t, ws.t, m.make_params(delta_out=delta.t))
    torch.cuda.synchronize()
    assert m.mla_device_status(ws.t) == 0
    for g, name in [(out, "out"), (delta, "delta"), (ws, "workspace")]:
        assert g.guards_intact(), f"{name}: bytes outside the buffer changed"
    assert torch.isfinite(delta.t).all()
