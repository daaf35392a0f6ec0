"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
* the numbers the pages print (parameter counts, cache sizes), kept in
  tests/golden/page_counts.json with their citations;
* closed forms (RMSNorm of a constant vector, RoPE of a unit vector);
* a brute-force, element-by-element loop implementation at tiny sizes
  (no max subtraction, no numpy matmul);
* an independent torch restatement that follows the layout steps of the
  pages' code (view to heads, split nope|pe and k_nope|v, transpose back);
* invariants: uniform scores give the mean of V, causal row 0 sees only
  itself, decode is invariant to permuting cached positions, prefill and
  decode agree, latent (absorbed) and rebuilt decodes agree, batch rows are
  independent.
``test_planted_mistakes`` checks that plausible mistakes planted in the
oracle do make these pins fail.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import mla_oracle as om

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_counts.json")))

TINY = om.Dims(d=16, H=2, q_lora=8, kv_lora=8, nope=4, rope=4, v=4)
TINY2 = om.Dims(d=24, H=3, q_lora=12, kv_lora=10, nope=6, rope=8, v=5)


def rand_weights(dims, seed, wstd=0.3):
    rng = np.random.default_rng(seed)
    w = {}
    for name, shape in om.weight_shapes(dims).items():
        if name.startswith("g_"):
            w[name] = 1.0 + 0.1 * rng.standard_normal(shape)
        else:
            w[name] = wstd * rng.standard_normal(shape)
    return w


def rand_x(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------
# printed numbers
# ---------------------------------------------------------------------------
def test_mla_parameter_count_matches_page():
    assert om.mla_param_count() == GOLDEN["mla_parameters"]["value"]


def test_component_counts_match_pages():
    s = om.weight_shapes()
    assert int(np.prod(s["w_o"])) == GOLDEN["o_proj_parameters"]["value"]
    # nn.Linear(8192 -> 7168) stores [out, in] = [7168, 8192]
    assert s["w_o"] == (GOLDEN["o_proj_parameters"]["cols"], GOLDEN["o_proj_parameters"]["rows"])
    assert int(np.prod(s["w_o"])) * GOLDEN["o_proj_all_moe_blocks"]["blocks"] == \
        GOLDEN["o_proj_all_moe_blocks"]["value"]
    # key-value compression page counts the 512-wide latent part of
    # kv_a_proj_with_mqa plus its norm (the rotary 64 columns are not in it)
    latent_rows = s["g_kva"][0]
    assert latent_rows * s["w_kv_a"][1] == GOLDEN["kv_down_projection_parameters"]["value"]
    assert latent_rows * s["w_kv_a"][1] + s["g_kva"][0] == GOLDEN["kv_compression_total"]["value"]
    assert s["w_kv_a"][0] == GOLDEN["kv_a_proj_with_mqa_outputs"]["value"]
    assert s["g_in"][0] == GOLDEN["attention_rmsnorm_parameters"]["value"]


def test_dense_block_total_matches_page():
    # block = attention norm + MLA + MLP norm + SwiGLU MLP (three d x I matrices)
    mlp = GOLDEN["swiglu_mlp_parameters"]["value"]
    d = om.KIMI_K2.d
    assert mlp % (3 * d) == 0          # intermediate size 18,432
    total = (GOLDEN["attention_rmsnorm_parameters"]["value"] + om.mla_param_count()
             + GOLDEN["mlp_rmsnorm_parameters"]["value"] + mlp)
    assert total == GOLDEN["dense_block_parameters"]["value"]


def test_cache_sizes_match_page():
    dd = om.KIMI_K2
    assert dd.kv_lora + dd.rope == GOLDEN["latent_cache_values_per_position"]["value"]
    assert dd.H * (dd.qk + dd.v) == GOLDEN["rebuilt_cache_values_per_position"]["value"]
    assert dd.rope // 2 == GOLDEN["rope_pairs"]["value"]


def test_decode_shapes_match_page():
    # P = 1000 cached positions -> the oracle attends over 1001 keys and
    # returns Delta of width d for one position
    dims = TINY
    w = rand_weights(dims, 1)
    P = 1000
    cache = om.cache_from_tokens(w, rand_x((1, P, dims.d), 2), dims)
    r = om.decode(w, rand_x((1, dims.d), 3), cache["K"], cache["V"], dims)
    assert cache["K"].shape[2] + 1 == GOLDEN["decode_keys_read"]["value"]
    assert r["delta"].shape == (1, dims.d)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def test_rmsnorm_constant_vector_closed_form():
    for c in (0.5, 2.0, -3.0):
        x = np.full((7,), c)
        g = np.linspace(0.5, 1.5, 7)
        y = om.rms_norm(x, g, 1e-6)
        np.testing.assert_allclose(y, g * c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rmsnorm_unit_gain_has_unit_rms_and_is_scale_invariant():
    x = rand_x((5, 64), 4)
    y = om.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(om.rms_norm(3.7 * x, np.ones(64), 0.0), y, rtol=1e-12)


def test_rope_unit_vector_closed_form():
    # pair 0 has theta = 1, so position t rotates (e_0) by exactly t radians;
    # pair 16 of 32 has theta = 10000^(-1/2) = 1/100.
    for t in (0, 1, 7, 1000, 8191):
        e0 = np.zeros(64); e0[0] = 1.0
        y = om.rope_rotate(e0, np.array(t), 10000.0)
        assert y[0] == pytest.approx(math.cos(t), abs=1e-12)
        assert y[32] == pytest.approx(math.sin(t), abs=1e-12)
        assert np.count_nonzero(np.abs(y) > 1e-15) <= 2
        e16 = np.zeros(64); e16[16 + 32] = 1.0
        y = om.rope_rotate(e16, np.array(t), 10000.0)
        assert y[16] == pytest.approx(-math.sin(t / 100.0), abs=1e-12)
        assert y[48] == pytest.approx(math.cos(t / 100.0), abs=1e-12)


def test_rope_preserves_pair_norms_and_t0_is_identity():
    x = rand_x((9, 64), 5)
    pos = np.arange(9) * 997
    y = om.rope_rotate(x, pos, 10000.0)
    n_in = x[:, :32] ** 2 + x[:, 32:] ** 2
    n_out = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)
    np.testing.assert_array_equal(om.rope_rotate(x, np.zeros(9), 10000.0), x)


def test_rope_scores_depend_only_on_relative_position():
    q, k = rand_x((64,), 6), rand_x((64,), 7)
    dots = []
    for m, n in ((5, 2), (105, 102), (8003, 8000)):
        dots.append(om.rope_rotate(q, np.array(m), 1e4) @ om.rope_rotate(k, np.array(n), 1e4))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ---------------------------------------------------------------------------
# brute force at tiny sizes: element loops, plain exp, no matmul
# ---------------------------------------------------------------------------
def _bf_rms(v, g, eps):
    ms = math.fsum(a * a for a in v) / len(v)
    r = 1.0 / math.sqrt(ms + eps)
    return [g[i] * v[i] * r for i in range(len(v))]


def _bf_lin(v, W):
    return [math.fsum(W[o][i] * v[i] for i in range(len(v))) for o in range(len(W))]


def _bf_rope(v, t, base):
    n = len(v); h = n // 2
    y = [0.0] * n
    for i in range(h):
        th = base ** (-2.0 * i / n)
        c, s = math.cos(t * th), math.sin(t * th)
        y[i] = v[i] * c - v[i + h] * s
        y[i + h] = v[i + h] * c + v[i] * s
    return y


def brute_force_prefill(w, x, dims, eps, base, scale):
    W = {k: v.tolist() for k, v in w.items()}
    B, T, d = x.shape
    out = np.zeros_like(x)
    for b in range(B):
        Q, K, V = [], [], []
        for t in range(T):
            xa = _bf_rms(list(x[b, t]), W["g_in"], eps)
            cq = _bf_rms(_bf_lin(xa, W["w_q_a"]), W["g_qa"], eps)
            q = _bf_lin(cq, W["w_q_b"])
            a = _bf_lin(xa, W["w_kv_a"])
            ckv = _bf_rms(a[:dims.kv_lora], W["g_kva"], eps)
            kr = _bf_rope(a[dims.kv_lora:], t, base)
            kv = _bf_lin(ckv, W["w_kv_b"])
            Qt, Kt, Vt = [], [], []
            for h in range(dims.H):
                qh = q[h * dims.qk:(h + 1) * dims.qk]
                Qt.append(qh[:dims.nope] + _bf_rope(qh[dims.nope:], t, base))
                kvh = kv[h * (dims.nope + dims.v):(h + 1) * (dims.nope + dims.v)]
                Kt.append(kvh[:dims.nope] + kr)
                Vt.append(kvh[dims.nope:])
            Q.append(Qt); K.append(Kt); V.append(Vt)
        for i in range(T):
            merged = []
            for h in range(dims.H):
                e = [math.exp(scale * math.fsum(Q[i][h][c] * K[j][h][c] for c in range(dims.qk)))
                     for j in range(i + 1)]
                z = math.fsum(e)
                merged += [math.fsum(e[j] * V[j][h][c] for j in range(i + 1)) / z for c in range(dims.v)]
            delta = _bf_lin(merged, W["w_o"])
            out[b, i] = x[b, i] + np.array(delta)
    return out


@pytest.mark.parametrize("dims,B,T", [(TINY, 2, 5), (TINY2, 1, 7)])
def test_prefill_matches_brute_force(dims, B, T):
    w = rand_weights(dims, 10)
    x = rand_x((B, T, dims.d), 11)
    ref = brute_force_prefill(w, x, dims, 1e-6, 10000.0, 1.0 / math.sqrt(dims.qk))
    got = om.prefill(w, x, dims)["out"]
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# independent torch restatement following the layout steps of the pages' code
# ---------------------------------------------------------------------------
def torch_restatement(w, x, dims, eps, base, scale):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    W = {k: torch.tensor(v, dtype=torch.float64) for k, v in w.items()}
    xs = torch.tensor(x, dtype=torch.float64)
    nb, n = xs.shape[0], xs.shape[1]

    def norm(t, g):
        return g * (t * torch.rsqrt(t.pow(2).mean(-1, keepdim=True) + eps))

    h = norm(xs, W["g_in"])
    q = F.linear(norm(F.linear(h, W["w_q_a"]), W["g_qa"]), W["w_q_b"])
    q = q.reshape(nb, n, dims.H, dims.qk).permute(0, 2, 1, 3)          # heads
    q_nope, q_pe = q[..., :dims.nope], q[..., dims.nope:]
    a = F.linear(h, W["w_kv_a"])
    latent, k_pe = a[..., :dims.kv_lora], a[..., dims.kv_lora:]
    k_pe = k_pe.reshape(nb, n, 1, dims.rope).permute(0, 2, 1, 3)
    kv = F.linear(norm(latent, W["g_kva"]), W["w_kv_b"])
    kv = kv.reshape(nb, n, dims.H, dims.nope + dims.v).permute(0, 2, 1, 3)
    k_nope, vals = kv[..., :dims.nope], kv[..., dims.nope:]
    # rotary table with the frequencies repeated over both halves
    inv = 1.0 / (base ** (torch.arange(0, dims.rope, 2, dtype=torch.float64) / dims.rope))
    fr = torch.outer(torch.arange(n, dtype=torch.float64), inv)
    cos, sin = torch.cat([fr, fr], -1).cos(), torch.cat([fr, fr], -1).sin()

    def rot(t):
        half = t.shape[-1] // 2
        return t * cos + torch.cat([-t[..., half:], t[..., :half]], -1) * sin

    q_pe, k_pe = rot(q_pe), rot(k_pe)
    Q = torch.cat([q_nope, q_pe], -1)
    K = torch.cat([k_nope, k_pe.expand(nb, dims.H, n, dims.rope)], -1)
    s = Q @ K.transpose(2, 3) * scale
    mask = torch.full((n, n), float("-inf"), dtype=torch.float64).triu(1)
    p = torch.softmax(s + mask, dim=-1)
    o = (p @ vals).permute(0, 2, 1, 3).reshape(nb, n, dims.H * dims.v)
    return (xs + F.linear(o, W["w_o"])).numpy()


@pytest.mark.parametrize("dims,B,T", [(TINY, 2, 6), (TINY2, 2, 9)])
def test_prefill_matches_torch_restatement(dims, B, T):
    w = rand_weights(dims, 20)
    x = rand_x((B, T, dims.d), 21)
    ref = torch_restatement(w, x, dims, 1e-6, 10000.0, 1.0 / math.sqrt(dims.qk))
    np.testing.assert_allclose(om.prefill(w, x, dims)["out"], ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def test_uniform_scores_give_mean_of_values():
    dims = TINY2
    w = rand_weights(dims, 30)
    w["w_q_b"] = np.zeros_like(w["w_q_b"])   # q = 0 -> every score is 0
    x = rand_x((1, 6, dims.d), 31)
    r = om.prefill(w, x, dims)
    V = r["V"][0]                              # [H, T, v]
    for i in range(6):
        o = V[:, :i + 1].mean(axis=1).reshape(-1)
        np.testing.assert_allclose(r["delta"][0, i], w["w_o"] @ o, rtol=1e-12, atol=1e-13)


def test_causal_row0_attends_only_to_itself():
    dims = TINY
    w = rand_weights(dims, 32)
    x = rand_x((2, 5, dims.d), 33)
    r = om.prefill(w, x, dims)
    for b in range(2):
        np.testing.assert_allclose(r["delta"][b, 0], w["w_o"] @ r["V"][b, :, 0].reshape(-1),
                                   rtol=1e-12, atol=1e-13)


def test_decode_invariant_to_permuting_cached_positions():
    dims = TINY2
    w = rand_weights(dims, 34)
    cache = om.cache_from_tokens(w, rand_x((2, 11, dims.d), 35), dims)
    xn = rand_x((2, dims.d), 36)
    perm = np.random.default_rng(0).permutation(11)
    a = om.decode(w, xn, cache["K"], cache["V"], dims)["out"]
    b = om.decode(w, xn, cache["K"][:, :, perm], cache["V"][:, :, perm], dims)["out"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T", [1, 2, 9])
def test_prefill_last_row_equals_decode(T):
    dims = TINY2
    w = rand_weights(dims, 37)
    x = rand_x((2, T, dims.d), 38)
    pre = om.prefill(w, x, dims)
    cache = om.cache_from_tokens(w, x[:, :T - 1], dims)
    dec = om.decode(w, x[:, T - 1], cache["K"], cache["V"], dims)
    np.testing.assert_allclose(dec["out"], pre["out"][:, T - 1], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dec["k_new"], pre["K"][:, :, T - 1], rtol=1e-12, atol=1e-13)
    lat = om.decode_latent(w, x[:, T - 1], cache["ckv"], cache["kpe"], dims)
    np.testing.assert_allclose(lat["out"], pre["out"][:, T - 1], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("T1,T2", [(1, 5), (4, 3), (6, 1)])
def test_chunked_prefill_equals_whole_prefill(T1, T2):
    """Prefill of T1 tokens, then a chunk of T2 tokens against the first
    T1's cache, reproduces one prefill of all T1 + T2 tokens: the chunk's
    positions start at T1 and its causal mask is offset by T1."""
    dims = TINY2
    w = rand_weights(dims, 61)
    x = rand_x((2, T1 + T2, dims.d), 62)
    whole = om.prefill(w, x, dims)
    cache = om.cache_from_tokens(w, x[:, :T1], dims)
    ch = om.prefill_with_past(w, x[:, T1:], cache["K"], cache["V"], dims)
    np.testing.assert_allclose(ch["out"], whole["out"][:, T1:], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ch["K"], whole["K"][:, :, T1:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ch["V"], whole["V"][:, :, T1:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ch["ckv"], whole["ckv"][:, T1:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ch["kpe"], whole["kpe"][:, T1:], rtol=1e-12, atol=1e-13)


def test_one_token_chunk_equals_decode():
    dims = TINY2
    w = rand_weights(dims, 63)
    cache = om.cache_from_tokens(w, rand_x((3, 7, dims.d), 64), dims)
    xn = rand_x((3, dims.d), 65)
    dec = om.decode(w, xn, cache["K"], cache["V"], dims)
    ch = om.prefill_with_past(w, xn[:, None], cache["K"], cache["V"], dims)
    np.testing.assert_allclose(ch["out"][:, 0], dec["out"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ch["K"][:, :, 0], dec["k_new"], rtol=1e-12, atol=1e-13)


def test_chunk_mask_without_offset_fails_the_pin(monkeypatch):
    """A planted mistake (the chunk's causal mask not offset by the past
    length) is caught by the whole-prefill pin."""
    dims = TINY2
    w = rand_weights(dims, 66)
    x = rand_x((1, 7, dims.d), 67)
    whole = om.prefill(w, x, dims)
    cache = om.cache_from_tokens(w, x[:, :4], dims)
    real_attend = om.attend
    monkeypatch.setattr(om, "attend", lambda Q, K, V, scale, q_pos, *rest: real_attend(
        Q, K, V, scale, None if q_pos is None else np.asarray(q_pos) - K.shape[0] + Q.shape[0], *rest))
    bad = om.prefill_with_past(w, x[:, 4:], cache["K"], cache["V"], dims)
    assert not np.allclose(bad["out"], whole["out"][:, 4:], rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("T1,T2", [(3, 4), (5, 1)])
def test_latent_chunk_equals_whole_prefill(T1, T2):
    """A chunk against the latent cache of the first T1 tokens reproduces
    the whole prefill's rows (the past keys and values rebuilt from the
    latent equal the ones the prefill computed from the tokens)."""
    dims = TINY2
    w = rand_weights(dims, 68)
    x = rand_x((2, T1 + T2, dims.d), 69)
    whole = om.prefill(w, x, dims)
    cache = om.cache_from_tokens(w, x[:, :T1], dims)
    ch = om.prefill_with_past_latent(w, x[:, T1:], cache["ckv"], cache["kpe"], dims)
    np.testing.assert_allclose(ch["out"], whole["out"][:, T1:], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ch["ckv"], whole["ckv"][:, T1:], rtol=1e-12, atol=1e-13)


def test_latent_chunk_rope_key_not_rebuilt_from_latent_fails(monkeypatch):
    """A planted mistake (the rebuilt keys' rotary part taken as zeros
    instead of the cached k^R) is caught by the whole-prefill pin."""
    dims = TINY2
    w = rand_weights(dims, 70)
    x = rand_x((1, 6, dims.d), 71)
    whole = om.prefill(w, x, dims)
    cache = om.cache_from_tokens(w, x[:, :4], dims)
    real = om.rebuild_kv
    monkeypatch.setattr(om, "rebuild_kv", lambda w_, c, r, d=om.KIMI_K2: real(w_, c, np.zeros_like(r), d))
    bad = om.prefill_with_past_latent(w, x[:, 4:], cache["ckv"], cache["kpe"], dims)
    assert not np.allclose(bad["out"], whole["out"][:, 4:], rtol=1e-6, atol=1e-8)


def test_varlen_decode_equal_lengths_is_batched_decode():
    dims = TINY2
    w = rand_weights(dims, 72)
    cache = om.cache_from_tokens(w, rand_x((3, 6, dims.d), 73), dims)
    xn = rand_x((3, dims.d), 74)
    ref = om.decode(w, xn, cache["K"], cache["V"], dims)
    got = om.decode_varlen(w, xn, cache["K"], cache["V"], [6, 6, 6], dims)
    for k in ("out", "k_new", "v_new"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-12, atol=1e-13)
    lat = om.decode_latent_varlen(w, xn, cache["ckv"], cache["kpe"], [6, 6, 6], dims)
    np.testing.assert_allclose(lat["out"], ref["out"], rtol=1e-10, atol=1e-11)


def test_varlen_decode_rows_equal_prefill_rows():
    """Sequence b of length P_b: its decode output equals row P_b of the
    prefill of its first P_b + 1 tokens (a ragged batch, both cache forms);
    rows of the cache beyond P_b (filled with noise) do not matter."""
    dims = TINY2
    w = rand_weights(dims, 75)
    lengths = [2, 7, 4]
    x = rand_x((3, 8, dims.d), 76)
    cache = om.cache_from_tokens(w, x, dims)
    K = cache["K"].copy()
    V = cache["V"].copy()
    C = cache["ckv"].copy()
    R = cache["kpe"].copy()
    for b, P in enumerate(lengths):  # noise where the sequence has no keys yet
        K[b, :, P:] = 50.0
        V[b, :, P:] = -50.0
        C[b, P:] = 50.0
        R[b, P:] = 50.0
    xn = np.stack([x[b, P] for b, P in enumerate(lengths)])
    got = om.decode_varlen(w, xn, K, V, lengths, dims)
    lat = om.decode_latent_varlen(w, xn, C, R, lengths, dims)
    for b, P in enumerate(lengths):
        ref = om.prefill(w, x[b:b + 1, :P + 1], dims, query_rows=[P])
        np.testing.assert_allclose(got["out"][b], ref["out"][0, 0], rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(lat["out"][b], ref["out"][0, 0], rtol=1e-10, atol=1e-11)


def test_latent_absorbed_equals_rebuilt():
    dims = TINY2
    w = rand_weights(dims, 39)
    cache = om.cache_from_tokens(w, rand_x((3, 13, dims.d), 40), dims)
    xn = rand_x((3, dims.d), 41)
    a = om.decode_latent(w, xn, cache["ckv"], cache["kpe"], dims)
    b = om.decode_latent_absorbed(w, xn, cache["ckv"], cache["kpe"], dims)
    np.testing.assert_allclose(a["delta"], b["delta"], rtol=1e-10, atol=1e-13)


def test_wuv_fold_blocks_and_folded_decode():
    """W_fold's block h is W_o's head-h columns times W_UV[h] (checked
    element by element against a triple loop), and the decode through the
    folded matrix equals the rebuilt-cache decode (associativity).  A fold
    with W_UV's rows and columns swapped per head, or the wrong head's
    block, fails both."""
    dims = TINY2
    w = rand_weights(dims, 45)
    F = om.fold_wuv_into_wo(w, dims)
    assert F.shape == (dims.d, dims.H * dims.kv_lora)
    wkvb = w["w_kv_b"]
    for h in range(dims.H):
        for i in range(dims.d):
            for c in range(dims.kv_lora):
                ref = sum(w["w_o"][i, h * dims.v + j] * wkvb[h * (dims.nope + dims.v) + dims.nope + j, c]
                          for j in range(dims.v))
                assert abs(F[i, h * dims.kv_lora + c] - ref) < 1e-12
    cache = om.cache_from_tokens(w, rand_x((2, 11, dims.d), 46), dims)
    xn = rand_x((2, dims.d), 47)
    a = om.decode_latent(w, xn, cache["ckv"], cache["kpe"], dims)
    b = om.decode_latent_folded(w, F, xn, cache["ckv"], cache["kpe"], dims)
    np.testing.assert_allclose(b["delta"], a["delta"], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(b["ckv_new"], a["ckv_new"], rtol=0, atol=1e-14)
    # a head-block permutation (each head given the next head's block) is caught
    Fp = np.concatenate([F[:, ((h + 1) % dims.H) * dims.kv_lora:((h + 1) % dims.H + 1) * dims.kv_lora]
                         for h in range(dims.H)], axis=1)
    bp = om.decode_latent_folded(w, Fp, xn, cache["ckv"], cache["kpe"], dims)
    assert not np.allclose(bp["delta"], a["delta"], rtol=1e-3, atol=1e-6)


def test_batch_rows_are_independent():
    dims = TINY
    w = rand_weights(dims, 42)
    x = rand_x((3, 4, dims.d), 43)
    a = om.prefill(w, x, dims)["out"]
    x2 = x.copy(); x2[1] = rand_x((4, dims.d), 44)
    b = om.prefill(w, x2, dims)["out"]
    np.testing.assert_array_equal(a[0], b[0]); np.testing.assert_array_equal(a[2], b[2])
    assert not np.allclose(a[1], b[1])


def test_query_rows_subset_matches_full():
    dims = TINY2
    w = rand_weights(dims, 45)
    x = rand_x((2, 10, dims.d), 46)
    full = om.prefill(w, x, dims)
    sub = om.prefill(w, x, dims, query_rows=[0, 3, 9])
    np.testing.assert_allclose(sub["out"], full["out"][:, [0, 3, 9]], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# the pins catch plausible mistakes (planted in the oracle, on the CPU)
# ---------------------------------------------------------------------------
def _pins_pass():
    try:
        test_rope_unit_vector_closed_form()
        test_prefill_matches_brute_force(TINY, 2, 5)
        test_prefill_matches_torch_restatement(TINY2, 2, 9)
        test_prefill_last_row_equals_decode(9)
        test_latent_absorbed_equals_rebuilt()
    except AssertionError:
        return False
    return True


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins_pass()
    orig_rope, orig_norm, orig_lin = om.rope_rotate, om.rms_norm, om._linear

    def rope_wrong_sign(x, pos, base):
        y = orig_rope(x, pos, base); h = x.shape[-1] // 2
        return np.concatenate([y[..., :h], -y[..., h:] + 2 * x[..., h:] * 0], axis=-1)

    def rope_interleaved(x, pos, base):
        y = orig_rope(x[..., np.r_[0:x.shape[-1]:2, 1:x.shape[-1]:2]], pos, base)
        out = np.empty_like(y); h = x.shape[-1] // 2
        out[..., 0::2], out[..., 1::2] = y[..., :h], y[..., h:]
        return out

    def norm_no_gain(x, g, eps):
        return orig_norm(x, np.ones_like(g), eps)

    def norm_no_eps(x, g, eps):
        return orig_norm(x, g, 0.5)

    mistakes = [("rope_rotate", rope_wrong_sign), ("rope_rotate", rope_interleaved),
                ("rms_norm", norm_no_gain), ("rms_norm", norm_no_eps)]
    for name, fn in mistakes:
        monkeypatch.setattr(om, name, fn)
        assert not _pins_pass(), f"planted mistake {fn.__name__} not caught"
        monkeypatch.setattr(om, name, {"rope_rotate": orig_rope, "rms_norm": orig_norm}[name])

    # scale applied twice / wrong scale
    orig_default = om.default_scale
    monkeypatch.setattr(om, "default_scale", lambda dims=om.KIMI_K2: 1.0 / dims.qk)
    assert not _pins_pass()
    monkeypatch.setattr(om, "default_scale", orig_default)

    # K and V swapped in the kv_b split
    def project_swapped(w, x, pos, dims, eps, base, want_q=True, bf16_storage=False):
        r = orig_project(w, x, pos, dims, eps, base, want_q, bf16_storage)
        if dims.nope == dims.v:
            r["V"] = r["K"][..., :dims.nope].copy()
        else:
            r["V"] = r["V"][..., ::-1].copy()
        return r
    orig_project = om.project_tokens
    monkeypatch.setattr(om, "project_tokens", project_swapped)
    assert not _pins_pass()
    monkeypatch.setattr(om, "project_tokens", orig_project)
    assert _pins_pass()


# ---------------------------------------------------------------------------
# the bf16-storage reading (activations handed on, probabilities and the
# attention output stored in bf16)
# ---------------------------------------------------------------------------
def _bf16_exact(a):
    return np.array_equal(om.round_to_bf16(a), a)


def _storage_cases(dims, seed):
    w = rand_weights(dims, seed)
    x = rand_x((2, 6, dims.d), seed + 1)
    xn = rand_x((2, dims.d), seed + 2)
    c = om.cache_from_tokens(w, x, dims)
    return [
        ("prefill", lambda st: om.prefill(w, x, dims, bf16_storage=st)),
        ("chunk", lambda st: om.prefill_with_past(w, x[:, 4:], c["K"][:, :, :4], c["V"][:, :, :4], dims,
                                                  bf16_storage=st)),
        ("decode", lambda st: om.decode(w, xn, c["K"], c["V"], dims, bf16_storage=st)),
        ("absorbed", lambda st: om.decode_latent_absorbed(w, xn, c["ckv"], c["kpe"], dims, bf16_storage=st)),
    ]


def test_bf16_storage_only_adds_rounding(monkeypatch):
    """With the rounding made the identity, the bf16-storage reading is the
    exact computation term for term; with it, every stored tensor the call
    returns holds bf16 values and the result stays within bf16-level
    distance of the exact one."""
    for name, run in _storage_cases(TINY2, 81):
        exact = run(False)
        st = run(True)
        d = st["delta"] - exact["delta"]
        rel = np.linalg.norm(d) / np.linalg.norm(exact["delta"])
        assert 1e-6 < rel < 2e-2, (name, rel)
        for k in ("K", "V", "ckv", "kpe", "ckv_new", "kpe_new"):
            if k in st:
                assert _bf16_exact(st[k]), (name, k)
    monkeypatch.setattr(om, "round_to_bf16", lambda a: np.asarray(a, dtype=np.float64))
    for name, run in _storage_cases(TINY2, 81):
        np.testing.assert_allclose(run(True)["delta"], run(False)["delta"], rtol=1e-12, atol=1e-14, err_msg=name)


def test_bf16_storage_rounds_probabilities_before_pv():
    """attend with bf16 storage: P cast to bf16 before P V and the output
    stored in bf16 (the page's cast of the float32 softmax to the query
    dtype).  A case where P is exactly representable (two equal scores, one
    masked) leaves only the output rounding."""
    Q = np.array([[1.0, 0.0]])
    K = np.array([[1.0, 0.0], [1.0, 0.0], [5.0, 0.0]])
    V = np.array([[1.0 + 2.0 ** -8, 3.0], [1.0, 1.0], [7.0, 7.0]])
    o = om.attend(Q, K, V, 1.0, np.array([1]), bf16_storage=True)       # keys 0, 1 visible, P = (1/2, 1/2)
    np.testing.assert_array_equal(o, om.round_to_bf16(np.array([[1.0 + 2.0 ** -9, 2.0]])))
    np.testing.assert_array_equal(o, np.array([[1.0, 2.0]]))              # 1 + 2^-9 rounds to 1
    p3 = om.attend(np.array([[0.0, 0.0]]), K, np.eye(3)[:, :2], 1.0, None, bf16_storage=True)
    np.testing.assert_array_equal(p3, om.round_to_bf16(np.array([[1.0 / 3.0, 1.0 / 3.0]])))
