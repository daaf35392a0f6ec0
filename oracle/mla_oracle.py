"""CPU oracle of the multi-head latent attention (MLA) sublayer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library and imports
nothing from it.

What it computes is the plain definition, in float64, with numpy matmul as
the only library primitive and no blocking or fusion:

* Kimi K2 "Dense transformer block" page, equation list: x_attn =
  RMSNorm(x_n); c^Q = x W_DQ; c^Q-hat = RMSNorm(c^Q); c^KV = x W_DKV;
  c^KV-hat = RMSNorm(c^KV); q^C, q^pe from c^Q-hat (W_UQ, W_QR); k^C, v from
  c^KV-hat (W_UK, W_UV); k^pe = x W_KR; RoPE on q^pe and k^pe; Q = [Q^C; Q^R];
  K_i = [K^C_i; k^R]; x'_n = x_n + Delta_attn.
* "Mix and project" page (decode, P = 1000), code excerpt: scores =
  Q K^T * softmax_scale, plus the additive mask, softmax in float32 (here:
  float64), P V, heads merged head-major, o_proj.
* "Key-value compression" page, code excerpt: one kv_a_proj_with_mqa matrix
  produces 512 latent + 64 rotary-key features, split after the product; only
  the 512-wide latent is normalised (kv_a_layernorm), the rotary key is not.

Readings where the pages are silent:
* RMSNorm(x; g) = g * x / sqrt(mean(x^2) + eps) with eps = 1e-6 for all three
  norms (the module bodies are not printed).
* q_b_proj output per head is [128 "nope" | 64 "pe"] in 192-wide blocks, the
  same view-then-split the pages print for kv_b_proj ([128 k_nope | 128 v]).
* RoPE is rotate-half on pairs (i, i + 32) with theta_i = base^(-2i/64),
  base 10000, no frequency scaling; position t rotates pair i by t*theta_i.
* Mask: causal (key j visible to query i iff j <= i) in prefill; none in
  decode, where the new token sits at position P and attends to all P + 1 keys.
* softmax_scale = 1/sqrt(192); dropout is the identity (inference).
* The latent cache holds the normalised c^KV-hat and the rotated k^R.

Every function below names the passage it follows.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Dims:
    """Sizes of one MLA instance (defaults: Kimi K2, checked against the
    101,124,096-parameter count in the dense-block page's parameter table)."""
    d: int = 7168
    H: int = 64
    q_lora: int = 1536
    kv_lora: int = 512
    nope: int = 128
    rope: int = 64
    v: int = 128

    @property
    def qk(self) -> int:
        return self.nope + self.rope


KIMI_K2 = Dims()
DEFAULT_EPS = 1e-6
DEFAULT_ROPE_BASE = 10000.0


def default_scale(dims: Dims = KIMI_K2) -> float:
    return 1.0 / np.sqrt(dims.qk)


def weight_shapes(dims: Dims = KIMI_K2) -> dict:
    """nn.Linear weights are [out, in] (key-value compression page, MLA
    __init__ excerpt); gains are vectors.  g_in is the block's attention
    RMSNorm, counted outside the MLA total on the dense-block page."""
    return {
        "g_in": (dims.d,),
        "w_q_a": (dims.q_lora, dims.d),
        "g_qa": (dims.q_lora,),
        "w_q_b": (dims.H * dims.qk, dims.q_lora),
        "w_kv_a": (dims.kv_lora + dims.rope, dims.d),
        "g_kva": (dims.kv_lora,),
        "w_kv_b": (dims.H * (dims.nope + dims.v), dims.kv_lora),
        "w_o": (dims.d, dims.H * dims.v),
    }


def mla_param_count(dims: Dims = KIMI_K2) -> int:
    """Learned parameters of one MLA sublayer (everything but g_in)."""
    return sum(int(np.prod(s)) for k, s in weight_shapes(dims).items() if k != "g_in")


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis (dense-block page: x_attn = RMSNorm(x_n),
    c^Q-hat = RMSNorm(c^Q), c^KV-hat = RMSNorm(c^KV))."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return g * (x / np.sqrt(ms + eps))


def rope_inv_freq(rope: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/rope) for i = 0 .. rope/2 - 1 (one per pair)."""
    i = np.arange(rope // 2, dtype=np.float64)
    return base ** (-2.0 * i / rope)


def rope_rotate(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """RoPE(x, R_t) of the dense-block page: rotate-half on pairs (i, i+half).

    ``pos`` broadcasts against x[..., 0].
    y_i = x_i cos(t th_i) - x_{i+half} sin(t th_i)
    y_{i+half} = x_{i+half} cos(t th_i) + x_i sin(t th_i)
    """
    half = x.shape[-1] // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(x.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """nn.Linear without bias: x W^T (attention_bias absent: the parameter
    count 101,124,096 holds only without biases)."""
    return x @ w.T


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """The nearest bfloat16 value of each float64 (8 significant bits,
    ties to even), for values in bfloat16's normal range: the storage of a
    module output in a bf16 model.  a = m 2^e with 1/2 <= |m| < 1; m is
    rounded to a multiple of 2^-8 (np.round rounds halves to even)."""
    m, e = np.frexp(np.asarray(a, dtype=np.float64))
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def _stored(a: np.ndarray, bf16: bool) -> np.ndarray:
    """a as the next step receives it: rounded to bf16 in the bf16-storage
    reading, unchanged otherwise."""
    return round_to_bf16(a) if bf16 else a


def project_tokens(w: dict, x: np.ndarray, pos: np.ndarray, dims: Dims, eps: float,
                   base: float, want_q: bool = True, bf16_storage: bool = False) -> dict:
    """Per-token part of MLA for tokens x [..., d] at positions ``pos``.

    Dense-block page equations c^Q .. v, and the key-value compression page's
    split of kv_a_proj_with_mqa into the 512 latent and the 64-wide rotary key
    (only the latent is normalised).  Returns per-head K rows [..., H, qk],
    V rows [..., H, v], the latent c^KV-hat [..., kv_lora], the rotated rotary
    key k^R [..., rope] and (if want_q) Q rows [..., H, qk].

    bf16_storage: the activations one step hands to the next are stored in
    bf16 (x_attn, the normalised latents, the rotated rotary keys, Q after
    RoPE, the kv_b output), as the pages' module does when it runs in bf16;
    the A-projection output stays unrounded until it is normalised or
    rotated (the A-projection precision reading).
    """
    st = bf16_storage
    x_attn = _stored(rms_norm(x, w["g_in"], eps), st)
    ckv_full = _linear(x_attn, w["w_kv_a"])
    ckv = ckv_full[..., :dims.kv_lora]
    kpe_raw = ckv_full[..., dims.kv_lora:]
    ckv_hat = _stored(rms_norm(ckv, w["g_kva"], eps), st)
    kv = _stored(_linear(ckv_hat, w["w_kv_b"]), st).reshape(x.shape[:-1] + (dims.H, dims.nope + dims.v))
    k_nope = kv[..., :dims.nope]
    v = kv[..., dims.nope:]
    k_r = _stored(rope_rotate(kpe_raw, pos, base), st)
    # K_i = [K^C_i ; k^R]: the one rotary key is shared by every head
    k_r_heads = np.broadcast_to(k_r[..., None, :], k_nope.shape[:-1] + (dims.rope,))
    out = {
        "K": np.concatenate([k_nope, k_r_heads], axis=-1),
        "V": v,
        "ckv": ckv_hat,
        "kpe": k_r,
    }
    if want_q:
        cq_hat = _stored(rms_norm(_linear(x_attn, w["w_q_a"]), w["g_qa"], eps), st)
        q = _linear(cq_hat, w["w_q_b"]).reshape(x.shape[:-1] + (dims.H, dims.qk))
        q_nope = _stored(q[..., :dims.nope], st)
        q_pe = _stored(rope_rotate(q[..., dims.nope:], np.asarray(pos)[..., None], base), st)
        out["Q"] = np.concatenate([q_nope, q_pe], axis=-1)
    return out


def softmax(s: np.ndarray) -> np.ndarray:
    """softmax over the last axis with max subtraction (masked entries are
    -inf and contribute exp(-inf) = 0)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
           q_pos: np.ndarray | None, bf16_storage: bool = False) -> np.ndarray:
    """One head: softmax(Q K^T * scale + M) V ("Mix and project" page code).

    Q [nq, qk], K [nk, qk], V [nk, v].  q_pos gives each query's position for
    the causal mask M (key j visible iff j <= q_pos); None means no mask.
    bf16_storage: the probabilities are cast to bf16 before P V and the
    output is stored in bf16, as the page's code casts the float32 softmax
    to the query dtype.
    """
    s = (Q @ K.T) * scale
    if q_pos is not None:
        j = np.arange(K.shape[0])
        s = np.where(j[None, :] <= np.asarray(q_pos)[:, None], s, -np.inf)
    return _stored(_stored(softmax(s), bf16_storage) @ V, bf16_storage)


def prefill(w: dict, x: np.ndarray, dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS,
            base: float = DEFAULT_ROPE_BASE, scale: float | None = None,
            query_rows=None, bf16_storage: bool = False) -> dict:
    """Causal prefill of x [B, T, d] at positions 0..T-1.

    Returns out = x + Delta [B, nq, d], Delta, the rebuilt caches
    K [B, H, T, qk], V [B, H, T, v], the latent cache ckv [B, T, kv_lora] and
    kpe [B, T, rope].  ``query_rows`` restricts the queries (and out/Delta
    rows) to those positions; keys and values always cover all T tokens.
    """
    if scale is None:
        scale = default_scale(dims)
    B, T, _ = x.shape
    rows = np.arange(T) if query_rows is None else np.asarray(query_rows)
    pos = np.arange(T)
    st = bf16_storage
    kv = project_tokens(w, x, pos[None, :], dims, eps, base, want_q=False, bf16_storage=st)
    qp = project_tokens(w, x[:, rows], rows[None, :], dims, eps, base, want_q=True, bf16_storage=st)
    O = np.empty((B, len(rows), dims.H, dims.v))
    for b in range(B):
        for h in range(dims.H):
            O[b, :, h] = attend(qp["Q"][b, :, h], kv["K"][b, :, h], kv["V"][b, :, h], scale, rows, st)
    delta = _linear(O.reshape(B, len(rows), dims.H * dims.v), w["w_o"])
    return {
        "out": x[:, rows] + delta,
        "delta": delta,
        "K": np.ascontiguousarray(kv["K"].transpose(0, 2, 1, 3)),
        "V": np.ascontiguousarray(kv["V"].transpose(0, 2, 1, 3)),
        "ckv": kv["ckv"],
        "kpe": kv["kpe"],
    }


def prefill_with_past(w: dict, x: np.ndarray, K_cache: np.ndarray, V_cache: np.ndarray,
                      dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
                      scale: float | None = None, query_rows=None, bf16_storage: bool = False) -> dict:
    """Chunked prefill: x [B, T, d] are the tokens at positions P0..P0+T-1,
    P0 = K_cache.shape[2]; K_cache [B, H, P0, qk] and V_cache [B, H, P0, v]
    hold positions 0..P0-1 (post-RoPE).

    "Mix and project" page: the cache update concatenates the new keys and
    values after the cached ones (past_key_value.update), and the additive
    mask of shape (B, 1, q_len, kv_seq_len) with kv_seq_len = P0 + T keeps the
    causal order: query t (position P0 + t) sees keys 0..P0+t.  Returns out,
    Delta and the new cache rows K/V [B, H, T, .], ckv, kpe [B, T, .].
    ``query_rows`` (indices into the chunk) restricts the queries.
    """
    if scale is None:
        scale = default_scale(dims)
    B, T, _ = x.shape
    P0 = K_cache.shape[2]
    rows = np.arange(T) if query_rows is None else np.asarray(query_rows)
    pos = P0 + np.arange(T)
    st = bf16_storage
    kv = project_tokens(w, x, pos[None, :], dims, eps, base, want_q=False, bf16_storage=st)
    qp = project_tokens(w, x[:, rows], (P0 + rows)[None, :], dims, eps, base, want_q=True, bf16_storage=st)
    O = np.empty((B, len(rows), dims.H, dims.v))
    for b in range(B):
        for h in range(dims.H):
            K = np.concatenate([K_cache[b, h], kv["K"][b, :, h]], axis=0)
            V = np.concatenate([V_cache[b, h], kv["V"][b, :, h]], axis=0)
            O[b, :, h] = attend(qp["Q"][b, :, h], K, V, scale, P0 + rows, st)
    delta = _linear(O.reshape(B, len(rows), dims.H * dims.v), w["w_o"])
    return {
        "out": x[:, rows] + delta,
        "delta": delta,
        "K": np.ascontiguousarray(kv["K"].transpose(0, 2, 1, 3)),
        "V": np.ascontiguousarray(kv["V"].transpose(0, 2, 1, 3)),
        "ckv": kv["ckv"],
        "kpe": kv["kpe"],
    }


def decode(w: dict, x_new: np.ndarray, K_cache: np.ndarray, V_cache: np.ndarray,
           dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
           scale: float | None = None, bf16_storage: bool = False) -> dict:
    """One decode step against the rebuilt per-head cache.

    x_new [B, d] is the token at position P = K_cache.shape[2]; K_cache
    [B, H, P, qk] and V_cache [B, H, P, v] hold positions 0..P-1 (post-RoPE).
    The cache update appends the new K/V and the query attends to all P + 1
    keys with no mask ("Mix and project" page: past_key_value.update, then
    scores over kv_seq_len = P + 1).
    """
    if scale is None:
        scale = default_scale(dims)
    B = x_new.shape[0]
    P = K_cache.shape[2]
    t = project_tokens(w, x_new, np.full((B,), P), dims, eps, base, want_q=True, bf16_storage=bf16_storage)
    O = np.empty((B, dims.H, dims.v))
    for b in range(B):
        for h in range(dims.H):
            K = np.concatenate([K_cache[b, h], t["K"][b, h][None]], axis=0)
            V = np.concatenate([V_cache[b, h], t["V"][b, h][None]], axis=0)
            O[b, h] = attend(t["Q"][b, h][None], K, V, scale, None, bf16_storage)[0]
    delta = _linear(O.reshape(B, dims.H * dims.v), w["w_o"])
    return {"out": x_new + delta, "delta": delta, "k_new": t["K"], "v_new": t["V"],
            "ckv_new": t["ckv"], "kpe_new": t["kpe"]}


def decode_varlen(w: dict, x_new: np.ndarray, K_cache: np.ndarray, V_cache: np.ndarray, lengths,
                  dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
                  scale: float | None = None) -> dict:
    """One decode step for sequences of different lengths: sequence b's new
    token sits at position P_b = lengths[b] and attends to the P_b + 1 keys
    of its own cache rows 0..P_b-1 plus itself ("Mix and project" page:
    every sequence is its own cache update and score row; sequences do not
    interact).  K_cache [B, H, >= max P_b, qk], V_cache likewise; rows at or
    beyond P_b are ignored.  Returns the stacked per-sequence results."""
    res = [decode(w, x_new[b:b + 1], K_cache[b:b + 1, :, :int(P)], V_cache[b:b + 1, :, :int(P)], dims, eps, base,
                  scale) for b, P in enumerate(lengths)]
    return {k: np.concatenate([r[k] for r in res], axis=0) for k in res[0]}


def decode_latent_varlen(w: dict, x_new: np.ndarray, ckv_cache: np.ndarray, kpe_cache: np.ndarray, lengths,
                         dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
                         scale: float | None = None) -> dict:
    """``decode_varlen`` against the latent cache (rows 0..P_b-1 of each
    sequence's ckv / kpe)."""
    res = [decode_latent(w, x_new[b:b + 1], ckv_cache[b:b + 1, :int(P)], kpe_cache[b:b + 1, :int(P)], dims, eps,
                         base, scale) for b, P in enumerate(lengths)]
    return {k: np.concatenate([r[k] for r in res], axis=0) for k in res[0]}


def rebuild_kv(w: dict, ckv: np.ndarray, kpe: np.ndarray, dims: Dims = KIMI_K2):
    """Per-head K/V from the latent cache (key-value compression page: the key
    content and values of all heads are rebuilt from one latent per position).
    ckv [..., P, kv_lora], kpe [..., P, rope] -> K [..., H, P, qk], V [..., H, P, v]."""
    kv = _linear(ckv, w["w_kv_b"]).reshape(ckv.shape[:-1] + (dims.H, dims.nope + dims.v))
    k_nope = kv[..., :dims.nope]
    k_r = np.broadcast_to(kpe[..., None, :], k_nope.shape[:-1] + (dims.rope,))
    K = np.concatenate([k_nope, k_r], axis=-1)
    V = kv[..., dims.nope:]
    return np.moveaxis(K, -2, -3), np.moveaxis(V, -2, -3)


def decode_latent(w: dict, x_new: np.ndarray, ckv_cache: np.ndarray, kpe_cache: np.ndarray,
                  dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS,
                  base: float = DEFAULT_ROPE_BASE, scale: float | None = None) -> dict:
    """Decode against the 576-value latent cache: rebuild, then attend.

    ckv_cache [B, P, kv_lora] (normalised latent) and kpe_cache [B, P, rope]
    (rotated rotary key) hold positions 0..P-1.  The per-head K/V are rebuilt
    from the latent exactly as in prefill, then ``decode`` runs.
    """
    K_cache, V_cache = rebuild_kv(w, ckv_cache, kpe_cache, dims)
    return decode(w, x_new, K_cache, V_cache, dims, eps, base, scale)


def decode_latent_absorbed(w: dict, x_new: np.ndarray, ckv_cache: np.ndarray,
                           kpe_cache: np.ndarray, dims: Dims = KIMI_K2,
                           eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
                           scale: float | None = None, bf16_storage: bool = False) -> dict:
    """Same step with W_UK / W_UV absorbed (the design the key-value
    compression page attributes to DeepSeek-V2: cache the latent instead of
    per-head K/V).  Used only as an invariant: it equals ``decode_latent`` up
    to float64 rounding, since q.(W_UK c) = (W_UK^T q).c and
    sum_j p_j W_UV c_j = W_UV sum_j p_j c_j.
    bf16_storage: the absorbed query q_lat, the probabilities, the latent
    output o_lat and the per-head output are stored in bf16 as well (the
    steps a bf16 implementation of this form hands on).
    """
    if scale is None:
        scale = default_scale(dims)
    B = x_new.shape[0]
    P = ckv_cache.shape[1]
    st = bf16_storage
    t = project_tokens(w, x_new, np.full((B,), P), dims, eps, base, want_q=True, bf16_storage=st)
    wkvb = w["w_kv_b"].reshape(dims.H, dims.nope + dims.v, dims.kv_lora)
    w_uk, w_uv = wkvb[:, :dims.nope], wkvb[:, dims.nope:]
    O = np.empty((B, dims.H, dims.v))
    for b in range(B):
        C = np.concatenate([ckv_cache[b], t["ckv"][b][None]], axis=0)      # [P+1, kv_lora]
        R = np.concatenate([kpe_cache[b], t["kpe"][b][None]], axis=0)      # [P+1, rope]
        for h in range(dims.H):
            q_lat = _stored(w_uk[h].T @ t["Q"][b, h, :dims.nope], st)
            s = (C @ q_lat + R @ t["Q"][b, h, dims.nope:]) * scale
            p = _stored(softmax(s[None])[0], st)
            O[b, h] = _stored(w_uv[h] @ _stored(p @ C, st), st)
    delta = _linear(O.reshape(B, dims.H * dims.v), w["w_o"])
    return {"out": x_new + delta, "delta": delta, "ckv_new": t["ckv"], "kpe_new": t["kpe"]}


def fold_wuv_into_wo(w: dict, dims: Dims = KIMI_K2) -> np.ndarray:
    """W_UV folded into the output projection (the latent-serving design of
    the key-value compression page carried one step further): head h's value
    up-projection W_UV[h] [v, kv_lora] and its columns of W_o [d, v] make one
    [d, kv_lora] block, W_fold[:, h*kv_lora:(h+1)*kv_lora] = W_o[:, h*v:(h+1)*v] W_UV[h],
    so the sublayer's output is o_lat (all heads' latent attention outputs,
    [H*kv_lora]) times W_fold^T."""
    wkvb = w["w_kv_b"].reshape(dims.H, dims.nope + dims.v, dims.kv_lora)
    w_uv = wkvb[:, dims.nope:]                                   # [H, v, kv_lora]
    w_o = w["w_o"].reshape(dims.d, dims.H, dims.v)               # [d, H, v]
    return np.concatenate([w_o[:, h] @ w_uv[h] for h in range(dims.H)], axis=1)


def decode_latent_folded(w: dict, w_fold: np.ndarray, x_new: np.ndarray, ckv_cache: np.ndarray,
                         kpe_cache: np.ndarray, dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS,
                         base: float = DEFAULT_ROPE_BASE, scale: float | None = None) -> dict:
    """Decode against the latent cache with W_UK absorbed into the query and
    W_UV folded into the output projection: per head the latent attention
    output o_lat[h] = sum_j p_j c_j ([kv_lora]), then
    Delta = [o_lat[0] .. o_lat[H-1]] W_fold^T.  Equal to ``decode_latent`` up to
    float64 rounding (associativity); the new token's cache rows as there."""
    if scale is None:
        scale = default_scale(dims)
    B = x_new.shape[0]
    P = ckv_cache.shape[1]
    t = project_tokens(w, x_new, np.full((B,), P), dims, eps, base, want_q=True)
    wkvb = w["w_kv_b"].reshape(dims.H, dims.nope + dims.v, dims.kv_lora)
    w_uk = wkvb[:, :dims.nope]
    o_lat = np.empty((B, dims.H, dims.kv_lora))
    for b in range(B):
        C = np.concatenate([ckv_cache[b], t["ckv"][b][None]], axis=0)      # [P+1, kv_lora]
        R = np.concatenate([kpe_cache[b], t["kpe"][b][None]], axis=0)      # [P+1, rope]
        for h in range(dims.H):
            q_lat = w_uk[h].T @ t["Q"][b, h, :dims.nope]
            s = (C @ q_lat + R @ t["Q"][b, h, dims.nope:]) * scale
            p = softmax(s[None])[0]
            o_lat[b, h] = p @ C
    delta = _linear(o_lat.reshape(B, dims.H * dims.kv_lora), w_fold)
    return {"out": x_new + delta, "delta": delta, "ckv_new": t["ckv"], "kpe_new": t["kpe"]}


def prefill_with_past_latent(w: dict, x: np.ndarray, ckv_cache: np.ndarray, kpe_cache: np.ndarray,
                             dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS, base: float = DEFAULT_ROPE_BASE,
                             scale: float | None = None, query_rows=None) -> dict:
    """Chunked prefill against the 576-value latent cache: ckv_cache
    [B, P0, kv_lora] and kpe_cache [B, P0, rope] hold positions 0..P0-1.
    The cached positions' per-head keys and values are rebuilt from the
    latent (key-value compression page: every head's key content and value
    come from the one latent of the position), then the chunk attends as in
    ``prefill_with_past``."""
    K, V = rebuild_kv(w, ckv_cache, kpe_cache, dims)
    return prefill_with_past(w, x, K, V, dims, eps, base, scale, query_rows)


def cache_from_tokens(w: dict, x: np.ndarray, dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS,
                      base: float = DEFAULT_ROPE_BASE) -> dict:
    """Both caches for tokens x [B, P, d] at positions 0..P-1 (what a prefill
    writes): K [B, H, P, qk], V [B, H, P, v], ckv [B, P, kv_lora], kpe [B, P, rope]."""
    P = x.shape[1]
    t = project_tokens(w, x, np.arange(P)[None, :], dims, eps, base, want_q=False)
    return {"K": np.ascontiguousarray(t["K"].transpose(0, 2, 1, 3)),
            "V": np.ascontiguousarray(t["V"].transpose(0, 2, 1, 3)),
            "ckv": t["ckv"], "kpe": t["kpe"]}


# ---------------------------------------------------------------------------
# The block's second half: post-attention RMSNorm and the dense SwiGLU MLP
# (dense-block page, equation list after x'_n = x_n + Delta_attn; the
# DecoderLayer forward excerpt of the same page).
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class FfnDims:
    """Sizes of the dense SwiGLU MLP.  The pages print its parameter count,
    396,361,728, not its width: three bias-free matrices d x I give
    I = 396,361,728 / (3 * 7168) = 18,432."""
    d: int = 7168
    inter: int = 18432


KIMI_K2_FFN = FfnDims()


def ffn_weight_shapes(fd: FfnDims = KIMI_K2_FFN) -> dict:
    """g_post: the MLP RMSNorm gain; w_1 (gate, g = x_ffn W_1) and w_3 (up,
    u = x_ffn W_3) map d -> I, w_2 (Delta_ffn = h W_2) maps I -> d; stored
    nn.Linear style [out, in]."""
    return {
        "g_post": (fd.d,),
        "w_1": (fd.inter, fd.d),
        "w_3": (fd.inter, fd.d),
        "w_2": (fd.d, fd.inter),
    }


def ffn_param_count(fd: FfnDims = KIMI_K2_FFN) -> int:
    """Parameters of the SwiGLU MLP row of the dense-block parameter table
    (the MLP RMSNorm gain has its own row)."""
    return sum(int(np.prod(s)) for k, s in ffn_weight_shapes(fd).items() if k != "g_post")


def dense_block_param_count(dims: Dims = KIMI_K2, fd: FfnDims = KIMI_K2_FFN) -> int:
    """Per-instance total of the dense-block parameter table: attention
    RMSNorm + MLA + MLP RMSNorm + SwiGLU MLP."""
    return dims.d + mla_param_count(dims) + fd.d + ffn_param_count(fd)


def sigmoid(z: np.ndarray) -> np.ndarray:
    """sigma(z) = 1 / (1 + e^-z), evaluated as (1 + tanh(z/2)) / 2, the same
    function without overflow for large |z|."""
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """The gating step of the SwiGLU MLP: a = g sigma(g) (SiLU of the gate),
    h = a (.) u."""
    a = g * sigmoid(g)
    return a * u


def ffn(w: dict, xp: np.ndarray, eps: float = DEFAULT_EPS, bf16_products: bool = False) -> dict:
    """x_{n+1} from x'_n (dense-block page): x_ffn = RMSNorm(x'_n);
    g = x_ffn W_1; u = x_ffn W_3; a = g sigma(g); h = a (.) u;
    Delta_ffn = h W_2; x_{n+1} = x'_n + Delta_ffn.  Any leading shape.

    bf16_products: the reading a bf16 model takes of the same equations
    (the MLP precision reading): the two product inputs, x_ffn and h, are
    module outputs stored in bfloat16, so each is rounded once to bf16
    before its product; everything else stays float64."""
    x_ffn = rms_norm(xp, w["g_post"], eps)
    if bf16_products:
        x_ffn = round_to_bf16(x_ffn)
    g = _linear(x_ffn, w["w_1"])
    u = _linear(x_ffn, w["w_3"])
    h = swiglu(g, u)
    if bf16_products:
        h = round_to_bf16(h)
    delta = _linear(h, w["w_2"])
    return {"out": xp + delta, "delta": delta, "h": h}


def dense_block_prefill(w: dict, w_ffn: dict, x: np.ndarray, dims: Dims = KIMI_K2, eps: float = DEFAULT_EPS,
                        base: float = DEFAULT_ROPE_BASE, scale: float | None = None) -> dict:
    """The whole dense block on x [B, T, d] at positions 0..T-1 (DecoderLayer
    forward excerpt): x' = x + MLA(RMSNorm(x)), then x_{n+1} = x' + MLP(RMSNorm(x'))."""
    attn = prefill(w, x, dims, eps, base, scale)
    f = ffn(w_ffn, attn["out"], eps)
    return {"out": f["out"], "x_mid": attn["out"], "delta_attn": attn["delta"], "delta_ffn": f["delta"]}


# ---------------------------------------------------------------------------
# FP8 block-scaled weights.  The dense-block page counts the checkpoint's
# tensors with its "FP8 block scales" left out, so the weights are stored in
# FP8 with one scale per block; the block size and the scale format are not
# printed.  Reading taken: E4M3 (4 exponent bits, bias 7, 3 mantissa bits,
# no infinities, largest finite 448) with one power-of-two scale per 128 x 128
# block of the [out, in] matrix: s = 2^k for the smallest k with
# amax(block) <= 448 * 2^k, q = E4M3 round-to-nearest-even of w / s, and the
# weight used is q * s (exact in bfloat16 and in float64).
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
FP8_BLOCK = 128


def block_scale_exponent(amax: float) -> int:
    """Smallest k with amax <= 448 * 2^k (0 for an all-zero block), from the
    exact binary exponents of amax and 448 = 0.875 * 2^9."""
    if amax == 0.0:
        return 0
    m, e = np.frexp(amax)  # amax = m * 2^e, m in [0.5, 1)
    return int(e - 9 if m <= 0.875 else e - 8)


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448.
    Normal values 2^e (1 + j/8), e in [-6, 8]; subnormals j 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -6)             # binade exponent (subnormals share e = -6)
    step = np.ldexp(1.0, e - 3)            # spacing of the binade: 3 mantissa bits
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.copysign(q, x)  # the sign survives rounding to zero


def e4m3_bits(q: np.ndarray) -> np.ndarray:
    """Encoding of E4M3 values (as produced by e4m3_round): sign, 4-bit
    exponent field (bias 7, 0 for subnormals), 3-bit mantissa."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    sign = (q < 0) | ((q == 0) & np.signbit(q))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex - 1
    normal = a >= 2.0 ** -6
    efield = np.where(normal, e + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, e) * 8 - 8, a / 2.0 ** -9)
    bits = (sign.astype(np.int64) << 7) | (efield.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    return bits.astype(np.uint8)


def e4m3_value(bits: np.ndarray) -> np.ndarray:
    """Value of E4M3 codes (the NaN codes 0x7F / 0xFF are never produced)."""
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    efield = (b >> 3) & 0xF
    mant = b & 0x7
    v = np.where(efield == 0, mant * 2.0 ** -9, np.ldexp(1.0 + mant / 8.0, efield - 7))
    return sign * v


def quantize_fp8_blocks(w: np.ndarray) -> dict:
    """Block quantization of one [rows, cols] matrix: E4M3 codes [rows, cols],
    scale exponents [ceil(rows/128), ceil(cols/128)], and the dequantized
    matrix q * s."""
    rows, cols = w.shape
    nb_r, nb_c = -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK)
    k = np.zeros((nb_r, nb_c), dtype=np.int64)
    deq = np.empty_like(w, dtype=np.float64)
    codes = np.empty(w.shape, dtype=np.uint8)
    for i in range(nb_r):
        for j in range(nb_c):
            blk = w[i * FP8_BLOCK:(i + 1) * FP8_BLOCK, j * FP8_BLOCK:(j + 1) * FP8_BLOCK]
            k[i, j] = block_scale_exponent(float(np.max(np.abs(blk))))
            q = e4m3_round(np.ldexp(blk, -k[i, j]))
            codes[i * FP8_BLOCK:(i + 1) * FP8_BLOCK, j * FP8_BLOCK:(j + 1) * FP8_BLOCK] = e4m3_bits(q)
            deq[i * FP8_BLOCK:(i + 1) * FP8_BLOCK, j * FP8_BLOCK:(j + 1) * FP8_BLOCK] = np.ldexp(q, k[i, j])
    return {"codes": codes, "exp": k, "w": deq}


FP8_MATRICES = ("w_q_a", "w_q_b", "w_kv_a", "w_kv_b", "w_o")


def quantize_weights_fp8(w: dict) -> dict:
    """The MLA weights with the five projection matrices replaced by their
    block-quantized values (gains unchanged); the decode functions above then
    compute with exactly the weights the FP8 path stores."""
    out = dict(w)
    for n in FP8_MATRICES:
        out[n] = quantize_fp8_blocks(w[n])["w"]
    return out
