"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the headers declare, sizes workspaces, and rejects bad
arguments before enqueueing anything (the pages' code raises ValueError /
asserts on shape mismatches; here they become status codes)."""
import ctypes
import os
import re

import pytest

import mla_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions(headers=None):
    names = []
    for h in headers or [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
                         if f.endswith(".h")]:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function():
    lib = m.lib()
    names = declared_functions()
    assert "mla_prefill" in names and "mla_decode_latent" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_product_library_carries_no_test_hooks_and_hooks_library_exports_them():
    import mla_hooks
    hooks = declared_functions([os.path.join(ROOT, "tests", "hooks", "mla_debug.h")])
    assert hooks == ["mla_debug_gemm", "mla_debug_umma_probe", "mla_debug_wait_timeout"]
    lib = m.lib()
    for n in hooks:
        assert not hasattr(lib, n), f"{n} exported by libmla.so"
    hl = mla_hooks.lib()
    for n in hooks:
        assert hasattr(hl, n), f"{n} not exported by the hooks library"


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert m.STATUS[code] in m.mla_status_string(code)


def test_workspace_sizes():
    p1 = m.workspace_size(m.MODE_PREFILL, 1, 16)
    p2 = m.workspace_size(m.MODE_PREFILL, 1, 2048)
    assert 0 < p1 < p2
    assert m.workspace_size(m.MODE_DECODE, 64, 1000) > 0
    assert m.workspace_size(m.MODE_DECODE_LATENT, 128, 8192) > 0
    assert m.lib().mla_workspace_size(m.MODE_PREFILL, 0, 16, 0) == 0
    assert m.lib().mla_workspace_size(m.MODE_PREFILL, 1, 0, 0) == 0
    assert m.lib().mla_workspace_size(7, 1, 16, 0) == 0
    assert m.lib().mla_workspace_size(m.MODE_DECODE, 1, -1, 0) == 0


FAKE = 1 << 40  # never dereferenced: every call below fails its host checks


def fake_weights(**override):
    vals = {n: FAKE + 4096 * i for i, n in enumerate(m.WEIGHT_NAMES)}
    vals.update(override)
    return m.MlaWeights(*[vals[n] for n in m.WEIGHT_NAMES])


def prefill(w, B=1, T=16, x=FAKE + (1 << 30), out=FAKE + (2 << 30), kc=None, vc=None, ckv=None, kpe=None,
            cap=0, ws=FAKE + (3 << 30), ws_bytes=None, params=None):
    if ws_bytes is None:
        ws_bytes = m.lib().mla_workspace_size(m.MODE_PREFILL, max(B, 1), max(T, 1), cap)
    return m.lib().mla_prefill(ctypes.byref(w), params, x, B, T, out, kc, vc, ckv, kpe, cap, ws, ws_bytes, None)


def test_prefill_argument_checks():
    w = fake_weights()
    assert prefill(w, B=0) == -1
    assert prefill(w, T=0) == -1
    assert prefill(fake_weights(w_o=None)) == -1
    assert prefill(fake_weights(w_q_b=FAKE + 8)) == -2
    assert prefill(w, x=FAKE + (1 << 30) + 2) == -2
    assert prefill(w, ws=None) == -3
    assert prefill(w, ws_bytes=1024) == -3
    # out overlapping x without being the same buffer
    assert prefill(w, out=FAKE + (1 << 30) + 4096) == -1
    # only one of a cache pair, or a cache smaller than T
    assert prefill(w, kc=FAKE + (4 << 30)) == -1
    assert prefill(w, ckv=FAKE + (4 << 30)) == -1
    assert prefill(w, kc=FAKE + (4 << 30), vc=FAKE + (5 << 30), cap=15) == -1
    bad = m.MlaParams(-1.0, 10000.0, 0.07, None, None)
    assert prefill(w, params=ctypes.byref(bad)) == -1


def test_decode_argument_checks():
    w = fake_weights()
    L = m.lib()
    ws_bytes = L.mla_workspace_size(m.MODE_DECODE, 4, 10, 11)
    args = dict(x=FAKE + (1 << 30), kc=FAKE + (2 << 30), vc=FAKE + (3 << 30), out=FAKE + (4 << 30),
                ws=FAKE + (5 << 30))

    def dec(B=4, P=10, cap=11, **kw):
        a = dict(args, **kw)
        return L.mla_decode(ctypes.byref(w), None, a["x"], B, P, a["kc"], a["vc"], cap, a["out"], a["ws"],
                            ws_bytes, None)

    assert dec(B=0) == -1
    assert dec(P=-1) == -1
    assert dec(cap=10) == -1            # P + 1 > cap
    assert dec(kc=None) == -1
    assert dec(vc=FAKE + 8) == -2

    ws_l = L.mla_workspace_size(m.MODE_DECODE_LATENT, 4, 10, 11)
    assert L.mla_decode_latent(ctypes.byref(w), None, args["x"], 4, 10, args["kc"], None, 11, args["out"],
                               args["ws"], ws_l, None) == -1
    assert L.mla_decode_latent(ctypes.byref(w), None, args["x"], 4, 10, args["kc"], args["vc"], 10, args["out"],
                               args["ws"], ws_l, None) == -1
    assert L.mla_decode_latent(ctypes.byref(w), None, args["x"], 4, 10, args["kc"], args["vc"], 11, args["out"],
                               args["ws"], 100, None) == -3


def chunk(w, B=1, T=16, P0=8, out=FAKE + (2 << 30), kc=FAKE + (4 << 30), vc=FAKE + (5 << 30), cap=64):
    ws_bytes = m.lib().mla_workspace_size(m.MODE_PREFILL, B, T, cap)
    return m.lib().mla_prefill_chunk(ctypes.byref(w), None, FAKE + (1 << 30), B, T, P0, out, kc, vc, None, None,
                                     cap, FAKE + (3 << 30), ws_bytes, None)


def test_prefill_chunk_argument_checks():
    w = fake_weights()
    assert chunk(w, P0=-1) == -1
    assert chunk(w, P0=49, T=16, cap=64) == -1       # P0 + T > cap
    assert chunk(w, kc=None, vc=None) == -1          # the rebuilt cache holds the past: required
    assert chunk(w, vc=None) == -1
    assert chunk(w, out=None) == -1
    assert chunk(w, kc=FAKE + (4 << 30) + 8) == -2


def fake_ffn_weights(**override):
    vals = {n: FAKE + 4096 * i for i, n in enumerate(m.FFN_WEIGHT_NAMES)}
    vals.update(override)
    return m.MlaFfnWeights(*[vals[n] for n in m.FFN_WEIGHT_NAMES])


def ffn(w, n=16, x=FAKE + (1 << 30), out=FAKE + (2 << 30), ws=FAKE + (3 << 30), ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = m.lib().mla_workspace_size(m.MODE_FFN, 1, max(n, 1), 0)
    return m.lib().mla_ffn(ctypes.byref(w), None, x, n, out, ws, ws_bytes, None)


def test_ffn_workspace_and_argument_checks():
    n = 2048
    assert m.workspace_size(m.MODE_FFN, 1, n) >= n * (m.D + m.FFN_INTER) * 2
    assert m.workspace_size(m.MODE_FFN, 4, 512) == m.workspace_size(m.MODE_FFN, 1, 2048)
    assert m.lib().mla_workspace_size(m.MODE_FFN, 1, 0, 0) == 0
    w = fake_ffn_weights()
    assert ffn(w, n=0) == -1
    assert ffn(fake_ffn_weights(w_2=None)) == -1
    assert ffn(fake_ffn_weights(w_1=FAKE + 8)) == -2
    assert ffn(w, x=None) == -1
    assert ffn(w, out=None) == -1
    assert ffn(w, ws=None) == -3
    assert ffn(w, ws_bytes=4096) == -3
    assert ffn(w, out=FAKE + (1 << 30) + 4096) == -1  # partial overlap with x


def test_prefill_chunk_latent_argument_checks():
    w = fake_weights()
    cap = 64
    ws_bytes = m.lib().mla_workspace_size(m.MODE_CHUNK_LATENT, 1, 16, cap)
    assert ws_bytes > m.lib().mla_workspace_size(m.MODE_PREFILL, 1, 16, cap)  # holds K/V of cap positions
    assert m.lib().mla_workspace_size(m.MODE_CHUNK_LATENT, 1, 16, 8) == 0     # cap < T

    def call(P0=8, T=16, out=FAKE + (2 << 30), ckv=FAKE + (4 << 30), kpe=FAKE + (5 << 30), nbytes=ws_bytes):
        return m.lib().mla_prefill_chunk_latent(ctypes.byref(w), None, FAKE + (1 << 30), 1, T, P0, out, ckv, kpe,
                                                cap, FAKE + (3 << 30), nbytes, None)
    assert call(P0=-1) == -1
    assert call(P0=49) == -1           # P0 + T > cap
    assert call(ckv=None) == -1
    assert call(kpe=None) == -1
    assert call(out=None) == -1
    assert call(kpe=FAKE + (5 << 30) + 8) == -2
    assert call(nbytes=ws_bytes - 256) == -3


def test_prefill_chunk_absorbed_argument_checks():
    w = fake_weights()
    cap = 64
    ws_bytes = m.lib().mla_workspace_size(m.MODE_CHUNK_ABSORBED, 2, 4, cap)
    assert ws_bytes > 0
    # one latent decode row per new token: the same bytes as a latent decode of B * T rows, plus positions
    assert ws_bytes >= m.lib().mla_workspace_size(m.MODE_DECODE_LATENT, 8, cap - 1, 0)
    # no rebuilt keys and values: much smaller than the rebuilt form's workspace at a long cache
    assert m.lib().mla_workspace_size(m.MODE_CHUNK_ABSORBED, 2, 4, 8192) < \
        m.lib().mla_workspace_size(m.MODE_CHUNK_LATENT, 2, 4, 8192) // 4
    assert m.lib().mla_workspace_size(m.MODE_CHUNK_ABSORBED, 2, 4, 3) == 0   # cap < T
    assert m.lib().mla_workspace_size(m.MODE_CHUNK_ABSORBED, 2, 0, cap) == 0  # T < 1

    def call(P0=8, T=4, out=FAKE + (2 << 30), ckv=FAKE + (4 << 30), kpe=FAKE + (5 << 30), nbytes=ws_bytes):
        return m.lib().mla_prefill_chunk_absorbed(ctypes.byref(w), None, FAKE + (1 << 30), 2, T, P0, out, ckv, kpe,
                                                  cap, FAKE + (3 << 30), nbytes, None)
    assert call(P0=-1) == -1
    assert call(P0=61) == -1           # P0 + T > cap
    assert call(T=0) == -1
    assert call(ckv=None) == -1
    assert call(kpe=None) == -1
    assert call(out=None) == -1
    assert call(ckv=FAKE + (4 << 30) + 8) == -2
    assert call(nbytes=ws_bytes - 256) == -3


def test_fold_entries_argument_checks():
    w = fake_weights()
    ws_bytes = m.lib().mla_workspace_size(m.MODE_FOLD, 1, 1, 0)
    assert ws_bytes > 0
    fold = m.lib().mla_fold_wuv_into_wo
    assert fold(ctypes.byref(w), None, FAKE + (3 << 30), ws_bytes, None) == -1
    assert fold(ctypes.byref(w), FAKE + (2 << 30) + 8, FAKE + (3 << 30), ws_bytes, None) == -2
    assert fold(ctypes.byref(w), FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes - 256, None) == -3
    assert fold(ctypes.byref(w), FAKE + (2 << 30), None, ws_bytes, None) == -3
    dws = m.lib().mla_workspace_size(m.MODE_DECODE_LATENT, 4, 10, 0)

    def dec(wf=FAKE + (6 << 30), P=10, cap=11):
        return m.lib().mla_decode_latent_folded(ctypes.byref(w), wf, None, FAKE + (1 << 30), 4, P, FAKE + (4 << 30),
                                                FAKE + (5 << 30), cap, FAKE + (2 << 30), FAKE + (3 << 30), dws, None)
    assert dec(wf=None) == -1
    assert dec(wf=FAKE + (6 << 30) + 8) == -2
    assert dec(cap=10) == -1           # P + 1 > cap


def test_fp8_entry_argument_checks():
    lib = m.lib()
    # quantizer: cols must be a multiple of 128, pointers 16-byte aligned (scales 4-byte)
    assert lib.mla_quantize_fp8(FAKE, 128, 100, FAKE + (1 << 30), FAKE + (2 << 30), None) == -1
    assert lib.mla_quantize_fp8(None, 128, 128, FAKE + (1 << 30), FAKE + (2 << 30), None) == -1
    assert lib.mla_quantize_fp8(FAKE + 8, 128, 128, FAKE + (1 << 30), FAKE + (2 << 30), None) == -2
    assert lib.mla_quantize_fp8(FAKE, 128, 128, FAKE + (1 << 30), FAKE + (2 << 30) + 2, None) == -2
    # FP8 decode: every scale pointer required
    vals = {f: FAKE + 4096 * i for i, (f, _) in enumerate(m.MlaWeightsFp8._fields_)}
    ws_bytes = lib.mla_workspace_size(m.MODE_DECODE, 4, 10, 0)
    for missing in ("s_q_a", "s_o"):
        w = m.MlaWeightsFp8(*[None if f == missing else vals[f] for f, _ in m.MlaWeightsFp8._fields_])
        assert lib.mla_decode_fp8(ctypes.byref(w), None, FAKE + (1 << 30), 4, 10, FAKE + (4 << 30), FAKE + (5 << 30),
                                  11, FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -1
    w = m.MlaWeightsFp8(*[vals[f] for f, _ in m.MlaWeightsFp8._fields_])
    assert lib.mla_decode_fp8(ctypes.byref(w), None, FAKE + (1 << 30), 4, 10, FAKE + (4 << 30), FAKE + (5 << 30),
                              10, FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -1  # cap < P + 1


def test_varlen_decode_argument_checks():
    lib = m.lib()
    w = fake_weights()
    ws_bytes = lib.mla_workspace_size(m.MODE_DECODE, 4, 10, 0)
    args = (FAKE + (1 << 30), 4)
    # the per-sequence positions are required and 4-byte aligned; P_max + 1 <= cap
    assert lib.mla_decode_varlen(ctypes.byref(w), None, *args, None, 10, FAKE + (4 << 30), FAKE + (5 << 30), 11,
                                 FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -1
    assert lib.mla_decode_varlen(ctypes.byref(w), None, *args, FAKE + (6 << 30) + 2, 10, FAKE + (4 << 30),
                                 FAKE + (5 << 30), 11, FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -2
    assert lib.mla_decode_varlen(ctypes.byref(w), None, *args, FAKE + (6 << 30), 11, FAKE + (4 << 30),
                                 FAKE + (5 << 30), 11, FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -1
    lws = lib.mla_workspace_size(m.MODE_DECODE_LATENT, 4, 10, 0)
    assert lib.mla_decode_latent_varlen(ctypes.byref(w), None, *args, None, 10, FAKE + (4 << 30), FAKE + (5 << 30),
                                        11, FAKE + (2 << 30), FAKE + (3 << 30), lws, None) == -1


def test_fp8_scales_alignment():
    lib = m.lib()
    vals = {f: FAKE + 4096 * i for i, (f, _) in enumerate(m.MlaWeightsFp8._fields_)}
    vals["s_kv_b"] += 2
    w = m.MlaWeightsFp8(*[vals[f] for f, _ in m.MlaWeightsFp8._fields_])
    ws_bytes = lib.mla_workspace_size(m.MODE_DECODE, 4, 10, 0)
    assert lib.mla_decode_fp8(ctypes.byref(w), None, FAKE + (1 << 30), 4, 10, FAKE + (4 << 30), FAKE + (5 << 30),
                              11, FAKE + (2 << 30), FAKE + (3 << 30), ws_bytes, None) == -2
