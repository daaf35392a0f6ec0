"""Python binding of libmla.so (the GB300 MLA sublayer).

Argument marshalling only: each function takes torch tensors for device
memory and the current torch stream, and calls the C entry point of the same
name (include/mla.h).  Every step of the computation runs in the library's
CUDA kernels; there is no fallback.  If the library has not been built the
import of ``lib()`` fails loudly.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

D, HEADS, Q_LORA, KV_LORA, QK_NOPE, QK_ROPE, QK, V = 7168, 64, 1536, 512, 128, 64, 192, 128
FFN_INTER = 18432
MODE_PREFILL, MODE_DECODE, MODE_DECODE_LATENT, MODE_FFN, MODE_CHUNK_LATENT, MODE_CHUNK_ABSORBED = 0, 1, 2, 3, 4, 5
MODE_FOLD = 6
STAGES = ["input_norm", "a_proj", "latent", "q_b", "kv_b", "attn", "combine", "absorb_q", "absorb_o", "o_proj",
          "ffn_norm", "gate_up", "down"]
MAX_STAGES = len(STAGES)

STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_ALIGNMENT", -3: "MLA_ERR_WORKSPACE",
          -4: "MLA_ERR_UNSUPPORTED", -5: "MLA_ERR_CUDA", -6: "MLA_ERR_TIMEOUT"}

WEIGHT_NAMES = ["w_in_norm", "w_q_a", "w_q_a_norm", "w_q_b", "w_kv_a", "w_kv_a_norm", "w_kv_b", "w_o"]
WEIGHT_SHAPES = {
    "w_in_norm": (D,), "w_q_a": (Q_LORA, D), "w_q_a_norm": (Q_LORA,), "w_q_b": (HEADS * QK, Q_LORA),
    "w_kv_a": (KV_LORA + QK_ROPE, D), "w_kv_a_norm": (KV_LORA,), "w_kv_b": (HEADS * (QK_NOPE + V), KV_LORA),
    "w_o": (D, HEADS * V),
}
FFN_WEIGHT_NAMES = ["w_post_norm", "w_1", "w_3", "w_2"]
FFN_WEIGHT_SHAPES = {"w_post_norm": (D,), "w_1": (FFN_INTER, D), "w_3": (FFN_INTER, D), "w_2": (D, FFN_INTER)}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MlaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_NAMES]


FP8_NAMES = ["w_q_a", "w_q_b", "w_kv_a", "w_kv_b", "w_o"]


class MlaWeightsFp8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ["w_in_norm", "w_q_a_norm", "w_kv_a_norm"] + FP8_NAMES] + \
               [("s_" + n[2:], ctypes.c_void_p) for n in FP8_NAMES]


class MlaFfnWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in FFN_WEIGHT_NAMES]


class MlaTiming(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p * MAX_STAGES), ("stop", ctypes.c_void_p * MAX_STAGES),
                ("n_launches", ctypes.c_int)]


class MlaParams(ctypes.Structure):
    _fields_ = [("eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("softmax_scale", ctypes.c_float),
                ("delta_out", ctypes.c_void_p), ("timing", ctypes.POINTER(MlaTiming))]


_lib = None

_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "mla_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "mla_prefill": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _VP, _VP, _VP, _VP,
                         _VP, _I, _VP, _SZ, _VP]),
    "mla_prefill_chunk": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _I, _VP, _VP,
                               _VP, _VP, _VP, _I, _VP, _SZ, _VP]),
    "mla_prefill_chunk_latent": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _I, _VP,
                                      _VP, _VP, _I, _VP, _SZ, _VP]),
    "mla_prefill_chunk_absorbed": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _I,
                                        _VP, _VP, _VP, _I, _VP, _SZ, _VP]),
    "mla_decode": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _VP, _VP, _I, _VP,
                        _VP, _SZ, _VP]),
    "mla_decode_latent": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _VP, _VP, _I,
                               _VP, _VP, _SZ, _VP]),
    "mla_fold_wuv_into_wo": (_I, [ctypes.POINTER(MlaWeights), _VP, _VP, _SZ, _VP]),
    "mla_decode_latent_folded": (_I, [ctypes.POINTER(MlaWeights), _VP, ctypes.POINTER(MlaParams), _VP, _I, _I, _VP,
                                      _VP, _I, _VP, _VP, _SZ, _VP]),
    "mla_decode_varlen": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _VP, _I, _VP, _VP,
                               _I, _VP, _VP, _SZ, _VP]),
    "mla_decode_latent_varlen": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _VP, _I, _VP,
                                      _VP, _I, _VP, _VP, _SZ, _VP]),
    "mla_decode_noalloc": (_I, [ctypes.POINTER(MlaWeights), ctypes.POINTER(MlaParams), _VP, _I, _I, _VP, _VP, _I,
                                _VP, _VP]),
    "mla_ffn": (_I, [ctypes.POINTER(MlaFfnWeights), ctypes.POINTER(MlaParams), _VP, _I, _VP, _VP, _SZ, _VP]),
    "mla_quantize_fp8": (_I, [_VP, _I, _I, _VP, _VP, _VP]),
    "mla_decode_fp8": (_I, [ctypes.POINTER(MlaWeightsFp8), ctypes.POINTER(MlaParams), _VP, _I, _I, _VP, _VP, _I, _VP,
                            _VP, _SZ, _VP]),
    "mla_device_status": (_I, [_VP, _VP]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
}


def lib():
    """The loaded libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: the CUDA library must be built "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise MlaError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_weights(w: dict) -> MlaWeights:
    """Pack a dict of bf16 CUDA tensors (names of WEIGHT_NAMES) into the C struct."""
    import torch
    for n in WEIGHT_NAMES:
        t = w[n]
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != WEIGHT_SHAPES[n]:
            raise ValueError(f"weight {n}: need contiguous bf16 CUDA tensor of shape {WEIGHT_SHAPES[n]}")
    s = MlaWeights(*[w[n].data_ptr() for n in WEIGHT_NAMES])
    s._keep = dict(w)  # the struct holds raw pointers: keep the tensors alive with it
    return s


def make_ffn_weights(w: dict) -> MlaFfnWeights:
    """Pack a dict of bf16 CUDA tensors (names of FFN_WEIGHT_NAMES) into the C struct."""
    import torch
    for n in FFN_WEIGHT_NAMES:
        t = w[n]
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or \
                tuple(t.shape) != FFN_WEIGHT_SHAPES[n]:
            raise ValueError(f"weight {n}: need contiguous bf16 CUDA tensor of shape {FFN_WEIGHT_SHAPES[n]}")
    s = MlaFfnWeights(*[w[n].data_ptr() for n in FFN_WEIGHT_NAMES])
    s._keep = dict(w)
    return s


def make_params(eps=1e-6, rope_base=10000.0, softmax_scale=None, delta_out=None, timing=None) -> MlaParams:
    if softmax_scale is None:
        softmax_scale = 1.0 / (QK ** 0.5)
    return MlaParams(eps, rope_base, softmax_scale,
                     None if delta_out is None else delta_out.data_ptr(),
                     None if timing is None else ctypes.pointer(timing))


def workspace_size(mode: int, B: int, t_or_p: int, cap: int = 0) -> int:
    n = lib().mla_workspace_size(mode, B, t_or_p, cap)
    if n == 0:
        raise MlaError(-1, "mla_workspace_size")
    return n


def alloc_workspace(mode: int, B: int, t_or_p: int, device="cuda", cap: int = 0):
    import torch
    return torch.empty(workspace_size(mode, B, t_or_p, cap), dtype=torch.uint8, device=device)


def mla_prefill(weights: MlaWeights, x, out, workspace, k_cache=None, v_cache=None, ckv_cache=None,
                kpe_cache=None, cap=0, params: MlaParams | None = None, stream=None):
    """x, out: bf16 [B, T, 7168] (out None: fill the given caches only); caches as in include/mla.h."""
    B, T = x.shape[0], x.shape[1]
    rc = lib().mla_prefill(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x), B, T,
                           _ptr(out), _ptr(k_cache), _ptr(v_cache), _ptr(ckv_cache), _ptr(kpe_cache), cap,
                           _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_prefill")


def mla_prefill_chunk(weights: MlaWeights, x, P0: int, out, k_cache, v_cache, workspace, ckv_cache=None,
                      kpe_cache=None, params: MlaParams | None = None, stream=None):
    """x, out: bf16 [B, T, 7168], the chunk at positions P0..P0+T-1; k_cache [B, 64, cap, 192] and
    v_cache [B, 64, cap, 128] hold rows 0..P0-1 and receive rows P0..P0+T-1."""
    B, T = x.shape[0], x.shape[1]
    cap = k_cache.shape[2]
    rc = lib().mla_prefill_chunk(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x),
                                 B, T, P0, _ptr(out), _ptr(k_cache), _ptr(v_cache), _ptr(ckv_cache),
                                 _ptr(kpe_cache), cap, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_prefill_chunk")


def mla_prefill_chunk_latent(weights: MlaWeights, x, P0: int, out, ckv_cache, kpe_cache, workspace,
                             params: MlaParams | None = None, stream=None):
    """x, out: bf16 [B, T, 7168] at positions P0..P0+T-1; ckv_cache [B, cap, 512] and kpe_cache
    [B, cap, 64] hold rows 0..P0-1 and receive rows P0..P0+T-1; workspace of MODE_CHUNK_LATENT
    sized with the same cap."""
    B, T = x.shape[0], x.shape[1]
    cap = ckv_cache.shape[1]
    rc = lib().mla_prefill_chunk_latent(ctypes.byref(weights), None if params is None else ctypes.byref(params),
                                        _ptr(x), B, T, P0, _ptr(out), _ptr(ckv_cache), _ptr(kpe_cache), cap,
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_prefill_chunk_latent")


def mla_prefill_chunk_absorbed(weights: MlaWeights, x, P0: int, out, ckv_cache, kpe_cache, workspace,
                               params: MlaParams | None = None, stream=None):
    """The same chunk as mla_prefill_chunk_latent in the absorbed form (one latent decode row per new
    token); workspace of MODE_CHUNK_ABSORBED sized with the same B, T and cap."""
    B, T = x.shape[0], x.shape[1]
    cap = ckv_cache.shape[1]
    rc = lib().mla_prefill_chunk_absorbed(ctypes.byref(weights), None if params is None else ctypes.byref(params),
                                          _ptr(x), B, T, P0, _ptr(out), _ptr(ckv_cache), _ptr(kpe_cache), cap,
                                          _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_prefill_chunk_absorbed")


def mla_decode(weights: MlaWeights, x, P: int, k_cache, v_cache, out, workspace,
               params: MlaParams | None = None, stream=None):
    """x, out: bf16 [B, 7168]; k_cache [B, 64, cap, 192], v_cache [B, 64, cap, 128]."""
    B = x.shape[0]
    cap = k_cache.shape[2]
    rc = lib().mla_decode(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x), B, P,
                          _ptr(k_cache), _ptr(v_cache), cap, _ptr(out), _ptr(workspace), workspace.numel(),
                          _stream(stream))
    _check(rc, "mla_decode")


def mla_decode_latent(weights: MlaWeights, x, P: int, ckv_cache, kpe_cache, out, workspace,
                      params: MlaParams | None = None, stream=None):
    """x, out: bf16 [B, 7168]; ckv_cache [B, cap, 512], kpe_cache [B, cap, 64]."""
    B = x.shape[0]
    cap = ckv_cache.shape[1]
    rc = lib().mla_decode_latent(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x),
                                 B, P, _ptr(ckv_cache), _ptr(kpe_cache), cap, _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(rc, "mla_decode_latent")


def mla_fold_wuv_into_wo(weights: MlaWeights, w_fold, workspace, stream=None):
    """w_fold: bf16 [7168, 64 * 512] receives W_o's head blocks times W_UV per head; workspace of MODE_FOLD."""
    rc = lib().mla_fold_wuv_into_wo(ctypes.byref(weights), _ptr(w_fold), _ptr(workspace), workspace.numel(),
                                    _stream(stream))
    _check(rc, "mla_fold_wuv_into_wo")


def mla_decode_latent_folded(weights: MlaWeights, w_fold, x, P: int, ckv_cache, kpe_cache, out, workspace,
                             params: MlaParams | None = None, stream=None):
    """mla_decode_latent with W_UV folded into o_proj (w_fold from mla_fold_wuv_into_wo)."""
    B = x.shape[0]
    cap = ckv_cache.shape[1]
    rc = lib().mla_decode_latent_folded(ctypes.byref(weights), _ptr(w_fold),
                                        None if params is None else ctypes.byref(params), _ptr(x), B, P,
                                        _ptr(ckv_cache), _ptr(kpe_cache), cap, _ptr(out), _ptr(workspace),
                                        workspace.numel(), _stream(stream))
    _check(rc, "mla_decode_latent_folded")


def mla_decode_varlen(weights: MlaWeights, x, P, P_max: int, k_cache, v_cache, out, workspace,
                      params: MlaParams | None = None, stream=None):
    """Ragged decode: P is an int32 CUDA tensor [B] of per-sequence positions (<= P_max)."""
    B = x.shape[0]
    cap = k_cache.shape[2]
    rc = lib().mla_decode_varlen(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x), B,
                                 _ptr(P), P_max, _ptr(k_cache), _ptr(v_cache), cap, _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(rc, "mla_decode_varlen")


def mla_decode_latent_varlen(weights: MlaWeights, x, P, P_max: int, ckv_cache, kpe_cache, out, workspace,
                             params: MlaParams | None = None, stream=None):
    """Ragged latent decode: P is an int32 CUDA tensor [B] of per-sequence positions (<= P_max)."""
    B = x.shape[0]
    cap = ckv_cache.shape[1]
    rc = lib().mla_decode_latent_varlen(ctypes.byref(weights), None if params is None else ctypes.byref(params),
                                        _ptr(x), B, _ptr(P), P_max, _ptr(ckv_cache), _ptr(kpe_cache), cap, _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_decode_latent_varlen")


def mla_decode_noalloc(weights: MlaWeights, x, P: int, k_cache, v_cache, out, params: MlaParams | None = None,
                       stream=None):
    """mla_decode with its scratch in the library's fixed static device array
    (for callers that cannot allocate device memory); no workspace argument."""
    B = x.shape[0]
    cap = k_cache.shape[2]
    rc = lib().mla_decode_noalloc(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x),
                                  B, P, _ptr(k_cache), _ptr(v_cache), cap, _ptr(out), _stream(stream))
    _check(rc, "mla_decode_noalloc")


def mla_ffn(weights: MlaFfnWeights, x, out, workspace, params: MlaParams | None = None, stream=None):
    """x, out: bf16 [..., 7168] (out = x + Delta_ffn, may be x itself)."""
    n_tok = x.numel() // D
    rc = lib().mla_ffn(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x), n_tok,
                       _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mla_ffn")


def mla_quantize_fp8(w, codes, scales, stream=None):
    """w: bf16 CUDA [rows, cols] (cols % 128 == 0) -> codes uint8 block-major
    [ceil(rows/128), cols/128, 128, 128], scales float32 [ceil(rows/128), cols/128]."""
    rows, cols = w.shape
    _check(lib().mla_quantize_fp8(_ptr(w), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)),
           "mla_quantize_fp8")


def make_weights_fp8(w: dict, stream=None):
    """FP8 block-scaled copies of the five projection matrices of a bf16
    weight dict (quantized by the library) packed with the bf16 gains;
    returns (struct, dict of the tensors it points to)."""
    import torch
    t = {n: w[n] for n in ("w_in_norm", "w_q_a_norm", "w_kv_a_norm")}
    for n in FP8_NAMES:
        rows, cols = w[n].shape
        t[n] = torch.empty(((rows + 127) // 128, cols // 128, 128, 128), dtype=torch.uint8, device=w[n].device)
        t["s_" + n[2:]] = torch.empty(((rows + 127) // 128, (cols + 127) // 128), dtype=torch.float32,
                                     device=w[n].device)
        mla_quantize_fp8(w[n], t[n], t["s_" + n[2:]], stream)
    st = MlaWeightsFp8(*[t[f].data_ptr() for f, _ in MlaWeightsFp8._fields_])
    st._keep = t
    return st, t


def mla_decode_fp8(weights: MlaWeightsFp8, x, P: int, k_cache, v_cache, out, workspace,
                   params: MlaParams | None = None, stream=None):
    """mla_decode with FP8 block-scaled weights (make_weights_fp8)."""
    B = x.shape[0]
    cap = k_cache.shape[2]
    rc = lib().mla_decode_fp8(ctypes.byref(weights), None if params is None else ctypes.byref(params), _ptr(x), B, P,
                              _ptr(k_cache), _ptr(v_cache), cap, _ptr(out), _ptr(workspace), workspace.numel(),
                              _stream(stream))
    _check(rc, "mla_decode_fp8")


def mla_device_status(workspace, stream=None) -> int:
    return lib().mla_device_status(_ptr(workspace), _stream(stream))


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()
