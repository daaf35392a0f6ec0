"""FP8 block-scaled weights on the GPU against the oracle.

* the quantizer (mla_quantize_fp8) on the five seeded projection matrices:
  codes (stored block-major) and scales bit-exact against the oracle's
  quantize_fp8_blocks (integer / byte work);
* mla_decode_fp8 against the oracle's decode computed with the oracle's own
  dequantized weights (the same tolerance as every decode: max abs <= 2e-2
  + half a bf16 ulp of |out|, relative Frobenius <= 1e-2), at decode sizes
  that take every tile configuration of the FP8-weight GEMM (M <= 64 and
  M <= 128, split-K A-projection).
"""
import functools

import numpy as np
import pytest

import synth
from oracle import mla_oracle as om
import mla_gb300 as m
from mla_testlib import (bits_to_cuda, cuda_to_f64, cuda_weights, oracle_weights, parity, parity_cache,
                         parity_out)
from test_parity_small import make_caches

pytestmark = pytest.mark.gpu

ORACLE = {"w_q_a": "w_q_a", "w_q_b": "w_q_b", "w_kv_a": "w_kv_a", "w_kv_b": "w_kv_b", "w_o": "w_o"}


@functools.lru_cache(maxsize=1)
def oracle_fp8():
    """Per matrix: the oracle's codes, scale exponents and dequantized weights."""
    w = oracle_weights(0)
    return {n: om.quantize_fp8_blocks(w[n]) for n in om.FP8_MATRICES}


@pytest.fixture(scope="module")
def WQ(gpu_available):
    wt = cuda_weights(0)
    st, tensors = m.make_weights_fp8(wt)
    import torch
    torch.cuda.synchronize()
    wq = dict(oracle_weights(0))
    for n, r in oracle_fp8().items():
        wq[n] = r["w"]
    return st, tensors, wq


def block_major(codes):
    """[rows, cols] -> [ceil(rows/128), cols/128, 128, 128], rows past the matrix zero."""
    rows, cols = codes.shape
    nb = -(-rows // 128)
    pad = np.zeros((nb * 128, cols), dtype=np.uint8)
    pad[:rows] = codes
    return pad.reshape(nb, 128, cols // 128, 128).transpose(0, 2, 1, 3)


def test_quantizer_bit_exact(WQ):
    _, t, _ = WQ
    for n, r in oracle_fp8().items():
        codes = t[n].cpu().numpy()
        ref = block_major(r["codes"])
        assert np.array_equal(codes, ref), f"{n}: {np.count_nonzero(codes != ref)} codes differ"
        scales = t["s_" + n[2:]].cpu().numpy().astype(np.float64)
        assert np.array_equal(scales, np.ldexp(1.0, r["exp"])), f"{n}: scales differ"


@pytest.mark.parametrize("B,P", [(3, 37), (2, 0), (100, 129), (64, 300)])
def test_decode_fp8_parity(WQ, B, P):
    import torch
    st, _, wq = WQ
    cap = P + 3
    W = (cuda_weights(0), None, oracle_weights(0))
    (Kb, Vb, _, _), (K64, V64, _, _) = make_caches(W, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    kc, vc = bits_to_cuda(Kb), bits_to_cuda(Vb)
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE, B, P)
    m.mla_decode_fp8(st, x, P, kc, vc, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.decode(wq, synth.bf16_bits_to_f64(xb), K64, V64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(kc[:, :, P]), ref["k_new"], "new K row")
    parity_cache(cuda_to_f64(vc[:, :, P]), ref["v_new"], "new V row")
