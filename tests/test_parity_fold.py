"""W_UV folded into o_proj on the GPU against the oracle.

* mla_fold_wuv_into_wo: sampled rows of W_fold against the oracle's fold of
  the same bf16 weights (each entry a 128-term sum rounded once to bf16: the
  cache tolerance, one bf16 ulp);
* mla_decode_latent_folded against the oracle's rebuilt-cache latent decode
  (the two are equal by associativity; the GPU rounds W_fold to bf16 once),
  with the decode tolerance, at sizes that take the M <= 64 and M = 128
  GEMM paths.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import mla_oracle as om
import mla_gb300 as m
from mla_testlib import (bits_to_cuda, cuda_to_f64, cuda_weights, oracle_weights, parity, parity_cache,
                         parity_out)
from test_parity_small import make_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def FOLD(gpu_available):
    import torch
    W = m.make_weights(cuda_weights(0))
    wf = torch.empty((7168, 64 * 512), dtype=torch.bfloat16, device="cuda")
    m.mla_fold_wuv_into_wo(W, wf, m.alloc_workspace(m.MODE_FOLD, 1, 1))
    torch.cuda.synchronize()
    return W, wf


def test_fold_rows(FOLD):
    _, wf = FOLD
    wo = oracle_weights(0)
    rows = [0, 1, 127, 128, 3583, 7040, 7167]
    w_rows = dict(wo)
    w_rows["w_o"] = wo["w_o"][rows]
    ref = om.fold_wuv_into_wo(w_rows, dataclasses.replace(om.KIMI_K2, d=len(rows)))
    parity_cache(cuda_to_f64(wf[rows]), ref, "W_fold rows")


@pytest.mark.parametrize("B,P", [(3, 37), (2, 0), (100, 129), (130, 20)])
def test_decode_latent_folded_parity(FOLD, B, P):
    """B = 130 takes the front end for more than 128 rows (the q_b TMA-store
    epilogue and the separate q^pe copy) and the folded product's M > 128
    tiles over K = 32768."""
    import torch
    W, wf = FOLD
    cap = P + 3
    Wt = (cuda_weights(0), None, oracle_weights(0))
    (_, _, Cb, Rb), (_, _, C64, R64) = make_caches(Wt, B, P, cap)
    xb = synth.tensor_bits(0, "new_x", (B, 7168), synth.X_DIST)
    x = bits_to_cuda(xb)
    ckv, kpe = bits_to_cuda(Cb), bits_to_cuda(Rb)
    out = torch.empty_like(x)
    delta = torch.empty((B, 7168), dtype=torch.float32, device="cuda")
    wsp = m.alloc_workspace(m.MODE_DECODE_LATENT, B, P)
    m.mla_decode_latent_folded(W, wf, x, P, ckv, kpe, out, wsp, m.make_params(delta_out=delta))
    torch.cuda.synchronize()
    assert m.mla_device_status(wsp) == 0
    ref = om.decode_latent(oracle_weights(0), synth.bf16_bits_to_f64(xb), C64, R64)
    parity(cuda_to_f64(delta), ref["delta"], "delta")
    parity_out(cuda_to_f64(out), ref["out"], "out")
    parity_cache(cuda_to_f64(ckv[:, P]), ref["ckv_new"], "new latent row")
