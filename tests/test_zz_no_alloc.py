"""mla_decode_noalloc, the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory (a host framework that
owns all device memory, a fixed memory budget, loops that cannot afford an
allocation's synchronisation): its scratch is a fixed static device array in
the library instead of a workspace argument.  Checked here through the C ABI
against mla_decode with a caller workspace, on the same inputs, for two calls
in a row (different shapes, so the second call runs on the array the first
one left behind).  The two entry points run the same kernels in the same
configuration (split-K and split-KV merges in a fixed order), so the
results must be identical bit for bit: a stale value left in the shared
array by the previous call would show.  This file is collected last on
purpose.
"""
import numpy as np
import pytest

import synth
import mla_gb300 as m
from mla_testlib import cuda_to_f64, cuda_weights, parity

pytestmark = pytest.mark.gpu


def _inputs(B, P, cap, seed):
    import torch
    x = synth.tensor_cuda(seed, "new_x", (B, 7168), synth.X_DIST)
    # cached positions 0..P-1: distribution-matched seeded values (both calls see the same bits)
    k = synth.tensor_cuda(seed, "cache_x", (B, 64, cap, 192), (0.0, 1.0))
    v = synth.tensor_cuda(seed + 1, "cache_x", (B, 64, cap, 128), (0.0, 0.5))
    return x, k, v


def test_decode_noalloc_matches_decode_two_calls(gpu_available):
    import torch
    wt = cuda_weights(0)
    W = m.make_weights(wt)
    for (B, P, seed) in [(3, 37, 5), (2, 300, 6)]:
        cap = P + 2
        x, k, v = _inputs(B, P, cap, seed)
        k1, v1, k2, v2 = k.clone(), v.clone(), k.clone(), v.clone()
        ref_out = torch.empty_like(x)
        ws = m.alloc_workspace(m.MODE_DECODE, B, P)
        m.mla_decode(W, x, P, k1, v1, ref_out, ws)
        out = torch.empty_like(x)
        m.mla_decode_noalloc(W, x, P, k2, v2, out)
        torch.cuda.synchronize()
        parity(cuda_to_f64(out), cuda_to_f64(ref_out), f"out B={B} P={P}")
        assert torch.equal(out, ref_out), f"out B={B} P={P} differs from mla_decode"
        assert torch.equal(k2, k1) and torch.equal(v2, v1), f"caches B={B} P={P} differ from mla_decode"


def test_decode_noalloc_rejects_oversized_batch(gpu_available):
    import torch
    wt = cuda_weights(0)
    W = m.make_weights(wt)
    B, P = 600, 4   # needs more scratch than the fixed array holds (limit: 455 sequences)
    x = torch.zeros((B, 7168), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, 64, P + 1, 192), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((B, 64, P + 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MlaError) as e:
        m.mla_decode_noalloc(W, x, P, k, v, torch.empty_like(x))
    assert e.value.status == -3
