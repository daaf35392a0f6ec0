"""Single kernels of the library on the GPU: the tcgen05 GEMM (both B
layouts, ragged M), the tensor-memory accumulator layout, and the bounded
device wait that reports a timeout instead of hanging."""
import numpy as np
import pytest

import mla_hooks as m

pytestmark = pytest.mark.gpu


def _rand_bf16(shape, seed, scale=1.0):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (64, 192, 512), (200, 384, 1536), (300, 2112, 7168),
                                   (129, 256, 128), (1000, 128, 64)])
def test_gemm_k_major(gpu_available, M, N, K):
    import torch
    A = _rand_bf16((M, K), 1)
    B = _rand_bf16((N, K), 2)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    m.mla_debug_gemm(A.cuda(), B.cuda(), C)
    ref = A.double() @ B.double().T
    got = C.double().cpu()
    err = (got - ref).abs().max().item()
    assert err <= 1e-2 * ref.abs().max().item() + 1e-3, f"max err {err}"


@pytest.mark.parametrize("M,N,K", [(64, 512, 128), (130, 256, 512), (7, 128, 64)])
def test_gemm_mn_major_b(gpu_available, M, N, K):
    import torch
    A = _rand_bf16((M, K), 3)
    Bt = _rand_bf16((K, N), 4)          # [K, N], N contiguous
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    m.mla_debug_gemm(A.cuda(), Bt.cuda(), C, b_mn_major=True)
    ref = A.double() @ Bt.double()
    got = C.double().cpu()
    err = (got - ref).abs().max().item()
    assert err <= 1e-2 * ref.abs().max().item() + 1e-3, f"max err {err}"


def test_tmem_layout_m128(gpu_available):
    import torch
    out = torch.full((128, 64), -1.0, device="cuda")
    m.mla_debug_umma_probe(out, 128)
    torch.cuda.synchronize()
    r = torch.arange(128).double()[:, None]
    n = torch.arange(64).double()[None, :]
    assert torch.equal(out.double().cpu(), r + 1 + 128 * n)


def test_tmem_layout_m64(gpu_available):
    """Where an M = 64 accumulator lives: row r is expected in lane
    32 * (r // 16) + r % 16 (16 lanes of each 32-lane quarter)."""
    import torch
    out = torch.full((128, 64), -1.0, device="cuda")
    m.mla_debug_umma_probe(out, 64)
    torch.cuda.synchronize()
    o = out.double().cpu().numpy()
    found = {}
    for lane in range(128):
        v = o[lane, 0]
        if float(v).is_integer() and 1 <= v <= 64 and np.allclose(o[lane], v + 128 * np.arange(64)):
            found[int(v) - 1] = lane
    expect = {r: 32 * (r // 16) + r % 16 for r in range(64)}
    assert found == expect, f"row -> lane map {found}"


def test_bounded_wait_reports_timeout(gpu_available):
    import torch
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mla_debug_wait_timeout(word, 20_000_000)   # 20 ms
    torch.cuda.synchronize()
    assert int(word.item()) & 1 == 1
    # the context is still usable
    assert float(torch.ones(1024, device="cuda").sum().item()) == 1024.0
