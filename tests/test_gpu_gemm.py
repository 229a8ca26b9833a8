"""GEMM kernel families (tcgen05/TMEM, mma.sync tiles, skinny split-K) against a
plain PyTorch fp32 matmul of the same bf16 operands, through the C ABI."""
import ctypes as C

import pytest

pytestmark = pytest.mark.gpu

SHAPES = [
    (128, 256, 64),      # one tile, one k-block
    (300, 512, 256),     # ragged M
    (1000, 384, 640),    # ragged last 256-column tile
    (37, 1024, 512),     # M below one tile
    (2048, 4096, 4096),  # many tiles per CTA (persistent loop, both accumulators)
]


def _run(impl, M, N, K, seed=0):
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    Bm = (torch.randn(N, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    Cm = torch.full((M, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = B.lib().swiftkv_gemm_bf16(A.data_ptr(), Bm.data_ptr(), Cm.data_ptr(), M, N, K, impl, st.data_ptr(),
                                   C.c_void_p(torch.cuda.current_stream().cuda_stream))
    B.check(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    torch.backends.cuda.matmul.allow_tf32 = False
    ref = A.float() @ Bm.float().T
    return Cm, ref


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("impl", [0, 1, 3, 4])
def test_gemm_matches_torch_fp32(impl, M, N, K):
    import torch
    Cm, ref = _run(impl, M, N, K)
    assert not torch.isnan(Cm).any()
    err = (Cm - ref).abs().max().item() / ref.abs().max().item()
    assert err < 2e-5, (impl, M, N, K, err)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 1024, 512), (64, 128, 14336)])
def test_skinny_gemm_matches_torch_fp32(M, N, K):
    import torch
    Cm, ref = _run(2, M, N, K)
    assert not torch.isnan(Cm).any()
    err = (Cm - ref).abs().max().item() / ref.abs().max().item()
    assert err < 2e-5, (M, N, K, err)


def test_tcgen05_is_deterministic():
    import torch
    c1, _ = _run(0, 777, 1024, 1024, seed=3)
    c2, _ = _run(0, 777, 1024, 1024, seed=3)
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 1024, 512), (64, 128, 14336), (37, 2048, 704),
                                   (48, 128256, 256)])
def test_gemv_matches_torch_fp32(M, N, K):
    import torch
    Cm, ref = _run(5, M, N, K)
    assert not torch.isnan(Cm).any()
    err = (Cm - ref).abs().max().item() / ref.abs().max().item()
    assert err < 2e-5, (M, N, K, err)
