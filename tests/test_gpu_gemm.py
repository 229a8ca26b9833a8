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
@pytest.mark.parametrize("impl", [0, 1, 4])
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


@pytest.mark.parametrize("M,N,K", [(24, 5120, 5120), (24, 5120, 13824), (16, 4096, 4096), (16, 8192, 1024),
                                   (64, 5120, 512), (1, 5120, 256)])
def test_residual_skinny_gemm_adds_the_impl6_product(M, N, K):
    """impl 7 (C += A B^T, the decode rows' O and down epilogue) runs impl 6's kernel and
    tiles with the residual epilogue: every column is accumulated over K in the same order,
    so the result equals C0 plus impl 6's product bit for bit, and matches the fp32
    reference. 64-row and 32-row weight tiles, M from 1 to 64."""
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    C0 = torch.randn(M, N, device="cuda", generator=g)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    prod = torch.full((M, N), float("nan"), device="cuda")
    B.check(B.lib().swiftkv_gemm_bf16(A.data_ptr(), W.data_ptr(), prod.data_ptr(), M, N, K, 6, st.data_ptr(), stream))
    acc = C0.clone()
    B.check(B.lib().swiftkv_gemm_bf16(A.data_ptr(), W.data_ptr(), acc.data_ptr(), M, N, K, 7, st.data_ptr(), stream))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(acc, C0 + prod)
    torch.backends.cuda.matmul.allow_tf32 = False
    ref = A.float() @ W.float().T
    err = ((acc - C0) - ref).abs().max().item() / ref.abs().max().item()
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


# N / 64 >= 76 tiles (the TMA kernel's range on 152 SMs); K = 704 and 320 end inside a
# 256-deep stage (the boxes past K read zeros)
@pytest.mark.parametrize("M,N,K", [(1, 5120, 4096), (16, 9728, 512), (64, 5120, 14336), (37, 10240, 704),
                                   (48, 128256, 256), (24, 7168, 5120), (5, 4864, 320),
                                   # 32-row tiles: N / 64 below half the SMs
                                   (16, 4096, 4096), (1, 4096, 14336), (64, 4096, 704), (33, 2432, 512)])
def test_tma_gemv_matches_torch_fp32(M, N, K):
    import torch
    Cm, ref = _run(6, M, N, K)
    assert not torch.isnan(Cm).any()
    err = (Cm - ref).abs().max().item() / ref.abs().max().item()
    assert err < 2e-5, (M, N, K, err)


def test_tma_gemv_rejects_narrow_weights():
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    with pytest.raises(B.SwiftKVError) as e:
        _run(6, 16, 1024, 4096)
    assert e.value.code == -9


@pytest.mark.parametrize("N,K", [(5120, 4096), (9728, 704), (7168, 5120), (4096, 4096)])
def test_tma_gemv_rows_do_not_depend_on_batch_size(N, K):
    """A row's result is the same bits whatever M is."""
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    g = torch.Generator(device="cuda").manual_seed(7)
    A = (torch.randn(64, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for M in (1, 17, 33, 64):
        Cm = torch.empty((M, N), device="cuda")
        B.check(B.lib().swiftkv_gemm_bf16(A.data_ptr(), W.data_ptr(), Cm.data_ptr(), M, N, K, 6, st.data_ptr(),
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream)))
        outs.append(Cm[0].clone())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_skinny_kernels_on_each_visible_device():
    """Kernels that raise their shared-memory limit do it once per device: the split-K
    skinny GEMM with more than 16 rows (55-74 KB of shared memory) and the persistent tcgen05
    GEMM run on every visible GPU in turn, twice each, in one process."""
    import torch
    n = torch.cuda.device_count()
    if n < 2:
        pytest.skip("one GPU visible")
    for rnd in range(2):
        for dev in range(n):
            with torch.cuda.device(dev):
                for impl, (M, N, K) in ((2, (40, 1024, 512)), (0, (300, 512, 256))):
                    Cm, ref = _run(impl, M, N, K, seed=rnd)
                    err = (Cm - ref).abs().max().item() / ref.abs().max().item()
                    assert err < 2e-5, (dev, impl, err)


def test_tensor_core_accumulation_error_against_float64():
    """The GEMMs' rounding error against the float64 product of the same bf16 operands: far
    below one bf16 rounding of the output (2^-9 relative) at every K the models use, and
    growing no faster than linearly in K. The tensor cores accumulate in fp32 range but round
    more coarsely than IEEE float32 (rms error ~3x IEEE's at K = 640, ~80x at K = 14336), which
    the parity tests' floors account for."""
    import numpy as np
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    rms = {}
    for K in (640, 4096, 14336):
        g = torch.Generator().manual_seed(K)
        A = (torch.randn(256, K, generator=g) * 0.5).to(torch.bfloat16)
        W = (torch.randn(256, K, generator=g) * 0.02).to(torch.bfloat16)
        ref = A.double().numpy() @ W.double().numpy().T
        Ad, Wd = A.cuda(), W.cuda()
        for impl in (4, 1):
            Cm = torch.empty(256, 256, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            B.check(B.lib().swiftkv_gemm_bf16(Ad.data_ptr(), Wd.data_ptr(), Cm.data_ptr(), 256, 256, K, impl,
                                              st.data_ptr(), C.c_void_p(torch.cuda.current_stream().cuda_stream)))
            torch.cuda.synchronize()
            d = (Cm.cpu().double().numpy() - ref) / np.abs(ref).mean()
            rms[(K, impl)] = float(np.sqrt(np.mean(d * d)))
            assert float(np.abs(d).max()) < 2.0 ** -12, (K, impl, float(np.abs(d).max()))
    for impl in (4, 1):
        assert rms[(14336, impl)] < 4 * (14336 / 640) * rms[(640, impl)], rms
    print({f"K={k} impl={i}": f"{v:.2e}" for (k, i), v in sorted(rms.items())})

