"""The no-allocation skinny GEMM entry point (swiftkv_gemm_skinny_noalloc).

It exists for callers that may not allocate device memory themselves or through
this library: hosts that keep the GPU's memory in their own pools, or that cannot
take cudaFree's device-wide synchronisation mid-pipeline. It must give the same
result as the allocating entry point (swiftkv_gemm_bf16, skinny impl 2) on two calls
in a row with different shapes, since every call reuses one fixed scratch array that
still holds the previous call's partial sums. This file is collected last so that a
stop-at-first-failure run has already run every other test when it gets here.
"""
import ctypes as C

import pytest

pytestmark = pytest.mark.gpu


def _mats(M, N, K, seed):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    B = (torch.randn(N, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    return A, B


def _stream():
    import torch
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_allocating_entry_two_calls_in_a_row():
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    lib = B.lib()
    # larger first, then smaller: the second call runs over the first call's leftovers
    for (M, N, K, seed) in [(16, 4096, 4096, 1), (7, 1024, 512, 2)]:
        A, W = _mats(M, N, K, seed)
        ref = torch.full((M, N), float("nan"), device="cuda")
        got = torch.full((M, N), float("nan"), device="cuda")
        B.check(lib.swiftkv_gemm_bf16(A.data_ptr(), W.data_ptr(), ref.data_ptr(), M, N, K, 2, None, _stream()))
        B.check(lib.swiftkv_gemm_skinny_noalloc(A.data_ptr(), W.data_ptr(), got.data_ptr(), M, N, K, _stream()))
        torch.cuda.synchronize()
        assert not torch.isnan(got).any()
        err = (got - ref).abs().max().item() / ref.abs().max().item()
        assert err < 2e-5, (M, N, K, err)
        torch.backends.cuda.matmul.allow_tf32 = False
        fp32 = A.float() @ W.float().T
        assert (got - fp32).abs().max().item() / fp32.abs().max().item() < 2e-5


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    lib = B.lib()
    A, W = _mats(64, 128256, 128, 3)   # LM-head-sized N: partials exceed the fixed 8 MiB
    out = torch.zeros((64, 128256), device="cuda")
    rc = lib.swiftkv_gemm_skinny_noalloc(A.data_ptr(), W.data_ptr(), out.data_ptr(), 64, 128256, 128, _stream())
    assert rc == -9
    assert b"fixed buffer" in lib.swiftkv_last_error()
    torch.cuda.synchronize()
    assert int(out.abs().sum().item()) == 0
    assert lib.swiftkv_gemm_skinny_noalloc(A.data_ptr(), W.data_ptr(), out.data_ptr(), 65, 128, 128, _stream()) == -1
