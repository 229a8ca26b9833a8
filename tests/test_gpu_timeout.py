"""The expiry path of the library's bounded waits, run on purpose without a fault.

Every mbarrier wait in the tcgen05 kernels gives up after a limit, raises
SWIFTKV_STATUS_TIMEOUT, drains its own work in flight, frees TMEM and returns. The
self-test entry runs that path with a short limit and a producer that issues nothing;
the status bit must be set, the wait must have lasted at least the limit and far less
than the library's 2 s ceiling, and the next ordinary calls on the same context must
succeed with a clean status."""
import ctypes as C

import numpy as np
import pytest

import synth
from gpu_helpers import LOGIT_ABS_TOL, oracle_prefill, run_gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_bounded_wait_expires_and_the_context_stays_usable(limit_ns):
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    lib = B.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    B.check(lib.swiftkv_selftest_wait_timeout(status.data_ptr(), elapsed.data_ptr(), limit_ns, stream))
    torch.cuda.synchronize()
    assert int(status.item()) == B.STATUS_TIMEOUT
    waited = int(elapsed.item())
    assert limit_ns <= waited < 500_000_000, waited

    # the same context runs an ordinary GEMM and a SwiftKV prefill afterwards
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = (torch.randn(256, 512, device="cuda") * 0.5).to(torch.bfloat16)
    w = (torch.randn(384, 512, device="cuda") * 0.5).to(torch.bfloat16)
    out = torch.empty(256, 384, device="cuda")
    B.check(lib.swiftkv_gemm_bf16(a.data_ptr(), w.data_ptr(), out.data_ptr(), 256, 384, 512, 4, st.data_ptr(),
                                  stream))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert float((out - a.float() @ w.float().T).abs().max()) < 1e-2

    batch = synth.prompt_batch(synth.TINY.vocab, 2, 0, 0, lens=[40, 90])
    m, kv, logits = run_gpu_prefill(synth.TINY, 2, 1, batch)
    assert m.status() == 0
    _, _, ref, _ = oracle_prefill(synth.TINY, 2, 1, batch)
    assert float(np.abs(logits.cpu().numpy() - np.stack(ref)).max()) <= LOGIT_ABS_TOL
    m.free()


def test_selftest_rejects_limits_outside_range():
    import torch
    from swiftkv_prefill_skipping_gb300 import binding as B
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, 999, 200_000_000):
        assert B.lib().swiftkv_selftest_wait_timeout(status.data_ptr(), None, bad, None) == -1
    assert B.lib().swiftkv_selftest_wait_timeout(None, None, 1_000_000, None) == -1
    assert int(status.item()) == 0
