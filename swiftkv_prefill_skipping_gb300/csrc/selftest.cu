// swiftkv_selftest_wait_timeout: exercises, on purpose and safely, the expiry path of the
// bounded mbarrier waits that every tcgen05 kernel of the library relies on.
//
// One CTA of three warps takes the shape of those kernels' abort protocol:
//   warp 1  allocates TMEM (as the GEMM and attention kernels do) and frees it at the end;
//   warp 0  the consumer: waits on the `full` barrier, whose producer issues nothing, with
//           the wait bounded by limit_ns of %globaltimer; when the limit passes it sets the
//           CTA's abort flag and records how long it waited;
//   warp 2  a second waiter (on `empty`, which only the consumer would have released): it
//           leaves its wait as soon as it sees the abort flag, without a limit of its own
//           expiring.
// Thread 0 then raises kStatusTimeout in the status word, TMEM is freed and the kernel
// returns. Nothing is left in flight: no TMA copy or MMA was issued.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "swiftkv.h"
#include "tc_common.cuh"

namespace skv {
namespace {

using namespace tc;

struct SelfTestCtrl {
  uint64_t full, empty;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(96, 1) wait_timeout_kernel(int* status, unsigned long long* elapsed_ns,
                                                             unsigned long long limit_ns) {
  __shared__ SelfTestCtrl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctl.abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl.full), 1);
    mbar_init(smem_u32(&ctl.empty), 1);
    ctl.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl.tmem_base)),
                 "r"(32)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0 && lane == 0) {
    const uint64_t t0 = global_ns();
    const bool ok = mbar_wait_for(smem_u32(&ctl.full), 0, abort_flag, limit_ns);
    if (elapsed_ns) *elapsed_ns = ok ? 0ull : (unsigned long long)(global_ns() - t0);
  } else if (warp == 2 && lane == 0) {
    // the phase this waits for never completes; only the consumer's abort ends the wait (the
    // 2 s library limit is far beyond any limit_ns this entry accepts)
    mbar_wait(smem_u32(&ctl.empty), 0, abort_flag);
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(status, kStatusTimeout);
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32) : "memory");
}

}  // namespace
}  // namespace skv

extern "C" int swiftkv_selftest_wait_timeout(int* status, unsigned long long* elapsed_ns, long long limit_ns,
                                             swiftkv_stream stream) {
  if (!status) return skv::set_error(SWIFTKV_EINVAL, "status is NULL");
  if (limit_ns < 1000 || limit_ns > 100000000)
    return skv::set_error(SWIFTKV_EINVAL, "limit_ns outside [1e3, 1e8]");
  skv::wait_timeout_kernel<<<1, 96, 0, (cudaStream_t)stream>>>(status, elapsed_ns, (unsigned long long)limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return skv::set_error(SWIFTKV_ECUDA, cudaGetErrorString(e));
  return SWIFTKV_OK;
}
