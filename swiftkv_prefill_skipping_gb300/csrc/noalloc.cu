// swiftkv_gemm_skinny_noalloc: the skinny split-K GEMM (C = A * B^T for at most 64
// rows) for callers that are not allowed to allocate device memory.
//
// Who needs it: a host program that hands this library no allocator and reserves the
// GPU's memory for itself (a serving engine that claims almost all of HBM for its KV
// cache at start-up), or one that cannot accept the device-wide synchronisation that
// cudaFree performs in the middle of its pipeline. The regular entry points size their
// workspace with cudaMalloc; this one takes its split-K scratch from a fixed array that
// is part of the library image instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes (8 MiB). Every GPU that
// loads the library holds one copy until the process exits. Host code cannot use the
// array's name as a device address, so the first call on each device looks the address
// up with cudaGetSymbolAddress (with that device current) and caches it.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "swiftkv.h"

namespace {

constexpr size_t kScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_skinny_scratch[kScratchBytes / sizeof(float)];

std::mutex g_setup_mu;
float* g_scratch_addr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Once per device, with that device current: the device address of the scratch array.
int scratch_for_device(int dev, float** addr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return skv::set_error(SWIFTKV_EUNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_skinny_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      return skv::set_error(SWIFTKV_ECUDA, msg);
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return skv::set_error(SWIFTKV_ECUDA, cudaGetErrorString(e));
    g_num_sms[dev] = n;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *addr = g_scratch_addr[dev];
  *sms = g_num_sms[dev];
  return SWIFTKV_OK;
}

}  // namespace

extern "C" int swiftkv_gemm_skinny_noalloc(const void* A, const void* B, float* C, int M, int N, int K,
                                           swiftkv_stream stream) {
  if (!A || !B || !C) return skv::set_error(SWIFTKV_EINVAL, "null matrix pointer");
  if (M < 1 || M > 64 || N < 1 || K < 1) return skv::set_error(SWIFTKV_EINVAL, "need 1 <= M <= 64, N >= 1, K >= 1");
  if (K % 64 || N % 128) return skv::set_error(SWIFTKV_EUNSUPPORTED, "need K % 64 == 0 and N % 128 == 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return skv::set_error(SWIFTKV_ECUDA, cudaGetErrorString(e));
  float* scratch = nullptr;
  int sms = 0;
  int r = scratch_for_device(dev, &scratch, &sms);
  if (r != SWIFTKV_OK) return r;
  const size_t need = skv::skinny_scratch_bytes(M, N, K, sms);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg, "M=%d N=%d K=%d needs %zu bytes of split-K scratch; the fixed buffer holds %zu", M, N,
             K, need, kScratchBytes);
    return skv::set_error(SWIFTKV_EUNSUPPORTED, msg);
  }
  // Nothing in the scratch has to start at zero: each split writes every partial the
  // reduction then reads, within this call.
  skv::EpiParams ep;
  memset(&ep, 0, sizeof ep);
  ep.kind = skv::EPI_STORE_F32;
  ep.M = M;
  ep.N = N;
  ep.ldo = N;
  ep.out_f32 = C;
  e = skv::launch_gemm_skinny(static_cast<const skv::bf16*>(A), K, static_cast<const skv::bf16*>(B), K, ep, scratch,
                              sms, (cudaStream_t)stream);
  if (e != cudaSuccess) return skv::set_error(SWIFTKV_ECUDA, cudaGetErrorString(e));
  return SWIFTKV_OK;
}
