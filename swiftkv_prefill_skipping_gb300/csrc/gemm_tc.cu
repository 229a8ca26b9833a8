// Blackwell (sm_103a) tensor-core GEMM: tcgen05.mma with the accumulator in
// tensor memory (TMEM), operands staged by TMA, warp-specialised and persistent.
//
//   C[M][N] = A[M][K] * B[N][K]^T  (bf16 in, fp32 accumulate), epilogue from common.cuh
//
// CTA = 6 warps, one CTA per SM (192 KB shared memory):
//   warp 0     TMA producer: 4-stage ring of (A 128x64, B 256x64) bf16 tiles, 128B swizzle
//   warp 1     allocates 512 TMEM columns; one lane issues tcgen05.mma (M=128, N=256, K=16)
//              into one of two 256-column fp32 accumulators, and tcgen05.commit frees
//              ring stages / publishes a finished accumulator
//   warps 2-5  epilogue: tcgen05.ld 32 rows x 32 columns per warp, fused epilogue, 16-byte
//              stores; the accumulator is released as soon as it has been read, so the
//              epilogue of tile i overlaps the main loop of tile i+1
// Tiles are visited in groups of m-tiles (see tile_coords) for L2 reuse.
//
// Every mbarrier wait is bounded (2 s of %globaltimer). On a timeout the CTA raises
// kStatusTimeout in the status word, stops issuing work, waits (bounded) for its own
// TMA copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;             // two accumulators

struct Ctrl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], fin;
  uint32_t tmem_base;
  int abort;
  int pending[STAGES];
};
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + (int)sizeof(Ctrl);

// kind::f16 instruction descriptor: D fp32, A/B bf16, both K-major, N = BN, M = BM.
constexpr uint32_t IDESC = tc::make_idesc(BM, BN, false, false);

// Tile order: groups of GROUP_M m-tiles; inside a group the m index runs fastest, then n.
// The CTAs running at any moment then share one activation panel (GROUP_M x 128 rows,
// 16 MB at K = 4096) that stays resident in L2 while the group sweeps every weight tile.
constexpr int GROUP_M = 16;

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int& mt, int& nt) {
  const int per_group = GROUP_M * n_tiles;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gm = min(GROUP_M, m_tiles - g * GROUP_M);
  mt = g * GROUP_M + r % gm;
  nt = r / gm;
}

__global__ void __launch_bounds__(THREADS, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB,
                                                             EpiParams ep, int K, int* status) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + STAGES * STAGE_BYTES);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = ep.M, N = ep.N;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = (N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kblocks = K / BK;
  volatile int* abort_flag = &ctl->abort;

  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto tfull = [&](int a) { return smem_u32(&ctl->tfull[a]); };
  auto tempty = [&](int a) { return smem_u32(&ctl->tempty[a]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      ctl->pending[s] = -1;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 128);
    }
    mbar_init(smem_u32(&ctl->fin), 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, m_tiles, n_tiles, mt, nt);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1, abort_flag)) break;
          mbar_expect_tx(full(stage), STAGE_BYTES);
          ctl->pending[stage] = (int)phase;
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          tma_load_2d(sa, &tmA, kb * BK, mt * BM, full(stage));
          tma_load_2d(sa + A_BYTES, &tmB, kb * BK, nt * BN, full(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(tempty(acc), aph ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          ctl->pending[stage] = -1;
          tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma(d, sdesc(sa + kk * 32), sdesc(sa + A_BYTES + kk * 32), IDESC, (kb | kk) != 0);
          tc_commit(empty(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
      }
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = pair_half(ep);
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int mt, nt;
      tile_coords(t, m_tiles, n_tiles, mt, nt);
      if (!mbar_wait(tfull(acc), aph, abort_flag)) break;
      tc_fence_after();
      const int row = mt * BM + q * 32 + lane;
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      for (int b0 = 0; b0 < BN; b0 += 2 * half) {
        const int ncol = nt * BN + b0;
        if (ncol >= N) break;
        for (int c = 0; c < half; c += 32) {
          float lo[32], hi[32];
          tmem_ld32(tb + b0 + c, lo);
          tmem_ld32(tb + b0 + half + c, hi);
          if (row < M) apply_chunk32(ep, row, ncol + c, ncol + half + c, lo, hi);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty(acc));
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(status, kStatusTimeout);
      for (int s = 0; s < STAGES; ++s) {  // TMA copies still in flight into this CTA's ring
        const int ph = ctl->pending[s];
        if (ph < 0) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(full(s), (uint32_t)ph) && global_ns() - t0 < kTimeoutNs) {
        }
      }
    }
    if (threadIdx.x == 32) {  // MMAs this thread issued
      tc_commit(smem_u32(&ctl->fin));
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(smem_u32(&ctl->fin), 0) && global_ns() - t0 < kTimeoutNs) {
      }
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace

cudaError_t launch_gemm_tc(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep, int num_sms,
                           int* status, cudaStream_t stream) {
  if (ep.M < 1 || ep.N < 1 || K < BK || K % BK || ep.N % 128 || lda % 8 ||
      (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))
    return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!tma_map_bf16_2d(&ta, A, ep.M, K, lda, BK, BM, true) || !tma_map_bf16_2d(&tb, B, ep.N, K, K, BK, BN, true))
    return cudaErrorNotSupported;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int tiles = ((ep.M + BM - 1) / BM) * ((ep.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, ep, K, status);
  return cudaGetLastError();
}

}  // namespace skv
