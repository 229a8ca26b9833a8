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

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
static_assert(BN == kNormTile, "fused RMSNorm sums of squares are kept per 256-column GEMM tile");
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

// FP8 cache, one K or V head (2 * H columns from TMEM column tcol) of row `row`: bias and RoPE,
// the bf16 values the cache would hold, their max, then codes, scale and expansion. The TMEM
// loads are warp-collective, so every lane runs them whether or not its row exists.
template <int H>
__device__ __forceinline__ void fp8_head_epilogue(const EpiParams& ep, int row, int M, int ncol, uint32_t tcol) {
  uint32_t pk[H];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < H; c += 32) {
    float lo[32], hi[32];
    tmem_ld32(tcol + c, lo);
    tmem_ld32(tcol + H + c, hi);
    if (row < M) kv_chunk_prep(ep, row, ncol + c, ncol + H + c, lo, hi);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const uint32_t pl = pack_bf16_(lo[i], lo[i + 1]), ph = pack_bf16_(hi[i], hi[i + 1]);
      pk[(c + i) >> 1] = pl;
      pk[(H + c + i) >> 1] = ph;
      amax = fmaxf(fmaxf(amax, fabsf(__uint_as_float(pl << 16))), fabsf(__uint_as_float(pl & 0xffff0000u)));
      amax = fmaxf(fmaxf(amax, fabsf(__uint_as_float(ph << 16))), fabsf(__uint_as_float(ph & 0xffff0000u)));
    }
  }
  if (row < M) store_head_fp8<2 * H>(ep, row, ncol, pk, amax);
}

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
  const int num_units = m_tiles * n_tiles;
  const int first_unit = blockIdx.x, unit_stride = gridDim.x;
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
      for (int u = first_unit; u < num_units && !*abort_flag; u += unit_stride) {
        int mt, nt;
        tile_coords(u, m_tiles, n_tiles, mt, nt);
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
      for (int u = first_unit; u < num_units && !*abort_flag; u += unit_stride, ++it) {
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
    for (int u = first_unit; u < num_units; u += unit_stride, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int mt, nt;
      tile_coords(u, m_tiles, n_tiles, mt, nt);
      if (!mbar_wait(tfull(acc), aph, abort_flag)) break;
      tc_fence_after();
      const int row = mt * BM + q * 32 + lane;
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      const float rs = (ep.norm_part && row < M) ? fused_norm_scale(ep, row) : 1.f;
      float ssq = 0.f;  // fused RMSNorm: the row's sum of squares over this 256-column tile
      for (int b0 = 0; b0 < BN; b0 += 2 * half) {
        const int ncol = nt * BN + b0;
        if (ncol >= N) break;
        if (fp8_head_block(ep, ncol)) {  // one K or V head of an FP8 cache
          if (half == 64) fp8_head_epilogue<64>(ep, row, M, ncol, tb + b0);
          else fp8_head_epilogue<32>(ep, row, M, ncol, tb + b0);
          continue;
        }
        for (int c = 0; c < half; c += 32) {
          float lo[32], hi[32];
          tmem_ld32(tb + b0 + c, lo);
          tmem_ld32(tb + b0 + half + c, hi);
          if (ep.norm_part) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              lo[i] *= rs;
              hi[i] *= rs;
            }
          }
          if (row < M) ssq += apply_chunk32(ep, row, ncol + c, ncol + half + c, lo, hi);
        }
      }
      if (ep.ss_out && row < M) ep.ss_out[(size_t)row * norm_tiles(N) + nt] = ssq;
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


// ---------------------------------------------------------------------------- CTA pairs
//
// 2-SM variant: a cluster of two CTAs computes a 256 x 256 tile with tcgen05.mma.cta_group::2
// (M = 256, N = 256). CTA r stages rows r*128.. of the A tile and rows r*128.. of the B tile
// (32 KB per stage instead of 48 KB), so each SM writes 64 B/clk into shared memory and the
// tensor core reads 64 B/clk from it: together within shared-memory bandwidth, where the
// 1-SM 128 x 256 tile needs ~192 B/clk. The even CTA issues the MMAs; both CTAs' TMA loads
// complete on its ring barriers; each of its commits arrives on the barrier of both CTAs; each CTA reads
// its own 128 accumulator rows from its own TMEM and releases them on the even CTA's barrier.
constexpr int P_STAGES = 6;
constexpr int P_STAGE_BYTES = 2 * BM * BK * 2;  // A half 16 KB + B half 16 KB
struct CtrlPair {
  uint64_t full[P_STAGES], empty[P_STAGES], tfull[2], tempty[2], fin;
  uint32_t tmem_base;
  int abort;
  int pending[P_STAGES];
};
constexpr int P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + (int)sizeof(CtrlPair);
constexpr uint32_t IDESC_PAIR = tc::make_idesc(2 * BM, BN, false, false);

// Unit order of the 2-SM kernel, `order` = group << 1 | by_n. by_n = 0: groups of `group`
// 256-row units, the row index running fastest, each group sweeping every weight tile while
// its activation panels stay in L2. by_n = 1: groups of `group` weight tiles, the weight index
// running fastest, each group sweeping every 256-row unit while its weight panels stay in L2.
__device__ __forceinline__ void unit_coords(int u, int m_units, int n_tiles, int order, int& mu, int& nt) {
  const int group = order >> 1;
  if (!(order & 1)) {
    const int per = group * n_tiles, g = u / per, r = u - g * per;
    const int gm = min(group, m_units - g * group);
    mu = g * group + r % gm;
    nt = r / gm;
  } else {
    const int per = group * m_units, g = u / per, r = u - g * per;
    const int gn = min(group, n_tiles - g * group);
    nt = g * group + r % gn;
    mu = r / gn;
  }
}

// Unit order per GEMM shape, chosen from DRAM traffic measured (ncu, one layer of the
// Llama-3.1-8B shape, 11 703 rows) over group kinds and sizes: reads per launch went from
// 455 to 356 MB for O (N = 4096) and from 2 246 to 1 666 MB for down (K = 14 336); row groups
// of 16 stayed best for QKV and gate/up, where larger and smaller groups both read more.
//   K > 8192 (panels over 4 MB): groups of 8 weight tiles, activation panels swept per group;
//   otherwise, at most 16 weight tiles: one group of all of them;
//   otherwise: groups of 256-row units holding 32 MiB of activation panels (16 at K = 4096,
//   between 4 and 16).
static int pair_order(int m_units, int n_tiles, int K) {
  if (K > 8192) return (std::min(8, n_tiles) << 1) | 1;
  if (n_tiles <= 16) return (n_tiles << 1) | 1;
  const int g = std::min(16, std::max(4, (32 << 20) / (512 * K)));
  return std::min(g, m_units) << 1;
}

__global__ void __launch_bounds__(THREADS, 1) gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                  const __grid_constant__ CUtensorMap tmB,
                                                                  EpiParams ep, int K, int order, int* status) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  CtrlPair* ctl = reinterpret_cast<CtrlPair*>(smem + P_STAGES * P_STAGE_BYTES);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = ep.M, N = ep.N;
  const int m_tiles = (M + BM - 1) / BM;
  const int n_tiles = (N + BN - 1) / BN;
  const int m_units = (m_tiles + 1) / 2;
  const int num_units = m_units * n_tiles;
  const int kblocks = K / BK;
  const int crank = (int)cluster_ctarank();
  const bool leader = crank == 0;
  const int first_unit = blockIdx.x / 2, unit_stride = gridDim.x / 2;
  volatile int* abort_flag = &ctl->abort;

  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto tfull = [&](int a) { return smem_u32(&ctl->tfull[a]); };
  auto tempty = [&](int a) { return smem_u32(&ctl->tempty[a]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      ctl->pending[s] = -1;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 256);
    }
    mbar_init(smem_u32(&ctl->fin), 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA of the pair allocates collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int u = first_unit; u < num_units && !*abort_flag; u += unit_stride) {
        int mu, nt;
        unit_coords(u, m_units, n_tiles, order, mu, nt);
        const int mt = mu * 2 + crank;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1, abort_flag)) break;
          const uint32_t fb = mapa_shared(full(stage), 0);
          if (leader) {
            mbar_expect_tx(full(stage), 2 * P_STAGE_BYTES);
            ctl->pending[stage] = (int)phase;
          }
          const uint32_t sa = sbase + stage * P_STAGE_BYTES;
          tma_load_2d_pair(sa, &tmA, kb * BK, mt * BM, fb);
          tma_load_2d_pair(sa + BM * BK * 2, &tmB, kb * BK, nt * BN + crank * BM, fb);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      for (int u = first_unit; u < num_units && !*abort_flag; u += unit_stride, ++it) {
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
          const uint32_t sa = sbase + stage * P_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_pair(d, sdesc(sa + kk * 32), sdesc(sa + BM * BK * 2 + kk * 32), IDESC_PAIR, (kb | kk) != 0);
          tc_commit_pair_mc(empty(stage), 0x3);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull(acc), 0x3);
      }
    }
  } else {
    const int q = warp & 3;
    const int half = pair_half(ep);
    int it = 0;
    for (int u = first_unit; u < num_units; u += unit_stride, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int mu, nt;
      unit_coords(u, m_units, n_tiles, order, mu, nt);
      const int mt = mu * 2 + crank;
      if (!mbar_wait(tfull(acc), aph, abort_flag)) break;
      tc_fence_after();
      const int row = mt * BM + q * 32 + lane;
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      const float rs = (ep.norm_part && row < M) ? fused_norm_scale(ep, row) : 1.f;
      float ssq = 0.f;  // fused RMSNorm: the row's sum of squares over this 256-column tile
      for (int b0 = 0; b0 < BN; b0 += 2 * half) {
        const int ncol = nt * BN + b0;
        if (ncol >= N) break;
        if (fp8_head_block(ep, ncol)) {  // one K or V head of an FP8 cache
          if (half == 64) fp8_head_epilogue<64>(ep, row, M, ncol, tb + b0);
          else fp8_head_epilogue<32>(ep, row, M, ncol, tb + b0);
          continue;
        }
        for (int c = 0; c < half; c += 32) {
          float lo[32], hi[32];
          tmem_ld32(tb + b0 + c, lo);
          tmem_ld32(tb + b0 + half + c, hi);
          if (ep.norm_part) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              lo[i] *= rs;
              hi[i] *= rs;
            }
          }
          if (row < M) ssq += apply_chunk32(ep, row, ncol + c, ncol + half + c, lo, hi);
        }
      }
      if (ep.ss_out && row < M) ep.ss_out[(size_t)row * norm_tiles(N) + nt] = ssq;
      tc_fence_before();
      mbar_arrive_cluster(mapa_shared(tempty(acc), 0));
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(status, kStatusTimeout);
      for (int s = 0; s < P_STAGES; ++s) {
        const int ph = ctl->pending[s];
        if (ph < 0) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(full(s), (uint32_t)ph) && global_ns() - t0 < kTimeoutNs) {
        }
      }
    }
    if (threadIdx.x == 32 && leader) {
      tc_commit_pair_mc(smem_u32(&ctl->fin), 0x3);
    }
    if (threadIdx.x == 32) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(smem_u32(&ctl->fin), 0) && global_ns() - t0 < kTimeoutNs) {
      }
    }
    __syncthreads();
  }
  cluster_sync();  // the leader's MMAs into both CTAs' TMEM are done before either frees it
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  cluster_sync();
}

}  // namespace

static cudaError_t launch_tc_single(const CUtensorMap& ta, const CUtensorMap& tb, const EpiParams& ep, int K,
                                    int num_sms, int* status, cudaStream_t stream) {
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tc_kernel), SMEM_BYTES, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const int units = ((ep.M + BM - 1) / BM) * ((ep.N + BN - 1) / BN);
  gemm_tc_kernel<<<units < num_sms ? units : num_sms, THREADS, SMEM_BYTES, stream>>>(ta, tb, ep, K, status);
  return cudaSuccess;
}

static cudaError_t launch_tc_pair(const CUtensorMap& ta, const CUtensorMap& tb, const EpiParams& ep, int K,
                                  int num_sms, int* status, cudaStream_t stream) {
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tc_pair_kernel), P_SMEM_BYTES, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const int m_units = ((ep.M + BM - 1) / BM + 1) / 2;
  const int n_tiles = (ep.N + BN - 1) / BN;
  const int units = m_units * n_tiles;
  const int order = pair_order(m_units, n_tiles, K);
  const int clusters = units < num_sms / 2 ? units : num_sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * 2);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel, ta, tb, ep, K, order, status);
}

cudaError_t launch_gemm_tc(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep, int num_sms,
                           int* status, cudaStream_t stream, int mode) {
  if (ep.M < 1 || ep.N < 1 || K < BK || K % BK || ep.N % 128 || lda % 8 ||
      (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))
    return cudaErrorNotSupported;
  if (mode != 0 && mode != 2) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  const int b_rows = mode == 0 ? BN : BN / 2;
  if (!tma_map_bf16_2d(&ta, A, ep.M, K, lda, BK, BM, true) || !tma_map_bf16_2d(&tb, B, ep.N, K, K, BK, b_rows, true))
    return cudaErrorNotSupported;
  cudaError_t e;
  if (mode == 2) e = launch_tc_pair(ta, tb, ep, K, num_sms, status, stream);
  else e = launch_tc_single(ta, tb, ep, K, num_sms, status, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace skv
