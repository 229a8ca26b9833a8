// Skinny GEMM (M <= 64 rows: decode tokens, the SwiftKV tail, the LM head) streaming the
// weights at HBM rate: C = A * W^T with the shared epilogue.
//
// Persistent: one CTA per SM walks the weight tiles (64 rows: two 32-row strips `half`
// apart, so RoPE and SwiGLU partners (n, n + half) stay in one thread; 32-row tiles of two
// 16-row strips for weights with fewer than SMs / 2 64-row tiles) over the whole K.
// One producer thread streams, per 256-deep k step, the tile's 32 x 64 weight boxes (four
// per strip, so each weight row is read 512 contiguous bytes at a time) and the matching
// slice of A (rows past M and columns past K zero-filled) with TMA into a ring of about
// 190 KB, running ahead across tiles; four consumer warps read each stage (warp w: rows
// 8w..8w+7 of both strips) with ldmatrix and accumulate on mma.sync (bf16 in, fp32
// accumulate, k in order), then run the epilogue from registers. No scratch; a row's
// arithmetic does not depend on M. Used when the matrix has at least half as many tiles as
// there are SMs (narrower ones would leave SMs idle and take the cp.async kernel). All waits are
// bounded: on a timeout the CTA flags kStatusTimeout, drains its own copies and exits.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int GT_BK = 64;        // k per box: one 128-byte swizzle row
constexpr int GT_KSUB = 4;       // boxes along k per stage (256 k)
constexpr int GT_RING_BYTES = 192 * 1024;
constexpr int GT_MAX_STAGES = 24;

// TR: weight rows per tile (two TR/2-row strips; 64, or 32 for weights with few rows);
// TR/16 consumer warps each own 8 rows of both strips.
template <int MB, int TR>
struct Gt {
  static constexpr int CONSUMERS = TR / 16;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
  static constexpr int A_ROWS = MB * 16;
  static constexpr int WBOX = TR / 2 * GT_BK * 2;             // one (TR/2) x 64 box
  static constexpr int ABOX = A_ROWS * GT_BK * 2;
  static constexpr int W_BYTES = 2 * GT_KSUB * WBOX;           // strip-major: [strip][ksub]
  static constexpr int A_BYTES = GT_KSUB * ABOX;
  static constexpr int STAGE = W_BYTES + A_BYTES;      // a multiple of 1024
  static constexpr int STAGES = GT_RING_BYTES / STAGE < GT_MAX_STAGES ? GT_RING_BYTES / STAGE : GT_MAX_STAGES;
};

struct GtCtrl {
  uint64_t full[GT_MAX_STAGES];
  uint64_t empty[GT_MAX_STAGES];
  int pending[GT_MAX_STAGES];
  int abort;
};

constexpr int gt_smem_bytes(int stage_bytes, int stages) { return 1024 + stages * stage_bytes + (int)sizeof(GtCtrl); }

// byte offset of 16-byte chunk `ch` of row `row` in a 128B-swizzled box (rows of 128 bytes)
__device__ __forceinline__ uint32_t sw128(int row, int ch) { return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4)); }

template <int MB, int TR>
__global__ void __launch_bounds__(Gt<MB, TR>::THREADS, 1) gemv_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                 const __grid_constant__ CUtensorMap tmW, int K,
                                                                 EpiParams ep, int* status) {
  using G = Gt<MB, TR>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t ring = smem_u32(smem);
  GtCtrl* ctl = reinterpret_cast<GtCtrl*>(smem + G::STAGES * G::STAGE);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = ep.M, N = ep.N;
  const int half = pair_half(ep);
  const int strips = half / (TR / 2);
  const int tiles = N / TR;
  const int ksteps = (K + GT_BK * GT_KSUB - 1) / (GT_BK * GT_KSUB);  // stages per tile
  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto col_of = [&](int tile) { return (tile / strips) * 2 * half + (tile % strips) * (TR / 2); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), G::CONSUMERS);
      ctl->pending[s] = -1;
    }
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // Launched as a programmatic dependent of the previous kernel on the stream: the first
  // stages' weight boxes (which no earlier kernel writes) are requested before waiting for
  // that kernel; everything that reads its output (A, and the epilogue's residual rows)
  // comes after griddepcontrol.wait.
  griddep_launch_dependents();
  if (warp == G::CONSUMERS) {
    // producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      auto load_w = [&](int st, int kt, int col_lo) {
        const uint32_t sw = ring + st * G::STAGE;
#pragma unroll
        for (int q = 0; q < GT_KSUB; ++q) {
          const int x = (kt * GT_KSUB + q) * GT_BK;
          tma_load_2d(sw + q * G::WBOX, &tmW, x, col_lo, full(st));
          tma_load_2d(sw + (GT_KSUB + q) * G::WBOX, &tmW, x, col_lo + half, full(st));
        }
      };
      auto load_a = [&](int st, int kt) {
        const uint32_t sw = ring + st * G::STAGE;
#pragma unroll
        for (int q = 0; q < GT_KSUB; ++q)
          tma_load_2d(sw + G::W_BYTES + q * G::ABOX, &tmA, (kt * GT_KSUB + q) * GT_BK, 0, full(st));
      };
      // prologue: weights of the first tile's first stages (the ring starts empty)
      const int pre = blockIdx.x < tiles ? min(ksteps, G::STAGES) : 0;
      for (int kt = 0; kt < pre; ++kt) {
        mbar_expect_tx(full(kt), G::STAGE);
        ctl->pending[kt] = 0;
        load_w(kt, kt, col_of(blockIdx.x));
      }
      griddep_wait();
      for (int kt = 0; kt < pre; ++kt) load_a(kt, kt);
      int issued = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x) {
        const int col_lo = col_of(tile);
        for (int kt = 0; kt < ksteps; ++kt, ++issued) {
          if (issued >= pre) {
            if (!mbar_wait(empty(stage), phase ^ 1, abort_flag)) break;
            mbar_expect_tx(full(stage), G::STAGE);
            ctl->pending[stage] = (int)phase;
            load_w(stage, kt, col_lo);
            load_a(stage, kt);
          }
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    } else {
      griddep_wait();
    }
  } else {
    griddep_wait();
    // consumers: warp w owns rows 8w..8w+7 of both strips
    int stage = 0;
    uint32_t phase = 0;
    const int brow = warp * 8 + (lane & 7);
    const int bstrip = lane >> 4, bch = (lane >> 3) & 1;
    const int arow = lane & 15, ach = lane >> 4;
    const int j = warp * 8 + 2 * (lane & 3);  // this thread's columns j, j+1 of each strip
    for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x) {
      const int col_lo = col_of(tile);
      float acc[MB][2][4];
#pragma unroll
      for (int mi = 0; mi < MB; ++mi)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mi][t][e] = 0.f;
      bool ok = true;
      for (int kt = 0; kt < ksteps; ++kt) {
        if (!mbar_wait(full(stage), phase, abort_flag)) {
          ok = false;
          break;
        }
        ctl->pending[stage] = -1;
        const uint32_t sw = ring + stage * G::STAGE;
        const uint32_t sa = sw + G::W_BYTES;
#pragma unroll
        for (int q = 0; q < GT_KSUB; ++q)
#pragma unroll
          for (int kk = 0; kk < GT_BK / 16; ++kk) {
            uint32_t b0[2], b1[2];
            ldmatrix_x4(sw + (bstrip * GT_KSUB + q) * G::WBOX + sw128(brow, 2 * kk + bch), b0[0], b0[1], b1[0],
                        b1[1]);
#pragma unroll
            for (int mi = 0; mi < MB; ++mi) {
              uint32_t af[4];
              ldmatrix_x4(sa + q * G::ABOX + sw128(mi * 16 + arow, 2 * kk + ach), af[0], af[1], af[2], af[3]);
              mma_bf16_16816(acc[mi][0], af, b0);
              mma_bf16_16816(acc[mi][1], af, b1);
            }
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(stage));
        if (++stage == G::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      const int lo = col_lo + j, hi = col_lo + half + j;
#pragma unroll
      for (int mi = 0; mi < MB; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = mi * 16 + (lane >> 2) + (e >> 1) * 8;
          if (m < M) apply_pair(ep, m, lo + (e & 1), hi + (e & 1), acc[mi][0][e], acc[mi][1][e]);
        }
    }
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    atomicOr(status, kStatusTimeout);
    for (int s = 0; s < G::STAGES; ++s) {  // TMA copies still in flight into this CTA's ring
      const int ph = ctl->pending[s];
      if (ph < 0) continue;
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full(s), (uint32_t)ph) && global_ns() - t0 < kTimeoutNs) {
      }
    }
  }
}

template <int MB, int TR>
cudaError_t launch_mb(const bf16* A, int lda, const bf16* W, int K, const EpiParams& ep, int num_sms, int* status,
                      cudaStream_t stream) {
  using G = Gt<MB, TR>;
  constexpr int smem = gt_smem_bytes(G::STAGE, G::STAGES);
  static_assert(smem <= 227 * 1024, "ring too large");
  static_assert(G::STAGE % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  CUtensorMap ma, mw;
  if (!tma_map_bf16_2d(&ma, A, ep.M, K, lda, GT_BK, G::A_ROWS, true) ||
      !tma_map_bf16_2d(&mw, W, ep.N, K, K, GT_BK, TR / 2, true))
    return cudaErrorNotSupported;
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_tma_kernel<MB, TR>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const int tiles = ep.N / TR;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles < num_sms ? tiles : num_sms);
  cfg.blockDim = dim3(G::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<MB, TR>, ma, mw, K, ep, status);
}

template <int TR>
cudaError_t launch_tr(const bf16* A, int lda, const bf16* W, int K, const EpiParams& ep, int num_sms, int* status,
                      cudaStream_t stream) {
  if (ep.M <= 16) return launch_mb<1, TR>(A, lda, W, K, ep, num_sms, status, stream);
  if (ep.M <= 32) return launch_mb<2, TR>(A, lda, W, K, ep, num_sms, status, stream);
  if (ep.M <= 48) return launch_mb<3, TR>(A, lda, W, K, ep, num_sms, status, stream);
  return launch_mb<4, TR>(A, lda, W, K, ep, num_sms, status, stream);
}

}  // namespace

cudaError_t launch_gemv_tma(const bf16* A, int lda, const bf16* W, int K, const EpiParams& ep, int num_sms,
                            int* status, cudaStream_t stream) {
  const int half = pair_half(ep);
  if (ep.M < 1 || ep.M > 64 || K % GT_BK || ep.N % 128 || half % 32 || (2 * half) > 128 || lda % 8 ||
      (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(W) & 15))
    return cudaErrorNotSupported;
  // 64-row tiles when there are enough of them for half the SMs, else 32-row tiles
  if (2 * (ep.N / 64) >= num_sms) return launch_tr<64>(A, lda, W, K, ep, num_sms, status, stream);
  if (2 * (ep.N / 32) >= num_sms) return launch_tr<32>(A, lda, W, K, ep, num_sms, status, stream);
  return cudaErrorNotSupported;
}

}  // namespace skv
