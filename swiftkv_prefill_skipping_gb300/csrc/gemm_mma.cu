// Warp-level tensor-core GEMMs (mma.sync m16n8k16 bf16 -> fp32) with the shared
// epilogues of common.cuh.
//
//   C[M][N] = A[M][K] * B[N][K]^T     A: activations, row-major (lda)
//                                     B: weights, nn.Linear layout [out][in] (ldb = K)
//
// gemm_tiled: 128x128x32 CTA tiles, 8 warps (64x32 each), 4-stage cp.async ring,
//             fp32 tile staged through shared memory for the pairwise epilogue.
// gemv:       M <= 64 rows (the last-token tail, decode, LM head): one CTA per pair of
//             16-column strips over the whole K, warps split K, fixed-order reduction in
//             shared memory; what the model uses for its M <= 64 GEMMs.
// gemm_skinny: the same rows with split-K across CTAs and fp32 partials in global scratch,
//             reduced in a fixed order by reduce_epilogue (used by the allocation-free entry
//             point and as a cross-check).
#include "common.cuh"
#include "launch.h"

namespace skv {

namespace {

constexpr int TM = 128, TN = 128, TK = 32, TSTAGES = 4, TTHREADS = 256;
constexpr int TLD = TK + 8;  // padded smem row (80 B): conflict-free ldmatrix
constexpr int TEPI_LD = TN + 4;
constexpr int kTiledSmem = TSTAGES * (TM + TN) * TLD * 2;  // 81920 B
static_assert(TM * TEPI_LD * 4 <= kTiledSmem, "epilogue tile must fit the ring");

__global__ void __launch_bounds__(TTHREADS) gemm_tiled_kernel(const bf16* __restrict__ A, int lda,
                                                              const bf16* __restrict__ B, int K,
                                                              EpiParams ep) {
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* sA = reinterpret_cast<bf16*>(smem);
  bf16* sB = sA + TSTAGES * TM * TLD;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int M = ep.M;
  const int ktiles = K / TK;

  auto load_stage = [&](int stage, int kt) {
    const int k0 = kt * TK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      int c = tid + i * TTHREADS;  // 0..511
      int row = c >> 2, kc = c & 3;
      int gm = m0 + row;
      const bf16* src = A + (size_t)(gm < M ? gm : 0) * lda + k0 + kc * 8;
      cp_async16(smem_u32(sA + (stage * TM + row) * TLD + kc * 8), src, gm < M ? 16 : 0);
      int gn = n0 + row;
      const bf16* srcb = B + (size_t)(gn < ep.N ? gn : 0) * K + k0 + kc * 8;
      cp_async16(smem_u32(sB + (stage * TN + row) * TLD + kc * 8), srcb, gn < ep.N ? 16 : 0);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;

#pragma unroll
  for (int s = 0; s < TSTAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    cp_async_commit();
  }

  for (int kt = 0; kt < ktiles; ++kt) {
    cp_async_wait<TSTAGES - 2>();
    __syncthreads();
    {
      int nk = kt + TSTAGES - 1;
      if (nk < ktiles) load_stage(nk % TSTAGES, nk);
      cp_async_commit();
    }
    const int stage = kt % TSTAGES;
    const bf16* a_base = sA + stage * TM * TLD;
    const bf16* b_base = sB + stage * TN * TLD;
#pragma unroll
    for (int kk = 0; kk < TK; kk += 16) {
      uint32_t af[4][4], bfr[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        int row = wm * 64 + mi * 16 + (lane & 15);
        int col = kk + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(a_base + row * TLD + col), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        int row = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        int col = kk + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(smem_u32(b_base + row * TLD + col), bfr[2 * nj][0], bfr[2 * nj][1],
                    bfr[2 * nj + 1][0], bfr[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_bf16_16816(acc[mi][ni], af[mi], bfr[ni]);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  float* tile = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
      int r = wm * 64 + mi * 16 + (lane >> 2);
      int c = wn * 32 + ni * 8 + 2 * (lane & 3);
      tile[r * TEPI_LD + c] = acc[mi][ni][0];
      tile[r * TEPI_LD + c + 1] = acc[mi][ni][1];
      tile[(r + 8) * TEPI_LD + c] = acc[mi][ni][2];
      tile[(r + 8) * TEPI_LD + c + 1] = acc[mi][ni][3];
    }
  __syncthreads();
  const int half = pair_half(ep);
  for (int u = tid; u < TM * (TN / 2); u += TTHREADS) {
    int r = u / (TN / 2), pi = u % (TN / 2);
    int m = m0 + r;
    if (m >= M) continue;
    int lo = pair_lo(pi, half);
    apply_pair(ep, m, n0 + lo, n0 + lo + half, tile[r * TEPI_LD + lo], tile[r * TEPI_LD + lo + half]);
  }
}

// ---------------------------------------------------------------------------- skinny split-K

constexpr int SN = 64, SK = 64, SSTAGES = 4, STHREADS = 128, SLD = SK + 8;

template <int MB>
__global__ void __launch_bounds__(STHREADS) gemm_skinny_kernel(const bf16* __restrict__ A, int lda,
                                                               const bf16* __restrict__ B, int K,
                                                               int M, int N, int kchunk,
                                                               float* __restrict__ part) {
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* sA = reinterpret_cast<bf16*>(smem);            // [SSTAGES][MB*16][SLD]
  bf16* sB = sA + SSTAGES * MB * 16 * SLD;             // [SSTAGES][SN][SLD]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * SN;
  const int split = blockIdx.y;
  const int kbeg = split * kchunk;
  const int ktiles = kchunk / SK;

  auto load_stage = [&](int stage, int kt) {
    const int k0 = kbeg + kt * SK;
#pragma unroll
    for (int i = 0; i < (SN * 8) / STHREADS; ++i) {
      int c = tid + i * STHREADS;
      int row = c >> 3, kc = c & 7;
      cp_async16(smem_u32(sB + (stage * SN + row) * SLD + kc * 8), B + (size_t)(n0 + row) * K + k0 + kc * 8,
                 16);
    }
#pragma unroll
    for (int i = 0; i < (MB * 16 * 8 + STHREADS - 1) / STHREADS; ++i) {
      int c = tid + i * STHREADS;
      if (c < MB * 16 * 8) {
        int row = c >> 3, kc = c & 7;
        const bf16* src = A + (size_t)(row < M ? row : 0) * lda + k0 + kc * 8;
        cp_async16(smem_u32(sA + (stage * MB * 16 + row) * SLD + kc * 8), src, row < M ? 16 : 0);
      }
    }
  };

  float acc[MB][2][4];
#pragma unroll
  for (int i = 0; i < MB; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;

#pragma unroll
  for (int s = 0; s < SSTAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    cp_async_commit();
  }
  for (int kt = 0; kt < ktiles; ++kt) {
    cp_async_wait<SSTAGES - 2>();
    __syncthreads();
    {
      int nk = kt + SSTAGES - 1;
      if (nk < ktiles) load_stage(nk % SSTAGES, nk);
      cp_async_commit();
    }
    const int stage = kt % SSTAGES;
    const bf16* a_base = sA + stage * MB * 16 * SLD;
    const bf16* b_base = sB + stage * SN * SLD;
#pragma unroll
    for (int kk = 0; kk < SK; kk += 16) {
      uint32_t bfr[2][2];
      {
        int row = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
        int col = kk + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(smem_u32(b_base + row * SLD + col), bfr[0][0], bfr[0][1], bfr[1][0], bfr[1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < MB; ++mi) {
        uint32_t af[4];
        int row = mi * 16 + (lane & 15);
        int col = kk + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(a_base + row * SLD + col), af[0], af[1], af[2], af[3]);
        mma_bf16_16816(acc[mi][0], af, bfr[0]);
        mma_bf16_16816(acc[mi][1], af, bfr[1]);
      }
    }
  }
  cp_async_wait<0>();

  float* out = part + (size_t)split * M * N;
#pragma unroll
  for (int mi = 0; mi < MB; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      int r = mi * 16 + (lane >> 2);
      int c = n0 + warp * 16 + ni * 8 + 2 * (lane & 3);
      if (r < M) {
        out[(size_t)r * N + c] = acc[mi][ni][0];
        out[(size_t)r * N + c + 1] = acc[mi][ni][1];
      }
      if (r + 8 < M) {
        out[(size_t)(r + 8) * N + c] = acc[mi][ni][2];
        out[(size_t)(r + 8) * N + c + 1] = acc[mi][ni][3];
      }
    }
}

__global__ void reduce_epilogue_kernel(const float* __restrict__ part, int splits, EpiParams ep) {
  const int M = ep.M, N = ep.N;
  const int half = pair_half(ep);
  const size_t total = (size_t)M * (N / 2);
  for (size_t u = blockIdx.x * (size_t)blockDim.x + threadIdx.x; u < total;
       u += (size_t)gridDim.x * blockDim.x) {
    int m = (int)(u / (N / 2));
    int pi = (int)(u % (N / 2));
    int lo = pair_lo(pi, half), hi = lo + half;
    float a = 0.f, b = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float* p = part + (size_t)s * M * N + (size_t)m * N;
      a += p[lo];
      b += p[hi];
    }
    apply_pair(ep, m, lo, hi, a, b);
  }
}


// ---------------------------------------------------------------------------- skinny, no split-K
//
// gemv_kernel: M <= 64 rows (the last-token tail, decode, LM head) streaming the weights
// once at HBM rate. A CTA owns two 16-column strips that are `half` apart, so RoPE and SwiGLU
// partners (n, n + half) stay inside the CTA; its 4 warps take interleaved 64-deep k-tiles,
// each with its own 4-stage cp.async ring, and their partial sums are added in a fixed order
// in shared memory before the epilogue. One launch, no global scratch, deterministic.
constexpr int GV_STAGES = 4, GV_LD = 64 + 8;

template <int MB>
__global__ void __launch_bounds__(128) gemv_kernel(const bf16* __restrict__ A, int lda,
                                                   const bf16* __restrict__ B, int K, EpiParams ep) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int WROWS = 32, AROWS = MB * 16;
  griddep_launch_dependents();  // a programmatic dependent may start as these blocks leave
  constexpr int STAGE = (WROWS + AROWS) * GV_LD;  // bf16 elements per stage per warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = ep.M;
  const int half = pair_half(ep);
  const int strips = half / 16;
  const int blk = blockIdx.x / strips, strip = blockIdx.x % strips;
  const int col_lo = blk * 2 * half + strip * 16;  // local cols 0..15 -> col_lo.., 16..31 -> col_lo+half..
  bf16* ring = reinterpret_cast<bf16*>(smem) + warp * GV_STAGES * STAGE;
  const int ktiles = K / 64;
  const int my_tiles = ktiles > warp ? (ktiles - warp + 3) / 4 : 0;

  auto load = [&](int stage, int i) {
    const int k0 = (warp + 4 * i) * 64;
    bf16* sw = ring + stage * STAGE;
    bf16* sa = sw + WROWS * GV_LD;
#pragma unroll
    for (int c = 0; c < (WROWS * 8) / 32; ++c) {  // 256 chunks of 16 B
      const int id = c * 32 + lane, row = id >> 3, kc = id & 7;
      const int n = row < 16 ? col_lo + row : col_lo + half + (row - 16);
      cp_async16(smem_u32(sw + row * GV_LD + kc * 8), B + (size_t)n * K + k0 + kc * 8, 16);
    }
#pragma unroll
    for (int c = 0; c < (AROWS * 8) / 32; ++c) {
      const int id = c * 32 + lane, row = id >> 3, kc = id & 7;
      const bf16* src = A + (size_t)(row < M ? row : 0) * lda + k0 + kc * 8;
      cp_async16(smem_u32(sa + row * GV_LD + kc * 8), src, row < M ? 16 : 0);
    }
  };

  float acc[MB][4][4];
#pragma unroll
  for (int a = 0; a < MB; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

#pragma unroll
  for (int s = 0; s < GV_STAGES - 1; ++s) {
    if (s < my_tiles) load(s, s);
    cp_async_commit();
  }
  for (int i = 0; i < my_tiles; ++i) {
    cp_async_wait<GV_STAGES - 2>();
    __syncwarp();
    if (i + GV_STAGES - 1 < my_tiles) load((i + GV_STAGES - 1) % GV_STAGES, i + GV_STAGES - 1);
    cp_async_commit();
    const bf16* sw = ring + (i % GV_STAGES) * STAGE;
    const bf16* sa = sw + WROWS * GV_LD;
#pragma unroll
    for (int kk = 0; kk < 64; kk += 16) {
      uint32_t bfr[4][2];
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int row = nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int col = kk + ((lane >> 3) & 1) * 8;
        ldmatrix_x4(smem_u32(sw + row * GV_LD + col), bfr[2 * nj][0], bfr[2 * nj][1], bfr[2 * nj + 1][0],
                    bfr[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < MB; ++mi) {
        uint32_t af[4];
        const int row = mi * 16 + (lane & 15);
        const int col = kk + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(sa + row * GV_LD + col), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) mma_bf16_16816(acc[mi][nb], af, bfr[nb]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();
  // partial sums -> shared memory [warp][row][32], then a fixed-order sum over the warps
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int mi = 0; mi < MB; ++mi)
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int r = mi * 16 + (lane >> 2), c = nb * 8 + 2 * (lane & 3);
      float* base = red + (warp * AROWS) * 32;
      base[r * 32 + c] = acc[mi][nb][0];
      base[r * 32 + c + 1] = acc[mi][nb][1];
      base[(r + 8) * 32 + c] = acc[mi][nb][2];
      base[(r + 8) * 32 + c + 1] = acc[mi][nb][3];
    }
  __syncthreads();
  for (int u = threadIdx.x; u < M * 16; u += 128) {
    const int m = u >> 4, c = u & 15;
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      a += red[(w * AROWS + m) * 32 + c];
      b += red[(w * AROWS + m) * 32 + 16 + c];
    }
    apply_pair(ep, m, col_lo + c, col_lo + half + c, a, b);
  }
}

template <int MB>
static cudaError_t launch_gemv_mb(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                                  cudaStream_t stream) {
  constexpr int smem = 4 * GV_STAGES * (32 + MB * 16) * GV_LD * 2;
  static_assert(4 * MB * 16 * 32 * 4 <= smem, "reduction buffer must fit the rings");
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_kernel<MB>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  gemv_kernel<MB><<<ep.N / 32, 128, smem, stream>>>(A, lda, B, K, ep);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep, cudaStream_t stream) {
  if (ep.M < 1 || ep.M > 64 || K % 64 || ep.N % 128) return cudaErrorNotSupported;
  if (ep.M <= 16) return launch_gemv_mb<1>(A, lda, B, K, ep, stream);
  if (ep.M <= 32) return launch_gemv_mb<2>(A, lda, B, K, ep, stream);
  if (ep.M <= 48) return launch_gemv_mb<3>(A, lda, B, K, ep, stream);
  return launch_gemv_mb<4>(A, lda, B, K, ep, stream);
}

int skinny_splits(int M, int N, int K, int num_sms) {
  (void)M;
  int tiles = N / SN;
  int s = 1;
  while (tiles * s < 2 * num_sms && K % (SK * s * 2) == 0 && K / (s * 2) >= 256) s *= 2;
  return s;
}

size_t skinny_scratch_bytes(int M, int N, int K, int num_sms) {
  return (size_t)skinny_splits(M, N, K, num_sms) * M * N * sizeof(float);
}

cudaError_t launch_gemm_tiled(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                              cudaStream_t stream) {
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tiled_kernel), kTiledSmem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(ep.N / TN, (ep.M + TM - 1) / TM);
  gemm_tiled_kernel<<<grid, TTHREADS, kTiledSmem, stream>>>(A, lda, B, K, ep);
  return cudaGetLastError();
}

template <int MB>
static cudaError_t launch_skinny_mb(const bf16* A, int lda, const bf16* B, int K, int M, int N,
                                    int splits, float* part, cudaStream_t stream) {
  constexpr int smem = SSTAGES * (MB * 16 + SN) * SLD * 2;
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm_skinny_kernel<MB>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(N / SN, splits);
  gemm_skinny_kernel<MB><<<grid, STHREADS, smem, stream>>>(A, lda, B, K, M, N, K / splits, part);
  return cudaGetLastError();
}

cudaError_t launch_gemm_skinny(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                               float* scratch, int num_sms, cudaStream_t stream) {
  const int M = ep.M, N = ep.N;
  const int splits = skinny_splits(M, N, K, num_sms);
  cudaError_t e;
  if (M <= 16) e = launch_skinny_mb<1>(A, lda, B, K, M, N, splits, scratch, stream);
  else if (M <= 32) e = launch_skinny_mb<2>(A, lda, B, K, M, N, splits, scratch, stream);
  else if (M <= 48) e = launch_skinny_mb<3>(A, lda, B, K, M, N, splits, scratch, stream);
  else e = launch_skinny_mb<4>(A, lda, B, K, M, N, splits, scratch, stream);
  if (e != cudaSuccess) return e;
  size_t total = (size_t)M * (N / 2);
  int blocks = (int)((total + 255) / 256);
  if (blocks > 8 * num_sms) blocks = 8 * num_sms;
  reduce_epilogue_kernel<<<blocks, 256, 0, stream>>>(scratch, splits, ep);
  return cudaGetLastError();
}

}  // namespace skv
