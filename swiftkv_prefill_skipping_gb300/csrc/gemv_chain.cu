// A chain of skinny GEMMs and RMSNorms (M <= 64 rows: decode tokens, the SwiftKV last-token
// tail) in one persistent, cooperative launch, each phase reading what the one before wrote:
// O (+residual) -> RMSNorm -> gate/up (+SwiGLU) -> down (+residual) -> RMSNorm -> the next
// layer's Q/QKV or the LM head. One CTA per SM; grid-wide barriers separate the phases.
//
// The weights do not depend on the activations, so each CTA's producer thread streams its
// weight tiles of every GEMM phase back to back into a ~190 KB TMA ring (64-row tiles: two
// 32-row strips `half` apart, 256-deep k steps of 32 x 64 boxes, as in the single-GEMM skinny
// kernel). The slice of A that goes with each stage is requested only once the phase's
// inputs are complete (the barrier before it has been passed); until then the stage waits
// with its weights already loaded, so the weight stream does not stop at the barriers. Tiles
// of phase p are dealt round-robin starting at the CTA after phase p - 1's last one, so SMs
// without work in a narrow phase are already streaming the next one's weights. Four
// consumer warps accumulate on mma.sync (bf16 in, fp32 accumulate, k in order: a row's result
// never depends on the batch) and run the shared epilogue from registers. An RMSNorm phase
// gives each of the M rows to one CTA, whose consumer warps compute the row's mean square
// (fixed order), then u = bf16(x * rsqrt(mean + eps) * gamma) - the model's own rounding point.
//
// Grid barrier: a 32-bit arrival counter that only grows (the host passes the count before
// this launch). After finishing phase p every CTA makes its stores visible (proxy fence for
// the TMA readers, then a release add); the next phase waits with acquire loads until all
// CTAs have arrived. Every wait is bounded (2 s); on a timeout the CTA raises kStatusTimeout,
// drains its own TMA copies and exits, and the others time out in turn.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int CH_BK = 64;        // k per box: one 128-byte swizzle row
constexpr int CH_KSUB = 4;       // boxes along k per stage (256 k)
constexpr int CH_TR = 64;        // weight rows per tile
constexpr int CH_CONSUMERS = CH_TR / 16;
constexpr int CH_THREADS = (CH_CONSUMERS + 1) * 32;
constexpr int CH_RING_BYTES = 192 * 1024;
constexpr int CH_MAX_STAGES = 24;

template <int MB>
struct Ch {
  static constexpr int A_ROWS = MB * 16;
  static constexpr int WBOX = CH_TR / 2 * CH_BK * 2;   // one 32 x 64 box
  static constexpr int ABOX = A_ROWS * CH_BK * 2;
  static constexpr int W_BYTES = 2 * CH_KSUB * WBOX;    // strip-major: [strip][ksub]
  static constexpr int A_BYTES = CH_KSUB * ABOX;
  static constexpr int STAGE = W_BYTES + A_BYTES;       // a multiple of 1024
  static constexpr int STAGES = CH_RING_BYTES / STAGE < CH_MAX_STAGES ? CH_RING_BYTES / STAGE : CH_MAX_STAGES;
};

struct ChCtrl {
  uint64_t full[CH_MAX_STAGES];
  uint64_t empty[CH_MAX_STAGES];
  uint64_t csync;                       // consumer-warp barrier (one arrival per warp)
  int pending[CH_MAX_STAGES];
  int abort;
  float red[CH_CONSUMERS];              // RMSNorm: per-warp sums of squares
};

constexpr int ch_smem_bytes(int stage_bytes, int stages) { return 1024 + stages * stage_bytes + (int)sizeof(ChCtrl); }

__device__ __forceinline__ uint32_t ch_sw128(int row, int ch) {
  return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ bool count_reached(const unsigned* c, unsigned target) {
  return (int)(ld_acquire_u32(c) - target) >= 0;
}
// Bounded wait until the arrival count reaches target; false on abort or timeout.
__device__ bool grid_wait(const unsigned* c, unsigned target, volatile int* abort_flag) {
  if (count_reached(c, target)) return true;
  const uint64_t t0 = global_ns();
  while (!count_reached(c, target)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > kTimeoutNs) {
      *abort_flag = 1;
      return false;
    }
    __nanosleep(100);
  }
  return true;
}


// Arrival count the barrier before phase p waits for (phases 1 .. n-1 each have one).
__device__ __forceinline__ unsigned barrier_target(const ChainParams& P, int p) {
  return P.count_base + (unsigned)p * gridDim.x;
}

template <int MB>
__global__ void __launch_bounds__(CH_THREADS, 1) gemv_chain_kernel(const __grid_constant__ ChainParams P,
                                                                  int* status) {
  using G = Ch<MB>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t ring = smem_u32(smem);
  ChCtrl* ctl = reinterpret_cast<ChCtrl*>(smem + G::STAGES * G::STAGE);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nG = (int)gridDim.x, me = (int)blockIdx.x;
  auto full = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty = [&](int s) { return smem_u32(&ctl->empty[s]); };
  // this CTA's first tile of phase p (then every nG-th)
  auto first_tile = [&](int p) { return ((me - P.ph[p].first_cta) % nG + nG) % nG; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CH_CONSUMERS);
      ctl->pending[s] = -1;
    }
    mbar_init(smem_u32(&ctl->csync), CH_CONSUMERS);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == CH_CONSUMERS) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      // A slices not yet requested: (stage, phase, k step), in issue order
      int pq_stage[CH_MAX_STAGES] = {}, pq_phase[CH_MAX_STAGES] = {}, pq_kt[CH_MAX_STAGES] = {};
      int pq_head = 0, pq_n = 0;
      int ready = -1;  // highest phase whose inputs are complete
      auto load_a = [&](int st, int p, int kt) {
        const uint32_t sa = ring + st * G::STAGE + G::W_BYTES;
#pragma unroll
        for (int q = 0; q < CH_KSUB; ++q)
          tma_load_2d(sa + q * G::ABOX, &P.ph[p].tmA, (kt * CH_KSUB + q) * CH_BK, 0, full(st));
      };
      // requests the A slices of every pending stage whose phase is ready (in order)
      auto drain = [&]() {
        while (pq_n > 0 && pq_phase[pq_head] <= ready) {
          load_a(pq_stage[pq_head], pq_phase[pq_head], pq_kt[pq_head]);
          pq_head = (pq_head + 1) % CH_MAX_STAGES;
          --pq_n;
        }
      };
      // advances `ready` past every barrier that has been passed (phase 0: the kernel start)
      auto poll = [&]() {
        bool moved = false;
        while (ready + 1 < P.n && ready >= 0 && count_reached(P.count, barrier_target(P, ready + 1))) {
          ++ready;
          moved = true;
        }
        if (moved) fence_proxy_async_global();  // the previous phases' stores, for the TMA reads
        drain();
      };
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int p = 0; ok && p < P.n; ++p) {
        const ChainPhase& ph = P.ph[p];
        if (ph.is_norm) continue;  // no weights
        const int half = pair_half(ph.ep);
        const int strips = half / (CH_TR / 2);
        const int ksteps = (ph.K + CH_BK * CH_KSUB - 1) / (CH_BK * CH_KSUB);
        for (int tile = first_tile(p); ok && tile < ph.tiles; tile += nG) {
          const int col_lo = (tile / strips) * 2 * half + (tile % strips) * (CH_TR / 2);
          for (int kt = 0; kt < ksteps; ++kt, ++issued) {
            if (issued >= G::STAGES) {  // the ring's first pass needs no wait
              const uint64_t t0 = global_ns();
              while (!mbar_test_wait(empty(stage), phase ^ 1)) {
                if (ready >= 0) poll();
                if (*abort_flag || global_ns() - t0 > kTimeoutNs) {
                  *abort_flag = 1;
                  ok = false;
                  break;
                }
              }
              if (!ok) break;
            }
            mbar_expect_tx(full(stage), G::STAGE);
            ctl->pending[stage] = (int)phase;
            const uint32_t sw = ring + stage * G::STAGE;
#pragma unroll
            for (int q = 0; q < CH_KSUB; ++q) {
              const int x = (kt * CH_KSUB + q) * CH_BK;
              tma_load_2d(sw + q * G::WBOX, &ph.tmW, x, col_lo, full(stage));
              tma_load_2d(sw + (CH_KSUB + q) * G::WBOX, &ph.tmW, x, col_lo + half, full(stage));
            }
            if (pq_n == 0 && p <= ready) {
              load_a(stage, p, kt);
            } else {
              const int slot = (pq_head + pq_n) % CH_MAX_STAGES;
              pq_stage[slot] = stage;
              pq_phase[slot] = p;
              pq_kt[slot] = kt;
              ++pq_n;
            }
            if (issued + 1 == G::STAGES && ready < 0) {
              // the ring is primed with weights: now wait for the kernels this one depends on
              griddep_wait();
              ready = 0;
              drain();
            }
            if (++stage == G::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (ok && ready < 0) {  // fewer stages than the ring holds
        griddep_wait();
        ready = 0;
        drain();
      }
      // the A slices still pending belong to phases whose barriers are ahead
      const uint64_t t0 = global_ns();
      while (ok && pq_n > 0) {
        poll();
        if (*abort_flag || global_ns() - t0 > kTimeoutNs) {
          *abort_flag = 1;
          break;
        }
        __nanosleep(100);
      }
    } else {
      griddep_wait();
    }
  } else {
    // ---------------------------------------------------------------- consumers
    griddep_wait();
    int stage = 0, nsync = 0;
    uint32_t phase = 0;
    const int tid = threadIdx.x;  // 0 .. 127
    // Barrier of the four consumer warps (shared-memory writes before it are visible after it).
    // Bounded, so a warp that aborted cannot leave the others waiting for ever.
    auto consumer_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->csync));
      const bool r = mbar_wait(smem_u32(&ctl->csync), (uint32_t)(nsync & 1), abort_flag);
      ++nsync;
      __syncwarp();
      return r;
    };
    const int brow = warp * 8 + (lane & 7);
    const int bstrip = lane >> 4, bch = (lane >> 3) & 1;
    const int arow = lane & 15, ach = lane >> 4;
    const int j = warp * 8 + 2 * (lane & 3);  // this thread's columns j, j+1 of each strip
    bool ok = true;
    for (int p = 0; ok && p < P.n; ++p) {
      const ChainPhase& ph = P.ph[p];
      const EpiParams& ep = ph.ep;
      const int M = ep.M;
      if (p > 0) {
        if (lane == 0) ok = grid_wait(P.count, barrier_target(P, p), abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        (void)ld_acquire_u32(P.count);  // every thread's own acquire of the earlier phases' stores
      }
      if (ph.is_norm) {
        // RMSNorm rows dealt round-robin like GEMM tiles: the row's sum of squares (thread
        // stripes of 4, then lanes, then warps, all in a fixed order), then the bf16 output
        const ChainNorm& nm = ph.norm;
        for (int row = first_tile(p); ok && row < ph.tiles; row += nG) {
          const float* xr = nm.x + (size_t)row * nm.ldx;
          float q = 0.f;
          for (int k = 4 * tid; k < nm.d; k += 4 * CH_CONSUMERS * 32) {
            const float4 v = *reinterpret_cast<const float4*>(xr + k);
            q += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
          if (lane == 0) ctl->red[warp] = q;
          if (!(ok = consumer_sync())) break;
          const float ssum = (ctl->red[0] + ctl->red[1]) + (ctl->red[2] + ctl->red[3]);
          const float r = rsqrtf(ssum / nm.d + nm.eps);
          bf16* ur = nm.u + (size_t)row * nm.ldu;
          for (int k = 4 * tid; k < nm.d; k += 4 * CH_CONSUMERS * 32) {
            const float4 v = *reinterpret_cast<const float4*>(xr + k);
            const float4 g = nm.gamma ? *reinterpret_cast<const float4*>(nm.gamma + k) : make_float4(1.f, 1.f, 1.f, 1.f);
            uint2 pk;
            pk.x = pack_bf16(v.x * r * g.x, v.y * r * g.y);
            pk.y = pack_bf16(v.z * r * g.z, v.w * r * g.w);
            *reinterpret_cast<uint2*>(ur + k) = pk;
          }
          if (!(ok = consumer_sync())) break;  // red[] is reused by the next row
        }
      } else {
        const int half = pair_half(ep);
        const int strips = half / (CH_TR / 2);
        const int ksteps = (ph.K + CH_BK * CH_KSUB - 1) / (CH_BK * CH_KSUB);
        for (int tile = first_tile(p); tile < ph.tiles; tile += nG) {
          const int col_lo = (tile / strips) * 2 * half + (tile % strips) * (CH_TR / 2);
          float acc[MB][2][4];
#pragma unroll
          for (int mi = 0; mi < MB; ++mi)
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[mi][t][e] = 0.f;
          for (int kt = 0; kt < ksteps; ++kt) {
            if (!mbar_wait(full(stage), phase, abort_flag)) {
              ok = false;
              break;
            }
            ctl->pending[stage] = -1;
            const uint32_t sw = ring + stage * G::STAGE;
            const uint32_t sa = sw + G::W_BYTES;
#pragma unroll
            for (int q = 0; q < CH_KSUB; ++q)
#pragma unroll
              for (int kk = 0; kk < CH_BK / 16; ++kk) {
                uint32_t b0[2], b1[2];
                ldmatrix_x4(sw + (bstrip * CH_KSUB + q) * G::WBOX + ch_sw128(brow, 2 * kk + bch), b0[0], b0[1],
                            b1[0], b1[1]);
#pragma unroll
                for (int mi = 0; mi < MB; ++mi) {
                  uint32_t af[4];
                  ldmatrix_x4(sa + q * G::ABOX + ch_sw128(mi * 16 + arow, 2 * kk + ach), af[0], af[1], af[2], af[3]);
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
      if (!ok) break;
      // this CTA's stores of phase p are done: publish them for the next phase (generic readers
      // and the TMA loads of the next phase's A)
      fence_proxy_async_global();
      if (!(ok = consumer_sync())) break;
      if (tid == 0 && p + 1 < P.n) {
        __threadfence();
        red_release_add_u32(P.count, 1u);
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

template <int MB>
cudaError_t launch_chain_mb(const ChainParams& P, int num_sms, int* status, cudaStream_t stream) {
  using G = Ch<MB>;
  constexpr int smem = ch_smem_bytes(G::STAGE, G::STAGES);
  static_assert(smem <= 227 * 1024, "ring too large");
  static_assert(G::STAGE % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_chain_kernel<MB>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // cooperative: every CTA is resident at once (the grid barriers rely on it), and a
  // programmatic dependent of the kernel before it, so the weight ring fills while that
  // kernel finishes
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel<MB>, P, status);
  if (e != cudaSuccess) {  // a cooperative launch that may not also be a programmatic dependent
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel<MB>, P, status);
  }
  return e;
}

}  // namespace

cudaError_t launch_gemv_chain(const ChainStep* steps, int n, int num_sms, unsigned* count, unsigned* count_base,
                              int* status, cudaStream_t stream) {
  if (n < 1 || n > kChainMaxPhases || num_sms < 1 || !count || !count_base) return cudaErrorNotSupported;
  int M = 0;
  for (int p = 0; p < n; ++p)
    if (steps[p].W) M = M ? M : steps[p].ep.M;
  if (M < 1 || M > 64) return cudaErrorNotSupported;
  ChainParams P;
  memset(&P, 0, sizeof P);
  int next_cta = 0;
  for (int p = 0; p < n; ++p) {
    const ChainStep& c = steps[p];
    ChainPhase& ph = P.ph[p];
    if (!c.W) {  // RMSNorm phase
      const ChainNorm& nm = c.norm;
      if (!nm.x || !nm.u || nm.rows < 1 || nm.rows > M || nm.d % 4 || nm.ldx % 4 || nm.ldu % 4 ||
          (reinterpret_cast<uintptr_t>(nm.x) & 15) || (reinterpret_cast<uintptr_t>(nm.u) & 7))
        return cudaErrorNotSupported;
      ph.is_norm = 1;
      ph.norm = nm;
      ph.tiles = nm.rows;
    } else {
      const int half = pair_half(c.ep);
      if (c.ep.M != M || c.K % CH_BK || c.ep.N % 128 || half % 32 || 2 * half > 128 || c.lda % 8 ||
          (reinterpret_cast<uintptr_t>(c.A) & 15) || (reinterpret_cast<uintptr_t>(c.W) & 15))
        return cudaErrorNotSupported;
      if (!tma_map_bf16_2d(&ph.tmA, c.A, M, c.K, c.lda, CH_BK, ((M + 15) / 16) * 16, true) ||
          !tma_map_bf16_2d(&ph.tmW, c.W, c.ep.N, c.K, c.K, CH_BK, CH_TR / 2, true))
        return cudaErrorNotSupported;
      ph.ep = c.ep;
      ph.K = c.K;
      ph.tiles = c.ep.N / CH_TR;
    }
    ph.first_cta = next_cta;
    next_cta = (next_cta + ph.tiles) % num_sms;
  }
  P.n = n;
  P.count = count;
  P.count_base = *count_base;
  cudaError_t e;
  if (M <= 16) e = launch_chain_mb<1>(P, num_sms, status, stream);
  else if (M <= 32) e = launch_chain_mb<2>(P, num_sms, status, stream);
  else if (M <= 48) e = launch_chain_mb<3>(P, num_sms, status, stream);
  else e = launch_chain_mb<4>(P, num_sms, status, stream);
  if (e == cudaSuccess) *count_base += (unsigned)(n - 1) * (unsigned)num_sms;
  return e;
}

}  // namespace skv
