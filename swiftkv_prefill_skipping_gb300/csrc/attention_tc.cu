// Varlen causal GQA flash attention on tcgen05 (sm_103a), d_head = 128, reading K/V
// straight out of the paged cache with TMA.
//
// One CTA = 128 query rows of one prompt chunk x one query head. A chunk may follow ctx
// tokens already in the cache (chunked prefill, decode rows): its rows then sit at
// positions ctx.. and see keys [0, ctx + row]. 6 warps:
//   warp 0     TMA producer: the Q tile once (two 64-column halves, 128B swizzle), then
//              per 64-key block the K and V rows of its four 16-token pages (each page
//              row block is contiguous in the pool) into a 3-stage ring
//   warp 1     allocates TMEM; one lane issues S = Q K^T (M=128, N=64, K=128) into one of
//              two 64-column S buffers, and O += P V (M=128, N=128, K=64; bf16 operands: P
//              read from TMEM as a high and a low part, two MMAs; V used as an MN-major
//              operand in the cache's own row layout) into one 128-column accumulator; S of
//              block j+1 is issued before P V of block j so the tensor core works while the
//              softmax warps do; an S buffer is refilled only after the P V that read the P
//              stored over it has completed
//   warps 2-5  one thread per query row: tcgen05.ld its S row, causal/length mask (only on
//              blocks that cross the diagonal or the prompt end), online softmax in the log2
//              domain with a running max allowed to lag by up to 2^8 (O, accumulated across
//              blocks in TMEM by the MMA, is rescaled in place only when it moves further),
//              P as bf16 high + low parts (about 17 significant bits) by tcgen05.st over
//              the S columns it came from; finally O / l from TMEM to global memory
// FP8 cache: the pools hold the e4m3 codes as (exact) bf16 values; the block's key and value
// scales come with its K/V, each score is multiplied by its key's scale and each P by its
// value's scale (float32). All mbarrier waits are bounded; on a timeout the CTA flags
// kStatusTimeout, drains its own TMA copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "attn_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int D = 128;          // head dim
constexpr int BQ = 128;         // query rows per CTA
constexpr int BKV = 64;         // keys per block (4 pages)
constexpr int KV_STAGES = 3;
constexpr int THREADS = 192;
constexpr int Q_BYTES = BQ * D * 2;            // 32 KB (two 16 KB halves)
constexpr int KV_HALF = BKV * 64 * 2;          // 8 KB: 64 keys x 64 dims
constexpr int K_BYTES = 2 * KV_HALF;           // 16 KB
constexpr int STAGE_BYTES = 2 * K_BYTES;       // K + V
constexpr int SCALE_BYTES = 2 * BKV * 4;       // FP8 cache: the block's key scales, then value scales
constexpr int TMEM_COLS = 256;                 // S: 2 x 64, O: 128 (accumulated across blocks)
constexpr int S_COL = 0, O_COL = 128;
constexpr float kStaleMax = 8.f;               // log2 headroom before O is rescaled
constexpr int P_LO_COL = 32;                   // P over S: high parts in columns 0-31, low parts 32-63

struct Ctrl {
  uint64_t q_full, kv_full[KV_STAGES], kv_empty[KV_STAGES], s_full[2], p_full[2], pv_done[2], fin;
  uint32_t tmem_base;
  int abort;
  int pending[KV_STAGES + 1];
};
constexpr int SMEM_BYTES = 1024 + Q_BYTES + KV_STAGES * (STAGE_BYTES + SCALE_BYTES) + (int)sizeof(Ctrl);

constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);  // Q (K-major) x K (K-major)
constexpr uint32_t IDESC_O = make_idesc(BQ, D, false, true);  // P (TMEM) x V (MN-major), bf16

__global__ void __launch_bounds__(THREADS, 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const float* __restrict__ kscale, const float* __restrict__ vscale,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ cu,
    const int* __restrict__ ctx, const int* __restrict__ tiles, int n_q, int n_kv, bf16* __restrict__ out, int ldo,
    float scale_log2, int* status) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + Q_BYTES;
  const uint32_t sScale = sKV + KV_STAGES * STAGE_BYTES;  // stage s at sScale + s * SCALE_BYTES
  const float* sScale_gen = reinterpret_cast<const float*>(smem + Q_BYTES + KV_STAGES * STAGE_BYTES);
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + Q_BYTES + KV_STAGES * (STAGE_BYTES + SCALE_BYTES));
  const bool fp8 = kscale != nullptr;
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = tiles[blockIdx.x];
  const int s = tile >> 16, qt = tile & 0xffff;
  const int h = blockIdx.y, kvh = h / (n_q / n_kv);
  const int seq0 = cu[s], n = cu[s + 1] - seq0;
  const int q0 = qt * BQ;
  // the chunk's rows sit at positions c0.. after c0 cached keys; keys [0, nk) are visible
  const int c0 = ctx ? ctx[s] : 0, nk = c0 + n;
  const int kv_end = min(nk, c0 + q0 + BQ);
  const int nblk = (kv_end + BKV - 1) / BKV;
  const int pool_rows = num_pages * n_kv * kPageSize;

  auto bar = [&](uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    mbar_init(bar(ctl->q_full), 1);
    for (int i = 0; i < KV_STAGES; ++i) {
      mbar_init(bar(ctl->kv_full[i]), 1);
      mbar_init(bar(ctl->kv_empty[i]), 1);
      ctl->pending[i] = -1;
    }
    ctl->pending[KV_STAGES] = -1;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(ctl->s_full[i]), 1);
      mbar_init(bar(ctl->p_full[i]), 128);
      mbar_init(bar(ctl->pv_done[i]), 1);
    }
    mbar_init(bar(ctl->fin), 1);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
      // Q: rows seq0+q0 .. +127 of this head's 128 columns (rows past the prompt are masked later)
      mbar_expect_tx(bar(ctl->q_full), Q_BYTES);
      ctl->pending[KV_STAGES] = 0;
      tma_load_2d(sQ, &tmQ, h * D, seq0 + q0, bar(ctl->q_full));
      tma_load_2d(sQ + Q_BYTES / 2, &tmQ, h * D + 64, seq0 + q0, bar(ctl->q_full));
      int stage = 0;
      uint32_t phase = 0;
      for (int j = 0; j < nblk; ++j) {
        if (!mbar_wait(bar(ctl->kv_empty[stage]), phase ^ 1, abort_flag)) break;
        mbar_expect_tx(bar(ctl->kv_full[stage]), STAGE_BYTES + (fp8 ? SCALE_BYTES : 0));
        ctl->pending[stage] = (int)phase;
        const uint32_t sk = sKV + stage * STAGE_BYTES, sv = sk + K_BYTES;
#pragma unroll
        for (int pg = 0; pg < BKV / kPageSize; ++pg) {
          const int key = j * BKV + pg * kPageSize;
          int page = key < nk ? bt[(size_t)s * max_pages + (key >> 4)] : -1;
          const bool valid = page >= 0 && page < num_pages;
          // a page outside the pool reads rows past the tensor's end: TMA fills zeros
          const int row = valid ? (page * n_kv + kvh) * kPageSize : pool_rows;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_2d(sk + hf * KV_HALF + pg * 2048, &tmK, hf * 64, row, bar(ctl->kv_full[stage]));
            tma_load_2d(sv + hf * KV_HALF + pg * 2048, &tmV, hf * 64, row, bar(ctl->kv_full[stage]));
          }
          if (fp8) {  // the page's 16 key and 16 value scales (page 0's for a page outside the pool)
            const size_t srow = valid ? (size_t)row : (size_t)kvh * kPageSize;
            const uint32_t ss = sScale + stage * SCALE_BYTES + pg * kPageSize * 4;
            bulk_load(ss, kscale + srow, kPageSize * 4, bar(ctl->kv_full[stage]));
            bulk_load(ss + BKV * 4, vscale + srow, kPageSize * 4, bar(ctl->kv_full[stage]));
          }
        }
        if (++stage == KV_STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(bar(ctl->q_full), 0, abort_flag);
      if (ok) ctl->pending[KV_STAGES] = -1;
      auto issue_s = [&](int j) -> bool {
        const int st = j % KV_STAGES;
        const uint32_t ph = (uint32_t)((j / KV_STAGES) & 1);
        if (!mbar_wait(bar(ctl->kv_full[st]), ph, abort_flag)) return false;
        ctl->pending[st] = -1;
        const int sb = j & 1;
        // the buffer holds P of block j - 2 until the P V that reads it has completed
        if (j >= 2 && !mbar_wait(bar(ctl->pv_done[sb]), (uint32_t)(((j - 2) >> 1) & 1), abort_flag)) return false;
        tc_fence_after();
        const uint32_t sk = sKV + st * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (Q_BYTES / 2) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * KV_HALF + (kk & 3) * 32;
          tc_mma(tmem + S_COL + sb * BKV, sdesc(sQ + off), sdesc(sk + koff), IDESC_S, kk != 0);
        }
        tc_commit(bar(ctl->s_full[sb]));
        return true;
      };
      if (ok && nblk > 0) ok = issue_s(0);
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + 1 < nblk && !issue_s(j + 1)) break;
        const int pb = j & 1;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        if (!mbar_wait(bar(ctl->p_full[pb]), ph, abort_flag)) break;
        const int st = j % KV_STAGES;
        tc_fence_after();
        const uint32_t sv = sKV + st * STAGE_BYTES + K_BYTES;
        const uint32_t pcol = tmem + S_COL + pb * BKV;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          // P: 16 keys = 8 TMEM columns per MMA (high part, then low part); V: MN-major,
          // 64-dim halves 8 KB apart, 8-key groups 1 KB apart
          const uint64_t vdesc = sdesc_sw128(sv + kk * 2048, KV_HALF, 1024);
          tc_mma_ts(tmem + O_COL, pcol + kk * 8, vdesc, IDESC_O, (j | kk) != 0);
          tc_mma_ts(tmem + O_COL, pcol + P_LO_COL + kk * 8, vdesc, IDESC_O, 1);
        }
        tc_commit(bar(ctl->pv_done[pb]));
        tc_commit(bar(ctl->kv_empty[st]));
      }
    }
  } else {
    // softmax / output warps: thread <-> query row. O accumulates in TMEM across blocks; the
    // probabilities use a running max that may lag the true one by up to 2^kStaleMax (they
    // then stay <= 256); only when a row's max moves further is O rescaled, by the warp, in
    // TMEM, after the previous block's P V has landed.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int qrow = q0 + r;     // row within the chunk
    const int qpos = c0 + qrow;  // its position
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    auto wait_pv = [&](int j) -> bool {
      return mbar_wait(bar(ctl->pv_done[j & 1]), (uint32_t)((j >> 1) & 1), abort_flag);
    };

    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(bar(ctl->s_full[sb]), (uint32_t)((j >> 1) & 1), abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sc[BKV];
      tmem_ld32(tmem + lane_off + S_COL + sb * BKV, sc);
      tmem_ld32(tmem + lane_off + S_COL + sb * BKV + 32, sc + 32);
      const float* kvs = nullptr;  // FP8: this block's key scales, then value scales
      if (fp8) {
        // the stage's scales arrived with its K/V (kv_full): wait on it directly so their
        // shared-memory writes are visible to this thread (the phase has long completed)
        const int st = j % KV_STAGES;
        if (!mbar_wait(bar(ctl->kv_full[st]), (uint32_t)((j / KV_STAGES) & 1), abort_flag)) {
          ok = false;
          break;
        }
        kvs = sScale_gen + st * (SCALE_BYTES / 4);
#pragma unroll
        for (int i = 0; i < BKV; ++i) sc[i] *= kvs[i];
      }
      const bool interior = (j + 1) * BKV - 1 <= c0 + q0 && (j + 1) * BKV <= nk;  // no key masked in any row
      if (!interior) {
#pragma unroll
        for (int i = 0; i < BKV; ++i) {
          const int key = j * BKV + i;
          if (key > qpos || key >= nk) sc[i] = -INFINITY;
        }
      }
      // row max and row sum over 8 independent partials (short dependency chains), combined
      // in a fixed order
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // sc[k], sc[k + 8], ..., sc[k + 56] with three-input max
        float v = fmax3f(sc[k], sc[k + 8], sc[k + 16]);
        v = fmax3f(v, sc[k + 24], sc[k + 32]);
        v = fmax3f(v, sc[k + 40], sc[k + 48]);
        pm[k] = fmaxf(v, sc[k + 56]);
      }
      float mx = fmax3f(fmax3f(pm[0], pm[1], pm[2]), fmax3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      mx *= scale_log2;
      const bool move = mx > m + kStaleMax;
      if (__any_sync(0xffffffffu, move)) {
        const float mn = move ? mx : m;
        const float factor = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
        if (j > 0) {  // O holds blocks 0..j-1: wait for the last of them, rescale the warp's rows
          if (!wait_pv(j - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            float t[32];
            tmem_ld32(tmem + lane_off + O_COL + c, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] *= factor;
            tmem_st32(tmem + lane_off + O_COL + c, t);
          }
        }
        l *= factor;
        m = mn;
      }
      const float mneg = -m;
      float ps[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ps[k] = 0.f;
#pragma unroll
      for (int i = 0; i < BKV; ++i) {
        sc[i] = ex2_approx(fmaf(sc[i], scale_log2, mneg));
        ps[i & 7] += sc[i];
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      if (fp8) {  // P V with V = code x scale: the value scale rides on P
#pragma unroll
        for (int i = 0; i < BKV; ++i) sc[i] *= kvs[BKV + i];
      }
      // P over this block's S columns (read above), as bf16 high and low parts
      {
        uint32_t pw[2 * 32];
        split_p_bf16(sc, pw);
        tmem_st64(tmem + lane_off + S_COL + sb * BKV, pw);
      }
      tc_fence_before();
      mbar_arrive(bar(ctl->p_full[sb]));
    }
    if (ok && nblk > 0) ok = wait_pv(nblk - 1);
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      bf16* dst = out + (size_t)(seq0 + min(qrow, n - 1)) * ldo + h * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        float t[32];
        tmem_ld32(tmem + lane_off + O_COL + c, t);
        if (qrow < n) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 u;
            u.x = pack_bf16(t[e] * inv, t[e + 1] * inv);
            u.y = pack_bf16(t[e + 2] * inv, t[e + 3] * inv);
            u.z = pack_bf16(t[e + 4] * inv, t[e + 5] * inv);
            u.w = pack_bf16(t[e + 6] * inv, t[e + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c + e) = u;
          }
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(status, kStatusTimeout);
      for (int i = 0; i <= KV_STAGES; ++i) {
        const int ph = ctl->pending[i];
        if (ph < 0) continue;
        const uint32_t b = i < KV_STAGES ? bar(ctl->kv_full[i]) : bar(ctl->q_full);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(b, (uint32_t)ph) && global_ns() - t0 < kTimeoutNs) {
        }
      }
    }
    if (threadIdx.x == 32) {
      tc_commit(bar(ctl->fin));
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(bar(ctl->fin), 0) && global_ns() - t0 < kTimeoutNs) {
      }
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace

cudaError_t launch_attention_prefill_tc(const bf16* q, int ldq, int T, const bf16* k_pool, const bf16* v_pool,
                                        const float* k_scale, const float* v_scale, const int* block_table,
                                        int max_pages, int num_pages, const int* cu, const int* ctx, const int* tiles,
                                        int num_tiles, int n_q, int n_kv, int d_head, bf16* out, int ldo, int* status,
                                        cudaStream_t stream) {
  if (num_tiles <= 0) return cudaSuccess;
  if (d_head != D || (reinterpret_cast<uintptr_t>(q) & 15) || ldq % 8 || (!k_scale != !v_scale) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 15) || (reinterpret_cast<uintptr_t>(v_scale) & 15))
    return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  const int pool_rows = num_pages * n_kv * kPageSize;
  if (!tma_map_bf16_2d(&mq, q, T, n_q * D, ldq, 64, BQ, true) ||
      !tma_map_bf16_2d(&mk, k_pool, pool_rows, D, D, 64, kPageSize, true) ||
      !tma_map_bf16_2d(&mv, v_pool, pool_rows, D, D, 64, kPageSize, true))
    return cudaErrorNotSupported;
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_tc_kernel), SMEM_BYTES, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(num_tiles, n_q);
  attn_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, k_scale, v_scale, block_table, max_pages,
                                                        num_pages, cu, ctx, tiles, n_q, n_kv, out, ldo, scale_log2,
                                                        status);
  return cudaGetLastError();
}

}  // namespace skv
