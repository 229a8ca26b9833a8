// Varlen causal GQA flash attention on tcgen05 (sm_103a), d_head = 128, two 128-row query
// tiles per CTA sharing every K/V block, reading K/V straight out of the paged cache.
//
// Work item: two 128-row query tiles that share every K/V block. With an even number of query
// heads per KV head (head_pairs), tile A and tile B are the same 128 rows [128p, 128p + 128) of
// one prompt chunk for two query heads of one KV head, so both need the same key blocks and
// finish together; otherwise tile A is rows [256p, 256p + 128) of one query head and tile B the
// next 128 rows (absent past the chunk's end), and tile A needs up to two fewer key blocks.
// A chunk may follow ctx cached tokens: its rows sit at positions ctx.. and see keys
// [0, ctx + row]. Persistent: one
// CTA per SM walks its share of the items (heaviest first, alternate rounds reversed) with
// TMEM, barriers and the K/V ring carried from item to item, so the next item's Q and K/V
// loads and first S MMAs run while the softmax warps write the current item's output. 11 warps:
//   warp 0      TMA: both Q tiles once (two 64-column halves each, 128B swizzle), then per
//               64-key block the K and V rows of its four 16-token pages into a 4-stage ring;
//               a block's page ids are read from the block table one block ahead of its
//               copies, and the next item's Q is requested into L2 while the current item runs
//   warps 1, 2  MMA issue for tile A and tile B (warp 1 also allocates all 512 TMEM columns):
//               one lane issues, per block, S = Q K^T (M=128, N=64, K=128; double-buffered)
//               ahead of O += P V (M=128, N=128, K=64, bf16 operands: P read from TMEM, where
//               the softmax warps left it over its S, as a high and a low part, two MMAs; V an
//               MN-major operand in the cache's own row layout); each tile's pipeline waits
//               only on its own softmax, and a K/V stage is released when both tiles' MMAs
//               that read it have completed
//   warps 3-6   softmax of tile A, warps 7-10 softmax of tile B: one thread per query row
//               (tcgen05.ld of its S row, causal/length mask only on blocks that cross the
//               diagonal or the chunk end, online softmax in the log2 domain with a running
//               max allowed to lag by up to 2^8 -- O is rescaled in TMEM only past that --, P
//               split into bf16 high + low parts (about 17 significant bits) and stored by
//               tcgen05.st over the S columns it came from), then O / l from TMEM to global
//               memory.
// While one tile's softmax warps work, the tensor core runs the other tile's MMAs, and each
// K/V block is loaded once for both tiles. Where tile A needs fewer keys than tile B (row
// pairs), its last blocks are skipped. An S buffer is refilled only after the P V that read the P
// stored over it has completed. Between items, Q is reloaded once the last S MMA of the item
// has completed (q_empty), and a tile's first P V of the next item waits until its O has been
// read out of TMEM (o_empty). FP8 cache: the K/V pools hold the e4m3 codes as (exact) bf16
// values; the TMA warp also brings each block's 64 key and 64 value scales into the stage,
// and the softmax multiplies each score by its key's scale and each P by its value's scale
// (float32) before the split, so K and V enter as code x scale without a bf16 rounding of
// the product. All mbarrier waits are bounded; on a timeout the CTA flags kStatusTimeout,
// drains its own TMA copies and MMAs, frees TMEM and exits.
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
constexpr int BQ = 128;         // query rows per tile
constexpr int BKV = 64;         // keys per block (4 pages)
constexpr int KV_STAGES = 4;
constexpr int THREADS = 352;
constexpr int SOFTMAX_WARP0 = 3;
constexpr int Q_BYTES = BQ * D * 2;            // 32 KB per tile (two 16 KB halves)
constexpr int KV_HALF = BKV * 64 * 2;          // 8 KB: 64 keys x 64 dims
constexpr int K_BYTES = 2 * KV_HALF;           // 16 KB
constexpr int STAGE_BYTES = 2 * K_BYTES;       // K + V
constexpr int SCALE_BYTES = 2 * BKV * 4;       // FP8 cache: the block's key scales, then value scales
constexpr int TMEM_COLS = 512;                 // S_A: 0, 64; S_B: 128, 192; O_A: 256; O_B: 384
constexpr int P_LO_COL = 32;                   // P over S: high parts in columns 0-31, low parts 32-63
constexpr int O_COL = 256;
constexpr float kStaleMax = 8.f;               // log2 headroom before O is rescaled

struct Ctrl {
  uint64_t q_full, q_empty, kv_full[KV_STAGES], kv_empty[KV_STAGES];
  uint64_t s_full[2][2], p_full[2][2], pv_done[2][2], fin[2];  // [tile][buffer]
  uint64_t o_empty[2];                                                     // [tile]
  uint32_t tmem_base;
  int abort;
  int pending[KV_STAGES + 1];
};
constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + KV_STAGES * (STAGE_BYTES + SCALE_BYTES) + (int)sizeof(Ctrl);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);  // Q (K-major) x K (K-major)
constexpr uint32_t IDESC_O = make_idesc(BQ, D, false, true);  // P (TMEM) x V (MN-major), bf16

// One work item: tile A (query head h, rows q0a..) and tile B (head hb, rows q0b..) of one chunk.
struct Item {
  int s, h, hb, seq0, n, c0, nk, q0a, q0b, nblk_a, nblk_b, nblk;
  bool has_b;
};

// This CTA's it-th item. Items are (tile, head) or (tile, head pair) pairs, tile-major over the
// tile list (sorted heaviest first), so consecutive items share their K/V rows in L2; CTA c
// takes item c of every round of gridDim.x items, counted from the other end in odd rounds, so
// every CTA gets a similar total. False past the last item.
__device__ __forceinline__ bool item_at(int it, const int* __restrict__ tiles, int n_items, int n_q,
                                        const int* __restrict__ cu, const int* __restrict__ ctx, Item& I,
                                        bool head_pairs) {
  const int G = gridDim.x, c = blockIdx.x;
  const long long w = (long long)it * G + ((it & 1) ? (G - 1 - c) : c);
  if (w >= n_items) return false;
  // head_pairs: items are (128-row tile, two query heads of one KV head), both tiles on the
  // same rows; else (256-row tile pair, one query head)
  const int per = head_pairs ? n_q / 2 : n_q;
  const int tile = tiles[w / per];
  const int k = (int)(w % per);
  I.s = tile >> 16;
  const int qp = tile & 0xffff;
  I.seq0 = cu[I.s];
  I.n = cu[I.s + 1] - I.seq0;
  // the chunk's rows sit at positions c0.. after c0 cached keys; keys [0, nk) are visible
  I.c0 = ctx ? ctx[I.s] : 0;
  I.nk = I.c0 + I.n;
  if (head_pairs) {
    I.h = 2 * k;
    I.hb = 2 * k + 1;
    I.q0a = I.q0b = qp * BQ;
    I.has_b = true;
  } else {
    I.h = I.hb = k;
    I.q0a = qp * 2 * BQ;
    I.q0b = I.q0a + BQ;
    I.has_b = I.q0b < I.n;
  }
  I.nblk_a = (min(I.nk, I.c0 + I.q0a + BQ) + BKV - 1) / BKV;
  I.nblk_b = I.has_b ? (min(I.nk, I.c0 + I.q0b + BQ) + BKV - 1) / BKV : 0;
  I.nblk = I.has_b ? I.nblk_b : I.nblk_a;  // blocks loaded (tile B's range covers tile A's)
  return true;
}

__global__ void __launch_bounds__(THREADS, 1) attn_tc2_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const float* __restrict__ kscale, const float* __restrict__ vscale,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ cu,
    const int* __restrict__ ctx, const int* __restrict__ tiles, int n_items, int n_q, int n_kv,
    bf16* __restrict__ out, int ldo, float scale_log2, int* status, bool head_pairs) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t sQ = smem_u32(smem);  // tile t at sQ + t * Q_BYTES
  const uint32_t sKV = sQ + 2 * Q_BYTES;
  const uint32_t sScale = sKV + KV_STAGES * STAGE_BYTES;  // stage s at sScale + s * SCALE_BYTES
  const float* sScale_gen = reinterpret_cast<const float*>(smem + 2 * Q_BYTES + KV_STAGES * STAGE_BYTES);
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + 2 * Q_BYTES + KV_STAGES * (STAGE_BYTES + SCALE_BYTES));
  const bool fp8 = kscale != nullptr;
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pool_rows = num_pages * n_kv * kPageSize;
  const int group = n_q / n_kv;

  auto bar = [&](uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    mbar_init(bar(ctl->q_full), 1);
    mbar_init(bar(ctl->q_empty), 2);  // both tiles' last S MMA of the item
    for (int i = 0; i < KV_STAGES; ++i) {
      mbar_init(bar(ctl->kv_full[i]), 1);
      mbar_init(bar(ctl->kv_empty[i]), 2);  // both tiles' MMAs done with the stage
      ctl->pending[i] = -1;
    }
    ctl->pending[KV_STAGES] = -1;
    for (int t = 0; t < 2; ++t) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(ctl->s_full[t][i]), 1);
        mbar_init(bar(ctl->p_full[t][i]), 128);
        mbar_init(bar(ctl->pv_done[t][i]), 1);
      }
      mbar_init(bar(ctl->o_empty[t]), 128);
    }
    mbar_init(bar(ctl->fin[0]), 1);
    mbar_init(bar(ctl->fin[1]), 1);
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
  Item I;

  if (warp == 0) {
    if (lane == 0) {
      // Page ids of block j of item X, read from the block table one block ahead of that
      // block's copies, so the reads' latency hides behind the copies of the block before
      auto block_pages = [&](const Item& X, int j, int* pg) {
#pragma unroll
        for (int p = 0; p < BKV / kPageSize; ++p) {
          const int key = j * BKV + p * kPageSize;
          pg[p] = key < X.nk ? bt[(size_t)X.s * max_pages + (key >> 4)] : -1;
        }
      };
      int kv_i = 0;  // K/V blocks loaded so far (all items): ring stage and phase
      bool ok = true;
      bool have = item_at(0, tiles, n_items, n_q, cu, ctx, I, head_pairs);
      int pg[BKV / kPageSize], pgn[BKV / kPageSize];
#pragma unroll
      for (int p = 0; p < BKV / kPageSize; ++p) pg[p] = pgn[p] = -1;
      if (have) block_pages(I, 0, pg);
      for (int it = 0; ok && have; ++it) {
        const int kvh = I.h / group;
        // Q of this item overwrites the previous item's, once its last S MMA has completed
        if (it > 0 && !mbar_wait(bar(ctl->q_empty), (uint32_t)((it - 1) & 1), abort_flag)) break;
        // Q: rows seq0 + q0 .. +127 of this head's 128 columns per tile (rows past the chunk
        // are masked later; rows past the tensor read zeros)
        mbar_expect_tx(bar(ctl->q_full), (I.has_b ? 2 : 1) * Q_BYTES);
        ctl->pending[KV_STAGES] = it & 1;
        for (int t = 0; t < (I.has_b ? 2 : 1); ++t) {
          const int row = I.seq0 + (t ? I.q0b : I.q0a);
          const int hq = t ? I.hb : I.h;
          tma_load_2d(sQ + t * Q_BYTES, &tmQ, hq * D, row, bar(ctl->q_full));
          tma_load_2d(sQ + t * Q_BYTES + Q_BYTES / 2, &tmQ, hq * D + 64, row, bar(ctl->q_full));
        }
        Item N;
        const bool have_next = item_at(it + 1, tiles, n_items, n_q, cu, ctx, N, head_pairs);
        for (int j = 0; j < I.nblk; ++j, ++kv_i) {
          const int stage = kv_i % KV_STAGES;
          const uint32_t phase = (uint32_t)((kv_i / KV_STAGES) & 1);
          if (j + 1 < I.nblk) {
            block_pages(I, j + 1, pgn);
          } else if (have_next) {
            block_pages(N, 0, pgn);
          }
          if (!mbar_wait(bar(ctl->kv_empty[stage]), phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(ctl->kv_full[stage]), STAGE_BYTES + (fp8 ? SCALE_BYTES : 0));
          ctl->pending[stage] = (int)phase;
          const uint32_t sk = sKV + stage * STAGE_BYTES, sv = sk + K_BYTES;
#pragma unroll
          for (int p = 0; p < BKV / kPageSize; ++p) {
            const int page = pg[p];
            const bool valid = page >= 0 && page < num_pages;
            // a page outside the pool reads rows past the tensor's end: TMA fills zeros
            const int row = valid ? (page * n_kv + kvh) * kPageSize : pool_rows;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              tma_load_2d(sk + hf * KV_HALF + p * 2048, &tmK, hf * 64, row, bar(ctl->kv_full[stage]));
              tma_load_2d(sv + hf * KV_HALF + p * 2048, &tmV, hf * 64, row, bar(ctl->kv_full[stage]));
            }
            if (fp8) {  // the page's 16 key and 16 value scales (page 0's for a page outside the pool)
              const size_t srow = valid ? (size_t)row : (size_t)kvh * kPageSize;
              const uint32_t ss = sScale + stage * SCALE_BYTES + p * kPageSize * 4;
              bulk_load(ss, kscale + srow, kPageSize * 4, bar(ctl->kv_full[stage]));
              bulk_load(ss + BKV * 4, vscale + srow, kPageSize * 4, bar(ctl->kv_full[stage]));
            }
          }
#pragma unroll
          for (int p = 0; p < BKV / kPageSize; ++p) pg[p] = pgn[p];
          // the next item's Q into L2 while this item runs, so its load after q_empty is short
          // (after the second block, by when the next item's descriptor reads have returned)
          if (j == min(1, I.nblk - 1) && have_next) {
            for (int t = 0; t < (N.has_b ? 2 : 1); ++t) {
              const int row = N.seq0 + (t ? N.q0b : N.q0a);
              const int hq = t ? N.hb : N.h;
              tma_prefetch_l2_2d(&tmQ, hq * D, row);
              tma_prefetch_l2_2d(&tmQ, hq * D + 64, row);
            }
          }
        }
        I = N;
        have = have_next;
      }
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      // tile t's MMAs. Counters over all items: K/V blocks, S/P blocks of this tile, items
      // that used this tile's O
      const int t = warp - 1;
      int kv_base = 0, sp = 0, oi = 0;
      bool ok = true;
      for (int it = 0; ok && item_at(it, tiles, n_items, n_q, cu, ctx, I, head_pairs); ++it) {
        const int nb = t ? I.nblk_b : I.nblk_a;  // blocks this tile reads (0: no tile B)
        // Releases block j's K/V stage for a block this tile does not read. The arrival counts
        // toward that block's phase only once the block has been loaded (kv_full), so it can
        // never complete an earlier phase the other tile's MMAs still depend on.
        auto release_unread = [&](int j) -> bool {
          const int kv = kv_base + j, st = kv % KV_STAGES;
          if (!mbar_wait(bar(ctl->kv_full[st]), (uint32_t)((kv / KV_STAGES) & 1), abort_flag)) return false;
          ctl->pending[st] = -1;
          mbar_arrive(bar(ctl->kv_empty[st]));
          return true;
        };
        // this item's Q has been loaded, so the previous item's q_empty phase has completed
        if (!mbar_wait(bar(ctl->q_full), (uint32_t)(it & 1), abort_flag)) break;
        ctl->pending[KV_STAGES] = -1;
        if (nb == 0) {  // no tile B in this item: release its Q and K/V stages
          mbar_arrive(bar(ctl->q_empty));
          for (int j = 0; ok && j < I.nblk; ++j) ok = release_unread(j);
          kv_base += I.nblk;
          continue;
        }
        auto issue_s = [&](int j) -> bool {
          const int kv = kv_base + j, st = kv % KV_STAGES;
          if (!mbar_wait(bar(ctl->kv_full[st]), (uint32_t)((kv / KV_STAGES) & 1), abort_flag)) return false;
          ctl->pending[st] = -1;
          const int g = sp + j, sb = g & 1;
          // the buffer holds P of block g - 2 until the P V that reads it has completed
          if (g >= 2 && !mbar_wait(bar(ctl->pv_done[t][sb]), (uint32_t)(((g - 2) >> 1) & 1), abort_flag))
            return false;
          tc_fence_after();
          const uint32_t sk = sKV + st * STAGE_BYTES;
          const uint32_t q = sQ + t * Q_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (Q_BYTES / 2) + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * KV_HALF + (kk & 3) * 32;
            tc_mma(tmem + t * 128 + sb * BKV, sdesc(q + off), sdesc(sk + koff), IDESC_S, kk != 0);
          }
          tc_commit(bar(ctl->s_full[t][sb]));
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int g = sp + j, pb = g & 1;
          if (!mbar_wait(bar(ctl->p_full[t][pb]), (uint32_t)((g >> 1) & 1), abort_flag)) return false;
          // the first P V of an item overwrites O: the previous item's output must have left TMEM
          if (j == 0 && oi > 0 && !mbar_wait(bar(ctl->o_empty[t]), (uint32_t)((oi - 1) & 1), abort_flag))
            return false;
          tc_fence_after();
          const int st = (kv_base + j) % KV_STAGES;
          const uint32_t sv = sKV + st * STAGE_BYTES + K_BYTES;
          const uint32_t pcol = tmem + t * 128 + pb * BKV;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            // P: 16 keys = 8 TMEM columns per MMA (high part, then low part); V: MN-major,
            // 64-dim halves 8 KB apart, 8-key groups 1 KB apart
            const uint64_t vdesc = sdesc_sw128(sv + kk * 2048, KV_HALF, 1024);
            tc_mma_ts(tmem + O_COL + t * 128, pcol + kk * 8, vdesc, IDESC_O, (j | kk) != 0);
            tc_mma_ts(tmem + O_COL + t * 128, pcol + P_LO_COL + kk * 8, vdesc, IDESC_O, 1);
          }
          tc_commit(bar(ctl->pv_done[t][pb]));
          tc_commit(bar(ctl->kv_empty[st]));
          return true;
        };
        // q_empty is committed after this tile's last S MMA of the item, so the next item's Q
        // can load while this item's P V and softmax finish
        ok = issue_s(0);
        if (ok && nb == 1) tc_commit(bar(ctl->q_empty));
        for (int j = 0; ok && j < nb; ++j) {
          // S of the next block first, so the tensor core has work while the softmax warps
          // turn this block's S into P
          if (j + 1 < nb) {
            if (!(ok = issue_s(j + 1))) break;
            if (j + 2 == nb) tc_commit(bar(ctl->q_empty));
          }
          if (!(ok = issue_pv(j))) break;
        }
        // blocks of the item past this tile's last (tile A needs fewer keys than tile B)
        for (int j = nb; ok && j < I.nblk; ++j) ok = release_unread(j);
        kv_base += I.nblk;
        sp += nb;
        oi += 1;
      }
    }
  } else {
    // softmax / output warps of tile t: thread <-> query row. O accumulates in TMEM across
    // blocks; the probabilities use a running max that may lag the true one by up to
    // 2^kStaleMax (they then stay <= 256); only when a row's max moves further is O
    // rescaled, by the warp, in TMEM, after the previous block's P V has landed.
    const int t = (warp - SOFTMAX_WARP0) >> 2;
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t s_col = t * 128, o_col = O_COL + t * 128;
    auto wait_pv = [&](int g) -> bool {
      return mbar_wait(bar(ctl->pv_done[t][g & 1]), (uint32_t)((g >> 1) & 1), abort_flag);
    };
    int sp = 0;   // S/P blocks of this tile over all items
    int kvb = 0;  // K/V blocks over all items (ring stage of block j: (kvb + j) % KV_STAGES)
    bool ok = true;
    for (int it = 0; ok && item_at(it, tiles, n_items, n_q, cu, ctx, I, head_pairs); kvb += I.nblk, ++it) {
      if (t == 1 && !I.has_b) continue;
      const int nb = t ? I.nblk_b : I.nblk_a;
      const int q0 = t ? I.q0b : I.q0a;
      const int qrow = q0 + r;       // row within the chunk
      const int qpos = I.c0 + qrow;  // its position
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nb; ++j) {
        const int g = sp + j, sb = g & 1;
        if (!mbar_wait(bar(ctl->s_full[t][sb]), (uint32_t)((g >> 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sc[BKV];
        tmem_ld64(tmem + lane_off + s_col + sb * BKV, sc);
        const float* kvs = nullptr;  // FP8: this block's key scales, then value scales
        if (fp8) {
          // the stage's scales arrived with its K/V (kv_full); wait on it directly so their
          // shared-memory writes are visible to this thread (the phase has long completed)
          const int kv = kvb + j, st = kv % KV_STAGES;
          if (!mbar_wait(bar(ctl->kv_full[st]), (uint32_t)((kv / KV_STAGES) & 1), abort_flag)) {
            ok = false;
            break;
          }
          kvs = sScale_gen + st * (SCALE_BYTES / 4);
#pragma unroll
          for (int i = 0; i < BKV; ++i) sc[i] *= kvs[i];
        }
        const bool interior = (j + 1) * BKV - 1 <= I.c0 + q0 && (j + 1) * BKV <= I.nk;  // no key masked in any row
        if (!interior) {
#pragma unroll
          for (int i = 0; i < BKV; ++i) {
            const int key = j * BKV + i;
            if (key > qpos || key >= I.nk) sc[i] = -INFINITY;
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
            if (!wait_pv(g - 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D; c += 32) {
              float v[32];
              tmem_ld32(tmem + lane_off + o_col + c, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= factor;
              tmem_st32(tmem + lane_off + o_col + c, v);
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
          tmem_st64(tmem + lane_off + s_col + sb * BKV, pw);
        }
        tc_fence_before();
        mbar_arrive(bar(ctl->p_full[t][sb]));
      }
      if (ok) ok = wait_pv(sp + nb - 1);
      if (ok) {
        tc_fence_after();
        const float inv = 1.f / l;
        bf16* dst = out + (size_t)(I.seq0 + min(qrow, I.n - 1)) * ldo + (t ? I.hb : I.h) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float v[32];
          tmem_ld32(tmem + lane_off + o_col + c, v);
          if (qrow < I.n) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 u;
              u.x = pack_bf16(v[e] * inv, v[e + 1] * inv);
              u.y = pack_bf16(v[e + 2] * inv, v[e + 3] * inv);
              u.z = pack_bf16(v[e + 4] * inv, v[e + 5] * inv);
              u.w = pack_bf16(v[e + 6] * inv, v[e + 7] * inv);
              *reinterpret_cast<uint4*>(dst + c + e) = u;
            }
          }
        }
        // O has left TMEM: the next item's first P V may overwrite it
        tc_fence_before();
        mbar_arrive(bar(ctl->o_empty[t]));
      }
      sp += nb;
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
    if (threadIdx.x == 32 || threadIdx.x == 64) {  // MMAs each issuing thread has in flight
      const uint32_t f = bar(ctl->fin[threadIdx.x == 64]);
      tc_commit(f);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(f, 0) && global_ns() - t0 < kTimeoutNs) {
      }
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace

cudaError_t launch_attention_prefill_tc2(const bf16* q, int ldq, int T, const bf16* k_pool, const bf16* v_pool,
                                         const float* k_scale, const float* v_scale,
                                         const int* block_table, int max_pages, int num_pages, const int* cu,
                                         const int* ctx, const int* tiles, int num_tiles, int n_q, int n_kv,
                                         int d_head, bf16* out, int ldo, int num_sms, int* status,
                                         cudaStream_t stream, bool head_pairs) {
  if (num_tiles <= 0) return cudaSuccess;
  // a head pair shares its KV head only when the group size is even
  if (head_pairs && (n_kv < 1 || n_q % n_kv || (n_q / n_kv) % 2)) return cudaErrorNotSupported;
  if (d_head != D || (reinterpret_cast<uintptr_t>(q) & 15) || ldq % 8 || num_sms < 1 || (!k_scale != !v_scale) ||
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
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_tc2_kernel), SMEM_BYTES, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const int n_items = num_tiles * (head_pairs ? n_q / 2 : n_q);
  attn_tc2_kernel<<<n_items < num_sms ? n_items : num_sms, THREADS, SMEM_BYTES, stream>>>(
      mq, mk, mv, k_scale, v_scale, block_table, max_pages, num_pages, cu, ctx, tiles, n_items, n_q, n_kv, out, ldo,
      scale_log2, status, head_pairs);
  return cudaGetLastError();
}

}  // namespace skv
