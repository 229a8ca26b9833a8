// Single-row GQA attention over the paged KV cache, split along the keys: decode tokens,
// the last token of each prompt in the SwiftKV tail, and rows of short chunks.
//
// The work is a list of items v = (unit, KV head), a unit being keys [k0, k0 + split) of row
// b (split 128 for rows of up to 1024 keys, else 256), so a long context is spread over
// many warps and short and long rows mix without stragglers; the split depends on the row's
// own length only, so no row's arithmetic depends on the batch. One CTA of 4 warps per SM; each warp walks its
// own items (v = global warp, + all warps, ...) one 16-key page at a time. Each (page, KV
// head) block is 16*d_head*2 contiguous bytes in the pool; the warp stages K and V (and,
// with an item's first page, its G query rows) with cp.async into a 3-slot ring of
// XOR-swizzled shared-memory tiles that runs ahead across item boundaries, so HBM reads
// stay in flight while it computes (7 warps per SM). The G = n_q/n_kv <= 8 query heads of
// the group are rows of an mma.sync m16n8k16 A operand (the other rows are zero), so one
// read of each K/V row serves the whole group: S = Q K^T (bf16, fp32 accumulate), online
// softmax in the log2 domain (O rescaled only when a row's running max moves), O += P V
// with V in bf16 and P as the sum of its bf16 high and low parts (about 16 significant
// bits), fp32 accumulate.
// An item that covers its whole row writes the output; otherwise it writes (max, sum,
// unnormalised O) per head and attn_split_combine merges the splits in order. No CTA-wide
// synchronisation at all.
#include <algorithm>
#include <cfloat>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "pdl.cuh"

namespace skv {

namespace {

constexpr int SW = 7;        // warps per CTA (one CTA per SM; 3 ring slots of 10 KB each fit 7)
constexpr int SSTAGES = 3;   // ring slots per warp
constexpr int SMAXG = 8;     // query heads per KV head (rows 0..7 of the mma A operand)

template <int D>
struct Sp {
  static constexpr int PAGE = kPageSize * D;      // elements of one (page, head) K or V block
  static constexpr int STAGE = 2 * PAGE + SMAXG * D;  // K, V, and the unit's Q when the page is its first
  static constexpr int SMEM = SW * SSTAGES * STAGE * 2;
};

template <int D>
__global__ void __launch_bounds__(SW * 32, 1) attn_split_kernel(
    const bf16* __restrict__ q, int ldq, const bf16* __restrict__ kpool, const bf16* __restrict__ vpool,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ qpos,
    const int* __restrict__ rows, const int* __restrict__ seqs, const int* __restrict__ units, int num_units,
    int n_q, int n_kv, bf16* __restrict__ out, int ldo, float* __restrict__ part, float scale_log2) {
  using S = Sp<D>;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) unsigned char smem[];
  griddep_launch_dependents();  // a programmatic dependent may start as these blocks leave
  griddep_wait();               // itself launched as one: q and the cache rows are fresh
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bf16* ring = reinterpret_cast<bf16*>(smem) + (size_t)warp * SSTAGES * S::STAGE;
  const int G = n_q / n_kv;
  const int total = num_units * n_kv;              // work items v = unit * n_kv + head
  const int gw = blockIdx.x * SW + warp, nw = gridDim.x * SW;

  auto swz = [](int row, int ch) { return row * D + ((ch ^ (row & 7)) * 8); };
  struct Geo {
    int r, kvh, k_begin, k_end, p_begin, npages, nkeys;
    const int* btrow;
  };
  auto geo = [&](int v) {
    Geo g;
    const int u = v / n_kv;
    g.kvh = v - u * n_kv;
    const int b = units[3 * u];
    g.r = rows ? rows[b] : b;
    const int sq = seqs ? seqs[b] : b;
    g.nkeys = qpos[g.r] + 1;
    g.k_begin = units[3 * u + 1];
    g.k_end = min(g.nkeys, g.k_begin + units[3 * u + 2]);
    g.p_begin = g.k_begin / kPageSize;
    g.npages = (g.k_end + kPageSize - 1) / kPageSize - g.p_begin;
    g.btrow = bt + (size_t)sq * max_pages;
    return g;
  };

  // loader: walks this warp's (work item, page) sequence SSTAGES - 1 pages ahead of the compute
  int lv = gw, lp = 0, lslot = 0;
  Geo lg;
  if (lv < total) lg = geo(lv);
  auto issue = [&]() {
    if (lv < total) {
      bf16* st = ring + lslot * S::STAGE;
      const int page = lg.btrow[lg.p_begin + lp];
      const bool ok = page >= 0 && page < num_pages;
      const size_t base = ok ? ((size_t)page * n_kv + lg.kvh) * S::PAGE : 0;
#pragma unroll
      for (int c = lane; c < kPageSize * CH; c += 32) {
        const int row = c / CH, ch = c % CH;
        cp_async16(smem_u32(st + swz(row, ch)), kpool + base + row * D + ch * 8, ok ? 16 : 0);
        cp_async16(smem_u32(st + S::PAGE + swz(row, ch)), vpool + base + row * D + ch * 8, ok ? 16 : 0);
      }
      if (lp == 0) {  // the unit's query heads ride with its first page
        const bf16* qsrc = q + (size_t)lg.r * ldq + (size_t)lg.kvh * G * D;
        for (int c = lane; c < G * CH; c += 32) {
          const int row = c / CH, ch = c % CH;
          cp_async16(smem_u32(st + 2 * S::PAGE + swz(row, ch)), qsrc + row * D + ch * 8, 16);
        }
      }
      if (++lslot == SSTAGES) lslot = 0;
      if (++lp == lg.npages) {
        lp = 0;
        lv += nw;
        if (lv < total) lg = geo(lv);
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
  };

  // heads are A rows 0..7 (groupID); rows 8..15 stay zero and are never read back
  const int g0 = lane >> 2, qc = 2 * (lane & 3);
  uint32_t qf[D / 16][4];
  float o[D / 8][4];
  float m0 = -FLT_MAX, l0 = 0.f;

#pragma unroll
  for (int i = 0; i < SSTAGES - 1; ++i) issue();
  int cv = gw, cp = 0, cslot = 0;
  Geo cg;
  if (cv < total) cg = geo(cv);
  while (cv < total) {
    issue();
    cp_async_wait<SSTAGES - 1>();
    __syncwarp();
    bf16* st = ring + cslot * S::STAGE;
    const bf16* kb = st;
    bf16* vb = st + S::PAGE;
    if (cp == 0) {  // new unit: Q fragments (rows = heads, zero past G), fresh softmax state
      const bf16* qs = st + 2 * S::PAGE;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks * 16 + qc;
        auto qat = [&](int g, int col) -> uint32_t {  // g < 8
          return g < G ? *reinterpret_cast<const uint32_t*>(qs + swz(g, col / 8) + (col & 7)) : 0u;
        };
        qf[ks][0] = qat(g0, c);
        qf[ks][1] = 0u;
        qf[ks][2] = qat(g0, c + 8);
        qf[ks][3] = 0u;
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
      m0 = -FLT_MAX;
      l0 = 0.f;
    }

    // S = Q K^T for the page's 16 keys: two n-tiles of 8 keys
    float sc[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[t][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t b0[2], b1[2];
      const int row = (lane & 7) + ((lane >> 4) << 3);
      const int ch = ks * 2 + ((lane >> 3) & 1);
      ldmatrix_x4(smem_u32(kb + swz(row, ch)), b0[0], b0[1], b1[0], b1[1]);
      mma_bf16_16816(sc[0], qf[ks], b0);
      mma_bf16_16816(sc[1], qf[ks], b1);
    }
    const int pg = cg.btrow[cg.p_begin + cp];
    const bool page_ok = pg >= 0 && pg < num_pages;
    const int key0 = (cg.p_begin + cp) * kPageSize;
    float mx0 = -FLT_MAX;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + 8 * t + qc + e;
        const bool valid = page_ok && key >= cg.k_begin && key < cg.k_end;
        sc[t][e] = valid ? sc[t][e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, sc[t][e]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    if (__any_sync(0xffffffffu, mx0 > m0)) {  // O and l rescale only when some row's max moves
      const float mn0 = fmaxf(m0, mx0);
      const float al0 = exp2f(m0 - mn0);
      m0 = mn0;
      l0 *= al0;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
      }
    }
    float ps0 = 0.f;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[t][e] = exp2f(sc[t][e] - m0);
        ps0 += sc[t][e];
      }
    l0 += ps0;
    // O += P V with V in bf16 straight from the cache: P (heads x 16 keys, the S accumulator
    // re-packed as an A operand) is split into bf16 high and low parts, P = hi + lo to about
    // 16 significant bits, and both are multiplied (fp32 accumulate)
    uint32_t ph[4], pl[4];
    {
      float hi[4], lo[4];
      const float p4[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hi[i] = __bfloat162float(__float2bfloat16_rn(p4[i]));
        lo[i] = p4[i] - hi[i];
      }
      ph[0] = pack_bf16(hi[0], hi[1]);
      ph[2] = pack_bf16(hi[2], hi[3]);
      pl[0] = pack_bf16(lo[0], lo[1]);
      pl[2] = pack_bf16(lo[2], lo[3]);
      ph[1] = ph[3] = pl[1] = pl[3] = 0u;
    }
#pragma unroll
    for (int dp = 0; dp < D / 16; ++dp) {
      uint32_t b0[2], b1[2];
      ldmatrix_x4_trans(smem_u32(vb + swz(lane & 15, dp * 2 + (lane >> 4))), b0[0], b0[1], b1[0], b1[1]);
      mma_bf16_16816(o[2 * dp], ph, b0);
      mma_bf16_16816(o[2 * dp + 1], ph, b1);
      mma_bf16_16816(o[2 * dp], pl, b0);
      mma_bf16_16816(o[2 * dp + 1], pl, b1);
    }
    __syncwarp();  // the slot is refilled by a later issue()
    if (++cslot == SSTAGES) cslot = 0;

    if (++cp == cg.npages) {
      // unit done: the whole row -> output; one split of it -> (max, sum, unnormalised O)
      float s0 = l0;
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      const bool whole = cg.k_begin == 0 && cg.k_end == cg.nkeys;
      const int u = cv / n_kv;
      if (whole) {
        const float i0 = s0 > 0.f ? 1.f / s0 : 0.f;
        bf16* orow = out + (size_t)cg.r * ldo + (size_t)cg.kvh * G * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          const int dim = n * 8 + qc;
          if (g0 < G) *reinterpret_cast<uint32_t*>(orow + g0 * D + dim) = pack_bf16(o[n][0] * i0, o[n][1] * i0);
        }
      } else {
        float* pp = part + ((size_t)u * n_kv + cg.kvh) * G * (D + 2);
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          const int dim = n * 8 + qc;
          if (g0 < G) *reinterpret_cast<float2*>(pp + g0 * (D + 2) + 2 + dim) = make_float2(o[n][0], o[n][1]);
        }
        if ((lane & 3) == 0) {
          if (g0 < G) *reinterpret_cast<float2*>(pp + g0 * (D + 2)) = make_float2(m0, s0);
        }
      }
      cp = 0;
      cv += nw;
      if (cv < total) cg = geo(cv);
    }
  }
  cp_async_wait<0>();
}

// FP8 cache variant of attn_split_kernel: pages hold e4m3 codes (16*d_head bytes per
// (page, head) block) and one float32 scale per key row. The ring stages K codes, V codes,
// both scale rows and the unit's Q. S: the K codes go to the tensor core without a
// shared-memory pass -- ldmatrix reads a 16-dim slice of 8 keys as 8 two-code elements, so a
// thread receives 4 consecutive dims of one key, converted (exactly) to f16; Q's fragments
// are built with the same dim order, so the dot products are unchanged -- with f16 Q,
// fp32 accumulate, then each score times its key's scale. P V: ldmatrix.trans on the V
// codes gives a thread two keys x two adjacent dims; byte permutes split them into an
// even-dim and an odd-dim fragment (exact f16). V's per-key scale rides on P: P' = p *
// s_v / S_ref in f16, S_ref the largest V scale seen so far in the unit (O is rescaled
// when it grows, like the softmax max), and O * S_ref is the unnormalised output.
constexpr int SSTAGES8 = 3;

template <int D>
struct Sp8 {
  static constexpr int CODES = kPageSize * D;        // bytes of one (page, head) K or V block
  static constexpr int QB = SMAXG * D * 2;            // bytes of the unit's query rows (bf16)
  static constexpr int STAGE = 2 * CODES + 2 * kPageSize * 4 + QB;
  static constexpr int SMEM = SW * SSTAGES8 * STAGE;
  static constexpr int CHB = D / 16;                  // 16-byte chunks per code row
};

template <int D>
__global__ void __launch_bounds__(SW * 32, 1) attn_split_fp8_kernel(
    const bf16* __restrict__ q, int ldq, const uint8_t* __restrict__ kpool, const uint8_t* __restrict__ vpool,
    const float* __restrict__ kscale, const float* __restrict__ vscale, const int* __restrict__ bt, int max_pages,
    int num_pages, const int* __restrict__ qpos, const int* __restrict__ rows, const int* __restrict__ seqs,
    const int* __restrict__ units, int num_units, int n_q, int n_kv, bf16* __restrict__ out, int ldo,
    float* __restrict__ part, float scale_log2) {
  using S = Sp8<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* ring = smem + (size_t)warp * SSTAGES8 * S::STAGE;
  const int G = n_q / n_kv;
  const int total = num_units * n_kv;
  const int gw = blockIdx.x * SW + warp, nw = gridDim.x * SW;

  // code rows of D bytes, 16-byte chunks XOR-swizzled so 8 rows of one chunk hit 8 bank groups
  auto swzb = [](int row, int ch) {
    const int sel = D == 128 ? (row & 7) : ((row >> 1) & 3);
    return row * D + ((ch ^ sel) << 4);
  };
  auto swzq = [](int row, int ch) { return row * D + ((ch ^ (row & 7)) * 8); };  // bf16 elements
  struct Geo {
    int r, kvh, k_begin, k_end, p_begin, npages, nkeys;
    const int* btrow;
  };
  auto geo = [&](int v) {
    Geo g;
    const int u = v / n_kv;
    g.kvh = v - u * n_kv;
    const int b = units[3 * u];
    g.r = rows ? rows[b] : b;
    const int sq = seqs ? seqs[b] : b;
    g.nkeys = qpos[g.r] + 1;
    g.k_begin = units[3 * u + 1];
    g.k_end = min(g.nkeys, g.k_begin + units[3 * u + 2]);
    g.p_begin = g.k_begin / kPageSize;
    g.npages = (g.k_end + kPageSize - 1) / kPageSize - g.p_begin;
    g.btrow = bt + (size_t)sq * max_pages;
    return g;
  };

  int lv = gw, lp = 0, lslot = 0;
  Geo lg;
  if (lv < total) lg = geo(lv);
  auto issue = [&]() {
    if (lv < total) {
      unsigned char* st = ring + lslot * S::STAGE;
      const int page = lg.btrow[lg.p_begin + lp];
      const bool ok = page >= 0 && page < num_pages;
      const size_t blk = ok ? (size_t)page * n_kv + lg.kvh : 0;
#pragma unroll
      for (int c = lane; c < kPageSize * S::CHB; c += 32) {
        const int row = c / S::CHB, ch = c % S::CHB;
        cp_async16(smem_u32(st + swzb(row, ch)), kpool + blk * S::CODES + row * D + ch * 16, ok ? 16 : 0);
        cp_async16(smem_u32(st + S::CODES + swzb(row, ch)), vpool + blk * S::CODES + row * D + ch * 16, ok ? 16 : 0);
      }
      if (lane < 8) {  // 16 K scales, then 16 V scales
        const float* sp = (lane < 4 ? kscale : vscale) + blk * kPageSize + (lane & 3) * 4;
        cp_async16(smem_u32(st + 2 * S::CODES + lane * 16), sp, ok ? 16 : 0);
      }
      if (lp == 0) {
        const bf16* qsrc = q + (size_t)lg.r * ldq + (size_t)lg.kvh * G * D;
        bf16* qs = reinterpret_cast<bf16*>(st + 2 * S::CODES + 2 * kPageSize * 4);
        for (int c = lane; c < G * (D / 8); c += 32) {
          const int row = c / (D / 8), ch = c % (D / 8);
          cp_async16(smem_u32(qs + swzq(row, ch)), qsrc + row * D + ch * 8, 16);
        }
      }
      if (++lslot == SSTAGES8) lslot = 0;
      if (++lp == lg.npages) {
        lp = 0;
        lv += nw;
        if (lv < total) lg = geo(lv);
      }
    }
    cp_async_commit();
  };

  const int g0 = lane >> 2, qd = lane & 3;
  uint32_t qf[D / 16][4];
  float o[D / 8][4];
  float m0 = -FLT_MAX, l0 = 0.f, sref = 0.f;

#pragma unroll
  for (int i = 0; i < SSTAGES8 - 1; ++i) issue();
  int cv = gw, cp = 0, cslot = 0;
  Geo cg;
  if (cv < total) cg = geo(cv);
  while (cv < total) {
    issue();
    cp_async_wait<SSTAGES8 - 1>();
    __syncwarp();
    const unsigned char* st = ring + cslot * S::STAGE;
    const float* sk = reinterpret_cast<const float*>(st + 2 * S::CODES);
    const float* sv = sk + kPageSize;
    if (cp == 0) {  // Q in f16, dims 16ks + 4qd .. +3 of head g0 (the order the K codes arrive in)
      const bf16* qs = reinterpret_cast<const bf16*>(st + 2 * S::CODES + 2 * kPageSize * 4);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t lo = 0u, hi = 0u;
        if (g0 < G) {
          const uint2 w = *reinterpret_cast<const uint2*>(qs + swzq(g0, 2 * ks + (qd >> 1)) + 4 * (qd & 1));
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
          const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
          lo = pack_f16(a.x, a.y);
          hi = pack_f16(b.x, b.y);
        }
        qf[ks][0] = lo;
        qf[ks][1] = 0u;
        qf[ks][2] = hi;
        qf[ks][3] = 0u;
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
      m0 = -FLT_MAX;
      l0 = 0.f;
      sref = 0.f;
    }

    // S = Q K^T straight from the codes
    float sc[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[t][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      uint32_t r[4];
      const int row = (lane & 7) + ((lane >> 4) << 3);
      const int ch = ks + ((lane >> 3) & 1);
      ldmatrix_x4(smem_u32(st + swzb(row, ch)), r[0], r[1], r[2], r[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // k-steps ks, ks + 1
        uint32_t b0[2], b1[2];
        b0[0] = f16x2_from_e4m3x2(r[h] & 0xffffu);
        b0[1] = f16x2_from_e4m3x2(r[h] >> 16);
        b1[0] = f16x2_from_e4m3x2(r[2 + h] & 0xffffu);
        b1[1] = f16x2_from_e4m3x2(r[2 + h] >> 16);
        mma_f16_16816(sc[0], qf[ks + h], b0);
        mma_f16_16816(sc[1], qf[ks + h], b1);
      }
    }
    const int pg = cg.btrow[cg.p_begin + cp];
    const bool page_ok = pg >= 0 && pg < num_pages;
    const int key0 = (cg.p_begin + cp) * kPageSize;
    float mx0 = -FLT_MAX, vmax = 0.f;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kk = 8 * t + 2 * qd + e;
        const int key = key0 + kk;
        const bool valid = page_ok && key >= cg.k_begin && key < cg.k_end;
        sc[t][e] = valid ? sc[t][e] * sk[kk] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, sc[t][e]);
        if (valid) vmax = fmaxf(vmax, sv[kk]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    }
    // one rescale for both moving references: the softmax max (O and l) and S_ref (O)
    if (__any_sync(0xffffffffu, mx0 > m0 || vmax > sref)) {
      const float mn0 = fmaxf(m0, mx0), sn = fmaxf(sref, vmax);
      const float al0 = exp2f(m0 - mn0);
      const float fo = al0 * (sn > 0.f ? sref / sn : 1.f);
      m0 = mn0;
      l0 *= al0;
      sref = sn;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= fo;
        o[n][1] *= fo;
      }
    }
    const float isref = sref > 0.f ? 1.f / sref : 0.f;
    float ps0 = 0.f, pv[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p = exp2f(sc[t][e] - m0);
        ps0 += p;
        pv[t][e] = p * (sv[8 * t + 2 * qd + e] * isref);
      }
    l0 += ps0;
    uint32_t pa[4];
    pa[0] = pack_f16(pv[0][0], pv[0][1]);
    pa[1] = 0u;
    pa[2] = pack_f16(pv[1][0], pv[1][1]);
    pa[3] = 0u;
    // O += P' V: per 16-dim chunk c, an even-dim and an odd-dim n-tile (O column order:
    // chunk c holds dims 16c + 4qd + {0, 2} in n-tile 2c and 16c + 4qd + {1, 3} in 2c + 1)
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
      uint32_t r[4];
      ldmatrix_x4_trans(smem_u32(st + S::CODES + swzb(lane & 15, c + (lane >> 4))), r[0], r[1], r[2], r[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // chunks c, c + 1: keys 0-7 in r[2h], keys 8-15 in r[2h+1]
        uint32_t be[2], bo[2];
        be[0] = f16x2_from_e4m3x2(__byte_perm(r[2 * h], 0, 0x0020));
        bo[0] = f16x2_from_e4m3x2(__byte_perm(r[2 * h], 0, 0x0031));
        be[1] = f16x2_from_e4m3x2(__byte_perm(r[2 * h + 1], 0, 0x0020));
        bo[1] = f16x2_from_e4m3x2(__byte_perm(r[2 * h + 1], 0, 0x0031));
        mma_f16_16816(o[2 * (c + h)], pa, be);
        mma_f16_16816(o[2 * (c + h) + 1], pa, bo);
      }
    }
    __syncwarp();
    if (++cslot == SSTAGES8) cslot = 0;

    if (++cp == cg.npages) {
      float s0 = l0;
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      const bool whole = cg.k_begin == 0 && cg.k_end == cg.nkeys;
      const int u = cv / n_kv;
      if (g0 < G) {
        if (whole) {
          const float f = s0 > 0.f ? sref / s0 : 0.f;
          bf16* orow = out + (size_t)cg.r * ldo + (size_t)(cg.kvh * G + g0) * D;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint2 w;
            w.x = pack_bf16(o[2 * c][0] * f, o[2 * c + 1][0] * f);
            w.y = pack_bf16(o[2 * c][1] * f, o[2 * c + 1][1] * f);
            *reinterpret_cast<uint2*>(orow + 16 * c + 4 * qd) = w;
          }
        } else {
          float* pp = part + (((size_t)u * n_kv + cg.kvh) * G + g0) * (D + 2);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {  // (D + 2)-float records: 8-byte alignment only
            *reinterpret_cast<float2*>(pp + 2 + 16 * c + 4 * qd) = make_float2(o[2 * c][0] * sref, o[2 * c + 1][0] * sref);
            *reinterpret_cast<float2*>(pp + 4 + 16 * c + 4 * qd) = make_float2(o[2 * c][1] * sref, o[2 * c + 1][1] * sref);
          }
          if (qd == 0) *reinterpret_cast<float2*>(pp) = make_float2(m0, s0);
        }
      }
      cp = 0;
      cv += nw;
      if (cv < total) cg = geo(cv);
    }
  }
  cp_async_wait<0>();
}

// Merges the splits of every item that has more than one, per head in split order: the
// split weights 2^(m_u - max) are computed once into shared memory, then each output
// element sums its splits' unnormalised O four loads at a time.
constexpr int CMB_THREADS = 256;
constexpr int CMB_MAX_W = 4096;  // split weights held in shared memory (splits x heads)

template <int D>
__global__ void __launch_bounds__(CMB_THREADS) attn_split_combine(const int* __restrict__ rows,
                                                                  const int* __restrict__ ubeg, int n_q, int n_kv,
                                                                  const float* __restrict__ part,
                                                                  bf16* __restrict__ out, int ldo) {
  __shared__ float s_w[CMB_MAX_W];
  __shared__ float s_mx[SMAXG], s_den[SMAXG];
  griddep_launch_dependents();
  griddep_wait();  // launched as a programmatic dependent of the split kernel: its partials
  const int b = blockIdx.x, kvh = blockIdx.y;
  const int u0 = ubeg[b], ns = ubeg[b + 1] - u0;
  if (ns <= 1) return;  // written directly by its only unit
  const int r = rows ? rows[b] : b;
  const int G = n_q / n_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto pp = [&](int i, int g) { return part + (((size_t)(u0 + i) * n_kv + kvh) * G + g) * (D + 2); };
  const bool cached = ns * G <= CMB_MAX_W;
  // per head: running max over the splits, then (cached) weights and the denominator
  for (int g = warp; g < G; g += CMB_THREADS / 32) {
    float mx = -INFINITY;
    for (int i = lane; i < ns; i += 32) mx = fmaxf(mx, pp(i, g)[0]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float den = 0.f;
    for (int i0 = 0; i0 < ns; i0 += 32) {  // in split order: lane partials, then a fixed tree
      const int i = i0 + lane;
      float w = 0.f, l = 0.f;
      if (i < ns) {
        w = exp2f(pp(i, g)[0] - mx);
        l = pp(i, g)[1] * w;
        if (cached) s_w[i * G + g] = w;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      den += l;
    }
    if (lane == 0) {
      s_mx[g] = mx;
      s_den[g] = den;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += CMB_THREADS) {
    const int g = idx / D, dim = idx % D;
    const float mx = s_mx[g];
    float num = 0.f;
    int i = 0;
    for (; i + 4 <= ns; i += 4) {
      float v[4], w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        v[t] = pp(i + t, g)[2 + dim];
        w[t] = cached ? s_w[(i + t) * G + g] : exp2f(pp(i + t, g)[0] - mx);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) num += v[t] * w[t];
    }
    for (; i < ns; ++i) num += pp(i, g)[2 + dim] * (cached ? s_w[i * G + g] : exp2f(pp(i, g)[0] - mx));
    const float den = s_den[g];
    out[(size_t)r * ldo + (size_t)(kvh * G + g) * D + dim] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
  }
}

template <int D>
cudaError_t split_d(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool, const int* bt, int max_pages,
                    int num_pages, const int* qpos, const int* rows, const int* seqs, const SplitPlan& plan,
                    int n_q, int n_kv, bf16* out, int ldo, int num_sms, cudaStream_t stream) {
  constexpr int smem = Sp<D>::SMEM;
  static_assert(smem <= 227 * 1024, "rings must fit in shared memory");
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_split_kernel<D>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const int total = plan.num_units * n_kv;
  const int ctas = std::min((total + SW - 1) / SW, num_sms);
  cudaError_t e = launch_pdl(attn_split_kernel<D>, dim3(ctas), dim3(SW * 32), smem, stream, q, ldq, k_pool, v_pool,
                             bt, max_pages, num_pages, qpos, rows, seqs, (const int*)plan.units, plan.num_units, n_q,
                             n_kv, out, ldo, plan.part, scale_log2);
  if (e != cudaSuccess || !plan.any_split) return e;
  return launch_pdl(attn_split_combine<D>, dim3(plan.num_items, n_kv), dim3(CMB_THREADS), 0, stream, rows,
                    (const int*)plan.ubeg, n_q, n_kv, (const float*)plan.part, out, ldo);
}

template <int D>
cudaError_t split_fp8_d(const bf16* q, int ldq, const uint8_t* k8, const uint8_t* v8, const float* ks,
                        const float* vs, const int* bt, int max_pages, int num_pages, const int* qpos,
                        const int* rows, const int* seqs, const SplitPlan& plan, int n_q, int n_kv, bf16* out,
                        int ldo, int num_sms, cudaStream_t stream) {
  constexpr int smem = Sp8<D>::SMEM;
  static_assert(smem <= 227 * 1024, "rings must fit in shared memory");
  static_assert(Sp8<D>::STAGE % 16 == 0, "ring slots must keep 16-byte alignment");
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_split_fp8_kernel<D>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const int total = plan.num_units * n_kv;
  const int ctas = std::min((total + SW - 1) / SW, num_sms);
  cudaError_t e = launch_pdl(attn_split_fp8_kernel<D>, dim3(ctas), dim3(SW * 32), smem, stream, q, ldq, k8, v8, ks,
                             vs, bt, max_pages, num_pages, qpos, rows, seqs, (const int*)plan.units, plan.num_units,
                             n_q, n_kv, out, ldo, plan.part, scale_log2);
  if (e != cudaSuccess || !plan.any_split) return e;
  return launch_pdl(attn_split_combine<D>, dim3(plan.num_items, n_kv), dim3(CMB_THREADS), 0, stream, rows,
                    (const int*)plan.ubeg, n_q, n_kv, (const float*)plan.part, out, ldo);
}

}  // namespace

cudaError_t launch_attention_decode_split_fp8(const bf16* q, int ldq, const uint8_t* k8, const uint8_t* v8,
                                              const float* k_scale, const float* v_scale, const int* block_table,
                                              int max_pages, int num_pages, const int* qpos, const int* rows,
                                              const int* seqs, const SplitPlan& plan, int n_q, int n_kv, int d_head,
                                              bf16* out, int ldo, int num_sms, cudaStream_t stream) {
  if (plan.num_units <= 0) return cudaSuccess;
  if (n_q % n_kv || n_q / n_kv > SMAXG) return cudaErrorNotSupported;
  if (d_head == 128)
    return split_fp8_d<128>(q, ldq, k8, v8, k_scale, v_scale, block_table, max_pages, num_pages, qpos, rows, seqs,
                            plan, n_q, n_kv, out, ldo, num_sms, stream);
  if (d_head == 64)
    return split_fp8_d<64>(q, ldq, k8, v8, k_scale, v_scale, block_table, max_pages, num_pages, qpos, rows, seqs,
                           plan, n_q, n_kv, out, ldo, num_sms, stream);
  return cudaErrorNotSupported;
}

int split_keys_for(int nkeys) { return nkeys <= kShortRowKeys ? kSplitKeys / 2 : kSplitKeys; }

void split_plan_host(const int* nkeys, int items, std::vector<int>* units, std::vector<int>* ubeg) {
  units->clear();
  ubeg->assign(1, 0);
  for (int b = 0; b < items; ++b) {
    const int split = split_keys_for(nkeys[b]);
    for (int k0 = 0; k0 < nkeys[b]; k0 += split) {
      units->push_back(b);
      units->push_back(k0);
      units->push_back(split);
    }
    ubeg->push_back((int)(units->size() / 3));
  }
}

size_t split_part_floats(int num_units, int n_q, int d_head) { return (size_t)num_units * n_q * (d_head + 2); }

cudaError_t launch_attention_decode_split(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                          const int* block_table, int max_pages, int num_pages, const int* qpos,
                                          const int* rows, const int* seqs, const SplitPlan& plan, int n_q,
                                          int n_kv, int d_head, bf16* out, int ldo, int num_sms, cudaStream_t stream) {
  if (plan.num_units <= 0) return cudaSuccess;
  // a group of more than 8 query heads takes the one-CTA-per-row kernel
  if (n_q % n_kv || n_q / n_kv > SMAXG) return cudaErrorNotSupported;
  if (d_head == 128)
    return split_d<128>(q, ldq, k_pool, v_pool, block_table, max_pages, num_pages, qpos, rows, seqs, plan, n_q,
                        n_kv, out, ldo, num_sms, stream);
  if (d_head == 64)
    return split_d<64>(q, ldq, k_pool, v_pool, block_table, max_pages, num_pages, qpos, rows, seqs, plan, n_q,
                       n_kv, out, ldo, num_sms, stream);
  return cudaErrorNotSupported;
}

}  // namespace skv
