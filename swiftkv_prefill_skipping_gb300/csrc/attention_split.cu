// Single-row GQA attention over the paged KV cache, split along the keys: decode tokens,
// the last token of each prompt in the SwiftKV tail, and rows of short chunks.
//
// The work is a list of units (item b, split j): keys [j*split, (j+1)*split) of item b,
// for one KV head per CTA (grid = units x n_kv), so a long context is spread over many
// SMs and short and long rows mix without stragglers. A CTA has 4 warps; warp w takes
// the split's pages w, w+4, ... Each (page, KV head) block of 16 keys is 16*d_head*2
// contiguous bytes in the pool; a warp stages its pages' K and V with cp.async into a
// 3-deep ring of XOR-swizzled shared-memory tiles, so HBM reads stay in flight while
// it computes. The G = n_q/n_kv query heads of the group are the 16 rows of an mma.sync
// m16n8k16 A operand (rows >= G are zero), so one read of each K/V row serves the whole
// group: S = Q K^T (bf16, fp32 accumulate), online softmax in the log2 domain, O += P V
// with P and V at fp16 (V converted in shared memory), fp32 accumulate. The warps merge
// through shared memory; a unit that covers its whole row writes the output, otherwise it
// writes (max, sum, unnormalised O) per head and attn_split_combine merges the splits.
#include <algorithm>
#include <cfloat>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace skv {

namespace {

constexpr int SW = 4;        // warps per CTA
constexpr int SSTAGES = 3;   // pages in flight per warp
constexpr int SMAXG = 16;    // query heads per KV head (rows of the mma A operand)

template <int D>
constexpr int split_smem_bytes() {
  return SW * SSTAGES * 2 * kPageSize * D * 2;
}

template <int D>
__global__ void __launch_bounds__(SW * 32) attn_split_kernel(
    const bf16* __restrict__ q, int ldq, const bf16* __restrict__ kpool, const bf16* __restrict__ vpool,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ qpos,
    const int* __restrict__ rows, const int* __restrict__ seqs, const int* __restrict__ units, int split_keys,
    int n_q, int n_kv, bf16* __restrict__ out, int ldo, float* __restrict__ part, float scale_log2) {
  constexpr int PAGE = kPageSize * D;  // elements of one (page, head) K or V block
  constexpr int CH = D / 8;            // 16-byte chunks per key row
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bf16* sK = reinterpret_cast<bf16*>(smem) + (size_t)warp * SSTAGES * 2 * PAGE;
  bf16* sV = sK + SSTAGES * PAGE;

  const int u = blockIdx.x, kvh = blockIdx.y;
  const int b = units[2 * u], j = units[2 * u + 1];
  const int r = rows ? rows[b] : b;    // row of q / out / qpos
  const int sq = seqs ? seqs[b] : b;   // block table row
  const int G = n_q / n_kv;
  const int nkeys = qpos[r] + 1;
  const int k_begin = j * split_keys, k_end = min(nkeys, k_begin + split_keys);
  const int p_begin = k_begin / kPageSize, p_end = (k_end + kPageSize - 1) / kPageSize;
  const int* btrow = bt + (size_t)sq * max_pages;

  auto swz = [](int row, int ch) { return row * D + ((ch ^ (row & 7)) * 8); };

  // Q of the group as A fragments: rows = heads (groupID, groupID + 8), zero past G
  const int g0 = lane >> 2, g1 = g0 + 8, qc = 2 * (lane & 3);
  const bf16* qrow = q + (size_t)r * ldq + (size_t)kvh * G * D;
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c = ks * 16 + qc;
    qf[ks][0] = g0 < G ? *reinterpret_cast<const uint32_t*>(qrow + g0 * D + c) : 0u;
    qf[ks][1] = g1 < G ? *reinterpret_cast<const uint32_t*>(qrow + g1 * D + c) : 0u;
    qf[ks][2] = g0 < G ? *reinterpret_cast<const uint32_t*>(qrow + g0 * D + c + 8) : 0u;
    qf[ks][3] = g1 < G ? *reinterpret_cast<const uint32_t*>(qrow + g1 * D + c + 8) : 0u;
  }

  const int npages = p_end - p_begin;
  const int my_pages = npages > warp ? (npages - warp + SW - 1) / SW : 0;
  auto page_of = [&](int i) { return btrow[p_begin + warp + SW * i]; };
  auto issue = [&](int i) {  // this warp's i-th page into ring slot i % SSTAGES
    if (i < my_pages) {
      const int page = page_of(i);
      const bool ok = page >= 0 && page < num_pages;
      const size_t base = ok ? ((size_t)page * n_kv + kvh) * PAGE : 0;
      bf16* dk = sK + (i % SSTAGES) * PAGE;
      bf16* dv = sV + (i % SSTAGES) * PAGE;
#pragma unroll
      for (int c = lane; c < kPageSize * CH; c += 32) {
        const int row = c / CH, ch = c % CH;
        cp_async16(smem_u32(dk + swz(row, ch)), kpool + base + row * D + ch * 8, ok ? 16 : 0);
        cp_async16(smem_u32(dv + swz(row, ch)), vpool + base + row * D + ch * 8, ok ? 16 : 0);
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
  };

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  float m0 = -FLT_MAX, m1 = -FLT_MAX, l0 = 0.f, l1 = 0.f;

#pragma unroll
  for (int i = 0; i < SSTAGES - 1; ++i) issue(i);
  for (int i = 0; i < my_pages; ++i) {
    issue(i + SSTAGES - 1);
    cp_async_wait<SSTAGES - 1>();
    __syncwarp();
    const bf16* kb = sK + (i % SSTAGES) * PAGE;
    bf16* vb = sV + (i % SSTAGES) * PAGE;
    // V bf16 -> fp16 in place (exact inside fp16's normal range, clamped to +-65504)
    {
      uint4* vt = reinterpret_cast<uint4*>(vb);
#pragma unroll
      for (int c = lane; c < PAGE / 8; c += 32) {
        uint4 raw = vt[c];
        uint32_t* w = reinterpret_cast<uint32_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[e]));
          w[e] = pack_f16(fminf(fmaxf(f.x, -65504.f), 65504.f), fminf(fmaxf(f.y, -65504.f), 65504.f));
        }
        vt[c] = raw;
      }
    }
    __syncwarp();

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
    const int pg = page_of(i);
    const bool page_ok = pg >= 0 && pg < num_pages;
    const int key0 = (p_begin + warp + SW * i) * kPageSize;
    float mx0 = -FLT_MAX, mx1 = -FLT_MAX;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + 8 * t + qc + e;
        const bool valid = page_ok && key >= k_begin && key < k_end;
        sc[t][e] = valid ? sc[t][e] * scale_log2 : -INFINITY;
        sc[t][2 + e] = valid ? sc[t][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, sc[t][e]);
        mx1 = fmaxf(mx1, sc[t][2 + e]);
      }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[t][e] = exp2f(sc[t][e] - mn0);
        sc[t][2 + e] = exp2f(sc[t][2 + e] - mn1);
        ps0 += sc[t][e];
        ps1 += sc[t][2 + e];
      }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }
    // O += P V: P (heads x 16 keys) is the S accumulator re-packed as an fp16 A operand
    uint32_t pa[4];
    pa[0] = pack_f16(sc[0][0], sc[0][1]);
    pa[1] = pack_f16(sc[0][2], sc[0][3]);
    pa[2] = pack_f16(sc[1][0], sc[1][1]);
    pa[3] = pack_f16(sc[1][2], sc[1][3]);
#pragma unroll
    for (int dp = 0; dp < D / 16; ++dp) {
      uint32_t b0[2], b1[2];
      ldmatrix_x4_trans(smem_u32(vb + swz(lane & 15, dp * 2 + (lane >> 4))), b0[0], b0[1], b1[0], b1[1]);
      mma_f16_16816(o[2 * dp], pa, b0);
      mma_f16_16816(o[2 * dp + 1], pa, b1);
    }
    __syncwarp();  // the slot is refilled by a later issue()
  }
  cp_async_wait<0>();
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every warp is done with its ring: the merge buffers alias it

  float* s_o = reinterpret_cast<float*>(smem);            // [SW][SMAXG][D]
  float* s_m = s_o + SW * SMAXG * D;                       // [SW][SMAXG]
  float* s_l = s_m + SW * SMAXG;                           // [SW][SMAXG]
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int dim = n * 8 + qc;
    if (g0 < G) {
      s_o[(warp * SMAXG + g0) * D + dim] = o[n][0];
      s_o[(warp * SMAXG + g0) * D + dim + 1] = o[n][1];
    }
    if (g1 < G) {
      s_o[(warp * SMAXG + g1) * D + dim] = o[n][2];
      s_o[(warp * SMAXG + g1) * D + dim + 1] = o[n][3];
    }
  }
  if ((lane & 3) == 0) {
    if (g0 < G) {
      s_m[warp * SMAXG + g0] = m0;
      s_l[warp * SMAXG + g0] = l0;
    }
    if (g1 < G) {
      s_m[warp * SMAXG + g1] = m1;
      s_l[warp * SMAXG + g1] = l1;
    }
  }
  __syncthreads();
  const bool whole = k_begin == 0 && k_end == nkeys;
  for (int idx = threadIdx.x; idx < G * D; idx += SW * 32) {
    const int g = idx / D, dim = idx % D;
    float mx = -FLT_MAX;
#pragma unroll
    for (int w = 0; w < SW; ++w) mx = fmaxf(mx, s_m[w * SMAXG + g]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < SW; ++w) {
      const float f = exp2f(s_m[w * SMAXG + g] - mx);
      num += s_o[(w * SMAXG + g) * D + dim] * f;
      den += s_l[w * SMAXG + g] * f;
    }
    if (whole) {
      out[(size_t)r * ldo + (size_t)(kvh * G + g) * D + dim] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
    } else {
      float* pp = part + (((size_t)u * n_kv + kvh) * G + g) * (D + 2);
      pp[2 + dim] = num;
      if (dim == 0) {
        pp[0] = mx;
        pp[1] = den;
      }
    }
  }
}

// Merges the splits of every item that has more than one: per head, the running maxima
// rescale each split's (sum, unnormalised O) to the largest one.
template <int D>
__global__ void __launch_bounds__(128) attn_split_combine(const int* __restrict__ rows, const int* __restrict__ ubeg,
                                                          int n_q, int n_kv, const float* __restrict__ part,
                                                          bf16* __restrict__ out, int ldo) {
  const int b = blockIdx.x, kvh = blockIdx.y;
  const int u0 = ubeg[b], u1 = ubeg[b + 1];
  if (u1 - u0 <= 1) return;  // written directly by its only unit
  const int r = rows ? rows[b] : b;
  const int G = n_q / n_kv;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, dim = idx % D;
    float mx = -FLT_MAX;
    for (int u = u0; u < u1; ++u) mx = fmaxf(mx, part[(((size_t)u * n_kv + kvh) * G + g) * (D + 2)]);
    float num = 0.f, den = 0.f;
    for (int u = u0; u < u1; ++u) {
      const float* pp = part + (((size_t)u * n_kv + kvh) * G + g) * (D + 2);
      const float f = exp2f(pp[0] - mx);
      num += pp[2 + dim] * f;
      den += pp[1] * f;
    }
    out[(size_t)r * ldo + (size_t)(kvh * G + g) * D + dim] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
  }
}

template <int D>
cudaError_t split_d(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool, const int* bt, int max_pages,
                    int num_pages, const int* qpos, const int* rows, const int* seqs, const SplitPlan& plan,
                    int n_q, int n_kv, bf16* out, int ldo, cudaStream_t stream) {
  constexpr int smem = split_smem_bytes<D>();
  static_assert(smem >= (SW * SMAXG * D + 2 * SW * SMAXG) * 4, "merge buffers must fit in the ring");
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  attn_split_kernel<D><<<dim3(plan.num_units, n_kv), SW * 32, smem, stream>>>(
      q, ldq, k_pool, v_pool, bt, max_pages, num_pages, qpos, rows, seqs, plan.units, plan.split_keys, n_q, n_kv,
      out, ldo, plan.part, scale_log2);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !plan.any_split) return e;
  attn_split_combine<D><<<dim3(plan.num_items, n_kv), 128, 0, stream>>>(rows, plan.ubeg, n_q, n_kv, plan.part,
                                                                        out, ldo);
  return cudaGetLastError();
}

}  // namespace

int split_plan_host(const int* nkeys, int items, std::vector<int>* units, std::vector<int>* ubeg) {
  // A fixed split keeps every row's arithmetic independent of the rest of the batch (a
  // prompt gives bit-identical logits alone or packed with others); 256 keys = 4 pages per
  // warp, 128 KB of K/V per CTA and KV head at d_head 128.
  const int split = kSplitKeys;
  units->clear();
  ubeg->assign(1, 0);
  for (int b = 0; b < items; ++b) {
    const int ns = (nkeys[b] + split - 1) / split;
    for (int j = 0; j < ns; ++j) {
      units->push_back(b);
      units->push_back(j);
    }
    ubeg->push_back((int)(units->size() / 2));
  }
  return split;
}

size_t split_part_floats(int num_units, int n_q, int d_head) { return (size_t)num_units * n_q * (d_head + 2); }

cudaError_t launch_attention_decode_split(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                          const int* block_table, int max_pages, int num_pages, const int* qpos,
                                          const int* rows, const int* seqs, const SplitPlan& plan, int n_q,
                                          int n_kv, int d_head, bf16* out, int ldo, cudaStream_t stream) {
  if (plan.num_units <= 0) return cudaSuccess;
  if (n_q % n_kv || n_q / n_kv > SMAXG || plan.split_keys % kPageSize) return cudaErrorNotSupported;
  if (d_head == 128)
    return split_d<128>(q, ldq, k_pool, v_pool, block_table, max_pages, num_pages, qpos, rows, seqs, plan, n_q,
                        n_kv, out, ldo, stream);
  if (d_head == 64)
    return split_d<64>(q, ldq, k_pool, v_pool, block_table, max_pages, num_pages, qpos, rows, seqs, plan, n_q,
                       n_kv, out, ldo, stream);
  return cudaErrorNotSupported;
}

}  // namespace skv
