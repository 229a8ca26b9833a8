// Causal GQA attention over the paged KV cache.
//
// attn_prefill_kernel: varlen prompts, one CTA per (64-row query tile, query head).
//   Q tile and double-buffered 64-key K/V tiles are staged in XOR-swizzled shared
//   memory with cp.async; each (page, head) block of 16 keys is 16*d_head*2
//   contiguous bytes. S = Q K^T and O += P V run on mma.sync bf16 tensor cores with fp32
//   accumulation; P V takes V in bf16 as cached and P as bf16 high + low parts (two MMAs,
//   about 17 significant bits of P); softmax is online (running max / sum in the log2
//   domain). FP8 cache: the pools hold the e4m3 codes as (exact) bf16 values, and each score
//   is multiplied by its key's scale and each P by its value's scale (float32).
//   Query tiles arrive longest-first (heaviest causal tiles scheduled first).
// attn_decode_kernel: one query per sequence (decode tokens and the last prompt
//   token of the SwiftKV tail), one CTA per (sequence, KV head) computing all query
//   heads of the GQA group from one read of each K/V row.
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace skv {

namespace {

constexpr int ABQ = 64, ABKV = 64, ATHREADS = 128;

template <int D>
__global__ void __launch_bounds__(ATHREADS) attn_prefill_kernel(
    const bf16* __restrict__ q, int ldq, const bf16* __restrict__ kpool, const bf16* __restrict__ vpool,
    const float* __restrict__ kscale, const float* __restrict__ vscale,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ cu,
    const int* __restrict__ ctx, const int* __restrict__ tiles, int n_q, int n_kv, bf16* __restrict__ out, int ldo,
    float scale_log2) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  __shared__ float s_scale[2][2][ABKV];  // FP8 cache: [buffer][key, value][key of the block]
  const bool fp8 = kscale != nullptr;
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + ABQ * D;
  bf16* sV = sK + 2 * ABKV * D;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = tiles[blockIdx.x];
  const int s = tile >> 16, qt = tile & 0xffff;
  const int h = blockIdx.y, kvh = h / (n_q / n_kv);
  const int seq0 = cu[s], n = cu[s + 1] - seq0;
  const int q0 = qt * ABQ;
  // the chunk's rows sit at positions c0.. after c0 cached keys; keys [0, nk) are visible
  const int c0 = ctx ? ctx[s] : 0, nk = c0 + n;

  auto swz = [](int row, int ch) { return row * D + ((ch ^ (row & 7)) * 8); };

  for (int c = tid; c < ABQ * CH; c += ATHREADS) {
    int r = c / CH, ch = c % CH;
    int tok = q0 + r;
    bool ok = tok < n;
    const bf16* src = q + (size_t)(seq0 + (ok ? tok : 0)) * ldq + h * D + ch * 8;
    cp_async16(smem_u32(sQ + swz(r, ch)), src, ok ? 16 : 0);
  }

  auto load_kv = [&](int buf, int kb) {
    for (int c = tid; c < ABKV * CH; c += ATHREADS) {
      int r = c / CH, ch = c % CH;
      int key = kb * ABKV + r;
      int page = key < nk ? bt[(size_t)s * max_pages + (key >> 4)] : -1;
      bool ok = page >= 0 && page < num_pages;
      size_t off = ok ? (((size_t)page * n_kv + kvh) * kPageSize + (key & 15)) * D + ch * 8 : 0;
      cp_async16(smem_u32(sK + buf * ABKV * D + swz(r, ch)), kpool + off, ok ? 16 : 0);
      cp_async16(smem_u32(sV + buf * ABKV * D + swz(r, ch)), vpool + off, ok ? 16 : 0);
    }
    if (fp8 && tid < ABKV) {  // this block's scales (keys past the chunk or off the pool: 1)
      const int key = kb * ABKV + tid;
      const int page = key < nk ? bt[(size_t)s * max_pages + (key >> 4)] : -1;
      const bool ok = page >= 0 && page < num_pages;
      const size_t si = ((size_t)page * n_kv + kvh) * kPageSize + (key & 15);
      s_scale[buf][0][tid] = ok ? kscale[si] : 1.f;
      s_scale[buf][1][tid] = ok ? vscale[si] : 1.f;
    }
  };

  const int kv_end = min(nk, c0 + q0 + ABQ);  // keys needed: [0, kv_end)
  const int nkv = (kv_end + ABKV - 1) / ABKV;
  load_kv(0, 0);
  cp_async_commit();

  uint32_t qf[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[i][j] = 0.f;
  float m_a = -FLT_MAX, m_b = -FLT_MAX, l_a = 0.f, l_b = 0.f;
  const int ra = warp * 16 + (lane >> 2);
  const int qa = q0 + ra, qb = qa + 8;            // rows within the chunk
  const int pa_ = c0 + qa, pb_ = c0 + qb;          // their positions

  for (int kb = 0; kb < nkv; ++kb) {
    if (kb + 1 < nkv) load_kv((kb + 1) & 1, kb + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        int row = warp * 16 + (lane & 15);
        int ch = ks * 2 + (lane >> 4);
        ldmatrix_x4(smem_u32(sQ + swz(row, ch)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const bf16* kb_s = sK + (kb & 1) * ABKV * D;
    const bf16* vb_s = sV + (kb & 1) * ABKV * D;
    const float* ksc = s_scale[kb & 1][0];
    const float* vsc = s_scale[kb & 1][1];
    float sc[ABKV / 8][4];
#pragma unroll
    for (int i = 0; i < ABKV / 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
#pragma unroll
    for (int np = 0; np < ABKV / 16; ++np) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b0[2], b1[2];
        int row = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        int ch = ks * 2 + ((lane >> 3) & 1);
        ldmatrix_x4(smem_u32(kb_s + swz(row, ch)), b0[0], b0[1], b1[0], b1[1]);
        mma_bf16_16816(sc[2 * np], qf[ks], b0);
        mma_bf16_16816(sc[2 * np + 1], qf[ks], b1);
      }
    }
    // mask, running max
    float mx_a = -FLT_MAX, mx_b = -FLT_MAX;
#pragma unroll
    for (int nb = 0; nb < ABKV / 8; ++nb) {
      int key = kb * ABKV + nb * 8 + 2 * (lane & 3);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int k = key + e;
        const float ks = fp8 ? ksc[k - kb * ABKV] : 1.f;  // FP8: the key's scale
        float va = (k <= pa_ && k < nk) ? sc[nb][e] * ks * scale_log2 : -INFINITY;
        float vb = (k <= pb_ && k < nk) ? sc[nb][2 + e] * ks * scale_log2 : -INFINITY;
        sc[nb][e] = va;
        sc[nb][2 + e] = vb;
        mx_a = fmaxf(mx_a, va);
        mx_b = fmaxf(mx_b, vb);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int nb = 0; nb < ABKV / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[nb][e] = exp2f(sc[nb][e] - mn_a);
        sc[nb][2 + e] = exp2f(sc[nb][2 + e] - mn_b);
        ps_a += sc[nb][e];
        ps_b += sc[nb][2 + e];
      }
    }
    l_a = l_a * al_a + ps_a;
    l_b = l_b * al_b + ps_b;
    if (fp8) {  // P V with V = code x scale: the value scale rides on P
#pragma unroll
      for (int nb = 0; nb < ABKV / 8; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float vs = vsc[nb * 8 + 2 * (lane & 3) + e];
          sc[nb][e] *= vs;
          sc[nb][2 + e] *= vs;
        }
    }
#pragma unroll
    for (int db = 0; db < D / 8; ++db) {
      o[db][0] *= al_a;
      o[db][1] *= al_a;
      o[db][2] *= al_b;
      o[db][3] *= al_b;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < ABKV / 16; ++kk) {
      uint32_t ph[4], pl[4];
      split_pair_bf16(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
      split_pair_bf16(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
      split_pair_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
      split_pair_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0[2], b1[2];
        int row = kk * 16 + (lane & 15);
        int ch = dp * 2 + (lane >> 4);
        ldmatrix_x4_trans(smem_u32(vb_s + swz(row, ch)), b0[0], b0[1], b1[0], b1[1]);
        mma_bf16_16816(o[2 * dp], ph, b0);
        mma_bf16_16816(o[2 * dp + 1], ph, b1);
        mma_bf16_16816(o[2 * dp], pl, b0);
        mma_bf16_16816(o[2 * dp + 1], pl, b1);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  const float ia = 1.f / l_a, ib = 1.f / l_b;
#pragma unroll
  for (int db = 0; db < D / 8; ++db) {
    int col = h * D + db * 8 + 2 * (lane & 3);
    if (qa < n)
      *reinterpret_cast<uint32_t*>(out + (size_t)(seq0 + qa) * ldo + col) = pack_bf16(o[db][0] * ia, o[db][1] * ia);
    if (qb < n)
      *reinterpret_cast<uint32_t*>(out + (size_t)(seq0 + qb) * ldo + col) = pack_bf16(o[db][2] * ib, o[db][3] * ib);
  }
}

constexpr int DTHREADS = 256, DWARPS = DTHREADS / 32, DMAXG = 8;

// One CTA per (sequence b, KV head): 8 warps walk the keys 32 at a time. In a round,
// lane i owns key k0 + i: it reads that key's K row (contiguous d_head*2 bytes) and
// computes the scores of every query head of the GQA group against it; one warp
// max/sum per head updates the running softmax; then the warp sweeps the round's 32
// V rows (coalesced, lane = 4 dims at d_head 128) with each key's probability
// broadcast by shuffle. Warps are merged through shared memory at the end.
template <int D>
__global__ void __launch_bounds__(DTHREADS) attn_decode_kernel(
    const bf16* __restrict__ q, int ldq, const bf16* __restrict__ kpool, const bf16* __restrict__ vpool,
    const int* __restrict__ bt, int max_pages, int num_pages, const int* __restrict__ qpos,
    const int* __restrict__ rows, const int* __restrict__ seqs, int n_q, int n_kv, bf16* __restrict__ out, int ldo,
    float scale_log2) {
  constexpr int DPL = D / 32;  // dims per lane in the PV sweep
  __shared__ float s_q[DMAXG][D];
  __shared__ float s_m[DWARPS][DMAXG], s_l[DWARPS][DMAXG];
  __shared__ float s_o[DWARPS][DMAXG][D];
  const int kvh = blockIdx.y;
  // item -> its row of q / out / qpos and its block table row (identity without maps)
  const int b = rows ? rows[blockIdx.x] : blockIdx.x;
  const int sq = seqs ? seqs[blockIdx.x] : blockIdx.x;
  const int G = n_q / n_kv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nkeys = qpos[b] + 1;

  for (int i = threadIdx.x; i < G * D; i += DTHREADS) {
    int g = i / D, dim = i % D;
    s_q[g][dim] = __bfloat162float(q[(size_t)b * ldq + (kvh * G + g) * D + dim]) * scale_log2;
  }
  __syncthreads();

  float m[DMAXG], l[DMAXG], o[DMAXG][DPL];
#pragma unroll
  for (int g = 0; g < DMAXG; ++g) {
    m[g] = -FLT_MAX;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[g][i] = 0.f;
  }
  const int* btrow = bt + (size_t)sq * max_pages;
  for (int k0 = warp * 32; k0 < nkeys; k0 += DWARPS * 32) {
    const int k = k0 + lane;
    int page = k < nkeys ? btrow[k >> 4] : -1;
    const bool ok = page >= 0 && page < num_pages;
    const size_t rowoff = ok ? (((size_t)page * n_kv + kvh) * kPageSize + (k & 15)) * D : 0;
    float sc[DMAXG];
#pragma unroll
    for (int g = 0; g < DMAXG; ++g) sc[g] = 0.f;
    if (ok) {
      const uint4* kr = reinterpret_cast<const uint4*>(kpool + rowoff);
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        uint4 raw = kr[c];
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
        float kf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(h2[e]);
          kf[2 * e] = f.x;
          kf[2 * e + 1] = f.y;
        }
#pragma unroll
        for (int g = 0; g < DMAXG; ++g) {
          if (g < G) {
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[g] += s_q[g][c * 8 + e] * kf[e];
          }
        }
      }
    }
    float p[DMAXG];
#pragma unroll
    for (int g = 0; g < DMAXG; ++g) {
      if (g >= G) break;
      float v = ok ? sc[g] : -INFINITY;
      float mx = v;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[g], mx);
      const float al = exp2f(m[g] - mn);
      p[g] = exp2f(v - mn);
      float ps = p[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      m[g] = mn;
      l[g] = l[g] * al + ps;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[g][i] *= al;
    }
    const int kcount = min(32, nkeys - k0);
    // issue all 32 V-row loads of the round before consuming any of them
    float vr[32][DPL];
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const int pg = __shfl_sync(0xffffffffu, page, kk);
      if (kk < kcount && pg >= 0 && pg < num_pages) {
        const bf16* vrow = vpool + (((size_t)pg * n_kv + kvh) * kPageSize + ((k0 + kk) & 15)) * D + lane * DPL;
        if constexpr (DPL == 4) {
          uint2 raw = *reinterpret_cast<const uint2*>(vrow);
          float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
          float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
          vr[kk][0] = f0.x;
          vr[kk][1] = f0.y;
          vr[kk][2] = f1.x;
          vr[kk][3] = f1.y;
        } else {
#pragma unroll
          for (int i = 0; i < DPL; ++i) vr[kk][i] = __bfloat162float(vrow[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < DPL; ++i) vr[kk][i] = 0.f;
      }
    }
#pragma unroll
    for (int g = 0; g < DMAXG; ++g) {
      if (g >= G) break;
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p[g], kk);
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[g][i] += pk * vr[kk][i];
      }
    }
  }
#pragma unroll
  for (int g = 0; g < DMAXG; ++g) {
    if (g >= G) break;
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) s_o[warp][g][lane * DPL + i] = o[g][i];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += DTHREADS) {
    int g = idx / D, dim = idx % D;
    float mx = -FLT_MAX;
    for (int w = 0; w < DWARPS; ++w) mx = fmaxf(mx, s_m[w][g]);
    float num = 0.f, den = 0.f;
    for (int w = 0; w < DWARPS; ++w) {
      float sc = exp2f(s_m[w][g] - mx);
      num += s_o[w][g][dim] * sc;
      den += s_l[w][g] * sc;
    }
    out[(size_t)b * ldo + (kvh * G + g) * D + dim] = __float2bfloat16_rn(num / den);
  }
}

template <int D>
cudaError_t prefill_d(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool, const float* k_scale,
                      const float* v_scale, const int* bt, int max_pages, int num_pages, const int* cu,
                      const int* ctx, const int* tiles, int num_tiles, int n_q, int n_kv, bf16* out, int ldo,
                      cudaStream_t stream) {
  constexpr int smem = (ABQ + 4 * ABKV) * D * 2;
  static PerDeviceOnce smem_attr;
  {
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_prefill_kernel<D>), smem, smem_attr);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(num_tiles, n_q);
  attn_prefill_kernel<D><<<grid, ATHREADS, smem, stream>>>(q, ldq, k_pool, v_pool, k_scale, v_scale, bt, max_pages,
                                                          num_pages, cu, ctx, tiles, n_q, n_kv, out, ldo, scale_log2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_prefill(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                     const float* k_scale, const float* v_scale,
                                     const int* block_table, int max_pages, int num_pages,
                                     const int* cu, const int* ctx, const int* tiles, int num_tiles, int n_q,
                                     int n_kv, int d_head, bf16* out, int ldo, cudaStream_t stream) {
  if (num_tiles <= 0) return cudaSuccess;
  if (!k_scale != !v_scale) return cudaErrorNotSupported;
  if (d_head == 128)
    return prefill_d<128>(q, ldq, k_pool, v_pool, k_scale, v_scale, block_table, max_pages, num_pages, cu, ctx,
                          tiles, num_tiles, n_q, n_kv, out, ldo, stream);
  if (d_head == 64)
    return prefill_d<64>(q, ldq, k_pool, v_pool, k_scale, v_scale, block_table, max_pages, num_pages, cu, ctx,
                         tiles, num_tiles, n_q, n_kv, out, ldo, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_attention_decode(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                    const int* block_table, int max_pages, int num_pages,
                                    const int* qpos, int B, int n_q, int n_kv, int d_head, bf16* out,
                                    int ldo, cudaStream_t stream, const int* rows, const int* seqs) {
  if (B <= 0) return cudaSuccess;
  if (n_q / n_kv > DMAXG) return cudaErrorNotSupported;
  dim3 grid(B, n_kv);
  if (d_head == 128) {
    attn_decode_kernel<128><<<grid, DTHREADS, 0, stream>>>(q, ldq, k_pool, v_pool, block_table, max_pages,
                                                           num_pages, qpos, rows, seqs, n_q, n_kv, out, ldo,
                                                           1.4426950408889634f / sqrtf(128.f));
  } else if (d_head == 64) {
    attn_decode_kernel<64><<<grid, DTHREADS, 0, stream>>>(q, ldq, k_pool, v_pool, block_table, max_pages,
                                                          num_pages, qpos, rows, seqs, n_q, n_kv, out, ldo,
                                                          1.4426950408889634f / sqrtf(64.f));
  } else {
    return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace skv
