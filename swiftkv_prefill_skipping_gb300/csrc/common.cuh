// Shared device definitions of the SwiftKV GB300 library: bf16 helpers, the
// device status word, and the GEMM epilogues (RoPE + paged KV write, residual
// add, SwiGLU, plain stores). Every GEMM variant (mma.sync tiles, skinny
// split-K, tcgen05) hands its fp32 accumulators to `apply_pair`, so all of them
// produce identical outputs for identical accumulators.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace skv {

typedef __nv_bfloat16 bf16;

constexpr int kPageSize = 16;

enum StatusBits : int { kStatusBadToken = 1, kStatusBadPage = 2, kStatusTimeout = 4 };

// Epilogue kinds. Column pairing: every GEMM hands columns to the epilogue in
// pairs (lo, hi = lo + half) inside aligned blocks of 2*half columns, where
// half = d_head/2 for the RoPE epilogues (rotate-half partners) and 64 for the
// others (SwiGLU gate/up partners in the 64-row interleaved packing).
enum EpiKind : int {
  EPI_STORE_F32 = 0,   // out_f32[m][n] = acc
  EPI_STORE_BF16 = 1,  // out_bf16[m][n] = bf16(acc)
  EPI_RESID = 2,       // out_f32[m][n] += acc           (fp32 residual stream)
  EPI_SWIGLU = 3,      // out_bf16[m][64*(n/128) + n%128] = bf16(silu(acc[n]) * acc[n+64]), n%128 < 64
  EPI_QKV = 4,         // cols [0,q_cols): Q -> RoPE -> out_bf16; then K (RoPE) and V -> paged cache
  EPI_WIDE_KV = 5,     // per AcrossKV group: [K | V] -> RoPE on K -> paged caches cache_base + group
};

struct EpiParams {
  int kind;
  int M, N;                  // rows, columns of the GEMM output
  int ldo;                   // leading dimension of out_f32 / out_bf16 (elements)
  float* out_f32;
  bf16* out_bf16;
  const float* bias;         // [N] or nullptr; added before RoPE
  int d_head, n_kv;
  int q_cols;                // EPI_QKV: n_q * d_head (0: no Q columns)
  const int* positions;      // [M] token position within its sequence
  const int* slots;          // [M] page*16 + row, or -1 (invalid page: write skipped)
  const float2* rope_tab;    // [rope_len][d_head/2] (cos, sin) for positions < rope_len
  int rope_len;
  const float* inv_freq;     // [d_head/2]
  bf16* const* k_pools;      // device array [num_caches] of K pools
  bf16* const* v_pools;      // device array [num_caches] of V pools
  int cache_base;            // EPI_QKV: the layer's cache; EPI_WIDE_KV: first skipped cache
  bf16* kv_stage;            // non-null (FP8 cache): K (after RoPE) and V rows go here instead,
  int kv_stage_ld;           //   [M][kv_stage_ld] at their K/V column, for the quantize pass
  // FP8 cache quantized in the epilogue (tcgen05 GEMMs; ks_pools non-null): k_pools / v_pools
  // hold uint8 e4m3 code pools, ks_pools / vs_pools the float scale pools [pages][n_kv][16];
  // exp_k / exp_v (optional) receive the codes as bf16 for the prompt-tile attention
  float* const* ks_pools;
  float* const* vs_pools;
  bf16* exp_k;
  bf16* exp_v;
  // RMSNorm fused into the GEMMs on either side of it (prompt rows on the tcgen05 GEMMs):
  const float* norm_part;    // non-null: the A operand holds bf16(gamma * x) of residual rows x and
  int norm_parts;            //   the kernel scales row m's accumulators by rsqrt(S_m / dim + eps),
  float norm_inv_dim;        //   S_m = the sum, in index order, of norm_part[m][0 .. norm_parts)
  float norm_eps;
  bf16* xb_out;              // EPI_RESID, non-null: also stores bf16(xb_gamma * updated row) at
  const float* xb_gamma;     //   [m][ldo] (xb_gamma NULL: 1), the next norm's input, and the row's
  float* ss_out;             //   sum of squares per 256-column GEMM tile at [m][norm_tiles(N)]
};

// Partial sums of squares an EPI_RESID row of width n leaves in ss_out: one per 256-column tile.
constexpr int kNormTile = 256;
constexpr int kMaxNormTiles = 32;  // widths up to 8192
__host__ __device__ __forceinline__ int norm_tiles(int n) { return (n + kNormTile - 1) / kNormTile; }

// Row scale of the fused RMSNorm: rsqrt(mean of squares + eps) with the tile sums added in
// index order (independent loads, one dependent add chain).
__device__ __forceinline__ float fused_norm_scale(const EpiParams& p, int m) {
  const float* s = p.norm_part + (size_t)m * p.norm_parts;
  float v[kMaxNormTiles];
#pragma unroll
  for (int i = 0; i < kMaxNormTiles; ++i) v[i] = i < p.norm_parts ? s[i] : 0.f;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxNormTiles; ++i) acc += v[i];
  return rsqrtf(acc * p.norm_inv_dim + p.norm_eps);
}

__host__ __device__ __forceinline__ int pair_half(const EpiParams& p) {
  return (p.kind == EPI_QKV || p.kind == EPI_WIDE_KV) ? (p.d_head >> 1) : 64;
}

// Column of the lo member of pair index `u` (0 <= u < ncols/2) in a block-aligned range.
__device__ __forceinline__ int pair_lo(int u, int half) { return (u / half) * (2 * half) + (u % half); }

__device__ __forceinline__ void rope_rotate(const EpiParams& p, int pos, int i, float& a, float& b) {
  float c, s;
  if (pos < p.rope_len) {
    float2 cs = p.rope_tab[(size_t)pos * (p.d_head >> 1) + i];
    c = cs.x;
    s = cs.y;
  } else {
    sincosf((float)pos * p.inv_freq[i], &s, &c);
  }
  float a2 = a * c - b * s;
  float b2 = b * c + a * s;
  a = a2;
  b = b2;
}

__device__ __forceinline__ void paged_store_pair(bf16* pool, int slot, int n_kv, int head, int d_head,
                                                 int i, float a, float b) {
  size_t page = (size_t)(slot >> 4);
  size_t row = ((page * n_kv + head) * kPageSize + (slot & 15)) * (size_t)d_head;
  pool[row + i] = __float2bfloat16_rn(a);
  pool[row + i + (d_head >> 1)] = __float2bfloat16_rn(b);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

// Applies the epilogue to the column pair (n_lo, n_hi = n_lo + half) of row m.
__device__ __forceinline__ void apply_pair(const EpiParams& p, int m, int n_lo, int n_hi, float a,
                                           float b) {
  switch (p.kind) {
    case EPI_STORE_F32: {
      float* o = p.out_f32 + (size_t)m * p.ldo;
      o[n_lo] = a;
      o[n_hi] = b;
      break;
    }
    case EPI_STORE_BF16: {
      bf16* o = p.out_bf16 + (size_t)m * p.ldo;
      o[n_lo] = __float2bfloat16_rn(a);
      o[n_hi] = __float2bfloat16_rn(b);
      break;
    }
    case EPI_RESID: {
      float* o = p.out_f32 + (size_t)m * p.ldo;
      o[n_lo] += a;
      o[n_hi] += b;
      break;
    }
    case EPI_SWIGLU: {
      int col = (n_lo >> 7) * 64 + (n_lo & 127);
      p.out_bf16[(size_t)m * p.ldo + col] = __float2bfloat16_rn(silu_f(a) * b);
      break;
    }
    case EPI_QKV: {
      if (p.bias) {
        a += p.bias[n_lo];
        b += p.bias[n_hi];
      }
      const int dh = p.d_head;
      if (n_lo < p.q_cols) {
        rope_rotate(p, p.positions[m], n_lo % dh, a, b);
        bf16* o = p.out_bf16 + (size_t)m * p.ldo;
        o[n_lo] = __float2bfloat16_rn(a);
        o[n_hi] = __float2bfloat16_rn(b);
      } else {
        int slot = p.slots[m];
        if (slot < 0) break;
        int c = n_lo - p.q_cols;
        const int kvc = p.n_kv * dh;
        const int cs = c;
        bool is_k = c < kvc;
        if (!is_k) c -= kvc;
        int head = c / dh, i = c % dh;
        if (is_k) rope_rotate(p, p.positions[m], i, a, b);
        if (p.kv_stage) {
          bf16* o = p.kv_stage + (size_t)m * p.kv_stage_ld + cs;
          o[0] = __float2bfloat16_rn(a);
          o[dh >> 1] = __float2bfloat16_rn(b);
        } else {
          paged_store_pair(is_k ? p.k_pools[p.cache_base] : p.v_pools[p.cache_base], slot, p.n_kv, head,
                           dh, i, a, b);
        }
      }
      break;
    }
    case EPI_WIDE_KV: {
      if (p.bias) {
        a += p.bias[n_lo];
        b += p.bias[n_hi];
      }
      int slot = p.slots[m];
      if (slot < 0) break;
      const int dh = p.d_head;
      const int kvc = p.n_kv * dh;
      int grp = n_lo / (2 * kvc);
      int c = n_lo - grp * 2 * kvc;
      bool is_k = c < kvc;
      if (!is_k) c -= kvc;
      int head = c / dh, i = c % dh;
      if (is_k) rope_rotate(p, p.positions[m], i, a, b);
      if (p.kv_stage) {
        bf16* o = p.kv_stage + (size_t)m * p.kv_stage_ld;
        o[n_lo] = __float2bfloat16_rn(a);
        o[n_hi] = __float2bfloat16_rn(b);
        break;
      }
      int cache = p.cache_base + grp;
      paged_store_pair(is_k ? p.k_pools[cache] : p.v_pools[cache], slot, p.n_kv, head, dh, i, a, b);
      break;
    }
    default:
      break;
  }
}

// ---------------------------------------------------------------------------- 32-column chunks

__device__ __forceinline__ uint32_t pack_bf16_(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// dst must be 16-byte aligned
__device__ __forceinline__ void store_bf16x32(bf16* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    uint4 u;
    u.x = pack_bf16_(v[i], v[i + 1]);
    u.y = pack_bf16_(v[i + 2], v[i + 3]);
    u.z = pack_bf16_(v[i + 4], v[i + 5]);
    u.w = pack_bf16_(v[i + 6], v[i + 7]);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}

// Same epilogue as apply_pair for the 32 pairs (n_lo + i, n_hi + i), i < 32, with
// 16-byte vector stores. A chunk never straddles a Q/K/V region or a head because
// half is a multiple of 32 and region widths are multiples of d_head.
// Returns, for EPI_RESID with xb_out, the sum of squares of the updated values (0 otherwise).
__device__ __forceinline__ float apply_chunk32(const EpiParams& p, int m, int n_lo, int n_hi, float* a,
                                              float* b) {
  float ssq = 0.f;
  switch (p.kind) {
    case EPI_STORE_F32: {
      float* o = p.out_f32 + (size_t)m * p.ldo;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        *reinterpret_cast<float4*>(o + n_lo + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
        *reinterpret_cast<float4*>(o + n_hi + i) = make_float4(b[i], b[i + 1], b[i + 2], b[i + 3]);
      }
      break;
    }
    case EPI_RESID: {
      float* o = p.out_f32 + (size_t)m * p.ldo;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 x = *reinterpret_cast<float4*>(o + n_lo + i);
        float4 y = *reinterpret_cast<float4*>(o + n_hi + i);
        x.x += a[i]; x.y += a[i + 1]; x.z += a[i + 2]; x.w += a[i + 3];
        y.x += b[i]; y.y += b[i + 1]; y.z += b[i + 2]; y.w += b[i + 3];
        *reinterpret_cast<float4*>(o + n_lo + i) = x;
        *reinterpret_cast<float4*>(o + n_hi + i) = y;
        a[i] = x.x; a[i + 1] = x.y; a[i + 2] = x.z; a[i + 3] = x.w;
        b[i] = y.x; b[i + 1] = y.y; b[i + 2] = y.z; b[i + 3] = y.w;
      }
      if (p.xb_out) {
        // the chunk's sum of squares (four interleaved partial sums combined in a fixed order)
        // and the next GEMM's input, bf16(gamma * x)
        float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          q[i & 3] = fmaf(a[i], a[i], q[i & 3]);
          q[i & 3] = fmaf(b[i], b[i], q[i & 3]);
        }
        ssq = (q[0] + q[1]) + (q[2] + q[3]);
        if (p.xb_gamma) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] *= p.xb_gamma[n_lo + i];
            b[i] *= p.xb_gamma[n_hi + i];
          }
        }
        bf16* xb = p.xb_out + (size_t)m * p.ldo;
        store_bf16x32(xb + n_lo, a);
        store_bf16x32(xb + n_hi, b);
      }
      break;
    }
    case EPI_STORE_BF16: {
      bf16* o = p.out_bf16 + (size_t)m * p.ldo;
      store_bf16x32(o + n_lo, a);
      store_bf16x32(o + n_hi, b);
      break;
    }
    case EPI_SWIGLU: {
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = silu_f(a[i]) * b[i];
      store_bf16x32(p.out_bf16 + (size_t)m * p.ldo + (n_lo >> 7) * 64 + (n_lo & 127), a);
      break;
    }
    case EPI_QKV:
    case EPI_WIDE_KV: {
      if (p.bias) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          a[i] += p.bias[n_lo + i];
          b[i] += p.bias[n_hi + i];
        }
      }
      const int dh = p.d_head;
      const int kvc = p.n_kv * dh;
      if (p.kind == EPI_QKV && n_lo < p.q_cols) {
        const int pos = p.positions[m], i0 = n_lo % dh;
#pragma unroll
        for (int i = 0; i < 32; ++i) rope_rotate(p, pos, i0 + i, a[i], b[i]);
        bf16* o = p.out_bf16 + (size_t)m * p.ldo;
        store_bf16x32(o + n_lo, a);
        store_bf16x32(o + n_hi, b);
        break;
      }
      const int slot = p.slots[m];
      if (slot < 0) break;
      int c, cache;
      if (p.kind == EPI_QKV) {
        c = n_lo - p.q_cols;
        cache = p.cache_base;
      } else {
        int grp = n_lo / (2 * kvc);
        c = n_lo - grp * 2 * kvc;
        cache = p.cache_base + grp;
      }
      const int cs = p.kind == EPI_QKV ? n_lo - p.q_cols : n_lo;  // K/V column of the stage
      const bool is_k = c < kvc;
      if (!is_k) c -= kvc;
      const int head = c / dh, i0 = c % dh;
      if (is_k) {
        const int pos = p.positions[m];
#pragma unroll
        for (int i = 0; i < 32; ++i) rope_rotate(p, pos, i0 + i, a[i], b[i]);
      }
      if (p.kv_stage) {
        bf16* o = p.kv_stage + (size_t)m * p.kv_stage_ld + cs;
        store_bf16x32(o, a);
        store_bf16x32(o + (dh >> 1), b);
        break;
      }
      bf16* pool = is_k ? p.k_pools[cache] : p.v_pools[cache];
      bf16* row = pool + ((size_t)(slot >> 4) * p.n_kv + head) * kPageSize * dh + (size_t)(slot & 15) * dh;
      store_bf16x32(row + i0, a);
      store_bf16x32(row + i0 + (dh >> 1), b);
      break;
    }
    default:
      break;
  }
  return ssq;
}

// ---------------------------------------------------------------------------- float8 e4m3

// Two floats to e4m3 codes (round to nearest even, saturating at +-448); lo in bits 0..7.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
// Two e4m3 codes (bits 0..7 and 8..15) to an f16x2 (exact), the low code in the low half.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t codes16) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes16, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// ---------------------------------------------------------------------------- FP8 cache epilogue
//
// Per-token FP8 quantization fused into the QKV / wide-KV epilogue of the tcgen05 GEMMs: the
// epilogue thread of a row holds every column of one K or V head (the 2 * half columns of a
// pair block), so it rounds the head's values to bf16 (the values a bf16 cache would hold),
// takes their max magnitude, and writes scale = amax / 448 and the e4m3 codes of value /
// scale (float32 division, round to nearest even) - the arithmetic of the separate quantize
// pass - straight into the cache.

// Whether the pair block starting at column n0 is a K or V head quantized in the epilogue.
__device__ __forceinline__ bool fp8_head_block(const EpiParams& p, int n0) {
  return p.ks_pools != nullptr && (p.kind == EPI_WIDE_KV || (p.kind == EPI_QKV && n0 >= p.q_cols));
}

// Bias and (for K) RoPE of the K/V columns (n_lo + i, n_hi + i), i < 32, in place.
__device__ __forceinline__ void kv_chunk_prep(const EpiParams& p, int m, int n_lo, int n_hi, float* a, float* b) {
  if (p.bias) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      a[i] += p.bias[n_lo + i];
      b[i] += p.bias[n_hi + i];
    }
  }
  const int dh = p.d_head, kvc = p.n_kv * dh;
  const int c = p.kind == EPI_QKV ? n_lo - p.q_cols : n_lo % (2 * kvc);
  if (c < kvc) {
    const int pos = p.positions[m], i0 = c % dh;
#pragma unroll
    for (int i = 0; i < 32; ++i) rope_rotate(p, pos, i0 + i, a[i], b[i]);
  }
}

// Codes, scale and expansion of the head whose pair block starts at column n0 for row m; pk
// holds its DH values as bf16 pairs in dimension order, amax their largest magnitude.
template <int DH>
__device__ __forceinline__ void store_head_fp8(const EpiParams& p, int m, int n0, const uint32_t* pk, float amax) {
  const int slot = p.slots[m];
  if (slot < 0) return;
  constexpr int dh = DH;
  const int kvc = p.n_kv * dh;
  int c, cache;
  if (p.kind == EPI_QKV) {
    c = n0 - p.q_cols;
    cache = p.cache_base;
  } else {
    const int grp = n0 / (2 * kvc);
    c = n0 - grp * 2 * kvc;
    cache = p.cache_base + grp;
  }
  const bool is_k = c < kvc;
  const int head = (is_k ? c : c - kvc) / dh;
  const size_t rowoff = ((size_t)(slot >> 4) * p.n_kv + head) * kPageSize + (slot & 15);
  const float scale = amax / 448.f;
  uint8_t* dst = reinterpret_cast<uint8_t* const*>(is_k ? p.k_pools : p.v_pools)[cache] + rowoff * dh;
  bf16* ex = is_k ? p.exp_k : p.exp_v;
#pragma unroll
  for (int q = 0; q < dh / 16; ++q) {  // 16 dimensions per 16-byte store
    uint32_t w[4], e[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      uint32_t cc = 0;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t pr = pk[q * 8 + r * 2 + h2];
        const float v0 = __uint_as_float(pr << 16), v1 = __uint_as_float(pr & 0xffff0000u);
        const uint16_t c2 = scale > 0.f ? e4m3x2_from_f32(v0 / scale, v1 / scale) : (uint16_t)0;
        cc |= (uint32_t)c2 << (16 * h2);
        if (ex) {
          const uint32_t hh = f16x2_from_e4m3x2(c2);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh));
          e[r * 2 + h2] = pack_bf16_(f.x, f.y);
        }
      }
      w[r] = cc;
    }
    *reinterpret_cast<uint4*>(dst + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    if (ex) {
      bf16* er = ex + rowoff * dh + q * 16;
      *reinterpret_cast<uint4*>(er) = make_uint4(e[0], e[1], e[2], e[3]);
      *reinterpret_cast<uint4*>(er + 8) = make_uint4(e[4], e[5], e[6], e[7]);
    }
  }
  (is_k ? p.ks_pools : p.vs_pools)[cache][rowoff] = scale;
}

// ---------------------------------------------------------------------------- programmatic launch

// Lets the next kernel on the stream, if it was launched as a programmatic dependent, start
// (its blocks are then scheduled as this kernel's blocks leave; it must griddep_wait()
// before reading anything this kernel writes). Harmless for ordinary successors.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the kernels this one depends on have completed and their writes are visible;
// returns at once for a kernel launched without a programmatic dependency.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col)
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two softmax weights p0, p1 (>= 0, finite) as bfloat16 high and low parts, packed bf16x2
// with p0's part in the low half: the high part is p rounded to the nearest bf16, the low part
// the remainder (exact in float32, at most half a bf16 ulp of p) rounded to the nearest bf16,
// so hi + lo equals p to within 2^-18 |p|.
__device__ __forceinline__ void split_pair_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(p0, p1);
  lo = pack_bf16(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xffff0000u));
}

}  // namespace skv
