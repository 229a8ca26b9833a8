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
};

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
__device__ __forceinline__ void apply_chunk32(const EpiParams& p, int m, int n_lo, int n_hi, float* a,
                                              float* b) {
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

}  // namespace skv
