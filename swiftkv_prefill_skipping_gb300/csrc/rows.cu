// Row-wise and bookkeeping kernels: parameter-carried uploads, the prefill/decode
// plan (positions, paged slots, last-token rows), embedding + RMSNorm, RMSNorm
// (optionally gathering rows), argmax, and the load-time column scaling that folds
// an RMSNorm gain into the wide W_KV.
//
// RMSNorm rows are HBM-bound: one 128-thread CTA per row, 16-byte loads/stores,
// fp32 statistics, bf16 output.
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "pdl.cuh"

namespace skv {

namespace {

__global__ void upload_kernel(int* dst, IntBlob blob) {
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i < blob.n; i += blockDim.x * gridDim.x)
    dst[i] = blob.v[i];
}

__global__ void plan_prefill_kernel(const int* __restrict__ cu, const int* __restrict__ ctx, int P, int T,
                                    const int* __restrict__ tokens,
                                    int vocab, const int* __restrict__ bt, int max_pages, int num_pages,
                                    int* positions, int* slots, int* last_idx, int* last_pos, int* status) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += blockDim.x * gridDim.x) {
    int lo = 0, hi = P - 1;  // largest s with cu[s] <= t
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    const int s = lo;
    const int c0 = ctx ? ctx[s] : 0;
    const int pos = c0 + t - cu[s];
    const int n = c0 + cu[s + 1] - cu[s];  // the sequence's length after this chunk
    const int page = bt[(size_t)s * max_pages + (pos >> 4)];
    const bool ok = page >= 0 && page < num_pages;
    if (!ok) atomicOr(status, kStatusBadPage);
    positions[t] = pos;
    slots[t] = ok ? page * kPageSize + (pos & 15) : -1;
    if (pos == n - 1) {
      last_idx[s] = t;
      last_pos[s] = pos;
    }
    const int tok = tokens[t];
    if (tok < 0 || tok >= vocab) atomicOr(status, kStatusBadToken);
  }
}

__global__ void plan_decode_kernel(const int* __restrict__ seq_lens, int B, const int* __restrict__ tokens,
                                   int vocab, const int* __restrict__ bt, int max_pages, int num_pages,
                                   int* positions, int* slots, int* status) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += blockDim.x * gridDim.x) {
    const int pos = seq_lens[b];
    const int page = bt[(size_t)b * max_pages + (pos >> 4)];
    const bool ok = page >= 0 && page < num_pages;
    if (!ok) atomicOr(status, kStatusBadPage);
    positions[b] = pos;
    slots[b] = ok ? page * kPageSize + (pos & 15) : -1;
    const int tok = tokens[b];
    if (tok < 0 || tok >= vocab) atomicOr(status, kStatusBadToken);
  }
}

constexpr int RN_THREADS = 128;
constexpr int RN_MAXV = 16;  // float4 per thread: d <= 8192

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < RN_THREADS / 32; ++w) s += red[w];
  return s;
}

__device__ __forceinline__ void store_bf16x4(bf16* dst, float4 v) {
  uint2 pk;
  pk.x = pack_bf16(v.x, v.y);
  pk.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = pk;
}

// Embedding row of each token into the fp32 residual stream x, and the first layer's input:
// without ss_part, u = bf16(RMSNorm(x) * gamma) (gamma NULL: 1); with ss_part (the fused-norm
// path), u = bf16(gamma * x) and the row's sum of squares goes to ss_part[t][0] with zeros in
// the other nparts - 1 slots, so a consumer summing the slots gets exactly the sum the unfused
// path normalises by.
__global__ void __launch_bounds__(RN_THREADS) embed_rmsnorm_kernel(const int* __restrict__ tokens,
                                                                   const bf16* __restrict__ embed, int vocab,
                                                                   int d, const float* __restrict__ gamma,
                                                                   float eps, float* __restrict__ x,
                                                                   bf16* __restrict__ u, float* __restrict__ ss_part,
                                                                   int nparts) {
  __shared__ float red[RN_THREADS / 32];
  const int t = blockIdx.x;
  int tok = tokens[t];
  if (tok < 0 || tok >= vocab) tok = 0;
  const bf16* e = embed + (size_t)tok * d;
  const int n4 = d >> 2;
  float4 v[RN_MAXV];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < RN_MAXV; ++i) {
    int c = threadIdx.x + i * RN_THREADS;
    if (c < n4) {
      uint2 raw = *reinterpret_cast<const uint2*>(e + 4 * c);
      __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
      __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
      float2 f0 = __bfloat1622float2(p0), f1 = __bfloat1622float2(p1);
      v[i] = make_float4(f0.x, f0.y, f1.x, f1.y);
      ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
      reinterpret_cast<float4*>(x + (size_t)t * d)[c] = v[i];
      if (ss_part) {
        const float4 g = gamma ? reinterpret_cast<const float4*>(gamma)[c] : make_float4(1.f, 1.f, 1.f, 1.f);
        store_bf16x4(u + (size_t)t * d + 4 * c, make_float4(v[i].x * g.x, v[i].y * g.y, v[i].z * g.z, v[i].w * g.w));
      }
    }
  }
  const float total = block_sum(ss, red);
  if (ss_part) {
    for (int i = threadIdx.x; i < nparts; i += RN_THREADS) ss_part[(size_t)t * nparts + i] = i ? 0.f : total;
    return;
  }
  const float r = rsqrtf(total / d + eps);
#pragma unroll
  for (int i = 0; i < RN_MAXV; ++i) {
    int c = threadIdx.x + i * RN_THREADS;
    if (c < n4) {
      const float4 g = gamma ? reinterpret_cast<const float4*>(gamma)[c] : make_float4(1.f, 1.f, 1.f, 1.f);
      float4 o = make_float4(v[i].x * r * g.x, v[i].y * r * g.y, v[i].z * r * g.z, v[i].w * r * g.w);
      store_bf16x4(u + (size_t)t * d + 4 * c, o);
    }
  }
}

// One row per CTA; each thread owns 8-element chunks (two 16-byte fp32 loads, one 16-byte
// bf16 store), so every global access is a full 16-byte vector.
__global__ void __launch_bounds__(RN_THREADS) rmsnorm_kernel(const float* __restrict__ x,
                                                             const int* __restrict__ rows, int d,
                                                             const float* __restrict__ gamma, float eps,
                                                             bf16* __restrict__ u, float* __restrict__ x_out) {
  griddep_launch_dependents();  // a programmatic dependent may start as these blocks leave
  griddep_wait();               // itself launched as one: x is the previous kernel's output
  __shared__ float red[RN_THREADS / 32];
  constexpr int MAXC = RN_MAXV / 2;  // 8-element chunks per thread: d <= 8192
  const int t = blockIdx.x;
  const int src = rows ? rows[t] : t;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)src * d);
  const int n8 = d >> 3;
  float4 v[MAXC][2];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    const int c = threadIdx.x + i * RN_THREADS;
    if (c < n8) {
      v[i][0] = xr[2 * c];
      v[i][1] = xr[2 * c + 1];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        ss += v[i][h].x * v[i][h].x + v[i][h].y * v[i][h].y + v[i][h].z * v[i][h].z + v[i][h].w * v[i][h].w;
      if (x_out) {
        reinterpret_cast<float4*>(x_out + (size_t)t * d)[2 * c] = v[i][0];
        reinterpret_cast<float4*>(x_out + (size_t)t * d)[2 * c + 1] = v[i][1];
      }
    }
  }
  const float r = rsqrtf(block_sum(ss, red) / d + eps);
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    const int c = threadIdx.x + i * RN_THREADS;
    if (c < n8) {
      float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
      if (gamma) {
        g0 = reinterpret_cast<const float4*>(gamma)[2 * c];
        g1 = reinterpret_cast<const float4*>(gamma)[2 * c + 1];
      }
      uint4 pk;
      pk.x = pack_bf16(v[i][0].x * r * g0.x, v[i][0].y * r * g0.y);
      pk.y = pack_bf16(v[i][0].z * r * g0.z, v[i][0].w * r * g0.w);
      pk.z = pack_bf16(v[i][1].x * r * g1.x, v[i][1].y * r * g1.y);
      pk.w = pack_bf16(v[i][1].z * r * g1.z, v[i][1].w * r * g1.w);
      *reinterpret_cast<uint4*>(u + (size_t)t * d + 8 * c) = pk;
    }
  }
}

__global__ void argmax_kernel(const float* __restrict__ logits, int V, int* __restrict__ out) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const float* row = logits + (size_t)blockIdx.x * V;
  float best = -FLT_MAX;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    float v = row[i];
    if (v > best) {  // strided scan visits indices in increasing order: keeps the first maximum
      best = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, best, o);
    int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (v2 > best || (v2 == best && i2 < bi)) {
      best = v2;
      bi = i2;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (sv[w] > best || (sv[w] == best && si[w] < bi)) {
        best = sv[w];
        bi = si[w];
      }
    out[blockIdx.x] = bi == 0x7fffffff ? 0 : bi;
  }
}

__global__ void scale_columns_kernel(bf16* W, size_t total, int K, const float* __restrict__ gamma) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x)
    W[i] = __float2bfloat16_rn(__bfloat162float(W[i]) * gamma[i % K]);
}

}  // namespace

cudaError_t launch_upload(int* dst, const IntBlob& blob, cudaStream_t stream) {
  if (blob.n <= 0) return cudaSuccess;
  upload_kernel<<<(blob.n + 255) / 256, 256, 0, stream>>>(dst, blob);
  return cudaGetLastError();
}

cudaError_t upload_ints(int* dst, const int* src, int n, cudaStream_t stream) {
  IntBlob blob;
  for (int off = 0; off < n; off += kBlobInts) {
    blob.n = n - off < kBlobInts ? n - off : kBlobInts;
    for (int i = 0; i < blob.n; ++i) blob.v[i] = src[off + i];
    cudaError_t e = launch_upload(dst + off, blob, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {

// ---------------------------------------------------------------------------- FP8 KV cache

// One warp per staged (row m, group, K/V, head) vector of d_head bf16 values: per-vector
// scale amax / 448, e4m3 codes of value / scale (float32 division, round to nearest even)
// into the paged uint8 pool at the row's slot, the scale into the scale pool; with `sk`/`sv`
// (groups == 1) the codes also go, as bf16 (exact: e4m3 values are bf16 values), into bf16
// expansion pools of the same layout for the prompt-tile attention, which applies the scales
// itself in float32.
template <int E>
__global__ void kv_quantize_kernel(const bf16* __restrict__ stage, int ld, int M, const int* __restrict__ slots,
                                   int groups, int n_kv, int cache_base, uint8_t* const* k8, uint8_t* const* v8,
                                   float* const* ks, float* const* vs, bf16* sk, bf16* sv) {
  constexpr int DH = E * 32;
  const int lane = threadIdx.x & 31;
  const long long vid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int per_row = groups * 2 * n_kv;
  if (vid >= (long long)M * per_row) return;
  const int m = (int)(vid / per_row);
  int r = (int)(vid - (long long)m * per_row);
  const int grp = r / (2 * n_kv);
  r -= grp * 2 * n_kv;
  const int kvsel = r / n_kv, head = r - kvsel * n_kv;
  const int slot = slots[m];
  if (slot < 0) return;
  const int kvc = n_kv * DH;
  const bf16* src = stage + (size_t)m * ld + (size_t)grp * 2 * kvc + kvsel * kvc + head * DH + lane * E;
  float v[E];
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i));
    v[i] = f.x;
    v[i + 1] = f.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax / 448.f;
  uint16_t c2[E / 2];
#pragma unroll
  for (int i = 0; i < E; i += 2)
    c2[i / 2] = scale > 0.f ? e4m3x2_from_f32(v[i] / scale, v[i + 1] / scale) : (uint16_t)0;
  const int cache = cache_base + grp;
  const size_t rowoff = ((size_t)(slot >> 4) * n_kv + head) * kPageSize + (slot & 15);
  uint8_t* dst = (kvsel ? v8[cache] : k8[cache]) + rowoff * DH + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint32_t*>(dst) = (uint32_t)c2[0] | ((uint32_t)c2[1] << 16);
  } else {
    *reinterpret_cast<uint16_t*>(dst) = c2[0];
  }
  if (lane == 0) (kvsel ? vs[cache] : ks[cache])[rowoff] = scale;
  bf16* ex = kvsel ? sv : sk;
  if (ex) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint32_t h = f16x2_from_e4m3x2(c2[i / 2]);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
      *reinterpret_cast<__nv_bfloat162*>(ex + rowoff * DH + lane * E + i) = __floats2bfloat162_rn(f.x, f.y);
    }
  }
}

// Expands whole (page, all heads) blocks of one cache's uint8 code pools into bf16 pools of
// the same layout (exact: e4m3 values are bf16 values; the attention applies the scales):
// item i = (sequence, page index) pairs; 16 codes per thread-step.
__global__ void kv_dequant_pages_kernel(const int* __restrict__ items, const int* __restrict__ bt, int max_pages,
                                        int num_pages, int n_kv, int dh, const uint8_t* __restrict__ k8,
                                        const uint8_t* __restrict__ v8, bf16* sk, bf16* sv) {
  const int s = items[2 * blockIdx.x], pidx = items[2 * blockIdx.x + 1];
  const int page = bt[(size_t)s * max_pages + pidx];
  if (page < 0 || page >= num_pages) return;
  const int per_page = n_kv * kPageSize * dh;  // codes of one page, all heads
  const size_t base = (size_t)page * per_page;
  for (int c = threadIdx.x; c < 2 * per_page / 16; c += blockDim.x) {
    const int kvsel = c >= per_page / 16;
    const int e = (c - kvsel * (per_page / 16)) * 16;  // element within the page
    const uint4 raw = *reinterpret_cast<const uint4*>((kvsel ? v8 : k8) + base + e);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t h = f16x2_from_e4m3x2((w[i] >> (16 * hh)) & 0xffffu);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x, f.y);
        o[2 * i + hh] = *reinterpret_cast<uint32_t*>(&b2);
      }
    }
    bf16* dst = (kvsel ? sv : sk) + base + e;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_kv_quantize(const bf16* stage, int ld, int M, const int* slots, int groups, int n_kv, int d_head,
                               int cache_base, uint8_t* const* k8, uint8_t* const* v8, float* const* ks,
                               float* const* vs, bf16* sk, bf16* sv, cudaStream_t stream) {
  const long long vecs = (long long)M * groups * 2 * n_kv;
  if (vecs <= 0) return cudaSuccess;
  const int blocks = (int)((vecs * 32 + 255) / 256);
  if (d_head == 128)
    kv_quantize_kernel<4><<<blocks, 256, 0, stream>>>(stage, ld, M, slots, groups, n_kv, cache_base, k8, v8, ks, vs,
                                                      sk, sv);
  else if (d_head == 64)
    kv_quantize_kernel<2><<<blocks, 256, 0, stream>>>(stage, ld, M, slots, groups, n_kv, cache_base, k8, v8, ks, vs,
                                                      sk, sv);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_kv_dequant_pages(const int* items, int num_items, const int* block_table, int max_pages,
                                    int num_pages, int n_kv, int d_head, const uint8_t* k8, const uint8_t* v8,
                                    bf16* sk, bf16* sv, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  kv_dequant_pages_kernel<<<num_items, 256, 0, stream>>>(items, block_table, max_pages, num_pages, n_kv, d_head, k8,
                                                          v8, sk, sv);
  return cudaGetLastError();
}

cudaError_t launch_plan_prefill(const int* cu, const int* ctx, int P, int T, const int* tokens, int vocab,
                                const int* block_table, int max_pages, int num_pages, int* positions,
                                int* slots, int* last_idx, int* last_pos, int* status,
                                cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  int blocks = (T + 255) / 256;
  plan_prefill_kernel<<<blocks, 256, 0, stream>>>(cu, ctx, P, T, tokens, vocab, block_table, max_pages,
                                                   num_pages, positions, slots, last_idx, last_pos,
                                                   status);
  return cudaGetLastError();
}

cudaError_t launch_plan_decode(const int* seq_lens, int B, const int* tokens, int vocab,
                               const int* block_table, int max_pages, int num_pages, int* positions,
                               int* slots, int* status, cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  plan_decode_kernel<<<(B + 255) / 256, 256, 0, stream>>>(seq_lens, B, tokens, vocab, block_table,
                                                          max_pages, num_pages, positions, slots, status);
  return cudaGetLastError();
}

cudaError_t launch_embed_rmsnorm(const int* tokens, int T, const bf16* embed, int vocab, int d,
                                 const float* gamma, float eps, float* x, bf16* u, float* ss_part, int nparts,
                                 cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  embed_rmsnorm_kernel<<<T, RN_THREADS, 0, stream>>>(tokens, embed, vocab, d, gamma, eps, x, u, ss_part, nparts);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, const int* rows, int T, int d, const float* gamma,
                           float eps, bf16* u, float* x_out, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  return launch_pdl(rmsnorm_kernel, dim3(T), dim3(RN_THREADS), 0, stream, x, rows, d, gamma, eps, u, x_out);
}

cudaError_t launch_argmax(const float* logits, int rows, int V, int* out, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  argmax_kernel<<<rows, 1024, 0, stream>>>(logits, V, out);
  return cudaGetLastError();
}

cudaError_t launch_scale_columns(bf16* W, int rows, int K, const float* gamma, cudaStream_t stream) {
  size_t total = (size_t)rows * K;
  if (total == 0) return cudaSuccess;
  scale_columns_kernel<<<1024, 256, 0, stream>>>(W, total, K, gamma);
  return cudaGetLastError();
}

}  // namespace skv
