// Internal launchers of the SwiftKV GB300 kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <vector>

#include "common.cuh"

namespace skv {

// Raises a kernel's dynamic shared-memory limit on the current device, once per device: the
// attribute belongs to the device that is current when it is set, so a process driving
// several GPUs sets it on each. Safe to call from several threads (setting it twice is
// harmless; the per-device bit is atomic). Devices past 63 set it on every call.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
};
inline cudaError_t set_max_dynamic_smem(const void* func, int bytes, PerDeviceOnce& once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (once.done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) once.done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Records `msg` as the calling thread's swiftkv_last_error() and returns `code`.
int set_error(int code, const char* msg);

// ---- GEMMs (C = A * B^T with an epilogue) -----------------------------------------------
cudaError_t launch_gemm_tiled(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                              cudaStream_t stream);
int skinny_splits(int M, int N, int K, int num_sms);
size_t skinny_scratch_bytes(int M, int N, int K, int num_sms);
cudaError_t launch_gemm_skinny(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                               float* scratch, int num_sms, cudaStream_t stream);
// M <= 64 without split-K: each CTA streams 32 weight rows over the full K (no scratch).
cudaError_t launch_gemv(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep, cudaStream_t stream);
// Persistent TMA-fed skinny GEMM for M <= 64 over 64-row weight tiles; cudaErrorNotSupported
// outside its shapes, including matrices with fewer than num_sms / 2 tiles (launch_gemv then).
cudaError_t launch_gemv_tma(const bf16* A, int lda, const bf16* W, int K, const EpiParams& ep, int num_sms,
                            int* status, cudaStream_t stream);
// A chain of skinny GEMM and RMSNorm phases (M <= 64 rows) in one cooperative persistent
// launch: phase p runs after every CTA has finished phase p - 1 (grid barrier on a
// monotonically growing arrival counter; count_base is the count before the launch and is
// advanced by the barriers the launch makes). Weights of later GEMM phases stream while
// earlier phases run. cudaErrorNotSupported outside its shapes.
constexpr int kChainMaxPhases = 6;
struct ChainNorm {        // u[m][:] = bf16(rmsnorm(x[m][:]) * gamma), m < rows
  const float* x;
  const float* gamma;     // NULL: 1
  bf16* u;
  int rows, d, ldx, ldu;
  float eps;
};
struct ChainStep {        // one phase: a GEMM (W != NULL) or an RMSNorm (W == NULL)
  const bf16* A;
  int lda;
  const bf16* W;          // [N][K]
  int K;
  EpiParams ep;
  ChainNorm norm;
};
struct ChainPhase {
  CUtensorMap tmA, tmW;
  EpiParams ep;
  ChainNorm norm;
  int is_norm, K, tiles, first_cta;  // tiles: 64-row weight tiles, or rows for a norm phase
};
struct ChainParams {
  ChainPhase ph[kChainMaxPhases];
  int n;
  unsigned* count;
  unsigned count_base;
};
cudaError_t launch_gemv_chain(const ChainStep* steps, int n, int num_sms, unsigned* count, unsigned* count_base,
                              int* status, cudaStream_t stream);
// tcgen05 (TMEM accumulator, TMA-fed) GEMM; returns cudaErrorNotSupported if the shape is not
// handled, so the caller can fall back to launch_gemm_tiled.
// mode 0: one CTA per 128 x 256 tile; 2: CTA pairs run tcgen05.mma.cta_group::2 on
// 256 x 256 tiles (any other mode: cudaErrorNotSupported).
cudaError_t launch_gemm_tc(const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
                           int num_sms, int* status, cudaStream_t stream, int mode = 0);

// ---- bookkeeping ------------------------------------------------------------------------
constexpr int kBlobInts = 2000;
struct IntBlob {
  int n;
  int v[kBlobInts];
};
// dst[0..blob.n) = blob.v (host data carried in the kernel's parameters).
cudaError_t launch_upload(int* dst, const IntBlob& blob, cudaStream_t stream);
cudaError_t upload_ints(int* dst, const int* src, int n, cudaStream_t stream);

// positions / slots / last index of a packed prefill batch; validates tokens and pages.
// ctx (device, nullable = all zero): tokens already cached per sequence; chunk row i of
// sequence s sits at position ctx[s] + i.
cudaError_t launch_plan_prefill(const int* cu, const int* ctx, int P, int T, const int* tokens, int vocab,
                                const int* block_table, int max_pages, int num_pages, int* positions,
                                int* slots, int* last_idx, int* last_pos, int* status,
                                cudaStream_t stream);
// decode: one token per sequence at position seq_lens[b].
cudaError_t launch_plan_decode(const int* seq_lens, int B, const int* tokens, int vocab,
                               const int* block_table, int max_pages, int num_pages, int* positions,
                               int* slots, int* status, cudaStream_t stream);

// ---- FP8 KV cache -------------------------------------------------------------------------
// Quantizes staged K/V rows (stage [M][ld]: per group [K heads | V heads] of d_head bf16
// values) per (row, group, K/V, head) into uint8 e4m3 pools (device arrays of pool pointers,
// cache cache_base + group) with float32 scales [num_pages][n_kv][16]; rows with slot < 0
// are skipped. sk/sv (groups == 1, may be null): bf16 expansion pools written as well.
cudaError_t launch_kv_quantize(const bf16* stage, int ld, int M, const int* slots, int groups, int n_kv, int d_head,
                               int cache_base, uint8_t* const* k8, uint8_t* const* v8, float* const* ks,
                               float* const* vs, bf16* sk, bf16* sv, cudaStream_t stream);
// Expands the (page, all heads) blocks named by items [2 * num_items] = (sequence, page index
// in its block-table row) of one cache into bf16 pools sk/sv of the same layout.
cudaError_t launch_kv_dequant_pages(const int* items, int num_items, const int* block_table, int max_pages,
                                    int num_pages, int n_kv, int d_head, const uint8_t* k8, const uint8_t* v8,
                                    bf16* sk, bf16* sv, cudaStream_t stream);

// ---- row kernels -------------------------------------------------------------------------
// x[t] = embed[tok[t]] (fp32); u[t] = bf16(rmsnorm(x[t]) * gamma) (gamma NULL: 1), or with
// ss_part (fused-norm path) u[t] = bf16(gamma * x[t]) and the row's sum of squares in
// ss_part[t][0] (zeros in the other nparts - 1 slots)
cudaError_t launch_embed_rmsnorm(const int* tokens, int T, const bf16* embed, int vocab, int d,
                                 const float* gamma, float eps, float* x, bf16* u, float* ss_part, int nparts,
                                 cudaStream_t stream);
// u[t] = bf16(rmsnorm(x[rows ? rows[t] : t]) * gamma); if x_out, x_out[t] = x[row] (gather).
// gamma == nullptr means a gain of one.
cudaError_t launch_rmsnorm(const float* x, const int* rows, int T, int d, const float* gamma,
                           float eps, bf16* u, float* x_out, cudaStream_t stream);
cudaError_t launch_argmax(const float* logits, int rows, int V, int* out, cudaStream_t stream);
// W[n][k] = bf16(float(W[n][k]) * gamma[k]) for n < rows
cudaError_t launch_scale_columns(bf16* W, int rows, int K, const float* gamma, cudaStream_t stream);

// ---- attention ---------------------------------------------------------------------------
// Varlen causal GQA attention of packed prompt chunks against their own paged K/V.
// tiles: [num_tiles] (seq << 16 | q_tile) 64-row query tiles; cu: [P+1] device; ctx: [P]
// device or nullptr: cached tokens before each chunk (row i at position ctx[s] + i sees
// keys [0, ctx[s] + i]).
// k_scale / v_scale (all three prompt kernels): NULL for a bf16 cache; for an FP8 cache the
// pools hold the e4m3 codes as bf16 values and these the per-(page, head, row) float scales
// [num_pages][n_kv][16]: scores take the key's scale and P the value's, in float32.
cudaError_t launch_attention_prefill(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                     const float* k_scale, const float* v_scale,
                                     const int* block_table, int max_pages, int num_pages,
                                     const int* cu, const int* ctx, const int* tiles, int num_tiles, int n_q,
                                     int n_kv, int d_head, bf16* out, int ldo, cudaStream_t stream);
// Same on tcgen05 with two 128-row query tiles per CTA sharing every K/V block (d_head 128
// only), heaviest tiles first. head_pairs (n_q / n_kv even): tiles are 128-row tiles
// (seq << 16 | tile) and an item is one tile for two query heads of one KV head; otherwise
// tiles are 256-row tile pairs (seq << 16 | pair) and an item is one pair for one head.
// Persistent: at most num_sms CTAs, each walking its share of the items.
cudaError_t launch_attention_prefill_tc2(const bf16* q, int ldq, int T, const bf16* k_pool, const bf16* v_pool,
                                         const float* k_scale, const float* v_scale, const int* block_table, int max_pages, int num_pages, const int* cu,
                                         const int* ctx, const int* tiles, int num_tiles, int n_q, int n_kv,
                                         int d_head, bf16* out, int ldo, int num_sms, int* status,
                                         cudaStream_t stream, bool head_pairs);
// Same on tcgen05 (d_head 128 only; cudaErrorNotSupported otherwise). tiles are 128-row tiles;
// T = rows of q. status receives kStatusTimeout if a bounded wait expires.
cudaError_t launch_attention_prefill_tc(const bf16* q, int ldq, int T, const bf16* k_pool, const bf16* v_pool,
                                        const float* k_scale, const float* v_scale, const int* block_table, int max_pages, int num_pages, const int* cu,
                                        const int* ctx, const int* tiles, int num_tiles, int n_q, int n_kv,
                                        int d_head, bf16* out, int ldo, int* status, cudaStream_t stream);
// B single query rows: item b is row r = rows[b] of q / out (r = b if rows is null) at
// position qpos[r], attending to keys 0..qpos[r] of block table row seqs[b] (b if null).
cudaError_t launch_attention_decode(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                    const int* block_table, int max_pages, int num_pages,
                                    const int* qpos, int B, int n_q, int n_kv, int d_head, bf16* out,
                                    int ldo, cudaStream_t stream, const int* rows = nullptr,
                                    const int* seqs = nullptr);

// Key-split single-row attention (decode tokens, SwiftKV tail rows, rows of short chunks).
// Items b = 0..num_items-1 are mapped as in launch_attention_decode (rows / seqs / qpos);
// units [3 * num_units] = (item, first key, keys), item-major with keys ascending; ubeg
// [num_items + 1] = first unit of each item; part = split_part_floats(num_units, ...) floats.
struct SplitPlan {
  const int* units;
  const int* ubeg;
  int num_units, num_items;
  bool any_split;  // some item has more than one unit (the combine pass runs)
  float* part;
};
// Host: splits item b's nkeys[b] keys into units of split_keys_for(nkeys[b]) keys (a
// multiple of 64 that depends on nothing but the row's own length): 128 for rows of up to
// kShortRowKeys keys (more, smaller units keep short-context decode batches busy), 256 above
// (fewer partials to combine for long contexts).
constexpr int kSplitKeys = 256;
constexpr int kShortRowKeys = 1024;
int split_keys_for(int nkeys);
void split_plan_host(const int* nkeys, int items, std::vector<int>* units, std::vector<int>* ubeg);
size_t split_part_floats(int num_units, int n_q, int d_head);
// The same over an FP8 cache: uint8 e4m3 pools and float32 scales [num_pages][n_kv][16].
cudaError_t launch_attention_decode_split_fp8(const bf16* q, int ldq, const uint8_t* k8, const uint8_t* v8,
                                              const float* k_scale, const float* v_scale, const int* block_table,
                                              int max_pages, int num_pages, const int* qpos, const int* rows,
                                              const int* seqs, const SplitPlan& plan, int n_q, int n_kv, int d_head,
                                              bf16* out, int ldo, int num_sms, cudaStream_t stream);
cudaError_t launch_attention_decode_split(const bf16* q, int ldq, const bf16* k_pool, const bf16* v_pool,
                                          const int* block_table, int max_pages, int num_pages, const int* qpos,
                                          const int* rows, const int* seqs, const SplitPlan& plan, int n_q,
                                          int n_kv, int d_head, bf16* out, int ldo, int num_sms,
                                          cudaStream_t stream);

}  // namespace skv
