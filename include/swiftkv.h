/*
 * swiftkv.h — C ABI of the SwiftKV prefill-skipping library for one NVIDIA GB300 (sm_103a).
 *
 * The method ("SwiftKV: Fast Prefill-Optimized Inference with Knowledge-Preserving
 * Model Transformation", section 3.2 and section 3.4 "The SwiftKV Rewiring Mechanism",
 * Eq. 2; the paper's section 3.5 "Optimized Implementation for Inference"):
 * prompt tokens run the decoder only through layer l; the K/V caches of every
 * later layer j > l are projected from x_{l+1}, the output of layer l, as
 * KV_j = W_KV^j x_{l+1}; with AcrossKV each group of g consecutive skipped
 * layers shares one cache projected with the group's first layer's W_KV; the
 * skipped layers' Q/attention/O/MLP never run on prompt tokens, except for the
 * last token of each prompt, which runs every layer to produce the logits of
 * the first output token.
 *
 * Conventions
 *  - l counts full layers (layers 1..l run in full); 1 <= l <= L. l == L is the
 *    ordinary model. acrosskv_group g >= 1 must divide L - l.
 *  - Matrices are bfloat16 bit patterns (uint16_t) in nn.Linear layout [out][in],
 *    row-major. Gains and biases are float.
 *  - "device" pointers are CUDA device memory of the current device; "host"
 *    pointers are ordinary (pageable or pinned) host memory.
 *  - All GPU work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) without synchronising, unless a function says otherwise. Host
 *    arrays are fully read before the call returns.
 *  - Return value: SWIFTKV_OK (0) or a negative swiftkv_error. Errors never abort
 *    the process and never trap on the device; swiftkv_last_error() describes the
 *    last failure of the calling thread.
 *  - Data-dependent checks that need device data (token ids < vocab, page ids <
 *    num_pages) are done by the kernels: a violation sets a bit in the model's
 *    device status word (swiftkv_status) and the offending read/write is skipped
 *    or clamped in bounds.
 */
#ifndef SWIFTKV_H
#define SWIFTKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* swiftkv_stream; /* == cudaStream_t */

enum swiftkv_error {
  SWIFTKV_OK = 0,
  SWIFTKV_EINVAL = -1,         /* null pointer, bad size or config field */
  SWIFTKV_EINVAL_L = -2,       /* l outside [1, L], or different from the loaded model's */
  SWIFTKV_EINVAL_GROUP = -3,   /* g < 1, (L - l) % g != 0, or different from the model's */
  SWIFTKV_EINVAL_SEQLENS = -4, /* cu_seqlens not starting at 0 / a prompt shorter than 1 token */
  SWIFTKV_ENO_PAGES = -5,      /* a sequence needs more pages than its block-table row holds */
  SWIFTKV_EOOM = -6,           /* device allocation failed */
  SWIFTKV_ECUDA = -7,          /* a CUDA runtime call or launch failed */
  SWIFTKV_EDEVICE = -8,        /* reserved: device status word reported a violation */
  SWIFTKV_EUNSUPPORTED = -9,   /* shape outside what the kernels implement */
  SWIFTKV_ESTATE = -10         /* weights not (fully) loaded */
};

/* Bits of the device status word. */
enum swiftkv_status_bits {
  SWIFTKV_STATUS_BAD_TOKEN = 1, /* a token id outside [0, vocab): row 0 was used */
  SWIFTKV_STATUS_BAD_PAGE = 2,  /* a block-table entry outside [0, num_pages): access skipped */
  SWIFTKV_STATUS_TIMEOUT = 4    /* a bounded wait inside a kernel expired; that kernel's output is invalid */
};

/* Shape of the decoder (Llama / Qwen family: RMSNorm, GQA attention with RoPE,
 * SwiGLU MLP, untied LM head). Supported: d_head in {64, 128}; n_q % n_kv == 0;
 * d, n_q*d_head multiples of 128; vocab a multiple of 128. */
typedef struct {
  int L;            /* decoder layers */
  int d;            /* model width */
  int n_q;          /* query heads */
  int n_kv;         /* key/value heads */
  int d_head;       /* head dim */
  int ffn;          /* SwiGLU intermediate width */
  int vocab;        /* vocabulary size */
  int qkv_bias;     /* 1: Q/K/V projections carry a bias (added before RoPE) */
  float rope_theta; /* RoPE base; rotate-half pairs (i, i + d_head/2), no scaling */
  float rms_eps;    /* RMSNorm epsilon */
} swiftkv_model_config;

/* One decoder layer's weights in host memory. */
typedef struct {
  const float* gamma_attn; /* [d] input RMSNorm gain */
  const uint16_t* wq;      /* [n_q*d_head][d] */
  const uint16_t* wk;      /* [n_kv*d_head][d] */
  const uint16_t* wv;      /* [n_kv*d_head][d] */
  const float* bq;         /* [n_q*d_head]  (NULL unless qkv_bias) */
  const float* bk;         /* [n_kv*d_head] (NULL unless qkv_bias) */
  const float* bv;         /* [n_kv*d_head] (NULL unless qkv_bias) */
  const uint16_t* wo;      /* [d][n_q*d_head] */
  const float* gamma_mlp;  /* [d] */
  const uint16_t* w_gate;  /* [ffn][d] */
  const uint16_t* w_up;    /* [ffn][d] */
  const uint16_t* w_down;  /* [d][ffn] */
} swiftkv_layer_weights;

/* All weights in host memory. */
typedef struct {
  const uint16_t* embed;              /* [vocab][d] */
  const float* gamma_final;           /* [d] */
  const uint16_t* lm_head;            /* [vocab][d] */
  const swiftkv_layer_weights* layers; /* [L] */
} swiftkv_host_weights;

/* Paged KV cache, owned by the caller (device memory).
 * There are num_caches = swiftkv_cache_count(L, l, g) caches: caches 0..l-1
 * belong to the full layers, cache l + i to the i-th group of skipped layers.
 * Each cache has a K pool and a V pool of [num_pages][n_kv][page_size][d_head]
 * elements: one (page, head) block of page_size * d_head elements is contiguous.
 * Token at position p of sequence s lives in page block_table[s][p / page_size],
 * row p % page_size.
 * kv_dtype 0: bf16 elements. kv_dtype 1: per-token FP8 ("SwiftKV" summary, AcrossKV,
 * complementarity with KV quantization, Appendix B.1 / Table B.1): uint8 float8-e4m3
 * codes, and for every (page, head, row) one float32 scale in k_scale / v_scale pools of
 * [num_pages][n_kv][page_size]; the value is code * scale, scale = max|v| / 448 over the
 * token's d_head values of that head (K after RoPE). */
typedef struct {
  void* const* k_pool;        /* host array [num_caches] of device pointers */
  void* const* v_pool;        /* host array [num_caches] of device pointers */
  int num_caches;
  int num_pages;
  int page_size;              /* must be 16 */
  const int32_t* block_table; /* device int32 [num_seqs][max_pages_per_seq] */
  int max_pages_per_seq;
  int kv_dtype;               /* 0 bf16, 1 fp8 e4m3 + per-token scales */
  void* const* k_scale;       /* kv_dtype 1: host array [num_caches] of device float pools; else NULL */
  void* const* v_scale;
} swiftkv_kv_pages;

typedef struct swiftkv_model swiftkv_model; /* opaque; owns device weights + workspace */

/* Number of KV caches for (L, l, g): l + (L - l)/g ("SwiftKV" summary, section 3.4
 * AcrossKV, "Memory reduction"). Negative swiftkv_error for invalid arguments. */
int swiftkv_cache_count(int L, int l, int acrosskv_group);

/* Creates an empty model for (cfg, l, g) on the current device. Device memory for
 * all weights is allocated here. The W_KV packing of the skipped layers depends on
 * (l, g), so both are fixed for the model's lifetime. */
int swiftkv_model_create(const swiftkv_model_config* cfg, int l, int acrosskv_group,
                         swiftkv_model** out);

/* Copies layer j's (0-based) weights from host memory, packing them for the kernels:
 * Q/K/V concatenated (full layers), gate/up interleaved in 64-row blocks, and for a
 * skipped layer that represents an AcrossKV group, its W_K/W_V (rows scaled by its
 * gamma_attn, rounded to bf16) into the wide W_KV of all groups. Synchronises `stream`. */
int swiftkv_load_layer(swiftkv_model* m, int j, const swiftkv_layer_weights* w,
                       swiftkv_stream stream);

/* Copies embedding, final gain and LM head from host memory. Synchronises `stream`. */
int swiftkv_load_globals(swiftkv_model* m, const uint16_t* embed, const float* gamma_final,
                         const uint16_t* lm_head, swiftkv_stream stream);

/* swiftkv_model_create + swiftkv_load_layer for every layer + swiftkv_load_globals.
 * On failure *out is NULL and nothing is leaked. */
int swiftkv_load_weights(const swiftkv_model_config* cfg, const swiftkv_host_weights* w, int l,
                         int acrosskv_group, swiftkv_stream stream, swiftkv_model** out);

/* SwiftKV prefill of num_seqs packed prompts.
 *   tokens      device int32 [T], T = cu_seqlens[num_seqs]; prompt s is
 *               tokens[cu_seqlens[s] .. cu_seqlens[s+1]), positions 0.. within it
 *   cu_seqlens  HOST int32 [num_seqs + 1], cu_seqlens[0] == 0, every prompt >= 1 token
 *   l, acrosskv_group  must equal the model's
 *   kv          caches to fill (all num_caches of them, positions 0..n_s-1 of each sequence)
 *   logits      device float [num_seqs][vocab]: logits of each prompt's last token
 * Workspace grows on demand (cudaMalloc) and is kept by the model. num_seqs == 0 is a no-op. */
int swiftkv_prefill(swiftkv_model* m, const int32_t* tokens, const int32_t* cu_seqlens,
                    int num_seqs, int l, int acrosskv_group, const swiftkv_kv_pages* kv,
                    float* logits, swiftkv_stream stream);

/* swiftkv_prefill with HOST tokens [T] and HOST logits [num_seqs][vocab]: copies in,
 * runs, copies out and synchronises `stream` before returning. */
int swiftkv_prefill_host(swiftkv_model* m, const int32_t* tokens_host, const int32_t* cu_seqlens,
                         int num_seqs, int l, int acrosskv_group, const swiftkv_kv_pages* kv,
                         float* logits_host, swiftkv_stream stream);

/* Serving forward over a batch that mixes prompt chunks and decode tokens ("SwiftKV"
 * blog and paper, section on the inference implementation in production serving
 * frameworks: with chunked prefill and decode tokens batched together, every token runs
 * the first l layers against its sequence's cached prefix, the skipped layers' KV is
 * projected from x_l, and only the tokens whose logits are needed, the last of each
 * chunk, run layers l+1..L).
 *   tokens      device int32 [T], T = cu_seqlens[num_seqs]; chunk s is
 *               tokens[cu_seqlens[s] .. cu_seqlens[s+1]), every chunk >= 1 token
 *   cu_seqlens  HOST int32 [num_seqs + 1], cu_seqlens[0] == 0
 *   ctx_lens    HOST int32 [num_seqs] or NULL (all 0): tokens sequence s already has in
 *               every cache (positions 0..ctx_lens[s]-1, written by earlier calls with the
 *               same block table row). Chunk token i sits at position ctx_lens[s] + i,
 *               writes its K/V there in every cache and attends to positions
 *               0..ctx_lens[s] + i. A decode token is a chunk of 1 with ctx_lens[s] equal
 *               to the sequence's length; a fresh prompt is a chunk with ctx_lens[s] = 0.
 *   kv, l, acrosskv_group, logits, stream  as for swiftkv_prefill; logits of row s are
 *               those of chunk s's last token (for a chunk that does not end its prompt
 *               they are computed and may be ignored).
 * ctx_lens[s] + n_s must fit the block table row (else SWIFTKV_ENO_PAGES); a negative
 * ctx_lens[s] is SWIFTKV_EINVAL_SEQLENS. With ctx_lens NULL this is swiftkv_prefill. */
int swiftkv_forward(swiftkv_model* m, const int32_t* tokens, const int32_t* cu_seqlens,
                    const int32_t* ctx_lens, int num_seqs, int l, int acrosskv_group,
                    const swiftkv_kv_pages* kv, float* logits, swiftkv_stream stream);

/* One decode token for each of `batch` sequences ("SwiftKV" summary, section 3.2:
 * decode tokens run every layer). Sequence b holds seq_lens[b] cached tokens; its
 * new token (position seq_lens[b]) writes its K/V at that position into every cache
 * (for skipped layers projected from its own x_{l+1}, like a prompt token), attends
 * to positions 0..seq_lens[b], and produces logits and the greedy next token.
 *   tokens      device int32 [batch]
 *   seq_lens    HOST int32 [batch]
 *   logits      device float [batch][vocab]
 *   next_tokens device int32 [batch]: argmax of the logits, lowest id on ties (may be NULL) */
int swiftkv_decode_step(swiftkv_model* m, const int32_t* tokens, const int32_t* seq_lens,
                        int batch, const swiftkv_kv_pages* kv, float* logits,
                        int32_t* next_tokens, swiftkv_stream stream);

/* Reads (synchronously) the device status word; clears it when clear != 0.
 * Returns the swiftkv_status_bits that are set, or a negative swiftkv_error. */
int swiftkv_status(swiftkv_model* m, int clear);

/* Bytes of device memory the model holds for weights and for workspace. */
int swiftkv_memory(const swiftkv_model* m, size_t* weight_bytes, size_t* workspace_bytes);

/* Kernel family for GEMMs with more than 64 rows: 0 = tcgen05 on CTA pairs (cta_group::2,
 * 256 x 256 tiles, default), 1 = warp-level mma.sync tiles, 2 = tcgen05 on single CTAs
 * (128 x 256 tiles); 1 and 2 are kept as cross-checks. All are fed by TMA where tcgen05 is
 * used. GEMMs with at most 64 rows use the persistent TMA-fed skinny kernel (impl 6 of
 * swiftkv_gemm_bf16) when the weight has at least SMs / 2 tiles of 64 rows, else the
 * cp.async one (impl 5). */
int swiftkv_set_gemm_impl(swiftkv_model* m, int impl);

/* How the rows that run layers one token at a time (the last-token tail of the skipped
 * layers, decode tokens) go through a layer after its attention. 1 (default) = one launch per
 * GEMM and per RMSNorm, each GEMM a programmatic dependent that starts streaming its weights
 * while the kernel before it finishes. 0 = one cooperative persistent launch per layer: O
 * (+residual), RMSNorm, gate/up (+SwiGLU), down (+residual), the next RMSNorm and the next
 * layer's Q (tail) or Q/K/V (decode), separated by grid-wide barriers, each SM streaming its
 * share of all those weights back to back; measured slower than 1 at the Qwen2.5-14B decode
 * shape (its ~3 us of prefetched weights per SM do not cover a barrier and a norm phase), kept
 * as a cross-check. Both give every row the same kernels' arithmetic order; where a device
 * cannot take the cooperative launch, 0 falls back to 1. Returns SWIFTKV_EINVAL for other
 * values. */
int swiftkv_set_rows_impl(swiftkv_model* m, int impl);

/* Where the RMSNorm of the prompt rows runs (batches of more than 64 rows on the tcgen05
 * GEMMs). 0 (default) = a separate RMSNorm pass before each GEMM that reads normalised rows:
 * the GEMM input is bf16(gamma * x / rms(x)), rounded where the model definition rounds it.
 * 1 = inside the GEMM epilogues: the O and down GEMMs also write bf16(gamma * x) and per-tile
 * sums of squares of x, and the next GEMM scales its fp32 accumulators by the row's 1/rms, so
 * no pass re-reads the fp32 residual stream (about 3 % faster on the Llama-3.1-8B-shaped
 * prefill). Mode 1 rounds the GEMM input at another point (gamma * x instead of
 * gamma * x / rms), so its results move by about one bf16 ulp against mode 0 and the
 * definition. The tail and decode rows always use the exact separate pass.
 * Returns SWIFTKV_EINVAL for other values. */
int swiftkv_set_norm_fusion(swiftkv_model* m, int on);

/* Kernel family for the prompt tokens' attention: 0 = tcgen05 with TMA-staged paged K/V,
 * persistent, two 128-row query tiles per work item (default; d_head 128), 1 = warp-level
 * mma.sync (always used for d_head 64), 2 = tcgen05 with one 128-row query tile per CTA
 * (cross-check: the same prompt-attention outputs as 0, bit for bit). The single-row
 * attention (decode tokens, the last-token tail, chunks of at most 4 rows) runs on the
 * key-split kernel under 0 and on the per-(row, KV head) kernel under 1 and 2, so logits
 * differ between settings by rounding. An FP8 cache always uses the key-split kernel. */
int swiftkv_set_attention_impl(swiftkv_model* m, int impl);

/* Kernel self-test entry (no model needed): C = A * B^T on the current device.
 *   A  device bf16 [M][K] row-major; B device bf16 [N][K] row-major; C device float [M][N]
 *   impl 0 = tcgen05 single CTA, 1 = mma.sync tiles, 2 = skinny split-K (M <= 64; allocates
 *   and frees its own scratch and synchronises the device), 3 = not used (SWIFTKV_EINVAL),
 *   4 = tcgen05 CTA pairs (cta_group::2),
 *   5 = skinny, one CTA per pair of 16-column strips over the whole K (M <= 64),
 *   6 = skinny, persistent, TMA-fed, 64-row weight tiles over the whole K (M <= 64 and
 *       N / 64 >= SMs / 2, else SWIFTKV_EUNSUPPORTED)
 *   7 = impl 6's kernel and tiles with the residual epilogue of the decode rows' O and
 *       down projections: C += A * B^T on the C passed in
 *   status  device int or NULL: receives SWIFTKV_STATUS_TIMEOUT if a bounded wait expired
 * Requires K % 64 == 0 and N % 128 == 0. */
int swiftkv_gemm_bf16(const void* A, const void* B, float* C, int M, int N, int K, int impl, int* status,
                      swiftkv_stream stream);

/* Test-only entry for the bounded waits of the tcgen05 kernels (no model needed; the pages
 * define no such operation: it checks this library's own failure handling). Every mbarrier
 * wait in the library gives up after a time limit instead of spinning forever; this runs
 * that expiry path on purpose with a short limit: one CTA allocates TMEM, one warp waits
 * on a barrier whose producer issues nothing, bounded by limit_ns nanoseconds of the GPU
 * clock; when the limit passes the CTA raises SWIFTKV_STATUS_TIMEOUT in *status, a second
 * waiting warp leaves its wait on seeing the abort, TMEM is freed and the kernel returns.
 * No fault, no endless wait, and the context stays usable for the next call.
 *   status      device int, OR-ed with SWIFTKV_STATUS_TIMEOUT (caller-owned)
 *   elapsed_ns  device unsigned 64-bit or NULL: nanoseconds the expired wait took
 *   limit_ns    1000 .. 100000000, else SWIFTKV_EINVAL
 * Enqueued on `stream`; returns SWIFTKV_OK once launched, SWIFTKV_ECUDA on a launch error. */
int swiftkv_selftest_wait_timeout(int* status, unsigned long long* elapsed_ns, long long limit_ns,
                                  swiftkv_stream stream);

/* swiftkv_gemm_bf16 with impl 2 (skinny split-K, M <= 64) for callers that may not
 * allocate device memory, e.g. a host that reserves the GPU's memory for its own pools
 * (a serving engine holding nearly all of HBM for its KV cache) or that cannot accept
 * the device-wide synchronisation of cudaFree mid-pipeline. It has no counterpart in
 * the SwiftKV paper; it is a deployment convenience of this library.
 *   A  device bf16 [M][K]; B device bf16 [N][K]; C device float [M][N] (caller-owned)
 *   Needs 1 <= M <= 64, K % 64 == 0, N % 128 == 0.
 * Calls no cudaMalloc/cudaFree: the split-K scratch is a fixed 8 MiB device array in the
 * library (one per GPU that loads it, held until the process exits). A shape whose
 * scratch (splits * M * N * 4 bytes) exceeds 8 MiB returns SWIFTKV_EUNSUPPORTED without
 * launching anything. The first call on a device looks the array's address up
 * (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture. All calls on a device share the one array and it keeps the last
 * call's contents: calls whose kernels overlap on the GPU (different streams without
 * ordering) race on it and must be serialised by the caller. */
int swiftkv_gemm_skinny_noalloc(const void* A, const void* B, float* C, int M, int N, int K,
                                swiftkv_stream stream);

/* Per-kernel-class timing of the model's own launches, for roofline reporting.
 * swiftkv_profile_begin clears the records and, until swiftkv_profile_end, brackets
 * every launch the model enqueues with a pair of CUDA events recorded on the launch's
 * stream. swiftkv_profile_end synchronises on those events, aggregates them by class
 * and writes up to max_entries entries; it returns the number of classes (or an error).
 *   name     kernel class ("gemm_layers", "gemm_wide_kv", "attn_prefill", "rmsnorm", ...)
 *   calls    launch sites recorded; kernels: CUDA kernels they launched
 *   ms       summed event time; flops / bytes: summed algorithmic work of those calls */
typedef struct {
  char name[32];
  int calls;
  int kernels;
  double ms;
  double flops;
  double bytes;
} swiftkv_profile_entry;

int swiftkv_profile_begin(swiftkv_model* m);
int swiftkv_profile_end(swiftkv_model* m, swiftkv_profile_entry* out, int max_entries);

/* Message for the last failed call on this thread ("" if none). */
const char* swiftkv_last_error(void);

/* Frees the model and everything it allocated. NULL is ignored. */
void swiftkv_free(swiftkv_model* m);

#ifdef __cplusplus
}
#endif
#endif /* SWIFTKV_H */
