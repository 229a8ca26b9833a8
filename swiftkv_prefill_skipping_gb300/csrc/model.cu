// C-ABI implementation: model creation and weight packing, the SwiftKV prefill
// orchestration (plan -> layers 1..l -> boundary norm + wide KV GEMM -> last-token
// tail -> LM head) and the decode step. One stream, no host synchronisation inside
// prefill/decode; per-call host data reaches the device through kernel parameters.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "launch.h"
#include "swiftkv.h"

using namespace skv;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail(SWIFTKV_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

#define RET(x)                 \
  do {                         \
    int r_ = (x);              \
    if (r_ != SWIFTKV_OK) return r_; \
  } while (0)

constexpr int kRopeLen = 32768;

struct LayerW {
  float* g_attn = nullptr;
  float* g_mlp = nullptr;
  bf16* wqkv = nullptr;  // full layer: [Nq + 2 Nkv][d]; skipped layer: W_Q only [Nq][d]
  float* bqkv = nullptr;
  bf16* wo = nullptr;    // [d][Nq]
  bf16* wgu = nullptr;   // [2 Fp][d], gate/up interleaved in 64-row blocks
  bf16* wd = nullptr;    // [d][Fp]
  bool loaded = false;
};

struct Workspace {
  int *cu, *tiles, *pools, *positions, *slots, *last_idx, *last_pos, *tokens, *ctx, *srow, *sseq, *dint;
  float *x, *xt, *part, *logits, *dpart;
  bf16 *u, *q, *attn, *h, *ut, *qt, *at, *ht;
  bf16 *kv_stage;         // FP8 cache: staged K/V rows before quantization
  bf16 *exp_k, *exp_v;    // FP8 cache: bf16 expansion of one cache for the prompt-tile attention
  int* deq_items;         // FP8 cache: (sequence, page) pairs of cached prefixes to expand
  float *ss_attn, *ss_mlp;  // fused RMSNorm: per-256-column sums of squares of x after the O / down GEMM
};

constexpr int kShortChunk = 4;  // chunks up to this many rows take the single-row attention kernel

// NVTX range over a host-side phase of a call (plan, layers 1..l, wide KV, tail, LM head,
// decode): visible in a profiler timeline, a no-op without one.
struct PhaseRange {
  explicit PhaseRange(const char* name) { nvtxRangePushA(name); }
  ~PhaseRange() { nvtxRangePop(); }
  PhaseRange(const PhaseRange&) = delete;
  PhaseRange& operator=(const PhaseRange&) = delete;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace skv {
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace skv

struct swiftkv_model {
  swiftkv_model_config cfg;
  int l, g, C, G;
  int Nq, Nkv, Fp, Nwide;
  int device, num_sms;
  std::vector<LayerW> layers;
  bf16 *embed = nullptr, *lm_head = nullptr;
  float* g_final = nullptr;
  bf16* w_wide = nullptr;
  float* b_wide = nullptr;
  float2* rope_tab = nullptr;
  float* inv_freq = nullptr;
  int* status = nullptr;
  std::vector<void*> allocs;
  size_t weight_bytes = 0;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  bool globals_loaded = false;
  int gemm_impl = 0;  // 0 tcgen05 CTA pairs, 1 mma.sync tiles, 2 tcgen05 single CTA (GEMMs with > 64 rows)
  int attn_impl = 0;  // 0 tcgen05 when d_head == 128, 1 mma.sync
  bool norm_fusion = false;  // prompt rows: RMSNorm in the tcgen05 GEMM epilogues (else its own pass)
  int rows_impl = 1;  // tail / decode rows after attention: 0 one chained launch, 1 a launch per GEMM / norm
  unsigned* chain_count = nullptr;  // grid-barrier arrivals of the chained launches (device)
  unsigned chain_base = 0;          // ... and their count so far (host)
  // profiling (swiftkv_profile_begin/end)
  bool prof_on = false;
  struct Rec {
    std::string name;
    cudaEvent_t a, b;
    int kernels;
    double flops, bytes;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
};

namespace {

int dalloc(swiftkv_model* m, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    cudaGetLastError();
    return fail(SWIFTKV_EOOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  }
  m->allocs.push_back(*p);
  m->weight_bytes += bytes;
  return SWIFTKV_OK;
}

template <typename T>
int dalloc_t(swiftkv_model* m, T** p, size_t count) {
  void* v = nullptr;
  int r = dalloc(m, &v, count * sizeof(T));
  *p = static_cast<T*>(v);
  return r;
}

int check_lg(int L, int l, int g) {
  if (l < 1 || l > L) return fail(SWIFTKV_EINVAL_L, "l=%d outside [1, %d]", l, L);
  if (g < 1 || (L - l) % g != 0) return fail(SWIFTKV_EINVAL_GROUP, "AcrossKV group %d does not divide L-l=%d", g, L - l);
  return SWIFTKV_OK;
}

int check_cfg(const swiftkv_model_config* c) {
  if (!c) return fail(SWIFTKV_EINVAL, "null config");
  if (c->L < 1 || c->d < 1 || c->n_q < 1 || c->n_kv < 1 || c->ffn < 1 || c->vocab < 1)
    return fail(SWIFTKV_EINVAL, "non-positive config field");
  if (c->n_q % c->n_kv) return fail(SWIFTKV_EUNSUPPORTED, "n_q %% n_kv != 0");
  if (c->n_q / c->n_kv > 8) return fail(SWIFTKV_EUNSUPPORTED, "GQA group > 8");
  if (c->d_head != 64 && c->d_head != 128) return fail(SWIFTKV_EUNSUPPORTED, "d_head must be 64 or 128");
  if (c->d % 128 || c->d > 8192) return fail(SWIFTKV_EUNSUPPORTED, "d must be a multiple of 128, <= 8192");
  if ((c->n_q * c->d_head) % 128) return fail(SWIFTKV_EUNSUPPORTED, "n_q*d_head must be a multiple of 128");
  if (c->vocab % 128) return fail(SWIFTKV_EUNSUPPORTED, "vocab must be a multiple of 128");
  if (!(c->rope_theta > 0.f) || !(c->rms_eps > 0.f)) return fail(SWIFTKV_EINVAL, "bad rope_theta / rms_eps");
  return SWIFTKV_OK;
}

int h2d(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (!src) return fail(SWIFTKV_EINVAL, "null host weight pointer");
  CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s));
  return SWIFTKV_OK;
}

int cache_of_layer(const swiftkv_model* m, int j) { return j < m->l ? j : m->l + (j - m->l) / m->g; }

// ---------------------------------------------------------------------------- workspace


// dec_ints / dec_floats: key-split plans of the single-row attention (units + ubeg) and
// their partial results.
int ensure_workspace(swiftkv_model* m, int T, int P, int C, int ntiles, size_t part_bytes, Workspace* w,
                     size_t dec_ints = 0, size_t dec_floats = 0, size_t stage_elems = 0, size_t exp_elems = 0,
                     size_t deq_ints = 0) {
  const auto& c = m->cfg;
  const size_t A = 256;
  size_t sizes[] = {
      (size_t)(P + 1) * 4,           // cu / seq lens
      (size_t)std::max(ntiles, 1) * 4,  // tiles
      (size_t)8 * C * 4,             // pool pointers: K, V, K scale, V scale (4C x 8 bytes)
      (size_t)T * 4, (size_t)T * 4,  // positions, slots
      (size_t)P * 4, (size_t)P * 4,  // last idx / pos
      (size_t)T * 4,                 // tokens (host-buffer entry)
      (size_t)T * c.d * 4,           // x
      (size_t)P * c.d * 4,           // xt
      part_bytes,                    // skinny partials
      (size_t)P * c.vocab * 4,       // logits (host-buffer entry)
      (size_t)T * c.d * 2,           // u
      (size_t)T * m->Nq * 2,         // q
      (size_t)T * m->Nq * 2,         // attn
      (size_t)T * m->Fp * 2,         // h
      (size_t)P * c.d * 2,           // ut
      (size_t)P * m->Nq * 2,         // qt
      (size_t)P * m->Nq * 2,         // at
      (size_t)P * m->Fp * 2,         // ht
      (size_t)P * 4,                 // cached tokens before each chunk
      (size_t)T * 4, (size_t)T * 4,  // rows of short chunks and their sequences
      dec_ints * 4,                  // key-split plans
      dec_floats * 4,                // key-split partials
      stage_elems * 2,               // staged K/V rows (FP8 cache)
      exp_elems * 2, exp_elems * 2,  // bf16 expansion of one cache (FP8 cache)
      deq_ints * 4,                  // prefix pages to expand
      (size_t)T * norm_tiles(c.d) * 4,  // fused RMSNorm sums of squares after attention
      (size_t)T * norm_tiles(c.d) * 4,  // ... and after the MLP (or the embedding)
  };
  const int n = sizeof(sizes) / sizeof(sizes[0]);
  size_t off[32], total = 0;
  for (int i = 0; i < n; ++i) {
    off[i] = total;
    total += align_up(sizes[i] ? sizes[i] : 16, A);
  }
  if (total > m->ws_bytes) {
    if (m->ws) {
      cudaFree(m->ws);  // synchronises the device: no enqueued work still uses it
      m->ws = nullptr;
      m->ws_bytes = 0;
    }
    size_t want = align_up(total + total / 8, 1 << 20);
    cudaError_t e = cudaMalloc(&m->ws, want);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(SWIFTKV_EOOM, "workspace cudaMalloc(%zu): %s", want, cudaGetErrorString(e));
    }
    m->ws_bytes = want;
  }
  char* b = m->ws;
  w->cu = (int*)(b + off[0]);
  w->tiles = (int*)(b + off[1]);
  w->pools = (int*)(b + off[2]);
  w->positions = (int*)(b + off[3]);
  w->slots = (int*)(b + off[4]);
  w->last_idx = (int*)(b + off[5]);
  w->last_pos = (int*)(b + off[6]);
  w->tokens = (int*)(b + off[7]);
  w->x = (float*)(b + off[8]);
  w->xt = (float*)(b + off[9]);
  w->part = (float*)(b + off[10]);
  w->logits = (float*)(b + off[11]);
  w->u = (bf16*)(b + off[12]);
  w->q = (bf16*)(b + off[13]);
  w->attn = (bf16*)(b + off[14]);
  w->h = (bf16*)(b + off[15]);
  w->ut = (bf16*)(b + off[16]);
  w->qt = (bf16*)(b + off[17]);
  w->at = (bf16*)(b + off[18]);
  w->ht = (bf16*)(b + off[19]);
  w->ctx = (int*)(b + off[20]);
  w->srow = (int*)(b + off[21]);
  w->sseq = (int*)(b + off[22]);
  w->dint = (int*)(b + off[23]);
  w->dpart = (float*)(b + off[24]);
  w->kv_stage = (bf16*)(b + off[25]);
  w->exp_k = (bf16*)(b + off[26]);
  w->exp_v = (bf16*)(b + off[27]);
  w->deq_items = (int*)(b + off[28]);
  w->ss_attn = (float*)(b + off[29]);
  w->ss_mlp = (float*)(b + off[30]);
  return SWIFTKV_OK;
}

size_t skinny_part_bytes(const swiftkv_model* m, int M) {
  if (M > 64) return 16;
  const auto& c = m->cfg;
  size_t mx = 16;
  int shapes[][2] = {{m->Nq + 2 * m->Nkv, c.d}, {m->Nq, c.d}, {c.d, m->Nq}, {2 * m->Fp, c.d},
                     {c.d, m->Fp}, {c.vocab, c.d}, {std::max(m->Nwide, 64), c.d}};
  for (auto& s : shapes) {
    mx = std::max(mx, skinny_scratch_bytes(M, s[0], s[1], m->num_sms));
  }
  return mx;
}

// ---------------------------------------------------------------------------- launches

struct Ctx {
  swiftkv_model* m;
  Workspace w;
  cudaStream_t s;
  const swiftkv_kv_pages* kv;
  bf16* const* k_dev;  // device arrays of pool pointers
  bf16* const* v_dev;
  bool tc_attn = false;  // prefill attention on tcgen05 (attn_impl 0: two tiles per item, 2: one 128-row tile)
  const int* ctx = nullptr;  // device [P]: cached tokens before each chunk (nullptr: none)
  int nshort = 0;            // rows of short chunks, attended one row at a time (w.srow / w.sseq)
  SplitPlan sp_short{};      // key-split plan of those rows
  SplitPlan sp_rows{};       // key-split plan of the single-row attention (tail / decode rows)
  bool fp8 = false;          // the caches hold e4m3 codes + per-token scales
  float* const* ks_dev = nullptr;  // device arrays of scale pools
  float* const* vs_dev = nullptr;
  bool expand = false;       // FP8: prompt tiles read a bf16 expansion of the layer's cache
  int n_deq = 0;             // FP8: prefix pages to expand per full layer (w.deq_items)
  // RMSNorm fused into the prompt rows' tcgen05 GEMMs: the O and down epilogues leave
  // bf16(gamma * x) in w.u (gamma: the next norm's gain) and per-tile sums of squares of x in
  // w.ss_attn / w.ss_mlp, which the next GEMM's epilogue turns into the row's 1/rms; no
  // separate norm pass over the prompt rows
  bool fused = false;
};

// Host side of a key-split plan: units then ubeg in one vector (one upload).
struct HostSplit {
  std::vector<int> units, ubeg;
  size_t ints() const { return units.size() + ubeg.size(); }
  int num_units() const { return (int)(units.size() / 3); }
};

HostSplit make_split(const std::vector<int>& nkeys) {
  HostSplit h;
  if (!nkeys.empty()) split_plan_host(nkeys.data(), (int)nkeys.size(), &h.units, &h.ubeg);
  return h;
}

// Uploads h into dst and describes it (partials in the shared key-split buffer).
int upload_split(Ctx& x, const HostSplit& h, int* dst, SplitPlan* p) {
  if (h.units.empty()) return SWIFTKV_OK;
  std::vector<int> blob(h.units);
  blob.insert(blob.end(), h.ubeg.begin(), h.ubeg.end());
  CK(upload_ints(dst, blob.data(), (int)blob.size(), x.s));
  p->units = dst;
  p->ubeg = dst + h.units.size();
  p->num_units = h.num_units();
  p->num_items = (int)h.ubeg.size() - 1;
  p->any_split = p->num_units > p->num_items;
  p->part = x.w.dpart;
  return SWIFTKV_OK;
}

// Bytes of one key's K and V vectors over every KV head in a cache (codes + scales for FP8).
double kv_bytes_per_key(const swiftkv_model* m, bool fp8) {
  return 2.0 * m->cfg.n_kv * (fp8 ? m->cfg.d_head + 4.0 : 2.0 * m->cfg.d_head);
}

cudaEvent_t prof_event(swiftkv_model* m) {
  if (m->ev_used == m->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    m->ev_pool.push_back(e);
  }
  return m->ev_pool[m->ev_used++];
}

// Brackets one launch site with events on the launch stream while profiling is on.
struct Prof {
  swiftkv_model* m;
  cudaStream_t s;
  int idx = -1;
  Prof(swiftkv_model* m_, cudaStream_t s_, const char* name, int kernels, double flops, double bytes)
      : m(m_), s(s_) {
    if (!m->prof_on) return;
    cudaEvent_t a = prof_event(m), b = prof_event(m);
    if (!a || !b) return;
    m->recs.push_back({name, a, b, kernels, flops, bytes});
    idx = (int)m->recs.size() - 1;
    cudaEventRecord(a, s);
  }
  ~Prof() {
    if (idx >= 0) cudaEventRecord(m->recs[idx].b, s);
  }
  // The bracketed launch did not happen: drop the record (the last one taken).
  void cancel() {
    if (idx < 0) return;
    m->recs.pop_back();
    m->ev_used -= 2;
    idx = -1;
  }
};

int gemm(Ctx& x, const char* name, const bf16* A, int lda, const bf16* B, int K, const EpiParams& ep,
         double flops) {
  const bool skinny = ep.M <= 64;
  const double bytes = (double)ep.N * K * 2 + (double)ep.M * K * 2;
  const bool fused = ep.norm_part || ep.xb_out || ep.ks_pools;
  if (fused && (skinny || x.m->gemm_impl == 1))
    return fail(SWIFTKV_EUNSUPPORTED, "fused RMSNorm / FP8 epilogue needs the tcgen05 GEMM (M=%d)", ep.M);
  Prof pr(x.m, x.s, name, 1, flops, bytes);
  cudaError_t e;
  if (skinny) {
    e = launch_gemv_tma(A, lda, B, K, ep, x.m->num_sms, x.m->status, x.s);
    if (e == cudaErrorNotSupported) e = launch_gemv(A, lda, B, K, ep, x.s);
    if (e == cudaErrorNotSupported) e = launch_gemm_skinny(A, lda, B, K, ep, x.w.part, x.m->num_sms, x.s);
  } else {
    e = cudaErrorNotSupported;
    if (x.m->gemm_impl == 0) e = launch_gemm_tc(A, lda, B, K, ep, x.m->num_sms, x.m->status, x.s, 2);
    else if (x.m->gemm_impl == 2) e = launch_gemm_tc(A, lda, B, K, ep, x.m->num_sms, x.m->status, x.s, 0);
    if (e == cudaErrorNotSupported && !fused) e = launch_gemm_tiled(A, lda, B, K, ep, x.s);
  }
  if (e != cudaSuccess) return fail(SWIFTKV_ECUDA, "gemm M=%d N=%d K=%d: %s", ep.M, ep.N, K, cudaGetErrorString(e));
  return SWIFTKV_OK;
}

EpiParams epi_base(Ctx& x, int kind, int M, int N) {
  EpiParams p;
  memset(&p, 0, sizeof p);
  p.kind = kind;
  p.M = M;
  p.N = N;
  p.d_head = x.m->cfg.d_head;
  p.n_kv = x.m->cfg.n_kv;
  p.rope_tab = x.m->rope_tab;
  p.rope_len = kRopeLen;
  p.inv_freq = x.m->inv_freq;
  p.k_pools = x.k_dev;
  p.v_pools = x.v_dev;
  return p;
}

// The GEMM's A operand is bf16(gamma * x) from the fused path; its epilogue applies the
// RMSNorm row scale from the sums of squares in ss.
void fuse_input(Ctx& x, EpiParams& e, const float* ss) {
  e.norm_part = ss;
  e.norm_parts = norm_tiles(x.m->cfg.d);
  e.norm_inv_dim = 1.f / (float)x.m->cfg.d;
  e.norm_eps = x.m->cfg.rms_eps;
}

// A residual-update GEMM of the fused path also leaves bf16(gamma * x) in xb (gamma: the gain
// of the norm that reads x next; NULL for the wide KV GEMM, whose weights carry their gains)
// and the new row's sums of squares in ss.
void fuse_output(EpiParams& e, bf16* xb, const float* gamma, float* ss) {
  e.xb_out = xb;
  e.xb_gamma = gamma;
  e.ss_out = ss;
}

// Whether an FP8 cache is quantized in the K/V GEMM's own epilogue: the tcgen05 GEMMs (more
// than 64 rows) do it; the skinny ones stage the bf16 rows for the quantize pass.
bool fp8_in_epilogue(const Ctx& x, int M) { return x.fp8 && M > 64 && x.m->gemm_impl != 1; }

void set_fp8_epilogue(Ctx& x, EpiParams& e, bool expand) {
  e.ks_pools = const_cast<float* const*>(x.ks_dev);
  e.vs_pools = const_cast<float* const*>(x.vs_dev);
  if (expand) {
    e.exp_k = x.w.exp_k;
    e.exp_v = x.w.exp_v;
  }
}

int norm(Ctx& x, const float* src, const int* rows, int T, const float* gamma, bf16* u, float* xout) {
  Prof pr(x.m, x.s, "rmsnorm", 1, 0.0, (double)T * x.m->cfg.d * (xout ? 10 : 6));
  CK(launch_rmsnorm(src, rows, T, x.m->cfg.d, gamma, x.m->cfg.rms_eps, u, xout, x.s));
  return SWIFTKV_OK;
}

// Attention output + O projection + MLP of layer j for rows [0, M) of (xres, q), reading
// the layer's cache; `prefill` selects the varlen prompt kernel, else one query per row.
int layer_rest(Ctx& x, int j, int M, float* xres, bf16* qb, bf16* ab, bf16* ub, bf16* hb, bool prefill,
               const int* qpos, int ntiles, const char* gname, double attn_flops, double attn_bytes,
               bool attn_only = false) {
  swiftkv_model* m = x.m;
  const auto& c = m->cfg;
  const LayerW& L = m->layers[j];
  const int cidx = cache_of_layer(m, j);
  const bf16* kp = static_cast<const bf16*>(x.kv->k_pool[cidx]);
  const bf16* vp = static_cast<const bf16*>(x.kv->v_pool[cidx]);
  cudaError_t e;
  // single-row attention: key-split kernel (default), else / if unsupported the one-CTA-per-row kernel
  auto rows_attn = [&](const int* pos, int items, const int* rows, const int* seqs, const SplitPlan& sp) {
    if (x.fp8)  // no fallback: only the key-split kernel reads e4m3 pages
      return launch_attention_decode_split_fp8(
          qb, m->Nq, static_cast<const uint8_t*>(x.kv->k_pool[cidx]), static_cast<const uint8_t*>(x.kv->v_pool[cidx]),
          static_cast<const float*>(x.kv->k_scale[cidx]), static_cast<const float*>(x.kv->v_scale[cidx]),
          x.kv->block_table, x.kv->max_pages_per_seq, x.kv->num_pages, pos, rows, seqs, sp, c.n_q, c.n_kv, c.d_head,
          ab, m->Nq, m->num_sms, x.s);
    cudaError_t r = cudaErrorNotSupported;
    if (m->attn_impl == 0 && sp.num_units > 0)
      r = launch_attention_decode_split(qb, m->Nq, kp, vp, x.kv->block_table, x.kv->max_pages_per_seq,
                                        x.kv->num_pages, pos, rows, seqs, sp, c.n_q, c.n_kv, c.d_head, ab, m->Nq,
                                        m->num_sms, x.s);
    if (r == cudaErrorNotSupported)
      r = launch_attention_decode(qb, m->Nq, kp, vp, x.kv->block_table, x.kv->max_pages_per_seq, x.kv->num_pages,
                                  pos, items, c.n_q, c.n_kv, c.d_head, ab, m->Nq, x.s, rows, seqs);
    return r;
  };
  auto launches = [&](const SplitPlan& sp) { return m->attn_impl == 0 || x.fp8 ? 1 + (int)sp.any_split : 1; };
  // prompt tiles read the bf16 expansion (the e4m3 codes as bf16) of the layer's cache when
  // the cache is FP8, with its scales applied in the attention kernel
  const bf16* tkp = x.fp8 ? x.w.exp_k : kp;
  const bf16* tvp = x.fp8 ? x.w.exp_v : vp;
  const float* tks = x.fp8 ? static_cast<const float*>(x.kv->k_scale[cidx]) : nullptr;
  const float* tvs = x.fp8 ? static_cast<const float*>(x.kv->v_scale[cidx]) : nullptr;
  {
  Prof pr(x.m, x.s, prefill ? "attn_prefill" : "attn_decode",
          prefill ? (ntiles > 0) + (x.nshort > 0 ? launches(x.sp_short) : 0) : launches(x.sp_rows), attn_flops,
          attn_bytes);
  if (prefill && x.tc_attn && m->attn_impl == 0)
    e = launch_attention_prefill_tc2(qb, m->Nq, M, tkp, tvp, tks, tvs, x.kv->block_table, x.kv->max_pages_per_seq,
                                     x.kv->num_pages, x.w.cu, x.ctx, x.w.tiles, ntiles, c.n_q, c.n_kv, c.d_head, ab,
                                     m->Nq, m->num_sms, m->status, x.s, (c.n_q / c.n_kv) % 2 == 0);
  else if (prefill && x.tc_attn)
    e = launch_attention_prefill_tc(qb, m->Nq, M, tkp, tvp, tks, tvs, x.kv->block_table, x.kv->max_pages_per_seq,
                                    x.kv->num_pages, x.w.cu, x.ctx, x.w.tiles, ntiles, c.n_q, c.n_kv, c.d_head, ab,
                                    m->Nq, m->status, x.s);
  else if (prefill)
    e = launch_attention_prefill(qb, m->Nq, tkp, tvp, tks, tvs, x.kv->block_table, x.kv->max_pages_per_seq,
                                 x.kv->num_pages,
                                 x.w.cu, x.ctx, x.w.tiles, ntiles, c.n_q, c.n_kv, c.d_head, ab, m->Nq, x.s);
  else
    e = rows_attn(qpos, M, nullptr, nullptr, x.sp_rows);
  if (e == cudaSuccess && prefill && x.nshort > 0) e = rows_attn(x.w.positions, x.nshort, x.w.srow, x.w.sseq, x.sp_short);
  }
  if (e != cudaSuccess) return fail(SWIFTKV_ECUDA, "attention layer %d: %s", j, cudaGetErrorString(e));
  if (attn_only) return SWIFTKV_OK;
  const bool fused = prefill && x.fused;  // prompt rows on the fused-norm path
  EpiParams eo = epi_base(x, EPI_RESID, M, c.d);
  eo.ldo = c.d;
  eo.out_f32 = xres;
  if (fused) fuse_output(eo, ub, L.g_mlp, x.w.ss_attn);
  RET(gemm(x, gname, ab, m->Nq, L.wo, m->Nq, eo, 2.0 * M * c.d * m->Nq));
  if (!fused) RET(norm(x, xres, nullptr, M, L.g_mlp, ub, nullptr));
  EpiParams eg = epi_base(x, EPI_SWIGLU, M, 2 * m->Fp);
  eg.ldo = m->Fp;
  eg.out_bf16 = hb;
  if (fused) fuse_input(x, eg, x.w.ss_attn);
  RET(gemm(x, gname, ub, c.d, L.wgu, c.d, eg, 2.0 * M * 2 * c.ffn * c.d));
  EpiParams ed = epi_base(x, EPI_RESID, M, c.d);
  ed.ldo = c.d;
  ed.out_f32 = xres;
  // the next norm: layer j + 1's input norm, or none before the wide KV GEMM (l = j + 1)
  if (fused) fuse_output(ed, ub, j + 1 < m->l ? m->layers[j + 1].g_attn : nullptr, x.w.ss_mlp);
  RET(gemm(x, gname, hb, m->Fp, L.wd, m->Fp, ed, 2.0 * M * c.d * c.ffn));
  return SWIFTKV_OK;
}

// FP8 cache: staged K/V rows of `groups` consecutive caches from cache_base -> e4m3 codes
// and scales; with `expand`, the bf16 expansion pools get the dequantized rows too.
int quantize(Ctx& x, int M, const int* slots, int groups, int cache_base, int ld, bool expand) {
  swiftkv_model* m = x.m;
  Prof pr(m, x.s, "kv_quantize", 1, 0.0, (double)M * ld * (2 + 1) + (double)M * groups * 2 * m->cfg.n_kv * 4);
  CK(launch_kv_quantize(x.w.kv_stage, ld, M, slots, groups, m->cfg.n_kv, m->cfg.d_head, cache_base,
                        reinterpret_cast<uint8_t* const*>(x.k_dev), reinterpret_cast<uint8_t* const*>(x.v_dev),
                        const_cast<float* const*>(x.ks_dev), const_cast<float* const*>(x.vs_dev),
                        expand ? x.w.exp_k : nullptr, expand ? x.w.exp_v : nullptr, x.s));
  return SWIFTKV_OK;
}

// Epilogue of layer j's Q/K/V (full layer: cache_base = j) or Q only (skipped layer)
// projection with RoPE.
EpiParams qkv_epi(Ctx& x, int j, int M, bf16* qb, const int* pos, const int* slots) {
  swiftkv_model* m = x.m;
  const LayerW& L = m->layers[j];
  const bool full = j < m->l;
  EpiParams e = epi_base(x, EPI_QKV, M, full ? m->Nq + 2 * m->Nkv : m->Nq);
  e.ldo = m->Nq;
  e.out_bf16 = qb;
  e.bias = L.bqkv;
  e.q_cols = m->Nq;
  e.positions = pos;
  e.slots = slots;
  e.cache_base = j;
  if (full && x.fp8) {
    if (fp8_in_epilogue(x, M)) {
      set_fp8_epilogue(x, e, x.expand);
    } else {
      e.kv_stage = x.w.kv_stage;
      e.kv_stage_ld = 2 * m->Nkv;
    }
  }
  return e;
}

int qkv(Ctx& x, int j, int M, const bf16* ub, bf16* qb, const int* pos, const int* slots, const char* gname,
        bool fused = false) {
  swiftkv_model* m = x.m;
  const bool full = j < m->l;
  EpiParams e = qkv_epi(x, j, M, qb, pos, slots);
  if (fused) fuse_input(x, e, x.w.ss_mlp);
  RET(gemm(x, gname, ub, m->cfg.d, m->layers[j].wqkv, m->cfg.d, e, 2.0 * M * e.N * m->cfg.d));
  if (full && x.fp8 && !fp8_in_epilogue(x, M)) RET(quantize(x, M, slots, 1, j, 2 * m->Nkv, x.expand));
  return SWIFTKV_OK;
}

// Rows after layer j's attention (in ab), one launch per step: O (+ residual into xres) ->
// RMSNorm (gamma_mlp) -> gate/up (+ SwiGLU) -> down (+ residual).
int mlp_rows(Ctx& x, int j, int M, float* xres, const bf16* ab, bf16* ub, bf16* hb, const char* gname) {
  swiftkv_model* m = x.m;
  const auto& c = m->cfg;
  const LayerW& L = m->layers[j];
  EpiParams eo = epi_base(x, EPI_RESID, M, c.d);
  eo.ldo = c.d;
  eo.out_f32 = xres;
  RET(gemm(x, gname, ab, m->Nq, L.wo, m->Nq, eo, 2.0 * M * c.d * m->Nq));
  RET(norm(x, xres, nullptr, M, L.g_mlp, ub, nullptr));
  EpiParams eg = epi_base(x, EPI_SWIGLU, M, 2 * m->Fp);
  eg.ldo = m->Fp;
  eg.out_bf16 = hb;
  RET(gemm(x, gname, ub, c.d, L.wgu, c.d, eg, 2.0 * M * 2 * c.ffn * c.d));
  EpiParams ed = epi_base(x, EPI_RESID, M, c.d);
  ed.ldo = c.d;
  ed.out_f32 = xres;
  RET(gemm(x, gname, hb, m->Fp, L.wd, m->Fp, ed, 2.0 * M * c.d * c.ffn));
  return SWIFTKV_OK;
}

// Rows M <= 64 after layer j's attention (in ab), as one chained launch: O (+ residual into
// xres) -> RMSNorm (gamma_mlp) -> gate/up (+ SwiGLU) -> down (+ residual) -> RMSNorm with
// g_next (if g_next_set) -> the next GEMM (if next_W: A = ub, weight next_W, epilogue
// next_ep). Returns SWIFTKV_EUNSUPPORTED, with nothing enqueued, where the chained kernel
// does not apply; the caller then runs the same steps one launch each.
int chain_rest(Ctx& x, int j, int M, float* xres, const bf16* ab, bf16* ub, bf16* hb, bool g_next_set,
               const float* g_next, const bf16* next_W, const EpiParams* next_ep, const char* gname) {
  swiftkv_model* m = x.m;
  const auto& c = m->cfg;
  const LayerW& L = m->layers[j];
  if (m->rows_impl != 0 || M > 64) return SWIFTKV_EUNSUPPORTED;
  ChainStep st[kChainMaxPhases];
  memset(st, 0, sizeof st);
  int n = 0;
  double flops = 0, bytes = 0;
  auto add_gemm = [&](const bf16* A, int lda, const bf16* W, int K, const EpiParams& ep) {
    st[n].A = A;
    st[n].lda = lda;
    st[n].W = W;
    st[n].K = K;
    st[n].ep = ep;
    ++n;
    flops += 2.0 * M * ep.N * K;
    bytes += (double)ep.N * K * 2 + (double)M * K * 2;
  };
  auto add_norm = [&](const float* gamma) {
    st[n].norm = ChainNorm{xres, gamma, ub, M, c.d, c.d, c.d, c.rms_eps};
    ++n;
    bytes += (double)M * c.d * 6;
  };
  EpiParams eo = epi_base(x, EPI_RESID, M, c.d);
  eo.ldo = c.d;
  eo.out_f32 = xres;
  add_gemm(ab, m->Nq, L.wo, m->Nq, eo);
  add_norm(L.g_mlp);
  EpiParams eg = epi_base(x, EPI_SWIGLU, M, 2 * m->Fp);
  eg.ldo = m->Fp;
  eg.out_bf16 = hb;
  add_gemm(ub, c.d, L.wgu, c.d, eg);
  EpiParams ed = epi_base(x, EPI_RESID, M, c.d);
  ed.ldo = c.d;
  ed.out_f32 = xres;
  add_gemm(hb, m->Fp, L.wd, m->Fp, ed);
  if (g_next_set) add_norm(g_next);
  if (next_W) add_gemm(ub, c.d, next_W, c.d, *next_ep);
  Prof pr(m, x.s, gname, 1, flops, bytes);
  const cudaError_t e = launch_gemv_chain(st, n, m->num_sms, m->chain_count, &m->chain_base, m->status, x.s);
  if (e != cudaSuccess) {
    // nothing was enqueued (unsupported shape, or a cooperative launch this device cannot
    // take): the caller runs the same steps one launch each
    cudaGetLastError();
    pr.cancel();
    return SWIFTKV_EUNSUPPORTED;
  }
  return SWIFTKV_OK;
}

// Boundary: one row-RMS of x_l (gains folded into W_KV) and the wide KV GEMM into the
// skipped caches. On the fused path the RMS comes from the last down GEMM's sums of squares.
int wide_kv(Ctx& x, int M, const float* xres, bf16* ub, const int* pos, const int* slots, bool fused = false) {
  swiftkv_model* m = x.m;
  if (!fused) RET(norm(x, xres, nullptr, M, nullptr, ub, nullptr));
  EpiParams e = epi_base(x, EPI_WIDE_KV, M, m->Nwide);
  if (fused) fuse_input(x, e, x.w.ss_mlp);
  e.bias = m->b_wide;
  e.positions = pos;
  e.slots = slots;
  e.cache_base = m->l;
  const bool in_epi = fp8_in_epilogue(x, M);
  if (x.fp8 && in_epi) {
    set_fp8_epilogue(x, e, false);  // skipped caches are read only by the single-row attention
  } else if (x.fp8) {
    e.kv_stage = x.w.kv_stage;
    e.kv_stage_ld = m->Nwide;
  }
  RET(gemm(x, "gemm_wide_kv", ub, m->cfg.d, m->w_wide, m->cfg.d, e, 2.0 * M * m->Nwide * m->cfg.d));
  if (x.fp8 && !in_epi) RET(quantize(x, M, slots, m->G, m->l, m->Nwide, false));
  return SWIFTKV_OK;
}

int check_ready(const swiftkv_model* m) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (!m->globals_loaded) return fail(SWIFTKV_ESTATE, "globals not loaded");
  for (int j = 0; j < m->cfg.L; ++j)
    if (!m->layers[j].loaded) return fail(SWIFTKV_ESTATE, "layer %d not loaded", j);
  return SWIFTKV_OK;
}

int check_kv(const swiftkv_model* m, const swiftkv_kv_pages* kv) {
  if (!kv || !kv->k_pool || !kv->v_pool || !kv->block_table) return fail(SWIFTKV_EINVAL, "null kv pages");
  if (kv->num_caches != m->C) return fail(SWIFTKV_EINVAL, "num_caches %d != %d", kv->num_caches, m->C);
  if (kv->page_size != kPageSize) return fail(SWIFTKV_EINVAL, "page_size must be 16");
  if (kv->num_pages < 1 || kv->max_pages_per_seq < 1) return fail(SWIFTKV_EINVAL, "empty page pool");
  for (int c = 0; c < m->C; ++c)
    if (!kv->k_pool[c] || !kv->v_pool[c]) return fail(SWIFTKV_EINVAL, "null pool pointer for cache %d", c);
  if (kv->kv_dtype != 0 && kv->kv_dtype != 1) return fail(SWIFTKV_EINVAL, "kv_dtype %d", kv->kv_dtype);
  if (kv->kv_dtype == 1) {
    if (!kv->k_scale || !kv->v_scale) return fail(SWIFTKV_EINVAL, "fp8 cache without scale pools");
    for (int c = 0; c < m->C; ++c)
      if (!kv->k_scale[c] || !kv->v_scale[c]) return fail(SWIFTKV_EINVAL, "null scale pool for cache %d", c);
    if (m->cfg.n_q / m->cfg.n_kv > 8)
      return fail(SWIFTKV_EUNSUPPORTED, "fp8 cache needs at most 8 query heads per KV head");
  }
  return SWIFTKV_OK;
}

int upload_pools(Ctx& x) {
  const int C = x.m->C;
  const int n = x.fp8 ? 4 * C : 2 * C;
  std::vector<void*> ptrs(n);
  for (int c = 0; c < C; ++c) {
    ptrs[c] = x.kv->k_pool[c];
    ptrs[C + c] = x.kv->v_pool[c];
    if (x.fp8) {
      ptrs[2 * C + c] = x.kv->k_scale[c];
      ptrs[3 * C + c] = x.kv->v_scale[c];
    }
  }
  CK(upload_ints(x.w.pools, reinterpret_cast<const int*>(ptrs.data()), 2 * n, x.s));
  x.k_dev = reinterpret_cast<bf16* const*>(x.w.pools);
  x.v_dev = reinterpret_cast<bf16* const*>(x.w.pools) + C;
  if (x.fp8) {
    x.ks_dev = reinterpret_cast<float* const*>(x.w.pools) + 2 * C;
    x.vs_dev = reinterpret_cast<float* const*>(x.w.pools) + 3 * C;
  }
  return SWIFTKV_OK;
}

}  // namespace

// ============================================================================ C ABI

extern "C" {

const char* swiftkv_last_error(void) { return g_err.c_str(); }

int swiftkv_cache_count(int L, int l, int g) {
  if (L < 1) return fail(SWIFTKV_EINVAL, "L < 1");
  RET(check_lg(L, l, g));
  return l + (L - l) / g;
}

void swiftkv_free(swiftkv_model* m) {
  if (!m) return;
  for (void* p : m->allocs) cudaFree(p);
  if (m->ws) cudaFree(m->ws);
  for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
  delete m;
}

int swiftkv_model_create(const swiftkv_model_config* cfg, int l, int g, swiftkv_model** out) {
  if (!out) return fail(SWIFTKV_EINVAL, "null out");
  *out = nullptr;
  RET(check_cfg(cfg));
  RET(check_lg(cfg->L, l, g));
  swiftkv_model* m = new swiftkv_model();
  m->cfg = *cfg;
  m->l = l;
  m->g = g;
  m->G = (cfg->L - l) / g;
  m->C = l + m->G;
  m->Nq = cfg->n_q * cfg->d_head;
  m->Nkv = cfg->n_kv * cfg->d_head;
  m->Fp = (cfg->ffn + 63) / 64 * 64;
  m->Nwide = m->G * 2 * m->Nkv;
  CK(cudaGetDevice(&m->device));
  CK(cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device));
  m->layers.resize(cfg->L);
  const size_t d = cfg->d;
  auto bail = [&](int r) {
    swiftkv_free(m);
    return r;
  };
  int r;
  for (int j = 0; j < cfg->L; ++j) {
    LayerW& L = m->layers[j];
    const int nrows = j < l ? m->Nq + 2 * m->Nkv : m->Nq;
    if ((r = dalloc_t(m, &L.g_attn, d)) || (r = dalloc_t(m, &L.g_mlp, d)) ||
        (r = dalloc_t(m, &L.wqkv, (size_t)nrows * d)) || (r = dalloc_t(m, &L.wo, d * m->Nq)) ||
        (r = dalloc_t(m, &L.wgu, (size_t)2 * m->Fp * d)) || (r = dalloc_t(m, &L.wd, d * m->Fp)))
      return bail(r);
    if (cfg->qkv_bias && (r = dalloc_t(m, &L.bqkv, nrows))) return bail(r);
    if (m->Fp != cfg->ffn) {
      if (cudaMemset(L.wgu, 0, (size_t)2 * m->Fp * d * 2) != cudaSuccess ||
          cudaMemset(L.wd, 0, d * m->Fp * 2) != cudaSuccess)
        return bail(fail(SWIFTKV_ECUDA, "memset"));
    }
  }
  if (m->Nwide > 0) {
    if ((r = dalloc_t(m, &m->w_wide, (size_t)m->Nwide * d))) return bail(r);
    if (cfg->qkv_bias && (r = dalloc_t(m, &m->b_wide, m->Nwide))) return bail(r);
  }
  if ((r = dalloc_t(m, &m->embed, (size_t)cfg->vocab * d)) || (r = dalloc_t(m, &m->lm_head, (size_t)cfg->vocab * d)) ||
      (r = dalloc_t(m, &m->g_final, d)) || (r = dalloc_t(m, &m->status, 1)) ||
      (r = dalloc_t(m, &m->chain_count, 1)))
    return bail(r);
  const int half = cfg->d_head / 2;
  if ((r = dalloc_t(m, &m->inv_freq, half)) || (r = dalloc_t(m, &m->rope_tab, (size_t)kRopeLen * half)))
    return bail(r);
  std::vector<float> inv(half);
  std::vector<double> invd(half);
  for (int i = 0; i < half; ++i) {
    invd[i] = std::pow((double)cfg->rope_theta, -2.0 * i / cfg->d_head);
    inv[i] = (float)invd[i];
  }
  std::vector<float2> tab((size_t)kRopeLen * half);
  for (int p = 0; p < kRopeLen; ++p)
    for (int i = 0; i < half; ++i) {
      double a = p * invd[i];
      tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  if (cudaMemcpy(m->inv_freq, inv.data(), half * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(m->rope_tab, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(m->status, 0, 4) != cudaSuccess || cudaMemset(m->chain_count, 0, 4) != cudaSuccess)
    return bail(fail(SWIFTKV_ECUDA, "rope table upload"));
  *out = m;
  return SWIFTKV_OK;
}

int swiftkv_load_layer(swiftkv_model* m, int j, const swiftkv_layer_weights* w, swiftkv_stream stream) {
  if (!m || !w) return fail(SWIFTKV_EINVAL, "null argument");
  const auto& c = m->cfg;
  if (j < 0 || j >= c.L) return fail(SWIFTKV_EINVAL, "layer %d out of range", j);
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaSetDevice(m->device));
  LayerW& L = m->layers[j];
  const size_t d = c.d, Nq = m->Nq, Nkv = m->Nkv, F = c.ffn, Fp = m->Fp;
  const bool full = j < m->l;
  const bool rep = !full && (j - m->l) % m->g == 0;
  if (c.qkv_bias && (!w->bq || ((full || rep) && (!w->bk || !w->bv))))
    return fail(SWIFTKV_EINVAL, "qkv_bias model needs bq/bk/bv");
  if ((full || rep) && (!w->wk || !w->wv)) return fail(SWIFTKV_EINVAL, "layer %d needs wk/wv", j);
  RET(h2d(L.g_attn, w->gamma_attn, d * 4, s));
  RET(h2d(L.g_mlp, w->gamma_mlp, d * 4, s));
  RET(h2d(L.wqkv, w->wq, Nq * d * 2, s));
  if (full) {
    RET(h2d(L.wqkv + Nq * d, w->wk, Nkv * d * 2, s));
    RET(h2d(L.wqkv + (Nq + Nkv) * d, w->wv, Nkv * d * 2, s));
  }
  if (c.qkv_bias) {
    RET(h2d(L.bqkv, w->bq, Nq * 4, s));
    if (full) {
      RET(h2d(L.bqkv + Nq, w->bk, Nkv * 4, s));
      RET(h2d(L.bqkv + Nq + Nkv, w->bv, Nkv * 4, s));
    }
  }
  RET(h2d(L.wo, w->wo, d * Nq * 2, s));
  if (!w->w_gate || !w->w_up || !w->w_down) return fail(SWIFTKV_EINVAL, "null MLP weights");
  for (size_t blk = 0; blk < Fp / 64; ++blk) {
    size_t r0 = blk * 64;
    if (r0 >= F) break;
    size_t rows = std::min<size_t>(64, F - r0);
    RET(h2d(L.wgu + (blk * 128) * d, w->w_gate + r0 * d, rows * d * 2, s));
    RET(h2d(L.wgu + (blk * 128 + 64) * d, w->w_up + r0 * d, rows * d * 2, s));
  }
  CK(cudaMemcpy2DAsync(L.wd, Fp * 2, w->w_down, F * 2, F * 2, d, cudaMemcpyHostToDevice, s));
  if (rep) {
    const size_t gi = (j - m->l) / m->g;
    const size_t base = gi * 2 * Nkv;
    RET(h2d(m->w_wide + base * d, w->wk, Nkv * d * 2, s));
    RET(h2d(m->w_wide + (base + Nkv) * d, w->wv, Nkv * d * 2, s));
    CK(launch_scale_columns(m->w_wide + base * d, (int)(2 * Nkv), (int)d, L.g_attn, s));
    if (c.qkv_bias) {
      RET(h2d(m->b_wide + base, w->bk, Nkv * 4, s));
      RET(h2d(m->b_wide + base + Nkv, w->bv, Nkv * 4, s));
    }
  }
  CK(cudaStreamSynchronize(s));
  L.loaded = true;
  return SWIFTKV_OK;
}

int swiftkv_load_globals(swiftkv_model* m, const uint16_t* embed, const float* gamma_final,
                         const uint16_t* lm_head, swiftkv_stream stream) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaSetDevice(m->device));
  const size_t V = m->cfg.vocab, d = m->cfg.d;
  RET(h2d(m->embed, embed, V * d * 2, s));
  RET(h2d(m->lm_head, lm_head, V * d * 2, s));
  RET(h2d(m->g_final, gamma_final, d * 4, s));
  CK(cudaStreamSynchronize(s));
  m->globals_loaded = true;
  return SWIFTKV_OK;
}

int swiftkv_load_weights(const swiftkv_model_config* cfg, const swiftkv_host_weights* w, int l, int g,
                         swiftkv_stream stream, swiftkv_model** out) {
  if (!out) return fail(SWIFTKV_EINVAL, "null out");
  *out = nullptr;
  if (!w || !w->layers) return fail(SWIFTKV_EINVAL, "null weights");
  swiftkv_model* m = nullptr;
  RET(swiftkv_model_create(cfg, l, g, &m));
  int r = SWIFTKV_OK;
  for (int j = 0; j < cfg->L && r == SWIFTKV_OK; ++j) r = swiftkv_load_layer(m, j, &w->layers[j], stream);
  if (r == SWIFTKV_OK) r = swiftkv_load_globals(m, w->embed, w->gamma_final, w->lm_head, stream);
  if (r != SWIFTKV_OK) {
    std::string keep = g_err;
    swiftkv_free(m);
    g_err = keep;
    return r;
  }
  *out = m;
  return SWIFTKV_OK;
}

int swiftkv_memory(const swiftkv_model* m, size_t* weight_bytes, size_t* workspace_bytes) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (weight_bytes) *weight_bytes = m->weight_bytes;
  if (workspace_bytes) *workspace_bytes = m->ws_bytes;
  return SWIFTKV_OK;
}

int swiftkv_status(swiftkv_model* m, int clear) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  CK(cudaSetDevice(m->device));
  int v = 0;
  CK(cudaMemcpy(&v, m->status, 4, cudaMemcpyDeviceToHost));
  if (clear) CK(cudaMemset(m->status, 0, 4));
  if (clear && v != 0) {  // an expired wait may have left the chained launches' barrier count short
    CK(cudaMemset(m->chain_count, 0, 4));
    m->chain_base = 0;
  }
  return v;
}

int swiftkv_set_gemm_impl(swiftkv_model* m, int impl) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (impl < 0 || impl > 2) return fail(SWIFTKV_EINVAL, "gemm impl %d", impl);
  m->gemm_impl = impl;
  return SWIFTKV_OK;
}

int swiftkv_set_rows_impl(swiftkv_model* m, int impl) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (impl != 0 && impl != 1) return fail(SWIFTKV_EINVAL, "rows impl %d", impl);
  m->rows_impl = impl;
  return SWIFTKV_OK;
}

int swiftkv_set_norm_fusion(swiftkv_model* m, int on) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (on != 0 && on != 1) return fail(SWIFTKV_EINVAL, "norm fusion %d", on);
  m->norm_fusion = on != 0;
  return SWIFTKV_OK;
}

int swiftkv_set_attention_impl(swiftkv_model* m, int impl) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  if (impl < 0 || impl > 2) return fail(SWIFTKV_EINVAL, "attention impl %d", impl);
  m->attn_impl = impl;
  return SWIFTKV_OK;
}

int swiftkv_gemm_bf16(const void* A, const void* B, float* C, int M, int N, int K, int impl, int* status,
                      swiftkv_stream stream) {
  if (!A || !B || !C || M < 1 || N < 1 || K < 1) return fail(SWIFTKV_EINVAL, "bad gemm arguments");
  if (impl < 0 || impl > 7 || impl == 3) return fail(SWIFTKV_EINVAL, "gemm impl %d", impl);
  if (K % 64 || N % 128) return fail(SWIFTKV_EUNSUPPORTED, "gemm needs K %% 64 == 0 and N %% 128 == 0");
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  EpiParams ep;
  memset(&ep, 0, sizeof ep);
  ep.kind = EPI_STORE_F32;
  ep.M = M;
  ep.N = N;
  ep.ldo = N;
  ep.out_f32 = C;
  int* st = status;
  int* own = nullptr;
  if (!st) {
    CK(cudaMalloc(&own, 4));
    CK(cudaMemset(own, 0, 4));
    st = own;
  }
  cudaError_t e = cudaSuccess;
  const bf16* a = static_cast<const bf16*>(A);
  const bf16* b = static_cast<const bf16*>(B);
  if (impl == 0 || impl == 4) {
    e = launch_gemm_tc(a, K, b, K, ep, sms, st, s, impl == 0 ? 0 : 2);
  } else if (impl == 1) {
    e = launch_gemm_tiled(a, K, b, K, ep, s);
  } else if (impl == 5) {
    e = M > 64 ? cudaErrorNotSupported : launch_gemv(a, K, b, K, ep, s);
  } else if (impl == 6 || impl == 7) {
    if (impl == 7) ep.kind = EPI_RESID;  // C += A * B^T: the decode rows' O and down epilogue
    e = M > 64 ? cudaErrorNotSupported : launch_gemv_tma(a, K, b, K, ep, sms, st, s);
  } else if (impl == 2) {
    if (M > 64) e = cudaErrorNotSupported;
    else {
      float* scratch = nullptr;
      e = cudaMalloc(&scratch, skinny_scratch_bytes(M, N, K, sms));
      if (e == cudaSuccess) e = launch_gemm_skinny(a, K, b, K, ep, scratch, sms, s);
      cudaDeviceSynchronize();
      if (scratch) cudaFree(scratch);
    }
  } else {
    e = cudaErrorInvalidValue;
  }
  if (own) {
    cudaDeviceSynchronize();
    cudaFree(own);
  }
  if (e != cudaSuccess) return fail(e == cudaErrorNotSupported ? SWIFTKV_EUNSUPPORTED : SWIFTKV_ECUDA,
                                    "gemm impl %d: %s", impl, cudaGetErrorString(e));
  return SWIFTKV_OK;
}

int swiftkv_profile_begin(swiftkv_model* m) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  m->recs.clear();
  m->ev_used = 0;
  m->prof_on = true;
  return SWIFTKV_OK;
}

int swiftkv_profile_end(swiftkv_model* m, swiftkv_profile_entry* out, int max_entries) {
  if (!m) return fail(SWIFTKV_EINVAL, "null model");
  m->prof_on = false;
  std::vector<swiftkv_profile_entry> agg;
  for (auto& r : m->recs) {
    CK(cudaEventSynchronize(r.b));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, r.a, r.b));
    swiftkv_profile_entry* e = nullptr;
    for (auto& a : agg)
      if (r.name == a.name) e = &a;
    if (!e) {
      agg.push_back(swiftkv_profile_entry{});
      e = &agg.back();
      snprintf(e->name, sizeof e->name, "%s", r.name.c_str());
    }
    e->calls += 1;
    e->kernels += r.kernels;
    e->ms += ms;
    e->flops += r.flops;
    e->bytes += r.bytes;
  }
  m->recs.clear();
  m->ev_used = 0;
  for (int i = 0; i < (int)agg.size() && i < max_entries; ++i) out[i] = agg[i];
  return (int)agg.size();
}

// Prefill of packed prompt chunks; ctx (host, nullable) = tokens each sequence already has
// in the cache (0 for a fresh prompt, its length for a decode token).
static int prefill_impl(swiftkv_model* m, const int32_t* tokens, const int32_t* cu, const int32_t* ctx, int P,
                        int l, int g, const swiftkv_kv_pages* kv, float* logits, cudaStream_t s, bool host_io) {
  RET(check_ready(m));
  if (l != m->l) return fail(SWIFTKV_EINVAL_L, "l=%d but the model was packed for l=%d", l, m->l);
  if (g != m->g) return fail(SWIFTKV_EINVAL_GROUP, "g=%d but the model was packed for g=%d", g, m->g);
  if (P < 0 || P > 32767) return fail(SWIFTKV_EINVAL, "num_seqs %d outside [0, 32767]", P);
  if (P == 0) return SWIFTKV_OK;
  if (!cu || !tokens || !logits) return fail(SWIFTKV_EINVAL, "null tokens / cu_seqlens / logits");
  RET(check_kv(m, kv));
  if (cu[0] != 0) return fail(SWIFTKV_EINVAL_SEQLENS, "cu_seqlens[0] != 0");
  for (int i = 0; i < P; ++i) {
    const int n = cu[i + 1] - cu[i];
    const int c0 = ctx ? ctx[i] : 0;
    if (n < 1) return fail(SWIFTKV_EINVAL_SEQLENS, "prompt %d has %d tokens", i, n);
    if (c0 < 0) return fail(SWIFTKV_EINVAL_SEQLENS, "ctx_lens[%d] = %d < 0", i, c0);
    if ((long long)c0 + n > (long long)kv->max_pages_per_seq * kPageSize)
      return fail(SWIFTKV_ENO_PAGES, "sequence %d needs %lld pages, block table holds %d", i,
                  ((long long)c0 + n + 15) / 16, kv->max_pages_per_seq);
  }
  const int T = cu[P];
  if ((long long)T * std::max(m->Fp, m->cfg.d) >= (1LL << 31)) return fail(SWIFTKV_EUNSUPPORTED, "batch too large");
  CK(cudaSetDevice(m->device));

  const bool tc_attn = m->attn_impl != 1 && m->cfg.d_head == 128;
  // the default tcgen05 attention pairs two query heads of one KV head on 128-row tiles when
  // the group size is even, else two 128-row tiles of one head (256-row tile pairs)
  const bool head_pairs = tc_attn && m->attn_impl == 0 && (m->cfg.n_q / m->cfg.n_kv) % 2 == 0;
  const int tile_rows = tc_attn ? (m->attn_impl == 0 && !head_pairs ? 256 : 128) : 64;
  // Chunks of at most kShortChunk rows (decode tokens) are attended one row at a time by
  // the GQA-grouped single-row kernel: a 128-row query tile would be nearly empty and its CTA
  // per query head would read the sequence's keys once per head. The rest go in query
  // tiles, heaviest first (a tile's keys grow with its last row's position).
  const int short_max = m->cfg.n_q / m->cfg.n_kv <= 8 ? kShortChunk : 0;
  std::vector<int> tiles, srow, sseq;
  for (int i = 0; i < P; ++i) {
    const int n = cu[i + 1] - cu[i];
    if (n <= short_max) {
      for (int r = 0; r < n; ++r) {
        srow.push_back(cu[i] + r);
        sseq.push_back(i);
      }
      continue;
    }
    int nt = (n + tile_rows - 1) / tile_rows;
    for (int t = 0; t < nt; ++t) tiles.push_back((i << 16) | t);
  }
  auto keys_of = [&](int tl) { return (ctx ? ctx[tl >> 16] : 0) + (tl & 0xffff) * tile_rows; };
  std::stable_sort(tiles.begin(), tiles.end(), [&](int a, int b) { return keys_of(a) > keys_of(b); });

  Ctx x;
  x.m = m;
  x.s = s;
  x.kv = kv;
  x.tc_attn = tc_attn;
  // FP8 cache: prompt tiles attend over a bf16 expansion of the layer's cache (chunk rows
  // written by the quantize pass, cached prefixes expanded page by page before each layer)
  x.fp8 = kv->kv_dtype == 1;
  x.expand = x.fp8 && !tiles.empty();
  std::vector<int> deq;
  if (x.expand)
    for (int i = 0; i < P; ++i) {
      const int n = cu[i + 1] - cu[i], c0 = ctx ? ctx[i] : 0;
      if (n <= short_max) continue;
      for (int pidx = 0; pidx < (c0 + kPageSize - 1) / kPageSize; ++pidx) {
        deq.push_back(i);
        deq.push_back(pidx);
      }
    }
  x.n_deq = (int)deq.size() / 2;
  const size_t stage_elems = x.fp8 ? (size_t)T * std::max(2 * m->Nkv, m->Nwide) : 0;
  const size_t exp_elems = x.expand ? (size_t)kv->num_pages * m->cfg.n_kv * kPageSize * m->cfg.d_head : 0;
  size_t part = std::max(skinny_part_bytes(m, P), skinny_part_bytes(m, T));
  std::vector<int> nk_short, nk_tail(P);
  for (size_t i = 0; i < srow.size(); ++i) {
    const int sq = sseq[i];
    nk_short.push_back((ctx ? ctx[sq] : 0) + srow[i] - cu[sq] + 1);
  }
  for (int i = 0; i < P; ++i) nk_tail[i] = (ctx ? ctx[i] : 0) + cu[i + 1] - cu[i];
  const HostSplit hs_short = make_split(nk_short), hs_tail = make_split(nk_tail);
  RET(ensure_workspace(m, T, P, m->C, (int)tiles.size(), part, &x.w, hs_short.ints() + hs_tail.ints(),
                       std::max(split_part_floats(hs_short.num_units(), m->cfg.n_q, m->cfg.d_head),
                                split_part_floats(hs_tail.num_units(), m->cfg.n_q, m->cfg.d_head)),
                       stage_elems, exp_elems, deq.size()));
  const int* tok = tokens;
  if (host_io) {
    CK(cudaMemcpyAsync(x.w.tokens, tokens, (size_t)T * 4, cudaMemcpyHostToDevice, s));
    tok = x.w.tokens;
  }
  // algorithmic attention work per layer: causal score/PV flops; bytes = Q and O rows plus
  // every key's K and V vectors of each KV head read once (prompt rows); the last rows read
  // their sequence's keys once per layer
  double attn_flops = 0, tail_keys = 0;
  for (int i = 0; i < P; ++i) {
    const double n = cu[i + 1] - cu[i], c0 = ctx ? ctx[i] : 0;
    attn_flops += 4.0 * m->cfg.n_q * m->cfg.d_head * (n * c0 + n * (n + 1) / 2);
    tail_keys += c0 + n;
  }
  const double kv_key_bytes = kv_bytes_per_key(m, x.fp8);
  const double attn_bytes = tail_keys * kv_key_bytes + 2.0 * T * m->Nq * 2;
  const double tail_bytes = tail_keys * kv_key_bytes + 2.0 * P * m->Nq * 2;
  {
  PhaseRange nv("swiftkv plan");
  Prof pr(m, s, "plan", 1 + (P + 1 + kBlobInts - 1) / kBlobInts + ((int)tiles.size() + kBlobInts - 1) / kBlobInts +
          (4 * m->C + kBlobInts - 1) / kBlobInts + (ctx ? (P + kBlobInts - 1) / kBlobInts : 0) +
          2 * (((int)srow.size() + kBlobInts - 1) / kBlobInts) +
          ((int)hs_short.ints() + kBlobInts - 1) / kBlobInts + ((int)hs_tail.ints() + kBlobInts - 1) / kBlobInts +
          ((int)deq.size() + kBlobInts - 1) / kBlobInts,
          0.0, 0.0);
  if (!deq.empty()) CK(upload_ints(x.w.deq_items, deq.data(), (int)deq.size(), s));
  CK(upload_ints(x.w.cu, cu, P + 1, s));
  CK(upload_ints(x.w.tiles, tiles.data(), (int)tiles.size(), s));
  if (ctx) {
    CK(upload_ints(x.w.ctx, ctx, P, s));
    x.ctx = x.w.ctx;
  }
  if (!srow.empty()) {
    CK(upload_ints(x.w.srow, srow.data(), (int)srow.size(), s));
    CK(upload_ints(x.w.sseq, sseq.data(), (int)sseq.size(), s));
    x.nshort = (int)srow.size();
  }
  RET(upload_split(x, hs_short, x.w.dint, &x.sp_short));
  RET(upload_split(x, hs_tail, x.w.dint + hs_short.ints(), &x.sp_rows));
  RET(upload_pools(x));
  CK(launch_plan_prefill(x.w.cu, x.ctx, P, T, tok, m->cfg.vocab, kv->block_table, kv->max_pages_per_seq, kv->num_pages,
                         x.w.positions, x.w.slots, x.w.last_idx, x.w.last_pos, m->status, s));
  }
  const auto& c = m->cfg;
  // more than 64 prompt rows run on the tcgen05 GEMMs, which take the RMSNorm in their epilogues
  x.fused = m->norm_fusion && T > 64 && m->gemm_impl != 1;
  {
  Prof pr(m, s, "embed_rmsnorm", 1, 0.0, (double)T * c.d * 8);
  CK(launch_embed_rmsnorm(tok, T, m->embed, c.vocab, c.d, m->layers[0].g_attn, c.rms_eps, x.w.x, x.w.u,
                          x.fused ? x.w.ss_mlp : nullptr, norm_tiles(c.d), s));
  }
  // layers 1..l in full for every prompt token
  std::unique_ptr<PhaseRange> nv_layers(new PhaseRange("swiftkv layers 1..l"));
  for (int j = 0; j < m->l; ++j) {
    if (j > 0 && !x.fused) RET(norm(x, x.w.x, nullptr, T, m->layers[j].g_attn, x.w.u, nullptr));
    if (x.n_deq > 0) {
      Prof pr(m, s, "kv_dequant", 1, 0.0,
              (double)x.n_deq * 2 * c.n_kv * kPageSize * (c.d_head * 3.0 + 4.0));
      CK(launch_kv_dequant_pages(x.w.deq_items, x.n_deq, kv->block_table, kv->max_pages_per_seq, kv->num_pages,
                                 c.n_kv, c.d_head, static_cast<const uint8_t*>(kv->k_pool[j]),
                                 static_cast<const uint8_t*>(kv->v_pool[j]), x.w.exp_k, x.w.exp_v, s));
    }
    RET(qkv(x, j, T, x.w.u, x.w.q, x.w.positions, x.w.slots, "gemm_layers", x.fused));
    RET(layer_rest(x, j, T, x.w.x, x.w.q, x.w.attn, x.w.u, x.w.h, true, nullptr, (int)tiles.size(),
                   "gemm_layers", attn_flops, attn_bytes));
  }
  nv_layers.reset();
  // caches of every skipped layer / AcrossKV group from x_l
  if (m->G > 0) {
    PhaseRange nv("swiftkv wide KV");
    RET(wide_kv(x, T, x.w.x, x.w.u, x.w.positions, x.w.slots, x.fused));
  }
  std::unique_ptr<PhaseRange> nv_tail(new PhaseRange("swiftkv last-token tail"));
  // last prompt token of each sequence: layers l+1..L
  RET(norm(x, x.w.x, x.w.last_idx, P, m->l < c.L ? m->layers[m->l].g_attn : m->g_final, x.w.ut, x.w.xt));
  bool q_ready = false;  // the previous chained launch already computed this layer's Q
  for (int j = m->l; j < c.L; ++j) {
    if (!q_ready) RET(qkv(x, j, P, x.w.ut, x.w.qt, x.w.last_pos, nullptr, "gemm_tail"));
    RET(layer_rest(x, j, P, x.w.xt, x.w.qt, x.w.at, x.w.ut, x.w.ht, false, x.w.last_pos, 0, "gemm_tail",
                   4.0 * c.n_q * c.d_head * tail_keys, tail_bytes, true));
    const float* g_next = j + 1 < c.L ? m->layers[j + 1].g_attn : m->g_final;
    EpiParams eq;
    if (j + 1 < c.L) eq = qkv_epi(x, j + 1, P, x.w.qt, x.w.last_pos, nullptr);
    const int r = chain_rest(x, j, P, x.w.xt, x.w.at, x.w.ut, x.w.ht, true, g_next,
                             j + 1 < c.L ? m->layers[j + 1].wqkv : nullptr, &eq, "gemm_tail");
    q_ready = r == SWIFTKV_OK;
    if (r == SWIFTKV_EUNSUPPORTED) {
      RET(mlp_rows(x, j, P, x.w.xt, x.w.at, x.w.ut, x.w.ht, "gemm_tail"));
      RET(norm(x, x.w.xt, nullptr, P, g_next, x.w.ut, nullptr));
    } else {
      RET(r);
    }
  }
  nv_tail.reset();
  PhaseRange nv_lm("swiftkv LM head");
  EpiParams el = epi_base(x, EPI_STORE_F32, P, c.vocab);
  el.ldo = c.vocab;
  el.out_f32 = host_io ? x.w.logits : logits;
  RET(gemm(x, "lm_head", x.w.ut, c.d, m->lm_head, c.d, el, 2.0 * P * c.vocab * c.d));
  if (host_io) {
    CK(cudaMemcpyAsync(logits, x.w.logits, (size_t)P * c.vocab * 4, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
  }
  CK(cudaGetLastError());
  return SWIFTKV_OK;
}

int swiftkv_prefill(swiftkv_model* m, const int32_t* tokens, const int32_t* cu_seqlens, int num_seqs, int l,
                    int g, const swiftkv_kv_pages* kv, float* logits, swiftkv_stream stream) {
  return prefill_impl(m, tokens, cu_seqlens, nullptr, num_seqs, l, g, kv, logits, (cudaStream_t)stream, false);
}

int swiftkv_prefill_host(swiftkv_model* m, const int32_t* tokens_host, const int32_t* cu_seqlens, int num_seqs,
                         int l, int g, const swiftkv_kv_pages* kv, float* logits_host, swiftkv_stream stream) {
  return prefill_impl(m, tokens_host, cu_seqlens, nullptr, num_seqs, l, g, kv, logits_host, (cudaStream_t)stream,
                      true);
}

int swiftkv_forward(swiftkv_model* m, const int32_t* tokens, const int32_t* cu_seqlens, const int32_t* ctx_lens,
                    int num_seqs, int l, int g, const swiftkv_kv_pages* kv, float* logits, swiftkv_stream stream) {
  return prefill_impl(m, tokens, cu_seqlens, ctx_lens, num_seqs, l, g, kv, logits, (cudaStream_t)stream, false);
}

int swiftkv_decode_step(swiftkv_model* m, const int32_t* tokens, const int32_t* seq_lens, int B,
                        const swiftkv_kv_pages* kv, float* logits, int32_t* next_tokens, swiftkv_stream stream) {
  RET(check_ready(m));
  if (B < 0 || B > 32767) return fail(SWIFTKV_EINVAL, "batch %d outside [0, 32767]", B);
  if (B == 0) return SWIFTKV_OK;
  if (!tokens || !seq_lens || !logits) return fail(SWIFTKV_EINVAL, "null tokens / seq_lens / logits");
  RET(check_kv(m, kv));
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return fail(SWIFTKV_EINVAL_SEQLENS, "seq_lens[%d] < 0", b);
    if (seq_lens[b] + 1 > kv->max_pages_per_seq * kPageSize)
      return fail(SWIFTKV_ENO_PAGES, "sequence %d has no page for position %d", b, seq_lens[b]);
  }
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaSetDevice(m->device));
  PhaseRange nv("swiftkv decode step");
  Ctx x;
  x.m = m;
  x.s = s;
  x.kv = kv;
  std::vector<int> nk(B);
  double dec_keys = 0;
  for (int b = 0; b < B; ++b) {
    nk[b] = seq_lens[b] + 1;
    dec_keys += nk[b];
  }
  const HostSplit hs = make_split(nk);
  x.fp8 = kv->kv_dtype == 1;
  RET(ensure_workspace(m, B, B, m->C, 1, skinny_part_bytes(m, B), &x.w, hs.ints(),
                       split_part_floats(hs.num_units(), m->cfg.n_q, m->cfg.d_head),
                       x.fp8 ? (size_t)B * std::max(2 * m->Nkv, m->Nwide) : 0));
  CK(upload_ints(x.w.cu, seq_lens, B, s));
  RET(upload_pools(x));
  RET(upload_split(x, hs, x.w.dint, &x.sp_rows));
  const auto& c = m->cfg;
  CK(launch_plan_decode(x.w.cu, B, tokens, c.vocab, kv->block_table, kv->max_pages_per_seq, kv->num_pages,
                        x.w.positions, x.w.slots, m->status, s));
  CK(launch_embed_rmsnorm(tokens, B, m->embed, c.vocab, c.d, m->layers[0].g_attn, c.rms_eps, x.w.x, x.w.u, nullptr,
                          0, s));
  bool q_ready = false;  // the previous chained launch already computed this layer's Q/K/V
  for (int j = 0; j < c.L; ++j) {
    if (j == m->l && m->G > 0) {
      RET(wide_kv(x, B, x.w.x, x.w.u, x.w.positions, x.w.slots));
      RET(norm(x, x.w.x, nullptr, B, m->layers[j].g_attn, x.w.u, nullptr));
    }
    if (!q_ready) RET(qkv(x, j, B, x.w.u, x.w.q, x.w.positions, x.w.slots, "gemm_decode"));
    RET(layer_rest(x, j, B, x.w.x, x.w.q, x.w.attn, x.w.u, x.w.h, false, x.w.positions, 0, "gemm_decode",
                   4.0 * c.n_q * c.d_head * dec_keys, dec_keys * kv_bytes_per_key(m, x.fp8) + 2.0 * B * m->Nq * 2,
                   true));
    // the chained launch also runs the next layer's input norm and Q/K/V projection, except
    // before the SwiftKV boundary (the wide KV GEMM normalises x_l itself)
    const bool boundary_next = j + 1 == m->l && m->G > 0;
    const bool next_qkv = j + 1 < c.L && !boundary_next;
    const float* g_next = j + 1 < c.L ? m->layers[j + 1].g_attn : m->g_final;
    EpiParams eq;
    if (next_qkv) eq = qkv_epi(x, j + 1, B, x.w.q, x.w.positions, x.w.slots);
    const int r = chain_rest(x, j, B, x.w.x, x.w.attn, x.w.u, x.w.h, !boundary_next, g_next,
                             next_qkv ? m->layers[j + 1].wqkv : nullptr, &eq, "gemm_decode");
    q_ready = r == SWIFTKV_OK && next_qkv;
    if (r == SWIFTKV_EUNSUPPORTED) {
      RET(mlp_rows(x, j, B, x.w.x, x.w.attn, x.w.u, x.w.h, "gemm_decode"));
      RET(norm(x, x.w.x, nullptr, B, g_next, x.w.u, nullptr));
    } else {
      RET(r);
      // K/V of the next full layer went to the staging rows: quantize them into the FP8 cache
      if (q_ready && x.fp8 && j + 1 < m->l) RET(quantize(x, B, x.w.slots, 1, j + 1, 2 * m->Nkv, x.expand));
    }
  }
  EpiParams el = epi_base(x, EPI_STORE_F32, B, c.vocab);
  el.ldo = c.vocab;
  el.out_f32 = logits;
  RET(gemm(x, "lm_head", x.w.u, c.d, m->lm_head, c.d, el, 2.0 * B * c.vocab * c.d));
  if (next_tokens) CK(launch_argmax(logits, B, c.vocab, next_tokens, s));
  CK(cudaGetLastError());
  return SWIFTKV_OK;
}

}  // extern "C"
