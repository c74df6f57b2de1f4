// Runtime behind the C ABI: model object, device-budget ledger, paged KV
// pool, CUDA-graph replay of the decode step, two-buffer layer streaming and
// the KV fork.  Host logic only; the arithmetic is in the kernels.
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <map>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/dls.h"
#include "kernels.h"

using namespace dls;

namespace {

thread_local std::string g_err;

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// prompt tokens per prefill pass (bounded scratch; longer prompts run in chunks)
constexpr int kPrefillChunk = 2048;
// split-K limits of the tensor-core GEMM at batch sizes <= 16
constexpr int kTgMaxSplit = 16;
constexpr int kTgCounters = 4096;
constexpr int kRgMaxRows = 4;  // batched steps of up to this many rows use the multi-row GEMV

struct MatOff {
  size_t qs = 0, d = 0;
  int rows = 0, cols = 0, nb = 0, ds = 0;
  size_t qs_bytes = 0, d_bytes = 0;
};

struct LayerLayout {
  size_t attn_norm = 0, ffn_norm = 0;
  MatOff qkv, o, gu, down;
  size_t bytes = 0;
};

MatOff mat_off(size_t& cur, int rows, int cols, int wtype) {
  MatOff m;
  m.rows = rows;
  m.cols = cols;
  m.nb = (cols + 31) / 32;
  m.ds = (m.nb + 7) & ~7;  // 16-byte scale rows
  m.qs_bytes = (size_t)rows * m.nb * (wtype == 8 ? 32 : 16);
  m.d_bytes = (size_t)rows * m.ds * 2;
  m.qs = cur;
  cur = a256(cur + m.qs_bytes);
  m.d = cur;
  cur = a256(cur + m.d_bytes);
  return m;
}

MatDev mat_at(const uint8_t* base, const MatOff& o, int row0 = 0, int rows = -1) {
  MatDev m;
  const size_t rb = o.qs_bytes / (o.rows ? o.rows : 1);
  m.qs = base + o.qs + (size_t)row0 * rb;
  m.d = reinterpret_cast<const __half*>(base + o.d) + (size_t)row0 * o.ds;
  m.rows = rows < 0 ? o.rows - row0 : rows;
  m.cols = o.cols;
  m.nb = o.nb;
  m.ds = o.ds;
  m.rstep = 1;
  return m;
}

struct Seq {
  bool live = false;
  int len = 0;
  std::vector<int> pages;
};

struct GraphEntry {
  int rows;
  bool head, argmax, drafting;
  int casc;  // suffix split count of a cascade step (0: no shared prefix)
  cudaGraphExec_t exec;
  int launches;  // kernels in the graph
};

}  // namespace

struct dls_model {
  // shapes
  int L, H, nh, nkv, hd, F, V, wtype, pt, max_seqs, max_ctx, max_batch, max_pages;
  float theta, eps;
  bool tied;
  int q_rows, kv_rows;
  LayerLayout lay;
  size_t emb_bytes = 0;
  int num_sms = 0;
  // streams, allocator, ledger
  cudaStream_t stream = nullptr, copy_stream = nullptr;
  bool own_stream = false;
  dls_allocator alloc{};
  bool have_alloc = false;
  uint64_t used = 0, budget = 0;
  uint64_t credit = 0;  // bytes an in-progress layout change will free (counted as gone by the ledger)
  std::vector<std::pair<void*, size_t>> allocs;
  // weights
  std::vector<uint8_t*> layer_dev, layer_host;
  uint8_t* stage[2] = {nullptr, nullptr};
  cudaEvent_t ev_filled[2] = {}, ev_free[2] = {}, ev_start = nullptr;
  int resident = 0;
  uint8_t* emb_block = nullptr;
  uint8_t* out_block = nullptr;
  MatOff emb_off, out_off;
  float* out_norm = nullptr;
  // KV
  __half* k_pool = nullptr;
  __half* v_pool = nullptr;
  size_t page_elems = 0, kv_layer_elems = 0;
  int n_pages = 0;
  std::vector<int> free_pages;
  std::vector<int> page_ref;  // sequences holding each page (a shared fork makes it > 1)
  std::vector<uint8_t> skip_host;  // layers skipped by decode steps (dls_set_layer_skip)
  uint8_t* skip_dev = nullptr;     // the same flags for the step kernel
  std::vector<uint8_t> draft_host; // layers the speculative draft skips (dls_generate_speculative)
  uint8_t* draft_dev = nullptr;
  bool drafting = false;           // decode steps run the draft (its mask instead of skip_host)
  bool verifying = false;          // a speculative verify pass: every layer runs
  std::vector<uint8_t> no_skip;    // all zero
  bool pass_streams = false;       // the current pass over the layers copies streamed layers in
  std::vector<Seq> seqs;
  int32_t* pt_dev = nullptr;
  std::vector<int32_t> pt_host;
  // workspaces
  float *x = nullptr, *q = nullptr, *o = nullptr, *gu = nullptr, *logits = nullptr;
  int32_t* next_tok = nullptr;
  int32_t* tokens_dev = nullptr;
  size_t tokens_cap = 0;
  int32_t* argmax_buf = nullptr;
  int2* argmax_part = nullptr;
  int* argmax_cnt = nullptr;
  StepParams* sp = nullptr;
  float2* rope = nullptr;
  int rope_len = 0;
  void* attn_ws = nullptr;
  float *part_o = nullptr, *part_ml = nullptr;
  int* counters = nullptr;
  int attn_splits = 1;
  int2* pairs_dev = nullptr;
  size_t pairs_cap = 0;
  // prefill scratch for chunks of up to pf_cap tokens (tensor-core path)
  int pf_cap = 0, pf_ldh = 0;
  int pf_bn = 0;  // prompt-chunk GEMM tile width: 0 choose, 128 or 256 (DLS_PREFILL_BN)
  float *pf_x = nullptr, *pf_qkv = nullptr, *pf_q = nullptr;
  __half *pf_a = nullptr, *pf_h = nullptr;        // fp16 GEMM operands (hi planes)
  __half *pf_a_lo = nullptr, *pf_h_lo = nullptr;  // their lo planes (fp16 of the rounding residual)
  int32_t* pf_tok = nullptr;
  // batched decode (2..max_batch rows): attention scratch for that many rows
  void* attn_ws_b = nullptr;
  float *part_o_b = nullptr, *part_ml_b = nullptr;
  int* counters_b = nullptr;
  int attn_splits_b = 1;
  // cascade attention for batched steps whose rows share leading KV pages
  // (DLS_CASCADE=0 turns it off): prefix partials, their split count, and
  // this step's shared length (0 = none) and suffix split count
  float *casc_o = nullptr, *casc_ml = nullptr;
  int casc_splits = 0;
  bool casc_tc = false;  // the shared-prefix pass runs on the tensor cores (casc_tc.cu)
  bool cascade = true;
  int casc_len = 0, casc_suffix_splits = 0;
  bool batch_tc = false;  // every batched step through the small-batch tensor-core GEMM
  bool batch_rg = false;  // every batched step through the multi-row GEMV
  bool pf_planes = true;  // prompt chunks through the split-plane GEMM (false: the exact-code one)
  std::map<std::tuple<int, int, int>, RgLaunch> rg_plans;  // (matrix kind, rows, T) -> multi-row GEMV plan
  // tensor-core GEMM split-K workspace: partial sums and per-tile counters
  float* tg_part = nullptr;
  int* tg_cnt = nullptr;
  size_t tg_part_elems = 0;
  GemvLaunch plan_qkv{}, plan_o{}, plan_gu{}, plan_down{}, plan_head{};
  // graphs and hooks
  std::vector<GraphEntry> graphs;
  float* capture = nullptr;
  int launches_per_step = 0;
  int launch_count = 0;
  // persistent decode-step kernel (all layers resident, one row)
  StepPlan step{};
  bool use_step = false;
  bool step_graph_ok = true;  // false: the cooperative launch could not be captured; run it eagerly
  StepLayer* step_layers = nullptr;
  float *step_part_o = nullptr, *step_part_ml = nullptr;
  int* step_att_cnt = nullptr;
  int2* step_am = nullptr;
  unsigned* step_bar = nullptr;  // [0] barrier counter, [1] abort flag
  unsigned long long* step_trace = nullptr;  // phase timestamps when profiling
  unsigned long long* step_ctrace = nullptr; // per-CTA phase timestamps when profiling
  // per-kernel timing (dls_debug_profile_step): an event after every launch
  bool profiling = false;
  // programmatic dependent launch between the step's kernels; off by default
  // (measured slower on this path), DLS_PDL=1 turns it on
  bool pdl = false;
  // per-matrix weight types ("mixed" model: some matrix in a K-quant format):
  // matrices wq wk wv wo w_gate w_up w_down stored one by one in the layer
  // block, K-quant ones packed (mkq: offset), the others in the wtype's
  // layout (mleg); run through the mixed-format path
  bool mixed = false;
  int mtype[7] = {0, 0, 0, 0, 0, 0, 0};
  size_t mkq[7] = {0, 0, 0, 0, 0, 0, 0};
  MatOff mleg[7];
  int emb_type = 0, out_type = 0;
  size_t out_bytes = 0;
  std::map<std::tuple<int, int, int>, KqLaunch> kq_plans;      // (type, rows, cols)
  std::map<std::pair<int, int>, GemvLaunch> mix_gemv_plans;   // (rows, blocks per row)
  float* mix_buf = nullptr;  // normalised activations [H] | projection output [max(H, q_rows)]
  // streamed layers: copy-engine cudaMemcpyAsync (0), or the SM-driven copy
  // kernel with this many CTAs on the copy stream (DLS_STREAM_COPY=sm:<ctas>)
  int stream_sm_ctas = 0;
  std::vector<cudaEvent_t> prof_events;
  std::vector<int> prof_kinds;
  std::string err;
};

namespace {

const char* status_str(int s) {
  switch (s) {
    case DLS_OK: return "OK";
    case DLS_ERR_ARG: return "ARG";
    case DLS_ERR_BUDGET: return "BUDGET";
    case DLS_ERR_CAPACITY: return "CAPACITY";
    case DLS_ERR_CUDA: return "CUDA";
    case DLS_ERR_TIMEOUT: return "TIMEOUT";
    case DLS_ERR_STATE: return "STATE";
    default: return "UNKNOWN";
  }
}

int fail(dls_model* m, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  std::string s = std::string("ERR ") + status_str(code) + " " + buf;
  if (m) m->err = s;
  g_err = s;
  return code;
}

#define CK(call)                                                                                      \
  do {                                                                                                \
    cudaError_t e_ = (call);                                                                          \
    if (e_ != cudaSuccess) return fail(m, DLS_ERR_CUDA, "call=%s cuda=%s", #call, cudaGetErrorString(e_)); \
  } while (0)

#define TRY(expr)            \
  do {                       \
    int r_ = (expr);         \
    if (r_ != DLS_OK) return r_; \
  } while (0)

// ---- ledger: reserve before allocating, commit only on success --------------

int dev_alloc(dls_model* m, size_t bytes, void** out, const char* what) {
  bytes = a256(bytes ? bytes : 256);
  const uint64_t used = m->used > m->credit ? m->used - m->credit : 0;
  if (m->budget && (bytes > m->budget || used > m->budget - bytes))
    return fail(m, DLS_ERR_BUDGET, "what=%s bytes=%zu used=%llu budget=%llu", what, bytes,
                (unsigned long long)m->used, (unsigned long long)m->budget);
  void* p = nullptr;
  if (m->have_alloc) {
    p = m->alloc.alloc(m->alloc.ctx, bytes, m->stream);
  } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  if (!p) return fail(m, DLS_ERR_CUDA, "what=%s bytes=%zu allocation failed", what, bytes);
  m->used += bytes;
  m->allocs.push_back({p, bytes});
  *out = p;
  return DLS_OK;
}

void dev_free(dls_model* m, void* p) {
  if (!p) return;
  for (size_t i = 0; i < m->allocs.size(); ++i)
    if (m->allocs[i].first == p) {
      m->used -= m->allocs[i].second;
      m->allocs.erase(m->allocs.begin() + i);
      if (m->have_alloc) m->alloc.free(m->alloc.ctx, p, m->stream);
      else cudaFree(p);
      return;
    }
}

template <class T>
int dev_alloc_t(dls_model* m, size_t count, T** out, const char* what) {
  void* p = nullptr;
  TRY(dev_alloc(m, count * sizeof(T), &p, what));
  *out = static_cast<T*>(p);
  return DLS_OK;
}

// Bounded host wait: poll the stream until it drains or the deadline passes.
int sync_stream(dls_model* m, cudaStream_t s, double seconds = 900.0) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaStreamQuery(s);
    if (e == cudaSuccess) return DLS_OK;
    if (e != cudaErrorNotReady) return fail(m, DLS_ERR_CUDA, "stream=%p cuda=%s", (void*)s, cudaGetErrorString(e));
    const double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (dt > seconds) return fail(m, DLS_ERR_TIMEOUT, "waited_s=%.1f", dt);
  }
}

int check_status(dls_model* m) {
  int32_t st = 0;
  CK(cudaMemcpyAsync(&st, &m->sp->status, sizeof st, cudaMemcpyDeviceToHost, m->stream));
  TRY(sync_stream(m, m->stream));
  if (st) {
    const int32_t zero = 0;
    CK(cudaMemcpyAsync(&m->sp->status, &zero, sizeof zero, cudaMemcpyHostToDevice, m->stream));
    TRY(sync_stream(m, m->stream));
    if (st & kTimeout) return fail(m, DLS_ERR_TIMEOUT, "device_status=0x%x (8=a bounded device wait ran out)", st);
    return fail(m, DLS_ERR_STATE, "device_status=0x%x (1=page 2=token 4=position)", st);
  }
  return DLS_OK;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// copy device results to a caller pointer (device or host); syncs for host
int copy_out(dls_model* m, void* dst, const void* src, size_t bytes) {
  if (!dst) return DLS_OK;
  const bool dev = is_device_ptr(dst);
  CK(cudaMemcpyAsync(dst, src, bytes, dev ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, m->stream));
  if (!dev) TRY(sync_stream(m, m->stream));
  return DLS_OK;
}

// ---- layers ------------------------------------------------------------------

struct LayerPtrs {
  const float *attn_norm, *ffn_norm;
  MatDev qkv, o, gu, down;
  const uint8_t* base;  // the layer block (mixed-format matrices are found from it)
};

LayerPtrs layer_ptrs(const dls_model* m, const uint8_t* base) {
  LayerPtrs p;
  p.attn_norm = reinterpret_cast<const float*>(base + m->lay.attn_norm);
  p.ffn_norm = reinterpret_cast<const float*>(base + m->lay.ffn_norm);
  p.qkv = mat_at(base, m->lay.qkv);
  p.o = mat_at(base, m->lay.o);
  p.gu = mat_at(base, m->lay.gu);
  p.down = mat_at(base, m->lay.down);
  p.base = base;
  return p;
}

MatDev head_mat(const dls_model* m) {
  return m->tied ? mat_at(m->emb_block, m->emb_off) : mat_at(m->out_block, m->out_off);
}

// ---- the decode step -------------------------------------------------------------
// Per batch row b (values in m->sp): embedding -> per layer [QKV+RoPE+KV
// append, attention, O + residual, gate/up, SwiGLU->down + residual] ->
// final norm + LM head [-> greedy pick].  With streamed layers the copy
// stream fills buffer (l - resident) % 2 while the previous layer computes.

enum KernelKind { K_EMBED = 1, K_QKV = 2, K_ATTN = 3, K_O = 4, K_GATE_UP = 5, K_DOWN = 6, K_HEAD = 7, K_ARGMAX = 8,
                  K_ADVANCE = 9, K_STEP = 10 };

int prof_mark(dls_model* m, int kind) {
  const size_t i = m->prof_kinds.size();
  if (i >= m->prof_events.size()) {
    cudaEvent_t e;
    CK(cudaEventCreate(&e));
    m->prof_events.push_back(e);
  }
  CK(cudaEventRecord(m->prof_events[i], m->stream));
  m->prof_kinds.push_back(kind);
  return DLS_OK;
}

#define LK(kind, call)                                                                                 \
  do {                                                                                                \
    cudaError_t e_ = (call);                                                                          \
    ++m->launch_count;                                                                                \
    if (e_ != cudaSuccess) return fail(m, DLS_ERR_CUDA, "launch=%s cuda=%s", #call, cudaGetErrorString(e_)); \
    if (m->profiling) TRY(prof_mark(m, kind));                                                        \
  } while (0)

int enqueue_copy_layer(dls_model* m, int l) {
  const int buf = (l - m->resident) & 1;
  CK(cudaStreamWaitEvent(m->copy_stream, m->ev_free[buf], 0));
  void* src_dev = nullptr;
  if (m->stream_sm_ctas > 0 && m->lay.bytes % 16 == 0 &&
      cudaHostGetDevicePointer(&src_dev, m->layer_host[l], 0) == cudaSuccess && src_dev) {
    // the pinned copy is mapped: SM-driven copy over the host link
    CK(launch_h2d_sm(m->stage[buf], src_dev, m->lay.bytes, m->stream_sm_ctas, m->copy_stream));
  } else {
    cudaGetLastError();
    CK(cudaMemcpyAsync(m->stage[buf], m->layer_host[l], m->lay.bytes, cudaMemcpyHostToDevice, m->copy_stream));
  }
  CK(cudaEventRecord(m->ev_filled[buf], m->copy_stream));
  return DLS_OK;
}

// Layers the decode steps skip right now: the draft's mask while drafting.
const uint8_t* step_skip(const dls_model* m) {
  return m->verifying ? m->no_skip.data() : m->drafting ? m->draft_host.data() : m->skip_host.data();
}

// Start a pass over the layers: with streamed layers, the copy stream joins
// the compute stream here and fills both buffers with the first two.  A pass
// that skips every streamed layer (`skip`, or NULL for none) copies nothing.
int stream_begin(dls_model* m, const uint8_t* skip) {
  m->pass_streams = false;
  for (int l = m->resident; l < m->L; ++l) m->pass_streams |= !(skip && skip[l]);
  if (!m->pass_streams) return DLS_OK;
  CK(cudaEventRecord(m->ev_start, m->stream));
  CK(cudaStreamWaitEvent(m->copy_stream, m->ev_start, 0));
  // both buffers are free at the start of a pass
  CK(cudaEventRecord(m->ev_free[0], m->stream));
  CK(cudaEventRecord(m->ev_free[1], m->stream));
  for (int l = m->resident; l < std::min(m->L, m->resident + 2); ++l) TRY(enqueue_copy_layer(m, l));
  return DLS_OK;
}

// Weights of layer l for the compute stream (waits for its buffer if streamed).
int layer_begin(dls_model* m, int l, LayerPtrs* P) {
  const bool streamed = l >= m->resident;
  const int buf = (l - m->resident) & 1;
  if (streamed && !m->pass_streams) {  // a skipped layer of a pass that copies nothing: no weights
    *P = LayerPtrs{};
    return DLS_OK;
  }
  if (streamed) CK(cudaStreamWaitEvent(m->stream, m->ev_filled[buf], 0));
  *P = layer_ptrs(m, streamed ? m->stage[buf] : m->layer_dev[l]);
  return DLS_OK;
}

// Layer l's last kernel is enqueued: release its buffer, refill it with l + 2.
int layer_end(dls_model* m, int l) {
  if (l < m->resident || !m->pass_streams) return DLS_OK;
  CK(cudaEventRecord(m->ev_free[(l - m->resident) & 1], m->stream));
  if (l + 2 < m->L) TRY(enqueue_copy_layer(m, l + 2));
  return DLS_OK;
}

int enqueue_row(dls_model* m, int b, bool head, bool argmax, float* capture) {
  cudaStream_t s = m->stream;
  const bool pdl = m->pdl && !m->profiling;  // profiled kernels run strictly one after another
  float* x = m->x + (size_t)b * m->H;
  float* logits = m->logits + (size_t)b * m->V;
  LK(K_EMBED, launch_embed(mat_at(m->emb_block, m->emb_off), m->wtype, m->sp, b, x, m->V, s, pdl));
  const uint8_t* skip = step_skip(m);
  TRY(stream_begin(m, skip));
  for (int l = 0; l < m->L; ++l) {
    LayerPtrs P;
    TRY(layer_begin(m, l, &P));
    if (skip[l]) {  // skipped: the residual passes through (a streamed layer's copy still runs if any streamed layer does)
      if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * m->H, x, m->H * sizeof(float), cudaMemcpyDeviceToDevice, s));
      TRY(layer_end(m, l));
      continue;
    }
    KvView kv{m->k_pool + (size_t)l * m->kv_layer_elems, m->v_pool + (size_t)l * m->kv_layer_elems, m->pt_dev,
              m->nkv, m->hd, m->pt, m->max_pages};
    // (1) RMSNorm -> QKV GEMV -> RoPE -> fp16 K/V append
    GemvArgs g{};
    g.w = P.qkv;
    g.unit = 2;
    g.x = x;
    g.g = P.attn_norm;
    g.eps = m->eps;
    g.y = m->q;
    g.q_rows = m->q_rows;
    g.kv_rows = m->kv_rows;
    g.kv = kv;
    g.rope_cs = m->rope;
    g.rope_len = m->rope_len;
    g.sp = m->sp;
    g.brow = b;
    LK(K_QKV, launch_gemv(m->wtype, PRO_RMSNORM, EPI_QKV, g, m->plan_qkv, s, pdl));
    // (2) split-K GQA attention over the paged cache
    AttnArgs a{};
    a.q = m->q;
    a.o = m->o;
    a.k_pool = kv.k_pool;
    a.v_pool = kv.v_pool;
    a.page_table = m->pt_dev;
    a.max_pages = m->max_pages;
    a.pt_row = m->sp->seq;
    a.len = m->sp->pos;
    a.len_add = 1;
    a.n_heads = m->nh;
    a.n_kv = m->nkv;
    a.head_dim = m->hd;
    a.page_tokens = m->pt;
    a.n_splits = m->attn_splits;
    a.row0 = b;
    a.part_o = m->part_o;
    a.part_ml = m->part_ml;
    a.counters = m->counters;
    a.status = &m->sp->status;
    a.max_len = m->max_ctx;
    LK(K_ATTN, launch_attention(a, 1, s, pdl));
    // (3) O projection + residual
    GemvArgs go{};
    go.w = P.o;
    go.unit = 1;
    go.x = m->o;
    go.y = x;
    LK(K_O, launch_gemv(m->wtype, PRO_COPY, EPI_RESID, go, m->plan_o, s, pdl));
    // (4) RMSNorm -> interleaved gate|up GEMV -> SwiGLU: h = silu(gate) * up
    GemvArgs gg{};
    gg.w = P.gu;
    gg.unit = 2;
    gg.x = x;
    gg.g = P.ffn_norm;
    gg.eps = m->eps;
    gg.y = m->gu;
    LK(K_GATE_UP, launch_gemv(m->wtype, PRO_RMSNORM, EPI_SWIGLU, gg, m->plan_gu, s, pdl));
    // (5) down GEMV on h + residual
    GemvArgs gd{};
    gd.w = P.down;
    gd.unit = 1;
    gd.x = m->gu;
    gd.y = x;
    LK(K_DOWN, launch_gemv(m->wtype, PRO_COPY, EPI_RESID, gd, m->plan_down, s, pdl));
    if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * m->H, x, m->H * sizeof(float), cudaMemcpyDeviceToDevice, s));
    TRY(layer_end(m, l));
  }
  if (head || argmax) {
    GemvArgs gh{};
    gh.w = head_mat(m);
    gh.unit = 1;
    gh.x = x;
    gh.g = m->out_norm;
    gh.eps = m->eps;
    gh.y = logits;
    LK(K_HEAD, launch_gemv(m->wtype, PRO_RMSNORM, EPI_STORE, gh, m->plan_head, s, pdl));
  }
  if (argmax)
    LK(K_ARGMAX, launch_argmax(logits, m->V, 1, m->next_tok + b, m->argmax_part, m->argmax_cnt,
                               argmax_blocks(1, m->num_sms), s, pdl));
  return DLS_OK;
}

// ---- the mixed-format path (models with K-quant matrices) ------------------------

// Shape of layer matrix i (wq, wk, wv, wo, w_gate, w_up, w_down).
void mix_shape(const dls_model* m, int i, int* rows, int* cols) {
  const int r[7] = {m->q_rows, m->kv_rows, m->kv_rows, m->H, m->F, m->F, m->H};
  const int c[7] = {m->H, m->H, m->H, m->q_rows, m->H, m->H, m->F};
  *rows = r[i];
  *cols = c[i];
}

size_t kq_host_bytes(int type, int rows, int cols) {
  return (size_t)rows * (cols / 256) * (type == DLS_Q4_K ? 144 : type == DLS_Q5_K ? 176 : 210);
}

// y = W x for one matrix: a K-quant matrix (packed at w) through the K-quant
// GEMV, a Q8_0 / Q4_0 matrix (md) through the decode GEMV with a plain
// prologue and epilogue.
int mix_gemv(dls_model* m, int type, const uint8_t* w, const MatDev& md, int rows, int cols, const float* x,
             float* y, int kind) {
  if (type) {
    const auto key = std::make_tuple(type, rows, cols);
    auto it = m->kq_plans.find(key);
    if (it == m->kq_plans.end()) it = m->kq_plans.emplace(key, kq_plan(type, rows, cols, m->num_sms)).first;
    if (it->second.grid < 1) return fail(m, DLS_ERR_ARG, "no K-quant GEMV for type=%d rows=%d cols=%d", type, rows, cols);
    KqArgs a{};
    a.w = w;
    a.d6 = type == DLS_Q6_K ? kq_d6(w, rows, cols) : nullptr;
    a.rows = rows;
    a.cols = cols;
    a.x = x;
    a.y = y;
    a.status = &m->sp->status;
    LK(kind, launch_kq_gemv(type, a, it->second, m->stream));
    return DLS_OK;
  }
  const auto key = std::make_pair(md.rows, md.nb);
  auto it = m->mix_gemv_plans.find(key);
  if (it == m->mix_gemv_plans.end())
    it = m->mix_gemv_plans.emplace(key, gemv_plan(m->wtype, PRO_COPY, EPI_STORE, md.rows, md.nb, m->num_sms, 1)).first;
  GemvArgs g{};
  g.w = md;
  g.unit = 1;
  g.x = x;
  g.y = y;
  LK(kind, launch_gemv(m->wtype, PRO_COPY, EPI_STORE, g, it->second, m->stream, false));
  return DLS_OK;
}

int mix_layer_gemv(dls_model* m, const uint8_t* base, int i, const float* x, float* y, int kind) {
  int rows, cols;
  mix_shape(m, i, &rows, &cols);
  const MatDev md = m->mtype[i] ? MatDev{} : mat_at(base, m->mleg[i]);
  return mix_gemv(m, m->mtype[i], base + m->mkq[i], md, rows, cols, x, y, kind);
}

// The decode step of `n` batch rows (values in m->sp) on a mixed-format
// model: per layer, each row in turn runs RMSNorm, the Q, K and V GEMVs, the
// RoPE + K/V append, split-K attention, the O GEMV + residual, RMSNorm,
// the gate and up GEMVs, SwiGLU and the down GEMV + residual.  Rows of one
// sequence at consecutive positions (a prefill chunk) see the keys the
// earlier rows appended.  head_row >= 0: the LM head for that row only,
// into logits row 0; head_row == -1 with `head`: every row's logits.
int enqueue_mixed(dls_model* m, int n, bool head, int head_row, bool argmax, float* capture, int cap_row) {
  cudaStream_t s = m->stream;
  const int H = m->H, qkv_ld = m->q_rows + 2 * m->kv_rows;
  float* xn = m->mix_buf;
  float* tmp = m->mix_buf + H;
  float* gbuf = m->gu;  // [F] gate | [F] up | [F] h (m->gu holds 2 F per batch row, 16 rows or more)
  float* ubuf = m->gu + m->F;
  float* hbuf = m->gu + 2 * (size_t)m->F;
  for (int r = 0; r < n; ++r) {
    float* x = m->x + (size_t)r * H;
    if (m->emb_type)
      LK(K_EMBED, launch_kq_dequant_rows(m->emb_type, m->emb_block, m->V, H, 0, m->sp->token + r, 1, x, H,
                                         &m->sp->status, s));
    else
      LK(K_EMBED, launch_embed(mat_at(m->emb_block, m->emb_off), m->wtype, m->sp, r, x, m->V, s, false));
  }
  const uint8_t* skip = step_skip(m);
  TRY(stream_begin(m, skip));
  for (int l = 0; l < m->L; ++l) {
    LayerPtrs P;
    TRY(layer_begin(m, l, &P));
    for (int r = 0; r < n; ++r) {
      float* x = m->x + (size_t)r * H;
      if (skip[l]) {
        if (capture && r == cap_row)
          CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
        continue;
      }
      KvView kv{m->k_pool + (size_t)l * m->kv_layer_elems, m->v_pool + (size_t)l * m->kv_layer_elems, m->pt_dev,
                m->nkv, m->hd, m->pt, m->max_pages};
      float* qkv = m->pf_qkv + (size_t)r * qkv_ld;
      float* q = m->pf_q + (size_t)r * m->q_rows;
      LK(K_QKV, launch_rmsnorm_vec(x, H, P.attn_norm, m->eps, xn, s));
      TRY(mix_layer_gemv(m, P.base, 0, xn, qkv, K_QKV));
      TRY(mix_layer_gemv(m, P.base, 1, xn, qkv + m->q_rows, K_QKV));
      TRY(mix_layer_gemv(m, P.base, 2, xn, qkv + m->q_rows + m->kv_rows, K_QKV));
      LK(K_QKV, launch_rope_kv_batch(qkv, 1, qkv_ld, m->q_rows, m->kv_rows, kv, m->sp->seq + r, m->sp->pos + r,
                                     m->rope, m->rope_len, q, &m->sp->status, s));
      AttnArgs a{};
      a.q = q;
      a.o = m->o;
      a.k_pool = kv.k_pool;
      a.v_pool = kv.v_pool;
      a.page_table = m->pt_dev;
      a.max_pages = m->max_pages;
      a.pt_row = m->sp->seq;
      a.len = m->sp->pos;
      a.len_add = 1;
      a.n_heads = m->nh;
      a.n_kv = m->nkv;
      a.head_dim = m->hd;
      a.page_tokens = m->pt;
      a.n_splits = m->attn_splits;
      a.row0 = r;
      a.part_o = m->part_o;
      a.part_ml = m->part_ml;
      a.counters = m->counters;
      a.status = &m->sp->status;
      a.max_len = m->max_ctx;
      LK(K_ATTN, launch_attention(a, 1, s, false));
      TRY(mix_layer_gemv(m, P.base, 3, m->o, tmp, K_O));
      LK(K_O, launch_add_vec(x, tmp, H, s));
      LK(K_GATE_UP, launch_rmsnorm_vec(x, H, P.ffn_norm, m->eps, xn, s));
      TRY(mix_layer_gemv(m, P.base, 4, xn, gbuf, K_GATE_UP));
      TRY(mix_layer_gemv(m, P.base, 5, xn, ubuf, K_GATE_UP));
      LK(K_GATE_UP, launch_swiglu_vec(gbuf, ubuf, hbuf, m->F, s));
      TRY(mix_layer_gemv(m, P.base, 6, hbuf, tmp, K_DOWN));
      LK(K_DOWN, launch_add_vec(x, tmp, H, s));
      if (capture && r == cap_row)
        CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
    }
    TRY(layer_end(m, l));
  }
  if (head || argmax) {
    const int htype = m->tied ? m->emb_type : m->out_type;
    const uint8_t* hblk = m->tied ? m->emb_block : m->out_block;
    const MatDev md = htype ? MatDev{} : head_mat(m);
    for (int r = 0; r < n; ++r) {
      if (head_row >= 0 && r != head_row) continue;
      float* logits = m->logits + (size_t)(head_row >= 0 ? 0 : r) * m->V;
      LK(K_HEAD, launch_rmsnorm_vec(m->x + (size_t)r * H, H, m->out_norm, m->eps, xn, s));
      TRY(mix_gemv(m, htype, hblk, md, m->V, H, xn, logits, K_HEAD));
    }
  }
  if (argmax)
    LK(K_ARGMAX, launch_argmax(m->logits, m->V, n, m->next_tok, m->argmax_part, m->argmax_cnt,
                               argmax_blocks(n, m->num_sms), s, false));
  return DLS_OK;
}

// ---- tensor-core GEMM -----------------------------------------------------------

int run_tgemm(dls_model* m, int kind, int epi, PgArgs g) {
  const TgPlan p = tgemm_plan(g.w.rows, g.w.nb * 32, g.T, m->num_sms, kTgMaxSplit, m->pf_bn);
  if (p.bn >= 128 && !m->pf_planes) {  // a prompt chunk
    LK(kind, launch_cgemm(m->wtype, epi, g, m->stream));
    return DLS_OK;
  }
  if (p.split > 1) {
    if ((size_t)p.split * g.T * g.w.rows > m->tg_part_elems || (size_t)((g.w.rows + 127) / 128) > (size_t)kTgCounters)
      return fail(m, DLS_ERR_CAPACITY, "gemm split workspace rows=%d T=%d split=%d", g.w.rows, g.T, p.split);
    g.part = m->tg_part;
    g.counters = m->tg_cnt;
  }
  LK(kind, launch_tgemm(m->wtype, epi, g, p, m->stream));
  return DLS_OK;
}

// One multi-row GEMV over `a.T` activation rows (plan cached per matrix kind).
int run_rgemv(dls_model* m, int kind, int pro, int epi, RgArgs a) {
  const auto key = std::make_tuple(kind * 4 + epi, a.w.rows, a.T);
  auto it = m->rg_plans.find(key);
  if (it == m->rg_plans.end())
    it = m->rg_plans.emplace(key, rgemv_plan(m->wtype, pro, epi, a.w.rows, a.w.nb, a.T, m->num_sms, a.unit)).first;
  const RgLaunch& l = it->second;
  if (l.grid < 1) return fail(m, DLS_ERR_ARG, "no multi-row GEMV plan rows=%d T=%d", a.w.rows, a.T);
  if (l.split > 1) {
    if ((size_t)l.split * a.T * a.w.rows > m->tg_part_elems || l.grid > kTgCounters)
      return fail(m, DLS_ERR_CAPACITY, "multi-row GEMV split workspace rows=%d T=%d split=%d", a.w.rows, a.T, l.split);
    a.part = m->tg_part;
    a.counters = m->tg_cnt;
  }
  a.status = &m->sp->status;
  LK(kind, launch_rgemv(m->wtype, pro, epi, a, l, m->stream));
  return DLS_OK;
}

// ---- prefill ---------------------------------------------------------------------
// T prompt tokens at positions pos0 .. pos0+T-1 of `seq`, all at once: the
// projections run as tensor-core GEMMs over the T tokens (fp16 operands,
// fp32 accumulation), attention as a causal flash pass over the paged cache
// (which already holds positions < pos0 and receives the chunk's K/V here).
// Token ids come from host `tokens`, or are already in pf_tok when it is
// NULL.  head: HEAD_NONE, HEAD_LAST (the last row's logits into logits row
// 0) or HEAD_ALL (every row's logits into logits rows 0..T-1, and their
// greedy picks into next_tok[0..T-1]).  Layer skip masks do not apply.
enum { HEAD_NONE = 0, HEAD_LAST = 1, HEAD_ALL = 2 };
int enqueue_prefill(dls_model* m, int seq, const int32_t* tokens, int T, int pos0, int head, float* capture) {
  cudaStream_t s = m->stream;
  const int H = m->H, qkv_ld = m->q_rows + 2 * m->kv_rows;
  if (tokens) CK(cudaMemcpyAsync(m->pf_tok, tokens, (size_t)T * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  LK(K_EMBED, launch_embed_rows(mat_at(m->emb_block, m->emb_off), m->wtype, m->pf_tok, T, m->V, m->pf_x, H,
                                &m->sp->status, s));
  TRY(stream_begin(m, nullptr));
  for (int l = 0; l < m->L; ++l) {
    LayerPtrs P;
    TRY(layer_begin(m, l, &P));
    KvView kv{m->k_pool + (size_t)l * m->kv_layer_elems, m->v_pool + (size_t)l * m->kv_layer_elems, m->pt_dev,
              m->nkv, m->hd, m->pt, m->max_pages};
    // (1) RMSNorm -> fp16 -> QKV GEMM -> RoPE, fp16 K/V into the pages
    LK(K_QKV, launch_rmsnorm_rows(m->pf_x, T, H, H, P.attn_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs g{};
    g.w = P.qkv;
    g.x = m->pf_a;
    g.xlo = m->pf_a_lo;
    g.kx = H;
    g.T = T;
    g.y = m->pf_qkv;
    g.ldy = qkv_ld;
    g.status = &m->sp->status;
    TRY(run_tgemm(m, K_QKV, EPI_STORE, g));
    LK(K_QKV, launch_rope_kv_rows(m->pf_qkv, T, qkv_ld, m->q_rows, m->kv_rows, kv, seq, pos0, m->rope, m->rope_len,
                                  m->pf_q, &m->sp->status, s));
    // (2) causal attention -> fp16 operand of the O projection (tensor cores
    // for head_dim 64/128; CUDA cores otherwise, through the qkv buffer)
    if (fattn_supported(m->hd, m->nh / m->nkv, m->pt)) {
      FattnArgs fa{};
      fa.q = m->pf_q;
      fa.n_heads = m->nh;
      fa.n_kv = m->nkv;
      fa.head_dim = m->hd;
      fa.T = T;
      fa.pos0 = pos0;
      fa.ptab = m->pt_dev + (size_t)seq * m->max_pages;
      fa.max_pages = m->max_pages;
      fa.page_tokens = m->pt;
      fa.pool_rows = m->n_pages * m->nkv * m->pt;
      fa.out = m->pf_a;
      fa.out_lo = m->pf_a_lo;
      fa.ld_out = m->q_rows;
      fa.status = &m->sp->status;
      LK(K_ATTN, launch_fattn(fa, kv.k_pool, kv.v_pool, s));
    } else {
      float* o = m->pf_qkv;
      LK(K_ATTN, launch_pattn(m->pf_q, o, kv, m->pt_dev + (size_t)seq * m->max_pages, m->nh, T, pos0, s));
      LK(K_O, launch_to_f16_rows(o, T, m->q_rows, m->q_rows, m->pf_a, m->pf_a_lo, m->q_rows, s));
    }
    // (3) O projection + residual
    PgArgs go = g;
    go.w = P.o;
    go.kx = m->q_rows;
    go.y = m->pf_x;
    go.ldy = H;
    TRY(run_tgemm(m, K_O, EPI_RESID, go));
    // (4) RMSNorm -> fp16 -> gate/up GEMM with SwiGLU -> fp16 h
    LK(K_GATE_UP, launch_rmsnorm_rows(m->pf_x, T, H, H, P.ffn_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs gg = g;
    gg.w = P.gu;
    gg.y = nullptr;
    gg.h = m->pf_h;
    gg.hlo = m->pf_h_lo;
    gg.ldh = m->pf_ldh;
    TRY(run_tgemm(m, K_GATE_UP, EPI_SWIGLU, gg));
    // (5) down GEMM + residual
    PgArgs gd = g;
    gd.w = P.down;
    gd.x = m->pf_h;
    gd.xlo = m->pf_h_lo;
    gd.kx = m->pf_ldh;
    gd.y = m->pf_x;
    gd.ldy = H;
    TRY(run_tgemm(m, K_DOWN, EPI_RESID, gd));
    if (capture)
      CK(cudaMemcpyAsync(capture + (size_t)l * H, m->pf_x + (size_t)(T - 1) * H, H * sizeof(float),
                         cudaMemcpyDeviceToDevice, s));
    TRY(layer_end(m, l));
  }
  if (head == HEAD_ALL) {
    LK(K_HEAD, launch_rmsnorm_rows(m->pf_x, T, H, H, m->out_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs gh{};
    gh.w = head_mat(m);
    gh.x = m->pf_a;
    gh.xlo = m->pf_a_lo;
    gh.kx = H;
    gh.T = T;
    gh.y = m->logits;
    gh.ldy = m->V;
    gh.status = &m->sp->status;
    TRY(run_tgemm(m, K_HEAD, EPI_STORE, gh));
    LK(K_ARGMAX, launch_argmax(m->logits, m->V, T, m->next_tok, m->argmax_part, m->argmax_cnt,
                               argmax_blocks(T, m->num_sms), s, false));
  } else if (head == HEAD_LAST) {
    GemvArgs gh{};
    gh.w = head_mat(m);
    gh.unit = 1;
    gh.x = m->pf_x + (size_t)(T - 1) * H;
    gh.g = m->out_norm;
    gh.eps = m->eps;
    gh.y = m->logits;
    LK(K_HEAD, launch_gemv(m->wtype, PRO_RMSNORM, EPI_STORE, gh, m->plan_head, s, false));
  }
  return DLS_OK;
}

// ---- batched decode ------------------------------------------------------------
// n = 2..max_batch rows (row b: sequence sp->seq[b], token sp->token[b] at
// position sp->pos[b]) in one pass over the weights: each projection is one
// tensor-core GEMM over the n rows (fp16 operands, fp32 accumulation), so a
// weight byte is read once per step for the whole batch.
int enqueue_batch_tc(dls_model* m, int n, bool head, bool argmax, float* capture);

// Batched step through the multi-row CUDA-core GEMV: fp32 activations end to
// end, RMSNorm fused into the projections that follow it.
// Split-K attention of a batched step, one row per (sequence, position); q
// in pf_q, o to m->o.  With a shared prefix (m->casc_len > 0) the cascade
// kernel first covers the prefix once for all rows, and the per-row launch
// covers the rest and merges both parts.
int enqueue_batch_attention(dls_model* m, const KvView& kv, int n) {
  cudaStream_t s = m->stream;
  AttnArgs a{};
  a.q = m->pf_q;
  a.o = m->o;
  a.k_pool = kv.k_pool;
  a.v_pool = kv.v_pool;
  a.page_table = m->pt_dev;
  a.max_pages = m->max_pages;
  a.pt_row = m->sp->seq;
  a.len = m->sp->pos;
  a.len_add = 1;
  a.n_heads = m->nh;
  a.n_kv = m->nkv;
  a.head_dim = m->hd;
  a.page_tokens = m->pt;
  a.n_splits = m->attn_splits_b;
  a.row0 = 0;
  a.part_o = m->part_o_b;
  a.part_ml = m->part_ml_b;
  a.counters = m->counters_b;
  a.status = &m->sp->status;
  a.max_len = m->max_ctx;
  if (m->casc_len > 0) {
    CascArgs c{};
    c.q = m->pf_q;
    c.k_pool = kv.k_pool;
    c.v_pool = kv.v_pool;
    c.page_table = m->pt_dev;
    c.max_pages = m->max_pages;
    c.pt_row = m->sp->seq;
    c.shared_len = &m->sp->shared_len;
    c.rows = n;
    c.n_heads = m->nh;
    c.n_kv = m->nkv;
    c.head_dim = m->hd;
    c.page_tokens = m->pt;
    c.n_splits = m->casc_splits;
    c.part_o = m->casc_o;
    c.part_ml = m->casc_ml;
    c.status = &m->sp->status;
    c.max_len = m->max_ctx;
    c.pool_rows = m->n_pages * m->nkv * m->pt;
    LK(K_ATTN, m->casc_tc ? launch_cascade_prefix_tc(c, s) : launch_cascade_prefix(c, s));
    a.start_len = &m->sp->shared_len;
    a.pre_o = m->casc_o;
    a.pre_ml = m->casc_ml;
    a.pre_splits = m->casc_splits;
    a.n_splits = m->casc_suffix_splits;
  }
  LK(K_ATTN, launch_attention(a, n, s, false));
  return DLS_OK;
}

int enqueue_batch(dls_model* m, int n, bool head, bool argmax, float* capture) {
  if (m->batch_tc || (n > kRgMaxRows && !m->batch_rg)) return enqueue_batch_tc(m, n, head, argmax, capture);
  cudaStream_t s = m->stream;
  const int H = m->H, qkv_ld = m->q_rows + 2 * m->kv_rows;
  float* x = m->x;  // [n][H]
  LK(K_EMBED, launch_embed_rows(mat_at(m->emb_block, m->emb_off), m->wtype, m->sp->token, n, m->V, x, H,
                                &m->sp->status, s));
  const uint8_t* skip = step_skip(m);
  TRY(stream_begin(m, skip));
  for (int l = 0; l < m->L; ++l) {
    LayerPtrs P;
    TRY(layer_begin(m, l, &P));
    if (skip[l]) {
      if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
      TRY(layer_end(m, l));
      continue;
    }
    KvView kv{m->k_pool + (size_t)l * m->kv_layer_elems, m->v_pool + (size_t)l * m->kv_layer_elems, m->pt_dev,
              m->nkv, m->hd, m->pt, m->max_pages};
    // (1) RMSNorm -> QKV -> RoPE + fp16 K/V append per row
    RgArgs g{};
    g.w = P.qkv;
    g.unit = 2;
    g.x = x;
    g.ldx = H;
    g.T = n;
    g.g = P.attn_norm;
    g.eps = m->eps;
    g.y = m->pf_qkv;
    g.ldy = qkv_ld;
    TRY(run_rgemv(m, K_QKV, PRO_RMSNORM, EPI_STORE, g));
    LK(K_QKV, launch_rope_kv_batch(m->pf_qkv, n, qkv_ld, m->q_rows, m->kv_rows, kv, m->sp->seq, m->sp->pos, m->rope,
                                   m->rope_len, m->pf_q, &m->sp->status, s));
    // (2) split-K attention, one row per (sequence, position)
    TRY(enqueue_batch_attention(m, kv, n));
    // (3) O projection + residual
    RgArgs go = g;
    go.w = P.o;
    go.unit = 1;
    go.x = m->o;
    go.ldx = m->q_rows;
    go.g = nullptr;
    go.y = x;
    go.ldy = H;
    TRY(run_rgemv(m, K_O, PRO_COPY, EPI_RESID, go));
    // (4) RMSNorm -> gate/up -> SwiGLU: h [n][F]
    RgArgs gg = g;
    gg.w = P.gu;
    gg.g = P.ffn_norm;
    gg.y = m->gu;
    gg.ldy = m->F;
    TRY(run_rgemv(m, K_GATE_UP, PRO_RMSNORM, EPI_SWIGLU, gg));
    // (5) down + residual
    RgArgs gd = go;
    gd.w = P.down;
    gd.x = m->gu;
    gd.ldx = m->F;
    TRY(run_rgemv(m, K_DOWN, PRO_COPY, EPI_RESID, gd));
    if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
    TRY(layer_end(m, l));
  }
  if (head || argmax) {
    RgArgs gh{};
    gh.w = head_mat(m);
    gh.unit = 1;
    gh.x = x;
    gh.ldx = H;
    gh.T = n;
    gh.g = m->out_norm;
    gh.eps = m->eps;
    gh.y = m->logits;
    gh.ldy = m->V;
    TRY(run_rgemv(m, K_HEAD, PRO_RMSNORM, EPI_STORE, gh));
  }
  if (argmax)
    LK(K_ARGMAX, launch_argmax(m->logits, m->V, n, m->next_tok, m->argmax_part, m->argmax_cnt,
                               argmax_blocks(n, m->num_sms), s, false));
  return DLS_OK;
}

int enqueue_batch_tc(dls_model* m, int n, bool head, bool argmax, float* capture) {
  cudaStream_t s = m->stream;
  const int H = m->H, qkv_ld = m->q_rows + 2 * m->kv_rows;
  float* x = m->x;  // [n][H]
  LK(K_EMBED, launch_embed_rows(mat_at(m->emb_block, m->emb_off), m->wtype, m->sp->token, n, m->V, x, H,
                                &m->sp->status, s));
  const uint8_t* skip = step_skip(m);
  TRY(stream_begin(m, skip));
  for (int l = 0; l < m->L; ++l) {
    LayerPtrs P;
    TRY(layer_begin(m, l, &P));
    if (skip[l]) {  // skipped: the residuals pass through
      if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
      TRY(layer_end(m, l));
      continue;
    }
    KvView kv{m->k_pool + (size_t)l * m->kv_layer_elems, m->v_pool + (size_t)l * m->kv_layer_elems, m->pt_dev,
              m->nkv, m->hd, m->pt, m->max_pages};
    // (1) RMSNorm -> fp16 -> QKV GEMM -> RoPE + fp16 K/V append per row
    LK(K_QKV, launch_rmsnorm_rows(x, n, H, H, P.attn_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs g{};
    g.w = P.qkv;
    g.x = m->pf_a;
    g.xlo = m->pf_a_lo;
    g.kx = H;
    g.T = n;
    g.y = m->pf_qkv;
    g.ldy = qkv_ld;
    g.status = &m->sp->status;
    TRY(run_tgemm(m, K_QKV, EPI_STORE, g));
    LK(K_QKV, launch_rope_kv_batch(m->pf_qkv, n, qkv_ld, m->q_rows, m->kv_rows, kv, m->sp->seq, m->sp->pos, m->rope,
                                   m->rope_len, m->pf_q, &m->sp->status, s));
    // (2) split-K attention, one row per sequence
    TRY(enqueue_batch_attention(m, kv, n));
    // (3) O GEMM + residual
    LK(K_O, launch_to_f16_rows(m->o, n, m->q_rows, m->q_rows, m->pf_a, m->pf_a_lo, m->q_rows, s));
    PgArgs go = g;
    go.w = P.o;
    go.kx = m->q_rows;
    go.y = x;
    go.ldy = H;
    TRY(run_tgemm(m, K_O, EPI_RESID, go));
    // (4) RMSNorm -> gate/up GEMM with SwiGLU -> (5) down GEMM + residual
    LK(K_GATE_UP, launch_rmsnorm_rows(x, n, H, H, P.ffn_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs gg = g;
    gg.w = P.gu;
    gg.y = nullptr;
    gg.h = m->pf_h;
    gg.hlo = m->pf_h_lo;
    gg.ldh = m->pf_ldh;
    TRY(run_tgemm(m, K_GATE_UP, EPI_SWIGLU, gg));
    PgArgs gd = g;
    gd.w = P.down;
    gd.x = m->pf_h;
    gd.xlo = m->pf_h_lo;
    gd.kx = m->pf_ldh;
    gd.y = x;
    gd.ldy = H;
    TRY(run_tgemm(m, K_DOWN, EPI_RESID, gd));
    if (capture) CK(cudaMemcpyAsync(capture + (size_t)l * H, x, H * sizeof(float), cudaMemcpyDeviceToDevice, s));
    TRY(layer_end(m, l));
  }
  if (head || argmax) {
    LK(K_HEAD, launch_rmsnorm_rows(x, n, H, H, m->out_norm, m->eps, m->pf_a, m->pf_a_lo, H, s));
    PgArgs gh{};
    gh.w = head_mat(m);
    gh.x = m->pf_a;
    gh.xlo = m->pf_a_lo;
    gh.kx = H;
    gh.T = n;
    gh.y = m->logits;
    gh.ldy = m->V;
    gh.status = &m->sp->status;
    TRY(run_tgemm(m, K_HEAD, EPI_STORE, gh));
  }
  if (argmax)
    LK(K_ARGMAX, launch_argmax(m->logits, m->V, n, m->next_tok, m->argmax_part, m->argmax_cnt,
                               argmax_blocks(n, m->num_sms), s, false));
  return DLS_OK;
}

int enqueue_persistent(dls_model* m, bool head, bool argmax, float* capture) {
  StepArgs a{};
  a.layers = m->step_layers;
  a.n_layers = m->L;
  a.emb = mat_at(m->emb_block, m->emb_off);
  a.head = head_mat(m);
  a.out_norm = m->out_norm;
  a.H = m->H;
  a.q_rows = m->q_rows;
  a.kv_rows = m->kv_rows;
  a.n_heads = m->nh;
  a.n_kv = m->nkv;
  a.hd = m->hd;
  a.F = m->F;
  a.vocab = m->V;
  a.eps = m->eps;
  a.page_table = m->pt_dev;
  a.max_pages = m->max_pages;
  a.page_tokens = m->pt;
  a.max_len = m->max_ctx;
  a.rope_cs = m->rope;
  a.rope_len = m->rope_len;
  a.sp = m->sp;
  a.x = m->x;
  a.q = m->q;
  a.o = m->o;
  a.h = m->gu;
  a.logits = m->logits;
  a.part_o = m->step_part_o;
  a.part_ml = m->step_part_ml;
  a.att_counters = m->step_att_cnt;
  a.am_part = m->step_am;
  a.tokens_out = argmax ? m->tokens_dev : nullptr;
  a.greedy = argmax ? 1 : 0;
  a.head_rows = (head || argmax) ? m->V : 0;
  a.bar = m->step_bar;
  a.abort = reinterpret_cast<int*>(m->step_bar + 1);
  a.S = m->step.splits;
  a.trace = m->profiling ? m->step_trace : nullptr;
  a.ctrace = m->profiling ? m->step_ctrace : nullptr;
  a.skip = m->drafting ? m->draft_dev : m->skip_dev;
  a.capture = capture;
  a.ns = m->step.ns;
  a.stage_bytes = m->step.stage_bytes;
  {
    // L2 hints during the attention and O phases: skip the gate/up bytes the
    // ring will already hold (~96 KB per CTA), then hint the next ~384 KB
    // (152 CTAs x 384 KB = 58 MB, well inside the L2).  Measured on the 8B
    // Q8_0 model at ctx 2048: 529 tok/s with the hints, 518 without.
    const int nb = (m->H + 31) / 32;
    const int row = (m->wtype == 8 ? nb * 32 : nb * 16) + ((nb + 7) & ~7) * 2;
    const char* e1 = getenv("DLS_STEP_PF_KB");
    const char* e2 = getenv("DLS_STEP_PF_SKIP_KB");
    const long kb = e1 ? std::max(0L, atol(e1)) : 384;
    const long skip = e2 ? std::max(0L, atol(e2)) : 96;
    a.pf_rows = (int)(kb * 1024 / row);
    a.pf_skip = (int)(skip * 1024 / row);
  }
  CK(cudaMemsetAsync(m->step_bar, 0, 2 * sizeof(unsigned), m->stream));
  LK(K_STEP, launch_step(m->step, a, m->stream));
  return DLS_OK;
}

int enqueue_step(dls_model* m, int rows, bool head, bool argmax, float* capture) {
  m->launch_count = 0;
  if (m->mixed) {
    TRY(enqueue_mixed(m, rows, head, -1, argmax, capture, 0));
    if (argmax) LK(K_ADVANCE, launch_advance(m->sp, m->next_tok, m->tokens_dev, rows, m->stream, false));
    m->launches_per_step = m->launch_count;
    return DLS_OK;
  }
  if (m->use_step && rows == 1) {
    TRY(enqueue_persistent(m, head, argmax, capture));
    m->launches_per_step = m->launch_count;
    return DLS_OK;
  }
  if (rows >= 2) TRY(enqueue_batch(m, rows, head, argmax, capture));
  else TRY(enqueue_row(m, 0, head, argmax, capture));
  if (argmax) LK(K_ADVANCE, launch_advance(m->sp, m->next_tok, m->tokens_dev, rows, m->stream, m->pdl));
  m->launches_per_step = m->launch_count;
  return DLS_OK;
}

void drop_graphs(dls_model* m) {
  for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
  m->graphs.clear();
}

// Replay the step as one CUDA graph (captured on first use per shape).
int run_step(dls_model* m, int rows, bool head, bool argmax) {
  if (m->capture) {
    float* cap = m->capture;
    m->capture = nullptr;
    return enqueue_step(m, rows, head, argmax, cap);
  }
  const bool persistent = m->use_step && rows == 1;
  if (persistent && !m->step_graph_ok) return enqueue_step(m, rows, head, argmax, nullptr);
  for (auto& g : m->graphs)
    if (g.rows == rows && g.head == head && g.argmax == argmax && g.drafting == m->drafting &&
        g.casc == (rows >= 2 ? m->casc_suffix_splits : 0)) {
      CK(cudaGraphLaunch(g.exec, m->stream));
      m->launches_per_step = g.launches;
      return DLS_OK;
    }
  cudaGraph_t graph = nullptr;
  CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
  const int r = enqueue_step(m, rows, head, argmax, nullptr);
  cudaError_t e = cudaStreamEndCapture(m->stream, &graph);
  cudaGraphExec_t exec = nullptr;
  if (r == DLS_OK && e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
  if (graph) cudaGraphDestroy(graph);
  if (persistent && (r != DLS_OK || e != cudaSuccess)) {
    // a cooperative launch that cannot live in a graph: launch it directly
    cudaGetLastError();
    m->step_graph_ok = false;
    return enqueue_step(m, rows, head, argmax, nullptr);
  }
  if (r != DLS_OK) return r;
  if (e != cudaSuccess) return fail(m, DLS_ERR_CUDA, "capture cuda=%s", cudaGetErrorString(e));
  m->graphs.push_back({rows, head, argmax, m->drafting, rows >= 2 ? m->casc_suffix_splits : 0, exec,
                       m->launches_per_step});
  CK(cudaGraphLaunch(exec, m->stream));
  return DLS_OK;
}

// ---- paged KV ------------------------------------------------------------------

int pages_needed(const dls_model* m, int len) { return (len + m->pt - 1) / m->pt; }

// Give `seq` pages for positions [0, len); all-or-nothing.
int ensure_pages(dls_model* m, int seq, int len) {
  Seq& s = m->seqs[seq];
  const int need = pages_needed(m, len) - (int)s.pages.size();
  if (need <= 0) return DLS_OK;
  if (need > (int)m->free_pages.size())
    return fail(m, DLS_ERR_CAPACITY, "seq=%d need_pages=%d free_pages=%zu", seq, need, m->free_pages.size());
  const int first = (int)s.pages.size();
  for (int i = 0; i < need; ++i) {
    const int p = m->free_pages.back();
    m->free_pages.pop_back();
    m->page_ref[p] = 1;
    s.pages.push_back(p);
    m->pt_host[(size_t)seq * m->max_pages + first + i] = p;
  }
  // pageable source: staged before the call returns, so the mirror may change later
  CK(cudaMemcpyAsync(m->pt_dev + (size_t)seq * m->max_pages + first, &m->pt_host[(size_t)seq * m->max_pages + first],
                     need * sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
  return DLS_OK;
}

int release_pages(dls_model* m, int seq) {
  Seq& s = m->seqs[seq];
  for (int p : s.pages)
    if (--m->page_ref[p] == 0) m->free_pages.push_back(p);  // shared pages stay with their other holders
  const int n = (int)s.pages.size();
  s.pages.clear();
  s.len = 0;
  if (n) {
    std::fill(m->pt_host.begin() + (size_t)seq * m->max_pages, m->pt_host.begin() + (size_t)seq * m->max_pages + n, -1);
    CK(cudaMemcpyAsync(m->pt_dev + (size_t)seq * m->max_pages, &m->pt_host[(size_t)seq * m->max_pages],
                       n * sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
  }
  return DLS_OK;
}

// Pages that releasing all of `seqs` would return to the pool (pages shared
// with sequences outside the set stay allocated).
size_t reclaimable_pages(const dls_model* m, const int32_t* seqs, int n) {
  std::unordered_map<int, int> held;
  for (int i = 0; i < n; ++i)
    for (int p : m->seqs[seqs[i]].pages) ++held[p];
  size_t r = 0;
  for (const auto& kv : held)
    if (kv.second == m->page_ref[kv.first]) ++r;
  return r;
}

int check_seq(dls_model* m, int seq) {
  if (seq < 0 || seq >= m->max_seqs || !m->seqs[seq].live) return fail(m, DLS_ERR_ARG, "seq=%d not live", seq);
  return DLS_OK;
}

// Positions [0, len) that every row of a batched step reads from the same
// physical KV pages (a shared fork, or rows of one sequence): whole leading
// pages common to all rows, no further than the shortest row's length,
// rounded down to whole 32-token tiles.  0 below four tiles (not worth the
// extra launch) or with the cascade off.
int shared_prefix_len(const dls_model* m, int n, const int32_t* seqs, const int32_t* pos) {
  if (n < 2 || !m->cascade || !m->casc_o || m->mixed) return 0;
  int minpos = pos[0];
  for (int i = 1; i < n; ++i) minpos = std::min(minpos, pos[i]);
  const std::vector<int>& p0 = m->seqs[seqs[0]].pages;
  int k = 0;
  for (; k < (int)p0.size(); ++k) {
    bool same = true;
    for (int i = 1; i < n && same; ++i) {
      const std::vector<int>& pi = m->seqs[seqs[i]].pages;
      same = k < (int)pi.size() && pi[k] == p0[k];
    }
    if (!same) break;
  }
  const int len = std::min(k * m->pt, minpos) / 32 * 32;
  return len >= 128 ? len : 0;
}

int set_params(dls_model* m, int n, const int32_t* seqs, const int32_t* tokens, const int32_t* pos, bool reset) {
  StepParams h{};
  h.n = n;
  for (int i = 0; i < n; ++i) {
    h.seq[i] = seqs[i];
    h.token[i] = tokens[i];
    h.pos[i] = pos[i];
  }
  h.shared_len = shared_prefix_len(m, n, seqs, pos);
  m->casc_len = h.shared_len;
  m->casc_suffix_splits = 0;
  if (m->casc_len > 0) {
    // the per-row launch only covers the keys after the shared prefix; up
    // to 8 tiles of them take one split (its partial never leaves the CTA)
    int maxpos = pos[0];
    for (int i = 1; i < n; ++i) maxpos = std::max(maxpos, pos[i]);
    const int sfx_tiles = (maxpos + 1 - m->casc_len + 31) / 32;
    const int s = sfx_tiles <= 8 ? 1 : attn_default_splits(n, m->nkv, m->num_sms, m->max_ctx - m->casc_len);
    m->casc_suffix_splits = std::max(1, std::min(std::min(s, m->attn_splits_b), 128 - m->casc_splits));
  }
  CK(launch_set_params(m->sp, h, reset, m->stream));
  return DLS_OK;
}

// ---- weights: host blocks -> device layout -------------------------------------

int upload_matrix(dls_model* m, const void* host_blocks, int rows, int cols, uint8_t* dst_base, const MatOff& off,
                  int row0, uint8_t* temp, int row_step = 1) {
  const int nb = (cols + 31) / 32;
  const size_t bsz = m->wtype == 8 ? 34 : 18;
  const size_t bytes = (size_t)rows * nb * bsz;
  CK(cudaMemcpyAsync(temp, host_blocks, bytes, cudaMemcpyHostToDevice, m->stream));
  const size_t rb = off.qs_bytes / off.rows;
  CK(launch_repack(temp, m->wtype, rows, nb, off.ds, row_step, dst_base + off.qs + (size_t)row0 * rb,
                   reinterpret_cast<__half*>(dst_base + off.d) + (size_t)row0 * off.ds, m->stream));
  return DLS_OK;
}

// host GGUF K-quant super-blocks -> the packed device layout at dst
int upload_kq(dls_model* m, const void* host_blocks, int type, int rows, int cols, uint8_t* dst, uint8_t* temp) {
  CK(cudaMemcpyAsync(temp, host_blocks, kq_host_bytes(type, rows, cols), cudaMemcpyHostToDevice, m->stream));
  CK(launch_kq_pack(type, temp, rows, cols, dst, m->stream));
  // the next upload reuses temp: the pack must have read it
  return sync_stream(m, m->stream);
}

int upload_layer(dls_model* m, const dls_layer_desc& ld, uint8_t* dst, uint8_t* temp) {
  CK(cudaMemcpyAsync(dst + m->lay.attn_norm, ld.attn_norm, m->H * sizeof(float), cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(dst + m->lay.ffn_norm, ld.ffn_norm, m->H * sizeof(float), cudaMemcpyHostToDevice, m->stream));
  if (m->mixed) {
    const void* src[7] = {ld.wq, ld.wk, ld.wv, ld.wo, ld.w_gate, ld.w_up, ld.w_down};
    for (int i = 0; i < 7; ++i) {
      int rows, cols;
      mix_shape(m, i, &rows, &cols);
      if (m->mtype[i]) TRY(upload_kq(m, src[i], m->mtype[i], rows, cols, dst + m->mkq[i], temp));
      else TRY(upload_matrix(m, src[i], rows, cols, dst, m->mleg[i], 0, temp));
    }
    return DLS_OK;
  }
  TRY(upload_matrix(m, ld.wq, m->q_rows, m->H, dst, m->lay.qkv, 0, temp));
  TRY(upload_matrix(m, ld.wk, m->kv_rows, m->H, dst, m->lay.qkv, m->q_rows, temp));
  TRY(upload_matrix(m, ld.wv, m->kv_rows, m->H, dst, m->lay.qkv, m->q_rows + m->kv_rows, temp));
  TRY(upload_matrix(m, ld.wo, m->H, m->q_rows, dst, m->lay.o, 0, temp));
  // gate and up rows interleaved: row 2i = gate_i, row 2i+1 = up_i
  TRY(upload_matrix(m, ld.w_gate, m->F, m->H, dst, m->lay.gu, 0, temp, 2));
  TRY(upload_matrix(m, ld.w_up, m->F, m->H, dst, m->lay.gu, 1, temp, 2));
  TRY(upload_matrix(m, ld.w_down, m->H, m->F, dst, m->lay.down, 0, temp));
  return DLS_OK;
}

size_t staging_bytes(const dls_model* m) { return 2 * a256(m->lay.bytes); }

// Largest resident count the budget allows given what else is allocated.
int auto_resident(const dls_model* m, uint64_t other_bytes) {
  if (!m->budget) return m->L;
  const uint64_t lb = a256(m->lay.bytes);
  if (other_bytes + (uint64_t)m->L * lb <= m->budget) return m->L;
  if (other_bytes + staging_bytes(m) > m->budget) return -1;
  const uint64_t room = m->budget - other_bytes - staging_bytes(m);
  return (int)std::min<uint64_t>(room / lb, (uint64_t)m->L - 1);
}

int setup_persistent(dls_model* m);

int step_scratch(dls_model* m, std::vector<void*>* made);

// Change the resident count to n, all or nothing (the LayerStreamer page's
// ledger: reserve, commit on success, roll back on failure).  Everything the
// new layout needs -- pinned host copies of the layers to evict, the two
// staging buffers, device copies of the layers to load, the persistent
// kernel's scratch -- is allocated first; if any allocation fails, what this
// call allocated is released and the model is unchanged.  Only then are
// layers copied and the old buffers freed.  While it allocates, the ledger
// credits the bytes the commit will free, so the budget is checked against
// the final layout (the device briefly holds both).
int apply_resident(dls_model* m, int n) {
  std::vector<int> evict, load;
  for (int l = n; l < m->L; ++l)
    if (m->layer_dev[l]) evict.push_back(l);
  for (int l = 0; l < n; ++l)
    if (!m->layer_dev[l]) load.push_back(l);
  const bool need_stage = n < m->L && !m->stage[0];
  const bool drop_stage = n >= m->L && m->stage[0];
  std::vector<int> new_host;   // layers whose pinned host copy this call made
  std::vector<void*> new_dev;  // device buffers this call allocated
  auto rollback = [&](int r) {
    m->credit = 0;
    cudaStreamSynchronize(m->stream);  // no copy into a buffer about to be released is left in flight
    for (void* p : new_dev) dev_free(m, p);
    for (int l : new_host) {
      cudaFreeHost(m->layer_host[l]);
      m->layer_host[l] = nullptr;
    }
    return r;
  };
  // 1. pinned host copies of the layers to evict
  for (int l : evict) {
    if (m->layer_host[l]) continue;
    void* h = nullptr;
    if (cudaHostAlloc(&h, m->lay.bytes, cudaHostAllocDefault) != cudaSuccess || !h) {
      cudaGetLastError();
      return rollback(fail(m, DLS_ERR_CUDA, "what=pinned_layer_copy layer=%d bytes=%zu allocation failed", l,
                           m->lay.bytes));
    }
    m->layer_host[l] = static_cast<uint8_t*>(h);
    new_host.push_back(l);
    if (cudaMemcpyAsync(h, m->layer_dev[l], m->lay.bytes, cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
      return rollback(fail(m, DLS_ERR_CUDA, "layer=%d copy to host failed", l));
  }
  // 2. device memory of the new layout
  m->credit = (uint64_t)evict.size() * a256(m->lay.bytes) + (drop_stage ? staging_bytes(m) : 0);
  uint8_t* stage_new[2] = {nullptr, nullptr};
  if (need_stage) {
    for (auto& st : stage_new) {
      void* p = nullptr;
      const int r = dev_alloc(m, m->lay.bytes, &p, "stream_buffer");
      if (r != DLS_OK) return rollback(r);
      new_dev.push_back(p);
      st = static_cast<uint8_t*>(p);
    }
  }
  std::vector<uint8_t*> load_ptr;
  for (int l : load) {
    void* p = nullptr;
    const int r = dev_alloc(m, m->lay.bytes, &p, "layer");
    if (r != DLS_OK) return rollback(r);
    (void)l;
    new_dev.push_back(p);
    load_ptr.push_back(static_cast<uint8_t*>(p));
  }
  if (n >= m->L) {
    const int r = step_scratch(m, &new_dev);
    if (r != DLS_OK) return rollback(r);
  }
  m->credit = 0;
  {
    const int r = sync_stream(m, m->stream);  // the host copies have landed
    if (r != DLS_OK) return rollback(r);
  }
  // 3. commit
  for (size_t i = 0; i < load.size(); ++i) {
    m->layer_dev[load[i]] = load_ptr[i];
    CK(cudaMemcpyAsync(load_ptr[i], m->layer_host[load[i]], m->lay.bytes, cudaMemcpyHostToDevice, m->stream));
  }
  for (int l : evict) {
    dev_free(m, m->layer_dev[l]);
    m->layer_dev[l] = nullptr;
  }
  if (drop_stage) {
    for (auto& st : m->stage) {
      dev_free(m, st);
      st = nullptr;
    }
  }
  if (need_stage) {
    m->stage[0] = stage_new[0];
    m->stage[1] = stage_new[1];
  }
  TRY(sync_stream(m, m->stream));
  m->resident = n;
  drop_graphs(m);
  return setup_persistent(m);
}

// Scratch of the persistent step kernel for the model's plan, allocated once;
// `made` (may be NULL) collects what this call allocated.
int step_scratch(dls_model* m, std::vector<void*>* made) {
  const char* e = getenv("DLS_STEP_KERNEL");
  if (e && atoi(e) == 0) return DLS_OK;
  if (m->mixed) return DLS_OK;
  if (!m->step.fn) m->step = step_plan(m->wtype, m->H, m->q_rows, m->F, m->nh, m->nkv, m->hd, m->num_sms);
  if (!m->step.fn || m->step_layers) return DLS_OK;
  const int g = m->nh / m->nkv, S = m->step.splits;
  std::vector<void*> got;
  auto one = [&](size_t bytes, const char* what, void** out) {
    const int r = dev_alloc(m, bytes, out, what);
    if (r == DLS_OK) got.push_back(*out);
    return r;
  };
  void* p[8] = {};
  int r = one((size_t)m->L * sizeof(StepLayer), "step_layers", &p[0]);
  if (r == DLS_OK) r = one((size_t)m->nkv * S * g * m->hd * sizeof(float), "step_attention_partials", &p[1]);
  if (r == DLS_OK) r = one((size_t)m->nkv * S * g * 2 * sizeof(float), "step_attention_ml", &p[2]);
  if (r == DLS_OK) r = one((size_t)m->nkv * sizeof(int), "step_attention_counters", &p[3]);
  if (r == DLS_OK) r = one((size_t)m->step.grid * sizeof(int2), "step_argmax", &p[4]);
  if (r == DLS_OK) r = one(2 * sizeof(unsigned), "step_barrier", &p[5]);
  if (r == DLS_OK) r = one((size_t)(5 * m->L + 8) * sizeof(unsigned long long), "step_trace", &p[6]);
  if (r == DLS_OK)
    r = one((size_t)(5 * m->L + 8) * m->step.grid * 8 * sizeof(unsigned long long), "step_cta_trace", &p[7]);
  if (r == DLS_OK && cudaMemsetAsync(p[3], 0, m->nkv * sizeof(int), m->stream) != cudaSuccess)
    r = fail(m, DLS_ERR_CUDA, "clearing the step counters failed");
  if (r != DLS_OK) {
    for (void* q : got) dev_free(m, q);
    return r;
  }
  m->step_layers = static_cast<StepLayer*>(p[0]);
  m->step_part_o = static_cast<float*>(p[1]);
  m->step_part_ml = static_cast<float*>(p[2]);
  m->step_att_cnt = static_cast<int*>(p[3]);
  m->step_am = static_cast<int2*>(p[4]);
  m->step_bar = static_cast<unsigned*>(p[5]);
  m->step_trace = static_cast<unsigned long long*>(p[6]);
  m->step_ctrace = static_cast<unsigned long long*>(p[7]);
  if (made) made->insert(made->end(), got.begin(), got.end());
  return DLS_OK;
}

// Plan the persistent step kernel when every layer is resident; allocate its
// scratch once.  Without a plan the step runs as separate kernels.
int setup_persistent(dls_model* m) {
  m->use_step = false;
  // the default for batch-1 steps of a resident model; DLS_STEP_KERNEL=0
  // runs them as separate kernels instead
  const char* e = getenv("DLS_STEP_KERNEL");
  if (e && atoi(e) == 0) return DLS_OK;
  if (m->resident < m->L || m->mixed) return DLS_OK;
  TRY(step_scratch(m, nullptr));
  if (!m->step.fn) return DLS_OK;
  std::vector<StepLayer> hl(m->L);
  for (int l = 0; l < m->L; ++l) {
    const LayerPtrs P = layer_ptrs(m, m->layer_dev[l]);
    hl[l].attn_norm = P.attn_norm;
    hl[l].ffn_norm = P.ffn_norm;
    hl[l].qkv = P.qkv;
    hl[l].o = P.o;
    hl[l].gu = P.gu;
    hl[l].down = P.down;
    hl[l].k_pool = m->k_pool + (size_t)l * m->kv_layer_elems;
    hl[l].v_pool = m->v_pool + (size_t)l * m->kv_layer_elems;
  }
  CK(cudaMemcpyAsync(m->step_layers, hl.data(), hl.size() * sizeof(StepLayer), cudaMemcpyHostToDevice, m->stream));
  TRY(sync_stream(m, m->stream));
  m->use_step = true;
  return DLS_OK;
}

void destroy(dls_model* m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  if (m->copy_stream) cudaStreamSynchronize(m->copy_stream);
  drop_graphs(m);
  while (!m->allocs.empty()) dev_free(m, m->allocs.back().first);
  for (auto* h : m->layer_host)
    if (h) cudaFreeHost(h);
  for (int i = 0; i < 2; ++i) {
    if (m->ev_filled[i]) cudaEventDestroy(m->ev_filled[i]);
    if (m->ev_free[i]) cudaEventDestroy(m->ev_free[i]);
  }
  if (m->ev_start) cudaEventDestroy(m->ev_start);
  for (auto e : m->prof_events) cudaEventDestroy(e);
  if (m->copy_stream) cudaStreamDestroy(m->copy_stream);
  if (m->own_stream && m->stream) cudaStreamDestroy(m->stream);
  delete m;
}

int validate_desc(const dls_model_desc* d) {
  dls_model* m = nullptr;
  if (!d) return fail(m, DLS_ERR_ARG, "desc=NULL");
  if (d->n_layers < 1 || d->hidden < 32 || d->n_heads < 1 || d->n_kv_heads < 1 || d->ffn < 1 || d->vocab < 1)
    return fail(m, DLS_ERR_ARG, "shape n_layers=%d hidden=%d n_heads=%d n_kv_heads=%d ffn=%d vocab=%d", d->n_layers,
                d->hidden, d->n_heads, d->n_kv_heads, d->ffn, d->vocab);
  if (d->hidden % 32) return fail(m, DLS_ERR_ARG, "hidden=%d not a multiple of 32", d->hidden);
  if (d->n_heads % d->n_kv_heads || d->n_heads / d->n_kv_heads > 16)
    return fail(m, DLS_ERR_ARG, "n_heads=%d n_kv_heads=%d (groups of at most 16)", d->n_heads, d->n_kv_heads);
  if (d->head_dim != 32 && d->head_dim != 64 && d->head_dim != 128)
    return fail(m, DLS_ERR_ARG, "head_dim=%d (32, 64 or 128)", d->head_dim);
  if (d->wtype != DLS_Q8_0 && d->wtype != DLS_Q4_0) return fail(m, DLS_ERR_ARG, "wtype=%d", d->wtype);
  const int pt = d->page_tokens ? d->page_tokens : 64;
  if (pt != 32 && pt != 64 && pt != 128 && pt != 256) return fail(m, DLS_ERR_ARG, "page_tokens=%d", d->page_tokens);
  if (d->max_seqs < 1 || d->max_ctx < 1) return fail(m, DLS_ERR_ARG, "max_seqs=%d max_ctx=%d", d->max_seqs, d->max_ctx);
  if (d->max_batch < 0 || d->max_batch > DLS_MAX_BATCH) return fail(m, DLS_ERR_ARG, "max_batch=%d", d->max_batch);
  if (d->kv_pool_pages < 0) return fail(m, DLS_ERR_ARG, "kv_pool_pages=%d", d->kv_pool_pages);
  if (!(d->rope_theta > 0.f) || !(d->rms_eps >= 0.f))
    return fail(m, DLS_ERR_ARG, "rope_theta=%g rms_eps=%g", d->rope_theta, d->rms_eps);
  if (!d->tok_embd || !d->output_norm || !d->layers || (!d->tied_embeddings && !d->output))
    return fail(m, DLS_ERR_ARG, "missing tensor pointer");
  auto kq = [](int t) { return t == DLS_Q4_K || t == DLS_Q5_K || t == DLS_Q6_K; };
  const int in_cols[7] = {d->hidden, d->hidden, d->hidden, d->n_heads * d->head_dim, d->hidden, d->hidden, d->ffn};
  for (int l = 0; l < d->n_layers; ++l) {
    const dls_layer_desc& L = d->layers[l];
    if (!L.attn_norm || !L.ffn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.w_gate || !L.w_up || !L.w_down)
      return fail(m, DLS_ERR_ARG, "layer=%d missing tensor pointer", l);
    for (int i = 0; i < 7; ++i) {
      const int t = L.types[i];
      if (t != 0 && !kq(t)) return fail(m, DLS_ERR_ARG, "layer=%d matrix=%d type=%d (0 or a K-quant type)", l, i, t);
      if (t != d->layers[0].types[i])
        return fail(m, DLS_ERR_ARG, "layer=%d matrix=%d type=%d differs from layer 0 (%d)", l, i, t,
                    d->layers[0].types[i]);
      if (kq(t) && (in_cols[i] % 256 || in_cols[i] > 32768))
        return fail(m, DLS_ERR_ARG, "matrix=%d input width %d: a K-quant matrix needs a multiple of 256 up to 32768",
                    i, in_cols[i]);
    }
  }
  for (int t : {d->tok_embd_type, d->output_type}) {
    if (t != 0 && !kq(t)) return fail(m, DLS_ERR_ARG, "embedding/output type=%d", t);
    if (kq(t) && d->hidden % 256) return fail(m, DLS_ERR_ARG, "K-quant embedding/output needs hidden %% 256 == 0");
  }
  return DLS_OK;
}

}  // namespace

int dls::report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = std::string("ERR ") + status_str(code) + " " + buf;
  return code;
}

// =================================================================== C ABI

extern "C" {

int dls_abi_version(void) { return DLS_ABI_VERSION; }
const char* dls_status_name(int s) { return status_str(s); }
const char* dls_last_error(const dls_model* m) { return m ? m->err.c_str() : g_err.c_str(); }
uint64_t dls_device_bytes(const dls_model* m) { return m ? m->used : 0; }
uint64_t dls_device_budget(const dls_model* m) { return m ? m->budget : 0; }
int32_t dls_resident_layers(const dls_model* m) { return m ? m->resident : -1; }
uint64_t dls_layer_bytes(const dls_model* m) { return m ? m->lay.bytes : 0; }
int32_t dls_debug_launches_per_step(const dls_model* m) { return m ? m->launches_per_step : -1; }

int dls_h2d_copy_sm(void* dst, const void* src_host, size_t bytes, int32_t ctas, void* cuda_stream) {
  if (!dst || !src_host || ctas < 1 || ctas > 4096)
    return fail(nullptr, DLS_ERR_ARG, "h2d_copy_sm dst=%p src=%p ctas=%d", dst, src_host, ctas);
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src_host) | bytes) & 15)
    return fail(nullptr, DLS_ERR_ARG, "h2d_copy_sm: pointers and bytes must be 16-byte multiples (bytes=%zu)", bytes);
  // the kernel dereferences src on the device: only pinned (page-locked,
  // mapped) host memory and device memory of this GPU are accepted
  cudaPointerAttributes as, ad;
  if (cudaPointerGetAttributes(&as, src_host) != cudaSuccess || cudaPointerGetAttributes(&ad, dst) != cudaSuccess) {
    cudaGetLastError();
    return fail(nullptr, DLS_ERR_ARG, "h2d_copy_sm: pointer attributes unavailable");
  }
  if (as.type != cudaMemoryTypeHost || !as.devicePointer || ad.type != cudaMemoryTypeDevice)
    return fail(nullptr, DLS_ERR_ARG, "h2d_copy_sm: src must be pinned host memory, dst device memory "
                "(types %d, %d)", (int)as.type, (int)ad.type);
  const cudaError_t e = launch_h2d_sm(dst, as.devicePointer, bytes, ctas, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return fail(nullptr, DLS_ERR_CUDA, "h2d_copy_sm cuda=%s", cudaGetErrorString(e));
  return DLS_OK;
}

int dls_check_context_budget(int32_t prefix_tokens, int32_t max_branch_tokens, int32_t headroom, int32_t n_ctx) {
  dls_model* m = nullptr;
  if (prefix_tokens < 0 || max_branch_tokens < 0 || headroom < 0 || n_ctx < 0)
    return fail(m, DLS_ERR_ARG, "negative token count");
  const long long required = (long long)prefix_tokens + max_branch_tokens + headroom;
  if (required > n_ctx)
    return fail(m, DLS_ERR_CAPACITY, "prefix_tokens=%d max_branch_tokens=%d headroom=%d required=%lld n_ctx=%d",
                prefix_tokens, max_branch_tokens, headroom, required, n_ctx);
  return DLS_OK;
}

int dls_model_create(const dls_model_desc* desc, const dls_allocator* allocator, void* cuda_stream, dls_model** out) {
  if (!out) return fail(nullptr, DLS_ERR_ARG, "out=NULL");
  *out = nullptr;
  TRY(validate_desc(desc));
  if (allocator && (!allocator->alloc || !allocator->free)) return fail(nullptr, DLS_ERR_ARG, "allocator callbacks");
  dls_model* m = new dls_model();
  const dls_model_desc& d = *desc;
  m->L = d.n_layers;
  m->H = d.hidden;
  m->nh = d.n_heads;
  m->nkv = d.n_kv_heads;
  m->hd = d.head_dim;
  m->F = d.ffn;
  m->V = d.vocab;
  m->wtype = d.wtype;
  m->pt = d.page_tokens ? d.page_tokens : 64;
  m->max_seqs = d.max_seqs;
  m->max_ctx = d.max_ctx;
  m->max_batch = d.max_batch ? d.max_batch : 1;
  m->max_pages = (d.max_ctx + m->pt - 1) / m->pt;
  m->theta = d.rope_theta;
  m->eps = d.rms_eps;
  m->tied = d.tied_embeddings != 0;
  m->q_rows = d.n_heads * d.head_dim;
  m->kv_rows = d.n_kv_heads * d.head_dim;
  m->budget = d.device_budget_bytes;
  if (allocator) {
    m->alloc = *allocator;
    m->have_alloc = true;
  }
  if (const char* e = getenv("DLS_PDL")) m->pdl = atoi(e) != 0;
  if (const char* e = getenv("DLS_STREAM_COPY"))
    if (strncmp(e, "sm:", 3) == 0) m->stream_sm_ctas = std::max(0, std::min(4096, atoi(e + 3)));
  auto bail = [&](int r) {
    std::string e = m->err;
    destroy(m);
    g_err = e;
    return r;
  };
#define CKC(call)                                                                                           \
  do {                                                                                                      \
    cudaError_t e_ = (call);                                                                                \
    if (e_ != cudaSuccess) return bail(fail(m, DLS_ERR_CUDA, "call=%s cuda=%s", #call, cudaGetErrorString(e_))); \
  } while (0)
#define TRYC(expr)                 \
  do {                             \
    int r_ = (expr);               \
    if (r_ != DLS_OK) return bail(r_); \
  } while (0)

  int dev = 0;
  CKC(cudaGetDevice(&dev));
  CKC(cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev));
  if (cuda_stream) {
    m->stream = static_cast<cudaStream_t>(cuda_stream);
  } else {
    CKC(cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking));
    m->own_stream = true;
  }
  CKC(cudaStreamCreateWithFlags(&m->copy_stream, cudaStreamNonBlocking));
  for (int i = 0; i < 2; ++i) {
    CKC(cudaEventCreateWithFlags(&m->ev_filled[i], cudaEventDisableTiming));
    CKC(cudaEventCreateWithFlags(&m->ev_free[i], cudaEventDisableTiming));
  }
  CKC(cudaEventCreateWithFlags(&m->ev_start, cudaEventDisableTiming));
  CKC(gemv_setup_attributes());
  CKC(tgemm_setup_attributes());
  CKC(cgemm_setup_attributes());
  // prompt chunks: the split-plane GEMM (default, faster as measured) or the
  // exact-code GEMM (DLS_PREFILL_GEMM=codes)
  if (const char* e = getenv("DLS_PREFILL_GEMM")) m->pf_planes = strcmp(e, "codes") != 0;
  if (const char* e = getenv("DLS_PREFILL_BN")) m->pf_bn = atoi(e) == 128 ? 128 : atoi(e) == 256 ? 256 : 0;
  CKC(sgemm_setup_attributes());
  CKC(rgemv_setup_attributes());
  // batched steps: the multi-row CUDA-core GEMV for 2-4 rows, the
  // small-batch tensor-core GEMM for 5-8 (measured on the 8B Q8_0 model at
  // ctx 2048, per step: 3.5 vs 5.5 ms at 2 rows, 4.6 vs 5.9 at 4, 7.4 vs 6.5
  // at 8); DLS_BATCH_GEMM=tc or =rg selects one for every batch size
  if (const char* e = getenv("DLS_BATCH_GEMM")) {
    m->batch_tc = strcmp(e, "tc") == 0;
    m->batch_rg = strcmp(e, "rg") == 0;
  }
  CKC(prefill_setup_attributes());
  CKC(fattn_setup_attributes());

  // per-matrix types (validated: every layer gives the same)
  for (int i = 0; i < 7; ++i) m->mtype[i] = d.layers[0].types[i];
  m->emb_type = d.tok_embd_type;
  m->out_type = m->tied ? 0 : d.output_type;
  m->mixed = m->emb_type || m->out_type;
  for (int i = 0; i < 7; ++i) m->mixed |= m->mtype[i] != 0;
  if (m->mixed) CKC(kq_setup_attributes());

  // layouts
  size_t cur = 0;
  m->lay.attn_norm = cur;
  cur = a256(cur + m->H * sizeof(float));
  m->lay.ffn_norm = cur;
  cur = a256(cur + m->H * sizeof(float));
  if (!m->mixed) {
    m->lay.qkv = mat_off(cur, m->q_rows + 2 * m->kv_rows, m->H, m->wtype);
    m->lay.o = mat_off(cur, m->H, m->q_rows, m->wtype);
    m->lay.gu = mat_off(cur, 2 * m->F, m->H, m->wtype);
    m->lay.down = mat_off(cur, m->H, m->F, m->wtype);
  } else {
    // the seven matrices one after another, each in its own format
    for (int i = 0; i < 7; ++i) {
      int rows, cols;
      mix_shape(m, i, &rows, &cols);
      if (m->mtype[i]) {
        m->mkq[i] = cur;
        cur = a256(cur + kq_packed_bytes(m->mtype[i], rows, cols));
      } else {
        m->mleg[i] = mat_off(cur, rows, cols, m->wtype);
      }
    }
  }
  m->lay.bytes = cur;
  cur = 0;
  m->emb_off = mat_off(cur, m->V, m->H, m->wtype);
  m->emb_bytes = m->emb_type ? kq_packed_bytes(m->emb_type, m->V, m->H) : cur;
  cur = 0;
  m->out_off = mat_off(cur, m->V, m->H, m->wtype);
  m->out_bytes = m->out_type ? kq_packed_bytes(m->out_type, m->V, m->H) : cur;

  m->plan_qkv = gemv_plan(m->wtype, PRO_RMSNORM, EPI_QKV, m->lay.qkv.rows, m->lay.qkv.nb, m->num_sms, 2);
  m->plan_o = gemv_plan(m->wtype, PRO_COPY, EPI_RESID, m->lay.o.rows, m->lay.o.nb, m->num_sms, 1);
  m->plan_gu = gemv_plan(m->wtype, PRO_RMSNORM, EPI_SWIGLU, m->lay.gu.rows, m->lay.gu.nb, m->num_sms, 2);
  m->plan_down = gemv_plan(m->wtype, PRO_COPY, EPI_RESID, m->lay.down.rows, m->lay.down.nb, m->num_sms, 1);
  m->plan_head = gemv_plan(m->wtype, PRO_RMSNORM, EPI_STORE, m->V, m->emb_off.nb, m->num_sms, 1);
  m->attn_splits = attn_default_splits(1, m->nkv, m->num_sms, m->max_ctx);

  // fixed allocations (everything but the layers)
  const int B = m->max_batch;
  m->n_pages = d.kv_pool_pages > 0 ? d.kv_pool_pages : m->max_seqs * m->max_pages;
  m->page_elems = (size_t)m->nkv * m->pt * m->hd;
  m->kv_layer_elems = (size_t)m->n_pages * m->page_elems;
  m->rope_len = m->max_ctx;
  const size_t bsz = m->wtype == 8 ? 34 : 18;
  size_t temp_bytes = (size_t)m->V * m->emb_off.nb * bsz;
  temp_bytes = std::max(temp_bytes, (size_t)2 * m->F * ((m->H + 31) / 32) * bsz);
  temp_bytes = std::max(temp_bytes, (size_t)m->H * ((m->F + 31) / 32) * bsz);
  for (int i = 0; i < 7; ++i)
    if (m->mtype[i]) {
      int rows, cols;
      mix_shape(m, i, &rows, &cols);
      temp_bytes = std::max(temp_bytes, kq_host_bytes(m->mtype[i], rows, cols));
    }
  for (int t : {m->emb_type, m->out_type})
    if (t) temp_bytes = std::max(temp_bytes, kq_host_bytes(t, m->V, m->H));
  void* p = nullptr;
  TRYC(dev_alloc(m, m->emb_bytes, &p, "tok_embd"));
  m->emb_block = static_cast<uint8_t*>(p);
  // padding (the scale rows' round-up to 8 blocks, alignment gaps) stays zero:
  // the tensor-core GEMMs read whole 64-column tiles, and a zero-filled code
  // times a stale scale could be 0 * inf
  CKC(cudaMemsetAsync(m->emb_block, 0, m->emb_bytes, m->stream));
  if (!m->tied) {
    TRYC(dev_alloc(m, m->out_bytes, &p, "output"));
    m->out_block = static_cast<uint8_t*>(p);
    CKC(cudaMemsetAsync(m->out_block, 0, m->out_bytes, m->stream));
  }
  if (m->mixed) TRYC(dev_alloc_t(m, (size_t)m->H + std::max(m->H, m->q_rows), &m->mix_buf, "mixed_path_vectors"));
  TRYC(dev_alloc_t(m, m->H, &m->out_norm, "output_norm"));
  TRYC(dev_alloc_t(m, (size_t)m->L * m->kv_layer_elems, &m->k_pool, "k_cache"));
  TRYC(dev_alloc_t(m, (size_t)m->L * m->kv_layer_elems, &m->v_pool, "v_cache"));
  // positions past a sequence's length inside its last page are read (and
  // given zero weight) by the prefill attention: keep them finite
  CKC(cudaMemsetAsync(m->k_pool, 0, (size_t)m->L * m->kv_layer_elems * sizeof(__half), m->stream));
  CKC(cudaMemsetAsync(m->v_pool, 0, (size_t)m->L * m->kv_layer_elems * sizeof(__half), m->stream));
  TRYC(dev_alloc_t(m, (size_t)m->max_seqs * m->max_pages, &m->pt_dev, "page_table"));
  // per-row scratch for batched steps: a user batch, or the rows of one
  // speculative verify pass (up to kMaxBatch)
  const int BR = std::max(B, kMaxBatch);
  TRYC(dev_alloc_t(m, (size_t)BR * m->H, &m->x, "x"));
  TRYC(dev_alloc_t(m, (size_t)BR * m->q_rows, &m->q, "q"));
  TRYC(dev_alloc_t(m, (size_t)BR * m->q_rows, &m->o, "o"));
  TRYC(dev_alloc_t(m, (size_t)BR * 2 * m->F, &m->gu, "gate_up"));
  // logits rows: a batch, or the rows of one dls_verify pass
  TRYC(dev_alloc_t(m, (size_t)std::max(B, DLS_MAX_VERIFY) * m->V, &m->logits, "logits"));
  TRYC(dev_alloc_t(m, (size_t)std::max(kMaxBatch, DLS_MAX_VERIFY), &m->next_tok, "next_token"));
  TRYC(dev_alloc_t(m, (size_t)4096, &m->argmax_buf, "argmax"));
  TRYC(dev_alloc_t(m, (size_t)4096 + 2 * m->num_sms, &m->argmax_part, "argmax_partials"));
  TRYC(dev_alloc_t(m, (size_t)4096, &m->argmax_cnt, "argmax_counters"));
  TRYC(dev_alloc_t(m, 1, &m->sp, "step_params"));
  TRYC(dev_alloc_t(m, (size_t)m->rope_len * (m->hd / 2), &m->rope, "rope_table"));
  const size_t ws = attn_workspace_bytes(1, m->nh, m->nkv, m->hd, m->attn_splits);
  TRYC(dev_alloc(m, ws, &m->attn_ws, "attention_scratch"));
  attn_workspace_carve(m->attn_ws, 1, m->nh, m->nkv, m->hd, m->attn_splits, &m->part_o, &m->part_ml, &m->counters);
  m->pairs_cap = (size_t)m->max_pages * std::max(1, m->max_seqs - 1);
  TRYC(dev_alloc_t(m, m->pairs_cap, &m->pairs_dev, "fork_pairs"));
  m->pf_cap = std::min(m->max_ctx, kPrefillChunk);
  if (const char* e = getenv("DLS_PREFILL_CHUNK")) m->pf_cap = std::max(1, std::min(m->max_ctx, atoi(e)));
  m->pf_ldh = (m->F + 31) & ~31;
  // token-major scratch shared by prefill chunks and batched decode rows
  const size_t pf_rows = (size_t)std::max(std::max(m->pf_cap, B), DLS_MAX_VERIFY);
  TRYC(dev_alloc_t(m, pf_rows * m->H, &m->pf_x, "prefill_x"));
  TRYC(dev_alloc_t(m, 2 * pf_rows * std::max(m->H, m->q_rows), &m->pf_a, "prefill_a16"));
  m->pf_a_lo = m->pf_a + pf_rows * std::max(m->H, m->q_rows);
  TRYC(dev_alloc_t(m, pf_rows * (m->q_rows + 2 * m->kv_rows), &m->pf_qkv, "prefill_qkv"));
  TRYC(dev_alloc_t(m, pf_rows * m->q_rows, &m->pf_q, "prefill_q"));
  TRYC(dev_alloc_t(m, 2 * pf_rows * m->pf_ldh, &m->pf_h, "prefill_h16"));
  m->pf_h_lo = m->pf_h + pf_rows * m->pf_ldh;
  TRYC(dev_alloc_t(m, pf_rows, &m->pf_tok, "prefill_tokens"));
  {
    m->attn_splits_b = attn_default_splits(BR, m->nkv, m->num_sms, m->max_ctx);
    const size_t wsb = attn_workspace_bytes(BR, m->nh, m->nkv, m->hd, m->attn_splits_b);
    TRYC(dev_alloc(m, wsb, &m->attn_ws_b, "attention_scratch_batch"));
    attn_workspace_carve(m->attn_ws_b, BR, m->nh, m->nkv, m->hd, m->attn_splits_b, &m->part_o_b, &m->part_ml_b,
                         &m->counters_b);
    CKC(cudaMemsetAsync(m->counters_b, 0, (size_t)BR * m->nkv * sizeof(int), m->stream));
  }
  if (const char* e = getenv("DLS_CASCADE")) m->cascade = atoi(e) != 0;
  if (BR >= 2 && cascade_supported(m->nh, m->nkv, m->hd)) {
    // the shared-prefix pass: on the tensor cores where the shape allows
    // (DLS_CASCADE_TC=0 keeps the CUDA-core kernel), one CTA per SM; the
    // CUDA-core kernel runs two CTAs per SM
    m->casc_tc = cascade_tc_supported(m->nh, m->nkv, m->hd, m->pt);
    if (const char* e = getenv("DLS_CASCADE_TC")) m->casc_tc = m->casc_tc && atoi(e) != 0;
    if (m->casc_tc) CKC(cascade_tc_setup_attributes());
    // prefix partials of cascade attention: [rows][n_kv][splits][group][head_dim]
    m->casc_splits = std::max(1, std::min((m->casc_tc ? 1 : 2) * m->num_sms / m->nkv, 64));
    const size_t slots = (size_t)std::min(BR, kMaxBatch) * m->nkv * m->casc_splits;
    const int g = m->nh / m->nkv;
    TRYC(dev_alloc_t(m, slots * g * m->hd, &m->casc_o, "cascade_partials"));
    TRYC(dev_alloc_t(m, slots * g * 2, &m->casc_ml, "cascade_ml"));
  }
  {
    // split-K partials for batches of up to 16 rows: [split][16][rows]
    // (the LM head of a batch or of a dls_verify pass included)
    const int max_rows = std::max(std::max(std::max(m->q_rows + 2 * m->kv_rows, 2 * m->F), m->H), m->V);
    m->tg_part_elems = (size_t)kTgMaxSplit * 16 * max_rows;
    TRYC(dev_alloc_t(m, m->tg_part_elems, &m->tg_part, "gemm_split_partials"));
    TRYC(dev_alloc_t(m, (size_t)kTgCounters, &m->tg_cnt, "gemm_split_counters"));
    CKC(cudaMemsetAsync(m->tg_cnt, 0, (size_t)kTgCounters * sizeof(int), m->stream));
  }
  // columns F .. pf_ldh of h are read by the down GEMM and never written
  CKC(cudaMemsetAsync(m->pf_h, 0, 2 * pf_rows * m->pf_ldh * sizeof(__half), m->stream));
  void* temp = nullptr;
  TRYC(dev_alloc(m, temp_bytes, &temp, "upload_temp"));

  // resident layers: as many as the budget allows (first layers first)
  m->layer_dev.assign(m->L, nullptr);
  m->layer_host.assign(m->L, nullptr);
  const int nres = auto_resident(m, m->used);
  if (nres < 0) return bail(fail(m, DLS_ERR_BUDGET, "fixed_bytes=%llu budget=%llu", (unsigned long long)m->used,
                                 (unsigned long long)m->budget));
  if (nres < m->L) {
    for (auto& st : m->stage) {
      TRYC(dev_alloc(m, m->lay.bytes, &p, "stream_buffer"));
      st = static_cast<uint8_t*>(p);
    }
  }
  for (int l = 0; l < nres; ++l) {
    TRYC(dev_alloc(m, m->lay.bytes, &p, "layer"));
    m->layer_dev[l] = static_cast<uint8_t*>(p);
  }
  m->resident = nres;

  // upload: norms, embeddings, layers (streamed layers go through buffer 0
  // and then to pinned host memory)
  CKC(cudaMemcpyAsync(m->out_norm, d.output_norm, m->H * sizeof(float), cudaMemcpyHostToDevice, m->stream));
  if (m->emb_type) TRYC(upload_kq(m, d.tok_embd, m->emb_type, m->V, m->H, m->emb_block, static_cast<uint8_t*>(temp)));
  else TRYC(upload_matrix(m, d.tok_embd, m->V, m->H, m->emb_block, m->emb_off, 0, static_cast<uint8_t*>(temp)));
  if (!m->tied) {
    if (m->out_type) TRYC(upload_kq(m, d.output, m->out_type, m->V, m->H, m->out_block, static_cast<uint8_t*>(temp)));
    else TRYC(upload_matrix(m, d.output, m->V, m->H, m->out_block, m->out_off, 0, static_cast<uint8_t*>(temp)));
  }
  for (int l = 0; l < m->L; ++l) {
    uint8_t* dst = l < nres ? m->layer_dev[l] : m->stage[0];
    CKC(cudaMemsetAsync(dst, 0, m->lay.bytes, m->stream));  // padding stays zero (as for the embedding)
    TRYC(upload_layer(m, d.layers[l], dst, static_cast<uint8_t*>(temp)));
    if (l >= nres) {
      void* h = nullptr;
      CKC(cudaHostAlloc(&h, m->lay.bytes, cudaHostAllocDefault));
      m->layer_host[l] = static_cast<uint8_t*>(h);
      CKC(cudaMemcpyAsync(h, dst, m->lay.bytes, cudaMemcpyDeviceToHost, m->stream));
    }
  }
  CKC(launch_rope_table(m->rope, m->rope_len, m->hd, m->theta, m->stream));
  m->pt_host.assign((size_t)m->max_seqs * m->max_pages, -1);
  CKC(cudaMemcpyAsync(m->pt_dev, m->pt_host.data(), m->pt_host.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                      m->stream));
  CKC(cudaMemsetAsync(m->attn_ws, 0, ws, m->stream));
  CKC(cudaMemsetAsync(m->argmax_cnt, 0, 4096 * sizeof(int), m->stream));
  CKC(cudaMemsetAsync(m->sp, 0, sizeof(StepParams), m->stream));
  TRYC(sync_stream(m, m->stream));
  dev_free(m, temp);
  m->free_pages.clear();
  for (int i = m->n_pages - 1; i >= 0; --i) m->free_pages.push_back(i);
  m->page_ref.assign(m->n_pages, 0);
  m->skip_host.assign(m->L, 0);
  TRYC(dev_alloc_t(m, (size_t)m->L, &m->skip_dev, "layer_skip"));
  CKC(cudaMemsetAsync(m->skip_dev, 0, m->L, m->stream));
  m->draft_host.assign(m->L, 0);
  m->no_skip.assign(m->L, 0);
  TRYC(dev_alloc_t(m, (size_t)m->L, &m->draft_dev, "draft_skip"));
  CKC(cudaMemsetAsync(m->draft_dev, 0, m->L, m->stream));
  TRYC(sync_stream(m, m->stream));
  m->seqs.assign(m->max_seqs, Seq());
  TRYC(setup_persistent(m));
  *out = m;
  return DLS_OK;
#undef CKC
#undef TRYC
}

void dls_model_destroy(dls_model* m) { destroy(m); }

int dls_seq_create(dls_model* m, int32_t* seq_out) {
  if (!m || !seq_out) return fail(m, DLS_ERR_ARG, "NULL argument");
  for (int i = 0; i < m->max_seqs; ++i)
    if (!m->seqs[i].live) {
      m->seqs[i].live = true;
      m->seqs[i].len = 0;
      *seq_out = i;
      return DLS_OK;
    }
  return fail(m, DLS_ERR_CAPACITY, "max_seqs=%d all live", m->max_seqs);
}

int dls_seq_free(dls_model* m, int32_t seq) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  TRY(release_pages(m, seq));
  m->seqs[seq].live = false;
  return DLS_OK;
}

int32_t dls_seq_length(const dls_model* m, int32_t seq) {
  if (!m || seq < 0 || seq >= m->max_seqs || !m->seqs[seq].live) return DLS_ERR_ARG;
  return m->seqs[seq].len;
}

int dls_prefill(dls_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  if (n < 1 || !tokens) return fail(m, DLS_ERR_ARG, "n=%d tokens=%p", n, (const void*)tokens);
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(m, DLS_ERR_ARG, "token[%d]=%d vocab=%d", i, tokens[i], m->V);
  Seq& s = m->seqs[seq];
  if ((long long)s.len + n > m->max_ctx)
    return fail(m, DLS_ERR_CAPACITY, "seq=%d length=%d n=%d max_ctx=%d", seq, s.len, n, m->max_ctx);
  TRY(ensure_pages(m, seq, s.len + n));
  const int32_t pos0 = s.len;
  TRY(set_params(m, 1, &seq, &tokens[0], &pos0, true));  // clears the device status word
  float* cap = m->capture;
  m->capture = nullptr;
  if (m->mixed) {
    // a mixed-format model: up to 8 prompt tokens per pass over the layers,
    // each token through the decode-step kernels (a streamed layer is copied
    // once per pass)
    for (int c0 = 0; c0 < n; c0 += kMaxBatch) {
      const int T = std::min(kMaxBatch, n - c0);
      int32_t seqs[kMaxBatch], poss[kMaxBatch];
      for (int t = 0; t < T; ++t) {
        seqs[t] = seq;
        poss[t] = pos0 + c0 + t;
      }
      if (c0 > 0) TRY(set_params(m, T, seqs, tokens + c0, poss, false));
      else TRY(set_params(m, T, seqs, tokens + c0, poss, true));
      m->launch_count = 0;
      const bool last = c0 + T == n;
      TRY(enqueue_mixed(m, T, last && logits_out, last ? T - 1 : -1, false, last ? cap : nullptr, T - 1));
    }
  } else {
    for (int c0 = 0; c0 < n; c0 += m->pf_cap) {
      const int T = std::min(m->pf_cap, n - c0);
      const bool last = c0 + T == n;
      TRY(enqueue_prefill(m, seq, tokens + c0, T, pos0 + c0, last && logits_out ? HEAD_LAST : HEAD_NONE,
                          last ? cap : nullptr));
    }
  }
  TRY(copy_out(m, logits_out, m->logits, (size_t)m->V * sizeof(float)));
  TRY(sync_stream(m, m->stream));
  TRY(check_status(m));
  s.len += n;
  return DLS_OK;
}

int dls_decode_step(dls_model* m, int32_t seq, int32_t token, int32_t pos, float* logits_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  if (token < 0 || token >= m->V) return fail(m, DLS_ERR_ARG, "token=%d vocab=%d", token, m->V);
  Seq& s = m->seqs[seq];
  if (pos != s.len) return fail(m, DLS_ERR_STATE, "seq=%d pos=%d length=%d", seq, pos, s.len);
  if (pos >= m->max_ctx) return fail(m, DLS_ERR_CAPACITY, "seq=%d pos=%d max_ctx=%d", seq, pos, m->max_ctx);
  TRY(ensure_pages(m, seq, pos + 1));
  TRY(set_params(m, 1, &seq, &token, &pos, true));
  TRY(run_step(m, 1, logits_out != nullptr, false));
  TRY(copy_out(m, logits_out, m->logits, (size_t)m->V * sizeof(float)));
  s.len += 1;
  return DLS_OK;
}

int dls_decode_batch(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, const int32_t* pos,
                     float* logits_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (n < 1 || n > m->max_batch || !seqs || !tokens || !pos)
    return fail(m, DLS_ERR_ARG, "n=%d max_batch=%d", n, m->max_batch);
  for (int i = 0; i < n; ++i) {
    TRY(check_seq(m, seqs[i]));
    for (int j = 0; j < i; ++j)
      if (seqs[j] == seqs[i]) return fail(m, DLS_ERR_ARG, "seq=%d repeated", seqs[i]);
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(m, DLS_ERR_ARG, "token[%d]=%d", i, tokens[i]);
    if (pos[i] != m->seqs[seqs[i]].len)
      return fail(m, DLS_ERR_STATE, "seq=%d pos=%d length=%d", seqs[i], pos[i], m->seqs[seqs[i]].len);
    if (pos[i] >= m->max_ctx) return fail(m, DLS_ERR_CAPACITY, "seq=%d pos=%d", seqs[i], pos[i]);
  }
  int need = 0;
  for (int i = 0; i < n; ++i)
    need += std::max(0, pages_needed(m, pos[i] + 1) - (int)m->seqs[seqs[i]].pages.size());
  if (need > (int)m->free_pages.size()) return fail(m, DLS_ERR_CAPACITY, "need_pages=%d free=%zu", need, m->free_pages.size());
  for (int i = 0; i < n; ++i) TRY(ensure_pages(m, seqs[i], pos[i] + 1));
  TRY(set_params(m, n, seqs, tokens, pos, true));
  TRY(run_step(m, n, logits_out != nullptr, false));
  TRY(copy_out(m, logits_out, m->logits, (size_t)n * m->V * sizeof(float)));
  for (int i = 0; i < n; ++i) m->seqs[seqs[i]].len += 1;
  return DLS_OK;
}

int dls_generate(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, int32_t n_steps,
                 int32_t* tokens_out, float* last_logits) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (n < 1 || n > m->max_batch || !seqs || !tokens || n_steps < 1 || !tokens_out)
    return fail(m, DLS_ERR_ARG, "n=%d n_steps=%d", n, n_steps);
  std::vector<int32_t> pos(n);
  int need = 0;
  for (int i = 0; i < n; ++i) {
    TRY(check_seq(m, seqs[i]));
    for (int j = 0; j < i; ++j)
      if (seqs[j] == seqs[i]) return fail(m, DLS_ERR_ARG, "seq=%d repeated", seqs[i]);
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(m, DLS_ERR_ARG, "token[%d]=%d", i, tokens[i]);
    pos[i] = m->seqs[seqs[i]].len;
    if ((long long)pos[i] + n_steps > m->max_ctx)
      return fail(m, DLS_ERR_CAPACITY, "seq=%d length=%d n_steps=%d max_ctx=%d", seqs[i], pos[i], n_steps, m->max_ctx);
    need += std::max(0, pages_needed(m, pos[i] + n_steps) - (int)m->seqs[seqs[i]].pages.size());
  }
  if (need > (int)m->free_pages.size()) return fail(m, DLS_ERR_CAPACITY, "need_pages=%d free=%zu", need, m->free_pages.size());
  const size_t ntok = (size_t)n * n_steps;
  if (ntok > m->tokens_cap) {
    int32_t* t = nullptr;
    TRY(dev_alloc_t(m, std::max<size_t>(ntok, 1024), &t, "generated_tokens"));
    dev_free(m, m->tokens_dev);
    m->tokens_dev = t;
    m->tokens_cap = std::max<size_t>(ntok, 1024);
    drop_graphs(m);  // graphs bake the output pointer in
  }
  for (int i = 0; i < n; ++i) TRY(ensure_pages(m, seqs[i], pos[i] + n_steps));
  TRY(set_params(m, n, seqs, tokens, pos.data(), true));
  for (int t = 0; t < n_steps; ++t) TRY(run_step(m, n, true, true));
  CK(cudaMemcpyAsync(tokens_out, m->tokens_dev, ntok * sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
  TRY(copy_out(m, last_logits, m->logits, (size_t)n * m->V * sizeof(float)));
  TRY(sync_stream(m, m->stream));
  TRY(check_status(m));
  for (int i = 0; i < n; ++i) m->seqs[seqs[i]].len += n_steps;
  return DLS_OK;
}

// Cut `seq` back to `len` positions: pages past them return to the pool
// (a shared page stays with its other holders), and the page position len
// falls in, when partly kept and shared, is replaced by a private copy so
// that later appends never write into a page another sequence reads.
int truncate_seq(dls_model* m, int seq, int len) {
  Seq& s = m->seqs[seq];
  if (len < 0 || len > s.len) return fail(m, DLS_ERR_ARG, "seq=%d truncate to %d of length %d", seq, len, s.len);
  const int keep = std::min(pages_needed(m, len), (int)s.pages.size());
  const bool cow = len % m->pt && keep > 0 && m->page_ref[s.pages[keep - 1]] > 1;
  if (cow) {
    size_t avail = m->free_pages.size();
    for (size_t k = keep; k < s.pages.size(); ++k) avail += m->page_ref[s.pages[k]] == 1 ? 1 : 0;
    if (avail < 1) return fail(m, DLS_ERR_CAPACITY, "seq=%d truncate needs a page for its shared tail", seq);
  }
  const int n_drop = (int)s.pages.size() - keep;
  for (int k = keep; k < (int)s.pages.size(); ++k) {
    const int p = s.pages[k];
    if (--m->page_ref[p] == 0) m->free_pages.push_back(p);
    m->pt_host[(size_t)seq * m->max_pages + k] = -1;
  }
  s.pages.resize(keep);
  if (n_drop > 0)  // pageable source: staged before the call returns
    CK(cudaMemcpyAsync(m->pt_dev + (size_t)seq * m->max_pages + keep, &m->pt_host[(size_t)seq * m->max_pages + keep],
                       n_drop * sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
  if (cow) {
    const int old = s.pages[keep - 1];
    const int fresh = m->free_pages.back();
    m->free_pages.pop_back();
    m->page_ref[fresh] = 1;
    --m->page_ref[old];
    s.pages[keep - 1] = fresh;
    m->pt_host[(size_t)seq * m->max_pages + keep - 1] = fresh;
    const int2 pair = make_int2(old, fresh);
    CK(cudaMemcpyAsync(m->pairs_dev, &pair, sizeof(int2), cudaMemcpyHostToDevice, m->stream));
    CK(launch_kv_copy(m->k_pool, m->v_pool, m->kv_layer_elems, m->L, m->page_elems, m->pairs_dev, 1, m->stream));
    CK(cudaMemcpyAsync(m->pt_dev + (size_t)seq * m->max_pages + keep - 1,
                       &m->pt_host[(size_t)seq * m->max_pages + keep - 1], sizeof(int32_t), cudaMemcpyHostToDevice,
                       m->stream));
    TRY(sync_stream(m, m->stream));  // `pair` lives on this stack frame
  }
  s.len = len;
  return DLS_OK;
}

int dls_seq_truncate(dls_model* m, int32_t seq, int32_t len) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  return truncate_seq(m, seq, len);
}

int dls_verify(dls_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out, int32_t* argmax_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  if (n < 1 || n > DLS_MAX_VERIFY || !tokens) return fail(m, DLS_ERR_ARG, "n=%d (1..%d) tokens=%p", n, DLS_MAX_VERIFY,
                                                          (const void*)tokens);
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(m, DLS_ERR_ARG, "token[%d]=%d vocab=%d", i, tokens[i], m->V);
  Seq& s = m->seqs[seq];
  if ((long long)s.len + n > m->max_ctx)
    return fail(m, DLS_ERR_CAPACITY, "seq=%d length=%d n=%d max_ctx=%d", seq, s.len, n, m->max_ctx);
  TRY(ensure_pages(m, seq, s.len + n));
  const int32_t pos0 = s.len;
  TRY(set_params(m, 1, &seq, &tokens[0], &pos0, true));
  TRY(enqueue_prefill(m, seq, tokens, n, pos0, HEAD_ALL, nullptr));
  TRY(copy_out(m, logits_out, m->logits, (size_t)n * m->V * sizeof(float)));
  if (argmax_out) CK(cudaMemcpyAsync(argmax_out, m->next_tok, n * sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
  TRY(sync_stream(m, m->stream));
  TRY(check_status(m));
  s.len += n;
  return DLS_OK;
}

// Self-speculative greedy decoding: per round, r draft steps (decode steps
// with the draft's layers skipped, tokens fed back on the device), the
// sequence cut back, one pass of the current token and the r drafts through
// every layer (a batched step over the one sequence for up to kMaxBatch
// positions, else a prefill chunk keeping every row's logits), and the
// longest agreeing prefix kept.  One host round trip per round (the drafts
// and the full model's picks).
int dls_generate_speculative(dls_model* m, int32_t seq, int32_t token, int32_t n_tokens, const uint8_t* draft_skip,
                             int32_t draft_k, int32_t* tokens_out, int32_t* stats) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  if (token < 0 || token >= m->V) return fail(m, DLS_ERR_ARG, "token=%d vocab=%d", token, m->V);
  if (n_tokens < 1 || !tokens_out || !draft_skip || draft_k < 0 || draft_k >= DLS_MAX_VERIFY)
    return fail(m, DLS_ERR_ARG, "n_tokens=%d draft_k=%d (0..%d) draft_skip=%p", n_tokens, draft_k, DLS_MAX_VERIFY - 1,
                (const void*)draft_skip);
  Seq& s = m->seqs[seq];
  const int P0 = s.len;
  if ((long long)P0 + n_tokens > m->max_ctx)
    return fail(m, DLS_ERR_CAPACITY, "seq=%d length=%d n_tokens=%d max_ctx=%d", seq, P0, n_tokens, m->max_ctx);
  const int need = std::max(0, pages_needed(m, P0 + n_tokens) - (int)s.pages.size());
  if (need > (int)m->free_pages.size()) return fail(m, DLS_ERR_CAPACITY, "need_pages=%d free=%zu", need, m->free_pages.size());
  bool same = true;
  for (int l = 0; l < m->L; ++l) same &= (m->draft_host[l] != 0) == (draft_skip[l] != 0);
  if (!same) {
    for (int l = 0; l < m->L; ++l) m->draft_host[l] = draft_skip[l] ? 1 : 0;
    CK(cudaMemcpyAsync(m->draft_dev, m->draft_host.data(), m->L, cudaMemcpyHostToDevice, m->stream));
    TRY(sync_stream(m, m->stream));  // pageable source
    drop_graphs(m);                   // captured draft steps hold the old mask
  }
  if (m->tokens_cap < (size_t)DLS_MAX_VERIFY) {
    int32_t* t = nullptr;
    TRY(dev_alloc_t(m, (size_t)1024, &t, "generated_tokens"));
    dev_free(m, m->tokens_dev);
    m->tokens_dev = t;
    m->tokens_cap = 1024;
    drop_graphs(m);  // graphs bake the output pointer in
  }
  int rounds = 0, drafted = 0, accepted = 0, done = 0, cur = token;
  int32_t host[2 * DLS_MAX_VERIFY];
  while (done < n_tokens) {
    const int P = s.len;
    const int r = std::min(draft_k, n_tokens - done - 1);
    TRY(ensure_pages(m, seq, P + r + 1));
    TRY(set_params(m, 1, &seq, &cur, &P, true));
    if (r > 0) {
      m->drafting = true;
      int rc = DLS_OK;
      for (int t = 0; t < r && rc == DLS_OK; ++t) rc = run_step(m, 1, false, true);
      m->drafting = false;
      TRY(rc);
    }
    if (r > 0 && r + 1 <= kMaxBatch) {
      // rows t = 0..r at positions P + t of this one sequence through the
      // batched step (each row attends to the positions up to its own)
      int32_t vs[kMaxBatch], vt[kMaxBatch], vp[kMaxBatch];
      for (int t = 0; t <= r; ++t) {
        vs[t] = seq;
        vt[t] = cur;
        vp[t] = P + t;
      }
      TRY(set_params(m, r + 1, vs, vt, vp, false));
      CK(cudaMemcpyAsync(m->sp->token + 1, m->tokens_dev, r * sizeof(int32_t), cudaMemcpyDeviceToDevice, m->stream));
      m->verifying = true;
      const int rc = enqueue_batch(m, r + 1, true, true, nullptr);
      m->verifying = false;
      TRY(rc);
    } else {
      // the prefill chunk reads [cur, d_1 .. d_r]: cur from the host, the drafts where the steps left them
      if (r > 0)
        CK(cudaMemcpyAsync(m->pf_tok + 1, m->tokens_dev, r * sizeof(int32_t), cudaMemcpyDeviceToDevice, m->stream));
      CK(cudaMemcpyAsync(m->pf_tok, &cur, sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
      TRY(enqueue_prefill(m, seq, nullptr, r + 1, P, HEAD_ALL, nullptr));
    }
    // read back after the whole round is enqueued (pageable destinations block the host)
    if (r > 0)
      CK(cudaMemcpyAsync(host + DLS_MAX_VERIFY, m->tokens_dev, r * sizeof(int32_t), cudaMemcpyDeviceToHost,
                         m->stream));
    CK(cudaMemcpyAsync(host, m->next_tok, (r + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
    TRY(sync_stream(m, m->stream));
    TRY(check_status(m));
    int n = 0;
    while (n < r && host[DLS_MAX_VERIFY + n] == host[n]) ++n;
    for (int i = 0; i < n; ++i) tokens_out[done + i] = host[DLS_MAX_VERIFY + i];
    tokens_out[done + n] = host[n];
    done += n + 1;
    cur = host[n];
    s.len = P + r + 1;  // the verify pass filled positions P .. P+r
    TRY(truncate_seq(m, seq, P + n + 1));
    ++rounds;
    drafted += r;
    accepted += n;
  }
  if (stats) {
    stats[0] = rounds;
    stats[1] = drafted;
    stats[2] = accepted;
  }
  return DLS_OK;
}

int dls_argmax(dls_model* m, const float* logits, int32_t n_rows, int32_t* out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!logits || !out || n_rows < 1 || n_rows > 4096) return fail(m, DLS_ERR_ARG, "n_rows=%d", n_rows);
  CK(launch_argmax(logits, m->V, n_rows, m->argmax_buf, m->argmax_part, m->argmax_cnt,
                   argmax_blocks(n_rows, m->num_sms), m->stream, false));
  TRY(copy_out(m, out, m->argmax_buf, (size_t)n_rows * sizeof(int32_t)));
  return DLS_OK;
}

int dls_kv_fork(dls_model* m, int32_t src, const int32_t* dsts, int32_t n_dst) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, src));
  if (n_dst < 1 || !dsts) return fail(m, DLS_ERR_ARG, "n_dst=%d", n_dst);
  for (int i = 0; i < n_dst; ++i) {
    TRY(check_seq(m, dsts[i]));
    if (dsts[i] == src) return fail(m, DLS_ERR_ARG, "dst=%d equals src", dsts[i]);
    for (int j = 0; j < i; ++j)
      if (dsts[j] == dsts[i]) return fail(m, DLS_ERR_ARG, "dst=%d repeated", dsts[i]);
  }
  const int len = m->seqs[src].len;
  const int np = pages_needed(m, len);
  // capacity: the destinations' pages that only they hold come back first
  const size_t avail = m->free_pages.size() + reclaimable_pages(m, dsts, n_dst);
  if ((size_t)np * n_dst > avail)
    return fail(m, DLS_ERR_CAPACITY, "src=%d length=%d pages_per_branch=%d branches=%d free_pages=%zu", src, len, np,
                n_dst, avail);
  if ((size_t)np * n_dst > m->pairs_cap)
    return fail(m, DLS_ERR_CAPACITY, "copy list %zu > %zu", (size_t)np * n_dst, m->pairs_cap);
  std::vector<int2> pairs;
  for (int i = 0; i < n_dst; ++i) {
    TRY(release_pages(m, dsts[i]));
    TRY(ensure_pages(m, dsts[i], len));
    for (int k = 0; k < np; ++k) pairs.push_back(make_int2(m->seqs[src].pages[k], m->seqs[dsts[i]].pages[k]));
  }
  if (!pairs.empty()) {
    CK(cudaMemcpyAsync(m->pairs_dev, pairs.data(), pairs.size() * sizeof(int2), cudaMemcpyHostToDevice, m->stream));
    CK(launch_kv_copy(m->k_pool, m->v_pool, m->kv_layer_elems, m->L, m->page_elems, m->pairs_dev, (int)pairs.size(),
                      m->stream));
    TRY(sync_stream(m, m->stream));  // pairs is a pageable host vector
  }
  for (int i = 0; i < n_dst; ++i) m->seqs[dsts[i]].len = len;
  return DLS_OK;
}

int dls_kv_fork_shared(dls_model* m, int32_t src, const int32_t* dsts, int32_t n_dst) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, src));
  if (n_dst < 1 || !dsts) return fail(m, DLS_ERR_ARG, "n_dst=%d", n_dst);
  for (int i = 0; i < n_dst; ++i) {
    TRY(check_seq(m, dsts[i]));
    if (dsts[i] == src) return fail(m, DLS_ERR_ARG, "dst=%d equals src", dsts[i]);
    for (int j = 0; j < i; ++j)
      if (dsts[j] == dsts[i]) return fail(m, DLS_ERR_ARG, "dst=%d repeated", dsts[i]);
  }
  const int len = m->seqs[src].len;
  const int n_full = len / m->pt;        // pages no position at or after len falls in: shared as they are
  const int tail = len % m->pt ? 1 : 0;  // the page the next position falls in: each branch gets its own copy
  const size_t avail = m->free_pages.size() + reclaimable_pages(m, dsts, n_dst);
  if ((size_t)tail * n_dst > avail)
    return fail(m, DLS_ERR_CAPACITY, "src=%d length=%d branches=%d free_pages=%zu", src, len, n_dst, avail);
  std::vector<int2> pairs;
  for (int i = 0; i < n_dst; ++i) {
    const int d = dsts[i];
    TRY(release_pages(m, d));
    Seq& sd = m->seqs[d];
    const Seq& ss = m->seqs[src];
    for (int k = 0; k < n_full; ++k) {
      const int p = ss.pages[k];
      ++m->page_ref[p];
      sd.pages.push_back(p);
      m->pt_host[(size_t)d * m->max_pages + k] = p;
    }
    if (n_full) {
      // pageable source: staged before the call returns
      CK(cudaMemcpyAsync(m->pt_dev + (size_t)d * m->max_pages, &m->pt_host[(size_t)d * m->max_pages],
                         n_full * sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
    }
    if (tail) {
      TRY(ensure_pages(m, d, len));  // one fresh page after the shared ones
      pairs.push_back(make_int2(ss.pages[n_full], sd.pages[n_full]));
    }
  }
  if (!pairs.empty()) {
    CK(cudaMemcpyAsync(m->pairs_dev, pairs.data(), pairs.size() * sizeof(int2), cudaMemcpyHostToDevice, m->stream));
    CK(launch_kv_copy(m->k_pool, m->v_pool, m->kv_layer_elems, m->L, m->page_elems, m->pairs_dev, (int)pairs.size(),
                      m->stream));
    TRY(sync_stream(m, m->stream));  // pairs is a pageable host vector
  }
  for (int i = 0; i < n_dst; ++i) m->seqs[dsts[i]].len = len;
  return DLS_OK;
}

int dls_set_layer_skip(dls_model* m, const uint8_t* skip, int32_t n_layers) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (skip && n_layers != m->L) return fail(m, DLS_ERR_ARG, "n_layers=%d model has %d", n_layers, m->L);
  for (int l = 0; l < m->L; ++l) m->skip_host[l] = skip && skip[l] ? 1 : 0;
  CK(cudaMemcpyAsync(m->skip_dev, m->skip_host.data(), m->L, cudaMemcpyHostToDevice, m->stream));
  TRY(sync_stream(m, m->stream));  // pageable source
  drop_graphs(m);                   // captured separate-kernel steps hold the old mask
  return DLS_OK;
}

int dls_layer_cosines(dls_model* m, int32_t seq, int32_t token, int32_t pos, float* cos_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!cos_out) return fail(m, DLS_ERR_ARG, "cos_out=NULL");
  // one decode step with the residual after every layer captured, the
  // embedding row beside it, then cos(input, output) per layer on the device
  float* buf = nullptr;
  TRY(dev_alloc_t(m, (size_t)(m->L + 1) * m->H + m->L, &buf, "layer_cosines"));
  float* emb = buf;
  float* cap = buf + m->H;
  float* cosd = buf + (size_t)(m->L + 1) * m->H;
  int r = (seq < 0 || seq >= m->max_seqs || !m->seqs[seq].live || token < 0 || token >= m->V)
              ? fail(m, DLS_ERR_ARG, "seq=%d token=%d", seq, token)
              : set_params(m, 1, &seq, &token, &pos, false);
  if (r == DLS_OK) {
    cudaError_t e = launch_embed(mat_at(m->emb_block, m->emb_off), m->wtype, m->sp, 0, emb, m->V, m->stream, false);
    if (e != cudaSuccess) r = fail(m, DLS_ERR_CUDA, "embed cuda=%s", cudaGetErrorString(e));
  }
  if (r == DLS_OK) {
    m->capture = cap;
    r = dls_decode_step(m, seq, token, pos, nullptr);
    m->capture = nullptr;
  }
  if (r == DLS_OK) {
    cudaError_t e = launch_layer_cosines(emb, cap, m->L, m->H, cosd, m->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(cos_out, cosd, m->L * sizeof(float), cudaMemcpyDeviceToHost, m->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
    if (e != cudaSuccess) r = fail(m, DLS_ERR_CUDA, "layer_cosines cuda=%s", cudaGetErrorString(e));
  }
  const int rs = sync_stream(m, m->stream);
  dev_free(m, buf);
  return r != DLS_OK ? r : rs;
}

int32_t dls_kv_free_pages(const dls_model* m) {
  if (!m) return DLS_ERR_ARG;
  return (int32_t)m->free_pages.size();
}

int dls_set_resident_layers(dls_model* m, int32_t n) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (n < -1 || n > m->L) return fail(m, DLS_ERR_ARG, "n=%d n_layers=%d", n, m->L);
  const uint64_t lb = a256(m->lay.bytes);
  uint64_t cur_layers = 0;
  for (auto* p : m->layer_dev)
    if (p) cur_layers += lb;
  const uint64_t cur_stage = m->stage[0] ? staging_bytes(m) : 0;
  const uint64_t other = m->used - cur_layers - cur_stage;
  if (n == -1) {
    n = auto_resident(m, other);
    if (n < 0) return fail(m, DLS_ERR_BUDGET, "no layout fits budget=%llu", (unsigned long long)m->budget);
  }
  const uint64_t want = other + (uint64_t)n * lb + (n < m->L ? staging_bytes(m) : 0);
  if (m->budget && want > m->budget)
    return fail(m, DLS_ERR_BUDGET, "resident=%d needs=%llu budget=%llu", n, (unsigned long long)want,
                (unsigned long long)m->budget);
  if (n == m->resident) return DLS_OK;
  return apply_resident(m, n);
}

int dls_debug_profile_step(dls_model* m, int32_t seq, int32_t token, int32_t pos, int32_t max_kernels,
                           float* kernel_ms, int32_t* kernel_kind, int32_t* n_kernels) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!kernel_ms || !kernel_kind || !n_kernels || max_kernels < 1) return fail(m, DLS_ERR_ARG, "output arrays");
  TRY(check_seq(m, seq));
  if (token < 0 || token >= m->V) return fail(m, DLS_ERR_ARG, "token=%d vocab=%d", token, m->V);
  Seq& s = m->seqs[seq];
  if (pos != s.len) return fail(m, DLS_ERR_STATE, "seq=%d pos=%d length=%d", seq, pos, s.len);
  if (pos >= m->max_ctx) return fail(m, DLS_ERR_CAPACITY, "seq=%d pos=%d max_ctx=%d", seq, pos, m->max_ctx);
  TRY(ensure_pages(m, seq, pos + 1));
  TRY(set_params(m, 1, &seq, &token, &pos, true));
  // hold the GPU for a few ms so the whole step is queued before it starts:
  // the event deltas then measure kernels, not host launch gaps
  CK(launch_delay(2000000, m->stream));
  m->prof_kinds.clear();
  m->profiling = true;
  TRY(prof_mark(m, 0));
  const int r = enqueue_step(m, 1, true, false, nullptr);
  m->profiling = false;
  TRY(r);
  TRY(sync_stream(m, m->stream));
  if (m->use_step) {
    // one persistent launch: per-phase durations from its timestamps
    int active = 0;  // layers the step computed
    for (int l = 0; l < m->L; ++l) active += m->skip_host[l] ? 0 : 1;
    const int nph = 5 * active + 2;  // embed, 5 per computed layer, head
    std::vector<unsigned long long> ts(nph + 1);
    CK(cudaMemcpy(ts.data(), m->step_trace, ts.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
    const int kinds[5] = {K_QKV, K_ATTN, K_O, K_GATE_UP, K_DOWN};
    if (nph > max_kernels) return fail(m, DLS_ERR_ARG, "max_kernels=%d < %d phases", max_kernels, nph);
    for (int i = 0; i < nph; ++i) {
      kernel_ms[i] = (float)((ts[i + 1] - ts[i]) * 1e-6);
      kernel_kind[i] = i == 0 ? K_EMBED : (i == nph - 1 ? K_HEAD : kinds[(i - 1) % 5]);
    }
    *n_kernels = nph;
    s.len += 1;
    return DLS_OK;
  }
  const int n = (int)m->prof_kinds.size() - 1;
  if (n > max_kernels) return fail(m, DLS_ERR_ARG, "max_kernels=%d < %d launches", max_kernels, n);
  for (int i = 0; i < n; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, m->prof_events[i], m->prof_events[i + 1]));
    kernel_ms[i] = ms;
    kernel_kind[i] = m->prof_kinds[i + 1];
  }
  *n_kernels = n;
  s.len += 1;
  return DLS_OK;
}

int dls_debug_profile_batch(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, const int32_t* pos,
                            int32_t max_kernels, float* kernel_ms, int32_t* kernel_kind, int32_t* n_kernels) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!kernel_ms || !kernel_kind || !n_kernels || max_kernels < 1) return fail(m, DLS_ERR_ARG, "output arrays");
  if (n < 2 || n > m->max_batch || !seqs || !tokens || !pos)
    return fail(m, DLS_ERR_ARG, "n=%d max_batch=%d (batches of 2 or more rows)", n, m->max_batch);
  for (int i = 0; i < n; ++i) {
    TRY(check_seq(m, seqs[i]));
    for (int j = 0; j < i; ++j)
      if (seqs[j] == seqs[i]) return fail(m, DLS_ERR_ARG, "seq=%d repeated", seqs[i]);
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(m, DLS_ERR_ARG, "token[%d]=%d", i, tokens[i]);
    if (pos[i] != m->seqs[seqs[i]].len)
      return fail(m, DLS_ERR_STATE, "seq=%d pos=%d length=%d", seqs[i], pos[i], m->seqs[seqs[i]].len);
    if (pos[i] >= m->max_ctx) return fail(m, DLS_ERR_CAPACITY, "seq=%d pos=%d", seqs[i], pos[i]);
  }
  int need = 0;
  for (int i = 0; i < n; ++i)
    need += std::max(0, pages_needed(m, pos[i] + 1) - (int)m->seqs[seqs[i]].pages.size());
  if (need > (int)m->free_pages.size()) return fail(m, DLS_ERR_CAPACITY, "need_pages=%d free=%zu", need, m->free_pages.size());
  for (int i = 0; i < n; ++i) TRY(ensure_pages(m, seqs[i], pos[i] + 1));
  TRY(set_params(m, n, seqs, tokens, pos, true));
  // hold the GPU so the whole step is queued before it starts
  CK(launch_delay(2000000, m->stream));
  m->prof_kinds.clear();
  m->profiling = true;
  TRY(prof_mark(m, 0));
  const int r = enqueue_step(m, n, true, false, nullptr);
  m->profiling = false;
  TRY(r);
  TRY(sync_stream(m, m->stream));
  const int nk = (int)m->prof_kinds.size() - 1;
  if (nk > max_kernels) return fail(m, DLS_ERR_ARG, "max_kernels=%d < %d launches", max_kernels, nk);
  for (int i = 0; i < nk; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, m->prof_events[i], m->prof_events[i + 1]));
    kernel_ms[i] = ms;
    kernel_kind[i] = m->prof_kinds[i + 1];
  }
  *n_kernels = nk;
  for (int i = 0; i < n; ++i) m->seqs[seqs[i]].len += 1;
  return DLS_OK;
}

int32_t dls_step_kernel_in_use(const dls_model* m, const char** why) {
  if (why) *why = nullptr;
  if (!m) return 0;
  if (m->use_step) return 1;
  if (why) {
    const char* e = getenv("DLS_STEP_KERNEL");
    if (e && atoi(e) == 0) *why = "disabled";
    else if (m->mixed) *why = "mixed weight formats";
    else if (m->resident < m->L) *why = "not all layers resident";
    else if (!m->step.fn) *why = m->step.why ? m->step.why : "not planned";
    else *why = "not set up";
  }
  return 0;
}

int dls_debug_step_trace(dls_model* m, uint64_t* out, int32_t max_entries, int32_t* n_entries) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!out || !n_entries || max_entries < 0) return fail(m, DLS_ERR_ARG, "output arrays");
  if (!m->use_step || !m->step_ctrace) return fail(m, DLS_ERR_STATE, "no persistent step kernel in use");
  const size_t n = (size_t)(5 * m->L + 8) * m->step.grid * 8;
  if ((size_t)max_entries < n) return fail(m, DLS_ERR_ARG, "max_entries=%d < %zu", max_entries, n);
  TRY(sync_stream(m, m->stream));
  CK(cudaMemcpy(out, m->step_ctrace, n * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  *n_entries = (int32_t)n;
  return DLS_OK;
}

int dls_debug_capture(dls_model* m, float* per_layer_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  m->capture = per_layer_out;
  return DLS_OK;
}

int dls_debug_bounded_wait(dls_model* m, int64_t limit_ns) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (limit_ns < 1000 || limit_ns > 10000000000LL)
    return fail(m, DLS_ERR_ARG, "limit_ns=%lld (1e3..1e10)", (long long)limit_ns);
  CK(launch_unarrived_wait((unsigned long long)limit_ns, &m->sp->status, m->stream));
  TRY(sync_stream(m, m->stream));
  return check_status(m);
}

int dls_debug_read_kv(dls_model* m, int32_t seq, int32_t layer, void* k_out, void* v_out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  TRY(check_seq(m, seq));
  if (layer < 0 || layer >= m->L || !k_out || !v_out) return fail(m, DLS_ERR_ARG, "layer=%d", layer);
  const Seq& s = m->seqs[seq];
  if (s.len == 0) return DLS_OK;
  const __half* kp = m->k_pool + (size_t)layer * m->kv_layer_elems;
  const __half* vp = m->v_pool + (size_t)layer * m->kv_layer_elems;
  const int32_t* pages = m->pt_dev + (size_t)seq * m->max_pages;
  CK(launch_kv_gather(kp, pages, s.len, m->nkv, m->pt, m->hd, static_cast<__half*>(k_out), m->stream));
  CK(launch_kv_gather(vp, pages, s.len, m->nkv, m->pt, m->hd, static_cast<__half*>(v_out), m->stream));
  return DLS_OK;
}

static int find_matrix(dls_model* m, int32_t layer, int32_t tensor, MatDev* out) {
  if (tensor == 7) {
    *out = mat_at(m->emb_block, m->emb_off);
    return DLS_OK;
  }
  if (tensor == 8) {
    *out = head_mat(m);
    return DLS_OK;
  }
  if (tensor < 0 || tensor > 8 || layer < 0 || layer >= m->L) return fail(m, DLS_ERR_ARG, "layer=%d tensor=%d", layer, tensor);
  const uint8_t* base = m->layer_dev[layer];
  if (!base) return fail(m, DLS_ERR_STATE, "layer=%d is not resident", layer);
  switch (tensor) {
    case 0: *out = mat_at(base, m->lay.qkv, 0, m->q_rows); break;
    case 1: *out = mat_at(base, m->lay.qkv, m->q_rows, m->kv_rows); break;
    case 2: *out = mat_at(base, m->lay.qkv, m->q_rows + m->kv_rows, m->kv_rows); break;
    case 3: *out = mat_at(base, m->lay.o); break;
    case 4:  // gate rows are the even rows of the interleaved gate|up matrix
    case 5:  // up rows are the odd rows
      *out = mat_at(base, m->lay.gu, tensor - 4, m->F);
      out->rstep = 2;
      break;
    case 6: *out = mat_at(base, m->lay.down); break;
  }
  return DLS_OK;
}

// A mixed-format model's matrix `tensor` (ids of dls_debug_dequant): its
// type, K-quant data, Q8_0 / Q4_0 view, and shape.
int find_matrix_mixed(dls_model* m, int32_t layer, int32_t tensor, int* type, const uint8_t** w, MatDev* md,
                      int* rows, int* cols) {
  *rows = m->V;
  *cols = m->H;
  if (tensor == 7 || (tensor == 8 && m->tied)) {
    *type = m->emb_type;
    *w = m->emb_block;
    *md = mat_at(m->emb_block, m->emb_off);
    return DLS_OK;
  }
  if (tensor == 8) {
    *type = m->out_type;
    *w = m->out_block;
    *md = mat_at(m->out_block, m->out_off);
    return DLS_OK;
  }
  if (tensor < 0 || tensor > 8 || layer < 0 || layer >= m->L) return fail(m, DLS_ERR_ARG, "layer=%d tensor=%d", layer, tensor);
  const uint8_t* base = m->layer_dev[layer];
  if (!base) return fail(m, DLS_ERR_STATE, "layer=%d is not resident", layer);
  mix_shape(m, tensor, rows, cols);
  *type = m->mtype[tensor];
  *w = base + m->mkq[tensor];
  *md = m->mtype[tensor] ? MatDev{} : mat_at(base, m->mleg[tensor]);
  return DLS_OK;
}

int dls_debug_dequant(dls_model* m, int32_t layer, int32_t tensor, float* out) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!out) return fail(m, DLS_ERR_ARG, "out=NULL");
  if (m->mixed) {
    int type, rows, cols;
    const uint8_t* w;
    MatDev md;
    TRY(find_matrix_mixed(m, layer, tensor, &type, &w, &md, &rows, &cols));
    if (type) CK(launch_kq_dequant_rows(type, w, rows, cols, 0, nullptr, rows, out, cols, nullptr, m->stream));
    else CK(launch_dequant(md, m->wtype, out, m->stream));
    return DLS_OK;
  }
  MatDev md;
  TRY(find_matrix(m, layer, tensor, &md));
  CK(launch_dequant(md, m->wtype, out, m->stream));
  return DLS_OK;
}

int dls_debug_gemv(dls_model* m, int32_t layer, int32_t tensor, const float* x, float* y) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!x || !y) return fail(m, DLS_ERR_ARG, "x/y NULL");
  if (m->mixed) {
    int type, rows, cols;
    const uint8_t* w;
    MatDev md;
    TRY(find_matrix_mixed(m, layer, tensor, &type, &w, &md, &rows, &cols));
    return mix_gemv(m, type, w, md, rows, cols, x, y, K_HEAD);
  }
  MatDev md;
  TRY(find_matrix(m, layer, tensor, &md));
  GemvArgs g{};
  g.unit = 1;
  g.x = x;
  if (md.rstep == 2) {
    // gate or up: run the whole interleaved matrix, then pick every other row
    g.w = mat_at(m->layer_dev[layer], m->lay.gu);
    g.y = m->gu;
    const GemvLaunch l = gemv_plan(m->wtype, PRO_COPY, EPI_STORE, g.w.rows, g.w.nb, m->num_sms, 1);
    CK(launch_gemv(m->wtype, PRO_COPY, EPI_STORE, g, l, m->stream, false));
    CK(cudaMemcpy2DAsync(y, sizeof(float), m->gu + (tensor - 4), 2 * sizeof(float), sizeof(float), m->F,
                         cudaMemcpyDeviceToDevice, m->stream));
    return DLS_OK;
  }
  g.w = md;
  g.y = y;
  const GemvLaunch l = gemv_plan(m->wtype, PRO_COPY, EPI_STORE, md.rows, md.nb, m->num_sms, 1);
  CK(launch_gemv(m->wtype, PRO_COPY, EPI_STORE, g, l, m->stream, false));
  return DLS_OK;
}

int dls_debug_gemm(dls_model* m, int32_t layer, int32_t tensor, int32_t n_tokens, const float* x, float* y) {
  if (!m) return fail(m, DLS_ERR_ARG, "model=NULL");
  if (!x || !y || n_tokens < 1) return fail(m, DLS_ERR_ARG, "x/y NULL or n_tokens=%d", n_tokens);
  if (m->mixed) return fail(m, DLS_ERR_STATE, "a mixed-format model has no tensor-core GEMM");
  MatDev md;
  TRY(find_matrix(m, layer, tensor, &md));
  const bool pair = md.rstep == 2;  // gate or up: run the interleaved matrix, keep every other column
  const MatDev w = pair ? mat_at(m->layer_dev[layer], m->lay.gu) : md;
  const int kx = w.nb * 32;
  void *xh = nullptr, *yt = nullptr;
  TRY(dev_alloc(m, 2 * (size_t)n_tokens * kx * sizeof(__half), &xh, "debug_gemm_x"));
  int r = pair ? dev_alloc(m, (size_t)n_tokens * w.rows * sizeof(float), &yt, "debug_gemm_y") : DLS_OK;
  if (r == DLS_OK) {
    __half* xhi = static_cast<__half*>(xh);
    __half* xlo = xhi + (size_t)n_tokens * kx;
    cudaError_t e = launch_to_f16_rows(x, n_tokens, w.cols, w.cols, xhi, xlo, kx, m->stream);
    PgArgs g{};
    g.w = w;
    g.x = xhi;
    g.xlo = xlo;
    g.kx = kx;
    g.T = n_tokens;
    g.y = pair ? static_cast<float*>(yt) : y;
    g.ldy = w.rows;
    g.status = &m->sp->status;
    const TgPlan p = tgemm_plan(w.rows, kx, n_tokens, m->num_sms, kTgMaxSplit, m->pf_bn);
    if (p.split > 1) {
      if ((size_t)p.split * n_tokens * w.rows > m->tg_part_elems) e = cudaErrorInvalidValue;
      g.part = m->tg_part;
      g.counters = m->tg_cnt;
    }
    if (e == cudaSuccess) e = launch_tgemm(m->wtype, EPI_STORE, g, p, m->stream);
    if (e == cudaSuccess && pair)
      e = cudaMemcpy2DAsync(y, sizeof(float), static_cast<float*>(yt) + (tensor - 4), 2 * sizeof(float), sizeof(float),
                            (size_t)n_tokens * m->F, cudaMemcpyDeviceToDevice, m->stream);
    if (e != cudaSuccess) r = fail(m, DLS_ERR_CUDA, "debug_gemm cuda=%s", cudaGetErrorString(e));
    if (r == DLS_OK) r = sync_stream(m, m->stream);
  }
  const int rs = sync_stream(m, m->stream);
  dev_free(m, xh);
  dev_free(m, yt);
  TRY(r);
  TRY(rs);
  return check_status(m);
}

}  // extern "C"
