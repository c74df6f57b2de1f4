// Host-side launchers of the library's kernels (one declaration per kernel
// family); the runtime in api.cu composes them into the decode step.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace dls {

enum Pro { PRO_COPY = 0, PRO_RMSNORM = 1 };
// EPI_SWIGLU: rows come in (gate, up) pairs; y[r/2] = silu(gate) * up
enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3 };

// Where a decode row finds its KV pages (model path: row b is sequence
// sp->seq[b] at position sp->pos[b]).
struct KvView {
  __half* k_pool;            // layer base, [n_pages][n_kv][page_tokens][head_dim]
  __half* v_pool;
  const int32_t* page_table; // [max_seqs][max_pages]
  int n_kv, head_dim, page_tokens, max_pages;
};

struct GemvArgs {
  MatDev w;
  int unit;                  // rows are split across CTAs in multiples of this
  const float* x;            // activation [cols]
  const float* g;            // RMSNorm gain [cols]
  float eps;
  float* y;                  // STORE: y[r] = acc; RESID: y[r] += acc; QKV: q rows -> y; SWIGLU: y[r/2]
  // EPI_QKV
  int q_rows, kv_rows;
  KvView kv;
  const float2* rope_cs;     // [rope_len][head_dim/2] cos, sin
  int rope_len;
  StepParams* sp;
  int brow;                  // batch row of sp this launch serves
};

struct GemvLaunch {
  int grid, threads, smem;
  int nwc;  // consumer warps (plus one producer warp)
  int rs;   // rows per ring stage
  int ns;   // ring stages
  int mc;   // K-chunks per consumer warp
};

// Choose grid/threads/smem for a matrix and check the kernel can run it.
GemvLaunch gemv_plan(int wtype, int pro, int epi, int rows, int nb, int num_sms, int unit);
cudaError_t gemv_setup_attributes();   // raise dynamic smem limits once
cudaError_t launch_gemv(int wtype, int pro, int epi, const GemvArgs& a, const GemvLaunch& l, cudaStream_t s,
                        bool pdl);

// ---- attention ------------------------------------------------------------------

struct AttnArgs {
  const float* q;            // [rows of this launch][n_heads*head_dim]
  float* o;                  // [rows of this launch][n_heads*head_dim]
  const __half* k_pool;
  const __half* v_pool;
  const int32_t* page_table; // rows of max_pages entries
  int max_pages;
  const int32_t* pt_row;     // page-table row per batch row (NULL: row b)
  const int32_t* len;        // per batch row: keys attended = len[b] + len_add
  int len_add;
  int n_heads, n_kv, head_dim, page_tokens;
  int n_splits;
  int row0;                  // first batch row of this launch
  float* part_o;             // scratch
  float* part_ml;
  int* counters;             // [rows][n_kv], zero between launches
  int32_t* status;           // optional status word (may be NULL)
  int max_len;               // upper bound on keys (guards page-table reads)
  // cascade (shared-prefix) attention: keys [0, *start_len) were covered by
  // launch_cascade_prefix, whose P = pre_splits partials per (row, kv head)
  // join this launch's merge (start_len NULL / pre_splits 0: no prefix part)
  const int32_t* start_len;  // device, a multiple of 32
  const float* pre_o;        // [rows][n_kv][P][G][head_dim]
  const float* pre_ml;       // [rows][n_kv][P][G] (m, l) pairs
  int pre_splits;
};

// The shared-prefix half of cascade attention: the keys [0, *shared_len) that
// every batch row holds in the same KV pages (a shared fork), read once per
// KV head for all rows.  CTA (kv head, split) streams its run of 32-token
// tiles through shared memory; warp r applies each tile to batch row r's G
// query heads.  Writes one (m, l, o) partial per (row, kv head, split).
struct CascArgs {
  const float* q;             // [rows][n_heads*head_dim]
  const __half* k_pool;
  const __half* v_pool;
  const int32_t* page_table;
  int max_pages;
  const int32_t* pt_row;      // page-table row of batch row 0 (the prefix pages are every row's)
  const int32_t* shared_len;  // device: shared prefix length, a multiple of 32 (0: nothing to do)
  int rows;                   // 1..8
  int n_heads, n_kv, head_dim, page_tokens;
  int n_splits;               // splits per KV head
  float* part_o;              // [rows][n_kv][n_splits][G][head_dim]
  float* part_ml;             // [rows][n_kv][n_splits][G]
  int32_t* status;
  int max_len;
  int pool_rows;              // rows of head_dim in one layer's K (or V) pool (the tensor-core kernel's maps)
};
cudaError_t launch_cascade_prefix(const CascArgs& a, cudaStream_t s);
bool cascade_supported(int n_heads, int n_kv, int head_dim);
// The same pass on the tensor cores (casc_tc.cu): head_dim 64 or 128, any
// group size up to 8, pages a multiple or a divisor of 64 tokens.
bool cascade_tc_supported(int n_heads, int n_kv, int head_dim, int page_tokens);
cudaError_t cascade_tc_setup_attributes();
cudaError_t launch_cascade_prefix_tc(const CascArgs& a, cudaStream_t s);

size_t attn_workspace_bytes(int rows, int n_heads, int n_kv, int head_dim, int n_splits);
void attn_workspace_carve(void* ws, int rows, int n_heads, int n_kv, int head_dim, int n_splits, float** part_o,
                          float** part_ml, int** counters);
int attn_default_splits(int rows, int n_kv, int num_sms, int max_len);
cudaError_t launch_attention(const AttnArgs& a, int rows, cudaStream_t s, bool pdl);

// ---- small kernels --------------------------------------------------------------

// cos(input, output) of every layer's residual: emb [H] (layer 0's input),
// cap [L][H] (the residual after each layer) -> out [L]
cudaError_t launch_layer_cosines(const float* emb, const float* cap, int L, int H, float* out, cudaStream_t s);
cudaError_t launch_embed(const MatDev& emb, int wtype, StepParams* sp, int brow, float* x, int vocab,
                         cudaStream_t s, bool pdl);
// greedy pick per row over [rows][vocab]; part/counters: scratch of
// argmax_scratch_entries(rows, num_sms) int2 and `rows` ints (zero between calls)
int argmax_blocks(int rows, int num_sms);
cudaError_t launch_argmax(const float* logits, int vocab, int rows, int32_t* out, int2* part, int* counters,
                          int nblk, cudaStream_t s, bool pdl);
cudaError_t launch_advance(StepParams* sp, const int32_t* next, int32_t* tokens_out, int rows, cudaStream_t s,
                           bool pdl);
cudaError_t launch_set_params(StepParams* sp, const StepParams& h, bool reset_step, cudaStream_t s);
// source row r goes to destination row r * row_step (qs, d point at the first destination row)
cudaError_t launch_repack(const uint8_t* src, int wtype, int rows, int nb, int ds, int row_step, uint8_t* qs,
                          __half* d, cudaStream_t s);
cudaError_t launch_rope_table(float2* cs, int len, int head_dim, float theta, cudaStream_t s);
cudaError_t launch_dequant(const MatDev& m, int wtype, float* out, cudaStream_t s);
// copy whole KV pages: pairs[i] = (src_page, dst_page), for every layer
cudaError_t launch_kv_copy(__half* k_pool, __half* v_pool, size_t layer_stride_elems, int n_layers,
                           size_t page_elems, const int2* pairs, int n_pairs, cudaStream_t s);
// host -> device copy by the SMs reading pinned (mapped) host memory; 16-byte aligned, bytes % 16 == 0
cudaError_t launch_h2d_sm(void* dst, const void* src, size_t bytes, int ctas, cudaStream_t s);
// a bounded mbarrier wait that is never satisfied: kTimeout into *status after limit_ns
cudaError_t launch_unarrived_wait(unsigned long long limit_ns, int32_t* status, cudaStream_t s);
// spin (bounded by the global timer) for `ns` nanoseconds on the stream
cudaError_t launch_delay(long long ns, cudaStream_t s);
cudaError_t launch_kv_gather(const __half* pool, const int32_t* pages, int len, int n_kv, int page_tokens,
                             int head_dim, __half* out, cudaStream_t s);

// ---- persistent decode step ------------------------------------------------------

struct StepLayer {
  const float* attn_norm;
  const float* ffn_norm;
  MatDev qkv, o, gu, down;  // gu: interleaved (gate, up) rows
  __half* k_pool;           // this layer's KV pools
  __half* v_pool;
};

struct StepArgs {
  const StepLayer* layers;  // device array [n_layers]
  int n_layers;
  MatDev emb, head;
  const float* out_norm;
  int H, q_rows, kv_rows, n_heads, n_kv, hd, F, vocab;
  float eps;
  const int32_t* page_table;  // [max_seqs][max_pages]; the step serves row 0 of sp
  int max_pages, page_tokens, max_len;
  const float2* rope_cs;
  int rope_len;
  StepParams* sp;
  float *x, *q, *o, *h, *logits;
  float *part_o, *part_ml;  // attention partials [n_kv * S]
  int* att_counters;        // [n_kv], zero between launches
  int2* am_part;            // [grid]
  int32_t* tokens_out;      // greedy: token of step sp->step goes to tokens_out[step]
  int greedy;               // pick argmax and advance sp at the end
  int head_rows;            // 0: skip the LM head (prefill tokens before the last)
  unsigned* bar;            // grid barrier counter, zero at launch
  int* abort;               // set when a bounded wait gives up, zero at launch
  int S;                    // attention splits per KV head (one per CTA)
  unsigned long long* trace;  // optional: CTA 0 writes the global timer after each phase
  unsigned long long* ctrace; // optional: per phase and CTA {consumer arrival, release, producer first issue,
                              // producer last issue, prologue done, stages done, epilogue done, -}: [phase][grid][8]
  int ns;                   // ring stages
  uint32_t stage_bytes;     // ring slot size
  int pf_skip, pf_rows;     // gate/up rows [pf_skip, pf_skip + pf_rows) of each CTA hinted into L2 during attention/O
  const uint8_t* skip;      // [n_layers]: layers this step does not compute (their residual passes through)
  float* capture;           // optional [n_layers][H]: the residual stream after every layer
};

struct StepPlan {
  const void* fn;  // NULL: no persistent kernel for this shape
  int grid, threads, smem, ns, splits;
  uint32_t stage_bytes;
  const char* why;  // when fn is NULL: the reason
};

StepPlan step_plan(int wtype, int H, int q_rows, int F, int n_heads, int n_kv, int hd, int num_sms);
cudaError_t launch_step(const StepPlan& p, const StepArgs& a, cudaStream_t s);

// ---- prefill (T tokens at once) --------------------------------------------------

// Activations enter the tensor cores as two fp16 planes, x = x_hi + x_lo
// with x_hi = fp16(x) and x_lo = fp16(x - x_hi), and the dequantised weights
// likewise (w_hi = fp16(d*q), w_lo = fp16(d*q - w_hi)); the GEMM accumulates
// w_hi x_hi + w_hi x_lo + w_lo x_hi in fp32, which carries both operands to
// about 22 bits instead of fp16's 11.
struct PgArgs {
  MatDev w;            // weight rows = GEMM M
  const __half* x;     // activations [T][kx] fp16 (hi plane), kx >= w.nb * 32, zero beyond the true width
  const __half* xlo;   // lo plane, same layout
  int kx;              // row stride of x in elements (multiple of 8)
  int T;               // tokens = GEMM N
  float* y;            // STORE / RESID: y[t * ldy + m]
  int ldy;
  __half* h;           // SWIGLU: h[t * ldh + m / 2] = silu(gate) * up (rows interleaved gate, up), hi plane
  __half* hlo;         // SWIGLU: lo plane of h
  int ldh;
  int32_t* status;     // kTimeout on a wait that gave up
  float* part;         // split-K partial sums [split][T][rows] (split > 1)
  int* counters;       // one per output tile, zero between launches (split > 1)
};

// tile width (tokens per CTA: 16 or 128) and K splits of one GEMM
struct TgPlan {
  int bn, split;
};
TgPlan tgemm_plan(int rows, int kpad, int T, int num_sms, int max_split, int chunk_bn = 0);
cudaError_t tgemm_setup_attributes();  // smem limits; fails if tensor maps cannot be made
// the prompt-chunk GEMM with the codes as exact MMA operands and the block
// scales applied per 32 columns by the epilogue (gemm_codes.cu): 128 x 128 tiles, no split
cudaError_t cgemm_setup_attributes();
cudaError_t launch_cgemm(int wtype, int epi, const PgArgs& a, cudaStream_t s);
cudaError_t launch_tgemm(int wtype, int epi, const PgArgs& a, const TgPlan& p, cudaStream_t s);
// the small-batch form (T <= 8): raw codes as exact fp16 operands, block
// scales applied per 32-column block from tensor memory (gemm_small.cu)
cudaError_t sgemm_setup_attributes();

// ---- multi-row dequant-GEMV (2..8 activation rows; gemv_rows.cu) ---------------
struct RgArgs {
  MatDev w;
  int unit;              // rows are split across CTAs in multiples of this (2 for SwiGLU pairs)
  const float* x;        // activations [T][ldx] fp32
  int ldx;
  int T;                 // activation rows, 1..8
  const float* g;        // RMSNorm gain [cols] (PRO_RMSNORM)
  float eps;
  float* y;              // STORE: y[t*ldy + r]; RESID: +=; SWIGLU: y[t*ldy + r/2] = silu(gate) * up
  int ldy;
  int32_t* status;       // kTimeout when a bounded wait ran out
  float* part;           // split-K partials [split][T][rows] (split > 1)
  int* counters;         // one per row range (grid.x), zero between launches (split > 1)
};

struct RgLaunch {
  int grid, threads, smem;
  int nt, rs, mc, ns, split;  // rows padded to nt, weight rows per stage, chunks per lane, stages, K splits
  int stage;                  // ring stage stride in bytes
};

RgLaunch rgemv_plan(int wtype, int pro, int epi, int rows, int nb, int T, int num_sms, int unit);  // grid 0: unsupported
cudaError_t rgemv_setup_attributes();
cudaError_t launch_rgemv(int wtype, int pro, int epi, const RgArgs& a, const RgLaunch& l, cudaStream_t s);

// ---- K-quant dequant-GEMV (Q4_K, Q6_K; kquant.cu) ------------------------------
enum KqFormat { KQ_Q4_K = 12, KQ_Q5_K = 13, KQ_Q6_K = 14 };  // the GGUF type ids

struct KqArgs {
  const uint8_t* w;   // packed super-blocks (Q4_K 144, Q5_K 176, Q6_K 208 bytes each), row-major
  const __half* d6;   // Q6_K: super-block scales [rows][nsb rounded up to 8]; unused for Q4_K
  int rows, cols;     // cols a multiple of 256
  const float* x;     // [cols], 16-byte aligned
  float* y;           // [rows]
  int* status;        // kTimeout is or-ed in when a bounded wait runs out (may be NULL)
};

struct KqLaunch {
  int grid, threads, smem;
  int nwc, rs, ns, mc;  // consumer warps, rows per ring stage, stages, units per lane
  int wide;             // Q4_K / Q5_K: 64-weight units (else 32)
};

size_t kq_packed_bytes(int fmt, int rows, int cols);
const __half* kq_d6(const void* packed, int rows, int cols);
cudaError_t launch_kq_pack(int fmt, const void* blocks, int rows, int cols, void* packed, cudaStream_t s);
KqLaunch kq_plan(int fmt, int rows, int cols, int num_sms);  // grid 0: unsupported shape
// rows row0 .. row0+n-1 (idx NULL) or idx[0..n) of a packed K-quant matrix -> fp32 out [n][ldo]
cudaError_t launch_kq_dequant_rows(int fmt, const void* packed, int rows, int cols, int row0, const int32_t* idx,
                                   int n, float* out, int ldo, int32_t* status, cudaStream_t s);
// single-vector helpers of the mixed-format decode path
cudaError_t launch_rmsnorm_vec(const float* x, int H, const float* g, float eps, float* out, cudaStream_t s);
cudaError_t launch_add_vec(float* x, const float* y, int n, cudaStream_t s);
cudaError_t launch_swiglu_vec(const float* gate, const float* up, float* h, int n, cudaStream_t s);
cudaError_t kq_setup_attributes();
cudaError_t launch_kq_gemv(int fmt, const KqArgs& a, const KqLaunch& l, cudaStream_t s);
cudaError_t launch_sgemm(int wtype, int epi, const PgArgs& a, int split, cudaStream_t s);
cudaError_t prefill_setup_attributes();
cudaError_t launch_embed_rows(const MatDev& emb, int wtype, const int32_t* tokens, int T, int vocab, float* x, int ldx,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_rmsnorm_rows(const float* x, int T, int H, int ldx, const float* g, float eps, __half* out,
                                __half* out_lo, int ldo,
                                cudaStream_t s);
cudaError_t launch_to_f16_rows(const float* x, int T, int cols, int ldx, __half* out, __half* out_lo, int ldo,
                               cudaStream_t s);
cudaError_t launch_rope_kv_rows(const float* qkv, int T, int ld, int q_rows, int kv_rows, const KvView& kv, int seq,
                                int pos0, const float2* rope_cs, int rope_len, float* q_out, int32_t* status,
                                cudaStream_t s);
// the same for n batch rows, row t being sequence seqs[t] at position poss[t]
cudaError_t launch_rope_kv_batch(const float* qkv, int n, int ld, int q_rows, int kv_rows, const KvView& kv,
                                 const int32_t* seqs, const int32_t* poss, const float2* rope_cs, int rope_len,
                                 float* q_out, int32_t* status, cudaStream_t s);
// causal attention of T query tokens at positions pos0 .. pos0+T-1 over one
// sequence (ptab_row = its page-table row); q, o: [T][n_heads][head_dim]
cudaError_t launch_pattn(const float* q, float* o, const KvView& kv, const int32_t* ptab_row, int n_heads, int T,
                         int pos0, cudaStream_t s);

// 2-D tiled tensor map (row-major, dim0 contiguous; strides in bytes)
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                  uint64_t stride1, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw);

// ---- prefill attention on the tensor cores ---------------------------------------

struct FattnArgs {
  const float* q;            // [T][n_heads][head_dim] fp32 (RoPE applied)
  int n_heads, n_kv, head_dim;
  int T, pos0;               // query tokens at positions pos0 .. pos0+T-1
  const int32_t* ptab;       // the sequence's page-table row
  int max_pages, page_tokens;
  int pool_rows;             // rows of head_dim in one layer's K (or V) pool: n_pages * n_kv * page_tokens
  __half* out;               // [T][ld_out] fp16 hi plane, head h at columns h * head_dim
  __half* out_lo;            // lo plane (fp16 of the rounding residual), same layout
  int ld_out;
  int32_t* status;
};

bool fattn_supported(int head_dim, int g, int page_tokens);
cudaError_t fattn_setup_attributes();
cudaError_t launch_fattn(const FattnArgs& a, const __half* k_pool, const __half* v_pool, cudaStream_t s);

// Record a failure for dls_last_error(NULL) (calls without a model) and
// return `code`.
int report_error(int code, const char* fmt, ...);

}  // namespace dls
