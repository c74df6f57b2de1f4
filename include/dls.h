/*
 * dls.h - C ABI of the GB300 (sm_103a) decode-step library for quantised
 * Llama-architecture models.
 *
 * What it computes (one token per sequence per decode step, every step on
 * the GPU in this library's own CUDA kernels):
 *
 *   x = dequant(tok_embd[token])
 *   per layer:  xn = rmsnorm(x) * g_attn
 *               q, k, v = Wq xn, Wk xn, Wv xn            (Q8_0 / Q4_0 dequant-GEMV)
 *               q, k = rope(q, pos), rope(k, pos)         (adjacent pairs)
 *               K[pos], V[pos] = fp16(k), fp16(v)         (paged fp16 KV cache)
 *               o = softmax(q K[0..pos]^T / sqrt(hd)) V   (GQA, causal)
 *               x += Wo o
 *               x += Wdown (silu(Wgate xn') * (Wup xn')), xn' = rmsnorm(x) * g_ffn
 *   logits = Wout (rmsnorm(x) * g_out)                    (Wout = tok_embd if tied)
 *
 * Sources, by page and section: the pure C + CUDA LLM inference engine page
 * (rskf.cn), section 1 (Llama architecture with RoPE, GQA, SwiGLU, RMSNorm and
 * a KV cache; Q4_0 and Q8_0 weights; 8B Q8_0 resident decode) and section 4.4
 * (single-token GEMV, fused RMSNorm, RoPE with a precomputed sin/cos table,
 * SwiGLU fused with the projection, causal softmax with the mask inside);
 * sections 3.3 and 4.2 (two-buffer layer streaming, SLEP) and 4.1 (the
 * resident-layer count from the device budget); the "3 Agents. 3 LLMs. 1 Aging
 * GPU" page (LayerStreamer: pinned host region, two device buffers, two
 * streams, per-layer events; the admission ledger that reserves before it
 * allocates and rolls back on failure); the SwarmKV page ("Prefill once, fan
 * out"), sections 2-4 (prefill fills the KV cache once, the snapshot is copied
 * per branch, branches continue RoPE at the prefix length, the context budget
 * is checked before anything is allocated, a restore must match the snapshot
 * size exactly).
 *
 * Conventions
 *  - Every call is ordered on the model's CUDA stream.  A model handle is not
 *    thread-safe: use it from one host thread at a time.
 *  - Status codes: DLS_OK (0) or a negative dls_status.  A failed call leaves
 *    the model as it was (sequences, lengths, resident layers), except
 *    DLS_ERR_CUDA, after which the model should be destroyed.
 *  - dls_last_error() returns "ERR <CODE> key=value ..." for the last failed
 *    call on that model (or, for a NULL model, on the calling thread).
 *  - Pointers marked "host" are host memory; "device" are device memory of
 *    the model's GPU; "host or device" accepts either (detected per call).
 *  - Nothing here traps or asserts on the device: kernels that detect a bad
 *    index or a wait that runs out record it in a status word that the host
 *    reads, and the call returns DLS_ERR_STATE or DLS_ERR_TIMEOUT.
 */
#ifndef DLS_H
#define DLS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DLS_ABI_VERSION 2
#define DLS_MAX_BATCH 8
/* Most positions one dls_verify pass scores (and 1 + the longest draft). */
#define DLS_MAX_VERIFY 16

typedef struct dls_model dls_model;

typedef enum dls_status {
  DLS_OK = 0,
  DLS_ERR_ARG = -1,      /* bad argument or descriptor */
  DLS_ERR_BUDGET = -2,   /* the device budget (ledger) cannot hold the request */
  DLS_ERR_CAPACITY = -3, /* out of sequences, KV pages or context */
  DLS_ERR_CUDA = -4,     /* a CUDA call failed */
  DLS_ERR_TIMEOUT = -5,  /* a bounded wait ran out */
  DLS_ERR_STATE = -6     /* call does not fit the model's state (e.g. pos != length) */
} dls_status;

/* Weight block formats (as the workloads define them):
 *  DLS_Q8_0: 34-byte block = little-endian fp16 d, 32 x int8 q;  w = d*q
 *  DLS_Q4_0: 18-byte block = fp16 d, 16 bytes; byte j = element j (low
 *            nibble) and element j+16 (high nibble); w = d*(nibble - 8)
 * A matrix [rows x in] is row-major with ceil(in/32) blocks per row; columns
 * past `in` in the last block must be zero weights. */
typedef enum dls_wtype { DLS_Q4_0 = 4, DLS_Q8_0 = 8 } dls_wtype;
/* GGUF K-quant types (layouts under "K-quant dequant-GEMV" below); allowed
 * per matrix (dls_layer_desc.types, tok_embd_type, output_type). */
#define DLS_Q4_K 12
#define DLS_Q5_K 13
#define DLS_Q6_K 14

/* Device memory source.  alloc returns device memory of at least `bytes`
 * (256-byte aligned) or NULL; free releases it.  `stream` is the model's
 * cudaStream_t.  Pass NULL for the allocator to use cudaMalloc/cudaFree.
 * Every byte the library holds on the device goes through this, and is
 * counted by the model's budget ledger. */
typedef struct dls_allocator {
  void* (*alloc)(void* ctx, size_t bytes, void* stream);
  void (*free)(void* ctx, void* ptr, void* stream);
  void* ctx;
} dls_allocator;

/* One layer's weights, all host memory, read only during dls_model_create. */
typedef struct dls_layer_desc {
  const float* attn_norm; /* fp32 [hidden] */
  const float* ffn_norm;  /* fp32 [hidden] */
  const void* wq;         /* blocks [n_heads*head_dim x hidden] */
  const void* wk;         /* blocks [n_kv_heads*head_dim x hidden] */
  const void* wv;         /* blocks [n_kv_heads*head_dim x hidden] */
  const void* wo;         /* blocks [hidden x n_heads*head_dim] */
  const void* w_gate;     /* blocks [ffn x hidden] */
  const void* w_up;       /* blocks [ffn x hidden] */
  const void* w_down;     /* blocks [hidden x ffn] (ffn padded to 32 with zero weights) */
  /* Weight type of wq, wk, wv, wo, w_gate, w_up, w_down in that order: 0 =
   * the model's wtype, or DLS_Q4_K / DLS_Q5_K / DLS_Q6_K for GGUF K-quant
   * super-blocks (the matrix's input width a multiple of 256).  Every layer
   * must give the same types.  A model with any K-quant matrix ("mixed")
   * runs its decode steps, batched steps and prefill through per-matrix
   * dequant-GEMVs with separate RMSNorm, RoPE/KV-append, attention, SwiGLU
   * and residual kernels, one row at a time (prefill: up to 8 tokens per
   * pass over the layers); the persistent step kernel and the tensor-core
   * paths serve Q8_0 / Q4_0 models. */
  int32_t types[7];
} dls_layer_desc;

typedef struct dls_model_desc {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  float rope_theta; /* RoPE base; pair i of a head rotates by pos * theta^(-2i/head_dim) */
  float rms_eps;    /* RMSNorm epsilon */
  int32_t tied_embeddings; /* nonzero: the LM head is tok_embd, `output` is ignored */
  int32_t wtype;           /* dls_wtype of every matrix */
  int32_t page_tokens;     /* KV page size in tokens: 32, 64, 128 or 256; 0 = 64 */
  int32_t max_seqs;        /* sequences the KV pool serves (>= 1) */
  int32_t max_ctx;         /* tokens per sequence (>= 1) */
  int32_t max_batch;       /* largest n of dls_decode_batch, 1..DLS_MAX_BATCH; 0 = 1 */
  uint64_t device_budget_bytes; /* cap on library device memory; 0 = no cap */
  const void* tok_embd;    /* host blocks [vocab x hidden] */
  const void* output;      /* host blocks [vocab x hidden], or NULL when tied */
  const float* output_norm;/* host fp32 [hidden] */
  const dls_layer_desc* layers; /* host array [n_layers] */
  int32_t kv_pool_pages;   /* KV pages shared by all sequences; 0 = max_seqs * ceil(max_ctx / page_tokens),
                              which lets every sequence reach max_ctx on private pages.  A smaller pool
                              oversubscribes: a call that needs a page when none is free fails with
                              DLS_ERR_CAPACITY and changes nothing. */
  int32_t tok_embd_type;   /* 0 = wtype, or a K-quant type (hidden a multiple of 256) */
  int32_t output_type;     /* the LM head's type likewise (ignored when tied) */
} dls_model_desc;

/* ---- model ------------------------------------------------------------- */

/* Validate `desc`, place the weights (re-laid-out for the kernels) and the
 * paged KV pool on the device, and return a model in *out.
 * Shape rules (else DLS_ERR_ARG): hidden a multiple of 32; head_dim 32, 64
 * or 128; n_heads a multiple of n_kv_heads with at most 16 query heads per
 * KV head; ffn and vocab any positive size.  With device_budget_bytes set, as many layers as
 * fit stay resident (first layers first) and the rest are streamed from
 * pinned host memory each step; DLS_ERR_BUDGET if not even that fits.
 * `cuda_stream` (cudaStream_t) orders all work; NULL makes a private stream.
 * The caller keeps ownership of every desc buffer (they are copied). */
int dls_model_create(const dls_model_desc* desc, const dls_allocator* allocator, void* cuda_stream,
                     dls_model** out);
void dls_model_destroy(dls_model* m);

/* Device bytes the ledger holds for this model, and its cap (0 = none). */
uint64_t dls_device_bytes(const dls_model* m);
uint64_t dls_device_budget(const dls_model* m);

/* ---- sequences ---------------------------------------------------------- */

/* Claim a free sequence id in [0, max_seqs).  It starts empty (length 0) and
 * holds no KV pages until tokens are written.  DLS_ERR_CAPACITY if none free. */
int dls_seq_create(dls_model* m, int32_t* seq_out);
/* Release a sequence and its KV pages. */
int dls_seq_free(dls_model* m, int32_t seq);
/* Tokens held in the sequence's KV cache, or a negative status. */
int32_t dls_seq_length(const dls_model* m, int32_t seq);

/* ---- the hot path --------------------------------------------------------- */

/* Run n prompt tokens (host int32 [n], each in [0, vocab)) through every
 * layer at positions length..length+n-1 of `seq`, filling its KV cache
 * (SwarmKV, section 2: prefill computes and stores the K/V of every prompt
 * token once).  The tokens go through in chunks of up to 2048 (the
 * environment variable DLS_PREFILL_CHUNK, read at model creation, sets
 * another size): each projection of a chunk is one tensor-core GEMM with
 * split fp16 operands (weights d*q and activations each as an fp16 value
 * plus the fp16 of its rounding residual, three products per K step) and
 * fp32 accumulation; attention is causal over the cache.  The
 * chunking changes a token's results at most by the fp32 summation order of
 * the GEMM tiling (chunks of up to 16 tokens split K across CTAs).  logits_out (host or device fp32
 * [vocab], or NULL) receives the logits of the last token.  DLS_ERR_CAPACITY
 * if length + n > max_ctx. */
int dls_prefill(dls_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out);

/* One decode step: `token` at position `pos`, which must equal the
 * sequence's length (else DLS_ERR_STATE: a fork must continue at the prefix
 * length).  Appends the token's K/V and writes logits (host or device fp32
 * [vocab]; NULL skips the copy-out). */
int dls_decode_step(dls_model* m, int32_t seq, int32_t token, int32_t pos, float* logits_out);

/* n decode steps in one pass over the weights (1 <= n <= max_batch): row i
 * is token tokens[i] of sequence seqs[i] at position pos[i] (host arrays;
 * distinct sequences).  logits_out: host or device fp32 [n][vocab] or NULL.
 * With n >= 2 each projection is one pass over the weights for all n rows,
 * so each weight byte is read once per step for the whole batch (SwarmKV,
 * section 4: the branches of a fork decode together): for n = 2..4 a
 * multi-row CUDA-core dequant-GEMV (exact int32 code x int16-slice
 * products, fp32 scaling), for n = 5..8 a tensor-core GEMM with the raw
 * codes as exact fp16 operands and the activations as hi + lo fp16 planes,
 * fp32 accumulation (the environment variable DLS_BATCH_GEMM=rg or tc,
 * read at model creation, forces one of the two); n = 1 is
 * dls_decode_step. */
int dls_decode_batch(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, const int32_t* pos,
                     float* logits_out);

/* Greedy generation kept on the device: n_steps decode steps of sequences
 * seqs[0..n-1] starting from tokens[i] at each sequence's end; each step's
 * argmax (lowest index on ties) is the next step's token.  tokens_out (host
 * int32 [n_steps][n]) receives the chosen tokens; last_logits (host or
 * device fp32 [n][vocab], or NULL) the final step's logits. */
int dls_generate(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, int32_t n_steps,
                 int32_t* tokens_out, float* last_logits);

/* Greedy pick per row: out[i] = argmax logits[i][0..vocab) (lowest index on
 * ties).  logits: device fp32 [n_rows][vocab]; out: host or device int32. */
int dls_argmax(dls_model* m, const float* logits, int32_t n_rows, int32_t* out);

/* KV fork: copy the first length(src) positions of every layer's K and V of
 * `src_seq` into each destination sequence (bit-exact device-to-device copy)
 * and set each destination's length to length(src).  Destinations must be
 * distinct live sequences other than src; their previous contents are
 * dropped.  DLS_ERR_CAPACITY if the KV pool cannot hold the copies. */
int dls_kv_fork(dls_model* m, int32_t src_seq, const int32_t* dst_seqs, int32_t n_dst);

/* KV fork by reference (the shared-prefix form of the fork: the SwarmKV
 * page, section 3, notes that paged KV sharing is the same idea as its
 * snapshot copy).  Each destination's page table takes the pages of
 * `src_seq` that hold only positions below length(src) as they are (a page
 * count per page keeps them allocated until every holder is freed); the page
 * the next position falls in, when partly filled, is copied into a fresh
 * page per destination, so appends never touch a shared page.  Destinations
 * read exactly the source's K/V bytes and get length(src).  Same argument
 * rules as dls_kv_fork; DLS_ERR_CAPACITY if the pool cannot hold one fresh
 * page per destination. */
int dls_kv_fork_shared(dls_model* m, int32_t src_seq, const int32_t* dst_seqs, int32_t n_dst);

/* Free pages in the KV pool (pages held by no sequence). */
int32_t dls_kv_free_pages(const dls_model* m);

/* ---- layer skip (the engine page, sections 2.5, 3.5, 4.5) ---------------------- */

/* Layers that decode steps skip from now on: skip[l] != 0 makes layer l's
 * output its input (the layer's projections, attention and cache append are
 * not run).  Host uint8 [n_layers] with n_layers equal to the model's, or
 * NULL to compute every layer.  Prefill is unaffected.  A layer skipped at
 * some positions has no cache entries there; compute it again only on
 * sequences started after the change.  Graph-captured steps are dropped and
 * captured again. */
int dls_set_layer_skip(dls_model* m, const uint8_t* skip, int32_t n_layers);

/* The calibration the engine page describes: one decode step of `token` at
 * `pos` of `seq` (exactly as dls_decode_step, the sequence grows by one),
 * and for every layer l the cosine similarity of its output with its input
 * (the previous layer's output; the embedding row for layer 0) written to
 * host cos_out [n_layers].  Layers above a threshold (0.98 on the page) are
 * the ones to pass to dls_set_layer_skip. */
int dls_layer_cosines(dls_model* m, int32_t seq, int32_t token, int32_t pos, float* cos_out);

/* ---- self-speculative decoding (the engine page, sections 3.5 and 5.3) ------- */

/* Cut `seq` back to its first `len` positions (0 <= len <= length, else
 * DLS_ERR_ARG); decoding continues at position len.  Pages past them return
 * to the pool (pages shared by a dls_kv_fork_shared stay with their other
 * holders); when the page that position len falls in is shared, it is first
 * replaced by a private copy (DLS_ERR_CAPACITY, nothing changed, if the pool
 * has no page for it). */
int dls_seq_truncate(dls_model* m, int32_t seq, int32_t len);

/* Score n tokens at once (1 <= n <= DLS_MAX_VERIFY): tokens (host int32
 * [n]) go through every layer at positions length..length+n-1 as one
 * dls_prefill chunk (the cache receives their K/V, the sequence grows by n),
 * and every position's logits are kept: logits_out (host or device fp32
 * [n][vocab], or NULL) and their greedy picks argmax_out (host int32 [n],
 * lowest index on ties, or NULL).  Row i is the model's prediction after
 * tokens[0..i].  The layer skip mask does not apply. */
int dls_verify(dls_model* m, int32_t seq, const int32_t* tokens, int32_t n, float* logits_out, int32_t* argmax_out);

/* Greedy self-speculative generation of n_tokens tokens from `token` at the
 * end of `seq` (the same tokens_out as dls_generate with one sequence, and
 * the sequence grows by n_tokens).  The draft is this model with the layers
 * draft_skip[l] != 0 skipped (host uint8 [n_layers]; e.g. the streamed
 * layers, or those dls_layer_cosines finds above a threshold).  Each round:
 * r = min(draft_k, tokens still wanted - 1) draft decode steps from the
 * current token t at position P; the sequence cut back to P; one pass of
 * [t, d_1..d_r] at positions P..P+r through every layer (a batched decode
 * step over the one sequence when r + 1 <= 8, else a dls_verify prefill
 * chunk); the longest prefix of drafts the full model also picks is
 * accepted, and the round emits those drafts plus the full model's next pick
 * (so the output is the full model's greedy continuation).  0 <= draft_k < DLS_MAX_VERIFY.  stats (host int32 [3], or
 * NULL) receives rounds, drafted and accepted token counts.  Draft steps
 * skip streamed layers' copies when the draft skips every streamed layer.
 * The mask of dls_set_layer_skip is not used by this call. */
int dls_generate_speculative(dls_model* m, int32_t seq, int32_t token, int32_t n_tokens, const uint8_t* draft_skip,
                             int32_t draft_k, int32_t* tokens_out, int32_t* stats);

/* Context-budget check done before any allocation (SwarmKV page, section 4,
 * step 0): DLS_OK if prefix_tokens + max_branch_tokens + headroom <= n_ctx,
 * else DLS_ERR_CAPACITY with the numbers in dls_last_error(NULL). */
int dls_check_context_budget(int32_t prefix_tokens, int32_t max_branch_tokens, int32_t headroom, int32_t n_ctx);

/* ---- layer residency and streaming ----------------------------------------- */

/* Keep layers [0, n) resident on the device and stream layers [n, n_layers)
 * from pinned host memory through two device buffers on a copy stream,
 * overlapped with compute.  n = -1 picks the largest n the budget allows.
 * DLS_ERR_BUDGET (model unchanged) if the layout does not fit the budget. */
int dls_set_resident_layers(dls_model* m, int32_t n);
int32_t dls_resident_layers(const dls_model* m);
/* Bytes of one layer's weights as the kernels read them (the per-layer H2D
 * transfer of a streamed layer). */
uint64_t dls_layer_bytes(const dls_model* m);

/* Host -> device copy performed by `ctas` CTAs of 512 threads that read the
 * pinned host buffer directly over the host link (on a Grace host, NVLink-C2C)
 * instead of through the copy engines that cudaMemcpyAsync uses (the engine
 * page, sections 3.3 and 4.2: streamed layers are bound by the host link, so
 * the faster path matters).  src_host: pinned host memory (cudaHostAlloc or
 * registered); dst: device memory; both 16-byte aligned, bytes a multiple of
 * 16.  Enqueued on cuda_stream.  DLS_ERR_ARG for any other pointer kind
 * (checked with cudaPointerGetAttributes before anything is launched). */
int dls_h2d_copy_sm(void* dst, const void* src_host, size_t bytes, int32_t ctas, void* cuda_stream);

/* ---- standalone op ----------------------------------------------------------- */

/* Split-K (flash-decoding) GQA attention of one query position over an fp16
 * paged KV cache, for `n_batch` independent rows (the engine page, section
 * 4.4: causal softmax with the mask inside the kernel; section 1: GQA over a
 * KV cache).  All pointers device:
 *   q         fp32 [n_batch][n_heads][head_dim] (already rotated)
 *   k_pages,  fp16 pools [n_pages][n_kv_heads][page_tokens][head_dim]
 *   v_pages
 *   page_table int32 [n_batch][max_pages]: logical page -> physical page
 *   lengths   int32 [n_batch]: keys 0..lengths[b]-1 are attended
 *             (1 <= lengths[b] <= page_tokens * max_pages)
 *   o         fp32 [n_batch][n_heads][head_dim]
 *   workspace scratch of dls_attention_workspace_bytes(...) bytes; its
 *             counter words must be zero before the first call (the call
 *             leaves them zero again).
 *   status    int32 [1] or NULL.  The call zeroes it on cuda_stream; the
 *             kernel ORs in 1 when a page-table entry it needs is negative,
 *             4 when a length is outside 1..page_tokens*max_pages (the
 *             kernel then clamps it) and 8 when a bounded wait ran out.  Read
 *             it with dls_attention_status once the work is done.
 * `n_splits` = how many CTAs share one (row, kv head), 1..128; 0 = choose.
 * Returns DLS_ERR_ARG on a bad shape or a workspace too small for the split
 * count; the work is enqueued on cuda_stream (the outputs are valid once it
 * completes). */
int dls_attention_decode(const float* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                         const int32_t* lengths, float* o, void* workspace, size_t workspace_bytes,
                         int32_t n_batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                         int32_t page_tokens, int32_t max_pages, int32_t n_splits, int32_t* status,
                         void* cuda_stream);
size_t dls_attention_workspace_bytes(int32_t n_batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                     int32_t n_splits);

/* Wait for cuda_stream, read the status word of a standalone attention call
 * and turn it into a status code: DLS_OK (0), DLS_ERR_TIMEOUT (bit 8: a
 * bounded wait ran out), DLS_ERR_STATE (bits 1 or 4: a missing page or a bad
 * length; the output is not meaningful), with the flags in
 * dls_last_error(NULL). */
int dls_attention_status(const int32_t* status, void* cuda_stream);

/* Allocation-free dls_attention_decode.  The pages have no counterpart of
 * this call: it serves callers that may not allocate device memory at all
 * (a process that fixes its device memory plan at start-up, or code where
 * an allocator call could block or synchronise).  Same arguments and result
 * as dls_attention_decode minus the workspace: the split-K scratch is a
 * fixed array of DLS_ATTENTION_NOALLOC_SCRATCH_BYTES inside the library,
 * present on every GPU that loads the library until the process exits.
 * Nothing is allocated (no cudaMalloc, no allocating library call).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture on that device.
 *  - Every call shares the one array; the call zeroes the arrival counters
 *    it needs on `cuda_stream`, but calls that overlap on the GPU (other
 *    streams, concurrent threads) race on the scratch and must not be issued.
 *  - n_splits = 0 takes the usual split count, lowered until the partials
 *    fit the array.  DLS_ERR_CAPACITY if the shape needs more scratch than
 *    the array holds even so, or for an explicit n_splits
 *    (dls_attention_workspace_bytes tells the need); DLS_ERR_ARG on a bad
 *    shape; the message is in dls_last_error(NULL). */
#define DLS_ATTENTION_NOALLOC_SCRATCH_BYTES (4u << 20)
int dls_attention_decode_noalloc(const float* q, const void* k_pages, const void* v_pages,
                                 const int32_t* page_table, const int32_t* lengths, float* o, int32_t n_batch,
                                 int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t page_tokens,
                                 int32_t max_pages, int32_t n_splits, int32_t* status, void* cuda_stream);

/* ---- K-quant dequant-GEMV (the engine page, section 1: Q4_K_M, Q5_K, Q6_K) ----- */

/* GGUF K-quant types: 256 weights per super-block; Q4_K 144 bytes (fp16 d,
 * fp16 dmin, twelve bytes of 6-bit sub-block scales and minimums, 128 bytes
 * of 4-bit codes; weight = d*sc*q - dmin*m per sub-block of 32), Q5_K 176
 * bytes (Q4_K's first 16, then 32 bytes holding a fifth code bit per weight,
 * then the 128 bytes of low 4 bits; the same weight formula), Q6_K 210
 * bytes (128 bytes of low code bits, 64 of high bits, sixteen int8 scales,
 * fp16 d; weight = d*scale*(code - 32) per group of 16).  A [rows][cols]
 * matrix is row-major with cols/256 super-blocks per row (cols a multiple of
 * 256). */

/* Bytes of the device layout dls_kquant_gemv reads (0 for a bad type or
 * shape). */
uint64_t dls_kquant_packed_bytes(int32_t type, int32_t rows, int32_t cols);

/* Lay out `blocks` (device, GGUF super-blocks as above) for the GEMV into
 * `packed` (device, 256-byte aligned, dls_kquant_packed_bytes bytes, owned by
 * the caller): Q4_K and Q5_K as they are; Q6_K with the fp16 scales moved to a separate
 * array so that every row is 16-byte aligned.  Enqueued on cuda_stream. */
int dls_kquant_pack(int32_t type, const void* blocks, int32_t rows, int32_t cols, void* packed, void* cuda_stream);

/* y = W x, the decode step's projection on a K-quant matrix: x device fp32
 * [cols] (16-byte aligned), y device fp32 [rows], packed from
 * dls_kquant_pack.  Each weight row streams through shared memory once;
 * activations are held as int16 slices with one scale per 32 (Q4_K, Q5_K) or 64
 * (Q6_K) columns, so the code-activation products are exact int32 and the
 * result is within 2^-16 of each slice's largest activation of the exact
 * product.  status (device int32, or NULL) gets bit 8 or-ed in when a
 * bounded wait inside the kernel runs out (the output is then invalid).
 * Enqueued on cuda_stream; DLS_ERR_ARG on a bad type, shape (cols above
 * 32768 included) or alignment. */
int dls_kquant_gemv(int32_t type, const void* packed, int32_t rows, int32_t cols, const float* x, float* y,
                    int32_t* status, void* cuda_stream);

/* ---- test and profiling hooks ------------------------------------------------ */

/* Arm a capture of the residual stream after every layer for the next
 * decode call (batch row 0) or prefill call (its last prompt token):
 * per_layer_out device fp32 [n_layers][hidden].  NULL disarms.  A captured
 * decode call runs the same kernels as an uncaptured one (the persistent
 * step kernel for batch-1 steps of a resident model, which then also writes
 * each layer's residual), launched without CUDA-graph replay. */
int dls_debug_capture(dls_model* m, float* per_layer_out);
/* Run, on the model's stream, the library's bounded mbarrier wait against
 * a barrier that nothing arrives at, with a limit of limit_ns (1e3..1e10;
 * the kernels' own limit is 2 s).  The wait gives up, records the timeout
 * in the model's device status word, and the call returns DLS_ERR_TIMEOUT
 * like any call whose kernel saw a wait run out; the model stays usable.
 * DLS_ERR_ARG for a limit out of range.  Synchronises the stream. */
int dls_debug_bounded_wait(dls_model* m, int64_t limit_ns);
/* Copy positions [0, length) of one layer's K and V of `seq` into device
 * fp16 [length][n_kv_heads][head_dim] buffers. */
int dls_debug_read_kv(dls_model* m, int32_t seq, int32_t layer, void* k_out, void* v_out);
/* Dequantise one weight matrix as the kernels see it into device fp32
 * [rows][cols].  tensor: 0 wq, 1 wk, 2 wv, 3 wo, 4 w_gate, 5 w_up, 6 w_down,
 * 7 tok_embd, 8 output (layer ignored for 7 and 8). */
int dls_debug_dequant(dls_model* m, int32_t layer, int32_t tensor, float* out);
/* y = W x with the decode GEMV kernel for one matrix (ids as above);
 * x device fp32 [cols], y device fp32 [rows]. */
int dls_debug_gemv(dls_model* m, int32_t layer, int32_t tensor, const float* x, float* y);
/* Y = X W^T with the prefill GEMM for one matrix (ids as above): X device
 * fp32 [n_tokens][cols], rounded to fp16 on the device; Y device fp32
 * [n_tokens][rows].  Synchronises the model's stream. */
int dls_debug_gemm(dls_model* m, int32_t layer, int32_t tensor, int32_t n_tokens, const float* x, float* y);
/* One decode step (same contract as dls_decode_step, logits left in the
 * model's buffer) run with a CUDA event after every kernel and without
 * programmatic dependent launch, so each kernel's device time is measured
 * alone.  Writes up to max_kernels durations (host float ms) and kernel
 * kinds (host int32: 1 embedding, 2 QKV GEMV, 3 attention, 4 O GEMV, 5
 * gate/up GEMV, 6 down GEMV, 7 LM head GEMV) and the count to *n_kernels. */
int dls_debug_profile_step(dls_model* m, int32_t seq, int32_t token, int32_t pos, int32_t max_kernels,
                           float* kernel_ms, int32_t* kernel_kind, int32_t* n_kernels);
/* dls_debug_profile_step for a batch of n >= 2 rows (the arguments of
 * dls_decode_batch): every kernel of one batched step timed alone; each
 * row's sequence grows by one.  Profiling only. */
int dls_debug_profile_batch(dls_model* m, int32_t n, const int32_t* seqs, const int32_t* tokens, const int32_t* pos,
                            int32_t max_kernels, float* kernel_ms, int32_t* kernel_kind, int32_t* n_kernels);
/* Per-CTA phase timestamps (global timer, ns) of the last profiled step of
 * the persistent step kernel: [phase][cta][8] = {consumer arrival at the
 * grid barrier that ends the phase, its release, producer's first issue of
 * the phase's copies, producer's last issue, consumers' prologue done, last
 * stage consumed, epilogue done, first stage's data ready}; phase 0 is the embedding,
 * 1 + 5 l + k layer l's k-th phase (QKV, attention, O, gate/up, down), then
 * the LM head.  Entries not written hold stale values.  Copies
 * (5 n_layers + 8) * grid * 8 values to host `out`; DLS_ERR_STATE when the
 * step does not run as the persistent kernel.  Profiling only. */
int dls_debug_step_trace(dls_model* m, uint64_t* out, int32_t max_entries, int32_t* n_entries);
/* Kernel launches issued by the last decode / generate step (all of this
 * library's kernels, per step). */
int32_t dls_debug_launches_per_step(const dls_model* m);

/* Whether batch-1 steps run as the one persistent step kernel (1) or as
 * separate kernels (0).  When 0 and the persistent kernel was wanted,
 * *why (may be NULL) receives the reason as a static string ("disabled",
 * "not all layers resident", "mixed weight formats", or the planner's
 * reason: no instantiation for the shape, shared memory or registers do
 * not fit one CTA per SM, ...); NULL when in use. */
int32_t dls_step_kernel_in_use(const dls_model* m, const char** why);

/* ---- errors -------------------------------------------------------------------- */

const char* dls_last_error(const dls_model* m);
const char* dls_status_name(int status);
int dls_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DLS_H */
