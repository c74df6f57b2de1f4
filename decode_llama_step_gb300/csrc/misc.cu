// The decode step's small kernels: embedding-row dequant, greedy pick,
// step-parameter upkeep, weight re-layout, the RoPE sin/cos table, the KV
// fork copy and test-only gathers.
#include <math.h>

#include <algorithm>

#include "kernels.h"

namespace dls {

namespace {

cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, cudaStream_t s, bool pdl, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// one dequantised weight: exact in fp32 (11-bit scale times a code of at most 8 bits)
__device__ __forceinline__ float dq(const MatDev& m, int wtype, int row, int col) {
  const int blk = col >> 5, e = col & 31;
  row *= m.rstep;
  const float d = __half2float(m.d[(size_t)row * m.ds + blk]);
  if (wtype == 8) {
    const uint32_t u = (uint32_t)m.qs[(size_t)row * m.nb * 32 + col];  // stored biased: q + 128
    return d * (mag_byte(u, 0) - 8388736.0f);
  }
  const uint8_t byte = m.qs[((size_t)row * m.nb + blk) * 16 + (e & 15)];
  const uint32_t nib = e < 16 ? (byte & 15u) : (byte >> 4);
  return d * (mag_byte(nib, 0) - 8388616.0f);
}

// ---------------------------------------------------------------- embedding

// one 32-element block per thread iteration, all loads issued up front
__global__ void embed_kernel(const MatDev emb, int wtype, StepParams* sp, int brow, float* x, int vocab) {
  griddep_wait();
  griddep_launch();
  int tok = sp->token[brow];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(&sp->status, kBadToken);
    tok = 0;
  }
  for (int blk = threadIdx.x; blk < emb.nb; blk += blockDim.x) {
    const float d = __half2float(emb.d[(size_t)tok * emb.ds + blk]);
    float v[32];
    if (wtype == 8) {
      const uint4* q = reinterpret_cast<const uint4*>(emb.qs + ((size_t)tok * emb.nb + blk) * 32);
      const uint4 q0 = q[0], q1 = q[1];
      const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t u = w[k];  // stored biased: q + 128
#pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * k + e] = mag_byte(u, e) - 8388736.0f;
      }
    } else {
      const uint4 q = *reinterpret_cast<const uint4*>(emb.qs + ((size_t)tok * emb.nb + blk) * 16);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = w[k] & 0x0F0F0F0Fu, hi = (w[k] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[4 * k + e] = mag_byte(lo, e) - 8388616.0f;
          v[16 + 4 * k + e] = mag_byte(hi, e) - 8388616.0f;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = blk * 32 + e;
      if (c < emb.cols) x[c] = d * v[e];
    }
  }
}

// ---------------------------------------------------------------- greedy pick

// CTA (blk, row) reduces a contiguous slice of one row to (value, index);
// the last CTA of the row to finish reduces the slices in order.  Ties go
// to the lowest index; NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void argmax_kernel(const float* logits, int vocab, int32_t* out, int2* part, int* counters) {
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.y, nblk = gridDim.x;
  const int per = (vocab + nblk - 1) / nblk;
  const int lo = blockIdx.x * per, hi = min(vocab, lo + per);
  const float* r = logits + (size_t)row * vocab;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const float v = r[i];
    if (better(v, i, best, bi)) {
      best = v;
      bi = i;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, best, bi)) {
      best = ov;
      bi = oi;
    }
  }
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (better(sv[w], si[w], best, bi)) {
        best = sv[w];
        bi = si[w];
      }
    part[(size_t)row * nblk + blockIdx.x] = make_int2(__float_as_int(best), bi);
    __threadfence();
    s_last = atomicAdd(&counters[row], 1) == nblk - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  best = -INFINITY;
  bi = 0x7fffffff;
  for (int b = 0; b < nblk; ++b) {
    const int2 p = __ldcg(&part[(size_t)row * nblk + b]);
    if (better(__int_as_float(p.x), p.y, best, bi)) {
      best = __int_as_float(p.x);
      bi = p.y;
    }
  }
  out[row] = bi == 0x7fffffff ? 0 : bi;  // all-NaN row: 0
  counters[row] = 0;
}

// next token := argmax, position += 1, record the token for the host
__global__ void advance_kernel(StepParams* sp, const int32_t* next, int32_t* tokens_out, int rows) {
  griddep_wait();
  griddep_launch();
  const int b = threadIdx.x;
  const int step = sp->step;
  __syncthreads();
  if (b < rows) {
    sp->token[b] = next[b];
    sp->pos[b] += 1;
    if (tokens_out) tokens_out[(size_t)step * rows + b] = next[b];
  }
  __syncthreads();
  if (b == 0) sp->step = step + 1;
}

__global__ void set_params_kernel(StepParams* sp, const StepParams h, int reset_step) {
  const int b = threadIdx.x;
  if (b < kMaxBatch) {
    sp->token[b] = h.token[b];
    sp->pos[b] = h.pos[b];
    sp->seq[b] = h.seq[b];
  }
  if (b == 0) {
    sp->n = h.n;
    sp->shared_len = h.shared_len;
    if (reset_step) {
      sp->step = 0;
      sp->status = 0;
    }
  }
}

// ---------------------------------------------------------------- weight layout

// GGUF-style blocks (2-byte scale + codes) -> scale array + code array
__global__ void repack_kernel(const uint8_t* src, int wtype, long long n_blocks, int nb, int ds, int row_step,
                              uint8_t* qs, __half* d) {
  const int bsz = wtype == 8 ? 34 : 18, nq = bsz - 2;
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < n_blocks;
       b += (long long)gridDim.x * blockDim.x) {
    const uint8_t* s = src + b * bsz;
    const long long r = (b / nb) * row_step, j = b % nb;
    d[r * ds + j] = __ushort_as_half((unsigned short)(s[0] | (s[1] << 8)));
    uint8_t* q = qs + (r * nb + j) * nq;
    // Q8_0 codes are stored biased (q + 128, as unsigned bytes) so the
    // kernels' exact byte -> float conversion needs no per-word XOR
    const uint8_t bias = wtype == 8 ? 0x80 : 0x00;
    for (int i = 0; i < nq; ++i) q[i] = s[2 + i] ^ bias;
  }
}

// RoPE table: entry (p, i) = (cos, sin) of p * theta^(-2i/hd), computed in
// fp64 and rounded once to fp32 (the engine page, section 4.4, precomputes
// the sin/cos table; fp64 keeps angles of up to ~1e4 radians accurate)
__global__ void rope_table_kernel(float2* cs, int len, int hd, double theta) {
  const int half = hd / 2;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < (long long)len * half;
       k += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(k / half), i = (int)(k % half);
    const double ang = (double)p * pow(theta, -2.0 * i / hd);
    double s, c;
    sincos(ang, &s, &c);
    cs[k] = make_float2((float)c, (float)s);
  }
}

__global__ void dequant_kernel(const MatDev m, int wtype, float* out) {
  const long long total = (long long)m.rows * m.cols;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < total;
       k += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(k / m.cols), c = (int)(k % m.cols);
    out[k] = dq(m, wtype, r, c);
  }
}

// ---------------------------------------------------------------- KV fork copy

// Whole pages, every layer, K and V: a plain 16-byte vector copy (HBM-bound).
// blockIdx.y = pair, blockIdx.z = layer*2 + (0: K, 1: V).
__global__ void kv_copy_kernel(__half* k_pool, __half* v_pool, size_t layer_stride, size_t page_elems,
                               const int2* pairs) {
  const int2 pr = pairs[blockIdx.y];
  const int layer = blockIdx.z >> 1;
  __half* pool = (blockIdx.z & 1) ? v_pool : k_pool;
  const uint4* src = reinterpret_cast<const uint4*>(pool + layer * layer_stride + (size_t)pr.x * page_elems);
  uint4* dst = reinterpret_cast<uint4*>(pool + layer * layer_stride + (size_t)pr.y * page_elems);
  const size_t n16 = page_elems * sizeof(__half) / 16;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __ldcs(src + i);
}

__global__ void kv_gather_kernel(const __half* pool, const int32_t* pages, int len, int n_kv, int pt, int hd,
                                 __half* out) {
  const long long total = (long long)len * n_kv * hd;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < total;
       k += (long long)gridDim.x * blockDim.x) {
    const int dim = (int)(k % hd);
    const int h = (int)((k / hd) % n_kv);
    const int p = (int)(k / ((long long)hd * n_kv));
    const int page = pages[p / pt];
    out[k] = pool[(((size_t)page * n_kv + h) * pt + (p % pt)) * hd + dim];
  }
}

__global__ void delay_kernel(long long ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < (1 << 24); ++i) {  // bounded: at most ~16M polls
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if ((long long)(t - t0) >= ns) break;
    __nanosleep(1000);
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

// cos(x_in, x_out) of every layer: block l reduces the dot product and
// the two squared norms of (layer l's input, its output), the input of
// layer 0 being the embedding row and of layer l > 0 layer l-1's output
__global__ void layer_cosines_kernel(const float* emb, const float* cap, int H, float* out) {
  const int l = blockIdx.x;
  const float* xi = l == 0 ? emb : cap + (size_t)(l - 1) * H;
  const float* xo = cap + (size_t)l * H;
  float d = 0.f, a = 0.f, b = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float p = xi[i], q = xo[i];
    d = fmaf(p, q, d);
    a = fmaf(p, p, a);
    b = fmaf(q, q, b);
  }
  __shared__ float red[3][32];
  d = warp_sum(d);
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][w] = d;
    red[1][w] = a;
    red[2][w] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float dd = 0.f, aa = 0.f, bb = 0.f;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
      dd += red[0][k];
      aa += red[1][k];
      bb += red[2][k];
    }
    out[l] = (aa > 0.f && bb > 0.f) ? dd / (sqrtf(aa) * sqrtf(bb)) : 0.f;
  }
}

cudaError_t launch_layer_cosines(const float* emb, const float* cap, int L, int H, float* out, cudaStream_t s) {
  layer_cosines_kernel<<<L, 256, 0, s>>>(emb, cap, H, out);
  return cudaGetLastError();
}

cudaError_t launch_embed(const MatDev& emb, int wtype, StepParams* sp, int brow, float* x, int vocab,
                         cudaStream_t s, bool pdl) {
  MatDev e = emb;
  void* args[] = {&e, &wtype, &sp, &brow, &x, &vocab};
  return launch_ex((const void*)embed_kernel, dim3(1), dim3(256), s, pdl, args);
}

int argmax_blocks(int rows, int num_sms) {
  int n = (2 * num_sms) / (rows > 0 ? rows : 1);
  return n < 1 ? 1 : (n > num_sms ? num_sms : n);
}

cudaError_t launch_argmax(const float* logits, int vocab, int rows, int32_t* out, int2* part, int* counters,
                          int nblk, cudaStream_t s, bool pdl) {
  void* args[] = {&logits, &vocab, &out, &part, &counters};
  return launch_ex((const void*)argmax_kernel, dim3(nblk, rows), dim3(256), s, pdl, args);
}

cudaError_t launch_advance(StepParams* sp, const int32_t* next, int32_t* tokens_out, int rows, cudaStream_t s,
                           bool pdl) {
  void* args[] = {&sp, &next, &tokens_out, &rows};
  return launch_ex((const void*)advance_kernel, dim3(1), dim3(32), s, pdl, args);
}

cudaError_t launch_set_params(StepParams* sp, const StepParams& h, bool reset_step, cudaStream_t s) {
  set_params_kernel<<<1, 32, 0, s>>>(sp, h, reset_step ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_repack(const uint8_t* src, int wtype, int rows, int nb, int ds, int row_step, uint8_t* qs,
                          __half* d, cudaStream_t s) {
  const long long n = (long long)rows * nb;
  repack_kernel<<<grid_for(n, 256), 256, 0, s>>>(src, wtype, n, nb, ds, row_step, qs, d);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* cs, int len, int head_dim, float theta, cudaStream_t s) {
  rope_table_kernel<<<grid_for((long long)len * head_dim / 2, 256), 256, 0, s>>>(cs, len, head_dim, (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const MatDev& m, int wtype, float* out, cudaStream_t s) {
  dequant_kernel<<<grid_for((long long)m.rows * m.cols, 256), 256, 0, s>>>(m, wtype, out);
  return cudaGetLastError();
}

cudaError_t launch_kv_copy(__half* k_pool, __half* v_pool, size_t layer_stride_elems, int n_layers,
                           size_t page_elems, const int2* pairs, int n_pairs, cudaStream_t s) {
  if (n_pairs <= 0) return cudaSuccess;
  const size_t n16 = page_elems * sizeof(__half) / 16;
  int gx = (int)((n16 + 255) / 256);
  if (gx > 64) gx = 64;
  for (int p0 = 0; p0 < n_pairs; p0 += 65535) {  // grid.y limit
    const int np = n_pairs - p0 < 65535 ? n_pairs - p0 : 65535;
    kv_copy_kernel<<<dim3(gx, np, 2 * n_layers), 256, 0, s>>>(k_pool, v_pool, layer_stride_elems, page_elems,
                                                                 pairs + p0);
  }
  return cudaGetLastError();
}

// One thread waits, with the library's bounded mbarrier wait, on a barrier
// that nothing arrives at; when the limit runs out it records kTimeout in
// the status word, exactly as a kernel whose copy never landed would.
__global__ void unarrived_wait_kernel(unsigned long long limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  mbar_fence_init();
  if (!mbar_wait(smem_u32(&bar), 0, 1000, limit_ns)) atomicOr(status, kTimeout);
}

cudaError_t launch_unarrived_wait(unsigned long long limit_ns, int32_t* status, cudaStream_t s) {
  unarrived_wait_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

// ---- single-vector helpers (the mixed-format decode path) ------------------------
//
// Launched with programmatic dependent launch: each waits for the previous
// kernel's results before it reads or writes anything, then lets the next
// kernel (a GEMV that streams its weights meanwhile) start.

// out = x / sqrt(mean(x^2) + eps) * g, one CTA, fixed-order reduction
__global__ void rmsnorm_vec_kernel(const float* x, int H, const float* g, float eps, float* out) {
  griddep_wait();
  griddep_launch();
  __shared__ float red[32];
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  const float rs = 1.0f / sqrtf(t / (float)H + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x) out[i] = x[i] * rs * g[i];
}

__global__ void add_vec_kernel(float* x, const float* y, int n) {
  griddep_wait();
  griddep_launch();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) x[i] += y[i];
}

__global__ void swiglu_vec_kernel(const float* gate, const float* up, float* h, int n) {
  griddep_wait();
  griddep_launch();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    h[i] = silu(gate[i]) * up[i];
}

cudaError_t launch_rmsnorm_vec(const float* x, int H, const float* g, float eps, float* out, cudaStream_t s) {
  void* args[] = {(void*)&x, &H, (void*)&g, &eps, &out};
  return launch_ex((const void*)rmsnorm_vec_kernel, dim3(1), dim3(1024), s, true, args);
}

cudaError_t launch_add_vec(float* x, const float* y, int n, cudaStream_t s) {
  void* args[] = {&x, (void*)&y, &n};
  return launch_ex((const void*)add_vec_kernel, dim3(std::min((n + 255) / 256, 1024)), dim3(256), s, true, args);
}

cudaError_t launch_swiglu_vec(const float* gate, const float* up, float* h, int n, cudaStream_t s) {
  void* args[] = {(void*)&gate, (void*)&up, &h, &n};
  return launch_ex((const void*)swiglu_vec_kernel, dim3(std::min((n + 255) / 256, 1024)), dim3(256), s, true,
                   args);
}

// Host -> device copy driven by the SMs: every thread reads 16-byte words of
// pinned host memory straight over the host link (four loads in flight per
// thread before the stores) and writes them to device memory.  Both
// pointers 16-byte aligned, bytes a multiple of 16 (checked by the caller).
__global__ void __launch_bounds__(512) h2d_sm_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                     size_t n16) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
                d = __ldcs(src + i + 3 * stride);
    __stcg(dst + i, a);
    __stcg(dst + i + stride, b);
    __stcg(dst + i + 2 * stride, c);
    __stcg(dst + i + 3 * stride, d);
  }
  for (; i < n16; i += stride) __stcg(dst + i, __ldcs(src + i));
}

cudaError_t launch_h2d_sm(void* dst, const void* src, size_t bytes, int ctas, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  h2d_sm_kernel<<<ctas, 512, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), bytes / 16);
  return cudaGetLastError();
}

cudaError_t launch_delay(long long ns, cudaStream_t s) {
  delay_kernel<<<1, 1, 0, s>>>(ns);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const __half* pool, const int32_t* pages, int len, int n_kv, int page_tokens,
                             int head_dim, __half* out, cudaStream_t s) {
  kv_gather_kernel<<<grid_for((long long)len * n_kv * head_dim, 256), 256, 0, s>>>(pool, pages, len, n_kv,
                                                                                 page_tokens, head_dim, out);
  return cudaGetLastError();
}

}  // namespace dls
