// Prefill kernels besides the projections (those are the tensor-core GEMM
// in gemm.cu): the layer math for T prompt tokens at once (SwarmKV page,
// section 2: prefill runs every prompt token through every layer once and
// fills the KV cache).
//
//  * pattn_kernel: causal attention of T query tokens over the sequence's
//    paged fp16 cache, flash style on CUDA cores (64 query-head rows per CTA,
//    32-key tiles, online softmax in registers).
//  * row kernels: embedding rows, RMSNorm -> fp16, RoPE + fp16 K/V append,
//    fp32 -> fp16.
#include <math.h>

#include <utility>

#include "kernels.h"

namespace dls {

namespace {

// ---------------------------------------------------------------- row kernels

// hi and lo fp16 planes of four fp32 values: hi = fp16(v), lo = fp16(v - hi)
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint2& hi, uint2& lo) {
  const __half2 h0 = __floats2half2_rn(a, b), h1 = __floats2half2_rn(c, d);
  const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
  const __half2 l0 = __floats2half2_rn(a - f0.x, b - f0.y), l1 = __floats2half2_rn(c - f1.x, d - f1.y);
  hi.x = *reinterpret_cast<const uint32_t*>(&h0);
  hi.y = *reinterpret_cast<const uint32_t*>(&h1);
  lo.x = *reinterpret_cast<const uint32_t*>(&l0);
  lo.y = *reinterpret_cast<const uint32_t*>(&l1);
}

// out[t] = fp16 planes of rmsnorm(x[t]) * g, zero-padded to ldo columns (H % 4 == 0)
__global__ void rmsnorm_rows_kernel(const float* x, int H, int ldx, const float* g, float eps, __half* out,
                                    __half* out_lo, int ldo) {
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * ldx);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const int n4 = H >> 2;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i];
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  const float rs = 1.0f / sqrtf(t / (float)H + eps);
  __half* o = out + (size_t)blockIdx.x * ldo;
  __half* ol = out_lo + (size_t)blockIdx.x * ldo;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i], gg = g4[i];
    uint2 hi, lo;
    split4(v.x * rs * gg.x, v.y * rs * gg.y, v.z * rs * gg.z, v.w * rs * gg.w, hi, lo);
    *reinterpret_cast<uint2*>(o + 4 * i) = hi;
    *reinterpret_cast<uint2*>(ol + 4 * i) = lo;
  }
  for (int i = H + threadIdx.x; i < ldo; i += blockDim.x) o[i] = ol[i] = __float2half_rn(0.f);
}

// out[t][0..cols) = fp16 planes of x[t], zero up to ldo (cols % 4 == 0)
__global__ void to_f16_rows_kernel(const float* x, int cols, int ldx, __half* out, __half* out_lo, int ldo) {
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * ldx);
  __half* o = out + (size_t)blockIdx.x * ldo;
  __half* ol = out_lo + (size_t)blockIdx.x * ldo;
  for (int i = threadIdx.x; i < (cols >> 2); i += blockDim.x) {
    const float4 v = xr[i];
    uint2 hi, lo;
    split4(v.x, v.y, v.z, v.w, hi, lo);
    *reinterpret_cast<uint2*>(o + 4 * i) = hi;
    *reinterpret_cast<uint2*>(ol + 4 * i) = lo;
  }
  for (int i = cols + threadIdx.x; i < ldo; i += blockDim.x) o[i] = ol[i] = __float2half_rn(0.f);
}

int row_threads(int elems) {
  int t = (elems + 31) / 32 * 32;
  return t < 64 ? 64 : t > 1024 ? 1024 : t;
}

// RoPE on the q and k rows of token t at position pos0 + t; q -> q_out
// (fp32), k and v -> the sequence's pages (fp16)
__global__ void rope_kv_rows_kernel(const float* qkv, int ld, int q_rows, int kv_rows, KvView kv, int seq, int pos0,
                                    const int32_t* seqs, const int32_t* poss, const float2* rope_cs, int rope_len,
                                    float* q_out, int32_t* status) {
  const int t = blockIdx.x;
  const int pos = poss ? poss[t] : pos0 + t;
  if (seqs) seq = seqs[t];
  const float* row = qkv + (size_t)t * ld;
  const int hd = kv.head_dim;
  const int lp = pos / kv.page_tokens;
  const int page = lp < kv.max_pages ? kv.page_table[(size_t)seq * kv.max_pages + lp] : -1;
  if (pos >= rope_len || page < 0) {
    if (threadIdx.x == 0 && status) atomicOr(status, page < 0 ? kBadPage : kBadPos);
    return;
  }
  const int npairs = (q_rows + 2 * kv_rows) / 2;
  for (int pi = threadIdx.x; pi < npairs; pi += blockDim.x) {
    const int r = 2 * pi;
    float v0 = row[r], v1 = row[r + 1];
    if (r < q_rows + kv_rows) {
      const float2 cs = rope_cs[(size_t)pos * (hd >> 1) + ((r % hd) >> 1)];
      const float t0 = v0 * cs.x - v1 * cs.y;
      v1 = v0 * cs.y + v1 * cs.x;
      v0 = t0;
    }
    if (r < q_rows) {
      q_out[(size_t)t * q_rows + r] = v0;
      q_out[(size_t)t * q_rows + r + 1] = v1;
    } else {
      const bool is_k = r < q_rows + kv_rows;
      const int rk = r - q_rows - (is_k ? 0 : kv_rows);
      const int kvh = rk / hd, dim = rk % hd;
      const size_t off = (((size_t)page * kv.n_kv + kvh) * kv.page_tokens + (pos % kv.page_tokens)) * hd + dim;
      *reinterpret_cast<__half2*>((is_k ? kv.k_pool : kv.v_pool) + off) = __floats2half2_rn(v0, v1);
    }
  }
}

// ---------------------------------------------------------------- causal prefill attention

constexpr int PA_ROWS = 64;   // query-head rows per CTA
constexpr int PA_KT = 32;     // keys per tile
constexpr int PA_T = 256;
template <int HD>
constexpr int PA_KROW = HD + 8;  // padded fp16 key row (16 extra bytes: no bank conflicts)
template <int HD>
constexpr int pa_smem_bytes() {
  return PA_ROWS * HD * 4 + PA_KT * PA_KROW<HD> * 2 + PA_KT * HD * 2 + PA_ROWS * (PA_KT + 1) * 4;
}

// CTA (kv head, query block): QB = 64/G consecutive query tokens x the G
// query heads of the group = 64 rows.  Thread t: row t/4; when scoring it
// owns keys 8*(t%4) .. +7 of the tile, when accumulating P V the 32 output
// dims 32*(t%4) .. (HD = 128; proportionally fewer for smaller HD).
template <int HD, int G>
__global__ void __launch_bounds__(PA_T) pattn_kernel(const float* q, float* o, const __half* k_pool,
                                                     const __half* v_pool, const int32_t* ptab, int n_kv,
                                                     int page_tokens, int T, int pos0) {
  constexpr int QB = PA_ROWS / G;
  constexpr int DPT = HD / 4;           // output dims per thread
  constexpr int KROW = PA_KROW<HD>;
  extern __shared__ float4 pa_smem[];
  float (*s_q)[HD] = reinterpret_cast<float (*)[HD]>(pa_smem);
  __half (*s_k)[KROW] = reinterpret_cast<__half (*)[KROW]>(&s_q[PA_ROWS][0]);
  __half (*s_v)[HD] = reinterpret_cast<__half (*)[HD]>(&s_k[PA_KT][0]);
  float (*s_p)[PA_KT + 1] = reinterpret_cast<float (*)[PA_KT + 1]>(&s_v[PA_KT][0]);
  const int kvh = blockIdx.x, qb = blockIdx.y;
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  const int qi = r / G, hh = r % G;
  const int t_tok = qb * QB + qi;             // query token index within the prefill
  const bool row_ok = t_tok < T;
  const int qpos = pos0 + t_tok;
  const float scale = 1.0f / sqrtf((float)HD);
  const int n_heads = n_kv * G;
  for (int i = tid; i < PA_ROWS * HD; i += PA_T) {
    const int rr = i / HD, d = i % HD;
    const int tt = qb * QB + rr / G;
    s_q[rr][d] = tt < T ? q[((size_t)tt * n_heads + (size_t)kvh * G + rr % G) * HD + d] * scale : 0.f;
  }
  float m_run = -INFINITY, l_run = 0.f, acc[DPT];
#pragma unroll
  for (int e = 0; e < DPT; ++e) acc[e] = 0.f;
  const int last_pos = pos0 + min(T, (qb + 1) * QB) - 1;  // newest query of the block
  const int n_tiles = last_pos / PA_KT + 1;
  for (int jt = 0; jt < n_tiles; ++jt) {
    __syncthreads();  // previous tile's K/V/P consumed
    // K and V tile: 32 keys x HD fp16, 16-byte chunks
    constexpr int CH = PA_KT * HD / 8;
    for (int c = tid; c < CH; c += PA_T) {
      const int kk = c / (HD / 8), part = c % (HD / 8);
      const int kp = jt * PA_KT + kk;
      uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
      if (kp <= last_pos) {
        const int page = ptab[kp / page_tokens];
        const size_t off = (((size_t)page * n_kv + kvh) * page_tokens + (kp % page_tokens)) * HD + part * 8;
        kv4 = *reinterpret_cast<const uint4*>(k_pool + off);
        vv4 = *reinterpret_cast<const uint4*>(v_pool + off);
      }
      *reinterpret_cast<uint4*>(&s_k[kk][part * 8]) = kv4;
      *reinterpret_cast<uint4*>(&s_v[kk][part * 8]) = vv4;
    }
    __syncthreads();
    // scores of row r for keys 8*sub .. +7
    float sc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) sc[u] = 0.f;
    for (int d = 0; d < HD; d += 4) {
      const float4 qv = *reinterpret_cast<const float4*>(&s_q[r][d]);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const __half2* kr = reinterpret_cast<const __half2*>(&s_k[8 * sub + u][d]);
        const float2 k01 = __half22float2(kr[0]), k23 = __half22float2(kr[1]);
        sc[u] = fmaf(qv.x, k01.x, fmaf(qv.y, k01.y, fmaf(qv.z, k23.x, fmaf(qv.w, k23.y, sc[u]))));
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int kp = jt * PA_KT + 8 * sub + u;
      if (!row_ok || kp > qpos) sc[u] = -INFINITY;  // causal mask
      mx = fmaxf(mx, sc[u]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    float ps = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float p = m_new == -INFINITY ? 0.f : expf(sc[u] - m_new);
      s_p[r][8 * sub + u] = p;
      ps += p;
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    const float al = m_new == -INFINITY ? 1.f : expf(m_run - m_new);
    l_run = l_run * al + ps;
    m_run = m_new;
    __syncthreads();
    // acc[r][dims] = al * acc + sum_k p[r][k] v[k][dims]
#pragma unroll
    for (int e = 0; e < DPT; ++e) acc[e] *= al;
    for (int kk = 0; kk < PA_KT; ++kk) {
      const float p = s_p[r][kk];
      const __half2* vr = reinterpret_cast<const __half2*>(&s_v[kk][sub * DPT]);
#pragma unroll
      for (int e = 0; e < DPT / 2; ++e) {
        const float2 vf = __half22float2(vr[e]);
        acc[2 * e] = fmaf(p, vf.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(p, vf.y, acc[2 * e + 1]);
      }
    }
  }
  if (row_ok) {
    const float inv = 1.0f / l_run;
    float* orow = o + ((size_t)t_tok * n_heads + (size_t)kvh * G + hh) * HD + sub * DPT;
#pragma unroll
    for (int e = 0; e < DPT; ++e) orow[e] = acc[e] * inv;
  }
}

using PaFn = void (*)(const float*, float*, const __half*, const __half*, const int32_t*, int, int, int, int);

template <int HD>
PaFn pa_pick(int g) {
  switch (g) {
    case 1: return pattn_kernel<HD, 1>;
    case 2: return pattn_kernel<HD, 2>;
    case 4: return pattn_kernel<HD, 4>;
    case 8: return pattn_kernel<HD, 8>;
    case 16: return pattn_kernel<HD, 16>;
  }
  return nullptr;
}

// one prompt token per block: x[t] = dequantised embedding row tokens[t]
__global__ void embed_rows_kernel(const MatDev emb, int wtype, const int32_t* tokens, int vocab, float* x, int ldx,
                                  int32_t* status) {
  int tok = tokens[blockIdx.x];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0 && status) atomicOr(status, kBadToken);
    tok = 0;
  }
  float* xr = x + (size_t)blockIdx.x * ldx;
  for (int c = threadIdx.x * 4; c < emb.cols; c += blockDim.x * 4) {
    const float d = __half2float(emb.d[(size_t)tok * emb.ds + (c >> 5)]);
    uint32_t u;
    if (wtype == 8) {
      u = *reinterpret_cast<const uint32_t*>(emb.qs + (size_t)tok * emb.nb * 32 + c);
    } else {
      const uint32_t b = *reinterpret_cast<const uint32_t*>(emb.qs + ((size_t)tok * emb.nb + (c >> 5)) * 16 + (c & 15));
      u = (c & 31) < 16 ? (b & 0x0F0F0F0Fu) : ((b >> 4) & 0x0F0F0F0Fu);
    }
    const float bias = wtype == 8 ? 8388736.0f : 8388616.0f;
    float4 v;
    v.x = d * (mag_byte(u, 0) - bias);
    v.y = d * (mag_byte(u, 1) - bias);
    v.z = d * (mag_byte(u, 2) - bias);
    v.w = d * (mag_byte(u, 3) - bias);
    *reinterpret_cast<float4*>(xr + c) = v;
  }
}

}  // namespace

cudaError_t prefill_setup_attributes() {
  for (int g : {1, 2, 4, 8, 16}) {
    const std::pair<PaFn, int> fs[] = {{pa_pick<32>(g), pa_smem_bytes<32>()},
                                       {pa_pick<64>(g), pa_smem_bytes<64>()},
                                       {pa_pick<128>(g), pa_smem_bytes<128>()}};
    for (const auto& f : fs) {
      cudaError_t err = cudaFuncSetAttribute(f.first, cudaFuncAttributeMaxDynamicSharedMemorySize, f.second);
      if (err != cudaSuccess) return err;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_embed_rows(const MatDev& emb, int wtype, const int32_t* tokens, int T, int vocab, float* x, int ldx,
                              int32_t* status, cudaStream_t s) {
  if (emb.cols % 4) return cudaErrorInvalidValue;
  embed_rows_kernel<<<T, 256, 0, s>>>(emb, wtype, tokens, vocab, x, ldx, status);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows(const float* x, int T, int H, int ldx, const float* g, float eps, __half* out,
                                __half* out_lo, int ldo, cudaStream_t s) {
  if (H % 4 || ldx % 4 || ldo % 4 || !out_lo) return cudaErrorInvalidValue;
  rmsnorm_rows_kernel<<<T, row_threads(H / 4), 0, s>>>(x, H, ldx, g, eps, out, out_lo, ldo);
  return cudaGetLastError();
}

cudaError_t launch_to_f16_rows(const float* x, int T, int cols, int ldx, __half* out, __half* out_lo, int ldo,
                               cudaStream_t s) {
  if (cols % 4 || ldx % 4 || ldo % 4 || !out_lo) return cudaErrorInvalidValue;
  to_f16_rows_kernel<<<T, row_threads(cols / 4), 0, s>>>(x, cols, ldx, out, out_lo, ldo);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_rows(const float* qkv, int T, int ld, int q_rows, int kv_rows, const KvView& kv, int seq,
                                int pos0, const float2* rope_cs, int rope_len, float* q_out, int32_t* status,
                                cudaStream_t s) {
  rope_kv_rows_kernel<<<T, row_threads((q_rows + 2 * kv_rows) / 2), 0, s>>>(
      qkv, ld, q_rows, kv_rows, kv, seq, pos0, nullptr, nullptr, rope_cs, rope_len, q_out, status);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_batch(const float* qkv, int n, int ld, int q_rows, int kv_rows, const KvView& kv,
                                 const int32_t* seqs, const int32_t* poss, const float2* rope_cs, int rope_len,
                                 float* q_out, int32_t* status, cudaStream_t s) {
  rope_kv_rows_kernel<<<n, row_threads((q_rows + 2 * kv_rows) / 2), 0, s>>>(qkv, ld, q_rows, kv_rows, kv, 0, 0, seqs,
                                                                              poss, rope_cs, rope_len, q_out, status);
  return cudaGetLastError();
}

cudaError_t launch_pattn(const float* q, float* o, const KvView& kv, const int32_t* ptab_row, int n_heads, int T,
                         int pos0, cudaStream_t s) {
  const int g = n_heads / kv.n_kv;
  const int qb = PA_ROWS / g;
  if (qb < 1) return cudaErrorInvalidValue;
  dim3 grid(kv.n_kv, (T + qb - 1) / qb);
  PaFn f = nullptr;
  int smem = 0;
  switch (kv.head_dim) {
    case 32: f = pa_pick<32>(g), smem = pa_smem_bytes<32>(); break;
    case 64: f = pa_pick<64>(g), smem = pa_smem_bytes<64>(); break;
    case 128: f = pa_pick<128>(g), smem = pa_smem_bytes<128>(); break;
  }
  if (!f) return cudaErrorInvalidValue;
  f<<<grid, PA_T, smem, s>>>(q, o, kv.k_pool, kv.v_pool, ptab_row, kv.n_kv, kv.page_tokens, T, pos0);
  return cudaGetLastError();
}

}  // namespace dls
