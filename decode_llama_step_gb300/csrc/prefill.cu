// Prefill: the same layer math for T prompt tokens at once (SwarmKV page,
// section 2: prefill runs every prompt token through every layer once and
// fills the KV cache; its cost grows with the prompt length, so it is where
// the dense tensor-core work is).
//
//  * pgemm_kernel: D[m, t] = sum_k W[m, k] X[t, k] on tcgen05 (kind::f16,
//    M = 128 weight rows, N = 128 tokens, K = 16 per instruction, fp32
//    accumulators in tensor memory).  Loader warps dequantise the Q8_0/Q4_0
//    weight tile (fp16(d * q), one rounding) and copy the fp16 token tile
//    into 128-byte-swizzled shared memory; one thread issues the MMAs and
//    commits them to the stage's "empty" barrier; four epilogue warps read the
//    accumulators back (tcgen05.ld) and store, add to the residual, or apply
//    SwiGLU to interleaved (gate, up) row pairs.
//  * pattn_kernel: causal attention of T query tokens over the sequence's
//    paged fp16 cache, flash style on CUDA cores (64 query-head rows per CTA,
//    32-key tiles, online softmax in registers).
//  * row kernels: RMSNorm -> fp16, RoPE + fp16 K/V append, fp32 -> fp16.
#include <math.h>

#include <utility>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int PBM = 128, PBN = 128, PBK = 64, PNST = 4;
constexpr int PTHREADS = 256;               // warp 0: MMA issue; warps 1-7: loaders; 4-7: epilogue
constexpr int NLOAD = PTHREADS - 32;        // loader threads
constexpr int kTileA = PBM * PBK * 2;       // 16 KB
constexpr int kTileB = PBN * PBK * 2;       // 16 KB
constexpr int kStageP = kTileA + kTileB;
constexpr int kChunks = PBM * PBK / 8;      // 16-byte chunks per tile (1024)
constexpr int kCPT = (kChunks + NLOAD - 1) / NLOAD;  // chunks per loader thread
constexpr uint64_t kWaitNsP = 2000000000ull;

struct PgShared {
  uint64_t full[PNST];
  uint64_t empty[PNST];
  uint64_t done;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 4) __nanosleep(32);
    if ((i & 63) == 0) {
      if (*(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsP) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

// 8 weights (row, cols col..col+7) dequantised to fp16(d * q), packed
template <int WT>
__device__ __forceinline__ uint4 dequant8(uint2 u, float d, int e) {
  float v[8];
  if (WT == 8) {  // bytes hold q + 128
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = d * (mag_byte(u.x, i) - 8388736.0f);
      v[4 + i] = d * (mag_byte(u.y, i) - 8388736.0f);
    }
  } else {  // 8 bytes of the block; low nibbles for elements 0-15, high for 16-31
    const uint32_t lo = e < 16 ? (u.x & 0x0F0F0F0Fu) : ((u.x >> 4) & 0x0F0F0F0Fu);
    const uint32_t hi = e < 16 ? (u.y & 0x0F0F0F0Fu) : ((u.y >> 4) & 0x0F0F0F0Fu);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = d * (mag_byte(lo, i) - 8388616.0f);
      v[4 + i] = d * (mag_byte(hi, i) - 8388616.0f);
    }
  }
  uint4 r;
  __half2 h;
  h = __floats2half2_rn(v[0], v[1]);
  r.x = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2half2_rn(v[2], v[3]);
  r.y = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2half2_rn(v[4], v[5]);
  r.z = *reinterpret_cast<uint32_t*>(&h);
  h = __floats2half2_rn(v[6], v[7]);
  r.w = *reinterpret_cast<uint32_t*>(&h);
  return r;
}

// shared offset of 16-byte chunk j of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

template <int WT, int EPI>
__global__ void __launch_bounds__(PTHREADS, 1) pgemm_kernel(const PgArgs a) {
  extern __shared__ uint8_t psmem[];
  const uint32_t raw = smem_u32(psmem);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t sbase = raw + pad;                       // 1024-aligned stage area
  PgShared& sh = *reinterpret_cast<PgShared*>(psmem + pad + PNST * kStageP);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev& w = a.w;
  const int m0 = blockIdx.x * PBM, n0 = blockIdx.y * PBN;
  const int kpad = w.nb * 32;
  const int nk = (kpad + PBK - 1) / PBK;
  const size_t rb = WT == 8 ? (size_t)w.nb * 32 : (size_t)w.nb * 16;

  if (warp == 0) {
    tmem_alloc(smem_u32(&sh.tmem), PBN);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < PNST; ++s) {
      mbar_init(smem_u32(&sh.full[s]), PTHREADS / 32 - 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    mbar_init(smem_u32(&sh.done), 1);
    sh.abort = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  constexpr uint32_t idesc = umma_idesc_f16(PBM, PBN);

  if (warp == 0) {
    // ---------------- MMA issue (one thread)
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % PNST;
        if (!pwait(smem_u32(&sh.full[s]), (kt / PNST) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t sa = sbase + s * kStageP, sb = sa + kTileA;
#pragma unroll
        for (int ks = 0; ks < PBK / 16; ++ks)
          umma_f16(tmem, umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + ks * 32), idesc, (kt | ks) != 0);
        umma_commit(smem_u32(&sh.empty[s]));
      }
      umma_commit(smem_u32(&sh.done));
    }
    __syncwarp();
  } else {
    // ---------------- loaders: weight tile (dequantised) and token tile
    const int lt = tid - 32;
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % PNST;
      const int k0 = kt * PBK;
      const uint32_t sa = sbase + s * kStageP, sb = sa + kTileA;
      // global loads first (registers), then wait for the slot
      uint2 cu[kCPT];
      float cd[kCPT];
      uint4 xv[kCPT];
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = lt + i * NLOAD;
        const int r = c >> 3, j = c & 7;
        const int col = k0 + 8 * j;
        cu[i] = make_uint2(0, 0);
        cd[i] = 0.f;
        xv[i] = make_uint4(0, 0, 0, 0);
        if (c < kChunks) {
          const int row = m0 + r;
          if (row < w.rows && col < kpad) {
            cd[i] = __half2float(w.d[(size_t)row * w.ds + (col >> 5)]);
            const size_t off = WT == 8 ? (size_t)row * rb + col : (size_t)row * rb + (col >> 5) * 16 + (col & 15);
            cu[i] = *reinterpret_cast<const uint2*>(w.qs + off);
          }
          const int tok = n0 + r;
          if (tok < a.T && col < kpad) xv[i] = *reinterpret_cast<const uint4*>(a.x + (size_t)tok * a.kx + col);
        }
      }
      if (kt >= PNST && !pwait(smem_u32(&sh.empty[s]), ((kt / PNST) - 1) & 1, &sh.abort)) break;
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = lt + i * NLOAD;
        if (c < kChunks) {
          const int r = c >> 3, j = c & 7;
          sts128(sa + swz(r, j), dequant8<WT>(cu[i], cd[i], (k0 + 8 * j) & 31));
          sts128(sb + swz(r, j), xv[i]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.full[s]));
    }
  }

  // ---------------- epilogue: warps 4-7 read TMEM lanes 32*(warp-4) ..
  if (warp >= 4) {
    const bool waited = pwait(smem_u32(&sh.done), 0, &sh.abort);
    const bool ok = __all_sync(0xffffffffu, waited && !*(volatile int*)&sh.abort);
    tc_fence_after();
    const int m = m0 + (warp - 4) * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)((warp - 4) * 32) << 16);
    for (int c0 = 0; c0 < PBN; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(taddr + c0, r);
      tmem_wait_ld();
      if (!ok) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = n0 + c0 + j;
        const float v = __uint_as_float(r[j]);
        if (EPI == EPI_SWIGLU) {
          const float up = __shfl_down_sync(0xffffffffu, v, 1);
          if ((lane & 1) == 0 && t < a.T && m + 1 < w.rows)
            a.h[(size_t)t * a.ldh + (m >> 1)] = __float2half_rn(silu(v) * up);
        } else if (t < a.T && m < w.rows) {
          float* dst = a.y + (size_t)t * a.ldy + m;
          if (EPI == EPI_RESID) *dst += v;
          else *dst = v;
        }
      }
    }
    if (!ok && a.status && lane == 0) atomicOr(a.status, kTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, PBN);
  }
}

using PgFn = void (*)(const PgArgs);

template <int WT>
PgFn pg_pick(int epi) {
  switch (epi) {
    case EPI_STORE: return pgemm_kernel<WT, EPI_STORE>;
    case EPI_RESID: return pgemm_kernel<WT, EPI_RESID>;
    case EPI_SWIGLU: return pgemm_kernel<WT, EPI_SWIGLU>;
  }
  return nullptr;
}

// ---------------------------------------------------------------- row kernels

// out[t] = fp16(rmsnorm(x[t]) * g), zero-padded to ldo columns
__global__ void rmsnorm_rows_kernel(const float* x, int H, int ldx, const float* g, float eps, __half* out, int ldo) {
  const float* xr = x + (size_t)blockIdx.x * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  const float rs = 1.0f / sqrtf(t / (float)H + eps);
  __half* o = out + (size_t)blockIdx.x * ldo;
  for (int i = threadIdx.x; i < ldo; i += blockDim.x) o[i] = __float2half_rn(i < H ? xr[i] * rs * g[i] : 0.f);
}

__global__ void to_f16_rows_kernel(const float* x, int cols, int ldx, __half* out, int ldo) {
  const float* xr = x + (size_t)blockIdx.x * ldx;
  __half* o = out + (size_t)blockIdx.x * ldo;
  for (int i = threadIdx.x; i < ldo; i += blockDim.x) o[i] = __float2half_rn(i < cols ? xr[i] : 0.f);
}

// RoPE on the q and k rows of token t at position pos0 + t; q -> q_out
// (fp32), k and v -> the sequence's pages (fp16)
__global__ void rope_kv_rows_kernel(const float* qkv, int ld, int q_rows, int kv_rows, KvView kv, int seq, int pos0,
                                    const float2* rope_cs, int rope_len, float* q_out, int32_t* status) {
  const int t = blockIdx.x, pos = pos0 + t;
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

int pgemm_smem_bytes() { return PNST * kStageP + (int)sizeof(PgShared) + 1024; }

cudaError_t pgemm_setup_attributes() {
  for (int e : {EPI_STORE, EPI_RESID, EPI_SWIGLU}) {
    for (PgFn f : {pg_pick<8>(e), pg_pick<4>(e)}) {
      cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, pgemm_smem_bytes());
      if (err != cudaSuccess) return err;
    }
  }
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

cudaError_t launch_pgemm(int wtype, int epi, const PgArgs& a, cudaStream_t s) {
  if (a.kx % 8 || a.kx < a.w.nb * 32 || a.T < 1) return cudaErrorInvalidValue;
  PgFn f = wtype == 8 ? pg_pick<8>(epi) : pg_pick<4>(epi);
  if (!f) return cudaErrorInvalidValue;
  dim3 grid((a.w.rows + PBM - 1) / PBM, (a.T + PBN - 1) / PBN);
  f<<<grid, PTHREADS, pgemm_smem_bytes(), s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows(const float* x, int T, int H, int ldx, const float* g, float eps, __half* out, int ldo,
                                cudaStream_t s) {
  rmsnorm_rows_kernel<<<T, 256, 0, s>>>(x, H, ldx, g, eps, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_to_f16_rows(const float* x, int T, int cols, int ldx, __half* out, int ldo, cudaStream_t s) {
  to_f16_rows_kernel<<<T, 256, 0, s>>>(x, cols, ldx, out, ldo);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_rows(const float* qkv, int T, int ld, int q_rows, int kv_rows, const KvView& kv, int seq,
                                int pos0, const float2* rope_cs, int rope_len, float* q_out, int32_t* status,
                                cudaStream_t s) {
  rope_kv_rows_kernel<<<T, 256, 0, s>>>(qkv, ld, q_rows, kv_rows, kv, seq, pos0, rope_cs, rope_len, q_out, status);
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
