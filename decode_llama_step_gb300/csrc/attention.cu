// Split-K ("flash-decoding") GQA attention of one query position over an
// fp16 paged KV cache: the causal softmax of the decode step with the mask
// inside the kernel (engine page, section 4.4: causal softmax with the mask
// fused; section 1: GQA, KV cache).
//
// Grid (n_kv * S, rows): CTA (kv head, split s) reads one contiguous range of
// positions of that KV head once and serves all g = n_heads / n_kv query
// heads of the group from it.  Positions go in 32-token tiles that never
// cross a page; V of a tile is loaded while its scores are computed.  Each
// CTA keeps an online softmax (running max m, sum l, unnormalised o) per
// head, writes (m, l, o) to scratch, and the last CTA of a (row, kv head) to
// finish combines the S partials in split order (deterministic) and resets
// the arrival counter to zero for the next launch.
#include <math.h>

#include "../../include/dls.h"
#include "kernels.h"

namespace dls {

namespace {

constexpr int TILE = 32;
constexpr int NT = 128;
constexpr int kMaxG = 16;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int NSTAGE = 4;   // K/V tile ring depth

template <int HD>
__global__ void __launch_bounds__(NT) attn_kernel(const AttnArgs a) {
  constexpr int DPL = HD / 32;            // dims per lane when scoring
  constexpr int HPT = NT / HD;            // head slots per pass (threads share d)
  constexpr int OPT = (kMaxG + HPT - 1) / HPT;
  constexpr int TILE_B = TILE * HD * 2;   // bytes of one K (or V) tile
  constexpr int kMaxSplits = 128;
  extern __shared__ __align__(128) uint8_t s_dyn[];
  // K/V tile ring in dynamic shared memory: [NSTAGE][K|V][TILE*HD] halves
  auto kv_tile = [&](int st, int which) { return reinterpret_cast<__half*>(s_dyn) + ((size_t)st * 2 + which) * TILE * HD; };
  __shared__ __align__(16) float s_q[kMaxG * HD];
  __shared__ float s_s[kMaxG][TILE];
  __shared__ float s_alpha[kMaxG], s_m[kMaxG], s_l[kMaxG];
  __shared__ __align__(8) uint64_t s_full[NSTAGE];
  __shared__ float s_w[kMaxG][kMaxSplits];
  __shared__ int s_last;

  const int g = a.n_heads / a.n_kv;
  const int S = a.n_splits;
  const int kvh = blockIdx.x / S, sp = blockIdx.x - kvh * S;
  const int brel = blockIdx.y, b = a.row0 + brel;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = tid % HD, hslot = tid / HD;
  const int pt = a.page_tokens;

  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(smem_u32(&s_full[i]), 1);
    mbar_fence_init();
  }
  griddep_wait();
  griddep_launch();

  int n = a.len[b] + a.len_add;
  if (n < 1 || n > a.max_len) {
    if (a.status && tid == 0) atomicOr(a.status, kBadPos);
    n = n < 1 ? 1 : a.max_len;
  }
  const int ptrow = a.pt_row ? a.pt_row[b] : b;
  const int32_t* ptab = a.page_table + (size_t)ptrow * a.max_pages;
  int per = (n + S - 1) / S;
  per = (per + TILE - 1) / TILE * TILE;
  const int t0 = sp * per, t1 = min(n, t0 + per);
  const int ntiles = t1 > t0 ? (t1 - t0 + TILE - 1) / TILE : 0;

  // thread 0 issues the K and V copies of a tile (a tile never crosses a page)
  auto issue = [&](int i) -> bool {
    const int t = t0 + i * TILE;
    const int nt = min(TILE, t1 - t);
    const int page = ptab[t / pt];
    const uint32_t bar = smem_u32(&s_full[i % NSTAGE]);
    if (page < 0) {
      mbar_arrive(bar);  // complete the phase with nothing copied
      return false;
    }
    const size_t base = (((size_t)page * a.n_kv + kvh) * pt + (t % pt)) * HD;
    const uint32_t bytes = (uint32_t)nt * HD * 2;
    mbar_expect_tx(bar, 2 * bytes);
    bulk_g2s(smem_u32(kv_tile(i % NSTAGE, 0)), a.k_pool + base, bytes, bar);
    bulk_g2s(smem_u32(kv_tile(i % NSTAGE, 1)), a.v_pool + base, bytes, bar);
    return true;
  };
  __syncthreads();  // barriers initialised
  if (tid == 0) {
    bool ok = true;
    for (int i = 0; i < min(NSTAGE, ntiles); ++i) ok &= issue(i);
    if (!ok && a.status) atomicOr(a.status, kBadPage);
  }

  const float scale = 1.0f / sqrtf((float)HD);
  const float* qrow = a.q + ((size_t)brel * a.n_heads + (size_t)kvh * g) * HD;
  for (int i = tid; i < g * HD; i += NT) s_q[i] = qrow[i] * scale;
  if (tid < g) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  float oacc[OPT];
#pragma unroll
  for (int k = 0; k < OPT; ++k) oacc[k] = 0.f;
  __syncthreads();

  bool failed = false;
  for (int i = 0; i < ntiles; ++i) {
    const int t = t0 + i * TILE;
    const int nt = min(TILE, t1 - t);
    if (!mbar_wait(smem_u32(&s_full[i % NSTAGE]), (i / NSTAGE) & 1)) failed = true;
    const __half* kt = kv_tile(i % NSTAGE, 0);
    const __half* vt = kv_tile(i % NSTAGE, 1);
    // scores: warp w scores tokens w, w+4, ...; lanes split the head dim
    for (int j = warp; j < nt; j += NT / 32) {
      float kf[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) kf[e] = __half2float(kt[j * HD + lane * DPL + e]);
      for (int h = 0; h < g; ++h) {
        float p = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) p = fmaf(s_q[h * HD + lane * DPL + e], kf[e], p);
        p = warp_sum(p);
        if (lane == 0) s_s[h][j] = p;
      }
    }
    __syncthreads();
    // online softmax update, one warp per head
    for (int h = warp; h < g; h += NT / 32) {
      const float sv = lane < nt ? s_s[h][lane] : -INFINITY;
      const float mx = warp_max(sv);
      const float m_old = s_m[h];
      const float m_new = fmaxf(m_old, mx);
      const float p = lane < nt ? expf(sv - m_new) : 0.f;
      const float ps = warp_sum(p);
      s_s[h][lane] = p;
      if (lane == 0) {
        const float al = expf(m_old - m_new);  // 0 on the first tile (m_old = -inf)
        s_alpha[h] = al;
        s_l[h] = s_l[h] * al + ps;
        s_m[h] = m_new;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
      const int h = hslot + k * HPT;
      if (h < g) {
        float o = oacc[k] * s_alpha[h];
        for (int j = 0; j < nt; ++j) o = fmaf(s_s[h][j], __half2float(vt[j * HD + d]), o);
        oacc[k] = o;
      }
    }
    __syncthreads();  // slot i % NSTAGE is free again
    if (tid == 0 && i + NSTAGE < ntiles && !issue(i + NSTAGE) && a.status) atomicOr(a.status, kBadPage);
  }
  if (failed && a.status && tid == 0) atomicOr(a.status, kTimeout);

  // ---- partials to scratch
  const size_t slot = ((size_t)brel * a.n_kv + kvh) * S + sp;
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int h = hslot + k * HPT;
    if (h < g) a.part_o[(slot * g + h) * HD + d] = oacc[k];
  }
  if (tid < g) reinterpret_cast<float2*>(a.part_ml)[slot * g + tid] = make_float2(s_m[tid], s_l[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[(size_t)brel * a.n_kv + kvh], 1);
    s_last = prev == S - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of this (row, kv head): combine the S splits
  // weights w_s = exp(m_s - M) / sum_s l_s exp(m_s - M), one warp per head
  const size_t slot0 = ((size_t)brel * a.n_kv + kvh) * S;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  for (int h = warp; h < g; h += NT / 32) {
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(&ml[(slot0 + s) * g + h]).x);
    M = warp_max(M);
    float den = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float2 v = __ldcg(&ml[(slot0 + s) * g + h]);
      const float e = v.y > 0.f ? expf(v.x - M) : 0.f;  // empty split: weight 0
      s_w[h][s] = e;
      den = fmaf(v.y, e, den);
    }
    den = warp_sum(den);
    for (int s = lane; s < S; s += 32) s_w[h][s] /= den;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int h = hslot + k * HPT;
    if (h >= g) continue;
    float acc = 0.f;
    const float* po = a.part_o + (slot0 * g + h) * HD + d;
#pragma unroll 8
    for (int s = 0; s < S; ++s) acc = fmaf(s_w[h][s], __ldcg(po + (size_t)s * g * HD), acc);
    a.o[((size_t)brel * a.n_heads + (size_t)kvh * g + h) * HD + d] = acc;
  }
  if (tid == 0) a.counters[(size_t)brel * a.n_kv + kvh] = 0;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t attn_workspace_bytes(int rows, int n_heads, int n_kv, int head_dim, int n_splits) {
  const int g = n_heads / n_kv;
  const size_t slots = (size_t)rows * n_kv * n_splits;
  return align256((size_t)rows * n_kv * sizeof(int)) + align256(slots * g * head_dim * sizeof(float)) +
         align256(slots * g * 2 * sizeof(float));
}

void attn_workspace_carve(void* ws, int rows, int n_heads, int n_kv, int head_dim, int n_splits, float** part_o,
                          float** part_ml, int** counters) {
  const int g = n_heads / n_kv;
  const size_t slots = (size_t)rows * n_kv * n_splits;
  char* p = static_cast<char*>(ws);
  *counters = reinterpret_cast<int*>(p);  // counters first, so "zero the head" clears them
  p += align256((size_t)rows * n_kv * sizeof(int));
  *part_o = reinterpret_cast<float*>(p);
  p += align256(slots * g * head_dim * sizeof(float));
  *part_ml = reinterpret_cast<float*>(p);
}

int attn_default_splits(int rows, int n_kv, int num_sms, int max_len) {
  int s = (2 * num_sms + rows * n_kv - 1) / (rows * n_kv);
  const int cap = (max_len + TILE - 1) / TILE;
  if (s > cap) s = cap;
  if (s > 128) s = 128;  // combine weights live in shared memory
  if (s < 1) s = 1;
  return s;
}

template <int HD>
cudaError_t attn_attr() {
  static bool done = false;  // one process-wide attribute per instantiation
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       NSTAGE * 2 * TILE * HD * 2);
  done = e == cudaSuccess;
  return e;
}

cudaError_t launch_attention(const AttnArgs& a, int rows, cudaStream_t s, bool pdl) {
  if (a.n_splits > 128 || a.n_splits < 1) return cudaErrorInvalidValue;
  cudaError_t e = a.head_dim == 32 ? attn_attr<32>() : a.head_dim == 64 ? attn_attr<64>() : attn_attr<128>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_kv * a.n_splits, rows);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = NSTAGE * 2 * TILE * a.head_dim * 2;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (a.head_dim) {
    case 32: return cudaLaunchKernelEx(&cfg, attn_kernel<32>, a);
    case 64: return cudaLaunchKernelEx(&cfg, attn_kernel<64>, a);
    case 128: return cudaLaunchKernelEx(&cfg, attn_kernel<128>, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dls

// ---- standalone C-ABI op ---------------------------------------------------------

extern "C" size_t dls_attention_workspace_bytes(int32_t n_batch, int32_t n_heads, int32_t n_kv_heads,
                                                int32_t head_dim, int32_t n_splits) {
  if (n_batch < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || n_splits < 1) return 0;
  return dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits);
}

extern "C" int dls_attention_decode(const float* q, const void* k_pages, const void* v_pages,
                                    const int32_t* page_table, const int32_t* lengths, float* o, void* workspace,
                                    size_t workspace_bytes, int32_t n_batch, int32_t n_heads, int32_t n_kv_heads,
                                    int32_t head_dim, int32_t page_tokens, int32_t max_pages, int32_t n_splits,
                                    void* cuda_stream) {
  if (!q || !k_pages || !v_pages || !page_table || !lengths || !o || !workspace) return DLS_ERR_ARG;
  if (n_splits > 128) return DLS_ERR_ARG;
  if (n_batch < 1 || n_kv_heads < 1 || n_heads < 1 || n_heads % n_kv_heads || n_heads / n_kv_heads > dls::kMaxG ||
      (head_dim != 32 && head_dim != 64 && head_dim != 128) || page_tokens < 32 || page_tokens % 32 ||
      max_pages < 1)
    return DLS_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return DLS_ERR_CUDA;
  const int max_len = page_tokens * max_pages;
  if (n_splits <= 0) n_splits = dls::attn_default_splits(n_batch, n_kv_heads, sms, max_len);
  if (workspace_bytes < dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits))
    return DLS_ERR_ARG;
  dls::AttnArgs a = {};
  a.q = q;
  a.o = o;
  a.k_pool = static_cast<const __half*>(k_pages);
  a.v_pool = static_cast<const __half*>(v_pages);
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.pt_row = nullptr;
  a.len = lengths;
  a.len_add = 0;
  a.n_heads = n_heads;
  a.n_kv = n_kv_heads;
  a.head_dim = head_dim;
  a.page_tokens = page_tokens;
  a.n_splits = n_splits;
  a.row0 = 0;
  a.status = nullptr;
  a.max_len = max_len;
  dls::attn_workspace_carve(workspace, n_batch, n_heads, n_kv_heads, head_dim, n_splits, &a.part_o, &a.part_ml,
                            &a.counters);
  cudaError_t e = dls::launch_attention(a, n_batch, static_cast<cudaStream_t>(cuda_stream), false);
  return e == cudaSuccess ? DLS_OK : DLS_ERR_CUDA;
}
