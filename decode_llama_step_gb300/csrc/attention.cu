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
#include <stdlib.h>

#include <algorithm>

#include <mutex>

#include "../../include/dls.h"
#include "kernels.h"

namespace dls {

namespace {

constexpr int TILE = 32;   // tokens per tile: one lane per token when scoring
constexpr int NW = 8;      // warps per CTA
constexpr int NT = 32 * NW;
constexpr int kMaxG = 16;
constexpr int kMaxSplits = 128;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp's online-softmax update over one 32-token tile staged in shared
// memory (K rows at kt, V rows at vt, head_dim halves each), for HPW query
// heads whose pre-scaled q lies at q2 (float2 words, HD/2 per head).  Scores
// take one lane per token (the head dimension walked from a lane-dependent
// start, so the 32 lanes hit 32 different banks) in two accumulator chains;
// P V gives each lane HD/32 output dimensions, unrolled over the tile with
// rows past nt zeroed (their p is 0 as well).
template <int HD, int HPW>
__device__ __forceinline__ void tile_update(const __half* kt, const __half* vt, const float2* q2, int nt, int lane,
                                            float (&m_run)[HPW], float (&l_run)[HPW], float (&o)[HPW][HD / 32]) {
  constexpr int DPL = HD / 32, W2 = HD / 2;
  float sc[HPW];
  {
    float2 acc[HPW][2];
#pragma unroll
    for (int h = 0; h < HPW; ++h) acc[h][0] = acc[h][1] = make_float2(0.f, 0.f);
    const __half2* krow = reinterpret_cast<const __half2*>(kt + lane * HD);
#pragma unroll 8
    for (int w2 = 0; w2 < W2; ++w2) {
      const int wi = (w2 + lane) & (W2 - 1);
      const float2 kf = __half22float2(krow[wi]);
#pragma unroll
      for (int h = 0; h < HPW; ++h) acc[h][w2 & 1] = __ffma2_rn(kf, q2[h * W2 + wi], acc[h][w2 & 1]);
    }
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      const float2 a = __fadd2_rn(acc[h][0], acc[h][1]);
      sc[h] = lane < nt ? a.x + a.y : -INFINITY;
    }
  }
  float p[HPW];
#pragma unroll
  for (int h = 0; h < HPW; ++h) {
    const float m_new = fmaxf(m_run[h], warp_max(sc[h]));
    p[h] = lane < nt ? expf(sc[h] - m_new) : 0.f;
    const float al = expf(m_run[h] - m_new);  // 0 on the warp's first tile
    l_run[h] = l_run[h] * al + warp_sum(p[h]);
    m_run[h] = m_new;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] *= al;
  }
  const __half* vl = vt + lane * DPL;
#pragma unroll
  for (int j = 0; j < TILE; ++j) {
    float vf[DPL];
    if (DPL == 4) {
      uint2 raw = *reinterpret_cast<const uint2*>(vl + j * HD);
      if (j >= nt) raw = make_uint2(0u, 0u);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      vf[0] = v01.x;
      vf[1] = v01.y;
      vf[2 % DPL] = v23.x;
      vf[3 % DPL] = v23.y;
    } else {
#pragma unroll
      for (int e = 0; e < DPL; ++e) vf[e] = j < nt ? __half2float(vl[j * HD + e]) : 0.f;
    }
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      const float pj = __shfl_sync(0xffffffffu, p[h], j);
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pj, vf[e], o[h][e]);
    }
  }
}

// CTA (kv head, split sp) covers a contiguous run of 32-token tiles of one
// sequence.  Its 8 warps form TS tile slots x HG head groups: warp w works
// on tiles slot, slot + TS, ... (slot = w % TS) for the query heads of group
// w / TS, so two warps share each tile when the group has 2+ heads.  Per
// tile: one bulk copy brings K and V into the slot's shared-memory stage;
// each warp scores the tile with one lane per token (the head dimension
// walked from a lane-dependent start so the 32 lanes read 32 different
// banks), keeps its heads' online softmax in registers, and accumulates P V
// with each lane owning HD/32 output dimensions.  The warps then merge in
// shared memory into one (m, l, o) partial per CTA; the last CTA of a
// (row, kv head) merges the S partials in split order.
template <int HD, int G>
__global__ void __launch_bounds__(NT) attn_kernel(const AttnArgs a) {
  constexpr int HG = G >= 2 ? 2 : 1;        // head groups
  constexpr int TS = NW / HG;               // tile slots
  constexpr int HPW = G / HG;               // heads per warp
  constexpr int DPL = HD / 32;              // output dims per lane
  constexpr int W2 = HD / 2;                // 2-element words per row
  constexpr int STAGE = 2 * TILE * HD;      // halves per slot stage (K then V)
  extern __shared__ __align__(128) uint8_t s_dyn[];
  __half* s_stage = reinterpret_cast<__half*>(s_dyn);          // [TS][STAGE]
  __shared__ __align__(16) float s_q[G * HD];
  __shared__ float s_wm[NW][HPW], s_wl[NW][HPW];
  __shared__ __align__(8) uint64_t s_full[TS];
  __shared__ float s_w[G][kMaxSplits];
  __shared__ int s_last;

  const int S = a.n_splits;
  const int kvh = blockIdx.x / S, sp = blockIdx.x - kvh * S;
  const int brel = blockIdx.y, b = a.row0 + brel;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot = warp % TS, hg = warp / TS;
  const int pt = a.page_tokens;

  if (tid < TS) mbar_init(smem_u32(&s_full[tid]), 1);
  mbar_fence_init();
  griddep_wait();

  int n = a.len[b] + a.len_add;
  if (n < 1 || n > a.max_len) {
    if (a.status && tid == 0) atomicOr(a.status, kBadPos);
    n = n < 1 ? 1 : a.max_len;
  }
  const int ptrow = a.pt_row ? a.pt_row[b] : b;
  const int32_t* ptab = a.page_table + (size_t)ptrow * a.max_pages;
  const int n_tiles = (n + TILE - 1) / TILE;
  // with a shared prefix computed by the cascade kernel, this launch covers
  // only the tiles from the prefix's end on
  int t0 = 0;
  if (a.start_len) t0 = min(max(*a.start_len, 0), n) / TILE;
  const int per = (n_tiles - t0 + S - 1) / S;
  const int tb = t0 + sp * per, te = min(n_tiles, tb + per);

  // the first warp of a slot copies tile i (K then V) into the slot's stage
  __half* st = s_stage + (size_t)slot * STAGE;
  const uint32_t bar = smem_u32(&s_full[slot]);
  auto issue = [&](int i) -> bool {
    const int t = i * TILE;
    const int nt = min(TILE, n - t);
    const int page = ptab[t / pt];
    if (page < 0) {
      mbar_arrive(bar);  // complete the phase with nothing copied
      return false;
    }
    const size_t base = (((size_t)page * a.n_kv + kvh) * pt + (t % pt)) * HD;
    const uint32_t bytes = (uint32_t)nt * HD * 2;
    mbar_expect_tx(bar, 2 * bytes);
    bulk_g2s(smem_u32(st), a.k_pool + base, bytes, bar);
    bulk_g2s(smem_u32(st + TILE * HD), a.v_pool + base, bytes, bar);
    return true;
  };
  __syncthreads();  // barriers initialised
  if (hg == 0 && lane == 0 && tb + slot < te && !issue(tb + slot) && a.status) atomicOr(a.status, kBadPage);

  const float scale = 1.0f / sqrtf((float)HD);
  const float* qrow = a.q + ((size_t)brel * a.n_heads + (size_t)kvh * G) * HD;
  for (int i = tid; i < G * HD; i += NT) s_q[i] = qrow[i] * scale;
  __syncthreads();
  griddep_launch();

  float m_run[HPW], l_run[HPW], o[HPW][DPL];
#pragma unroll
  for (int h = 0; h < HPW; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  }
  const float2* q2 = reinterpret_cast<const float2*>(s_q) + (size_t)hg * HPW * W2;
  bool failed = false;
  int use = 0;
  for (int i = tb + slot; i < te; i += TS, ++use) {
    const int nt = min(TILE, n - i * TILE);
    if (!mbar_wait(bar, use & 1)) failed = true;
    tile_update<HD, HPW>(st, st + TILE * HD, q2, nt, lane, m_run, l_run, o);
    // both warps of the slot are done with the stage before it is refilled
    if (HG > 1) named_bar(1 + slot, 32 * HG);
    else __syncwarp();
    if (hg == 0 && lane == 0 && i + TS < te && !issue(i + TS) && a.status) atomicOr(a.status, kBadPage);
  }
  if (failed && a.status) atomicOr(a.status, kTimeout);

  // ---- merge the warps of this CTA; per-warp outputs reuse the (now idle)
  // stage memory: NW*HPW*HD floats <= TS*2*TILE*HD halves
  __syncthreads();
  float(*s_wo)[HPW * HD] = reinterpret_cast<float(*)[HPW * HD]>(s_dyn);
  static_assert(NW * HPW * HD * 4 <= TS * 2 * TILE * HD * 2, "merge buffer must fit the stages");
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      s_wm[warp][h] = m_run[h];
      s_wl[warp][h] = l_run[h];
    }
  }
#pragma unroll
  for (int h = 0; h < HPW; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) s_wo[warp][h * HD + lane * DPL + e] = o[h][e];
  __syncthreads();
  const size_t slot0 = ((size_t)brel * a.n_kv + kvh) * S;
  // one split (S == 1): its partial stays in shared memory, after the
  // per-warp outputs, and this CTA merges it with the prefix partials (if
  // any) without the global round trip and the arrival counter
  const bool solo = S == 1;
  float* s_po = reinterpret_cast<float*>(s_dyn + NW * HPW * HD * 4);          // [G * HD]
  float2* s_pml = reinterpret_cast<float2*>(s_dyn + NW * HPW * HD * 4 + G * HD * 4);  // [G]
  static_assert(NW * HPW * HD * 4 + G * HD * 4 + G * 8 <= TS * 2 * TILE * HD * 2, "solo partial must fit the stages");
  for (int idx = tid; idx < G * HD; idx += NT) {
    const int h = idx / HD, hl = h % HPW, g0 = (h / HPW) * TS;  // warps g0 .. g0+TS-1 hold head h
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < TS; ++t) M = fmaxf(M, s_wm[g0 + t][hl]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      const float e = s_wl[g0 + t][hl] > 0.f ? expf(s_wm[g0 + t][hl] - M) : 0.f;
      acc = fmaf(e, s_wo[g0 + t][hl * HD + (idx % HD)], acc);
      L = fmaf(e, s_wl[g0 + t][hl], L);
    }
    if (solo) {
      s_po[idx] = acc;
      if ((idx % HD) == 0) s_pml[h] = make_float2(M, L);
    } else {
      a.part_o[(slot0 + sp) * G * HD + idx] = acc;
      if ((idx % HD) == 0) reinterpret_cast<float2*>(a.part_ml)[(slot0 + sp) * G + h] = make_float2(M, L);
    }
  }
  if (solo) {
    __syncthreads();
  } else {
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int prev = atomicAdd(&a.counters[(size_t)brel * a.n_kv + kvh], 1);
      s_last = prev == S - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }

  // ---- last CTA of this (row, kv head): merge the S splits (and the P
  // splits of the shared prefix from the cascade kernel, after them in split
  // order), all loads in flight
  const int P = a.pre_splits;
  const size_t pslot0 = ((size_t)brel * a.n_kv + kvh) * (size_t)P;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  const float2* pml = reinterpret_cast<const float2*>(a.pre_ml);
  for (int h = warp; h < G; h += NW) {
    // every lane's (at most four) splits in one round of loads
    float2 v[kMaxSplits / 32];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      const int s = lane + 32 * k;
      v[k] = s < S ? (solo ? s_pml[h] : __ldcg(&ml[(slot0 + s) * G + h]))
           : s < S + P ? __ldcg(&pml[(pslot0 + s - S) * G + h]) : make_float2(-INFINITY, 0.f);
      M = fmaxf(M, v[k].x);
    }
    M = warp_max(M);
    float den = 0.f, e[kMaxSplits / 32];
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      e[k] = v[k].y > 0.f ? expf(v[k].x - M) : 0.f;  // empty split: weight 0
      den = fmaf(v[k].y, e[k], den);
    }
    den = warp_sum(den);
    const float inv = 1.0f / den;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k)
      if (lane + 32 * k < S + P) s_w[h][lane + 32 * k] = e[k] * inv;
  }
  __syncthreads();
  for (int idx = tid; idx < G * HD; idx += NT) {
    const int h = idx / HD;
    const float* po = a.part_o + slot0 * G * HD + idx;
    const float* pp = a.pre_o + pslot0 * G * HD + idx;
    float acc = 0.f;
    // sixteen partials' loads in flight per round
    for (int s0 = 0; s0 < S + P; s0 += 16) {
      float pv[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int s = s0 + k;
        pv[k] = s < S ? (solo ? s_po[idx] : __ldcg(po + (size_t)s * G * HD))
              : s < S + P ? __ldcg(pp + (size_t)(s - S) * G * HD) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (s0 + k < S + P) acc = fmaf(s_w[h][s0 + k], pv[k], acc);
    }
    a.o[((size_t)brel * a.n_heads + (size_t)kvh * G) * HD + idx] = acc;
  }
  if (tid == 0) a.counters[(size_t)brel * a.n_kv + kvh] = 0;
}

// The per-tile update of the cascade kernel.  Eight warps (one per batch
// row) read every tile, so the tile's K is first transposed in shared
// memory into kt2[i][token] = (K[token][2i], K[token][2i+1]): a lane (one
// token) then reads one 4-byte word per dimension pair without bank
// conflicts while every lane reads the same q pair (a broadcast), instead of
// each lane walking q at its own offset.  Softmax and P V as tile_update.
template <int HD, int HPW>
__device__ __forceinline__ void tile_update_kt(const __half2* kt2, const __half* vt, const float2* q2, int lane,
                                               float (&m_run)[HPW], float (&l_run)[HPW], float (&o)[HPW][HD / 32]) {
  constexpr int DPL = HD / 32, W2 = HD / 2;
  float sc[HPW];
  {
    float2 acc[HPW][2];
#pragma unroll
    for (int h = 0; h < HPW; ++h) acc[h][0] = acc[h][1] = make_float2(0.f, 0.f);
#pragma unroll 8
    for (int i = 0; i < W2; ++i) {
      const float2 kf = __half22float2(kt2[i * TILE + lane]);
#pragma unroll
      for (int h = 0; h < HPW; ++h) acc[h][i & 1] = __ffma2_rn(kf, q2[h * W2 + i], acc[h][i & 1]);
    }
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      const float2 a = __fadd2_rn(acc[h][0], acc[h][1]);
      sc[h] = a.x + a.y;
    }
  }
  float p[HPW];
#pragma unroll
  for (int h = 0; h < HPW; ++h) {
    const float m_new = fmaxf(m_run[h], warp_max(sc[h]));
    p[h] = expf(sc[h] - m_new);
    const float al = expf(m_run[h] - m_new);
    l_run[h] = l_run[h] * al + warp_sum(p[h]);
    m_run[h] = m_new;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] *= al;
  }
  const __half* vl = vt + lane * DPL;
#pragma unroll
  for (int j = 0; j < TILE; ++j) {
    float vf[DPL];
    if (DPL == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(vl + j * HD);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      vf[0] = v01.x;
      vf[1] = v01.y;
      vf[2 % DPL] = v23.x;
      vf[3 % DPL] = v23.y;
    } else {
#pragma unroll
      for (int e = 0; e < DPL; ++e) vf[e] = __half2float(vl[j * HD + e]);
    }
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      const float pj = __shfl_sync(0xffffffffu, p[h], j);
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pj, vf[e], o[h][e]);
    }
  }
}

// ---- cascade attention: the shared prefix, once for every batch row --------------

constexpr int kCascStages = 4;

// Grid (n_kv * S): CTA (kv head, split sp) covers a contiguous run of the
// prefix's 32-token tiles.  Warp NW (the producer) streams the tiles -- K
// then V, one bulk copy each, from the pages of batch row 0, which every row
// shares -- through a ring of kCascStages stages; consumer warp r < rows
// applies each tile to row r's G query heads (the same per-tile update as the
// per-row kernel) and writes one (m, l, o) partial per head.  The prefix
// bytes are read once per step instead of once per row.
template <int HD, int G>
__global__ void __launch_bounds__(NT + 32) cascade_prefix_kernel(const CascArgs a) {
  constexpr int DPL = HD / 32;
  constexpr int STAGE = 2 * TILE * HD;  // halves: K then V
  extern __shared__ __align__(128) uint8_t s_dyn[];
  __half* s_stage = reinterpret_cast<__half*>(s_dyn);
  __half2* s_kt2 = reinterpret_cast<__half2*>(s_dyn + (size_t)kCascStages * STAGE * 2);  // [HD/2][TILE]
  float* s_q = reinterpret_cast<float*>(s_dyn + (size_t)kCascStages * STAGE * 2 + (size_t)HD / 2 * TILE * 4);
  __shared__ __align__(8) uint64_t s_full[kCascStages], s_empty[kCascStages];
  const int S = a.n_splits;
  const int kvh = blockIdx.x / S, sp = blockIdx.x - kvh * S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows = a.rows;
  if (tid == 0) {
    for (int i = 0; i < kCascStages; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_empty[i]), rows);
    }
    mbar_fence_init();
  }
  int n = *a.shared_len;
  if (n < 0 || n > a.max_len || n % TILE) {
    if (a.status && tid == 0) atomicOr(a.status, kBadPos);
    n = 0;
  }
  const int n_tiles = n / TILE;
  const int per = (n_tiles + S - 1) / S;
  const int tb = min(n_tiles, sp * per), te = min(n_tiles, tb + per);
  const int pt = a.page_tokens;
  const float scale = 1.0f / sqrtf((float)HD);
  for (int i = tid; i < rows * G * HD; i += NT + 32) {
    const int r = i / (G * HD), j = i - r * (G * HD);
    s_q[i] = a.q[(size_t)r * a.n_heads * HD + (size_t)kvh * G * HD + j] * scale;
  }
  __syncthreads();

  if (warp == NW) {  // producer
    if (lane == 0) {
      const int ptrow = a.pt_row ? a.pt_row[0] : 0;
      const int32_t* ptab = a.page_table + (size_t)ptrow * a.max_pages;
      int k = 0;
      for (int i = tb; i < te; ++i, ++k) {
        const int st = k % kCascStages;
        const uint32_t full = smem_u32(&s_full[st]);
        if (k >= kCascStages && !mbar_wait(smem_u32(&s_empty[st]), ((k / kCascStages) - 1) & 1)) {
          if (a.status) atomicOr(a.status, kTimeout);
          break;
        }
        const int t = i * TILE;
        const int page = ptab[t / pt];
        if (page < 0) {
          if (a.status) atomicOr(a.status, kBadPage);
          mbar_arrive(full);  // the phase completes with nothing copied
          continue;
        }
        const size_t base = (((size_t)page * a.n_kv + kvh) * pt + (t % pt)) * HD;
        const uint32_t bytes = TILE * HD * 2;
        __half* dst = s_stage + (size_t)st * STAGE;
        mbar_expect_tx(full, 2 * bytes);
        bulk_g2s(smem_u32(dst), a.k_pool + base, bytes, full);
        bulk_g2s(smem_u32(dst + TILE * HD), a.v_pool + base, bytes, full);
      }
      // never leave with copies in flight
      for (int j = max(0, k - kCascStages); j < k; ++j) mbar_wait(smem_u32(&s_full[j % kCascStages]), (j / kCascStages) & 1);
    }
    return;
  }
  if (warp >= rows) return;

  float m_run[G], l_run[G], o[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  }
  const float2* q2 = reinterpret_cast<const float2*>(s_q + (size_t)warp * G * HD);
  bool failed = false;
  const int ctid = tid;  // consumer threads: 0 .. rows * 32 - 1
  for (int i = tb, k = 0; i < te; ++i, ++k) {
    const int st = k % kCascStages;
    // every consumer waits (bounded) even after a failure, so the named
    // barriers below always see all of them
    if (!mbar_wait(smem_u32(&s_full[st]), (k / kCascStages) & 1)) failed = true;
    const __half* kt = s_stage + (size_t)st * STAGE;
    named_bar(1, rows * 32);  // every warp is done with the previous tile's transpose
    // transpose: word i of token t -> kt2[i][t]; lanes walk the words from a
    // token-dependent start so reads and writes both spread over the banks
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(kt);
    uint32_t* tw = reinterpret_cast<uint32_t*>(s_kt2);
    for (int e = ctid; e < TILE * (HD / 2); e += rows * 32) {
      const int t = e % TILE, i = ((e / TILE) + t) % (HD / 2);
      tw[i * TILE + t] = kw[t * (HD / 2) + i];
    }
    named_bar(1, rows * 32);
    tile_update_kt<HD, G>(s_kt2, kt + TILE * HD, q2, lane, m_run, l_run, o);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s_empty[st]));
  }
  if (failed && a.status && lane == 0) atomicOr(a.status, kTimeout);
  const size_t slot = ((size_t)warp * a.n_kv + kvh) * S + sp;
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int e = 0; e < DPL; ++e) a.part_o[(slot * G + h) * HD + lane * DPL + e] = o[h][e];
    if (lane == 0) reinterpret_cast<float2*>(a.part_ml)[slot * G + h] = make_float2(m_run[h], l_run[h]);
  }
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

// Splits per (row, kv head): about one tile per slot at the longest context.
int attn_default_splits(int rows, int n_kv, int num_sms, int max_len) {
  const int tiles = (max_len + TILE - 1) / TILE;
  int s = (tiles + 3) / 4;  // about one tile per slot
  // at most ~16 CTAs per SM over the grid: short splits keep every tile's
  // copy in flight at once (batches of 8 rows at ctx ~4K measured 2.06 ms
  // per 32-layer step with this cap against 2.29 with a cap of 4)
  const int cap = (16 * num_sms + rows * n_kv - 1) / (rows * n_kv);
  if (s > cap) s = cap;
  if (s > kMaxSplits) s = kMaxSplits;  // merge weights live in shared memory
  if (s < 1) s = 1;
  return s;
}

using AttnFn = void (*)(const AttnArgs);

int attn_smem(int hd, int g) {
  const int ts = g >= 2 ? NW / 2 : NW;
  return ts * 2 * TILE * hd * 2;
}

// The dynamic shared memory limit is a per-device function attribute: raise
// it once on every device the kernel runs on (flags per device id, under a
// lock, since calls may come from several host threads).
constexpr int kMaxDevices = 256;
std::mutex g_attr_mu;

template <int HD, int G>
AttnFn attn_fn() {
  static bool done[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(attn_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem(HD, G)) != cudaSuccess)
      return nullptr;
    done[dev] = true;
  }
  return attn_kernel<HD, G>;
}

template <int HD>
AttnFn attn_fn_g(int g) {
  switch (g) {
    case 1: return attn_fn<HD, 1>();
    case 2: return attn_fn<HD, 2>();
    case 4: return attn_fn<HD, 4>();
    case 8: return attn_fn<HD, 8>();
    case 16: return attn_fn<HD, 16>();
  }
  return nullptr;
}

using CascFn = void (*)(const CascArgs);

size_t casc_smem(int hd, int g, int rows) {
  return (size_t)kCascStages * 2 * TILE * hd * 2 + (size_t)hd / 2 * TILE * 4 + (size_t)rows * g * hd * 4;
}

template <int HD, int G>
CascFn casc_fn() {
  static bool done[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(cascade_prefix_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)casc_smem(HD, G, kMaxBatch)) != cudaSuccess)
      return nullptr;
    done[dev] = true;
  }
  return cascade_prefix_kernel<HD, G>;
}

template <int HD>
CascFn casc_fn_g(int g) {
  switch (g) {
    case 1: return casc_fn<HD, 1>();
    case 2: return casc_fn<HD, 2>();
    case 4: return casc_fn<HD, 4>();
    case 8: return casc_fn<HD, 8>();
  }
  return nullptr;
}

cudaError_t launch_attention(const AttnArgs& a, int rows, cudaStream_t s, bool pdl) {
  if (a.n_splits > kMaxSplits || a.n_splits < 1 || a.n_kv < 1 || a.n_heads % a.n_kv) return cudaErrorInvalidValue;
  if (a.pre_splits < 0 || a.n_splits + a.pre_splits > kMaxSplits || (a.pre_splits && (!a.pre_o || !a.pre_ml)))
    return cudaErrorInvalidValue;
  const int g = a.n_heads / a.n_kv;
  AttnFn f = a.head_dim == 32 ? attn_fn_g<32>(g) : a.head_dim == 64 ? attn_fn_g<64>(g)
           : a.head_dim == 128 ? attn_fn_g<128>(g) : nullptr;
  if (!f) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_kv * a.n_splits, rows);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = attn_smem(a.head_dim, a.n_heads / a.n_kv);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, f, a);
}

bool cascade_supported(int n_heads, int n_kv, int head_dim) {
  if (n_kv < 1 || n_heads % n_kv) return false;
  const int g = n_heads / n_kv;
  return (g == 1 || g == 2 || g == 4 || g == 8) && (head_dim == 32 || head_dim == 64 || head_dim == 128);
}

cudaError_t launch_cascade_prefix(const CascArgs& a, cudaStream_t s) {
  if (a.rows < 1 || a.rows > kMaxBatch || a.n_splits < 1 || !cascade_supported(a.n_heads, a.n_kv, a.head_dim))
    return cudaErrorInvalidValue;
  const int g = a.n_heads / a.n_kv;
  CascFn f = a.head_dim == 32 ? casc_fn_g<32>(g) : a.head_dim == 64 ? casc_fn_g<64>(g) : casc_fn_g<128>(g);
  if (!f) return cudaErrorInvalidValue;
  f<<<a.n_kv * a.n_splits, NT + 32, casc_smem(a.head_dim, g, a.rows), s>>>(a);
  return cudaGetLastError();
}

}  // namespace dls

// ---- standalone C-ABI op ---------------------------------------------------------

namespace {

bool bad_shape(int32_t n_batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t page_tokens,
               int32_t max_pages, int32_t n_splits) {
  return n_splits > dls::kMaxSplits || n_batch < 1 || n_kv_heads < 1 || n_heads < 1 || n_heads % n_kv_heads ||
         n_heads / n_kv_heads > dls::kMaxG || (head_dim != 32 && head_dim != 64 && head_dim != 128) ||
         page_tokens < 32 || page_tokens % 32 || max_pages < 1;
}

// Launch arguments shared by both entry points (scratch carved from `ws`).
dls::AttnArgs standalone_args(const float* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                              const int32_t* lengths, float* o, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, int32_t page_tokens, int32_t max_pages, int32_t n_splits,
                              int32_t* status, void* ws, int32_t n_batch) {
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
  a.status = status;
  a.max_len = page_tokens * max_pages;
  dls::attn_workspace_carve(ws, n_batch, n_heads, n_kv_heads, head_dim, n_splits, &a.part_o, &a.part_ml,
                            &a.counters);
  return a;
}

}  // namespace

extern "C" size_t dls_attention_workspace_bytes(int32_t n_batch, int32_t n_heads, int32_t n_kv_heads,
                                                int32_t head_dim, int32_t n_splits) {
  if (n_batch < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || n_splits < 1) return 0;
  return dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits);
}

extern "C" int dls_attention_decode(const float* q, const void* k_pages, const void* v_pages,
                                    const int32_t* page_table, const int32_t* lengths, float* o, void* workspace,
                                    size_t workspace_bytes, int32_t n_batch, int32_t n_heads, int32_t n_kv_heads,
                                    int32_t head_dim, int32_t page_tokens, int32_t max_pages, int32_t n_splits,
                                    int32_t* status, void* cuda_stream) {
  if (!q || !k_pages || !v_pages || !page_table || !lengths || !o || !workspace)
    return dls::report_error(DLS_ERR_ARG, "attention: NULL pointer argument");
  if (bad_shape(n_batch, n_heads, n_kv_heads, head_dim, page_tokens, max_pages, n_splits))
    return dls::report_error(DLS_ERR_ARG, "attention: bad shape n_batch=%d n_heads=%d n_kv_heads=%d head_dim=%d "
                             "page_tokens=%d max_pages=%d n_splits=%d", n_batch, n_heads, n_kv_heads, head_dim,
                             page_tokens, max_pages, n_splits);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return dls::report_error(DLS_ERR_CUDA, "attention: no current device");
  if (n_splits <= 0) n_splits = dls::attn_default_splits(n_batch, n_kv_heads, sms, page_tokens * max_pages);
  const size_t need = dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits);
  if (workspace_bytes < need)
    return dls::report_error(DLS_ERR_ARG, "attention: workspace_bytes=%zu < %zu needed for n_splits=%d",
                             workspace_bytes, need, n_splits);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "attention: clearing the status word failed");
  const dls::AttnArgs a = standalone_args(q, k_pages, v_pages, page_table, lengths, o, n_heads, n_kv_heads, head_dim,
                                          page_tokens, max_pages, n_splits, status, workspace, n_batch);
  if (dls::launch_attention(a, n_batch, st, false) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "attention: launch failed");
  return DLS_OK;
}

extern "C" int dls_attention_status(const int32_t* status, void* cuda_stream) {
  if (!status) return dls::report_error(DLS_ERR_ARG, "attention status: NULL status word");
  int32_t v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "attention status: reading the status word failed");
  if (v & dls::kTimeout)
    return dls::report_error(DLS_ERR_TIMEOUT, "attention: a bounded wait ran out device_status=0x%x", v);
  if (v)
    return dls::report_error(DLS_ERR_STATE, "attention: device_status=0x%x (1=missing page 4=length outside "
                             "1..page_tokens*max_pages)", v);
  return DLS_OK;
}

// ---- allocation-free variant -------------------------------------------------------
//
// Some callers cannot call cudaMalloc or any allocating routine: a serving
// process that carves all device memory into fixed pools at start-up and
// forbids allocations afterwards (an allocation could fail or fragment the
// plan mid-request), or code on a latency-critical path where an allocator
// call may take a lock or synchronise the device.  For them this entry point
// takes the split-K scratch from a file-scope device array instead of a
// caller-provided workspace.

namespace {

// Scratch of dls_attention_decode_noalloc.  Every GPU that loads this library
// holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[DLS_ATTENTION_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[dls::kMaxDevices] = {};  // device address of the scratch, per device id

// Device address of the scratch on the current device, looked up once per
// device (host code sees only a host-side stand-in under the symbol's name).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= dls::kMaxDevices) return DLS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_noalloc_scratch) != cudaSuccess || !p) return DLS_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DLS_OK;
}

}  // namespace

extern "C" int dls_attention_decode_noalloc(const float* q, const void* k_pages, const void* v_pages,
                                            const int32_t* page_table, const int32_t* lengths, float* o,
                                            int32_t n_batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                            int32_t page_tokens, int32_t max_pages, int32_t n_splits,
                                            int32_t* status, void* cuda_stream) {
  if (!q || !k_pages || !v_pages || !page_table || !lengths || !o)
    return dls::report_error(DLS_ERR_ARG, "noalloc attention: NULL pointer argument");
  if (bad_shape(n_batch, n_heads, n_kv_heads, head_dim, page_tokens, max_pages, n_splits))
    return dls::report_error(DLS_ERR_ARG, "noalloc attention: bad shape n_batch=%d n_heads=%d n_kv_heads=%d "
                             "head_dim=%d page_tokens=%d max_pages=%d n_splits=%d", n_batch, n_heads, n_kv_heads,
                             head_dim, page_tokens, max_pages, n_splits);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return dls::report_error(DLS_ERR_CUDA, "noalloc attention: no current device");
  const size_t cap = DLS_ATTENTION_NOALLOC_SCRATCH_BYTES;
  if (n_splits <= 0) {
    // the usual choice, cut down to the largest split count whose partials
    // fit the array (any count gives the same result up to fp32 rounding)
    n_splits = dls::attn_default_splits(n_batch, n_kv_heads, sms, page_tokens * max_pages);
    while (n_splits > 1 && dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits) > cap)
      --n_splits;
  }
  const size_t need = dls::attn_workspace_bytes(n_batch, n_heads, n_kv_heads, head_dim, n_splits);
  if (need > cap)
    return dls::report_error(DLS_ERR_CAPACITY, "noalloc attention: needs %zu bytes of scratch for n_splits=%d, the "
                             "built-in array holds %zu (fewer rows or splits fit)", need, n_splits, cap);
  void* ws = nullptr;
  if (noalloc_scratch(&ws) != DLS_OK)
    return dls::report_error(DLS_ERR_CUDA, "noalloc attention: cudaGetSymbolAddress failed");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // the arrival counters at the head of the scratch must start at zero
  const size_t counter_bytes = ((size_t)n_batch * n_kv_heads * sizeof(int) + 255) & ~(size_t)255;
  if (cudaMemsetAsync(ws, 0, counter_bytes, st) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "noalloc attention: clearing the counters failed");
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "noalloc attention: clearing the status word failed");
  const dls::AttnArgs a = standalone_args(q, k_pages, v_pages, page_table, lengths, o, n_heads, n_kv_heads, head_dim,
                                          page_tokens, max_pages, n_splits, status, ws, n_batch);
  if (dls::launch_attention(a, n_batch, st, false) != cudaSuccess)
    return dls::report_error(DLS_ERR_CUDA, "noalloc attention: launch failed");
  return DLS_OK;
}
