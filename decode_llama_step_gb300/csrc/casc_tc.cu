// Cascade attention's shared-prefix pass on the 5th-generation tensor cores
// (SwarmKV page, section 3: branches hold the prefix's KV pages by
// reference; section 10: the prefix is read once per step for all of them).
//
// CTA = (KV head, split of the prefix).  Its MMA rows are the (batch row,
// query head) pairs of the head's group, row r = batch row r / G, head
// r % G (at most 8 x 8 = 64 live rows; rows past rows * G are zero).  Per
// 64-key tile of the prefix:
//   S = Q K^T       tcgen05.mma kind::f16, M = 128, N = 64 keys, K = hd, with
//                   Q as two fp16 planes q_hi = fp16(q), q_lo = fp16(q - q_hi):
//                   q_hi k + q_lo k carries q to ~22 bits (k is fp16 exactly)
//   softmax         warps 2-17, four threads per row (each a quarter of the
//                   tile's keys and of the output columns; a row's threads
//                   exchange their maxima through shared memory): scale, mask
//                   keys past the prefix, running max, p = exp(s - max) as the
//                   planes p_hi, p_lo
//   O_t = P V       M = 128, N = hd, K = 64 keys (V an MN-major operand),
//                   p_hi V + p_lo V
//   o = o * exp(max_old - max_new) + O_t   in the softmax threads' registers,
//                   one tile late: P and O_t have two buffers each, so tile
//                   j's P V runs while the softmax threads score tile j + 1
// and the CTA writes one (m, l, o) partial per live row in the layout of the
// CUDA-core cascade kernel (o unnormalised, relative to m; natural-log
// units), which the per-row suffix kernel merges.  K/V tiles come from batch
// row 0's pages (every row shares them) by 2-D TMA in the 128-byte swizzle.
// Every wait is bounded (2 s) and sets an abort flag; the partials of an
// aborted CTA are not written and the status word reports the timeout.
#include <math.h>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int CBK = 64;     // keys per tile
constexpr int CROWS = 128;  // MMA rows
constexpr int NSW = 16;     // softmax warps: HPR per TMEM lane quarter
constexpr int HPR = NSW / 4;  // threads per row
constexpr int CTHR = 32 * (NSW + 2);  // warp 0 TMA, warp 1 MMA, warps 2 .. NSW+1 softmax
constexpr int CNS = 2;      // K/V ring stages
constexpr uint64_t kWaitNsT = 2000000000ull;

template <int HD>
struct TCfg {
  static constexpr int KA = HD / 64;          // 64-wide swizzle atoms along the head dimension
  static constexpr int kQ = CROWS * HD * 2;   // one fp16 plane of Q
  static constexpr int kKV = CBK * HD * 2;    // one K or V tile
  static constexpr int kP = CROWS * CBK * 2;  // one fp16 plane of P (one swizzle atom wide)
  static constexpr int kKVOff = 2 * kQ;       // stage s: K at + 2 s kKV, V at + (2 s + 1) kKV
  static constexpr int kPOff = kKVOff + CNS * 2 * kKV;  // P buffer b: hi at + 2 b kP, lo at + (2 b + 1) kP
  static constexpr int kXOff = kPOff + 4 * kP;  // float [3][HPR parts][128 rows]: row maxima (by tile parity), l
  static constexpr int kBarOff = kXOff + 3 * HPR * CROWS * 4;
  static constexpr int kSmem = kBarOff + 256 + 1024;
  static constexpr int kTmemCols = 512;       // S: columns 0-63, O buffer b: 64 + b hd .. 64 + (b + 1) hd
  static_assert(kSmem <= 227 * 1024, "shared memory");
  // the CTA allocates all of tensor memory: its shared memory must keep a
  // second CTA of the kernel off the SM
  static_assert(2 * kSmem > 227 * 1024, "one CTA per SM");
};

struct TBars {
  uint64_t kv_full[CNS], kv_empty[CNS], q_full, s_full, s_free, p_full, o_full[2], o_free[2];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool twait(uint32_t bar, uint32_t parity, int* abort_flag, bool heed_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 63) == 0) {
      if (heed_abort && *(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsT) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// (a, b) -> fp16 hi plane word and lo plane word (the rounding residual)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  hi = h2bits(h);
  lo = h2bits(__floats2half2_rn(a - f.x, b - f.y));
}

template <int HD, int G>
__global__ void __launch_bounds__(CTHR, 1) casc_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v, const CascArgs a) {
  using C = TCfg<HD>;
  extern __shared__ uint8_t tsm[];
  const uint32_t raw = smem_u32(tsm);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t qhi = raw + pad, qlo = qhi + C::kQ;
  const uint32_t kvbase = raw + pad + C::kKVOff;
  const uint32_t pbase = raw + pad + C::kPOff;
  TBars& sh = *reinterpret_cast<TBars*>(tsm + pad + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.n_splits;
  const int kvh = blockIdx.x / S, sp = blockIdx.x - kvh * S;
  const int R = a.rows * G;  // live rows

  int n = *a.shared_len;
  if (n < 0 || n > a.max_len || n % 32) {
    if (a.status && tid == 0) atomicOr(a.status, kBadPos);
    n = 0;
  }
  const int n_tiles = (n + CBK - 1) / CBK;
  const int per = (n_tiles + S - 1) / S;
  const int tb = min(n_tiles, sp * per), te = min(n_tiles, tb + per);
  const int nt = te - tb;
  const int pr = a.page_tokens < CBK ? a.page_tokens : CBK;  // keys per TMA piece
  const int n_pieces = CBK / pr;

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem), C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < CNS; ++i) {
      mbar_init(smem_u32(&sh.kv_full[i]), 1);
      mbar_init(smem_u32(&sh.kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&sh.q_full), NSW);
    mbar_init(smem_u32(&sh.s_full), 1);
    mbar_init(smem_u32(&sh.s_free), NSW);
    mbar_init(smem_u32(&sh.p_full), NSW);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh.o_full[b]), 1);
      mbar_init(smem_u32(&sh.o_free[b]), NSW);
    }
    sh.abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ---------------- TMA producer: the prefix tiles of batch row 0's pages
    if (lane == 0) {
      const int ptrow = a.pt_row ? a.pt_row[0] : 0;
      const int32_t* ptab = a.page_table + (size_t)ptrow * a.max_pages;
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j % CNS;
        if (j >= CNS && !twait(smem_u32(&sh.kv_empty[s]), ((j / CNS) - 1) & 1, &sh.abort)) break;
        const uint32_t bar = smem_u32(&sh.kv_full[s]);
        mbar_expect_tx(bar, 2 * C::kKV);
        const uint32_t kd = kvbase + 2 * s * C::kKV, vd = kd + C::kKV;
        for (int p = 0; p < n_pieces; ++p) {
          const int key0 = (tb + j) * CBK + p * pr;
          const int lp = key0 / a.page_tokens;
          const int page = (key0 < n && lp < a.max_pages) ? ptab[lp] : -1;
          if (page < 0 && key0 < n && a.status) atomicOr(a.status, kBadPage);
          // a piece past the prefix (or without a page) is read from past
          // the end of the pool: the TMA fills it with zeros
          const int y = page >= 0 ? (page * a.n_kv + kvh) * a.page_tokens + (key0 % a.page_tokens) : a.pool_rows;
#pragma unroll
          for (int at = 0; at < C::KA; ++at) {
            tma_load_2d(kd + at * (CBK * 128) + p * pr * 128, &tm_k, at * 64, y, bar);
            tma_load_2d(vd + at * (CBK * 128) + p * pr * 128, &tm_v, at * 64, y, bar);
          }
        }
        issued = j + 1;
      }
      // copies still in flight (after an abort) land before the CTA exits
      for (int j = issued > CNS ? issued - CNS : 0; j < issued; ++j)
        twait(smem_u32(&sh.kv_full[j % CNS]), (j / CNS) & 1, &sh.abort, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t id_s = umma_idesc_f16(CROWS, CBK);
      constexpr uint32_t id_o = umma_idesc_f16_bmn(CROWS, HD);
      const uint32_t t_s = tmem;
      bool go = twait(smem_u32(&sh.q_full), 0, &sh.abort);
      for (int j = 0; go && j < nt; ++j) {
        const int s = j % CNS;
        if (!twait(smem_u32(&sh.kv_full[s]), (j / CNS) & 1, &sh.abort)) break;
        if (j > 0 && !twait(smem_u32(&sh.s_free), (j - 1) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t kd = kvbase + 2 * s * C::kKV, vd = kd + C::kKV;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t oq = (ks >> 2) * (CROWS * 128) + (ks & 3) * 32;
          const uint32_t ok = (ks >> 2) * (CBK * 128) + (ks & 3) * 32;
          const uint64_t bk = umma_desc_k128(kd + ok);
          umma_f16(t_s, umma_desc_k128(qhi + oq), bk, id_s, ks != 0);
          umma_f16(t_s, umma_desc_k128(qlo + oq), bk, id_s, 1);
        }
        umma_commit(smem_u32(&sh.s_full));
        // P V of tile j into O buffer b (from P buffer b), once the softmax
        // threads have taken that buffer's previous tile (j - 2)
        const int b = j & 1;
        if (!twait(smem_u32(&sh.p_full), j & 1, &sh.abort)) break;
        if (j >= 2 && !twait(smem_u32(&sh.o_free[b]), ((j >> 1) - 1) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t t_o = tmem + CBK + b * HD, ph = pbase + 2 * b * C::kP, pl = ph + C::kP;
#pragma unroll
        for (int ks = 0; ks < CBK / 16; ++ks) {
          const uint64_t bv = umma_desc_mn128(vd + ks * 16 * 128, CBK * 128, 1024);
          umma_f16(t_o, umma_desc_k128(ph + ks * 32), bv, id_o, ks != 0);
          umma_f16(t_o, umma_desc_k128(pl + ks * 32), bv, id_o, 1);
        }
        umma_commit(smem_u32(&sh.o_full[b]));
        umma_commit(smem_u32(&sh.kv_empty[s]));
      }
    }
    __syncwarp();
  } else {
    // ---------------- softmax: warp w handles TMEM lane quarter w & 3 (rows
    // r = 32 (w & 3) + lane) and part hf = (w - 2) / 4 of the tile's keys and
    // of the output columns
    const int quarter = warp & 3, hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const bool live = r < R;
    const int rb = live ? r / G : 0, h = r % G;
    constexpr int KH = CBK / HPR, OH = HD / HPR;  // keys, output columns per thread
    static_assert(KH % 16 == 0 && OH % 16 == 0, "whole 16-column TMEM loads");
    float* xch = reinterpret_cast<float*>(tsm + pad + C::kXOff);  // [tile parity | l][part][row]
    // Q -> the two fp16 planes, swizzled (atom at = d / 64, 16-byte chunk
    // (d % 64) / 8): the 256 softmax threads read the live rows' q as 8-float
    // chunks, consecutive threads consecutive chunks (a batch row's G heads
    // are contiguous), every load in flight at once; rows past the live ones
    // are zero
    {
      constexpr int CPR = HD / 8;                      // chunks per MMA row
      constexpr int NCH = CROWS * CPR / (32 * NSW);    // chunks per thread
      const int st = tid - 64;                         // 0 .. 255
      float4 v0[NCH], v1[NCH];
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const int e = st + k * 32 * NSW, rr = e / CPR, c = e % CPR;
        v0[k] = v1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rr < R) {
          const float* qr = a.q + (size_t)(rr / G) * a.n_heads * HD + ((size_t)kvh * G + rr % G) * HD + 8 * c;
          v0[k] = *reinterpret_cast<const float4*>(qr);
          v1[k] = *reinterpret_cast<const float4*>(qr + 4);
        }
      }
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const int e = st + k * 32 * NSW, rr = e / CPR, c = e % CPR;
        uint4 hi, lo;
        split2(v0[k].x, v0[k].y, hi.x, lo.x);
        split2(v0[k].z, v0[k].w, hi.y, lo.y);
        split2(v1[k].x, v1[k].y, hi.z, lo.z);
        split2(v1[k].z, v1[k].w, hi.w, lo.w);
        const uint32_t off = (c >> 3) * (CROWS * 128) + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
        sts128(qhi + off, hi);
        sts128(qlo + off, lo);
      }
      fence_async_smem();
      // the MMA reads every row, written by any of the eight warps
      named_bar(5, 32 * NSW);
      if (lane == 0) mbar_arrive(smem_u32(&sh.q_full));
    }
    const float scale = 1.0f / sqrtf((float)HD);
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    float o[OH];
#pragma unroll
    for (int d = 0; d < OH; ++d) o[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, alpha_prev = 1.f;  // l_run: this half's keys only
    bool ok = true;
    // o = o * alpha + (this half of tile jj's P V, in O buffer jj & 1)
    auto accumulate_o = [&](int jj, float alpha) {
      const int b = jj & 1;
      if (ok && !twait(smem_u32(&sh.o_full[b]), (jj >> 1) & 1, &sh.abort)) ok = false;
      if (ok) {
        tc_fence_after();
#pragma unroll
        uint32_t v[OH / 16][16];  // every load of this part's columns in flight per wait
#pragma unroll
        for (int c = 0; c < OH / 16; ++c) tmem_ld16(trow + CBK + b * HD + hf * OH + c * 16, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < OH / 16; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) o[c * 16 + i] = fmaf(o[c * 16 + i], alpha, __uint_as_float(v[c][i]));
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.o_free[b]));
    };
    // every iteration runs the pair's exchange barrier, even after a failed
    // wait (the partner could otherwise wait on it for ever)
    for (int j = 0; j < nt; ++j) {
      if (ok && !twait(smem_u32(&sh.s_full), j & 1, &sh.abort)) ok = false;
      tc_fence_after();
      const int kbase = (tb + j) * CBK + hf * KH;  // this half's first key
      // P buffer j & 1: its previous tile's P V (j - 2) has completed, as
      // has every MMA issued before this tile's S = Q K^T
      const uint32_t pbuf = pbase + 2 * (j & 1) * C::kP;
      uint32_t sv[KH / 16][16];
      if (ok) {
#pragma unroll
        for (int c = 0; c < KH / 16; ++c) tmem_ld16(trow + hf * KH + c * 16, sv[c]);
        tmem_wait_ld();
      }
      float mx = -INFINITY;
#pragma unroll
      for (int hh = 0; hh < KH / 16; ++hh)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (ok && kbase + hh * 16 + i < n) mx = fmaxf(mx, __uint_as_float(sv[hh][i]) * scale);
      // the row's max over all its parts
      float* xm = xch + (j & 1) * HPR * CROWS;
      xm[hf * CROWS + r] = mx;
      named_bar(1 + quarter, 32 * HPR);
#pragma unroll
      for (int o2 = 1; o2 < HPR; ++o2) mx = fmaxf(mx, xm[((hf + o2) % HPR) * CROWS + r]);
      const float m_new = fmaxf(m_run, mx);
      // p = exp(s - m_new) into this part's chunks of the two planes, and this part's sum
      float sum = 0.f;
#pragma unroll
      for (int c1 = 0; c1 < KH / 16; ++c1) {
        float p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool in = ok && live && kbase + c1 * 16 + i < n && m_new != -INFINITY;
          p[i] = in ? expf(__uint_as_float(sv[c1][i]) * scale - m_new) : 0.f;
          sum += p[i];
        }
        // keys 16 (hf KH / 16 + c1) .. +15 = 16-byte chunks 2 (hf KH / 16 + c1) and +1 of the row
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kc = 2 * (hf * (KH / 16) + c1) + hh;
          uint4 hi, lo;
          split2(p[8 * hh + 0], p[8 * hh + 1], hi.x, lo.x);
          split2(p[8 * hh + 2], p[8 * hh + 3], hi.y, lo.y);
          split2(p[8 * hh + 4], p[8 * hh + 5], hi.z, lo.z);
          split2(p[8 * hh + 6], p[8 * hh + 7], hi.w, lo.w);
          const uint32_t off = r * 128 + ((kc ^ (r & 7)) << 4);
          sts128(pbuf + off, hi);
          sts128(pbuf + C::kP + off, lo);
        }
      }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.s_free));
        mbar_arrive(smem_u32(&sh.p_full));
      }
      const float alpha = m_new == -INFINITY ? 1.f : expf(m_run - m_new);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      // the previous tile's P V -> the running sum, rescaled by that tile's
      // alpha (this tile's P V runs meanwhile)
      if (j > 0) accumulate_o(j - 1, alpha_prev);
      alpha_prev = alpha;
    }
    if (nt > 0) accumulate_o(nt - 1, alpha_prev);
    // the row's l: all parts' sums (the same m), in part order
    xch[2 * HPR * CROWS + hf * CROWS + r] = l_run;
    named_bar(1 + quarter, 32 * HPR);
    l_run = 0.f;
#pragma unroll
    for (int o2 = 0; o2 < HPR; ++o2) l_run += xch[2 * HPR * CROWS + o2 * CROWS + r];
    ok = __all_sync(0xffffffffu, ok && !*(volatile int*)&sh.abort);
    if (ok && live) {
      const size_t slot = ((size_t)rb * a.n_kv + kvh) * S + sp;
      float* po = a.part_o + (slot * G + h) * HD + hf * OH;
#pragma unroll
      for (int c = 0; c < OH / 4; ++c)
        *reinterpret_cast<float4*>(po + 4 * c) = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      if (hf == 0) reinterpret_cast<float2*>(a.part_ml)[slot * G + h] = make_float2(m_run, l_run);
    }
    if (!ok && a.status && lane == 0) atomicOr(a.status, kTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

using CtFn = void (*)(const CUtensorMap, const CUtensorMap, const CascArgs);

template <int HD>
CtFn ct_pick(int g) {
  switch (g) {
    case 1: return casc_tc_kernel<HD, 1>;
    case 2: return casc_tc_kernel<HD, 2>;
    case 4: return casc_tc_kernel<HD, 4>;
    case 8: return casc_tc_kernel<HD, 8>;
  }
  return nullptr;
}

CtFn ct_select(int hd, int g, int* smem) {
  if (hd == 128) {
    *smem = TCfg<128>::kSmem;
    return ct_pick<128>(g);
  }
  if (hd == 64) {
    *smem = TCfg<64>::kSmem;
    return ct_pick<64>(g);
  }
  return nullptr;
}

}  // namespace

bool cascade_tc_supported(int n_heads, int n_kv, int head_dim, int page_tokens) {
  if (n_kv < 1 || n_heads % n_kv) return false;
  const int g = n_heads / n_kv;
  int smem = 0;
  return ct_select(head_dim, g, &smem) != nullptr && g * kMaxBatch <= CROWS && page_tokens >= 8 &&
         page_tokens % 8 == 0 && (page_tokens >= CBK ? page_tokens % CBK == 0 : CBK % page_tokens == 0);
}

cudaError_t cascade_tc_setup_attributes() {
  for (int hd : {64, 128})
    for (int g : {1, 2, 4, 8}) {
      int smem = 0;
      CtFn f = ct_select(hd, g, &smem);
      cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
  return cudaSuccess;
}

cudaError_t launch_cascade_prefix_tc(const CascArgs& a, cudaStream_t s) {
  if (a.rows < 1 || a.rows > kMaxBatch || a.n_splits < 1 || a.pool_rows < 1 ||
      !cascade_tc_supported(a.n_heads, a.n_kv, a.head_dim, a.page_tokens))
    return cudaErrorInvalidValue;
  const int g = a.n_heads / a.n_kv;
  int smem = 0;
  CtFn f = ct_select(a.head_dim, g, &smem);
  CUtensorMap tk, tv;
  const int pr = a.page_tokens < CBK ? a.page_tokens : CBK;
  if (!make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.k_pool, a.head_dim, a.pool_rows, a.head_dim * 2, 64, pr,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.v_pool, a.head_dim, a.pool_rows, a.head_dim * 2, 64, pr,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  f<<<a.n_kv * a.n_splits, CTHR, smem, s>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace dls
