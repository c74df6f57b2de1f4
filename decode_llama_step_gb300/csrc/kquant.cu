// Batch-1 dequant-GEMV y = W x for K-quant weights (Q4_K, Q6_K): the
// projection of a decode step on the GGUF K-quant files the engine page runs
// its 70B model from (section 1: Q4_K_M and Q6_K among its formats).
//
// Device layout ("packed"), 16-byte aligned throughout so that whole rows
// move with 1-D bulk async copies:
//  * Q4_K: the GGUF super-block as it is, 144 bytes = 16 bytes of scales
//    (d, dmin, twelve bytes of 6-bit sub-block scales and minimums) + 128
//    bytes of 4-bit codes; a row is cols/256 consecutive super-blocks.
//  * Q6_K: the first 208 bytes of each GGUF super-block (low code bits, high
//    code bits, sixteen int8 scales) row-major, then a separate fp16 array of
//    the super-block scales d, [rows][nsb rounded up to 8].
//
// Same HBM-bound scheme as the Q8_0 / Q4_0 GEMV: one CTA per SM (two where
// registers allow) owns a contiguous row range; a producer warp streams its
// rows through a shared-memory ring with cp.async.bulk and mbarriers; each
// consumer lane owns a fixed slice of the columns ("unit"), holds that slice
// of x as int16 with one scale in registers, and takes exact int32 dot
// products of codes and activations (dp2a) per row.
//  * Q4_K unit: the low nibbles of sub-block 2g and the high nibbles of
//    sub-block 2g+1 (one pair of 6-bit scales and minimums, decoded once per
//    unit).  Wide units (rows of 16K columns or more): all 32 code bytes of
//    the pair = 64 weights, four per super-block.  Narrow units (shorter
//    rows, where more lanes per row keep more warps in flight): 16 code
//    bytes = 32 weights, eight per super-block.
//    y += xs * (d * (sc_a I_a + sc_b I_b) - dmin * (m_a S_a + m_b S_b)), with
//    I the integer code-activation dots and S the sums of the int16 slice.
//    The high nibbles enter the dot product in place (byte & 0xF0 = 16 x
//    code) and I_b is the exact quotient by 16 (Q5_K, whose fifth bit sits
//    above the nibble, shifts them down instead).
//  * Q6_K unit: 48 code bytes = 64 weights in four groups of 16, each group
//    with its int8 scale; y += xs * d * sum_g sc_g (I_g - 32 S_g).
#include <stdlib.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/dls.h"
#include "gemv_core.cuh"
#include "kernels.h"

namespace dls {

namespace {

// Consumer warps per CTA: as many as one unit per lane needs (a warp per 32
// units of a row) while registers allow, else fewer warps with 2-4 units per
// lane.  Cols up to 32768 fit.
constexpr int kMaxWarps = 31;
constexpr int kMaxWarpsMC = 8;
template <int FMT, int MC, int W>
struct KqBounds {
  static constexpr int threads = MC > 1 ? 32 * (kMaxWarpsMC + 1) : (FMT != KQ_Q6_K && !W) ? 1024 : 512;
};
constexpr int kRB = 64;              // rows per reduction block
constexpr int kStageBytes = 16384;   // target code bytes per ring stage
constexpr int kRing = 64 * 1024;

struct KqShared {
  uint64_t full[16];
  uint64_t empty[16];
  int abort;
};

// W: wide Q4_K / Q5_K units (64 weights) or narrow ones (32); Q6_K units
// are 64 weights either way.
template <int FMT, int W>
struct KqGeo {
  static constexpr bool K4 = FMT != KQ_Q6_K;               // Q4_K and Q5_K share the unit geometry
  static constexpr bool WIDE = !K4 || W;
  static constexpr int UPB = WIDE ? 4 : 8;                  // units per super-block
  static constexpr int NP = WIDE ? 32 : 16;                 // int16 pairs per unit
  static constexpr int NGL = NP / 8;                        // groups of 16 weights per unit
  static constexpr int NG = K4 ? 2 : 4;                     // sums kept: per sub-block (Q4_K) or scale group (Q6_K)
  static constexpr int SB = FMT == KQ_Q4_K ? 144 : FMT == KQ_Q5_K ? 176 : 208;  // packed super-block bytes
  static constexpr int MCMAX = WIDE ? 2 : 4;                // units per lane (registers)
};

template <int FMT, int W>
struct KqX {
  uint32_t p[KqGeo<FMT, W>::NP];  // int16 pairs: element 2e in the low half of p[e]
  int sum[KqGeo<FMT, W>::NG];     // per sum group: sum of the int16 values
  float s;                        // x_i ~= s * X_i
};

// Byte i (0..15) of a 16-byte vector.
__device__ __forceinline__ uint32_t byte_of(const uint4& v, int i) {
  const uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
  return (w >> (8 * (i & 3))) & 0xFFu;
}

// The element offsets (within the row) of one unit's groups of 16.
template <int FMT, int W>
__device__ __forceinline__ int group_col(int unit, int g) {
  if (FMT != KQ_Q6_K && W) {
    // 64 consecutive columns: the low nibbles' 32 (sub-block 2gg), then the
    // high nibbles' 32 (sub-block 2gg + 1)
    const int sb = unit >> 2, gg = unit & 3;
    return sb * 256 + 64 * gg + 16 * g;
  } else if (FMT != KQ_Q6_K) {
    // 16 columns of sub-block 2gg (g = 0, low nibbles) and the same 16 of 2gg + 1 (g = 1)
    const int sb = unit >> 3, v = unit & 7, gg = v >> 1, l0 = (v & 1) * 16;
    return sb * 256 + 64 * gg + 32 * g + l0;
  } else {
    const int sb = unit >> 2, v = unit & 3, h = v >> 1, l0 = (v & 1) * 16;
    return sb * 256 + 128 * h + 32 * g + l0;
  }
}

template <int FMT, int W>
__device__ __forceinline__ void load_unit_x(const float* x, int unit, bool valid, KqX<FMT, W>& xq) {
  constexpr int NG = KqGeo<FMT, W>::NG, NGL = KqGeo<FMT, W>::NGL;
  float v[NGL * 16];
#pragma unroll
  for (int g = 0; g < NGL; ++g) {
    const int c0 = valid ? group_col<FMT, W>(unit, g) : 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 f = *reinterpret_cast<const float4*>(x + c0 + 4 * j);
      if (!valid) f = make_float4(0.f, 0.f, 0.f, 0.f);
      v[g * 16 + 4 * j] = f.x;
      v[g * 16 + 4 * j + 1] = f.y;
      v[g * 16 + 4 * j + 2] = f.z;
      v[g * 16 + 4 * j + 3] = f.w;
    }
  }
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < NGL * 16; ++i) mx = fmaxf(mx, fabsf(v[i]));
  const float s = mx > 0.f ? mx / 32767.0f : 1.0f;
  const float inv = 1.0f / s;
#pragma unroll
  for (int g = 0; g < NG; ++g) xq.sum[g] = 0;
#pragma unroll
  for (int g = 0; g < NGL; ++g) {
    int sum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int a = __float2int_rn(v[g * 16 + 2 * e] * inv), b = __float2int_rn(v[g * 16 + 2 * e + 1] * inv);
      sum += a + b;
      xq.p[g * 8 + e] = (uint32_t)(a & 0xFFFF) | ((uint32_t)b << 16);
    }
    xq.sum[g * NG / NGL] += sum;  // wide Q4_K / Q5_K units: two groups per sub-block
  }
  xq.s = s;
}

// 16 unsigned code bytes (one per element, 4 words) against 8 int16 pairs.
__device__ __forceinline__ int dot16(const uint32_t (&c)[4], const uint32_t* p) {
  int s0 = 0, s1 = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    s0 = dp2a_lo(p[2 * k], c[k], s0);
    s1 = dp2a_hi(p[2 * k + 1], c[k], s1);
  }
  return s0 + s1;
}

// Per-lane byte selectors for the Q4_K scale bytes of the lane's two
// sub-blocks s = 2g, 2g+1 (g = lane & 3 for wide units, (lane & 7) >> 1 for
// narrow ones; fixed for the kernel).
// Scale bytes 0-7 are words y, z of the super-block's first 16 bytes (after
// d, dmin), bytes 8-11 word w.
//   g < 2:  [sc_a, sc_b, m_a, m_b] = low 6 bits of bytes (s, s, s+4, s+4)
//   g >= 2: low 4 bits from the nibbles of bytes s+4 (word w), top 2 bits
//           from the top of bytes s-4 (sc) and s (m)
struct Q4kSel {
  uint32_t s1, s2;
  bool split;
};

__device__ __forceinline__ Q4kSel q4k_sel(int lane, bool wide) {
  const int g = wide ? lane & 3 : (lane & 7) >> 1, a = 2 * g;
  Q4kSel q;
  q.split = g >= 2;
  q.s1 = q.split ? (uint32_t)((a - 4) | (a - 3) << 4 | a << 8 | (a + 1) << 12)
                 : (uint32_t)(a | (a + 1) << 4 | (a + 4) << 8 | (a + 5) << 12);
  q.s2 = (uint32_t)((a - 4) & 7) * 0x0101u | (uint32_t)((a - 3) & 7) * 0x1010u;
  return q;
}

// The scale bytes [sc_a, sc_b, m_a, m_b] of the lane's sub-block pair and
// the super-block's d and dmin, from its 16-byte head.
__device__ __forceinline__ uint32_t q4k_scales(const uint4& m, const Q4kSel& sel, float& d, float& dmin) {
  d = __half2float(__ushort_as_half((unsigned short)(m.x & 0xFFFF)));
  dmin = __half2float(__ushort_as_half((unsigned short)(m.x >> 16)));
  const uint32_t t1 = __byte_perm(m.y, m.z, sel.s1);
  const uint32_t t2 = __byte_perm(m.w, 0u, sel.s2);
  return sel.split ? ((t2 & 0x00000F0Fu) | ((t2 >> 4) & 0x0F0F0000u) | (((t1 >> 6) & 0x03030303u) << 4))
                   : (t1 & 0x3F3F3F3Fu);
}

// One narrow Q4_K unit of one row: codes at qa (16 bytes), super-block head
// at ma.  Q5_K (FIFTH): the fifth code bits at ha, bit 2g of byte l for the
// low nibbles' weights and bit 2g + 1 for the high nibbles'.
template <bool FIFTH, int FMT>
__device__ __forceinline__ float unit_q4_k_narrow(uint32_t qa, uint32_t ma, uint32_t ha, int g, const Q4kSel& sel,
                                                  const KqX<FMT, 0>& xq) {
  const uint4 q = lds128(qa);
  float d, dmin;
  const uint32_t v = q4k_scales(lds128(ma), sel, d, dmin);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    lo[k] = w[k] & 0x0F0F0F0Fu;
    hi[k] = (w[k] >> 4) & 0x0F0F0F0Fu;
  }
  if constexpr (FIFTH) {
    const uint4 h = lds128(ha);
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      lo[k] |= ((hw[k] >> (2 * g)) & 0x01010101u) << 4;
      hi[k] |= ((hw[k] >> (2 * g + 1)) & 0x01010101u) << 4;
    }
  }
  const int ia = dot16(lo, xq.p), ib = dot16(hi, xq.p + 8);
  // exact in int32: |sc * I| <= 63 * 16 * 31 * 32767 (twice that < 2^31),
  // |m * S| <= 63 * 16 * 32767
  const int isc = (int)(v & 0xFFu) * ia + (int)((v >> 8) & 0xFFu) * ib;
  const int imn = (int)((v >> 16) & 0xFFu) * xq.sum[0] + (int)(v >> 24) * xq.sum[1];
  return xq.s * fmaf(d, (float)isc, -dmin * (float)imn);
}

// One wide Q4_K unit of one row: codes at qa (32 bytes), super-block head at
// ma.  Q5_K (FIFTH): the fifth code bits at ha (32 bytes), bit 2g of byte l
// for the low nibbles' weights and bit 2g + 1 for the high nibbles'.
template <bool FIFTH, int FMT>
__device__ __forceinline__ float unit_q4_k(uint32_t qa, uint32_t ma, uint32_t ha, int g, const Q4kSel& sel,
                                           const KqX<FMT, 1>& xq) {
  const uint4 q0 = lds128(qa), q1 = lds128(qa + 16);
  float d, dmin;
  const uint32_t v = q4k_scales(lds128(ma), sel, d, dmin);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint32_t lo[8], hi[8];
  int ia, ib;
  if constexpr (FIFTH) {
    const uint4 h0 = lds128(ha), h1 = lds128(ha + 16);
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo[k] = (w[k] & 0x0F0F0F0Fu) | (((hw[k] >> (2 * g)) & 0x01010101u) << 4);
      hi[k] = ((w[k] >> 4) & 0x0F0F0F0Fu) | (((hw[k] >> (2 * g + 1)) & 0x01010101u) << 4);
    }
    ia = dot16(*reinterpret_cast<const uint32_t(*)[4]>(lo), xq.p) +
         dot16(*reinterpret_cast<const uint32_t(*)[4]>(lo + 4), xq.p + 8);
    ib = dot16(*reinterpret_cast<const uint32_t(*)[4]>(hi), xq.p + 16) +
         dot16(*reinterpret_cast<const uint32_t(*)[4]>(hi + 4), xq.p + 24);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo[k] = w[k] & 0x0F0F0F0Fu;
      hi[k] = w[k] & 0xF0F0F0F0u;  // 16 x the high nibble
    }
    ia = dot16(*reinterpret_cast<const uint32_t(*)[4]>(lo), xq.p) +
         dot16(*reinterpret_cast<const uint32_t(*)[4]>(lo + 4), xq.p + 8);
    // |16 I_b| <= 32 x 240 x 32767 < 2^31; a multiple of 16, so the shift is exact
    ib = (dot16(*reinterpret_cast<const uint32_t(*)[4]>(hi), xq.p + 16) +
          dot16(*reinterpret_cast<const uint32_t(*)[4]>(hi + 4), xq.p + 24)) >> 4;
  }
  // exact in int32: |sc * I| <= 63 * 32 * 31 * 32767 (twice that < 2^31),
  // |m * S| <= 63 * 32 * 32767
  const int isc = (int)(v & 0xFFu) * ia + (int)((v >> 8) & 0xFFu) * ib;
  const int imn = (int)((v >> 16) & 0xFFu) * xq.sum[0] + (int)(v >> 24) * xq.sum[1];
  return xq.s * fmaf(d, (float)isc, -dmin * (float)imn);
}

// One Q6_K unit of one row: ql halves at aa / ba, qh at ha, scales at sa.
__device__ __forceinline__ float unit_q6_k(uint32_t aa, uint32_t ba, uint32_t ha, uint32_t sa, float d, int lane,
                                           const KqX<KQ_Q6_K, 1>& xq) {
  const uint4 A = lds128(aa), B = lds128(ba), Q = lds128(ha), S = lds128(sa);
  const uint32_t a[4] = {A.x, A.y, A.z, A.w}, b[4] = {B.x, B.y, B.z, B.w}, qh[4] = {Q.x, Q.y, Q.z, Q.w};
  const int base = 8 * ((lane & 3) >> 1) + (lane & 1);   // scale of group 0 (8h + l0/16)
  float acc = 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t src = (g & 1) ? b[k] : a[k];
      const uint32_t low = (g < 2 ? src : src >> 4) & 0x0F0F0F0Fu;
      const uint32_t high = (qh[k] >> (2 * g)) & 0x03030303u;
      c[k] = low | (high << 4);
    }
    const int ig = dot16(c, xq.p + 8 * g) - 32 * xq.sum[g];
    const float scg = (float)(int)(int8_t)byte_of(S, base + 2 * g);
    acc = fmaf(scg, (float)ig, acc);
  }
  return xq.s * d * acc;
}

template <int FMT, int RS, int MC, int W>
__global__ void __launch_bounds__(KqBounds<FMT, RS * 0 + MC, W>::threads) kq_gemv_kernel(const KqArgs a,
                                                                                       const KqLaunch L) {
  using G = KqGeo<FMT, W>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  KqShared& sh = *reinterpret_cast<KqShared*>(smem_raw);
  float* s_part = reinterpret_cast<float*>(smem_raw + sizeof(KqShared));   // [nwc][kRB]
  uint8_t* ring = smem_raw + ((sizeof(KqShared) + L.nwc * kRB * 4 + 127) & ~127);
  const int nsb = a.cols / 256;
  const int nsb_pad = (nsb + 7) & ~7;
  const int nwc = L.nwc, NS = L.ns;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t row_bytes = (uint32_t)nsb * G::SB;
  const uint32_t drow_bytes = FMT == KQ_Q6_K ? (uint32_t)nsb_pad * 2 : 0;
  const uint32_t stage_q = RS * row_bytes;
  const uint32_t stage_bytes = stage_q + RS * drow_bytes;
  const int r0 = (int)((long long)a.rows * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)a.rows * (blockIdx.x + 1) / gridDim.x);
  const int nrows = max(r1 - r0, 0);
  const int nst = (nrows + RS - 1) / RS;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), nwc);
    }
    sh.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the next kernel may start now (it waits
  // for this grid's completion before reading its output); the weight
  // stream below does not depend on the previous kernel, the consumers wait
  // for it before reading x.
  griddep_launch();

  if (warp == nwc) {
    // ---------------- producer: this CTA's rows through the ring
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nst; ++s) {
        const int slot = s % NS;
        if (s >= NS && !mbar_wait(smem_u32(&sh.empty[slot]), ((s / NS) - 1) & 1)) {
          if (a.status) atomicOr(a.status, kTimeout);
          sh.abort = 1;
          break;
        }
        const int rows_s = min(RS, nrows - s * RS);
        const int row = r0 + s * RS;
        uint8_t* dst = ring + (size_t)slot * stage_bytes;
        const uint32_t qb = rows_s * row_bytes, db = rows_s * drow_bytes;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_expect_tx(bar, qb + db);
        bulk_g2s(smem_u32(dst), a.w + (size_t)row * row_bytes, qb, bar);
        if (FMT == KQ_Q6_K)
          bulk_g2s(smem_u32(dst + stage_q), reinterpret_cast<const uint8_t*>(a.d6) + (size_t)row * drow_bytes, db, bar);
        ++issued;
      }
      // never leave with copies in flight
      for (int s = max(0, issued - NS); s < issued; ++s) mbar_wait(smem_u32(&sh.full[s % NS]), (s / NS) & 1);
    }
  } else {
    // ---------------- consumers
    griddep_wait();
    const int nunits = nsb * G::UPB;
    KqX<FMT, G::WIDE ? 1 : 0> xq[MC];
    bool valid[MC];
    int ubase[MC];
#pragma unroll
    for (int k = 0; k < MC; ++k) {
      const int unit = (warp + k * nwc) * 32 + lane;
      valid[k] = unit < nunits;
      ubase[k] = valid[k] ? unit : 0;
      load_unit_x<FMT, G::WIDE ? 1 : 0>(a.x, ubase[k], valid[k], xq[k]);
    }
    const Q4kSel qsel = q4k_sel(lane, G::WIDE);
    const int stages_per_block = kRB / RS;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NS;
      if (!sh.abort && !mbar_wait(smem_u32(&sh.full[slot]), (s / NS) & 1)) {
        if (a.status) atomicOr(a.status, kTimeout);
        sh.abort = 1;
      }
      const int rows_s = min(RS, nrows - s * RS);
      const uint32_t st = smem_u32(ring) + (uint32_t)slot * stage_bytes;
      float acc[RS];
#pragma unroll
      for (int rr = 0; rr < RS; ++rr) acc[rr] = 0.f;
      if (!sh.abort) {
#pragma unroll
        for (int k = 0; k < MC; ++k) {
          const int unit = ubase[k];
#pragma unroll
          for (int rr = 0; rr < RS; ++rr) {
            const uint32_t rowa = st + rr * row_bytes;
            float t;
            if constexpr (FMT != KQ_Q6_K && G::WIDE) {
              constexpr bool Q5 = FMT == KQ_Q5_K;
              const int sb = unit >> 2, gg = unit & 3;
              const uint32_t blk = rowa + (uint32_t)sb * G::SB;
              t = unit_q4_k<Q5>(blk + (Q5 ? 48 : 16) + 32 * gg, blk, blk + 16, gg, qsel, xq[k]);
            } else if constexpr (FMT != KQ_Q6_K) {
              constexpr bool Q5 = FMT == KQ_Q5_K;
              const int sb = unit >> 3, v = unit & 7;
              const uint32_t blk = rowa + (uint32_t)sb * G::SB;
              t = unit_q4_k_narrow<Q5>(blk + (Q5 ? 48 : 16) + 32 * (v >> 1) + 16 * (v & 1), blk, blk + 16 + 16 * (v & 1),
                                       v >> 1, qsel, xq[k]);
            } else {
              const int sb = unit >> 2, v = unit & 3, h = v >> 1, l0 = (v & 1) * 16;
              const uint32_t blk = rowa + (uint32_t)sb * 208;
              const float d = lds_half_as_float(st + stage_q + rr * drow_bytes + sb * 2);
              t = unit_q6_k(blk + 64 * h + l0, blk + 64 * h + 32 + l0, blk + 128 + 32 * h + l0, blk + 192, d, lane,
                            xq[k]);
            }
            acc[rr] = valid[k] ? acc[rr] + t : acc[rr];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
      const float t = butterfly<RS>(acc, lane);
      const int rr = RS == 1 ? 0 : (lane >> (5 - (RS == 2 ? 1 : RS == 4 ? 2 : 3)));
      const int lrow = s * RS + rr - (s / stages_per_block) * kRB;
      if ((lane & ((32 / RS) - 1)) == 0 && rr < rows_s) s_part[warp * kRB + lrow] = t;
      if ((s + 1) % stages_per_block == 0 || s == nst - 1) {
        named_bar(1, nwc * 32);
        const int b0 = r0 + (s / stages_per_block) * kRB;
        const int bn = min(kRB, r1 - b0);
        for (int lr = tid; lr < bn; lr += nwc * 32) {
          float v = 0.f;
          for (int ww = 0; ww < nwc; ++ww) v += s_part[ww * kRB + lr];   // fixed order
          a.y[b0 + lr] = v;
        }
        named_bar(1, nwc * 32);
      }
    }
  }
  __syncthreads();
}

using KqFn = void (*)(const KqArgs, const KqLaunch);

template <int FMT, int MC, int W>
KqFn kq_pick_rs(int rs) {
  switch (rs) {
    case 1: return &kq_gemv_kernel<FMT, 1, MC, W>;
    case 2: return &kq_gemv_kernel<FMT, 2, MC, W>;
    case 4: return &kq_gemv_kernel<FMT, 4, MC, W>;
    case 8: return &kq_gemv_kernel<FMT, 8, MC, W>;
  }
  return nullptr;
}

template <int FMT, int W>
KqFn kq_pick_mc(int rs, int mc) {
  if (mc <= 1) return kq_pick_rs<FMT, 1, W>(rs);
  if (mc <= 2) return kq_pick_rs<FMT, 2, W>(rs);
  if constexpr (!W) {
    if (mc <= 4) return kq_pick_rs<FMT, 4, W>(rs);
  }
  return nullptr;
}

// wide: 64-weight Q4_K / Q5_K units (ignored for Q6_K, whose units always are)
KqFn kq_pick(int fmt, int rs, int mc, bool wide) {
  if (fmt == KQ_Q4_K) return wide ? kq_pick_mc<KQ_Q4_K, 1>(rs, mc) : kq_pick_mc<KQ_Q4_K, 0>(rs, mc);
  if (fmt == KQ_Q5_K) return wide ? kq_pick_mc<KQ_Q5_K, 1>(rs, mc) : kq_pick_mc<KQ_Q5_K, 0>(rs, mc);
  if (fmt == KQ_Q6_K) return kq_pick_mc<KQ_Q6_K, 1>(rs, mc);
  return nullptr;
}

// Q6_K GGUF super-blocks (210 bytes, not 16-byte aligned) -> the packed
// layout: one thread per 32-bit word of the 208-byte part, one per d.
__global__ void kq_pack_q6_k_kernel(const uint8_t* src, int rows, int nsb, uint8_t* dst, __half* d6) {
  const int nsb_pad = (nsb + 7) & ~7;
  const long long words = (long long)rows * nsb * 52;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < words;
       i += (long long)gridDim.x * blockDim.x) {
    const long long blk = i / 52;
    const int w = (int)(i % 52);
    const uint8_t* s = src + blk * 210 + 4 * w;
    const uint32_t v = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16) | ((uint32_t)s[3] << 24);
    reinterpret_cast<uint32_t*>(dst)[i] = v;
    if (w == 0) {
      const long long r = blk / nsb, sb = blk % nsb;
      const uint8_t* dp = src + blk * 210 + 208;
      d6[r * nsb_pad + sb] = __ushort_as_half((unsigned short)(dp[0] | (dp[1] << 8)));
    }
  }
}

}  // namespace

size_t kq_packed_bytes(int fmt, int rows, int cols) {
  const size_t nsb = (size_t)cols / 256, nsb_pad = (nsb + 7) & ~(size_t)7;
  if (fmt == KQ_Q4_K) return (size_t)rows * nsb * 144;
  if (fmt == KQ_Q5_K) return (size_t)rows * nsb * 176;
  const size_t main = ((size_t)rows * nsb * 208 + 255) & ~(size_t)255;
  return main + (size_t)rows * nsb_pad * 2;
}

const __half* kq_d6(const void* packed, int rows, int cols) {
  const size_t nsb = (size_t)cols / 256;
  const size_t main = ((size_t)rows * nsb * 208 + 255) & ~(size_t)255;
  return reinterpret_cast<const __half*>(static_cast<const uint8_t*>(packed) + main);
}

// ---- dequantisation of single weights (embedding rows, test hooks) ---------------

// Weight (row, col) of a packed K-quant matrix, from the fields of its
// super-block (the layouts in the header comment), computed in fp64 and
// rounded once to fp32.
__device__ double kq_weight(int fmt, const uint8_t* w, const __half* d6, int nsb, int row, int col) {
  const int sbi = col >> 8, i = col & 255;
  if (fmt == KQ_Q6_K) {
    const uint8_t* b = w + ((size_t)row * nsb + sbi) * 208;
    const int h = i >> 7, o = i & 127, g = o >> 5, l = o & 31;
    const uint32_t qlb = b[64 * h + 32 * (g & 1) + l];
    const int low = g < 2 ? (int)(qlb & 15u) : (int)(qlb >> 4);
    const int high = (b[128 + 32 * h + l] >> (2 * g)) & 3;
    const int sc = (int)(int8_t)b[192 + (i >> 4)];
    const double d = (double)__half2float(d6[(size_t)row * ((nsb + 7) & ~7) + sbi]);
    return d * (double)(sc * ((low | (high << 4)) - 32));
  }
  const int sbb = fmt == KQ_Q4_K ? 144 : 176;
  const uint8_t* b = w + ((size_t)row * nsb + sbi) * sbb;
  const double d = (double)__half2float(__ushort_as_half((uint16_t)(b[0] | (b[1] << 8))));
  const double dmin = (double)__half2float(__ushort_as_half((uint16_t)(b[2] | (b[3] << 8))));
  const uint8_t* sb = b + 4;
  const int s = i >> 5;
  int sc, m;
  if (s < 4) {
    sc = sb[s] & 63;
    m = sb[s + 4] & 63;
  } else {
    sc = (sb[s + 4] & 15) | ((sb[s - 4] >> 6) << 4);
    m = (sb[s + 4] >> 4) | ((sb[s] >> 6) << 4);
  }
  const int g = i >> 6, l = i & 31, hi = (i >> 5) & 1;
  const uint8_t* qs = b + (fmt == KQ_Q4_K ? 16 : 48);
  int q = hi ? (qs[32 * g + l] >> 4) : (qs[32 * g + l] & 15);
  if (fmt == KQ_Q5_K) q |= ((b[16 + l] >> (2 * g + hi)) & 1) << 4;
  return d * (double)(sc * q) - dmin * (double)m;
}

// out[i][c] = weight(row_i, c): rows row0.. (idx NULL) or idx[i] (clamped to
// [0, rows), a bad index flagged in *status)
__global__ void kq_dequant_rows_kernel(int fmt, const uint8_t* w, const __half* d6, int rows, int cols, int row0,
                                       const int32_t* idx, int n, float* out, int ldo, int32_t* status) {
  const int nsb = cols / 256;
  const size_t total = (size_t)n * cols;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / cols), c = (int)(e % cols);
    int r = idx ? idx[i] : row0 + i;
    if (r < 0 || r >= rows) {
      if (status && c == 0) atomicOr(status, kBadToken);
      r = 0;
    }
    out[(size_t)i * ldo + c] = (float)kq_weight(fmt, w, d6, nsb, r, c);
  }
}

cudaError_t launch_kq_dequant_rows(int fmt, const void* packed, int rows, int cols, int row0, const int32_t* idx,
                                   int n, float* out, int ldo, int32_t* status, cudaStream_t s) {
  if ((fmt != KQ_Q4_K && fmt != KQ_Q5_K && fmt != KQ_Q6_K) || cols % 256 || n < 1) return cudaErrorInvalidValue;
  const size_t total = (size_t)n * cols;
  const int grid = (int)std::min<size_t>((total + 255) / 256, 4096);
  kq_dequant_rows_kernel<<<grid, 256, 0, s>>>(fmt, static_cast<const uint8_t*>(packed),
                                              fmt == KQ_Q6_K ? kq_d6(packed, rows, cols) : nullptr, rows, cols, row0,
                                              idx, n, out, ldo, status);
  return cudaGetLastError();
}

cudaError_t launch_kq_pack(int fmt, const void* blocks, int rows, int cols, void* packed, cudaStream_t s) {
  if (fmt == KQ_Q4_K || fmt == KQ_Q5_K)
    return cudaMemcpyAsync(packed, blocks, kq_packed_bytes(fmt, rows, cols), cudaMemcpyDeviceToDevice, s);
  const int nsb = cols / 256;
  uint8_t* dst = static_cast<uint8_t*>(packed);
  __half* d6 = const_cast<__half*>(kq_d6(packed, rows, cols));
  const size_t nsb_pad = ((size_t)nsb + 7) & ~(size_t)7;
  cudaError_t e = cudaMemsetAsync(d6, 0, (size_t)rows * nsb_pad * 2, s);
  if (e != cudaSuccess) return e;
  const long long words = (long long)rows * nsb * 52;
  const int grid = (int)std::min<long long>((words + 255) / 256, 65535);
  kq_pack_q6_k_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(blocks), rows, nsb, dst, d6);
  return cudaGetLastError();
}

KqLaunch kq_plan(int fmt, int rows, int cols, int num_sms) {
  KqLaunch l{};
  if ((fmt != KQ_Q4_K && fmt != KQ_Q5_K && fmt != KQ_Q6_K) || cols % 256 || cols <= 0 || rows <= 0) return l;
  const int nsb = cols / 256;
  // wide Q4_K / Q5_K units (fewer instructions per weight) where a row has
  // 256 of them or more, or where there are 16K rows or more (long streams
  // per CTA); narrow units otherwise, whose lighter lanes keep more warps in
  // flight.  Measured on the 70B shapes: 28672 x 8192 wide 4290 GB/s, narrow
  // 3788; 8192 x 8192 wide 2297, narrow 2608; 8192 x 28672 wide 3282, narrow 3124.
  const bool k4 = fmt != KQ_Q6_K, wide = !k4 || nsb * 4 >= 256 || rows >= 16384;
  const int upb = wide ? 4 : 8, mcmax = wide ? 2 : 4;
  const int max1 = (wide ? 512 : 1024) / 32 - 1;  // consumer warps at one unit per lane
  const int nchunk = (nsb * upb + 31) / 32;
  int nwc = 0, mc = 0;
  if (nchunk <= max1) {
    nwc = nchunk;
    mc = 1;
  } else {
    for (int d = 1; d <= kMaxWarpsMC; ++d)
      if (nchunk % d == 0 && nchunk / d <= mcmax) nwc = d;
    if (!nwc) nwc = std::min(kMaxWarpsMC, (nchunk + mcmax - 1) / mcmax);
    mc = (nchunk + nwc - 1) / nwc;
  }
  if (mc > mcmax) return l;
  const int row_bytes = nsb * (fmt == KQ_Q4_K ? 144 : fmt == KQ_Q5_K ? 176 : 208);
  const int drow = fmt == KQ_Q6_K ? ((nsb + 7) & ~7) * 2 : 0;
  int rs = 1;
  while (rs < 8 && (rs * 2) * row_bytes <= kStageBytes) rs *= 2;
  const int stage = rs * (row_bytes + drow);
  KqFn f = kq_pick(fmt, rs, mc, wide);
  if (!f) return l;
  const int threads = 32 * (nwc + 1);
  const int head = (int)((sizeof(KqShared) + nwc * kRB * 4 + 127) & ~127);
  // two CTAs per SM with a 64 KB ring, or up to four with ~40 KB rings when
  // registers allow (more warps to hide the shared-memory and dp2a latency)
  int best_occ = 0, best_ns = 0;
  for (int ring : {kRing, 40 * 1024}) {
    const int ns = std::max(2, std::min(16, ring / stage));
    const int smem = head + ns * stage;
    if (smem > 200 * 1024) continue;
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, threads, smem) != cudaSuccess) {
      cudaGetLastError();
      occ = 1;
    }
    occ = std::max(1, std::min(ring == kRing ? 2 : 4, occ));
    if (occ > best_occ) {
      best_occ = occ;
      best_ns = ns;
    }
  }
  if (!best_occ) return l;
  l.nwc = nwc;
  l.mc = mc;
  l.wide = wide ? 1 : 0;
  l.rs = rs;
  l.ns = best_ns;
  l.threads = threads;
  l.smem = head + best_ns * stage;
  l.grid = std::max(1, std::min(num_sms * best_occ, rows));
  return l;
}

cudaError_t kq_setup_attributes() {
  for (int fmt : {(int)KQ_Q4_K, (int)KQ_Q5_K, (int)KQ_Q6_K})
    for (int rs : {1, 2, 4, 8})
      for (int mc : {1, 2, 4})
        for (bool wide : {false, true}) {
          KqFn f = kq_pick(fmt, rs, mc, wide);
          if (!f) continue;
          cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
          if (e != cudaSuccess) return e;
        }
  return cudaSuccess;
}

cudaError_t launch_kq_gemv(int fmt, const KqArgs& a, const KqLaunch& l, cudaStream_t s) {
  KqFn f = kq_pick(fmt, l.rs, l.mc, l.wide != 0);
  if (!f || l.grid < 1 || l.ns > 16 || l.nwc < 1 || l.nwc > kMaxWarps || a.cols % 256 || !a.w || !a.x || !a.y ||
      (fmt == KQ_Q6_K && !a.d6))
    return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.w) | reinterpret_cast<uintptr_t>(a.d6) | reinterpret_cast<uintptr_t>(a.x)) & 15)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.grid);
  cfg.blockDim = dim3(l.threads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see the kernel's griddep calls
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f, a, l);
}

}  // namespace dls

// ---- C ABI ------------------------------------------------------------------------

namespace {

bool kq_type_ok(int32_t type) { return type == DLS_Q4_K || type == DLS_Q5_K || type == DLS_Q6_K; }

std::mutex g_kq_mu;
std::map<std::tuple<int, int, int, int>, dls::KqLaunch> g_kq_plans;  // (device, type, rows, cols)
bool g_kq_attr[64] = {};

// The launch plan of one shape on the current device (cached), with the
// kernels' shared-memory limit raised once per device.
int kq_launch_for(int32_t type, int32_t rows, int32_t cols, dls::KqLaunch* out) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return dls::report_error(DLS_ERR_CUDA, "kquant: no current device");
  std::lock_guard<std::mutex> g(g_kq_mu);
  if (dev >= 0 && dev < 64 && !g_kq_attr[dev]) {
    if (dls::kq_setup_attributes() != cudaSuccess) return dls::report_error(DLS_ERR_CUDA, "kquant: attributes");
    g_kq_attr[dev] = true;
  }
  const auto key = std::make_tuple(dev, (int)type, (int)rows, (int)cols);
  auto it = g_kq_plans.find(key);
  if (it == g_kq_plans.end()) it = g_kq_plans.emplace(key, dls::kq_plan(type, rows, cols, sms)).first;
  if (it->second.grid < 1)
    return dls::report_error(DLS_ERR_ARG, "kquant: unsupported shape type=%d rows=%d cols=%d", type, rows, cols);
  *out = it->second;
  return DLS_OK;
}

}  // namespace

extern "C" uint64_t dls_kquant_packed_bytes(int32_t type, int32_t rows, int32_t cols) {
  if (!kq_type_ok(type) || rows < 1 || cols < 256 || cols % 256) return 0;
  return dls::kq_packed_bytes(type, rows, cols);
}

extern "C" int dls_kquant_pack(int32_t type, const void* blocks, int32_t rows, int32_t cols, void* packed,
                               void* cuda_stream) {
  if (!kq_type_ok(type) || rows < 1 || cols < 256 || cols % 256 || !blocks || !packed)
    return dls::report_error(DLS_ERR_ARG, "kquant pack: type=%d rows=%d cols=%d", type, rows, cols);
  if (reinterpret_cast<uintptr_t>(packed) & 255)
    return dls::report_error(DLS_ERR_ARG, "kquant pack: the packed buffer must be 256-byte aligned");
  const cudaError_t e = dls::launch_kq_pack(type, blocks, rows, cols, packed, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return dls::report_error(DLS_ERR_CUDA, "kquant pack: cuda=%s", cudaGetErrorString(e));
  return DLS_OK;
}

extern "C" int dls_kquant_gemv(int32_t type, const void* packed, int32_t rows, int32_t cols, const float* x,
                               float* y, int32_t* status, void* cuda_stream) {
  if (!kq_type_ok(type) || rows < 1 || cols < 256 || cols % 256 || !packed || !x || !y)
    return dls::report_error(DLS_ERR_ARG, "kquant gemv: type=%d rows=%d cols=%d", type, rows, cols);
  if ((reinterpret_cast<uintptr_t>(packed) & 255) || (reinterpret_cast<uintptr_t>(x) & 15))
    return dls::report_error(DLS_ERR_ARG, "kquant gemv: packed must be 256-byte and x 16-byte aligned");
  dls::KqLaunch l;
  const int r = kq_launch_for(type, rows, cols, &l);
  if (r != DLS_OK) return r;
  dls::KqArgs a{};
  a.w = static_cast<const uint8_t*>(packed);
  a.d6 = type == DLS_Q6_K ? dls::kq_d6(packed, rows, cols) : nullptr;
  a.rows = rows;
  a.cols = cols;
  a.x = x;
  a.y = y;
  a.status = status;
  const cudaError_t e = dls::launch_kq_gemv(type, a, l, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return dls::report_error(DLS_ERR_CUDA, "kquant gemv: cuda=%s", cudaGetErrorString(e));
  return DLS_OK;
}
