// Device building blocks shared by the decode GEMV kernel and the
// persistent decode-step kernel: chunk geometry, the per-lane dot product of
// 16 code bytes with the lane's activations, and the cross-lane reduction.
#pragma once
#include "common.cuh"

namespace dls {

template <int WT>
struct Geo {
  static constexpr int CH = WT == 8 ? 512 : 1024;   // columns per chunk
  static constexpr int XV = WT == 8 ? 8 : 16;       // x pairs per lane per chunk
  static constexpr int MCMAX = WT == 8 ? 4 : 2;     // max chunks per warp (register budget)
};

template <int RS>
__device__ __forceinline__ float butterfly(float (&acc)[RS], int lane) {
  // After this, lane holds the warp total of row (lane >> (5 - log2 RS)).
  if (RS == 1) return warp_sum(acc[0]);
  float v[RS];
#pragma unroll
  for (int i = 0; i < RS; ++i) v[i] = acc[i];
  int n = RS, off = 16;
#pragma unroll
  for (; n > 1; n >>= 1, off >>= 1) {
    const bool hi = lane & off;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = hi ? v[j] : v[n / 2 + j];
      const float keep = hi ? v[n / 2 + j] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float t = v[0];
#pragma unroll
  for (; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  return t;
}

// A lane's activation slice for one chunk as int16 pairs (element 2e in the
// low half of p[e]) with one scale: x_i ~= s * X_i, |X_i| <= 32767, so the
// code-activation products are exact int32 dot products (dp2a) and the error
// is at most s/2 per element (2^-16 of the slice's largest magnitude).
// corr = bias * sum(X) removes the code bias (128 for Q8_0, 8 for Q4_0).
template <int WT>
struct XQ {
  static constexpr int N = WT == 8 ? 8 : 16;  // int16 pairs (16 or 32 elements)
  uint32_t p[N];
  float s;
  int corr;
};

template <int WT>
__device__ __forceinline__ void quantize_slice(const float* v, XQ<WT>& xq) {
  constexpr int n = 2 * XQ<WT>::N;
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < n; ++i) mx = fmaxf(mx, fabsf(v[i]));
  const float s = mx > 0.f ? mx / 32767.0f : 1.0f;
  const float inv = 1.0f / s;
  int sum = 0;
#pragma unroll
  for (int e = 0; e < XQ<WT>::N; ++e) {
    const int a = __float2int_rn(v[2 * e] * inv), b = __float2int_rn(v[2 * e + 1] * inv);
    sum += a + b;
    xq.p[e] = (uint32_t)(a & 0xFFFF) | ((uint32_t)b << 16);
  }
  xq.s = s;
  xq.corr = sum * (WT == 8 ? 128 : 8);
}

// integer dot of one lane's 16 code bytes with its quantised activations:
// sum_i q_i X_i exactly (two accumulator chains)
template <int WT>
__device__ __forceinline__ int idot16(uint4 q, const XQ<WT>& xq) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  int s0 = 0, s1 = 0;
  if (WT == 8) {  // bytes hold q + 128
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s0 = dp2a_lo(xq.p[2 * k], w[k], s0);
      s1 = dp2a_hi(xq.p[2 * k + 1], w[k], s1);
    }
  } else {  // byte j: element j in the low nibble, j + 16 in the high nibble
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = w[k] & 0x0F0F0F0Fu, hi = (w[k] >> 4) & 0x0F0F0F0Fu;
      s0 = dp2a_lo(xq.p[2 * k], lo, s0);
      s1 = dp2a_hi(xq.p[2 * k + 1], lo, s1);
      s0 = dp2a_lo(xq.p[8 + 2 * k], hi, s0);
      s1 = dp2a_hi(xq.p[8 + 2 * k + 1], hi, s1);
    }
  }
  return s0 + s1 - xq.corr;
}

// dot of 16 code bytes (one lane's slice of one row) with its activations
// Two independent accumulator chains per call keep the FMA pipe fed.
template <int WT>
__device__ __forceinline__ float dot16(uint4 q, const float2* xr) {
  float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if (WT == 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 p01, p23;
      i8x4_to_f2(w[k], p01, p23);
      s0 = __ffma2_rn(p01, xr[2 * k], s0);
      s1 = __ffma2_rn(p23, xr[2 * k + 1], s1);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bytes 4k..: low nibbles = elements 4k.., high = 16+4k..
      float2 a01, a23, b01, b23;
      u4x4_to_f2(w[k] & 0x0F0F0F0Fu, a01, a23);
      u4x4_to_f2((w[k] >> 4) & 0x0F0F0F0Fu, b01, b23);
      s0 = __ffma2_rn(a01, xr[2 * k], s0);
      s1 = __ffma2_rn(a23, xr[2 * k + 1], s1);
      s0 = __ffma2_rn(b01, xr[8 + 2 * k], s0);
      s1 = __ffma2_rn(b23, xr[8 + 2 * k + 1], s1);
    }
  }
  const float2 s = __fadd2_rn(s0, s1);
  return s.x + s.y;
}


}  // namespace dls
