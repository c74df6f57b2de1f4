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

// dot of 16 code bytes (one lane's slice of one row) with its activations
template <int WT>
__device__ __forceinline__ float dot16(uint4 q, const float2* xr) {
  float2 s = make_float2(0.f, 0.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if (WT == 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 p01, p23;
      i8x4_to_f2(w[k], p01, p23);
      s = __ffma2_rn(p01, xr[2 * k], s);
      s = __ffma2_rn(p23, xr[2 * k + 1], s);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bytes 4k..: low nibbles = elements 4k.., high = 16+4k..
      float2 a01, a23, b01, b23;
      u4x4_to_f2(w[k] & 0x0F0F0F0Fu, a01, a23);
      u4x4_to_f2((w[k] >> 4) & 0x0F0F0F0Fu, b01, b23);
      s = __ffma2_rn(a01, xr[2 * k], s);
      s = __ffma2_rn(a23, xr[2 * k + 1], s);
      s = __ffma2_rn(b01, xr[8 + 2 * k], s);
      s = __ffma2_rn(b23, xr[8 + 2 * k + 1], s);
    }
  }
  return s.x + s.y;
}


}  // namespace dls
