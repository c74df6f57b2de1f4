// Shared device helpers and launch structures of the decode-step library.
// sm_103a only: packed fp32 (f32x2) arithmetic, programmatic dependent launch
// (griddepcontrol), bulk L2 prefetch, non-allocating streaming loads.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dls {

constexpr int kMaxBatch = 8;

// Per-step inputs read by the kernels from device memory, so that one
// captured CUDA graph serves every position.  Written by set_params_kernel
// (decode) or advanced in place by argmax_kernel (greedy generation).
struct StepParams {
  int32_t n;                   // batch rows in this step
  int32_t token[kMaxBatch];
  int32_t pos[kMaxBatch];      // position of the new token (= KV length before the step)
  int32_t seq[kMaxBatch];
  int32_t step;                // generation step counter (argmax output slot)
  int32_t status;              // nonzero: a kernel saw an invalid index (bit flags)
  int32_t shared_len;          // batched steps: leading positions every row holds in the same KV pages (a
                               // multiple of 32; their attention runs once for all rows), 0 = none
};

enum StatusBits : int32_t {
  kBadPage = 1,   // page table entry missing for a position being written/read
  kBadToken = 2,  // token id outside [0, vocab)
  kBadPos = 4,    // position outside the rope table / context
  kTimeout = 8,   // a bounded wait on an mbarrier ran out
};

// One weight matrix in the kernels' layout: codes and fp16 scales in two
// arrays ("structure of arrays"), so rows of codes are contiguous, 16-byte
// aligned and can be moved by bulk copies.
//   Q8_0: qs u8 [rows][nb*32] holding q + 128                d fp16 [rows][ds]
//   Q4_0: qs u8   [rows][nb][16] (GGUF nibble order kept)   d fp16 [rows][ds]
struct MatDev {
  const uint8_t* qs;
  const __half* d;
  int rows, cols, nb;
  int ds;     // scale row stride in elements: nb rounded up to 8 (16-byte rows)
  int rstep;  // storage rows per logical row (2 for one half of an interleaved pair); GEMVs need 1
};

// ---- small PTX wrappers -----------------------------------------------------

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  // bytes: multiple of 16, address 16-byte aligned
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// one 128-byte line into L2 (a hint issued by one thread)
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

typedef unsigned long long f2_t;  // two fp32 lanes in one 64-bit register pair

__device__ __forceinline__ f2_t pk2(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk2(f2_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f2_t ffma2(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t fadd2(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- exact int8 / int4 -> fp32 --------------------------------------------------
// A byte b placed in the low byte of the pattern 0x4B0000bb is the float
// 2^23 + b exactly; subtracting 2^23 + bias recovers the signed code with no
// rounding.  One PRMT per value and one packed add per two values.

__device__ __forceinline__ float mag_byte(uint32_t u, int k) {
  return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540 | k));
}

// four biased Q8_0 codes (q + 128 per byte, one 32-bit word) -> (q0,q1), (q2,q3)
__device__ __forceinline__ void i8x4_to_f2(uint32_t u, float2& p01, float2& p23) {
  const float2 bias = make_float2(-8388736.0f, -8388736.0f);
  p01 = __fadd2_rn(make_float2(mag_byte(u, 0), mag_byte(u, 1)), bias);
  p23 = __fadd2_rn(make_float2(mag_byte(u, 2), mag_byte(u, 3)), bias);
}

// two-way integer dot: c + a.lo16*b.byte(0|2) + a.hi16*b.byte(1|3), a signed
// 16-bit pair, b unsigned bytes; exact in int32
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// four nibble codes already isolated one per byte (values 0..15) -> (n-8)
__device__ __forceinline__ void u4x4_to_f2(uint32_t b, float2& p01, float2& p23) {
  const float2 bias = make_float2(-8388616.0f, -8388616.0f);  // 2^23 + 8
  p01 = __fadd2_rn(make_float2(mag_byte(b, 0), mag_byte(b, 1)), bias);
  p23 = __fadd2_rn(make_float2(mag_byte(b, 2), mag_byte(b, 3)), bias);
}

// ---- mbarrier + bulk async copy (TMA, non-tensor form) ---------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of an mbarrier, backing off with `sleep_ns` naps
// after a few polls so a waiting warp does not take issue slots from working
// ones; gives up after `limit_ns` of global time and returns false (the
// caller records an error and stops).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t sleep_ns = 20,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 4) __nanosleep(sleep_ns);
    if ((i & 63) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes and
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// shared-memory loads by 32-bit shared address
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_half_as_float(uint32_t a) {
  uint16_t h;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace dls
