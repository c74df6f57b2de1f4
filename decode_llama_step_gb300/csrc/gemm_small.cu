// Small-batch dequantising GEMM on the 5th-generation tensor cores, for a
// batched decode step of up to 8 rows (each weight byte read once for all of
// them):
//   y[t, m] = sum_b d[m, b] * sum_{k in block b} q[m, k] x[t, k]
// with Q8_0 / Q4_0 codes q (exact small integers), per-32-column block
// scales d (fp16) and fp32 activations x.
//
// Why not the prefill GEMM's scheme (w = fp16(d q) split into hi + lo
// planes): with 8 tokens per weight pass the tensor cores idle and the CUDA
// cores writing two fp16 planes per weight into shared memory set the pace.
// Here the codes enter the MMA as they are, converted to fp16 (exact), and
// the scale is applied per block after the MMA, in fp32:
//   * the activations are the two fp16 planes x_hi = fp16(x), x_lo =
//     fp16(x - x_hi), packed as the 16 columns of one N = 16 operand (tokens
//     0-7 hi, then 0-7 lo): the products q x_hi, q x_lo are exact in the fp32
//     accumulator;
//   * each 32-column block's two MMAs (K = 16 each) land in a tensor-memory
//     region of their own;
//   * epilogue warps read the region (tcgen05.ld), add the hi and lo
//     columns and accumulate d * (sum) into fp32 registers, one weight row
//     per thread, then free the region.
//
// One CTA: 128 weight rows x up to 8 tokens over a range of 64-column K
// steps (split-K across CTAs as in the prefill GEMM; partial sums meet in a
// workspace and the last CTA of a tile adds them in split order).
//   warp 0     TMA: per K step, the two 8-token activation planes (128-byte
//              swizzle, rows 0-7 and 8-15 of the MMA's B operand), the raw
//              codes of 128 weight rows and their scales
//   warp 1     tensor-memory owner; one thread issues the MMAs
//   warps 2-5  convert: one thread per weight row turns its 64 codes into
//              fp16 (exact) in the MMA's A layout and copies the row's two
//              block scales for the epilogue
//   warps 6-9  epilogue: per K step, scale and accumulate the two blocks
// Every wait is bounded (2 s); a wait that gives up sets an abort flag that
// all roles see, the kernel stores nothing and reports kTimeout.
#include <cuda.h>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int SBM = 128, SBK = 64;     // weight rows per CTA, K per step
constexpr int STHREADS = 320;
constexpr int kSR = 8;                 // tensor-memory regions (K steps in flight between MMA and epilogue)
constexpr int kSSplitMax = 16;
constexpr uint64_t kWaitNsS = 2000000000ull;
constexpr int kSATile = SBM * SBK * 2;  // 16 KB fp16 A operand

template <int WT>
struct SCfg {
  static constexpr int kCodes = WT == 8 ? SBM * 64 : SBM * 32;
  static constexpr int kB = 2048;                          // 16 rows (8 hi + 8 lo) x 128 bytes
  static constexpr int kStage = kB + kCodes + SBM * 16;     // B | codes | scales (8 per row)
  static constexpr int NR = WT == 8 ? 5 : 8;  // ring stages: the bytes in flight set the pace
  static constexpr int NA = 2;                // A tiles: converts run at most two steps ahead of the MMA
  static constexpr int kScOff = NA * kSATile + NR * kStage;  // float2 scales [kSR][SBM]
  static constexpr int kBarOff = kScOff + kSR * SBM * 8;
  static constexpr int kSmem = kBarOff + 512 + 1024;
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
  static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
};

template <int NR, int NA>
struct SBars {
  uint64_t rfull[NR], rempty[NR], afull[NA], aempty[NA], tfull[kSR], tfree[kSR], sfull[kSR];
  uint32_t tmem;
  int abort;
  int last;
};

__device__ __forceinline__ bool swait(uint32_t bar, uint32_t parity, int* abort_flag, bool heed_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 63) == 0) {
      if (heed_abort && *(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsS) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t lds32s(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// two codes (bytes selected from u) -> two exact fp16 values (byte - bias)
__device__ __forceinline__ uint32_t cv2(uint32_t u, uint32_t sel, __half2 bias) {
  const uint32_t p = __byte_perm(u, 0x64646464u, sel);  // fp16 1024 + byte in each half
  const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&p), bias);
  return *reinterpret_cast<const uint32_t*>(&q);
}

// Row r of one K step: its codes at `qrow` (swizzled by the TMA) -> 64 fp16
// codes at `arow` (128-byte swizzle, the MMA's A layout).  `kval`: columns
// of this step inside the matrix (the rest are written as zeros).
template <int WT>
__device__ __forceinline__ void convert_row(uint32_t qrow, uint32_t arow, int r, int kval) {
  const int sw = r & 7;
  if (WT == 8) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1024 + 128
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 16 codes: columns 16c .. 16c+15
      uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
      if (16 * c < kval) {
        const uint4 u = lds128(qrow + ((c ^ ((r >> 1) & 3)) << 4));
        o0 = make_uint4(cv2(u.x, 0x4140u, bias), cv2(u.x, 0x4342u, bias), cv2(u.y, 0x4140u, bias),
                        cv2(u.y, 0x4342u, bias));
        o1 = make_uint4(cv2(u.z, 0x4140u, bias), cv2(u.z, 0x4342u, bias), cv2(u.w, 0x4140u, bias),
                        cv2(u.w, 0x4342u, bias));
      }
      sts128(arow + (((2 * c) ^ sw) << 4), o0);
      sts128(arow + (((2 * c + 1) ^ sw) << 4), o1);
    }
  } else {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1024 + 8
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {  // one 16-byte block: low nibbles = columns 0-15, high = 16-31
      const bool in = 32 * hf < kval;
      const uint4 u = in ? lds128(qrow + ((hf ^ ((r >> 2) & 1)) << 4)) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // output chunk j: columns 8j .. 8j+7 of the block
        const uint32_t a = w[(2 * j) & 3], b = w[(2 * j + 1) & 3];
        const uint32_t sa = j < 2 ? a & 0x0F0F0F0Fu : (a >> 4) & 0x0F0F0F0Fu;
        const uint32_t sb = j < 2 ? b & 0x0F0F0F0Fu : (b >> 4) & 0x0F0F0F0Fu;
        uint4 o = make_uint4(cv2(sa, 0x4140u, bias), cv2(sa, 0x4342u, bias), cv2(sb, 0x4140u, bias),
                             cv2(sb, 0x4342u, bias));
        if (!in) o = make_uint4(0, 0, 0, 0);
        sts128(arow + (((4 * hf + j) ^ sw) << 4), o);
      }
    }
  }
}

template <int EPI>
__device__ __forceinline__ void sepi_store(const PgArgs& a, int t, int m, int rows, float v) {
  if (EPI == EPI_SWIGLU) {
    const float up = __shfl_down_sync(0xffffffffu, v, 1);
    if ((threadIdx.x & 1) == 0 && t < a.T && m + 1 < rows) {
      const float hv = silu(v) * up;
      const __half hh = __float2half_rn(hv);
      a.h[(size_t)t * a.ldh + (m >> 1)] = hh;
      a.hlo[(size_t)t * a.ldh + (m >> 1)] = __float2half_rn(hv - __half2float(hh));
    }
  } else if (t < a.T && m < rows) {
    float* dst = a.y + (size_t)t * a.ldy + m;
    if (EPI == EPI_RESID) *dst += v;
    else *dst = v;
  }
}

template <int WT, int EPI>
__global__ void __launch_bounds__(STHREADS) sgemm_kernel(const __grid_constant__ CUtensorMap tm_xh,
                                                         const __grid_constant__ CUtensorMap tm_xl,
                                                         const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_d, const PgArgs a) {
  using C = SCfg<WT>;
  using Bars = SBars<C::NR, C::NA>;
  extern __shared__ uint8_t ssm[];
  const uint32_t raw = smem_u32(ssm);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t abase = raw + pad;                // NA fp16 A tiles
  const uint32_t rbase = abase + C::NA * kSATile;  // NR stages: B | codes | scales
  float2* sc = reinterpret_cast<float2*>(ssm + pad + C::kScOff);  // [kSR][SBM] block scales
  Bars& sh = *reinterpret_cast<Bars*>(ssm + pad + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev& w = a.w;
  const int m0 = blockIdx.y * SBM;
  const int kpad = w.nb * 32;
  const int nk_all = (kpad + SBK - 1) / SBK;
  const int S = gridDim.z, z = blockIdx.z;
  const int kt0 = (int)((long long)nk_all * z / S);
  const int nk = (int)((long long)nk_all * (z + 1) / S) - kt0;  // >= 1: the host keeps S <= nk_all

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem), 32 * kSR);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < C::NR; ++i) {
      mbar_init(smem_u32(&sh.rfull[i]), 1);
      mbar_init(smem_u32(&sh.rempty[i]), 1);
    }
    for (int i = 0; i < C::NA; ++i) {
      mbar_init(smem_u32(&sh.afull[i]), 4);
      mbar_init(smem_u32(&sh.aempty[i]), 1);
    }
    for (int i = 0; i < kSR; ++i) {
      mbar_init(smem_u32(&sh.tfull[i]), 1);
      mbar_init(smem_u32(&sh.tfree[i]), 4);
      mbar_init(smem_u32(&sh.sfull[i]), 4);
    }
    sh.abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_xh);
    prefetch_tmap(&tm_xl);
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_d);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  // Programmatic dependent launch: the next kernel in the stream may start
  // its prologue now (it waits for this grid's completion before it reads
  // what this one writes); this one's weights stream before its own wait.
  griddep_launch();

  if (warp == 0) {
    // ---------------- TMA producer: the first stages' codes and scales go
    // out before the wait on the previous kernel (they do not depend on it),
    // the activations after it
    if (lane == 0) {
      int issued = 0;
      const int pre = nk < C::NR ? nk : C::NR;
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = rbase + i * C::kStage;
        const uint32_t bar = smem_u32(&sh.rfull[i]);
        const int kt = kt0 + i;
        mbar_expect_tx(bar, C::kStage);
        tma_load_2d(st + C::kB, &tm_q, kt * (WT == 8 ? 64 : 32), m0, bar);
        tma_load_2d(st + C::kB + C::kCodes, &tm_d, (kt * 2) & ~7, m0, bar);
      }
      griddep_wait();
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = rbase + i * C::kStage;
        const uint32_t bar = smem_u32(&sh.rfull[i]);
        const int kt = kt0 + i;
        tma_load_2d(st, &tm_xh, kt * SBK, 0, bar);
        tma_load_2d(st + 1024, &tm_xl, kt * SBK, 0, bar);
        issued = i + 1;
      }
      for (int i = pre; i < nk; ++i) {
        const int s = i % C::NR;
        if (!swait(smem_u32(&sh.rempty[s]), ((i / C::NR) - 1) & 1, &sh.abort)) break;
        const uint32_t st = rbase + s * C::kStage;
        const uint32_t bar = smem_u32(&sh.rfull[s]);
        const int kt = kt0 + i;
        mbar_expect_tx(bar, C::kStage);
        tma_load_2d(st, &tm_xh, kt * SBK, 0, bar);
        tma_load_2d(st + 1024, &tm_xl, kt * SBK, 0, bar);
        tma_load_2d(st + C::kB, &tm_q, kt * (WT == 8 ? 64 : 32), m0, bar);
        tma_load_2d(st + C::kB + C::kCodes, &tm_d, (kt * 2) & ~7, m0, bar);
        issued = i + 1;
      }
      // copies still in flight (after an abort) land before the CTA exits
      for (int i = issued > C::NR ? issued - C::NR : 0; i < issued; ++i)
        swait(smem_u32(&sh.rfull[i % C::NR]), (i / C::NR) & 1, &sh.abort, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue: two 16-wide K slices per 32-column block,
    // block 0 of the step into columns 32r .. 32r+15, block 1 into +16
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16(SBM, 16);
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::NR, ai = i % C::NA, r = i % kSR;
        if (!swait(smem_u32(&sh.afull[ai]), (i / C::NA) & 1, &sh.abort)) break;
        if (!swait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t sa = abase + ai * kSATile, sb = rbase + s * C::kStage;
#pragma unroll
        for (int ks = 0; ks < SBK / 16; ++ks)
          umma_f16(tmem + 32 * r + 16 * (ks >> 1), umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + ks * 32), idesc,
                   ks & 1);
        umma_commit(smem_u32(&sh.rempty[s]));
        umma_commit(smem_u32(&sh.aempty[ai]));
        umma_commit(smem_u32(&sh.tfull[r]));
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- convert: thread = weight row
    const int r = tid - 64;
    for (int i = 0; i < nk; ++i) {
      const int s = i % C::NR, ai = i % C::NA, rg = i % kSR;
      if (!swait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
      if (i >= C::NA && !swait(smem_u32(&sh.aempty[ai]), ((i / C::NA) - 1) & 1, &sh.abort)) break;
      if (i >= kSR && !swait(smem_u32(&sh.tfree[rg]), ((i / kSR) - 1) & 1, &sh.abort)) break;
      const int kt = kt0 + i;
      const uint32_t st = rbase + s * C::kStage;
      const uint32_t dsc = lds32s(st + C::kB + C::kCodes + r * 16 + (((kt * 2) & 7) << 1));
      const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&dsc));
      sc[rg * SBM + r] = dd;
      convert_row<WT>(st + C::kB + r * (WT == 8 ? 64 : 32), abase + ai * kSATile + r * 128, r, kpad - kt * SBK);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.sfull[rg]));  // the block scales, straight to the epilogue
        mbar_arrive(smem_u32(&sh.afull[ai]));
      }
    }
  } else {
    // ---------------- epilogue: thread = weight row (its TMEM lane); it
    // reads and writes what neighbouring kernels touch, so only after the
    // previous kernel has completed
    griddep_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int m = m0 + row;
    float y[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) y[t] = 0.f;
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int rg = i % kSR;
      ok = swait(smem_u32(&sh.sfull[rg]), (i / kSR) & 1, &sh.abort) &&
           swait(smem_u32(&sh.tfull[rg]), (i / kSR) & 1, &sh.abort);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[16], u[16];
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + 32 * rg;
      tmem_ld16(taddr, v);
      tmem_ld16(taddr + 16, u);
      tmem_wait_ld();
      const float2 dd = sc[rg * SBM + row];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        y[t] = fmaf(dd.x, __uint_as_float(v[t]) + __uint_as_float(v[t + 8]), y[t]);
        y[t] = fmaf(dd.y, __uint_as_float(u[t]) + __uint_as_float(u[t + 8]), y[t]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.tfree[rg]));
    }
    ok = __all_sync(0xffffffffu, ok && !*(volatile int*)&sh.abort);
    if (S == 1) {
      if (ok)
#pragma unroll
        for (int t = 0; t < 8; ++t) sepi_store<EPI>(a, t, m, w.rows, y[t]);
    } else {
      // partials -> workspace [S][T][rows]; the last CTA of the tile adds them in split order
      if (ok && m < w.rows)
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (t < a.T) a.part[((size_t)z * a.T + t) * w.rows + m] = y[t];
      __threadfence();
      named_bar(1, 128);
      if (warp == 6 && lane == 0) {
        const int prev = atomicAdd(&a.counters[blockIdx.y], 1);
        sh.last = prev == S - 1;
        if (sh.last) a.counters[blockIdx.y] = 0;  // ready for the next launch
      }
      named_bar(1, 128);
      if (sh.last && ok) {
        __threadfence();
        float acc[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = 0.f;
        for (int zz = 0; zz < S; ++zz)
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (t < a.T && m < w.rows) acc[t] += __ldcg(&a.part[((size_t)zz * a.T + t) * w.rows + m]);
#pragma unroll
        for (int t = 0; t < 8; ++t) sepi_store<EPI>(a, t, m, w.rows, acc[t]);
      }
    }
    if (!ok && a.status && lane == 0) atomicOr(a.status, kTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 32 * kSR);
  }
}

using SgFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const PgArgs);

template <int WT>
SgFn sg_pick(int epi) {
  switch (epi) {
    case EPI_STORE: return sgemm_kernel<WT, EPI_STORE>;
    case EPI_RESID: return sgemm_kernel<WT, EPI_RESID>;
    case EPI_SWIGLU: return sgemm_kernel<WT, EPI_SWIGLU>;
  }
  return nullptr;
}

SgFn sg_select(int wtype, int epi, int* smem) {
  if (wtype == 8) {
    *smem = SCfg<8>::kSmem;
    return sg_pick<8>(epi);
  }
  *smem = SCfg<4>::kSmem;
  return sg_pick<4>(epi);
}

}  // namespace

cudaError_t sgemm_setup_attributes() {
  for (int wt : {8, 4})
    for (int e : {EPI_STORE, EPI_RESID, EPI_SWIGLU}) {
      int smem = 0;
      SgFn f = sg_select(wt, e, &smem);
      cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
  return cudaSuccess;
}

cudaError_t launch_sgemm(int wtype, int epi, const PgArgs& a, int split, cudaStream_t s) {
  const MatDev& w = a.w;
  const int kpad = w.nb * 32;
  const int nk = (kpad + SBK - 1) / SBK;
  if (a.kx % 8 || a.kx < kpad || a.T < 1 || a.T > 8 || w.rstep != 1 || split < 1 || split > nk || !a.xlo ||
      split > kSSplitMax)
    return cudaErrorInvalidValue;
  if (split > 1 && (!a.part || !a.counters)) return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && !a.hlo) return cudaErrorInvalidValue;
  int smem = 0;
  SgFn f = sg_select(wtype, epi, &smem);
  if (!f) return cudaErrorInvalidValue;
  CUtensorMap th, tl, tq, td;
  const uint64_t rb = wtype == 8 ? (uint64_t)w.nb * 32 : (uint64_t)w.nb * 16;
  if (!make_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, SBK, 8,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.xlo, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, SBK,
                    8, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.qs, rb, (uint64_t)w.rows, rb, wtype == 8 ? 64 : 32, SBM,
                    wtype == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.d, (uint64_t)w.ds, (uint64_t)w.rows, (uint64_t)w.ds * 2, 8,
                    SBM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, (w.rows + SBM - 1) / SBM, split);
  cfg.blockDim = dim3(STHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f, th, tl, tq, td, a);
}

}  // namespace dls
