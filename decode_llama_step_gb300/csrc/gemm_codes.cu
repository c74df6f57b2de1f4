// Prompt-chunk dequantising GEMM on the 5th-generation tensor cores with the
// weight codes as exact MMA operands:
//   y[t, m] = sum_b d[m, b] * sum_{k in block b} q[m, k] x[t, k]
// Q8_0 / Q4_0 codes q are small integers, exact in fp16; the activations
// enter as two fp16 planes x_hi = fp16(x), x_lo = fp16(x - x_hi) whose
// products with q are exact in the fp32 accumulator; the per-32-column block
// scale d is applied afterwards, in fp32, by the epilogue warps.  Two MMAs
// (x_hi, x_lo) per 16-column K slice, accumulated into the same tensor-memory
// region, carry the full product to ~2^-22 of each operand; the scheme of the
// first prefill GEMM (fp16 weight planes w_hi + w_lo, three MMAs per slice)
// needs 1.5x the tensor work and CUDA-core time to write two weight planes.
//
// CTA = 128 weight rows x 128 tokens over the whole K range:
//   warp 0       TMA: per 64-column K step the two activation planes of the
//                128 tokens (128-byte swizzle, the MMA's B operand), the raw
//                codes of the 128 rows and their block scales
//   warp 1       tensor-memory owner; one thread issues the MMAs: each
//                32-column block of a step into a 128-column region of its
//                own (two regions per step, two steps in flight)
//   warps 2-5    convert: thread = weight row; 64 codes -> fp16 in the A
//                layout (128-byte swizzle), the row's two block scales
//   warps 6-21   epilogue: thread = (weight row, 32 tokens); reads its
//                columns of both block regions of a step (tcgen05.ld, one
//                wait), y += d * region, frees the regions;
//                at the end stores y (plain, residual add, or SwiGLU over the
//                interleaved gate/up rows into the fp16 h planes)
// Every wait is bounded (2 s); a wait that gives up sets an abort flag that
// all roles see, the kernel stores nothing and reports kTimeout.
#include <cuda.h>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int CBM = 128, CBN = 128, CBK = 64;
constexpr int kCEpiWarps = 16;          // epilogue warps: (lane quarter, 32-token group)
constexpr int CTHREADS = 32 * (6 + kCEpiWarps);
constexpr int kCR = 2;                 // tensor-memory step regions (256 columns each)
constexpr int kCNA = 2;                // fp16 A tiles
constexpr uint64_t kWaitNsC = 2000000000ull;
constexpr int kCATile = CBM * CBK * 2;  // 16 KB

template <int WT>
struct CCfg {
  static constexpr int kX = CBN * 128;                      // one activation plane: 128 tokens x 64 fp16
  static constexpr int kCodes = WT == 8 ? CBM * 64 : CBM * 32;
  static constexpr int kStage = 2 * kX + kCodes + CBM * 16;  // x_hi | x_lo | codes | scales (8 per row)
  static constexpr int NR = 4;
  static constexpr int kScOff = kCNA * kCATile + NR * kStage;  // float2 scales [kCR][CBM]
  static constexpr int kBarOff = kScOff + kCR * CBM * 8;
  static constexpr int kSmem = kBarOff + 512 + 1024;
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
  static_assert(kSmem <= 227 * 1024, "one CTA per SM");
};

template <int NR>
struct CBars {
  uint64_t rfull[NR], rempty[NR], afull[kCNA], aempty[kCNA], tfull[kCR], tfree[kCR], sfull[kCR];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool cwait(uint32_t bar, uint32_t parity, int* abort_flag, bool heed_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 63) == 0) {
      if (heed_abort && *(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsC) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t lds32c(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// two codes (bytes selected from u) -> two exact fp16 values (byte - bias)
__device__ __forceinline__ uint32_t cvc(uint32_t u, uint32_t sel, __half2 bias) {
  const uint32_t p = __byte_perm(u, 0x64646464u, sel);  // fp16 1024 + byte in each half
  const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&p), bias);
  return *reinterpret_cast<const uint32_t*>(&q);
}

// Row r of one K step: its codes at `qrow` (swizzled by the TMA: 64-byte rows
// for Q8_0, 32-byte rows for Q4_0) -> 64 fp16 codes at `arow` (128-byte
// swizzle, the MMA's A layout).  `kval`: columns of this step inside the
// matrix (the rest are written as zeros).
template <int WT>
__device__ __forceinline__ void convert_codes(uint32_t qrow, uint32_t arow, int r, int kval) {
  const int sw = r & 7;
  if (WT == 8) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1024 + 128
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 16 codes: columns 16c .. 16c+15
      uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
      if (16 * c < kval) {
        const uint4 u = lds128(qrow + ((c ^ ((r >> 1) & 3)) << 4));
        o0 = make_uint4(cvc(u.x, 0x4140u, bias), cvc(u.x, 0x4342u, bias), cvc(u.y, 0x4140u, bias),
                        cvc(u.y, 0x4342u, bias));
        o1 = make_uint4(cvc(u.z, 0x4140u, bias), cvc(u.z, 0x4342u, bias), cvc(u.w, 0x4140u, bias),
                        cvc(u.w, 0x4342u, bias));
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
        uint4 o = make_uint4(cvc(sa, 0x4140u, bias), cvc(sa, 0x4342u, bias), cvc(sb, 0x4140u, bias),
                             cvc(sb, 0x4342u, bias));
        if (!in) o = make_uint4(0, 0, 0, 0);
        sts128(arow + (((4 * hf + j) ^ sw) << 4), o);
      }
    }
  }
}

template <int EPI>
__device__ __forceinline__ void cepi_store(const PgArgs& a, int t, int m, int rows, float v) {
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
__global__ void __launch_bounds__(CTHREADS, 1) cgemm_kernel(const __grid_constant__ CUtensorMap tm_xh,
                                                            const __grid_constant__ CUtensorMap tm_xl,
                                                            const __grid_constant__ CUtensorMap tm_q,
                                                            const __grid_constant__ CUtensorMap tm_d, const PgArgs a) {
  using C = CCfg<WT>;
  using Bars = CBars<C::NR>;
  extern __shared__ uint8_t csm[];
  const uint32_t raw = smem_u32(csm);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t abase = raw + pad;                  // kCNA fp16 A tiles
  const uint32_t rbase = abase + kCNA * kCATile;     // NR stages: x_hi | x_lo | codes | scales
  float2* sc = reinterpret_cast<float2*>(csm + pad + C::kScOff);  // [kCR][CBM] block scales
  Bars& sh = *reinterpret_cast<Bars*>(csm + pad + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev& w = a.w;
  const int n0 = blockIdx.x * CBN;  // token tile
  const int m0 = blockIdx.y * CBM;  // weight-row tile
  const int kpad = w.nb * 32;
  const int nk = (kpad + CBK - 1) / CBK;

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < C::NR; ++i) {
      mbar_init(smem_u32(&sh.rfull[i]), 1);
      mbar_init(smem_u32(&sh.rempty[i]), 1);
    }
    for (int i = 0; i < kCNA; ++i) {
      mbar_init(smem_u32(&sh.afull[i]), 4);
      mbar_init(smem_u32(&sh.aempty[i]), 1);
    }
    for (int i = 0; i < kCR; ++i) {
      mbar_init(smem_u32(&sh.tfull[i]), 1);
      mbar_init(smem_u32(&sh.tfree[i]), kCEpiWarps);
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

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::NR;
        if (i >= C::NR && !cwait(smem_u32(&sh.rempty[s]), ((i / C::NR) - 1) & 1, &sh.abort)) break;
        const uint32_t st = rbase + s * C::kStage;
        const uint32_t bar = smem_u32(&sh.rfull[s]);
        mbar_expect_tx(bar, C::kStage);
        tma_load_2d(st, &tm_xh, i * CBK, n0, bar);
        tma_load_2d(st + C::kX, &tm_xl, i * CBK, n0, bar);
        tma_load_2d(st + 2 * C::kX, &tm_q, i * (WT == 8 ? 64 : 32), m0, bar);
        tma_load_2d(st + 2 * C::kX + C::kCodes, &tm_d, (i * 2) & ~7, m0, bar);
        issued = i + 1;
      }
      // copies still in flight (after an abort) land before the CTA exits
      for (int i = issued > C::NR ? issued - C::NR : 0; i < issued; ++i)
        cwait(smem_u32(&sh.rfull[i % C::NR]), (i / C::NR) & 1, &sh.abort, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue: per 16-column K slice, codes x x_hi then
    // codes x x_lo into the slice's block region (columns 256 rg + 128 bb)
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16(CBM, CBN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::NR, ai = i % kCNA, rg = i % kCR;
        if (!cwait(smem_u32(&sh.afull[ai]), (i / kCNA) & 1, &sh.abort)) break;
        if (!cwait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t sa = abase + ai * kCATile, sb = rbase + s * C::kStage;
#pragma unroll
        for (int ks = 0; ks < CBK / 16; ++ks) {
          const uint32_t d = tmem + 256 * rg + 128 * (ks >> 1);
          umma_f16(d, umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + ks * 32), idesc, ks & 1);
          umma_f16(d, umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + C::kX + ks * 32), idesc, 1);
        }
        umma_commit(smem_u32(&sh.rempty[s]));
        umma_commit(smem_u32(&sh.aempty[ai]));
        umma_commit(smem_u32(&sh.tfull[rg]));
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------- convert: thread = weight row
    const int r = tid - 64;
    for (int i = 0; i < nk; ++i) {
      const int s = i % C::NR, ai = i % kCNA, rg = i % kCR;
      if (!cwait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
      if (i >= kCNA && !cwait(smem_u32(&sh.aempty[ai]), ((i / kCNA) - 1) & 1, &sh.abort)) break;
      if (i >= kCR && !cwait(smem_u32(&sh.tfree[rg]), ((i / kCR) - 1) & 1, &sh.abort)) break;
      const uint32_t st = rbase + s * C::kStage;
      const uint32_t dsc = lds32c(st + 2 * C::kX + C::kCodes + r * 16 + (((i * 2) & 7) << 1));
      sc[rg * CBM + r] = __half22float2(*reinterpret_cast<const __half2*>(&dsc));
      convert_codes<WT>(st + 2 * C::kX + r * (WT == 8 ? 64 : 32), abase + ai * kCATile + r * 128, r,
                        kpad - i * CBK);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.sfull[rg]));  // the block scales, straight to the epilogue
        mbar_arrive(smem_u32(&sh.afull[ai]));
      }
    }
  } else {
    // ---------------- epilogue: thread = weight row (its TMEM lane), 32 tokens
    const int q = warp & 3;
    const int grp = (warp - 6) >> 2;
    const int row = q * 32 + lane;
    const int m = m0 + row;
    float y[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) y[t] = 0.f;
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int rg = i % kCR;
      ok = cwait(smem_u32(&sh.sfull[rg]), (i / kCR) & 1, &sh.abort) &&
           cwait(smem_u32(&sh.tfull[rg]), (i / kCR) & 1, &sh.abort);
      if (!ok) break;
      tc_fence_after();
      const float2 dd = sc[rg * CBM + row];
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + 256 * rg + 32 * grp;
      uint32_t v[32], u[32];
      tmem_ld32(tbase, v);        // block 0 of the step
      tmem_ld32(tbase + 128, u);  // block 1
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        y[j] = fmaf(dd.y, __uint_as_float(u[j]), fmaf(dd.x, __uint_as_float(v[j]), y[j]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.tfree[rg]));
    }
    ok = __all_sync(0xffffffffu, ok && !*(volatile int*)&sh.abort);
    if (ok)
#pragma unroll
      for (int t = 0; t < 32; ++t) cepi_store<EPI>(a, n0 + 32 * grp + t, m, w.rows, y[t]);
    if (!ok && a.status && lane == 0) atomicOr(a.status, kTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

using CgFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const PgArgs);

template <int WT>
CgFn cg_pick(int epi) {
  switch (epi) {
    case EPI_STORE: return cgemm_kernel<WT, EPI_STORE>;
    case EPI_RESID: return cgemm_kernel<WT, EPI_RESID>;
    case EPI_SWIGLU: return cgemm_kernel<WT, EPI_SWIGLU>;
  }
  return nullptr;
}

CgFn cg_select(int wtype, int epi, int* smem) {
  if (wtype == 8) {
    *smem = CCfg<8>::kSmem;
    return cg_pick<8>(epi);
  }
  *smem = CCfg<4>::kSmem;
  return cg_pick<4>(epi);
}

}  // namespace

cudaError_t cgemm_setup_attributes() {
  for (int wt : {8, 4})
    for (int e : {EPI_STORE, EPI_RESID, EPI_SWIGLU}) {
      int smem = 0;
      CgFn f = cg_select(wt, e, &smem);
      cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
  return cudaSuccess;
}

cudaError_t launch_cgemm(int wtype, int epi, const PgArgs& a, cudaStream_t s) {
  const MatDev& w = a.w;
  const int kpad = w.nb * 32;
  if (a.kx % 8 || a.kx < kpad || a.T < 1 || w.rstep != 1 || !a.xlo) return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && (!a.h || !a.hlo)) return cudaErrorInvalidValue;
  int smem = 0;
  CgFn f = cg_select(wtype, epi, &smem);
  if (!f) return cudaErrorInvalidValue;
  CUtensorMap th, tl, tq, td;
  const uint64_t rb = wtype == 8 ? (uint64_t)w.nb * 32 : (uint64_t)w.nb * 16;
  if (!make_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, CBK,
                    CBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.xlo, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, CBK,
                    CBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.qs, rb, (uint64_t)w.rows, rb, wtype == 8 ? 64 : 32, CBM,
                    wtype == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.d, (uint64_t)w.ds, (uint64_t)w.rows, (uint64_t)w.ds * 2, 8,
                    CBM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // token tiles along x: the CTAs that share a weight tile run together (it
  // stays in L2), and the activation planes of a chunk fit L2 as well
  dim3 grid((a.T + CBN - 1) / CBN, (w.rows + CBM - 1) / CBM);
  f<<<grid, CTHREADS, smem, s>>>(th, tl, tq, td, a);
  return cudaGetLastError();
}

}  // namespace dls
