// Dequantising GEMM on the 5th-generation tensor cores:
//   D[m, t] = sum_k W[m, k] X[t, k],  W Q8_0/Q4_0 (repacked codes + fp16
//   scales), X fp16 [T][kx], fp32 accumulation in tensor memory.
// It serves the prefill projections (T = a prompt chunk; SwarmKV page,
// section 2: prefill runs every prompt token through every layer) and the
// batched decode step (T = the batch; each weight byte is read once for all
// rows of the batch).
//
// One CTA computes a 128-row x BN-token tile over a range of 64-column K
// steps (split-K spreads small matrices over the GPU; partial sums meet in
// a workspace and the last-arriving CTA of a tile adds them in split order).
//   warp 0    TMA producer: per K step one ring stage receives the fp16
//             token tile (128-byte swizzle, the MMA's B layout), the raw
//             codes of 128 weight rows (64- or 32-byte swizzle, which makes
//             the dequantising reads bank-conflict free) and their scales.
//   warp 1    owns the tensor memory; one thread issues 4 MMAs (K = 16) per
//             step and commits them to the barriers that free the stage.
//   warps 2-9 dequantise: two threads per weight row, each turning 32 of
//             the row's 64 codes into fp16(d * q) (packed half2 arithmetic,
//             one rounding, bit-identical to rounding the exact fp32
//             product) and writing them swizzled as the MMA's A operand;
//             afterwards they read the accumulators (tcgen05.ld; two warps
//             per 32-lane quarter of tensor memory, each half the columns)
//             and run the epilogue.
// Every wait is bounded (2 s); a wait that gives up sets an abort flag that
// all roles see, the kernel stores nothing and reports kTimeout.
#include <cuda.h>

#include <mutex>
#include <stdlib.h>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int GBM = 128, GBK = 64;
constexpr int GTHREADS = 320;
constexpr int NDQ = 8;  // dequantising / epilogue warps
constexpr int kSplitMax = 16;  // K splits of one tile (the partial sums are added in registers)
constexpr int kATile = GBM * GBK * 2;  // 16 KB fp16 A operand per stage
constexpr int kScaleBox = GBM * 16;    // 8 fp16 scales per row
constexpr uint64_t kWaitNsG = 2000000000ull;

template <int WT, int BN>
struct GCfg {
  static constexpr int kCodes = WT == 8 ? GBM * 64 : GBM * 32;
  static constexpr int kB = BN * 128;                          // one activation plane
  static constexpr int kStage = 2 * kB + kCodes + kScaleBox;  // bytes the TMA lands per stage: x hi | x lo | codes | scales
  // small batches: two CTAs per SM (<= 113 KB each), one streaming while
  // the other starts up or finishes
  // prompt chunks: 128-token tiles with three stages, or 256-token tiles
  // (each dequantised weight tile feeds twice the tokens) with two
  static constexpr int NR = BN >= 256 ? 2 : BN >= 128 ? 3 : (WT == 8 ? 3 : 4);
  static constexpr int NA = BN >= 256 ? 2 : BN >= 128 ? 3 : 2;  // fp16 weight tiles (hi and lo planes)
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr int kBarOff = NA * 2 * kATile + NR * kStage;
  static constexpr int kSmem = kBarOff + 256 + 1024;
  static_assert(BN >= 128 || kSmem <= 113 * 1024, "two CTAs per SM");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

template <int NR, int NA>
struct GBars {
  uint64_t rfull[NR], rempty[NR], afull[NA], aempty[NA], done;
  uint32_t tmem;
  int abort;
  int last;
};

__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, int* abort_flag, bool heed_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 63) == 0) {
      if (heed_abort && *(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsG) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// two codes (bytes k0, k1 of u as selected) -> hi = fp16(d * q) and
// lo = fp16(d * q - hi) pairs.  d * q has at most 19 significant bits, so
// the fused multiply-add gives the exact residual (lo is representable).
__device__ __forceinline__ void dq2(uint32_t u, uint32_t sel, __half2 bias, __half2 d, uint32_t& hi, uint32_t& lo) {
  const uint32_t p = __byte_perm(u, 0x64646464u, sel);  // fp16 1024 + byte in each half
  const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&p), bias);
  const __half2 v = __hmul2(q, d);
  const __half2 r = __hfma2(q, d, __hneg2(v));
  hi = *reinterpret_cast<const uint32_t*>(&v);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// 4 codes of one 32-bit word -> 4 fp16 of each plane (two words each)
__device__ __forceinline__ void dq4(uint32_t u, __half2 bias, __half2 d, uint32_t& h0, uint32_t& h1, uint32_t& l0,
                                    uint32_t& l1) {
  dq2(u, 0x4140u, bias, d, h0, l0);
  dq2(u, 0x4342u, bias, d, h1, l1);
}

// Half hf (columns 32hf .. 32hf+31) of row r of one K step: codes at `qrow`
// (swizzled by the TMA), scales of the step's two blocks in `dsc`, fp16
// output planes at `arow` (hi) and `arow + kATile` (lo), 128-byte swizzle.
// `zero`: these columns lie outside the matrix (the second half of a K
// step past the last block).
template <int WT>
__device__ __forceinline__ void dequant_half(uint32_t qrow, uint32_t dsc, uint32_t arow, int r, int hf, bool zero) {
  const __half2 dh = *reinterpret_cast<const __half2*>(&dsc);
  const __half2 d = hf ? __high2half2(dh) : __low2half2(dh);
  const int sw = r & 7;
  const uint32_t lrow = arow + kATile;
  if (zero) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sts128(arow + (((4 * hf + j) ^ sw) << 4), make_uint4(0, 0, 0, 0));
      sts128(lrow + (((4 * hf + j) ^ sw) << 4), make_uint4(0, 0, 0, 0));
    }
    return;
  }
  if (WT == 8) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1024 + 128
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {  // 16 codes: columns 16c .. 16c+15
      const int c = 2 * hf + cc;
      const uint4 u = lds128(qrow + ((c ^ ((r >> 1) & 3)) << 4));
      uint4 h0, h1, l0, l1;
      dq4(u.x, bias, d, h0.x, h0.y, l0.x, l0.y);
      dq4(u.y, bias, d, h0.z, h0.w, l0.z, l0.w);
      dq4(u.z, bias, d, h1.x, h1.y, l1.x, l1.y);
      dq4(u.w, bias, d, h1.z, h1.w, l1.z, l1.w);
      sts128(arow + (((2 * c) ^ sw) << 4), h0);
      sts128(arow + (((2 * c + 1) ^ sw) << 4), h1);
      sts128(lrow + (((2 * c) ^ sw) << 4), l0);
      sts128(lrow + (((2 * c + 1) ^ sw) << 4), l1);
    }
  } else {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1024 + 8
    // one 16-byte block: low nibbles = columns 0-15, high nibbles = 16-31
    const uint4 u = lds128(qrow + ((hf ^ ((r >> 2) & 1)) << 4));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // output chunk j: columns 8j .. 8j+7
      const uint32_t a = w[(2 * j) & 3], b = w[(2 * j + 1) & 3];
      const uint32_t sa = j < 2 ? a & 0x0F0F0F0Fu : (a >> 4) & 0x0F0F0F0Fu;
      const uint32_t sb = j < 2 ? b & 0x0F0F0F0Fu : (b >> 4) & 0x0F0F0F0Fu;
      uint4 h, l;
      dq4(sa, bias, d, h.x, h.y, l.x, l.y);
      dq4(sb, bias, d, h.z, h.w, l.z, l.w);
      sts128(arow + (((4 * hf + j) ^ sw) << 4), h);
      sts128(lrow + (((4 * hf + j) ^ sw) << 4), l);
    }
  }
}

template <int EPI>
__device__ __forceinline__ void epi_store(const PgArgs& a, int t, int m, int rows, float v) {
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

template <int WT, int EPI, int BN>
__global__ void __launch_bounds__(GTHREADS) tgemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_xl,
                                                         const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_d, const PgArgs a) {
  using C = GCfg<WT, BN>;
  using Bars = GBars<C::NR, C::NA>;
  extern __shared__ uint8_t gsm[];
  const uint32_t raw = smem_u32(gsm);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t abase = raw + pad;                   // NA fp16 A tiles, each hi plane | lo plane
  const uint32_t rbase = abase + C::NA * 2 * kATile;  // NR stages: B hi | B lo | codes | scales
  Bars& sh = *reinterpret_cast<Bars*>(gsm + pad + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MatDev& w = a.w;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * GBM;
  const int kpad = w.nb * 32;
  const int nk_all = (kpad + GBK - 1) / GBK;
  const int S = gridDim.z, z = blockIdx.z;
  const int kt0 = (int)((long long)nk_all * z / S);
  const int nk = (int)((long long)nk_all * (z + 1) / S) - kt0;  // >= 1: the host keeps S <= nk_all

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem), C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < C::NR; ++i) {
      mbar_init(smem_u32(&sh.rfull[i]), 1);
      mbar_init(smem_u32(&sh.rempty[i]), 1);
    }
    for (int i = 0; i < C::NA; ++i) {
      mbar_init(smem_u32(&sh.afull[i]), NDQ);
      mbar_init(smem_u32(&sh.aempty[i]), 1);
    }
    mbar_init(smem_u32(&sh.done), 1);
    sh.abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_x);
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
        if (i >= C::NR && !gwait(smem_u32(&sh.rempty[s]), ((i / C::NR) - 1) & 1, &sh.abort)) break;
        const uint32_t st = rbase + s * C::kStage;
        const uint32_t bar = smem_u32(&sh.rfull[s]);
        const int kt = kt0 + i;
        mbar_expect_tx(bar, C::kStage);
        tma_load_2d(st, &tm_x, kt * GBK, n0, bar);
        tma_load_2d(st + C::kB, &tm_xl, kt * GBK, n0, bar);
        tma_load_2d(st + 2 * C::kB, &tm_q, kt * (WT == 8 ? 64 : 32), m0, bar);
        tma_load_2d(st + 2 * C::kB + C::kCodes, &tm_d, (kt * 2) & ~7, m0, bar);
        issued = i + 1;
      }
      // copies still in flight (after an abort) land before the CTA exits
      for (int i = issued > C::NR ? issued - C::NR : 0; i < issued; ++i)
        gwait(smem_u32(&sh.rfull[i % C::NR]), (i / C::NR) & 1, &sh.abort, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16(GBM, BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::NR, ai = i % C::NA;
        if (!gwait(smem_u32(&sh.afull[ai]), (i / C::NA) & 1, &sh.abort)) break;
        if (!gwait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t sa = abase + ai * 2 * kATile, sb = rbase + s * C::kStage;
        // w x = w_hi x_hi + w_hi x_lo + w_lo x_hi (w_lo x_lo is below fp32 rounding)
#pragma unroll
        for (int ks = 0; ks < GBK / 16; ++ks) {
          umma_f16(tmem, umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + ks * 32), idesc, (i | ks) != 0);
          umma_f16(tmem, umma_desc_k128(sa + ks * 32), umma_desc_k128(sb + C::kB + ks * 32), idesc, true);
          umma_f16(tmem, umma_desc_k128(sa + kATile + ks * 32), umma_desc_k128(sb + ks * 32), idesc, true);
        }
        umma_commit(smem_u32(&sh.rempty[s]));
        umma_commit(smem_u32(&sh.aempty[ai]));
      }
      umma_commit(smem_u32(&sh.done));
    }
    __syncwarp();
  } else {
    // ---------------- dequantise (thread pair per weight row)
    const int dt = tid - 64, r = dt & (GBM - 1), hf = dt >> 7;
    for (int i = 0; i < nk; ++i) {
      const int s = i % C::NR, ai = i % C::NA;
      if (!gwait(smem_u32(&sh.rfull[s]), (i / C::NR) & 1, &sh.abort)) break;
      if (i >= C::NA && !gwait(smem_u32(&sh.aempty[ai]), ((i / C::NA) - 1) & 1, &sh.abort)) break;
      const int kt = kt0 + i;
      const uint32_t st = rbase + s * C::kStage;
      const uint32_t qrow = st + 2 * C::kB + r * (WT == 8 ? 64 : 32);
      const uint32_t dsc = lds32(st + 2 * C::kB + C::kCodes + r * 16 + (((kt * 2) & 7) << 1));
      dequant_half<WT>(qrow, dsc, abase + ai * 2 * kATile + r * 128, r, hf, hf && kpad - kt * GBK < GBK);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.afull[ai]));
    }

    // ---------------- epilogue: warp w reads TMEM lanes 32 * (w % 4) .., half the columns
    const bool waited = gwait(smem_u32(&sh.done), 0, &sh.abort, false);
    const bool ok = __all_sync(0xffffffffu, waited && !*(volatile int*)&sh.abort);
    tc_fence_after();
    const int q = warp & 3;
    constexpr int CW = BN / 2;                  // columns per warp
    const int cb = ((warp - 2) >> 2) * CW;       // this warp's first column
    const int m = m0 + q * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + cb;
    if (S == 1) {
#pragma unroll 1
      for (int c0 = 0; c0 < CW; c0 += 8) {
        uint32_t v[8];
        tmem_ld8(taddr + c0, v);
        tmem_wait_ld();
        if (!ok || n0 + cb + c0 >= a.T) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) epi_store<EPI>(a, n0 + cb + c0 + j, m, w.rows, __uint_as_float(v[j]));
      }
    } else {
      // partial tile -> workspace [S][T][rows]; the last CTA of the tile adds the S parts in order
#pragma unroll 1
      for (int c0 = 0; c0 < CW; c0 += 8) {
        uint32_t v[8];
        tmem_ld8(taddr + c0, v);
        tmem_wait_ld();
        if (!ok) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int t = n0 + cb + c0 + j;
          if (t < a.T && m < w.rows) a.part[((size_t)z * a.T + t) * w.rows + m] = __uint_as_float(v[j]);
        }
      }
      __threadfence();
      named_bar(1, 32 * NDQ);
      const int tile = blockIdx.y * gridDim.x + blockIdx.x;
      if (tid == 64) {
        const int prev = atomicAdd(&a.counters[tile], 1);
        sh.last = prev == S - 1;
        if (sh.last) a.counters[tile] = 0;  // ready for the next launch
      }
      named_bar(1, 32 * NDQ);
      if (sh.last && ok) {
        // add the S partials in split order; all of a column pair's loads are
        // issued before the first add (the split count is at most kSplitMax)
        __threadfence();
        const int tmax = min(CW, a.T - n0 - cb);
        for (int j = 0; j < tmax; j += 2) {
          const int t0 = n0 + cb + j, t1 = t0 + 1;
          const bool r_ok = m < w.rows, ok1 = j + 1 < tmax;
          float v0[kSplitMax], v1[kSplitMax];
#pragma unroll
          for (int zz = 0; zz < kSplitMax; ++zz) {
            const bool in = zz < S && r_ok;
            v0[zz] = in ? __ldcg(&a.part[((size_t)zz * a.T + t0) * w.rows + m]) : 0.f;
            v1[zz] = in && ok1 ? __ldcg(&a.part[((size_t)zz * a.T + t1) * w.rows + m]) : 0.f;
          }
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int zz = 0; zz < kSplitMax; ++zz) {
            acc0 += v0[zz];
            acc1 += v1[zz];
          }
          epi_store<EPI>(a, t0, m, w.rows, acc0);
          if (ok1) epi_store<EPI>(a, t1, m, w.rows, acc1);
        }
      }
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

// ---- host ----------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                  uint64_t stride1, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

using TgFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const PgArgs);

template <int WT, int BN>
TgFn tg_pick(int epi) {
  switch (epi) {
    case EPI_STORE: return tgemm_kernel<WT, EPI_STORE, BN>;
    case EPI_RESID: return tgemm_kernel<WT, EPI_RESID, BN>;
    case EPI_SWIGLU: return tgemm_kernel<WT, EPI_SWIGLU, BN>;
  }
  return nullptr;
}

template <int BN>
TgFn tg_pick(int wtype, int epi, int* smem) {
  if (wtype == 8) {
    *smem = GCfg<8, BN>::kSmem;
    return tg_pick<8, BN>(epi);
  }
  *smem = GCfg<4, BN>::kSmem;
  return tg_pick<4, BN>(epi);
}

TgFn tg_select(int wtype, int epi, int bn, int* smem) {
  switch (bn) {
    case 16: return tg_pick<16>(wtype, epi, smem);
    case 128: return tg_pick<128>(wtype, epi, smem);
    case 256: return tg_pick<256>(wtype, epi, smem);
  }
  return nullptr;
}

}  // namespace

cudaError_t tgemm_setup_attributes() {
  for (int wt : {8, 4})
    for (int e : {EPI_STORE, EPI_RESID, EPI_SWIGLU})
      for (int bn : {16, 128, 256}) {
        int smem = 0;
        TgFn f = tg_select(wt, e, bn, &smem);
        cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
      }
  return encode_fn() ? cudaSuccess : cudaErrorNotSupported;
}

TgPlan tgemm_plan(int rows, int kpad, int T, int num_sms, int max_split, int chunk_bn) {
  TgPlan p{};
  const int mt = (rows + GBM - 1) / GBM;
  const int nk = (kpad + GBK - 1) / GBK;
  if (T <= 16) {
    // decode batch (two CTAs per SM): split K so that the CTAs fill whole
    // waves; the fewest splits among the best fills, at least 8 K steps each
    p.bn = 16;
    num_sms *= 2;
    const int smax = std::max(1, std::min(std::min(max_split, kSplitMax), nk / 8));
    double best = -1.0;
    p.split = 1;
    for (int s = 1; s <= smax; ++s) {
      const int ctas = mt * s;
      const double fill = (double)ctas / ((double)((ctas + num_sms - 1) / num_sms) * num_sms);
      if (fill > best + 0.02) {
        best = fill;
        p.split = s;
      }
    }
  } else {
    // prompt chunk: 256-token tiles when they still give every SM a tile
    // (half the dequantising work per token of 128-token tiles), else 128;
    // chunk_bn 128 or 256 fixes the width (0: choose)
    const int t256 = mt * ((T + 255) / 256);
    p.bn = chunk_bn == 128 ? 128 : chunk_bn == 256 ? 256 : (T >= 256 && t256 >= num_sms) ? 256 : 128;
    p.split = 1;
  }
  return p;
}

cudaError_t launch_tgemm(int wtype, int epi, const PgArgs& a, const TgPlan& p, cudaStream_t s) {
  if (a.T <= 8 && p.bn == 16) return launch_sgemm(wtype, epi, a, p.split, s);
  const MatDev& w = a.w;
  const int kpad = w.nb * 32;
  const int nk = (kpad + GBK - 1) / GBK;
  if (a.kx % 8 || a.kx < kpad || a.T < 1 || w.rstep != 1 || p.split < 1 || p.split > nk || !a.xlo)
    return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && !a.hlo) return cudaErrorInvalidValue;
  if (p.split > 1 && (!a.part || !a.counters)) return cudaErrorInvalidValue;
  int smem = 0;
  TgFn f = tg_select(wtype, epi, p.bn, &smem);
  if (!f) return cudaErrorInvalidValue;
  CUtensorMap tx, txl, tq, td;
  const uint64_t rb = wtype == 8 ? (uint64_t)w.nb * 32 : (uint64_t)w.nb * 16;
  if (!make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, GBK,
              (uint32_t)p.bn, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&txl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.xlo, (uint64_t)a.kx, (uint64_t)a.T, (uint64_t)a.kx * 2, GBK,
              (uint32_t)p.bn, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.qs, rb, (uint64_t)w.rows, rb, wtype == 8 ? 64 : 32, GBM,
              wtype == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.d, (uint64_t)w.ds, (uint64_t)w.rows, (uint64_t)w.ds * 2, 8, GBM,
              CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  dim3 grid((a.T + p.bn - 1) / p.bn, (w.rows + GBM - 1) / GBM, p.split);
  f<<<grid, GTHREADS, smem, s>>>(tx, txl, tq, td, a);
  return cudaGetLastError();
}

}  // namespace dls
