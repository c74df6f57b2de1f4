// Multi-row dequant-GEMV Y = X W^T for 2..8 activation rows (a batched
// decode step: the branches of a fork, or the positions a speculative round
// checks), Q8_0 / Q4_0 weights.  Each weight byte is read from HBM once for
// all rows; the arithmetic stays on the CUDA cores (at 8 rows a weight byte
// feeds 8-16 multiply-adds, far below what would make tensor cores pay).
//
// Per CTA: a contiguous range of weight rows and a range of K (split-K when
// the activation slices of all rows would not fit in registers).
//  * A producer warp streams the CTA's weight rows (codes and block scales)
//    through a shared-memory ring with 1-D bulk async copies and mbarriers.
//  * Consumer lanes own 16 columns of each 512-column chunk (Q8_0: 16 code
//    bytes; Q4_0: 8 code bytes = the low and high nibbles of half a block)
//    and hold every activation row's slice as int16 with one scale per
//    (row, slice), so each code-activation product is an exact int32 dp2a
//    term; the fp32 accumulation adds d * s * dot per block and row.
//  * RMSNorm prologue: every CTA takes each row's sum of squares over the
//    full width (the rows are a few KB and L2-resident), then scales its
//    slice by the row's 1/rms and the gain.
//  * Lanes reduce with a halving butterfly over (weight row, activation row)
//    pairs, warps through shared memory in a fixed order.  With split-K the
//    partial sums meet in a workspace and the last CTA of a row range adds
//    them in split order: the results do not depend on timing.
//  * Epilogues: store, residual add, or SwiGLU on interleaved (gate, up)
//    row pairs, all fp32 [row][ld] outputs.
#include <stdlib.h>

#include <algorithm>

#include "gemv_core.cuh"
#include "kernels.h"

namespace dls {

namespace {

constexpr int kRW = 8;                 // consumer warps
constexpr int kRRB = 32;               // weight rows per reduction block
constexpr int kRStage = 16384;         // target code bytes per ring stage
constexpr int kRRing = 64 * 1024;

struct RgShared {
  uint64_t full[16];
  uint64_t empty[16];
  float ss[kRW][8];                    // RMSNorm partial sums [warp][row]
  int abort;
  int last;                            // this CTA adds the split-K partials
};

// A lane's 16 activations of one row and chunk: int16 pairs and one scale.
struct X16 {
  uint32_t p[8];
  float s;
  int corr;     // code bias (128 for Q8_0, 8 for Q4_0) times the sum of the int16 values
};

template <int WT>
__device__ __forceinline__ void quant16(const float (&v)[16], X16& x) {
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(v[i]));
  const float s = mx > 0.f ? mx / 32767.0f : 1.0f;
  const float inv = 1.0f / s;
  int sum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int a = __float2int_rn(v[2 * e] * inv), b = __float2int_rn(v[2 * e + 1] * inv);
    sum += a + b;
    x.p[e] = (uint32_t)(a & 0xFFFF) | ((uint32_t)b << 16);
  }
  x.s = s;
  x.corr = sum * (WT == 8 ? 128 : 8);
}

// columns of the lane's 16 elements in chunk c: Q8_0 one run of 16, Q4_0
// two runs of 8 (low nibbles, then high nibbles of the same 8 bytes)
template <int WT>
__device__ __forceinline__ int run_col(int c, int lane, int run) {
  if (WT == 8) return c * 512 + lane * 16;
  return c * 512 + (lane >> 1) * 32 + (lane & 1) * 8 + run * 16;
}

// The lane's 16 codes of one row as 4 words of one code per byte (Q4_0:
// the low nibbles of the 8 bytes, then the high nibbles), matching X16's pairs.
template <int WT>
__device__ __forceinline__ void code_words(const uint8_t* q, uint32_t (&c)[4]) {
  if (WT == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(q);
    c[0] = v.x, c[1] = v.y, c[2] = v.z, c[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(q);
    c[0] = v.x & 0x0F0F0F0Fu, c[1] = v.y & 0x0F0F0F0Fu;
    c[2] = (v.x >> 4) & 0x0F0F0F0Fu, c[3] = (v.y >> 4) & 0x0F0F0F0Fu;
  }
}

// sum_i code_i X_i minus the code bias: one dp2a chain started at -corr
__device__ __forceinline__ int code_dot(const uint32_t (&c)[4], const X16& x) {
  int s = -x.corr;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    s = dp2a_lo(x.p[2 * k], c[k], s);
    s = dp2a_hi(x.p[2 * k + 1], c[k], s);
  }
  return s;
}

template <int WT, int PRO, int EPI, int RS, int NT, int MC>
__global__ void __launch_bounds__(32 * (kRW + 1), 2) rgemv_kernel(const RgArgs a, const RgLaunch L) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  RgShared& sh = *reinterpret_cast<RgShared*>(smem_raw);
  float* s_part = reinterpret_cast<float*>(smem_raw + sizeof(RgShared));   // [kRW][kRRB][NT]
  uint8_t* ring = smem_raw + ((sizeof(RgShared) + kRW * kRRB * NT * 4 + 127) & ~127);
  const MatDev& w = a.w;
  const int nb = w.nb, kpad = nb * 32;
  const int NS = L.ns;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t row_bytes = WT == 8 ? (size_t)nb * 32 : (size_t)nb * 16;
  const size_t drow_bytes = (size_t)w.ds * 2;
  const int T = a.T;

  // rows: balanced over blockIdx.x in multiples of `unit`; K: chunks
  // [c0, c1) of 512 columns for split blockIdx.y
  const int units = (w.rows + a.unit - 1) / a.unit;
  const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
  const int r0 = u0 * a.unit, r1 = min(w.rows, u1 * a.unit);
  const int nrows = max(r1 - r0, 0);
  const int nst = (nrows + RS - 1) / RS;
  const int nchunk = (kpad + 511) / 512;
  const int split = gridDim.y, sp = blockIdx.y;
  const int c0 = nchunk * sp / split, c1 = nchunk * (sp + 1) / split;
  // this split's segment of every weight row: codes of chunks [c0, c1) (512
  // columns = 512 or 256 bytes each) and their block scales (32 bytes each)
  constexpr uint32_t CB = WT == 8 ? 512 : 256;
  const uint32_t qbeg = c0 * CB, qseg = min((uint32_t)c1 * CB, (uint32_t)row_bytes) - qbeg;
  const uint32_t dbeg = c0 * 32, dseg = min((uint32_t)c1 * 32, (uint32_t)drow_bytes) - dbeg;
  const uint32_t stage_q = RS * qseg;
  const uint32_t stage_bytes = L.stage;  // >= RS * (qseg + dseg), set by the plan for the widest split

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), kRW);
    }
    sh.abort = 0;
    sh.last = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the next kernel may start its prologue
  // (it waits for this grid's completion before reading its outputs); the
  // weight stream below does not depend on the previous kernel, the
  // consumers wait for it before reading the activations.
  griddep_launch();

  if (warp == kRW) {
    // ---------------- producer
    if (lane == 0) {
      int issued = 0, slot = 0;
      uint32_t phase = 0;  // parity of the ring pass this stage is in
      for (int s = 0; s < nst; ++s) {
        if (s >= NS && !mbar_wait(smem_u32(&sh.empty[slot]), phase ^ 1u)) {
          atomicOr(a.status, kTimeout);
          sh.abort = 1;
          break;
        }
        const int rows_s = min(RS, nrows - s * RS);
        const int row = r0 + s * RS;
        uint8_t* dst = ring + (size_t)slot * stage_bytes;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_expect_tx(bar, rows_s * (qseg + dseg));
        if (split == 1) {  // whole rows: one copy of each kind
          bulk_g2s(smem_u32(dst), w.qs + (size_t)row * row_bytes, rows_s * qseg, bar);
          bulk_g2s(smem_u32(dst + stage_q), reinterpret_cast<const uint8_t*>(w.d) + (size_t)row * drow_bytes,
                   rows_s * dseg, bar);
        } else {
          for (int rr = 0; rr < rows_s; ++rr) {
            bulk_g2s(smem_u32(dst + rr * qseg), w.qs + (size_t)(row + rr) * row_bytes + qbeg, qseg, bar);
            bulk_g2s(smem_u32(dst + stage_q + rr * dseg),
                     reinterpret_cast<const uint8_t*>(w.d) + (size_t)(row + rr) * drow_bytes + dbeg, dseg, bar);
          }
        }
        ++issued;
        if (++slot == NS) {
          slot = 0;
          phase ^= 1u;
        }
      }
      for (int s = max(0, issued - NS); s < issued; ++s) mbar_wait(smem_u32(&sh.full[s % NS]), (s / NS) & 1);
    }
  } else {
    // ---------------- consumers
    griddep_wait();
    float rs[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) rs[t] = 1.0f;
    if (PRO == PRO_RMSNORM) {
      // each row's sum of squares over the full width (cols % 4 == 0)
      float ss[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        ss[t] = 0.f;
        if (t < T)
          for (int i = tid * 4; i < w.cols; i += kRW * 32 * 4) {
            const float4 v = *reinterpret_cast<const float4*>(a.x + (size_t)t * a.ldx + i);
            ss[t] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[t]))));
          }
        ss[t] = warp_sum(ss[t]);
      }
      if (lane == 0)
#pragma unroll
        for (int t = 0; t < NT; ++t) sh.ss[warp][t] = ss[t];
      named_bar(1, kRW * 32);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float tot = 0.f;
        for (int i = 0; i < kRW; ++i) tot += sh.ss[i][t];  // fixed order
        rs[t] = 1.0f / sqrtf(tot / (float)w.cols + a.eps);
      }
    }
    X16 xq[MC][NT];
    bool valid[MC];
    int qoff[MC], blk[MC];
#pragma unroll
    for (int k = 0; k < MC; ++k) {
      const int c = c0 + warp + k * kRW;
      valid[k] = c < c1 && run_col<WT>(c, lane, 0) < kpad;
      qoff[k] = valid[k] ? (WT == 8 ? (c - c0) * 512 + lane * 16 : (c - c0) * 256 + lane * 8) : 0;
      blk[k] = valid[k] ? ((c - c0) * 16 + (lane >> 1)) : 0;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float v[16];
#pragma unroll
        for (int run = 0; run < (WT == 8 ? 1 : 2); ++run) {
          const int col = valid[k] ? run_col<WT>(c, lane, run) : 0;
#pragma unroll
          for (int j = 0; j < (WT == 8 ? 16 : 8); j += 4) {
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f), g = make_float4(1.f, 1.f, 1.f, 1.f);
            if (valid[k] && t < T && col + j < w.cols) {
              f = *reinterpret_cast<const float4*>(a.x + (size_t)t * a.ldx + col + j);
              if (PRO == PRO_RMSNORM) g = *reinterpret_cast<const float4*>(a.g + col + j);
            }
            const int o = run * 8 + j;
            v[o] = f.x * rs[t] * g.x;
            v[o + 1] = f.y * rs[t] * g.y;
            v[o + 2] = f.z * rs[t] * g.z;
            v[o + 3] = f.w * rs[t] * g.w;
          }
        }
        quant16<WT>(v, xq[k][t]);
      }
    }

    // lanes past the matrix hold zero activations (X = 0, corr = 0): their
    // products are exactly 0 whatever the codes they read
    const int stages_per_block = kRRB / RS;
    int slot = 0;
    uint32_t phase = 0;
    for (int s = 0; s < nst; ++s) {
      if (!sh.abort && !mbar_wait(smem_u32(&sh.full[slot]), phase)) {
        atomicOr(a.status, kTimeout);
        sh.abort = 1;
      }
      const int rows_s = min(RS, nrows - s * RS);
      const uint8_t* stp = ring + (size_t)slot * stage_bytes;
      float acc[RS * NT];
#pragma unroll
      for (int i = 0; i < RS * NT; ++i) acc[i] = 0.f;
      if (!sh.abort) {
#pragma unroll
        for (int k = 0; k < MC; ++k) {
#pragma unroll
          for (int rr = 0; rr < RS; ++rr) {
            uint32_t cw[4];
            code_words<WT>(stp + rr * qseg + qoff[k], cw);
            const float d = __half2float(*reinterpret_cast<const __half*>(stp + stage_q + rr * dseg + blk[k] * 2));
#pragma unroll
            for (int t = 0; t < NT; ++t)
              acc[rr * NT + t] = fmaf(d * xq[k][t].s, (float)code_dot(cw, xq[k][t]), acc[rr * NT + t]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
      if (++slot == NS) {
        slot = 0;
        phase ^= 1u;
      }
      constexpr int N = RS * NT;
      const float tot = butterfly<N>(acc, lane);
      constexpr int LG = N == 1 ? 0 : N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
      const int idx = lane >> (5 - LG);
      const int rr = idx / NT, t = idx % NT;
      const int lrow = s * RS + rr - (s / stages_per_block) * kRRB;
      if ((lane & ((32 >> LG) - 1)) == 0 && rr < rows_s) s_part[(warp * kRRB + lrow) * NT + t] = tot;

      if ((s + 1) % stages_per_block == 0 || s == nst - 1) {
        named_bar(1, kRW * 32);
        const int b0 = r0 + (s / stages_per_block) * kRRB;
        const int bn = min(kRRB, r1 - b0);
        for (int i = tid; i < bn * NT; i += kRW * 32) {
          const int lr = i / NT, tt = i % NT;
          if (tt >= T) continue;
          float v = 0.f;
          for (int ww = 0; ww < kRW; ++ww) v += s_part[(ww * kRRB + lr) * NT + tt];
          const int r = b0 + lr;
          if (split > 1) {
            a.part[((size_t)sp * T + tt) * w.rows + r] = v;
          } else if (EPI == EPI_SWIGLU) {
            // rows (2i, 2i+1) are (gate_i, up_i): the pair sits in this block (rows split in pairs)
            s_part[(0 * kRRB + lr) * NT + tt] = v;  // reuse warp 0's slot: read back below
          } else if (EPI == EPI_RESID) {
            a.y[(size_t)tt * a.ldy + r] += v;
          } else {
            a.y[(size_t)tt * a.ldy + r] = v;
          }
        }
        if (EPI == EPI_SWIGLU && split == 1) {
          named_bar(1, kRW * 32);
          for (int i = tid; i < (bn >> 1) * NT; i += kRW * 32) {
            const int pi = i / NT, tt = i % NT;
            if (tt >= T) continue;
            const float g = s_part[(2 * pi) * NT + tt], u = s_part[(2 * pi + 1) * NT + tt];
            a.y[(size_t)tt * a.ldy + ((b0 + 2 * pi) >> 1)] = silu(g) * u;
          }
        }
        named_bar(1, kRW * 32);
      }
    }

    if (split > 1) {
      // the last CTA of this row range adds the partials in split order
      __threadfence();
      named_bar(1, kRW * 32);
      if (tid == 0) {
        const int prev = atomicAdd(&a.counters[blockIdx.x], 1);
        sh.last = prev == split - 1;
        if (sh.last) atomicExch(&a.counters[blockIdx.x], 0);
      }
      named_bar(1, kRW * 32);
      if (sh.last) {
        __threadfence();
        const int step = EPI == EPI_SWIGLU ? 2 : 1;
        for (int i = tid; i < (nrows / step) * T; i += kRW * 32) {
          const int j = i / T, tt = i % T;
          const int r = r0 + j * step;
          float v0 = 0.f, v1 = 0.f;
          for (int q = 0; q < split; ++q) {
            v0 += __ldcg(&a.part[((size_t)q * T + tt) * w.rows + r]);
            if (step == 2) v1 += __ldcg(&a.part[((size_t)q * T + tt) * w.rows + r + 1]);
          }
          if (EPI == EPI_SWIGLU) a.y[(size_t)tt * a.ldy + (r >> 1)] = silu(v0) * v1;
          else if (EPI == EPI_RESID) a.y[(size_t)tt * a.ldy + r] += v0;
          else a.y[(size_t)tt * a.ldy + r] = v0;
        }
      }
    }
  }
  __syncthreads();
}

using RgFn = void (*)(const RgArgs, const RgLaunch);

template <int WT, int P, int E, int NT, int MC>
RgFn rg_pick_rs(int rs) {
  switch (rs) {
    case 1: return &rgemv_kernel<WT, P, E, 1, NT, MC>;
    case 2: return &rgemv_kernel<WT, P, E, 2, NT, MC>;
    case 4: return NT <= 4 ? &rgemv_kernel<WT, P, E, 4, NT <= 4 ? NT : 4, MC> : nullptr;
  }
  return nullptr;
}

template <int WT, int P, int E>
RgFn rg_pick_nt(int nt, int rs, int mc) {
  if (nt == 2) return mc == 1 ? rg_pick_rs<WT, P, E, 2, 1>(rs) : mc == 2 ? rg_pick_rs<WT, P, E, 2, 2>(rs) : nullptr;
  if (nt == 4) return mc == 1 ? rg_pick_rs<WT, P, E, 4, 1>(rs) : nullptr;
  if (nt == 8) return mc == 1 ? rg_pick_rs<WT, P, E, 8, 1>(rs) : nullptr;
  return nullptr;
}

RgFn rg_pick(int wtype, int pro, int epi, int nt, int rs, int mc) {
#define DLS_RPICK(WT, P, E) \
  if (wtype == WT && pro == P && epi == E) return rg_pick_nt<WT, P, E>(nt, rs, mc);
  DLS_RPICK(8, PRO_RMSNORM, EPI_STORE)
  DLS_RPICK(8, PRO_COPY, EPI_RESID)
  DLS_RPICK(8, PRO_RMSNORM, EPI_SWIGLU)
  DLS_RPICK(4, PRO_RMSNORM, EPI_STORE)
  DLS_RPICK(4, PRO_COPY, EPI_RESID)
  DLS_RPICK(4, PRO_RMSNORM, EPI_SWIGLU)
#undef DLS_RPICK
  return nullptr;
}

}  // namespace

RgLaunch rgemv_plan(int wtype, int pro, int epi, int rows, int nb, int T, int num_sms, int unit) {
  RgLaunch l{};
  if (T < 1 || T > 8 || rows < 1) return l;
  const int nt = T <= 2 ? 2 : T <= 4 ? 4 : 8;
  const int mcmax = nt == 2 ? 2 : 1;
  const int nchunk = (nb * 32 + 511) / 512;
  // K splits: each CTA's chunks fit kRW warps x mcmax chunks
  const int split = (nchunk + kRW * mcmax - 1) / (kRW * mcmax);
  const int per = (nchunk + split - 1) / split;
  const int mc = (per + kRW - 1) / kRW;
  const int row_bytes = wtype == 8 ? nb * 32 : nb * 16;
  const int ds = (nb + 7) & ~7;
  // the widest split's segment of a row (splits differ by at most one chunk)
  const int qseg = std::min(per * (wtype == 8 ? 512 : 256), row_bytes);
  const int dseg = std::min(per * 32, ds * 2);
  const int rsmax = nt == 8 ? 2 : 4;
  int rs = 1;
  while (rs < rsmax && (rs * 2) * qseg <= kRStage) rs *= 2;
  const int stage = rs * (qseg + dseg);
  const int ns = std::max(2, std::min(16, kRRing / stage));
  RgFn f = rg_pick(wtype, pro, epi, nt, rs, mc);
  if (!f) return l;
  l.nt = nt;
  l.rs = rs;
  l.mc = mc;
  l.ns = ns;
  l.split = split;
  l.stage = stage;
  l.threads = 32 * (kRW + 1);
  l.smem = (int)((sizeof(RgShared) + kRW * kRRB * nt * 4 + 127) & ~127) + ns * stage;
  if (l.smem > 200 * 1024) return RgLaunch{};
  int occ = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, l.threads, l.smem) != cudaSuccess) {
    cudaGetLastError();
    occ = 1;
  }
  occ = std::max(1, std::min(2, occ));
  const int units = (rows + unit - 1) / unit;
  l.grid = std::max(1, std::min(num_sms * occ / split, units));
  return l;
}

cudaError_t rgemv_setup_attributes() {
  for (int wt : {8, 4})
    for (int p : {(int)PRO_COPY, (int)PRO_RMSNORM})
      for (int e : {(int)EPI_STORE, (int)EPI_RESID, (int)EPI_SWIGLU})
        for (int nt : {2, 4, 8})
          for (int rs : {1, 2, 4})
            for (int mc : {1, 2}) {
              RgFn f = rg_pick(wt, p, e, nt, rs, mc);
              if (!f) continue;
              cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
              if (err != cudaSuccess) return err;
            }
  return cudaSuccess;
}

cudaError_t launch_rgemv(int wtype, int pro, int epi, const RgArgs& a, const RgLaunch& l, cudaStream_t s) {
  RgFn f = rg_pick(wtype, pro, epi, l.nt, l.rs, l.mc);
  if (!f || l.grid < 1 || l.split < 1 || a.T < 1 || a.T > l.nt || a.w.ds % 8 || a.w.cols % 4 || a.ldx % 4 ||
      a.w.rstep != 1 || !a.status || (pro == PRO_RMSNORM && !a.g))
    return cudaErrorInvalidValue;
  if (l.split > 1 && (!a.part || !a.counters)) return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && (a.unit % 2 || a.w.rows % 2)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.grid, l.split);
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
