// Batch-1 dequant-GEMV y = W x for Q8_0 / Q4_0 weights: the decode step's
// projections (engine page, section 4.4: a GEMV specialised for the
// single-token vector-matrix product, RMSNorm fused into it, SwiGLU fused
// with the projection).
//
// HBM-bound design for sm_103a:
//  * One CTA per SM owns a contiguous, balanced range of rows; its slice of
//    the code array and of the scale array is contiguous.
//  * A producer warp streams that slice through a shared-memory ring with
//    1-D bulk async copies (TMA, cp.async.bulk) and mbarriers: stages of RS
//    whole rows (~16 KB of codes plus their scales), 64 KB in flight per CTA,
//    two CTAs per SM where registers allow.
//    The first stages are issued before waiting on the previous kernel
//    (programmatic dependent launch): weights never depend on it.
//  * Consumer warps own K-chunks (512 columns for Q8_0, 1024 for Q4_0); each
//    lane holds its activation slice in registers for the whole kernel and
//    reads 16 bytes of codes per row per chunk from shared memory.
//  * Codes become exact fp32 through the 0x4B0000bb pattern (one byte permute
//    per value); products accumulate in packed f32x2 FMAs; per-row partials
//    reduce across lanes with a halving butterfly and across warps in a fixed
//    order (deterministic results).
//  * Prologues: copy or rmsnorm(x) * g, computed while the activation is
//    loaded into registers.  Epilogues: store, residual add, RoPE on adjacent
//    (q, k) pairs plus the fp16 K/V append into the cache, or SwiGLU on
//    interleaved (gate, up) row pairs (engine page, section 4.4: SwiGLU
//    fused with the projection), which feeds the down projection directly.
#include <stdlib.h>

#include "gemv_core.cuh"
#include "kernels.h"

namespace dls {

namespace {

constexpr int kMaxConsumers = 14;
constexpr int kRB = 64;              // rows per epilogue block
constexpr int kStageCodes = 16384;   // target code bytes per ring stage
constexpr int kRingBytes = 64 * 1024;
constexpr int kRingBytesSmall = 44 * 1024;  // ring when more than two CTAs share an SM

struct Shared {
  uint64_t full[16];
  uint64_t empty[16];
  float red[32];
  float rs;
  int abort;
};

template <int WT, int PRO, int EPI, int RS, int MC>
__global__ void __launch_bounds__(32 * (kMaxConsumers + 1)) gemv_kernel(const GemvArgs a, const GemvLaunch L) {
  using G = Geo<WT>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  float* s_part = reinterpret_cast<float*>(smem_raw + sizeof(Shared));   // [nwc][kRB]
  uint8_t* ring = smem_raw + ((sizeof(Shared) + L.nwc * kRB * 4 + 127) & ~127);
  const MatDev& w = a.w;
  const int nb = w.nb, kpad = nb * 32, cols = w.cols;
  const int nwc = L.nwc, NS = L.ns;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t row_bytes = WT == 8 ? (size_t)nb * 32 : (size_t)nb * 16;
  const size_t drow_bytes = (size_t)w.ds * 2;
  const uint32_t stage_q = RS * (uint32_t)row_bytes;
  const uint32_t stage_bytes = stage_q + RS * (uint32_t)drow_bytes;

  const int units = (w.rows + a.unit - 1) / a.unit;
  const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
  const int r0 = u0 * a.unit, r1 = min(w.rows, u1 * a.unit);
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

  if (warp == nwc) {
    // ---------------- producer: stream this CTA's rows through the ring
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nst; ++s) {
        const int slot = s % NS;
        if (s >= NS && !mbar_wait(smem_u32(&sh.empty[slot]), ((s / NS) - 1) & 1)) {
          atomicOr(&a.sp->status, kTimeout);
          sh.abort = 1;
          break;
        }
        const int rows_s = min(RS, nrows - s * RS);
        const int row = r0 + s * RS;
        uint8_t* dst = ring + (size_t)slot * stage_bytes;
        const uint32_t qb = rows_s * (uint32_t)row_bytes, db = rows_s * (uint32_t)drow_bytes;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_expect_tx(bar, qb + db);
        bulk_g2s(smem_u32(dst), w.qs + (size_t)row * row_bytes, qb, bar);
        bulk_g2s(smem_u32(dst + stage_q), reinterpret_cast<const uint8_t*>(w.d) + (size_t)row * drow_bytes, db, bar);
        ++issued;
      }
      griddep_launch();  // all of this CTA's weights are in flight
      // never leave with copies in flight: wait for every issued stage
      for (int s = max(0, issued - NS); s < issued; ++s)
        mbar_wait(smem_u32(&sh.full[s % NS]), (s / NS) & 1);
    }
  } else {
    // ---------------- consumers
    griddep_wait();
    if (nst == 0) griddep_launch();
    // prologue: this lane's activation slice in registers, loaded with one
    // round of float4 loads.  The consumer lanes' slices partition [0, kpad),
    // so their squares also give the RMSNorm sum of squares.
    const int nchunk = (kpad + G::CH - 1) / G::CH;
    const int mc = warp < nchunk ? min(MC, (nchunk - warp + nwc - 1) / nwc) : 0;
    constexpr int V4 = G::XV / 2;  // float4 per lane per chunk
    float4 raw[MC][V4];
    float4 gg[PRO == PRO_RMSNORM ? MC : 1][V4];
    bool valid[MC];
    // branch-free: all of the lane's float4 loads (x and gains) go out
    // together; a slice past the matrix reads element 0 and is zeroed
    // (cols % 4 == 0 is checked at launch: a float4 is all in or all out)
    bool in4[MC][V4];
#pragma unroll
    for (int k = 0; k < MC; ++k) {
      const int c = warp + k * nwc;
      const int col0 = WT == 8 ? c * 512 + lane * 16 : (c * 32 + lane) * 32;
      valid[k] = k < mc && col0 < kpad;
#pragma unroll
      for (int m4 = 0; m4 < V4; ++m4) {
        const int i0 = col0 + 4 * m4;
        in4[k][m4] = valid[k] && i0 < cols;
        const int j0 = in4[k][m4] ? i0 : 0;
        raw[k][m4] = *reinterpret_cast<const float4*>(a.x + j0);
        if (PRO == PRO_RMSNORM) gg[PRO == PRO_RMSNORM ? k : 0][m4] = *reinterpret_cast<const float4*>(a.g + j0);
      }
    }
#pragma unroll
    for (int k = 0; k < MC; ++k)
#pragma unroll
      for (int m4 = 0; m4 < V4; ++m4)
        if (!in4[k][m4]) raw[k][m4] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (PRO == PRO_RMSNORM) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < MC; ++k)
#pragma unroll
        for (int m4 = 0; m4 < V4; ++m4) {
          const float4 v = raw[k][m4];
          ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
      ss = warp_sum(ss);
      if (lane == 0) sh.red[warp] = ss;
      named_bar(1, nwc * 32);
      float t = 0.f;
      for (int i = 0; i < nwc; ++i) t += sh.red[i];  // fixed order, same in every thread
      const float rs = 1.0f / sqrtf(t / (float)cols + a.eps);
#pragma unroll
      for (int k = 0; k < MC; ++k)
#pragma unroll
        for (int m4 = 0; m4 < V4; ++m4) {
          const float4 g = gg[PRO == PRO_RMSNORM ? k : 0][m4];
          raw[k][m4] = make_float4(raw[k][m4].x * rs * g.x, raw[k][m4].y * rs * g.y, raw[k][m4].z * rs * g.z,
                                   raw[k][m4].w * rs * g.w);
        }
    }
    XQ<WT> xq[MC];
#pragma unroll
    for (int k = 0; k < MC; ++k) quantize_slice<WT>(reinterpret_cast<const float*>(raw[k]), xq[k]);

    int32_t pos = 0, seq = 0;
    if (EPI == EPI_QKV) {
      pos = a.sp->pos[a.brow];
      seq = a.sp->seq[a.brow];
    }
    const int stages_per_block = kRB / RS;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % NS;
      if (!sh.abort && !mbar_wait(smem_u32(&sh.full[slot]), (s / NS) & 1)) {
        atomicOr(&a.sp->status, kTimeout);
        sh.abort = 1;
      }
      if (s == nst - 1) griddep_launch();  // last stage arrived: let the next kernel start
      const int rows_s = min(RS, nrows - s * RS);
      const uint32_t st = smem_u32(ring) + (uint32_t)slot * stage_bytes;
      float acc[RS];
#pragma unroll
      for (int rr = 0; rr < RS; ++rr) acc[rr] = 0.f;
      if (!sh.abort) {
        // branch-free: every row slot is computed (rows past rows_s read
        // stale stage bytes and are discarded), invalid lanes read offset 0
        // and contribute exactly 0 through a select
#pragma unroll
        for (int k = 0; k < MC; ++k) {
          const int c = warp + k * nwc;
          const int qoff = valid[k] ? (WT == 8 ? c * 512 + lane * 16 : (c * 32 + lane) * 16) : 0;
          const int blk = valid[k] ? (WT == 8 ? (c * 512 + lane * 16) >> 5 : c * 32 + lane) : 0;
          const uint32_t qa = st + (uint32_t)qoff, da = st + stage_q + (uint32_t)blk * 2;
#pragma unroll
          for (int rr = 0; rr < RS; ++rr) {
            const uint4 q = lds128(qa + rr * (uint32_t)row_bytes);
            const float d = lds_half_as_float(da + rr * (uint32_t)drow_bytes);
            const float t = (float)idot16<WT>(q, xq[k]);
            acc[rr] = valid[k] ? fmaf(d * xq[k].s, t, acc[rr]) : acc[rr];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
      const float t = butterfly<RS>(acc, lane);
      const int rr = RS == 1 ? 0 : (lane >> (5 - (RS == 2 ? 1 : RS == 4 ? 2 : 3)));
      const int lrow = s * RS + rr - (s / stages_per_block) * kRB;
      if ((lane & ((32 / RS) - 1)) == 0 && rr < rows_s) s_part[warp * kRB + lrow] = t;

      // ---- end of an epilogue block (or the last stage): reduce + epilogue
      if ((s + 1) % stages_per_block == 0 || s == nst - 1) {
        named_bar(1, nwc * 32);
        const int b0 = r0 + (s / stages_per_block) * kRB;
        const int bn = min(kRB, r1 - b0);
        const int nwa = min(nwc, nchunk);
        if (EPI == EPI_QKV) {
          const int hd = a.kv.head_dim;
          for (int pi = tid; pi < (bn >> 1); pi += nwc * 32) {
            const int lr = pi * 2, r = b0 + lr;
            float v0 = 0.f, v1 = 0.f;
            for (int ww = 0; ww < nwa; ++ww) {
              v0 += s_part[ww * kRB + lr];
              v1 += s_part[ww * kRB + lr + 1];
            }
            if (r < a.q_rows + a.kv_rows) {  // q or k: rotate the adjacent pair
              if (pos < 0 || pos >= a.rope_len) {
                atomicOr(&a.sp->status, kBadPos);
                continue;
              }
              const float2 cs = a.rope_cs[(size_t)pos * (hd >> 1) + ((r % hd) >> 1)];
              const float t0 = v0 * cs.x - v1 * cs.y;
              v1 = v0 * cs.y + v1 * cs.x;
              v0 = t0;
            }
            if (r < a.q_rows) {
              a.y[r] = v0;
              a.y[r + 1] = v1;
            } else {
              const bool is_k = r < a.q_rows + a.kv_rows;
              const int rk = r - a.q_rows - (is_k ? 0 : a.kv_rows);
              const int kvh = rk / hd, dim = rk % hd;
              const int pt = a.kv.page_tokens;
              const int lp = pos / pt;
              const int page =
                  (pos >= 0 && lp < a.kv.max_pages) ? a.kv.page_table[(size_t)seq * a.kv.max_pages + lp] : -1;
              if (page < 0) {
                atomicOr(&a.sp->status, kBadPage);
                continue;
              }
              const size_t off = (((size_t)page * a.kv.n_kv + kvh) * pt + (pos % pt)) * hd + dim;
              __half* dst = (is_k ? a.kv.k_pool : a.kv.v_pool) + off;
              *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(v0, v1);
            }
          }
        } else if (EPI == EPI_SWIGLU) {
          // rows (2i, 2i+1) are (gate_i, up_i): h_i = silu(gate_i) * up_i
          for (int pi = tid; pi < (bn >> 1); pi += nwc * 32) {
            const int lr = pi * 2;
            float g0 = 0.f, u0 = 0.f;
            for (int ww = 0; ww < nwa; ++ww) {
              g0 += s_part[ww * kRB + lr];
              u0 += s_part[ww * kRB + lr + 1];
            }
            a.y[(b0 + lr) >> 1] = silu(g0) * u0;
          }
        } else {
          for (int lr = tid; lr < bn; lr += nwc * 32) {
            float v = 0.f;
            for (int ww = 0; ww < nwa; ++ww) v += s_part[ww * kRB + lr];
            if (EPI == EPI_RESID) a.y[b0 + lr] += v;
            else a.y[b0 + lr] = v;
          }
        }
        named_bar(1, nwc * 32);
      }
    }
  }
  __syncthreads();
}

using KernelFn = void (*)(const GemvArgs, const GemvLaunch);

template <int WT, int P, int E, int MC>
KernelFn pick_rs(int rs) {
  switch (rs) {
    case 1: return &gemv_kernel<WT, P, E, 1, MC>;
    case 2: return &gemv_kernel<WT, P, E, 2, MC>;
    case 4: return &gemv_kernel<WT, P, E, 4, MC>;
    case 8: return &gemv_kernel<WT, P, E, 8, MC>;
  }
  return nullptr;
}

template <int WT, int P, int E>
KernelFn pick_mc(int rs, int mc) {
  if (mc <= 1) return pick_rs<WT, P, E, 1>(rs);
  if (mc <= 2) return pick_rs<WT, P, E, 2>(rs);
  if (WT == 8 && mc <= 4) return pick_rs<WT, P, E, (WT == 8 ? 4 : 2)>(rs);
  return nullptr;
}

KernelFn pick(int wtype, int pro, int epi, int rs, int mc) {
#define DLS_PICK(WT, P, E) \
  if (wtype == WT && pro == P && epi == E) return pick_mc<WT, P, E>(rs, mc);
  DLS_PICK(8, PRO_RMSNORM, EPI_QKV)
  DLS_PICK(8, PRO_COPY, EPI_RESID)
  DLS_PICK(8, PRO_RMSNORM, EPI_STORE)
  DLS_PICK(8, PRO_RMSNORM, EPI_SWIGLU)
  DLS_PICK(8, PRO_COPY, EPI_STORE)
  DLS_PICK(4, PRO_RMSNORM, EPI_QKV)
  DLS_PICK(4, PRO_COPY, EPI_RESID)
  DLS_PICK(4, PRO_RMSNORM, EPI_STORE)
  DLS_PICK(4, PRO_RMSNORM, EPI_SWIGLU)
  DLS_PICK(4, PRO_COPY, EPI_STORE)
#undef DLS_PICK
  return nullptr;
}

}  // namespace

GemvLaunch gemv_plan(int wtype, int pro, int epi, int rows, int nb, int num_sms, int unit) {
  const int kpad = nb * 32;
  const int CH = wtype == 8 ? 512 : 1024;
  const int MC = wtype == 8 ? 4 : 2;  // Geo<WT>::MCMAX
  const int nchunk = (kpad + CH - 1) / CH;
  // consumer warps: the largest divisor of the chunk count <= 8 that keeps
  // chunks per warp within the register budget; else a divisor up to 14;
  // else an uneven split
  int nwc = 0;
  for (int d = 1; d <= 8; ++d)
    if (nchunk % d == 0 && nchunk / d <= MC) nwc = d;
  if (!nwc)
    for (int d = 9; d <= kMaxConsumers && !nwc; ++d)
      if (nchunk % d == 0 && nchunk / d <= MC) nwc = d;
  if (!nwc) nwc = std::min(kMaxConsumers, (nchunk + MC - 1) / MC);
  const int row_bytes = wtype == 8 ? nb * 32 : nb * 16;
  const int ds = (nb + 7) & ~7;
  int rs = 1;
  while (rs < 8 && (rs * 2) * row_bytes <= kStageCodes) rs *= 2;
  const int stage = rs * row_bytes + rs * ds * 2;
  const char* cps_env = getenv("DLS_GEMV_CTAS");
  const int cps_max = cps_env ? std::max(1, std::min(4, atoi(cps_env))) : 2;
  int ns = (cps_max > 2 ? kRingBytesSmall : kRingBytes) / stage;
  ns = std::max(2, std::min(16, ns));
  GemvLaunch l;
  l.threads = (nwc + 1) * 32;
  l.nwc = nwc;
  l.rs = rs;
  l.ns = ns;
  l.mc = (nchunk + nwc - 1) / nwc;
  const int head = (int)((sizeof(Shared) + nwc * kRB * 4 + 127) & ~127);
  l.smem = head + ns * stage;
  // CTAs per SM from the occupancy the kernel actually achieves (registers,
  // shared memory), at most 2
  int occ = 1;
  KernelFn f = pick(wtype, pro, epi, rs, l.mc);
  if (f && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, l.threads, l.smem) != cudaSuccess) {
    cudaGetLastError();
    occ = 1;
  }
  occ = std::max(1, std::min(cps_max, occ));
  const int units = (rows + unit - 1) / unit;
  int grid = std::min(num_sms * occ, units);
  if (grid < 1) grid = 1;
  l.grid = grid;
  return l;
}

cudaError_t gemv_setup_attributes() {
  const int pros[2] = {PRO_COPY, PRO_RMSNORM};
  const int epis[4] = {EPI_STORE, EPI_RESID, EPI_QKV, EPI_SWIGLU};
  for (int wt : {8, 4})
    for (int p : pros)
      for (int e : epis)
        for (int rs : {1, 2, 4, 8})
          for (int mc : {1, 2, 4}) {
            KernelFn f = pick(wt, p, e, rs, mc);
            if (!f) continue;
            cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
            if (err != cudaSuccess) return err;
          }
  return cudaSuccess;
}

cudaError_t launch_gemv(int wtype, int pro, int epi, const GemvArgs& a, const GemvLaunch& l, cudaStream_t s,
                        bool pdl) {
  KernelFn f = pick(wtype, pro, epi, l.rs, l.mc);
  if (!f || l.ns > 16 || l.nwc > kMaxConsumers || a.w.ds % 8 || a.w.cols % 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.grid);
  cfg.blockDim = dim3(l.threads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, f, a, l);
}

}  // namespace dls
