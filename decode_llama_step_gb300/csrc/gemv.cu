// Batch-1 dequant-GEMV y = W x for Q8_0 / Q4_0 weights, the decode step's
// projections (engine page, section 4.4: a GEMV specialised for the
// single-token vector-matrix product; RMSNorm fused into it; SwiGLU fused
// with the projection).
//
// Design (HBM-bound, ~2.4 ALU ops per weight):
//  * Each CTA owns a contiguous, balanced range of rows, so it streams one
//    contiguous slice of the code array and of the scale array.
//  * A warp owns K-chunks of 512 (Q8_0) / 1024 (Q4_0) columns: per row each
//    lane issues one 16-byte non-allocating load, R = 8 rows at a time,
//    double-buffered, so 128-256 bytes per lane are in flight.
//  * Codes become exact fp32 through the 0x4B0000bb magic pattern (one byte
//    permute per value); products accumulate with packed f32x2 FMAs.
//  * Per row the R partial sums reduce across lanes with a halving
//    butterfly (9 shuffles for 8 rows), then across warps in shared memory
//    in a fixed order: the result is deterministic.
//  * Prologue: the activation vector goes to shared memory, optionally as
//    rmsnorm(x) * g or as silu(gate) * up.  Before waiting on the previous
//    kernel (programmatic dependent launch) the CTA asks L2 to prefetch the
//    head of its weight slice: weights never depend on the previous kernel.
//  * Epilogues: store, residual add, or RoPE on (q, k) pairs plus the fp16
//    K/V append into the paged cache.
#include "kernels.h"

namespace dls {

namespace {

constexpr int R = 8;             // rows in flight per warp
constexpr int kMaxThreads = 256;   // at most 8 warps (gemv_plan)
constexpr int kPrefetchBytes = 48 * 1024;

template <int WT>
struct Geo {
  static constexpr int CH = WT == 8 ? 512 : 1024;  // columns per warp chunk
};

template <int WT>
__device__ __forceinline__ size_t row_bytes(int nb) {
  return WT == 8 ? (size_t)nb * 32 : (size_t)nb * 16;
}

struct Item {
  uint4 v[R];
  uint32_t d[R];   // fp16 bits of the scale (0 when the slot is empty)
};

template <int WT>
__device__ __forceinline__ void load_item(Item& it, const MatDev& w, int row0, int nrows, int chunk, int lane) {
  const int nb = w.nb;
  const int kpad = nb * 32;
  bool ok;
  size_t qoff;
  int blk;
  if (WT == 8) {
    const int col = chunk * 512 + lane * 16;
    ok = col < kpad;
    qoff = (size_t)col;
    blk = col >> 5;
  } else {
    blk = chunk * 32 + lane;
    ok = blk < nb;
    qoff = (size_t)blk * 16;
  }
  const size_t rb = row_bytes<WT>(nb);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (ok && r < nrows) {
      const int row = row0 + r;
      it.v[r] = ld_stream(w.qs + (size_t)row * rb + qoff);
      it.d[r] = ld_stream_u16(w.d + (size_t)row * nb + blk);
    } else {
      it.v[r] = make_uint4(0, 0, 0, 0);
      it.d[r] = 0;
    }
  }
}

template <int WT>
__device__ __forceinline__ void compute_item(const Item& it, float (&acc)[R], const float* s_x, int nb, int chunk,
                                             int lane) {
  const int kpad = nb * 32;
  if (WT == 8) {
    const int col = chunk * 512 + lane * 16;
    if (col >= kpad) return;
    const float4* xv = reinterpret_cast<const float4*>(s_x + col);
    f2_t x2[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 t = xv[m];
      x2[2 * m] = pk2(t.x, t.y);
      x2[2 * m + 1] = pk2(t.z, t.w);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      f2_t s = pk2(0.f, 0.f);
      const uint32_t wv[4] = {it.v[r].x, it.v[r].y, it.v[r].z, it.v[r].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f2_t p01, p23;
        i8x4_to_f2(wv[k], p01, p23);
        s = ffma2(p01, x2[2 * k], s);
        s = ffma2(p23, x2[2 * k + 1], s);
      }
      const float2 sf = upk2(s);
      acc[r] = fmaf(__half2float(__ushort_as_half((unsigned short)it.d[r])), sf.x + sf.y, acc[r]);
    }
  } else {
    const int blk = chunk * 32 + lane;
    if (blk >= nb) return;
    const float4* xv = reinterpret_cast<const float4*>(s_x + blk * 32);
    f2_t x2[16];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 t = xv[m];
      x2[2 * m] = pk2(t.x, t.y);
      x2[2 * m + 1] = pk2(t.z, t.w);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      f2_t s = pk2(0.f, 0.f);
      const uint32_t wv[4] = {it.v[r].x, it.v[r].y, it.v[r].z, it.v[r].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // bytes 4k..4k+3: low nibbles = elements 4k.., high nibbles = 16+4k..
        const uint32_t lo = wv[k] & 0x0F0F0F0Fu;
        const uint32_t hi = (wv[k] >> 4) & 0x0F0F0F0Fu;
        f2_t a01, a23, b01, b23;
        u4x4_to_f2(lo, a01, a23);
        u4x4_to_f2(hi, b01, b23);
        s = ffma2(a01, x2[2 * k], s);
        s = ffma2(a23, x2[2 * k + 1], s);
        s = ffma2(b01, x2[8 + 2 * k], s);
        s = ffma2(b23, x2[8 + 2 * k + 1], s);
      }
      const float2 sf = upk2(s);
      acc[r] = fmaf(__half2float(__ushort_as_half((unsigned short)it.d[r])), sf.x + sf.y, acc[r]);
    }
  }
}

// Sum acc[0..7] over the warp; the total of row (lane >> 2) & 7 ends in
// every lane of that quad.
__device__ __forceinline__ float butterfly8(const float (&acc)[R], int lane) {
  float t4[4], t2[2];
  const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = b16 ? acc[j] : acc[4 + j];
    const float keep = b16 ? acc[4 + j] : acc[j];
    t4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = b8 ? t4[j] : t4[2 + j];
    const float keep = b8 ? t4[2 + j] : t4[j];
    t2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float t1 = (b4 ? t2[1] : t2[0]) + __shfl_xor_sync(0xffffffffu, b4 ? t2[0] : t2[1], 4);
  t1 += __shfl_xor_sync(0xffffffffu, t1, 2);
  t1 += __shfl_xor_sync(0xffffffffu, t1, 1);
  return t1;
}

__device__ __forceinline__ float block_sum(float v, float* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < nw; ++w) t += s_red[w];  // fixed order: deterministic
  return t;
}

template <int WT, int PRO, int EPI>
__global__ void __launch_bounds__(kMaxThreads) gemv_kernel(const GemvArgs a, const int rb_cap) {
  extern __shared__ __align__(16) float smem[];
  const MatDev& w = a.w;
  const int nb = w.nb, kpad = nb * 32, cols = w.cols;
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* s_x = smem;                  // [kpad]
  float* s_part = smem + kpad;        // [nw][rb_cap]
  __shared__ float s_red[32];

  const int units = (w.rows + a.unit - 1) / a.unit;
  const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
  const int r0 = u0 * a.unit, r1 = min(w.rows, u1 * a.unit);

  // Weights do not depend on the previous kernel: start pulling this CTA's
  // slice into L2 before waiting for it.
  if (threadIdx.x == 0 && r1 > r0) {
    const size_t rbytes = row_bytes<WT>(nb);
    const uint8_t* qa = w.qs + (size_t)r0 * rbytes;
    const size_t qn = min((size_t)(r1 - r0) * rbytes, (size_t)kPrefetchBytes) & ~(size_t)15;
    if (qn) prefetch_l2(qa, (uint32_t)qn);
    const uintptr_t da = reinterpret_cast<uintptr_t>(w.d + (size_t)r0 * nb);
    const uintptr_t da16 = da & ~(uintptr_t)15;
    const size_t dn = (min((size_t)(r1 - r0) * nb * 2, (size_t)kPrefetchBytes / 16) + (da - da16)) & ~(size_t)15;
    if (dn) prefetch_l2(reinterpret_cast<const void*>(da16), (uint32_t)dn);
  }

  griddep_wait();

  // ---- prologue: activation vector -> shared memory
  if (PRO == PRO_RMSNORM) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < cols; i += blockDim.x) {
      const float v = a.x[i];
      ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, s_red);
    const float rs = 1.0f / sqrtf(ss / (float)cols + a.eps);
    for (int i = threadIdx.x; i < kpad; i += blockDim.x) s_x[i] = i < cols ? a.x[i] * rs * a.g[i] : 0.f;
  } else if (PRO == PRO_SWIGLU) {
    for (int i = threadIdx.x; i < kpad; i += blockDim.x) s_x[i] = i < cols ? silu(a.x[i]) * a.x[cols + i] : 0.f;
  } else {
    for (int i = threadIdx.x; i < kpad; i += blockDim.x) s_x[i] = i < cols ? a.x[i] : 0.f;
  }
  __syncthreads();
  griddep_launch();

  constexpr int CH = Geo<WT>::CH;
  const int nchunk = (kpad + CH - 1) / CH;
  const int mc = warp < nchunk ? (nchunk - warp + nw - 1) / nw : 0;
  const int nwa = min(nw, nchunk);

  int32_t pos = 0, seq = 0;
  if (EPI == EPI_QKV) {
    pos = a.sp->pos[a.brow];
    seq = a.sp->seq[a.brow];
  }

  for (int rb0 = r0; rb0 < r1; rb0 += rb_cap) {
    const int rbn = min(rb_cap, r1 - rb0);
    const int ngroups = (rbn + R - 1) / R;
    const int nitems = ngroups * mc;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    Item A, B;
    auto item_rows = [&](int i, int& row0, int& nrows, int& chunk) {
      const int g = i / mc, j = i - g * mc;
      row0 = rb0 + g * R;
      nrows = min(R, rb0 + rbn - row0);
      chunk = warp + j * nw;
    };
    auto finish_group = [&](int i) {
      const int g = i / mc;
      const float t = butterfly8(acc, lane);
      const int rr = g * R + ((lane >> 2) & 7);
      if ((lane & 3) == 0 && rr < rbn) s_part[warp * rb_cap + rr] = t;
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = 0.f;
    };
    if (nitems > 0) {
      int row0, nrows, chunk;
      item_rows(0, row0, nrows, chunk);
      load_item<WT>(A, w, row0, nrows, chunk, lane);
    }
    for (int i = 0; i < nitems; i += 2) {
      int row0, nrows, chunk;
      if (i + 1 < nitems) {
        item_rows(i + 1, row0, nrows, chunk);
        load_item<WT>(B, w, row0, nrows, chunk, lane);
      }
      item_rows(i, row0, nrows, chunk);
      compute_item<WT>(A, acc, s_x, nb, chunk, lane);
      if ((i % mc) == mc - 1) finish_group(i);
      if (i + 1 < nitems) {
        if (i + 2 < nitems) {
          item_rows(i + 2, row0, nrows, chunk);
          load_item<WT>(A, w, row0, nrows, chunk, lane);
        }
        item_rows(i + 1, row0, nrows, chunk);
        compute_item<WT>(B, acc, s_x, nb, chunk, lane);
        if (((i + 1) % mc) == mc - 1) finish_group(i + 1);
      }
    }
    __syncthreads();

    // ---- cross-warp reduction (fixed order) and epilogue
    if (EPI == EPI_QKV) {
      const int hd = a.kv.head_dim;
      for (int pi = threadIdx.x; pi < (rbn >> 1); pi += blockDim.x) {
        const int rr = pi * 2, r = rb0 + rr;
        float v0 = 0.f, v1 = 0.f;
        for (int ww = 0; ww < nwa; ++ww) {
          v0 += s_part[ww * rb_cap + rr];
          v1 += s_part[ww * rb_cap + rr + 1];
        }
        if (r < a.q_rows + a.kv_rows) {  // q or k: rotate the adjacent pair
          if (pos < 0 || pos >= a.rope_len) {
            atomicOr(&a.sp->status, kBadPos);
            continue;
          }
          const int i = (r % hd) >> 1;
          const float2 cs = a.rope_cs[(size_t)pos * (hd >> 1) + i];
          const float t0 = v0 * cs.x - v1 * cs.y;
          const float t1 = v0 * cs.y + v1 * cs.x;
          v0 = t0;
          v1 = t1;
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
          const int page = (pos >= 0 && lp < a.kv.max_pages) ? a.kv.page_table[(size_t)seq * a.kv.max_pages + lp] : -1;
          if (page < 0) {
            atomicOr(&a.sp->status, kBadPage);
            continue;
          }
          const size_t off = (((size_t)page * a.kv.n_kv + kvh) * pt + (pos % pt)) * hd + dim;
          __half* dst = (is_k ? a.kv.k_pool : a.kv.v_pool) + off;
          *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(v0, v1);
        }
      }
    } else {
      for (int rr = threadIdx.x; rr < rbn; rr += blockDim.x) {
        float v = 0.f;
        for (int ww = 0; ww < nwa; ++ww) v += s_part[ww * rb_cap + rr];
        if (EPI == EPI_RESID) a.y[rb0 + rr] += v;
        else a.y[rb0 + rr] = v;
      }
    }
    __syncthreads();
  }
}

template <int WT, int PRO, int EPI>
constexpr auto kernel_ptr() {
  return &gemv_kernel<WT, PRO, EPI>;
}

using KernelFn = void (*)(const GemvArgs, const int);

KernelFn pick(int wtype, int pro, int epi) {
#define DLS_PICK(WT, P, E) \
  if (wtype == WT && pro == P && epi == E) return kernel_ptr<WT, P, E>();
  DLS_PICK(8, PRO_RMSNORM, EPI_QKV)
  DLS_PICK(8, PRO_COPY, EPI_RESID)
  DLS_PICK(8, PRO_RMSNORM, EPI_STORE)
  DLS_PICK(8, PRO_SWIGLU, EPI_RESID)
  DLS_PICK(8, PRO_COPY, EPI_STORE)
  DLS_PICK(4, PRO_RMSNORM, EPI_QKV)
  DLS_PICK(4, PRO_COPY, EPI_RESID)
  DLS_PICK(4, PRO_RMSNORM, EPI_STORE)
  DLS_PICK(4, PRO_SWIGLU, EPI_RESID)
  DLS_PICK(4, PRO_COPY, EPI_STORE)
#undef DLS_PICK
  return nullptr;
}

constexpr int kRbCapRows = 2048;

}  // namespace

GemvLaunch gemv_plan(int wtype, int rows, int nb, int num_sms, int unit) {
  const int kpad = nb * 32;
  const int CH = wtype == 8 ? 512 : 1024;
  const int nchunk = (kpad + CH - 1) / CH;
  // warps per CTA: the largest divisor of the chunk count that is <= 8, so
  // every warp owns the same number of chunks
  int nw = 1;
  for (int d = 1; d <= 8; ++d)
    if (nchunk % d == 0) nw = d;
  if (nchunk > 8 && nw < 4) nw = 8;  // awkward counts: accept a short last round
  const int ctas_per_sm = nw >= 8 ? 1 : (nw >= 4 ? 2 : 4);
  const int units = (rows + unit - 1) / unit;
  int grid = num_sms * ctas_per_sm;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  const int rows_cta = ((units + grid - 1) / grid) * unit;
  int rb = rows_cta < kRbCapRows ? rows_cta : kRbCapRows;
  rb = (rb + 1) & ~1;
  GemvLaunch l;
  l.grid = grid;
  l.threads = nw * 32;
  l.smem = (kpad + nw * rb) * 4;
  return l;
}

cudaError_t gemv_setup_attributes() {
  const int pros[3] = {PRO_COPY, PRO_RMSNORM, PRO_SWIGLU};
  const int epis[3] = {EPI_STORE, EPI_RESID, EPI_QKV};
  for (int wt : {8, 4})
    for (int p : pros)
      for (int e : epis) {
        KernelFn f = pick(wt, p, e);
        if (!f) continue;
        cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (err != cudaSuccess) return err;
      }
  return cudaSuccess;
}

cudaError_t launch_gemv(int wtype, int pro, int epi, const GemvArgs& a, const GemvLaunch& l, cudaStream_t s,
                        bool pdl) {
  KernelFn f = pick(wtype, pro, epi);
  if (!f) return cudaErrorInvalidValue;
  const int nw = l.threads / 32;
  const int rb = (l.smem / 4 - a.w.nb * 32) / nw;
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
  return cudaLaunchKernelEx(&cfg, f, a, rb);
}

}  // namespace dls
