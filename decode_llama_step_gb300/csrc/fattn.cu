// Causal prefill attention on the 5th-generation tensor cores (flash
// attention): T query tokens at positions pos0 .. pos0+T-1 of one sequence
// attend to keys 0 .. their own position in the sequence's paged fp16 cache
// (engine page, section 4.4: causal softmax with the mask fused; SwarmKV
// page, section 2: prefill computes attention over the whole prompt once).
//
// CTA = (KV head, block of 128 / G query tokens): its 128 query rows are the
// G heads of the group for each of those tokens (row r = token r / G, head
// r % G), so one K/V tile serves all of them.  Per 128-key tile:
//   S = Q K^T   tcgen05.mma kind::f16, M = 128 rows, N = 128 keys, K = hd,
//               fp32 accumulators in tensor memory
//   softmax     warps 2-5, thread = row: scale, causal mask, running max,
//               P = exp(S - max) rounded to fp16 into shared memory
//   O_t = P V   M = 128, N = hd, K = 128 keys (V read as an MN-major operand)
//   o = o * exp(max_old - max_new) + O_t   in the softmax threads' registers
// K/V tiles come from the pages by 2-D TMA (128-byte swizzle, the MMA's
// operand layout); pieces of a tile that lie past the sequence's pages are
// loaded from outside the tensor, which the TMA fills with zeros.
// Every wait is bounded (2 s) and sets an abort flag; nothing is stored then.
#include <math.h>

#include "kernels.h"
#include "tc.cuh"

namespace dls {

namespace {

constexpr int FBK = 128;      // keys per tile
constexpr int FROWS = 128;    // query rows per CTA
constexpr int FTHREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int FNS = 2;        // K/V ring stages
constexpr uint64_t kWaitNsF = 2000000000ull;

template <int HD>
struct FCfg {
  static constexpr int KA = HD / 64;              // 64-wide swizzle atoms along the head dimension
  static constexpr int kQ = FROWS * HD * 2;       // fp16 Q tile
  static constexpr int kKV = FBK * HD * 2;        // one K or V tile
  static constexpr int kP = FROWS * FBK * 2;      // fp16 P tile
  static constexpr int kBarOff = kQ + FNS * 2 * kKV + kP;
  static constexpr int kSmem = kBarOff + 256 + 1024;
  static constexpr int kTmemCols = 256;           // S: columns 0-127, O: 128 .. 128+HD
};

struct FBars {
  uint64_t kv_full[FNS], kv_empty[FNS], q_full, s_full, s_free, p_full, o_full, o_free;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, int* abort_flag, bool heed_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 63) == 0) {
      if (heed_abort && *(volatile int*)abort_flag) return false;
      if (global_ns() - t0 > kWaitNsF) {
        *(volatile int*)abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int HD, int G>
__global__ void __launch_bounds__(FTHREADS, 1) fattn_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                            const __grid_constant__ CUtensorMap tm_v,
                                                            const FattnArgs a) {
  using C = FCfg<HD>;
  constexpr int BQ = FROWS / G;  // query tokens per CTA
  extern __shared__ uint8_t fsm[];
  const uint32_t raw = smem_u32(fsm);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t qbase = raw + pad;
  const uint32_t kvbase = qbase + C::kQ;                 // stage s: K at + 2 s kKV, V at + (2 s + 1) kKV
  const uint32_t pbase = kvbase + FNS * 2 * C::kKV;
  FBars& sh = *reinterpret_cast<FBars*>(fsm + pad + C::kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.x;
  const int qb = gridDim.y - 1 - blockIdx.y;             // the longest blocks start first
  const int q0 = qb * BQ;
  const int last_pos = a.pos0 + min(a.T, q0 + BQ) - 1;  // newest query of the block
  const int n_tiles = last_pos / FBK + 1;
  const int pr = a.page_tokens < FBK ? a.page_tokens : FBK;  // keys per TMA piece
  const int n_pieces = FBK / pr;

  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem), C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < FNS; ++i) {
      mbar_init(smem_u32(&sh.kv_full[i]), 1);
      mbar_init(smem_u32(&sh.kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&sh.q_full), 4);
    mbar_init(smem_u32(&sh.s_full), 1);
    mbar_init(smem_u32(&sh.s_free), 4);
    mbar_init(smem_u32(&sh.p_full), 4);
    mbar_init(smem_u32(&sh.o_full), 1);
    mbar_init(smem_u32(&sh.o_free), 4);
    sh.abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ---------------- TMA producer: K and V tiles, piece by piece (pages)
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % FNS;
        if (j >= FNS && !fwait(smem_u32(&sh.kv_empty[s]), ((j / FNS) - 1) & 1, &sh.abort)) break;
        const uint32_t bar = smem_u32(&sh.kv_full[s]);
        mbar_expect_tx(bar, 2 * C::kKV);
        const uint32_t kd = kvbase + 2 * s * C::kKV, vd = kd + C::kKV;
        for (int p = 0; p < n_pieces; ++p) {
          const int key0 = j * FBK + p * pr;
          const int lp = key0 / a.page_tokens;
          const int page = (key0 <= last_pos && lp < a.max_pages) ? a.ptab[lp] : -1;
          // a piece with no page is read from past the end of the pool: zeros
          const int y = page >= 0 ? (page * a.n_kv + kvh) * a.page_tokens + (key0 % a.page_tokens) : a.pool_rows;
#pragma unroll
          for (int at = 0; at < C::KA; ++at) {
            tma_load_2d(kd + at * (FBK * 128) + p * pr * 128, &tm_k, at * 64, y, bar);
            tma_load_2d(vd + at * (FBK * 128) + p * pr * 128, &tm_v, at * 64, y, bar);
          }
        }
        issued = j + 1;
      }
      for (int j = issued > FNS ? issued - FNS : 0; j < issued; ++j)
        fwait(smem_u32(&sh.kv_full[j % FNS]), (j / FNS) & 1, &sh.abort, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t id_s = umma_idesc_f16(FROWS, FBK);
      constexpr uint32_t id_o = umma_idesc_f16_bmn(FROWS, HD);
      const uint32_t t_s = tmem, t_o = tmem + 128;
      bool go = fwait(smem_u32(&sh.q_full), 0, &sh.abort);
      for (int j = 0; go && j < n_tiles; ++j) {
        const int s = j % FNS;
        if (!fwait(smem_u32(&sh.kv_full[s]), (j / FNS) & 1, &sh.abort)) break;
        if (j > 0 && !fwait(smem_u32(&sh.s_free), (j - 1) & 1, &sh.abort)) break;
        tc_fence_after();
        const uint32_t kd = kvbase + 2 * s * C::kKV, vd = kd + C::kKV;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (FROWS * 128) + (ks & 3) * 32;
          umma_f16(t_s, umma_desc_k128(qbase + off), umma_desc_k128(kd + off), id_s, ks != 0);
        }
        umma_commit(smem_u32(&sh.s_full));
        if (!fwait(smem_u32(&sh.p_full), j & 1, &sh.abort)) break;
        if (j > 0 && !fwait(smem_u32(&sh.o_free), (j - 1) & 1, &sh.abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < FBK / 16; ++ks) {
          const uint32_t aoff = (ks >> 2) * (FROWS * 128) + (ks & 3) * 32;
          umma_f16(t_o, umma_desc_k128(pbase + aoff), umma_desc_mn128(vd + ks * 16 * 128, FBK * 128, 1024), id_o,
                   ks != 0);
        }
        umma_commit(smem_u32(&sh.o_full));
        umma_commit(smem_u32(&sh.kv_empty[s]));
      }
    }
    __syncwarp();
  } else {
    // ---------------- softmax (thread = query row r; TMEM lane r)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int tl = r / G, h = r % G;
    const int t = q0 + tl;
    const bool row_ok = t < a.T;
    const int qpos = a.pos0 + t;
    // Q row -> fp16, swizzled (atom at = d / 64, 16-byte chunk (d % 64) / 8)
    {
      const float* qr = a.q + ((size_t)t * a.n_heads + (size_t)kvh * G + h) * HD;
#pragma unroll
      for (int c = 0; c < HD / 8; ++c) {
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (row_ok) {
          v0 = *reinterpret_cast<const float4*>(qr + 8 * c);
          v1 = *reinterpret_cast<const float4*>(qr + 8 * c + 4);
        }
        uint4 pk;
        pk.x = pack_h2(v0.x, v0.y);
        pk.y = pack_h2(v0.z, v0.w);
        pk.z = pack_h2(v1.x, v1.y);
        pk.w = pack_h2(v1.z, v1.w);
        const int at = c >> 3, j8 = c & 7;
        sts128(qbase + at * (FROWS * 128) + r * 128 + ((j8 ^ (r & 7)) << 4), pk);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.q_full));
    }
    const float sl2 = 1.4426950408889634f / sqrtf((float)HD);  // log2(e) / sqrt(hd)
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    float o[HD];
#pragma unroll
    for (int d = 0; d < HD; ++d) o[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!fwait(smem_u32(&sh.s_full), j & 1, &sh.abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kbase = j * FBK;
      // pass 1: row max of the masked, scaled scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < FBK / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(trow + c * 16, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (kbase + c * 16 + i <= qpos) mx = fmaxf(mx, __uint_as_float(v[i]));
      }
      const float m_new = fmaxf(m_run, mx * sl2);
      // pass 2: P = exp2(s * sl2 - m_new) as fp16, row sum
      float sum = 0.f;
#pragma unroll 1
      for (int c = 0; c < FBK / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(trow + c * 16, v);
        tmem_wait_ld();
        float p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool in = kbase + c * 16 + i <= qpos && m_new != -INFINITY;
          p[i] = in ? exp2f(__uint_as_float(v[i]) * sl2 - m_new) : 0.f;
          sum += p[i];
        }
        // keys 16c .. 16c+15 = 16-byte chunks 2c, 2c+1 of the row (atom = chunk / 8)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kc = 2 * c + hh, at = kc >> 3, j8 = kc & 7;
          uint4 pk;
          pk.x = pack_h2(p[8 * hh + 0], p[8 * hh + 1]);
          pk.y = pack_h2(p[8 * hh + 2], p[8 * hh + 3]);
          pk.z = pack_h2(p[8 * hh + 4], p[8 * hh + 5]);
          pk.w = pack_h2(p[8 * hh + 6], p[8 * hh + 7]);
          sts128(pbase + at * (FROWS * 128) + r * 128 + ((j8 ^ (r & 7)) << 4), pk);
        }
      }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.s_free));
        mbar_arrive(smem_u32(&sh.p_full));
      }
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      // O tile of this key block -> rescaled running sum
      if (!fwait(smem_u32(&sh.o_full), j & 1, &sh.abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < HD / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(trow + 128 + c * 16, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[c * 16 + i] = fmaf(o[c * 16 + i], alpha, __uint_as_float(v[i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.o_free));
    }
    ok = __all_sync(0xffffffffu, ok && !*(volatile int*)&sh.abort);
    if (ok && row_ok) {
      const float inv = 1.0f / l_run;
      const size_t off = (size_t)t * a.ld_out + ((size_t)kvh * G + h) * HD;
      __half* orow = a.out + off;
      __half* lrow = a.out_lo + off;
#pragma unroll
      for (int c = 0; c < HD / 8; ++c) {
        uint4 pk, pl;
        pk.x = pack_h2(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
        pk.y = pack_h2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
        pk.z = pack_h2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
        pk.w = pack_h2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
        // lo plane: what fp16 rounding dropped
        const uint32_t* hw = &pk.x;
        uint32_t* lw = &pl.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
          lw[j] = pack_h2(o[8 * c + 2 * j] * inv - f.x, o[8 * c + 2 * j + 1] * inv - f.y);
        }
        *reinterpret_cast<uint4*>(orow + 8 * c) = pk;
        *reinterpret_cast<uint4*>(lrow + 8 * c) = pl;
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

using FaFn = void (*)(const CUtensorMap, const CUtensorMap, const FattnArgs);

template <int HD>
FaFn fa_pick(int g) {
  switch (g) {
    case 1: return fattn_kernel<HD, 1>;
    case 2: return fattn_kernel<HD, 2>;
    case 4: return fattn_kernel<HD, 4>;
    case 8: return fattn_kernel<HD, 8>;
    case 16: return fattn_kernel<HD, 16>;
  }
  return nullptr;
}

FaFn fa_select(int hd, int g, int* smem) {
  if (hd == 128) {
    *smem = FCfg<128>::kSmem;
    return fa_pick<128>(g);
  }
  if (hd == 64) {
    *smem = FCfg<64>::kSmem;
    return fa_pick<64>(g);
  }
  return nullptr;
}

}  // namespace

bool fattn_supported(int head_dim, int g, int page_tokens) {
  int smem = 0;
  return fa_select(head_dim, g, &smem) != nullptr && page_tokens >= 8 && (page_tokens % 8) == 0 &&
         (page_tokens >= FBK ? page_tokens % FBK == 0 : FBK % page_tokens == 0);
}

cudaError_t fattn_setup_attributes() {
  for (int hd : {64, 128})
    for (int g : {1, 2, 4, 8, 16}) {
      int smem = 0;
      FaFn f = fa_select(hd, g, &smem);
      cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
  return cudaSuccess;
}

cudaError_t launch_fattn(const FattnArgs& a, const __half* k_pool, const __half* v_pool, cudaStream_t s) {
  const int g = a.n_heads / a.n_kv;
  int smem = 0;
  FaFn f = fa_select(a.head_dim, g, &smem);
  if (!f || !fattn_supported(a.head_dim, g, a.page_tokens) || a.T < 1 || a.ld_out % 8 || !a.out_lo)
    return cudaErrorInvalidValue;
  CUtensorMap tk, tv;
  const int pr = a.page_tokens < FBK ? a.page_tokens : FBK;
  if (!make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k_pool, a.head_dim, a.pool_rows, a.head_dim * 2, 64, pr,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, v_pool, a.head_dim, a.pool_rows, a.head_dim * 2, 64, pr,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int bq = FROWS / g;
  dim3 grid(a.n_kv, (a.T + bq - 1) / bq);
  f<<<grid, FTHREADS, smem, s>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace dls
