// Persistent decode-step kernel: the whole single-token decode step of a
// resident model (embedding, every layer's QKV GEMV + RoPE + KV append,
// attention, O GEMV, gate/up GEMV + SwiGLU, down GEMV, final norm + LM head,
// and optionally the greedy pick) in one cooperative launch with one CTA per
// SM.
//
// Why: the step is HBM-bound on weights, but run as ~160 separate kernels
// every boundary costs a launch, a pipeline ramp and a latency-bound
// prologue while HBM idles.  Here one producer warp per CTA streams this
// CTA's slice of every phase's weights -- and the K/V tiles of its
// attention task -- through one shared-memory ring in program order, never
// waiting on the phase boundaries (weights and past K/V do not depend on
// them).  Eight consumer warps run the phases in order, separated by grid
// barriers; while they wait at a barrier the ring keeps filling.
//
// Phases per token (pages: the engine page, sections 1 and 4.4):
//   embed -> for each layer: QKV | attention | O | gate/up | down -> head [-> argmax]
// with a grid barrier after each.  Row slices, chunk ownership, reduction
// orders and epilogues follow the standalone decode GEMV (gemv.cu), and the
// attention task follows attention.cu's split-K scheme with the splits
// mapped one per CTA.
//
// Every wait is bounded: an mbarrier or grid-barrier wait that runs out
// sets a global abort flag that ends all other waits, and a status bit the
// host reads.  The producer never leaves with copies in flight.
#include <math.h>
#include <stdlib.h>

#include "gemv_core.cuh"
#include "kernels.h"

namespace dls {

namespace {

constexpr int NWC = 8;               // consumer warps
constexpr int NTHR = 32 * (NWC + 2);  // consumers, the producer warp, the L2-hint warp
constexpr int kRB = 64;              // rows per epilogue block
constexpr int kTile = 32;            // attention tokens per ring stage
constexpr int kMaxStages = 16;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kTr = 8;               // per-CTA trace slots per phase

// Consumer-side timestamp of this CTA in the current phase (profiling only):
// slot 4 = prologue done, 5 = last stage consumed, 6 = epilogue done, 7 =
// first stage's data ready (thread 0's warp).
__device__ __forceinline__ void ctmark(const StepArgs& A, unsigned epoch, int slot) {
  if (A.ctrace && threadIdx.x == 0) A.ctrace[((size_t)epoch * gridDim.x + blockIdx.x) * kTr + slot] = global_ns();
}

constexpr int kMaxSkipLayers = 256;  // layer-skip flags kept in shared memory

struct Sh {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float red[32];
  int last;
  unsigned epoch_pub;  // grid barriers the consumers have passed
  uint8_t skip[kMaxSkipLayers];  // the step's layer-skip flags (copied once from global memory)
};

struct Ctx {
  const StepArgs* A;
  Sh* sh;
  uint8_t* ring;
  float* s_part;   // [NWC][kRB]
  float* s_q;      // [G*HD]
  float* s_wm;     // [NWC][G]
  float* s_wl;     // [NWC][G]
  float* s_wo;     // [NWC][G*HD]
  __half* s_kvpos; // [2][HD]: K and V of position pos (attention), loaded with q
  int sidx;        // ring stages consumed / produced so far
  int slot;        // sidx % ns
  uint32_t par;    // (sidx / ns) & 1: the phase parity of the current slot's use
  unsigned epoch;  // grid barriers passed (thread 0)
  int pos, seq;
  int pos_page;    // page holding position pos, -1 if none
};

__device__ __forceinline__ void advance(Ctx& c, int ns) {
  ++c.sidx;
  if (++c.slot == ns) {
    c.slot = 0;
    c.par ^= 1u;
  }
}

__device__ __forceinline__ bool aborted(const StepArgs& A) { return *(volatile int*)A.abort != 0; }

__device__ __forceinline__ void set_abort(const StepArgs& A) {
  atomicExch(A.abort, 1);
  atomicOr(&A.sp->status, kTimeout);
}

// mbarrier wait that also gives up when another CTA aborted
__device__ __forceinline__ bool wait_bar(const StepArgs& A, uint32_t bar, uint32_t parity, uint32_t sleep_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 4) __nanosleep(sleep_ns);
    if ((i & 63) == 0) {
      if (aborted(A)) return false;
      if (global_ns() - t0 > kWaitNs) {
        set_abort(A);
        return false;
      }
    }
  }
}

// All consumer warps of all CTAs; the producer warp never takes part.
// Thread 0 publishes the CTA's writes with a release add on the counter and
// waits for the whole grid with acquire loads (the CTA barriers on either
// side order the other threads' accesses around it).
__device__ __forceinline__ void grid_sync(Ctx& c) {
  const StepArgs& A = *c.A;
  named_bar(1, NWC * 32);
  if (A.trace && blockIdx.x == 0 && threadIdx.x == 0) A.trace[c.epoch + 1] = global_ns();  // phase end
  if (threadIdx.x == 0) {
    if (A.ctrace) A.ctrace[((size_t)c.epoch * gridDim.x + blockIdx.x) * kTr + 0] = global_ns();
    const unsigned target = (++c.epoch) * gridDim.x;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(A.bar) : "memory");
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(A.bar) : "memory");
      if (v >= target) break;
      if ((i & 15) == 15) {
        if (aborted(A)) break;
        const uint64_t now = global_ns();
        if (!t0) t0 = now;
        if (now - t0 > kWaitNs) {
          set_abort(A);
          break;
        }
      }
      if (i >= 64) __nanosleep(32);
    }
    if (A.ctrace) A.ctrace[((size_t)(c.epoch - 1) * gridDim.x + blockIdx.x) * kTr + 1] = global_ns();
    *(volatile unsigned*)&c.sh->epoch_pub = c.epoch;
  }
  named_bar(1, NWC * 32);
}

__device__ __forceinline__ void row_split(int rows, int unit, int& r0, int& r1) {
  const int units = (rows + unit - 1) / unit;
  const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
  r0 = u0 * unit;
  r1 = min(rows, u1 * unit);
}

template <int WT>
__device__ __forceinline__ size_t row_bytes_of(const MatDev& w) {
  return WT == 8 ? (size_t)w.nb * 32 : (size_t)w.nb * 16;
}

// While the consumers sit in the latency-bound attention and O phases, HBM
// would idle once the ring is full.  A warp of its own follows the
// consumers' phase counter and, when layer l's
// attention phase begins, hint this CTA's gate/up rows [pf_skip, pf_skip +
// pf_rows) of layer l (codes and scales) into L2, so the gate/up phase's
// stage copies find them there.  Bounded: gives up on an abort or after the
// wait limit.
template <int WT>
__device__ void hint_lanes(const Ctx& c) {
  const StepArgs& A = *c.A;
  const int lane = threadIdx.x & 31;
  int r0, r1;
  row_split(A.layers[0].gu.rows, 2, r0, r1);
  const int lo = min(r1, r0 + A.pf_skip), hi = min(r1, r0 + A.pf_skip + A.pf_rows);
  if (lo >= hi) return;
  const volatile unsigned* ep = &c.sh->epoch_pub;
  const uint64_t t0 = global_ns();
  unsigned done = 0;  // computed layers before l
  for (int l = 0; l < A.n_layers; ++l) {
    if (c.sh->skip[l]) continue;
    const unsigned target = 2u + 5u * done++;  // barriers passed when layer l's attention starts
    for (uint32_t i = 0; *ep < target; ++i) {
      __nanosleep(256);
      if ((i & 63) == 63 && (aborted(A) || global_ns() - t0 > kWaitNs)) return;
    }
    const MatDev& w = A.layers[l].gu;
    const size_t rb = row_bytes_of<WT>(w), db = (size_t)w.ds * 2;
    const uint8_t* q = w.qs + (size_t)lo * rb;
    const size_t nq = (size_t)(hi - lo) * rb;
    for (size_t off = (size_t)lane * 128; off < nq; off += 32 * 128) prefetch_line_l2(q + off);
    const uint8_t* d = reinterpret_cast<const uint8_t*>(w.d) + (size_t)lo * db;
    const size_t nd = (size_t)(hi - lo) * db;
    for (size_t off = (size_t)lane * 128; off < nd; off += 32 * 128) prefetch_line_l2(d + off);
  }
}

// ------------------------------------------------------------------ producer
//
// This CTA's copy stream in program order: per layer its QKV rows, its
// attention tiles, its O rows, gate/up rows and down rows; then its LM head
// rows.  One chunk fills one ring stage: RS whole rows (codes, then their
// scales at offset RS * row bytes) or one 32-token K/V tile (K, then V at
// offset kTile * HD * 2).

// Row ranges of this CTA in each GEMV phase (the same for every layer).
struct Rows {
  int qkv0, qkv1, o0, o1, gu0, gu1, dn0, dn1, hd0, hd1;
};

// A cursor over the stream.  Entering a phase sets up its base pointers
// and counts once, so a chunk costs a few adds.
struct PCur {
  int l = 0;    // layer; n_layers = the LM head
  int ph = -1;  // 0 QKV, 1 attention, 2 O, 3 gate/up, 4 down; -1 = not started
  int i = 0, n = 0;  // chunk index and count in the phase
  // GEMV phase: rows [row, row_end) remain; codes and scales of `row`
  const uint8_t* q;
  const uint8_t* d;
  uint32_t rb, db;
  int rs, row, row_end;
  // attention phase: tiles [tb, te) of this CTA's task
  int tb, te;
  const __half* kp;
  const __half* vp;
};

// One ring stage's copies: codes at 0 and scales at off_b (RS rows of a
// GEMV), or K at 0 and V at off_b of a 32-token tile, plus K2 and V2 of the
// next tile at 2 and 3 tile sizes (attention: two tiles per stage).
struct Chunk {
  const uint8_t* a;
  const uint8_t* b;
  const uint8_t* a2;
  const uint8_t* b2;
  uint32_t na, nb, n2;  // bytes (all 0: an empty stage)
  uint32_t off_b;
  bool bad_page;
};

__device__ __forceinline__ void attn_task(const StepArgs& A, int n, int& kvh, int& tb, int& te) {
  const int ntask = A.n_kv * A.S;
  kvh = blockIdx.x / A.S;
  const int sp = blockIdx.x % A.S;
  const int n_tiles = (n + kTile - 1) / kTile;
  const int per = (n_tiles + A.S - 1) / A.S;
  tb = sp * per;
  te = min(n_tiles, tb + per);
  if ((int)blockIdx.x >= ntask) te = tb;  // no task for this CTA
}

template <int WT>
__device__ __forceinline__ void gemv_phase(PCur& u, const MatDev& w, int r0, int r1, int rs) {
  u.rb = (uint32_t)row_bytes_of<WT>(w);
  u.db = (uint32_t)w.ds * 2;
  u.rs = rs;
  u.row = r0;
  u.row_end = r1;
  u.q = w.qs + (size_t)r0 * u.rb;
  u.d = reinterpret_cast<const uint8_t*>(w.d) + (size_t)r0 * u.db;
  u.n = r1 > r0 ? (r1 - r0 + rs - 1) / rs : 0;
}

// Set up phase (u.l, u.ph).
template <int WT, int HD, int RSA, int RSB>
__device__ void begin_phase(const Ctx& c, const Rows& R, PCur& u) {
  const StepArgs& A = *c.A;
  u.i = 0;
  if (u.l >= A.n_layers) {
    gemv_phase<WT>(u, A.head, R.hd0, R.hd1, RSA);
    if (!A.head_rows) u.n = 0;
    return;
  }
  if (c.sh->skip[u.l]) {  // a skipped layer streams nothing
    u.n = 0;
    return;
  }
  const StepLayer& L = A.layers[u.l];
  switch (u.ph) {
    case 0: gemv_phase<WT>(u, L.qkv, R.qkv0, R.qkv1, RSA); break;
    case 1: {
      int kvh;
      attn_task(A, c.pos + 1, kvh, u.tb, u.te);
      u.n = max(0, (u.te - u.tb + 1) / 2);  // two tiles per stage
      const size_t head_off = (size_t)kvh * A.page_tokens * HD;
      u.kp = L.k_pool + head_off;
      u.vp = L.v_pool + head_off;
      break;
    }
    case 2: gemv_phase<WT>(u, L.o, R.o0, R.o1, RSA); break;
    case 3: gemv_phase<WT>(u, L.gu, R.gu0, R.gu1, RSA); break;
    default: gemv_phase<WT>(u, L.down, R.dn0, R.dn1, RSB); break;
  }
}

// The next chunk of the stream at cursor u (advancing it); false at the end.
template <int WT, int HD, int RSA, int RSB>
__device__ bool next_chunk(const Ctx& c, const Rows& R, PCur& u, Chunk& ch) {
  const StepArgs& A = *c.A;
  while (u.ph < 0 || u.i >= u.n) {
    if (u.ph >= 0) {  // leave the finished phase
      if (u.l >= A.n_layers) return false;  // the LM head was the last phase
      if (++u.ph == 5) {
        u.ph = 0;
        ++u.l;
      }
    } else {
      u.ph = 0;
    }
    if (u.l > A.n_layers) return false;
    begin_phase<WT, HD, RSA, RSB>(c, R, u);
  }
  ch.bad_page = false;
  ch.n2 = 0;
  if (u.l < A.n_layers && u.ph == 1) {
    // tiles 2i and 2i + 1 of the task: K | V | K2 | V2
    ch.na = ch.nb = 0;
    ch.off_b = kTile * HD * 2;
    const int t = u.tb + 2 * u.i;
    // positions before pos are final; pos itself is written by this step
    const int n_old = max(0, min(kTile, c.pos - t * kTile));
    const int page = A.page_table[(size_t)c.seq * A.max_pages + (t * kTile) / A.page_tokens];
    ch.bad_page = page < 0;
    if (n_old > 0 && page >= 0) {
      const size_t base = ((size_t)page * A.n_kv * A.page_tokens + (t * kTile) % A.page_tokens) * HD;
      ch.a = reinterpret_cast<const uint8_t*>(u.kp + base);
      ch.b = reinterpret_cast<const uint8_t*>(u.vp + base);
      ch.na = ch.nb = (uint32_t)n_old * HD * 2;
    }
    if (t + 1 < u.te) {
      const int n_old2 = max(0, min(kTile, c.pos - (t + 1) * kTile));
      const int page2 = A.page_table[(size_t)c.seq * A.max_pages + ((t + 1) * kTile) / A.page_tokens];
      ch.bad_page |= page2 < 0;
      if (n_old2 > 0 && page2 >= 0) {
        const size_t base = ((size_t)page2 * A.n_kv * A.page_tokens + ((t + 1) * kTile) % A.page_tokens) * HD;
        ch.a2 = reinterpret_cast<const uint8_t*>(u.kp + base);
        ch.b2 = reinterpret_cast<const uint8_t*>(u.vp + base);
        ch.n2 = (uint32_t)n_old2 * HD * 2;
      }
    }
  } else {
    const int n = min(u.rs, u.row_end - u.row);
    ch.a = u.q;
    ch.na = (uint32_t)n * u.rb;
    ch.b = u.d;
    ch.nb = (uint32_t)n * u.db;
    ch.off_b = (uint32_t)u.rs * u.rb;
    u.q += ch.na;
    u.d += ch.nb;
    u.row += n;
  }
  ++u.i;
  return true;
}

// The producer warp's lane 0: fill the ring in stream order.
template <int WT, int HD, int RSA, int RSB>
__device__ void produce(Ctx& c) {
  const StepArgs& A = *c.A;
  Rows R;
  {
    const StepLayer& L0 = A.layers[0];  // every layer has the same shapes
    row_split(L0.qkv.rows, 2, R.qkv0, R.qkv1);
    row_split(L0.o.rows, 1, R.o0, R.o1);
    row_split(L0.gu.rows, 2, R.gu0, R.gu1);
    row_split(L0.down.rows, 1, R.dn0, R.dn1);
  }
  row_split(A.head.rows, 1, R.hd0, R.hd1);
  PCur rc;
  Chunk ch;
  int last_phase = -1;
  // the abort flag is checked inside waits only: a global load per chunk
  // would serialise an L2 round trip into every stage issue
  for (;;) {
    if (!next_chunk<WT, HD, RSA, RSB>(c, R, rc, ch)) break;
    const int phase = 1 + 5 * rc.l + (rc.l < A.n_layers ? rc.ph : 0);
    if (A.ctrace) {
      unsigned long long* t = A.ctrace + ((size_t)phase * gridDim.x + blockIdx.x) * kTr;
      const unsigned long long now = global_ns();
      if (phase != last_phase) t[2] = now;
      t[3] = now;
      last_phase = phase;
    }
    const int slot = c.slot;
    if (c.sidx >= A.ns) {
      const uint32_t bar = smem_u32(&c.sh->empty[slot]);
      const uint32_t parity = c.par ^ 1u;  // the slot's previous use
      if (!mbar_try_wait(bar, parity)) {
        const uint64_t t0 = global_ns();
        bool ok = true;
        for (uint32_t it = 1;; ++it) {
          if (mbar_try_wait(bar, parity)) break;
          if (it > 4) __nanosleep(200);
          if ((it & 63) == 0) {
            if (aborted(A)) {
              ok = false;
              break;
            }
            if (global_ns() - t0 > kWaitNs) {
              set_abort(A);
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
      }
    }
    const uint32_t bar = smem_u32(&c.sh->full[slot]);
    uint8_t* dst = c.ring + (size_t)slot * A.stage_bytes;
    if (ch.bad_page) atomicOr(&A.sp->status, kBadPage);
    const uint32_t total = ch.na + ch.nb + 2 * ch.n2;
    if (total == 0) {
      mbar_arrive(bar);
    } else {
      mbar_expect_tx(bar, total);
      if (ch.na) bulk_g2s(smem_u32(dst), ch.a, ch.na, bar);
      if (ch.nb) bulk_g2s(smem_u32(dst + ch.off_b), ch.b, ch.nb, bar);
      if (ch.n2) {
        bulk_g2s(smem_u32(dst + 2 * kTile * HD * 2), ch.a2, ch.n2, bar);
        bulk_g2s(smem_u32(dst + 3 * kTile * HD * 2), ch.b2, ch.n2, bar);
      }
    }
    advance(c, A.ns);
  }
  // never leave with copies in flight
  for (int s = max(0, c.sidx - A.ns); s < c.sidx; ++s) {
    const uint32_t bar = smem_u32(&c.sh->full[s % A.ns]);
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, (s / A.ns) & 1) && global_ns() - t0 < kWaitNs) __nanosleep(100);
  }
}

// ------------------------------------------------------------------ consumers

// The lane's activation slice (chunks warp, warp+NWC, ...), from L2.
template <int WT, int PRO, int MC>
__device__ __forceinline__ void load_x(Ctx& c, const MatDev& w, const float* x, const float* gain,
                                       XQ<WT> (&xq)[MC], bool (&valid)[MC]) {
  using Gm = Geo<WT>;
  constexpr int V4 = Gm::XV / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kpad = w.nb * 32, cols = w.cols;
  const int nchunk = (kpad + Gm::CH - 1) / Gm::CH;
  const int mc = warp < nchunk ? min(MC, (nchunk - warp + NWC - 1) / NWC) : 0;
  float4 raw[MC][V4];
  float4 gg[PRO == PRO_RMSNORM ? MC : 1][V4];
  // branch-free: every float4 of the lane's slices is loaded at once (a
  // slice past the matrix reads element 0 and is zeroed afterwards), so the
  // loads of all chunks, x and gains, are in flight together.  cols % 4 == 0
  // (checked when the kernel is planned): a float4 is all in or all out.
  bool in4[MC][V4];
#pragma unroll
  for (int k = 0; k < MC; ++k) {
    const int ch = warp + k * NWC;
    const int col0 = WT == 8 ? ch * 512 + lane * 16 : (ch * 32 + lane) * 32;
    valid[k] = k < mc && col0 < kpad;
#pragma unroll
    for (int m4 = 0; m4 < V4; ++m4) {
      const int i0 = col0 + 4 * m4;
      in4[k][m4] = valid[k] && i0 < cols;
      const int j0 = in4[k][m4] ? i0 : 0;
      raw[k][m4] = __ldcg(reinterpret_cast<const float4*>(x + j0));
      if (PRO == PRO_RMSNORM) gg[PRO == PRO_RMSNORM ? k : 0][m4] = *reinterpret_cast<const float4*>(gain + j0);
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
    named_bar(1, NWC * 32);  // previous readers of red[] are done
    if (lane == 0) c.sh->red[warp] = ss;
    named_bar(1, NWC * 32);
    float t = 0.f;
    for (int i = 0; i < NWC; ++i) t += c.sh->red[i];  // fixed order
    const float rs = 1.0f / sqrtf(t / (float)cols + c.A->eps);
#pragma unroll
    for (int k = 0; k < MC; ++k)
#pragma unroll
      for (int m4 = 0; m4 < V4; ++m4) {
        const float4 g = gg[PRO == PRO_RMSNORM ? k : 0][m4];
        raw[k][m4] = make_float4(raw[k][m4].x * rs * g.x, raw[k][m4].y * rs * g.y, raw[k][m4].z * rs * g.z,
                                 raw[k][m4].w * rs * g.w);
      }
  }
#pragma unroll
  for (int k = 0; k < MC; ++k) quantize_slice<WT>(reinterpret_cast<const float*>(raw[k]), xq[k]);
}

struct EpiArgs {
  float* y;
  // EPI_QKV
  __half* k_pool;
  __half* v_pool;
  // EPI_RESID: optional copy of the updated rows (the residual stream
  // after a layer, for the per-layer capture)
  float* cap;
};

template <int WT, int PRO, int EPI, int RS, int MC>
__device__ void consume_gemv(Ctx& c, const MatDev& w, int unit, const float* x, const float* gain, const EpiArgs& e) {
  using Gm = Geo<WT>;
  const StepArgs& A = *c.A;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  XQ<WT> xq[MC];
  bool valid[MC];
  load_x<WT, PRO, MC>(c, w, x, gain, xq, valid);
  ctmark(A, c.epoch, 4);
  int r0, r1;
  row_split(w.rows, unit, r0, r1);
  const int nrows = max(r1 - r0, 0);
  const int nst = (nrows + RS - 1) / RS;
  const size_t rb = row_bytes_of<WT>(w), db = (size_t)w.ds * 2;
  const int kpad = w.nb * 32;
  const int nchunk = (kpad + Gm::CH - 1) / Gm::CH;
  const int nwa = min(NWC, nchunk);
  constexpr int spb = kRB / RS;  // stages per epilogue block
  // residual rows of the first two epilogue blocks, read before the stages
  // arrive (no other CTA writes this CTA's rows during the phase)
  float res_pre[2] = {0.f, 0.f};
  if (EPI == EPI_RESID && tid < kRB) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int r = r0 + b * kRB + tid;
      if (r < r1) res_pre[b] = __ldcg(e.y + r);
    }
  }
  // RoPE factors of this thread's pair in the first two epilogue blocks,
  // loaded before the stages arrive (the position is fixed for the step)
  float2 cs_pre[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
  if (EPI == EPI_QKV && c.pos >= 0 && c.pos < A.rope_len && tid < kRB / 2) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int r = r0 + b * kRB + 2 * tid;
      if (r < r1 && r < A.q_rows + A.kv_rows) cs_pre[b] = A.rope_cs[(size_t)c.pos * (A.hd >> 1) + ((r % A.hd) >> 1)];
    }
  }
  for (int s = 0; s < nst; ++s) {
    const int slot = c.slot;
    const bool ok = wait_bar(A, smem_u32(&c.sh->full[slot]), c.par, 20);
    if (s == 0) ctmark(A, c.epoch, 7);
    const int rows_s = min(RS, nrows - s * RS);
    const uint32_t st = smem_u32(c.ring) + (uint32_t)slot * A.stage_bytes;
    float acc[RS];
#pragma unroll
    for (int rr = 0; rr < RS; ++rr) acc[rr] = 0.f;
    if (ok) {
      // branch-free: see the standalone GEMV
#pragma unroll
      for (int k = 0; k < MC; ++k) {
        const int ch = warp + k * NWC;
        const int qoff = valid[k] ? (WT == 8 ? ch * 512 + lane * 16 : (ch * 32 + lane) * 16) : 0;
        const int blk = valid[k] ? (WT == 8 ? (ch * 512 + lane * 16) >> 5 : ch * 32 + lane) : 0;
        const uint32_t qa = st + (uint32_t)qoff, da = st + (uint32_t)(RS * rb) + (uint32_t)blk * 2;
#pragma unroll
        for (int rr = 0; rr < RS; ++rr) {
          const uint4 q = lds128(qa + rr * (uint32_t)rb);
          const float d = lds_half_as_float(da + rr * (uint32_t)db);
          const float t = (float)idot16<WT>(q, xq[k]);
          acc[rr] = valid[k] ? fmaf(d * xq[k].s, t, acc[rr]) : acc[rr];
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&c.sh->empty[slot]));
    advance(c, A.ns);
    const float t = butterfly<RS>(acc, lane);
    const int rr = RS == 1 ? 0 : (lane >> (5 - (RS == 2 ? 1 : RS == 4 ? 2 : 3)));
    const int lrow = s * RS + rr - (s / spb) * kRB;
    if ((lane & ((32 / RS) - 1)) == 0 && rr < rows_s) c.s_part[warp * kRB + lrow] = t;

    if ((s + 1) % spb == 0 || s == nst - 1) {
      named_bar(1, NWC * 32);
      if (s == nst - 1) ctmark(A, c.epoch, 5);
      const int b0 = r0 + (s / spb) * kRB;
      const int bn = min(kRB, r1 - b0);
      if (EPI == EPI_QKV || EPI == EPI_SWIGLU) {
        for (int pi = tid; pi < (bn >> 1); pi += NWC * 32) {
          const int lr = pi * 2, r = b0 + lr;
          float v0 = 0.f, v1 = 0.f;
          for (int ww = 0; ww < nwa; ++ww) {
            v0 += c.s_part[ww * kRB + lr];
            v1 += c.s_part[ww * kRB + lr + 1];
          }
          if (EPI == EPI_SWIGLU) {
            e.y[r >> 1] = silu(v0) * v1;
            continue;
          }
          const int hd = A.hd;
          if (r < A.q_rows + A.kv_rows) {
            if (c.pos < 0 || c.pos >= A.rope_len) {
              atomicOr(&A.sp->status, kBadPos);
              continue;
            }
            const int blk = s / spb;
            const float2 cs = (pi == tid && blk < 2) ? (blk == 0 ? cs_pre[0] : cs_pre[1])
                                                     : A.rope_cs[(size_t)c.pos * (hd >> 1) + ((r % hd) >> 1)];
            const float t0 = v0 * cs.x - v1 * cs.y;
            v1 = v0 * cs.y + v1 * cs.x;
            v0 = t0;
          }
          if (r < A.q_rows) {
            e.y[r] = v0;
            e.y[r + 1] = v1;
          } else {
            const bool is_k = r < A.q_rows + A.kv_rows;
            const int rk = r - A.q_rows - (is_k ? 0 : A.kv_rows);
            const int kvh = rk / hd, dim = rk % hd;
            const int pt = A.page_tokens;
            const int page = c.pos_page;
            if (page < 0) {
              atomicOr(&A.sp->status, kBadPage);
              continue;
            }
            const size_t off = (((size_t)page * A.n_kv + kvh) * pt + (c.pos % pt)) * hd + dim;
            *reinterpret_cast<__half2*>((is_k ? e.k_pool : e.v_pool) + off) = __floats2half2_rn(v0, v1);
          }
        }
      } else {
        for (int lr = tid; lr < bn; lr += NWC * 32) {
          float v = 0.f;
          for (int ww = 0; ww < nwa; ++ww) v += c.s_part[ww * kRB + lr];
          if (EPI == EPI_RESID) {
            const int blk = s / spb;
            const float old = (lr == tid && blk < 2) ? (blk == 0 ? res_pre[0] : res_pre[1]) : __ldcg(e.y + b0 + lr);
            e.y[b0 + lr] = old + v;
            if (e.cap) e.cap[b0 + lr] = old + v;
          } else {
            e.y[b0 + lr] = v;
          }
        }
      }
      named_bar(1, NWC * 32);
    }
  }
  ctmark(A, c.epoch, 6);
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One CTA's attention task: split sp of KV head kvh, tiles tb .. te-1, two
// consecutive 32-token tiles per ring stage.  The eight consumer warps are
// (stage parity) x (tile of the stage) x (head group): warp w works on the
// stages j with j % 2 == w >> 2, on tile (w >> 1) & 1 of each, for the HPW
// query heads of group w & 1.  Position pos (written by this step's QKV
// phase) is copied from global into its tile before scoring.  The four
// warps of a head group merge in shared memory into one (m, l, o) partial
// per CTA; the last CTA of a KV head merges the S partials in split order
// with all loads in flight.
template <int HD, int G>
__device__ void consume_attention(Ctx& c, const __half* k_pool, const __half* v_pool) {
  static_assert(G >= 2 && NWC == 8, "two head groups over eight warps");
  constexpr int HG = 2;               // head groups
  constexpr int HPW = G / HG;         // heads per warp
  constexpr int WPG = NWC / HG;       // warps per head group
  constexpr int DPL = HD / 32, W2 = HD / 2;
  const StepArgs& A = *c.A;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hg = warp & 1, tis = (warp >> 1) & 1, par = warp >> 2;
  const int n = c.pos + 1;
  int kvh, tb, te;
  attn_task(A, n, kvh, tb, te);
  const bool has_task = (int)blockIdx.x < A.n_kv * A.S;
  const int sp = blockIdx.x % A.S;
  const float scale = 1.0f / sqrtf((float)HD);
  // the tile holding position pos (written by this step's QKV phase, so not
  // in the ring): its K and V rows are loaded here, beside q, rather than
  // after the stage arrives, which keeps that L2 round trip off the
  // critical path of the CTA that holds the newest tile
  const int pos_tile = c.pos / kTile;
  const bool has_pos = has_task && pos_tile >= tb && pos_tile < te && c.pos_page >= 0;
  if (has_task) {
    const float* qrow = A.q + (size_t)kvh * G * HD;
    for (int i = tid; i < G * HD; i += NWC * 32) c.s_q[i] = __ldcg(qrow + i) * scale;
    if (has_pos) {
      const size_t off = (((size_t)c.pos_page * A.n_kv + kvh) * A.page_tokens + (c.pos % A.page_tokens)) * HD;
      for (int i = tid; i < HD / 2; i += NWC * 32) {
        reinterpret_cast<__half2*>(c.s_kvpos)[i] = __ldcg(reinterpret_cast<const __half2*>(k_pool + off) + i);
        reinterpret_cast<__half2*>(c.s_kvpos + HD)[i] = __ldcg(reinterpret_cast<const __half2*>(v_pool + off) + i);
      }
    }
  }
  named_bar(1, NWC * 32);
  ctmark(A, c.epoch, 4);
  float m_run[HPW], l_run[HPW], o[HPW][DPL];
#pragma unroll
  for (int h = 0; h < HPW; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  }
  const float2* q2 = reinterpret_cast<const float2*>(c.s_q) + (size_t)hg * HPW * W2;
  const int nst = max(0, (te - tb + 1) / 2);
  for (int j = 0; j < nst; ++j) {
    const int slot = c.slot;
    const int t = tb + 2 * j + tis;
    if ((j & 1) == par && t < te) {
      const int nt = min(kTile, n - t * kTile);
      const bool ok = wait_bar(A, smem_u32(&c.sh->full[slot]), c.par, 20);
      if (j == 0) ctmark(A, c.epoch, 7);
      __half* kt = reinterpret_cast<__half*>(c.ring + (size_t)slot * A.stage_bytes) + 2 * tis * kTile * HD;
      __half* vt = kt + kTile * HD;
      const int jp = c.pos - t * kTile;  // the new position inside this tile, if any
      if (has_pos && t == pos_tile) {
        // the two head-group warps of this tile write the same bytes
        for (int i = lane; i < HD / 2; i += 32) {
          reinterpret_cast<__half2*>(kt + jp * HD)[i] = reinterpret_cast<const __half2*>(c.s_kvpos)[i];
          reinterpret_cast<__half2*>(vt + jp * HD)[i] = reinterpret_cast<const __half2*>(c.s_kvpos + HD)[i];
        }
        __syncwarp();
      }
      if (ok) {
        float sc[HPW];
        {
          // two accumulator chains per head halve the dependent FMA chain
          float2 acc[HPW][2];
#pragma unroll
          for (int h = 0; h < HPW; ++h) acc[h][0] = acc[h][1] = make_float2(0.f, 0.f);
          const __half2* krow = reinterpret_cast<const __half2*>(kt + lane * HD);
#pragma unroll 8
          for (int w2 = 0; w2 < W2; ++w2) {
            const int wi = (w2 + lane) & (W2 - 1);
            const float2 kf = __half22float2(krow[wi]);
#pragma unroll
            for (int h = 0; h < HPW; ++h) acc[h][w2 & 1] = __ffma2_rn(kf, q2[h * W2 + wi], acc[h][w2 & 1]);
          }
#pragma unroll
          for (int h = 0; h < HPW; ++h) {
            const float2 a = __fadd2_rn(acc[h][0], acc[h][1]);
            sc[h] = lane < nt ? a.x + a.y : -INFINITY;
          }
        }
        float p[HPW];
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const float m_new = fmaxf(m_run[h], warp_max_f(sc[h]));
          p[h] = lane < nt ? expf(sc[h] - m_new) : 0.f;
          const float al = expf(m_run[h] - m_new);
          l_run[h] = l_run[h] * al + warp_sum(p[h]);
          m_run[h] = m_new;
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[h][e] *= al;
        }
        // o += P V over the tile's tokens, fully unrolled and branch-free so
        // the V loads and the p broadcasts of all 32 tokens are in flight
        // together; rows past nt hold stale bytes and are zeroed (their p
        // is 0 too)
        const __half* vl = vt + lane * DPL;
#pragma unroll
        for (int jj = 0; jj < kTile; ++jj) {
          float vf[DPL];
          if (DPL == 4) {
            uint2 raw = *reinterpret_cast<const uint2*>(vl + jj * HD);
            if (jj >= nt) raw = make_uint2(0u, 0u);
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            vf[0] = v01.x;
            vf[1] = v01.y;
            vf[2 % DPL] = v23.x;
            vf[3 % DPL] = v23.y;
          } else {
#pragma unroll
            for (int e = 0; e < DPL; ++e) vf[e] = jj < nt ? __half2float(vl[jj * HD + e]) : 0.f;
          }
#pragma unroll
          for (int h = 0; h < HPW; ++h) {
            const float pj = __shfl_sync(0xffffffffu, p[h], jj);
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pj, vf[e], o[h][e]);
          }
        }
      }
      // the generic writes of the new position's row into the slot must be
      // ordered before the next bulk copy into it (a slot that was only read
      // needs no proxy fence: the empty-barrier arrival orders the reads)
      if (has_pos && t == pos_tile) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(smem_u32(&c.sh->empty[slot]));
    advance(c, A.ns);
  }
  // merge the TS warps of each head group
  ctmark(A, c.epoch, 5);
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      c.s_wm[warp * HPW + h] = m_run[h];
      c.s_wl[warp * HPW + h] = l_run[h];
    }
  }
#pragma unroll
  for (int h = 0; h < HPW; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) c.s_wo[(warp * HPW + h) * HD + lane * DPL + e] = o[h][e];
  named_bar(1, NWC * 32);
  if (has_task) {
    const size_t slot = (size_t)kvh * A.S + sp;
    for (int idx = tid; idx < G * HD; idx += NWC * 32) {
      const int h = idx / HD, hh = h % HPW, g0 = h / HPW;  // warps g0, g0 + 2, g0 + 4, g0 + 6 hold head h
      float M = -INFINITY;
#pragma unroll
      for (int t = 0; t < WPG; ++t) M = fmaxf(M, c.s_wm[(g0 + HG * t) * HPW + hh]);
      float acc = 0.f, L = 0.f;
#pragma unroll
      for (int t = 0; t < WPG; ++t) {
        const int wi = (g0 + HG * t) * HPW + hh;
        const float ew = c.s_wl[wi] > 0.f ? expf(c.s_wm[wi] - M) : 0.f;
        acc = fmaf(ew, c.s_wo[wi * HD + (idx % HD)], acc);
        L = fmaf(ew, c.s_wl[wi], L);
      }
      A.part_o[slot * G * HD + idx] = acc;
      if ((idx % HD) == 0) reinterpret_cast<float2*>(A.part_ml)[slot * G + h] = make_float2(M, L);
    }
  }
  named_bar(1, NWC * 32);
  // thread 0 publishes the CTA's partials (release, after the CTA barrier)
  // and, on the last arrival, acquires everyone else's
  if (tid == 0) {
    int prev = 0;
    if (has_task)
      asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(A.att_counters + kvh) : "memory");
    c.sh->last = has_task && prev == A.S - 1;
  }
  named_bar(1, NWC * 32);
  if (c.sh->last) {
    // merge the S splits of this KV head in split order: every thread's
    // partial loads go out first, one warp per head turns the (m, l) pairs
    // into split weights exp(m_s - M) / sum_s l_s exp(m_s - M), then each
    // output is the weighted sum of its S partials
    constexpr int kOut = (G * HD + NWC * 32 - 1) / (NWC * 32);  // outputs per thread
    constexpr int kMB = kOut <= 2 ? 20 : 1;                      // splits loaded up front
    const size_t slot0 = (size_t)kvh * A.S;
    const float2* ml = reinterpret_cast<const float2*>(A.part_ml);
    float* s_w = c.s_wo;  // [G][S] (G * S <= NWC * G * HD)
    const bool one_round = A.S <= kMB;
    float pv[kOut][kMB];
#pragma unroll
    for (int oi = 0; oi < kOut; ++oi) {
      const int idx = tid + oi * NWC * 32;
#pragma unroll
      for (int k = 0; k < kMB; ++k)
        pv[oi][k] = (one_round && k < A.S && idx < G * HD) ? __ldcg(A.part_o + (slot0 + k) * G * HD + idx) : 0.f;
    }
    for (int h = warp; h < G; h += NWC) {
      // each lane holds up to kMl splits' (m, l) pairs: one round of loads
      constexpr int kMl = 4;
      float2 v[kMl];
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kMl; ++k) {
        const int s2 = lane + 32 * k;
        v[k] = s2 < A.S ? __ldcg(&ml[(slot0 + s2) * G + h]) : make_float2(-INFINITY, 0.f);
        M = fmaxf(M, v[k].x);
      }
      M = warp_max_f(M);
      float den = 0.f, ew[kMl];
#pragma unroll
      for (int k = 0; k < kMl; ++k) {
        ew[k] = v[k].y > 0.f ? expf(v[k].x - M) : 0.f;  // empty split: weight 0
        den = fmaf(v[k].y, ew[k], den);
      }
      den = warp_sum(den);
      const float inv = 1.0f / den;
#pragma unroll
      for (int k = 0; k < kMl; ++k)
        if (lane + 32 * k < A.S) s_w[h * A.S + lane + 32 * k] = ew[k] * inv;
    }
    named_bar(1, NWC * 32);
#pragma unroll
    for (int oi = 0; oi < kOut; ++oi) {
      const int idx = tid + oi * NWC * 32;
      if (idx >= G * HD) continue;
      const float* wv = s_w + (idx / HD) * A.S;
      float acc = 0.f;
      if (one_round) {
#pragma unroll
        for (int k = 0; k < kMB; ++k)
          if (k < A.S) acc = fmaf(wv[k], pv[oi][k], acc);
      } else {
        const float* po = A.part_o + slot0 * G * HD + idx;
#pragma unroll 8
        for (int s2 = 0; s2 < A.S; ++s2) acc = fmaf(wv[s2], __ldcg(po + (size_t)s2 * G * HD), acc);
      }
      A.o[(size_t)kvh * G * HD + idx] = acc;
    }
    if (tid == 0) A.att_counters[kvh] = 0;
  }
  ctmark(A, c.epoch, 6);
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// At most 168 registers a thread: the 10 warps spread 3-3-2-2 over the
// SM's four schedulers, and three warps x 32 threads x 168 registers fill
// one scheduler's 16K-entry register file (at 200 the CTA does not launch).
template <int WT, int HD, int G, int RSA, int MCA, int RSB, int MCB>
__global__ void __maxnreg__(168) step_kernel(const StepArgs A) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ctx c;
  c.A = &A;
  c.sh = reinterpret_cast<Sh*>(smem);
  size_t off = (sizeof(Sh) + 127) & ~(size_t)127;
  c.s_part = reinterpret_cast<float*>(smem + off);
  off += NWC * kRB * 4;
  c.s_q = reinterpret_cast<float*>(smem + off);
  off += G * HD * 4;
  c.s_wm = reinterpret_cast<float*>(smem + off);
  off += NWC * G * 4;
  c.s_wl = reinterpret_cast<float*>(smem + off);
  off += NWC * G * 4;
  c.s_wo = reinterpret_cast<float*>(smem + off);
  off += NWC * G * HD * 4;
  c.s_kvpos = reinterpret_cast<__half*>(smem + off);
  off += 2 * HD * 2;
  c.ring = smem + ((off + 127) & ~(size_t)127);
  c.sidx = 0;
  c.slot = 0;
  c.par = 0;
  c.epoch = 0;
  c.pos = A.sp->pos[0];
  c.seq = A.sp->seq[0];
  {
    const int lp = c.pos >= 0 ? c.pos / A.page_tokens : -1;
    c.pos_page = (lp >= 0 && lp < A.max_pages) ? A.page_table[(size_t)c.seq * A.max_pages + lp] : -1;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < A.ns; ++s) {
      mbar_init(smem_u32(&c.sh->full[s]), 1);
      mbar_init(smem_u32(&c.sh->empty[s]), NWC);
    }
    c.sh->epoch_pub = 0;
    mbar_fence_init();
    if (A.trace && blockIdx.x == 0) A.trace[0] = global_ns();
  }
  for (int l = tid; l < kMaxSkipLayers; l += blockDim.x) c.sh->skip[l] = (A.skip && l < A.n_layers) ? A.skip[l] : 0;
  __syncthreads();

  if (warp == NWC) {
    // ---------------- producer: every phase's stages, in consumer order
    if (lane == 0) produce<WT, HD, RSA, RSB>(c);
  } else if (warp == NWC + 1) {
    // ---------------- L2 hints for the gate/up rows
    if (A.pf_rows) hint_lanes<WT>(c);
  } else {
    // ---------------- consumers
    // embedding row -> x (rows split like the residual epilogues)
    {
      int tok = A.sp->token[0];
      if (tok < 0 || tok >= A.vocab) {
        if (tid == 0) atomicOr(&A.sp->status, kBadToken);
        tok = 0;
      }
      int r0, r1;
      row_split(A.H, 1, r0, r1);
      const MatDev& E = A.emb;
      for (int col = r0 + tid; col < r1; col += NWC * 32) {
        const int blk = col >> 5, e = col & 31;
        const float d = __half2float(E.d[(size_t)tok * E.ds + blk]);
        float q;
        if (WT == 8) {
          q = mag_byte((uint32_t)E.qs[(size_t)tok * E.nb * 32 + col], 0) - 8388736.0f;  // stored q + 128
        } else {
          const uint8_t byte = E.qs[((size_t)tok * E.nb + blk) * 16 + (e & 15)];
          q = mag_byte(e < 16 ? (byte & 15u) : (byte >> 4), 0) - 8388616.0f;
        }
        A.x[col] = d * q;
      }
    }
    grid_sync(c);
    for (int l = 0; l < A.n_layers; ++l) {
      if (c.sh->skip[l]) {  // the residual passes through; every CTA reads the same flags
        if (A.capture) {
          // this CTA's rows of x, which no CTA writes before the next layer's
          // O phase (two grid barriers later)
          int r0, r1;
          row_split(A.H, 1, r0, r1);
          for (int r = r0 + tid; r < r1; r += NWC * 32) A.capture[(size_t)l * A.H + r] = __ldcg(A.x + r);
        }
        continue;
      }
      const StepLayer& L = A.layers[l];
      EpiArgs e{};
      e.y = A.q;
      e.k_pool = L.k_pool;
      e.v_pool = L.v_pool;
      consume_gemv<WT, PRO_RMSNORM, EPI_QKV, RSA, MCA>(c, L.qkv, 2, A.x, L.attn_norm, e);
      grid_sync(c);
      consume_attention<HD, G>(c, L.k_pool, L.v_pool);
      grid_sync(c);
      e.y = A.x;
      consume_gemv<WT, PRO_COPY, EPI_RESID, RSA, MCA>(c, L.o, 1, A.o, nullptr, e);
      grid_sync(c);
      e.y = A.h;
      consume_gemv<WT, PRO_RMSNORM, EPI_SWIGLU, RSA, MCA>(c, L.gu, 2, A.x, L.ffn_norm, e);
      grid_sync(c);
      e.y = A.x;
      e.cap = A.capture ? A.capture + (size_t)l * A.H : nullptr;
      consume_gemv<WT, PRO_COPY, EPI_RESID, RSB, MCB>(c, L.down, 1, A.h, nullptr, e);
      grid_sync(c);
    }
    EpiArgs e{};
    e.y = A.logits;
    if (A.head_rows) consume_gemv<WT, PRO_RMSNORM, EPI_STORE, RSA, MCA>(c, A.head, 1, A.x, A.out_norm, e);
    if (A.head_rows && A.greedy) {
      grid_sync(c);
      // greedy pick: each CTA reduces a slice of the logits, CTA 0 the slices
      int r0, r1;
      row_split(A.vocab, 1, r0, r1);
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int i = r0 + tid; i < r1; i += NWC * 32) {
        const float v = __ldcg(A.logits + i);
        if (better(v, i, best, bi)) {
          best = v;
          bi = i;
        }
      }
      for (int o2 = 16; o2 > 0; o2 >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o2);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o2);
        if (better(ov, oi, best, bi)) {
          best = ov;
          bi = oi;
        }
      }
      if (lane == 0) {
        c.s_wm[warp] = best;
        reinterpret_cast<int*>(c.s_wl)[warp] = bi;
      }
      named_bar(1, NWC * 32);
      if (tid == 0) {
        for (int w = 1; w < NWC; ++w)
          if (better(c.s_wm[w], reinterpret_cast<int*>(c.s_wl)[w], best, bi)) {
            best = c.s_wm[w];
            bi = reinterpret_cast<int*>(c.s_wl)[w];
          }
        A.am_part[blockIdx.x] = make_int2(__float_as_int(best), bi);
      }
      grid_sync(c);
      if (blockIdx.x == 0 && tid == 0) {
        best = -INFINITY;
        bi = 0x7fffffff;
        for (int b = 0; b < (int)gridDim.x; ++b) {
          const int2 p2 = __ldcg(&A.am_part[b]);
          if (better(__int_as_float(p2.x), p2.y, best, bi)) {
            best = __int_as_float(p2.x);
            bi = p2.y;
          }
        }
        const int tok = bi == 0x7fffffff ? 0 : bi;
        const int step = A.sp->step;
        if (A.tokens_out) A.tokens_out[step] = tok;
        A.sp->token[0] = tok;
        A.sp->pos[0] = c.pos + 1;
        A.sp->step = step + 1;
      }
    }
    if (A.trace && blockIdx.x == 0 && tid == 0) A.trace[c.epoch + 1] = global_ns();
  }
  __syncthreads();
}

template <int WT, int HD, int G, int RSA, int MCA, int RSB, int MCB>
const void* step_fn() {
  return reinterpret_cast<const void*>(&step_kernel<WT, HD, G, RSA, MCA, RSB, MCB>);
}

struct Variant {
  int wt, hd, g, rsa, mca, rsb, mcb;
  const void* (*fn)();
};

// The shapes with a persistent-kernel instantiation (others use the
// multi-kernel step).
const Variant kVariants[] = {
    {8, 128, 4, 8, 1, 2, 4, &step_fn<8, 128, 4, 8, 1, 2, 4>},  // 8B-shape Q8_0
    {4, 128, 4, 8, 1, 4, 2, &step_fn<4, 128, 4, 8, 1, 4, 2>},  // 8B-shape Q4_0
    {8, 64, 4, 8, 1, 4, 2, &step_fn<8, 64, 4, 8, 1, 4, 2>},    // 1B-shape Q8_0
    {8, 64, 2, 8, 1, 8, 1, &step_fn<8, 64, 2, 8, 1, 8, 1>},    // tiny Q8_0
    {4, 64, 2, 8, 1, 8, 1, &step_fn<4, 64, 2, 8, 1, 8, 1>},    // tiny Q4_0
    {4, 128, 8, 8, 1, 2, 4, &step_fn<4, 128, 8, 8, 1, 2, 4>},  // 70B-shape Q4_0
};

// rows per ring stage: as many whole rows as fit 32 KB of codes, at most 8
int pow2_rows(int row_bytes) {
  int rs = 1;
  while (rs < 8 && (rs * 2) * row_bytes <= 32768) rs *= 2;
  return rs;
}

}  // namespace

StepPlan step_plan(int wtype, int H, int q_rows, int F, int n_heads, int n_kv, int hd, int num_sms) {
  StepPlan p{};
  p.fn = nullptr;
  p.why = "the O projection's input width differs from the hidden size";
  if (q_rows != H) return p;  // O projection must share the hidden-size geometry
  p.why = "hidden or FFN size not a multiple of 4";
  if (H % 4 || F % 4) return p;  // activation slices are read as whole float4
  const int G = n_heads / n_kv;
  const int nb_h = (H + 31) / 32, nb_f = (F + 31) / 32;
  const int rb_h = wtype == 8 ? nb_h * 32 : nb_h * 16, rb_f = wtype == 8 ? nb_f * 32 : nb_f * 16;
  const int CH = wtype == 8 ? 512 : 1024;
  const int rsa = pow2_rows(rb_h), rsb = pow2_rows(rb_f);
  const int mca = ((nb_h * 32 + CH - 1) / CH + NWC - 1) / NWC;
  const int mcb = ((nb_f * 32 + CH - 1) / CH + NWC - 1) / NWC;
  for (const Variant& v : kVariants)
    if (v.wt == wtype && v.hd == hd && v.g == G && v.rsa == rsa && v.mca == mca && v.rsb == rsb && v.mcb == mcb) {
      p.fn = v.fn();
      break;
    }
  p.why = "no instantiation for this shape";
  if (!p.fn) return p;
  const int ds_h = (nb_h + 7) & ~7, ds_f = (nb_f + 7) & ~7;
  size_t stage = std::max((size_t)rsa * (rb_h + ds_h * 2), (size_t)rsb * (rb_f + ds_f * 2));
  stage = std::max(stage, (size_t)4 * kTile * hd * 2);  // two K/V tiles
  stage = (stage + 127) & ~(size_t)127;
  size_t head = ((sizeof(Sh) + 127) & ~(size_t)127) + NWC * kRB * 4 + G * hd * 4 + 2 * NWC * G * 4 + NWC * G * hd * 4 +
                2 * hd * 2;
  head = (head + 127) & ~(size_t)127;
  const size_t budget = 220 * 1024;
  int ns = (int)((budget - head) / stage);
  ns = std::min(ns, kMaxStages);
  if (const char* e = getenv("DLS_STEP_STAGES")) ns = std::min(ns, std::max(2, atoi(e)));  // tuning knob
  if (ns < 2) {
    p.why = "fewer than two ring stages fit in shared memory";
    p.fn = nullptr;
    return p;
  }
  p.ns = ns;
  p.stage_bytes = (uint32_t)stage;
  p.smem = (int)(head + ns * stage);
  p.grid = num_sms;
  p.threads = NTHR;
  p.why = nullptr;
  p.splits = std::min(num_sms / n_kv, 128);  // the merge holds up to 4 x 32 splits' (m, l) pairs per warp
  if (p.splits < 1) {
    p.why = "more KV heads than SMs";
    p.fn = nullptr;
    return p;
  }
  if (cudaFuncSetAttribute(p.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem) != cudaSuccess) {
    cudaGetLastError();
    p.why = "the shared-memory size was refused";
    p.fn = nullptr;
    return p;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p.fn, p.threads, p.smem) != cudaSuccess || occ < 1) {
    cudaGetLastError();
    p.why = "one CTA per SM does not fit (registers or shared memory)";
    p.fn = nullptr;
  }
  return p;
}

cudaError_t launch_step(const StepPlan& p, const StepArgs& a, cudaStream_t s) {
  if (!p.fn || a.n_layers > kMaxSkipLayers) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the grid barriers rely on it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<StepArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, p.fn, args);
}

}  // namespace dls
