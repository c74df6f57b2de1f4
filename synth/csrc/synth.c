/*
 * Seeded synthetic inputs for the Llama-architecture decode step: normal
 * weights, GGUF-style Q8_0 / Q4_0 block quantisation of them, and uniform
 * token ids.  This file is an INPUT GENERATOR shared by the CUDA library's
 * tests/benchmarks and by the fp64 oracle; it contains none of the decode
 * step's arithmetic (no dequantisation, no norm, no attention).
 *
 * Random numbers: one counter-based generator, SplitMix64 (Steele, Lea and
 * Flood, "Fast Splittable Pseudorandom Number Generators", OOPSLA 2014).  The
 * i-th draw of stream `key` is mix64(key + (i + 1) * GOLDEN): every element
 * is a pure function of (key, index), so the output does not depend on the
 * thread count or the order of evaluation.
 *
 * Normals: Box-Muller on two consecutive uniforms, element 2p taking the
 * cosine branch and element 2p+1 the sine branch of pair p.
 *
 * Block formats (as the workloads define them):
 *   Q8_0: 34-byte block = fp16 scale d, then 32 int8 q;      weight = d*q
 *   Q4_0: 18-byte block = fp16 scale d, then 16 bytes; byte j holds element j
 *         in its low nibble and element j+16 in its high nibble; weight = d*(q-8)
 * A matrix [rows x cols] is stored row-major, ceil(cols/32) blocks per row;
 * the columns past `cols` in the last block are zero weights.
 *
 * Quantiser (our reading; the workloads only say "drawn then quantised"):
 *   Q8_0: d = amax/127 (0 when amax = 0); q = round_half_away(x/d), clamped
 *         to [-127, 127]; d stored as fp16.
 *   Q4_0: m = the element of largest magnitude (first one on ties, sign kept);
 *         d = m / -8; q = clamp(round_half_away(x/d) + 8, 0, 15); fp16 d.
 *
 * Portability: built with -ffp-contract=off and no target-specific flags;
 * fp64 -> fp16 conversion is written out here (round to nearest even).  The
 * libm functions (log, sqrt, cos, sin) may differ in the last bit between C
 * libraries, so bytes are compared only between two consumers on one machine.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* standard normals for pair p of stream `key`: elements 2p (cosine branch)
   and 2p+1 (sine branch) */
static inline void normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
  const double two53 = 9007199254740992.0;
  const double u1 = ((double)(draw(key, 2 * p) >> 11) + 1.0) / two53; /* (0, 1] */
  const double u2 = (double)(draw(key, 2 * p + 1) >> 11) / two53;     /* [0, 1) */
  const double r = sqrt(-2.0 * log(u1));
  const double a = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(a);
  *z1 = r * sin(a);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

/* fp64 -> IEEE binary16 bits, round to nearest, ties to even. */
static uint16_t f64_to_f16_bits(double v) {
  uint64_t b;
  memcpy(&b, &v, 8);
  const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  const int exp = (int)((b >> 52) & 0x7FF);
  uint64_t man = b & 0xFFFFFFFFFFFFFULL;
  if (exp == 0x7FF) return sign | 0x7C00u | (man ? 0x200u : 0u);
  if (exp == 0 && man == 0) return sign;
  /* value = 1.man * 2^(exp-1023) (doubles below 2^-1022 round to 0 in fp16 anyway) */
  const int e = exp - 1023;
  if (e > 15) return sign | 0x7C00u; /* overflow -> inf */
  /* significand with implicit bit, 53 bits */
  uint64_t sig = man | (1ULL << 52);
  int shift; /* number of low bits to drop */
  uint16_t hexp;
  if (e >= -14) { /* normal fp16 */
    shift = 52 - 10;
    hexp = (uint16_t)(e + 15);
  } else { /* subnormal fp16: value = m * 2^-24 */
    shift = 52 - 10 + (-14 - e);
    hexp = 0;
    if (shift > 63) return sign;
  }
  uint64_t keep = sig >> shift;
  const uint64_t rem = sig & ((1ULL << shift) - 1);
  const uint64_t half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (keep & 1))) keep++;
  if (hexp == 0) {
    /* subnormal; rounding may carry into the smallest normal (bit 10) */
    return sign | (uint16_t)keep;
  }
  /* normal: keep has the implicit bit at bit 10; carry may bump exponent */
  if (keep >> 11) {
    keep >>= 1;
    hexp++;
    if (hexp >= 31) return sign | 0x7C00u;
  }
  return sign | (uint16_t)(hexp << 10) | (uint16_t)(keep & 0x3FF);
}

static double f16_bits_to_f64(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 1024), e - 25);
  return s ? -v : v;
}

static inline double round_half_away(double v) { return v < 0 ? -floor(-v + 0.5) : floor(v + 0.5); }

static void quant_block_q8_0(const double* x, uint8_t* out) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(x[i]));
  const double d = amax / 127.0;
  const uint16_t dh = f64_to_f16_bits(d);
  memcpy(out, &dh, 2); /* little-endian on every target we build for */
  for (int i = 0; i < 32; ++i) {
    double q = d > 0.0 ? round_half_away(x[i] / d) : 0.0;
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    out[2 + i] = (uint8_t)(int8_t)(int)q;
  }
}

static void quant_block_q4_0(const double* x, uint8_t* out) {
  double m = 0.0, amax = 0.0;
  for (int i = 0; i < 32; ++i)
    if (fabs(x[i]) > amax) { amax = fabs(x[i]); m = x[i]; }
  const double d = m / -8.0;
  const uint16_t dh = f64_to_f16_bits(d);
  memcpy(out, &dh, 2);
  uint8_t q[32];
  for (int i = 0; i < 32; ++i) {
    double v = d != 0.0 ? round_half_away(x[i] / d) + 8.0 : 8.0;
    if (v < 0.0) v = 0.0;
    if (v > 15.0) v = 15.0;
    q[i] = (uint8_t)v;
  }
  for (int j = 0; j < 16; ++j) out[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/*
 * K-quant super-blocks (256 weights; the GGUF layouts the engine page's Q4_K_M
 * and Q6_K files use), for drawing synthetic K-quant matrices.  Quantiser
 * (our reading; any valid blocks serve as inputs, since both consumers read
 * the bytes): per 32-weight sub-block (Q4_K, Q5_K) the range [min(lo, 0),
 * hi] is split into 15 (31) steps, the step sizes and the offsets -min are
 * coded as 6-bit multiples of the super-block's d and dmin (their maxima over
 * 63, stored fp16); per 16-weight group (Q6_K) the step is amax / 31, coded
 * as an int8 multiple of d (the largest step over 127, stored fp16).  Codes
 * are round-half-away of (x + offset) / step, clamped to the code range.
 *   Q4_K 144 bytes: d, dmin, 12 scale bytes, 128 bytes of nibbles (byte
 *     32g + l: weight 64g + l low, 64g + 32 + l high).
 *   Q5_K 176 bytes: d, dmin, 12 scale bytes, 32 bytes qh (bit 2g / 2g + 1 of
 *     qh[l]: fifth bit of weight 64g + l / 64g + 32 + l), 128 bytes of nibbles.
 *   Q6_K 210 bytes: 128 bytes ql, 64 bytes qh, 16 int8 scales, fp16 d.
 */
static void pack_scales_k(const int* sc, const int* m, uint8_t* b) {
  for (int s = 0; s < 4; ++s) {
    b[s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
    b[s + 4] = (uint8_t)((m[s] & 63) | ((m[s + 4] >> 4) << 6));
    b[s + 8] = (uint8_t)((sc[s + 4] & 15) | ((m[s + 4] & 15) << 4));
  }
}

static void quant_super_k45(const double* x, int qmax, uint8_t* out) {
  double step[8], off[8], dmax = 0.0, omax = 0.0;
  for (int s = 0; s < 8; ++s) {
    double lo = 0.0, hi = -INFINITY;
    for (int i = 0; i < 32; ++i) {
      lo = fmin(lo, x[32 * s + i]);
      hi = fmax(hi, x[32 * s + i]);
    }
    step[s] = (hi - lo) / qmax;
    off[s] = -lo;
    dmax = fmax(dmax, step[s]);
    omax = fmax(omax, off[s]);
  }
  const uint16_t dh = f64_to_f16_bits(dmax / 63.0), mh = f64_to_f16_bits(omax / 63.0);
  const double d = f16_bits_to_f64(dh), dmin = f16_bits_to_f64(mh);
  int sc[8], m[8];
  for (int s = 0; s < 8; ++s) {
    double a = d > 0.0 ? round_half_away(step[s] / d) : 0.0;
    double b = dmin > 0.0 ? round_half_away(off[s] / dmin) : 0.0;
    sc[s] = (int)fmin(fmax(a, 0.0), 63.0);
    m[s] = (int)fmin(fmax(b, 0.0), 63.0);
  }
  memcpy(out, &dh, 2);
  memcpy(out + 2, &mh, 2);
  pack_scales_k(sc, m, out + 4);
  uint8_t* qh = qmax == 31 ? out + 16 : NULL;
  uint8_t* qs = out + (qmax == 31 ? 48 : 16);
  if (qh) memset(qh, 0, 32);
  for (int i = 0; i < 256; ++i) {
    const int s = i / 32;
    const double w = d * sc[s];
    double q = w > 0.0 ? round_half_away((x[i] + dmin * m[s]) / w) : 0.0;
    q = fmin(fmax(q, 0.0), (double)qmax);
    const int qi = (int)q, g = i / 64, l = i % 32, high = (i / 32) & 1;
    uint8_t* byte = &qs[32 * g + l];
    if (high) *byte = (uint8_t)((*byte & 0x0F) | ((qi & 15) << 4));
    else *byte = (uint8_t)((*byte & 0xF0) | (qi & 15));
    if (qh && (qi >> 4)) qh[l] |= (uint8_t)(1u << (2 * g + high));
  }
}

static void quant_super_q6_k(const double* x, uint8_t* out) {
  double step[16], dmax = 0.0;
  for (int k = 0; k < 16; ++k) {
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) amax = fmax(amax, fabs(x[16 * k + i]));
    step[k] = amax / 31.0;
    dmax = fmax(dmax, step[k]);
  }
  const uint16_t dh = f64_to_f16_bits(dmax / 127.0);
  const double d = f16_bits_to_f64(dh);
  uint8_t* ql = out;
  uint8_t* qh = out + 128;
  int8_t* scales = (int8_t*)(out + 192);
  memset(out, 0, 192);
  for (int k = 0; k < 16; ++k) {
    const double a = d > 0.0 ? round_half_away(step[k] / d) : 0.0;
    scales[k] = (int8_t)(int)fmin(fmax(a, 0.0), 127.0);
  }
  for (int i = 0; i < 256; ++i) {
    const double w = d * scales[i / 16];
    double q = w > 0.0 ? round_half_away(x[i] / w) : 0.0;
    q = fmin(fmax(q, -32.0), 31.0);
    const int code = (int)q + 32, h = i / 128, o = i % 128, g = o / 32, l = o % 32;
    uint8_t* lb = &ql[64 * h + 32 * (g % 2) + l];
    if (g < 2) *lb = (uint8_t)((*lb & 0xF0) | (code & 15));
    else *lb = (uint8_t)((*lb & 0x0F) | ((code & 15) << 4));
    qh[32 * h + l] |= (uint8_t)(((code >> 4) & 3) << (2 * g));
  }
  memcpy(out + 208, &dh, 2);
}

/* ---- exported API ------------------------------------------------------- */

/* n normals * sigma, elements [start, start+n) of stream key */
void synth_normal(uint64_t key, uint64_t start, int64_t n, double sigma, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = sigma * normal_at(key, start + (uint64_t)i);
}

/* uniform token ids in [0, vocab) */
void synth_tokens(uint64_t key, int64_t n, int32_t vocab, int32_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = (int32_t)(((draw(key, (uint64_t)i) >> 32) * (uint64_t)vocab) >> 32);
}

/*
 * Quantised matrix [rows x cols] of sigma*N(0,1): element (r, c) is element
 * r*cols + c of stream key.  wtype 8 = Q8_0, 4 = Q4_0.  `out` holds
 * rows * ceil(cols/32) blocks.  Returns 0, or -1 on a bad wtype.
 */
int synth_quant_matrix(uint64_t key, int64_t rows, int64_t cols, double sigma, int wtype, uint8_t* out) {
  if (wtype != 8 && wtype != 4) return -1;
  const int64_t nb = (cols + 31) / 32;
  const int64_t bsz = wtype == 8 ? 34 : 18;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double x[32];
    for (int64_t b = 0; b < nb; ++b) {
      for (int i = 0; i < 32;) {
        const int64_t c = b * 32 + i;
        const uint64_t idx = (uint64_t)(r * cols + c);
        if (c + 1 < cols && (idx & 1) == 0) { /* both elements of a pair in this row */
          double z0, z1;
          normal_pair(key, idx >> 1, &z0, &z1);
          x[i] = sigma * z0;
          x[i + 1] = sigma * z1;
          i += 2;
        } else {
          x[i] = c < cols ? sigma * normal_at(key, idx) : 0.0;
          i += 1;
        }
      }
      uint8_t* o = out + (r * nb + b) * bsz;
      if (wtype == 8) quant_block_q8_0(x, o);
      else quant_block_q4_0(x, o);
    }
  }
  return 0;
}

/*
 * K-quant matrix [rows x cols] (cols a multiple of 256) of sigma*N(0,1),
 * element (r, c) = element r*cols + c of stream key, as the normals of
 * synth_quant_matrix.  kind 12 = Q4_K (144-byte super-blocks), 13 = Q5_K
 * (176), 14 = Q6_K (210).  Returns 0, or -1 on a bad kind or shape.
 */
int synth_quant_matrix_k(uint64_t key, int64_t rows, int64_t cols, double sigma, int kind, uint8_t* out) {
  if ((kind != 12 && kind != 13 && kind != 14) || cols % 256) return -1;
  const int64_t nsb = cols / 256;
  const int64_t bsz = kind == 12 ? 144 : kind == 13 ? 176 : 210;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double x[256];
    for (int64_t b = 0; b < nsb; ++b) {
      const uint64_t base = (uint64_t)(r * cols + b * 256);  /* even: cols is a multiple of 256 */
      for (int i = 0; i < 256; i += 2) {
        double z0, z1;
        normal_pair(key, (base + (uint64_t)i) >> 1, &z0, &z1);
        x[i] = sigma * z0;
        x[i + 1] = sigma * z1;
      }
      uint8_t* o = out + (r * nsb + b) * bsz;
      if (kind == 14) quant_super_q6_k(x, o);
      else quant_super_k45(x, kind == 12 ? 15 : 31, o);
    }
  }
  return 0;
}

/* Quantise caller-given values (n a multiple of 32) into blocks. */
int synth_quantize(const double* x, int64_t n, int wtype, uint8_t* out) {
  if ((wtype != 8 && wtype != 4) || n % 32) return -1;
  const int64_t bsz = wtype == 8 ? 34 : 18;
  for (int64_t b = 0; b < n / 32; ++b) {
    if (wtype == 8) quant_block_q8_0(x + b * 32, out + b * bsz);
    else quant_block_q4_0(x + b * 32, out + b * bsz);
  }
  return 0;
}

/* fp16 helpers exposed for the generator's own self-test */
uint16_t synth_f64_to_f16(double v) { return f64_to_f16_bits(v); }
double synth_f16_to_f64(uint16_t h) { return f16_bits_to_f64(h); }
