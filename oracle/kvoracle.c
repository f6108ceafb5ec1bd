/*
 * kvoracle.c -- plain, slow, scalar CPU reference of the KV-page codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product library
 * (the CUDA codec) shares no code, header, table or constant generator with it.
 *
 * Build:  gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *             -o liboracle.so kvoracle.c -lm
 * "-ffp-contract=off" matters: every float operation below is one IEEE
 * binary32 operation rounded to nearest-even; no fused multiply-add.
 *
 * Sources (web pages; cited by title and section):
 *   [OKV]  "KV precision and storage encoding" (OrbitKV docs, storage formats),
 *          sections "FP8 and TurboQuant" and "Ownership, storage and GDS".
 *   [ASYM] "Asymmetric KV: methods and results" (knlp), sections
 *          "Precision and scaling reference" and "Actual-worker comparison".
 *   [HIQ]  "Building a quantized HiCache for SGLang", sections "Building the
 *          INT8 codec" and "Why exactly 1,152 bytes?".
 * Readings taken where the pages are silent are marked READING and are listed
 * with their reasons in the design notes of the repository.
 *
 * Everything works on plain arrays with plain loops.  Floating point is FP32
 * where the pages fix FP32 (the FP8 scale rule) or where the codec's stored
 * results depend on FP32 rounding (TurboQuant / uniform codes); the
 * Lloyd-Max codebook is solved in FP64 and rounded once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Identifiers shared with the product only as an interface (same numbers,   */
/* separately written): codec kinds, dtypes, layouts, segment statuses.      */
/* ------------------------------------------------------------------------ */
enum { O_FP16 = 1, O_BF16 = 2 };
enum { O_SEPARATE = 1, O_PACKED = 2 };
enum {
  O_NONE = 0, O_FP8_CAST = 1, O_FP8_FIXED = 2, O_FP8_DYNAMIC = 3,
  O_TQ3 = 4, O_TQ4 = 5, O_UNI3 = 6, O_UNI4 = 7, O_UNI8 = 8, O_INT8 = 9,
  O_TQ2 = 10, O_UNI2 = 11
};
enum {
  S_ENCODED = 1, S_RAW_NONFINITE = 2, S_RAW_RANGE = 3, S_RAW_PROTECTED = 4,
  S_RAW_POLICY = 5, S_RAW_OVERSIZE = 6, S_RAW_NO_SAVING = 7, S_BAD_DESC = 8,
  S_CORRUPT = 9
};

/* ======================================================================== */
/* 1. Number formats, written from their definitions.                       */
/* ======================================================================== */

/* IEEE binary16: 1 sign, 5 exponent bits (bias 15), 10 fraction bits. */
float kvo_f16_to_f32(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0x1f) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -24);            /* subnormal m*2^-24 */
  else v = ldexp((double)(1024 + m), e - 25);           /* (1+m/1024)*2^(e-15) */
  return (float)(s ? -v : v);
}

/* bfloat16 is by definition the upper half of a binary32. */
float kvo_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a finite double to a binary format with `mant` stored fraction bits
 * and minimum normal exponent `emin`, nearest-even (rint in the default
 * rounding mode).  No overflow handling here. */
static double round_to_format(double x, int mant, int emin) {
  if (x == 0.0) return x;
  int e;
  frexp(fabs(x), &e);                  /* |x| = f*2^e, f in [0.5, 1) */
  int ex = e - 1;                      /* floor(log2|x|) */
  if (ex < emin) ex = emin;            /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, ex - mant);
  return copysign(rint(fabs(x) / quantum) * quantum, x);
}

uint16_t kvo_f32_to_f16(float x) {
  uint16_t s = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return s | 0x7e00;
  if (isinf(x)) return s | 0x7c00;
  double a = fabs(round_to_format((double)x, 10, -14));
  if (a > 65504.0) return s | 0x7c00;                   /* rounds past max finite */
  if (a == 0.0) return s;
  int e;
  frexp(a, &e);
  int ex = e - 1;
  if (ex < -14) return s | (uint16_t)(a / ldexp(1.0, -24));           /* subnormal */
  return s | (uint16_t)((ex + 15) << 10) | (uint16_t)(a / ldexp(1.0, ex - 10) - 1024.0);
}

uint16_t kvo_f32_to_bf16(float x) {
  uint16_t s = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return s | 0x7fc0;
  if (isinf(x)) return s | 0x7f80;
  float r = (float)round_to_format((double)x, 7, -126);  /* exact, or inf on overflow */
  uint32_t u;
  memcpy(&u, &r, 4);
  return (uint16_t)(u >> 16);
}

/* E4M3FN: 1 sign, 4 exponent bits (bias 7), 3 fraction bits, no infinities,
 * S.1111.111 is NaN, largest finite 0x7E = 448, subnormals m*2^-9. */
static double e4m3_magnitude(int c) {           /* c in 0..0x7E */
  int e = (c >> 3) & 0xf, m = c & 7;
  if (e == 0) return ldexp((double)m, -9);
  return ldexp(8.0 + m, e - 10);                /* (1+m/8)*2^(e-7) */
}

float kvo_e4m3_to_f32(uint8_t c) {
  if ((c & 0x7f) == 0x7f) return NAN;
  double v = e4m3_magnitude(c & 0x7f);
  return (float)((c & 0x80) ? -v : v);
}

/* Nearest E4M3FN code, ties to the even code (even fraction), sign kept
 * (so -0 and tiny negatives give 0x80).  [OKV "FP8 and TurboQuant"]: round
 * to nearest, ties to even, signed zero and subnormals.  Precondition: q
 * finite with |q| <= 448 (callers clip or reject first). */
uint8_t kvo_f32_to_e4m3(float q) {
  double a = fabs((double)q);
  int best = 0;
  double bestd = a;                              /* distance to code 0 (= 0.0) */
  for (int c = 1; c <= 0x7e; ++c) {
    double d = fabs(a - e4m3_magnitude(c));
    if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
  }
  return (uint8_t)(best | (signbit(q) ? 0x80 : 0));
}

static float src_to_f32(uint16_t h, int dtype) {
  return dtype == O_FP16 ? kvo_f16_to_f32(h) : kvo_bf16_to_f32(h);
}
static uint16_t f32_to_src(float x, int dtype) {
  return dtype == O_FP16 ? kvo_f32_to_f16(x) : kvo_f32_to_bf16(x);
}

/* ======================================================================== */
/* 2. Reductions.  READING: sums use the pairwise (recursive halving) order  */
/* over the element index; max/min need no order.                           */
/* ======================================================================== */
float kvo_pairwise_sum(const float* a, int n) {          /* n a power of two */
  if (n == 1) return a[0];
  float lo = kvo_pairwise_sum(a, n / 2);
  float hi = kvo_pairwise_sum(a + n / 2, n / 2);
  return lo + hi;
}

/* ======================================================================== */
/* 3. FP8 E4M3FN, [ASYM "Precision and scaling reference"]: the absolute      */
/* maximum is clamped at 1e-12 (FP32), multiplied by the FP32-rounded        */
/* reciprocal of 448, operands are divided in FP32, clipped to +-448 and      */
/* rounded to E4M3FN nearest-even.  Dynamic mode: one scale per token/head   */
/* vector.  Fixed mode: one scale per (layer, K/V component) from            */
/* calibration.  Cast mode ([OKV]): scale 1.                                  */
/* ======================================================================== */
float kvo_fp8_scale_from_amax(float amax) {
  const float recip448 = 1.0f / 448.0f;          /* fl32(1/448) */
  float a = amax > 1e-12f ? amax : 1e-12f;
  return a * recip448;
}

float kvo_absmax(const float* x, int n) {
  float m = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > m) m = a;
  }
  return m;
}

void kvo_fp8_encode_vec(const float* x, int D, float s, uint8_t* codes) {
  for (int i = 0; i < D; ++i) {
    float q = x[i] / s;
    if (q > 448.0f) q = 448.0f;
    if (q < -448.0f) q = -448.0f;
    codes[i] = kvo_f32_to_e4m3(q);
  }
}

/* Restore: native operand = code * scale in FP32 ([ASYM]: each layer
 * reconstructs native attention operands from codes and FP32 scales). */
void kvo_fp8_decode_vec(const uint8_t* codes, int D, float s, float* out) {
  for (int i = 0; i < D; ++i) out[i] = kvo_e4m3_to_f32(codes[i]) * s;
}

/* ======================================================================== */
/* 4. TurboQuant K ([OKV "FP8 and TurboQuant"]): normalize the head vector,  */
/* apply deterministic random signs and an orthonormal Walsh-Hadamard        */
/* transform, encode Gaussian Lloyd-Max centroid indices; restore corrects   */
/* the centroid-vector norm, applies the inverse transform and the original  */
/* FP16 norm.                                                                */
/* ======================================================================== */

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): state advances by the golden-gamma constant,
 * output is the state passed through the variant-13 64-bit finalizer.
 * READING: sign i is bit (i mod 64) of output floor(i/64); 1 means negate. */
uint64_t kvo_splitmix64_next(uint64_t* state) {
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void kvo_signs(uint64_t seed, int D, uint8_t* neg) {
  uint64_t st = seed, w = 0;
  for (int i = 0; i < D; ++i) {
    if ((i & 63) == 0) w = kvo_splitmix64_next(&st);
    neg[i] = (uint8_t)((w >> (i & 63)) & 1u);
  }
}

/* Format version 2: one sign vector per (seed, layer, head dim).  READING of
 * [OKV "FP8 and TurboQuant"] ("versioned sign generator"): layer l takes its
 * W = ceil(D/64) words from the same SplitMix64 stream, after the W*l words of
 * the layers below it, so sign i of layer l is bit (i mod 64) of output
 * l*W + floor(i/64).  Layer 0 is the version-1 vector. */
void kvo_signs_layer(uint64_t seed, int layer, int D, uint8_t* neg) {
  const int W = (D + 63) / 64;
  uint64_t st = seed, w = 0;
  for (long k = 0; k < (long)layer * W; ++k) kvo_splitmix64_next(&st);  /* the layers below */
  for (int i = 0; i < D; ++i) {
    if ((i & 63) == 0) w = kvo_splitmix64_next(&st);
    neg[i] = (uint8_t)((w >> (i & 63)) & 1u);
  }
}

/* 1/sqrt(D) rounded to FP32 (exact for D = 64, 256). */
float kvo_wht_scale(int D) { return (float)(1.0 / sqrt((double)D)); }

/* Orthonormal Walsh-Hadamard transform, natural (Sylvester) order.
 * READING: butterflies with ascending stride h = 1, 2, ..., D/2, pair
 * (i, i+h) -> (a_i + a_{i+h}, a_i - a_{i+h}); the 1/sqrt(D) scale is applied
 * once at the end.  The transform is its own inverse in exact arithmetic. */
void kvo_wht(float* a, int D) {
  for (int h = 1; h < D; h <<= 1)
    for (int i = 0; i < D; ++i)
      if ((i & h) == 0) {
        float u = a[i], v = a[i + h];
        a[i] = u + v;
        a[i + h] = u - v;
      }
  float c = kvo_wht_scale(D);
  for (int i = 0; i < D; ++i) a[i] = a[i] * c;
}

/* Probability mass of N(0,1) on (a, b), written to avoid cancellation. */
static double gauss_mass(double a, double b) {
  const double r2 = 1.4142135623730950488;
  if (a >= 0.0) return 0.5 * (erfc(a / r2) - erfc(b / r2));
  if (b <= 0.0) return 0.5 * (erfc(-b / r2) - erfc(-a / r2));
  return 0.5 * (erf(b / r2) - erf(a / r2));
}
static double gauss_pdf(double t) {
  if (isinf(t)) return 0.0;
  return exp(-0.5 * t * t) / 2.5066282746310005024;   /* sqrt(2*pi) */
}

/* Lloyd-Max quantizer of N(0,1) with K = 2^bits levels (Lloyd's iteration:
 * boundaries at centroid midpoints, centroids at conditional means
 * E[X | t_j < X < t_{j+1}] = (pdf(t_j) - pdf(t_{j+1})) / mass(t_j, t_{j+1})),
 * FP64, iterated to its fixed point.  Centroids ascending. */
void kvo_lloyd_max_gauss(int bits, double* c) {
  int K = 1 << bits;
  double t[257], nc[256];
  for (int j = 0; j < K; ++j) c[j] = -2.0 + 4.0 * (j + 0.5) / K;
  for (int it = 0; it < 200000; ++it) {
    t[0] = -INFINITY;
    t[K] = INFINITY;
    for (int j = 1; j < K; ++j) t[j] = 0.5 * (c[j - 1] + c[j]);
    double dmax = 0.0;
    for (int j = 0; j < K; ++j) {
      nc[j] = (gauss_pdf(t[j]) - gauss_pdf(t[j + 1])) / gauss_mass(t[j], t[j + 1]);
      double d = fabs(nc[j] - c[j]);
      if (d > dmax) dmax = d;
    }
    for (int j = 0; j < K; ++j) c[j] = nc[j];
    if (dmax <= 4e-16) break;
  }
}

/* READING: a rotated unit vector of dimension D has coordinates ~ N(0, 1/D),
 * so the codebook is the N(0,1) Lloyd-Max quantizer scaled by 1/sqrt(D):
 * cent[j] = fl32(c_j / sqrt(D)), bnd[j] = fl32(((c_j + c_{j+1}) / 2) / sqrt(D)). */
void kvo_codebook(int bits, int D, float* cent, float* bnd) {
  double c[256];
  int K = 1 << bits;
  kvo_lloyd_max_gauss(bits, c);
  double sd = sqrt((double)D);
  for (int j = 0; j < K; ++j) cent[j] = (float)(c[j] / sd);
  for (int j = 0; j + 1 < K; ++j) bnd[j] = (float)((0.5 * (c[j] + c[j + 1])) / sd);
}

/* code = number of boundaries strictly below y (READING: a value equal to a
 * boundary takes the lower index). */
static int tq_index(float y, const float* bnd, int K) {
  int code = 0;
  for (int j = 0; j + 1 < K; ++j)
    if (bnd[j] < y) code++;
  return code;
}

/* Encode one K vector.  n = sqrt(pairwise sum of x_i^2); r = 1/n (0 when
 * that is not finite); u_i = +-(x_i * r); y = WHT(u); codes; FP16 norm. */
void kvo_tq_encode_vec(const float* x, int D, int bits, const uint8_t* neg,
                       const float* bnd, uint8_t* codes, uint16_t* norm16) {
  float sq[256], u[256];
  for (int i = 0; i < D; ++i) sq[i] = x[i] * x[i];
  float n = sqrtf(kvo_pairwise_sum(sq, D));
  float r = 1.0f / n;
  if (!isfinite(r)) r = 0.0f;
  for (int i = 0; i < D; ++i) {
    u[i] = x[i] * r;
    if (neg[i]) u[i] = -u[i];
  }
  kvo_wht(u, D);
  for (int i = 0; i < D; ++i) codes[i] = (uint8_t)tq_index(u[i], bnd, 1 << bits);
  *norm16 = kvo_f32_to_f16(n);
}

/* Restore one K vector: c_i = cent[code_i]; nc = sqrt(pairwise sum c_i^2);
 * g = norm/nc; t = WHT(c); undo the signs; out_i = t_i * g. */
void kvo_tq_decode_vec(const uint8_t* codes, uint16_t norm16, int D, int bits,
                       const uint8_t* neg, const float* cent, float* out) {
  float c[256], sq[256];
  (void)bits;
  for (int i = 0; i < D; ++i) c[i] = cent[codes[i]];
  for (int i = 0; i < D; ++i) sq[i] = c[i] * c[i];
  float nc = sqrtf(kvo_pairwise_sum(sq, D));
  float g = kvo_f16_to_f32(norm16) / nc;
  kvo_wht(c, D);
  for (int i = 0; i < D; ++i) {
    float t = neg[i] ? -c[i] : c[i];
    out[i] = t * g;
  }
}

/* ======================================================================== */
/* 5. Per-vector uniform quantization with FP16 minimum and scale            */
/* ([OKV "FP8 and TurboQuant"], V).  READING: codes are taken against the    */
/* FP16-rounded minimum m and scale s: code = rint((x - m)/s) clamped to      */
/* [0, 2^b - 1], code 0 when s == 0; restore = code*s + m.                   */
/* ======================================================================== */
void kvo_uniform_encode_vec(const float* x, int D, int bits, uint8_t* codes,
                            uint16_t* m16, uint16_t* s16) {
  /* READING: the sign of a zero minimum or maximum carries no information for
   * the step or the offset; a zero extreme is taken as +0 (x + 0 in FP32), so
   * the stored FP16 minimum of a vector whose minimum is a zero is 0x0000 */
  float mn = x[0], mx = x[0];
  for (int i = 1; i < D; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  float levels = (float)((1 << bits) - 1);
  *m16 = kvo_f32_to_f16(mn);
  *s16 = kvo_f32_to_f16((mx - mn) / levels);
  float m = kvo_f16_to_f32(*m16), s = kvo_f16_to_f32(*s16);
  for (int i = 0; i < D; ++i) {
    if (s == 0.0f) { codes[i] = 0; continue; }
    float q = rintf((x[i] - m) / s);
    /* READING: a quotient that is not a number takes the lower clamp.  It
     * arises only when the FP16 minimum and step overflow (m = -inf and
     * s = inf), i.e. when an admission bound above the FP16 range lets BF16
     * values beyond +-65504 through. */
    if (!(q >= 0.0f)) q = 0.0f;
    if (q > levels) q = levels;
    codes[i] = (uint8_t)q;
  }
}

void kvo_uniform_decode_vec(const uint8_t* codes, uint16_t m16, uint16_t s16, int D,
                            float* out) {
  float m = kvo_f16_to_f32(m16), s = kvo_f16_to_f32(s16);
  for (int i = 0; i < D; ++i) out[i] = (float)codes[i] * s + m;
}

/* ======================================================================== */
/* 5b. Symmetric per-head INT8 ([HIQ "Building the INT8 codec"]), BF16 KV.  */
/* One scale per head vector (token, layer, K or V, head), in the page's     */
/* order of operations on BF16 tensors:                                     */
/*   amax  = max |x| raised to a floor (BF16 tensor: the floor is rounded to */
/*           BF16 when it applies; READING: floor 1e-12, the FP8 rule's, as  */
/*           the page names only "a small nonzero floor");                    */
/*   scale = amax / 127, divided in FP32 and rounded to BF16 (BF16 tensor     */
/*           divided by an integer);                                         */
/*   code  = round half to even of FP32(x) / FP32(scale), clamped to          */
/*           [-127, 127] (the rounded scale can push the quotient past 127);  */
/*   restore = code * scale as BF16 tensors: the FP32 product (exact)         */
/*           rounded to BF16.                                                  */
/* ======================================================================== */
static const float kInt8AmaxFloor = 1e-12f;

uint16_t kvo_int8_scale(float amax) {
  float a = amax < kInt8AmaxFloor ? kvo_bf16_to_f32(kvo_f32_to_bf16(kInt8AmaxFloor)) : amax;
  float q = a / 127.0f;
  return kvo_f32_to_bf16(q);
}

void kvo_int8_encode_vec(const float* x, int D, int8_t* codes, uint16_t* scale16) {
  *scale16 = kvo_int8_scale(kvo_absmax(x, D));
  float s = kvo_bf16_to_f32(*scale16);
  for (int i = 0; i < D; ++i) {
    float q = rintf(x[i] / s);   /* default rounding mode: nearest, ties to even */
    if (q > 127.0f) q = 127.0f;
    if (q < -127.0f) q = -127.0f;
    codes[i] = (int8_t)q;
  }
}

void kvo_int8_decode_vec(const int8_t* codes, uint16_t scale16, int D, float* out) {
  float s = kvo_bf16_to_f32(scale16);
  for (int i = 0; i < D; ++i) out[i] = (float)codes[i] * s;   /* exact; rounded by the caller */
}

/* ======================================================================== */
/* 6. Code packing.  READING: little-endian bit stream, code i occupies bits */
/* [b*i, b*i + b) (byte k, bit m is stream bit 8k + m); b = 8 is one byte    */
/* per code.  Gives D*b/8 bytes per vector ([OKV]: 64 + 2 = 66 for 4-bit K). */
/* ======================================================================== */
void kvo_pack_bits(const uint8_t* codes, int n, int bits, uint8_t* out) {
  memset(out, 0, (size_t)(n * bits + 7) / 8);
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < bits; ++k)
      if ((codes[i] >> k) & 1) {
        int pos = i * bits + k;
        out[pos >> 3] |= (uint8_t)(1u << (pos & 7));
      }
}

void kvo_unpack_bits(const uint8_t* in, int n, int bits, uint8_t* codes) {
  for (int i = 0; i < n; ++i) {
    int v = 0;
    for (int k = 0; k < bits; ++k) {
      int pos = i * bits + k;
      v |= ((in[pos >> 3] >> (pos & 7)) & 1) << k;
    }
    codes[i] = (uint8_t)v;
  }
}

/* ======================================================================== */
/* 7. Segments: the codec's unit of admission and storage.                    */
/* READING: a segment is all vectors of one role (K or V) of one page (block) */
/* of one layer, vectors ordered v = token*H + head; encoded slot =           */
/* [codes of all vectors][metadata of all vectors], zero-padded to 128 B.    */
/* [OKV "Ownership, storage and GDS"]: segments with nonfinite values stay    */
/* raw, as do oversized (> 16 MiB source) segments and encodings that save   */
/* less than 12.5%; [OKV "FP8 and TurboQuant"]: values outside the range      */
/* stay raw rather than being clipped, and the first and last two layers of  */
/* the stage stay exact under the TurboQuant policy.                         */
/* ======================================================================== */
typedef struct {
  int32_t dtype, layout, head_dim, num_heads, block_tokens, num_layers;
  int64_t num_blocks, stride_block, stride_token, stride_head;
  int32_t codec[2];                 /* per role: 0 = K, 1 = V */
  int32_t protect_first, protect_last;
  uint64_t seed;
  float reject_abs;
  int32_t sign_version;             /* 0 or 1: one sign vector per (seed, D); 2: per layer too */
  const float* fixed_amax;          /* [num_layers][2] calibration absmax */
  int32_t fixed_overflow;           /* FP8_FIXED: 0 = clip quotients to +-448, 1 = keep the segment raw */
  int32_t reserved;
} kvo_geom;

/* The sign vector of a layer under the geometry's format version. */
static void layer_signs(const kvo_geom* g, int layer, uint8_t* neg) {
  if (g->sign_version == 2) kvo_signs_layer(g->seed, layer, g->head_dim, neg);
  else kvo_signs(g->seed, g->head_dim, neg);
}
static uint32_t format_version(const kvo_geom* g) { return g->sign_version == 2 ? 2u : 1u; }

typedef struct {
  uint32_t layer, block, role, reserved;
  uint64_t enc_offset;
} kvo_desc;

static int codec_bits(int codec) {
  switch (codec) {
    case O_TQ2: case O_UNI2: return 2;
    case O_TQ3: case O_UNI3: return 3;
    case O_TQ4: case O_UNI4: return 4;
    case O_UNI8: return 8;
    default: return 0;
  }
}
static int is_fp8(int c) { return c == O_FP8_CAST || c == O_FP8_FIXED || c == O_FP8_DYNAMIC; }
static int is_tq(int c) { return c == O_TQ2 || c == O_TQ3 || c == O_TQ4; }
static int is_uni(int c) { return c == O_UNI2 || c == O_UNI3 || c == O_UNI4 || c == O_UNI8; }

/* [HIQ "Why exactly 1,152 bytes?"]: the INT8 codec stores one record per
 * token row of a role: the H heads' int8 codes (H*D bytes), then their H BF16
 * scales, zero-padded to a multiple of 128 bytes (8 heads x 128: 1,040 ->
 * 1,152).  A segment's slot is its block_tokens records in token order. */
int64_t kvo_int8_record_bytes(int H, int D) {
  int64_t b = (int64_t)H * (D + 2);
  return (b + 127) / 128 * 128;
}

/* Bytes per vector: codes and metadata. */
static void vec_bytes(int codec, int D, int* code_b, int* meta_b) {
  if (is_fp8(codec)) { *code_b = D; *meta_b = codec == O_FP8_DYNAMIC ? 4 : 0; }
  else if (is_tq(codec)) { *code_b = D * codec_bits(codec) / 8; *meta_b = 2; }
  else if (is_uni(codec)) { *code_b = D * codec_bits(codec) / 8; *meta_b = 4; }
  else { *code_b = 0; *meta_b = 0; }
}

int64_t kvo_segment_enc_bytes(const kvo_geom* g, int role) {
  if (g->codec[role] == O_INT8)
    return (int64_t)g->block_tokens * kvo_int8_record_bytes(g->num_heads, g->head_dim);
  int cb, mb;
  vec_bytes(g->codec[role], g->head_dim, &cb, &mb);
  int64_t nv = (int64_t)g->num_heads * g->block_tokens;
  int64_t b = nv * (cb + mb);
  return (b + 127) / 128 * 128;
}
int64_t kvo_segment_raw_bytes(const kvo_geom* g) {
  return (int64_t)g->num_heads * g->block_tokens * g->head_dim * 2;
}

static uint16_t* vec_ptr(const kvo_geom* g, void* const* ptrs, const kvo_desc* d, int t, int h) {
  uint16_t* base;
  int64_t off = (int64_t)d->block * g->stride_block + (int64_t)t * g->stride_token +
                (int64_t)h * g->stride_head;
  if (g->layout == O_SEPARATE) base = (uint16_t*)ptrs[2 * d->layer + d->role];
  else { base = (uint16_t*)ptrs[d->layer]; off += (int64_t)d->role * g->head_dim; }
  return base + off;
}

/* Descriptor validity (shared contract with the product, written separately). */
static int desc_ok(const kvo_geom* g, void* const* ptrs, const kvo_desc* d, uint64_t buf_bytes) {
  if (d->layer >= (uint32_t)g->num_layers || d->role > 1) return 0;
  if ((int64_t)d->block >= g->num_blocks) return 0;
  void* p = g->layout == O_SEPARATE ? ptrs[2 * d->layer + d->role] : ptrs[d->layer];
  if (!p) return 0;
  if (d->enc_offset % 16) return 0;
  uint64_t need = (uint64_t)kvo_segment_enc_bytes(g, (int)d->role);
  if (d->enc_offset > buf_bytes || need > buf_bytes - d->enc_offset) return 0;
  return 1;
}

static int policy_status(const kvo_geom* g, const kvo_desc* d) {
  int codec = g->codec[d->role];
  if (codec == O_NONE) return S_RAW_POLICY;
  if ((int)d->layer < g->protect_first || (int)d->layer >= g->num_layers - g->protect_last)
    return S_RAW_PROTECTED;
  int64_t raw = kvo_segment_raw_bytes(g);
  if (raw > (int64_t)16 << 20) return S_RAW_OVERSIZE;
  /* keep only if the aligned footprint saves >= 12.5%: enc <= 7/8 raw */
  if (8 * kvo_segment_enc_bytes(g, (int)d->role) > 7 * raw) return S_RAW_NO_SAVING;
  return 0;
}

void kvo_encode(const kvo_geom* g, void* const* ptrs, const kvo_desc* descs, uint32_t n,
                uint8_t* out, uint64_t out_bytes, uint8_t* status) {
  int D = g->head_dim, H = g->num_heads, T = g->block_tokens;
  int nv = H * T;
  uint8_t neg[256];
  float cent[16], bnd[16];
  int neg_layer = -1;               /* layer whose signs neg holds */
  float reject = g->reject_abs > 0.0f ? g->reject_abs : 448.0f;
  float* x = (float*)malloc(sizeof(float) * (size_t)D);
  uint8_t* codes = (uint8_t*)malloc((size_t)D);
  int cb_bits_done = 0;
  for (uint32_t i = 0; i < n; ++i) {
    const kvo_desc* d = &descs[i];
    if (!desc_ok(g, ptrs, d, out_bytes)) { status[i] = S_BAD_DESC; continue; }
    int st = policy_status(g, d);
    if (st) { status[i] = (uint8_t)st; continue; }
    int codec = g->codec[d->role];
    /* admission: scan the source segment */
    int nonfinite = 0, range = 0;
    for (int t = 0; t < T; ++t)
      for (int h = 0; h < H; ++h) {
        const uint16_t* p = vec_ptr(g, ptrs, d, t, h);
        for (int e = 0; e < D; ++e) {
          float v = src_to_f32(p[e], g->dtype);
          if (!isfinite(v)) nonfinite = 1;
          else if (fabsf(v) > reject) range = 1;
        }
      }
    if (nonfinite) { status[i] = S_RAW_NONFINITE; continue; }
    if (range) { status[i] = S_RAW_RANGE; continue; }
    int cbytes, mbytes;
    vec_bytes(codec, D, &cbytes, &mbytes);
    int bits = codec_bits(codec);
    if (is_tq(codec) && cb_bits_done != bits) { kvo_codebook(bits, D, cent, bnd); cb_bits_done = bits; }
    if (is_tq(codec) && neg_layer != (int)d->layer) { layer_signs(g, (int)d->layer, neg); neg_layer = (int)d->layer; }
    uint8_t* slot = out + d->enc_offset;
    int64_t seg_bytes = kvo_segment_enc_bytes(g, (int)d->role);
    memset(slot, 0, (size_t)seg_bytes);
    uint8_t* meta = slot + (size_t)nv * cbytes;
    int64_t rec = kvo_int8_record_bytes(H, D);
    /* READING: FP16 metadata that overflows (a TurboQuant norm, a uniform
     * minimum or step beyond +-65504) cannot be stored, so the segment stays
     * raw as out of range.  Under the default bound (448) this never happens;
     * it needs an admission bound above the FP16 range and BF16 sources. */
    int meta_overflow = 0;
    for (int t = 0; t < T; ++t)
      for (int h = 0; h < H; ++h) {
        int v = t * H + h;
        const uint16_t* p = vec_ptr(g, ptrs, d, t, h);
        for (int e = 0; e < D; ++e) x[e] = src_to_f32(p[e], g->dtype);
        uint8_t* vc = slot + (size_t)v * cbytes;
        if (codec == O_INT8) {
          uint8_t* r = slot + (size_t)(t * rec);
          uint16_t s16;
          kvo_int8_encode_vec(x, D, (int8_t*)(r + (size_t)h * D), &s16);
          memcpy(r + (size_t)H * D + 2 * (size_t)h, &s16, 2);
        } else if (is_fp8(codec)) {
          float s;
          if (codec == O_FP8_CAST) s = 1.0f;
          else if (codec == O_FP8_FIXED) s = kvo_fp8_scale_from_amax(g->fixed_amax[2 * d->layer + d->role]);
          else {
            s = kvo_fp8_scale_from_amax(kvo_absmax(x, D));
            memcpy(meta + (size_t)v * 4, &s, 4);
          }
          /* READING: [OKV "FP8 and TurboQuant"] keeps values outside the
           * range raw rather than clipping them; [ASYM "Precision and scaling
           * reference"] clips quotients to +-448.  The clip is the default;
           * with fixed_overflow = 1 a fixed-scale segment in which some FP32
           * quotient x / s lies beyond +-448 stays raw (out of range). */
          if (codec == O_FP8_FIXED && g->fixed_overflow == 1)
            for (int e = 0; e < D; ++e)
              if (fabsf(x[e] / s) > 448.0f) meta_overflow = 1;
          kvo_fp8_encode_vec(x, D, s, vc);
        } else if (is_tq(codec)) {
          uint16_t n16;
          kvo_tq_encode_vec(x, D, bits, neg, bnd, codes, &n16);
          if ((n16 & 0x7FFFu) >= 0x7C00u) meta_overflow = 1;
          kvo_pack_bits(codes, D, bits, vc);
          memcpy(meta + (size_t)v * 2, &n16, 2);
        } else {
          uint16_t mm[2];
          kvo_uniform_encode_vec(x, D, bits, codes, &mm[0], &mm[1]);
          if ((mm[0] & 0x7FFFu) >= 0x7C00u || (mm[1] & 0x7FFFu) >= 0x7C00u) meta_overflow = 1;
          if (bits == 8) memcpy(vc, codes, (size_t)D);
          else kvo_pack_bits(codes, D, bits, vc);
          memcpy(meta + (size_t)v * 4, mm, 4);
        }
      }
    status[i] = meta_overflow ? S_RAW_RANGE : S_ENCODED;
  }
  free(x);
  free(codes);
}

/* Restore ENCODED segments into the engine layout; every other status is
 * left to the caller's raw path.  result[i] (optional): S_ENCODED when
 * restored, S_BAD_DESC for an invalid descriptor, else the input status. */
void kvo_decode(const kvo_geom* g, void* const* ptrs, const kvo_desc* descs, uint32_t n,
                const uint8_t* in, uint64_t in_bytes, const uint8_t* status, uint8_t* result) {
  int D = g->head_dim, H = g->num_heads, T = g->block_tokens;
  int nv = H * T;
  uint8_t neg[256];
  float cent[16], bnd[16];
  int neg_layer = -1;               /* layer whose signs neg holds */
  float* y = (float*)malloc(sizeof(float) * (size_t)D);
  uint8_t* codes = (uint8_t*)malloc((size_t)D);
  int cb_bits_done = 0;
  for (uint32_t i = 0; i < n; ++i) {
    const kvo_desc* d = &descs[i];
    if (!desc_ok(g, ptrs, d, in_bytes) || g->codec[d->role] == O_NONE) {
      if (result) result[i] = S_BAD_DESC;
      continue;
    }
    if (status[i] != S_ENCODED) {
      if (result) result[i] = status[i];
      continue;
    }
    int codec = g->codec[d->role];
    int cbytes, mbytes;
    vec_bytes(codec, D, &cbytes, &mbytes);
    int bits = codec_bits(codec);
    if (is_tq(codec) && cb_bits_done != bits) { kvo_codebook(bits, D, cent, bnd); cb_bits_done = bits; }
    if (is_tq(codec) && neg_layer != (int)d->layer) { layer_signs(g, (int)d->layer, neg); neg_layer = (int)d->layer; }
    const uint8_t* slot = in + d->enc_offset;
    const uint8_t* meta = slot + (size_t)nv * cbytes;
    int64_t rec = kvo_int8_record_bytes(H, D);
    /* READING: FP16 metadata that overflows (a TurboQuant norm, a uniform
     * minimum or step beyond +-65504) cannot be stored, so the segment stays
     * raw as out of range.  Under the default bound (448) this never happens;
     * it needs an admission bound above the FP16 range and BF16 sources. */
    int meta_overflow = 0;
    for (int t = 0; t < T; ++t)
      for (int h = 0; h < H; ++h) {
        int v = t * H + h;
        const uint8_t* vc = slot + (size_t)v * cbytes;
        if (codec == O_INT8) {
          const uint8_t* r = slot + (size_t)(t * rec);
          uint16_t s16;
          memcpy(&s16, r + (size_t)H * D + 2 * (size_t)h, 2);
          kvo_int8_decode_vec((const int8_t*)(r + (size_t)h * D), s16, D, y);
        } else if (is_fp8(codec)) {
          float s;
          if (codec == O_FP8_CAST) s = 1.0f;
          else if (codec == O_FP8_FIXED) s = kvo_fp8_scale_from_amax(g->fixed_amax[2 * d->layer + d->role]);
          else memcpy(&s, meta + (size_t)v * 4, 4);
          kvo_fp8_decode_vec(vc, D, s, y);
        } else if (is_tq(codec)) {
          uint16_t n16;
          memcpy(&n16, meta + (size_t)v * 2, 2);
          kvo_unpack_bits(vc, D, bits, codes);
          kvo_tq_decode_vec(codes, n16, D, bits, neg, cent, y);
        } else {
          uint16_t mm[2];
          memcpy(mm, meta + (size_t)v * 4, 4);
          if (bits == 8) memcpy(codes, vc, (size_t)D);
          else kvo_unpack_bits(vc, D, bits, codes);
          kvo_uniform_decode_vec(codes, mm[0], mm[1], D, y);
        }
        uint16_t* p = vec_ptr(g, ptrs, d, t, h);
        for (int e = 0; e < D; ++e) p[e] = f32_to_src(y[e], g->dtype);
      }
    if (result) result[i] = S_ENCODED;
  }
  free(y);
  free(codes);
}

/* ======================================================================== */
/* 7b. Segment header and CRC-32 ([OKV "Ownership, storage and GDS"]: every  */
/* encoded segment carries a version, its original length, its format, its  */
/* stored length and a CRC32; checksums are validated before GPU decode and  */
/* a damaged object becomes a miss).  READINGS: CRC-32 is the common IEEE    */
/* 802.3 / zlib one (reflected polynomial 0xEDB88320, register preset to all */
/* ones, result complemented) over the stored slot bytes; the header is      */
/* {u32 version = 1, u32 format = codec | dtype << 8 | log2(head_dim) << 16, */
/* u64 original bytes, u64 stored bytes (0 when the segment stayed raw),     */
/* u32 crc32, u32 status}; a verified segment keeps status ENCODED, a header */
/* or checksum mismatch gives CORRUPT, raw headers pass their status on.     */
/* ======================================================================== */
typedef struct {
  uint32_t version, format;
  uint64_t orig_bytes, stored_bytes;
  uint32_t crc32, status;
} kvo_header;

/* Bit-serial CRC-32, one message bit at a time, straight from the definition
 * of the reflected shift register. */
uint32_t kvo_crc32(const uint8_t* p, uint64_t n) {
  uint32_t r = 0xFFFFFFFFu;
  for (uint64_t i = 0; i < n; ++i) {
    r ^= p[i];
    for (int k = 0; k < 8; ++k) r = (r & 1u) ? (r >> 1) ^ 0xEDB88320u : (r >> 1);
  }
  return ~r;
}

static uint32_t header_format(const kvo_geom* g, int role) {
  int lg = 0;
  while ((1 << lg) < g->head_dim) ++lg;
  return (uint32_t)g->codec[role] | ((uint32_t)g->dtype << 8) | ((uint32_t)lg << 16);
}

/* Descriptor checks that need no layer pointers (sealing and verifying touch
 * only the slot buffer). */
static int slot_desc_ok(const kvo_geom* g, const kvo_desc* d, uint64_t buf_bytes) {
  if (d->layer >= (uint32_t)g->num_layers || d->role > 1) return 0;
  if ((int64_t)d->block >= g->num_blocks) return 0;
  if (d->enc_offset % 16) return 0;
  if (g->codec[d->role] == O_NONE) return 1;
  uint64_t need = (uint64_t)kvo_segment_enc_bytes(g, (int)d->role);
  if (d->enc_offset > buf_bytes || need > buf_bytes - d->enc_offset) return 0;
  return 1;
}

void kvo_seal(const kvo_geom* g, const kvo_desc* descs, uint32_t n, const uint8_t* buf,
              uint64_t buf_bytes, const uint8_t* status, kvo_header* out) {
  for (uint32_t i = 0; i < n; ++i) {
    const kvo_desc* d = &descs[i];
    kvo_header h;
    memset(&h, 0, sizeof h);
    h.version = format_version(g);
    h.orig_bytes = (uint64_t)kvo_segment_raw_bytes(g);
    if (!slot_desc_ok(g, d, buf_bytes)) {
      h.status = S_BAD_DESC;
    } else {
      h.format = header_format(g, (int)d->role);
      h.status = status[i];
      if (status[i] == S_ENCODED && g->codec[d->role] != O_NONE) {
        h.stored_bytes = (uint64_t)kvo_segment_enc_bytes(g, (int)d->role);
        h.crc32 = kvo_crc32(buf + d->enc_offset, h.stored_bytes);
      }
    }
    out[i] = h;
  }
}

void kvo_verify(const kvo_geom* g, const kvo_desc* descs, uint32_t n, const uint8_t* buf,
                uint64_t buf_bytes, const kvo_header* hdr, uint8_t* result) {
  for (uint32_t i = 0; i < n; ++i) {
    const kvo_desc* d = &descs[i];
    const kvo_header* h = &hdr[i];
    if (!slot_desc_ok(g, d, buf_bytes) || g->codec[d->role] == O_NONE) { result[i] = S_BAD_DESC; continue; }
    int ok = h->version == format_version(g) && h->format == header_format(g, (int)d->role) &&
             h->orig_bytes == (uint64_t)kvo_segment_raw_bytes(g) &&
             h->status >= S_ENCODED && h->status <= S_BAD_DESC;
    if (ok && h->status == S_ENCODED)
      ok = h->stored_bytes == (uint64_t)kvo_segment_enc_bytes(g, (int)d->role) &&
           kvo_crc32(buf + d->enc_offset, h->stored_bytes) == h->crc32;
    else if (ok)
      ok = h->stored_bytes == 0;
    result[i] = ok ? (uint8_t)h->status : (uint8_t)S_CORRUPT;
  }
}

/* ======================================================================== */
/* 8. Array forms of the scalar conversions (for exhaustive tests).         */
/* ======================================================================== */
void kvo_f16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_f16_to_f32(h[i]);
}
void kvo_bf16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_bf16_to_f32(h[i]);
}
void kvo_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_f32_to_f16(x[i]);
}
void kvo_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_f32_to_bf16(x[i]);
}
void kvo_f32_to_e4m3_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_f32_to_e4m3(x[i]);
}
void kvo_e4m3_to_f32_array(const uint8_t* c, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvo_e4m3_to_f32(c[i]);
}
/* FP8 encode of n vectors of length D, per-vector scales given in s[] */
void kvo_fp8_encode_many(const float* x, int64_t nvec, int D, const float* s, uint8_t* codes) {
  for (int64_t v = 0; v < nvec; ++v) kvo_fp8_encode_vec(x + v * D, D, s[v], codes + v * D);
}
void kvo_tq_encode_many(const float* x, int64_t nvec, int D, int bits, uint64_t seed,
                        uint8_t* codes, uint16_t* norm16) {
  uint8_t neg[256];
  float cent[16], bnd[16];
  kvo_signs(seed, D, neg);
  kvo_codebook(bits, D, cent, bnd);
  for (int64_t v = 0; v < nvec; ++v)
    kvo_tq_encode_vec(x + v * D, D, bits, neg, bnd, codes + v * D, norm16 + v);
}
void kvo_tq_decode_many(const uint8_t* codes, const uint16_t* norm16, int64_t nvec, int D,
                        int bits, uint64_t seed, float* out) {
  uint8_t neg[256];
  float cent[16], bnd[16];
  kvo_signs(seed, D, neg);
  kvo_codebook(bits, D, cent, bnd);
  for (int64_t v = 0; v < nvec; ++v)
    kvo_tq_decode_vec(codes + v * D, norm16[v], D, bits, neg, cent, out + v * D);
}
/* The same with the sign vector given (one byte per element, 1 = negate). */
void kvo_tq_encode_many_signs(const float* x, int64_t nvec, int D, int bits, const uint8_t* neg,
                              uint8_t* codes, uint16_t* norm16) {
  float cent[16], bnd[16];
  kvo_codebook(bits, D, cent, bnd);
  for (int64_t v = 0; v < nvec; ++v)
    kvo_tq_encode_vec(x + v * D, D, bits, neg, bnd, codes + v * D, norm16 + v);
}
void kvo_tq_decode_many_signs(const uint8_t* codes, const uint16_t* norm16, int64_t nvec, int D,
                              int bits, const uint8_t* neg, float* out) {
  float cent[16], bnd[16];
  kvo_codebook(bits, D, cent, bnd);
  for (int64_t v = 0; v < nvec; ++v)
    kvo_tq_decode_vec(codes + v * D, norm16[v], D, bits, neg, cent, out + v * D);
}
void kvo_uniform_encode_many(const float* x, int64_t nvec, int D, int bits, uint8_t* codes,
                             uint16_t* m16, uint16_t* s16) {
  for (int64_t v = 0; v < nvec; ++v)
    kvo_uniform_encode_vec(x + v * D, D, bits, codes + v * D, m16 + v, s16 + v);
}
void kvo_uniform_decode_many(const uint8_t* codes, const uint16_t* m16, const uint16_t* s16,
                             int64_t nvec, int D, float* out) {
  for (int64_t v = 0; v < nvec; ++v)
    kvo_uniform_decode_vec(codes + v * D, m16[v], s16[v], D, out + v * D);
}
void kvo_int8_encode_many(const float* x, int64_t nvec, int D, int8_t* codes, uint16_t* scale16) {
  for (int64_t v = 0; v < nvec; ++v) kvo_int8_encode_vec(x + v * D, D, codes + v * D, scale16 + v);
}
void kvo_int8_decode_many(const int8_t* codes, const uint16_t* scale16, int64_t nvec, int D,
                          float* out) {
  for (int64_t v = 0; v < nvec; ++v) kvo_int8_decode_vec(codes + v * D, scale16[v], D, out + v * D);
}
void kvo_tq_index_many(const float* y, int64_t n, int bits, int D, uint8_t* codes) {
  float cent[16], bnd[16];
  kvo_codebook(bits, D, cent, bnd);
  for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)tq_index(y[i], bnd, 1 << bits);
}
