// turboquant.cu -- TurboQuant-style K encode / decode kernels (2, 3 and 4 bits).
//
// "KV precision and storage encoding" (OrbitKV), section "FP8 and
// TurboQuant": normalize each head vector, apply deterministic random signs
// and an orthonormal Walsh-Hadamard transform, then encode Gaussian
// Lloyd-Max centroids; restore corrects the centroid-vector norm, applies
// the inverse transform and the original FP16 norm.
//
// Encode, per vector: n = sqrt(pairwise sum of x_i^2), r = 1/n (0 if not
// finite), u_i = +-x_i * r (the sign flip is applied to the 16-bit source,
// which is exact), w = Walsh-Hadamard butterflies of u (ascending stride),
// y = RN(w * 1/sqrt(D)), code_i = number of codebook boundaries below y_i,
// FP16(n) stored.  The scale is folded into the boundaries (an exact
// rewriting, see Params::lut_thr), and the index comes from a cell table:
// one FFMA, one shared-memory load and one compare per element.
// Decode: c_i = centroid[code_i], g = f32(n16) / sqrt(pairwise sum c_i^2),
// out_i = +-(RN(RN(WHT(c)_i * 1/sqrt(D)) * g)).
//
// Thread mapping: a lane owns 64 contiguous elements of a vector when
// D >= 64 (the "64 elements per lane" kernels below), else 32 (64 bytes of
// FP16/BF16), G = D/32 lanes per vector, held as 16 FP32 pairs (element 2m,
// 2m+1).  Butterflies with stride
// 2..16 are packed FP32x2 ops between pairs, stride 1 is inside a pair, and
// strides >= 32 are warp shuffles across the vector's lanes.
#include "device_common.cuh"

namespace kvc {
namespace {

constexpr int kTqE = 32;               // elements per lane
constexpr float kCellMagic = 12582912.0f;  // 1.5 * 2^23: FFMA(w, 4, magic) has rint(4 w) in its low bits
constexpr uint32_t kCellMagicBits = 0x4b400000u;

// Sign mask word k (elements 2k, 2k+1 of a lane's 32) for sign word `bits`.
__device__ __forceinline__ uint32_t sign_mask_word(uint32_t bits, int k) {
  return (((bits >> (2 * k)) & 1u) << 15) | (((bits >> (2 * k + 1)) & 1u) << 31);
}

// Output k (k = 0, 1, ...) of the SplitMix64 stream seeded with `seed`
// (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014): the seed advanced by k + 1 golden-gamma increments, through
// the variant-13 finalizer.
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t k) {
  uint64_t z = seed + (k + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Sign bits of elements 32 w .. 32 w + 31 (bit i = negate element 32 w + i)
// of the TurboQuant sign vector of `layer`: bit i mod 64 of stream output
// layer * ceil(D / 64) + i / 64 (format version 2), or of layer 0's outputs
// for every layer (version 1).
__device__ __forceinline__ uint32_t tq_sign_word(const Params& p, uint32_t layer, uint32_t w) {
  const uint32_t per_layer = (p.D + 63u) / 64u;
  const uint64_t z = splitmix64_at(p.sign_seed, (uint64_t)(p.sign_per_layer ? layer : 0u) * per_layer + (w >> 1));
  return (w & 1u) ? (uint32_t)(z >> 32) : (uint32_t)z;
}

// Pairwise sum of the squares of pairs [M0, M0 + N) (2N elements), written
// depth first so that few partial sums are live at a time.
template <int M0, int N>
struct PairSumSq {
  template <int P>
  static __device__ __forceinline__ float run(const float2 (&a)[P]) {
    if constexpr (N == 1) {
      const float2 q = mul2(a[M0], a[M0]);
      return __fadd_rn(q.x, q.y);
    } else {
      const float lo = PairSumSq<M0, N / 2>::run(a);
      const float hi = PairSumSq<M0 + N / 2, N / 2>::run(a);
      return __fadd_rn(lo, hi);
    }
  }
};

// Pairwise sum of squares over the vector: the lane's 2P contiguous elements
// as an in-thread tree, then xor-shuffles over the G lanes with ascending
// distance.
template <int G, int P>
__device__ __forceinline__ float vector_sumsq(const float2 (&a)[P]) {
  float c = PairSumSq<0, P>::run(a);
#pragma unroll
  for (int o = 1; o < G; o <<= 1) c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, o));
  return c;
}

// Walsh-Hadamard butterflies of the 32-element decoder.  Strides 1 .. 16
// inside the lane (stride 1 inside each pair, 2 .. 16 between pairs); a cross-lane stage (lanes l and l ^ o, stride 32 o) is split
// between the two lanes instead of doubled: the lower lane computes the sums
// and differences of slots 0..15, the upper lane those of slots 16..31, so
// each sends only the half the other needs (16 shuffles per stage, not 32).
// Sums land in slots 0..15 and differences in 16..31 of both lanes.  After the
// J = log2(G) stages, slot s of lane l holds element
//   (s & 15) | (l << 4) | ((s >> 4) << (4 + J))
// (the half bit of the slot and the lane bits have traded places).  Each sum
// and difference is the single rounding of the same operands as in the
// ascending-stride transform.
template <int G>
__device__ __forceinline__ void butterflies_split(float2 (&a)[16], uint32_t li) {
#pragma unroll
  for (int m = 0; m < 16; ++m) {  // stride 1: inside each pair
    const float u = a[m].x, v = a[m].y;
    a[m] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {  // strides 2, 4, 8, 16
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m & h) continue;
      const float2 u = a[m], v = a[m + h];
      a[m] = add2(u, v);
      a[m + h] = sub2(u, v);
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {  // strides 32 o: across lanes, split
    const bool low = (li & (uint32_t)o) == 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float2 send = low ? a[8 + m] : a[m];
      const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, send.x, o),
                                   __shfl_xor_sync(0xffffffffu, send.y, o));
      const float2 u = low ? a[m] : r, v = low ? r : a[8 + m];
      a[m] = add2(u, v);
      a[8 + m] = sub2(u, v);
    }
  }
}

// First element of the 8 slots 8c .. 8c + 7 of lane li after butterflies_split.
template <int G>
__device__ __forceinline__ uint32_t split_group_start(uint32_t li, int c) {
  constexpr int J = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  return (uint32_t)((8 * c) & 15) | (li << 4) | ((uint32_t)(c >> 1) << (4 + J));
}



// ---------------------------------------------------------------- 64 elements per lane
// For D >= 64 a lane owns 64 contiguous elements (G = D/64 lanes per vector):
// the 64-point transform inside the lane needs no shuffles, and D = 128 has
// a single cross-lane stage.  That stage is split between the two partner
// lanes without any lane-dependent selects:
//  * the odd lane negates its inputs 32..63 (folded into its sign masks, so
//    free).  Negating the upper half of a transform's inputs swaps the two
//    halves of its outputs, so after the in-lane stages its register s holds
//    in-lane coefficient s ^ 32, exactly (each sum or difference is the
//    single rounding of the same operands, up to sign);
//  * both lanes keep registers 0..31 and send 32..63, and both compute
//    X = keep + recv, Y = keep - recv.  The even lane gets the sums of
//    elements 0..31 and the differences of elements 0..31 of the stage
//    (vector elements A + s and A + 64 + s), the odd lane the sums and the
//    negated differences of elements 32..63, negated once more afterwards.
// D = 256 splits its second stage (lanes li, li ^ 2) the same way, after
// the first one has put the upper lanes' sums and differences in swapped
// registers (butterflies64).  Lane li ends with elements 32 li + s
// (registers 0..31) and 32 G + 32 li + s (32..63); tq64_run_negated names
// the runs that come out negated.
constexpr int kTq64Threads = 128;

__device__ __forceinline__ uint4 xor4(const uint4& a, uint32_t m) {
  return make_uint4(a.x ^ m, a.y ^ m, a.z ^ m, a.w ^ m);
}

// After butterflies64 (without the fix), run R (0: registers 0..31, 1:
// 32..63) of lane li holds the negated elements: lane 1's second run at
// G = 2; lane 3's first and lane 2's second at G = 4.
template <int G>
__device__ __forceinline__ bool tq64_run_negated(uint32_t li, int run) {
  if constexpr (G == 2) return run == 1 && li == 1u;
  if constexpr (G == 4) return run == 0 ? li == 3u : li == 2u;
  return false;
}

// Elements of run R of lane li: 32 li + s (R = 0) and 32 G + 32 li + s (R = 1).
template <int G>
__device__ __forceinline__ uint32_t tq64_run_start(uint32_t li, int run) {
  return 32u * li + (run ? 32u * G : 0u);
}

template <int G, bool FIX>
__device__ __forceinline__ void butterflies64(float2 (&a)[32], uint32_t li) {
#pragma unroll
  for (int m = 0; m < 32; ++m) {  // stride 1: inside each pair
    const float u = a[m].x, v = a[m].y;
    a[m] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
  }
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {  // strides 2 .. 32: pair m with pair m + h
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      if (m & h) continue;
      const float2 u = a[m], v = a[m + h];
      a[m] = add2(u, v);
      a[m + h] = sub2(u, v);
    }
  }
  if constexpr (G == 2) {  // stride 64: lanes li, li ^ 1, split (see above)
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 1),
                                   __shfl_xor_sync(0xffffffffu, a[16 + m].y, 1));
      const float2 k = a[m];
      a[m] = add2(k, r);
      a[16 + m] = sub2(k, r);
    }
  }
  if constexpr (G == 4) {
    // stride 64 (lanes li, li ^ 1) as above, except that lanes 2 and 3 put
    // the differences in registers 0..31 and the sums in 32..63: r * t + k
    // with t = -1 is the single rounding of k - r.  Stride 128 (lanes li,
    // li ^ 2) then pairs registers 0..31 of the lower lane with 32..63 of the
    // upper one and splits the same way.
    const float t = (li & 2u) ? -1.0f : 1.0f;
    const float2 t2 = make_float2(t, t), nt2 = make_float2(-t, -t);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 1),
                                   __shfl_xor_sync(0xffffffffu, a[16 + m].y, 1));
      const float2 k = a[m];
      a[m] = fma2(r, t2, k);
      a[16 + m] = fma2(r, nt2, k);
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 2),
                                   __shfl_xor_sync(0xffffffffu, a[16 + m].y, 2));
      const float2 k = a[m];
      a[m] = add2(k, r);
      a[16 + m] = sub2(k, r);
    }
  }
  if constexpr (G >= 2 && FIX) {  // the negated runs (see tq64_run_negated)
    const float fa = tq64_run_negated<G>(li, 0) ? -1.0f : 1.0f;
    const float fb = tq64_run_negated<G>(li, 1) ? -1.0f : 1.0f;
    const float2 fa2 = make_float2(fa, fa), fb2 = make_float2(fb, fb);
    if constexpr (G == 4) {
#pragma unroll
      for (int m = 0; m < 16; ++m) a[m] = mul2(a[m], fa2);
    }
#pragma unroll
    for (int m = 16; m < 32; ++m) a[m] = mul2(a[m], fb2);
  }
}

// (c << 2 BITS) | (a << BITS) | b for codes a, b < 2^BITS (BITS = 2 or 4):
// one saturating pack, which leaves in-range codes unchanged
template <int BITS>
__device__ __forceinline__ uint32_t tq_pack2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if (BITS == 4) asm("cvt.pack.sat.u4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else asm("cvt.pack.sat.u2.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Store the codes of 32 consecutive elements (4 words of 8 codes, element 0
// lowest) at byte `dst` (the element index of the first times BITS / 8).
template <int BITS>
__device__ __forceinline__ void tq_store32(uint8_t* dst, const uint32_t (&acc)[4]) {
  if (BITS == 4) {
    st16(dst, make_uint4(acc[0], acc[1], acc[2], acc[3]));
  } else if (BITS == 2) {
    st8(dst, make_uint2(acc[0] | (acc[1] << 16), acc[2] | (acc[3] << 16)));
  } else {
    st4(dst, acc[0] | (acc[1] << 24));
    st4(dst + 4, (acc[1] >> 8) | (acc[2] << 16));
    st4(dst + 8, (acc[2] >> 16) | (acc[3] << 8));
  }
}

// Encoder for D >= 64.  Lane li of a vector's G = D/64 lanes owns elements
// 64 li .. 64 li + 63 ("in-lane index" k = 0..63), held as 32 FP32 pairs
// a[P] = (element k, element k + 16) with k = (P & 15) | ((P & 16) << 1):
// the in-lane index bits 0..3 are the pair bits 0..3, bit 4 is the pair's
// component and bit 5 is pair bit 4.  So the pairwise sum of squares and the
// transform stages of strides 1, 2, 4, 8 and 32 are packed FP32x2 operations
// between pairs; only stride 16 works inside the pairs.  The next vector's
// 128 bytes are loaded into registers while the current one is coded.
//
// The odd lane's inputs with k >= 32 are negated through its sign masks, so
// after the in-lane stages its pair P holds what the even lane's pair P ^ 16
// holds (see tq64_run_negated): both lanes keep pairs 0..15 and exchange
// 16..31 for the stride-64 stage.  Negated output runs are coded through the
// mirrored index table, whose codes are the bitwise complement of the
// direct ones; the packed words are complemented back.
// Pairwise sum of squares over pairs [P0, P0 + N), componentwise.  The
// squares are FMAs with the -0 addend nz2 (see the normalisation in the
// encoder): a packed product feeding a packed addition would be fused with
// it, which rounds differently when a square falls below the normal range.
template <int P0, int N>
struct PairTree {
  template <int NP>
  static __device__ __forceinline__ float2 run(const float2 (&a)[NP], float2 nz2) {
    if constexpr (N == 1) {
      return fma2(a[P0], a[P0], nz2);
    } else {
      return add2(PairTree<P0, N / 2>::run(a, nz2), PairTree<P0 + N / 2, N / 2>::run(a, nz2));
    }
  }
};

// Codes of the 32 elements of run R (pairs 16 R .. 16 R + 15; run element o
// in pair 16 R + (o & 15), component o >> 4), 8 per word, element 0 lowest;
// `lut` is the direct or the mirrored table of this lane and run, `cm` the
// complement that turns the table's codes into the element's.
template <int BITS, int R, int NP>
__device__ __forceinline__ void tq_run_codes(const float2 (&a)[NP], uint32_t lut, uint32_t cm,
                                             uint32_t (&acc)[4]) {
  const float2 k4 = make_float2(4.0f, 4.0f), mg = make_float2(kCellMagic, kCellMagic);
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // pairs 16 R + 8 half .. + 7: words half, half + 2
    uint32_t cx[8], cy[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 v = a[16 * R + 8 * half + e];
      const float2 cell = fma2(v, k4, mg);
      uint2 tx, ty;
      asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(tx.x), "=r"(tx.y) : "r"(__float_as_uint(cell.x) * 128u + lut));
      asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(ty.x), "=r"(ty.y) : "r"(__float_as_uint(cell.y) * 128u + lut));
      cx[e] = tx.y + (v.x > __uint_as_float(tx.x) ? 1u : 0u);
      cy[e] = ty.y + (v.y > __uint_as_float(ty.x) ? 1u : 0u);
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t* c = s ? cy : cx;
      uint32_t v;
      if (BITS == 4 || BITS == 2) {
        v = tq_pack2<BITS>(c[7], c[6], 0u);
        v = tq_pack2<BITS>(c[5], c[4], v);
        v = tq_pack2<BITS>(c[3], c[2], v);
        v = tq_pack2<BITS>(c[1], c[0], v);
      } else {
        const uint32_t p0 = c[0] + (c[1] << BITS), p1 = c[2] + (c[3] << BITS);
        const uint32_t p2 = c[4] + (c[5] << BITS), p3 = c[6] + (c[7] << BITS);
        v = (p0 + (p1 << (2 * BITS))) + ((p2 + (p3 << (2 * BITS))) << (4 * BITS));
      }
      acc[half + 2 * s] = v ^ cm;
    }
  }
}

// The lane's part of vector j (16 NC bytes): 32-byte loads when every vector
// is 32-byte aligned, else 16-byte loads.
template <int NC>
__device__ __forceinline__ void tq_lane_load(const uint16_t* src, bool v32, uint4 (&w)[NC]) {
  if (v32) {
#pragma unroll
    for (int k = 0; k < NC / 2; ++k) ld_nc32(src + 16 * k, w[2 * k], w[2 * k + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < NC; ++k) w[k] = ld_nc16(src + 8 * k);
  }
}

// E = 64 elements per lane for head dims 64 .. 256; E = 32 (one lane per
// vector, pairs (k, k + 16), no stride-32 stage) for head dim 32.
template <int DT, int D, int BITS, int E>
__global__ void __launch_bounds__(kTq64Threads, E == 64 ? 3 : 5) tq_encode_lanes_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / E, VPW = 32 / G, W = kTq64Threads / 32;
  constexpr int NP = E / 2, NCH = E / 8;       // pairs and 16-byte chunks of a lane
  constexpr int CB = D * BITS / 8;
  constexpr int NT = G >= 2 ? 2 : 1;           // index tables: direct (+ mirrored)
  static_assert((E == 64 && G >= 1 && G <= 4) || (E == 32 && G == 1), "head dim 32 .. 256");
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  __shared__ uint2 s_lut[NT][kLutCells * 16];
  // each warp's sign masks of its current layer, source word t (elements 2t,
  // 2t + 1) of lane position l: BF16: [l][t] bit 31 = sign of element 2t,
  // [l][NP + t] bit 31 = sign of element 2t + 1; FP16: [l][t] bits 15 and 31.
  // Rows padded by 8 words: the lanes of a vector read different banks.
  __shared__ uint32_t s_mask[W][G][2 * NP + 8];
  for (int k = threadIdx.x; k < NT * kLutCells * 16; k += blockDim.x) {
    const int t = k / (kLutCells * 16), c = (k >> 4) % kLutCells;
    s_lut[t][k % (kLutCells * 16)] =
        t ? make_uint2(__float_as_uint(p.lut_mthr[c]), p.lut_mlo[c]) : make_uint2(__float_as_uint(p.lut_thr[c]), p.lut_lo[c]);
  }
  __syncthreads();
  // this warp's masks for `layer` (lanes of position li write row li)
  auto build_masks = [&](uint32_t layer) {
    __syncwarp();  // every lane is done with the previous layer's masks
    for (uint32_t t = grp; t < (uint32_t)NP; t += VPW) {
      const uint32_t e0 = li * E + 2u * t;
      const uint32_t bits = tq_sign_word(p, layer, e0 >> 5);
      uint32_t s0 = (bits >> (e0 & 31u)) & 1u, s1 = (bits >> ((e0 + 1u) & 31u)) & 1u;
      if (G >= 2 && (li & 1u) && t >= 16u) {  // the odd lane's inputs 32..63
        s0 ^= 1u;
        s1 ^= 1u;
      }
      s_mask[warp][li][t] = DT == 1 ? s0 << 31 : (s0 << 15) | (s1 << 31);
      s_mask[warp][li][NP + t] = DT == 1 ? s1 << 31 : 0u;
    }
    __syncwarp();
  };
  uint32_t mask_layer = 0xffffffffu;
  const uint32_t lane_off = (lane & 15u) * 8u + (uint32_t)(kLutHalf * 128) - kCellMagicBits * 128u;
  const uint32_t lut_d = (uint32_t)__cvta_generic_to_shared(&s_lut[0][0]) + lane_off;
  const uint32_t lut_m = (uint32_t)__cvta_generic_to_shared(&s_lut[NT - 1][0]) + lane_off;
  const bool neg_a = tq64_run_negated<G>(li, 0), neg_b = tq64_run_negated<G>(li, 1);
  const uint32_t lut_a = neg_a ? lut_m : lut_d, lut_b = neg_b ? lut_m : lut_d;
  constexpr uint32_t kAll = BITS == 4 ? 0xffffffffu : (1u << (8 * BITS)) - 1u;
  const uint32_t cm_a = neg_a ? kAll : 0u, cm_b = neg_b ? kAll : 0u;
  const uint32_t mask_addr = (uint32_t)__cvta_generic_to_shared(&s_mask[warp][li][0]);
  const uint32_t run_a = tq64_run_start<G>(li, 0), run_b = tq64_run_start<G>(li, 1);
  const uint32_t nv = p.nv;
  const bool v32 = p.vec32 != 0;
  const float admit_ss = p.reject_abs * p.reject_abs * 0.99609375f;

  // lanes past the end of a segment load (and code, without storing) its
  // last vector, so that every lane works on admitted-or-flagged page data
  auto src_of = [&](const uint16_t* page, uint32_t j) {
    return page + vec_off(p, j < nv ? j : nv - 1u) + E * li;
  };

  // each warp codes whole segments: no CTA-wide barrier, so the warps of an
  // SM drift apart and their table lookups overlap other warps' arithmetic
  SegCursor cursor;
  warp_cursor_init(cursor, W);
  Seg cur;
  uint32_t ci = cursor_next<kEncode, true>(p, cursor, cur);
  uint4 pw[NCH];
  if (ci != 0xffffffffu) tq_lane_load(src_of(cur.page, grp), v32, pw);
  while (ci != 0xffffffffu) {
    const uint16_t* npage;  // the next segment's page: the rest of its plan is redone below
    uint32_t ni;
    {
      Seg nxt;
      ni = cursor_next<kEncode, true>(p, cursor, nxt);
      npage = nxt.page;
    }
    uint8_t* codes = cur.slot;
    uint8_t* meta = cur.slot + (uint64_t)nv * CB;
    uint32_t flags = 0;
    const uint32_t layer = p.sign_per_layer ? cur.layer : 0u;
    if (layer != mask_layer) {
      build_masks(layer);
      mask_layer = layer;
    }
    for (uint32_t j0 = 0; j0 < nv; j0 += VPW) {
      const uint32_t j = j0 + grp;
      // source words -> pairs, sign flips on the 16-bit values (exact)
      float2 a[NP];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 m0 = lds16(mask_addr + 16u * c);
        uint4 m1 = make_uint4(0, 0, 0, 0);
        if (DT == 1) m1 = lds16(mask_addr + 4u * NP + 16u * c);
        const uint32_t ww[4] = {pw[c].x, pw[c].y, pw[c].z, pw[c].w};
        const uint32_t k0[4] = {m0.x, m0.y, m0.z, m0.w}, k1[4] = {m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int t = 4 * c + q;                    // elements 2t, 2t + 1
          const int P = ((2 * t) & 15) | ((t >> 4) << 4), comp = (t >> 3) & 1;
          float lo, hi;
          if (DT == 1) {
            lo = __uint_as_float(ww[q] * 65536u + k0[q]);   // + 2^31 flips the sign bit
            hi = __uint_as_float((ww[q] & 0xffff0000u) ^ k1[q]);
          } else {
            const uint32_t v = ww[q] ^ k0[q];
            lo = lo_f32<0>(v);
            hi = hi_f32<0>(v);
          }
          if (comp) {
            a[P].y = lo;
            a[P + 1].y = hi;
          } else {
            a[P].x = lo;
            a[P + 1].x = hi;
          }
        }
      }
      // the page data is in registers now: load the next vector
      if (j0 + VPW < nv) tq_lane_load(src_of(cur.page, j + VPW), v32, pw);
      else if (ni != 0xffffffffu) tq_lane_load(src_of(npage, grp), v32, pw);
      // pairwise sum of squares: in-lane index bits 0..3, then 4, then 5
      const float2 nz2 = make_float2(p.neg_zero, p.neg_zero);
      float ss;
      if constexpr (E == 64) {
        const float2 ta = PairTree<0, 16>::run(a, nz2), tb = PairTree<16, 16>::run(a, nz2);
        ss = __fadd_rn(__fadd_rn(ta.x, ta.y), __fadd_rn(tb.x, tb.y));
      } else {
        const float2 ta = PairTree<0, 16>::run(a, nz2);
        ss = __fadd_rn(ta.x, ta.y);
      }
#pragma unroll
      for (int o = 1; o < G; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      // Admission.  ss is within 2^-20 (relative) of the exact sum of
      // squares, so ss <= 0.996 reject^2 shows every |x| <= reject; a
      // nonfinite element makes ss NaN or inf.  Otherwise the warp takes the
      // exact maximum of every vector.
      if (__any_sync(0xffffffffu, !(ss <= admit_ss))) {
        float amax = 0.0f;
        uint32_t nonfinite = 0;
#pragma unroll
        for (int m = 0; m < NP; ++m) {
          nonfinite |= !isfinite(a[m].x) | !isfinite(a[m].y);
          amax = fmaxf(amax, fmaxf(fabsf(a[m].x), fabsf(a[m].y)));
        }
#pragma unroll
        for (int o = 1; o < G; o <<= 1) {
          nonfinite |= __shfl_xor_sync(0xffffffffu, nonfinite, o);
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        }
        const uint32_t vflags = nonfinite ? 1u : (amax > p.reject_abs ? 2u : 0u);
        flags |= vflags;
        if (vflags) {  // keep NaN / inf out of the arithmetic (the segment stays raw)
#pragma unroll
          for (int m = 0; m < NP; ++m) a[m] = make_float2(0.0f, 0.0f);
        }
      }
      const float n = __fsqrt_rn(ss);
      float r = __frcp_rn(n);
      if (!isfinite(r)) r = 0.0f;
      // u = x r, rounded on its own.  A packed product whose result feeds
      // packed additions is fused with them into packed FMAs by the compiler
      // (measured on sm_103a, with contraction disabled and with an explicit
      // .rn modifier alike), which changes the roundings of the first
      // butterfly stage.  An FMA with a -0 addend is the same single
      // rounding of x r, zero signs included, and cannot be fused further as
      // long as the compiler cannot see that the addend is -0: it comes from
      // the launch parameters.
      const float2 r2 = make_float2(r, r);
#pragma unroll
      for (int m = 0; m < NP; ++m) a[m] = fma2(a[m], r2, nz2);
      // Walsh-Hadamard butterflies, ascending stride
#pragma unroll
      for (int h = 1; h < 16; h <<= 1) {  // strides 1, 2, 4, 8: pair P with pair P + h
#pragma unroll
        for (int m = 0; m < NP; ++m) {
          if (m & h) continue;
          const float2 u = a[m], v = a[m + h];
          a[m] = add2(u, v);
          a[m + h] = sub2(u, v);
        }
      }
#pragma unroll
      for (int m = 0; m < NP; ++m) {  // stride 16: inside each pair
        const float u = a[m].x, v = a[m].y;
        a[m] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
      }
      if constexpr (E == 64) {
#pragma unroll
        for (int m = 0; m < 16; ++m) {  // stride 32: pair P with pair P + 16
          const float2 u = a[m], v = a[m + 16];
          a[m] = add2(u, v);
          a[m + 16] = sub2(u, v);
        }
      }
      if constexpr (G == 2) {  // stride 64: lanes li, li ^ 1 (split, see above)
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 rv = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 1),
                                        __shfl_xor_sync(0xffffffffu, a[16 + m].y, 1));
          const float2 k = a[m];
          a[m] = add2(k, rv);
          a[16 + m] = sub2(k, rv);
        }
      }
      if constexpr (G == 4) {
        // stride 64 as above, except that lanes 2 and 3 put the differences
        // in pairs 0..15 and the sums in 16..31 (rv * t + k with t = -1 is the
        // single rounding of k - rv); stride 128 (lanes li, li ^ 2) then pairs
        // 0..15 of the lower lane with 16..31 of the upper one, split alike.
        const float t = (li & 2u) ? -1.0f : 1.0f;
        const float2 t2 = make_float2(t, t), nt2 = make_float2(-t, -t);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 rv = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 1),
                                        __shfl_xor_sync(0xffffffffu, a[16 + m].y, 1));
          const float2 k = a[m];
          a[m] = fma2(rv, t2, k);
          a[16 + m] = fma2(rv, nt2, k);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 rv = make_float2(__shfl_xor_sync(0xffffffffu, a[16 + m].x, 2),
                                        __shfl_xor_sync(0xffffffffu, a[16 + m].y, 2));
          const float2 k = a[m];
          a[m] = add2(k, rv);
          a[16 + m] = sub2(k, rv);
        }
      }
      if (n < 0x1p-62f) {
        // Norms this small may come from squares that underflowed, so |w|
        // can exceed sqrt(D); clamp into the table (beyond +-17 every code
        // is already the first or the last).
#pragma unroll
        for (int m = 0; m < NP; ++m)
          a[m] = make_float2(fminf(fmaxf(a[m].x, -17.0f), 17.0f), fminf(fmaxf(a[m].y, -17.0f), 17.0f));
      }
      uint32_t acc_a[4], acc_b[4];
      tq_run_codes<BITS, 0>(a, lut_a, cm_a, acc_a);
      if constexpr (E == 64) tq_run_codes<BITS, 1>(a, lut_b, cm_b, acc_b);
      if (j < nv) {
        uint8_t* vc = codes + (uint64_t)j * CB;
        tq_store32<BITS>(vc + run_a * BITS / 8, acc_a);
        if constexpr (E == 64) tq_store32<BITS>(vc + run_b * BITS / 8, acc_b);
        if (li == 0)
          st_u16(meta + (uint64_t)j * 2, __half_as_ushort(__float2half_rn(n)));
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    for (uint64_t b = (uint64_t)nv * (CB + 2) + lane; b < p.seg_bytes[cur.role]; b += 32) st_u8(cur.slot + b, 0);
    if (lane == 0)
      st_u8(p.status + ci, (flags & 1u) ? KV_SEG_RAW_NONFINITE : (flags & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED);
    if (ni != 0xffffffffu) cur = plan_segment(p, ni, kEncode);
    ci = ni;
  }
}

// Decoder for D >= 64, the same lane layout as tq_encode64_kernel.  Lane li
// reads the codes of elements 64 li .. 64 li + 63.  The odd lane's inputs
// 32..63 are negated by complementing their codes (the codebook is symmetric:
// centroid[c] = -centroid[2^b - 1 - c], exactly), and its negated
// differences are corrected by its output sign masks.
template <int DT, int D, int BITS>
__global__ void __launch_bounds__(kTq64Threads, 4) tq_decode64_kernel(const __grid_constant__ Params p) {
  constexpr int E = 64, G = D / E, VPW = 32 / G, W = kTq64Threads / 32;
  constexpr int CB = D * BITS / 8;
  constexpr int NW = 2 * BITS;                  // code words of a lane (64 codes)
  constexpr int NPAIR = 1 << (2 * BITS);        // table of two consecutive codes
  constexpr int REP = 16;                       // copies: each lane of a half warp has its own banks
  static_assert(G >= 1 && G <= 4, "head dim 64 .. 256");
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  // each warp's output sign masks of its current layer: row l, chunk c
  __shared__ uint4 s_sign[W][4][9];
  // (centroid[lo code], centroid[hi code]) for every pair of codes, REP copies;
  // 2-bit codes: the four centroids of every code byte instead, REPQ copies
  // (a quarter warp's eight 16-byte reads then fall in distinct banks)
  constexpr int REPQ = 8;
  __shared__ float2 s_pair[BITS == 2 ? 1 : NPAIR * REP];
  __shared__ float4 s_quad[BITS == 2 ? 256 * REPQ : 1];
  // D = 64 (one lane per vector): 16 restored vectors of each warp at a time,
  // 128 bytes a row, 16-byte chunk q of row r at position q ^ (r & 7)
  __shared__ uint4 s_out[G == 1 ? W : 1][G == 1 ? 16 : 1][8];
  auto build_signs = [&](uint32_t layer) {
    __syncwarp();  // every lane is done with the previous layer's masks
    for (uint32_t q = lane; q < (uint32_t)G * 32u; q += 32u) {
      // word k4 of output chunk c of lane l: elements A + 8c (c < 4) or B + 8(c - 4), + 2 k4
      const uint32_t l = q / 32u, c = (q % 32u) / 4u, k4 = q % 4u;
      const uint32_t e0 = tq64_run_start<G>(l, c < 4 ? 0 : 1) + 8u * (c & 3u) + 2u * k4;
      uint32_t m = sign_mask_word(tq_sign_word(p, layer, e0 >> 5), (int)((e0 & 31u) >> 1));
      if (tq64_run_negated<G>(l, c < 4 ? 0 : 1)) m ^= 0x80008000u;  // negated runs
      reinterpret_cast<uint32_t*>(&s_sign[warp][l][c])[k4] = m;
    }
    __syncwarp();
  };
  uint32_t sign_layer = 0xffffffffu;
  if (BITS == 2) {
    for (int k = threadIdx.x; k < 256 * REPQ; k += blockDim.x) {
      const int v = k / REPQ;
      s_quad[k] = make_float4(p.cent[v & 3], p.cent[(v >> 2) & 3], p.cent[(v >> 4) & 3], p.cent[v >> 6]);
    }
  } else {
    for (int k = threadIdx.x; k < NPAIR * REP; k += blockDim.x) {
      const int v = k / REP;
      s_pair[k] = make_float2(p.cent[v & ((1 << BITS) - 1)], p.cent[v >> BITS]);
    }
  }
  __syncthreads();
  const uint32_t pair_base = BITS == 2 ? (uint32_t)__cvta_generic_to_shared(s_quad) + (lane % REPQ) * 16u
                                       : (uint32_t)__cvta_generic_to_shared(s_pair) + (lane % REP) * 8u;
  const uint32_t sign_addr = (uint32_t)__cvta_generic_to_shared(&s_sign[warp][li][0]);
  const uint32_t run_a = tq64_run_start<G>(li, 0), run_b = tq64_run_start<G>(li, 1);
  const uint32_t cmask = (G >= 2 && (li & 1u)) ? 0xffffffffu : 0u;  // complement the upper codes
  const bool vec32 = p.vec32 != 0;
  // one lane per vector and the warp's vectors side by side in the page:
  // stage them and store 1 KB runs (8 cache lines a store instead of 32)
  const bool stage_out = G == 1 && vec32 && p.heads_contig != 0 && p.sh == (int64_t)D;
  const float cD = p.wht_scale;
  const float2 cD2 = make_float2(cD, cD);
  const uint32_t nv = p.nv;
  const uint32_t jw = grp;  // one warp per segment: this lane's first vector

  // codes and norm of vector j of segment s (registers; issued ahead of use)
  auto fetch = [&](const Seg& s, uint32_t j, uint32_t (&cw)[NW], uint16_t& n16) {
#pragma unroll
    for (int k = 0; k < NW; ++k) cw[k] = 0;
    n16 = 0;
    if (j < nv) {
      const uint8_t* vc = s.slot + (uint64_t)j * CB + 8 * BITS * li;
      if (BITS == 3) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const uint2 t = ld_nc8(vc + 8 * k);
          cw[2 * k] = t.x;
          cw[2 * k + 1] = t.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
          const uint4 t = ld_nc16(vc + 16 * k);
          cw[4 * k] = t.x; cw[4 * k + 1] = t.y; cw[4 * k + 2] = t.z; cw[4 * k + 3] = t.w;
        }
      }
      n16 = ld_nc2(s.slot + (uint64_t)nv * CB + (uint64_t)j * 2);
    }
  };

  SegCursor cursor;
  warp_cursor_init(cursor, W);
  Seg cur;
  uint32_t ci = cursor_next<kDecode, true>(p, cursor, cur);
  uint32_t cwn[NW];
  uint16_t nn = 0;
#pragma unroll
  for (int k = 0; k < NW; ++k) cwn[k] = 0;
  if (ci != 0xffffffffu) fetch(cur, jw, cwn, nn);
  while (ci != 0xffffffffu) {
    Seg nxt;
    const uint32_t ni = cursor_next<kDecode, true>(p, cursor, nxt);
    uint16_t* page = const_cast<uint16_t*>(cur.page);
    const uint32_t layer = p.sign_per_layer ? cur.layer : 0u;
    if (layer != sign_layer) {
      build_signs(layer);
      sign_layer = layer;
    }
    for (uint32_t j0 = 0; j0 < nv; j0 += VPW) {
      const uint32_t j = j0 + grp;
      uint32_t cw[NW];
#pragma unroll
      for (int k = 0; k < NW; ++k) cw[k] = k < NW / 2 ? cwn[k] : cwn[k] ^ cmask;
      const uint16_t n16 = nn;
      if (j0 + VPW < nv) fetch(cur, j + VPW, cwn, nn);
      else if (ni != 0xffffffffu) fetch(nxt, jw, cwn, nn);
      float2 a[32];
      if (BITS == 2) {  // code byte q: elements 4q .. 4q + 3
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t v = __byte_perm(cw[q >> 2], 0, 0x4440 | (q & 3));
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(a[2 * q].x), "=f"(a[2 * q].y), "=f"(a[2 * q + 1].x), "=f"(a[2 * q + 1].y)
                       : "r"(v * (16u * REPQ) + pair_base));
        }
      } else {
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          uint32_t v;
          if (BITS == 4) {
            v = __byte_perm(cw[m >> 2], 0, 0x4440 | (m & 3));
          } else {
            const int bit = 6 * m;
            v = (bit & 31) <= 26 ? (cw[bit >> 5] >> (bit & 31)) & 63u
                                 : __funnelshift_r(cw[bit >> 5], cw[(bit >> 5) + 1], bit & 31) & 63u;
          }
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a[m].x), "=f"(a[m].y) : "r"(v * (8u * REP) + pair_base));
        }
      }
      const float nc = __fsqrt_rn(vector_sumsq<G>(a));
      const float g = __fdiv_rn(__half2float(__ushort_as_half(n16)), nc);
      const float2 g2 = make_float2(g, g);
      // D = 64, 256: 1/sqrt(D) is a power of two, and neither t * (1/sqrt(D))
      // (|t| >= 2^-30 or 0: sums of centroids) nor (1/sqrt(D)) * g
      // (g >= 2^-26) leaves the normal range, so both products are exact and
      // RN(RN(t / sqrt(D)) * g) = RN(t * (g / sqrt(D))): one multiply.
      constexpr bool kPow2Scale = D == 64 || D == 256;
      const float2 gc2 = make_float2(__fmul_rn(g, cD), __fmul_rn(g, cD));
      butterflies64<G, false>(a, li);
      uint32_t o[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 m = lds16(sign_addr + 16u * c);
        const uint32_t mk[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 t = kPow2Scale ? mul2(a[4 * c + k], gc2) : mul2(mul2(a[4 * c + k], cD2), g2);
          o[4 * c + k] = pack2<DT>(t.x, t.y) ^ mk[k];
        }
      }
      if (G == 1 && stage_out && j0 + VPW <= nv) {
        uint16_t* base = page + vec_off(p, j0);  // the warp's 32 vectors, 64 elements apart
#pragma unroll
        for (uint32_t half = 0; half < 2; ++half) {
          __syncwarp();  // the previous reads of the stage are done
          if ((lane >> 4) == half) {
            const uint32_t r = lane & 15u;
#pragma unroll
            for (uint32_t q = 0; q < 8; ++q)
              s_out[G == 1 ? warp : 0][G == 1 ? r : 0][q ^ (r & 7u)] =
                  make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
          __syncwarp();
#pragma unroll
          for (uint32_t kk = 0; kk < 2; ++kk) {  // rows 8 kk .. 8 kk + 7, four lanes a row
            const uint32_t r = 8u * kk + (lane >> 2), c = 2u * (lane & 3u);
            const uint4 lo = s_out[G == 1 ? warp : 0][G == 1 ? r : 0][c ^ (r & 7u)];
            const uint4 hi = s_out[G == 1 ? warp : 0][G == 1 ? r : 0][(c + 1u) ^ (r & 7u)];
            st32(base + (uint64_t)(16u * half + r) * D + 8u * c, lo, hi);
          }
        }
      } else if (j < nv) {
        uint16_t* dst = page + vec_off(p, j);
        if (vec32) {  // 32 bytes per store: twice the bytes per line of each warp store
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            st32(dst + run_a + 8 * c, make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]),
                 make_uint4(o[4 * c + 4], o[4 * c + 5], o[4 * c + 6], o[4 * c + 7]));
            st32(dst + run_b + 8 * c, make_uint4(o[16 + 4 * c], o[17 + 4 * c], o[18 + 4 * c], o[19 + 4 * c]),
                 make_uint4(o[20 + 4 * c], o[21 + 4 * c], o[22 + 4 * c], o[23 + 4 * c]));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            st16(dst + run_a + 8 * c, make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
            st16(dst + run_b + 8 * c, make_uint4(o[16 + 4 * c], o[17 + 4 * c], o[18 + 4 * c], o[19 + 4 * c]));
          }
        }
      }
    }
    if (lane == 0 && p.result) st_u8(p.result + ci, KV_SEG_ENCODED);
    cur = nxt;
    ci = ni;
  }
}

template <int DT, int D, int BITS>
__global__ void __launch_bounds__(kThreads, 3) tq_decode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kTqE, VPW = 32 / G, W = kThreads / 32;
  constexpr int CB = D * BITS / 8;
  constexpr int NPAIR = 1 << (2 * BITS);        // table of two consecutive codes
  constexpr int REP = 16;                       // copies: each lane of a half warp has its own banks
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  // each warp's output sign masks of its current layer: row li, group c covers
  // the 8 elements from split_group_start<G>(li, c)
  __shared__ uint4 s_sign[W][G][5];
  // (centroid[lo code], centroid[hi code]) for every pair of codes, REP copies;
  // 2-bit codes: the four centroids of every code byte instead, REPQ copies
  // (a quarter warp's eight 16-byte reads then fall in distinct banks)
  constexpr int REPQ = 8;
  __shared__ float2 s_pair[BITS == 2 ? 1 : NPAIR * REP];
  __shared__ float4 s_quad[BITS == 2 ? 256 * REPQ : 1];
  auto build_signs = [&](uint32_t layer) {
    __syncwarp();  // every lane is done with the previous layer's masks
    for (uint32_t q = lane; q < (uint32_t)G * 16u; q += 32u) {
      const uint32_t l = q / 16u, c = (q % 16u) / 4u, k4 = q % 4u;
      const uint32_t e0 = split_group_start<G>(l, (int)c) + 2u * k4;
      reinterpret_cast<uint32_t*>(&s_sign[warp][l][c])[k4] =
          sign_mask_word(tq_sign_word(p, layer, e0 >> 5), (int)((e0 & 31u) >> 1));
    }
    __syncwarp();
  };
  uint32_t sign_layer = 0xffffffffu;
  if (BITS == 2) {
    for (int k = threadIdx.x; k < 256 * REPQ; k += blockDim.x) {
      const int v = k / REPQ;
      s_quad[k] = make_float4(p.cent[v & 3], p.cent[(v >> 2) & 3], p.cent[(v >> 4) & 3], p.cent[v >> 6]);
    }
  } else {
    for (int k = threadIdx.x; k < NPAIR * REP; k += blockDim.x) {
      const int v = k / REP;
      s_pair[k] = make_float2(p.cent[v & ((1 << BITS) - 1)], p.cent[v >> BITS]);
    }
  }
  __syncthreads();
  const uint32_t pair_base = BITS == 2 ? (uint32_t)__cvta_generic_to_shared(s_quad) + (lane % REPQ) * 16u
                                       : (uint32_t)__cvta_generic_to_shared(s_pair) + (lane % REP) * 8u;
  const uint32_t sign_addr = (uint32_t)__cvta_generic_to_shared(&s_sign[warp][li][0]);
  const float cD = p.wht_scale;
  const float2 cD2 = make_float2(cD, cD);
  const uint32_t nv = p.nv;
  const uint32_t jw = grp;  // one warp per segment: this lane's first vector
  const bool vec32 = p.vec32 != 0;

  // codes and norm of vector j of segment s (registers; issued ahead of use)
  auto fetch = [&](const Seg& s, uint32_t j, uint32_t (&cw)[4], uint16_t& n16) {
    cw[0] = cw[1] = cw[2] = cw[3] = 0;
    n16 = 0;
    if (j < nv) {
      const uint8_t* vc = s.slot + (uint64_t)j * CB;
      if (BITS == 4) {
        const uint4 t = ld_nc16(vc + 16 * li);
        cw[0] = t.x; cw[1] = t.y; cw[2] = t.z; cw[3] = t.w;
      } else if (BITS == 2) {
        const uint2 t = ld_nc8(vc + 8 * li);
        cw[0] = t.x; cw[1] = t.y;
      } else {
        cw[0] = ld_nc4(vc + 12 * li);
        cw[1] = ld_nc4(vc + 12 * li + 4);
        cw[2] = ld_nc4(vc + 12 * li + 8);
      }
      n16 = ld_nc2(s.slot + (uint64_t)nv * CB + (uint64_t)j * 2);
    }
  };

  SegCursor cursor;
  warp_cursor_init(cursor, W);
  Seg cur;
  uint32_t ci = cursor_next<kDecode, true>(p, cursor, cur);
  uint32_t cwn[4] = {0, 0, 0, 0};
  uint16_t nn = 0;
  if (ci != 0xffffffffu) fetch(cur, jw, cwn, nn);
  while (ci != 0xffffffffu) {
    Seg nxt;
    const uint32_t ni = cursor_next<kDecode, true>(p, cursor, nxt);
    uint16_t* page = const_cast<uint16_t*>(cur.page);
    const uint32_t layer = p.sign_per_layer ? cur.layer : 0u;
    if (layer != sign_layer) {
      build_signs(layer);
      sign_layer = layer;
    }
    for (uint32_t j0 = 0; j0 < nv; j0 += VPW) {
      const uint32_t j = j0 + grp;
      const uint32_t cw[4] = {cwn[0], cwn[1], cwn[2], cwn[3]};
      const uint16_t n16 = nn;
      if (j0 + VPW < nv) fetch(cur, j + VPW, cwn, nn);
      else if (ni != 0xffffffffu) fetch(nxt, jw, cwn, nn);
      float2 a[16];
      if (BITS == 2) {  // code byte q: elements 4q .. 4q + 3
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t v = __byte_perm(cw[q >> 2], 0, 0x4440 | (q & 3));
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(a[2 * q].x), "=f"(a[2 * q].y), "=f"(a[2 * q + 1].x), "=f"(a[2 * q + 1].y)
                       : "r"(v * (16u * REPQ) + pair_base));
        }
      } else {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          uint32_t v;
          if (BITS == 4) {
            v = __byte_perm(cw[m >> 2], 0, 0x4440 | (m & 3));
          } else {
            const int bit = 6 * m;
            v = __funnelshift_r(cw[bit >> 5], cw[(bit >> 5) + 1], bit & 31) & 63u;
          }
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a[m].x), "=f"(a[m].y) : "r"(v * (8u * REP) + pair_base));
        }
      }
      const float nc = __fsqrt_rn(vector_sumsq<G>(a));
      const float g = __fdiv_rn(__half2float(__ushort_as_half(n16)), nc);
      const float2 g2 = make_float2(g, g);
      butterflies_split<G>(a, li);
      uint32_t o[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 m = lds16(sign_addr + 16u * c);
        const uint32_t mk[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 t = mul2(mul2(a[4 * c + k], cD2), g2);
          o[4 * c + k] = pack2<DT>(t.x, t.y) ^ mk[k];
        }
      }
      if (j < nv) {
        uint16_t* dst = page + vec_off(p, j);
        if (vec32) {  // groups 2c, 2c + 1 are 16 consecutive elements starting on a 16-element boundary
#pragma unroll
          for (int c = 0; c < 4; c += 2)
            st32(dst + split_group_start<G>(li, c), make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]),
                 make_uint4(o[4 * c + 4], o[4 * c + 5], o[4 * c + 6], o[4 * c + 7]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st16(dst + split_group_start<G>(li, c), make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
        }
      }
    }
    if (lane == 0 && p.result) st_u8(p.result + ci, KV_SEG_ENCODED);
    cur = nxt;
    ci = ni;
  }
}

template <int DT, int D, int BITS>
int encode(const Params& p, void* stream) {
  constexpr int E = D >= 64 ? 64 : 32;
  return launch_codec_kernel(tq_encode_lanes_kernel<DT, D, BITS, E>, p, stream, 8, kTq64Threads, true);
}

template <int DT, int D, int BITS>
int decode(const Params& p, void* stream) {
  if constexpr (D >= 64)
    return launch_codec_kernel(tq_decode64_kernel<DT, D, BITS>, p, stream, 8, kTq64Threads, true);
  else
    return launch_codec_kernel(tq_decode_kernel<DT, D, BITS>, p, stream, 8, kThreads, true);
}

template <int DT, int D>
int dispatch_bits(const Params& p, int dir, uint32_t codec, void* stream) {
  const bool enc = dir == kEncode;
  switch (codec) {
    case KV_CODEC_TQ2:
      return enc ? encode<DT, D, 2>(p, stream) : decode<DT, D, 2>(p, stream);
    case KV_CODEC_TQ3:
      return enc ? encode<DT, D, 3>(p, stream) : decode<DT, D, 3>(p, stream);
    case KV_CODEC_TQ4:
      return enc ? encode<DT, D, 4>(p, stream) : decode<DT, D, 4>(p, stream);
  }
  return KV_ERR_INVALID_ARG;
}

template <int DT>
int dispatch_dim(const Params& p, int dir, uint32_t codec, void* stream) {
  switch (p.D) {
    case 32: return dispatch_bits<DT, 32>(p, dir, codec, stream);
    case 64: return dispatch_bits<DT, 64>(p, dir, codec, stream);
    case 128: return dispatch_bits<DT, 128>(p, dir, codec, stream);
    case 256: return dispatch_bits<DT, 256>(p, dir, codec, stream);
  }
  return KV_ERR_UNSUPPORTED_HEAD_DIM;
}

}  // namespace

int launch_turboquant(const Params& p, int dir, uint32_t codec, void* stream) {
  return p.dtype == KV_DT_FP16 ? dispatch_dim<0>(p, dir, codec, stream)
                               : dispatch_dim<1>(p, dir, codec, stream);
}

}  // namespace kvc
