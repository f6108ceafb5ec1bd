// uniform.cu -- per-vector uniform quantization with FP16 minimum and step.
//
// "KV precision and storage encoding" (OrbitKV), section "FP8 and TurboQuant":
// V uses per-vector uniform quantization with an FP16 minimum and scale
// (3 and 4 bits on the page; 2 and 8 bits here as well).
// Per vector: m = fp16(min x), s = fp16((max x - min x) / (2^b - 1)), codes
// clamp(rint((x - m) / s), 0, 2^b - 1) against the stored (rounded) m and s,
// code 0 when s == 0; restore code * s + m.  Codes are a little-endian bit
// stream (b = 2, 3, 4) or one byte each (b = 8); metadata is (m, s) as two FP16.
#include "crc_common.cuh"

namespace kvc {
namespace {

#define LV(b) ((1u << (b)) - 1u)

constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4b400000u;
constexpr int kEncodeCtas = 5;  // resident CTAs per SM (see launch_codec_kernel)
constexpr int kDecodeCtas = 5;

// Codes of 8 elements: clamp(rint((x - m) / s), 0, L).  The quotient is
// correctly rounded (q0 = RN(d r), e = RN(d - q0 s) exact, q = RN(q0 + e r));
// clamping to [0, L] before rounding gives the same integer (0 and L are
// integers), and RN(q + 1.5 * 2^23) holds rint(q) in its low byte, which is
// what t[] returns (the higher bits are the magic's).  The caller passes r = 0
// when s == 0, which makes every quotient 0.
//
// SAT (2, 4 and 8 bits): t[] is rint(q) itself, unclamped, as a signed
// integer, and the saturating packs (pack_codes8) clamp it.  Admitted vectors
// have |x| <= 448, so |m - min| <= 0.125 (half the FP16 spacing below 512)
// and s >= 2^-24 whenever s != 0; hence |q| <= 0.125 * 2^24 + 1.5 L < 2^22,
// the range in which RN(q + 1.5 * 2^23) - 1.5 * 2^23 is rint(q).  (Codes of
// vectors that fail admission are never used: their segment stays raw.)
template <uint32_t LEVELS, bool SAT>
__device__ __forceinline__ void uniform_codes8(const float (&x)[8], float m, float sc, float r,
                                               uint32_t (&t)[8]) {
  const float2 m2 = make_float2(m, m), ns2 = make_float2(-sc, -sc), r2 = make_float2(r, r);
  const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 d = sub2(make_float2(x[e], x[e + 1]), m2);
    const float2 q0 = mul2(d, r2);
    const float2 res = fma2(q0, ns2, d);
    float2 q = fma2(res, r2, q0);
    if (!SAT) {
      q.x = fminf(fmaxf(q.x, 0.0f), (float)LEVELS);
      q.y = fminf(fmaxf(q.y, 0.0f), (float)LEVELS);
    }
    const float2 v = add2(q, mg2);
    t[e] = __float_as_uint(v.x) - (SAT ? kRoundMagicBits : 0u);
    t[e + 1] = __float_as_uint(v.y) - (SAT ? kRoundMagicBits : 0u);
  }
}

// (c << 2 BITS) | (sat(a) << BITS) | sat(b), with a and b signed and sat the
// clamp to [0, 2^BITS - 1]
template <int BITS>
__device__ __forceinline__ uint32_t pack_sat(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if (BITS == 8) asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else if (BITS == 4) asm("cvt.pack.sat.u4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else asm("cvt.pack.sat.u2.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Codes of 8 elements (t[] from uniform_codes8) as the little-endian bit
// stream of BITS-bit codes: 8 bytes (BITS = 8) or the low 8 * BITS bits.
// 2, 4 and 8 bits: saturating packs, two codes each; 3 bits: the clamped
// codes' low bits shifted into place.
template <int BITS>
__device__ __forceinline__ uint2 pack_codes8(const uint32_t (&t)[8]) {
  if (BITS == 8)
    return make_uint2(pack_sat<8>(t[1], t[0], pack_sat<8>(t[3], t[2], 0u)),
                      pack_sat<8>(t[5], t[4], pack_sat<8>(t[7], t[6], 0u)));
  if (BITS == 4 || BITS == 2) {
    uint32_t v = pack_sat<BITS>(t[7], t[6], 0u);
    v = pack_sat<BITS>(t[5], t[4], v);
    v = pack_sat<BITS>(t[3], t[2], v);
    return make_uint2(pack_sat<BITS>(t[1], t[0], v), 0u);
  }
  uint32_t v = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) v |= (t[e] & ((1u << BITS) - 1u)) << (BITS * e);
  return make_uint2(v, 0u);
}

// (max - min) / L correctly rounded, from the rounded reciprocal of L
template <uint32_t LEVELS>
__device__ __forceinline__ float div_levels(float range) {
  constexpr float L = (float)LEVELS;
  constexpr float rL = 1.0f / (float)LEVELS;
  const float q0 = __fmul_rn(range, rL);
  const float e = __fmaf_rn(-q0, L, range);
  return __fmaf_rn(e, rL, q0);
}

// Thread mapping (as for TurboQuant): lane li of a vector's G = D/32 lanes owns
// its 32 contiguous elements [32 li, 32 li + 32) as four 16-byte chunks, so the
// per-vector work (minimum / maximum over G lanes, the FP16 metadata, the
// step's reciprocal) is shared by few lanes and every lane packs and stores its
// own 32 codes (4 * BITS bytes) in one piece.
constexpr int kUniE = 32;

// Little-endian stream of a lane's 32 codes (four chunks of 8), stored at
// `dst` (4 * BITS bytes, aligned to that size for BITS = 2, 4, 8 and to 4
// bytes for BITS = 3).
template <int BITS>
__device__ __forceinline__ void store_codes32(uint8_t* dst, const uint2 (&v)[4]) {
  if (BITS == 8) {
    st16(dst, make_uint4(v[0].x, v[0].y, v[1].x, v[1].y));
    st16(dst + 16, make_uint4(v[2].x, v[2].y, v[3].x, v[3].y));
  } else if (BITS == 4) {
    st16(dst, make_uint4(v[0].x, v[1].x, v[2].x, v[3].x));
  } else if (BITS == 2) {
    st8(dst, make_uint2(v[0].x | (v[1].x << 16), v[2].x | (v[3].x << 16)));
  } else {  // 4 x 24 bits -> three words
    st4(dst, v[0].x | (v[1].x << 24));
    st4(dst + 4, (v[1].x >> 8) | (v[2].x << 16));
    st4(dst + 8, (v[2].x >> 16) | (v[3].x << 8));
  }
}

// 8-bit codes: the chunk layout of the FP8 kernels (G lanes of a vector take
// its 16-byte chunks round-robin), so each lane's 8-byte code stores and each
// warp's loads stay coalesced.  Q selects the variant (NoSeal / WarpSeg /
// CrcParams).  The sealing encoder is the FP8 one's scheme: a step
// of one warp writes 1 KB of codes, and at the start of every second step,
// with that step's loads in flight, the warp folds the 2 KB CRC row its last
// two steps wrote (re-read from L2) and prefetches the vectors two steps
// ahead into L2; the rows left after the last step and the header follow.
template <int DT, int D, int BITS, int NT, typename Q>
__global__ void __launch_bounds__(Variant<Q, NT>::kCtaThreads)
    uniform_encode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q, NT>::kSeal, WARP = Variant<Q, NT>::kWarp;
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = M::U, W = Variant<Q, NT>::kCtaThreads / 32;
  constexpr uint32_t STEP = WARP ? VPW * U : W * VPW * U;
  constexpr uint32_t LEVELS = (1u << BITS) - 1u;
  constexpr int CB = D * BITS / 8;  // code bytes per vector
  static_assert(!SEAL || (BITS == 8 && VPW * U * CB == kCrcRow / 2), "a sealing step writes half a CRC row");
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t j_first = WARP ? 0u : warp * VPW * U;
  __shared__ uint32_t s_flag[2];
  crc::NibbleTables* t = nullptr;
  uint32_t tb = 0;
  uint32_t i = blockIdx.x, i_step = gridDim.x;  // no wrap: n_segments < 2^31
  if constexpr (WARP) {
    if constexpr (SEAL) tb = crc::load_tables(q, t);
    SegCursor c;
    warp_cursor_init(c, W);
    i = c.base;
    i_step = c.stride;
  } else {
    if (threadIdx.x < 2) s_flag[threadIdx.x] = 0;
    __syncthreads();
  }
  const uint32_t nv = p.nv;
  int it = 0;
  for (; i < p.n_segments; i += i_step) {
    const Seg s = plan_segment(p, i, kEncode);
    if (s.action != kProcess) {
      if constexpr (WARP) {
        if (s.action == kReport) {
          if (lane == 0) st_u8(p.status + i, s.status);
          if constexpr (SEAL) crc::seal_segment<true>(q, *t, tb, i, s.status, lane);
        }
      } else {
        if (s.action == kReport && threadIdx.x == 0) st_u8(p.status + i, s.status);
      }
      continue;
    }
    if (!WARP && threadIdx.x == 0) s_flag[(it + 1) & 1] = 0;
    uint8_t* codes = s.slot;
    uint8_t* meta = s.slot + (uint64_t)nv * CB;
    uint32_t flags = 0;
    uint32_t crc_s = 0, crc_m = 0;  // sealing: rows folded so far, and their register
    const bool al32 = ((uintptr_t)s.slot & 31u) == 0;
    for (uint32_t j0 = j_first, k = 0; j0 < nv; j0 += STEP, ++k) {
      uint4 w[U][NC];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const uint16_t* src = s.page + (j < nv ? vec_off(p, j) : 0);
#pragma unroll
        for (int c = 0; c < NC; ++c)
          w[u][c] = j < nv ? ld_stream16<SEAL>(src + 8 * (li + G * c)) : make_uint4(0, 0, 0, 0);
      }
      if constexpr (SEAL) {
        const uint32_t jn = j0 + 2u * STEP + lane;
        if (lane < STEP && jn < nv) prefetch_l2(s.page + vec_off(p, jn), D * 2);
        if (k >= 2u && (k & 1u) == 0u) {
          __syncwarp();
          crc_s = crc::fold_row<false>(*t, tb, s.slot, crc_m, al32, crc_s, lane);
          ++crc_m;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        float mn, mx;
        vec_minmax<DT, G, NC>(w[u], mn, mx);
        flags |= admission(mn, mx, p.reject_abs);
        mn = __fadd_rn(mn, 0.0f);  // a zero minimum / maximum is +0
        mx = __fadd_rn(mx, 0.0f);
        const __half m16 = __float2half_rn(mn);
        const __half s16 = __float2half_rn(div_levels<LEVELS>(__fsub_rn(mx, mn)));
        const float m = __half2float(m16), sc = __half2float(s16);
        const float r = sc == 0.0f ? 0.0f : __frcp_rn(sc);
        const bool in = j < nv;
        uint8_t* vc = codes + (uint64_t)j * CB;
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) {
          const uint32_t cidx = li + G * ch;
          float x[8];
          unpack8<DT>(w[u][ch], x);
          uint32_t t[8];
          uniform_codes8<LEVELS, BITS != 3>(x, m, sc, r, t);
          const uint2 v = pack_codes8<BITS>(t);
          if (BITS == 8) {
            if (in) st8(vc + 8 * cidx, v);
          } else if (BITS == 4) {
            if (in) st4(vc + 4 * cidx, v.x);
          } else if (BITS == 2) {
            if (in) st_u16(vc + 2 * cidx, (uint16_t)v.x);
          } else {
            store_3bit(vc, v.x, cidx, in);
          }
        }
        if (in && li == 0)
          st4(meta + (uint64_t)j * 4,
              (uint32_t)__half_as_ushort(m16) | ((uint32_t)__half_as_ushort(s16) << 16));
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if constexpr (WARP) {
      zero_padding(s.slot, (uint64_t)nv * (CB + 4), p.seg_bytes[s.role], lane, 32);
      const uint32_t st = status_of_flags(flags);
      __syncwarp();
      if (lane == 0) st_u8(p.status + i, (uint8_t)st);
      if constexpr (SEAL) crc::seal_segment<false>(q, *t, tb, i, st, lane, crc_m, crc_s);
    } else {
      if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
      zero_padding(s.slot, (uint64_t)nv * (CB + 4), p.seg_bytes[s.role], threadIdx.x, blockDim.x);
      __syncthreads();
      if (threadIdx.x == 0) st_u8(p.status + i, status_of_flags(s_flag[it & 1]));
      ++it;
    }
  }
}

// 2-, 3- and 4-bit codes: each lane codes its own 32 elements (see kUniE), so
// the per-vector work is shared by D/32 lanes and the lane's codes (8, 12 or
// 16 bytes) go out in one store, adjacent to its neighbours'.
template <int DT, int D, int BITS, int NT>
__global__ void __launch_bounds__(NT) uniform_encode_lanes_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kUniE, VPW = 32 / G, U = 2, W = NT / 32;
  constexpr int STEP = W * VPW * U;
  constexpr uint32_t LEVELS = (1u << BITS) - 1u;
  constexpr int CB = D * BITS / 8;        // code bytes per vector
  constexpr int LB = kUniE * BITS / 8;    // code bytes per lane
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  __shared__ uint32_t s_flag[2];
  if (threadIdx.x < 2) s_flag[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t nv = p.nv;
  const bool vec32 = p.vec32 != 0;
  int it = 0;
  for (uint32_t i = blockIdx.x; i < p.n_segments; i += gridDim.x) {
    const Seg s = plan_segment(p, i, kEncode);
    if (s.action != kProcess) {
      if (s.action == kReport && threadIdx.x == 0) st_u8(p.status + i, s.status);
      continue;
    }
    if (threadIdx.x == 0) s_flag[(it + 1) & 1] = 0;
    uint8_t* codes = s.slot;
    uint8_t* meta = s.slot + (uint64_t)nv * CB;
    uint32_t flags = 0;
    for (uint32_t j0 = warp * VPW * U; j0 < nv; j0 += STEP) {
      uint4 w[U][4];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const uint16_t* src = s.page + (j < nv ? vec_off(p, j) : 0) + kUniE * li;
        if (j >= nv) {
#pragma unroll
          for (int c = 0; c < 4; ++c) w[u][c] = make_uint4(0, 0, 0, 0);
        } else if (D >= 64 && vec32) {  // two 32-byte loads: a whole sector each (1% slower at D = 32)
          ld_nc32(src, w[u][0], w[u][1]);
          ld_nc32(src + 16, w[u][2], w[u][3]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) w[u][c] = ld_nc16(src + 8 * c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        float mn, mx;
        vec_minmax<DT, G, 4>(w[u], mn, mx);
        flags |= admission(mn, mx, p.reject_abs);
        mn = __fadd_rn(mn, 0.0f);  // a zero minimum / maximum is +0
        mx = __fadd_rn(mx, 0.0f);
        const __half m16 = __float2half_rn(mn);
        const __half s16 = __float2half_rn(div_levels<LEVELS>(__fsub_rn(mx, mn)));
        const float m = __half2float(m16), sc = __half2float(s16);
        const float r = sc == 0.0f ? 0.0f : __frcp_rn(sc);
        uint2 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float x[8];
          unpack8<DT>(w[u][c], x);
          uint32_t t[8];
          uniform_codes8<LEVELS, BITS != 3>(x, m, sc, r, t);
          v[c] = pack_codes8<BITS>(t);
        }
        if (j < nv) {
          store_codes32<BITS>(codes + (uint64_t)j * CB + LB * li, v);
          if (li == 0)
            st4(meta + (uint64_t)j * 4,
                (uint32_t)__half_as_ushort(m16) | ((uint32_t)__half_as_ushort(s16) << 16));
        }
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
    zero_padding(s.slot, (uint64_t)nv * (CB + 4), p.seg_bytes[s.role], threadIdx.x, blockDim.x);
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t f = s_flag[it & 1];
      st_u8(p.status + i, (f & 1u) ? KV_SEG_RAW_NONFINITE : (f & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED);
    }
    ++it;
  }
}

// exact float of a small unsigned integer: (2^23 + c) - 2^23
__device__ __forceinline__ float small_u2f(uint32_t c) {
  return __fsub_rn(__uint_as_float(0x4b000000u | c), 8388608.0f);
}

// ADJ (segments of kAdjacentChunkMinVectors or more, D >= 64, 2/4/8-bit codes): lane li owns the
// adjacent chunks 2 li, 2 li + 1 -- one code load and, when every vector is
// 32-byte aligned, one 32-byte store per vector (as the FP8 decoder).
//
// Q selects the variant (NoSeal / CrcParams).  The verifying decoder (8-bit
// codes) is the FP8 one's scheme: one warp per segment checks the header and
// the CRC-32 as kv_codec_verify does (loads with an L2 evict_last policy) and
// only then restores the segment, re-reading the slot from L2 last vectors
// first (loads and page stores with evict_first).
template <int DT, int D, int BITS, int NT, bool ADJ, typename Q>
__global__ void __launch_bounds__(Variant<Q, NT>::kCtaThreads)
    uniform_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q, NT>::kSeal;
  static_assert(!SEAL || BITS == 8, "verifying decoders for 8-bit codes");
  // 3-bit codes (two dependent word loads per chunk) keep twice as many
  // vectors in flight per step at D >= 64: uniform-3 decode 0.82 -> 0.84 of
  // HBM on a GB300, while 2/4/8 bits lose 1-11% that way.
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = (BITS == 3 && D >= 64 ? 2 : 1) * M::U;
  constexpr int W = Variant<Q, NT>::kCtaThreads / 32;
  constexpr uint32_t STEP = SEAL ? VPW * U : W * VPW * U;
  constexpr int CB = D * BITS / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t j_first = SEAL ? 0u : warp * VPW * U;
  const uint32_t nv = p.nv;
  const bool vec32 = p.vec32 != 0;
  crc::NibbleTables* t = nullptr;
  uint32_t tb = 0;
  uint32_t i = blockIdx.x, i_step = gridDim.x;  // no wrap: n_segments < 2^31
  uint64_t keep = 0, once = 0;
  if constexpr (SEAL) {
    tb = crc::load_tables(q, t);
    SegCursor c;
    warp_cursor_init(c, W);
    i = c.base;
    i_step = c.stride;
    keep = l2_evict_last();
    once = l2_evict_first();
  }
  for (; i < p.n_segments; i += i_step) {
    Seg s;
    if constexpr (SEAL) {
      if (!owns_segment(p, ldg_u32(&p.descs[i].role))) continue;  // another launch's: no CRC
      s = plan_segment(p, i, kDecode, (int)crc::verify_segment<true>(q, *t, tb, i, lane, keep));
      if (s.action != kProcess) {
        if (lane == 0) st_u8(p.result + i, s.status);
        continue;
      }
    } else {
      s = plan_segment(p, i, kDecode);
      if (s.action != kProcess) {
        if (s.action == kReport && threadIdx.x == 0 && p.result) st_u8(p.result + i, s.status);
        continue;
      }
    }
    const uint8_t* codes = s.slot;
    const uint8_t* meta = s.slot + (uint64_t)nv * CB;
    uint16_t* page = const_cast<uint16_t*>(s.page);
    // verifying: the steps last to first (the rows the check read last first)
    const uint32_t n_steps = SEAL ? (nv + STEP - 1u) / STEP : 0u;
    for (uint32_t kk = 0, j0 = SEAL ? (n_steps - 1u) * STEP : j_first; SEAL ? kk < n_steps : j0 < nv;
         ++kk, j0 = SEAL ? (n_steps - 1u - kk) * STEP : j0 + STEP) {
      uint2 cw[U][NC];
      uint32_t mw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const bool in = j < nv;
        const uint8_t* vc = codes + (uint64_t)j * CB;
        if (ADJ && NC == 2) {  // chunks 2 li, 2 li + 1: 2 * BITS bytes at 2 * BITS * li
          cw[u][0] = cw[u][NC - 1] = make_uint2(0, 0);
          if (in) {
            if (BITS == 8) {
              const uint4 t = ld_nc16_h<SEAL>(vc + 16 * li, once);
              cw[u][0] = make_uint2(t.x, t.y);
              cw[u][NC - 1] = make_uint2(t.z, t.w);
            } else if (BITS == 4) {
              const uint2 t = ld_nc8(vc + 8 * li);
              cw[u][0].x = t.x;
              cw[u][NC - 1].x = t.y;
            } else {
              const uint32_t t = ld_nc4(vc + 4 * li);
              cw[u][0].x = t & 0xffffu;
              cw[u][NC - 1].x = t >> 16;
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < NC; ++ch) {
            const uint32_t cidx = li + G * ch;
            cw[u][ch] = make_uint2(0, 0);
            if (in) {
              if (BITS == 8) cw[u][ch] = ld_nc8_h<SEAL>(vc + 8 * cidx, once);
              else if (BITS == 4) cw[u][ch].x = ld_nc4(vc + 4 * cidx);
              else if (BITS == 2) cw[u][ch].x = ld_nc2(vc + 2 * cidx);
              else cw[u][ch].x = load_3bit(vc, cidx);
            }
          }
        }
        mw[u] = in ? ld_nc4_h<SEAL>(meta + (uint64_t)j * 4, once) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const float m = __half2float(__ushort_as_half((unsigned short)(mw[u] & 0xffffu)));
        const float sc = __half2float(__ushort_as_half((unsigned short)(mw[u] >> 16)));
        const float2 m2 = make_float2(m, m), s2 = make_float2(sc, sc);
        uint16_t* dst = page + (j < nv ? vec_off(p, j) : 0);
        uint4 oc[NC];
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) {
          uint32_t r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t c0, c1;
            if (BITS == 8) {
              const uint32_t wd = k < 2 ? cw[u][ch].x : cw[u][ch].y;
              c0 = (wd >> (16 * (k & 1))) & 0xffu;
              c1 = (wd >> (16 * (k & 1) + 8)) & 0xffu;
            } else {
              c0 = (cw[u][ch].x >> (BITS * 2 * k)) & LV(BITS);
              c1 = (cw[u][ch].x >> (BITS * (2 * k + 1))) & LV(BITS);
            }
            const float2 y = add2(mul2(make_float2(small_u2f(c0), small_u2f(c1)), s2), m2);
            r[k] = pack2<DT>(y.x, y.y);
          }
          if (ADJ && NC == 2) oc[ch] = make_uint4(r[0], r[1], r[2], r[3]);
          else if (j < nv) st16_h<SEAL>(dst + 8 * (li + G * ch), make_uint4(r[0], r[1], r[2], r[3]), once);
        }
        if (ADJ && NC == 2 && j < nv) {
          if (vec32) {
            st32_h<SEAL>(dst + 16 * li, oc[0], oc[NC - 1], once);
          } else {
            st16_h<SEAL>(dst + 16 * li, oc[0], once);
            st16_h<SEAL>(dst + 16 * li + 8, oc[NC - 1], once);
          }
        }
      }
    }
    if constexpr (SEAL) {
      if (lane == 0) st_u8(p.result + i, KV_SEG_ENCODED);
    } else {
      if (threadIdx.x == 0 && p.result) st_u8(p.result + i, KV_SEG_ENCODED);
    }
  }
}

// Encoder segments that fit in one step of a 256-thread CTA are too short to
// keep a CTA's warps busy between its per-segment barriers.  For the lanes
// encoders they run on 128-thread CTAs, twice as many per SM (measured on the
// GB300: uniform-3/2 packed 0.64/0.62 -> 0.74/0.72 of HBM); the 8-bit encoder
// gives each such segment a warp of its own (WarpSeg, 4 CTAs of 256 threads
// per SM at its 55 registers): uniform-8 on 64-vector segments 0.70 with
// 256-thread CTAs, 0.87 with 128-thread CTAs, 0.92 with a warp per segment.
template <int DT, int D, int BITS>
int launch_encode(const Params& p, void* stream) {
  if constexpr (BITS == 8) {
    constexpr uint32_t step = 8u * ChunkMap<D>::VPW * ChunkMap<D>::U;
    if (p.nv <= step) return launch_warp(uniform_encode_kernel<DT, D, 8, kThreads, WarpSeg>, p, stream, 4);
    return launch_plain(uniform_encode_kernel<DT, D, 8, kThreads, NoSeal>, p, stream, kEncodeCtas);
  } else {
    constexpr uint32_t step = 8u * (32 / (D / kUniE)) * 2;
    if (p.nv <= step)
      return launch_codec_kernel(uniform_encode_lanes_kernel<DT, D, BITS, 128>, p, stream, 2 * kEncodeCtas, 128);
    return launch_codec_kernel(uniform_encode_lanes_kernel<DT, D, BITS, kThreads>, p, stream, kEncodeCtas);
  }
}

// (The decoders stay at 256 threads: 128-thread CTAs lose 10% on 64-vector
// segments.)
template <int DT, int D, int BITS>
int launch_decode(const Params& p, void* stream) {
  if (BITS != 3 && p.nv >= kAdjacentChunkMinVectors)
    return launch_plain(uniform_decode_kernel<DT, D, BITS, kThreads, BITS != 3, NoSeal>, p, stream, kDecodeCtas);
  return launch_plain(uniform_decode_kernel<DT, D, BITS, kThreads, false, NoSeal>, p, stream, kDecodeCtas);
}

// Uniform-8 with segment headers: the sealing encoder / verifying decoder.
template <int DT, int D>
int launch_sealed8(const Params& p, const CrcParams& q, int dir, void* stream) {
  if (dir == kEncode) return launch_sealed(uniform_encode_kernel<DT, D, 8, kThreads, CrcParams>, p, q, stream);
  if (p.nv >= kAdjacentChunkMinVectors)
    return launch_sealed(uniform_decode_kernel<DT, D, 8, kThreads, true, CrcParams>, p, q, stream);
  return launch_sealed(uniform_decode_kernel<DT, D, 8, kThreads, false, CrcParams>, p, q, stream);
}

template <int DT>
int sealed_dim(const Params& p, const CrcParams& q, int dir, void* stream) {
  switch (p.D) {
    case 32: return launch_sealed8<DT, 32>(p, q, dir, stream);
    case 64: return launch_sealed8<DT, 64>(p, q, dir, stream);
    case 128: return launch_sealed8<DT, 128>(p, q, dir, stream);
    case 256: return launch_sealed8<DT, 256>(p, q, dir, stream);
  }
  return KV_ERR_UNSUPPORTED_HEAD_DIM;
}

template <int DT, int D>
int dispatch_bits(const Params& p, int dir, uint32_t codec, void* stream) {
  const bool enc = dir == kEncode;
  switch (codec) {
    case KV_CODEC_UNIFORM2: return enc ? launch_encode<DT, D, 2>(p, stream) : launch_decode<DT, D, 2>(p, stream);
    case KV_CODEC_UNIFORM3: return enc ? launch_encode<DT, D, 3>(p, stream) : launch_decode<DT, D, 3>(p, stream);
    case KV_CODEC_UNIFORM4: return enc ? launch_encode<DT, D, 4>(p, stream) : launch_decode<DT, D, 4>(p, stream);
    case KV_CODEC_UNIFORM8: return enc ? launch_encode<DT, D, 8>(p, stream) : launch_decode<DT, D, 8>(p, stream);
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

int launch_uniform(const Params& p, int dir, uint32_t codec, void* stream) {
  return p.dtype == KV_DT_FP16 ? dispatch_dim<0>(p, dir, codec, stream)
                               : dispatch_dim<1>(p, dir, codec, stream);
}

int launch_uniform_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream) {
  if (codec != KV_CODEC_UNIFORM8) return KV_ERR_INVALID_ARG;
  return p.dtype == KV_DT_FP16 ? sealed_dim<0>(p, q, dir, stream) : sealed_dim<1>(p, q, dir, stream);
}

}  // namespace kvc
