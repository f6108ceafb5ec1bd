// fp8.cu -- FP8 E4M3FN encode / decode kernels.
//
// "Asymmetric KV: methods and results" (knlp), section "Precision and scaling
// reference": scale = max(FP32 absmax, 1e-12) * fl32(1/448); operands divided
// in FP32, clipped to +-448, rounded to E4M3FN nearest-even; dynamic mode
// applies the rule per token/head vector; codes stored as E4M3FN, scales as
// FP32.  "KV precision and storage encoding" (OrbitKV), section "FP8 and
// TurboQuant": E4M3FN nearest-even with signed zero and subnormals, hardware
// conversion on newer GPUs, segments with nonfinite or out-of-range values
// stay raw.
//
// Per element the encoder does one correctly rounded division (reciprocal of
// the vector's scale + one FMA correction) and the hardware conversion
// cvt.rn.satfinite.e4m3x2.f32, whose saturation to +-448 is the clip.
//
// Besides the plain kernels (one CTA per segment) there are sealing encoders
// and verifying decoders (one warp per segment) that give the segment
// headers' CRC-32 without a second pass over the slots in HBM: section
// "Ownership, storage and GDS" of the same OrbitKV page asks for a CRC32 per
// stored segment, checked before GPU decode.
#include "crc_common.cuh"

namespace kvc {
namespace {

constexpr float kRecip448 = 1.0f / 448.0f;  // fl32(1/448)
// Resident CTAs per SM (see launch_plain), from sweeps of 2-8 on the
// GB300: the dynamic-scale encoder (more work per vector) and the head_dim 32
// encoders want 6, the fixed-scale / cast encoders 4; the decoders 3.
template <uint32_t CODEC, int D>
constexpr int encode_ctas() { return (CODEC == KV_CODEC_FP8_DYNAMIC || D == 32) ? 6 : 4; }
constexpr int kDecodeCtas = 3;

// four floats -> four E4M3FN bytes (first element in the low byte), RNE,
// saturating to +-448 (the clip); NaN stays NaN
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t d;
  asm("{ .reg .b16 lo, hi; cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3; mov.b32 %0, {lo, hi}; }"
      : "=r"(d)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return d;
}
// four E4M3 bytes -> two f16x2 words (exact)
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& h01, uint32_t& h23) {
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo;"
      " cvt.rn.f16x2.e4m3x2 %1, hi; }"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
}

// E4M3 codes of 8 elements.  CAST: code(x).  FIXED / DYNAMIC: code(x / s),
// the quotient correctly rounded: with nr = -RN(1/s), qn = RN(x nr) = -RN(x/s)
// approximately, e = RN(x + qn s) is the exact residual x - q0 s, and
// RN(qn + e nr) = -RN(x / s) exactly; the codes of -q have the sign bits
// flipped back.  Zero inputs keep their sign through every step.
template <uint32_t CODEC>
__device__ __forceinline__ uint2 fp8_codes8(const float (&x)[8], float s, float nr) {
  if (CODEC == KV_CODEC_FP8_CAST)
    return make_uint2(e4m3x4(x[0], x[1], x[2], x[3]), e4m3x4(x[4], x[5], x[6], x[7]));
  const float2 s2 = make_float2(s, s), nr2 = make_float2(nr, nr);
  float q[8];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 xx = make_float2(x[e], x[e + 1]);
    const float2 q0n = mul2(xx, nr2);
    const float2 res = fma2(q0n, s2, xx);
    const float2 qn = fma2(res, nr2, q0n);
    q[e] = qn.x;
    q[e + 1] = qn.y;
  }
  return make_uint2(e4m3x4(q[0], q[1], q[2], q[3]) ^ 0x80808080u,
                    e4m3x4(q[4], q[5], q[6], q[7]) ^ 0x80808080u);
}

template <uint32_t CODEC, int D>
__device__ __forceinline__ uint64_t fp8_used_bytes(uint32_t nv) {
  return (uint64_t)nv * (D + (CODEC == KV_CODEC_FP8_DYNAMIC ? 4 : 0));
}

// Variants (NoSeal: the plain kernel, one CTA of kThreads per segment;
// CrcParams: one warp per segment):
//  * Sealing encoder: every encode step writes 1 KB of codes.  At the start of
//    every second step, with that step's loads in flight, the warp folds the
//    2 KB CRC row its last two steps wrote (after __syncwarp, with plain loads:
//    the bytes were just written and sit in L2) and prefetches the vectors two
//    steps ahead into L2.  The rows left after the last step follow, then the
//    header kv_codec_seal would write.
//  * Verifying decoder: checks header and CRC-32 exactly as kv_codec_verify
//    does (loads with an L2 evict_last policy) and restores the segment only
//    when they match, re-reading the slot from L2 (evict_first, like the page
//    stores) last vectors first: a damaged slot is never scattered.
// (The vector loop is written out in the kernel bodies: moved into a helper
// function it compiled to half again as many registers, which cost the plain
// encoder two of its six CTAs per SM.)

template <int DT, int D, uint32_t CODEC, typename Q>
__global__ void __launch_bounds__(Variant<Q>::kCtaThreads)
    fp8_encode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q>::kSeal;
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = M::U, W = Variant<Q>::kCtaThreads / 32;
  // a warp's vector rows: a CTA's warps interleave over the segment; a sealing
  // warp walks its segment alone
  constexpr uint32_t STEP = SEAL ? VPW * U : W * VPW * U;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t j_first = SEAL ? 0u : warp * VPW * U;
  __shared__ uint32_t s_flag[2];
  crc::NibbleTables* t = nullptr;
  uint32_t tb = 0;
  uint32_t i = blockIdx.x, i_step = gridDim.x;  // no wrap: n_segments < 2^31
  if constexpr (SEAL) {
    tb = crc::load_tables(q, t);
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
      if constexpr (SEAL) {
        if (s.action == kReport) {
          if (lane == 0) st_u8(p.status + i, s.status);
          crc::seal_segment<true>(q, *t, tb, i, s.status, lane);
        }
      } else {
        if (s.action == kReport && threadIdx.x == 0) st_u8(p.status + i, s.status);
      }
      continue;
    }
    if (!SEAL && threadIdx.x == 0) s_flag[(it + 1) & 1] = 0;
    float fixed = 1.0f;
    if (CODEC == KV_CODEC_FP8_FIXED) fixed = p.fixed_scale[s.layer][s.role];
    const float fixed_nr = -__frcp_rn(fixed);
    uint8_t* codes = s.slot;
    uint8_t* meta = s.slot + (uint64_t)nv * D;
    uint32_t flags = 0;
    // sealing: the slot's CRC rows (2 KB) folded so far into this lane's
    // register; a step writes 1 KB of codes, so row m is complete once step
    // 2m + 1 is, and is folded during the loads of step 2m + 2
    static_assert(!SEAL || VPW * U * D == kCrcRow / 2, "a step writes half a CRC row");
    uint32_t crc_s = 0, crc_m = 0;
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
        // the vectors two steps ahead into L2 meanwhile, one per lane
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
        const float amax = vec_absmax<DT, G, NC>(w[u]);
        flags |= admission_abs(amax, p.reject_abs);
        float sc = fixed, nr = fixed_nr;
        if (CODEC == KV_CODEC_FP8_DYNAMIC) {
          sc = __fmul_rn(fmaxf(amax, 1e-12f), kRecip448);
          nr = -__frcp_rn(sc);
        }
        if (CODEC == KV_CODEC_FP8_FIXED && p.fixed_reject) {
          // the vector's largest |x / s| is RN(amax / s) (correctly rounded
          // division is monotonic), formed as -RN(amax / s) by the steps of
          // fp8_codes8; beyond 448 the segment stays raw (out of range)
          const float q0 = __fmul_rn(amax, nr);
          const float qn = __fmaf_rn(__fmaf_rn(q0, sc, amax), nr, q0);
          if (qn < -448.0f) flags |= 2u;
        }
        const bool in = j < nv;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float x[8];
          unpack8<DT>(w[u][c], x);
          const uint2 out = fp8_codes8<CODEC>(x, sc, nr);
          if (in) st8(codes + (uint64_t)j * D + 8 * (li + G * c), out);
        }
        if (CODEC == KV_CODEC_FP8_DYNAMIC && in && li == 0)
          st4(meta + (uint64_t)j * 4, __float_as_uint(sc));
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if constexpr (SEAL) {
      zero_padding(s.slot, fp8_used_bytes<CODEC, D>(nv), p.seg_bytes[s.role], lane, 32);
      const uint32_t st = status_of_flags(flags);
      __syncwarp();
      if (lane == 0) st_u8(p.status + i, (uint8_t)st);
      crc::seal_segment<false>(q, *t, tb, i, st, lane, crc_m, crc_s);
    } else {
      if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
      zero_padding(s.slot, fp8_used_bytes<CODEC, D>(nv), p.seg_bytes[s.role], threadIdx.x, blockDim.x);
      __syncthreads();
      if (threadIdx.x == 0) st_u8(p.status + i, status_of_flags(s_flag[it & 1]));
      ++it;
    }
  }
}

// ADJ (segments of kAdjacentChunkMinVectors or more, D >= 64): lane li owns the
// adjacent chunks 2 li, 2 li + 1 -- one 16-byte code load and, when every vector
// is 32-byte aligned, one 32-byte store per vector.  Measured on a GB300: FP8
// decode of 512-vector segments 0.93-0.97 -> 0.97-0.98 of HBM, of 128-vector
// segments 0.968 -> 0.958, so smaller segments keep chunks li, li + G.
template <int DT, int D, uint32_t CODEC, bool ADJ, typename Q>
__global__ void __launch_bounds__(Variant<Q>::kCtaThreads)
    fp8_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q>::kSeal;
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = M::U, W = Variant<Q>::kCtaThreads / 32;
  constexpr uint32_t STEP = SEAL ? VPW * U : W * VPW * U;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t j_first = SEAL ? 0u : warp * VPW * U;
  const uint32_t nv = p.nv;
  const bool vec32 = p.vec32 != 0;
  crc::NibbleTables* t = nullptr;
  uint32_t tb = 0;
  uint32_t i = blockIdx.x, i_step = gridDim.x;  // no wrap: n_segments < 2^31
  // verifying: the check's reads keep the slot in L2 (evict_last) for the
  // restore's reads right after, which with the page stores go first
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
    float fixed = 1.0f;
    if (CODEC == KV_CODEC_FP8_FIXED) fixed = p.fixed_scale[s.layer][s.role];
    const uint8_t* codes = s.slot;
    const uint8_t* meta = s.slot + (uint64_t)nv * D;
    uint16_t* page = const_cast<uint16_t*>(s.page);
    // verifying: the restore walks the steps last to first, so that it starts
    // on the rows the check read last (the likeliest still in L2)
    const uint32_t n_steps = SEAL ? (nv + STEP - 1u) / STEP : 0u;
    for (uint32_t kk = 0, j0 = SEAL ? (n_steps - 1u) * STEP : j_first; SEAL ? kk < n_steps : j0 < nv;
         ++kk, j0 = SEAL ? (n_steps - 1u - kk) * STEP : j0 + STEP) {
      uint2 cw[U][NC];
      float sc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const bool in = j < nv;
        if (ADJ && NC == 2) {  // lane li owns the adjacent chunks 2 li, 2 li + 1: one 16-byte load
          const uint4 tt = in ? ld_nc16_h<SEAL>(codes + (uint64_t)j * D + 16 * li, once) : make_uint4(0, 0, 0, 0);
          cw[u][0] = make_uint2(tt.x, tt.y);
          cw[u][NC - 1] = make_uint2(tt.z, tt.w);
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            cw[u][c] = in ? ld_nc8_h<SEAL>(codes + (uint64_t)j * D + 8 * (li + G * c), once) : make_uint2(0, 0);
        }
        sc[u] = fixed;
        if (CODEC == KV_CODEC_FP8_DYNAMIC)
          sc[u] = in ? __uint_as_float(ld_nc4_h<SEAL>(meta + (uint64_t)j * 4, once)) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        uint16_t* dst = page + (j < nv ? vec_off(p, j) : 0);
        const float2 s2 = make_float2(sc[u], sc[u]);
        uint4 oc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint32_t h[4];
          e4m3x4_to_f16(cw[u][c].x, h[0], h[1]);
          e4m3x4_to_f16(cw[u][c].y, h[2], h[3]);
          uint4 o;
          if (DT == 0 && CODEC == KV_CODEC_FP8_CAST) {
            o = make_uint4(h[0], h[1], h[2], h[3]);   // code value is already the FP16 result
          } else {
            uint32_t r[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 y = mul2(make_float2(lo_f32<0>(h[k]), hi_f32<0>(h[k])), s2);
              r[k] = pack2<DT>(y.x, y.y);
            }
            o = make_uint4(r[0], r[1], r[2], r[3]);
          }
          if (ADJ && NC == 2) oc[c] = o;
          else if (j < nv) st16_h<SEAL>(dst + 8 * (li + G * c), o, once);
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

template <int DT, int D, uint32_t CODEC>
int sealed_mode(const Params& p, const CrcParams& q, int dir, void* stream) {
  if (dir == kEncode) return launch_sealed(fp8_encode_kernel<DT, D, CODEC, CrcParams>, p, q, stream);
  if (p.nv >= kAdjacentChunkMinVectors)
    return launch_sealed(fp8_decode_kernel<DT, D, CODEC, true, CrcParams>, p, q, stream);
  return launch_sealed(fp8_decode_kernel<DT, D, CODEC, false, CrcParams>, p, q, stream);
}

template <int DT, int D>
int sealed_codec(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream) {
  switch (codec) {
    case KV_CODEC_FP8_CAST: return sealed_mode<DT, D, KV_CODEC_FP8_CAST>(p, q, dir, stream);
    case KV_CODEC_FP8_FIXED: return sealed_mode<DT, D, KV_CODEC_FP8_FIXED>(p, q, dir, stream);
    case KV_CODEC_FP8_DYNAMIC: return sealed_mode<DT, D, KV_CODEC_FP8_DYNAMIC>(p, q, dir, stream);
  }
  return KV_ERR_INVALID_ARG;
}

template <int DT>
int sealed_dim(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream) {
  switch (p.D) {
    case 32: return sealed_codec<DT, 32>(p, q, dir, codec, stream);
    case 64: return sealed_codec<DT, 64>(p, q, dir, codec, stream);
    case 128: return sealed_codec<DT, 128>(p, q, dir, codec, stream);
    case 256: return sealed_codec<DT, 256>(p, q, dir, codec, stream);
  }
  return KV_ERR_UNSUPPORTED_HEAD_DIM;
}

template <int DT, int D, uint32_t CODEC>
int decode(const Params& p, void* stream) {
  if (p.nv >= kAdjacentChunkMinVectors)
    return launch_plain(fp8_decode_kernel<DT, D, CODEC, true, NoSeal>, p, stream, kDecodeCtas);
  return launch_plain(fp8_decode_kernel<DT, D, CODEC, false, NoSeal>, p, stream, kDecodeCtas);
}

template <int DT, int D>
int dispatch_mode(const Params& p, int dir, uint32_t codec, void* stream) {
  if (dir == kEncode) {
    switch (codec) {
      case KV_CODEC_FP8_CAST:
        return launch_plain(fp8_encode_kernel<DT, D, KV_CODEC_FP8_CAST, NoSeal>, p, stream,
                                   encode_ctas<KV_CODEC_FP8_CAST, D>());
      case KV_CODEC_FP8_FIXED:
        return launch_plain(fp8_encode_kernel<DT, D, KV_CODEC_FP8_FIXED, NoSeal>, p, stream,
                                   encode_ctas<KV_CODEC_FP8_FIXED, D>());
      case KV_CODEC_FP8_DYNAMIC:
        return launch_plain(fp8_encode_kernel<DT, D, KV_CODEC_FP8_DYNAMIC, NoSeal>, p, stream,
                                   encode_ctas<KV_CODEC_FP8_DYNAMIC, D>());
    }
  } else {
    switch (codec) {
      case KV_CODEC_FP8_CAST: return decode<DT, D, KV_CODEC_FP8_CAST>(p, stream);
      case KV_CODEC_FP8_FIXED: return decode<DT, D, KV_CODEC_FP8_FIXED>(p, stream);
      case KV_CODEC_FP8_DYNAMIC: return decode<DT, D, KV_CODEC_FP8_DYNAMIC>(p, stream);
    }
  }
  return KV_ERR_INVALID_ARG;
}

template <int DT>
int dispatch_dim(const Params& p, int dir, uint32_t codec, void* stream) {
  switch (p.D) {
    case 32: return dispatch_mode<DT, 32>(p, dir, codec, stream);
    case 64: return dispatch_mode<DT, 64>(p, dir, codec, stream);
    case 128: return dispatch_mode<DT, 128>(p, dir, codec, stream);
    case 256: return dispatch_mode<DT, 256>(p, dir, codec, stream);
  }
  return KV_ERR_UNSUPPORTED_HEAD_DIM;
}

}  // namespace

int launch_fp8(const Params& p, int dir, uint32_t codec, void* stream) {
  return p.dtype == KV_DT_FP16 ? dispatch_dim<0>(p, dir, codec, stream)
                               : dispatch_dim<1>(p, dir, codec, stream);
}

int launch_fp8_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream) {
  return p.dtype == KV_DT_FP16 ? sealed_dim<0>(p, q, dir, codec, stream)
                               : sealed_dim<1>(p, q, dir, codec, stream);
}

}  // namespace kvc
