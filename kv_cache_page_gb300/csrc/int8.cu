// int8.cu -- symmetric per-head INT8 encode / decode in token-row records.
//
// "Building a quantized HiCache for SGLang", section "Building the INT8
// codec": one scale per KV head vector (token, layer, K or V, head); amax =
// max|x| raised to a small floor, scale = amax / 127 (a BF16 tensor divided
// by an integer: FP32 quotient rounded to BF16), code = round(FP32(x) /
// FP32(scale)) clamped to [-127, 127]; restore = code * scale as BF16.
// Section "Why exactly 1,152 bytes?": per token row of one role the H heads'
// codes (H*D bytes) then their H BF16 scales, padded with zeros to a multiple
// of 128 bytes; a segment's slot is its block_tokens records in token order.
//
// The source is BF16 (the page's KV dtype; the host refuses FP16).  Per
// element the encoder does one correctly rounded division (reciprocal of the
// scale + one FMA correction) and a magic-number rounding whose low byte is
// the two's-complement code.  The clamp to [-127, 127] is implied for BF16
// sources: over every BF16 maximum a (floored), a / scale <= 127.33 < 127.5,
// and |x| <= a, so every rounded quotient is already in range.
#include "crc_common.cuh"

namespace kvc {
namespace {

constexpr int kEncodeCtas = 6;  // resident CTAs per SM (see launch_codec_kernel)
constexpr int kDecodeCtas = 4;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: RN(q + magic) holds rint(q) in its low byte
constexpr float kAmaxFloor = 1e-12f;        // floor of the head maximum
constexpr uint32_t kAmaxFloorBf16 = 0x2B8D0000u;  // BF16(1e-12f) as FP32 bits (the floored value)

// Codes of 8 elements: rint(x / s) as 8 int8 bytes (|x / s| < 127.5, see
// above).  The quotient is correctly rounded: q0 = RN(x r), e = RN(x - q0 s)
// is exact, q = RN(q0 + e r).
__device__ __forceinline__ uint2 int8_codes8(const float (&x)[8], float s, float r) {
  const float2 ns2 = make_float2(-s, -s), r2 = make_float2(r, r);
  const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
  uint32_t t[8];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 xx = make_float2(x[e], x[e + 1]);
    const float2 q0 = mul2(xx, r2);
    const float2 res = fma2(q0, ns2, xx);
    const float2 q = fma2(res, r2, q0);
    const float2 m = add2(q, mg2);
    t[e] = __float_as_uint(m.x);
    t[e + 1] = __float_as_uint(m.y);
  }
  // low bytes in element order
  const uint32_t lo = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
  return make_uint2(lo, hi);
}

// a / 127 correctly rounded, for a BF16 maximum a >= the floor: q0 = RN(a
// RN(1/127)), one FMA residual and correction (equal to the IEEE quotient for
// every such a; checked exhaustively).
__device__ __forceinline__ float div127(float a) {
  constexpr float r = 1.0f / 127.0f;
  const float q0 = __fmul_rn(a, r);
  const float e = __fmaf_rn(-q0, 127.0f, a);
  return __fmaf_rn(e, r, q0);
}

// Byte offset of vector j's codes and of its scale inside the slot.
__device__ __forceinline__ void record_offsets(const Params& p, uint32_t j, uint32_t& code_off,
                                               uint32_t& scale_off) {
  const uint32_t t = (uint32_t)(((uint64_t)j * p.h_magic) >> 32);
  const uint32_t h = j - t * p.H;
  const uint32_t rec = t * p.rec_bytes;
  code_off = rec + h * p.D;
  scale_off = rec + p.H * p.D + 2u * h;
}

// Zero the padding of every record of a slot (whole CTA, 16-bit stores: the
// used part H*(D+2) and the record size are even).
__device__ __forceinline__ void zero_record_padding(const Params& p, uint8_t* slot) {
  const uint32_t pad16 = (p.rec_bytes - p.rec_used) / 2u;
  if (pad16 == 0) return;
  const uint32_t total = p.T * pad16;
  for (uint32_t k = threadIdx.x; k < total; k += blockDim.x) {
    const uint32_t t = k / pad16, o = k - t * pad16;
    st_u16(slot + (uint64_t)t * p.rec_bytes + p.rec_used + 2u * o, 0);
  }
}

// Q selects the variant (NoSeal: a CTA of kThreads per segment; CrcParams: one
// warp per segment, as for the FP8 kernels).  The sealing encoder writes the
// slot's records in token order: the step that completes a token's record
// also zeroes its padding, and at the start of a step, with its loads in
// flight, the warp folds the next 2 KB CRC row if the records completed by
// the earlier steps cover it (re-read from L2).  The rows left after the last
// step and the header follow.
template <int D, typename Q>
__global__ void __launch_bounds__(Variant<Q>::kCtaThreads)
    int8_encode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q>::kSeal;
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = M::U, W = Variant<Q>::kCtaThreads / 32;
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
    uint32_t flags = 0;
    // sealing: records [0, rec_done) complete (codes, scales, zeroed padding),
    // rows [0, crc_m) of the slot folded into crc_s
    uint32_t rec_done = 0, crc_s = 0, crc_m = 0;
    const bool al32 = ((uintptr_t)s.slot & 31u) == 0;
    for (uint32_t j0 = j_first; j0 < nv; j0 += STEP) {
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
        if ((crc_m + 1u) * kCrcRow <= rec_done * p.rec_bytes) {
          __syncwarp();
          crc_s = crc::fold_row<false>(*t, tb, s.slot, crc_m, al32, crc_s, lane);
          ++crc_m;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const float amax = vec_absmax<1, G, NC>(w[u]);
        flags |= admission_abs(amax, p.reject_abs);
        const float a = amax < kAmaxFloor ? __uint_as_float(kAmaxFloorBf16) : amax;
        const __nv_bfloat16 s16 = __float2bfloat16_rn(div127(a));
        const float sc = __bfloat162float(s16);
        const float r = __frcp_rn(sc);
        const bool in = j < nv;
        uint32_t code_off = 0, scale_off = 0;
        if (in) record_offsets(p, j, code_off, scale_off);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float x[8];
          unpack8<1>(w[u][c], x);
          const uint2 out = int8_codes8(x, sc, r);
          if (in) st8(s.slot + code_off + 8 * (li + G * c), out);
        }
        if (in && li == 0)
          st_u16(s.slot + scale_off, __bfloat16_as_ushort(s16));
      }
      if constexpr (SEAL) {
        // zero the padding of the records this step completed, with the widest
        // stores the used part's size allows (16, 4 or 2 bytes; the record
        // size is a multiple of 128)
        const uint32_t end = min(nv, j0 + STEP), n = p.rec_bytes - p.rec_used;
        for (; (rec_done + 1u) * p.H <= end; ++rec_done) {
          uint8_t* pad = s.slot + (uint64_t)rec_done * p.rec_bytes + p.rec_used;
          if ((p.rec_used & 15u) == 0u) {
            for (uint32_t o = 16u * lane; o < n; o += 512u) st16(pad + o, make_uint4(0, 0, 0, 0));
          } else if ((p.rec_used & 3u) == 0u) {
            for (uint32_t o = 4u * lane; o < n; o += 128u) st4(pad + o, 0u);
          } else {
            for (uint32_t o = 2u * lane; o < n; o += 64u) st_u16(pad + o, 0);
          }
        }
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if constexpr (SEAL) {
      const uint32_t st = status_of_flags(flags);
      __syncwarp();
      if (lane == 0) st_u8(p.status + i, (uint8_t)st);
      crc::seal_segment<false>(q, *t, tb, i, st, lane, crc_m, crc_s);
    } else {
      if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
      zero_record_padding(p, s.slot);
      __syncthreads();
      if (threadIdx.x == 0) {
        const uint32_t f = s_flag[it & 1];
        st_u8(p.status + i, (f & 1u) ? KV_SEG_RAW_NONFINITE : (f & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED);
      }
      ++it;
    }
  }
}

// Verifying variant (CrcParams): one warp per segment checks the header and
// the CRC-32 as kv_codec_verify does (loads with an L2 evict_last policy) and
// only then restores the segment, re-reading the slot from L2 last vectors
// first (code loads and page stores with evict_first).
template <int D, typename Q>
__global__ void __launch_bounds__(Variant<Q>::kCtaThreads)
    int8_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ Q q) {
  using M = ChunkMap<D>;
  constexpr bool SEAL = Variant<Q>::kSeal;
  constexpr int G = M::G, NC = M::NC, VPW = M::VPW, U = M::U, W = Variant<Q>::kCtaThreads / 32;
  constexpr uint32_t STEP = SEAL ? VPW * U : W * VPW * U;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t j_first = SEAL ? 0u : warp * VPW * U;
  const uint32_t nv = p.nv;
  // float(c) for a two's-complement byte c: the word 0x4B0000(c ^ 0x80) is
  // 2^23 + c + 128 exactly
  const float2 bias2 = make_float2(-8388736.0f, -8388736.0f);
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
    uint16_t* page = const_cast<uint16_t*>(s.page);
    // verifying: the steps last to first (the rows the check read last first)
    const uint32_t n_steps = SEAL ? (nv + STEP - 1u) / STEP : 0u;
    for (uint32_t kk = 0, j0 = SEAL ? (n_steps - 1u) * STEP : j_first; SEAL ? kk < n_steps : j0 < nv;
         ++kk, j0 = SEAL ? (n_steps - 1u - kk) * STEP : j0 + STEP) {
      uint2 cw[U][NC];
      float sc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const bool in = j < nv;
        uint32_t code_off = 0, scale_off = 0;
        if (in) record_offsets(p, j, code_off, scale_off);
#pragma unroll
        for (int c = 0; c < NC; ++c)
          cw[u][c] = in ? ld_nc8_h<SEAL>(s.slot + code_off + 8 * (li + G * c), once) : make_uint2(0, 0);
        sc[u] = in ? __uint_as_float((uint32_t)ld_nc2(s.slot + scale_off) << 16) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        uint16_t* dst = page + (j < nv ? vec_off(p, j) : 0);
        const float2 s2 = make_float2(sc[u], sc[u]);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint32_t r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wd = (k < 2 ? cw[u][c].x : cw[u][c].y) ^ 0x80808080u;
            const uint32_t b = 2u * (k & 1);
            const float2 f = make_float2(__uint_as_float(__byte_perm(wd, 0x4B000000u, 0x7440u | b)),
                                         __uint_as_float(__byte_perm(wd, 0x4B000000u, 0x7440u | (b + 1))));
            const float2 y = mul2(add2(f, bias2), s2);
            r[k] = pack2<1>(y.x, y.y);
          }
          if (j < nv) st16_h<SEAL>(dst + 8 * (li + G * c), make_uint4(r[0], r[1], r[2], r[3]), once);
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

template <int D>
int launch_dim(const Params& p, const CrcParams* q, int dir, void* stream) {
  if (q)
    return dir == kEncode ? launch_sealed(int8_encode_kernel<D, CrcParams>, p, *q, stream)
                          : launch_sealed(int8_decode_kernel<D, CrcParams>, p, *q, stream);
  return dir == kEncode ? launch_plain(int8_encode_kernel<D, NoSeal>, p, stream, kEncodeCtas)
                        : launch_plain(int8_decode_kernel<D, NoSeal>, p, stream, kDecodeCtas);
}

int launch_any(const Params& p, const CrcParams* q, int dir, uint32_t codec, void* stream) {
  if (codec != KV_CODEC_INT8_HEAD || p.dtype != KV_DT_BF16) return KV_ERR_INVALID_ARG;
  switch (p.D) {
    case 32: return launch_dim<32>(p, q, dir, stream);
    case 64: return launch_dim<64>(p, q, dir, stream);
    case 128: return launch_dim<128>(p, q, dir, stream);
    case 256: return launch_dim<256>(p, q, dir, stream);
  }
  return KV_ERR_UNSUPPORTED_HEAD_DIM;
}

}  // namespace

int launch_int8(const Params& p, int dir, uint32_t codec, void* stream) {
  return launch_any(p, nullptr, dir, codec, stream);
}

int launch_int8_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream) {
  return launch_any(p, &q, dir, codec, stream);
}

}  // namespace kvc
