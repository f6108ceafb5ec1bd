// turboquant.cu -- TurboQuant-style K encode / decode kernels (3 and 4 bits).
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
// Thread mapping: each lane owns 32 contiguous elements of a vector (64
// bytes of FP16/BF16), G = D/32 lanes per vector, held as 16 FP32 pairs
// (element 2m, 2m+1).  Butterflies with stride 2..16 are packed FP32x2 ops
// between pairs, stride 1 is inside a pair, and strides >= 32 are warp
// shuffles across the vector's lanes.
#include "device_common.cuh"

namespace kvc {
namespace {

constexpr int kTqE = 32;               // elements per lane
constexpr float kCellMagic = 12582912.0f;  // 1.5 * 2^23: FFMA(w, 4, magic) has rint(4 w) in its low bits
constexpr uint32_t kCellMagicBits = 0x4b400000u;

// Sign masks of the lane's 16 packed words (elements 2m, 2m+1): bit 15 / 31.
__device__ __forceinline__ void sign_masks(const Params& p, uint32_t li, uint32_t (&m)[16]) {
  const uint32_t bits = p.sign_words[li];
#pragma unroll
  for (int k = 0; k < 16; ++k)
    m[k] = (((bits >> (2 * k)) & 1u) << 15) | (((bits >> (2 * k + 1)) & 1u) << 31);
}

// Pairwise sum over the vector: in-thread tree over the lane's 32 elements
// (pairs first), then xor-shuffles over the G lanes with ascending distance.
template <int G>
__device__ __forceinline__ float vector_sum(const float2 (&a)[16]) {
  float s[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) s[m] = __fadd_rn(a[m].x, a[m].y);
#pragma unroll
  for (int w = 1; w < 16; w <<= 1)
#pragma unroll
    for (int m = 0; m < 16; m += 2 * w) s[m] = __fadd_rn(s[m], s[m + w]);
  float c = s[0];
#pragma unroll
  for (int o = 1; o < G; o <<= 1) c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, o));
  return c;
}

// Unscaled Walsh-Hadamard butterflies over the vector, strides 1 .. D/2.
template <int G>
__device__ __forceinline__ void butterflies(float2 (&a)[16], uint32_t li) {
#pragma unroll
  for (int m = 0; m < 16; ++m) {  // stride 1: inside each pair
    const float u = a[m].x, v = a[m].y;
    a[m] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {  // strides 2, 4, 8, 16: pair m with pair m + h
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m & h) continue;
      const float2 u = a[m], v = a[m + h];
      a[m] = add2(u, v);
      a[m + h] = sub2(u, v);
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {  // strides 32 o: across lanes
    const float sg = (li & (uint32_t)o) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float2 partner = make_float2(__shfl_xor_sync(0xffffffffu, a[m].x, o),
                                         __shfl_xor_sync(0xffffffffu, a[m].y, o));
      a[m] = fma2(a[m], sg2, partner);  // low lane: mine + partner; high lane: partner - mine
    }
  }
}

template <int DT, int D, int BITS>
__global__ void __launch_bounds__(kThreads) tq_encode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kTqE, VPW = 32 / G, W = kThreads / 32;
  constexpr int STEP = W * VPW;
  constexpr int CB = D * BITS / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  // cell table, 16 copies so that the lanes of a half warp never share a bank
  __shared__ uint2 s_lut[kLutCells * 16];
  __shared__ uint32_t s_flag[2];
  for (int k = threadIdx.x; k < kLutCells * 16; k += blockDim.x)
    s_lut[k] = make_uint2(__float_as_uint(p.lut_thr[k >> 4]), p.lut_lo[k >> 4]);
  if (threadIdx.x < 2) s_flag[threadIdx.x] = 0;
  __syncthreads();
  uint32_t smask[16];
  sign_masks(p, li, smask);
  // byte address of cell c for this lane = bits(FFMA(w, 4, magic)) * 128 + lut_base
  const uint32_t lut_base = (uint32_t)__cvta_generic_to_shared(s_lut) + (lane & 15u) * 8u +
                            (uint32_t)(kLutHalf * 128) - kCellMagicBits * 128u;
  const uint32_t nv = p.nv;
  int it = 0;
  for (uint32_t i = blockIdx.x; i < p.n_segments; i += gridDim.x) {
    const Seg s = plan_segment(p, i, kEncode);
    if (s.action != kProcess) {
      if (s.action == kReport && threadIdx.x == 0) p.status[i] = s.status;
      continue;
    }
    if (threadIdx.x == 0) s_flag[(it + 1) & 1] = 0;
    uint8_t* codes = s.slot;
    uint8_t* meta = s.slot + (uint64_t)nv * CB;
    uint32_t flags = 0;
    for (uint32_t j0 = warp * VPW; j0 < nv; j0 += STEP) {
      const uint32_t j = j0 + grp;
      const bool in = j < nv;
      uint4 w[4];
      const uint16_t* src = s.page + (in ? vec_off(p, j) : 0) + kTqE * li;
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = in ? ld_nc16(src + 8 * c) : make_uint4(0, 0, 0, 0);
      float mn, mx;
      vec_minmax<DT, G, 4>(w, mn, mx);
      const uint32_t vflags = admission(mn, mx, p.reject_abs);
      flags |= vflags;
      if (vflags) {  // keep NaN / inf out of the arithmetic (the segment stays raw)
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = make_uint4(0, 0, 0, 0);
      }
      float2 a[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t ww[4] = {w[c].x ^ smask[4 * c], w[c].y ^ smask[4 * c + 1],
                                w[c].z ^ smask[4 * c + 2], w[c].w ^ smask[4 * c + 3]};
#pragma unroll
        for (int k = 0; k < 4; ++k) a[4 * c + k] = make_float2(lo_f32<DT>(ww[k]), hi_f32<DT>(ww[k]));
      }
      float2 sq[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) sq[m] = mul2(a[m], a[m]);
      const float n = __fsqrt_rn(vector_sum<G>(sq));
      float r = __frcp_rn(n);
      if (!isfinite(r)) r = 0.0f;
      const float2 r2 = make_float2(r, r);
#pragma unroll
      for (int m = 0; m < 16; ++m) a[m] = mul2(a[m], r2);
      butterflies<G>(a, li);
      if (n < 0x1p-62f) {
        // Norms this small may come from squares that underflowed, so |w|
        // can exceed sqrt(D); clamp into the table (beyond +-17 every code
        // is already the first or the last).
#pragma unroll
        for (int m = 0; m < 16; ++m)
          a[m] = make_float2(fminf(fmaxf(a[m].x, -17.0f), 17.0f), fminf(fmaxf(a[m].y, -17.0f), 17.0f));
      }
      // codes, element 0 in the lowest bits: accumulate from the last element
      uint32_t acc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v = 0;
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          const float x = (e & 1) ? a[4 * q + e / 2].y : a[4 * q + e / 2].x;
          const uint32_t cell = __float_as_uint(__fmaf_rn(x, 4.0f, kCellMagic));
          uint2 ent;
          asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(ent.x), "=r"(ent.y) : "r"(cell * 128u + lut_base));
          v = (v << BITS) + ent.y + (x > __uint_as_float(ent.x) ? 1u : 0u);
        }
        acc[q] = v;
      }
      uint8_t* vc = codes + (uint64_t)j * CB;
      if (in) {
        if (BITS == 4) {
          st16(vc + 16 * li, make_uint4(acc[0], acc[1], acc[2], acc[3]));
        } else {
          const uint32_t w0 = acc[0] | (acc[1] << 24);
          const uint32_t w1 = (acc[1] >> 8) | (acc[2] << 16);
          const uint32_t w2 = (acc[2] >> 16) | (acc[3] << 8);
          st4(vc + 12 * li, w0);
          st4(vc + 12 * li + 4, w1);
          st4(vc + 12 * li + 8, w2);
        }
        if (li == 0)
          *reinterpret_cast<uint16_t*>(meta + (uint64_t)j * 2) = __half_as_ushort(__float2half_rn(n));
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
    zero_padding(s.slot, (uint64_t)nv * (CB + 2), p.seg_bytes[s.role]);
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t f = s_flag[it & 1];
      p.status[i] = (f & 1u) ? KV_SEG_RAW_NONFINITE : (f & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED;
    }
    ++it;
  }
}

template <int DT, int D, int BITS>
__global__ void __launch_bounds__(kThreads) tq_decode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kTqE, VPW = 32 / G, W = kThreads / 32;
  constexpr int STEP = W * VPW;
  constexpr int CB = D * BITS / 8;
  constexpr int NPAIR = BITS == 4 ? 256 : 64;  // table of two consecutive codes
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  // (centroid[lo code], centroid[hi code]) for every pair of codes, 16 copies
  __shared__ float2 s_pair[NPAIR * 16];
  for (int k = threadIdx.x; k < NPAIR * 16; k += blockDim.x) {
    const int v = k >> 4;
    s_pair[k] = make_float2(p.cent[v & ((1 << BITS) - 1)], p.cent[v >> BITS]);
  }
  __syncthreads();
  uint32_t smask[16];
  sign_masks(p, li, smask);
  const uint32_t pair_base = (uint32_t)__cvta_generic_to_shared(s_pair) + (lane & 15u) * 8u;
  const float cD = p.wht_scale;
  const float2 cD2 = make_float2(cD, cD);
  const uint32_t nv = p.nv;
  for (uint32_t i = blockIdx.x; i < p.n_segments; i += gridDim.x) {
    const Seg s = plan_segment(p, i, kDecode);
    if (s.action != kProcess) {
      if (s.action == kReport && threadIdx.x == 0 && p.result) p.result[i] = s.status;
      continue;
    }
    const uint8_t* codes = s.slot;
    const uint8_t* meta = s.slot + (uint64_t)nv * CB;
    uint16_t* page = const_cast<uint16_t*>(s.page);
    for (uint32_t j0 = warp * VPW; j0 < nv; j0 += STEP) {
      const uint32_t j = j0 + grp;
      const bool in = j < nv;
      const uint8_t* vc = codes + (uint64_t)j * CB;
      uint32_t cw[4] = {0, 0, 0, 0};
      uint16_t n16 = 0;
      if (in) {
        if (BITS == 4) {
          const uint4 t = ld_nc16(vc + 16 * li);
          cw[0] = t.x; cw[1] = t.y; cw[2] = t.z; cw[3] = t.w;
        } else {
          cw[0] = ld_nc4(vc + 12 * li);
          cw[1] = ld_nc4(vc + 12 * li + 4);
          cw[2] = ld_nc4(vc + 12 * li + 8);
        }
        n16 = ld_nc2(meta + (uint64_t)j * 2);
      }
      float2 a[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        uint32_t v;
        if (BITS == 4) {
          v = __byte_perm(cw[m >> 2], 0, 0x4440 | (m & 3));
        } else {
          const int bit = 6 * m;
          v = __funnelshift_r(cw[bit >> 5], cw[(bit >> 5) + 1], bit & 31) & 63u;
        }
        asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a[m].x), "=f"(a[m].y) : "r"(v * 128u + pair_base));
      }
      float2 sq[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) sq[m] = mul2(a[m], a[m]);
      const float nc = __fsqrt_rn(vector_sum<G>(sq));
      const float g = __fdiv_rn(__half2float(__ushort_as_half(n16)), nc);
      const float2 g2 = make_float2(g, g);
      butterflies<G>(a, li);
      uint32_t o[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float2 t = mul2(mul2(a[m], cD2), g2);
        o[m] = pack2<DT>(t.x, t.y) ^ smask[m];
      }
      uint16_t* dst = page + (in ? vec_off(p, j) : 0) + kTqE * li;
      if (in) {
#pragma unroll
        for (int c = 0; c < 4; ++c) st16(dst + 8 * c, make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
      }
    }
    if (threadIdx.x == 0 && p.result) p.result[i] = KV_SEG_ENCODED;
  }
}

template <int DT, int D>
int dispatch_bits(const Params& p, int dir, uint32_t codec, void* stream) {
  const bool enc = dir == kEncode;
  switch (codec) {
    case KV_CODEC_TQ3:
      return enc ? launch_codec_kernel(tq_encode_kernel<DT, D, 3>, p, stream)
                 : launch_codec_kernel(tq_decode_kernel<DT, D, 3>, p, stream);
    case KV_CODEC_TQ4:
      return enc ? launch_codec_kernel(tq_encode_kernel<DT, D, 4>, p, stream)
                 : launch_codec_kernel(tq_decode_kernel<DT, D, 4>, p, stream);
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
