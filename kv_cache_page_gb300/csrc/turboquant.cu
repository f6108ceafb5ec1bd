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
// which is exact), y = WHT(u) (ascending-stride butterflies, then * 1/sqrt(D)),
// code_i = number of codebook boundaries strictly below y_i, FP16(n) stored.
// Decode: c_i = centroid[code_i], g = f32(n16) / sqrt(pairwise sum c_i^2),
// out_i = +-(WHT(c)_i * g).  All register-resident; the WHT's cross-lane
// stages are warp shuffles.
#include "device_common.cuh"

namespace kvc {
namespace {

// Sign-bit masks for the lane's 8 elements: bit 15 / 31 of word k flips
// element 2k / 2k+1 of the packed 16-bit data.
__device__ __forceinline__ void sign_masks(const Params& p, uint32_t li, uint32_t (&m)[4]) {
  const uint32_t bits = (p.sign_words[li >> 2] >> (8u * (li & 3u))) & 0xffu;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    m[k] = (((bits >> (2 * k)) & 1u) << 15) | (((bits >> (2 * k + 1)) & 1u) << 31);
}

// number of boundaries b[0..K-2] (ascending) strictly below y
template <int K>
__device__ __forceinline__ uint32_t centroid_index(float y, const float* b) {
  uint32_t pos = 0;
#pragma unroll
  for (int step = K / 2; step >= 1; step >>= 1)
    if (b[pos + step - 1] < y) pos += step;
  return pos;
}

template <int DT, int D, int BITS>
__global__ void __launch_bounds__(kThreads) tq_encode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kE, VPW = 32 / G, U = 2, W = kThreads / 32;
  constexpr int STEP = W * VPW * U;
  constexpr int K = 1 << BITS;
  constexpr int CB = D * BITS / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  __shared__ float s_bnd[16];
  __shared__ uint32_t s_flag[2];
  if (threadIdx.x < 16) s_bnd[threadIdx.x] = p.bnd[threadIdx.x];
  if (threadIdx.x < 2) s_flag[threadIdx.x] = 0;
  __syncthreads();
  uint32_t smask[4];
  sign_masks(p, li, smask);
  const float cD = p.wht_scale;
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
    for (uint32_t j0 = warp * VPW * U; j0 < nv; j0 += STEP) {
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        w[u] = j < nv ? ld_stream16(s.page + vec_off(p, j) + li * kE) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        float mn, mx;
        vec_minmax<DT, G>(w[u], mn, mx);
        flags |= admission(mn, mx, p.reject_abs);
        uint4 ws = w[u];
        ws.x ^= smask[0]; ws.y ^= smask[1]; ws.z ^= smask[2]; ws.w ^= smask[3];
        float x[8], a[8];
        unpack8<DT>(ws, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = __fmul_rn(x[e], x[e]);
        const float n = __fsqrt_rn(pairwise_sum8<G>(a));
        float r = __frcp_rn(n);
        if (!isfinite(r)) r = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = __fmul_rn(x[e], r);
        wht_butterflies<G>(a, li);
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) v |= centroid_index<K>(__fmul_rn(a[e], cD), s_bnd) << (BITS * e);
        const bool in = j < nv;
        uint8_t* vc = codes + (uint64_t)j * CB;
        if (BITS == 4) {
          if (in) st4(vc + li * 4, v);
        } else {
          store_3bit(vc, v, li, in);
        }
        if (in && li == 0)
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
  constexpr int G = D / kE, VPW = 32 / G, U = 2, W = kThreads / 32;
  constexpr int STEP = W * VPW * U;
  constexpr int CB = D * BITS / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  __shared__ float s_cent[16];
  if (threadIdx.x < 16) s_cent[threadIdx.x] = p.cent[threadIdx.x];
  __syncthreads();
  uint32_t smask[4];
  sign_masks(p, li, smask);
  const float cD = p.wht_scale;
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
    for (uint32_t j0 = warp * VPW * U; j0 < nv; j0 += STEP) {
      uint32_t cw[U];
      uint16_t nw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const bool in = j < nv;
        const uint8_t* vc = codes + (uint64_t)j * CB;
        cw[u] = 0;
        nw[u] = 0;
        if (in) {
          cw[u] = BITS == 4 ? ld_nc4(vc + li * 4) : load_3bit(vc, li);
          nw[u] = ld_nc2(meta + (uint64_t)j * 2);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        float c[8], a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = s_cent[(cw[u] >> (BITS * e)) & ((1u << BITS) - 1u)];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = __fmul_rn(c[e], c[e]);
        const float nc = __fsqrt_rn(pairwise_sum8<G>(a));
        const float g = __fdiv_rn(__half2float(__ushort_as_half(nw[u])), nc);
        wht_butterflies<G>(c, li);
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = __fmul_rn(__fmul_rn(c[e], cD), g);
        uint4 o = pack8<DT>(c);
        o.x ^= smask[0]; o.y ^= smask[1]; o.z ^= smask[2]; o.w ^= smask[3];
        if (j < nv) st16(page + vec_off(p, j) + li * kE, o);
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
