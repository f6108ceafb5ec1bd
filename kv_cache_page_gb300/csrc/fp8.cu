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
#include "device_common.cuh"

namespace kvc {
namespace {

constexpr float kRecip448 = 1.0f / 448.0f;  // fl32(1/448)

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }"
      : "=r"(d)
      : "f"(hi), "f"(lo));
  return d;
}
// two E4M3 bytes (low byte = first element) -> f16x2 (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(d) : "r"(two));
  return d;
}

template <int DT, int D, uint32_t CODEC>
__global__ void __launch_bounds__(kThreads) fp8_encode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kE, VPW = 32 / G, U = 4, W = kThreads / 32;
  constexpr int STEP = W * VPW * U;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  __shared__ uint32_t s_flag[2];
  if (threadIdx.x < 2) s_flag[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t nv = p.nv;
  int it = 0;
  for (uint32_t i = blockIdx.x; i < p.n_segments; i += gridDim.x) {
    const Seg s = plan_segment(p, i, kEncode);
    if (s.action != kProcess) {
      if (s.action == kReport && threadIdx.x == 0) p.status[i] = s.status;
      continue;
    }
    if (threadIdx.x == 0) s_flag[(it + 1) & 1] = 0;
    float scale = 1.0f;
    if (CODEC == KV_CODEC_FP8_FIXED) scale = p.fixed_scale[s.layer][s.role];
    const float rscale = __frcp_rn(scale);
    uint8_t* codes = s.slot;
    uint8_t* meta = s.slot + (uint64_t)nv * D;
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
        float x[8];
        unpack8<DT>(w[u], x);
        float sc = scale, r = rscale;
        if (CODEC == KV_CODEC_FP8_DYNAMIC) {
          const float amax = fmaxf(-mn, mx);
          sc = __fmul_rn(fmaxf(amax, 1e-12f), kRecip448);
          r = __frcp_rn(sc);
        }
        if (CODEC != KV_CODEC_FP8_CAST) {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = div_by(x[e], sc, r);
        }
        const uint32_t b01 = e4m3x2(x[0], x[1]), b23 = e4m3x2(x[2], x[3]);
        const uint32_t b45 = e4m3x2(x[4], x[5]), b67 = e4m3x2(x[6], x[7]);
        const uint2 out = make_uint2(b01 | (b23 << 16), b45 | (b67 << 16));
        if (j < nv) {
          st8(codes + (uint64_t)j * D + li * kE, out);
          if (CODEC == KV_CODEC_FP8_DYNAMIC && li == 0) st4(meta + (uint64_t)j * 4, __float_as_uint(sc));
        }
      }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags) atomicOr(&s_flag[it & 1], flags);
    const uint64_t used = (uint64_t)nv * (D + (CODEC == KV_CODEC_FP8_DYNAMIC ? 4 : 0));
    zero_padding(s.slot, used, p.seg_bytes[s.role]);
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t f = s_flag[it & 1];
      p.status[i] = (f & 1u) ? KV_SEG_RAW_NONFINITE : (f & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED;
    }
    ++it;
  }
}

template <int DT, int D, uint32_t CODEC>
__global__ void __launch_bounds__(kThreads) fp8_decode_kernel(const __grid_constant__ Params p) {
  constexpr int G = D / kE, VPW = 32 / G, U = 4, W = kThreads / 32;
  constexpr int STEP = W * VPW * U;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t grp = lane / G, li = lane % G;
  const uint32_t nv = p.nv;
  for (uint32_t i = blockIdx.x; i < p.n_segments; i += gridDim.x) {
    const Seg s = plan_segment(p, i, kDecode);
    if (s.action != kProcess) {
      if (s.action == kReport && threadIdx.x == 0 && p.result) p.result[i] = s.status;
      continue;
    }
    float scale = 1.0f;
    if (CODEC == KV_CODEC_FP8_FIXED) scale = p.fixed_scale[s.layer][s.role];
    const uint8_t* codes = s.slot;
    const uint8_t* meta = s.slot + (uint64_t)nv * D;
    uint16_t* page = const_cast<uint16_t*>(s.page);
    for (uint32_t j0 = warp * VPW * U; j0 < nv; j0 += STEP) {
      uint2 c[U];
      float sc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const bool in = j < nv;
        c[u] = in ? ld_nc8(codes + (uint64_t)j * D + li * kE) : make_uint2(0, 0);
        sc[u] = scale;
        if (CODEC == KV_CODEC_FP8_DYNAMIC) sc[u] = in ? __uint_as_float(ld_nc4(meta + (uint64_t)j * 4)) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t j = j0 + u * VPW + grp;
        const uint32_t h[4] = {e4m3x2_to_f16x2(c[u].x & 0xffffu), e4m3x2_to_f16x2(c[u].x >> 16),
                               e4m3x2_to_f16x2(c[u].y & 0xffffu), e4m3x2_to_f16x2(c[u].y >> 16)};
        float y[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          y[2 * k] = __fmul_rn(lo_f32<0>(h[k]), sc[u]);
          y[2 * k + 1] = __fmul_rn(hi_f32<0>(h[k]), sc[u]);
        }
        if (j < nv) st16(page + vec_off(p, j) + li * kE, pack8<DT>(y));
      }
    }
    if (threadIdx.x == 0 && p.result) p.result[i] = KV_SEG_ENCODED;
  }
}

template <int DT, int D>
int dispatch_mode(const Params& p, int dir, uint32_t codec, void* stream) {
  if (dir == kEncode) {
    switch (codec) {
      case KV_CODEC_FP8_CAST: return launch_codec_kernel(fp8_encode_kernel<DT, D, KV_CODEC_FP8_CAST>, p, stream);
      case KV_CODEC_FP8_FIXED: return launch_codec_kernel(fp8_encode_kernel<DT, D, KV_CODEC_FP8_FIXED>, p, stream);
      case KV_CODEC_FP8_DYNAMIC: return launch_codec_kernel(fp8_encode_kernel<DT, D, KV_CODEC_FP8_DYNAMIC>, p, stream);
    }
  } else {
    switch (codec) {
      case KV_CODEC_FP8_CAST: return launch_codec_kernel(fp8_decode_kernel<DT, D, KV_CODEC_FP8_CAST>, p, stream);
      case KV_CODEC_FP8_FIXED: return launch_codec_kernel(fp8_decode_kernel<DT, D, KV_CODEC_FP8_FIXED>, p, stream);
      case KV_CODEC_FP8_DYNAMIC: return launch_codec_kernel(fp8_decode_kernel<DT, D, KV_CODEC_FP8_DYNAMIC>, p, stream);
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

}  // namespace kvc
