// crc.cu -- segment headers: CRC-32 of encoded slots (seal) and their check
// before decode (verify).
//
// "KV precision and storage encoding" (OrbitKV docs), section "Ownership,
// storage and GDS": each encoded segment carries a version, its original
// length, its format, its stored length and a CRC32; checksums are validated
// before GPU decode, and a damaged object becomes a miss.
//
// The standalone passes: two slots per warp at a time (one per half warp),
// one 1024-thread CTA per SM holding the lookup tables (the CRC itself is in
// crc_common.cuh).  The FP8, uniform-8 and
// INT8 codec kernels also seal while they encode and verify before they
// decode, without this second pass over the slots (fp8.cu, uniform.cu,
// int8.cu).
#include "crc_common.cuh"

namespace kvc {
namespace {

using namespace crc;

// Two slots per warp at a time, one per half warp (crc_rows_half): warp w
// takes slots 2 w + half, 2 (w + W) + half, ... for W warps in the grid.
__global__ void __launch_bounds__(kCrcThreads, 1) crc_seal_kernel(const __grid_constant__ CrcParams p) {
  NibbleTables* t;
  const uint32_t tb = load_tables(p, t);
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t nw = gridDim.x * kCrcWarps, w = blockIdx.x * kCrcWarps + warp;
  for (uint32_t i0 = 2u * w; i0 < p.n_segments; i0 += 2u * nw) {  // no wrap: n_segments < 2^31
    const uint32_t i = i0 + (lane >> 4);
    const bool have = i < p.n_segments;
    uint32_t role = 0;
    uint64_t off = 0;
    const bool ok = have && slot_ok(p, p.descs + i, role, off);
    const uint32_t st = have ? ld_u8(p.status + i) : 0u;
    const bool coded = ok && st == KV_SEG_ENCODED && p.codec[role] != KV_CODEC_NONE;
    const uint32_t n = coded ? (uint32_t)p.seg_bytes[role] : 0u;
    const uint32_t crc = crc_rows_half<true>(*t, tb, p.buf + (coded ? off : 0), n, coded ? p.crc_k[role] : 0u, lane);
    if (have && (lane & 15u) == 0u) {
      if (!ok) store_header(p.headers + i, p.version, 0, 0, 0, KV_SEG_BAD_DESC, p.orig_bytes);
      else store_header(p.headers + i, p.version, p.format[role], n, coded ? crc : 0u, st, p.orig_bytes);
    }
  }
}

__global__ void __launch_bounds__(kCrcThreads, 1) crc_verify_kernel(const __grid_constant__ CrcParams p) {
  NibbleTables* t;
  const uint32_t tb = load_tables(p, t);
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t nw = gridDim.x * kCrcWarps, w = blockIdx.x * kCrcWarps + warp;
  for (uint32_t i0 = 2u * w; i0 < p.n_segments; i0 += 2u * nw) {
    const uint32_t i = i0 + (lane >> 4);
    const bool have = i < p.n_segments;
    uint32_t role = 0;
    uint64_t off = 0;
    const bool desc = have && slot_ok(p, p.descs + i, role, off) && p.codec[role] != KV_CODEC_NONE;
    uint64_t w0 = 0, orig = 0, stored = 0, w3 = 0;
    if (desc) {
      const uint64_t* hw = reinterpret_cast<const uint64_t*>(p.headers + i);
      w0 = ldg_u64(hw);
      orig = ldg_u64(hw + 1);
      stored = ldg_u64(hw + 2);
      w3 = ldg_u64(hw + 3);
    }
    const uint32_t st = (uint32_t)(w3 >> 32);
    bool ok = desc && (uint32_t)w0 == p.version && (uint32_t)(w0 >> 32) == p.format[role] &&
              orig == p.orig_bytes && st >= KV_SEG_ENCODED && st <= KV_SEG_BAD_DESC;
    const bool check = ok && st == KV_SEG_ENCODED && stored == p.seg_bytes[role];
    const uint32_t n = check ? (uint32_t)stored : 0u;
    const uint32_t crc = crc_rows_half<true>(*t, tb, p.buf + (check ? off : 0), n, check ? p.crc_k[role] : 0u, lane);
    if (ok) ok = st == KV_SEG_ENCODED ? (check && crc == (uint32_t)w3) : stored == 0;
    if (have && (lane & 15u) == 0u)
      st_u8(p.result + i, !desc ? (uint8_t)KV_SEG_BAD_DESC : ok ? (uint8_t)st : (uint8_t)KV_SEG_CORRUPT);
  }
}

}  // namespace

int launch_crc(const CrcParams& p, int seal, void* stream) {
  const void* k = seal ? reinterpret_cast<const void*>(crc_seal_kernel)
                       : reinterpret_cast<const void*>(crc_verify_kernel);
  // the tables need more than the default 48 KB of dynamic shared memory (set
  // on every launch: the attribute belongs to the current device's context)
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCrcSmem) != cudaSuccess)
    return KV_ERR_CUDA;
  unsigned grid = 0;
  const int rc = grid_for_threads(k, (p.n_segments + 2 * kCrcWarps - 1) / (2 * kCrcWarps), 1, kCrcThreads, &grid,
                                  false);
  if (rc != KV_OK || grid == 0) return rc;
  void* args[] = {const_cast<CrcParams*>(&p)};
  return dbg_launch(stream, [&] {
    return cudaLaunchKernel(k, dim3(grid), dim3(kCrcThreads), args, kCrcSmem, (cudaStream_t)stream);
  }, p);
}

}  // namespace kvc
