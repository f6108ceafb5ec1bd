// crc.cu -- segment headers: CRC-32 of encoded slots (seal) and their check
// before decode (verify).
//
// "KV precision and storage encoding" (OrbitKV docs), section "Ownership,
// storage and GDS": each encoded segment carries a version, its original
// length, its format, its stored length and a CRC32; checksums are validated
// before GPU decode, and a damaged object becomes a miss.
//
// The standalone passes: one warp per slot, one 1024-thread CTA per SM holding
// the lookup tables (the CRC itself is in crc_common.cuh).  The FP8 codec
// kernels also seal while they encode and verify before they decode, without
// this second pass over the slots (fp8.cu).
#include "crc_common.cuh"

namespace kvc {
namespace {

using namespace crc;

__global__ void __launch_bounds__(kCrcThreads, 1) crc_seal_kernel(const __grid_constant__ CrcParams p) {
  NibbleTables* t;
  const uint32_t tb = load_tables(p, t);
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (uint32_t i = blockIdx.x * kCrcWarps + warp; i < p.n_segments; i += gridDim.x * kCrcWarps)
    seal_segment<true>(p, *t, tb, i, p.status[i], lane);
}

__global__ void __launch_bounds__(kCrcThreads, 1) crc_verify_kernel(const __grid_constant__ CrcParams p) {
  NibbleTables* t;
  const uint32_t tb = load_tables(p, t);
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (uint32_t i = blockIdx.x * kCrcWarps + warp; i < p.n_segments; i += gridDim.x * kCrcWarps) {
    const uint32_t r = verify_segment(p, *t, tb, i, lane);
    if (lane == 0) p.result[i] = (uint8_t)r;
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
  const int rc = grid_for_threads(k, (p.n_segments + kCrcWarps - 1) / kCrcWarps, 1, kCrcThreads, &grid, false);
  if (rc != KV_OK || grid == 0) return rc;
  void* args[] = {const_cast<CrcParams*>(&p)};
  const cudaError_t e =
      cudaLaunchKernel(k, dim3(grid), dim3(kCrcThreads), args, kCrcSmem, (cudaStream_t)stream);
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // namespace kvc
