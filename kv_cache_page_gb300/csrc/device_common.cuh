// device_common.cuh -- segment planning, streaming loads and number-format
// helpers shared by the codec kernels.
//
// Thread mapping: a vector of D elements is held by G consecutive lanes.  The
// streaming codecs (FP8, INT8, uniform-8 encode, every uniform decode) use
// ChunkMap below: the vector's 16-byte chunks dealt round-robin to its lanes,
// so each warp load and store covers whole contiguous runs.  TurboQuant and
// the 2/3/4-bit uniform encoders give each lane 32 contiguous elements
// (G = D/32).  A warp holds 32/G vectors at a time and each lane handles U
// such vectors per step, so that several independent 128-bit loads are in
// flight per thread.  A CTA owns one segment at a time and walks the
// segment's vectors in token-major order j = t*H + h, which is also the order
// of the encoded slot.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kv_internal.h"
#ifdef KVC_BOUNDS_CHECK
#include <cstdlib>
#include <mutex>
#endif

namespace kvc {

// ---------------------------------------------------------------- bounds check
// The debug build (-DKVC_BOUNDS_CHECK: libkvcodec_debug.so) checks every
// global load and store of the kernels.  Its bytes must lie inside one of the
// buffers the call was given: a layer tensor (from its first element to the
// last one the registered strides reach), the slot buffer, the descriptors,
// statuses, results or headers.  The launcher writes these ranges into this
// translation unit's g_dbg before each launch.  An access outside them is
// skipped (a load gives zeros) and counted, with the first such address, and
// the call returns KV_ERR_INTERNAL.  The release build compiles every check
// away.
#ifdef KVC_BOUNDS_CHECK
constexpr int kDbgMaxRanges = 2 * kMaxLayers + 8;
struct DbgRanges {
  uint32_t n;
  uint64_t lo[kDbgMaxRanges];
  uint64_t hi[kDbgMaxRanges];  // exclusive
};
static __constant__ DbgRanges g_dbg;
static __device__ unsigned int g_dbg_count;
static __device__ unsigned long long g_dbg_first;

static __device__ __noinline__ bool dbg_ok(const void* ptr, uint32_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(ptr), e = a + bytes;
  for (uint32_t k = 0; k < g_dbg.n; ++k)
    if (a >= g_dbg.lo[k] && e <= g_dbg.hi[k]) return true;
  if (atomicAdd(&g_dbg_count, 1u) == 0u) g_dbg_first = a;
  return false;
}
// On an access outside the call's buffers: the statements after `bytes`
// (typically a return) instead of the access.
#define KVC_GUARD(ptr, bytes, ...)                  \
  do {                                              \
    if (!::kvc::dbg_ok((ptr), (bytes))) {           \
      __VA_ARGS__;                                  \
    }                                               \
  } while (0)

inline void dbg_add(DbgRanges& r, const void* base, uint64_t bytes) {
  if (base && bytes && r.n < (uint32_t)kDbgMaxRanges) {
    r.lo[r.n] = reinterpret_cast<uint64_t>(base);
    r.hi[r.n] = r.lo[r.n] + bytes;
    ++r.n;
  }
}
// Slot-buffer bytes the check accepts.  KVC_DEBUG_SLOT_MARGIN (bytes) holds
// back the end of the buffer, so that a test can see the check fire on
// accesses that are in fact in bounds.
inline uint64_t dbg_slot_bytes(uint64_t buf_bytes) {
  const char* m = std::getenv("KVC_DEBUG_SLOT_MARGIN");
  const uint64_t cut = m ? std::strtoull(m, nullptr, 10) : 0u;
  return cut < buf_bytes ? buf_bytes - cut : 0u;
}
inline void dbg_ranges(DbgRanges& r, const Params& p) {
  const uint64_t row = p.layout == KV_LAYOUT_VLLM_PACKED ? 2ull * p.D : p.D;
  const uint64_t last = (uint64_t)p.sb * (p.num_blocks - 1u) + (uint64_t)p.st * (p.T - 1u) +
                        (uint64_t)p.sh * (p.H - 1u);
  const uint32_t nptr = p.layout == KV_LAYOUT_SEPARATE ? 2u * p.L : p.L;
  for (uint32_t k = 0; k < nptr; ++k) dbg_add(r, p.layer_ptr[k], 2u * (last + row));
  dbg_add(r, p.buf, dbg_slot_bytes(p.buf_bytes));
  dbg_add(r, p.descs, (uint64_t)p.n_segments * sizeof(kv_segment_desc));
  dbg_add(r, p.status, p.n_segments);
  dbg_add(r, p.result, p.n_segments);
}
inline void dbg_ranges(DbgRanges& r, const CrcParams& q) {
  dbg_add(r, q.buf, dbg_slot_bytes(q.buf_bytes));
  dbg_add(r, q.descs, (uint64_t)q.n_segments * sizeof(kv_segment_desc));
  dbg_add(r, q.status, q.n_segments);
  dbg_add(r, q.result, q.n_segments);
  dbg_add(r, q.headers, (uint64_t)q.n_segments * sizeof(kv_segment_header));
}
// One checked launch at a time per translation unit (the ranges and the
// counter are the unit's own); the launch is waited for.
static std::mutex& dbg_mutex() {
  static std::mutex m;
  return m;
}
static int dbg_begin(const DbgRanges& r, void* stream) {
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_dbg, &r, sizeof r, 0, cudaMemcpyHostToDevice, (cudaStream_t)stream) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_dbg_count, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              (cudaStream_t)stream) != cudaSuccess)
    return KV_ERR_CUDA;
  return KV_OK;
}
static int dbg_end(void* stream) {
  unsigned int n = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess ||
      cudaMemcpyFromSymbol(&n, g_dbg_count, sizeof n) != cudaSuccess)
    return KV_ERR_CUDA;
  return n ? KV_ERR_INTERNAL : KV_OK;
}
// Launch `launch` (a callable returning a cudaError_t) with the check armed
// for the ranges of the given parameter blocks.
template <typename F, typename... Ps>
static int dbg_launch(void* stream, F launch, const Ps&... ps) {
  DbgRanges r;
  r.n = 0;
  (dbg_ranges(r, ps), ...);
  std::lock_guard<std::mutex> g(dbg_mutex());
  if (dbg_begin(r, stream) != KV_OK) return KV_ERR_CUDA;
  if (launch() != cudaSuccess) return KV_ERR_CUDA;
  return dbg_end(stream);
}
#else
#define KVC_GUARD(ptr, bytes, ...) \
  do {                             \
  } while (0)
// Release: launch `launch` and map its status.
template <typename F, typename... Ps>
inline int dbg_launch(void*, F launch, const Ps&...) {
  return launch() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}
#endif

// Scalar global loads and stores of the kernels (every one bounds-checked in
// the debug build).
__device__ __forceinline__ uint32_t ldg_u32(const uint32_t* ptr) {
  KVC_GUARD(ptr, 4, return 0u);
  return __ldg(ptr);
}
__device__ __forceinline__ uint64_t ldg_u64(const void* ptr) {
  KVC_GUARD(ptr, 8, return 0u);
  return __ldg(reinterpret_cast<const unsigned long long*>(ptr));
}
__device__ __forceinline__ uint8_t ldg_u8(const uint8_t* ptr) {
  KVC_GUARD(ptr, 1, return 0u);
  return __ldg(ptr);
}
// coherent byte load (an array this launch also writes)
__device__ __forceinline__ uint8_t ld_volatile_u8(const uint8_t* ptr) {
  KVC_GUARD(ptr, 1, return 0u);
  return *(const volatile uint8_t*)ptr;
}
__device__ __forceinline__ uint8_t ld_u8(const uint8_t* ptr) {
  KVC_GUARD(ptr, 1, return 0u);
  return *ptr;
}
__device__ __forceinline__ void st_u8(uint8_t* ptr, uint8_t v) {
  KVC_GUARD(ptr, 1, return);
  *ptr = v;
}
__device__ __forceinline__ void st_u16(void* ptr, uint16_t v) {
  KVC_GUARD(ptr, 2, return);
  *reinterpret_cast<uint16_t*>(ptr) = v;
}
__device__ __forceinline__ void st_u64(void* ptr, uint64_t v) {
  KVC_GUARD(ptr, 8, return);
  *reinterpret_cast<uint64_t*>(ptr) = v;
}

// ---------------------------------------------------------------- planning
enum Action { kProcess = 0, kReport = 1, kSkip = 2 };

struct Seg {
  int action;
  uint8_t status;        // kReport: the byte to write
  uint32_t role;
  uint32_t layer;
  const uint16_t* page;  // first element of this role's vectors of the page
  uint8_t* slot;         // encoded slot
};

// Decide what this CTA does with segment i.  Uniform across the CTA.
// Ownership: a launch that codes one role (role_sel 0 or 1) owns the
// descriptors of that role; the first launch also owns descriptors with an
// invalid role or a role without codec.  Descriptors of the other coded role
// are skipped after reading just the role field.  Decode takes the segment's
// status from `given` when it is not negative, else from p.status (a coherent
// load when p.status is the result array this launch writes, each entry
// rewritten only by its owner with a value that leads to the same plan).
__device__ __forceinline__ bool owns_segment(const Params& p, uint32_t role) {
  const bool coded_role = role <= 1u && p.codec[role] != KV_CODEC_NONE;
  return coded_role ? (p.role_sel == 2u || role == p.role_sel) : (p.is_first != 0u);
}

__device__ __forceinline__ Seg plan_segment(const Params& p, uint32_t i, int dir, int given = -1) {
  Seg s;
  const kv_segment_desc* dp = p.descs + i;
  // all fields in one round trip
  const uint32_t layer = ldg_u32(&dp->layer), block = ldg_u32(&dp->block), role = ldg_u32(&dp->role);
  const uint64_t off = ldg_u64(&dp->enc_offset);
  s.role = role;
  s.layer = layer;
  s.page = nullptr;
  s.slot = nullptr;
  s.status = 0;
  const bool coded_role = role <= 1u && p.codec[role] != KV_CODEC_NONE;
  if (!owns_segment(p, role)) {
    s.action = kSkip;
    return s;
  }
  bool ok = layer < p.L && role <= 1u && (uint64_t)block < p.num_blocks && (off & 15u) == 0;
  const void* base = nullptr;
  if (ok) {
    base = p.layout == KV_LAYOUT_SEPARATE ? p.layer_ptr[2 * layer + role] : p.layer_ptr[layer];
    const uint64_t need = p.seg_bytes[role];
    ok = base != nullptr && off <= p.buf_bytes && need <= p.buf_bytes - off;
  }
  s.action = kReport;
  if (!ok) {
    s.status = (uint8_t)KV_SEG_BAD_DESC;
    return s;
  }
  if (!coded_role) {
    s.status = dir == kEncode ? (uint8_t)KV_SEG_RAW_POLICY : (uint8_t)KV_SEG_BAD_DESC;
    return s;
  }
  if (dir == kEncode) {
    if (layer < p.protect_first || layer + p.protect_last >= p.L) {
      s.status = (uint8_t)KV_SEG_RAW_PROTECTED;
      return s;
    }
    if (p.static_status[role]) {
      s.status = p.static_status[role];
      return s;
    }
  } else {
    const uint8_t st = given >= 0          ? (uint8_t)given
                       : p.status_is_result ? ld_volatile_u8(p.status + i)
                                            : ldg_u8(p.status + i);
    if (st != (uint8_t)KV_SEG_ENCODED) {
      s.status = st;
      return s;
    }
  }
  int64_t e = (int64_t)block * p.sb;
  if (p.layout == KV_LAYOUT_VLLM_PACKED) e += (int64_t)role * p.D;
  s.page = reinterpret_cast<const uint16_t*>(base) + e;
  s.slot = p.buf + off;
  s.action = kProcess;
  return s;
}

// The segments of a CTA are blockIdx.x, blockIdx.x + gridDim.x, ...  A cursor
// plans 32 upcoming candidates at once, one per lane (every warp of the CTA
// holds the same cursor), writes the status (encode) or result (decode) of
// those the launch only reports (warp 0 does the writing), and hands out the
// ones it codes in order, re-planning each from its (now cached) descriptor.
// The descriptor loads from memory are paid once per 32 segments.
struct SegCursor {
  uint32_t base;   // candidate index of lane 0
  uint32_t mask;   // candidates of this batch still to hand out
  uint32_t stride; // distance between the owner's segments
};

__device__ __forceinline__ void cursor_init(SegCursor& c) {
  c.base = blockIdx.x;
  c.mask = 0;
  c.stride = gridDim.x;
}

// One warp per segment: warp w of CTA b owns segments g, g + S, g + 2S, ...
// with g = b * warps_per_cta + w and S the number of warps, made odd (one
// warp idles when it is even) so that alternating K / V descriptors reach
// every warp.  Such a cursor is private to its warp, which writes the
// statuses of the segments it only reports.
__device__ __forceinline__ void warp_cursor_init(SegCursor& c, uint32_t warps_per_cta) {
  const uint32_t total = gridDim.x * warps_per_cta;
  c.stride = (total > 1u && (total & 1u) == 0u) ? total - 1u : total;
  c.base = blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
  if (c.base >= c.stride) c.base = 0xffffffffu;  // the idle warp of an even count
  c.mask = 0;
}

// Next segment index to code (and its plan in s), or 0xffffffff when done.
// WARP: the cursor was set up by warp_cursor_init (every warp reports its own
// candidates); otherwise warp 0 of the CTA reports.
template <int DIR, bool WARP = false>
__device__ __forceinline__ uint32_t cursor_next(const Params& p, SegCursor& c, Seg& s) {
  while (c.mask == 0u) {
    if (c.base >= p.n_segments) return 0xffffffffu;
    const uint32_t i = c.base + (threadIdx.x & 31u) * c.stride;
    bool go = false;
    if (i < p.n_segments) {
      const Seg m = plan_segment(p, i, DIR);
      go = m.action == kProcess;
      if (m.action == kReport && (WARP || threadIdx.x < 32u)) {
        if (DIR == kEncode) st_u8(p.status + i, m.status);
        else if (p.result) st_u8(p.result + i, m.status);
      }
    }
    c.mask = __ballot_sync(0xffffffffu, go);
    if (c.mask == 0u) c.base += 32u * c.stride;
  }
  const uint32_t k = (uint32_t)(__ffs(c.mask) - 1);
  c.mask &= c.mask - 1u;
  const uint32_t idx = c.base + k * c.stride;
  if (c.mask == 0u) c.base += 32u * c.stride;
  s = plan_segment(p, idx, DIR);
  return idx;
}

// Element offset of vector j (token-major) inside its page.
__device__ __forceinline__ int64_t vec_off(const Params& p, uint32_t j) {
  if (p.heads_contig) return (int64_t)j * p.sh;
  const uint32_t t = (uint32_t)(((uint64_t)j * p.h_magic) >> 32);
  const uint32_t h = j - t * p.H;
  return (int64_t)t * p.st + (int64_t)h * p.sh;
}

// ---------------------------------------------------------------- memory
// V: volatile, so that the load stays ahead of later volatile asm (table
// reads a kernel overlaps with the load's latency)
template <bool V = false>
__device__ __forceinline__ uint4 ld_stream16(const void* ptr) {
  KVC_GUARD(ptr, 16, return make_uint4(0, 0, 0, 0));
  uint4 v;
  if (V)
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
  else
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
  return v;
}
// read-only 16-byte load that allocates in L1 (for lanes reading 64-byte
// blocks, whose second half-sector is then served from L1)
__device__ __forceinline__ uint4 ld_nc16(const void* ptr) {
  KVC_GUARD(ptr, 16, return make_uint4(0, 0, 0, 0));
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(ptr));
  return v;
}
// read-only 32-byte load (sm_100+); ptr must be 32-byte aligned
__device__ __forceinline__ void ld_nc32(const void* ptr, uint4& a, uint4& b) {
  KVC_GUARD(ptr, 32, a = b = make_uint4(0, 0, 0, 0); return);
  asm("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(ptr));
}
// coherent 32- and 16-byte loads, for data written earlier in the same launch
// (ordered after the writers' barrier by the memory clobber)
__device__ __forceinline__ void ld_plain32(const void* ptr, uint4& a, uint4& b) {
  KVC_GUARD(ptr, 32, a = b = make_uint4(0, 0, 0, 0); return);
  asm volatile("ld.global.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(ptr)
               : "memory");
}
__device__ __forceinline__ uint4 ld_plain16(const void* ptr) {
  KVC_GUARD(ptr, 16, return make_uint4(0, 0, 0, 0));
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_nc8(const void* ptr) {
  KVC_GUARD(ptr, 8, return make_uint2(0, 0));
  uint2 v;
  asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint32_t ld_nc4(const void* ptr) {
  KVC_GUARD(ptr, 4, return 0u);
  uint32_t v;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint16_t ld_nc2(const void* ptr) {
  KVC_GUARD(ptr, 2, return (uint16_t)0);
  uint16_t v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint4 lds16(uint32_t smem) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem));
  return v;
}
__device__ __forceinline__ void st16(void* ptr, uint4 v) {
  KVC_GUARD(ptr, 16, return);
  *reinterpret_cast<uint4*>(ptr) = v;
}
// 32-byte store (sm_100+); ptr must be 32-byte aligned
__device__ __forceinline__ void st32(void* ptr, const uint4& a, const uint4& b) {
  KVC_GUARD(ptr, 32, return);
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a.x), "r"(a.y),
               "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
__device__ __forceinline__ void st8(void* ptr, uint2 v) {
  KVC_GUARD(ptr, 8, return);
  *reinterpret_cast<uint2*>(ptr) = v;
}
__device__ __forceinline__ void st4(void* ptr, uint32_t v) {
  KVC_GUARD(ptr, 4, return);
  *reinterpret_cast<uint32_t*>(ptr) = v;
}

// L2 eviction priorities.  A policy from createpolicy rides on a load or a
// store as a cache hint: evict_last for bytes that are read again soon (a slot
// checked before it is decoded), evict_first for bytes read or written once.
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Read-only loads and stores, with the policy when H (else as above).
template <bool H>
__device__ __forceinline__ void ld_nc32_h(const void* ptr, uint4& a, uint4& b, uint64_t pol) {
  if (!H) return ld_nc32(ptr, a, b);
  KVC_GUARD(ptr, 32, a = b = make_uint4(0, 0, 0, 0); return);
  asm("ld.global.nc.L2::cache_hint.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(ptr), "l"(pol));
}
template <bool H>
__device__ __forceinline__ uint4 ld_nc16_h(const void* ptr, uint64_t pol) {
  if (!H) return ld_nc16(ptr);
  KVC_GUARD(ptr, 16, return make_uint4(0, 0, 0, 0));
  uint4 v;
  asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(ptr), "l"(pol));
  return v;
}
template <bool H>
__device__ __forceinline__ uint2 ld_nc8_h(const void* ptr, uint64_t pol) {
  if (!H) return ld_nc8(ptr);
  KVC_GUARD(ptr, 8, return make_uint2(0, 0));
  uint2 v;
  asm("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(ptr), "l"(pol));
  return v;
}
template <bool H>
__device__ __forceinline__ uint32_t ld_nc4_h(const void* ptr, uint64_t pol) {
  if (!H) return ld_nc4(ptr);
  KVC_GUARD(ptr, 4, return 0u);
  uint32_t v;
  asm("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(pol));
  return v;
}
template <bool H>
__device__ __forceinline__ void st16_h(void* ptr, uint4 v, uint64_t pol) {
  if (!H) return st16(ptr, v);
  KVC_GUARD(ptr, 16, return);
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
template <bool H>
__device__ __forceinline__ void st32_h(void* ptr, const uint4& a, const uint4& b, uint64_t pol) {
  if (!H) return st32(ptr, a, b);
  KVC_GUARD(ptr, 32, return);
  asm volatile("st.global.L2::cache_hint.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(ptr),
               "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w), "l"(pol)
               : "memory");
}

// Bring `bytes` (a multiple of 16) at `ptr` (16-byte aligned) into L2 without
// waiting for them; a plain hint, its completion is never awaited.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  KVC_GUARD(ptr, bytes, return);
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Zero the alignment padding [used, seg_bytes) of a slot: threads first,
// first + step, ... (the whole CTA: threadIdx.x, blockDim.x; one warp: lane, 32).
__device__ __forceinline__ void zero_padding(uint8_t* slot, uint64_t used, uint64_t total, uint32_t first,
                                             uint32_t step) {
  for (uint64_t k = used + first; k < total; k += step) st_u8(slot + k, 0);
}

// ---------------------------------------------------------------- 16-bit formats
// DT = 0: FP16, DT = 1: BF16.  Two elements per 32-bit word, element 2k in the
// low half (little endian).
template <int DT>
__device__ __forceinline__ uint32_t min_nan2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (DT == 0) asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <int DT>
__device__ __forceinline__ uint32_t max_nan2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (DT == 0) asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <int DT>
__device__ __forceinline__ float lo_f32(uint32_t w) {
  if (DT == 0) return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
  return __uint_as_float(w << 16);
}
template <int DT>
__device__ __forceinline__ float hi_f32(uint32_t w) {
  if (DT == 0) return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
  return __uint_as_float(w & 0xffff0000u);
}
// Round two floats to the 16-bit format (nearest-even), lo in the low half.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t d;
  if (DT == 0) asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  else asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

template <int DT>
__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  x[0] = lo_f32<DT>(w.x); x[1] = hi_f32<DT>(w.x);
  x[2] = lo_f32<DT>(w.y); x[3] = hi_f32<DT>(w.y);
  x[4] = lo_f32<DT>(w.z); x[5] = hi_f32<DT>(w.z);
  x[6] = lo_f32<DT>(w.w); x[7] = hi_f32<DT>(w.w);
}
template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
  return make_uint4(pack2<DT>(y[0], y[1]), pack2<DT>(y[2], y[3]), pack2<DT>(y[4], y[5]),
                    pack2<DT>(y[6], y[7]));
}

// Minimum and maximum of the vector held by G lanes (NC 8-element chunks
// each), NaN propagating, returned as floats (exact: min/max of 16-bit values).
template <int DT, int G, int NC>
__device__ __forceinline__ void vec_minmax(const uint4 (&w)[NC], float& mn, float& mx) {
  uint32_t a = min_nan2<DT>(min_nan2<DT>(w[0].x, w[0].y), min_nan2<DT>(w[0].z, w[0].w));
  uint32_t b = max_nan2<DT>(max_nan2<DT>(w[0].x, w[0].y), max_nan2<DT>(w[0].z, w[0].w));
#pragma unroll
  for (int c = 1; c < NC; ++c) {
    a = min_nan2<DT>(a, min_nan2<DT>(min_nan2<DT>(w[c].x, w[c].y), min_nan2<DT>(w[c].z, w[c].w)));
    b = max_nan2<DT>(b, max_nan2<DT>(max_nan2<DT>(w[c].x, w[c].y), max_nan2<DT>(w[c].z, w[c].w)));
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    a = min_nan2<DT>(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max_nan2<DT>(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  a = min_nan2<DT>(a, __byte_perm(a, 0, 0x1032));
  b = max_nan2<DT>(b, __byte_perm(b, 0, 0x1032));
  mn = lo_f32<DT>(a);
  mx = lo_f32<DT>(b);
}

// max(|a|, |b|) per half, NaN propagating (the sign of the result is the xor
// of the input signs and is ignored by the callers)
template <int DT>
__device__ __forceinline__ uint32_t absmax_nan2(uint32_t a, uint32_t b) {
  uint32_t d;
  if (DT == 0) asm("max.NaN.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest |x| of the vector held by G lanes (NC chunks each), NaN propagating,
// as a float (exact).
template <int DT, int G, int NC>
__device__ __forceinline__ float vec_absmax(const uint4 (&w)[NC]) {
  uint32_t a = absmax_nan2<DT>(absmax_nan2<DT>(w[0].x, w[0].y), absmax_nan2<DT>(w[0].z, w[0].w));
#pragma unroll
  for (int c = 1; c < NC; ++c)
    a = absmax_nan2<DT>(a, absmax_nan2<DT>(absmax_nan2<DT>(w[c].x, w[c].y), absmax_nan2<DT>(w[c].z, w[c].w)));
#pragma unroll
  for (int o = 1; o < G; o <<= 1) a = absmax_nan2<DT>(a, __shfl_xor_sync(0xffffffffu, a, o));
  a = absmax_nan2<DT>(a, __byte_perm(a, 0, 0x1032));
  return fabsf(lo_f32<DT>(a));
}

// Chunk assignment for the order-free codecs (FP8, uniform): the vector's
// 16-byte chunks c = 0 .. D/8-1 are dealt round-robin to its G lanes, lane li
// holding chunks li, li + G, ... (NC of them), so one warp load instruction
// reads G contiguous chunks of each of the warp's 32/G vectors.  G is a
// multiple of 4 for every head dim (the 3-bit packer combines 4 chunks).
// Segments of at least this many vectors take the decoders' adjacent-chunk
// mapping (lane li owns chunks 2li, 2li + 1: one 16-byte code load and one
// 32-byte page store per vector); shorter segments keep the round-robin
// chunks, which measured faster on 128-vector segments.  Shared by the FP8 and
// the uniform decoders so that both switch at the same size.
constexpr uint32_t kAdjacentChunkMinVectors = 256;

template <int D>
struct ChunkMap {
  static constexpr int E = D == 32 ? 8 : 16;   // elements per lane
  static constexpr int G = D / E;               // lanes per vector
  static constexpr int NC = E / 8;              // chunks per lane
  static constexpr int VPW = 32 / G;            // vectors per warp row
  static constexpr int U = NC == 1 ? 4 : 2;     // warp rows per step: 32 or 64 B of loads per lane
};

// ---------------------------------------------------------------- packed FP32x2
// One instruction on two independent FP32 lanes, each rounded to nearest-even
// as its scalar counterpart (sm_100+ packed FP32 arithmetic).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Admission flags of one vector from its largest |x|: bit 0 nonfinite, bit 1 range.
__device__ __forceinline__ uint32_t admission_abs(float amax, float reject) {
  return isfinite(amax) ? (amax > reject ? 2u : 0u) : 1u;
}

// Admission flags of one vector from its min/max: bit 0 nonfinite, bit 1 range.
__device__ __forceinline__ uint32_t admission(float mn, float mx, float reject) {
  const bool nonfinite = !(isfinite(mn) && isfinite(mx));
  const bool range = (mn < -reject) || (mx > reject);
  return nonfinite ? 1u : (range ? 2u : 0u);
}

// ---------------------------------------------------------------- arithmetic
// Correctly rounded x / s from the correctly rounded reciprocal r = RN(1/s):
// q0 = RN(x r), residual e = x - q0 s (exact by FMA), q = RN(q0 + e r) (one
// Newton correction, Markstein 1990), sign copied from x so that -0 / s = -0.
__device__ __forceinline__ float div_by(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q0, s, x);
  return copysignf(__fmaf_rn(e, r, q0), x);
}

// Pairwise sum over the vector (element order) held by G lanes of 8: an
// in-thread tree over the 8 elements, then xor-shuffles with ascending lane
// distance.  Every lane of the group ends with the same bits.
template <int G>
__device__ __forceinline__ float pairwise_sum8(const float (&a)[8]) {
  const float b0 = __fadd_rn(a[0], a[1]), b1 = __fadd_rn(a[2], a[3]);
  const float b2 = __fadd_rn(a[4], a[5]), b3 = __fadd_rn(a[6], a[7]);
  float c = __fadd_rn(__fadd_rn(b0, b1), __fadd_rn(b2, b3));
#pragma unroll
  for (int o = 1; o < G; o <<= 1) c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, o));
  return c;
}

// Walsh-Hadamard butterflies (no scale) over the vector held by G lanes, stride
// h = 1, 2, 4 inside the thread, then h = 8, 16, ... across lanes (lane
// distance h/8).  Pair (a_lo, a_hi) -> (a_lo + a_hi, a_lo - a_hi); across
// lanes each side computes its own output as fma(mine, +-1, partner), which
// is the single rounding of the same sum or difference.
template <int G>
__device__ __forceinline__ void wht_butterflies(float (&a)[8], uint32_t li) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & h) continue;
      const float u = a[i], v = a[i + h];
      a[i] = __fadd_rn(u, v);
      a[i + h] = __fsub_rn(u, v);
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    const float sgn = (li & (uint32_t)o) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float partner = __shfl_xor_sync(0xffffffffu, a[i], o);
      a[i] = __fmaf_rn(a[i], sgn, partner);
    }
  }
}

// 3-bit codes of one 8-element chunk (24 bits, chunk index c of the vector)
// -> the 12-byte little-endian stream of chunks 4q..4q+3, written as three
// words by the lanes holding chunks 4q..4q+2 (the four chunks sit on four
// consecutive lanes).  `dst` points at the vector's code bytes.
__device__ __forceinline__ void store_3bit(uint8_t* dst, uint32_t v24, uint32_t c, bool active) {
  const uint32_t next = __shfl_down_sync(0xffffffffu, v24, 1);
  const uint32_t k = c & 3u;
  if (active && k < 3u) {
    const uint32_t w = (v24 >> (8u * k)) | (next << (24u - 8u * k));
    st4(dst + 12u * (c >> 2) + 4u * k, w);
  }
}

// Inverse of store_3bit: the 24 bits of chunk c from the vector's code bytes.
// Reads at most one word past the chunk, which stays inside the slot (the
// metadata region follows the codes).
__device__ __forceinline__ uint32_t load_3bit(const uint8_t* src, uint32_t c) {
  const uint32_t bit = 24u * c;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(src) + (bit >> 5);
  const uint32_t lo = ld_nc4(w), hi = ld_nc4(w + 1);
  return __funnelshift_r(lo, hi, bit & 31u) & 0xffffffu;
}

// Launch a codec kernel (signature void(Params)) on the caller's stream with
// `threads` threads per CTA and at most `max_per_sm` resident CTAs per SM.
// The caps come from sweeps on a GB300 (one CTA codes one segment): the
// write-heavy decodes stream best with few CTAs per SM, the encodes with more.
// (static: in the debug build each translation unit arms its own
// bounds-check state)
template <typename K>
static int launch_codec_kernel(K kernel, const Params& p, void* stream, int max_per_sm,
                               int threads = kThreads, bool warp_segments = false) {
  unsigned grid = 0;
  // one warp per segment: enough CTAs for every segment to have its warp
  const uint32_t units = warp_segments ? (p.n_segments + (uint32_t)threads / 32u - 1u) / ((uint32_t)threads / 32u)
                                       : p.n_segments;
  const int rc = grid_for_threads(reinterpret_cast<const void*>(kernel), units, max_per_sm,
                                  threads, &grid, !warp_segments);
  if (rc != KV_OK || grid == 0) return rc;
  void* args[] = {const_cast<Params*>(&p)};
  return dbg_launch(stream, [&] {
    return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(grid), dim3(threads), args, 0,
                            (cudaStream_t)stream);
  }, p);
}

}  // namespace kvc
