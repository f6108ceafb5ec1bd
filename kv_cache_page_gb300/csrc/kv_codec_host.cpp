// kv_codec_host.cpp -- the C ABI: geometry validation, codec tables, launches.
//
// The handle is a validated copy of the registered geometry plus the tables
// the kernels need (sign bits, Lloyd-Max codebook, FP8 fixed scales); it lives
// in host memory and travels to every launch as the kernel parameter block.
// "KV precision and storage encoding" (OrbitKV), section "FP8 and
// TurboQuant": the manager validates dtype, head dimension, strides and K/V
// roles for vLLM's packed [block, head, token, 2 x head_dim] layout and for
// separate K/V tensors, and never infers the head layout from byte counts.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>

#include <cstddef>

#include "kv_codec.h"
#include "kv_internal.h"

struct kv_codec_s {
  kvc::Params p;       // geometry part filled at create; call part per call
  kvc::CrcParams crc;  // seal / verify: tables and per-role constants filled at create
};

namespace {

using kvc::Params;

bool valid_codec(uint32_t c) { return c <= KV_CODEC_UNIFORM2; }
bool is_fp8(uint32_t c) { return c >= KV_CODEC_FP8_CAST && c <= KV_CODEC_FP8_DYNAMIC; }
bool is_tq(uint32_t c) { return c == KV_CODEC_TQ2 || c == KV_CODEC_TQ3 || c == KV_CODEC_TQ4; }
uint32_t codec_bits(uint32_t c) {
  switch (c) {
    case KV_CODEC_TQ2: case KV_CODEC_UNIFORM2: return 2;
    case KV_CODEC_TQ3: case KV_CODEC_UNIFORM3: return 3;
    case KV_CODEC_TQ4: case KV_CODEC_UNIFORM4: return 4;
    case KV_CODEC_UNIFORM8: return 8;
  }
  return 0;
}
bool supported_dim(uint32_t d) { return d == 32 || d == 64 || d == 128 || d == 256; }

// --- SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): golden-gamma increment and
// the variant-13 finalizer.  Bit i of the sign stream is bit (i mod 64) of the
// (i div 64)-th output; 1 negates element i.
uint64_t splitmix_next(uint64_t& state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void sign_words(uint64_t seed, uint32_t D, uint32_t* words /* D/32 */) {
  uint64_t st = seed;
  for (uint32_t k = 0; k < D / 64; ++k) {
    const uint64_t w = splitmix_next(st);
    words[2 * k] = (uint32_t)w;
    words[2 * k + 1] = (uint32_t)(w >> 32);
  }
  if (D == 32) words[0] = (uint32_t)splitmix_next(st);
}

// --- Gaussian Lloyd-Max quantizer with K = 2^bits levels, solved on the
// positive half-line (the density is symmetric and K is even): boundaries
// t_0 = 0, t_k = (c_k + c_{k+1}) / 2, t_{K/2} = inf; centroid of (a, b) is
// (pdf(a) - pdf(b)) / (Q(a) - Q(b)) with Q the upper tail.  Iterated in FP64
// to its fixed point.  Returns the K/2 positive centroids, ascending.
void lloyd_max_positive(uint32_t bits, double* c) {
  const uint32_t half = (1u << bits) / 2;
  const double inv_sqrt2pi = 0.39894228040143267794;
  auto pdf = [&](double t) { return std::isinf(t) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * t * t); };
  auto tail = [](double t) { return std::isinf(t) ? 0.0 : 0.5 * std::erfc(t / 1.41421356237309504880); };
  for (uint32_t k = 0; k < half; ++k) c[k] = (k + 0.5) * 3.0 / half;
  double t[130];
  for (int it = 0; it < 200000; ++it) {
    t[0] = 0.0;
    for (uint32_t k = 1; k < half; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
    t[half] = INFINITY;
    double change = 0.0;
    for (uint32_t k = 0; k < half; ++k) {
      const double nc = (pdf(t[k]) - pdf(t[k + 1])) / (tail(t[k]) - tail(t[k + 1]));
      change = std::max(change, std::fabs(nc - c[k]));
      c[k] = nc;
    }
    if (change <= 4e-16) break;
  }
}

void make_codebook(uint32_t bits, uint32_t D, float* cent, float* bnd) {
  const uint32_t K = 1u << bits, half = K / 2;
  double pos[64];
  lloyd_max_positive(bits, pos);
  double full[128];
  for (uint32_t k = 0; k < half; ++k) {
    full[half + k] = pos[k];
    full[half - 1 - k] = -pos[k];
  }
  const double rs = std::sqrt((double)D);
  for (uint32_t j = 0; j < K; ++j) cent[j] = (float)(full[j] / rs);
  for (uint32_t j = 0; j + 1 < K; ++j) bnd[j] = (float)((0.5 * (full[j] + full[j + 1])) / rs);
}

// Boundaries of the scaled domain moved to the unscaled WHT output:
// W_j = max{w : RN(w * c) <= b_j}; RN(w * c) is monotone in w, so
// RN(w * c) > b_j  <=>  w > W_j.
float unscaled_threshold(float b, float c) {
  volatile float cv = c;  // keep every product a single FP32 rounding
  float w = (float)((double)b / (double)c);
  auto prod = [&](float x) { volatile float y = x * cv; return (float)y; };
  while (prod(w) > b) w = std::nextafterf(w, -INFINITY);
  while (prod(std::nextafterf(w, INFINITY)) <= b) w = std::nextafterf(w, INFINITY);
  return w;
}

// Cell table over c = rint(4 w) in [-kLutHalf, kLutHalf] for the ascending
// thresholds W[0 .. nb): the number of thresholds below every w of the cell
// is lo + (w > thr), thr = the one threshold inside the cell or +inf.
// Returns false if a cell would hold two thresholds.
bool build_cells(const float* W, uint32_t nb, float* thr, uint32_t* lo) {
  for (int cell = -kvc::kLutHalf; cell <= kvc::kLutHalf; ++cell) {
    // floats w with rint(4 w) == cell (4 w is exact; ties go to the even cell)
    const float a = (float)((cell - 0.5) / 4.0), b = (float)((cell + 0.5) / 4.0);
    const float wlo = (cell & 1) ? std::nextafterf(a, INFINITY) : a;
    const float whi = (cell & 1) ? std::nextafterf(b, -INFINITY) : b;
    uint32_t below = 0, inside = 0;
    float t = INFINITY;
    for (uint32_t j = 0; j < nb; ++j) {
      if (W[j] < wlo) ++below;
      else if (W[j] < whi) { ++inside; t = W[j]; }
    }
    if (inside > 1) return false;
    thr[cell + kvc::kLutHalf] = t;
    lo[cell + kvc::kLutHalf] = below;
  }
  return true;
}

// The encoder's index tables.  Direct: code(w) = #{j : W_j < w} with
// W_j = unscaled_threshold(bnd_j).  Mirrored, for lanes that hold v = -w:
// #{j : W_j >= -v} = #{j : v > -succ(W_j)} (succ = next float up), so the
// mirrored table over the thresholds -succ(W_j) gives (2^bits - 1) - code(w),
// the complement of the code's bits.
bool build_index_table(const float* bnd, uint32_t nb, float c, float* thr, uint32_t* lo,
                       float* mthr, uint32_t* mlo) {
  float W[15], M[15];
  for (uint32_t j = 0; j < nb; ++j) W[j] = unscaled_threshold(bnd[j], c);
  for (uint32_t j = 0; j < nb; ++j) M[j] = -std::nextafterf(W[nb - 1 - j], INFINITY);
  return build_cells(W, nb, thr, lo) && build_cells(M, nb, mthr, mlo);
}

// --- CRC-32 (zlib's: reflected polynomial 0xEDB88320) register maps.  A
// GF(2)-linear map of the 32-bit register is kept as the images of its 32
// unit vectors; powers of "advance by one zero byte" come by squaring.
constexpr uint32_t kCrcPoly = 0xEDB88320u;

struct Gf2Map {
  uint32_t col[32];
};

uint32_t gf2_apply(const Gf2Map& m, uint32_t v) {
  uint32_t r = 0;
  for (int j = 0; v; ++j, v >>= 1)
    if (v & 1u) r ^= m.col[j];
  return r;
}

Gf2Map gf2_compose(const Gf2Map& a, const Gf2Map& b) {  // a after b
  Gf2Map c;
  for (int j = 0; j < 32; ++j) c.col[j] = gf2_apply(a, b.col[j]);
  return c;
}

uint32_t crc_bit_steps(uint32_t r, int bits) {
  for (int k = 0; k < bits; ++k) r = (r & 1u) ? (r >> 1) ^ kCrcPoly : (r >> 1);
  return r;
}

// The register r advanced through n zero bytes.
uint32_t crc_advance(uint32_t r, uint64_t n) {
  Gf2Map step;
  for (int j = 0; j < 32; ++j) step.col[j] = crc_bit_steps(1u << j, 8);
  while (n) {
    if (n & 1u) r = gf2_apply(step, r);
    step = gf2_compose(step, step);
    n >>= 1;
  }
  return r;
}

// Nibble tables of the kernels (see CrcTables).  Chunk nibble i = 8 w + k
// sits in byte 4 w + k/2 of the chunk (low half for even k) and is followed by
// 15 - that byte's index bytes of the chunk.
void build_crc_tables(kvc::CrcTables& t) {
  for (int k = 0; k < 4; ++k)
    for (uint32_t v = 0; v < 256; ++v) t.byte[k][v] = crc_advance(crc_bit_steps(v, 8), (uint64_t)k);
  for (int k = 0; k < 8; ++k)
    for (uint32_t v = 0; v < 16; ++v) {
      t.row[k][v] = crc_advance(v << (4 * k), kvc::kCrcRow);
      for (int b = 0; b < 5; ++b) t.fin[b][k][v] = crc_advance(v << (4 * k), (uint64_t)kvc::kCrcBlock << b);
    }
}

const kvc::CrcTables& crc_tables() {
  static kvc::CrcTables tab;
  static std::once_flag once;
  std::call_once(once, [] { build_crc_tables(tab); });
  return tab;
}

// FP8 scale rule: max(amax, 1e-12) * fl32(1/448), in FP32.
float fp8_scale(float amax) {
  const float recip = 1.0f / 448.0f;
  const float a = amax > 1e-12f ? amax : 1e-12f;
  return a * recip;
}

// Non-overlap of the page layout: dims sorted by stride must each step over
// the whole extent of the smaller ones (extent-1 dims do not matter).
bool strides_fit(uint64_t row, int64_t sb, uint64_t nb, int64_t st, uint64_t nt, int64_t sh,
                 uint64_t nh) {
  std::pair<uint64_t, uint64_t> dims[3] = {{(uint64_t)sh, nh}, {(uint64_t)st, nt}, {(uint64_t)sb, nb}};
  std::sort(dims, dims + 3);
  uint64_t span = row;  // elements covered by the smaller dims
  for (auto& d : dims) {
    if (d.second <= 1) continue;
    if (d.first < span) return false;
    // span = stride * (extent - 1) + previous span, watching overflow
    if (d.second - 1 > (uint64_t(1) << 62) / d.first) return false;
    span = d.first * (d.second - 1) + span;
    if (span > (uint64_t(1) << 62)) return false;
  }
  return true;
}

// --- launch bookkeeping: SM count per device, occupancy per (device, kernel)
std::mutex g_mu;
std::map<int, int> g_sms;
std::map<std::pair<int, const void*>, int> g_occ;

// The launches of one encode or decode call: one when both roles share a
// codec, else one per coded role.  With `seal` (one_pass: every coded role FP8,
// uniform-8 or INT8), the launches also write (encode) or first check (decode)
// the segment headers.
int launch_all(kv_codec_s* h, int dir, void* stream, const kvc::CrcParams* seal = nullptr) {
  Params& p = h->p;
  const uint32_t kc = p.codec[0], vc = p.codec[1];
  auto run = [&](uint32_t codec) -> int {
    if (seal)
      return is_fp8(codec)                    ? kvc::launch_fp8_sealed(p, *seal, dir, codec, stream)
             : codec == KV_CODEC_INT8_HEAD ? kvc::launch_int8_sealed(p, *seal, dir, codec, stream)
                                            : kvc::launch_uniform_sealed(p, *seal, dir, codec, stream);
    if (is_fp8(codec)) return kvc::launch_fp8(p, dir, codec, stream);
    if (is_tq(codec)) return kvc::launch_turboquant(p, dir, codec, stream);
    if (codec == KV_CODEC_INT8_HEAD) return kvc::launch_int8(p, dir, codec, stream);
    return kvc::launch_uniform(p, dir, codec, stream);
  };
  if (kc == vc) {
    p.is_first = 1;
    if (kc == KV_CODEC_NONE) {  // statuses only
      p.role_sel = 3;
      return seal ? kvc::launch_fp8_sealed(p, *seal, dir, KV_CODEC_FP8_CAST, stream)
                  : kvc::launch_fp8(p, dir, KV_CODEC_FP8_CAST, stream);
    }
    p.role_sel = 2;
    return run(kc);
  }
  int first = 1;
  for (uint32_t r = 0; r < 2; ++r) {
    const uint32_t c = p.codec[r];
    if (c == KV_CODEC_NONE) continue;
    p.role_sel = r;
    p.is_first = (uint32_t)first;
    first = 0;
    const int rc = run(c);
    if (rc != KV_OK) return rc;
  }
  return KV_OK;
}

// Every coded role takes a codec with sealing / verifying kernels (FP8,
// uniform-8 and HiQ INT8): the headers are written or checked in the codec's
// own pass.
bool one_pass(const Params& p) {
  for (int r = 0; r < 2; ++r) {
    const uint32_t c = p.codec[r];
    if (c != KV_CODEC_NONE && !is_fp8(c) && c != KV_CODEC_UNIFORM8 && c != KV_CODEC_INT8_HEAD) return false;
  }
  return true;
}

// Address under which the kernels reach a caller buffer: device and managed
// memory as they are, pinned host memory through its device mapping (the
// kernels then move its bytes over the CPU-GPU link themselves).  Pageable
// host memory has no such address.
int device_view(const void* ptr, const void** out) {
  *out = nullptr;
  if (!ptr) return KV_OK;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the error this query left
    return KV_ERR_CUDA;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      *out = ptr;
      return KV_OK;
    case cudaMemoryTypeHost:
      if (!a.devicePointer) return KV_ERR_NOT_ACCESSIBLE;
      *out = a.devicePointer;
      return KV_OK;
    default:
      return KV_ERR_NOT_ACCESSIBLE;
  }
}

// The device views of the descriptor, slot, status and result buffers of a call.
int resolve_buffers(Params& p, const kv_segment_desc* descs, const void* buf, const void* status,
                    const void* result) {
  const void* v = nullptr;
  int rc = device_view(descs, &v);
  if (rc != KV_OK) return rc;
  p.descs = static_cast<const kv_segment_desc*>(v);
  if ((rc = device_view(buf, &v)) != KV_OK) return rc;
  p.buf = const_cast<uint8_t*>(static_cast<const uint8_t*>(v));
  if ((rc = device_view(status, &v)) != KV_OK) return rc;
  p.status = const_cast<uint8_t*>(static_cast<const uint8_t*>(v));
  if ((rc = device_view(result, &v)) != KV_OK) return rc;
  p.result = const_cast<uint8_t*>(static_cast<const uint8_t*>(v));
  // a mapping keeps the offset within the page, so the alignment checks on the
  // caller's pointers hold for these addresses too
  return KV_OK;
}

int check_call(kv_codec_s* h, const void* const* layer_ptrs, uint32_t n_layer_ptrs,
               const kv_segment_desc* d_descs, const void* buf, const void* status) {
  const Params& p = h->p;
  const uint32_t want = p.layout == KV_LAYOUT_SEPARATE ? 2 * p.L : p.L;
  if (!layer_ptrs || n_layer_ptrs != want || !d_descs || !buf || !status) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)buf & 15u) || ((uintptr_t)d_descs & 7u)) return KV_ERR_MISALIGNED;
  for (uint32_t k = 0; k < n_layer_ptrs; ++k)
    if ((uintptr_t)layer_ptrs[k] & 15u) return KV_ERR_MISALIGNED;
  return KV_OK;
}

// The per-call CRC parameters: device views of descriptors, slots, statuses
// (seal), headers and result (verify).
int crc_call(kv_codec_t h, kvc::CrcParams& p, const kv_segment_desc* descs, uint32_t n_segments,
             const void* buf, uint64_t buf_bytes, const uint8_t* status, const kv_segment_header* headers,
             uint8_t* result) {
  p = h->crc;
  const void* v = nullptr;
  int rc;
  if ((rc = device_view(descs, &v)) != KV_OK) return rc;
  p.descs = static_cast<const kv_segment_desc*>(v);
  if ((rc = device_view(buf, &v)) != KV_OK) return rc;
  p.buf = static_cast<const uint8_t*>(v);
  if ((rc = device_view(status, &v)) != KV_OK) return rc;
  p.status = static_cast<const uint8_t*>(v);
  if ((rc = device_view(headers, &v)) != KV_OK) return rc;
  p.headers = const_cast<kv_segment_header*>(static_cast<const kv_segment_header*>(v));
  if ((rc = device_view(result, &v)) != KV_OK) return rc;
  p.result = static_cast<uint8_t*>(const_cast<void*>(v));
  p.n_segments = n_segments;
  p.buf_bytes = buf_bytes;
  return KV_OK;
}

}  // namespace

namespace kvc {
int grid_for(const void* kernel, uint32_t n_segments, int max_per_sm, unsigned* grid) {
  return grid_for_threads(kernel, n_segments, max_per_sm, kThreads, grid);
}

int grid_for_threads(const void* kernel, uint32_t n_segments, int max_per_sm, int threads, unsigned* grid,
                     bool odd) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  int sms = 0, occ = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) sms = it->second;
    auto jt = g_occ.find({dev, kernel});
    if (jt != g_occ.end()) occ = jt->second;
  }
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    g_sms[dev] = sms;
  }
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, 0) != cudaSuccess)
      return KV_ERR_CUDA;
    if (occ < 1) occ = 1;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[{dev, kernel}] = occ;
  }
  const int per_sm = std::max(1, std::min(occ, max_per_sm));
  uint64_t g = std::min<uint64_t>((uint64_t)sms * (uint64_t)per_sm, n_segments);
  // An odd stride deals segments of both roles to every CTA when K and V
  // segments alternate in the descriptor list (a launch that codes one role
  // only skips the other role's segments).  Kernels with a segment per warp
  // make their warp stride odd themselves (odd = false).
  if (odd && g > 1 && g < n_segments && (g & 1) == 0) --g;
  *grid = (unsigned)g;
  return KV_OK;
}
}  // namespace kvc

extern "C" {

uint32_t kv_codec_abi_version(void) { return KV_CODEC_ABI_VERSION; }

const char* kv_codec_strerror(int code) {
  switch (code) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_UNSUPPORTED_HEAD_DIM: return "head_dim must be 32, 64, 128 or 256";
    case KV_ERR_LAYOUT_MISMATCH: return "strides overlap or do not fit the layout";
    case KV_ERR_UNSUPPORTED_CODEC_FOR_ROLE: return "TurboQuant codecs are for the K role only";
    case KV_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case KV_ERR_NOT_ACCESSIBLE: return "buffer is pageable host memory (pin it or use device memory)";
    case KV_ERR_UNSUPPORTED_DTYPE: return "codec not defined for this source dtype (INT8_HEAD needs BF16)";
    case KV_ERR_INTERNAL: return "a kernel access fell outside the call's buffers (bounds-checked build)";
    case KV_ERR_CUDA: return "CUDA runtime error";
    case KV_ERR_ABI: return "geometry ABI version or size mismatch";
    case KV_ERR_TOO_MANY_LAYERS: return "num_layers must be 1..KV_CODEC_MAX_LAYERS";
  }
  return "unknown error";
}

int kv_codec_codebook(uint32_t bits, uint32_t head_dim, float* centroids, float* boundaries) {
  if (bits < 1 || bits > 4 || !centroids || !boundaries) return KV_ERR_INVALID_ARG;
  if (!supported_dim(head_dim)) return KV_ERR_UNSUPPORTED_HEAD_DIM;
  make_codebook(bits, head_dim, centroids, boundaries);
  return KV_OK;
}

int kv_codec_signs(uint64_t seed, uint32_t head_dim, uint8_t* negate) {
  if (!negate) return KV_ERR_INVALID_ARG;
  if (!supported_dim(head_dim)) return KV_ERR_UNSUPPORTED_HEAD_DIM;
  uint32_t w[8] = {0};
  sign_words(seed, head_dim, w);
  for (uint32_t i = 0; i < head_dim; ++i) negate[i] = (uint8_t)((w[i >> 5] >> (i & 31)) & 1u);
  return KV_OK;
}

int kv_codec_layer_signs(uint64_t seed, uint32_t layer, uint32_t head_dim, uint8_t* negate) {
  if (!negate || layer >= KV_CODEC_MAX_LAYERS) return KV_ERR_INVALID_ARG;
  if (!supported_dim(head_dim)) return KV_ERR_UNSUPPORTED_HEAD_DIM;
  const uint32_t W = (head_dim + 63) / 64;
  uint64_t st = seed, w = 0;
  for (uint64_t k = 0; k < (uint64_t)layer * W; ++k) splitmix_next(st);  // the layers below
  for (uint32_t i = 0; i < head_dim; ++i) {
    if ((i & 63u) == 0) w = splitmix_next(st);
    negate[i] = (uint8_t)((w >> (i & 63u)) & 1u);
  }
  return KV_OK;
}

static_assert(sizeof(kv_codec_geometry) == 112 && offsetof(kv_codec_geometry, fixed_overflow) == KV_CODEC_GEOMETRY_SIZE_V1,
              "the geometry grows at its end only");

int kv_codec_create(const kv_codec_geometry* g, kv_codec_t* out) {
  if (!out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!g) return KV_ERR_INVALID_ARG;
  if (g->abi_version != KV_CODEC_ABI_VERSION ||
      (g->struct_size != sizeof(kv_codec_geometry) && g->struct_size != KV_CODEC_GEOMETRY_SIZE_V1))
    return KV_ERR_ABI;
  // fields past the earlier 104-byte layout are read only when the caller has them
  const bool ext = g->struct_size >= sizeof(kv_codec_geometry);
  const uint32_t fixed_overflow = ext ? g->fixed_overflow : KV_FIXED_OVERFLOW_CLIP;
  if (fixed_overflow > KV_FIXED_OVERFLOW_REJECT || (ext && g->reserved != 0)) return KV_ERR_INVALID_ARG;
  if (g->dtype != KV_DT_FP16 && g->dtype != KV_DT_BF16) return KV_ERR_INVALID_ARG;
  if (g->layout != KV_LAYOUT_SEPARATE && g->layout != KV_LAYOUT_VLLM_PACKED) return KV_ERR_INVALID_ARG;
  if (!supported_dim(g->head_dim)) return KV_ERR_UNSUPPORTED_HEAD_DIM;
  if (g->num_layers == 0 || g->num_layers > KV_CODEC_MAX_LAYERS) return KV_ERR_TOO_MANY_LAYERS;
  if (g->num_kv_heads == 0 || g->block_tokens == 0 || g->num_blocks == 0 || g->sign_version > 2)
    return KV_ERR_INVALID_ARG;
  const uint64_t nv = (uint64_t)g->num_kv_heads * g->block_tokens;
  if (nv > (1u << 20) || g->num_kv_heads > 4096) return KV_ERR_INVALID_ARG;
  if (!valid_codec(g->k_codec) || !valid_codec(g->v_codec)) return KV_ERR_INVALID_ARG;
  if (is_tq(g->v_codec)) return KV_ERR_UNSUPPORTED_CODEC_FOR_ROLE;
  if ((g->k_codec == KV_CODEC_INT8_HEAD || g->v_codec == KV_CODEC_INT8_HEAD) && g->dtype != KV_DT_BF16)
    return KV_ERR_UNSUPPORTED_DTYPE;
  float reject = g->reject_abs == 0.0f ? 448.0f : g->reject_abs;
  if (!(reject > 0.0f && reject <= 448.0f)) return KV_ERR_INVALID_ARG;
  if (g->stride_block <= 0 || g->stride_token <= 0 || g->stride_head <= 0) return KV_ERR_LAYOUT_MISMATCH;
  if ((g->stride_block | g->stride_token | g->stride_head) & 7) return KV_ERR_MISALIGNED;
  const uint64_t row = g->layout == KV_LAYOUT_SEPARATE ? g->head_dim : 2ull * g->head_dim;
  if (!strides_fit(row, g->stride_block, g->num_blocks, g->stride_token, g->block_tokens,
                   g->stride_head, g->num_kv_heads))
    return KV_ERR_LAYOUT_MISMATCH;
  const bool fixed = g->k_codec == KV_CODEC_FP8_FIXED || g->v_codec == KV_CODEC_FP8_FIXED;
  if (fixed) {
    if (!g->fixed_amax) return KV_ERR_INVALID_ARG;
    for (uint32_t k = 0; k < 2 * g->num_layers; ++k)
      if (!(std::isfinite(g->fixed_amax[k]) && g->fixed_amax[k] >= 0.0f)) return KV_ERR_INVALID_ARG;
  }

  kv_codec_s* h = new (std::nothrow) kv_codec_s;
  if (!h) return KV_ERR_INVALID_ARG;
  std::memset(h, 0, sizeof(*h));
  Params& p = h->p;
  p.dtype = g->dtype;
  p.layout = g->layout;
  p.D = g->head_dim;
  p.H = g->num_kv_heads;
  p.T = g->block_tokens;
  p.L = g->num_layers;
  p.nv = (uint32_t)nv;
  p.n_layer_ptrs = g->layout == KV_LAYOUT_SEPARATE ? 2 * g->num_layers : g->num_layers;
  p.num_blocks = g->num_blocks;
  p.h_magic = ((1ull << 32) + p.H - 1) / p.H;
  p.heads_contig = (uint64_t)g->stride_token == (uint64_t)g->stride_head * g->num_kv_heads ? 1 : 0;
  p.sb = g->stride_block;
  p.st = g->stride_token;
  p.sh = g->stride_head;
  p.codec[0] = g->k_codec;
  p.codec[1] = g->v_codec;
  p.protect_first = g->protect_first;
  p.protect_last = g->protect_last;
  p.reject_abs = reject;
  p.wht_scale = (float)(1.0 / std::sqrt((double)g->head_dim));
  p.neg_zero = -0.0f;
  const uint64_t raw = nv * g->head_dim * 2;
  // INT8_HEAD token record: H int8 head vectors + H BF16 scales, 128-byte multiple
  p.rec_used = p.H * (p.D + 2);
  p.rec_bytes = (p.rec_used + 127) / 128 * 128;
  for (int r = 0; r < 2; ++r) {
    const uint32_t c = p.codec[r];
    uint32_t cb = 0, mb = 0;
    if (is_fp8(c)) {
      cb = p.D;
      mb = c == KV_CODEC_FP8_DYNAMIC ? 4 : 0;
    } else if (c == KV_CODEC_INT8_HEAD) {
      cb = p.D;
      mb = 2;
    } else if (c != KV_CODEC_NONE) {
      cb = p.D * codec_bits(c) / 8;
      mb = is_tq(c) ? 2 : 4;
    }
    p.code_bytes[r] = cb;
    p.meta_bytes[r] = mb;
    p.seg_bytes[r] = c == KV_CODEC_INT8_HEAD ? (uint64_t)p.T * p.rec_bytes
                                             : (nv * (cb + mb) + 127) / 128 * 128;
    uint8_t st = 0;
    if (c != KV_CODEC_NONE) {
      if (raw > (16ull << 20)) st = KV_SEG_RAW_OVERSIZE;
      else if (8 * p.seg_bytes[r] > 7 * raw) st = KV_SEG_RAW_NO_SAVING;
    }
    p.static_status[r] = st;
  }
  p.sign_seed = g->rotation_seed;
  p.sign_per_layer = g->sign_version == 2 ? 1u : 0u;
  p.fixed_reject = fixed_overflow == KV_FIXED_OVERFLOW_REJECT ? 1u : 0u;
  if (is_tq(g->k_codec)) {
    const uint32_t bits = codec_bits(g->k_codec);
    make_codebook(bits, p.D, p.cent, p.bnd);
    if (!build_index_table(p.bnd, (1u << bits) - 1u, p.wht_scale, p.lut_thr, p.lut_lo, p.lut_mthr,
                           p.lut_mlo)) {
      delete h;
      return KV_ERR_INVALID_ARG;
    }
  }
  if (fixed)
    for (uint32_t l = 0; l < p.L; ++l)
      for (int r = 0; r < 2; ++r) p.fixed_scale[l][r] = fp8_scale(g->fixed_amax[2 * l + r]);
  // seal / verify constants
  kvc::CrcParams& c = h->crc;
  c.tab = crc_tables();
  c.L = p.L;
  c.num_blocks = p.num_blocks;
  c.orig_bytes = raw;
  c.version = g->sign_version == 2 ? KV_SEGMENT_FORMAT_VERSION_2 : KV_SEGMENT_FORMAT_VERSION;
  uint32_t lg = 0;
  while ((1u << lg) < p.D) ++lg;
  for (int r = 0; r < 2; ++r) {
    c.codec[r] = p.codec[r];
    c.format[r] = p.codec[r] | (p.dtype << 8) | (lg << 16);
    c.seg_bytes[r] = p.seg_bytes[r];
    c.crc_k[r] = crc_advance(0xFFFFFFFFu, p.seg_bytes[r]) ^ 0xFFFFFFFFu;
  }
  *out = h;
  return KV_OK;
}

int kv_codec_destroy(kv_codec_t h) {
  if (!h) return KV_ERR_INVALID_ARG;
  delete h;
  return KV_OK;
}

int kv_codec_segment_bytes(kv_codec_t h, uint32_t role, uint64_t* enc_bytes, uint64_t* raw_bytes) {
  if (!h || role > 1) return KV_ERR_INVALID_ARG;
  if (enc_bytes) *enc_bytes = h->p.codec[role] == KV_CODEC_NONE ? 0 : h->p.seg_bytes[role];
  if (raw_bytes) *raw_bytes = (uint64_t)h->p.nv * h->p.D * 2;
  return KV_OK;
}

// Every vector of every page starts on a 32-byte boundary: the layer
// pointers are 32-byte aligned and every stride is a multiple of 16
// elements (the packed layout's V half starts D elements in, D >= 32).
uint8_t vectors_32b_aligned(const kvc::Params& p) {
  if ((p.sb | p.st | p.sh) & 15) return 0;
  for (uint32_t k = 0; k < p.n_layer_ptrs; ++k)
    if ((uintptr_t)p.layer_ptr[k] & 31u) return 0;
  return 1;
}

int kv_codec_encode(kv_codec_t h, const void* const* layer_ptrs, uint32_t n_layer_ptrs,
                    const kv_segment_desc* d_descs, uint32_t n_segments, void* d_out,
                    uint64_t out_bytes, uint8_t* d_status, void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  const int rc = check_call(h, layer_ptrs, n_layer_ptrs, d_descs, d_out, d_status);
  if (rc != KV_OK) return rc;
  kv_codec_s call = *h;  // per-call copy: the handle stays immutable
  Params& p = call.p;
  for (uint32_t k = 0; k < n_layer_ptrs; ++k) p.layer_ptr[k] = layer_ptrs[k];
  p.vec32 = vectors_32b_aligned(p);
  const int rv = resolve_buffers(p, d_descs, d_out, d_status, nullptr);
  if (rv != KV_OK) return rv;
  p.n_segments = n_segments;
  p.buf_bytes = out_bytes;
  return launch_all(&call, kvc::kEncode, stream);
}

int kv_codec_seal(kv_codec_t h, const kv_segment_desc* descs, uint32_t n_segments, const void* buf,
                  uint64_t buf_bytes, const uint8_t* status, kv_segment_header* headers, void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  if (!descs || !buf || !status || !headers) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)buf & 15u) || ((uintptr_t)descs & 7u) || ((uintptr_t)headers & 7u))
    return KV_ERR_MISALIGNED;
  kvc::CrcParams p;
  const int rc = crc_call(h, p, descs, n_segments, buf, buf_bytes, status, headers, nullptr);
  return rc != KV_OK ? rc : kvc::launch_crc(p, 1, stream);
}

int kv_codec_verify(kv_codec_t h, const kv_segment_desc* descs, uint32_t n_segments, const void* buf,
                    uint64_t buf_bytes, const kv_segment_header* headers, uint8_t* result,
                    void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  if (!descs || !buf || !headers || !result) return KV_ERR_INVALID_ARG;
  if (((uintptr_t)buf & 15u) || ((uintptr_t)descs & 7u) || ((uintptr_t)headers & 7u))
    return KV_ERR_MISALIGNED;
  kvc::CrcParams p;
  const int rc = crc_call(h, p, descs, n_segments, buf, buf_bytes, nullptr, headers, result);
  return rc != KV_OK ? rc : kvc::launch_crc(p, 0, stream);
}

int kv_codec_encode_sealed(kv_codec_t h, const void* const* layer_ptrs, uint32_t n_layer_ptrs,
                           const kv_segment_desc* descs, uint32_t n_segments, void* out, uint64_t out_bytes,
                           uint8_t* status, kv_segment_header* headers, void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  int rc = check_call(h, layer_ptrs, n_layer_ptrs, descs, out, status);
  if (rc != KV_OK) return rc;
  if (!headers) return KV_ERR_INVALID_ARG;
  if ((uintptr_t)headers & 7u) return KV_ERR_MISALIGNED;
  kv_codec_s call = *h;
  Params& p = call.p;
  for (uint32_t k = 0; k < n_layer_ptrs; ++k) p.layer_ptr[k] = layer_ptrs[k];
  p.vec32 = vectors_32b_aligned(p);
  if ((rc = resolve_buffers(p, descs, out, status, nullptr)) != KV_OK) return rc;
  p.n_segments = n_segments;
  p.buf_bytes = out_bytes;
  kvc::CrcParams q;
  if ((rc = crc_call(h, q, descs, n_segments, out, out_bytes, status, headers, nullptr)) != KV_OK) return rc;
  if (one_pass(p)) return launch_all(&call, kvc::kEncode, stream, &q);
  // other codecs: encode, then seal the slots in a second pass
  if ((rc = launch_all(&call, kvc::kEncode, stream)) != KV_OK) return rc;
  return kvc::launch_crc(q, 1, stream);
}

int kv_codec_decode_verified(kv_codec_t h, void* const* layer_ptrs, uint32_t n_layer_ptrs,
                             const kv_segment_desc* descs, uint32_t n_segments, const void* in,
                             uint64_t in_bytes, const kv_segment_header* headers, uint8_t* result,
                             void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  int rc = check_call(h, layer_ptrs, n_layer_ptrs, descs, in, result);
  if (rc != KV_OK) return rc;
  if (!headers) return KV_ERR_INVALID_ARG;
  if ((uintptr_t)headers & 7u) return KV_ERR_MISALIGNED;
  kv_codec_s call = *h;
  Params& p = call.p;
  for (uint32_t k = 0; k < n_layer_ptrs; ++k) p.layer_ptr[k] = layer_ptrs[k];
  p.vec32 = vectors_32b_aligned(p);
  // other codecs decode with the verified results as their statuses, which
  // they then overwrite with the final results (same array)
  if ((rc = resolve_buffers(p, descs, in, result, result)) != KV_OK) return rc;
  p.status_is_result = 1;
  p.n_segments = n_segments;
  p.buf_bytes = in_bytes;
  kvc::CrcParams q;
  if ((rc = crc_call(h, q, descs, n_segments, in, in_bytes, nullptr, headers, result)) != KV_OK) return rc;
  if (one_pass(p)) return launch_all(&call, kvc::kDecode, stream, &q);
  if ((rc = kvc::launch_crc(q, 0, stream)) != KV_OK) return rc;
  return launch_all(&call, kvc::kDecode, stream);
}

int kv_codec_decode(kv_codec_t h, void* const* layer_ptrs, uint32_t n_layer_ptrs,
                    const kv_segment_desc* d_descs, uint32_t n_segments, const void* d_in,
                    uint64_t in_bytes, const uint8_t* d_status, uint8_t* d_result, void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  if (n_segments == 0) return KV_OK;
  if (n_segments > KV_CODEC_MAX_SEGMENTS) return KV_ERR_INVALID_ARG;
  const int rc = check_call(h, layer_ptrs, n_layer_ptrs, d_descs, d_in, d_status);
  if (rc != KV_OK) return rc;
  kv_codec_s call = *h;
  Params& p = call.p;
  for (uint32_t k = 0; k < n_layer_ptrs; ++k) p.layer_ptr[k] = layer_ptrs[k];
  p.vec32 = vectors_32b_aligned(p);
  const int rv = resolve_buffers(p, d_descs, d_in, d_status, d_result);
  if (rv != KV_OK) return rv;
  p.n_segments = n_segments;
  p.buf_bytes = in_bytes;
  return launch_all(&call, kvc::kDecode, stream);
}

}  // extern "C"
