// crc_common.cuh -- CRC-32 of encoded slots by a warp (or a half warp), shared
// by the seal / verify kernels and the codec kernels that seal or verify a
// slot in the same pass as they encode or decode it.
//
// "KV precision and storage encoding" (OrbitKV docs), section "Ownership,
// storage and GDS": each encoded segment carries a version, its original
// length, its format, its stored length and a CRC32; checksums are validated
// before GPU decode, and a damaged object becomes a miss.
//
// CRC-32 here is zlib's (reflected polynomial 0xEDB88320, register preset to
// all ones, result complemented).  One warp codes one slot.  With R(M) the
// register of message M fed into a zero register and F_n the map "advance
// the register through n zero bytes" (both GF(2)-linear):
//   CRC(M) = R(M) ^ F_N(~0) ^ ~0,   R(A || B) = F_|B|(R(A)) ^ R(B).
// The slot is cut into rows of kCrcRow (2 KB) bytes from its start, the last
// row possibly short.  Lane l takes the 64-byte block l of every row, folds it
// from a zero register a word at a time with four byte tables (slicing by 4),
// and keeps s = F_2048(s) ^ R(block).  Finally it advances s by the bytes that
// follow its last block (a multiple of 64, below 4 KB); the xor of the lanes is
// R(M).  Rows can be folded as soon as they are written, which lets an encoder
// checksum its slot while it is still producing it.  The standalone passes
// give each half warp a slot of its own, with 1 KB rows (crc_rows_half).
//
// The byte tables sit in shared memory in 32 copies, entry e of copy l in bank
// l, so the 32 lookups of a warp never conflict: 4 x 256 x 32 words (128 KB),
// one 1024-thread CTA per SM.  Tables 2i and 2i + 1 share a 64 KB region on a
// 64 KB boundary: entry e of copy l of table k at (k >> 1) 64 KB + 256 e +
// 128 (k & 1) + 4 l, so a lookup address is one byte permute of the register
// (the index byte into bits 8..15) with the lane's constant (the other bytes).
// The advance maps are 16-entry nibble tables (a table fills 16 distinct
// banks, so any indices are conflict-free).
#pragma once
#include <type_traits>

#include "device_common.cuh"

namespace kvc {
namespace crc {


constexpr int kCrcThreads = 1024;       // one CTA per SM (the tables take 128 KB)
constexpr int kCrcWarps = kCrcThreads / 32;
static_assert(kCrcThreads % 32 == 0 && kCrcThreads >= 32, "the table fill and the slot loop work in whole warps");
constexpr uint32_t kByteTabBytes = 4u * 256u * 32u * 4u;   // 128 KB
constexpr uint32_t kTabAlign = 65536u;  // the byte tables start on a 64 KB boundary
struct NibbleTables {
  uint32_t row[8][16];
  uint32_t fin[5][8][16];
};
// dynamic shared memory: the nibble tables, then the byte tables at the next
// 64 KB boundary of the shared window
constexpr uint32_t kCrcSmem = (uint32_t)sizeof(NibbleTables) + kTabAlign + kByteTabBytes;

// Entry at byte offset `off` of nibble table q.
__device__ __forceinline__ uint32_t entry(const uint32_t (*t)[16], int q, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(t[q]) + off);
}

// A 32-bit GF(2)-linear map given as 8 nibble tables.  The even and the odd
// nibbles of r, each times 4 (a table offset), are spread over the bytes of
// two words with one shift and mask each; a byte permute then picks each.
__device__ __forceinline__ uint32_t apply8(const uint32_t (*t)[16], uint32_t r) {
  const uint32_t ev = (r << 2) & 0x3C3C3C3Cu;   // byte k: 4 * nibble 2k
  const uint32_t od = (r >> 2) & 0x3C3C3C3Cu;   // byte k: 4 * nibble 2k + 1
  const uint32_t a = entry(t, 0, __byte_perm(ev, 0, 0x4440)) ^ entry(t, 1, __byte_perm(od, 0, 0x4440)) ^
                     entry(t, 2, __byte_perm(ev, 0, 0x4441));
  const uint32_t b = entry(t, 3, __byte_perm(od, 0, 0x4441)) ^ entry(t, 4, __byte_perm(ev, 0, 0x4442)) ^
                     entry(t, 5, __byte_perm(od, 0, 0x4442));
  return a ^ b ^ entry(t, 6, __byte_perm(ev, 0, 0x4443)) ^ entry(t, 7, __byte_perm(od, 0, 0x4443));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// R of one 64-byte block (16 little-endian words) from a zero register.
// tb = the shared address of this lane's copy of byte table 0 (bits 8..15
// zero); table k adds (k >> 1) 64 KB + 128 (k & 1), and byte j of the
// register goes to bits 8..15: s = T3[b0] ^ T2[b1] ^ T1[b2] ^ T0[b3].
__device__ __forceinline__ uint32_t fold_block(uint32_t tb, const uint4 (&c)[4]) {
  const uint32_t t3 = tb + kTabAlign + 128u, t2 = tb + kTabAlign, t1 = tb + 128u, t0 = tb;
  uint32_t s = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s ^= w[k];
      s = lds32(__byte_perm(s, t3, 0x7604)) ^ lds32(__byte_perm(s, t2, 0x7614)) ^
          lds32(__byte_perm(s, t1, 0x7624)) ^ lds32(__byte_perm(s, t0, 0x7634));
    }
  }
  return s;
}

// R of two 64-byte blocks at once (two independent chains, interleaved word by
// word: the table reads are volatile asm, which the compiler keeps in order).
__device__ __forceinline__ void fold_block2(uint32_t tb, const uint4 (&c)[4], const uint4 (&d)[4], uint32_t& rc,
                                            uint32_t& rd) {
  const uint32_t t3 = tb + kTabAlign + 128u, t2 = tb + kTabAlign, t1 = tb + 128u, t0 = tb;
  uint32_t s = 0, u = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
    const uint32_t v[4] = {d[q].x, d[q].y, d[q].z, d[q].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s ^= w[k];
      u ^= v[k];
      const uint32_t a0 = lds32(__byte_perm(s, t3, 0x7604)), b0 = lds32(__byte_perm(u, t3, 0x7604));
      const uint32_t a1 = lds32(__byte_perm(s, t2, 0x7614)), b1 = lds32(__byte_perm(u, t2, 0x7614));
      const uint32_t a2 = lds32(__byte_perm(s, t1, 0x7624)), b2 = lds32(__byte_perm(u, t1, 0x7624));
      const uint32_t a3 = lds32(__byte_perm(s, t0, 0x7634)), b3 = lds32(__byte_perm(u, t0, 0x7634));
      s = a0 ^ a1 ^ a2 ^ a3;
      u = b0 ^ b1 ^ b2 ^ b3;
    }
  }
  rc = s;
  rd = u;
}

// 64 bytes at `src` (32-byte aligned when A32, else 16): read-only loads for a
// slot this kernel does not write (NC), plain loads for one it has just
// written (the writer's lanes synchronised with __syncwarp first).  H: the
// read-only loads carry the L2 policy `pol`.
template <bool NC, bool H = false>
__device__ __forceinline__ void load_block(const uint8_t* src, bool a32, uint4 (&c)[4], uint64_t pol = 0) {
  if (a32) {
    if (NC) {
      ld_nc32_h<H>(src, c[0], c[1], pol);
      ld_nc32_h<H>(src + 32, c[2], c[3], pol);
    } else {
      ld_plain32(src, c[0], c[1]);
      ld_plain32(src + 32, c[2], c[3]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = NC ? ld_nc16_h<H>(src + 16 * q, pol) : ld_plain16(src + 16 * q);
  }
}

// One row into this lane's register: s = F_row(s) ^ R(block `lane` of row m).
template <bool NC, bool H = false>
__device__ __forceinline__ uint32_t fold_row(const NibbleTables& T, uint32_t tb, const uint8_t* slot, uint32_t m,
                                             bool al32, uint32_t s, uint32_t lane, uint64_t pol = 0) {
  uint4 c[4];
  load_block<NC, H>(slot + (uint64_t)m * kCrcRow + kCrcBlock * lane, al32, c, pol);
  return apply8(T.row, s) ^ fold_block(tb, c);
}

// CRC-32 of the n-byte slot at `slot` (n a multiple of 64) by the calling warp,
// rows 0 .. m0 - 1 already folded into the lanes' registers s (m0 = 0, s = 0
// for a whole slot); every lane returns the value.  The slot is n / 2048 full
// rows and a tail row of t = (n mod 2048) / 64 blocks; lane l's last block is
// then followed by 64 after_l bytes, after_l = t - 1 - l for l < t, else
// 31 - l + t (at most 62), by which its register is advanced before the xor.
// PAIRS: fold two rows a step (two independent chains), which measured faster
// for a warp finishing a slot it has just written and slower for the
// standalone passes, whose 32 warps per SM already hide the chains' latency.
template <bool NC = true, bool H = false, bool PAIRS = false>
__device__ __forceinline__ uint32_t crc_rows(const NibbleTables& T, uint32_t tb, const uint8_t* slot, uint32_t n,
                                             uint32_t m0, uint32_t s, uint32_t crc_k, uint32_t lane,
                                             uint64_t pol = 0) {
  const uint32_t rows = n / kCrcRow, tail = (n % kCrcRow) / kCrcBlock;
  const bool al32 = ((uintptr_t)slot & 31u) == 0;  // blocks start on 64-byte offsets of the slot
  uint32_t m = m0;
  // two rows a step: s = F_row(F_row(s) ^ R(block of row m)) ^ R(block of row m + 1)
  for (; PAIRS && m + 2u <= rows; m += 2u) {
    const uint8_t* src = slot + (uint64_t)m * kCrcRow + kCrcBlock * lane;
    uint4 c[4], d[4];
    load_block<NC, H>(src, al32, c, pol);
    load_block<NC, H>(src + kCrcRow, al32, d, pol);
    uint32_t rc, rd;
    fold_block2(tb, c, d, rc, rd);
    s = apply8(T.row, apply8(T.row, s) ^ rc) ^ rd;
  }
  for (; m < rows; ++m) s = fold_row<NC, H>(T, tb, slot, m, al32, s, lane, pol);
  uint32_t after = 31u - lane + tail;
  if (lane < tail) {
    s = fold_row<NC, H>(T, tb, slot, rows, al32, s, lane, pol);
    after = tail - 1u - lane;
  }
#pragma unroll
  for (int b = 0; b < 5; ++b) {
    const uint32_t t = apply8(T.fin[b], s);
    s = ((after >> b) & 1u) ? t : s;
  }
  const uint32_t t32 = apply8(T.row, s);  // 64 * 32 bytes: one row
  s = ((after >> 5) & 1u) ? t32 : s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s ^= __shfl_xor_sync(0xffffffffu, s, o);
  return s ^ crc_k;
}

// The same by one half warp, the other half coding another slot at the same
// time: rows of 1 KB (16 blocks of 64 bytes), so a slot is rounded up to a
// whole number of 1 KB rows rather than 2 KB (FP8 dynamic slots of 16,896
// bytes: 17 half rows for 16.5, against 9 rows for 8.25).  Lane h = lane & 15
// folds block h of every row; its register is advanced by 1 KB per row
// (fin[4], 64 * 16 bytes) and at the end by the at most 30 blocks after its
// last block.  Every lane of the warp calls it (the final xor is a half-warp
// shuffle); n = 0 gives crc_k.  Every lane of a half returns its slot's CRC.
template <bool NC = true>
__device__ __forceinline__ uint32_t crc_rows_half(const NibbleTables& T, uint32_t tb, const uint8_t* slot,
                                                  uint32_t n, uint32_t crc_k, uint32_t lane) {
  constexpr uint32_t kHalfRow = kCrcRow / 2;
  const uint32_t h = lane & 15u;
  const uint32_t rows = n / kHalfRow, tail = (n % kHalfRow) / kCrcBlock;
  const bool al32 = ((uintptr_t)slot & 31u) == 0;
  uint32_t s = 0;
  for (uint32_t m = 0; m < rows; ++m) {
    uint4 c[4];
    load_block<NC>(slot + (uint64_t)m * kHalfRow + kCrcBlock * h, al32, c);
    s = apply8(T.fin[4], s) ^ fold_block(tb, c);
  }
  uint32_t after = 15u - h + tail;
  if (h < tail) {
    uint4 c[4];
    load_block<NC>(slot + (uint64_t)rows * kHalfRow + kCrcBlock * h, al32, c);
    s = apply8(T.fin[4], s) ^ fold_block(tb, c);
    after = tail - 1u - h;
  }
#pragma unroll
  for (int b = 0; b < 5; ++b) {
    const uint32_t t = apply8(T.fin[b], s);
    s = ((after >> b) & 1u) ? t : s;
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s ^= __shfl_xor_sync(0xffffffffu, s, o);
  return s ^ crc_k;
}

// Fill the shared tables; returns the shared address of this lane's copy of
// byte table 0.
__device__ __forceinline__ uint32_t load_tables(const CrcParams& p, NibbleTables*& nt) {
  extern __shared__ __align__(16) uint8_t crc_smem[];
  nt = reinterpret_cast<NibbleTables*>(crc_smem);
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(crc_smem);
  const uint32_t tab = (base + (uint32_t)sizeof(NibbleTables) + kTabAlign - 1u) & ~(kTabAlign - 1u);
  uint32_t* byte_tab = reinterpret_cast<uint32_t*>(crc_smem + (tab - base));
  const uint32_t* src = &p.tab.row[0][0];
  uint32_t* dst = &nt->row[0][0];
  for (uint32_t k = threadIdx.x; k < sizeof(NibbleTables) / 4; k += blockDim.x) dst[k] = src[k];
  // one table word per warp and step (a broadcast read of the parameters),
  // stored to its 32 copies: copy l of entry e of table k at word
  // (k >> 1) 16384 + 64 e + 32 (k & 1) + l
  const uint32_t lane = threadIdx.x & 31u;
  for (uint32_t t = threadIdx.x >> 5; t < 4u * 256u; t += blockDim.x >> 5) {
    const uint32_t k = t >> 8, e = t & 255u;
    byte_tab[(k >> 1) * 16384u + 64u * e + 32u * (k & 1u) + lane] = p.tab.byte[k][e];
  }
  __syncthreads();
  return tab + (threadIdx.x & 31u) * 4u;
}

// Descriptor checks that need no layer pointers.
__device__ __forceinline__ bool slot_ok(const CrcParams& p, const kv_segment_desc* dp, uint32_t& role,
                                        uint64_t& off) {
  const uint32_t layer = ldg_u32(&dp->layer), block = ldg_u32(&dp->block);
  role = ldg_u32(&dp->role);
  off = ldg_u64(&dp->enc_offset);
  if (layer >= p.L || role > 1u || (uint64_t)block >= p.num_blocks || (off & 15u)) return false;
  if (p.codec[role] == KV_CODEC_NONE) return true;
  return off <= p.buf_bytes && p.seg_bytes[role] <= p.buf_bytes - off;
}

__device__ __forceinline__ void store_header(kv_segment_header* h, uint32_t version, uint32_t format,
                                             uint64_t stored, uint32_t crc, uint32_t status, uint64_t orig) {
  uint64_t* w = reinterpret_cast<uint64_t*>(h);
  st_u64(w, (uint64_t)version | ((uint64_t)format << 32));
  st_u64(w + 1, orig);
  st_u64(w + 2, stored);
  st_u64(w + 3, (uint64_t)crc | ((uint64_t)status << 32));
}


// Seal segment i whose encode status is st: the header kv_codec_seal writes.
// NC: the slot was written by an earlier launch (read-only loads); otherwise
// by this warp in this launch.  Every lane of the warp calls it.
// m0 / s0: rows of the slot the caller has already folded (crc_rows).
template <bool NC>
__device__ __forceinline__ void seal_segment(const CrcParams& p, const NibbleTables& T, uint32_t tb,
                                             uint32_t i, uint32_t st, uint32_t lane, uint32_t m0 = 0,
                                             uint32_t s0 = 0) {
  uint32_t role;
  uint64_t off;
  if (!slot_ok(p, p.descs + i, role, off)) {
    if (lane == 0) store_header(p.headers + i, p.version, 0, 0, 0, KV_SEG_BAD_DESC, p.orig_bytes);
    return;
  }
  uint64_t stored = 0;
  uint32_t crc = 0;
  if (st == KV_SEG_ENCODED && p.codec[role] != KV_CODEC_NONE) {
    stored = p.seg_bytes[role];
    crc = crc_rows<NC, false, !NC>(T, tb, p.buf + off, (uint32_t)stored, m0, s0, p.crc_k[role], lane);
  }
  if (lane == 0) store_header(p.headers + i, p.version, p.format[role], stored, crc, st, p.orig_bytes);
}

// The result kv_codec_verify gives segment i: its header's status when the
// header matches the codec and the slot's CRC-32, else KV_SEG_CORRUPT
// (KV_SEG_BAD_DESC for an invalid descriptor).  Every lane returns it.  H: the
// slot's loads carry the L2 policy `pol` (a decoder that reads the slot again
// right after keeps it in L2 with evict_last).
template <bool H = false>
__device__ __forceinline__ uint32_t verify_segment(const CrcParams& p, const NibbleTables& T, uint32_t tb,
                                                   uint32_t i, uint32_t lane, uint64_t pol = 0) {
  uint32_t role;
  uint64_t off;
  if (!slot_ok(p, p.descs + i, role, off) || p.codec[role] == KV_CODEC_NONE) return KV_SEG_BAD_DESC;
  const uint64_t* w = reinterpret_cast<const uint64_t*>(p.headers + i);
  const uint64_t w0 = ldg_u64(w), orig = ldg_u64(w + 1), stored = ldg_u64(w + 2), w3 = ldg_u64(w + 3);
  const uint32_t st = (uint32_t)(w3 >> 32);
  bool ok = (uint32_t)w0 == p.version && (uint32_t)(w0 >> 32) == p.format[role] && orig == p.orig_bytes &&
            st >= KV_SEG_ENCODED && st <= KV_SEG_BAD_DESC;
  if (ok && st == KV_SEG_ENCODED) {
    ok = stored == p.seg_bytes[role];
    if (ok) ok = crc_rows<true, H>(T, tb, p.buf + off, (uint32_t)stored, 0, 0, p.crc_k[role], lane, pol) == (uint32_t)w3;
  } else if (ok) {
    ok = stored == 0;
  }
  return ok ? st : (uint32_t)KV_SEG_CORRUPT;
}

}  // namespace crc

// The codec kernels' second parameter selects their variant.  NoSeal: the
// plain kernel, a CTA of NT threads per segment.  CrcParams: one warp per
// segment in kCrcThreads-thread CTAs (one per SM) that hold the CRC tables;
// the encoder seals each slot as it writes it, the decoder verifies each slot
// before it restores it.  WarpSeg (kernels that offer it): one warp per
// segment in CTAs of NT threads, without the CRC -- no CTA barrier per
// segment, for segments too short to keep a CTA's warps busy.
struct NoSeal {};
struct WarpSeg {};
template <typename Q, int NT = kThreads>
struct Variant {
  static constexpr bool kSeal = std::is_same<Q, CrcParams>::value;
  static constexpr bool kWarp = !std::is_same<Q, NoSeal>::value;  // one warp per segment
  static constexpr int kCtaThreads = kSeal ? crc::kCrcThreads : NT;
};

// Status of an encoded segment from its admission flags (bit 0: a nonfinite
// value, bit 1: a value beyond the admission bound).
__device__ __forceinline__ uint8_t status_of_flags(uint32_t f) {
  return (f & 1u) ? KV_SEG_RAW_NONFINITE : (f & 2u) ? KV_SEG_RAW_RANGE : KV_SEG_ENCODED;
}

// Plain launch of a codec kernel's NoSeal variant: `threads` per CTA, at most
// max_per_sm CTAs per SM.  (The launch helpers are static: in the debug build
// each translation unit arms its own bounds-check state.)
static int launch_plain(void (*kernel)(Params, NoSeal), const Params& p, void* stream, int max_per_sm,
                        int threads = kThreads) {
  const void* k = reinterpret_cast<const void*>(kernel);
  unsigned grid = 0;
  const int rc = grid_for_threads(k, p.n_segments, max_per_sm, threads, &grid);
  if (rc != KV_OK || grid == 0) return rc;
  NoSeal none;
  void* args[] = {const_cast<Params*>(&p), &none};
  return dbg_launch(stream, [&] { return cudaLaunchKernel(k, dim3(grid), dim3(threads), args, 0, (cudaStream_t)stream); },
                    p);
}

// Launch of a codec kernel's WarpSeg variant: kThreads per CTA, at most
// max_per_sm CTAs per SM, a warp for every segment up to that.
static int launch_warp(void (*kernel)(Params, WarpSeg), const Params& p, void* stream, int max_per_sm) {
  const void* k = reinterpret_cast<const void*>(kernel);
  constexpr uint32_t kWarps = kThreads / 32;
  unsigned grid = 0;
  const int rc = grid_for_threads(k, (p.n_segments + kWarps - 1u) / kWarps, max_per_sm, kThreads, &grid, false);
  if (rc != KV_OK || grid == 0) return rc;
  WarpSeg none;
  void* args[] = {const_cast<Params*>(&p), &none};
  return dbg_launch(stream, [&] { return cudaLaunchKernel(k, dim3(grid), dim3(kThreads), args, 0, (cudaStream_t)stream); },
                    p);
}

// Launch of a codec kernel's CrcParams variant: one CTA of kCrcThreads per SM
// at most, kCrcSmem bytes of dynamic shared memory for the tables.
static int launch_sealed(void (*kernel)(Params, CrcParams), const Params& p, const CrcParams& q, void* stream) {
  const void* k = reinterpret_cast<const void*>(kernel);
  // the tables need more than the default 48 KB of dynamic shared memory (set
  // on every launch: the attribute belongs to the current device's context)
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)crc::kCrcSmem) != cudaSuccess)
    return KV_ERR_CUDA;
  unsigned grid = 0;
  const int rc = grid_for_threads(k, (p.n_segments + crc::kCrcWarps - 1) / crc::kCrcWarps, 1,
                                  crc::kCrcThreads, &grid, false);
  if (rc != KV_OK || grid == 0) return rc;
  void* args[] = {const_cast<Params*>(&p), const_cast<CrcParams*>(&q)};
  return dbg_launch(stream, [&] {
    return cudaLaunchKernel(k, dim3(grid), dim3(crc::kCrcThreads), args, crc::kCrcSmem, (cudaStream_t)stream);
  }, p, q);
}

}  // namespace kvc
