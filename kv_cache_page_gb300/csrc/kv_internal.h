// kv_internal.h -- launch parameters shared by the host library and the kernels.
//
// Everything a kernel needs travels in one __grid_constant__ parameter block
// (about 15 KB: per-layer pointers, fixed FP8 scales, the TurboQuant codebook
// and sign bits), so the codec holds no device memory and a launch needs no
// host-to-device copy.
#pragma once
#include <stdint.h>

#include "kv_codec.h"

namespace kvc {

constexpr int kMaxLayers = (int)KV_CODEC_MAX_LAYERS;
constexpr int kThreads = 256;           // threads per CTA for every codec kernel

// TurboQuant index table: cell c = rint(4 w) of the unscaled Walsh-Hadamard
// output w (|w| <= sqrt(D) <= 16 for a unit vector), c in [-kLutHalf, kLutHalf].
constexpr int kLutHalf = 68;
constexpr int kLutCells = 2 * kLutHalf + 1;

struct Params {
  // ---- registered geometry ----
  uint32_t dtype;                       // KV_DT_*
  uint32_t layout;                      // KV_LAYOUT_*
  uint32_t D;                           // head_dim
  uint32_t H;                           // num_kv_heads
  uint32_t T;                           // block_tokens
  uint32_t L;                           // num_layers
  uint32_t nv;                          // vectors per segment = H * T
  uint32_t n_layer_ptrs;
  uint64_t num_blocks;
  uint64_t h_magic;                     // ceil(2^32 / H): t = (j * h_magic) >> 32
  int64_t sb, st, sh;                   // strides (elements)
  uint32_t codec[2];                    // KV_CODEC_* per role
  uint32_t protect_first, protect_last;
  uint32_t code_bytes[2];               // per vector
  uint32_t meta_bytes[2];               // per vector
  uint64_t seg_bytes[2];                // encoded slot (multiple of 128)
  uint32_t rec_bytes;                   // INT8_HEAD token record: H * (D + 2) rounded up to 128
  uint32_t rec_used;                    // H * (D + 2): codes and scales; zeros follow
  uint8_t static_status[2];             // 0 = encodable, else KV_SEG_RAW_{POLICY,OVERSIZE,NO_SAVING}
  uint8_t heads_contig;                 // st == H * sh: vector j of a page sits at j * sh
  uint8_t vec32;                        // per call: every vector starts on a 32-byte boundary
  float reject_abs;                     // admission bound
  float wht_scale;                      // fl32(1/sqrt(D))
  float neg_zero;                       // -0.0f (an FMA addend the compiler cannot fold)
  uint64_t sign_seed;                   // TurboQuant sign stream (SplitMix64 seed)
  uint32_t sign_per_layer;              // 1: format version 2, a sign vector per layer
  uint32_t fixed_reject;                // FP8_FIXED: a quotient beyond +-448 keeps the segment raw
  float cent[16];                       // TurboQuant centroids (K codec)
  float bnd[16];                        // TurboQuant boundaries (K codec), bnd[15] unused
  // Index table of the unscaled WHT output w: code(w) = lut_lo[c] + (w > lut_thr[c]),
  // c = rint(4 w); built from the boundaries moved to the unscaled domain,
  // W_j = max{w : RN(w * wht_scale) <= bnd[j]}, so that no scale multiply is needed.
  float lut_thr[kLutCells];
  uint32_t lut_lo[kLutCells];
  // The same for lanes holding negated outputs v = -w: lut_mlo[c] + (v > lut_mthr[c])
  // = (2^bits - 1) - code(w), c = rint(4 v).
  float lut_mthr[kLutCells];
  uint32_t lut_mlo[kLutCells];
  float fixed_scale[kMaxLayers][2];     // FP8_FIXED scale per (layer, role)
  const void* layer_ptr[2 * kMaxLayers];
  // ---- per call ----
  const kv_segment_desc* descs;
  uint32_t n_segments;
  uint32_t role_sel;                    // 0 / 1: that role only; 2: both roles; 3: none
  uint32_t is_first;                    // this launch reports segments no launch encodes
  uint32_t status_is_result;            // decode: status and result are the same array
  uint8_t* buf;                         // encode: slots written; decode: slots read
  uint64_t buf_bytes;
  uint8_t* status;                      // encode: written; decode: read
  uint8_t* result;                      // decode: optional per-segment result
};

enum Dir { kEncode = 0, kDecode = 1 };

// Segment checksums (seal / verify).  CRC-32 over a slot is computed by one
// warp: lane l folds the 64-byte blocks l, l + 32, ... of the slot (rows of
// 2 KB from the slot's start, the last one possibly short) into a zero-preset
// CRC register with byte tables, advancing the register by 2 KB of zero bytes
// per row; the lanes' registers are then advanced by the bytes that follow
// their last block and xor-combined.  The advances are GF(2)-linear maps of 32
// bits, applied as 16-entry nibble tables.
constexpr uint32_t kCrcBlock = 64;               // bytes a lane folds per row
constexpr uint32_t kCrcRow = 32 * kCrcBlock;     // one row: a 64-byte block per lane
struct CrcTables {
  uint32_t byte[4][256];    // slicing by 4: register of byte v followed by k zero bytes
  uint32_t row[8][16];      // register advanced by kCrcRow zero bytes, per nibble
  uint32_t fin[5][8][16];   // register advanced by kCrcBlock * 2^b zero bytes, b = 0..4
};

struct CrcParams {
  CrcTables tab;
  const kv_segment_desc* descs;
  uint32_t n_segments;
  uint32_t L;
  uint64_t num_blocks;
  uint32_t codec[2];
  uint32_t version;                     // header version (the geometry's format version)
  uint32_t format[2];                   // header format word per role
  uint64_t seg_bytes[2];
  uint32_t crc_k[2];                    // CRC of a zero slot of seg_bytes[role] (preset and complement)
  uint64_t orig_bytes;
  const uint8_t* buf;
  uint64_t buf_bytes;
  const uint8_t* status;                // seal: input statuses
  kv_segment_header* headers;           // seal: written; verify: read
  uint8_t* result;                      // verify: written
};

int launch_crc(const CrcParams& p, int seal, void* stream);

// Kernel launchers (one per codec family), defined in the .cu files.  `codec`
// is the KV_CODEC_* kind the launch runs; grid size is chosen from the device.
int launch_fp8(const Params& p, int dir, uint32_t codec, void* stream);
// FP8 encode that also writes the segment headers (q.headers), or decode that
// first verifies them (result in p.result); one pass over the slots.
int launch_fp8_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream);
int launch_uniform(const Params& p, int dir, uint32_t codec, void* stream);
// The same for KV_CODEC_UNIFORM8 (KV_ERR_INVALID_ARG for another codec).
int launch_uniform_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream);
int launch_turboquant(const Params& p, int dir, uint32_t codec, void* stream);
int launch_int8(const Params& p, int dir, uint32_t codec, void* stream);
// The same for KV_CODEC_INT8_HEAD.
int launch_int8_sealed(const Params& p, const CrcParams& q, int dir, uint32_t codec, void* stream);

// Grid size for a codec kernel over n segments: one CTA per segment up to
// SM count x resident CTAs per SM, the latter the occupancy limit (cached per
// device and kernel) capped at `max_per_sm`.  Defined in the host library.
int grid_for(const void* kernel, uint32_t n_segments, int max_per_sm, unsigned* grid);
// The same for a kernel launched with `threads` threads per CTA; odd: make the
// grid odd (CTA-per-segment kernels), else the units are warps' segment groups.
int grid_for_threads(const void* kernel, uint32_t n_segments, int max_per_sm, int threads, unsigned* grid,
                     bool odd = true);

}  // namespace kvc
