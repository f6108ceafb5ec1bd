/*
 * kv_codec.h -- C ABI of the GB300 KV-cache page codec.
 *
 * The codec encodes KV-cache pages on the GPU before they are offloaded and
 * restores them into the engine's native FP16/BF16 layout, as described by
 * "KV precision and storage encoding" (OrbitKV docs), section "FP8 and
 * TurboQuant", and "Asymmetric KV: methods and results" (knlp), section
 * "Precision and scaling reference".
 *
 * Unit of work: a SEGMENT = all vectors of one role (K or V) of one page
 * (block) of one layer, i.e. num_kv_heads * block_tokens vectors of head_dim
 * elements.  The storage-format page attaches metadata and raw fallback per
 * segment (section "Ownership, storage and GDS").
 *
 * Encoded segment slot (little endian):
 *     [codes of vector 0 .. n-1][metadata of vector 0 .. n-1][zero padding]
 * with vectors ordered v = token * num_kv_heads + head, padded to a multiple of
 * 128 bytes (kv_codec_segment_bytes gives the size).  Codes per vector:
 *     FP8 (all modes)     head_dim bytes, E4M3FN
 *     TQ2 / TQ3 / TQ4     head_dim*bits/8 bytes, little-endian bit stream
 *                         (code i in bits [bits*i, bits*i + bits))
 *     UNIFORM2/3/4        head_dim*bits/8 bytes, same bit stream
 *     UNIFORM8            head_dim bytes
 * Metadata per vector:
 *     FP8_DYNAMIC         FP32 scale (4 bytes)
 *     FP8_CAST/FIXED      none
 *     TQ2 / TQ3 / TQ4     FP16 norm of the source vector (2 bytes)
 *     UNIFORM2/3/4/8      FP16 minimum, FP16 step (4 bytes)
 * E.g. head_dim 128: TQ4 K 66, UNIFORM4 V 68, TQ3 K 50, UNIFORM3 V 52 bytes per
 * vector (the storage-format page's payload sizes).
 *
 * INT8_HEAD slots follow instead the token-row record of "Building a quantized
 * HiCache for SGLang" (section "Why exactly 1,152 bytes?"): one record per
 * token of the page, in token order,
 *     [int8 codes of head 0 .. H-1 (H*D bytes)][BF16 scale of head 0 .. H-1]
 *     [zero padding to a multiple of 128 bytes]
 * (8 heads x 128: 1,024 + 16 = 1,040 -> 1,152 bytes), so a slot is
 * block_tokens records.  Per head vector (section "Building the INT8 codec"):
 * amax = max|x| floored at 1e-12, scale = BF16(FP32(amax / 127)), code =
 * round-half-even(FP32(x / scale)) clamped to [-127, 127]; restore =
 * BF16(code * scale).  Defined for BF16 sources only.
 *
 * Threading and streams: a handle is immutable after creation and may be used
 * from several host threads.  Encode/decode only enqueue work on the caller's
 * CUDA stream (no synchronisation, no allocation); all buffers belong to the
 * caller and must stay valid until that work completes.
 *
 * Host-resident slots (offload and restore without staging copies): the
 * descriptor, slot, status and result buffers of encode/decode may each be
 * device memory or PINNED host memory (cudaHostAlloc / cudaMallocHost /
 * cudaHostRegister).  For pinned host memory the kernels load and store the
 * bytes through its device mapping, i.e. over the CPU-GPU link (NVLink-C2C on
 * GB300), so an encode writes its slots straight into host memory and a decode
 * reads them from there and scatters the result into the engine pages.  This
 * is the restore path of "Building a quantized HiCache for SGLang" (section
 * "CPU to GPU: restoration": compressed copy, dequantization and scatter all
 * enqueued on the transfer stream before the layer is marked ready) and the
 * "upload encoded bytes and GPU decode" restore of the OrbitKV docs, with the
 * copy folded into the kernel.  Stream order gives the ordering: the caller records an event on
 * the stream it passes and makes the consuming stream wait on it.  Pageable
 * host memory is refused (KV_ERR_NOT_ACCESSIBLE).  The engine pages
 * (layer_ptrs) are device memory.
 *
 * All functions return KV_OK (0) or a negative KV_ERR_* code and never abort.
 */
#ifndef KV_CODEC_H
#define KV_CODEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV_CODEC_ABI_VERSION 1u
#define KV_CODEC_MAX_LAYERS 512u
/* Largest n_segments of one call (larger counts return KV_ERR_INVALID_ARG). */
#define KV_CODEC_MAX_SEGMENTS 0x7FFFFFFFu

/* ---- return codes ------------------------------------------------------ */
#define KV_OK 0
#define KV_ERR_INVALID_ARG -1          /* NULL pointer, zero size, bad enum value */
#define KV_ERR_UNSUPPORTED_HEAD_DIM -2 /* head_dim not in {32, 64, 128, 256} */
#define KV_ERR_LAYOUT_MISMATCH -3      /* strides overlap or do not fit the layout */
#define KV_ERR_UNSUPPORTED_CODEC_FOR_ROLE -4 /* a TurboQuant kind (TQ2/TQ3/TQ4) requested for V */
#define KV_ERR_MISALIGNED -5           /* pointer or stride not 16-byte aligned */
#define KV_ERR_CUDA -6                 /* a CUDA runtime call failed (launch, device query) */
#define KV_ERR_ABI -7                  /* abi_version / struct_size mismatch */
#define KV_ERR_TOO_MANY_LAYERS -8      /* num_layers = 0 or > KV_CODEC_MAX_LAYERS */
#define KV_ERR_NOT_ACCESSIBLE -9       /* a buffer is pageable host memory (not pinned) */
#define KV_ERR_UNSUPPORTED_DTYPE -10   /* codec not defined for the source dtype (INT8_HEAD: BF16) */
#define KV_ERR_INTERNAL -11            /* bounds-checked debug library only: a kernel access fell outside
                                          the call's buffers (skipped, not performed) */

/* ---- enums ------------------------------------------------------------- */
#define KV_DT_FP16 1u
#define KV_DT_BF16 2u

#define KV_LAYOUT_SEPARATE 1u    /* K and V tensors, each [block, token, head, D] by strides */
#define KV_LAYOUT_VLLM_PACKED 2u /* one tensor per layer, rows of 2*D: K = [0, D), V = [D, 2D) */

#define KV_CODEC_NONE 0u        /* role is not encoded: its segments get KV_SEG_RAW_POLICY */
#define KV_CODEC_FP8_CAST 1u    /* E4M3FN of x (scale 1) */
#define KV_CODEC_FP8_FIXED 2u   /* E4M3FN of x / s, s per (layer, role) from calibration */
#define KV_CODEC_FP8_DYNAMIC 3u /* E4M3FN of x / s, s per token/head vector, stored FP32 */
#define KV_CODEC_TQ3 4u         /* TurboQuant K, 3-bit codes (K role only) */
#define KV_CODEC_TQ4 5u         /* TurboQuant K, 4-bit codes (K role only) */
#define KV_CODEC_UNIFORM3 6u    /* per-vector uniform, FP16 min and step */
#define KV_CODEC_UNIFORM4 7u
#define KV_CODEC_UNIFORM8 8u
#define KV_CODEC_INT8_HEAD 9u   /* symmetric per-head INT8, BF16 scale, token-row records (BF16 only) */
#define KV_CODEC_TQ2 10u        /* TurboQuant K, 2-bit codes (K role only) */
#define KV_CODEC_UNIFORM2 11u   /* per-vector uniform, 2-bit codes */

/* ---- per-segment status bytes (written by encode, read by decode) ------- */
#define KV_SEG_ENCODED 1u       /* slot holds the encoding */
#define KV_SEG_RAW_NONFINITE 2u /* an element is inf or NaN: keep raw */
#define KV_SEG_RAW_RANGE 3u     /* an element has |x| > reject_abs (or, under KV_FIXED_OVERFLOW_REJECT,
                                   an FP8 fixed-scale quotient beyond +-448): keep raw, no clipping */
#define KV_SEG_RAW_PROTECTED 4u /* layer is in the protected first/last range */
#define KV_SEG_RAW_POLICY 5u    /* the role's codec is KV_CODEC_NONE */
#define KV_SEG_RAW_OVERSIZE 6u  /* source segment larger than 16 MiB */
#define KV_SEG_RAW_NO_SAVING 7u /* aligned encoding saves less than 12.5% */
#define KV_SEG_BAD_DESC 8u      /* descriptor invalid (see kv_segment_desc); nothing written */
#define KV_SEG_CORRUPT 9u       /* kv_codec_verify: header or CRC-32 mismatch; treat as a miss */
/* In every RAW_* / BAD_DESC case the segment's slot is not written (BAD_DESC)
 * or holds unspecified bytes (RAW_*); the caller keeps the raw page. */

/* ---- geometry ----------------------------------------------------------- */
/* Registered once per engine KV cache ("Python only registers engine tensor
 * geometry"; "quantization never infers head layout from byte count",
 * storage-format page, "FP8 and TurboQuant").  Strides are in ELEMENTS, the
 * element (head_dim) stride is 1, and for the 128-bit vector accesses every
 * stride must be a multiple of 8 elements (16 bytes). */
typedef struct kv_codec_geometry {
  uint32_t abi_version;   /* KV_CODEC_ABI_VERSION */
  uint32_t struct_size;   /* sizeof(kv_codec_geometry) */
  uint32_t dtype;         /* KV_DT_FP16 | KV_DT_BF16 */
  uint32_t layout;        /* KV_LAYOUT_SEPARATE | KV_LAYOUT_VLLM_PACKED */
  uint32_t head_dim;      /* 32, 64, 128 or 256 */
  uint32_t num_kv_heads;  /* H >= 1 */
  uint32_t block_tokens;  /* tokens per page >= 1 (16 in the pages' engines) */
  uint32_t num_layers;    /* 1 .. KV_CODEC_MAX_LAYERS */
  uint64_t num_blocks;    /* pages per layer tensor; descriptors with block >= this are rejected */
  int64_t stride_block;   /* elements between pages */
  int64_t stride_token;   /* elements between tokens of a page */
  int64_t stride_head;    /* elements between heads of a token */
  uint32_t k_codec;       /* KV_CODEC_* for the K role */
  uint32_t v_codec;       /* KV_CODEC_* for the V role (TQ kinds not allowed) */
  uint32_t protect_first; /* layers [0, protect_first) stay raw */
  uint32_t protect_last;  /* layers [num_layers - protect_last, num_layers) stay raw */
  uint64_t rotation_seed; /* seed of the TurboQuant sign vector */
  float reject_abs;       /* admission bound, 0 < reject_abs <= 448; 0 selects 448 */
  uint32_t sign_version;  /* TurboQuant sign vectors ("versioned sign generator", storage-format
                             page, "FP8 and TurboQuant"): 0 or 1 = one vector per (rotation_seed,
                             head_dim), segment format version 1; 2 = one per layer as well,
                             format version 2 (see kv_codec_layer_signs); other values are refused
                             with KV_ERR_INVALID_ARG */
  const float* fixed_amax; /* host, [num_layers][2] (K, V) calibration absolute maxima,
                              required iff a role uses FP8_FIXED; copied at create */
  uint32_t fixed_overflow; /* FP8_FIXED quotients x / s beyond +-448 (calibration below the
                              data's range): KV_FIXED_OVERFLOW_CLIP (0) clips them to +-448
                              ("Asymmetric KV: methods and results", "Precision and scaling
                              reference"); KV_FIXED_OVERFLOW_REJECT (1) keeps such a segment
                              raw, status KV_SEG_RAW_RANGE ("KV precision and storage
                              encoding", "FP8 and TurboQuant": out-of-range values stay raw
                              rather than being clipped); other values are refused */
  uint32_t reserved;       /* 0 */
} kv_codec_geometry;
/* struct_size: sizeof(kv_codec_geometry) (112 bytes), or 104 for the layout
 * without fixed_overflow and reserved (taken as 0). */
#define KV_CODEC_GEOMETRY_SIZE_V1 104u
#define KV_FIXED_OVERFLOW_CLIP 0u
#define KV_FIXED_OVERFLOW_REJECT 1u

/* One segment to encode or decode.  Device-resident array, 24 bytes each.
 * A descriptor is invalid (status KV_SEG_BAD_DESC, nothing read or written) when
 * layer >= num_layers, block >= num_blocks, role > 1, the layer pointer for it is
 * NULL, enc_offset is not a multiple of 16, or the slot does not fit in the
 * encoded buffer (enc_offset + kv_codec_segment_bytes(role) > buffer bytes). */
typedef struct kv_segment_desc {
  uint32_t layer;
  uint32_t block;
  uint32_t role;          /* 0 = K, 1 = V */
  uint32_t reserved;      /* ignored */
  uint64_t enc_offset;    /* byte offset of the segment's slot in the encoded buffer */
} kv_segment_desc;

/* Segment header ("KV precision and storage encoding", OrbitKV docs, section
 * "Ownership, storage and GDS": every encoded segment carries a version, its
 * original length, its format, its stored length and a CRC32).  32 bytes,
 * little endian, one per descriptor. */
#define KV_SEGMENT_FORMAT_VERSION 1u   /* geometry sign_version 0 or 1 */
#define KV_SEGMENT_FORMAT_VERSION_2 2u /* geometry sign_version 2: per-layer sign vectors */
typedef struct kv_segment_header {
  uint32_t version;       /* the geometry's format version: KV_SEGMENT_FORMAT_VERSION (1) or
                             KV_SEGMENT_FORMAT_VERSION_2; verify treats any other as a mismatch */
  uint32_t format;        /* codec kind | dtype << 8 | log2(head_dim) << 16 (0 for a bad descriptor) */
  uint64_t orig_bytes;    /* source segment bytes: num_kv_heads * block_tokens * head_dim * 2 */
  uint64_t stored_bytes;  /* encoded slot bytes; 0 when the segment stayed raw */
  uint32_t crc32;         /* CRC-32 of the stored bytes: reflected polynomial 0xEDB88320,
                             register preset to all ones, result complemented (zlib's) */
  uint32_t status;        /* the segment's status when sealed */
} kv_segment_header;

typedef struct kv_codec_s* kv_codec_t;

/* Validate a geometry and build the handle: sign vector (SplitMix64 of
 * rotation_seed), Lloyd-Max codebooks for TQ roles, FP8 fixed scales
 * s = max(amax, 1e-12) * fl32(1/448) per (layer, role).  Host only: touches no
 * GPU and allocates no device memory.  On error *out is set to NULL. */
int kv_codec_create(const kv_codec_geometry* geometry, kv_codec_t* out);

/* Release a handle (host memory only; no GPU work is pending on its behalf
 * beyond what the caller enqueued, which does not reference the handle). */
int kv_codec_destroy(kv_codec_t codec);

/* Bytes of one encoded segment slot for `role` (multiple of 128; 0 if the role
 * has no codec) and of one raw source segment (H * block_tokens * D * 2). */
int kv_codec_segment_bytes(kv_codec_t codec, uint32_t role, uint64_t* enc_bytes,
                           uint64_t* raw_bytes);

/* Encode n_segments segments.
 *   layer_ptrs   HOST array of DEVICE pointers, 16-byte aligned: separate layout
 *                [K_0, V_0, K_1, V_1, ...] (2 * num_layers entries), packed layout
 *                one per layer (num_layers entries).  NULL entries are allowed for
 *                roles that no descriptor references.  When every pointer is
 *                32-byte aligned and every stride a multiple of 16 elements, the
 *                kernels move page data 32 bytes at a time (faster; same result).
 *   n_layer_ptrs number of entries in layer_ptrs (must match the layout).
 *   d_descs      array of n_segments descriptors, 8-byte aligned (device or pinned host).
 *   d_out        encoded buffer of out_bytes bytes, 16-byte aligned (device or pinned host).
 *   d_status     array of n_segments status bytes, written for every segment
 *                (device or pinned host).
 *   stream       cudaStream_t (NULL = legacy default stream).
 * Segments are independent; descriptors may repeat a source page but must not
 * overlap slots.  n_segments = 0 is a no-op. */
int kv_codec_encode(kv_codec_t codec, const void* const* layer_ptrs, uint32_t n_layer_ptrs,
                    const kv_segment_desc* d_descs, uint32_t n_segments, void* d_out,
                    uint64_t out_bytes, uint8_t* d_status, void* stream);

/* Restore every segment whose status is KV_SEG_ENCODED into the engine layout;
 * all other segments are left untouched (the caller restores them from its raw
 * copy).  d_descs, d_in (in_bytes bytes, 16-byte aligned), d_status and
 * d_result may be device or pinned host memory, as for encode.  d_result
 * (optional array of n_segments bytes) receives
 * KV_SEG_ENCODED for restored segments, KV_SEG_BAD_DESC for invalid descriptors
 * (or a role without codec), and the input status otherwise. */
int kv_codec_decode(kv_codec_t codec, void* const* layer_ptrs, uint32_t n_layer_ptrs,
                    const kv_segment_desc* d_descs, uint32_t n_segments, const void* d_in,
                    uint64_t in_bytes, const uint8_t* d_status, uint8_t* d_result,
                    void* stream);

/* Seal n_segments encoded slots: write one kv_segment_header per descriptor,
 * with the CRC-32 of the slot for segments whose status is KV_SEG_ENCODED
 * (stored_bytes 0 and crc32 0 for the others; status KV_SEG_BAD_DESC and
 * format 0 for an invalid descriptor).  buf / buf_bytes: the encoded buffer
 * (16-byte aligned); status: the statuses kv_codec_encode wrote; headers: n
 * records, 8-byte aligned.  descs, buf, status and headers may be device or
 * pinned host memory.  Stream-ordered like encode. */
int kv_codec_seal(kv_codec_t codec, const kv_segment_desc* descs, uint32_t n_segments,
                  const void* buf, uint64_t buf_bytes, const uint8_t* status,
                  kv_segment_header* headers, void* stream);

/* Check n_segments slots against their headers before decode (section
 * "Ownership, storage and GDS": checksums are validated before GPU decode and a
 * damaged object becomes a miss).  result[i] = the header's status when the
 * header matches this geometry (version, format, original and stored length)
 * and, for KV_SEG_ENCODED, the slot's CRC-32 matches; KV_SEG_CORRUPT otherwise;
 * KV_SEG_BAD_DESC for an invalid descriptor or a role without codec.  Passing
 * result as the status of kv_codec_decode restores exactly the verified
 * segments.  Buffers as for kv_codec_seal; result: n bytes. */
int kv_codec_verify(kv_codec_t codec, const kv_segment_desc* descs, uint32_t n_segments,
                    const void* buf, uint64_t buf_bytes, const kv_segment_header* headers,
                    uint8_t* result, void* stream);

/* Encode and seal in one call (section "Ownership, storage and GDS": a CRC32
 * per stored segment).  Slots, statuses and headers equal those of
 * kv_codec_encode followed by kv_codec_seal on the same arguments.  When every
 * coded role takes an FP8 codec, KV_CODEC_UNIFORM8 or KV_CODEC_INT8_HEAD this
 * is one pass: each slot's CRC-32 is taken by the warp that encoded it, from
 * the bytes it has just written, so HBM carries the slots once; other codecs
 * run encode, then seal.  Arguments as
 * for kv_codec_encode, plus headers (n records, 8-byte aligned, device or
 * pinned host memory). */
int kv_codec_encode_sealed(kv_codec_t codec, const void* const* layer_ptrs, uint32_t n_layer_ptrs,
                           const kv_segment_desc* descs, uint32_t n_segments, void* out,
                           uint64_t out_bytes, uint8_t* status, kv_segment_header* headers,
                           void* stream);

/* Verify and decode in one call (same section: checksums validated before GPU
 * decode, a damaged object becomes a miss).  result[i] and the restored pages
 * equal those of kv_codec_verify into result followed by kv_codec_decode with
 * status = result and d_result = result: a segment whose header or CRC-32 does
 * not match is reported KV_SEG_CORRUPT and its page is not written.  When every
 * coded role takes an FP8 codec, KV_CODEC_UNIFORM8 or KV_CODEC_INT8_HEAD this is
 * one pass: the warp that checks a slot then restores it, re-reading the slot
 * from L2.  Arguments as for
 * kv_codec_decode, with the headers in place of the statuses and result (n
 * bytes) required. */
int kv_codec_decode_verified(kv_codec_t codec, void* const* layer_ptrs, uint32_t n_layer_ptrs,
                             const kv_segment_desc* descs, uint32_t n_segments, const void* in,
                             uint64_t in_bytes, const kv_segment_header* headers, uint8_t* result,
                             void* stream);

/* Static description of an error code. */
const char* kv_codec_strerror(int code);

/* The codebook the handle-independent TurboQuant path uses for (bits, head_dim):
 * 2^bits centroids ascending and 2^bits - 1 boundaries, FP32, host memory.
 * Gaussian Lloyd-Max levels scaled by 1/sqrt(head_dim). */
int kv_codec_codebook(uint32_t bits, uint32_t head_dim, float* centroids, float* boundaries);

/* The sign vector for (seed, head_dim): one byte per element, 1 = negate.
 * Sign i is bit (i mod 64) of output floor(i/64) of SplitMix64 seeded with
 * `seed` (Steele, Lea and Flood, OOPSLA 2014). */
int kv_codec_signs(uint64_t seed, uint32_t head_dim, uint8_t* negate);

/* Format version 2: the sign vector of `layer` for (seed, head_dim), one byte
 * per element, 1 = negate.  Layer l takes the W = ceil(head_dim / 64) outputs
 * l*W .. l*W + W - 1 of the same SplitMix64 stream (sign i is bit (i mod 64)
 * of output l*W + floor(i/64)), so layer 0 is the kv_codec_signs vector.
 * layer < KV_CODEC_MAX_LAYERS. */
int kv_codec_layer_signs(uint64_t seed, uint32_t layer, uint32_t head_dim, uint8_t* negate);

/* ABI version compiled into the library. */
uint32_t kv_codec_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KV_CODEC_H */
