/*
 * kvc.h -- C ABI of the GB300 KV-cache compression data path.
 *
 * The path (encode): per-channel key smoothing -> optional randomized Hadamard
 * rotation along head_dim -> group-wise asymmetric min-max quantization (2/3/4/8
 * bit codes, fp16 scale and zero) -> bit-packing into one all-layer payload ->
 * chunked lossless stage pipeline (tuple shuffle, bit shuffle, delta, zero-word
 * elimination).  Decode is the exact inverse.  Sources:
 *   "KVServe: Service-Aware KV Cache Compression for Communication-Efficient
 *    Disaggregated LLM Serving", §5.1 (pipeline BS = C(Q(T(X))): transformer,
 *    quantizer, codec; layer-/head-wise precision), §7.3 (KIVI metadata);
 *   "Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated
 *    LLM Serving", §4.1 (fused transform + quantization writing a preallocated
 *    all-layer buffer; fused reconstruction) and §4.2 (LC-style lossless backend
 *    TUPL8_1 -> BIT_8 -> RZE_2 with device-pointer encode/decode APIs, persistent
 *    scratch and a compressed-size scalar returned to the host).
 *
 * Conventions
 *  - Every pointer named d_* or documented as "device" is CUDA device memory of
 *    the current device; host pointers are documented as such.  The caller owns
 *    every buffer (inputs, outputs, stream, workspace).  A plan owns host memory
 *    only and never allocates device memory; encode/decode allocate nothing.
 *  - Work is enqueued asynchronously on the caller's CUDA stream.  Every entry
 *    point that enqueues work first resets the workspace status word, so
 *    kvc_query() reports the errors of the last call only.  Argument and
 *    profile errors are returned synchronously; errors found by the GPU (corrupt
 *    stream, non-finite input, fp16 metadata overflow, look-back timeout) set bits
 *    of a status word in the workspace, which kvc_query() reads after a sync.
 *  - Device buffers must be 16-byte aligned; token and page strides multiples of 16.
 *  - A plan is not thread-safe; use one plan per concurrently-issuing host thread.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *kvc_stream_t;

typedef enum kvc_status {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned buffer, bad block-table entry */
    KVC_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head_dim != 128) */
    KVC_ERR_CAPACITY = 3,    /* output or workspace smaller than required */
    KVC_ERR_CORRUPT = 4,     /* stream header / chunk table / chunk payload inconsistent */
    KVC_ERR_RANGE = 5,       /* an fp16 zero, scale or smoothing centre overflowed (saturated) */
    KVC_ERR_NONFINITE = 6,   /* NaN or Inf in the encode input (output bytes unspecified) */
    KVC_ERR_TIMEOUT = 7,     /* a bounded device wait gave up (chunk offset look-back) */
    KVC_ERR_CUDA = 8         /* a CUDA runtime call failed */
} kvc_status;

/* Bits of the device status word (kvc_query's host_flags). */
#define KVC_FLAG_RANGE 1u
#define KVC_FLAG_NONFINITE 2u
#define KVC_FLAG_CORRUPT 4u
#define KVC_FLAG_CAPACITY 8u
#define KVC_FLAG_TIMEOUT 16u
#define KVC_FLAG_BAD_PAGE 32u

enum { KVC_F16 = 1, KVC_BF16 = 2 };
/* Quantization axis ("Beyond Compression Ratio" §4.1: channel-wise keys, token-wise values). */
enum { KVC_AXIS_OVER_TOKENS = 0, KVC_AXIS_OVER_CHANNELS = 1 };
/* Lossless stage kinds ("Beyond Compression Ratio" §4.2). */
enum { KVC_ST_TUPL = 1, KVC_ST_BIT = 2, KVC_ST_DELTA = 3, KVC_ST_RZE = 4 };

#define KVC_MAX_STAGES 4
#define KVC_MAX_LAYERS 256
#define KVC_HEADER_BYTES 64 /* fixed part; a v2 width map follows it (kvc_header_bytes) */

/* One lossless stage: TUPL param k in {2,4,8} (k-byte tuples -> k byte columns);
 * BIT param 8 (bit planes of bytes); DELTA param w in {1,2,4} (w-byte words,
 * differences mod 2^(8w)); RZE param w in {1,2,4} (zero-word elimination with a
 * two-level bitmap; only as the last stage). */
typedef struct kvc_stage {
    uint8_t kind;
    uint8_t param;
} kvc_stage;

/* A compression profile, chosen per request and fixed for it ("KVServe" §3.1).
 * struct_size versions the struct: sizeof(kvc_profile), or KVC_PROFILE_V1_SIZE for
 * callers built before the format-v2 fields (they read as 0 / NULL). */
typedef struct kvc_profile {
    uint32_t struct_size;   /* = sizeof(kvc_profile) (or KVC_PROFILE_V1_SIZE) */
    uint8_t smooth_keys;    /* per-channel key smoothing (128-token blocks) */
    uint8_t hadamard;       /* randomized Hadamard rotation along head_dim (K and V) */
    uint8_t bits_k, bits_v; /* code width: 2, 3, 4 or 8 */
    uint16_t group_k, group_v; /* group size: 32, 64 or 128 */
    uint8_t axis_k, axis_v;    /* KVC_AXIS_*; defaults OVER_TOKENS for K, OVER_CHANNELS for V */
    uint8_t n_stages;          /* 0 = no lossless stage (the stream carries the payload as is) */
    uint8_t reserved0;
    kvc_stage stages[KVC_MAX_STAGES];
    uint32_t chunk_bytes;      /* lossless chunk size: multiple of 256 in [256, 65536] */
    uint32_t reserved1;
    uint64_t hadamard_seed;    /* seed of the +-1 sign vector (SplitMix64) */
    /* ---- format v2 (optional; a profile that uses neither writes v1 streams) ---- */
    /* Token delta ("KVServe" §5.1, the Delta transformer, after CacheGen): the first
     * token of every 128-token block is the anchor; K and V rows become their fp32
     * differences from it before smoothing and the Hadamard rotation, the anchors'
     * element bits go to payload sections 6 (K) and 7 (V). */
    uint8_t token_delta;
    uint8_t reserved2[7];
    /* Per-(layer, head) code widths ("KVServe" §5.1 layer- and head-wise mixed
     * precision; "Beyond Compression Ratio" §4.1 head-importance-aware mixed
     * precision): HOST arrays of layers * kv_heads widths in {2, 3, 4, 8}, entry
     * l * kv_heads + h, read (copied) by kvc_plan only; NULL = bits_k / bits_v for
     * every head.  With either map: layers * kv_heads <= KVC_MAX_MAP_ENTRIES. */
    const uint8_t *bits_map_k;
    const uint8_t *bits_map_v;
} kvc_profile;
#define KVC_PROFILE_V1_SIZE 40
#define KVC_MAX_MAP_ENTRIES 2048

/* KV tensor geometry.  Each layer's K (and V) is addressed as rows of
 * kv_heads*head_dim elements: token t lives at
 *     base + t*token_stride                                   (no block table)
 *     base + block_table[t/page_size]*page_stride + (t%page_size)*token_stride
 * and head h of that row at + h*head_dim*element_size. */
typedef struct kvc_shape {
    uint32_t struct_size;  /* = sizeof(kvc_shape) */
    uint32_t layers;       /* 0 .. KVC_MAX_LAYERS */
    uint32_t tokens;       /* 0 .. 2^31-1 */
    uint32_t kv_heads;     /* >= 1 */
    uint32_t head_dim;     /* 128 */
    uint32_t dtype;        /* KVC_F16 or KVC_BF16 */
    uint32_t page_size;    /* tokens per page, power of two (block table only) */
    uint32_t num_pages;    /* physical pages per layer buffer (block table only; bounds check) */
    uint64_t token_stride; /* bytes between token rows; 0 = kv_heads*head_dim*element_size */
    uint64_t page_stride;  /* bytes between physical pages (block table only) */
} kvc_shape;

/* Where the KV of every layer lives (encode input / decode output). */
typedef struct kvc_kv {
    void *const *k_layers;      /* HOST array of `layers` DEVICE pointers to K */
    void *const *v_layers;      /* HOST array of `layers` DEVICE pointers to V */
    const int32_t *block_table; /* DEVICE array of ceil(tokens/page_size) physical page
                                   ids shared by all layers; NULL = contiguous layout */
} kvc_kv;

typedef struct kvc_plan_s kvc_plan_t;

/* Validate a profile and shape and precompute the payload layout, stream bounds
 * and the Hadamard sign vector ("Beyond Compression Ratio" §4.1: signs and
 * workspaces cached and reused across layers and requests).  Host-only object.
 * Returns KVC_ERR_INVALID_ARG / KVC_ERR_UNSUPPORTED without creating a plan. */
kvc_status kvc_plan(const kvc_profile *profile, const kvc_shape *shape, kvc_plan_t **out);
void kvc_plan_destroy(kvc_plan_t *plan);

/* Bytes of the caller-provided device workspace encode/decode need ("persistent
 * runtime scratch", "Beyond Compression Ratio" §4.2): a 256-byte control block
 * (status word, stream size, chunk tickets), per-chunk look-back / offset /
 * chunk-address words (and one word per 4096 chunks for the decode's partial
 * sums) and, when lossless stages are on, the quantized payload. */
size_t kvc_workspace_bytes(const kvc_plan_t *plan);
/* Worst-case stream size (header + chunk table + every chunk stored raw): the
 * capacity of the caller's preallocated output buffer ("Beyond Compression
 * Ratio" §4.1, all-layer output buffer; §4.2, device bitstream). */
size_t kvc_max_stream_bytes(const kvc_plan_t *plan);
/* Bytes of the quantized payload Q (all sections, each 16-byte aligned). */
size_t kvc_payload_bytes(const kvc_plan_t *plan);
/* Offset and size of payload section i: 0 K codes, 1 K scale/zero, 2 V codes,
 * 3 V scale/zero, 4 K smoothing centres (fp16), 5 K smoothing exponents (int8),
 * 6 K delta anchors, 7 V delta anchors (element bits). */
kvc_status kvc_section(const kvc_plan_t *plan, int index, uint64_t *offset, uint64_t *size);
/* Number of lossless chunks (0 without stages). */
uint64_t kvc_num_chunks(const kvc_plan_t *plan);
/* Bytes of the stream header: 64, plus the 2-bit width map (padded to 16 bytes)
 * when the profile has per-(layer, head) widths.  The chunk table (or, without
 * stages, the payload) starts there. */
size_t kvc_header_bytes(const kvc_plan_t *plan);

/* Full encode ("KVServe" §5.1: BS = C(Q(T(X))); "Beyond Compression Ratio" §4.1
 * fused transform + quantization into the all-layer buffer, §4.2 device-pointer
 * encoding API): quantize all layers into the payload, then header + lossless
 * stream into d_stream (capacity stream_cap >= kvc_max_stream_bytes).  Inputs:
 * in->k_layers / v_layers as described by the plan's shape (device, read only).
 * d_workspace: kvc_workspace_bytes(plan) bytes of caller-owned device memory
 * (16-byte aligned), reused across calls.  The stream size is written to the
 * device word *d_stream_bytes (may be NULL) and to the workspace control block;
 * kvc_query() returns it to the host.  No host sync.  Returns INVALID_ARG for
 * null or misaligned pointers, CAPACITY for a short stream or workspace. */
kvc_status kvc_encode(kvc_plan_t *plan, const kvc_kv *in, void *d_stream, size_t stream_cap,
                      void *d_workspace, size_t workspace_bytes, uint64_t *d_stream_bytes,
                      kvc_stream_t stream);

/* Full decode ("Beyond Compression Ratio" §4.2 device-pointer decoding API, §4.1
 * fused reconstruction: dequantize, inverse Hadamard, normalization, sign
 * restoration) of a stream of stream_bytes bytes (device) into the layers of
 * *out (device, same geometry as the plan; written, never read).  The header and
 * chunk table are checked against the plan on the device; a corrupt stream sets
 * KVC_FLAG_CORRUPT and leaves *out untouched.  The stream must stay unchanged
 * until the decode has run: by default (kvc_decode_codes_in_place) the
 * reconstruction reads the codes of stored chunks from it.  No host sync. */
kvc_status kvc_decode(kvc_plan_t *plan, const void *d_stream, size_t stream_bytes, const kvc_kv *out,
                      void *d_workspace, size_t workspace_bytes, kvc_stream_t stream);

/* The four steps of the path, one call each (encode = quantize + lossless_encode,
 * decode = lossless_decode + dequantize).  d_payload holds kvc_payload_bytes. */
/* Smoothing, Hadamard, group statistics, quantization and packing (fused). */
kvc_status kvc_quantize(kvc_plan_t *plan, const kvc_kv *in, void *d_payload, void *d_workspace,
                        size_t workspace_bytes, kvc_stream_t stream);
/* Header + chunk table + lossless chunks of a payload; stream size to *d_stream_bytes. */
kvc_status kvc_lossless_encode(kvc_plan_t *plan, const void *d_payload, void *d_stream, size_t stream_cap,
                               void *d_workspace, size_t workspace_bytes, uint64_t *d_stream_bytes,
                               kvc_stream_t stream);
/* Validate a stream and restore its payload. */
kvc_status kvc_lossless_decode(kvc_plan_t *plan, const void *d_stream, size_t stream_bytes, void *d_payload,
                               void *d_workspace, size_t workspace_bytes, kvc_stream_t stream);
/* Dequantization, inverse Hadamard, normalization, sign restoration, unsmoothing
 * and conversion to the element type (fused).  (Inside kvc_decode this step is
 * skipped on the device when the lossless decode found the stream corrupt.) */
kvc_status kvc_dequantize(kvc_plan_t *plan, const void *d_payload, const kvc_kv *out, void *d_workspace,
                          size_t workspace_bytes, kvc_stream_t stream);

/* The compressed-size scalar returned to the host ("Beyond Compression Ratio"
 * §4.2: only the size crosses to the host, the stream stays on the device).
 * Synchronize `stream`, then read the workspace control block: the stream size of
 * the last encode (host_stream_bytes, may be NULL) and the status bits
 * (host_flags, may be NULL).  Returns the most severe error the bits encode
 * (CORRUPT > CAPACITY > TIMEOUT > INVALID_ARG (bad page) > NONFINITE > RANGE) or KVC_OK. */
kvc_status kvc_query(const void *d_workspace, kvc_stream_t stream, uint64_t *host_stream_bytes,
                     uint32_t *host_flags);

const char *kvc_status_str(kvc_status status);

/* Allocation-free variant of kvc_lossless_encode (no counterpart in the pages; an
 * addition for callers that cannot allocate device memory, e.g. a transport or
 * storage plugin called from inside another runtime's send path that receives
 * only the payload and output buffers and must not call cudaMalloc there, which
 * can synchronize the device or is barred by the host framework's memory pool).
 * The encoder's scratch -- the 256-byte control block and one 64-bit look-back
 * word per chunk -- lives in a device array of KVC_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the process
 * exits.  Plans whose 256 + 8 * kvc_num_chunks(plan) bytes exceed that size are
 * rejected with KVC_ERR_CAPACITY (1 MiB: up to 131040 chunks, i.e. 2 GiB of
 * payload at 16 KiB chunks).  Arguments as kvc_lossless_encode, except:
 * d_stream_bytes (device u64, required) receives the stream size, and d_status
 * (device u32, may be NULL) receives the status bits (KVC_FLAG_*); kvc_query does
 * not apply.  Allocates nothing (no cudaMalloc / cudaFree).  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and caches
 * it for that device's current context; make that first call before any stream
 * capture.  After the device is reset (cudaDeviceReset) the next call looks the
 * address up again in the new context (so, again, before any capture).  All calls share the one
 * array (its words are reset at the start of every call), so calls whose GPU work
 * overlaps -- on different streams or from different threads -- race; serialize them. */
#define KVC_NOALLOC_SCRATCH_BYTES (1u << 20)
kvc_status kvc_lossless_encode_noalloc(kvc_plan_t *plan, const void *d_payload, void *d_stream, size_t stream_cap,
                                       uint64_t *d_stream_bytes, uint32_t *d_status, kvc_stream_t stream);

/* ---- measurement hooks ---------------------------------------------------- */
/* Number of kernel launches this plan has enqueued so far. */
uint64_t kvc_launch_count(const kvc_plan_t *plan);
/* enable != 0: bracket every kernel launch with CUDA events (up to `capacity`
 * launches are kept); enable == 0 stops.  Returns KVC_ERR_CUDA if events fail. */
kvc_status kvc_timing_enable(kvc_plan_t *plan, int enable, int capacity);
/* After a sync: copy up to `max` records (kernel name, milliseconds) of the
 * launches recorded since kvc_timing_enable and return how many were written. */
typedef struct kvc_timing {
    const char *kernel;
    float ms;
} kvc_timing;
int kvc_timing_read(kvc_plan_t *plan, kvc_timing *out, int max);

/* Execution choice for kvc_encode (the stream is the same byte for byte either way):
 * with enable != 0 the value encoder itself writes the whole lossless chunks of the
 * value-code section into the stream -- it quantizes a chunk's rows into shared
 * memory, runs the chunk's stages there and takes the chunk's place through the
 * look-back -- between a lossless launch over the chunks before that section and
 * one over the rest ("Beyond Compression Ratio" §3 design goal G1, one kernel for
 * closely coupled operations; §4.1-4.2).  It applies when the values are grouped
 * over channels with a uniform width of 2, 4 or 8 bits and no token delta, the
 * stage list is TUPL_8 BIT_8 [DELTA_1] RZE_1/2 with 4, 8, 12 or 16 KiB chunks that
 * hold a multiple of 128 value rows, and the value-code section starts on a chunk
 * boundary; otherwise kvc_encode runs as usual.  Off by default: on a GB300 the
 * fused value encoder (llama8b, 16 KiB chunks) takes longer than the value encoder
 * and the lossless work it saves together.  Returns KVC_ERR_INVALID_ARG for a null
 * plan. */
kvc_status kvc_fuse_value_chunks(kvc_plan_t *plan, int enable);

/* Execution choice for kvc_decode (the reconstruction is the same either way): with
 * enable != 0 (the default) the dequantizers read the codes of stored (raw) chunks
 * straight from the stream, so those chunks never pass through the workspace
 * payload; the lossless decoder restores only the other chunks ("Beyond Compression
 * Ratio" §3 design goal G1 and §4.2: the decoder's output feeds reconstruction on
 * the device).  It applies per tensor to the whole chunks of its code section when
 * the width is a uniform 2, 4 or 8 bits, chunk_bytes is a power of two, the section
 * starts on a chunk boundary, and either the groups run over tokens with
 * ceil(T / group) * group a multiple of 128 and 2048 * bits dividing chunk_bytes,
 * or they run over channels without key smoothing.  kvc_lossless_decode always
 * writes the whole payload.  Returns KVC_ERR_INVALID_ARG for a null plan. */
kvc_status kvc_decode_codes_in_place(kvc_plan_t *plan, int enable);

/* ---- test hooks -------------------------------------------------------------- */
/* Fault injection on the host side of the look-back scan: the chunk with ticket
 * `ticket` (>= 0) does not publish its size, so its successor's bounded wait runs
 * out after `poll_limit` polls and sets KVC_FLAG_TIMEOUT.  ticket < 0 disables it;
 * poll_limit = 0 restores the default limit. */
kvc_status kvc_debug_lookback(kvc_plan_t *plan, int64_t ticket, uint32_t poll_limit);
/* Measurement hook for comparing stage lists on equal terms ("Beyond Compression
 * Ratio" §4.2, offline pipeline search): enable != 0 makes this plan's lossless
 * encode and decode use the generic stage kernels even for the stage lists and
 * chunk sizes that have a fast kernel (TUPL_8 [BIT_8] [DELTA_1] RZE_1/2, chunks of
 * 4, 8, 12 or 16 KiB).  Streams are identical either way.  Measurements name the
 * launches kvc_lossless_enc / kvc_lossless_dec (generic) or kvc_lossless_enc_fast /
 * kvc_lossless_dec_fast. */
kvc_status kvc_debug_generic_stages(kvc_plan_t *plan, int enable);
/* Self-check of the encoders' two quotient steps (no plan).  The min-max rule
 * ("Beyond Compression Ratio" §4.1, group-wise asymmetric quantization; "KVServe"
 * §5.1, KIVI-style min-max) divides twice: the group scale s = fp16_up(RN(w / Q))
 * with w = max - z and Q = 2^b - 1, and the code rint(RN(RN(y - z) / s)).  The
 * encoders form both quotients as q = RN(t * RN(1/d)) corrected once by the exact
 * residual t - q d (Markstein's correction).  Codes: each round tests every
 * positive finite binary16 divisor s against 256 x 256 dividends t drawn from
 * `seed + round` (uniform in [0, 256 s), within 4 ulps of k s and of (k + 1/2) s
 * for k < 256, and any normal value below 2^17) and compares with the correctly
 * rounded division: counts[0] = quotients that differ for t >= 1e-30, counts[1] =
 * codes that differ (quotients below 4096), counts[2] = dividends tested.  Scales:
 * every non-negative binary32 pattern w for b = 2, 3, 4, 8 (one pass, whatever
 * `rounds`): counts[3] = quotients that differ for finite w >= 1e-30, counts[4] =
 * binary16 scales that differ, counts[5] = patterns tested.  Host array of 6.
 * Synchronizes `stream`; allocates 48 bytes of device memory for the call.
 * Returns KVC_ERR_INVALID_ARG for a null `counts`, KVC_ERR_CUDA on a CUDA error. */
kvc_status kvc_debug_quotient_check(uint32_t seed, uint32_t rounds, unsigned long long *counts, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
