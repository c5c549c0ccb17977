// kvc_internal.h -- parameter blocks shared by the C-ABI host code and the kernels.
//
// Workspace control block (first 256 bytes of the caller's workspace):
//   u32 [0]  status flags (KVC_FLAG_*), set with atomicOr by any kernel
//   u64 @8   stream size written by the last encode
//   u32 [4]  chunk ticket counter of the lossless encoder ([5], [6]: the value
//            encoder that writes code chunks into the stream, and the encoder
//            launch after it)
// followed at byte 256 by one u64 per lossless chunk (encode: look-back words;
// decode: chunk byte offsets, then for chunks whose codes are read in place the
// address of their bytes) and one u64 per kDecodeSumSeg chunks (the decode
// prepare's partial sums), then (256-aligned) the quantized payload when lossless
// stages are on.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kHeadDim = 128;       // only head_dim = 128 is built
constexpr int kSmoothBlock = 128;   // tokens per key-smoothing block
constexpr uint32_t kCtrlBytes = 256;
constexpr int kCtrlFlags = 0;       // u32 index
constexpr int kCtrlStreamBytes = 1; // u64 index
constexpr int kCtrlTicket = 4;      // u32 index (a split encode also uses the next two words)
constexpr int kSections = 8;        // payload sections (kvc_section)
constexpr uint32_t kDecodeSumSeg = 4096;  // table entries per partial sum of the decode prepare
// largest stream header: 64 bytes + a 2-bit width map of KVC_MAX_MAP_ENTRIES
// (layer, head) entries for each of K and V
constexpr int kMaxHeaderBytes = KVC_HEADER_BYTES + 2 * KVC_MAX_MAP_ENTRIES * 2 / 8;

// Geometry of one KV tensor (K or V) of every layer.
struct KvGeom {
  uint32_t L, T, H;
  uint32_t bf16;            // 1 = bfloat16, 0 = binary16
  uint64_t token_stride;    // bytes
  uint64_t page_stride;     // bytes
  const int32_t *block_table;
  uint32_t page_shift, page_mask, num_pages;
  uint32_t pad_;
};

// One quantize or dequantize launch over one tensor.
struct QuantParams {
  KvGeom g;
  void *layers[KVC_MAX_LAYERS];  // K or V base pointer per layer (const on encode)
  uint32_t bits, group, axis, smooth;
  uint32_t n_tg;                 // token groups per (layer, head) = ceil(T / group)
  uint32_t n_sb;                 // smoothing blocks per (layer, head) = ceil(T / 128)
  uint32_t sign[4];              // bit j set => Hadamard sign j is -1
  uint8_t *codes;                // code section
  uint8_t *meta;                 // {scale, zero} section
  uint8_t *mu;                   // fp16 smoothing centres (keys)
  int8_t *ex;                    // int8 smoothing exponents (keys)
  uint32_t *status;              // workspace status word
  uint32_t check_corrupt;        // dequantize: skip when the status word carries CORRUPT
  uint32_t hadamard;             // randomized Hadamard on
  uint32_t tma;                  // key-tile encoder: tiles arrive through the tensor maps (TmaMaps)
  uint32_t delta;                // token delta: subtract (add back) each 128-token block's first row
  uint32_t mixed;                // per-(layer, head) widths: the launch also takes a WidthTable
  uint8_t *anchors;              // token delta: anchor element bits [layer][head][block][channel]
  // decode with codes read in place (in_lo < in_hi): the code bytes at payload
  // offset o = codes_off + (their offset from `codes`) lie in chunk c = o >> chunk_shift;
  // for in_lo <= c < in_hi they are read at src_of[c] + (o mod 2^chunk_shift), the
  // address the lossless decoder left there (the stored chunk in the stream when it
  // is stored raw, else the chunk decoded into the payload).  A decoder reads one
  // unit (a key tile, 16 value rows) from one such lookup, so the host enables it
  // only where no unit crosses a chunk boundary.
  const uint64_t *src_of;
  uint64_t codes_off;
  uint32_t chunk_shift, in_lo, in_hi, pad3_;
};

// Per-(layer, head) widths of one tensor: wsum[i] = sum of the widths of entries
// 0 .. i-1 (entry = layer * H + head), i = 0 .. L*H; the width of entry i is
// wsum[i + 1] - wsum[i].  Code offsets follow from it: groups over tokens, the
// (layer, head) block starts at 16 * n_tg * G * wsum[lh] bytes; groups over
// channels, layer l starts at 16 * T * wsum[l*H], token t of it at
// + 16 * t * (wsum[(l+1)*H] - wsum[l*H]) and head h at + 16 * (wsum[lh] - wsum[l*H]).
struct WidthTable {
  uint16_t wsum[KVC_MAX_MAP_ENTRIES + 1];
};

// Tensor maps of one tensor's layers for the key-tile encoder's TMA loads: rank 2
// (H*128 channels innermost, T tokens; row stride = token stride), box 64
// channels x 128 tokens, 128-byte swizzle, rows past T read as zero.  Passed as a
// kernel parameter, so at most kTmaMaxLayers layers (beyond that the encoder
// loads with cp.async).
constexpr int kTmaMaxLayers = 128;
struct TmaMaps {
  CUtensorMap map[kTmaMaxLayers];
};

// Prologue: reset workspace words, write the stream header.
struct PrologueParams {
  uint32_t *ctrl;
  uint64_t *state;      // look-back words to zero
  uint64_t n_state;
  uint32_t zero_flags;  // also clear the status word
  uint32_t write_header;
  uint8_t *stream;
  uint32_t header_bytes;
  uint8_t header[kMaxHeaderBytes];
  uint64_t static_size; // nonzero: the stream size is known now (no lossless chunks)
  uint64_t gap_off;     // zero padding between the chunk table and the first chunk
  uint32_t gap_len;
  uint32_t pad_;
  uint64_t *d_stream_bytes;
  // zero padding bytes of the payload sections
  uint8_t *payload;
  uint64_t pad_off[kSections];
  uint32_t pad_len[kSections];
};

struct LosslessParams {
  const uint8_t *payload;
  uint64_t payload_bytes;
  uint8_t *stream;         // encode output / decode input
  uint64_t stream_cap;     // encode: capacity; decode: stream bytes
  uint64_t data_start;
  uint32_t chunk_bytes, n_chunks;
  uint32_t n_stages;
  uint8_t kind[KVC_MAX_STAGES], param[KVC_MAX_STAGES];
  uint64_t *state;         // encode: look-back words; decode: chunk offsets
  uint32_t *ctrl;
  uint64_t *d_stream_bytes;
  uint8_t *out_payload;    // decode output
  int64_t skip_ticket;     // test hook: this ticket does not publish
  uint32_t poll_limit;
  uint32_t fused_offsets;  // decode: the decoder checks the table and computes the chunk offsets itself
  uint32_t header_bytes;   // the chunk table starts here
  uint32_t generic_only;   // measurement hook: the generic stage kernels even where a fast one exists
  // encode: this launch takes chunks first_chunk .. last_chunk - 1, in the order of
  // the ticket counter ctrl[ticket_word] (the whole stream: 0, n_chunks, kCtrlTicket)
  uint32_t first_chunk, last_chunk, ticket_word, pad2_;
  // decode: chunks c with inplace_lo[i] <= c < inplace_hi[i] hold codes that the
  // dequantizers read in place; the decoder leaves a raw one in the stream (no copy)
  // and sets state[c] to the address of the chunk's bytes (stream or payload)
  uint32_t inplace_lo[2], inplace_hi[2];
  uint8_t header[kMaxHeaderBytes];  // decode: expected header (header_bytes of it)
};

// Self-checks of the encoders' quotient steps (counts in device memory): the codes'
// quotients (one round of dividends) and the group scales' quotients (every pattern).
int launch_quotient_check(uint32_t seed, unsigned long long *d_counts, void *stream);
int launch_range_check(unsigned long long *d_counts, int sm_count, void *stream);

// Launchers (return cudaError_t as int).  `occ_grid` = resident-grid size to use.
// max_per_sm > 0 caps the resident CTAs per SM of the launch (so that a kernel
// launched beside it on another stream finds room on every SM).
int launch_quantize(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, int sm_count, int max_per_sm,
                    void *stream, uint64_t *launches, const char **name);
int launch_dequantize(const QuantParams &p, const WidthTable *widths, int sm_count, int max_per_sm, void *stream,
                      uint64_t *launches, const char **name);
int launch_prologue(const PrologueParams &p, void *stream);
int launch_lossless_encode(const LosslessParams &p, int sm_count, void *stream);
// The value encoder that writes the whole chunks of the value-code section into
// the stream itself (kvc_fused.cu): whether a profile takes it (the section, at
// byte codes_off of the payload, starts on a chunk boundary, its chunks hold whole
// rows, the stage list has the fast path with BIT_8), the chunk index of the
// section's start and its number of whole chunks; and the launch, which takes its
// chunks by the ticket counter ctrl[lp.ticket_word].
bool v_lossless_fusable(const QuantParams &v, const LosslessParams &lp, uint64_t codes_off, uint64_t codes_bytes,
                        uint32_t *c0, uint32_t *nfull);
int launch_v_lossless(const QuantParams &v, const LosslessParams &lp, uint32_t c0, uint32_t nfull, int sm_count,
                      void *stream);
int launch_decode_prepare(const LosslessParams &p, void *stream);
int launch_lossless_decode(const LosslessParams &p, int sm_count, void *stream);
// Whether launch_lossless_decode can take the prepare step into the decoder for
// this table size (nothing else needs to run first except the status reset).
bool lossless_decode_fusable(const LosslessParams &p, int sm_count);
// Whether the encoder / decoder launch for these parameters takes the fast path
// (worker/publisher encoder; fast chunk decode), for naming measurements.
bool lossless_encode_is_fast(const LosslessParams &p);
bool lossless_decode_is_fast(const LosslessParams &p);

}  // namespace kvc
