// kvc_api.cu -- the C ABI (include/kvc.h): plans, payload layout, launches.
//
// Payload layout (the "preallocated all-layer output buffer" of "Beyond
// Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
// Serving", §4.1), sections in this order, each starting 16-byte aligned:
//   0 K codes, 1 K {scale, zero}, 2 V codes, 3 V {scale, zero},
//   4 K smoothing centres (fp16), 5 K smoothing exponents (int8),
//   6 K delta anchors, 7 V delta anchors (element bits; token delta only).
// Groups over tokens: records [layer][head][token group][channel]; groups over
// channels: records [layer][token][head][channel group]; smoothing and anchor
// cells [layer][head][128-token block][channel].  A record holds G codes of b
// bits, least significant bit first.  With per-(layer, head) widths ("KVServe"
// §5.1 mixed precision) each (layer, head) -- or each head of a token row --
// keeps its own record size; the offsets follow from prefix sums of the widths.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <new>
#include <stdlib.h>
#include <string.h>
#include <vector>

#include "kvc_internal.h"

using namespace kvc;

struct TimingRec {
  const char *name;
  cudaEvent_t start, stop;
};

struct kvc_plan_s {
  kvc_profile prof;  // bits_map_* cleared: the plan keeps its own copies below
  kvc_shape shape;
  uint64_t off[kSections], size[kSections];
  uint64_t payload_bytes, n_chunks, data_start, max_stream_bytes, workspace_bytes;
  uint64_t n_tg_k, n_tg_v, n_sb;
  uint32_t sign[4];
  uint32_t header_bytes;
  uint8_t header[kMaxHeaderBytes];
  bool mixed;                    // per-(layer, head) widths
  std::vector<uint8_t> width[2]; // K, V: width of entry l * H + h (mixed only)
  WidthTable *wt[2];             // prefix sums of the widths (mixed only)
  int sm_count;
  uint64_t launches;
  // K and V kernels run side by side: V on this stream, forked from and joined
  // back into the caller's stream with two events (null: one after the other)
  cudaStream_t side;
  cudaEvent_t ev_fork, ev_join;
  // host-side tensor maps for the key-tile encoder's TMA loads, per tensor, and the
  // layer pointers they were encoded for
  TmaMaps *tm[2];
  const void *tm_ptr[2][kTmaMaxLayers];
  // timing
  bool timing;
  int timing_cap;
  std::vector<TimingRec> recs;
  std::vector<cudaEvent_t> pool;
  // test hooks
  int64_t skip_ticket;
  uint32_t poll_limit;
  bool generic_stages;
  // kvc_fuse_value_chunks: the value encoder writes its whole code chunks itself
  bool fuse_values;
  // kvc_decode_codes_in_place: kvc_decode's dequantizers read stored code chunks
  // from the stream
  bool codes_in_place;
};

static constexpr uint32_t kDefaultPollLimit = 1u << 22;

// Bytes of the workspace's per-chunk words: one u64 per chunk (look-back words,
// then decode offsets) and one per kDecodeSumSeg chunks (the decode prepare's
// partial sums), 256-aligned.
static uint64_t state_bytes(uint64_t n_chunks) {
  const uint64_t n_sums = (n_chunks + kDecodeSumSeg - 1) / kDecodeSumSeg;
  return (8 * (n_chunks + n_sums) + 255) / 256 * 256;
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t align_up(uint64_t a, uint64_t b) { return (a + b - 1) / b * b; }

// SplitMix64 (S. Vigna), the published 64-bit mixing generator.
static uint64_t splitmix64(uint64_t &state) {
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static bool valid_bits(uint32_t b) { return b == 2 || b == 3 || b == 4 || b == 8; }
static bool valid_group(uint32_t g) { return g == 32 || g == 64 || g == 128; }

// Copy a caller's profile of either struct version into a full one.
static kvc_status read_profile(const kvc_profile *in, kvc_profile *out) {
  memset(out, 0, sizeof *out);
  if (in->struct_size == sizeof(kvc_profile)) memcpy(out, in, sizeof *out);
  else if (in->struct_size == KVC_PROFILE_V1_SIZE) memcpy(out, in, KVC_PROFILE_V1_SIZE);
  else return KVC_ERR_INVALID_ARG;
  out->struct_size = sizeof(kvc_profile);
  return KVC_OK;
}

static kvc_status check_profile(const kvc_profile *p) {
  if (!valid_bits(p->bits_k) || !valid_bits(p->bits_v)) return KVC_ERR_INVALID_ARG;
  if (p->token_delta > 1) return KVC_ERR_INVALID_ARG;
  if (!valid_group(p->group_k) || !valid_group(p->group_v)) return KVC_ERR_INVALID_ARG;
  if (p->axis_k > 1 || p->axis_v > 1) return KVC_ERR_INVALID_ARG;
  if (p->smooth_keys > 1 || p->hadamard > 1) return KVC_ERR_INVALID_ARG;
  if (p->n_stages > KVC_MAX_STAGES) return KVC_ERR_INVALID_ARG;
  for (uint32_t s = 0; s < p->n_stages; s++) {
    const uint32_t k = p->stages[s].kind, prm = p->stages[s].param;
    bool ok = false;
    if (k == KVC_ST_TUPL) ok = prm == 2 || prm == 4 || prm == 8;
    else if (k == KVC_ST_BIT) ok = prm == 8;
    else if (k == KVC_ST_DELTA) ok = prm == 1 || prm == 2 || prm == 4;
    else if (k == KVC_ST_RZE) ok = (prm == 1 || prm == 2 || prm == 4) && s + 1 == p->n_stages;
    if (!ok) return KVC_ERR_INVALID_ARG;
  }
  if (p->n_stages && (p->chunk_bytes < 256 || p->chunk_bytes > 65536 || p->chunk_bytes % 256))
    return KVC_ERR_INVALID_ARG;
  return KVC_OK;
}

static uint64_t groups(const kvc_shape &s, uint32_t axis, uint32_t G) {
  const uint64_t L = s.layers, T = s.tokens, H = s.kv_heads, D = s.head_dim;
  return axis == KVC_AXIS_OVER_TOKENS ? L * H * ceil_div(T, G) * D : L * T * H * (D / G);
}

// Width code of the v2 header map: 2, 3, 4, 8 -> 0, 1, 2, 3.
static uint32_t width_code(uint32_t b) { return b == 2 ? 0u : b == 3 ? 1u : b == 4 ? 2u : 3u; }

static void put16(uint8_t *p, uint32_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }

// Stream header, 64 bytes little-endian: magic "KVC1", version (2 when the token
// delta or per-(layer, head) widths are used, else 1), header size, geometry,
// profile (flags: 1 smoothing, 2 Hadamard, 4 token delta, 8 width map), chunking,
// seed and payload size; with a width map, the map follows (2 bits per entry,
// entry i at bits 2i..2i+1, K entries then V entries, padded to 16 bytes).
static void build_header(kvc_plan_s *P) {
  uint8_t *h = P->header;
  memset(h, 0, sizeof P->header);
  const bool v2 = P->prof.token_delta || P->mixed;
  h[0] = 'K'; h[1] = 'V'; h[2] = 'C'; h[3] = '1';
  put16(h + 4, v2 ? 2 : 1);
  put16(h + 6, P->header_bytes);
  put32(h + 8, P->shape.layers);
  put32(h + 12, P->shape.tokens);
  put16(h + 16, P->shape.kv_heads);
  put16(h + 18, P->shape.head_dim);
  h[20] = (uint8_t)P->shape.dtype;
  h[21] = (uint8_t)((P->prof.smooth_keys ? 1 : 0) | (P->prof.hadamard ? 2 : 0) | (P->prof.token_delta ? 4 : 0) |
                    (P->mixed ? 8 : 0));
  h[22] = P->mixed ? 0 : P->prof.bits_k;
  h[23] = P->mixed ? 0 : P->prof.bits_v;
  if (P->mixed) {
    const uint64_t n = (uint64_t)P->shape.layers * P->shape.kv_heads;
    for (int t = 0; t < 2; t++)
      for (uint64_t i = 0; i < n; i++) {
        const uint64_t e = t * n + i;
        h[KVC_HEADER_BYTES + e / 4] |= (uint8_t)(width_code(P->width[t][i]) << (2 * (e % 4)));
      }
  }
  put16(h + 24, P->prof.group_k);
  put16(h + 26, P->prof.group_v);
  h[28] = P->prof.axis_k;
  h[29] = P->prof.axis_v;
  h[30] = P->prof.n_stages;
  for (uint32_t s = 0; s < P->prof.n_stages; s++) {
    h[32 + 2 * s] = P->prof.stages[s].kind;
    h[33 + 2 * s] = P->prof.stages[s].param;
  }
  put32(h + 40, P->prof.n_stages ? P->prof.chunk_bytes : 0);
  put32(h + 44, (uint32_t)P->n_chunks);
  put64(h + 48, P->prof.hadamard_seed);
  put64(h + 56, P->payload_bytes);
}

extern "C" kvc_status kvc_plan(const kvc_profile *profile_in, const kvc_shape *shape, kvc_plan_t **out) {
  if (!profile_in || !shape || !out) return KVC_ERR_INVALID_ARG;
  *out = nullptr;
  kvc_profile prof;
  kvc_status st = read_profile(profile_in, &prof);
  if (st != KVC_OK) return st;
  const kvc_profile *profile = &prof;
  if ((st = check_profile(profile)) != KVC_OK) return st;
  kvc_shape s = *shape;
  if (s.struct_size != sizeof(kvc_shape)) return KVC_ERR_INVALID_ARG;
  if (s.dtype != KVC_F16 && s.dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (s.head_dim != (uint32_t)kHeadDim) return KVC_ERR_UNSUPPORTED;
  if (s.kv_heads < 1 || s.kv_heads > 65535 || s.layers > KVC_MAX_LAYERS || s.tokens > 0x7fffffffu)
    return KVC_ERR_INVALID_ARG;
  if ((uint64_t)s.layers * s.tokens * s.kv_heads >= (1ull << 31)) return KVC_ERR_UNSUPPORTED;
  const uint64_t row_bytes = (uint64_t)s.kv_heads * s.head_dim * 2;
  if (s.token_stride == 0) s.token_stride = row_bytes;
  if (s.token_stride < row_bytes || s.token_stride % 16) return KVC_ERR_INVALID_ARG;
  if (s.page_size) {
    if (s.page_size & (s.page_size - 1)) return KVC_ERR_INVALID_ARG;
    if (s.page_stride % 16 || s.num_pages == 0) return KVC_ERR_INVALID_ARG;
    if (s.page_stride < (uint64_t)s.page_size * s.token_stride) return KVC_ERR_INVALID_ARG;
  }

  const bool mixed = profile->bits_map_k || profile->bits_map_v;
  const uint64_t n_lh = (uint64_t)s.layers * s.kv_heads;
  if (mixed && n_lh > KVC_MAX_MAP_ENTRIES) return KVC_ERR_UNSUPPORTED;
  if (mixed)
    for (int t = 0; t < 2; t++) {
      const uint8_t *m = t ? profile->bits_map_v : profile->bits_map_k;
      if (m)
        for (uint64_t i = 0; i < n_lh; i++)
          if (!valid_bits(m[i])) return KVC_ERR_INVALID_ARG;
    }

  kvc_plan_s *P = new (std::nothrow) kvc_plan_s();
  if (!P) return KVC_ERR_INVALID_ARG;
  P->prof = *profile;
  P->prof.bits_map_k = P->prof.bits_map_v = nullptr;
  P->shape = s;
  P->mixed = mixed;
  // code bytes per unit of width: one (layer, head) block of n_tg groups over
  // tokens, or one head of one token row (groups over channels)
  const uint64_t unit_k = profile->axis_k == KVC_AXIS_OVER_TOKENS ? 16 * ceil_div(s.tokens, profile->group_k) * profile->group_k
                                                                   : 16 * (uint64_t)s.tokens;
  const uint64_t unit_v = profile->axis_v == KVC_AXIS_OVER_TOKENS ? 16 * ceil_div(s.tokens, profile->group_v) * profile->group_v
                                                                   : 16 * (uint64_t)s.tokens;
  uint64_t wtot[2] = {n_lh * profile->bits_k, n_lh * profile->bits_v};
  if (mixed) {
    for (int t = 0; t < 2; t++) {
      const uint8_t *m = t ? profile->bits_map_v : profile->bits_map_k;
      const uint8_t def = t ? profile->bits_v : profile->bits_k;
      P->width[t].assign(n_lh, def);
      if (m) memcpy(P->width[t].data(), m, n_lh);
      P->wt[t] = new (std::nothrow) WidthTable();
      if (!P->wt[t]) {
        kvc_plan_destroy(P);
        return KVC_ERR_INVALID_ARG;
      }
      uint32_t acc = 0;
      for (uint64_t i = 0; i < n_lh; i++) {
        P->wt[t]->wsum[i] = (uint16_t)acc;
        acc += P->width[t][i];
      }
      P->wt[t]->wsum[n_lh] = (uint16_t)acc;
      wtot[t] = acc;
    }
  }
  const uint64_t gk = groups(s, profile->axis_k, profile->group_k), gv = groups(s, profile->axis_v, profile->group_v);
  const uint64_t nsb = (uint64_t)s.layers * s.kv_heads * ceil_div(s.tokens, kSmoothBlock) * s.head_dim;
  P->size[0] = unit_k * wtot[0];
  P->size[1] = gk * 4;
  P->size[2] = unit_v * wtot[1];
  P->size[3] = gv * 4;
  P->size[4] = profile->smooth_keys ? nsb * 2 : 0;
  P->size[5] = profile->smooth_keys ? nsb : 0;
  P->size[6] = profile->token_delta ? nsb * 2 : 0;
  P->size[7] = profile->token_delta ? nsb * 2 : 0;
  uint64_t o = 0;
  for (int i = 0; i < kSections; i++) {
    P->off[i] = o;
    o += align_up(P->size[i], 16);
  }
  P->payload_bytes = o;
  P->header_bytes = (uint32_t)(KVC_HEADER_BYTES + (mixed ? align_up(ceil_div(4 * n_lh, 8), 16) : 0));
  if (profile->n_stages) {
    P->n_chunks = ceil_div(o, profile->chunk_bytes);
    if (P->n_chunks >= (1ull << 31)) {
      kvc_plan_destroy(P);
      return KVC_ERR_UNSUPPORTED;
    }
    P->data_start = align_up(P->header_bytes + 4 * P->n_chunks, 16);
  } else {
    P->n_chunks = 0;
    P->data_start = P->header_bytes;
  }
  P->max_stream_bytes = P->data_start + o;
  P->workspace_bytes = kCtrlBytes + state_bytes(P->n_chunks) + (profile->n_stages ? o : 0);
  P->n_tg_k = ceil_div(s.tokens, profile->group_k);
  P->n_tg_v = ceil_div(s.tokens, profile->group_v);
  P->n_sb = ceil_div(s.tokens, kSmoothBlock);
  if (profile->hadamard) {
    uint64_t state = profile->hadamard_seed;
    for (int j = 0; j < kHeadDim; j++)
      if (splitmix64(state) >> 63) P->sign[j >> 5] |= 1u << (j & 31);
  }
  build_header(P);
  int dev = 0;
  P->sm_count = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&P->sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (P->sm_count <= 0) P->sm_count = 1;
  P->skip_ticket = -1;
  P->poll_limit = kDefaultPollLimit;
  P->codes_in_place = true;
  // the side stream and its events are made here, once, so that encode and decode
  // create nothing; without them the two tensors' kernels run one after the other
  P->side = nullptr;
  if (cudaStreamCreateWithFlags(&P->side, cudaStreamNonBlocking) == cudaSuccess) {
    if (cudaEventCreateWithFlags(&P->ev_fork, cudaEventDisableTiming) != cudaSuccess) {
      cudaStreamDestroy(P->side);
      P->side = nullptr;
    } else if (cudaEventCreateWithFlags(&P->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      cudaEventDestroy(P->ev_fork);
      cudaStreamDestroy(P->side);
      P->side = nullptr;
    }
  } else {
    P->side = nullptr;
    cudaGetLastError();
  }
  *out = P;
  return KVC_OK;
}

static void timing_clear(kvc_plan_s *P) {
  for (auto &r : P->recs) {
    P->pool.push_back(r.start);
    P->pool.push_back(r.stop);
  }
  P->recs.clear();
}

extern "C" void kvc_plan_destroy(kvc_plan_t *plan) {
  if (!plan) return;
  timing_clear(plan);
  for (cudaEvent_t e : plan->pool) cudaEventDestroy(e);
  delete plan->tm[0];
  delete plan->tm[1];
  delete plan->wt[0];
  delete plan->wt[1];
  if (plan->side) {
    cudaEventDestroy(plan->ev_fork);
    cudaEventDestroy(plan->ev_join);
    cudaStreamDestroy(plan->side);
  }
  delete plan;
}

extern "C" size_t kvc_workspace_bytes(const kvc_plan_t *p) { return p ? (size_t)p->workspace_bytes : 0; }
extern "C" size_t kvc_max_stream_bytes(const kvc_plan_t *p) { return p ? (size_t)p->max_stream_bytes : 0; }
extern "C" size_t kvc_payload_bytes(const kvc_plan_t *p) { return p ? (size_t)p->payload_bytes : 0; }
extern "C" uint64_t kvc_num_chunks(const kvc_plan_t *p) { return p ? p->n_chunks : 0; }
extern "C" uint64_t kvc_launch_count(const kvc_plan_t *p) { return p ? p->launches : 0; }
extern "C" size_t kvc_header_bytes(const kvc_plan_t *p) { return p ? (size_t)p->header_bytes : 0; }

extern "C" kvc_status kvc_section(const kvc_plan_t *p, int index, uint64_t *offset, uint64_t *size) {
  if (!p || index < 0 || index >= kSections) return KVC_ERR_INVALID_ARG;
  if (offset) *offset = p->off[index];
  if (size) *size = p->size[index];
  return KVC_OK;
}

// ---------------------------------------------------------------------------
// launch bracketing for kvc_timing_*
// ---------------------------------------------------------------------------
static cudaEvent_t take_event(kvc_plan_s *P) {
  if (!P->pool.empty()) {
    cudaEvent_t e = P->pool.back();
    P->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct Bracket {
  kvc_plan_s *P;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  Bracket(kvc_plan_s *p, cudaStream_t s, bool on = true) : P(p), st(s) {
    if (on && P->timing && (int)P->recs.size() < P->timing_cap) {
      a = take_event(P);
      b = take_event(P);
      if (a && b) cudaEventRecord(a, st);
    }
  }
  void done(const char *name) {
    if (a && b) {
      cudaEventRecord(b, st);
      P->recs.push_back({name, a, b});
    }
  }
};

static kvc_status cuda_status(int rc) { return rc == 0 ? KVC_OK : KVC_ERR_CUDA; }

extern "C" kvc_status kvc_timing_enable(kvc_plan_t *plan, int enable, int capacity) {
  if (!plan) return KVC_ERR_INVALID_ARG;
  timing_clear(plan);
  plan->timing = enable != 0;
  plan->timing_cap = capacity > 0 ? capacity : 4096;
  return KVC_OK;
}

extern "C" int kvc_timing_read(kvc_plan_t *plan, kvc_timing *out, int max) {
  if (!plan || !out) return 0;
  int n = 0;
  for (auto &r : plan->recs) {
    if (n >= max) break;
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      ms = -1.f;
    out[n].kernel = r.name;
    out[n].ms = ms;
    n++;
  }
  return n;
}

extern "C" kvc_status kvc_fuse_value_chunks(kvc_plan_t *plan, int enable) {
  if (!plan) return KVC_ERR_INVALID_ARG;
  plan->fuse_values = enable != 0;
  return KVC_OK;
}

extern "C" kvc_status kvc_decode_codes_in_place(kvc_plan_t *plan, int enable) {
  if (!plan) return KVC_ERR_INVALID_ARG;
  plan->codes_in_place = enable != 0;
  return KVC_OK;
}

extern "C" kvc_status kvc_debug_generic_stages(kvc_plan_t *plan, int enable) {
  if (!plan) return KVC_ERR_INVALID_ARG;
  plan->generic_stages = enable != 0;
  return KVC_OK;
}

extern "C" kvc_status kvc_debug_quotient_check(uint32_t seed, uint32_t rounds, unsigned long long *counts,
                                               void *stream) {
  if (!counts) return KVC_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KVC_ERR_CUDA;
  unsigned long long *d = nullptr;
  if (cudaMalloc(&d, 6 * sizeof(unsigned long long)) != cudaSuccess) return KVC_ERR_CUDA;
  bool ok = cudaMemsetAsync(d, 0, 6 * sizeof(unsigned long long), st) == cudaSuccess;
  for (uint32_t i = 0; ok && i < rounds; i++) ok = kvc::launch_quotient_check(seed + i, d, st) == (int)cudaSuccess;
  ok = ok && kvc::launch_range_check(d, sms, st) == (int)cudaSuccess;
  ok = ok && cudaMemcpyAsync(counts, d, 6 * sizeof(unsigned long long), cudaMemcpyDeviceToHost, st) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  cudaFree(d);
  return ok ? KVC_OK : KVC_ERR_CUDA;
}

extern "C" kvc_status kvc_debug_lookback(kvc_plan_t *plan, int64_t ticket, uint32_t poll_limit) {
  if (!plan) return KVC_ERR_INVALID_ARG;
  plan->skip_ticket = ticket < 0 ? -1 : ticket;
  plan->poll_limit = poll_limit ? poll_limit : kDefaultPollLimit;
  return KVC_OK;
}

// ---------------------------------------------------------------------------
// argument checks shared by the entry points
// ---------------------------------------------------------------------------
static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static kvc_status check_kv(const kvc_plan_s *P, const kvc_kv *kv) {
  if (!kv) return KVC_ERR_INVALID_ARG;
  if (P->shape.layers == 0 || P->shape.tokens == 0) return KVC_OK;
  if (!kv->k_layers || !kv->v_layers) return KVC_ERR_INVALID_ARG;
  for (uint32_t l = 0; l < P->shape.layers; l++)
    if (!kv->k_layers[l] || !kv->v_layers[l] || !aligned16(kv->k_layers[l]) || !aligned16(kv->v_layers[l]))
      return KVC_ERR_INVALID_ARG;
  if (kv->block_table && P->shape.page_size == 0) return KVC_ERR_INVALID_ARG;
  return KVC_OK;
}

static kvc_status check_ws(const kvc_plan_s *P, const void *ws, size_t bytes) {
  if (!ws || !aligned16(ws)) return KVC_ERR_INVALID_ARG;
  if (bytes < P->workspace_bytes) return KVC_ERR_CAPACITY;
  return KVC_OK;
}

static uint32_t *ctrl_of(void *ws) { return static_cast<uint32_t *>(ws); }
static uint64_t *state_of(void *ws) { return reinterpret_cast<uint64_t *>(static_cast<uint8_t *>(ws) + kCtrlBytes); }
static uint8_t *ws_payload(const kvc_plan_s *P, void *ws) {
  return static_cast<uint8_t *>(ws) + kCtrlBytes + state_bytes(P->n_chunks);
}

static void fill_geom(const kvc_plan_s *P, const kvc_kv *kv, KvGeom &g) {
  const kvc_shape &s = P->shape;
  g.L = s.layers;
  g.T = s.tokens;
  g.H = s.kv_heads;
  g.bf16 = s.dtype == KVC_BF16;
  g.token_stride = s.token_stride;
  g.page_stride = s.page_stride;
  g.block_table = kv->block_table;
  g.page_shift = 0;
  if (s.page_size)
    while ((1u << g.page_shift) < s.page_size) g.page_shift++;
  g.page_mask = s.page_size ? s.page_size - 1 : 0;
  g.num_pages = s.num_pages;
  g.pad_ = 0;
}

// ---------------------------------------------------------------------------
// tensor maps for the key-tile encoder (cuTensorMapEncodeTiled through the
// runtime's driver entry point; no link-time dependency on the driver library)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Maps of tensor `t`'s layers (see TmaMaps), re-encoded only for layers whose
// pointer changed since the last call.  nullptr when TMA cannot be used: too many
// layers, no encoder, or a layout the maps do not describe.
static const TmaMaps *tensor_maps(kvc_plan_s *P, int t, void *const *layers) {
  const kvc_shape &sh = P->shape;
  if (sh.layers > (uint32_t)kTmaMaxLayers || sh.token_stride % 16 != 0) return nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return nullptr;
  if (!P->tm[t]) {
    P->tm[t] = new (std::nothrow) TmaMaps();
    if (!P->tm[t]) return nullptr;
    for (int l = 0; l < kTmaMaxLayers; l++) P->tm_ptr[t][l] = nullptr;
  }
  for (uint32_t l = 0; l < sh.layers; l++) {
    if (P->tm_ptr[t][l] == layers[l]) continue;
    const cuuint64_t dim[2] = {(cuuint64_t)sh.kv_heads * sh.head_dim, (cuuint64_t)sh.tokens};
    const cuuint64_t stride[1] = {(cuuint64_t)sh.token_stride};
    const cuuint32_t box[2] = {64, 128}, estride[2] = {1, 1};
    const CUresult r = enc(&P->tm[t]->map[l], sh.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void *>(layers[l]), dim, stride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      P->tm_ptr[t][l] = nullptr;
      return nullptr;
    }
    P->tm_ptr[t][l] = layers[l];
  }
  return P->tm[t];
}

// The chunks [lo, hi) whose codes of tensor t (0 = K, 1 = V) kvc_decode's
// dequantizer reads in place: the whole chunks of the tensor's code section, where
// its decoder reads a unit's codes through one lookup -- the key-tile decoder
// (groups over tokens, every (layer, head) holding whole 128-token tiles, a tile of
// 2048 BITS bytes dividing the chunk) or the value-row decoder (groups over channels
// without smoothing, 16 rows of 16 BITS bytes dividing the chunk) -- with a uniform
// width of 2, 4 or 8 bits, chunks of a power of two bytes and the section starting
// on a chunk boundary.
static bool in_place_range(const kvc_plan_s *P, int t, uint32_t *lo, uint32_t *hi) {
  *lo = *hi = 0;
  if (!P->codes_in_place || P->prof.n_stages == 0 || P->mixed || P->n_chunks == 0) return false;
  const uint32_t bits = t ? P->prof.bits_v : P->prof.bits_k, G = t ? P->prof.group_v : P->prof.group_k;
  const uint32_t axis = t ? P->prof.axis_v : P->prof.axis_k;
  const bool smooth = t == 0 && P->prof.smooth_keys;
  const uint64_t cb = P->prof.chunk_bytes, off = P->off[t ? 2 : 0], size = P->size[t ? 2 : 0];
  if ((bits != 2 && bits != 4 && bits != 8) || cb == 0 || (cb & (cb - 1)) || off % cb) return false;
  if (axis == KVC_AXIS_OVER_TOKENS) {
    const uint64_t n_tg = t ? P->n_tg_v : P->n_tg_k;
    if ((n_tg * G) % kSmoothBlock || cb % (2048ull * bits)) return false;
  } else if (smooth || cb % (256ull * bits)) {
    return false;
  }
  const uint64_t l = off / cb, h = (off + size) / cb;
  if (h <= l || h > P->n_chunks) return false;
  *lo = (uint32_t)l;
  *hi = (uint32_t)h;
  return true;
}

// One quantize / dequantize launch per tensor.  Decoding runs K on the caller's
// stream and V beside it on the plan's side stream (forked after the work already
// queued on the caller's stream, joined back before anything queued after): the
// two reconstruction kernels share the SMs, each with its full persistent grid,
// and the pair is also timed as one launch.  Measured on one GB300, the overlap
// helps the decoders on every workload (llama8b dequantize 0.186 -> 0.181 ms) but
// not the encoders: with both grids the 70B encode got 3% slower, and with one
// CTA of each per SM the shorter kernel's SMs idle once it is done (70B and
// 8B@32K encodes 23-27% slower), so the encoders run one after the other.
// The launch parameters of one tensor (0 = K, 1 = V) over payload Q; returns the
// key tiles' tensor maps when the encoder can load them by TMA.
static const TmaMaps *fill_quant(kvc_plan_s *P, const kvc_kv *kv, uint8_t *Q, void *ws, int tensor, bool enc,
                                 bool check_corrupt, bool in_place, QuantParams &q) {
  memset(&q, 0, sizeof q);
  fill_geom(P, kv, q.g);
  void *const *src = tensor ? kv->v_layers : kv->k_layers;
  for (uint32_t l = 0; l < P->shape.layers; l++) q.layers[l] = src[l];
  q.bits = tensor ? P->prof.bits_v : P->prof.bits_k;
  q.group = tensor ? P->prof.group_v : P->prof.group_k;
  q.axis = tensor ? P->prof.axis_v : P->prof.axis_k;
  q.smooth = tensor == 0 && P->prof.smooth_keys;
  q.n_tg = (uint32_t)(tensor ? P->n_tg_v : P->n_tg_k);
  q.n_sb = (uint32_t)P->n_sb;
  q.hadamard = P->prof.hadamard;
  memcpy(q.sign, P->sign, sizeof q.sign);
  q.codes = Q + P->off[tensor ? 2 : 0];
  q.meta = Q + P->off[tensor ? 3 : 1];
  q.mu = Q + P->off[4];
  q.ex = reinterpret_cast<int8_t *>(Q + P->off[5]);
  q.status = ctrl_of(ws) + kCtrlFlags;
  q.check_corrupt = check_corrupt;
  q.delta = P->prof.token_delta;
  q.anchors = Q + P->off[tensor ? 7 : 6];
  q.mixed = P->mixed;
  uint32_t lo, hi;
  if (in_place && !enc && in_place_range(P, tensor, &lo, &hi)) {
    q.src_of = state_of(ws);
    q.codes_off = P->off[tensor ? 2 : 0];
    q.chunk_shift = (uint32_t)__builtin_ctz(P->prof.chunk_bytes);
    q.in_lo = lo;
    q.in_hi = hi;
  }
  const TmaMaps *maps = nullptr;
  if (enc && q.axis == KVC_AXIS_OVER_TOKENS && !kv->block_table) maps = tensor_maps(P, tensor, src);
  q.tma = maps != nullptr;
  return maps;
}

static kvc_status run_quant(kvc_plan_s *P, const kvc_kv *kv, uint8_t *Q, void *ws, bool enc, bool check_corrupt,
                            cudaStream_t st, bool in_place = false) {
  if (P->shape.layers == 0 || P->shape.tokens == 0) return KVC_OK;
  const bool fork = P->side != nullptr && !enc;
  const int cap = 0;
  Bracket pair(P, st, fork);  // an overlapped pair is also timed as one unit
  if (fork) {
    if (cudaEventRecord(P->ev_fork, st) != cudaSuccess || cudaStreamWaitEvent(P->side, P->ev_fork, 0) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  kvc_status status = KVC_OK;
  for (int tensor = 0; tensor < 2 && status == KVC_OK; tensor++) {
    cudaStream_t s = fork && tensor == 1 ? P->side : st;
    QuantParams q;
    const TmaMaps *maps = fill_quant(P, kv, Q, ws, tensor, enc, check_corrupt, in_place, q);
    const WidthTable *wt = P->mixed ? P->wt[tensor] : nullptr;
    Bracket br(P, s);
    const char *name = "";
    const int rc = enc ? launch_quantize(q, maps, wt, P->sm_count, cap, s, &P->launches, &name)
                       : launch_dequantize(q, wt, P->sm_count, cap, s, &P->launches, &name);
    br.done(name);
    if (rc) status = KVC_ERR_CUDA;
  }
  // joined even after a failed launch, so that nothing queued on the caller's
  // stream later can overtake work already queued on the side stream
  if (fork) {
    if (cudaEventRecord(P->ev_join, P->side) != cudaSuccess || cudaStreamWaitEvent(st, P->ev_join, 0) != cudaSuccess)
      status = KVC_ERR_CUDA;
  }
  pair.done(enc ? "kvc_quantize_kv" : "kvc_dequantize_kv");
  return status;
}

static kvc_status run_prologue(kvc_plan_s *P, void *ws, bool zero_flags, bool zero_state, uint8_t *stream,
                               uint64_t *d_stream_bytes, uint8_t *payload, cudaStream_t st) {
  PrologueParams pp;
  memset(&pp, 0, sizeof pp);
  pp.ctrl = ctrl_of(ws);
  pp.state = state_of(ws);
  pp.n_state = zero_state ? P->n_chunks : 0;
  pp.zero_flags = zero_flags;
  pp.write_header = stream != nullptr;
  pp.stream = stream;
  pp.header_bytes = P->header_bytes;
  memcpy(pp.header, P->header, P->header_bytes);
  if (stream) {
    if (P->prof.n_stages == 0 || P->n_chunks == 0) pp.static_size = P->data_start + (P->prof.n_stages ? 0 : P->payload_bytes);
    pp.d_stream_bytes = d_stream_bytes;
    if (P->prof.n_stages) {
      pp.gap_off = P->header_bytes + 4 * P->n_chunks;
      pp.gap_len = (uint32_t)(P->data_start - pp.gap_off);
    }
  }
  pp.payload = payload;
  if (payload)
    for (int i = 0; i < kSections; i++) {
      pp.pad_off[i] = P->off[i] + P->size[i];
      pp.pad_len[i] = (uint32_t)(align_up(P->size[i], 16) - P->size[i]);
    }
  Bracket br(P, st);
  const int rc = launch_prologue(pp, st);
  br.done("kvc_prologue");
  P->launches++;
  return cuda_status(rc);
}

static void fill_lossless(kvc_plan_s *P, LosslessParams &lp, void *ws) {
  memset(&lp, 0, sizeof lp);
  lp.payload_bytes = P->payload_bytes;
  lp.data_start = P->data_start;
  lp.chunk_bytes = P->prof.chunk_bytes;
  lp.n_chunks = (uint32_t)P->n_chunks;
  lp.n_stages = P->prof.n_stages;
  for (uint32_t s = 0; s < P->prof.n_stages; s++) {
    lp.kind[s] = P->prof.stages[s].kind;
    lp.param[s] = P->prof.stages[s].param;
  }
  lp.state = state_of(ws);
  lp.ctrl = ctrl_of(ws);
  lp.skip_ticket = P->skip_ticket;
  lp.poll_limit = P->poll_limit;
  lp.generic_only = P->generic_stages ? 1u : 0u;
  lp.header_bytes = P->header_bytes;
  lp.first_chunk = 0;
  lp.last_chunk = lp.n_chunks;
  lp.ticket_word = kCtrlTicket;
  memcpy(lp.header, P->header, P->header_bytes);
}

static kvc_status lossless_encode_impl(kvc_plan_s *P, const uint8_t *Q, void *d_stream, size_t cap, void *ws,
                                       uint64_t *d_stream_bytes, cudaStream_t st) {
  if (P->prof.n_stages == 0) {
    if (P->payload_bytes &&
        cudaMemcpyAsync(static_cast<uint8_t *>(d_stream) + P->header_bytes, Q, P->payload_bytes,
                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return KVC_ERR_CUDA;
    return KVC_OK;
  }
  LosslessParams lp;
  fill_lossless(P, lp, ws);
  lp.payload = Q;
  lp.stream = static_cast<uint8_t *>(d_stream);
  lp.stream_cap = cap;
  lp.d_stream_bytes = d_stream_bytes;
  Bracket br(P, st);
  const int rc = launch_lossless_encode(lp, P->sm_count, st);
  br.done(lossless_encode_is_fast(lp) ? "kvc_lossless_enc_fast" : "kvc_lossless_enc");
  if (P->n_chunks) P->launches++;
  return cuda_status(rc);
}

extern "C" kvc_status kvc_quantize(kvc_plan_t *plan, const kvc_kv *in, void *d_payload, void *d_workspace,
                                   size_t workspace_bytes, kvc_stream_t stream) {
  if (!plan || !d_payload || !aligned16(d_payload)) return KVC_ERR_INVALID_ARG;
  kvc_status s = check_kv(plan, in);
  if (s != KVC_OK) return s;
  if ((s = check_ws(plan, d_workspace, workspace_bytes)) != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *Q = static_cast<uint8_t *>(d_payload);
  if ((s = run_prologue(plan, d_workspace, true, false, nullptr, nullptr, Q, st)) != KVC_OK) return s;
  return run_quant(plan, in, Q, d_workspace, true, false, st);
}

extern "C" kvc_status kvc_lossless_encode(kvc_plan_t *plan, const void *d_payload, void *d_stream, size_t stream_cap,
                                          void *d_workspace, size_t workspace_bytes, uint64_t *d_stream_bytes,
                                          kvc_stream_t stream) {
  if (!plan || !d_stream || !aligned16(d_stream) || (!d_payload && plan->payload_bytes) ||
      (d_payload && !aligned16(d_payload)))
    return KVC_ERR_INVALID_ARG;
  if (stream_cap < plan->max_stream_bytes) return KVC_ERR_CAPACITY;
  kvc_status s = check_ws(plan, d_workspace, workspace_bytes);
  if (s != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = run_prologue(plan, d_workspace, true, true, static_cast<uint8_t *>(d_stream), d_stream_bytes, nullptr, st)) !=
      KVC_OK)
    return s;
  return lossless_encode_impl(plan, static_cast<const uint8_t *>(d_payload), d_stream, stream_cap, d_workspace,
                              d_stream_bytes, st);
}

// Encode with the value-code chunks written by the value encoder itself (see
// kvc_fused.cu): the key encoder; the lossless stages over the chunks before the
// value codes; the value encoder with the section's whole chunks; the lossless
// stages over the rest.  Every chunk takes its place through the one look-back, in
// chunk order across the three launches, so the stream is the one the unfused
// path writes.
static kvc_status encode_split(kvc_plan_s *P, const kvc_kv *in, uint8_t *Q, void *ws, const QuantParams &qv,
                               LosslessParams lp, uint32_t c0, uint32_t nfull, cudaStream_t st) {
  {
    QuantParams qk;
    const TmaMaps *maps = fill_quant(P, in, Q, ws, 0, true, false, false, qk);
    Bracket br(P, st);
    const char *name = "";
    const int rc = launch_quantize(qk, maps, nullptr, P->sm_count, 0, st, &P->launches, &name);
    br.done(name);
    if (rc) return KVC_ERR_CUDA;
  }
  lp.first_chunk = 0;
  lp.last_chunk = c0;
  lp.ticket_word = kCtrlTicket;
  if (c0) {
    Bracket br(P, st);
    const int rc = launch_lossless_encode(lp, P->sm_count, st);
    br.done("kvc_lossless_enc_fast_head");
    P->launches++;
    if (rc) return KVC_ERR_CUDA;
  }
  lp.ticket_word = kCtrlTicket + 1;
  {
    Bracket br(P, st);
    const int rc = launch_v_lossless(qv, lp, c0, nfull, P->sm_count, st);
    br.done("kvc_enc_rows_lc");
    P->launches++;
    if (rc) return KVC_ERR_CUDA;
  }
  lp.first_chunk = c0 + nfull;
  lp.last_chunk = lp.n_chunks;
  lp.ticket_word = kCtrlTicket + 2;
  Bracket br(P, st);
  const int rc = launch_lossless_encode(lp, P->sm_count, st);
  br.done("kvc_lossless_enc_fast_tail");
  P->launches++;
  return cuda_status(rc);
}

extern "C" kvc_status kvc_encode(kvc_plan_t *plan, const kvc_kv *in, void *d_stream, size_t stream_cap,
                                 void *d_workspace, size_t workspace_bytes, uint64_t *d_stream_bytes,
                                 kvc_stream_t stream) {
  if (!plan || !d_stream || !aligned16(d_stream)) return KVC_ERR_INVALID_ARG;
  kvc_status s = check_kv(plan, in);
  if (s != KVC_OK) return s;
  if (stream_cap < plan->max_stream_bytes) return KVC_ERR_CAPACITY;
  if ((s = check_ws(plan, d_workspace, workspace_bytes)) != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *out = static_cast<uint8_t *>(d_stream);
  // without lossless stages the payload is written in place after the header
  uint8_t *Q = plan->prof.n_stages ? ws_payload(plan, d_workspace) : out + plan->header_bytes;
  if ((s = run_prologue(plan, d_workspace, true, true, out, d_stream_bytes, Q, st)) != KVC_OK) return s;
  if (plan->fuse_values && plan->prof.n_stages && plan->shape.layers && plan->shape.tokens && !plan->mixed) {
    QuantParams qv;
    fill_quant(plan, in, Q, d_workspace, 1, true, false, false, qv);
    LosslessParams lp;
    fill_lossless(plan, lp, d_workspace);
    lp.payload = Q;
    lp.stream = out;
    lp.stream_cap = stream_cap;
    lp.d_stream_bytes = d_stream_bytes;
    uint32_t c0 = 0, nfull = 0;
    if (v_lossless_fusable(qv, lp, plan->off[2], plan->size[2], &c0, &nfull))
      return encode_split(plan, in, Q, d_workspace, qv, lp, c0, nfull, st);
  }
  if ((s = run_quant(plan, in, Q, d_workspace, true, false, st)) != KVC_OK) return s;
  if (plan->prof.n_stages == 0) return KVC_OK;
  return lossless_encode_impl(plan, Q, d_stream, stream_cap, d_workspace, d_stream_bytes, st);
}

static kvc_status lossless_decode_impl(kvc_plan_s *P, const void *d_stream, size_t stream_bytes, uint8_t *Q, void *ws,
                                       bool copy_plain, cudaStream_t st, bool in_place = false) {
  LosslessParams lp;
  fill_lossless(P, lp, ws);
  bool some = false;
  for (int t = 0; t < 2 && in_place; t++) some |= in_place_range(P, t, &lp.inplace_lo[t], &lp.inplace_hi[t]);
  lp.stream = static_cast<uint8_t *>(const_cast<void *>(d_stream));
  lp.stream_cap = stream_bytes;
  lp.out_payload = Q;
  lp.fused_offsets = lossless_decode_fusable(lp, P->sm_count) ? 1u : 0u;
  if (lp.fused_offsets) {  // the decoder checks the stream itself: only the status word is reset first
    if (cudaMemsetAsync(lp.ctrl + kCtrlFlags, 0, sizeof(uint32_t), st) != cudaSuccess) return KVC_ERR_CUDA;
  } else {
    Bracket br(P, st);
    const int rc = launch_decode_prepare(lp, st);
    br.done("kvc_decode_prepare");
    P->launches += lp.n_chunks ? 2 : 1;  // the sums (header checks) and the offsets
    if (rc) return KVC_ERR_CUDA;
  }
  if (P->prof.n_stages == 0) {
    // the payload sits after the header; copy only when the caller wants it elsewhere
    if (copy_plain && P->payload_bytes && stream_bytes >= P->header_bytes + P->payload_bytes &&
        cudaMemcpyAsync(Q, static_cast<const uint8_t *>(d_stream) + P->header_bytes, P->payload_bytes,
                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return KVC_ERR_CUDA;
    return KVC_OK;
  }
  Bracket br(P, st);
  const int rc = launch_lossless_decode(lp, P->sm_count, st);
  br.done(lossless_decode_is_fast(lp) ? (some ? "kvc_lossless_dec_fast_inplace" : "kvc_lossless_dec_fast")
                                      : (some ? "kvc_lossless_dec_inplace" : "kvc_lossless_dec"));
  if (P->n_chunks) P->launches++;
  return cuda_status(rc);
}

extern "C" kvc_status kvc_lossless_decode(kvc_plan_t *plan, const void *d_stream, size_t stream_bytes, void *d_payload,
                                          void *d_workspace, size_t workspace_bytes, kvc_stream_t stream) {
  if (!plan || !d_stream || !aligned16(d_stream) || (!d_payload && plan->payload_bytes) ||
      (d_payload && !aligned16(d_payload)))
    return KVC_ERR_INVALID_ARG;
  kvc_status s = check_ws(plan, d_workspace, workspace_bytes);
  if (s != KVC_OK) return s;
  return lossless_decode_impl(plan, d_stream, stream_bytes, static_cast<uint8_t *>(d_payload), d_workspace, true,
                              (cudaStream_t)stream);
}

extern "C" kvc_status kvc_dequantize(kvc_plan_t *plan, const void *d_payload, const kvc_kv *out, void *d_workspace,
                                     size_t workspace_bytes, kvc_stream_t stream) {
  if (!plan || (!d_payload && plan->payload_bytes) || (d_payload && !aligned16(d_payload))) return KVC_ERR_INVALID_ARG;
  kvc_status s = check_kv(plan, out);
  if (s != KVC_OK) return s;
  if ((s = check_ws(plan, d_workspace, workspace_bytes)) != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = run_prologue(plan, d_workspace, true, false, nullptr, nullptr, nullptr, st)) != KVC_OK) return s;
  return run_quant(plan, out, static_cast<uint8_t *>(const_cast<void *>(d_payload)), d_workspace, false, false, st);
}

extern "C" kvc_status kvc_decode(kvc_plan_t *plan, const void *d_stream, size_t stream_bytes, const kvc_kv *out,
                                 void *d_workspace, size_t workspace_bytes, kvc_stream_t stream) {
  if (!plan || !d_stream || !aligned16(d_stream)) return KVC_ERR_INVALID_ARG;
  kvc_status s = check_kv(plan, out);
  if (s != KVC_OK) return s;
  if ((s = check_ws(plan, d_workspace, workspace_bytes)) != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *Q = plan->prof.n_stages ? ws_payload(plan, d_workspace)
                                   : static_cast<uint8_t *>(const_cast<void *>(d_stream)) + plan->header_bytes;
  if ((s = lossless_decode_impl(plan, d_stream, stream_bytes, Q, d_workspace, false, st, true)) != KVC_OK) return s;
  return run_quant(plan, out, Q, d_workspace, false, true, st, true);
}

extern "C" kvc_status kvc_query(const void *d_workspace, kvc_stream_t stream, uint64_t *host_stream_bytes,
                                uint32_t *host_flags) {
  if (!d_workspace) return KVC_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
  uint64_t ctrl[2] = {0, 0};
  if (cudaMemcpy(ctrl, d_workspace, sizeof ctrl, cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ERR_CUDA;
  const uint32_t flags = (uint32_t)(ctrl[0] & 0xffffffffu);
  if (host_flags) *host_flags = flags;
  if (host_stream_bytes) *host_stream_bytes = ctrl[1];
  if (flags & KVC_FLAG_CORRUPT) return KVC_ERR_CORRUPT;
  if (flags & KVC_FLAG_CAPACITY) return KVC_ERR_CAPACITY;
  if (flags & KVC_FLAG_TIMEOUT) return KVC_ERR_TIMEOUT;
  if (flags & KVC_FLAG_BAD_PAGE) return KVC_ERR_INVALID_ARG;
  if (flags & KVC_FLAG_NONFINITE) return KVC_ERR_NONFINITE;
  if (flags & KVC_FLAG_RANGE) return KVC_ERR_RANGE;
  return KVC_OK;
}

extern "C" const char *kvc_status_str(kvc_status s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported";
    case KVC_ERR_CAPACITY: return "capacity too small";
    case KVC_ERR_CORRUPT: return "corrupt stream";
    case KVC_ERR_RANGE: return "fp16 metadata overflow (saturated)";
    case KVC_ERR_NONFINITE: return "non-finite input";
    case KVC_ERR_TIMEOUT: return "device wait timed out";
    case KVC_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

// ---------------------------------------------------------------------------
// Allocation-free lossless encode (kvc_lossless_encode_noalloc).
//
// The lossless encoder's scratch (256-byte control block + one 64-bit look-back
// word per chunk) lives in this file-scope device array instead of a caller
// workspace.  Every GPU that loads the library holds the array until the process
// exits.  In host code `g_noalloc_scratch` only names a host-side stand-in, so
// its device address is looked up with cudaGetSymbolAddress once per device
// context: the cache is keyed to the context's unique id (cuCtxGetId), so after a
// cudaDeviceReset (which destroys the primary context; the runtime makes a new
// one with a new id on the next call) the address is looked up again instead of
// pointing into the destroyed context.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);

static std::mutex g_noalloc_mutex;
struct NoallocSlot {
  unsigned long long ctx_id;  // id of the context the address belongs to (0 = none yet)
  void *addr;
};
static NoallocSlot g_noalloc_slot[256];  // per device ordinal

// Unique id of the calling thread's current context (0 when there is none or the
// driver entry points are missing).
static unsigned long long current_ctx_id() {
  static std::once_flag once;
  static PfnCtxGetCurrent get_current = nullptr;
  static PfnCtxGetId get_id = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PfnCtxGetId>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

static kvc_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
  if (dev < 0 || dev >= 256) return KVC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocSlot &slot = g_noalloc_slot[dev];
  unsigned long long id = current_ctx_id();
  if (slot.addr && id != 0 && slot.ctx_id == id) {
    *out = slot.addr;
    return KVC_OK;
  }
  // first call in this context: the lookup also makes the runtime set up the
  // device's primary context if it has none yet
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KVC_ERR_CUDA;
  if (id == 0) id = current_ctx_id();
  slot.ctx_id = id;    // 0 (no id available): looked up again on every call
  slot.addr = id ? p : nullptr;
  *out = p;
  return KVC_OK;
}

extern "C" kvc_status kvc_lossless_encode_noalloc(kvc_plan_t *plan, const void *d_payload, void *d_stream,
                                                  size_t stream_cap, uint64_t *d_stream_bytes, uint32_t *d_status,
                                                  kvc_stream_t stream) {
  if (!plan || !d_stream || !aligned16(d_stream) || !d_stream_bytes || (!d_payload && plan->payload_bytes) ||
      (d_payload && !aligned16(d_payload)))
    return KVC_ERR_INVALID_ARG;
  if (stream_cap < plan->max_stream_bytes) return KVC_ERR_CAPACITY;
  if ((uint64_t)kCtrlBytes + 8 * plan->n_chunks > KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_CAPACITY;
  void *ws = nullptr;
  kvc_status s = noalloc_scratch(&ws);
  if (s != KVC_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if ((s = run_prologue(plan, ws, true, true, static_cast<uint8_t *>(d_stream), d_stream_bytes, nullptr, st)) != KVC_OK)
    return s;
  if ((s = lossless_encode_impl(plan, static_cast<const uint8_t *>(d_payload), d_stream, stream_cap, ws,
                                d_stream_bytes, st)) != KVC_OK)
    return s;
  if (d_status && cudaMemcpyAsync(d_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}
