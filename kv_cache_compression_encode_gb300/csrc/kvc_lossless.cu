// kvc_lossless.cu -- chunked lossless stage pipeline over the quantized payload.
//
// "Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
// Serving", §4.2: composable GPU stages (tuple reordering, bit shuffling,
// zero-oriented encoding; pipeline TUPL8_1 -> BIT_8 -> RZE_2) over the device
// buffer of the fused frontend, producing a GPU-resident bitstream of which only
// a size scalar goes back to the host.
//
// One CTA encodes one chunk at a time entirely in shared memory: the stages run
// as block-wide passes, RZE's compaction offsets come from block scans of
// per-thread counts, and the chunk's place in the stream comes from a decoupled
// look-back over per-chunk words (chunks are taken in ticket order, so a CTA only
// ever waits for CTAs that are already running; every wait is bounded).
//
// Stream: header (64 bytes, plus the width map of a mixed-width profile) |
// u32 table[n_chunks] (bit 31 = stored raw, bits 0..30 = stored size) | chunk i
// at data_start + sum_{j<i} align16(size_j), zero padded.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc_internal.h"
#include "kvc_lossless_dev.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// Stages (block-wide; `in` and `out` are distinct shared buffers; n bytes).
// Every stage keeps the tail past the last whole tuple / word as is.
// ---------------------------------------------------------------------------
// TUPL_k: m = n/k tuples; column j (byte j of every tuple) is written contiguously.
template <int NT = LT>
__device__ void tupl_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t k) {
  const uint32_t m = n / k;
  if ((m & 3u) == 0) {
    // four tuples per thread: read 4k bytes, write k words of 4 bytes
    const uint32_t nq = m / 4;
    for (uint32_t idx = threadIdx.x; idx < nq; idx += NT) {
      uint32_t src[8];
      const uint32_t *in32 = reinterpret_cast<const uint32_t *>(in) + idx * k;
      for (uint32_t u = 0; u < k; u++) src[u] = in32[u];
      for (uint32_t j = 0; j < k; j++) {
        uint32_t word = 0;
#pragma unroll
        for (uint32_t q = 0; q < 4; q++) {
          const uint32_t b = q * k + j;  // byte index inside the 4k-byte block
          word |= ((src[b >> 2] >> (8 * (b & 3))) & 0xffu) << (8 * q);
        }
        reinterpret_cast<uint32_t *>(out + j * m)[idx] = word;
      }
    }
  } else {
    for (uint32_t j = 0; j < k; j++)
      for (uint32_t i = threadIdx.x; i < m; i += NT) out[j * m + i] = in[i * k + j];
  }
  for (uint32_t o = m * k + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

template <int NT = LT>
__device__ void tupl_decode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t k) {
  const uint32_t m = n / k;
  for (uint32_t i = threadIdx.x; i < m; i += NT) {
    if (k == 8) {
      uint64_t v = 0;
#pragma unroll
      for (uint32_t j = 0; j < 8; j++) v |= (uint64_t)in[j * m + i] << (8 * j);
      *reinterpret_cast<uint64_t *>(out + 8 * i) = v;
    } else if (k == 4) {
      uint32_t v = 0;
#pragma unroll
      for (uint32_t j = 0; j < 4; j++) v |= (uint32_t)in[j * m + i] << (8 * j);
      *reinterpret_cast<uint32_t *>(out + 4 * i) = v;
    } else {
      *reinterpret_cast<uint16_t *>(out + 2 * i) = (uint16_t)(in[i] | (in[m + i] << 8));
    }
  }
  for (uint32_t o = m * k + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

// BIT_8: plane p (n8/8 bytes) collects bit p of every byte, byte i -> bit i%8 of byte i/8.
template <int NT = LT>
__device__ void bit_encode(const uint8_t *in, uint8_t *out, uint32_t n) {
  const uint32_t n8 = n & ~7u, P = n8 / 8;
  if ((P & 3u) == 0) {
    for (uint32_t idx = threadIdx.x; idx < P / 4; idx += NT) {
      const uint4 a = reinterpret_cast<const uint4 *>(in)[2 * idx];
      const uint4 b = reinterpret_cast<const uint4 *>(in)[2 * idx + 1];
      const uint64_t x0 = transpose8(((uint64_t)a.y << 32) | a.x), x1 = transpose8(((uint64_t)a.w << 32) | a.z);
      const uint64_t x2 = transpose8(((uint64_t)b.y << 32) | b.x), x3 = transpose8(((uint64_t)b.w << 32) | b.z);
#pragma unroll
      for (int p = 0; p < 8; p++) {
        const uint32_t word = (uint32_t)((x0 >> (8 * p)) & 0xff) | (uint32_t)((x1 >> (8 * p)) & 0xff) << 8 |
                              (uint32_t)((x2 >> (8 * p)) & 0xff) << 16 | (uint32_t)((x3 >> (8 * p)) & 0xff) << 24;
        reinterpret_cast<uint32_t *>(out + p * P)[idx] = word;
      }
    }
  } else {
    for (uint32_t b = threadIdx.x; b < P; b += NT) {
      const uint64_t x = transpose8(*reinterpret_cast<const uint64_t *>(in + 8 * b));
#pragma unroll
      for (int p = 0; p < 8; p++) out[p * P + b] = (uint8_t)(x >> (8 * p));
    }
  }
  for (uint32_t o = n8 + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

template <int NT = LT>
__device__ void bit_decode(const uint8_t *in, uint8_t *out, uint32_t n) {
  const uint32_t n8 = n & ~7u, P = n8 / 8;
  for (uint32_t b = threadIdx.x; b < P; b += NT) {
    uint64_t x = 0;
#pragma unroll
    for (int p = 0; p < 8; p++) x |= (uint64_t)in[p * P + b] << (8 * p);
    *reinterpret_cast<uint64_t *>(out + 8 * b) = transpose8(x);
  }
  for (uint32_t o = n8 + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

// DELTA_w: word i -> word i - word (i-1) mod 2^(8w); word 0 kept.
template <int NT = LT>
__device__ void delta_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w) {
  const uint32_t m = n / w;
  const uint32_t mask = w == 4 ? 0xffffffffu : ((1u << (8 * w)) - 1u);
  for (uint32_t i = threadIdx.x; i < m; i += NT) {
    const uint32_t cur = ld_word(in + i * w, w), prev = i ? ld_word(in + (i - 1) * w, w) : 0u;
    st_word(out + i * w, w, (cur - prev) & mask);
  }
  for (uint32_t o = m * w + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

// Inverse: running sum mod 2^(8w); each thread sums a contiguous run, then a block scan.
template <int NT = LT>
__device__ void delta_decode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w, uint32_t *tmp) {
  const uint32_t m = n / w;
  const uint32_t mask = w == 4 ? 0xffffffffu : ((1u << (8 * w)) - 1u);
  const uint32_t S = (m + NT - 1) / NT;
  const uint32_t i0 = min(m, threadIdx.x * S), i1 = min(m, i0 + S);
  uint32_t sum = 0;
  for (uint32_t i = i0; i < i1; i++) sum += ld_word(in + i * w, w);
  uint32_t total;
  uint32_t acc = block_excl_scan<uint32_t, NT>(sum, tmp, total);
  for (uint32_t i = i0; i < i1; i++) {
    acc += ld_word(in + i * w, w);
    st_word(out + i * w, w, acc & mask);
  }
  for (uint32_t o = m * w + threadIdx.x; o < n; o += NT) out[o] = in[o];
  bsync<NT>();
}

// RZE_w: B = bitmap of nonzero words, B2 = bitmap of nonzero bytes of B; output
// B2 | nonzero B bytes | nonzero words | tail.  Returns the encoded size; when it
// is >= n nothing is written (the chunk will be stored raw).
template <int NT = LT>
__device__ uint32_t rze_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w, uint8_t *Bs,
                               uint32_t *tmp) {
  const uint32_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8, tail = n - m * w;
  const uint32_t S = (nb + NT - 1) / NT;
  const uint32_t j0 = min(nb, threadIdx.x * S), j1 = min(nb, j0 + S);
  uint32_t cw = 0, cb = 0;
  for (uint32_t j = j0; j < j1; j++) {
    uint32_t byte = 0;
    for (uint32_t q = 0; q < 8; q++) {
      const uint32_t i = 8 * j + q;
      if (i < m && ld_word(in + i * w, w) != 0u) byte |= 1u << q;
    }
    Bs[j] = (uint8_t)byte;
    cw += __popc(byte);
    cb += byte != 0;
  }
  uint32_t totW, totB;
  const uint32_t exW = block_excl_scan<uint32_t, NT>(cw, tmp, totW);
  const uint32_t exB = block_excl_scan<uint32_t, NT>(cb, tmp, totB);
  const uint32_t size = nb2 + totB + w * totW + tail;
  if (size >= n) return size;
  for (uint32_t b2 = threadIdx.x; b2 < nb2; b2 += NT) {
    uint32_t v = 0;
    for (uint32_t q = 0; q < 8; q++) {
      const uint32_t j = 8 * b2 + q;
      if (j < nb && Bs[j]) v |= 1u << q;
    }
    out[b2] = (uint8_t)v;
  }
  uint32_t oB = nb2 + exB, oW = nb2 + totB + w * exW;
  for (uint32_t j = j0; j < j1; j++) {
    const uint32_t byte = Bs[j];
    if (!byte) continue;
    out[oB++] = (uint8_t)byte;
    for (uint32_t q = 0; q < 8; q++)
      if ((byte >> q) & 1u) {
        const uint8_t *src = in + (8 * j + q) * w;
        for (uint32_t u = 0; u < w; u++) out[oW + u] = src[u];
        oW += w;
      }
  }
  const uint32_t t0 = nb2 + totB + w * totW;
  for (uint32_t o = threadIdx.x; o < tail; o += NT) out[t0 + o] = in[m * w + o];
  bsync<NT>();
  return size;
}

// Inverse of RZE for `size` stored bytes that must expand to exactly n bytes.
// Returns false (uniformly across the block) when the bytes are inconsistent.
template <int NT = LT>
__device__ bool rze_decode(const uint8_t *in, uint32_t size, uint8_t *out, uint32_t n, uint32_t w, uint8_t *Bs,
                           uint32_t *tmp) {
  const uint32_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8, tail = n - m * w;
  if (size < nb2) return false;
  // B bytes listed by B2 (only its first nb bits count)
  const uint32_t S2 = (nb2 + NT - 1) / NT;
  const uint32_t b0 = min(nb2, threadIdx.x * S2), b1 = min(nb2, b0 + S2);
  uint32_t cb = 0;
  for (uint32_t b = b0; b < b1; b++) {
    uint32_t v = in[b];
    if (8 * b + 8 > nb) v &= (1u << (nb - 8 * b)) - 1u;
    cb += __popc(v);
  }
  uint32_t totB;
  uint32_t rB = block_excl_scan<uint32_t, NT>(cb, tmp, totB);
  if (nb2 + totB > size) return false;
  for (uint32_t b = b0; b < b1; b++) {
    const uint32_t v = in[b];
    for (uint32_t q = 0; q < 8; q++) {
      const uint32_t j = 8 * b + q;
      if (j >= nb) break;
      Bs[j] = ((v >> q) & 1u) ? in[nb2 + rB++] : (uint8_t)0;
    }
  }
  bsync<NT>();
  // words listed by B (only its first m bits count)
  const uint32_t S = (nb + NT - 1) / NT;
  const uint32_t j0 = min(nb, threadIdx.x * S), j1 = min(nb, j0 + S);
  uint32_t cw = 0;
  for (uint32_t j = j0; j < j1; j++) {
    uint32_t v = Bs[j];
    if (8 * j + 8 > m) v &= (1u << (m - 8 * j)) - 1u;
    cw += __popc(v);
  }
  uint32_t totW;
  uint32_t rW = block_excl_scan<uint32_t, NT>(cw, tmp, totW);
  if (nb2 + totB + w * totW + tail != size) return false;
  const uint8_t *words = in + nb2 + totB;
  for (uint32_t j = j0; j < j1; j++) {
    const uint32_t v = Bs[j];
    for (uint32_t q = 0; q < 8; q++) {
      const uint32_t i = 8 * j + q;
      if (i >= m) break;
      if ((v >> q) & 1u) {
        for (uint32_t u = 0; u < w; u++) out[i * w + u] = words[rW * w + u];
        rW++;
      } else {
        for (uint32_t u = 0; u < w; u++) out[i * w + u] = 0;
      }
    }
  }
  const uint8_t *tl = words + w * totW;
  for (uint32_t o = threadIdx.x; o < tail; o += NT) out[m * w + o] = tl[o];
  bsync<NT>();
  return true;
}

// ---------------------------------------------------------------------------
// Prologue: reset workspace words, zero section padding, write the header.
// ---------------------------------------------------------------------------
__global__ void kvc_prologue(const PrologueParams P) {
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
  if (tid < kCtrlBytes / 4) {
    const bool keep = (tid == (uint32_t)kCtrlFlags) && !P.zero_flags;
    if (!keep) P.ctrl[tid] = 0u;
  }
  for (uint64_t i = tid; i < P.n_state; i += nt) P.state[i] = 0ull;
  if (P.write_header)
    for (uint32_t i = tid; i < P.header_bytes; i += nt) P.stream[i] = P.header[i];
  if (P.write_header && tid < P.gap_len) P.stream[P.gap_off + tid] = 0;
  if (P.payload && tid < kSections * 16) {
    const int s = tid / 16, b = tid % 16;
    if ((uint32_t)b < P.pad_len[s]) P.payload[P.pad_off[s] + b] = 0;
  }
  if (P.static_size && tid == 0) {
    reinterpret_cast<uint64_t *>(P.ctrl)[kCtrlStreamBytes] = P.static_size;
    if (P.d_stream_bytes) *P.d_stream_bytes = P.static_size;
  }
}

// ---------------------------------------------------------------------------
// Encode: one chunk per CTA iteration, in ticket order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(LT) kvc_lossless_enc(const LosslessParams P) {
  extern __shared__ uint4 smem_u4[];
  uint8_t *bufA = reinterpret_cast<uint8_t *>(smem_u4);
  uint8_t *bufB = bufA + P.chunk_bytes + 64;
  uint8_t *Bs = bufB + P.chunk_bytes + 64;
  uint32_t *tmp = reinterpret_cast<uint32_t *>(Bs + 8192);
  __shared__ uint32_t s_ticket;
  __shared__ uint64_t s_excl;
  uint32_t *ctrl = P.ctrl;
  const bool has_rze = P.n_stages > 0 && P.kind[P.n_stages - 1] == KVC_ST_RZE;

  for (;;) {
    if (threadIdx.x == 0) s_ticket = P.first_chunk + atomicAdd(ctrl + P.ticket_word, 1u);
    __syncthreads();
    const uint32_t ticket = s_ticket;
    if (ticket >= P.last_chunk) break;
    const uint64_t off = (uint64_t)ticket * P.chunk_bytes;
    const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
    const uint4 *src = reinterpret_cast<const uint4 *>(P.payload + off);

    uint32_t size = n;
    bool raw = true;
    uint8_t *res = bufA;
    if (has_rze) {  // without an RZE stage every stage keeps the length: the chunk is stored raw
      for (uint32_t i = threadIdx.x; i < n / 16; i += LT) reinterpret_cast<uint4 *>(bufA)[i] = __ldg(src + i);
      __syncthreads();
      uint8_t *cur = bufA, *nxt = bufB;
      for (uint32_t s = 0; s + 1 < P.n_stages; s++) {
        const uint32_t k = P.kind[s], prm = P.param[s];
        if (k == KVC_ST_TUPL) tupl_encode(cur, nxt, n, prm);
        else if (k == KVC_ST_BIT) bit_encode(cur, nxt, n);
        else delta_encode(cur, nxt, n, prm);
        uint8_t *t = cur; cur = nxt; nxt = t;
      }
      const uint32_t rs = rze_encode(cur, nxt, n, P.param[P.n_stages - 1], Bs, tmp);
      if (rs < n) {
        size = rs;
        raw = false;
        res = nxt;
        if (threadIdx.x < align16u(size) - size) res[size + threadIdx.x] = 0;
      }
    }
    const uint32_t asz = align16u(size);

    // decoupled look-back (warp 0): publish this chunk's aggregate, then add predecessors' until an inclusive prefix
    if (threadIdx.x < 32) {
      const uint64_t excl = lookback_warp(P, ticket, asz);
      if (threadIdx.x == 0) {
        s_excl = excl;
        const uint64_t dst = P.data_start + excl;
        if (dst + asz > P.stream_cap) atomicOr(ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CAPACITY);
        reinterpret_cast<uint32_t *>(P.stream + P.header_bytes)[ticket] = size | (raw ? 0x80000000u : 0u);
        if (ticket == P.n_chunks - 1) {
          const uint64_t total = dst + asz;
          reinterpret_cast<uint64_t *>(ctrl)[kCtrlStreamBytes] = total;
          if (P.d_stream_bytes) *P.d_stream_bytes = total;
        }
      }
    }
    __syncthreads();
    const uint64_t dst = P.data_start + s_excl;
    if (dst + asz <= P.stream_cap) {
      uint4 *out = reinterpret_cast<uint4 *>(P.stream + dst);
      if (raw) {
        for (uint32_t i = threadIdx.x; i < asz / 16; i += LT) out[i] = __ldg(src + i);
      } else {
        for (uint32_t i = threadIdx.x; i < asz / 16; i += LT) out[i] = reinterpret_cast<const uint4 *>(res)[i];
      }
    }
    __syncthreads();
  }
}

// ===========================================================================
// Fast encoder for the stage lists TUPL_8 [BIT_8] [DELTA_1] RZE_w (w = 1 or 2)
// and chunk sizes that are multiples of 4 KiB up to 16 KiB.  A CTA holds eight
// worker warps, two publisher warps and one loader warp, around a ring of
// kRing chunk slots.
//  * Loader: takes the CTA's next ticket (at most kAhead chunks ahead of the
//    workers), announces it to the publishers and fetches the chunk into its
//    slot with one bulk copy, completing on the slot's mbarrier.
//  * Workers: with BIT_8 the chunk's encoded size is first computed from the
//    chunk as loaded (fast_size_bit8) and published for the look-back at once;
//    an incompressible chunk is then done.  Otherwise TUPL_8 (and BIT_8) run
//    as one register transform per 8-tuple block (a 4x4 byte transpose gathers
//    byte j of the 8 tuples, an 8x8 bit transpose makes the 8 bit-plane bytes)
//    into a scratch buffer, stored swizzled so that the next pass reads it
//    without bank conflicts.  DELTA_1 and RZE run as one register pass: a
//    thread owns 64 contiguous bytes, takes the word bitmaps of the byte
//    differences, and one block scan of its counts gives its output offsets;
//    the encoded chunk is written over its slot.  The slot is then handed to a
//    publisher.
//  * Publishers (chunks k = p, p + 2, ... for warp p): each walks back over the
//    chunk's predecessors (32 at a time) as soon as its ticket is announced,
//    while the chunk is still being encoded.  When the slot is full it
//    publishes the inclusive prefix, writes the chunk-table entry, copies the
//    chunk to the stream with one bulk copy and hands the slot back once the
//    copy has read it.  Workers never wait on other CTAs, only on slots of
//    their own ring.
// Tickets, loaded, started, full and free slots pass between the warps through
// mbarriers; every wait is bounded and sets KVC_FLAG_TIMEOUT when it runs out.  A
// chunk whose length is not a multiple of 4 KiB (only the last one can be) runs
// the generic stage functions on the worker threads.
// ===========================================================================
__global__ void __launch_bounds__(FW, kFastCtasPerSm) kvc_lossless_enc_fast(const LosslessParams P, const FastSpec F) {
  extern __shared__ uint4 smem_u4[];
  const uint32_t cb = P.chunk_bytes, slot_bytes = cb + 64;
  uint8_t *const A = reinterpret_cast<uint8_t *>(smem_u4);  // transform output (swizzled)
  uint8_t *const ring = A + slot_bytes;                      // slot s at ring + s * slot_bytes
  uint16_t *Bs = reinterpret_cast<uint16_t *>(ring + kRing * slot_bytes);                       // generic-path bitmap
  uint32_t *wsum = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(Bs) + cb / 8 + 64);  // scan words
  // Chunk k of this CTA lives in slot k % kRing: loaded there, encoded over itself
  // when it compresses, copied out from there either way.  tick[j]: the ticket of
  // chunk k (k % 2kRing == j) is known, a value >= n_chunks meaning "no more
  // chunks"; loaded[s]: the chunk has arrived (or the stop is known);
  // started[s]: the workers have begun it; full[s]: the slot holds the chunk's
  // stored bytes; empty[s]: the publisher is done with the slot.
  __shared__ __align__(8) uint64_t s_tick[2 * kRing], s_loaded[kRing], s_started[kRing], s_full[kRing], s_empty[kRing];
  __shared__ uint32_t s_ticket[2 * kRing], s_word[kRing], s_from_payload[kRing];
  const uint32_t nc = P.n_chunks;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; s++) {
      mbar_init(&s_loaded[s], 1);
      mbar_init(&s_started[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    for (int j = 0; j < 2 * kRing; j++) mbar_init(&s_tick[j], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (threadIdx.x >= FT + 32 * kPubWarps) {  // ---- loader warp
    if ((threadIdx.x & 31) != 0) return;
    uint32_t *ticket_ctr = P.ctrl + P.ticket_word;
    uint32_t k = 0, first = 0;  // loads [first, k) may still be pending at the end
    for (;; k++) {
      const uint32_t s = k % kRing, j = k % (2 * kRing);
      // a ticket is taken only kAhead chunks ahead of the workers (a ticket held
      // while idle would hold up every later chunk's look-back), and the slot's
      // previous chunk must have been copied out
      if ((k >= kAhead && !mbar_wait(&s_started[(k - kAhead) % kRing], ((k - kAhead) / kRing) & 1u)) ||
          (k >= kRing && !mbar_wait(&s_empty[s], (k / kRing - 1) & 1u))) {
        atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
        break;
      }
      const uint32_t t = P.first_chunk + atomicAdd(ticket_ctr, 1u);
      if (t >= P.last_chunk) {  // every publisher warp and the workers learn of the stop
        for (uint32_t q = 0; q < (uint32_t)kPubWarps; q++) {
          const uint32_t jq = (k + q) % (2 * kRing);
          s_ticket[jq] = nc;
          mbar_arrive(&s_tick[jq]);
        }
        mbar_arrive(&s_loaded[s]);
        first = 1;  // chunk k - kRing's slot has been reused by the stop
        break;
      }
      s_ticket[j] = t;
      mbar_arrive(&s_tick[j]);
      const uint64_t off = (uint64_t)t * cb;
      const uint32_t n = (uint32_t)min((uint64_t)cb, P.payload_bytes - off);
      mbar_arrive_tx(&s_loaded[s], n);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_addr(ring + s * slot_bytes)),
          "l"(P.payload + off), "r"(n), "r"(smem_addr(&s_loaded[s]))
          : "memory");
    }
    // no load may still be landing when the CTA ends (only reachable with every
    // load consumed, or after a timeout)
    for (uint32_t q = k + first > kRing ? k + first - kRing : 0; q < k; q++)
      mbar_wait(&s_loaded[q % kRing], (q / kRing) & 1u);
    return;
  }

  if (threadIdx.x >= FT && threadIdx.x < FT + 32 * kPubWarps) {  // ---- publisher warps: chunks k = p, p + kPubWarps, ...
    const int lane = threadIdx.x & 31;
    for (uint32_t k = (threadIdx.x - FT) >> 5;; k += kPubWarps) {
      const uint32_t j = k % (2 * kRing), s = k % kRing;
      if (!mbar_wait(&s_tick[j], (k / (2 * kRing)) & 1u)) {
        if (lane == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
        break;
      }
      const uint32_t t = s_ticket[j];
      if (t >= nc) break;
      // the predecessors' sizes do not depend on this chunk: walk back while
      // the workers are still encoding it
      const uint64_t excl = t ? lookback_excl(P, t) : 0ull;
      if (!mbar_wait(&s_full[s], (k / kRing) & 1u)) {
        if (lane == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
        break;
      }
      const uint32_t word = s_word[s];
      const uint32_t asz = align16u(word & 0x7fffffffu);
      const uint64_t dst = P.data_start + excl;
      if (lane == 0) {
        if (t && (int64_t)t != P.skip_ticket) st_word64(P.state + t, kFlagIncl | (excl + asz));
        if (dst + asz > P.stream_cap) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CAPACITY);
        reinterpret_cast<uint32_t *>(P.stream + P.header_bytes)[t] = word;
        if (t == nc - 1) {
          const uint64_t total = dst + asz;
          reinterpret_cast<uint64_t *>(P.ctrl)[kCtrlStreamBytes] = total;
          if (P.d_stream_bytes) *P.d_stream_bytes = total;
        }
      }
      if (dst + asz <= P.stream_cap) {
        if (s_from_payload[s]) {  // a raw chunk whose slot the generic stages overwrote
          uint4 *o = reinterpret_cast<uint4 *>(P.stream + dst);
          const uint4 *g = reinterpret_cast<const uint4 *>(P.payload + (uint64_t)t * cb);
          for (uint32_t i = lane; i < asz / 16; i += 32) o[i] = __ldg(g + i);
        } else if (lane == 0) {
          // one bulk copy from the slot; the slot is free once it has been read
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(P.stream + dst),
                       "r"(smem_addr(ring + s * slot_bytes)), "r"(asz)
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    return;
  }

  // ---- workers
  for (uint32_t k = 0;; k++) {
    const uint32_t s = k % kRing;
    uint8_t *const S = ring + s * slot_bytes;
    if (!mbar_wait(&s_loaded[s], (k / kRing) & 1u)) {
      if (threadIdx.x == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
      break;
    }
    const uint32_t t = s_ticket[k % (2 * kRing)];
    if (t >= nc) break;
    if (threadIdx.x == 0) mbar_arrive(&s_started[s]);

    const uint64_t off = (uint64_t)t * cb;
    const uint32_t n = (uint32_t)min((uint64_t)cb, P.payload_bytes - off);
    uint32_t size = n;
    bool raw, from_payload = false;
    if (fast_len(n)) {
      // with BIT_8 the size is known from the chunk as loaded; an incompressible
      // chunk then skips the transform altogether
      uint32_t es = 0;
      if (F.bit8) {
        if (F.rze_w == 2) es = F.delta1 ? fast_size_bit8<2, true>(S, n, wsum) : fast_size_bit8<2, false>(S, n, wsum);
        else es = F.delta1 ? fast_size_bit8<1, true>(S, n, wsum) : fast_size_bit8<1, false>(S, n, wsum);
        if (threadIdx.x == 0) publish_size(P, t, align16u(es < n ? es : n));
      }
      if (F.bit8 && es >= n) {
        raw = true;  // the slot holds the chunk as loaded
      } else {
        if (F.bit8) fast_transform<true>(S, A, n);
        else fast_transform<false>(S, A, n);
        const bool pub = !F.bit8;  // with BIT_8 the size is already out
        uint32_t rs;
        if (F.rze_w == 2)
          rs = F.delta1 ? fast_delta_rze<2, true>(A, S, n, wsum, P, t, pub) : fast_delta_rze<2, false>(A, S, n, wsum, P, t, pub);
        else
          rs = F.delta1 ? fast_delta_rze<1, true>(A, S, n, wsum, P, t, pub) : fast_delta_rze<1, false>(A, S, n, wsum, P, t, pub);
        raw = rs >= n;  // stored raw: the slot still holds the chunk as loaded
        if (!raw) size = rs;
        if (F.bit8 && rs != es && threadIdx.x == 0)  // the two size computations must agree
          atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
      }
    } else {
      uint8_t *cur_b = S, *nxt_b = A;
      for (uint32_t st = 0; st + 1 < P.n_stages; st++) {
        const uint32_t kind = P.kind[st], prm = P.param[st];
        if (kind == KVC_ST_TUPL) tupl_encode<FT>(cur_b, nxt_b, n, prm);
        else if (kind == KVC_ST_BIT) bit_encode<FT>(cur_b, nxt_b, n);
        else delta_encode<FT>(cur_b, nxt_b, n, prm);
        uint8_t *tmpb = cur_b; cur_b = nxt_b; nxt_b = tmpb;
      }
      const uint32_t rs = rze_encode<FT>(cur_b, nxt_b, n, P.param[P.n_stages - 1], reinterpret_cast<uint8_t *>(Bs), wsum);
      raw = rs >= n;
      if (!raw) {
        size = rs;
        if (nxt_b != S) {
          for (uint32_t i = threadIdx.x; i < align16u(rs) / 16; i += FT)
            reinterpret_cast<uint4 *>(S)[i] = reinterpret_cast<const uint4 *>(nxt_b)[i];
        }
      } else {
        from_payload = P.n_stages > 1;  // the stages wrote over the slot
      }
      if (threadIdx.x == 0) publish_size(P, t, align16u(size));
    }
    const uint32_t asz = align16u(size);
    if (!raw && threadIdx.x < asz - size) S[size + threadIdx.x] = 0;
    if (threadIdx.x == 0) {
      s_word[s] = size | (raw ? 0x80000000u : 0u);
      s_from_payload[s] = from_payload;
    }
    // the publisher reads the slot through the bulk-copy (async) proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bsync<FT>();
    if (threadIdx.x == 0) mbar_arrive(&s_full[s]);
  }
}

// ---------------------------------------------------------------------------
// Fast decode of one compressed chunk for the stage lists TUPL_8 [BIT_8]
// [DELTA_1] RZE_w, n a multiple of 4 KiB: the inverse of the fast encoder's
// register passes.  `in` (shared) holds the chunk's `size` stored bytes; thread
// t < n/64 owns stream bytes 64t..64t+63:
//  * RZE: its level-2 bits, one block scan for its place in the list of nonzero
//    level-1 bytes, its level-1 bytes, a second scan for its place in the list of
//    nonzero words, its words;
//  * DELTA_1: byte-wise inclusive prefix sums inside its words (SWAR adds that
//    keep carries inside each byte), a block scan of the per-thread sums;
//  * the bytes go to `buf` (shared) swizzled like the encoder's transform output;
//    thread beta then gathers the 64 bit-plane bytes of block beta, undoes the
//    8x8 bit transposes and the 4x4 byte transposes (both are involutions) and
//    stores the 64-byte block to `dst`.
// The consistency checks are the generic decoder's: the level-1 list must fit in
// the stored bytes and the sizes must add up exactly; otherwise false (uniform).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t badd4(uint32_t a, uint32_t b) {  // byte-wise a + b mod 256
  return ((a & 0x7f7f7f7fu) + (b & 0x7f7f7f7fu)) ^ ((a ^ b) & 0x80808080u);
}

template <int W, bool DELTA, bool BIT8>
__device__ bool fast_decode_chunk(const uint8_t *in, uint32_t size, uint32_t n, uint8_t *buf, uint8_t *dst,
                                  uint32_t *tmp) {
  const uint32_t nthr = n / 64, nb = n / (8 * W), nb2 = nb / 8;
  const uint32_t t = threadIdx.x;
  const bool active = t < nthr;
  if (size < nb2) return false;
  uint32_t l2 = 0;  // this thread's level-2 bits (W = 2: a nibble, W = 1: a byte)
  if (active) l2 = W == 2 ? (in[t >> 1] >> (4 * (t & 1))) & 0xfu : in[t];
  uint32_t totB;
  uint32_t r = block_excl_scan<uint32_t, LT>(__popc(l2), tmp, totB);
  if (nb2 + totB > size) return false;
  uint32_t blo = 0, bhi = 0;  // element bits: W = 2 -> 32 in blo; W = 1 -> 64 in (bhi:blo)
  if (active) {
    const uint8_t *L1 = in + nb2;
#pragma unroll
    for (int k = 0; k < 8 / W; k++)
      if ((l2 >> k) & 1u) {
        const uint32_t b = L1[r++];
        if (k < 4) blo |= b << (8 * k);
        else bhi |= b << (8 * (k - 4));
      }
  }
  uint32_t totW;
  uint32_t e = block_excl_scan<uint32_t, LT>(__popc(blo) + __popc(bhi), tmp, totW);
  if (nb2 + totB + W * totW != size) return false;
  uint32_t x[16];
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = 0u;
  if (active && (blo | bhi)) {
    // this thread's nonzero elements are contiguous from byte nb2 + totB + W e of
    // the chunk: they are taken from a bit window refilled with aligned 32-bit
    // words (the reads stay inside the chunk buffer, which has 64 spare bytes)
    const uint32_t *Wd = reinterpret_cast<const uint32_t *>(in);
    const uint32_t a0 = nb2 + totB + W * e;
    uint32_t wi = a0 >> 2;
    uint64_t win = Wd[wi++] >> (8 * (a0 & 3u));
    uint32_t have = 32 - 8 * (a0 & 3u);
#pragma unroll
    for (int i = 0; i < 16; i++) {
      if (W == 2) {
#pragma unroll
        for (int hh = 0; hh < 2; hh++)
          if ((blo >> (2 * i + hh)) & 1u) {
            if (have < 16) {
              win |= (uint64_t)Wd[wi++] << have;
              have += 32;
            }
            x[i] |= ((uint32_t)win & 0xffffu) << (16 * hh);
            win >>= 16;
            have -= 16;
          }
      } else {
        const uint32_t bits = i < 8 ? (blo >> (4 * i)) : (bhi >> (4 * (i - 8)));
#pragma unroll
        for (int b = 0; b < 4; b++)
          if ((bits >> b) & 1u) {
            if (have < 8) {
              win |= (uint64_t)Wd[wi++] << have;
              have += 32;
            }
            x[i] |= ((uint32_t)win & 0xffu) << (8 * b);
            win >>= 8;
            have -= 8;
          }
      }
    }
  }
  if (DELTA) {
    uint32_t run = 0;
#pragma unroll
    for (int i = 0; i < 16; i++) {
      uint32_t p = badd4(x[i], x[i] << 8);
      p = badd4(p, p << 16);
      p = badd4(p, run * 0x01010101u);
      x[i] = p;
      run = p >> 24;
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan<uint32_t, LT>(active ? run : 0u, tmp, tot) & 0xffu;
#pragma unroll
    for (int i = 0; i < 16; i++) x[i] = badd4(x[i], ex * 0x01010101u);
  }
  if (active) {
    uint4 *d = reinterpret_cast<uint4 *>(buf) + 4 * t;
    const uint32_t rot = (t >> 1) & 3u;
#pragma unroll
    for (int k = 0; k < 4; k++) d[(k + rot) & 3u] = make_uint4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
  }
  bsync<LT>();
  if (active) {
    const uint32_t beta = t, m = n / 8, m8 = n / 64;
    uint32_t L0[4], L1[4], H0[4], H1[4];
    const uint32_t off8 = 64 * (beta >> 3) + 16 * (((beta >> 1) + (beta >> 4)) & 3u) + 8 * (beta & 1u);
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint32_t lo, hi;
      if (BIT8) {
        const uint8_t *ob = buf + swzb(j * m8 + beta);
        lo = (uint32_t)ob[0] | ((uint32_t)ob[m] << 8) | ((uint32_t)ob[2 * m] << 16) | ((uint32_t)ob[3 * m] << 24);
        hi = (uint32_t)ob[4 * m] | ((uint32_t)ob[5 * m] << 8) | ((uint32_t)ob[6 * m] << 16) | ((uint32_t)ob[7 * m] << 24);
        bits8x8(lo, hi);
      } else {
        const uint2 v = *reinterpret_cast<const uint2 *>(buf + j * m + off8);
        lo = v.x;
        hi = v.y;
      }
      if (j < 4) {
        L0[j] = lo;
        L1[j] = hi;
      } else {
        H0[j - 4] = lo;
        H1[j - 4] = hi;
      }
    }
    uint32_t a[4], b[4], c[4], d[4];
    byte_t4x4(L0[0], L0[1], L0[2], L0[3], a);  // a[i]: bytes 0..3 of tuple i
    byte_t4x4(H0[0], H0[1], H0[2], H0[3], b);  // b[i]: bytes 4..7 of tuple i
    byte_t4x4(L1[0], L1[1], L1[2], L1[3], c);  // tuples 4..7
    byte_t4x4(H1[0], H1[1], H1[2], H1[3], d);
    uint4 *o = reinterpret_cast<uint4 *>(dst + 64 * beta);
    o[0] = make_uint4(a[0], b[0], a[1], b[1]);
    o[1] = make_uint4(a[2], b[2], a[3], b[3]);
    o[2] = make_uint4(c[0], d[0], c[1], d[1]);
    o[3] = make_uint4(c[2], d[2], c[3], d[3]);
  }
  bsync<LT>();
  return true;
}

// ---------------------------------------------------------------------------
// Decode, step 1 (one CTA): check the header and the chunk table, compute the
// chunk offsets.  Any inconsistency sets KVC_FLAG_CORRUPT.
// ---------------------------------------------------------------------------
constexpr int PT = 1024;
constexpr uint32_t kPrepSeg = 4 * PT;  // table entries per CTA of the prepare kernels: one 16-byte load a thread
static_assert(kPrepSeg == kDecodeSumSeg, "one partial sum per prepare CTA");

// Block-wide exclusive scan (PT threads) of 64-bit values; tmp holds PT/32 + 1
// words and ends with the block total in tmp[PT/32].
__device__ __forceinline__ unsigned long long prep_scan(unsigned long long v, unsigned long long *tmp) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= (uint32_t)o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= (uint32_t)o) w += y;
    }
    tmp[lane] = w;
    if (lane == 31) tmp[PT / 32] = w;
  }
  __syncthreads();
  return x - v + (warp ? tmp[warp - 1] : 0ull);
}

// Decode, step 1 (tables too large for the decoder to scan in every CTA), first
// kernel: CTA b checks table entries [b kPrepSeg, (b + 1) kPrepSeg) against their
// chunks' lengths (a stored chunk holds exactly its length, a compressed one less)
// and writes the sum of their aligned sizes to sums[b]; CTA 0 also checks the
// header and that the stream reaches the chunk data (without stages: the whole
// payload after the header).  A failed check sets CORRUPT
// (the caller has cleared the status word).  The sums follow the chunks' words in
// the workspace (state[n_chunks + b]).
__global__ void __launch_bounds__(PT) kvc_decode_sums(const LosslessParams P) {
  __shared__ unsigned long long tmp[PT / 32 + 1];
  __shared__ int s_bad;
  const uint32_t tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const uint64_t stream_bytes = P.stream_cap;
  if (blockIdx.x == 0) {
    if (stream_bytes < P.header_bytes) {
      if (tid == 0) s_bad = 1;
    } else {
      if (tid < P.header_bytes / 4 &&
          reinterpret_cast<const uint32_t *>(P.stream)[tid] != reinterpret_cast<const uint32_t *>(P.header)[tid])
        atomicOr(&s_bad, 1);
      // without stages the payload follows the header as it is
      if (tid == 0 && (P.n_stages == 0 ? stream_bytes < P.header_bytes + P.payload_bytes : stream_bytes < P.data_start))
        s_bad = 1;
    }
  }
  const uint32_t nc = P.n_chunks, i = blockIdx.x * kPrepSeg + 4 * tid;
  unsigned long long sum = 0;
  int bad = 0;
  if (i < nc && stream_bytes >= P.data_start) {
    // the table is 16-byte aligned and padded to data_start
    const uint4 q = *reinterpret_cast<const uint4 *>(P.stream + P.header_bytes + 4 * (size_t)i);
    const uint32_t e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      if (i + k < nc) {
        const uint32_t e = e4[k], sz = e & 0x7fffffffu;
        const uint64_t off = (uint64_t)(i + k) * P.chunk_bytes;
        const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
        if (e >> 31) bad |= sz != n;
        else bad |= sz >= n;
        sum += align16u(sz);
      }
    }
  }
  if (bad) atomicOr(&s_bad, 1);
  prep_scan(sum, tmp);
  if (tid == 0) {
    if (nc) P.state[nc + blockIdx.x] = tmp[PT / 32];
    if (s_bad) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
  }
}

// Second kernel: CTA b adds the sums of the CTAs before it to data_start, scans
// its entries' aligned sizes and writes every chunk's byte offset in the stream
// to state[]; the last CTA checks that the chunks end inside the stream.
__global__ void __launch_bounds__(PT) kvc_decode_offsets(const LosslessParams P) {
  __shared__ unsigned long long tmp[PT / 32 + 1];
  __shared__ unsigned long long s_base;
  const uint32_t tid = threadIdx.x, lane = tid & 31;
  const uint64_t *sums = P.state + P.n_chunks;
  if (tid < 32) {  // sum of sums[0 .. blockIdx.x - 1] by the first warp
    unsigned long long x = 0;
    for (uint32_t j = lane; j < blockIdx.x; j += 32) x += sums[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) s_base = P.data_start + x;
  }
  const uint32_t nc = P.n_chunks, i = blockIdx.x * kPrepSeg + 4 * tid;
  uint32_t e4[4] = {0u, 0u, 0u, 0u};
  unsigned long long sum = 0;
  if (i < nc && P.stream_cap >= P.data_start) {
    const uint4 q = *reinterpret_cast<const uint4 *>(P.stream + P.header_bytes + 4 * (size_t)i);
    e4[0] = q.x; e4[1] = q.y; e4[2] = q.z; e4[3] = q.w;
#pragma unroll
    for (int k = 0; k < 4; k++)
      if (i + k < nc) sum += align16u(e4[k] & 0x7fffffffu);
  }
  unsigned long long pos = prep_scan(sum, tmp);  // also publishes s_base (barriers inside)
  pos += s_base;
  if (i < nc) {
    unsigned long long o4[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      o4[k] = pos;
      if (i + k < nc) pos += align16u(e4[k] & 0x7fffffffu);
    }
    if (i + 4 <= nc) {  // offsets of four chunks: two 16-byte stores
      reinterpret_cast<ulonglong2 *>(P.state + i)[0] = make_ulonglong2(o4[0], o4[1]);
      reinterpret_cast<ulonglong2 *>(P.state + i)[1] = make_ulonglong2(o4[2], o4[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; k++)
        if (i + k < nc) P.state[i + k] = o4[k];
    }
  }
  if (blockIdx.x == gridDim.x - 1 && tid == 0 && s_base + tmp[PT / 32] > P.stream_cap)
    atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
}

// ---------------------------------------------------------------------------
// Decode, step 1 inside the decoder (tables of up to kFusedMaxChunks chunks):
// every CTA checks the header and the whole table exactly as kvc_decode_sums
// does and takes the offsets of its own chunks (c = blockIdx.x + k gridDim.x) from
// one block scan; all CTAs reach the same verdict, CTA 0 reports a corrupt stream.
// ---------------------------------------------------------------------------
constexpr uint32_t kFusedMaxChunks = 32 * LT;  // 32 table words per thread
constexpr uint32_t kFusedMaxOwn = 64;           // chunks per CTA

__device__ bool decode_offsets(const LosslessParams &P, unsigned long long *tmp, unsigned long long *s_off,
                               int *s_bad) {
  const uint32_t tid = threadIdx.x, nc = P.n_chunks;
  const uint32_t *table = reinterpret_cast<const uint32_t *>(P.stream + P.header_bytes);
  if (tid == 0) *s_bad = 0;
  __syncthreads();
  for (uint32_t w = tid; w < P.header_bytes / 4; w += LT)
    if (reinterpret_cast<const uint32_t *>(P.stream)[w] != reinterpret_cast<const uint32_t *>(P.header)[w])
      atomicOr(s_bad, 1);
  // thread tid takes entries [S tid, S tid + S), S a multiple of 4 (16-byte reads;
  // the table is 16-byte aligned and padded to data_start)
  const uint32_t S = ((nc + LT - 1) / LT + 3) & ~3u;
  const uint32_t i0 = min(nc, tid * S), i1 = min(nc, i0 + S);
  unsigned long long sum = 0;
  int bad = 0;
  for (uint32_t i = i0; i < i1; i += 4) {
    const uint4 q = *reinterpret_cast<const uint4 *>(table + i);
    const uint32_t e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) {
      if (i + k < i1) {
        const uint32_t e = e4[k], sz = e & 0x7fffffffu;
        const uint64_t off = (uint64_t)(i + k) * P.chunk_bytes;
        const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
        if (e >> 31) bad |= sz != n;  // a stored chunk holds exactly its length, a compressed one less
        else bad |= sz >= n;
        sum += align16u(sz);
      }
    }
  }
  if (bad) atomicOr(s_bad, 1);
  unsigned long long total;
  unsigned long long run = P.data_start + block_excl_scan<unsigned long long>(sum, tmp, total);
  if (tid == 0 && P.data_start + total > P.stream_cap) atomicOr(s_bad, 1);
  // this CTA's chunks in the thread's range: the first at or after i0, then every gridDim.x
  const uint32_t b = blockIdx.x, grid = gridDim.x;
  uint32_t own = i0 <= b ? b : b + (i0 - b + grid - 1) / grid * grid;
  for (uint32_t i = i0; i < i1; i += 4) {
    const uint4 q = *reinterpret_cast<const uint4 *>(table + i);
    const uint32_t e4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (uint32_t k = 0; k < 4; k++) {
      if (i + k < i1) {
        if (i + k == own) {
          s_off[(own - b) / grid] = run;
          own += grid;
        }
        run += align16u(e4[k] & 0x7fffffffu);
      }
    }
  }
  __syncthreads();
  if (*s_bad) {
    if (b == 0 && tid == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
    return false;
  }
  return true;
}

__device__ __forceinline__ bool in_place_chunk(const LosslessParams &P, uint32_t c) {
  return (c >= P.inplace_lo[0] && c < P.inplace_hi[0]) || (c >= P.inplace_lo[1] && c < P.inplace_hi[1]);
}

// ---------------------------------------------------------------------------
// Decode, step 2: one chunk per CTA iteration back into the payload.  A chunk
// whose codes the dequantizers read in place (inplace_lo/hi) gets the address of
// its bytes in state[c]; stored raw, it is left in the stream.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(LT, 3) kvc_lossless_dec(const LosslessParams P, const FastSpec F) {
  extern __shared__ uint4 smem_u4[];
  __shared__ unsigned long long s_off[kFusedMaxOwn];
  __shared__ int s_bad;
  if (!P.fused_offsets) {
    // A stream the prepare step found corrupt is skipped.  The whole CTA takes one
    // decision from one read: other CTAs of this launch may set CORRUPT while it
    // starts, and a CTA split between warps that return and warps that go on
    // would leave the named barriers of the stage functions waiting.
    if (threadIdx.x == 0) s_bad = (*(volatile uint32_t *)(P.ctrl + kCtrlFlags) & KVC_FLAG_CORRUPT) != 0;
    __syncthreads();
    if (s_bad) return;
  }
  uint8_t *bufA = reinterpret_cast<uint8_t *>(smem_u4);
  uint8_t *bufB = bufA + P.chunk_bytes + 64;
  uint8_t *Bs = bufB + P.chunk_bytes + 64;
  uint32_t *tmp = reinterpret_cast<uint32_t *>(Bs + 8192);
  if (P.fused_offsets && !decode_offsets(P, reinterpret_cast<unsigned long long *>(tmp), s_off, &s_bad)) return;
  const uint32_t *table = reinterpret_cast<const uint32_t *>(P.stream + P.header_bytes);
  const uint32_t last = P.n_stages - 1;
  const bool has_rze = P.kind[last] == KVC_ST_RZE;

  // this CTA's chunks c = blockIdx.x + k gridDim.x, k < n_own, in batches of LT
  const uint32_t b = blockIdx.x, grid = gridDim.x;
  const uint32_t n_own = b < P.n_chunks ? (P.n_chunks - 1 - b) / grid + 1 : 0;
  const bool any_inpl = P.inplace_hi[0] > P.inplace_lo[0] || P.inplace_hi[1] > P.inplace_lo[1];
  __shared__ uint32_t s_skip[LT / 32];
  for (uint32_t kb = 0; kb < n_own; kb += LT) {
    if (any_inpl) {
      // one chunk of the batch per thread: a raw chunk whose codes are read in place
      // only gets its stream address in state[c] and is skipped below
      const uint32_t k = kb + threadIdx.x;
      bool skip = false;
      if (k < n_own) {
        const uint32_t c = b + k * grid;
        if (in_place_chunk(P, c)) {
          const uint32_t e = table[c];
          if (e >> 31) {
            const uint64_t soff = P.fused_offsets ? s_off[k] : P.state[c];
            P.state[c] = (uint64_t)(uintptr_t)(P.stream + soff);
            skip = true;
          }
        }
      }
      const uint32_t m = __ballot_sync(0xffffffffu, skip);
      if ((threadIdx.x & 31) == 0) s_skip[threadIdx.x >> 5] = m;
      __syncthreads();
    }
    const uint32_t kend = min(n_own, kb + (uint32_t)LT);
    for (uint32_t kc = kb; kc < kend; kc++) {
      if (any_inpl && ((s_skip[(kc - kb) >> 5] >> ((kc - kb) & 31)) & 1u)) continue;
      const uint32_t c = b + kc * grid;
      const uint32_t e = table[c], size = e & 0x7fffffffu;
      const uint64_t off = (uint64_t)c * P.chunk_bytes;
      const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
      const uint64_t soff = P.fused_offsets ? s_off[kc] : P.state[c];
      const uint4 *src = reinterpret_cast<const uint4 *>(P.stream + soff);
      uint4 *dst = reinterpret_cast<uint4 *>(P.out_payload + off);
      if (in_place_chunk(P, c)) {  // a compressed chunk read in place: restored into the payload
        if (!P.fused_offsets) __syncthreads();  // every thread has read state[c]
        if (threadIdx.x == 0) P.state[c] = (uint64_t)(uintptr_t)(P.out_payload + off);
      }
      if (e >> 31) {
        for (uint32_t i = threadIdx.x; i < n / 16; i += LT) dst[i] = __ldg(src + i);
        continue;
      }
      if (!has_rze) {  // a non-raw chunk needs an RZE stage (the prepare step allows size < n only)
        if (threadIdx.x == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
        continue;
      }
      for (uint32_t i = threadIdx.x; i < align16u(size) / 16; i += LT)
        reinterpret_cast<uint4 *>(bufA)[i] = __ldg(src + i);
      __syncthreads();
      if (F.rze_w != 0 && fast_len(n)) {
        uint8_t *d8 = P.out_payload + off;
        bool ok;
        if (F.rze_w == 2) {
          if (F.delta1) ok = F.bit8 ? fast_decode_chunk<2, true, true>(bufA, size, n, bufB, d8, tmp)
                                    : fast_decode_chunk<2, true, false>(bufA, size, n, bufB, d8, tmp);
          else ok = F.bit8 ? fast_decode_chunk<2, false, true>(bufA, size, n, bufB, d8, tmp)
                           : fast_decode_chunk<2, false, false>(bufA, size, n, bufB, d8, tmp);
        } else {
          if (F.delta1) ok = F.bit8 ? fast_decode_chunk<1, true, true>(bufA, size, n, bufB, d8, tmp)
                                    : fast_decode_chunk<1, true, false>(bufA, size, n, bufB, d8, tmp);
          else ok = F.bit8 ? fast_decode_chunk<1, false, true>(bufA, size, n, bufB, d8, tmp)
                           : fast_decode_chunk<1, false, false>(bufA, size, n, bufB, d8, tmp);
        }
        if (!ok) {
          if (threadIdx.x == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
          __syncthreads();
        }
        continue;
      }
      const bool ok = rze_decode(bufA, size, bufB, n, P.param[last], Bs, tmp);
      if (!ok) {
        if (threadIdx.x == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
        __syncthreads();
        continue;
      }
      uint8_t *cur = bufB, *nxt = bufA;
      for (int s = (int)last - 1; s >= 0; s--) {
        const uint32_t k = P.kind[s], prm = P.param[s];
        if (k == KVC_ST_TUPL) tupl_decode(cur, nxt, n, prm);
        else if (k == KVC_ST_BIT) bit_decode(cur, nxt, n);
        else delta_decode(cur, nxt, n, prm, tmp);
        uint8_t *t = cur; cur = nxt; nxt = t;
      }
      for (uint32_t i = threadIdx.x; i < n / 16; i += LT) dst[i] = reinterpret_cast<const uint4 *>(cur)[i];
      __syncthreads();
    }
    if (any_inpl) __syncthreads();  // s_skip is rewritten by the next batch
  }
}

// ---------------------------------------------------------------------------
static size_t lossless_smem(uint32_t chunk_bytes) { return 2 * ((size_t)chunk_bytes + 64) + kScratchBytes; }

int launch_prologue(const PrologueParams &p, void *stream) {
  uint64_t threads = 256, blocks = 1;
  if (p.n_state > 256) blocks = (p.n_state + 255) / 256 < 1024 ? (p.n_state + 255) / 256 : 1024;
  kvc_prologue<<<(unsigned)blocks, (unsigned)threads, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

bool lossless_fast_spec(const LosslessParams &p, FastSpec &f) {
  f = FastSpec{0, 0, 0, 0};
  if (p.chunk_bytes > kFastMaxChunk || p.chunk_bytes % 4096) return false;
  uint32_t s = 0;
  if (s >= p.n_stages || p.kind[s] != KVC_ST_TUPL || p.param[s] != 8) return false;
  s++;
  if (s < p.n_stages && p.kind[s] == KVC_ST_BIT) { f.bit8 = 1; s++; }
  if (s < p.n_stages && p.kind[s] == KVC_ST_DELTA && p.param[s] == 1) { f.delta1 = 1; s++; }
  if (s + 1 != p.n_stages || p.kind[s] != KVC_ST_RZE || (p.param[s] != 1 && p.param[s] != 2)) return false;
  f.rze_w = p.param[s];
  return true;
}

static size_t fast_smem(uint32_t cb) { return (1 + kRing) * ((size_t)cb + 64) + cb / 8 + 64 + 64 * 4; }

int launch_lossless_encode(const LosslessParams &p, int sm_count, void *stream) {
  if (p.last_chunk <= p.first_chunk || p.last_chunk > p.n_chunks) return 0;
  const uint32_t range = p.last_chunk - p.first_chunk;
  FastSpec f;
  if (!p.generic_only && lossless_fast_spec(p, f)) {
    const size_t smem = fast_smem(p.chunk_bytes);
    cudaError_t e = cudaFuncSetAttribute(kvc_lossless_enc_fast, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc_lossless_enc_fast, FW, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    uint64_t blocks = (uint64_t)sm_count * per_sm;
    if (blocks > range) blocks = range;
    kvc_lossless_enc_fast<<<(unsigned)blocks, FW, smem, (cudaStream_t)stream>>>(p, f);
    return (int)cudaGetLastError();
  }
  const size_t smem = lossless_smem(p.chunk_bytes);
  cudaError_t e = cudaFuncSetAttribute(kvc_lossless_enc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc_lossless_enc, LT, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  uint64_t blocks = (uint64_t)sm_count * per_sm;
  if (blocks > range) blocks = range;
  kvc_lossless_enc<<<(unsigned)blocks, LT, smem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

bool lossless_encode_is_fast(const LosslessParams &p) {
  FastSpec f;
  return p.n_chunks != 0 && !p.generic_only && lossless_fast_spec(p, f);
}

bool lossless_decode_is_fast(const LosslessParams &p) {
  FastSpec f;
  return p.n_chunks != 0 && p.n_stages != 0 && !p.generic_only && lossless_fast_spec(p, f);
}

int launch_decode_prepare(const LosslessParams &p, void *stream) {
  if (cudaMemsetAsync(p.ctrl + kCtrlFlags, 0, sizeof(uint32_t), (cudaStream_t)stream) != cudaSuccess)
    return (int)cudaGetLastError();
  const uint32_t blocks = p.n_chunks ? (p.n_chunks + kPrepSeg - 1) / kPrepSeg : 1;
  kvc_decode_sums<<<blocks, PT, 0, (cudaStream_t)stream>>>(p);  // with no chunks: the header checks only
  if (p.n_chunks) kvc_decode_offsets<<<blocks, PT, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

static uint64_t decode_blocks(const LosslessParams &p, int sm_count) {
  const size_t smem = lossless_smem(p.chunk_bytes);
  if (cudaFuncSetAttribute(kvc_lossless_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc_lossless_dec, LT, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  uint64_t blocks = (uint64_t)sm_count * per_sm;
  return blocks > p.n_chunks ? p.n_chunks : blocks;
}

bool lossless_decode_fusable(const LosslessParams &p, int sm_count) {
  if (p.n_stages == 0 || p.n_chunks == 0 || p.n_chunks > kFusedMaxChunks || p.stream_cap < p.data_start) return false;
  const uint64_t blocks = decode_blocks(p, sm_count);
  return blocks > 0 && (p.n_chunks + blocks - 1) / blocks <= kFusedMaxOwn;
}

int launch_lossless_decode(const LosslessParams &p, int sm_count, void *stream) {
  if (p.n_chunks == 0 || p.n_stages == 0) return 0;
  const size_t smem = lossless_smem(p.chunk_bytes);
  const uint64_t blocks = decode_blocks(p, sm_count);
  if (blocks == 0) return (int)cudaErrorInvalidValue;
  FastSpec f;
  if (p.generic_only || !lossless_fast_spec(p, f)) f = FastSpec{0, 0, 0, 0};  // rze_w == 0: generic stages for every chunk
  kvc_lossless_dec<<<(unsigned)blocks, LT, smem, (cudaStream_t)stream>>>(p, f);
  return (int)cudaGetLastError();
}

}  // namespace kvc
