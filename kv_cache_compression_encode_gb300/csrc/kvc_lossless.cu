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
// Stream: 64-byte header | u32 table[n_chunks] (bit 31 = stored raw, bits 0..30 =
// stored size) | chunk i at data_start + sum_{j<i} align16(size_j), zero padded.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc_internal.h"

namespace kvc {

constexpr int LT = 512;               // threads per lossless CTA
constexpr int kScratchBytes = 8192 + 1024 + 256;  // RZE bitmap (<= 64 KiB / 8) + scan temporaries
constexpr uint64_t kFlagAgg = 1ull << 62, kFlagIncl = 2ull << 62, kValMask = (1ull << 62) - 1;

__device__ __forceinline__ uint32_t align16u(uint32_t x) { return (x + 15u) & ~15u; }

__device__ __forceinline__ void st_release(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Block-wide exclusive scan of one value per thread (LT threads).  tmp holds
// LT/32 + 1 words.  Ends with a barrier, so tmp can be reused immediately.
template <typename U>
__device__ __forceinline__ U block_excl_scan(U v, U *tmp, U &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  U x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    U w = lane < LT / 32 ? tmp[lane] : U(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const U y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < LT / 32) tmp[lane] = w;
    if (lane == LT / 32 - 1) tmp[LT / 32] = w;
  }
  __syncthreads();
  const U excl = x - v + (warp ? tmp[warp - 1] : U(0));
  total = tmp[LT / 32];
  __syncthreads();
  return excl;
}

// 8x8 bit-matrix transpose: byte i of x = row i, bit j = column j.  Afterwards
// bit i of byte p is bit p of the original byte i.  Three block swaps (2x2, 4x4,
// 8x8 sub-blocks), each exchanging the off-diagonal blocks.
__device__ __forceinline__ uint64_t transpose8(uint64_t x) {
  uint64_t t;
  t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
  x ^= t ^ (t << 7);
  t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
  x ^= t ^ (t << 14);
  t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
  x ^= t ^ (t << 28);
  return x;
}

__device__ __forceinline__ uint32_t ld_word(const uint8_t *p, uint32_t w) {
  if (w == 4) return *reinterpret_cast<const uint32_t *>(p);
  if (w == 2) return *reinterpret_cast<const uint16_t *>(p);
  return *p;
}
__device__ __forceinline__ void st_word(uint8_t *p, uint32_t w, uint32_t v) {
  if (w == 4) *reinterpret_cast<uint32_t *>(p) = v;
  else if (w == 2) *reinterpret_cast<uint16_t *>(p) = (uint16_t)v;
  else *p = (uint8_t)v;
}

// ---------------------------------------------------------------------------
// Stages (block-wide; `in` and `out` are distinct shared buffers; n bytes).
// Every stage keeps the tail past the last whole tuple / word as is.
// ---------------------------------------------------------------------------
// TUPL_k: m = n/k tuples; column j (byte j of every tuple) is written contiguously.
__device__ void tupl_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t k) {
  const uint32_t m = n / k;
  if ((m & 3u) == 0) {
    // four tuples per thread: read 4k bytes, write k words of 4 bytes
    const uint32_t nq = m / 4;
    for (uint32_t idx = threadIdx.x; idx < nq; idx += LT) {
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
      for (uint32_t i = threadIdx.x; i < m; i += LT) out[j * m + i] = in[i * k + j];
  }
  for (uint32_t o = m * k + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

__device__ void tupl_decode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t k) {
  const uint32_t m = n / k;
  for (uint32_t i = threadIdx.x; i < m; i += LT) {
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
  for (uint32_t o = m * k + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

// BIT_8: plane p (n8/8 bytes) collects bit p of every byte, byte i -> bit i%8 of byte i/8.
__device__ void bit_encode(const uint8_t *in, uint8_t *out, uint32_t n) {
  const uint32_t n8 = n & ~7u, P = n8 / 8;
  if ((P & 3u) == 0) {
    for (uint32_t idx = threadIdx.x; idx < P / 4; idx += LT) {
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
    for (uint32_t b = threadIdx.x; b < P; b += LT) {
      const uint64_t x = transpose8(*reinterpret_cast<const uint64_t *>(in + 8 * b));
#pragma unroll
      for (int p = 0; p < 8; p++) out[p * P + b] = (uint8_t)(x >> (8 * p));
    }
  }
  for (uint32_t o = n8 + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

__device__ void bit_decode(const uint8_t *in, uint8_t *out, uint32_t n) {
  const uint32_t n8 = n & ~7u, P = n8 / 8;
  for (uint32_t b = threadIdx.x; b < P; b += LT) {
    uint64_t x = 0;
#pragma unroll
    for (int p = 0; p < 8; p++) x |= (uint64_t)in[p * P + b] << (8 * p);
    *reinterpret_cast<uint64_t *>(out + 8 * b) = transpose8(x);
  }
  for (uint32_t o = n8 + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

// DELTA_w: word i -> word i - word (i-1) mod 2^(8w); word 0 kept.
__device__ void delta_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w) {
  const uint32_t m = n / w;
  const uint32_t mask = w == 4 ? 0xffffffffu : ((1u << (8 * w)) - 1u);
  for (uint32_t i = threadIdx.x; i < m; i += LT) {
    const uint32_t cur = ld_word(in + i * w, w), prev = i ? ld_word(in + (i - 1) * w, w) : 0u;
    st_word(out + i * w, w, (cur - prev) & mask);
  }
  for (uint32_t o = m * w + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

// Inverse: running sum mod 2^(8w); each thread sums a contiguous run, then a block scan.
__device__ void delta_decode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w, uint32_t *tmp) {
  const uint32_t m = n / w;
  const uint32_t mask = w == 4 ? 0xffffffffu : ((1u << (8 * w)) - 1u);
  const uint32_t S = (m + LT - 1) / LT;
  const uint32_t i0 = min(m, threadIdx.x * S), i1 = min(m, i0 + S);
  uint32_t sum = 0;
  for (uint32_t i = i0; i < i1; i++) sum += ld_word(in + i * w, w);
  uint32_t total;
  uint32_t acc = block_excl_scan<uint32_t>(sum, tmp, total);
  for (uint32_t i = i0; i < i1; i++) {
    acc += ld_word(in + i * w, w);
    st_word(out + i * w, w, acc & mask);
  }
  for (uint32_t o = m * w + threadIdx.x; o < n; o += LT) out[o] = in[o];
  __syncthreads();
}

// RZE_w: B = bitmap of nonzero words, B2 = bitmap of nonzero bytes of B; output
// B2 | nonzero B bytes | nonzero words | tail.  Returns the encoded size; when it
// is >= n nothing is written (the chunk will be stored raw).
__device__ uint32_t rze_encode(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t w, uint8_t *Bs,
                               uint32_t *tmp) {
  const uint32_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8, tail = n - m * w;
  const uint32_t S = (nb + LT - 1) / LT;
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
  const uint32_t exW = block_excl_scan<uint32_t>(cw, tmp, totW);
  const uint32_t exB = block_excl_scan<uint32_t>(cb, tmp, totB);
  const uint32_t size = nb2 + totB + w * totW + tail;
  if (size >= n) return size;
  for (uint32_t b2 = threadIdx.x; b2 < nb2; b2 += LT) {
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
  for (uint32_t o = threadIdx.x; o < tail; o += LT) out[t0 + o] = in[m * w + o];
  __syncthreads();
  return size;
}

// Inverse of RZE for `size` stored bytes that must expand to exactly n bytes.
// Returns false (uniformly across the block) when the bytes are inconsistent.
__device__ bool rze_decode(const uint8_t *in, uint32_t size, uint8_t *out, uint32_t n, uint32_t w, uint8_t *Bs,
                           uint32_t *tmp) {
  const uint32_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8, tail = n - m * w;
  if (size < nb2) return false;
  // B bytes listed by B2 (only its first nb bits count)
  const uint32_t S2 = (nb2 + LT - 1) / LT;
  const uint32_t b0 = min(nb2, threadIdx.x * S2), b1 = min(nb2, b0 + S2);
  uint32_t cb = 0;
  for (uint32_t b = b0; b < b1; b++) {
    uint32_t v = in[b];
    if (8 * b + 8 > nb) v &= (1u << (nb - 8 * b)) - 1u;
    cb += __popc(v);
  }
  uint32_t totB;
  uint32_t rB = block_excl_scan<uint32_t>(cb, tmp, totB);
  if (nb2 + totB > size) return false;
  for (uint32_t b = b0; b < b1; b++) {
    const uint32_t v = in[b];
    for (uint32_t q = 0; q < 8; q++) {
      const uint32_t j = 8 * b + q;
      if (j >= nb) break;
      Bs[j] = ((v >> q) & 1u) ? in[nb2 + rB++] : (uint8_t)0;
    }
  }
  __syncthreads();
  // words listed by B (only its first m bits count)
  const uint32_t S = (nb + LT - 1) / LT;
  const uint32_t j0 = min(nb, threadIdx.x * S), j1 = min(nb, j0 + S);
  uint32_t cw = 0;
  for (uint32_t j = j0; j < j1; j++) {
    uint32_t v = Bs[j];
    if (8 * j + 8 > m) v &= (1u << (m - 8 * j)) - 1u;
    cw += __popc(v);
  }
  uint32_t totW;
  uint32_t rW = block_excl_scan<uint32_t>(cw, tmp, totW);
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
  for (uint32_t o = threadIdx.x; o < tail; o += LT) out[m * w + o] = tl[o];
  __syncthreads();
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
  if (P.write_header && tid < KVC_HEADER_BYTES) P.stream[tid] = P.header[tid];
  if (P.write_header && tid < P.gap_len) P.stream[P.gap_off + tid] = 0;
  if (P.payload && tid < 6 * 16) {
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
    if (threadIdx.x == 0) s_ticket = atomicAdd(ctrl + kCtrlTicket, 1u);
    __syncthreads();
    const uint32_t ticket = s_ticket;
    if (ticket >= P.n_chunks) break;
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

    // decoupled look-back: publish this chunk's aggregate, then add predecessors' until an inclusive prefix
    if (threadIdx.x == 0) {
      uint64_t *state = P.state;
      const bool publish = (int64_t)ticket != P.skip_ticket;
      uint64_t excl = 0;
      if (ticket == 0) {
        if (publish) st_release(state, kFlagIncl | asz);
      } else {
        if (publish) st_release(state + ticket, kFlagAgg | asz);
        uint32_t j = ticket - 1, polls = 0;
        for (;;) {
          const uint64_t v = ld_acquire(state + j);
          const uint64_t f = v & ~kValMask;
          if (f == 0) {
            if (++polls > P.poll_limit) {
              atomicOr(ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
              break;
            }
            __nanosleep(64);
            continue;
          }
          excl += v & kValMask;
          if (f == kFlagIncl || j == 0) break;
          --j;
        }
        if (publish) st_release(state + ticket, kFlagIncl | (excl + asz));
      }
      s_excl = excl;
      const uint64_t dst = P.data_start + excl;
      if (dst + asz > P.stream_cap) atomicOr(ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CAPACITY);
      reinterpret_cast<uint32_t *>(P.stream + KVC_HEADER_BYTES)[ticket] = size | (raw ? 0x80000000u : 0u);
      if (ticket == P.n_chunks - 1) {
        const uint64_t total = dst + asz;
        reinterpret_cast<uint64_t *>(ctrl)[kCtrlStreamBytes] = total;
        if (P.d_stream_bytes) *P.d_stream_bytes = total;
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

// ---------------------------------------------------------------------------
// Decode, step 1 (one CTA): check the header and the chunk table, compute the
// chunk offsets.  Any inconsistency sets KVC_FLAG_CORRUPT.
// ---------------------------------------------------------------------------
constexpr int PT = 1024;

__global__ void __launch_bounds__(PT) kvc_decode_prepare(const LosslessParams P) {
  __shared__ unsigned long long tmp[PT / 32 + 1];
  __shared__ int s_bad;
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bad = 0;
    P.ctrl[kCtrlFlags] = 0u;
  }
  __syncthreads();
  const uint64_t stream_bytes = P.stream_cap;
  if (stream_bytes < KVC_HEADER_BYTES) {
    if (tid == 0) s_bad = 1;
  } else if (tid < KVC_HEADER_BYTES / 4) {
    if (reinterpret_cast<const uint32_t *>(P.stream)[tid] != reinterpret_cast<const uint32_t *>(P.header)[tid])
      atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (!s_bad) {
    if (P.n_stages == 0) {
      if (tid == 0 && stream_bytes < KVC_HEADER_BYTES + P.payload_bytes) s_bad = 1;
    } else if (stream_bytes < P.data_start) {
      if (tid == 0) s_bad = 1;
    } else {
      const uint32_t nc = P.n_chunks;
      const uint32_t S = (nc + PT - 1) / PT;
      const uint32_t i0 = min(nc, tid * S), i1 = min(nc, i0 + S);
      const uint32_t *table = reinterpret_cast<const uint32_t *>(P.stream + KVC_HEADER_BYTES);
      unsigned long long sum = 0;
      int bad = 0;
      for (uint32_t i = i0; i < i1; i++) {
        const uint32_t e = table[i], sz = e & 0x7fffffffu;
        const uint64_t off = (uint64_t)i * P.chunk_bytes;
        const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
        if (e >> 31) bad |= sz != n;
        else bad |= sz >= n;
        sum += align16u(sz);
      }
      if (bad) atomicOr(&s_bad, 1);
      // exclusive scan of the aligned sizes (64-bit)
      unsigned long long x = sum;
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
      unsigned long long pos = P.data_start + x - sum + (warp ? tmp[warp - 1] : 0ull);
      for (uint32_t i = i0; i < i1; i++) {
        P.state[i] = pos;
        pos += align16u(table[i] & 0x7fffffffu);
      }
      if (tid == 0 && P.data_start + tmp[PT / 32] > stream_bytes) s_bad = 1;
    }
  }
  __syncthreads();
  if (tid == 0 && s_bad) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
}

// ---------------------------------------------------------------------------
// Decode, step 2: one chunk per CTA iteration back into the payload.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(LT) kvc_lossless_dec(const LosslessParams P) {
  if (*(volatile uint32_t *)(P.ctrl + kCtrlFlags) & KVC_FLAG_CORRUPT) return;
  extern __shared__ uint4 smem_u4[];
  uint8_t *bufA = reinterpret_cast<uint8_t *>(smem_u4);
  uint8_t *bufB = bufA + P.chunk_bytes + 64;
  uint8_t *Bs = bufB + P.chunk_bytes + 64;
  uint32_t *tmp = reinterpret_cast<uint32_t *>(Bs + 8192);
  const uint32_t *table = reinterpret_cast<const uint32_t *>(P.stream + KVC_HEADER_BYTES);
  const uint32_t last = P.n_stages - 1;
  const bool has_rze = P.kind[last] == KVC_ST_RZE;

  for (uint32_t c = blockIdx.x; c < P.n_chunks; c += gridDim.x) {
    const uint32_t e = table[c], size = e & 0x7fffffffu;
    const uint64_t off = (uint64_t)c * P.chunk_bytes;
    const uint32_t n = (uint32_t)min((uint64_t)P.chunk_bytes, P.payload_bytes - off);
    const uint4 *src = reinterpret_cast<const uint4 *>(P.stream + P.state[c]);
    uint4 *dst = reinterpret_cast<uint4 *>(P.out_payload + off);
    if (e >> 31) {
      for (uint32_t i = threadIdx.x; i < n / 16; i += LT) dst[i] = __ldg(src + i);
      continue;
    }
    if (!has_rze) {  // a non-raw chunk needs an RZE stage (the prepare step allows size < n only)
      if (threadIdx.x == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
      continue;
    }
    for (uint32_t i = threadIdx.x; i < align16u(size) / 16; i += LT) reinterpret_cast<uint4 *>(bufA)[i] = __ldg(src + i);
    __syncthreads();
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
}

// ---------------------------------------------------------------------------
static size_t lossless_smem(uint32_t chunk_bytes) { return 2 * ((size_t)chunk_bytes + 64) + kScratchBytes; }

int launch_prologue(const PrologueParams &p, void *stream) {
  uint64_t threads = 256, blocks = 1;
  if (p.n_state > 256) blocks = (p.n_state + 255) / 256 < 1024 ? (p.n_state + 255) / 256 : 1024;
  kvc_prologue<<<(unsigned)blocks, (unsigned)threads, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

int launch_lossless_encode(const LosslessParams &p, int sm_count, void *stream) {
  if (p.n_chunks == 0) return 0;
  const size_t smem = lossless_smem(p.chunk_bytes);
  cudaError_t e = cudaFuncSetAttribute(kvc_lossless_enc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc_lossless_enc, LT, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  uint64_t blocks = (uint64_t)sm_count * per_sm;
  if (blocks > p.n_chunks) blocks = p.n_chunks;
  kvc_lossless_enc<<<(unsigned)blocks, LT, smem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

int launch_decode_prepare(const LosslessParams &p, void *stream) {
  kvc_decode_prepare<<<1, PT, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

int launch_lossless_decode(const LosslessParams &p, int sm_count, void *stream) {
  if (p.n_chunks == 0 || p.n_stages == 0) return 0;
  const size_t smem = lossless_smem(p.chunk_bytes);
  cudaError_t e = cudaFuncSetAttribute(kvc_lossless_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc_lossless_dec, LT, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  uint64_t blocks = (uint64_t)sm_count * per_sm;
  if (blocks > p.n_chunks) blocks = p.n_chunks;
  kvc_lossless_dec<<<(unsigned)blocks, LT, smem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace kvc
