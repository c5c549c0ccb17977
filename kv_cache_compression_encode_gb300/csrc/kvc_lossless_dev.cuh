// kvc_lossless_dev.cuh -- device building blocks of the chunked lossless stages
// shared by the lossless kernels (kvc_lossless.cu) and the value encoder that
// writes its code chunks straight into the stream (kvc_fused.cu): look-back words,
// block scans, and the fast path's size, transform and delta/zero-elimination
// passes for TUPL_8 [BIT_8] [DELTA_1] RZE_w ("Beyond Compression Ratio: High-
// Throughput KV Compression for Disaggregated LLM Serving", §4.2).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc_internal.h"

namespace kvc {

constexpr int LT = 512;               // threads per generic lossless CTA
constexpr int kScratchBytes = 8192 + 1024 + 256;  // RZE bitmap (<= 64 KiB / 8) + scan temporaries
constexpr uint64_t kFlagAgg = 1ull << 62, kFlagIncl = 2ull << 62, kValMask = (1ull << 62) - 1;

__device__ __forceinline__ uint32_t align16u(uint32_t x) { return (x + 15u) & ~15u; }

// A look-back word carries its flag and its value in one 64-bit access and no
// other data is read through it, so relaxed (non-ordering) device-scope accesses
// suffice -- and unlike acquire loads, a lane's loads of a whole window can all
// be in flight at once.
__device__ __forceinline__ void st_word64(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_word64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Barrier over the first NT threads of the CTA (named barrier 1).  Stage functions
// use it instead of __syncthreads so that a CTA can hold threads outside the
// group that runs them (the encoder's publisher warp); in a CTA of exactly NT
// threads it is an ordinary CTA barrier.
template <int NT>
__device__ __forceinline__ void bsync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Block-wide exclusive scan of one value per thread (LT threads).  tmp holds
// LT/32 + 1 words.  Ends with a barrier, so tmp can be reused immediately.
template <typename U, int NT = LT>
__device__ __forceinline__ U block_excl_scan(U v, U *tmp, U &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  U x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  bsync<NT>();
  if (warp == 0) {
    U w = lane < NT / 32 ? tmp[lane] : U(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const U y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) tmp[lane] = w;
    if (lane == NT / 32 - 1) tmp[NT / 32] = w;
  }
  bsync<NT>();
  const U excl = x - v + (warp ? tmp[warp - 1] : U(0));
  total = tmp[NT / 32];
  bsync<NT>();
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

__device__ __forceinline__ uint64_t warp_sum64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Exclusive prefix of chunk `ticket` by the decoupled look-back of one warp:
// lane l reads the word of chunk base - l, 32 predecessors per round; aggregates
// are summed until an inclusive prefix is reached, and a predecessor that has not
// published yet is polled again (bounded by poll_limit, then KVC_FLAG_TIMEOUT).
// Publishes nothing.
static __device__ uint64_t lookback_excl(const LosslessParams &P, uint32_t ticket) {
  const int lane = threadIdx.x & 31;
  const uint64_t *state = P.state;
  uint64_t excl = 0;
  int64_t base = (int64_t)ticket - 1;  // lane i looks at chunk base - i
  uint32_t polls = 0;
  for (;;) {
    const int64_t j = base - lane;
    const uint64_t v = j >= 0 ? ld_word64(state + j) : kFlagIncl;  // before chunk 0: an inclusive prefix of 0
    const uint64_t f = v & ~kValMask;
    const uint32_t not_ready = __ballot_sync(0xffffffffu, f == 0);
    const uint32_t incl = __ballot_sync(0xffffffffu, f == kFlagIncl);
    const int first_nr = not_ready ? __ffs(not_ready) - 1 : 32;
    const int first_inc = incl ? __ffs(incl) - 1 : 32;
    if (first_inc < first_nr) {  // an inclusive prefix with only aggregates before it
      excl += warp_sum64(lane <= first_inc ? (v & kValMask) : 0ull);
      break;
    }
    excl += warp_sum64(lane < first_nr ? (v & kValMask) : 0ull);
    if (first_nr == 32) {  // 32 aggregates: keep walking back
      base -= 32;
      continue;
    }
    base -= first_nr;  // resume at the predecessor that has not published yet
    if (++polls > P.poll_limit) {
      if (lane == 0) atomicOr(P.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_TIMEOUT);
      break;
    }
    __nanosleep(64);
  }
  return excl;
}

// The whole look-back for one chunk of `agg` bytes: publish the aggregate, find
// the exclusive prefix, publish the inclusive one.
static __device__ uint64_t lookback_warp(const LosslessParams &P, uint32_t ticket, uint64_t agg) {
  const int lane = threadIdx.x & 31;
  const bool publish = (int64_t)ticket != P.skip_ticket;
  if (ticket == 0) {
    if (lane == 0 && publish) st_word64(P.state, kFlagIncl | agg);
    return 0;
  }
  if (lane == 0 && publish) st_word64(P.state + ticket, kFlagAgg | agg);
  const uint64_t excl = lookback_excl(P, ticket);
  if (lane == 0 && publish) st_word64(P.state + ticket, kFlagIncl | (excl + agg));
  return excl;
}

constexpr int FT = 256;        // worker threads
constexpr int kPubWarps = 2;  // publisher warps, taking the CTA's chunks in turn
constexpr int FW = FT + 32 * kPubWarps + 32;  // workers + publishers + the loader warp
constexpr uint32_t kAhead = 2;  // the loader takes a ticket at most this many chunks ahead
constexpr int kRing = 5;       // slots per CTA (16 KiB chunks: 2 CTAs per SM)
constexpr int kFastCtasPerSm = 2;
constexpr uint32_t kFastMaxChunk = 16384;
constexpr uint32_t kMbarTries = 1u << 20;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(b)),
               "r"(bytes)
               : "memory");
}
// Waits until the phase of parity `par` has completed; false after kMbarTries tries.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t par) {
  for (uint32_t i = 0; i < kMbarTries; i++) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_addr(b)), "r"(par)
                 : "memory");
    if (done) return true;
  }
  return false;
}

// The transform's output is stored swizzled: 16-byte unit u at unit
// (u & ~3) | ((u + (u >> 3)) & 3), i.e. within each 64-byte block the four units
// rotate by (block >> 1), so 8 lanes reading unit k of 8 consecutive blocks touch
// 8 distinct bank groups.  swzb is that map on a byte offset.
__device__ __forceinline__ uint32_t swzb(uint32_t x) { return (x & ~0x30u) | ((((x >> 4) + (x >> 7)) & 3u) << 4); }
__device__ __forceinline__ bool fast_len(uint32_t n) { return (n & 4095u) == 0 && n <= kFastMaxChunk; }

// 4x4 byte transpose: o[j] = byte j of a, b, c, d.
__device__ __forceinline__ void byte_t4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&o)[4]) {
  const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(c, d, 0x5140);
  const uint32_t t2 = __byte_perm(a, b, 0x7362), t3 = __byte_perm(c, d, 0x7362);
  o[0] = __byte_perm(t0, t1, 0x5410);
  o[1] = __byte_perm(t0, t1, 0x7632);
  o[2] = __byte_perm(t2, t3, 0x5410);
  o[3] = __byte_perm(t2, t3, 0x7632);
}

// transpose8 on the 64-bit value (hi:lo), both 32-bit halves at a time.
__device__ __forceinline__ void bits8x8(uint32_t &lo, uint32_t &hi) {
  uint32_t t;
  t = (lo ^ (lo >> 7)) & 0x00AA00AAu; lo ^= t ^ (t << 7);
  t = (hi ^ (hi >> 7)) & 0x00AA00AAu; hi ^= t ^ (t << 7);
  t = (lo ^ (lo >> 14)) & 0x0000CCCCu; lo ^= t ^ (t << 14);
  t = (hi ^ (hi >> 14)) & 0x0000CCCCu; hi ^= t ^ (t << 14);
  t = (lo ^ (hi << 4)) & 0xF0F0F0F0u;
  lo ^= t;
  hi ^= t >> 4;
}

// TUPL_8 (and BIT_8 after it) of a fast chunk, plain in and swizzled out.
// Without BIT_8, tuple byte j of block beta goes to byte 8*beta.. of row j (m
// bytes per row); with BIT_8, bit p of those 8 bytes forms byte beta of row j of
// bit plane p.  n is a multiple of 4 KiB, so a row start never changes the
// swizzle rotation and each thread computes its offsets once per row.
template <bool BIT8>
__device__ void fast_transform(const uint8_t *in, uint8_t *out, uint32_t n) {
  const uint32_t nblk = n / 64, m = n / 8, m8 = n / 64;
  for (uint32_t beta = threadIdx.x; beta < nblk; beta += FT) {
    uint32_t w[16];
    const uint4 *blk = reinterpret_cast<const uint4 *>(in) + 4 * beta;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint4 v = blk[k];
      w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
    }
    uint32_t L0[4], L1[4], H0[4], H1[4];  // byte j (0..3 / 4..7) of tuples 0..3 / 4..7
    byte_t4x4(w[0], w[2], w[4], w[6], L0);
    byte_t4x4(w[8], w[10], w[12], w[14], L1);
    byte_t4x4(w[1], w[3], w[5], w[7], H0);
    byte_t4x4(w[9], w[11], w[13], w[15], H1);
    const uint32_t off8 = 64 * (beta >> 3) + 16 * (((beta >> 1) + (beta >> 4)) & 3u) + 8 * (beta & 1u);
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint32_t lo = j < 4 ? L0[j & 3] : H0[j & 3], hi = j < 4 ? L1[j & 3] : H1[j & 3];
      if (BIT8) {
        bits8x8(lo, hi);
        uint8_t *ob = out + swzb(j * m8 + beta);
#pragma unroll
        for (int p = 0; p < 4; p++) ob[p * m] = (uint8_t)(lo >> (8 * p));
#pragma unroll
        for (int p = 0; p < 4; p++) ob[(p + 4) * m] = (uint8_t)(hi >> (8 * p));
      } else {
        *reinterpret_cast<uint2 *>(out + j * m + off8) = make_uint2(lo, hi);
      }
    }
  }
  bsync<FT>();
}

// The encoded size of a fast chunk under TUPL_8, BIT_8, [DELTA_1], RZE_w computed
// from the chunk as loaded (plain, in shared memory), without the transform.
// Bit-plane byte (p, j) of block beta holds bit p of byte j of the block's 8
// tuples, so it is nonzero iff bit p of OR_i tuple_i[j] is set; with DELTA_1 the
// stream byte is nonzero iff the plane byte differs from the one before it, which
// for beta > 0 is the same plane's byte in block beta - 1: bit p of
// OR_i (tuple_i[j] ^ prev_tuple_i[j]).  So 64 nonzero flags per block come from an
// OR-fold of the block (XOR'd with the previous one); block 0, whose predecessors
// are the last bytes of the previous planes, takes the real transform of blocks 0
// and n/64 - 1.  Elements (W = 2: the plane bytes of blocks 2u, 2u + 1) and
// level-1 bitmap bytes (8 elements: 8 W consecutive blocks of one plane) are ORs
// of these flags across neighbouring threads.  Returns nb2 + totB + W totW, the
// size the full pass computes (uniform across the CTA).
__device__ __forceinline__ uint64_t plane_bytes(const uint32_t (&w)[16], uint32_t j) {  // byte p = plane (p, j)
  const bool h = j >= 4;
  uint32_t L[4], M[4];
  byte_t4x4(h ? w[1] : w[0], h ? w[3] : w[2], h ? w[5] : w[4], h ? w[7] : w[6], L);
  byte_t4x4(h ? w[9] : w[8], h ? w[11] : w[10], h ? w[13] : w[12], h ? w[15] : w[14], M);
  const uint32_t q = j & 3u;
  uint32_t lo = q == 0 ? L[0] : q == 1 ? L[1] : q == 2 ? L[2] : L[3];
  uint32_t hi = q == 0 ? M[0] : q == 1 ? M[1] : q == 2 ? M[2] : M[3];
  bits8x8(lo, hi);
  return ((uint64_t)hi << 32) | lo;
}

template <int W, bool DELTA>
__device__ uint32_t fast_size_bit8(const uint8_t *S, uint32_t n, uint32_t *wsum) {
  const uint32_t nthr = n / 64, nb = n / (8 * W), nb2 = nb / 8;
  const uint32_t t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const bool active = t < nthr;
  uint32_t olo = 0, ohi = 0;  // flag of plane (p, j): bit 8j + p of (ohi:olo)
  if (active && !(DELTA && t == 0)) {
    // the fold does not depend on the order of the four units: reading them
    // rotated by (t >> 1) & 3 keeps 8 lanes on 8 distinct bank groups
    const uint4 *blk = reinterpret_cast<const uint4 *>(S) + 4 * t;
    const uint32_t rot = (t >> 1) & 3u;
    uint32_t x[16];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint4 v = blk[(k + rot) & 3u];
      x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
    }
    if (DELTA) {
      const uint4 *pb = blk - 4;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint4 v = pb[(k + rot) & 3u];
        x[4 * k] ^= v.x; x[4 * k + 1] ^= v.y; x[4 * k + 2] ^= v.z; x[4 * k + 3] ^= v.w;
      }
    }
    olo = x[0] | x[2] | x[4] | x[6] | x[8] | x[10] | x[12] | x[14];
    ohi = x[1] | x[3] | x[5] | x[7] | x[9] | x[11] | x[13] | x[15];
  }
  if (DELTA && warp == 0) {  // block 0: lane j < 8 compares plane (p, j) with its predecessor in the last block
    uint64_t pb0 = 0, pbl = 0;
    if (lane < 8) {
      uint32_t x[16], y[16];
      const uint4 *b0 = reinterpret_cast<const uint4 *>(S), *bl = b0 + 4 * (nthr - 1);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint4 v = b0[k], u = bl[k];
        x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
        y[4 * k] = u.x; y[4 * k + 1] = u.y; y[4 * k + 2] = u.z; y[4 * k + 3] = u.w;
      }
      pb0 = plane_bytes(x, lane);
      pbl = plane_bytes(y, lane);
    }
    // (p, j) follows (p, j - 1) of the last block; (p, 0) follows (p - 1, 7)
    const uint64_t up = __shfl_up_sync(0xffffffffu, pbl, 1), l7 = __shfl_sync(0xffffffffu, pbl, 7);
    const uint64_t pred = lane == 0 ? (l7 << 8) : up;
    const uint64_t d = pb0 ^ pred;
    const uint64_t f = (((d & 0x7f7f7f7f7f7f7f7full) + 0x7f7f7f7f7f7f7f7full) | d) & 0x8080808080808080ull;
    const uint32_t fb = lane < 8 ? (uint32_t)(((f >> 7) * 0x0102040810204080ull) >> 56) : 0u;  // bit p
    uint32_t lo0 = 0, hi0 = 0;
#pragma unroll
    for (int jj = 0; jj < 8; jj++) {
      const uint32_t b = __shfl_sync(0xffffffffu, fb, jj);
      if (jj < 4) lo0 |= b << (8 * jj);
      else hi0 |= b << (8 * (jj - 4));
    }
    if (t == 0) {
      olo = lo0;
      ohi = hi0;
    }
  }
  uint32_t cw = 0, cb = 0;
  if (W == 2) {  // elements: the flags of blocks 2u and 2u + 1; bitmap bytes: 16 blocks
    const uint32_t elo = olo | __shfl_xor_sync(0xffffffffu, olo, 1), ehi = ohi | __shfl_xor_sync(0xffffffffu, ohi, 1);
    uint32_t glo = elo, ghi = ehi;
#pragma unroll
    for (int o = 2; o < 16; o <<= 1) {
      glo |= __shfl_xor_sync(0xffffffffu, glo, o);
      ghi |= __shfl_xor_sync(0xffffffffu, ghi, o);
    }
    if (active && (t & 1) == 0) cw = __popc(elo) + __popc(ehi);
    if (active && (t & 15) == 0) cb = __popc(glo) + __popc(ghi);
  } else {  // elements: the plane bytes; bitmap bytes: 8 blocks
    uint32_t glo = olo, ghi = ohi;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      glo |= __shfl_xor_sync(0xffffffffu, glo, o);
      ghi |= __shfl_xor_sync(0xffffffffu, ghi, o);
    }
    if (active) cw = __popc(olo) + __popc(ohi);
    if (active && (t & 7) == 0) cb = __popc(glo) + __popc(ghi);
  }
  uint32_t c = (cb << 16) | cw;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (lane == 0) wsum[warp] = c;
  bsync<FT>();
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < FT / 32; i++) tot += wsum[i];
  bsync<FT>();  // wsum is reused right after
  return nb2 + (tot >> 16) + W * (tot & 0xffffu);
}

// DELTA_1 (optional) and RZE_w of a transformed fast chunk held swizzled in `in`;
// the encoded chunk goes to `out` (which may be `in` itself: every read happens
// before the first barrier).  Returns the encoded size; nothing is written when it
// is >= n.
// Publishes chunk t's aligned encoded size for the look-back of its successors
// (chunk 0's size is its inclusive prefix).
__device__ __forceinline__ void publish_size(const LosslessParams &P, uint32_t t, uint32_t asz) {
  if ((int64_t)t != P.skip_ticket) st_word64(P.state + t, (t == 0 ? kFlagIncl : kFlagAgg) | asz);
}

template <int W, bool DELTA>
__device__ uint32_t fast_delta_rze(const uint8_t *in, uint8_t *out, uint32_t n, uint32_t *wsum, const LosslessParams &P,
                                   uint32_t ticket, bool publish = true) {
  const uint32_t nthr = n / 64, nb = n / (8 * W), nb2 = nb / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t t = threadIdx.x;
  const bool active = t < nthr;
  uint32_t x[16], prevw = 0;  // prevw: byte 3 = the byte before this thread's first byte
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = 0u;
  if (active) {
    const uint4 *src = reinterpret_cast<const uint4 *>(in) + 4 * t;
    const uint32_t rot = (t >> 1) & 3u;  // logical unit k of this block sits at unit (k + rot) & 3
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint4 v = src[(k + rot) & 3u];
      x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
    }
    // last byte of the previous block: logical unit 3 of block t - 1
    if (DELTA && t) prevw = (uint32_t)in[16 * (4 * (t - 1) + ((3u + ((t - 1) >> 1)) & 3u)) + 15] << 24;
  }
  // A byte of DELTA_1's output is zero exactly when the byte equals the one before
  // it, so the bitmaps only need x ^ (x shifted by one byte); the differences
  // themselves are formed when a compressible chunk's elements are written.
  // Word bitmap: W = 2 -> 32 words (one bit each, 4 bitmap bytes); W = 1 -> 64
  // bytes (8 bitmap bytes).
  uint32_t blo = 0, bhi = 0;
#pragma unroll
  for (int i = 0; i < 16; i++) {
    const uint32_t e = DELTA ? x[i] ^ __byte_perm(i ? x[i - 1] : prevw, x[i], 0x6543) : x[i];
    if (W == 2) {
      blo |= (uint32_t)((e & 0xffffu) != 0u) << (2 * i);
      blo |= (uint32_t)((e >> 16) != 0u) << (2 * i + 1);
    } else {
#pragma unroll
      for (int b = 0; b < 4; b++) {
        const uint32_t bit = (uint32_t)(((e >> (8 * b)) & 0xffu) != 0u);
        if (i < 8) blo |= bit << (4 * i + b);
        else bhi |= bit << (4 * (i - 8) + b);
      }
    }
  }
  uint32_t nzB = 0;
#pragma unroll
  for (int j = 0; j < 4; j++) nzB += ((blo >> (8 * j)) & 0xffu) != 0u;
  if (W == 1) {
#pragma unroll
    for (int j = 0; j < 4; j++) nzB += ((bhi >> (8 * j)) & 0xffu) != 0u;
  }
  const uint32_t nzW = __popc(blo) + (W == 1 ? __popc(bhi) : 0u);
  const uint32_t c = (nzB << 16) | nzW;
  uint32_t sc = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, sc, o);
    if (lane >= o) sc += y;
  }
  if (lane == 31) wsum[warp] = sc;
  bsync<FT>();
  uint32_t wb = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < FT / 32; i++) {
    const uint32_t v = wsum[i];
    if (i < warp) wb += v;
    tot += v;
  }
  const uint32_t totB = tot >> 16, totW = tot & 0xffffu;
  const uint32_t size = nb2 + totB + W * totW;
  if (t == 0 && publish) publish_size(P, ticket, align16u(size < n ? size : n));  // before the compaction
  if (size >= n) return size;  // uniform: the chunk is stored raw
  const uint32_t ex = wb + sc - c;
  uint32_t rB = ex >> 16, rW = ex & 0xffffu;
  // second-level bitmap: W = 2 -> 4 bits per thread (two threads per byte); W = 1 -> one byte per thread
  uint32_t nib = 0;
#pragma unroll
  for (int j = 0; j < 4; j++) nib |= (uint32_t)(((blo >> (8 * j)) & 0xffu) != 0u) << j;
  if (W == 2) {
    const uint32_t hi = __shfl_down_sync(0xffffffffu, nib, 1);
    if (active && (t & 1) == 0) out[t >> 1] = (uint8_t)(nib | (hi << 4));
  } else {
#pragma unroll
    for (int j = 0; j < 4; j++) nib |= (uint32_t)(((bhi >> (8 * j)) & 0xffu) != 0u) << (4 + j);
    if (active) out[t] = (uint8_t)nib;
  }
  if (DELTA) {  // byte-wise differences, mod 256 (no borrow crosses a byte)
#pragma unroll
    for (int i = 15; i >= 0; i--) {
      const uint32_t a = x[i], b = __byte_perm(i ? x[i - 1] : prevw, x[i], 0x6543);
      x[i] = ((a | 0x80808080u) - (b & 0x7f7f7f7fu)) ^ ((a ^ ~b) & 0x80808080u);
    }
  }
  if (active) {
    uint8_t *oB = out + nb2, *oW = out + nb2 + totB;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const uint32_t b = (blo >> (8 * j)) & 0xffu;
      if (b) oB[rB++] = (uint8_t)b;
    }
    if (W == 1) {
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const uint32_t b = (bhi >> (8 * j)) & 0xffu;
        if (b) oB[rB++] = (uint8_t)b;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; i++) {
      if (W == 2) {
        if ((blo >> (2 * i)) & 1u) { oW[2 * rW] = (uint8_t)x[i]; oW[2 * rW + 1] = (uint8_t)(x[i] >> 8); rW++; }
        if ((blo >> (2 * i + 1)) & 1u) { oW[2 * rW] = (uint8_t)(x[i] >> 16); oW[2 * rW + 1] = (uint8_t)(x[i] >> 24); rW++; }
      } else {
        const uint32_t bits = i < 8 ? (blo >> (4 * i)) : (bhi >> (4 * (i - 8)));
#pragma unroll
        for (int b = 0; b < 4; b++)
          if ((bits >> b) & 1u) oW[rW++] = (uint8_t)(x[i] >> (8 * b));
      }
    }
  }
  return size;
}

struct FastSpec {
  uint32_t bit8, delta1, rze_w, pad;
};

// Whether the stage list and chunk size have the fast path (TUPL_8 [BIT_8]
// [DELTA_1] RZE_1/2, chunks of 4, 8, 12 or 16 KiB), and its switches.
bool lossless_fast_spec(const LosslessParams &p, FastSpec &f);

}  // namespace kvc
