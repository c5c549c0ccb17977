// kvc_device.cuh -- device building blocks of the quantize / dequantize kernels.
//
// Every floating-point step is written with explicit round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fmaf_rn) so the compiler cannot contract or
// reorder it: the results are the binary32 values that the stream format fixes
// ("Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated
// LLM Serving", §4.1: the fused kernel preserves the transformation and
// quantization semantics exactly).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvc_internal.h"

namespace kvc {

constexpr unsigned kFull = 0xffffffffu;
// 1/sqrt(128) rounded to binary32 (the Hadamard normalization).
__device__ __forceinline__ float hadamard_scale() { return __uint_as_float(0x3DB504F3u); }

__device__ __forceinline__ float elt_to_f32(uint32_t bits16, bool bf16) {
  return bf16 ? __uint_as_float(bits16 << 16) : __half2float(__ushort_as_half((unsigned short)bits16));
}

__device__ __forceinline__ uint32_t f32_to_elt(float x, bool bf16) {
  return bf16 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x))
              : (uint32_t)__half_as_ushort(__float2half_rn(x));
}

// Unpack 8 half-precision elements held in a 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4 &w, bool bf16, float *x) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    x[2 * i] = elt_to_f32(u[i] & 0xffffu, bf16);
    x[2 * i + 1] = elt_to_f32(u[i] >> 16, bf16);
  }
}

__device__ __forceinline__ uint4 pack8(const float *x, bool bf16) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; i++) u[i] = f32_to_elt(x[2 * i], bf16) | (f32_to_elt(x[2 * i + 1], bf16) << 16);
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// Byte offset of token t's row inside one layer's buffer, or ~0 for a block-table
// entry outside [0, num_pages) (the caller treats the row as absent and flags it).
// 32 bytes to global memory in one access when `p` is 32-byte aligned (the
// 256-bit vector store of sm_100 and later), else as two 16-byte stores.
__device__ __forceinline__ void st_global32(void *p, const uint32_t (&u)[8]) {
  if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(u[0]), "r"(u[1]), "r"(u[2]),
                 "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7])
                 : "memory");
  } else {
    uint4 *q = reinterpret_cast<uint4 *>(p);
    q[0] = make_uint4(u[0], u[1], u[2], u[3]);
    q[1] = make_uint4(u[4], u[5], u[6], u[7]);
  }
}

// 32 read-only bytes from global memory, one 256-bit access when `p` is 32-byte
// aligned, else two 16-byte loads.
__device__ __forceinline__ void ld_global32_nc(const void *p, uint4 &a, uint4 &b) {
  if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
  } else {
    a = __ldg(reinterpret_cast<const uint4 *>(p));
    b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
  }
}

__device__ __forceinline__ uint64_t row_offset(const KvGeom &g, uint32_t t) {
  if (g.block_table) {
    uint32_t page = (uint32_t)__ldg(g.block_table + (t >> g.page_shift));
    if (page >= g.num_pages) return ~0ull;
    return (uint64_t)page * g.page_stride + (uint64_t)(t & g.page_mask) * g.token_stride;
  }
  return (uint64_t)t * g.token_stride;
}

// ---------------------------------------------------------------------------
// Walsh-Hadamard butterflies in Sylvester order, strides 1, 2, ..., 64 in that
// order.  A lane holds 32 consecutive channels (channel bits 0..4 in registers);
// channel bits 5 and 6 live in lane bits 0 and 1 of a group of four lanes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fwht_in_thread(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; i++) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
}

// Stride held across lanes: the lane whose bit is clear keeps a + b, the other a - b.
__device__ __forceinline__ void fwht_across_lanes(float (&v)[32], int lane_mask, bool upper) {
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const float o = __shfl_xor_sync(kFull, v[i], lane_mask);
    v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
  }
}

// Full 128-point transform of the row held by the 4 lanes (part = lane & 3).
__device__ __forceinline__ void fwht128(float (&v)[32], int part) {
  fwht_in_thread(v);
  fwht_across_lanes(v, 1, part & 1);
  fwht_across_lanes(v, 2, part & 2);
}

// Multiply by the +-1 signs of channels 32*part .. 32*part+31 (bit i of `bits`).
__device__ __forceinline__ void apply_signs(float (&v)[32], uint32_t bits) {
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ (((bits >> i) & 1u) << 31));
}

__device__ __forceinline__ void scale_all(float (&v)[32], float c) {
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __fmul_rn(v[i], c);
}

// ---------------------------------------------------------------------------
// Min-max quantization parameters: z = fp16 toward -inf of the minimum,
// s = fp16 toward +inf of RN((max - z) / (2^b - 1)); an infinite z or s saturates
// to +-65504 and raises the RANGE flag.  Returns meta = scale | zero << 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t saturate_f16(uint32_t h, uint32_t &flags) {
  if ((h & 0x7fffu) == 0x7c00u) {
    flags |= KVC_FLAG_RANGE;
    return (h & 0x8000u) | 0x7bffu;
  }
  return h;
}

// RN(w / (2^BITS - 1)) for a group's range w >= 0, by the quotient correction step
// of P. Markstein ("Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990): with c = RN(1/Q) and q = RN(w c)
// within one ulp of w / Q, the residual w - q Q is exact in one fma and RN(q + e c)
// is the correctly rounded quotient, barring underflow.  Where the quotient is
// below 2^-100 it may be off by an ulp, but every positive value there rounds up to
// the same binary16 scale (2^-24), so the scale is unchanged.  An infinite or NaN
// range takes w c, which is what the division gives.
template <int BITS>
__device__ __forceinline__ float range_div(float w) {
  constexpr float Q = (float)((1u << BITS) - 1u);
  constexpr float c = 1.0f / Q;  // correctly rounded at compile time
  const float q = __fmul_rn(w, c);
  const float e = __fmaf_rn(-q, Q, w);
  const float d = __fmaf_rn(e, c, q);
  return fabsf(w) <= 3.402823466e38f ? d : __fmul_rn(w, c);
}

template <int BITS>
__device__ __forceinline__ uint32_t quant_params(float mn, float mx, float &s, float &z, float &r,
                                                 uint32_t &flags) {
  mn = __fadd_rn(mn, 0.0f);  // a zero extreme counts as +0
  mx = __fadd_rn(mx, 0.0f);
  const uint32_t zb = saturate_f16(__half_as_ushort(__float2half_rd(mn)), flags);
  z = __half2float(__ushort_as_half((unsigned short)zb));
  const float w = __fsub_rn(mx, z);
  const float v = range_div<BITS>(w);
  const uint32_t sb = saturate_f16(__half_as_ushort(__float2half_ru(v)), flags);
  s = __half2float(__ushort_as_half((unsigned short)sb));
  r = s == 0.0f ? 0.0f : __frcp_rn(s);  // 0: every code of the group is 0
  return sb | (zb << 16);
}

// Code of y: clamp(rint_even(RN(RN(y - z) / s)), 0, 2^b - 1), 0 when s == 0.
// Fast path: p = RN(RN(y - z) * RN(1/s)) differs from the exact quotient d by at
// most 2^-15 for |d| < 256, and RN(d) from d by at most 2^-17; when p is more than
// 2^-14 away from every half-integer, rint(p) = rint(RN(d)).  Otherwise (about one
// element in 8000) the correctly rounded division decides.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float y, float z, float s, float r) {
  const float Qf = (float)((1u << BITS) - 1u);
  const float t = __fsub_rn(y, z);
  const float p = __fmul_rn(t, r);
  float k = rintf(p);
  if (!(fabsf(__fsub_rn(p, k)) < 0.49993896484375f)) k = rintf(__fdiv_rn(t, s));  // 0.5 - 2^-14
  k = fminf(fmaxf(k, 0.0f), Qf);
  return s == 0.0f ? 0u : (uint32_t)k;
}

// ---------------------------------------------------------------------------
// Packing: code i of a record occupies bits [i*b, i*b + b), least significant
// bit first; 32 codes fill BITS 32-bit words (little-endian bytes).
// ---------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ void pack32(const uint32_t (&q)[32], uint32_t (&w)[BITS]) {
#pragma unroll
  for (int j = 0; j < BITS; j++) w[j] = 0u;
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const int bit = i * BITS, wi = bit >> 5, sh = bit & 31;
    w[wi] |= q[i] << sh;
    if (sh + BITS > 32) w[wi + 1] |= q[i] >> (32 - sh);
  }
}

template <int BITS>
__device__ __forceinline__ void unpack32(const uint32_t (&w)[BITS], uint32_t (&q)[32]) {
  constexpr uint32_t M = (1u << BITS) - 1u;
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const int bit = i * BITS, wi = bit >> 5, sh = bit & 31;
    uint32_t c = w[wi] >> sh;
    if (sh + BITS > 32) c |= w[wi + 1] << (32 - sh);
    q[i] = c & M;
  }
}

// Store / load BITS words (4*BITS bytes) at a 4-byte aligned address; 16-byte
// vectors where the width allows it (4*BITS is 8, 12, 16 or 32 bytes).
template <int BITS>
__device__ __forceinline__ void store_words(uint8_t *dst, const uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (BITS == 8) {
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else if constexpr (BITS == 2) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int j = 0; j < BITS; j++) reinterpret_cast<uint32_t *>(dst)[j] = w[j];
  }
}

template <int BITS>
__device__ __forceinline__ void load_words(const uint8_t *src, uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {
    const uint4 a = *reinterpret_cast<const uint4 *>(src);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else if constexpr (BITS == 8) {
    const uint4 a = reinterpret_cast<const uint4 *>(src)[0], b = reinterpret_cast<const uint4 *>(src)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if constexpr (BITS == 2) {
    const uint2 a = *reinterpret_cast<const uint2 *>(src);
    w[0] = a.x; w[1] = a.y;
  } else {
#pragma unroll
    for (int j = 0; j < BITS; j++) w[j] = reinterpret_cast<const uint32_t *>(src)[j];
  }
}

// ---------------------------------------------------------------------------
// Key smoothing: centre = fp16 RN of the midrange, exponent e = smallest integer
// with 2^e >= max |x - centre| (0 for 0), clamped to [-126, 127].
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ceil_log2_pos(float r) {
  if (!(r > 0.0f)) return 0;
  const uint32_t u = __float_as_uint(r);
  const int ex = (int)((u >> 23) & 0xffu);
  if (ex == 0xff) return 127;
  if (ex == 0) return -126;  // subnormal: below 2^-126
  const int e = ex - 127 + ((u & 0x7fffffu) ? 1 : 0);
  return e > 127 ? 127 : e;
}

// 2^k as binary32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2i(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void smooth_params(float mn, float mx, float &mu, float &inv, uint32_t &mu_bits,
                                              int &e, uint32_t &flags) {
  mn = __fadd_rn(mn, 0.0f);  // a zero extreme counts as +0
  mx = __fadd_rn(mx, 0.0f);
  const float mid = __fmul_rn(__fadd_rn(mn, mx), 0.5f);
  mu_bits = saturate_f16(__half_as_ushort(__float2half_rn(mid)), flags);
  mu = __half2float(__ushort_as_half((unsigned short)mu_bits));
  const float r = fmaxf(fabsf(__fsub_rn(mx, mu)), fabsf(__fsub_rn(mn, mu)));
  e = ceil_log2_pos(r);
  inv = pow2i(-e);
}

__device__ __forceinline__ bool all_finite8(const float *x) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 8; i++) ok &= (fabsf(x[i]) <= 3.402823466e38f);
  return ok;
}

// ---------------------------------------------------------------------------
// NaN-propagating min / max (PTX min.NaN / max.NaN, two or three operands): a
// NaN or infinity anywhere in a group reaches its statistics, so the finite
// check costs one test per group instead of one per element.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fmin_n(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmax_n(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmin3_n(float a, float b, float c) {
  float d;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3_n(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Element-wise minimum / maximum of two packed 16-bit pairs (bf16x2 or f16x2),
// NaN-propagating; exact, like the binary32 versions on the widened values.
template <bool BF16>
__device__ __forceinline__ uint32_t pmin2_n(uint32_t a, uint32_t b) {
  uint32_t d;
  if (BF16) asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <bool BF16>
__device__ __forceinline__ uint32_t pmax2_n(uint32_t a, uint32_t b) {
  uint32_t d;
  if (BF16) asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ bool finite2(float a, float b) { return fabsf(a) <= 3.402823466e38f && fabsf(b) <= 3.402823466e38f; }

// ---------------------------------------------------------------------------
// Packed binary32 pairs (Blackwell f32x2): every lane of a pair is rounded on its
// own, exactly as the scalar operation.  a - b is written fma(b, -1, a), which is
// the single rounding of the exact difference.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 bcast2(float a) { return make_float2(a, a); }

// ---------------------------------------------------------------------------
// Branch-free codes for a pair, from the correctly rounded quotient.  With
// t = RN(y - z) >= 0, r = RN(1/s) and q = RN(t r) (within one ulp of t / s), the
// residual e = t - q s is exact in one fma and RN(q + e r) is the correctly
// rounded t / s: the quotient correction step of P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Develop. 34(1), 1990.  The step assumes nothing underflows; a quotient that can
// round to code 1 or more has t >= s / 2 >= 2^-25 and a residual far above
// 2^-126, and a smaller one gives code 0 either way.  rint comes from adding
// 1.5 * 2^23 (round half to even); the code is the low mantissa bits of the sum.
// r = 0 when s = 0 makes every code 0, as the rule says.  Valid for finite
// y >= z and a finite s: a group with a saturated or non-finite parameter, where
// the rule's clamp is needed, takes qexact instead.
// ---------------------------------------------------------------------------
constexpr float kRintMagic = 12582912.0f;  // 1.5 * 2^23

// The corrected quotients t / s of a pair (r2 = RN(1/s), ns2 = -s in both halves).
__device__ __forceinline__ float2 qdiv2(float2 t, float2 r2, float2 ns2) {
  const float2 q = mul2(t, r2);
  const float2 e = __ffma2_rn(q, ns2, t);
  return __ffma2_rn(e, r2, q);
}

// Returns the sums of a pair; the code of a half is its low BITS bits.
__device__ __forceinline__ float2 qsum2(float2 y, float2 z2, float2 r2, float2 ns2) {
  return add2(qdiv2(sub2(y, z2), r2, ns2), bcast2(kRintMagic));
}

// The exact rule: clamp(rint_even(RN(RN(y - z) / s)), 0, 2^BITS - 1), 0 when s == 0.
template <int BITS>
__device__ __forceinline__ uint32_t qexact(float y, float z, float s) {
  const float Qf = (float)((1u << BITS) - 1u);
  if (s == 0.0f) return 0u;
  const float k = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(y, z), s)), 0.0f), Qf);
  return (uint32_t)k;
}

// Code bits of a qsum2 sum, already masked to BITS.
template <int BITS>
__device__ __forceinline__ uint32_t code_of(float u) { return __float_as_uint(u) & ((1u << BITS) - 1u); }

}  // namespace kvc
