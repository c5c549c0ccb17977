// kvc_quant_kernels.cuh -- fused transform + quantize + pack (encode) and fused
// reconstruction (decode) for one KV tensor of every layer.  Kernel templates
// only: kvc_quant.cu instantiates the format-v1 kernels, kvc_quant_v2.cu the
// ones with the token delta and per-(layer, head) widths (format v2).
//
// "Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
// Serving", §4.1: each KV tile is loaded once, the randomized Hadamard transform,
// the quantization statistics and the low-bit conversion run on chip, and the
// codes go straight into the all-layer payload; reconstruction dequantizes,
// applies the inverse Hadamard transform, normalization and sign restoration and
// writes only the final KV.  Key smoothing (a per-channel affine normalization,
// "KVServe" §5.1 transformer stage) is fused the same way.
//
// Two kernel shapes:
//  * rows  -- groups over channels, no smoothing (the value default).  A warp owns
//    16 rows (token, head) at a time, 2 lanes per row, 64 channels per lane; the
//    Hadamard butterflies run in registers (strides 1..32) and across the lane
//    pair (stride 64).  The decoder assembles its output rows in shared memory
//    and writes each with one bulk copy.
//  * key tile -- groups over tokens (the key default, kvc_enc_ktile /
//    kvc_dec_ktile).  A CTA owns a (layer, head, 128-token) tile in shared memory:
//    per-channel smoothing statistics over tokens, the row-wise Hadamard pass,
//    then a column pass that quantizes and packs each channel's token group (and
//    the reverse for decoding).
//  * tile  -- smoothing with groups over channels (kvc_enc_tile / kvc_dec_tile),
//    the general layout for the less common profiles.
#pragma once
#include <cuda_runtime.h>

#include <type_traits>

#include "kvc_device.cuh"

namespace kvc {

// The width table is a kernel parameter of the mixed-width kernels only.
struct NoWidths {
  uint32_t unused;
};
template <bool MIXED>
using WidthsArg = typename std::conditional<MIXED, WidthTable, NoWidths>::type;
template <bool MIXED>
__device__ __forceinline__ uint32_t width_of(const WidthsArg<MIXED> &W, uint32_t lh) {
  if constexpr (MIXED) return (uint32_t)W.wsum[lh + 1] - (uint32_t)W.wsum[lh];
  else return 0u;
}

constexpr int kThreads = 256;
constexpr int kTS = 144;  // floats per shared-memory tile row (128 + 16: conflict-free row and column access)
constexpr size_t kTileSmem = (size_t)(128 * kTS + 2 * 8 * 128 + 3 * 128) * sizeof(float);

// ---------------------------------------------------------------------------
// rows: encode.  Two lanes own a row (token, head): lane half h holds channels
// 64h .. 64h+63 as 32 packed pairs.  Butterfly stride 1 runs inside each pair,
// strides 2..32 between pairs, stride 64 across the two lanes; a warp handles 16
// rows per step.  Groups of 32 or 64 channels are lane-local, groups of 128 take
// one shuffle.  Codes come from the branch-free pair quantizer; a warp takes the
// exact division only when one of its lanes met a near-tie.
// ---------------------------------------------------------------------------
// Sign masks for the raw element pairs: bit 15 / 31 set where the channel's sign is -1.
__device__ __forceinline__ uint32_t pair_sign_mask(uint32_t sbits, int j) {
  return (((sbits >> j) & 1u) << 15) | (((sbits >> (j + 1)) & 1u) << 31);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16_q(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit_q() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_q() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float2 unpack_pair(uint32_t u, bool bf16) {
  if (bf16) return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}

__device__ __forceinline__ uint32_t pack_pair(float2 v, bool bf16) {
  if (bf16) return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
  return (uint32_t)__half_as_ushort(__float2half_rn(v.x)) | ((uint32_t)__half_as_ushort(__float2half_rn(v.y)) << 16);
}

// In-lane butterflies of 64 channels held as 32 pairs: stride 1 within pairs, 2..32 between pairs.
__device__ __forceinline__ void fwht64_pairs(float2 (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const float a = w[i].x, b = w[i].y;
    w[i] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
  }
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; i++)
      if ((i & h) == 0) {
        const float2 a = w[i], b = w[i + h];
        w[i] = add2(a, b);
        w[i + h] = sub2(a, b);
      }
  }
}

// Insert code c (low BITS bits of c, higher bits ignored) as field `idx` of a
// little-endian bit string held in 32-bit words.
template <int BITS, int NW>
__device__ __forceinline__ void put_code(uint32_t (&w)[NW], int idx, uint32_t c) {
  constexpr uint32_t M = (1u << BITS) - 1u;
  const int bit = idx * BITS, wi = bit >> 5, sh = bit & 31;
  w[wi] |= (c << sh) & (M << sh);
  if (sh + BITS > 32) w[wi + 1] |= (c & M) >> (32 - sh);
}

// 32 codes (BITS each, LSB first) -> 16 float pairs, exactly.
template <int BITS>
__device__ __forceinline__ void codes_to_f2(const uint32_t (&w)[BITS], float2 (&q)[16]) {
  constexpr uint32_t kE = 0x4B000000u;  // the bits of 2^23
  uint32_t b[32];
  if constexpr (BITS == 4) {
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint32_t lo = w[k] & 0x0F0F0F0Fu, hi = (w[k] >> 4) & 0x0F0F0F0Fu;  // byte j: codes 8k+2j, 8k+2j+1
#pragma unroll
      for (int j = 0; j < 4; j++) {
        b[8 * k + 2 * j] = __byte_perm(lo, kE, 0x7440u | j);
        b[8 * k + 2 * j + 1] = __byte_perm(hi, kE, 0x7440u | j);
      }
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int k = 0; k < 8; k++)
#pragma unroll
      for (int j = 0; j < 4; j++) b[4 * k + j] = __byte_perm(w[k], kE, 0x7440u | j);
  } else if constexpr (BITS == 2) {
#pragma unroll
    for (int k = 0; k < 2; k++)
#pragma unroll
      for (int f = 0; f < 4; f++) {
        const uint32_t m = (w[k] >> (2 * f)) & 0x03030303u;  // byte j: code 16k + 4j + f
#pragma unroll
        for (int j = 0; j < 4; j++) b[16 * k + 4 * j + f] = __byte_perm(m, kE, 0x7440u | j);
      }
  } else {
    uint32_t c[32];
    unpack32<BITS>(w, c);
#pragma unroll
    for (int i = 0; i < 32; i++) b[i] = c[i] | kE;
  }
  const float2 e2 = bcast2(8388608.0f);
#pragma unroll
  for (int i = 0; i < 16; i++) q[i] = sub2(make_float2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1])), e2);
}

// Codes of 32 qsum2 sums (bits 0x4B400000 + code, the code in the low byte) into
// BITS words, LSB first.  2 and 4 bits: the codes of a byte are gathered with
// integer multiply-adds (the magic's low byte is 0, so the low byte of
// u1 * 2^BITS + u0 is code0 | code1 << BITS), bytes into words by byte_perm.
template <int BITS>
__device__ __forceinline__ void pack_sums32(const uint32_t (&u)[32], uint32_t (&cw)[BITS]) {
  if constexpr (BITS == 4 || BITS == 2 || BITS == 8) {
    constexpr int per_byte = 8 / BITS;
    uint32_t b[4 * BITS];  // one byte (in the low 8 bits) per 8 / BITS codes
#pragma unroll
    for (int i = 0; i < 4 * BITS; i++) {
      uint32_t x = u[per_byte * i + per_byte - 1];
#pragma unroll
      for (int j = per_byte - 2; j >= 0; j--) x = x * (1u << BITS) + u[per_byte * i + j];
      b[i] = x;
    }
#pragma unroll
    for (int w = 0; w < BITS; w++)
      cw[w] = __byte_perm(__byte_perm(b[4 * w], b[4 * w + 1], 0x0040), __byte_perm(b[4 * w + 2], b[4 * w + 3], 0x0040),
                          0x5410);
  } else {
#pragma unroll
    for (int i = 0; i < BITS; i++) cw[i] = 0u;
#pragma unroll
    for (int i = 0; i < 32; i++) put_code<BITS>(cw, i, u[i]);
  }
}

// Decode with codes read in place: the address of the code unit at byte `rel` of
// the code section (a unit never crosses a chunk boundary where this is enabled).
__device__ __forceinline__ const uint8_t *code_unit(const QuantParams &P, size_t rel) {
  if (P.in_lo < P.in_hi) {
    const uint64_t o = P.codes_off + rel, c = o >> P.chunk_shift;
    if (c >= P.in_lo && c < P.in_hi)
      return reinterpret_cast<const uint8_t *>(__ldg(reinterpret_cast<const unsigned long long *>(P.src_of) + c)) +
             (o & ((1ull << P.chunk_shift) - 1u));
  }
  return P.codes + rel;
}

// Where a value row's codes go.  Uniform width: record row R = (l T + t) H + h at
// R * 16 BITS.  Per-(layer, head) widths: layer l's rows start at 16 T wsum[lH],
// token t's row at + 16 t (wsum[(l+1)H] - wsum[lH]), head h at + 16 (wsum[lH+h] - wsum[lH]).
template <int BITS, bool MIXED>
__device__ __forceinline__ size_t row_code_offset(const WidthsArg<MIXED> &W, uint32_t T, uint32_t H, uint32_t l,
                                                  uint32_t t, uint32_t h, uint32_t R) {
  if constexpr (MIXED) {
    const uint32_t a = W.wsum[l * H], e = W.wsum[(l + 1) * H];
    return 16 * ((size_t)T * a + (size_t)t * (e - a) + (W.wsum[l * H + h] - a));
  } else {
    (void)W; (void)T; (void)H; (void)l; (void)t; (void)h;
    return (size_t)R * (kHeadDim * BITS / 8);
  }
}

// One step of the rows encoder for the 16 rows of a warp: lane pair (2 rsub,
// 2 rsub + 1) quantizes row (l, t, h) if `valid`; R = (l T + t) H + h indexes the
// metadata; `cdst` is the row's code record start.  Every lane of the warp runs it.
template <int BITS, bool HAD, bool BF16, bool DELTA>
__device__ __forceinline__ void enc_row(const QuantParams &P, const uint32_t (*smask)[32], int half, bool valid,
                                        uint32_t l, uint32_t t, uint32_t h, uint32_t R, uint8_t *cdst,
                                        uint32_t &flags) {
  constexpr bool bf16 = BF16;
  const uint32_t G = P.group;
  const float sg = half ? -1.0f : 1.0f;  // stride 64: lower lane a + b, upper lane a - b = -b + a
  float2 w[32];
  {
    uint4 q[8];
#pragma unroll
    for (int j = 0; j < 8; j++) q[j] = make_uint4(0u, 0u, 0u, 0u);
    const uint8_t *abase = nullptr;  // token delta: the block's anchor row (first token of the 128-token block)
    if (valid) {
      const uint64_t ro = row_offset(P.g, t);
      if (ro == ~0ull) {
        flags |= KVC_FLAG_BAD_PAGE;
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.layers[l]) + ro +
                                                           (size_t)(h * kHeadDim + 64 * half) * 2);
#pragma unroll
        for (int j = 0; j < 4; j++) ld_global32_nc(src + 2 * j, q[2 * j], q[2 * j + 1]);
      }
      if constexpr (DELTA) {
        const uint64_t ao = row_offset(P.g, t & ~(uint32_t)(kSmoothBlock - 1));
        if (ao == ~0ull) flags |= KVC_FLAG_BAD_PAGE;
        else abase = static_cast<const uint8_t *>(P.layers[l]) + ao + (size_t)(h * kHeadDim + 64 * half) * 2;
      }
    }
    uint4 av[DELTA ? 8 : 1];  // token delta: the anchor half row, loaded beside the row itself
    if constexpr (DELTA) {
#pragma unroll
      for (int j = 0; j < 8; j++) av[j] = make_uint4(0u, 0u, 0u, 0u);
      if (abase) {
#pragma unroll
        for (int j = 0; j < 4; j++)
          ld_global32_nc(reinterpret_cast<const uint4 *>(abase) + 2 * j, av[2 * j], av[2 * j + 1]);
      }
    }
    if constexpr (DELTA) {
      if (valid && (t & (kSmoothBlock - 1)) == 0) {  // the anchor row keeps its element bits
        uint4 *cell = reinterpret_cast<uint4 *>(
            P.anchors + ((((size_t)l * P.g.H + h) * P.n_sb + (t >> 7)) * kHeadDim + 64 * half) * 2);
#pragma unroll
        for (int j = 0; j < 8; j++) cell[j] = q[j];
      }
    }
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint32_t r4[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
      uint32_t a4[4] = {0u, 0u, 0u, 0u};
      if constexpr (DELTA) {
        a4[0] = av[j].x; a4[1] = av[j].y; a4[2] = av[j].z; a4[3] = av[j].w;
      }
#pragma unroll
      for (int e = 0; e < 4; e++) {
        if (HAD) r4[e] ^= smask[half][4 * j + e];
        w[4 * j + e] = unpack_pair(r4[e], bf16);
        if constexpr (DELTA) {  // sign-flipped row minus sign-flipped anchor = sign * (row - anchor), exactly
          if (HAD) a4[e] ^= smask[half][4 * j + e];
          w[4 * j + e] = sub2(w[4 * j + e], unpack_pair(a4[e], bf16));
        }
      }
    }
  }
  if (HAD) {
    fwht64_pairs(w);
    const float2 c2 = bcast2(hadamard_scale()), sg2 = bcast2(sg);
#pragma unroll
    for (int i = 0; i < 32; i++) {
      const float2 o = make_float2(__shfl_xor_sync(kFull, w[i].x, 1), __shfl_xor_sync(kFull, w[i].y, 1));
      w[i] = mul2(__ffma2_rn(w[i], sg2, o), c2);
    }
  }
  // group statistics (NaN-propagating): G = 32 -> two groups per lane, 64 -> one, 128 -> lane pair
  float mn0 = fmin_n(w[0].x, w[0].y), mx0 = fmax_n(w[0].x, w[0].y);
  float mn1 = fmin_n(w[16].x, w[16].y), mx1 = fmax_n(w[16].x, w[16].y);
#pragma unroll
  for (int i = 1; i < 16; i++) {
    mn0 = fmin3_n(mn0, w[i].x, w[i].y);
    mx0 = fmax3_n(mx0, w[i].x, w[i].y);
    mn1 = fmin3_n(mn1, w[16 + i].x, w[16 + i].y);
    mx1 = fmax3_n(mx1, w[16 + i].x, w[16 + i].y);
  }
  if (G >= 64) {
    mn0 = mn1 = fmin_n(mn0, mn1);
    mx0 = mx1 = fmax_n(mx0, mx1);
  }
  if (G == 128) {
    mn0 = mn1 = fmin_n(mn0, __shfl_xor_sync(kFull, mn0, 1));
    mx0 = mx1 = fmax_n(mx0, __shfl_xor_sync(kFull, mx0, 1));
  }
  if (valid && !finite2(mn0, mx0)) flags |= KVC_FLAG_NONFINITE;
  if (valid && !finite2(mn1, mx1)) flags |= KVC_FLAG_NONFINITE;
  float s0, z0, r0, s1, z1, r1;
  uint32_t f0 = 0, f1 = 0, meta1;
  const uint32_t meta0 = quant_params<BITS>(mn0, mx0, s0, z0, r0, f0);
  if (G == 32) {
    meta1 = quant_params<BITS>(mn1, mx1, s1, z1, r1, f1);
  } else {  // one group per lane: the second half shares the first half's parameters
    meta1 = meta0;
    s1 = s0;
    z1 = z0;
    r1 = r0;
  }
  uint32_t wds[2 * BITS];
  {
    const float2 za = bcast2(z0), ra = bcast2(r0), zb = bcast2(z1), rb = bcast2(r1);
    const float2 na = bcast2(-s0), nb = bcast2(-s1);
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {  // codes 32 hh .. 32 hh + 31
      uint32_t u[32];
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const float2 s2 = qsum2(w[16 * hh + i], hh ? zb : za, hh ? rb : ra, hh ? nb : na);
        u[2 * i] = __float_as_uint(s2.x);
        u[2 * i + 1] = __float_as_uint(s2.y);
      }
      uint32_t cw[BITS];
      pack_sums32<BITS>(u, cw);
#pragma unroll
      for (int k = 0; k < BITS; k++) wds[hh * BITS + k] = cw[k];
    }
  }
  // a saturated or non-finite group takes the exact rule
  const bool bad = f0 != 0 || f1 != 0 || !finite2(mn0, mx0) || !finite2(mn1, mx1);
  if (__any_sync(kFull, bad)) {
    if (bad) {
#pragma unroll
      for (int j = 0; j < 2 * BITS; j++) wds[j] = 0u;
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const float z = i < 16 ? z0 : z1, sc = i < 16 ? s0 : s1;
        put_code<BITS>(wds, 2 * i, qexact<BITS>(w[i].x, z, sc));
        put_code<BITS>(wds, 2 * i + 1, qexact<BITS>(w[i].y, z, sc));
      }
    }
  }
  if (valid) {
    flags |= f0 | f1;
    uint8_t *dst = cdst + 8 * BITS * half;
    if constexpr ((2 * BITS) % 4 == 0) {
#pragma unroll
      for (int j = 0; j < 2 * BITS; j += 4)
        *reinterpret_cast<uint4 *>(dst + 4 * j) = make_uint4(wds[j], wds[j + 1], wds[j + 2], wds[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 2 * BITS; j += 2) *reinterpret_cast<uint2 *>(dst + 4 * j) = make_uint2(wds[j], wds[j + 1]);
    }
    uint32_t *mp = reinterpret_cast<uint32_t *>(P.meta);
    if (G == 32) *reinterpret_cast<uint2 *>(mp + (size_t)R * 4 + 2 * half) = make_uint2(meta0, meta1);
    else if (G == 64) mp[(size_t)R * 2 + half] = meta0;
    else if (half == 0) mp[R] = meta0;
  }
}

// Row position of a lane, advanced by a fixed number of rows without divisions.
// Uniform width: rows in (layer, token, head) order (head fastest).  Per-(layer,
// head) widths: (layer, head, token) order, so that the 16 rows of a warp step
// share their head and hence their width (except where a head's rows end).
struct RowPos {
  uint32_t a, b, l;  // uniform: a = h, b = t; mixed: a = t, b = h
  __device__ __forceinline__ void init(uint32_t R, uint32_t na, uint32_t nb) {
    a = R % na;
    b = (R / na) % nb;
    l = R / na / nb;
  }
  __device__ __forceinline__ void advance(uint32_t da, uint32_t db, uint32_t dl, uint32_t na, uint32_t nb) {
    a += da;
    uint32_t c = a >= na;
    a -= c ? na : 0u;
    b += db + c;
    c = b >= nb;
    b -= c ? nb : 0u;
    l += dl + c;
  }
};

// ---------------------------------------------------------------------------
// rows: encode.  Two lanes own a row (token, head): lane half h holds channels
// 64h .. 64h+63 as 32 packed pairs (see enc_row).
// ---------------------------------------------------------------------------
template <int BITS, bool HAD, bool BF16, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kThreads, 2) kvc_enc_rows(const QuantParams P, const __grid_constant__ WidthsArg<MIXED> W) {
  __shared__ uint32_t smask[2][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane & 1, rsub = lane >> 1;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  const uint32_t n_it = (NR + 15) / 16;
  if (HAD && threadIdx.x < 64) {
    const int hh = threadIdx.x >> 5, j = threadIdx.x & 31;  // pair j of half hh: channels 64hh + 2j, +1
    smask[hh][j] = pair_sign_mask(P.sign[2 * hh + (j >> 4)], (2 * j) & 31);
  }
  __syncthreads();
  uint32_t flags = 0;

  const uint32_t na = MIXED ? T : H, nb = MIXED ? H : T;
  const uint32_t it0 = blockIdx.x * (kThreads / 32) + warp, it_step = gridDim.x * (kThreads / 32);
  const uint32_t R0 = it0 * 16 + rsub, dR = it_step * 16;
  RowPos pos;
  pos.init(R0, na, nb);
  const uint32_t da = dR % na, db = (dR / na) % nb, dl = dR / na / nb;
  for (uint32_t it = it0; it < n_it; it += it_step) {
    const bool valid = it * 16 + rsub < NR;
    const uint32_t l = pos.l, t = MIXED ? pos.a : pos.b, h = MIXED ? pos.b : pos.a;
    pos.advance(da, db, dl, na, nb);
    const uint32_t R = (l * T + t) * H + h;
    if constexpr (MIXED) {
      const uint32_t b = valid ? width_of<MIXED>(W, l * H + h) : 0u;
      uint8_t *cdst = valid ? P.codes + row_code_offset<0, MIXED>(W, T, H, l, t, h, R) : P.codes;
      if (__any_sync(kFull, b == 2)) enc_row<2, HAD, BF16, DELTA>(P, smask, half, b == 2, l, t, h, R, cdst, flags);
      if (__any_sync(kFull, b == 3)) enc_row<3, HAD, BF16, DELTA>(P, smask, half, b == 3, l, t, h, R, cdst, flags);
      if (__any_sync(kFull, b == 4)) enc_row<4, HAD, BF16, DELTA>(P, smask, half, b == 4, l, t, h, R, cdst, flags);
      if (__any_sync(kFull, b == 8)) enc_row<8, HAD, BF16, DELTA>(P, smask, half, b == 8, l, t, h, R, cdst, flags);
    } else {
      enc_row<BITS, HAD, BF16, DELTA>(P, smask, half, valid, l, t, h, R,
                                      P.codes + row_code_offset<BITS, MIXED>(W, T, H, l, t, h, R), flags);
    }
  }
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// rows: decode
// ---------------------------------------------------------------------------
constexpr size_t kDecRowsSmem = (size_t)(kThreads / 32) * 16 * 512;  // the row slots of kvc_dec_rows
// Input staging of kvc_dec_rows (one code width): per warp two buffers of 16 rows'
// codes (16 BITS bytes each) and metadata (up to 4 words each).
__host__ __device__ constexpr size_t dec_rows_stage_bytes(int bits) { return (size_t)16 * (16 * bits + 16); }
constexpr size_t dec_rows_smem(int bits) { return kDecRowsSmem + (size_t)(kThreads / 32) * 2 * dec_rows_stage_bytes(bits); }

// One step of the rows decoder for the 16 rows of a warp: lanes rsub and
// rsub + 16 reconstruct row (l, t, h) if `valid` (codes at `csrc`, metadata by R)
// and send it out through the row's slot by one bulk copy.  Every lane runs it.
// Codes at `csrc` and metadata words at `mrow`: global memory, or (STAGED) this
// warp's shared staging buffer.
template <int BITS, bool HAD, bool BF16, bool DELTA, bool STAGED = false>
__device__ __forceinline__ void dec_row(const QuantParams &P, const uint32_t (*fsign)[64], uint4 *oslot, int half,
                                        bool valid, uint32_t l, uint32_t t, uint32_t h, uint32_t R,
                                        const uint8_t *csrc, const uint32_t *mrow, uint32_t &flags) {
  const uint32_t G = P.group;
  const float sg = half ? -1.0f : 1.0f;  // stride 64: lower lane a + b, upper lane a - b = -b + a
  float2 w[32];  // channels 64 half + 2i, +1
  {
    uint32_t cw[2 * BITS];
    uint32_t m0 = 0, m1 = 0;  // group metadata of channels 64 half + 0..31 / 32..63
#pragma unroll
    for (int k = 0; k < 2 * BITS; k++) cw[k] = 0u;
    if (valid) {
      const uint8_t *src = csrc + 8 * BITS * half;
      if constexpr ((2 * BITS) % 4 == 0) {
#pragma unroll
        for (int k = 0; k < 2 * BITS; k += 4) {
          const uint4 *p4 = reinterpret_cast<const uint4 *>(src + 4 * k);
          const uint4 a = STAGED ? *p4 : __ldg(p4);
          cw[k] = a.x; cw[k + 1] = a.y; cw[k + 2] = a.z; cw[k + 3] = a.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 2 * BITS; k += 2) {
          const uint2 *p2 = reinterpret_cast<const uint2 *>(src + 4 * k);
          const uint2 a = STAGED ? *p2 : __ldg(p2);
          cw[k] = a.x; cw[k + 1] = a.y;
        }
      }
      if (G == 32) {
        const uint2 *p2 = reinterpret_cast<const uint2 *>(mrow + 2 * half);
        const uint2 mm = STAGED ? *p2 : __ldg(p2);
        m0 = mm.x;
        m1 = mm.y;
      } else {
        const uint32_t *p1 = mrow + (G == 64 ? half : 0);
        m0 = m1 = STAGED ? *p1 : __ldg(p1);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {  // codes 32 hh .. 32 hh + 31
      uint32_t wv[BITS];
#pragma unroll
      for (int k = 0; k < BITS; k++) wv[k] = cw[hh * BITS + k];
      float2 qf[16];
      codes_to_f2<BITS>(wv, qf);
      const uint32_t m = hh ? m1 : m0;
      const float2 s2 = bcast2(__half2float(__ushort_as_half((unsigned short)(m & 0xffffu))));
      const float2 z2 = bcast2(__half2float(__ushort_as_half((unsigned short)(m >> 16))));
#pragma unroll
      for (int i = 0; i < 16; i++) w[16 * hh + i] = __ffma2_rn(qf[i], s2, z2);
    }
  }
  if (HAD) {
    fwht64_pairs(w);
    const float2 c2 = bcast2(hadamard_scale()), sg2 = bcast2(sg);
#pragma unroll
    for (int i = 0; i < 32; i++) {
      const float2 o = make_float2(__shfl_xor_sync(kFull, w[i].x, 16), __shfl_xor_sync(kFull, w[i].y, 16));
      w[i] = mul2(__ffma2_rn(w[i], sg2, o), c2);
    }
    const uint4 *fs = reinterpret_cast<const uint4 *>(fsign[half]);
#pragma unroll
    for (int k = 0; k < 16; k++) {  // signs of channels 4k .. 4k + 3 of this half
      const uint4 m = fs[k];
      w[2 * k].x = __uint_as_float(__float_as_uint(w[2 * k].x) ^ m.x);
      w[2 * k].y = __uint_as_float(__float_as_uint(w[2 * k].y) ^ m.y);
      w[2 * k + 1].x = __uint_as_float(__float_as_uint(w[2 * k + 1].x) ^ m.z);
      w[2 * k + 1].y = __uint_as_float(__float_as_uint(w[2 * k + 1].y) ^ m.w);
    }
  }
  if constexpr (DELTA) {  // plus the block's anchor row (element bits in the payload)
    if (valid) {
      const uint4 *ac = reinterpret_cast<const uint4 *>(
          P.anchors + ((((size_t)l * P.g.H + h) * P.n_sb + (t >> 7)) * kHeadDim + 64 * half) * 2);
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const uint4 a = __ldg(ac + j);
        const uint32_t a4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; e++) w[4 * j + e] = add2(w[4 * j + e], unpack_pair(a4[e], BF16));
      }
    }
  }
  bool put = false;
  uint8_t *dst = nullptr;
  if (valid) {
    const uint64_t ro = row_offset(P.g, t);
    if (ro == ~0ull) {
      flags |= KVC_FLAG_BAD_PAGE;
    } else {
      put = true;
      dst = static_cast<uint8_t *>(P.layers[l]) + ro + (size_t)h * kHeadDim * 2;
    }
  }
  // the previous row copy from this slot has read it
  if (half == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncwarp();
  if (put) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      uint32_t u[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const float2 x = w[4 * k + e];
        if (BF16) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(x.x, x.y);
          u[e] = *reinterpret_cast<const uint32_t *>(&b2);
        } else {
          const __half2 h2 = __floats2half2_rn(x.x, x.y);
          u[e] = *reinterpret_cast<const uint32_t *>(&h2);
        }
      }
      oslot[k] = make_uint4(u[0], u[1], u[2], u[3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stores above before the async read
  }
  __syncwarp();
  if (put && half == 0) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 256;" ::"l"(dst), "r"(smem_u32(oslot))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
}

template <int BITS, bool HAD, bool BF16, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kThreads, 2) kvc_dec_rows(const QuantParams P, const __grid_constant__ WidthsArg<MIXED> W) {
  if (P.check_corrupt && (*(volatile uint32_t *)P.status & KVC_FLAG_CORRUPT)) return;
  __shared__ __align__(16) uint32_t fsign[2][64];  // bit 31 set where channel 64 half + c has Hadamard sign -1
  extern __shared__ uint4 rows_out[];  // per warp 16 row slots of 512 B
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, rsub = lane & 15;  // lane: channels 64 half .. 64 half + 63 of row rsub
  // row rsub is assembled 16 (rsub % 8) bytes into its slot (the 8 rows of a
  // 16-byte store phase then sit in 8 distinct bank groups) and leaves by one
  // 256-byte bulk copy
  uint4 *const oslot = rows_out + (warp * 16 + rsub) * 32 + (rsub & 7) + 8 * half;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  const uint32_t n_it = (NR + 15) / 16;
  if (HAD && threadIdx.x < 128) {
    const int c = threadIdx.x;
    fsign[c >> 6][c & 63] = ((P.sign[c >> 5] >> (c & 31)) & 1u) << 31;
  }
  __syncthreads();
  uint32_t flags = 0;

  // rows in (layer, token, head) order, or (layer, head, token) with per-head widths
  const uint32_t na = MIXED ? T : H, nb = MIXED ? H : T;
  const uint32_t it0 = blockIdx.x * (kThreads / 32) + warp, it_step = gridDim.x * (kThreads / 32);
  const uint32_t R0 = it0 * 16 + rsub, dR = it_step * 16;
  RowPos pos;
  pos.init(R0, na, nb);
  const uint32_t da = dR % na, db = (dR / na) % nb, dl = dR / na / nb;
  if constexpr (MIXED) {
    for (uint32_t it = it0; it < n_it; it += it_step) {
      const bool valid = it * 16 + rsub < NR;
      const uint32_t l = pos.l, t = pos.a, h = pos.b;
      pos.advance(da, db, dl, na, nb);
      const uint32_t R = (l * T + t) * H + h;
      const uint32_t b = valid ? width_of<MIXED>(W, l * H + h) : 0u;
      const uint8_t *csrc = valid ? P.codes + row_code_offset<0, MIXED>(W, T, H, l, t, h, R) : P.codes;
      const uint32_t *mrow = reinterpret_cast<const uint32_t *>(P.meta) + (valid ? (size_t)R * (kHeadDim / P.group) : 0);
      if (__any_sync(kFull, b == 2)) dec_row<2, HAD, BF16, DELTA>(P, fsign, oslot, half, b == 2, l, t, h, R, csrc, mrow, flags);
      if (__any_sync(kFull, b == 3)) dec_row<3, HAD, BF16, DELTA>(P, fsign, oslot, half, b == 3, l, t, h, R, csrc, mrow, flags);
      if (__any_sync(kFull, b == 4)) dec_row<4, HAD, BF16, DELTA>(P, fsign, oslot, half, b == 4, l, t, h, R, csrc, mrow, flags);
      if (__any_sync(kFull, b == 8)) dec_row<8, HAD, BF16, DELTA>(P, fsign, oslot, half, b == 8, l, t, h, R, csrc, mrow, flags);
    }
  } else {
    // One code width: a warp step's 16 rows are consecutive records, so their codes
    // (16 x 16 BITS bytes) and metadata words are two contiguous runs.  They are
    // copied into this warp's staging buffer one step ahead (cp.async), so the
    // loads of step k + 1 are in flight while step k is reconstructed.
    constexpr uint32_t kStage = (uint32_t)dec_rows_stage_bytes(BITS);
    uint8_t *stage0 = reinterpret_cast<uint8_t *>(rows_out) + kDecRowsSmem + (size_t)warp * 2 * kStage;
    const uint32_t wpr = kHeadDim / P.group;  // metadata words per row
    // the codes of step itn's 16 rows: 256 BITS bytes, one unit for code_unit
    auto codes_of = [&](uint32_t itn) { return code_unit(P, (size_t)itn * (256 * BITS)); };
    auto issue = [&](uint32_t itn, const uint8_t *cg, uint8_t *buf) {
      const uint32_t r0 = itn * 16;
      const uint32_t nrow = NR - r0 < 16u ? NR - r0 : 16u;
      for (uint32_t u = lane; u < nrow * BITS; u += 32)  // 16-byte units, BITS per row
        cp_async16_q(buf + 16 * u, cg + 16 * (size_t)u);
      const uint32_t *mg = reinterpret_cast<const uint32_t *>(P.meta) + (size_t)r0 * wpr;
      uint32_t *mb = reinterpret_cast<uint32_t *>(buf + 16 * 16 * BITS);
      for (uint32_t u = lane; u < nrow * wpr; u += 32) {
        const uint32_t d = (uint32_t)__cvta_generic_to_shared(mb + (u / wpr) * 4 + u % wpr);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(mg + u) : "memory");
      }
      cp_async_commit_q();
    };
    uint32_t k = 0;
    if (it0 < n_it) issue(it0, codes_of(it0), stage0);
    // the code address of the step after the next is looked up one step early
    const uint8_t *cg_next = it0 + it_step < n_it ? codes_of(it0 + it_step) : nullptr;
    for (uint32_t it = it0; it < n_it; it += it_step, k ^= 1u) {
      const bool valid = it * 16 + rsub < NR;
      const uint32_t l = pos.l, t = pos.b, h = pos.a;
      pos.advance(da, db, dl, na, nb);
      const uint32_t R = (l * T + t) * H + h;
      const uint8_t *cg_after = it + 2 * it_step < n_it ? codes_of(it + 2 * it_step) : nullptr;
      if (it + it_step < n_it) issue(it + it_step, cg_next, stage0 + (k ^ 1u) * kStage);
      else cp_async_commit_q();  // an empty group keeps the wait count below uniform
      cg_next = cg_after;
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();
      const uint8_t *buf = stage0 + k * kStage;
      dec_row<BITS, HAD, BF16, DELTA, true>(P, fsign, oslot, half, valid, l, t, h, R, buf + 16 * BITS * rsub,
                                            reinterpret_cast<const uint32_t *>(buf + 16 * 16 * BITS) + 4 * rsub,
                                            flags);
      __syncwarp();  // every lane is done with this buffer before the next step refills it
    }
    cp_async_wait_all_q();
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// tile layout: logical float4 chunk q (0..7) of channel part p (32 channels) of a
// row is stored at physical chunk 8p + ((q + p) & 7).  A lane reading its part's
// chunks in the order q = 0..7 then touches, within each 8-lane shared-memory
// phase, 8 distinct bank groups (row stride 144 floats shifts odd rows by 16
// banks), while its register indices stay compile-time constants.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int phys_chunk(int lc) {  // lc = logical float4 chunk 0..31
  const int p = lc >> 3, q = lc & 7;
  return 8 * p + ((q + p) & 7);
}
__device__ __forceinline__ int phys_col(int col) { return 4 * phys_chunk(col >> 2) + (col & 3); }

__device__ __forceinline__ void tile_row_load(const float *Y, int r, int part, float (&v)[32]) {
  const float4 *row = reinterpret_cast<const float4 *>(Y + r * kTS) + 8 * part;
#pragma unroll
  for (int q = 0; q < 8; q++) {
    const float4 a = row[(q + part) & 7];
    v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
  }
}

__device__ __forceinline__ void tile_row_store(float *Y, int r, int part, const float (&v)[32]) {
  float4 *row = reinterpret_cast<float4 *>(Y + r * kTS) + 8 * part;
#pragma unroll
  for (int q = 0; q < 8; q++) row[(q + part) & 7] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// ---------------------------------------------------------------------------
// tile: encode
// ---------------------------------------------------------------------------
// Per-token groups of one row part (32 channels) of the tile kernel's row pass:
// parameters, codes, packing, one record store (and the metadata word by the
// group's first part).
template <int BITS>
__device__ __forceinline__ void tile_row_groups(const QuantParams &P, const float (&v)[32], int part, int gl,
                                                bool store, uint8_t *rec, size_t R, uint32_t &flags) {
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int i = 1; i < 32; i++) {
    mn = fminf(mn, v[i]);
    mx = fmaxf(mx, v[i]);
  }
  if (gl >= 2) {
    mn = fminf(mn, __shfl_xor_sync(kFull, mn, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  }
  if (gl >= 4) {
    mn = fminf(mn, __shfl_xor_sync(kFull, mn, 2));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  }
  float s, z, rr;
  uint32_t fl = 0;
  const uint32_t meta = quant_params<BITS>(mn, mx, s, z, rr, fl);
  uint32_t q[32], wds[BITS];
#pragma unroll
  for (int i = 0; i < 32; i++) q[i] = quant_code<BITS>(v[i], z, s, rr);
  pack32<BITS>(q, wds);
  if (store) {
    flags |= fl;
    store_words<BITS>(rec + 4 * BITS * part, wds);
    if ((part & (gl - 1)) == 0)
      *reinterpret_cast<uint32_t *>(P.meta + (R * (kHeadDim / P.group) + part / gl) * 4) = meta;
  }
}

template <int BITS, bool HAD, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kThreads) kvc_enc_tile(const QuantParams P, const __grid_constant__ WidthsArg<MIXED> W) {
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);  // [128][kTS]
  float *red = Y + 128 * kTS;                     // [2][8][128]
  float *mu_s = red + 2 * 8 * 128;                // [128]
  float *inv_s = mu_s + 128;                      // [128]
  float *anc_s = inv_s + 128;                     // [128] token delta: the block's anchor row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16 = P.g.bf16 != 0;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const int rg = tid >> 4, c8 = tid & 15;
  uint32_t flags = 0;

  for (uint32_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const uint32_t sb = tile % n_sb, lh = tile / n_sb, h = lh % H, l = lh / H;
    const uint32_t t0 = sb * kSmoothBlock;
    const uint32_t nvalid = min((uint32_t)kSmoothBlock, T - t0);
    const uint8_t *lbase = static_cast<const uint8_t *>(P.layers[l]);

    // ---- A: load the tile (a half-warp reads one 256-byte row segment)
    float x[8][8];
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const uint32_t r = rg + 16 * i;
      w[i] = make_uint4(0u, 0u, 0u, 0u);
      if (r < nvalid) {
        const uint64_t ro = row_offset(P.g, t0 + r);
        if (ro == ~0ull) flags |= KVC_FLAG_BAD_PAGE;
        else w[i] = __ldg(reinterpret_cast<const uint4 *>(lbase + ro + (size_t)(h * kHeadDim + 8 * c8) * 2));
      }
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
      unpack8(w[i], bf16, x[i]);
      if (!all_finite8(x[i])) flags |= KVC_FLAG_NONFINITE;
    }
    if constexpr (DELTA) {  // every row minus the block's first row (the anchor), whose bits are kept
      if (rg == 0) {
#pragma unroll
        for (int j = 0; j < 8; j++) anc_s[8 * c8 + j] = x[0][j];
        *reinterpret_cast<uint4 *>(P.anchors + (((size_t)lh * n_sb + sb) * kHeadDim + 8 * c8) * 2) = w[0];
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float a = anc_s[8 * c8 + j];
#pragma unroll
        for (int i = 0; i < 8; i++) x[i][j] = __fsub_rn(x[i][j], a);
      }
    }

    if (P.smooth) {
      // per-channel min / max over the valid tokens of the block
      float mn[8], mx[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        mn[j] = __int_as_float(0x7f800000);
        mx[j] = __int_as_float(0xff800000);
      }
#pragma unroll
      for (int i = 0; i < 8; i++)
        if (rg + 16 * i < nvalid)
#pragma unroll
          for (int j = 0; j < 8; j++) {
            mn[j] = fminf(mn[j], x[i][j]);
            mx[j] = fmaxf(mx[j], x[i][j]);
          }
#pragma unroll
      for (int j = 0; j < 8; j++) {
        mn[j] = fminf(mn[j], __shfl_xor_sync(kFull, mn[j], 16));
        mx[j] = fmaxf(mx[j], __shfl_xor_sync(kFull, mx[j], 16));
      }
      if (lane < 16)
#pragma unroll
        for (int j = 0; j < 8; j++) {
          red[warp * 128 + 8 * c8 + j] = mn[j];
          red[1024 + warp * 128 + 8 * c8 + j] = mx[j];
        }
      __syncthreads();
      if (tid < 128) {
        float a = red[tid], b = red[1024 + tid];
#pragma unroll
        for (int k = 1; k < 8; k++) {
          a = fminf(a, red[k * 128 + tid]);
          b = fmaxf(b, red[1024 + k * 128 + tid]);
        }
        float mu, inv;
        uint32_t mub;
        int e;
        smooth_params(a, b, mu, inv, mub, e, flags);
        mu_s[tid] = mu;
        inv_s[tid] = inv;
        const size_t cell = ((size_t)lh * n_sb + sb) * kHeadDim + tid;
        reinterpret_cast<uint16_t *>(P.mu)[cell] = (uint16_t)mub;
        P.ex[cell] = (int8_t)e;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float m = mu_s[8 * c8 + j], iv = inv_s[8 * c8 + j];
#pragma unroll
        for (int i = 0; i < 8; i++)
          x[i][j] = (rg + 16 * i < nvalid) ? __fmul_rn(__fsub_rn(x[i][j], m), iv) : 0.0f;
      }
    }
    const int pc0 = phys_chunk(2 * c8), pc1 = phys_chunk(2 * c8 + 1);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      float4 *row = reinterpret_cast<float4 *>(Y + (rg + 16 * i) * kTS);
      row[pc0] = make_float4(x[i][0], x[i][1], x[i][2], x[i][3]);
      row[pc1] = make_float4(x[i][4], x[i][5], x[i][6], x[i][7]);
    }
    __syncthreads();

    // ---- C: rows -- Hadamard, and the per-token groups when the axis is channels
    if (HAD || P.axis == KVC_AXIS_OVER_CHANNELS) {
      const int part = lane & 3, rsub = lane >> 2;
      const int gl = (int)(P.group >> 5);
#pragma unroll 1
      for (int k = 0; k < 2; k++) {
        const int r = warp * 16 + k * 8 + rsub;
        float v[32];
        tile_row_load(Y, r, part, v);
        if (HAD) {
          apply_signs(v, P.sign[part]);
          fwht128(v, part);
          scale_all(v, hadamard_scale());
        }
        if (P.axis == KVC_AXIS_OVER_CHANNELS) {
          const bool store = (uint32_t)r < nvalid;
          const size_t R = ((size_t)l * T + t0 + r) * H + h;
          if constexpr (MIXED) {
            uint8_t *rec = P.codes + (store ? row_code_offset<0, MIXED>(W, T, H, l, t0 + r, h, (uint32_t)R) : 0);
            switch (width_of<MIXED>(W, lh)) {  // one width per (layer, head): uniform over the CTA
              case 2: tile_row_groups<2>(P, v, part, gl, store, rec, R, flags); break;
              case 3: tile_row_groups<3>(P, v, part, gl, store, rec, R, flags); break;
              case 4: tile_row_groups<4>(P, v, part, gl, store, rec, R, flags); break;
              default: tile_row_groups<8>(P, v, part, gl, store, rec, R, flags); break;
            }
          } else {
            tile_row_groups<BITS>(P, v, part, gl, store, P.codes + R * (kHeadDim * BITS / 8), R, flags);
          }
        } else {
          tile_row_store(Y, r, part, v);
        }
      }
      __syncthreads();
    }

    // ---- D: columns -- groups of G tokens per channel (format v1 only: groups
    // over tokens otherwise run in the key-tile kernel)
    if constexpr (!MIXED) if (P.axis == KVC_AXIS_OVER_TOKENS) {
      const int c = tid & 127, half = tid >> 7, pcol = phys_col(c);
      const uint32_t G = P.group;
      float gmn[2], gmx[2];
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int seg = 2 * half + j;
        float a = __int_as_float(0x7f800000), b = __int_as_float(0xff800000);
        for (int q = 0; q < 32; q++) {
          const uint32_t rr = 32 * seg + q;
          if (rr < nvalid) {
            const float y = Y[rr * kTS + pcol];
            a = fminf(a, y);
            b = fmaxf(b, y);
          }
        }
        gmn[j] = a;
        gmx[j] = b;
      }
      if (G >= 64) {
        gmn[0] = gmn[1] = fminf(gmn[0], gmn[1]);
        gmx[0] = gmx[1] = fmaxf(gmx[0], gmx[1]);
      }
      if (G == 128) {
        red[half * 128 + c] = gmn[0];
        red[256 + half * 128 + c] = gmx[0];
        __syncthreads();
        gmn[0] = gmn[1] = fminf(red[c], red[128 + c]);
        gmx[0] = gmx[1] = fmaxf(red[256 + c], red[384 + c]);
      }
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const uint32_t row0 = 32 * (2 * half + j);
        const uint32_t tg = (t0 + row0) / G;
        if (tg < P.n_tg) {
          float s, z, rr;
          uint32_t fl = 0;
          const uint32_t meta = quant_params<BITS>(gmn[j], gmx[j], s, z, rr, fl);
          flags |= fl;
          uint32_t q[32], wds[BITS];
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const uint32_t rowi = row0 + i;
            q[i] = rowi < nvalid ? quant_code<BITS>(Y[rowi * kTS + pcol], z, s, rr) : 0u;
          }
          pack32<BITS>(q, wds);
          const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + c;
          store_words<BITS>(P.codes + g * (G * BITS / 8) + ((row0 % G) / 32) * 4 * BITS, wds);
          if (row0 % G == 0) *reinterpret_cast<uint32_t *>(P.meta + g * 4) = meta;
        }
      }
    }
    __syncthreads();
  }
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// key tile, groups over tokens (the key default): kvc_enc_ktile
//
// Per (layer, head, 128-token) tile, 512 threads, three barriers (four with smoothing and cp.async loads):
//  A  (smoothing only) warp w takes channel octet w over all 128 rows of the
//     stage (lane l: rows l + 32i).  The per-channel minima and maxima run on
//     the packed 16-bit pairs and are reduced across the warp by a halving
//     butterfly; then four warps, one lane per channel, turn them into the
//     smoothing parameters (sign folded into the power-of-two scale) in a
//     shared table.
//  C  thread (row r, part p) reads its 32 channels of row r from the stage and
//     smooths them (or flips their signs); the stage is then free for the next
//     tile's cp.async.  The Hadamard butterflies run with strides 1..16 in
//     registers and strides 32 and 64 with the lanes holding the row's other
//     parts (shuffles); the scaled row goes to the fp32 tile Y.
//  D  thread (channel c, quarter q) takes rows 32q..32q+31 of channel c from Y:
//     group minimum and maximum in registers plus one or two shuffles (groups
//     of 64 or 128 tokens), the group parameters, its 32 codes (packed by
//     integer multiply-adds), one store into the channel's record.
// Stage: the tile as two boxes of 64 channels x 128 rows (16 KiB each, rows of
// 128 bytes), each with the TMA 128-byte swizzle: 16-byte chunk k (0..15) of row
// r sits at byte (k >> 3) * 16384 + 128 r + 16 ((k & 7) ^ (r & 7)).
// Y: float4 column k of row r sits at k ^ (r & 1) ^ (((k >> 3) & 3) << 1) ^
// (((r >> 5) & 3) << 1).  With these, the loads into the stage, the A and C reads
// of the stage (C: two-way at most), the C writes and the D reads of Y are free of
// bank conflicts.
// ---------------------------------------------------------------------------
constexpr int kKT = 512;
constexpr int kTabStride = 36;  // floats per 32-channel part in the parameter tables (spreads the parts over banks)
// 1 KiB slack for aligning the stage to the swizzle's 1 KiB period
constexpr size_t kKtileSmem = 1024 + 128 * 256 + (size_t)128 * 128 * 4 + 3 * 4 * kTabStride * 4 + 256 * 4;

__device__ __forceinline__ uint32_t stage_off(uint32_t k, uint32_t r) {
  return (k >> 3) * 16384u + 128u * r + 16u * ((k & 7u) ^ (r & 7u));
}
__device__ __forceinline__ uint32_t ycol4(uint32_t k, uint32_t r) {
  return k ^ (r & 1u) ^ (((k >> 3) & 3u) << 1) ^ (((r >> 5) & 3u) << 1);
}


// The tile's two boxes by TMA (one thread): the mbarrier expects their 32 KiB.
__device__ __forceinline__ void ktile_tma(const CUtensorMap *map, uint32_t h, uint32_t t0, uint8_t *stage,
                                          uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
               "r"(32768u)
               : "memory");
#pragma unroll
  for (int b = 0; b < 2; b++)
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(stage + b * 16384)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"((int)(h * kHeadDim + 64 * b)), "r"((int)t0), "r"(smem_u32(bar))
        : "memory");
}
// Bounded wait for phase `par` of the stage barrier; false when it ran out.
__device__ __forceinline__ bool ktile_wait(uint64_t *bar, uint32_t par) {
  for (uint32_t i = 0; i < (1u << 22); i++) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_u32(bar)), "r"(par)
                 : "memory");
    if (done) return true;
  }
  return false;
}

// Thread (rg = tid / 16, k = tid % 16) copies chunk k of rows rg + 32i (i < 4) of
// the tile (sb, h, l) into the stage; rows past the end of the tensor are left as
// they are (no phase reads them), a bad page is zero-filled and flagged.
__device__ __forceinline__ void ktile_issue(const QuantParams &P, uint32_t sb, uint32_t h, uint32_t l, uint8_t *stage,
                                            int rg, int k, uint32_t &flags) {
  const uint32_t t0 = sb * kSmoothBlock, nvalid = min((uint32_t)kSmoothBlock, P.g.T - t0);
  const uint8_t *lbase = static_cast<const uint8_t *>(P.layers[l]) + (size_t)(h * kHeadDim + 8 * k) * 2;
  uint8_t *dst = stage + stage_off(k, rg);  // rows rg + 32i: + 4096 i
  if (!P.g.block_table) {
    const uint64_t ts = P.g.token_stride;
    const uint8_t *src = lbase + (uint64_t)(t0 + rg) * ts;
    if (nvalid == kSmoothBlock) {
#pragma unroll
      for (int i = 0; i < 4; i++) cp_async16_q(dst + i * 4096, src + (uint64_t)i * 32 * ts);
    } else {
#pragma unroll
      for (int i = 0; i < 4; i++)
        if (rg + 32 * i < (int)nvalid) cp_async16_q(dst + i * 4096, src + (uint64_t)i * 32 * ts);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t r = rg + 32 * i;
      if (r < nvalid) {
        const uint64_t ro = row_offset(P.g, t0 + r);
        if (ro == ~0ull) {
          flags |= KVC_FLAG_BAD_PAGE;
          *reinterpret_cast<uint4 *>(dst + i * 4096) = make_uint4(0u, 0u, 0u, 0u);
        } else {
          cp_async16_q(dst + i * 4096, lbase + ro);
        }
      }
    }
  }
  cp_async_commit_q();
}

// In-lane butterflies of 32 channels held as 16 pairs: stride 1 within pairs, 2..16 between pairs.
__device__ __forceinline__ void fwht32_pairs(float2 (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i++) {
    const float a = w[i].x, b = w[i].y;
    w[i] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i++)
      if ((i & h) == 0) {
        const float2 a = w[i], b = w[i + h];
        w[i] = add2(a, b);
        w[i + h] = sub2(a, b);
      }
  }
}

// 32 codes (BITS each, 4*BITS bytes) into a record segment.
template <int BITS>
__device__ __forceinline__ void store_codes32(uint8_t *dst, const uint32_t (&cw)[BITS]) {
  if constexpr (BITS == 2) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(cw[0], cw[1]);
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  } else if constexpr (BITS == 8) {
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  } else {
#pragma unroll
    for (int i = 0; i < BITS; i++) reinterpret_cast<uint32_t *>(dst)[i] = cw[i];
  }
}


// Tile coordinates, advanced by a fixed number of tiles without divisions.
struct TilePos {
  uint32_t sb, h, l;
  __device__ __forceinline__ void init(uint32_t tile, uint32_t n_sb, uint32_t H) {
    sb = tile % n_sb;
    const uint32_t lh = tile / n_sb;
    h = lh % H;
    l = lh / H;
  }
  // step = dsb + n_sb * (dh + H * dl) tiles, with dsb < n_sb and dh < H
  __device__ __forceinline__ void advance(uint32_t dsb, uint32_t dh, uint32_t dl, uint32_t n_sb, uint32_t H) {
    sb += dsb;
    uint32_t c = sb >= n_sb;
    sb -= c ? n_sb : 0u;
    h += dh + c;
    c = h >= H;
    h -= c ? H : 0u;
    l += dl + c;
  }
};

// D phase of kvc_enc_ktile for one (channel, 32-row quarter): the group
// parameters from the group's minimum and maximum, 32 codes from the correctly
// rounded quotients (the exact rule with its clamp for a saturated or non-finite
// group, warp-wide), codes of rows past the end zeroed, one store into the
// channel's record segment `dst` (and the metadata word at `meta` by the quarter
// that starts the group).
template <int BITS>
__device__ __forceinline__ void ktile_columns(const float (&v)[32], int nv, float mn, float mx, bool active,
                                              bool d_first, uint8_t *dst, uint8_t *meta, uint32_t &flags) {
  float sc = 0.0f, z = 0.0f, rr = 0.0f;
  uint32_t mword = 0, fl = 0;
  bool finite = true;
  if (active) {
    finite = finite2(mn, mx);
    if (!finite) flags |= KVC_FLAG_NONFINITE;
    mword = quant_params<BITS>(mn, mx, sc, z, rr, fl);
    flags |= fl;
  }
  uint32_t cw[BITS];
  {
    const float2 z2 = bcast2(z), r2 = bcast2(rr), ns2 = bcast2(-sc);
    uint32_t u[32];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const float2 s2 = qsum2(make_float2(v[2 * i], v[2 * i + 1]), z2, r2, ns2);
      u[2 * i] = __float_as_uint(s2.x);
      u[2 * i + 1] = __float_as_uint(s2.y);
    }
    pack_sums32<BITS>(u, cw);
  }
  // a saturated or non-finite group takes the exact rule
  const bool bad = active && (fl != 0 || !finite);
  if (__any_sync(kFull, bad)) {
    if (bad) {
#pragma unroll
      for (int i = 0; i < BITS; i++) cw[i] = 0u;
#pragma unroll
      for (int i = 0; i < 32; i++) put_code<BITS>(cw, i, qexact<BITS>(v[i], z, sc));
    }
  }
  if (nv < 32) {  // codes of rows past the end are 0
    const int keep = (nv > 0 ? nv : 0) * BITS;
#pragma unroll
    for (int i = 0; i < BITS; i++) {
      const int lo = 32 * i;
      if (keep <= lo) cw[i] = 0u;
      else if (keep < lo + 32) cw[i] &= (1u << (keep - lo)) - 1u;
    }
  }
  if (active) {
    if (d_first) *reinterpret_cast<uint32_t *>(meta) = mword;
    store_codes32<BITS>(dst, cw);
  }
}

template <int BITS, bool HAD, bool BF16, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kKT, 2)
    kvc_enc_ktile(const QuantParams P, const __grid_constant__ TmaMaps M, const __grid_constant__ WidthsArg<MIXED> W) {
  extern __shared__ float4 smem_f4[];
  __shared__ __align__(8) uint64_t stage_bar;
  uint8_t *stage = reinterpret_cast<uint8_t *>(smem_f4);
  stage += (1024u - (smem_u32(stage) & 1023u)) & 1023u;                // [2 boxes][128 rows][128 B], TMA swizzle
  float *Y = reinterpret_cast<float *>(stage + 128 * 256);             // [128][128] fp32, swizzled
  float *tab_mu = Y + 128 * 128;                                       // [4 parts][kTabStride]
  float *tab_inv = tab_mu + 4 * kTabStride;
  float *tab_nmi = tab_inv + 4 * kTabStride;                           // -mu * inv
  float *st = tab_nmi + 4 * kTabStride;  // A: channel c minimum at st[c], maximum at st[128 + c]
  __shared__ uint32_t s_wide;  // a channel of this tile has e > 100 (see the smoothing in C)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb, G = P.group;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const bool smooth = P.smooth != 0;
  uint32_t flags = 0;

  // tile-invariant thread roles and offsets
  const int rg = tid >> 4, kq = tid & 15;                  // cp.async: rows rg + 32i, chunk kq
  const uint32_t a_off = stage_off(warp, lane);             // A: chunk `warp` of rows lane + 32i: + 4096 i
  const int cr = tid >> 2, cp = tid & 3;                   // C: row cr, channels 32cp .. 32cp + 31
  const uint32_t c_off = stage_off(4 * cp, cr);             // C: chunk 4cp + i of row cr at c_off ^ 16 i
  const uint32_t c_xy = ycol4(8 * cp, cr) & 7u;            // C: Y float4 column 8cp + j sits at 8cp + (j ^ c_xy)
  const int dc = 8 * warp + (lane >> 2), dq = lane & 3;    // D: channel dc, rows 32dq .. 32dq + 31
  const float *Yd0 = Y + 32 * dq * 128 + 4 * (int)ycol4(dc >> 2, 32 * dq) + (dc & 3);      // even rows
  const float *Yd1 = Y + 32 * dq * 128 + 4 * (int)ycol4(dc >> 2, 32 * dq + 1) + (dc & 3);  // odd rows
  const int tiles_groups = 128 / (int)G;
  const uint32_t dq_group = (uint32_t)((32 * dq) / (int)G);  // D: this quarter's group within the tile
  const uint32_t rec_bytes = G * BITS / 8, seg_off = (uint32_t)((32 * dq) % (int)G) * BITS / 8;
  const bool d_first = ((32 * dq) % (int)G) == 0;          // D: the quarter that starts its group writes the metadata
  // the persistent grid advances by gridDim.x tiles
  const uint32_t step_lh = gridDim.x / n_sb, step_sb = gridDim.x % n_sb;
  const uint32_t step_h = step_lh % H, step_l = step_lh / H;

  const bool tma = P.tma != 0;
  if (tma && tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&stage_bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  uint32_t tile = blockIdx.x;
  TilePos cur, nxt;
  cur.init(tile < n_tiles ? tile : 0u, n_sb, H);
  if (tile < n_tiles) {
    if (!tma) ktile_issue(P, cur.sb, cur.h, cur.l, stage, rg, kq, flags);
    else if (tid == 0) ktile_tma(&M.map[cur.l], cur.h, cur.sb * kSmoothBlock, stage, &stage_bar);
  }
  for (uint32_t it = 0; tile < n_tiles; tile += gridDim.x, it++) {
    const uint32_t sb = cur.sb, lh = cur.l * H + cur.h;
    const uint32_t nvalid = min((uint32_t)kSmoothBlock, T - sb * kSmoothBlock);
    nxt = cur;
    nxt.advance(step_sb, step_h, step_l, n_sb, H);
    if (!tma) cp_async_wait_all_q();
    else if (!ktile_wait(&stage_bar, it & 1u)) flags |= KVC_FLAG_TIMEOUT;
    // the stage holds this tile.  With smoothing and TMA a warp that is done with
    // the previous tile's D goes straight on to A (which reads only the stage and
    // writes only st); the barrier after A then also ends every read of the
    // previous Y.  Otherwise a barrier here (cp.async data is visible to the
    // other threads only after it, and C writes Y).
    if (!tma || !smooth) __syncthreads();

    // ---- A: smoothing parameters.  Minima and maxima run on the packed 16-bit
    // pairs (exact); lanes 8j..8j+7 end with pair j (channels 2j, 2j+1 of the octet).
    // With the token delta they run on the fp32 differences from row 0 instead.
    if (smooth) {
      // every warp has left the previous tile's C (the barrier after C): the flag is free
      if (tid == 0) s_wide = 0u;
     if constexpr (DELTA) {
      float an[8];  // the octet's channels of row 0, the block's anchor
      {
        const uint4 u = *reinterpret_cast<const uint4 *>(stage + stage_off(warp, 0));
        const float2 p0 = unpack_pair(u.x, BF16), p1 = unpack_pair(u.y, BF16), p2 = unpack_pair(u.z, BF16),
                     p3 = unpack_pair(u.w, BF16);
        an[0] = p0.x; an[1] = p0.y; an[2] = p1.x; an[3] = p1.y; an[4] = p2.x; an[5] = p2.y; an[6] = p3.x; an[7] = p3.y;
      }
      float mn[8], mx[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        mn[j] = __int_as_float(0x7f800000);
        mx[j] = __int_as_float(0xff800000);
      }
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int r = lane + 32 * i;
        if (r < (int)nvalid) {
          const uint4 u = *reinterpret_cast<const uint4 *>(stage + a_off + 4096 * i);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const float2 x = unpack_pair(w4[k], BF16);
            const float d0 = __fsub_rn(x.x, an[2 * k]), d1 = __fsub_rn(x.y, an[2 * k + 1]);
            mn[2 * k] = fmin_n(mn[2 * k], d0); mx[2 * k] = fmax_n(mx[2 * k], d0);
            mn[2 * k + 1] = fmin_n(mn[2 * k + 1], d1); mx[2 * k + 1] = fmax_n(mx[2 * k + 1], d1);
          }
        }
      }
      // halving butterfly (offsets 16, 8, 4: 8 -> 4 -> 2 -> 1 channels per lane), then offsets 2, 1
#pragma unroll
      for (int s2 = 0; s2 < 3; s2++) {
        const int o = 16 >> s2, half = 4 >> s2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
          const float sn = up ? mn[i] : mn[i + half], sx = up ? mx[i] : mx[i + half];
          const float kn = up ? mn[i + half] : mn[i], kx = up ? mx[i + half] : mx[i];
          mn[i] = fmin_n(kn, __shfl_xor_sync(kFull, sn, o));
          mx[i] = fmax_n(kx, __shfl_xor_sync(kFull, sx, o));
        }
      }
#pragma unroll
      for (int o = 2; o >= 1; o >>= 1) {
        mn[0] = fmin_n(mn[0], __shfl_xor_sync(kFull, mn[0], o));
        mx[0] = fmax_n(mx[0], __shfl_xor_sync(kFull, mx[0], o));
      }
      if ((lane & 3) == 0) {  // lane bits 4, 3, 2 give the channel of the octet
        const int ch = 8 * warp + 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
        st[ch] = mn[0];
        st[128 + ch] = mx[0];
      }
     } else {
      const uint32_t pinf = BF16 ? 0x7f807f80u : 0x7c007c00u, ninf = pinf | 0x80008000u;
      uint32_t mn[4] = {pinf, pinf, pinf, pinf}, mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int r = lane + 32 * i;
        if (r < (int)nvalid) {
          const uint4 u = *reinterpret_cast<const uint4 *>(stage + a_off + 4096 * i);
          mn[0] = pmin2_n<BF16>(mn[0], u.x); mx[0] = pmax2_n<BF16>(mx[0], u.x);
          mn[1] = pmin2_n<BF16>(mn[1], u.y); mx[1] = pmax2_n<BF16>(mx[1], u.y);
          mn[2] = pmin2_n<BF16>(mn[2], u.z); mx[2] = pmax2_n<BF16>(mx[2], u.z);
          mn[3] = pmin2_n<BF16>(mn[3], u.w); mx[3] = pmax2_n<BF16>(mx[3], u.w);
        }
      }
      // halving butterfly (offsets 16, 8), then the rest of the lanes (4, 2, 1)
#pragma unroll
      for (int s = 0; s < 2; s++) {
        const int o = 16 >> s, half = 2 >> s;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
          const uint32_t sn = up ? mn[i] : mn[i + half], sx = up ? mx[i] : mx[i + half];
          const uint32_t kn = up ? mn[i + half] : mn[i], kx = up ? mx[i + half] : mx[i];
          mn[i] = pmin2_n<BF16>(kn, __shfl_xor_sync(kFull, sn, o));
          mx[i] = pmax2_n<BF16>(kx, __shfl_xor_sync(kFull, sx, o));
        }
      }
#pragma unroll
      for (int o = 4; o >= 1; o >>= 1) {
        mn[0] = pmin2_n<BF16>(mn[0], __shfl_xor_sync(kFull, mn[0], o));
        mx[0] = pmax2_n<BF16>(mx[0], __shfl_xor_sync(kFull, mx[0], o));
      }
      if ((lane & 3) == 0) {
        const int hi = (lane >> 2) & 1;  // lane 8j: channel 2j, lane 8j + 4: channel 2j + 1
        const int ch = 8 * warp + 2 * (lane >> 3) + hi;
        const float2 fa = unpack_pair(mn[0], BF16), fb = unpack_pair(mx[0], BF16);
        st[ch] = hi ? fa.y : fa.x;
        st[128 + ch] = hi ? fb.y : fb.x;
      }
     }
      __syncthreads();
      if (warp < 4) {  // one lane per channel turns the statistics into the smoothing parameters
        const int ch = 32 * warp + lane;
        float a = st[ch], b = st[128 + ch];
        if (a != a) a = __int_as_float(0x7fffffff);  // one NaN for every input NaN
        if (b != b) b = __int_as_float(0x7fffffff);
        if (!finite2(a, b)) flags |= KVC_FLAG_NONFINITE;
        float mu, inv;
        uint32_t mub;
        int e;
        smooth_params(a, b, mu, inv, mub, e, flags);
        if (HAD && ((P.sign[warp] >> lane) & 1u)) inv = -inv;  // sign folded into the exact scale
        tab_mu[kTabStride * warp + lane] = mu;
        tab_inv[kTabStride * warp + lane] = inv;
        tab_nmi[kTabStride * warp + lane] = __fmul_rn(-mu, inv);  // exact: mu is binary16, inv = +-2^-e
        if (e > 100) s_wide = 1u;
        const size_t cell = ((size_t)lh * n_sb + sb) * kHeadDim + ch;
        reinterpret_cast<uint16_t *>(P.mu)[cell] = (uint16_t)mub;
        P.ex[cell] = (int8_t)e;
      }
      // no barrier here: C reads only the stage until its own barrier, which also
      // publishes the parameter table before the smoothing uses it
    }

    // ---- C: row pass
    {
      float2 w[16];
      const bool live = cr < (int)nvalid;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (live) u = *reinterpret_cast<const uint4 *>(stage + (c_off ^ (16u * i)));
        w[4 * i] = unpack_pair(u.x, BF16);
        w[4 * i + 1] = unpack_pair(u.y, BF16);
        w[4 * i + 2] = unpack_pair(u.z, BF16);
        w[4 * i + 3] = unpack_pair(u.w, BF16);
        if constexpr (DELTA) {  // minus the block's anchor (row 0), whose bits row 0's threads keep
          const uint4 ua = *reinterpret_cast<const uint4 *>(stage + (stage_off(4 * cp, 0) ^ (16u * i)));
          w[4 * i] = sub2(w[4 * i], unpack_pair(ua.x, BF16));
          w[4 * i + 1] = sub2(w[4 * i + 1], unpack_pair(ua.y, BF16));
          w[4 * i + 2] = sub2(w[4 * i + 2], unpack_pair(ua.z, BF16));
          w[4 * i + 3] = sub2(w[4 * i + 3], unpack_pair(ua.w, BF16));
          if (cr == 0)
            reinterpret_cast<uint4 *>(P.anchors + (((size_t)lh * n_sb + sb) * kHeadDim + 32 * cp) * 2)[i] = ua;
        }
      }
      __syncthreads();  // every row has been read: the stage takes the next tile
      if (tile + gridDim.x < n_tiles) {
        if (!tma) {
          ktile_issue(P, nxt.sb, nxt.h, nxt.l, stage, rg, kq, flags);
        } else if (tid == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the reads above before the async writes
          ktile_tma(&M.map[nxt.l], nxt.h, nxt.sb * kSmoothBlock, stage, &stage_bar);
        }
      }
      if (smooth) {
        // x' = RN(x - mu) 2^-e.  One fma, RN(x inv + (-mu inv)), rounds the exact
        // (x - mu) inv once: the same value whenever x - mu is exact or the result is
        // normal.  An inexact x - mu has |x - mu| >= |mu| / 2 >= 2^-25 (binary16 mu,
        // Sterbenz), so with e <= 100 the result is normal; a tile with a larger e
        // (a range beyond 2^100) takes the two roundings as written.
        const float4 *ti = reinterpret_cast<const float4 *>(tab_inv + kTabStride * cp);
        if (!s_wide) {
          const float4 *tn = reinterpret_cast<const float4 *>(tab_nmi + kTabStride * cp);
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const float4 n = tn[k], iv = ti[k];
            w[2 * k] = __ffma2_rn(w[2 * k], make_float2(iv.x, iv.y), make_float2(n.x, n.y));
            w[2 * k + 1] = __ffma2_rn(w[2 * k + 1], make_float2(iv.z, iv.w), make_float2(n.z, n.w));
          }
        } else {
          const float4 *tm = reinterpret_cast<const float4 *>(tab_mu + kTabStride * cp);
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const float4 m = tm[k], iv = ti[k];
            w[2 * k] = mul2(sub2(w[2 * k], make_float2(m.x, m.y)), make_float2(iv.x, iv.y));
            w[2 * k + 1] = mul2(sub2(w[2 * k + 1], make_float2(m.z, m.w)), make_float2(iv.z, iv.w));
          }
        }
        if (nvalid < 128 && !live) {  // rows past the end stay 0 (only the last tile has any)
#pragma unroll
          for (int k = 0; k < 16; k++) w[k] = make_float2(0.0f, 0.0f);
        }
      } else if (HAD) {
        const uint32_t sbits = P.sign[cp];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          w[i].x = __uint_as_float(__float_as_uint(w[i].x) ^ (((sbits >> (2 * i)) & 1u) << 31));
          w[i].y = __uint_as_float(__float_as_uint(w[i].y) ^ (((sbits >> (2 * i + 1)) & 1u) << 31));
        }
      }
      if (HAD) {
        fwht32_pairs(w);
        const float2 s32 = bcast2((cp & 1) ? -1.0f : 1.0f), s64 = bcast2((cp & 2) ? -1.0f : 1.0f);
#pragma unroll
        for (int i = 0; i < 16; i++) {  // stride 32: the partner part is lane ^ 1
          const float2 x = make_float2(__shfl_xor_sync(kFull, w[i].x, 1), __shfl_xor_sync(kFull, w[i].y, 1));
          w[i] = __ffma2_rn(w[i], s32, x);  // lower channel: own + other; upper: other - own
        }
#pragma unroll
        for (int i = 0; i < 16; i++) {  // stride 64: the partner part is lane ^ 2
          const float2 x = make_float2(__shfl_xor_sync(kFull, w[i].x, 2), __shfl_xor_sync(kFull, w[i].y, 2));
          w[i] = __ffma2_rn(w[i], s64, x);
        }
        const float2 c2 = bcast2(hadamard_scale());
#pragma unroll
        for (int i = 0; i < 16; i++) w[i] = mul2(w[i], c2);
      }
      float4 *yrow = reinterpret_cast<float4 *>(Y + cr * 128) + 8 * cp;
#pragma unroll
      for (int j = 0; j < 8; j++) yrow[j ^ c_xy] = make_float4(w[2 * j].x, w[2 * j].y, w[2 * j + 1].x, w[2 * j + 1].y);
    }
    __syncthreads();

    // ---- D: column pass
    {
      const int nv = (int)nvalid - 32 * dq;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = ((i & 1) ? Yd1 : Yd0)[i * 128];
      float mn, mx;
      if (nv >= 32) {
        mn = fmin3_n(v[0], v[1], v[2]);
        mx = fmax3_n(v[0], v[1], v[2]);
#pragma unroll
        for (int i = 3; i < 31; i += 2) {
          mn = fmin3_n(mn, v[i], v[i + 1]);
          mx = fmax3_n(mx, v[i], v[i + 1]);
        }
        mn = fmin_n(mn, v[31]);
        mx = fmax_n(mx, v[31]);
      } else {
        mn = __int_as_float(0x7f800000);
        mx = __int_as_float(0xff800000);
#pragma unroll
        for (int i = 0; i < 32; i++)
          if (i < nv) {
            mn = fmin_n(mn, v[i]);
            mx = fmax_n(mx, v[i]);
          }
      }
      for (int o = 1; o < (int)G / 32; o <<= 1) {  // the group's other quarters are lanes ^ 1 (and ^ 2)
        mn = fmin_n(mn, __shfl_xor_sync(kFull, mn, o));
        mx = fmax_n(mx, __shfl_xor_sync(kFull, mx, o));
      }
      const uint32_t tg = sb * tiles_groups + dq_group;
      const bool active = tg < P.n_tg;  // a quarter past the end of an existing group still writes its (zero) codes
      if constexpr (MIXED) {
        // this (layer, head)'s width and code block (blocks of 16 n_tg G bytes per unit of width)
        const uint32_t b = width_of<MIXED>(W, lh);
        uint8_t *blk = P.codes + (size_t)16 * P.n_tg * G * W.wsum[lh];
        const size_t rec = (size_t)tg * kHeadDim + dc;  // record index in the block
        const uint32_t seg = (uint32_t)((32 * dq) % (int)G);
        uint8_t *meta = P.meta + (((size_t)lh * P.n_tg + tg) * kHeadDim + dc) * 4;
        switch (b) {
          case 2: ktile_columns<2>(v, nv, mn, mx, active, d_first, blk + rec * (G * 2 / 8) + seg * 2 / 8, meta, flags); break;
          case 3: ktile_columns<3>(v, nv, mn, mx, active, d_first, blk + rec * (G * 3 / 8) + seg * 3 / 8, meta, flags); break;
          case 4: ktile_columns<4>(v, nv, mn, mx, active, d_first, blk + rec * (G * 4 / 8) + seg * 4 / 8, meta, flags); break;
          default: ktile_columns<8>(v, nv, mn, mx, active, d_first, blk + rec * G + seg, meta, flags); break;
        }
      } else {
        const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + dc;
        ktile_columns<BITS>(v, nv, mn, mx, active, d_first, P.codes + g * rec_bytes + seg_off, P.meta + g * 4,
                            flags);
      }
    }
    cur = nxt;
  }
  cp_async_wait_all_q();
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// key tile decode, groups over tokens (the key default): kvc_dec_ktile
//
// Per (layer, head, 128-token) tile, 128 threads (three CTAs per SM), two
// barriers, no shuffles:
//  D  thread c: the 128 codes of channel c (loaded a tile ahead) become floats
//     through the exponent field (0x4B000000 | code is 2^23 + code, so one exact
//     subtraction per pair leaves the code), are dequantized with one packed
//     fma per pair and go down column c of the fp32 tile Y;
//  C  thread r: all 128 channels of row r in registers: the inverse Hadamard
//     transform (strides 1..64, then the scale), the signs and the smoothing
//     undone by one packed fma per pair (sign folded into the power-of-two
//     scale), rounding to the element type, the 256-byte row stored.
// Each thread cp.asyncs its next tile's codes and metadata into its own slots of
// shared buffers while C runs.
// Y: float4 column k of row r sits at k ^ (r & 31), so a warp's column writes
// (one row, 32 channels) and row reads (32 rows, one float4 column) are free of
// bank conflicts.
// ---------------------------------------------------------------------------
constexpr int kKD = 128;


// Byte offset `o` of channel c's code slot, rotated so that the 8 lanes of a
// 16-byte shared access phase hit 8 distinct bank groups: 16-byte unit u of the
// slot is stored at unit u ^ kdec_rot<BITS>(c) (BITS = 3: slots of 3 units, not
// rotated).
template <int BITS>
__device__ __forceinline__ uint32_t kdec_rot(int c) {
  if constexpr (BITS == 2) return ((uint32_t)c >> 2) & 1u;
  else if constexpr (BITS == 4) return ((uint32_t)c >> 1) & 3u;
  else if constexpr (BITS == 8) return (uint32_t)c & 7u;
  else return 0u;
}

// The D-phase inputs of a tile for channel c, copied by thread c into its own
// slots of the shared buffers (so only thread c reads them, after its own
// cp.async wait): its codes over the tile's 128 rows (16*BITS bytes: a segment of
// each of the tile's 128 / G token-group records) at cbuf + 16*BITS*c, 16-byte
// units rotated by kdec_rot, and the group metadata words at mbuf[128 gi + c].
// Groups past the end are zero.
// `blk` is the (layer, head)'s code block: records [token group][channel].  SB:
// the slot width (BITS, or 8 in a mixed-width launch).
template <int BITS, int SB = BITS>
__device__ __forceinline__ void kdec_issue(const QuantParams &P, uint32_t sb, uint32_t lh, const uint8_t *blk, int c,
                                           uint8_t *cbuf, uint32_t *mbuf) {
  const uint32_t G = P.group, ng = 128u >> (31 - __clz(G)), rec = G * BITS / 8;  // G is 32, 64 or 128
  const size_t g0 = ((size_t)lh * P.n_tg + sb * ng) * kHeadDim + c;  // record of the tile's first group
  const size_t r0 = (size_t)sb * ng * kHeadDim + c;                   // the same inside the block
  uint8_t *dst = cbuf + 16 * SB * c;
  const uint32_t rot = kdec_rot<BITS>(c) << 4;
  for (uint32_t gi = 0; gi < ng; gi++) {
    const size_t g = g0 + (size_t)gi * kHeadDim;
    if (sb * ng + gi < P.n_tg) {
      const uint32_t m = (uint32_t)__cvta_generic_to_shared(mbuf + 128 * gi + c);
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(m), "l"(P.meta + g * 4) : "memory");
      const uint8_t *src = blk + (r0 + (size_t)gi * kHeadDim) * rec;
      if ((rec & 15) == 0) {
        for (uint32_t o = 0; o < rec; o += 16) cp_async16_q(dst + ((gi * rec + o) ^ rot), src + o);
      } else {
        for (uint32_t o = 0; o < rec; o += 4) {
          const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst + ((gi * rec + o) ^ rot));
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src + o) : "memory");
        }
      }
    } else {
      mbuf[128 * gi + c] = 0u;
      for (uint32_t o = 0; o < rec; o += 4) *reinterpret_cast<uint32_t *>(dst + ((gi * rec + o) ^ rot)) = 0u;
    }
  }
  cp_async_commit_q();
}

// Y, the smoothing table, the code slots, the metadata words, and (token delta)
// the tile's anchor row as floats.
template <int BITS>
constexpr size_t kdec_smem(uint32_t G, bool delta = false) {
  return (size_t)128 * 128 * 4 + 64 * 16 + 16 * BITS * 128 + 4 * 128 * (128 / G) + (delta ? 128 * 4 : 0);
}

// D phase of kvc_dec_ktile for one tile: column `tid` of Y from this thread's
// code and metadata slots, the smoothing table entry of channel `tid`.
// SB: the width the code slots were laid out for (BITS, or 8 in a mixed-width
// launch; kdec_issue packs the slot's first 16*BITS bytes either way).
template <int BITS, bool HAD, int SB = BITS>
__device__ __forceinline__ void kdec_columns(const QuantParams &P, float *Y, float4 *tab, const uint8_t *cbuf,
                                             const uint32_t *mbuf, bool smooth, uint32_t mub, int ex) {
  const int tid = threadIdx.x, kc = tid >> 2;
  const uint32_t G = P.group;
  float *Yc = Y + (tid & 3);  // element (row i, channel tid) at Yc + 128 i + 4 (kc ^ (i & 31))
  uint32_t cw[4 * BITS];
  const uint32_t *cs = reinterpret_cast<const uint32_t *>(cbuf + 16 * SB * tid);
  if constexpr (BITS == 3) {
#pragma unroll
    for (int k = 0; k < 12; k++) cw[k] = cs[k];
  } else {
    const uint32_t rot = kdec_rot<BITS>(tid);
#pragma unroll
    for (int k = 0; k < BITS; k++) {
      const uint4 a = reinterpret_cast<const uint4 *>(cs)[k ^ rot];
      cw[4 * k] = a.x; cw[4 * k + 1] = a.y; cw[4 * k + 2] = a.z; cw[4 * k + 3] = a.w;
    }
  }
  const uint32_t gsh = 31 - __clz(G), ng = 128u >> gsh;  // G is 32, 64 or 128
  uint32_t meta[4];
#pragma unroll
  for (uint32_t gi = 0; gi < 4; gi++) meta[gi] = gi < ng ? mbuf[128 * gi + tid] : 0u;
  float2 qf[16];
#pragma unroll
  for (int seg = 0; seg < 4; seg++) {  // rows 32 seg .. 32 seg + 31
    uint32_t w[BITS];
#pragma unroll
    for (int k = 0; k < BITS; k++) w[k] = cw[seg * BITS + k];
    codes_to_f2<BITS>(w, qf);
    const uint32_t gi = (uint32_t)(32 * seg) >> gsh;
    const uint32_t m = gi == 0 ? meta[0] : gi == 1 ? meta[1] : gi == 2 ? meta[2] : meta[3];
    const float2 s2 = bcast2(__half2float(__ushort_as_half((unsigned short)(m & 0xffffu))));
    const float2 z2 = bcast2(__half2float(__ushort_as_half((unsigned short)(m >> 16))));
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const float2 y = __ffma2_rn(qf[i], s2, z2);
      const int r0 = 32 * seg + 2 * i;
      Yc[r0 * 128 + 4 * (kc ^ (r0 & 31))] = y.x;
      Yc[(r0 + 1) * 128 + 4 * (kc ^ ((r0 + 1) & 31))] = y.y;
    }
  }
  if (smooth) {
    float sc = pow2i(ex < -126 ? -126 : ex);
    if (HAD && ((P.sign[tid >> 5] >> (tid & 31)) & 1u)) sc = -sc;  // sign folded into the exact scale
    float *t = reinterpret_cast<float *>(tab + (tid >> 1)) + (tid & 1);
    t[0] = __half2float(__ushort_as_half((unsigned short)mub));
    t[2] = sc;
  }
}

// The code block of (layer, head) lh as kdec_issue addresses tile sb of it: with
// codes read in place, shifted so that tile sb's records land where code_unit puts
// them (the tile, 2048 BITS bytes, is one unit: the host enables this only where
// every (layer, head) holds whole tiles).
template <int BITS>
__device__ __forceinline__ const uint8_t *kdec_block(const QuantParams &P, uint32_t sb, uint32_t lh) {
  const size_t rec = P.group * BITS / 8, blk = (size_t)lh * P.n_tg * kHeadDim * rec;
  if (P.in_lo >= P.in_hi) return P.codes + blk;
  const size_t lead = (size_t)sb * (128u / P.group) * kHeadDim * rec;  // tile sb's first record in the block
  return reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(code_unit(P, blk + lead)) - lead);
}

// The D-phase inputs of tile (sb, lh) for channel c: its (layer, head)'s width
// decides the record size (a mixed-width launch dispatches per tile).  `blk`: the
// uniform-width launch's kdec_block for this tile.
template <int BITS, bool MIXED>
__device__ __forceinline__ void kdec_issue_any(const QuantParams &P, const WidthsArg<MIXED> &W, uint32_t sb,
                                               uint32_t lh, int c, uint8_t *cbuf, uint32_t *mbuf,
                                               const uint8_t *blk) {
  if constexpr (MIXED) {
    const uint8_t *blk = P.codes + (size_t)16 * P.n_tg * P.group * W.wsum[lh];
    switch (width_of<MIXED>(W, lh)) {
      case 2: kdec_issue<2, BITS>(P, sb, lh, blk, c, cbuf, mbuf); break;
      case 3: kdec_issue<3, BITS>(P, sb, lh, blk, c, cbuf, mbuf); break;
      case 4: kdec_issue<4, BITS>(P, sb, lh, blk, c, cbuf, mbuf); break;
      default: kdec_issue<8, BITS>(P, sb, lh, blk, c, cbuf, mbuf); break;
    }
  } else {
    kdec_issue<BITS>(P, sb, lh, blk, c, cbuf, mbuf);
  }
}

template <int BITS, bool HAD, bool BF16, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kKD, 3) kvc_dec_ktile(const QuantParams P, const __grid_constant__ WidthsArg<MIXED> W) {
  if (P.check_corrupt && (*(volatile uint32_t *)P.status & KVC_FLAG_CORRUPT)) return;
  constexpr int SB = MIXED ? 8 : BITS;             // code slot width
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);   // [128][128] fp32, swizzled
  float4 *tab = smem_f4 + 128 * 128 / 4;           // pair j: {mu_2j, mu_2j+1, sc_2j, sc_2j+1}
  uint8_t *cbuf = reinterpret_cast<uint8_t *>(tab + 64);                 // [128 channels][16*SB] codes
  uint32_t *mbuf = reinterpret_cast<uint32_t *>(cbuf + 16 * SB * 128);  // [groups][128] metadata
  float *anc = reinterpret_cast<float *>(mbuf + 128 * (128 / P.group));  // token delta: the tile's anchor row
  const int tid = threadIdx.x;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const bool smooth = P.smooth != 0;
  uint32_t flags = 0;
  const uint32_t step_lh = gridDim.x / n_sb, step_sb = gridDim.x % n_sb;
  const uint32_t step_h = step_lh % H, step_l = step_lh / H;

  uint32_t tile = blockIdx.x;
  if (tile >= n_tiles) return;
  TilePos cur, nxt;
  cur.init(tile, n_sb, H);
  uint32_t mub = 0, anb = 0;
  int ex = 0;
  kdec_issue_any<SB, MIXED>(P, W, cur.sb, cur.l * H + cur.h, tid, cbuf, mbuf,
                            MIXED ? nullptr : kdec_block<SB>(P, cur.sb, cur.l * H + cur.h));
  if (smooth || DELTA) {
    const size_t cell = ((size_t)(cur.l * H + cur.h) * n_sb + cur.sb) * kHeadDim + tid;
    if (smooth) {
      mub = reinterpret_cast<const uint16_t *>(P.mu)[cell];
      ex = P.ex[cell];
    }
    if (DELTA) anb = reinterpret_cast<const uint16_t *>(P.anchors)[cell];
  }
  for (; tile < n_tiles; tile += gridDim.x) {
    const uint32_t sb = cur.sb, l = cur.l, h = cur.h;
    const uint32_t t0 = sb * kSmoothBlock, nvalid = min((uint32_t)kSmoothBlock, T - t0);
    nxt = cur;
    nxt.advance(step_sb, step_h, step_l, n_sb, H);
    const bool more = tile + gridDim.x < n_tiles;
    // the next tile's code block, looked up before this tile's D phase
    const uint8_t *blk_n = !MIXED && more ? kdec_block<SB>(P, nxt.sb, nxt.l * H + nxt.h) : nullptr;

    // ---- D: column tid
    cp_async_wait_all_q();
    if constexpr (MIXED) {
      switch (width_of<MIXED>(W, l * H + h)) {
        case 2: kdec_columns<2, HAD, SB>(P, Y, tab, cbuf, mbuf, smooth, mub, ex); break;
        case 3: kdec_columns<3, HAD, SB>(P, Y, tab, cbuf, mbuf, smooth, mub, ex); break;
        case 4: kdec_columns<4, HAD, SB>(P, Y, tab, cbuf, mbuf, smooth, mub, ex); break;
        default: kdec_columns<8, HAD, SB>(P, Y, tab, cbuf, mbuf, smooth, mub, ex); break;
      }
    } else {
      kdec_columns<BITS, HAD, SB>(P, Y, tab, cbuf, mbuf, smooth, mub, ex);
    }
    if constexpr (DELTA) anc[tid] = elt_to_f32(anb, BF16);
    if (more) {  // this thread's slots are read: the next tile's inputs go there
      kdec_issue_any<SB, MIXED>(P, W, nxt.sb, nxt.l * H + nxt.h, tid, cbuf, mbuf, blk_n);
      if (smooth || DELTA) {
        const size_t cell = ((size_t)(nxt.l * H + nxt.h) * n_sb + nxt.sb) * kHeadDim + tid;
        if (smooth) {
          mub = reinterpret_cast<const uint16_t *>(P.mu)[cell];
          ex = P.ex[cell];
        }
        if (DELTA) anb = reinterpret_cast<const uint16_t *>(P.anchors)[cell];
      }
    }
    __syncthreads();

    // ---- C: row tid
    const int r = tid;
    if (r < (int)nvalid) {
      float2 v[64];  // v[j] = channels 2j, 2j+1
      const float4 *yrow = reinterpret_cast<const float4 *>(Y + r * 128);
#pragma unroll
      for (int k = 0; k < 32; k++) {
        const float4 a = yrow[k ^ (r & 31)];
        v[2 * k] = make_float2(a.x, a.y);
        v[2 * k + 1] = make_float2(a.z, a.w);
      }
      if (HAD) {
#pragma unroll
        for (int j = 0; j < 64; j++) {  // stride 1, inside each pair
          const float a = v[j].x, b = v[j].y;
          v[j] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
        }
#pragma unroll
        for (int hs = 1; hs < 64; hs <<= 1)  // strides 2 .. 64: pairs j and j + hs
#pragma unroll
          for (int j = 0; j < 64; j++)
            if ((j & hs) == 0) {
              const float2 a = v[j], b = v[j + hs];
              v[j] = add2(a, b);
              v[j + hs] = sub2(a, b);
            }
        const float2 c2 = bcast2(hadamard_scale());
#pragma unroll
        for (int j = 0; j < 64; j++) v[j] = mul2(v[j], c2);
      }
      if (smooth) {
#pragma unroll
        for (int j = 0; j < 64; j++) {
          const float4 t = tab[j];
          v[j] = __ffma2_rn(v[j], make_float2(t.z, t.w), make_float2(t.x, t.y));
        }
      } else if (HAD) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const uint32_t sbits = P.sign[q];
#pragma unroll
          for (int i = 0; i < 16; i++) {
            float2 &x = v[16 * q + i];
            x.x = __uint_as_float(__float_as_uint(x.x) ^ (((sbits >> (2 * i)) & 1u) << 31));
            x.y = __uint_as_float(__float_as_uint(x.y) ^ (((sbits >> (2 * i + 1)) & 1u) << 31));
          }
        }
      }
      if constexpr (DELTA) {  // plus the block's anchor row
        const float2 *an2 = reinterpret_cast<const float2 *>(anc);
#pragma unroll
        for (int j = 0; j < 64; j++) v[j] = add2(v[j], an2[j]);
      }
      const uint64_t ro = row_offset(P.g, t0 + r);
      if (ro == ~0ull) {
        flags |= KVC_FLAG_BAD_PAGE;
      } else {
        uint8_t *dst = static_cast<uint8_t *>(P.layers[l]) + ro + (size_t)h * kHeadDim * 2;
        // the 256-byte row goes out by one bulk copy from this thread's own Y row,
        // which it has read already; starting it 16 (r % 16) bytes into that row
        // spreads the 8 rows of a 16-byte store phase over 8 bank groups
        uint4 *srow = reinterpret_cast<uint4 *>(Y + r * 128) + (r & 15);
#pragma unroll
        for (int k = 0; k < 16; k++) {
          uint32_t u[4];
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 x = v[4 * k + i];
            if (BF16) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(x.x, x.y);
              u[i] = *reinterpret_cast<const uint32_t *>(&b2);
            } else {
              const __half2 h2 = __floats2half2_rn(x.x, x.y);
              u[i] = *reinterpret_cast<const uint32_t *>(&h2);
            }
          }
          srow[k] = make_uint4(u[0], u[1], u[2], u[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stores above before the async read
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 256;" ::"l"(dst),
                     "r"(smem_u32(srow))
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    // the next tile's D writes Y: every row copy must have read its bytes
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncthreads();
    cur = nxt;
  }
  cp_async_wait_all_q();
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// tile: decode
// ---------------------------------------------------------------------------
// Dequantized per-token groups of one row part (32 channels) of the tile decoder.
template <int BITS>
__device__ __forceinline__ void tile_row_dequant(const QuantParams &P, float (&v)[32], int part, int gl,
                                                 const uint8_t *rec, size_t R) {
  uint32_t wds[BITS], q[32];
  load_words<BITS>(rec + 4 * BITS * part, wds);
  const uint32_t meta = *reinterpret_cast<const uint32_t *>(P.meta + (R * (kHeadDim / P.group) + part / gl) * 4);
  const float s = __half2float(__ushort_as_half((unsigned short)(meta & 0xffffu)));
  const float z = __half2float(__ushort_as_half((unsigned short)(meta >> 16)));
  unpack32<BITS>(wds, q);
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __fmaf_rn((float)q[i], s, z);
}

template <int BITS, bool HAD, bool DELTA = false, bool MIXED = false>
__global__ void __launch_bounds__(kThreads) kvc_dec_tile(const QuantParams P, const __grid_constant__ WidthsArg<MIXED> W) {
  if (P.check_corrupt && (*(volatile uint32_t *)P.status & KVC_FLAG_CORRUPT)) return;
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);
  float *mu_s = Y + 128 * kTS + 2 * 8 * 128;
  float *sc_s = mu_s + 128;
  float *anc_s = sc_s + 128;  // token delta: the block's anchor row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16 = P.g.bf16 != 0;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const int rg = tid >> 4, c8 = tid & 15;
  uint32_t flags = 0;

  for (uint32_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const uint32_t sb = tile % n_sb, lh = tile / n_sb, h = lh % H, l = lh / H;
    const uint32_t t0 = sb * kSmoothBlock;
    const uint32_t nvalid = min((uint32_t)kSmoothBlock, T - t0);

    if (P.smooth && tid < 128) {
      const size_t cell = ((size_t)lh * n_sb + sb) * kHeadDim + tid;
      const uint16_t mub = reinterpret_cast<const uint16_t *>(P.mu)[cell];
      int e = P.ex[cell];
      if (e < -126) e = -126;
      mu_s[tid] = __half2float(__ushort_as_half(mub));
      sc_s[tid] = pow2i(e);
    }
    if (DELTA && tid < 128)
      anc_s[tid] = elt_to_f32(reinterpret_cast<const uint16_t *>(P.anchors)[((size_t)lh * n_sb + sb) * kHeadDim + tid], bf16);

    // ---- D': columns -- dequantize each channel's token groups into the tile
    // (format v1 only: groups over tokens otherwise run in the key-tile kernel)
    if constexpr (!MIXED) if (P.axis == KVC_AXIS_OVER_TOKENS) {
      const int c = tid & 127, half = tid >> 7, pcol = phys_col(c);
      const uint32_t G = P.group;
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const uint32_t row0 = 32 * (2 * half + j);
        const uint32_t tg = (t0 + row0) / G;
        if (tg < P.n_tg) {
          const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + c;
          uint32_t wds[BITS], q[32];
          load_words<BITS>(P.codes + g * (G * BITS / 8) + ((row0 % G) / 32) * 4 * BITS, wds);
          const uint32_t meta = *reinterpret_cast<const uint32_t *>(P.meta + g * 4);
          const float s = __half2float(__ushort_as_half((unsigned short)(meta & 0xffffu)));
          const float z = __half2float(__ushort_as_half((unsigned short)(meta >> 16)));
          unpack32<BITS>(wds, q);
#pragma unroll
          for (int i = 0; i < 32; i++) Y[(row0 + i) * kTS + pcol] = __fmaf_rn((float)q[i], s, z);
        }
      }
    }
    __syncthreads();

    // ---- C': rows -- per-token groups, inverse Hadamard, normalization, signs
    if (HAD || P.axis == KVC_AXIS_OVER_CHANNELS) {
      const int part = lane & 3, rsub = lane >> 2;
      const int gl = (int)(P.group >> 5);
#pragma unroll 1
      for (int k = 0; k < 2; k++) {
        const int r = warp * 16 + k * 8 + rsub;
        float v[32];
        if (P.axis == KVC_AXIS_OVER_CHANNELS) {
#pragma unroll
          for (int i = 0; i < 32; i++) v[i] = 0.0f;
          if ((uint32_t)r < nvalid) {
            const size_t R = ((size_t)l * T + t0 + r) * H + h;
            if constexpr (MIXED) {
              const uint8_t *rec = P.codes + row_code_offset<0, MIXED>(W, T, H, l, t0 + r, h, (uint32_t)R);
              switch (width_of<MIXED>(W, lh)) {
                case 2: tile_row_dequant<2>(P, v, part, gl, rec, R); break;
                case 3: tile_row_dequant<3>(P, v, part, gl, rec, R); break;
                case 4: tile_row_dequant<4>(P, v, part, gl, rec, R); break;
                default: tile_row_dequant<8>(P, v, part, gl, rec, R); break;
              }
            } else {
              tile_row_dequant<BITS>(P, v, part, gl, P.codes + R * (kHeadDim * BITS / 8), R);
            }
          }
        } else {
          tile_row_load(Y, r, part, v);
        }
        if (HAD) {
          fwht128(v, part);
          scale_all(v, hadamard_scale());
          apply_signs(v, P.sign[part]);
        }
        tile_row_store(Y, r, part, v);
      }
    }
    __syncthreads();

    // ---- A': undo the smoothing, round to the element type, write the rows
    uint8_t *lbase = static_cast<uint8_t *>(P.layers[l]);
    float m8[8], s8[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      m8[j] = P.smooth ? mu_s[8 * c8 + j] : 0.0f;
      s8[j] = P.smooth ? sc_s[8 * c8 + j] : 1.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const uint32_t r = rg + 16 * i;
      if (r < nvalid) {
        const float4 *src = reinterpret_cast<const float4 *>(Y + r * kTS);
        const float4 a = src[phys_chunk(2 * c8)], b = src[phys_chunk(2 * c8 + 1)];
        float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (P.smooth) {
#pragma unroll
          for (int j = 0; j < 8; j++) xv[j] = __fmaf_rn(xv[j], s8[j], m8[j]);
        }
        if constexpr (DELTA) {
#pragma unroll
          for (int j = 0; j < 8; j++) xv[j] = __fadd_rn(xv[j], anc_s[8 * c8 + j]);
        }
        const uint64_t ro = row_offset(P.g, t0 + r);
        if (ro == ~0ull) flags |= KVC_FLAG_BAD_PAGE;
        else *reinterpret_cast<uint4 *>(lbase + ro + (size_t)(h * kHeadDim + 8 * c8) * 2) = pack8(xv, bf16);
      }
    }
    __syncthreads();
  }
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// launchers (instantiated by kvc_quant.cu and the format-v2 translation units)
// ---------------------------------------------------------------------------

template <typename K>
static int resident_blocks(K kernel, size_t smem, int threads = kThreads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
  return n;
}

// One launch of `kernel` with `smem` dynamic shared bytes on a grid of at most the
// resident CTAs (at most `cap` per SM when cap > 0) and at most `work_units`.
template <typename K, typename... Args>
static int run_k(K kernel, size_t smem, int threads, int sm_count, int cap, void *stream, uint64_t work_units,
                 const Args &...args) {
  if (smem > 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  int per_sm = resident_blocks(kernel, smem, threads);
  if (cap > 0 && per_sm > cap) per_sm = cap;
  uint64_t blocks = (uint64_t)sm_count * per_sm;
  if (work_units < blocks) blocks = work_units;
  if (blocks == 0) return 0;
  kernel<<<(unsigned)blocks, threads, smem, (cudaStream_t)stream>>>(args...);
  return (int)cudaGetLastError();
}

static bool use_tile(const QuantParams &p) { return p.smooth || p.axis == KVC_AXIS_OVER_TOKENS; }

// The kernel for one tensor of one profile.  BITS is the code width of a uniform
// launch (ignored, 0, when MIXED).
template <int BITS, bool DELTA, bool MIXED>
static int dispatch_v(const QuantParams &p, const TmaMaps *maps, const WidthsArg<MIXED> &W, bool enc, int sm,
                      int cap, void *st, const char **name) {
  static const TmaMaps no_maps = {};
  const bool had = p.hadamard != 0, bf = p.g.bf16 != 0;
  const bool tile = use_tile(p);
  const uint64_t rows = (uint64_t)p.g.L * p.g.T * p.g.H;
  const uint64_t units = tile ? (uint64_t)p.g.L * p.g.H * p.n_sb : (rows + 127) / 128;
  const TmaMaps &M = maps ? *maps : no_maps;
  if (p.axis == KVC_AXIS_OVER_TOKENS) {
    if (enc) {
      *name = "kvc_enc_ktile";
      auto k = had ? (bf ? kvc_enc_ktile<BITS, true, true, DELTA, MIXED> : kvc_enc_ktile<BITS, true, false, DELTA, MIXED>)
                   : (bf ? kvc_enc_ktile<BITS, false, true, DELTA, MIXED> : kvc_enc_ktile<BITS, false, false, DELTA, MIXED>);
      return run_k(k, kKtileSmem, kKT, sm, cap, st, units, p, M, W);
    }
    *name = "kvc_dec_ktile";
    constexpr int SB = MIXED ? 8 : BITS;
    auto k = had ? (bf ? kvc_dec_ktile<BITS, true, true, DELTA, MIXED> : kvc_dec_ktile<BITS, true, false, DELTA, MIXED>)
                 : (bf ? kvc_dec_ktile<BITS, false, true, DELTA, MIXED> : kvc_dec_ktile<BITS, false, false, DELTA, MIXED>);
    return run_k(k, kdec_smem<SB>(p.group, DELTA), kKD, sm, cap, st, units, p, W);
  }
  if (tile) {
    if (enc) {
      *name = "kvc_enc_tile";
      return run_k(had ? kvc_enc_tile<BITS, true, DELTA, MIXED> : kvc_enc_tile<BITS, false, DELTA, MIXED>, kTileSmem,
                   kThreads, sm, cap, st, units, p, W);
    }
    *name = "kvc_dec_tile";
    return run_k(had ? kvc_dec_tile<BITS, true, DELTA, MIXED> : kvc_dec_tile<BITS, false, DELTA, MIXED>, kTileSmem,
                 kThreads, sm, cap, st, units, p, W);
  }
  if (enc) {
    *name = "kvc_enc_rows";
    auto k = had ? (bf ? kvc_enc_rows<BITS, true, true, DELTA, MIXED> : kvc_enc_rows<BITS, true, false, DELTA, MIXED>)
                 : (bf ? kvc_enc_rows<BITS, false, true, DELTA, MIXED> : kvc_enc_rows<BITS, false, false, DELTA, MIXED>);
    return run_k(k, 0, kThreads, sm, cap, st, units, p, W);
  }
  *name = "kvc_dec_rows";
  auto k = had ? (bf ? kvc_dec_rows<BITS, true, true, DELTA, MIXED> : kvc_dec_rows<BITS, true, false, DELTA, MIXED>)
               : (bf ? kvc_dec_rows<BITS, false, true, DELTA, MIXED> : kvc_dec_rows<BITS, false, false, DELTA, MIXED>);
  return run_k(k, MIXED ? kDecRowsSmem : dec_rows_smem(BITS), kThreads, sm, cap, st, units, p, W);
}

// Format-v2 launches (kvc_quant_delta.cu: token delta, uniform widths;
// kvc_quant_mixed.cu: per-(layer, head) widths, with or without the delta).
int launch_quant_delta(const QuantParams &p, const TmaMaps *maps, bool enc, int sm, int cap, void *st,
                       const char **name);
int launch_quant_mixed(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, bool enc, int sm, int cap,
                       void *st, const char **name);

}  // namespace kvc
