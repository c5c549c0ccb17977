// kvc_quant.cu -- fused transform + quantize + pack (encode) and fused
// reconstruction (decode) for one KV tensor of every layer.
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
//    8 rows (token, head) at a time, 4 lanes per row, 32 channels per lane; the
//    Hadamard butterflies run in registers (strides 1..16) and across the 4 lanes
//    (strides 32, 64).  No shared memory.
//  * tile  -- groups over tokens and/or smoothing (the key default).  A CTA owns a
//    (layer, head, 128-token) tile in shared memory: per-channel statistics over
//    tokens, the row-wise Hadamard pass, then a column pass that quantizes and
//    packs each channel's token group.
#include <cuda_runtime.h>

#include "kvc_device.cuh"

namespace kvc {

constexpr int kThreads = 256;
constexpr int kTS = 144;  // floats per shared-memory tile row (128 + 16: conflict-free row and column access)
constexpr size_t kTileSmem = (size_t)(128 * kTS + 2 * 8 * 128 + 2 * 128) * sizeof(float);

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

template <int BITS, bool HAD, bool BF16>
__global__ void __launch_bounds__(kThreads, 2) kvc_enc_rows(const QuantParams P) {
  __shared__ uint32_t smask[2][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane & 1, rsub = lane >> 1;
  constexpr bool bf16 = BF16;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  const uint32_t n_it = (NR + 15) / 16;
  const uint32_t G = P.group;
  if (HAD && threadIdx.x < 64) {
    const int hh = threadIdx.x >> 5, j = threadIdx.x & 31;  // pair j of half hh: channels 64hh + 2j, +1
    smask[hh][j] = pair_sign_mask(P.sign[2 * hh + (j >> 4)], (2 * j) & 31);
  }
  __syncthreads();
  const float sg = half ? -1.0f : 1.0f;  // stride 64: lower lane a + b, upper lane a - b = -b + a
  uint32_t flags = 0;

  for (uint32_t it = blockIdx.x * (kThreads / 32) + warp; it < n_it; it += gridDim.x * (kThreads / 32)) {
    const uint32_t R = it * 16 + rsub;
    const bool valid = R < NR;
    float2 w[32];
    {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; j++) q[j] = make_uint4(0u, 0u, 0u, 0u);
      if (valid) {
        const uint32_t h = R % H, lt = R / H, t = lt % T, l = lt / T;
        const uint64_t ro = row_offset(P.g, t);
        if (ro == ~0ull) {
          flags |= KVC_FLAG_BAD_PAGE;
        } else {
          const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.layers[l]) + ro +
                                                             (size_t)(h * kHeadDim + 64 * half) * 2);
#pragma unroll
          for (int j = 0; j < 8; j++) q[j] = __ldg(src + j);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; j++) {
        uint32_t r4[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          if (HAD) r4[e] ^= smask[half][4 * j + e];
          w[4 * j + e] = unpack_pair(r4[e], bf16);
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
    uint32_t f0 = 0, f1 = 0;
    const uint32_t meta0 = quant_params<BITS>(mn0, mx0, s0, z0, r0, f0);
    const uint32_t meta1 = quant_params<BITS>(mn1, mx1, s1, z1, r1, f1);
    bool bad = f0 != 0 || f1 != 0;
    uint32_t wds[2 * BITS];
#pragma unroll
    for (int j = 0; j < 2 * BITS; j++) wds[j] = 0u;
    {
      const float2 za = bcast2(z0), ra = bcast2(r0), zb = bcast2(z1), rb = bcast2(r1);
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const float2 u = qfast2<BITS>(w[i], i < 16 ? za : zb, i < 16 ? ra : rb, bad);
        put_code<BITS>(wds, 2 * i, __float_as_uint(u.x));
        put_code<BITS>(wds, 2 * i + 1, __float_as_uint(u.y));
      }
    }
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
      uint8_t *dst = P.codes + (size_t)R * (kHeadDim * BITS / 8) + 8 * BITS * half;
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
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// rows: decode
// ---------------------------------------------------------------------------
template <int BITS, bool HAD>
__global__ void __launch_bounds__(kThreads) kvc_dec_rows(const QuantParams P) {
  if (P.check_corrupt && (*(volatile uint32_t *)P.status & KVC_FLAG_CORRUPT)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = lane & 3, rsub = lane >> 2;
  const bool bf16 = P.g.bf16 != 0;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  const uint32_t n_it = (NR + 7) / 8;
  const int gl = (int)(P.group >> 5);
  const uint32_t row_code_bytes = kHeadDim * BITS / 8;
  const uint32_t groups_per_row = kHeadDim / P.group;
  const uint32_t sbits = P.sign[part];
  uint32_t flags = 0;

  for (uint32_t it = blockIdx.x * (kThreads / 32) + warp; it < n_it; it += gridDim.x * (kThreads / 32)) {
    const uint32_t R = it * 8 + rsub;
    const bool valid = R < NR;
    float v[32];
    if (valid) {
      uint32_t wds[BITS], q[32];
      load_words<BITS>(P.codes + (size_t)R * row_code_bytes + 4 * BITS * part, wds);
      const uint32_t meta =
          *reinterpret_cast<const uint32_t *>(P.meta + ((size_t)R * groups_per_row + part / gl) * 4);
      const float s = __half2float(__ushort_as_half((unsigned short)(meta & 0xffffu)));
      const float z = __half2float(__ushort_as_half((unsigned short)(meta >> 16)));
      unpack32<BITS>(wds, q);
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = __fmaf_rn((float)q[i], s, z);
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = 0.0f;
    }
    if (HAD) {
      fwht128(v, part);
      scale_all(v, hadamard_scale());
      apply_signs(v, sbits);
    }
    if (valid) {
      const uint32_t h = R % H, lt = R / H, t = lt % T, l = lt / T;
      const uint64_t ro = row_offset(P.g, t);
      if (ro == ~0ull) {
        flags |= KVC_FLAG_BAD_PAGE;
      } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.layers[l]) + ro +
                                               (size_t)(h * kHeadDim + 32 * part) * 2);
#pragma unroll
        for (int j = 0; j < 4; j++) dst[j] = pack8(v + 8 * j, bf16);
      }
    }
  }
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
template <int BITS, bool HAD>
__global__ void __launch_bounds__(kThreads) kvc_enc_tile(const QuantParams P) {
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);  // [128][kTS]
  float *red = Y + 128 * kTS;                     // [2][8][128]
  float *mu_s = red + 2 * 8 * 128;                // [128]
  float *inv_s = mu_s + 128;                      // [128]
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
          if ((uint32_t)r < nvalid) {
            flags |= fl;
            const size_t R = ((size_t)l * T + t0 + r) * H + h;
            store_words<BITS>(P.codes + R * (kHeadDim * BITS / 8) + 4 * BITS * part, wds);
            if ((part & (gl - 1)) == 0)
              *reinterpret_cast<uint32_t *>(P.meta + (R * (kHeadDim / P.group) + part / gl) * 4) = meta;
          }
        } else {
          tile_row_store(Y, r, part, v);
        }
      }
      __syncthreads();
    }

    // ---- D: columns -- groups of G tokens per channel
    if (P.axis == KVC_AXIS_OVER_TOKENS) {
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
// Per (layer, head, 128-token) tile, 256 threads:
//  A  each thread reads 8 rows x 8 channels of the raw tile from the stage buffer
//     (filled by cp.async during the previous tile), takes the smoothing
//     statistics, applies the smoothing and stores x' into Y;
//  C  (Hadamard) a lane owns 32 consecutive channels of a row and runs the
//     butterfly strides 1..16 in registers;
//  D  a thread owns channels {c, c+32, c+64, c+96} x 16 tokens: strides 32 and 64
//     in registers, normalization, per-channel group statistics (combined across
//     the token segments through shared memory), quantization and packing of
//     its 16 codes per channel straight into the channel's record.
// Y has no padding: float4 chunk q of part p (32 channels) of row r sits at
// chunk 8p + ((q + p + 4(r & 1)) & 7), which keeps the row pass, the column pass
// and the phase-A stores free of bank conflicts.
// ---------------------------------------------------------------------------
constexpr size_t kKtileSmem = (size_t)128 * 128 * 4 + 128 * 256 + 2 * 8 * 128 * 4 + 2 * 128 * 4;

__device__ __forceinline__ int kchunk(int lc, int r) {
  const int p = lc >> 3, q = lc & 7;
  return 8 * p + ((q + p + 4 * (r & 1)) & 7);
}
__device__ __forceinline__ int kcol(int col, int r) { return 4 * kchunk(col >> 2, r) + (col & 3); }

__device__ __forceinline__ void cp_async16_q(void *smem, const void *gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit_q() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_q() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Copy the raw rows of `tile` this thread will read in phase A (rows rg + 16i,
// 16-byte chunk c8) into the stage buffer; absent rows are zero-filled.
__device__ __forceinline__ void ktile_issue(const QuantParams &P, uint32_t tile, uint8_t *stage, int rg, int c8,
                                            uint32_t &flags) {
  const uint32_t n_sb = P.n_sb, H = P.g.H;
  const uint32_t sb = tile % n_sb, lh = tile / n_sb, h = lh % H, l = lh / H;
  const uint32_t t0 = sb * kSmoothBlock, nvalid = min((uint32_t)kSmoothBlock, P.g.T - t0);
  const uint8_t *lbase = static_cast<const uint8_t *>(P.layers[l]);
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const uint32_t r = rg + 16 * i;
    uint8_t *dst = stage + r * 256 + 16 * c8;
    if (r < nvalid) {
      const uint64_t ro = row_offset(P.g, t0 + r);
      if (ro == ~0ull) {
        flags |= KVC_FLAG_BAD_PAGE;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
      } else {
        cp_async16_q(dst, lbase + ro + (size_t)(h * kHeadDim + 8 * c8) * 2);
      }
    }
  }
  cp_async_commit_q();
}

// 16 codes (BITS each) -> the channel's 2*BITS bytes inside its record.
template <int BITS>
__device__ __forceinline__ void store_code_words(uint8_t *dst, const uint32_t (&w)[(16 * BITS + 31) / 32]) {
  if constexpr (BITS == 2) {
    *reinterpret_cast<uint32_t *>(dst) = w[0];
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
  } else if constexpr (BITS == 8) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // 48 bits, 2-byte aligned
    uint16_t *d16 = reinterpret_cast<uint16_t *>(dst);
    d16[0] = (uint16_t)w[0];
    d16[1] = (uint16_t)(w[0] >> 16);
    d16[2] = (uint16_t)w[1];
  }
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

// Key tile with 512 threads (kvc_enc_ktile): per (layer, head, 128-token) tile
//  A  thread (rg = tid/16, c8 = tid%16) takes rows rg + 32i (i < 4) x 8 channels
//     from the stage buffer; smoothing statistics combine through the idle tile
//     buffer; the smoothed rows (signs folded into the power-of-two scale) go to Y;
//  C  one row per lane quarter-warp: butterfly strides 1..16 in registers;
//  D  thread (cq = lane, rs = warp) takes channels {cq + 32k} x rows 8rs .. 8rs+7:
//     strides 32/64 and the normalization in registers, per-channel statistics of
//     its 8 rows; one thread per (group, channel) then turns the segment partials
//     into the group's parameters (written once to a shared table and to the
//     metadata section); every thread quantizes and packs its 8 codes per channel.
constexpr int kKT = 512;
constexpr size_t kKtile3Smem = (size_t)128 * 128 * 4 + 128 * 256 + 4 * 128 * 16 + 2 * 128 * 4;

__device__ __forceinline__ void ktile3_issue(const QuantParams &P, uint32_t tile, uint8_t *stage, int rg, int c8,
                                             uint32_t &flags) {
  const uint32_t n_sb = P.n_sb, H = P.g.H;
  const uint32_t sb = tile % n_sb, lh = tile / n_sb, h = lh % H, l = lh / H;
  const uint32_t t0 = sb * kSmoothBlock, nvalid = min((uint32_t)kSmoothBlock, P.g.T - t0);
  const uint8_t *lbase = static_cast<const uint8_t *>(P.layers[l]) + (size_t)(h * kHeadDim + 8 * c8) * 2;
  uint8_t *dst = stage + rg * 256 + 16 * c8;
  if (!P.g.block_table) {
    const uint64_t ts = P.g.token_stride;
    const uint8_t *src = lbase + (uint64_t)(t0 + rg) * ts;
#pragma unroll
    for (int i = 0; i < 4; i++)
      if (rg + 32 * i < (int)nvalid) cp_async16_q(dst + i * 32 * 256, src + (uint64_t)i * 32 * ts);
  } else {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t r = rg + 32 * i;
      if (r < nvalid) {
        const uint64_t ro = row_offset(P.g, t0 + r);
        if (ro == ~0ull) {
          flags |= KVC_FLAG_BAD_PAGE;
          *reinterpret_cast<uint4 *>(dst + i * 32 * 256) = make_uint4(0u, 0u, 0u, 0u);
        } else {
          cp_async16_q(dst + i * 32 * 256, lbase + ro);
        }
      }
    }
  }
  cp_async_commit_q();
}

template <int BITS>
__device__ __forceinline__ void store_codes8(uint8_t *dst, uint32_t lo, uint32_t hi) {
  if constexpr (BITS == 2) *reinterpret_cast<uint16_t *>(dst) = (uint16_t)lo;
  else if constexpr (BITS == 4) *reinterpret_cast<uint32_t *>(dst) = lo;
  else if constexpr (BITS == 8) *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
  else {
    dst[0] = (uint8_t)lo;
    dst[1] = (uint8_t)(lo >> 8);
    dst[2] = (uint8_t)(lo >> 16);
  }
}

template <int BITS, bool HAD, bool BF16>
__global__ void __launch_bounds__(kKT, 2) kvc_enc_ktile(const QuantParams P) {
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);                       // [128][128] swizzled; also reduction space
  uint8_t *stage = reinterpret_cast<uint8_t *>(Y + 128 * 128);          // [128][256] raw rows of the next tile
  float4 *prm = reinterpret_cast<float4 *>(stage + 128 * 256);          // [4 groups][128] {z, r, s, meta}
  float *mu_s = reinterpret_cast<float *>(prm + 4 * 128);
  float *inv_s = mu_s + 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr bool bf16 = BF16;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb, G = P.group;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const int rg = tid >> 4, c8 = tid & 15;
  const bool smooth = P.smooth != 0;
  uint32_t flags = 0;

  // tile-invariant quantities
  const int spg = (int)(G >> 3);                      // 8-row segments per group
  const int tiles_groups = 128 / (int)G;              // token groups per tile
  const int my_gi = (8 * warp) / (int)G;              // phase-D group of this warp's rows
  const uint32_t rec_bytes = G * BITS / 8;
  const uint32_t my_seg_off = (uint32_t)(((8 * warp) % (int)G) / 8) * BITS;
  const int chA = kchunk(2 * c8, rg), chB = kchunk(2 * c8 + 1, rg);  // phase-A store chunks (rg parity fixed)
  // phase-D column offsets: channel cq + 32k of an even / odd row
  int coff[8];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    coff[2 * k] = kcol(lane + 32 * k, 0);
    coff[2 * k + 1] = kcol(lane + 32 * k, 1);
  }

  uint32_t tile = blockIdx.x;
  if (tile < n_tiles) ktile3_issue(P, tile, stage, rg, c8, flags);
  for (; tile < n_tiles; tile += gridDim.x) {
    const uint32_t sb = tile % n_sb, lh = tile / n_sb;
    const uint32_t t0 = sb * kSmoothBlock;
    const uint32_t nvalid = min((uint32_t)kSmoothBlock, T - t0);

    // ---- A
    cp_async_wait_all_q();
    float2 x[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t r = rg + 32 * i;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (r < nvalid) w = *reinterpret_cast<const uint4 *>(stage + r * 256 + 16 * c8);
      x[i][0] = unpack_pair(w.x, bf16);
      x[i][1] = unpack_pair(w.y, bf16);
      x[i][2] = unpack_pair(w.z, bf16);
      x[i][3] = unpack_pair(w.w, bf16);
    }
    if (tile + gridDim.x < n_tiles) ktile3_issue(P, tile + gridDim.x, stage, rg, c8, flags);

    if (smooth) {
      float mn[8], mx[8];
#pragma unroll
      for (int j = 0; j < 4; j++) {
        mn[2 * j] = mx[2 * j] = x[0][j].x;
        mn[2 * j + 1] = mx[2 * j + 1] = x[0][j].y;
      }
      if (nvalid == 128) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
          mn[2 * j] = fmin3_n(mn[2 * j], x[1][j].x, x[2][j].x);
          mn[2 * j] = fmin_n(mn[2 * j], x[3][j].x);
          mx[2 * j] = fmax3_n(mx[2 * j], x[1][j].x, x[2][j].x);
          mx[2 * j] = fmax_n(mx[2 * j], x[3][j].x);
          mn[2 * j + 1] = fmin3_n(mn[2 * j + 1], x[1][j].y, x[2][j].y);
          mn[2 * j + 1] = fmin_n(mn[2 * j + 1], x[3][j].y);
          mx[2 * j + 1] = fmax3_n(mx[2 * j + 1], x[1][j].y, x[2][j].y);
          mx[2 * j + 1] = fmax_n(mx[2 * j + 1], x[3][j].y);
        }
      } else {
#pragma unroll
        for (int i = 1; i < 4; i++)
          if (rg + 32 * i < (int)nvalid)
#pragma unroll
            for (int j = 0; j < 4; j++) {
              mn[2 * j] = fmin_n(mn[2 * j], x[i][j].x);
              mx[2 * j] = fmax_n(mx[2 * j], x[i][j].x);
              mn[2 * j + 1] = fmin_n(mn[2 * j + 1], x[i][j].y);
              mx[2 * j + 1] = fmax_n(mx[2 * j + 1], x[i][j].y);
            }
      }
      const bool mine = rg < (int)nvalid, other = (rg ^ 1) < (int)nvalid;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float oa = __shfl_xor_sync(kFull, mn[j], 16), ob = __shfl_xor_sync(kFull, mx[j], 16);
        if (!mine) { mn[j] = oa; mx[j] = ob; }
        else if (other) { mn[j] = fmin_n(mn[j], oa); mx[j] = fmax_n(mx[j], ob); }
      }
      float *red = Y;  // [16 warps][128] minima, then maxima
      if (lane < 16) {
        reinterpret_cast<float4 *>(red + warp * 128 + 8 * c8)[0] = make_float4(mn[0], mn[1], mn[2], mn[3]);
        reinterpret_cast<float4 *>(red + warp * 128 + 8 * c8)[1] = make_float4(mn[4], mn[5], mn[6], mn[7]);
        reinterpret_cast<float4 *>(red + 2048 + warp * 128 + 8 * c8)[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
        reinterpret_cast<float4 *>(red + 2048 + warp * 128 + 8 * c8)[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
      }
      __syncthreads();
      if (tid < 128) {
        float a = red[tid], b = red[2048 + tid];
        for (int k = 1; k < 16; k++) {
          if (2 * k < (int)nvalid) {  // warp k holds rows 2k, 2k+1, 2k+32, ...
            a = fmin_n(a, red[k * 128 + tid]);
            b = fmax_n(b, red[2048 + k * 128 + tid]);
          }
        }
        if (!finite2(a, b)) flags |= KVC_FLAG_NONFINITE;
        float mu, inv;
        uint32_t mub;
        int e;
        smooth_params(a, b, mu, inv, mub, e, flags);
        if (HAD && ((P.sign[tid >> 5] >> (tid & 31)) & 1u)) inv = -inv;  // sign folded into the exact scale
        mu_s[tid] = mu;
        inv_s[tid] = inv;
        const size_t cell = ((size_t)lh * n_sb + sb) * kHeadDim + tid;
        reinterpret_cast<uint16_t *>(P.mu)[cell] = (uint16_t)mub;
        P.ex[cell] = (int8_t)e;
      }
      __syncthreads();
      const float4 m0 = reinterpret_cast<const float4 *>(mu_s + 8 * c8)[0];
      const float4 m1 = reinterpret_cast<const float4 *>(mu_s + 8 * c8)[1];
      const float4 s0 = reinterpret_cast<const float4 *>(inv_s + 8 * c8)[0];
      const float4 s1 = reinterpret_cast<const float4 *>(inv_s + 8 * c8)[1];
      const float2 m[4] = {make_float2(m0.x, m0.y), make_float2(m0.z, m0.w), make_float2(m1.x, m1.y),
                           make_float2(m1.z, m1.w)};
      const float2 iv[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                            make_float2(s1.z, s1.w)};
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) x[i][j] = mul2(sub2(x[i][j], m[j]), iv[j]);
      if (nvalid < 128) {
#pragma unroll
        for (int i = 0; i < 4; i++)
          if (rg + 32 * i >= (int)nvalid)
#pragma unroll
            for (int j = 0; j < 4; j++) x[i][j] = make_float2(0.0f, 0.0f);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
      float4 *row = reinterpret_cast<float4 *>(Y + (rg + 32 * i) * 128);
      row[chA] = make_float4(x[i][0].x, x[i][0].y, x[i][1].x, x[i][1].y);
      row[chB] = make_float4(x[i][2].x, x[i][2].y, x[i][3].x, x[i][3].y);
    }
    __syncthreads();

    // ---- C
    if (HAD) {
      const int part = lane & 3, r = warp * 8 + (lane >> 2);
      float4 *row = reinterpret_cast<float4 *>(Y + r * 128) + 8 * part;
      const int rot = (part + 4 * (r & 1)) & 7;
      float2 w[16];
#pragma unroll
      for (int q = 0; q < 8; q++) {
        const float4 a = row[(q + rot) & 7];
        w[2 * q] = make_float2(a.x, a.y);
        w[2 * q + 1] = make_float2(a.z, a.w);
      }
      if (!smooth) {
        const uint32_t sbits = P.sign[part];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          w[i].x = __uint_as_float(__float_as_uint(w[i].x) ^ (((sbits >> (2 * i)) & 1u) << 31));
          w[i].y = __uint_as_float(__float_as_uint(w[i].y) ^ (((sbits >> (2 * i + 1)) & 1u) << 31));
        }
      }
      fwht32_pairs(w);
#pragma unroll
      for (int q = 0; q < 8; q++) row[(q + rot) & 7] = make_float4(w[2 * q].x, w[2 * q].y, w[2 * q + 1].x, w[2 * q + 1].y);
      __syncthreads();
    }

    // ---- D1: 8 rows x 4 channels into registers, strides 32 / 64, per-channel partials
    const int cq = lane, rs = warp;
    const int nv = (int)nvalid - 8 * rs;
    float2 v[4][4];
    {
      const float *Yr = Y + 8 * rs * 128;
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int k = 0; k < 4; k++)
          v[k][i] = make_float2(Yr[2 * i * 128 + coff[2 * k]], Yr[(2 * i + 1) * 128 + coff[2 * k + 1]]);
    }
    if (HAD) {
      const float2 c2 = bcast2(hadamard_scale());
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float2 a0 = add2(v[0][i], v[1][i]), a1 = sub2(v[0][i], v[1][i]);
        const float2 a2 = add2(v[2][i], v[3][i]), a3 = sub2(v[2][i], v[3][i]);
        v[0][i] = mul2(add2(a0, a2), c2);
        v[2][i] = mul2(sub2(a0, a2), c2);
        v[1][i] = mul2(add2(a1, a3), c2);
        v[3][i] = mul2(sub2(a1, a3), c2);
      }
    }
    float pmn[4], pmx[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      if (nv >= 8) {
        pmn[k] = fmin3_n(fmin_n(v[k][0].x, v[k][0].y), v[k][1].x, v[k][1].y);
        pmx[k] = fmax3_n(fmax_n(v[k][0].x, v[k][0].y), v[k][1].x, v[k][1].y);
        pmn[k] = fmin3_n(fmin3_n(pmn[k], v[k][2].x, v[k][2].y), v[k][3].x, v[k][3].y);
        pmx[k] = fmax3_n(fmax3_n(pmx[k], v[k][2].x, v[k][2].y), v[k][3].x, v[k][3].y);
      } else {
        pmn[k] = pmx[k] = v[k][0].x;
#pragma unroll
        for (int i = 0; i < 4; i++) {
          if (2 * i < nv) { pmn[k] = fmin_n(pmn[k], v[k][i].x); pmx[k] = fmax_n(pmx[k], v[k][i].x); }
          if (2 * i + 1 < nv) { pmn[k] = fmin_n(pmn[k], v[k][i].y); pmx[k] = fmax_n(pmx[k], v[k][i].y); }
        }
      }
    }
    __syncthreads();  // every thread has read Y: its space holds the partials now
    float *red = Y;   // [16 segments][128] minima at 0, maxima at 2048
#pragma unroll
    for (int k = 0; k < 4; k++) {
      red[rs * 128 + cq + 32 * k] = pmn[k];
      red[2048 + rs * 128 + cq + 32 * k] = pmx[k];
    }
    __syncthreads();

    // ---- D2: one thread per (group, channel) of the tile
    {
      const int nseg_valid = (int)((nvalid + 7) / 8);
      const uint32_t tg_base = sb * tiles_groups;    // first token group of the tile
      for (int j = tid; j < tiles_groups * 128; j += kKT) {
        const int gi = j >> 7, ch = j & 127;
        const int s0 = gi * spg;
        const uint32_t tg = tg_base + gi;
        if (s0 < nseg_valid && tg < P.n_tg) {
          float a = red[s0 * 128 + ch], b = red[2048 + s0 * 128 + ch];
          const int ns = min(spg, nseg_valid - s0);
          for (int sg = 1; sg < ns; sg++) {
            a = fmin_n(a, red[(s0 + sg) * 128 + ch]);
            b = fmax_n(b, red[2048 + (s0 + sg) * 128 + ch]);
          }
          if (!finite2(a, b)) flags |= KVC_FLAG_NONFINITE;
          float sc, z, rr;
          uint32_t fl = 0;
          const uint32_t meta = quant_params<BITS>(a, b, sc, z, rr, fl);
          flags |= fl;
          // a saturated group (fl != 0) is marked by r = NaN: its codes take the exact path
          prm[gi * 128 + ch] = make_float4(z, fl ? __int_as_float(0x7fc00000) : rr, sc, __uint_as_float(meta));
          const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + ch;
          *reinterpret_cast<uint32_t *>(P.meta + g * 4) = meta;
        }
      }
    }
    __syncthreads();

    // ---- D3: codes
    {
      const uint32_t tg = sb * tiles_groups + my_gi;
      if (tg < P.n_tg) {  // a segment past the end of an existing group still writes its (zero) codes
        const int gi = my_gi;
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int ch = cq + 32 * k;
          const float4 pp = prm[gi * 128 + ch];
          const float z = pp.x, rr = pp.y, sc = pp.z;
          bool bad = false;
          uint32_t cw[2] = {0u, 0u};
          const float2 z2 = bcast2(z), r2 = bcast2(rr);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 u = qfast2<BITS>(v[k][i], z2, r2, bad);
            put_code<BITS>(cw, 2 * i, __float_as_uint(u.x));
            put_code<BITS>(cw, 2 * i + 1, __float_as_uint(u.y));
          }
          if (__any_sync(kFull, bad)) {
            if (bad) {
              cw[0] = cw[1] = 0u;
#pragma unroll
              for (int i = 0; i < 4; i++) {
                put_code<BITS>(cw, 2 * i, qexact<BITS>(v[k][i].x, z, sc));
                put_code<BITS>(cw, 2 * i + 1, qexact<BITS>(v[k][i].y, z, sc));
              }
            }
          }
          if (nv < 8) {  // codes of rows past the end are 0
            const int keep = (nv > 0 ? nv : 0) * BITS;
            if (keep < 32) { cw[0] &= (1u << keep) - 1u; cw[1] = 0u; }
            else if (keep < 64) cw[1] &= (1u << (keep - 32)) - 1u;
          }
          const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + ch;
          store_codes8<BITS>(P.codes + g * rec_bytes + my_seg_off, cw[0], cw[1]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait_all_q();
  if (flags) atomicOr(P.status, flags);
}

// ---------------------------------------------------------------------------
// tile: decode
// ---------------------------------------------------------------------------
template <int BITS, bool HAD>
__global__ void __launch_bounds__(kThreads) kvc_dec_tile(const QuantParams P) {
  if (P.check_corrupt && (*(volatile uint32_t *)P.status & KVC_FLAG_CORRUPT)) return;
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);
  float *mu_s = Y + 128 * kTS + 2 * 8 * 128;
  float *sc_s = mu_s + 128;
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

    // ---- D': columns -- dequantize each channel's token groups into the tile
    if (P.axis == KVC_AXIS_OVER_TOKENS) {
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
            uint32_t wds[BITS], q[32];
            load_words<BITS>(P.codes + R * (kHeadDim * BITS / 8) + 4 * BITS * part, wds);
            const uint32_t meta =
                *reinterpret_cast<const uint32_t *>(P.meta + (R * (kHeadDim / P.group) + part / gl) * 4);
            const float s = __half2float(__ushort_as_half((unsigned short)(meta & 0xffffu)));
            const float z = __half2float(__ushort_as_half((unsigned short)(meta >> 16)));
            unpack32<BITS>(wds, q);
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] = __fmaf_rn((float)q[i], s, z);
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
// launchers
// ---------------------------------------------------------------------------
template <typename K>
static int resident_blocks(K kernel, size_t smem, int threads = kThreads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
  return n;
}

template <typename K>
static int run(K kernel, bool tile, const QuantParams &p, int sm_count, void *stream, uint64_t work_units,
               size_t smem_override = 0, int threads = kThreads) {
  const size_t smem = smem_override ? smem_override : (tile ? kTileSmem : 0);
  if (tile) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  const uint64_t want = work_units;  // tiles, or CTAs of 8 warps
  uint64_t blocks = (uint64_t)sm_count * resident_blocks(kernel, smem, threads);
  if (want < blocks) blocks = want;
  if (blocks == 0) return 0;
  kernel<<<(unsigned)blocks, threads, smem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

static bool use_tile(const QuantParams &p) { return p.smooth || p.axis == KVC_AXIS_OVER_TOKENS; }

template <int BITS>
static int dispatch(const QuantParams &p, bool had, bool enc, int sm, void *st, const char **name) {
  const bool tile = use_tile(p);
  const uint64_t rows = (uint64_t)p.g.L * p.g.T * p.g.H;
  const uint64_t units = tile ? (uint64_t)p.g.L * p.g.H * p.n_sb : (enc ? (rows + 127) / 128 : (rows + 63) / 64);
  if (enc) {
    if (p.axis == KVC_AXIS_OVER_TOKENS) {
      *name = "kvc_enc_ktile";
      if (p.g.bf16)
        return had ? run(kvc_enc_ktile<BITS, true, true>, true, p, sm, st, units, kKtile3Smem, kKT)
                   : run(kvc_enc_ktile<BITS, false, true>, true, p, sm, st, units, kKtile3Smem, kKT);
      return had ? run(kvc_enc_ktile<BITS, true, false>, true, p, sm, st, units, kKtile3Smem, kKT)
                 : run(kvc_enc_ktile<BITS, false, false>, true, p, sm, st, units, kKtile3Smem, kKT);
    }
    if (tile) {
      *name = "kvc_enc_tile";
      return had ? run(kvc_enc_tile<BITS, true>, true, p, sm, st, units)
                 : run(kvc_enc_tile<BITS, false>, true, p, sm, st, units);
    }
    *name = "kvc_enc_rows";
    if (p.g.bf16)
      return had ? run(kvc_enc_rows<BITS, true, true>, false, p, sm, st, units)
                 : run(kvc_enc_rows<BITS, false, true>, false, p, sm, st, units);
    return had ? run(kvc_enc_rows<BITS, true, false>, false, p, sm, st, units)
               : run(kvc_enc_rows<BITS, false, false>, false, p, sm, st, units);
  }
  if (tile) {
    *name = "kvc_dec_tile";
    return had ? run(kvc_dec_tile<BITS, true>, true, p, sm, st, units)
               : run(kvc_dec_tile<BITS, false>, true, p, sm, st, units);
  }
  *name = "kvc_dec_rows";
  return had ? run(kvc_dec_rows<BITS, true>, false, p, sm, st, units)
             : run(kvc_dec_rows<BITS, false>, false, p, sm, st, units);
}

static int dispatch_bits(const QuantParams &p, bool enc, int sm, void *st, uint64_t *launches, const char **name) {
  const bool had = p.hadamard != 0;
  int rc;
  switch (p.bits) {
    case 2: rc = dispatch<2>(p, had, enc, sm, st, name); break;
    case 3: rc = dispatch<3>(p, had, enc, sm, st, name); break;
    case 4: rc = dispatch<4>(p, had, enc, sm, st, name); break;
    default: rc = dispatch<8>(p, had, enc, sm, st, name); break;
  }
  if (launches) ++*launches;
  return rc;
}

int launch_quantize(const QuantParams &p, int sm_count, void *stream, uint64_t *launches, const char **name) {
  return dispatch_bits(p, true, sm_count, stream, launches, name);
}

int launch_dequantize(const QuantParams &p, int sm_count, void *stream, uint64_t *launches, const char **name) {
  return dispatch_bits(p, false, sm_count, stream, launches, name);
}

}  // namespace kvc
