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
// rows: encode
// ---------------------------------------------------------------------------
template <int BITS, bool HAD>
__global__ void __launch_bounds__(kThreads) kvc_enc_rows(const QuantParams P) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = lane & 3, rsub = lane >> 2;
  const bool bf16 = P.g.bf16 != 0;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  const uint32_t n_it = (NR + 7) / 8;
  const int gl = (int)(P.group >> 5);  // lanes per group: 1, 2 or 4
  const uint32_t row_code_bytes = kHeadDim * BITS / 8;
  const uint32_t groups_per_row = kHeadDim / P.group;
  const uint32_t sbits = P.sign[part];
  uint32_t flags = 0;

  for (uint32_t it = blockIdx.x * (kThreads / 32) + warp; it < n_it; it += gridDim.x * (kThreads / 32)) {
    const uint32_t R = it * 8 + rsub;
    const bool valid = R < NR;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = 0.0f;
    if (valid) {
      const uint32_t h = R % H, lt = R / H, t = lt % T, l = lt / T;
      const uint64_t ro = row_offset(P.g, t);
      if (ro == ~0ull) {
        flags |= KVC_FLAG_BAD_PAGE;
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.layers[l]) + ro +
                                                           (size_t)(h * kHeadDim + 32 * part) * 2);
        uint4 w[4];
#pragma unroll
        for (int j = 0; j < 4; j++) w[j] = __ldg(src + j);
#pragma unroll
        for (int j = 0; j < 4; j++) {
          unpack8(w[j], bf16, v + 8 * j);
          if (!all_finite8(v + 8 * j)) flags |= KVC_FLAG_NONFINITE;
        }
      }
    }
    if (HAD) {
      apply_signs(v, sbits);
      fwht128(v, part);
      scale_all(v, hadamard_scale());
    }
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
    float s, z, r;
    uint32_t fl = 0;
    const uint32_t meta = quant_params<BITS>(mn, mx, s, z, r, fl);
    uint32_t q[32];
#pragma unroll
    for (int i = 0; i < 32; i++) q[i] = quant_code<BITS>(v[i], z, s, r);
    uint32_t wds[BITS];
    pack32<BITS>(q, wds);
    if (valid) {
      flags |= fl;
      store_words<BITS>(P.codes + (size_t)R * row_code_bytes + 4 * BITS * part, wds);
      if ((part & (gl - 1)) == 0)
        *reinterpret_cast<uint32_t *>(P.meta + ((size_t)R * groups_per_row + part / gl) * 4) = meta;
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

template <int BITS>
__device__ __forceinline__ void store_codes16(uint8_t *dst, const uint32_t (&q)[16]) {
  if constexpr (BITS == 2) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 16; i++) w |= q[i] << (2 * i);
    *reinterpret_cast<uint32_t *>(dst) = w;
  } else if constexpr (BITS == 4) {
    uint32_t a = 0, b = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      a |= q[i] << (4 * i);
      b |= q[i + 8] << (4 * i);
    }
    *reinterpret_cast<uint2 *>(dst) = make_uint2(a, b);
  } else if constexpr (BITS == 8) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; j++) w[j] = q[4 * j] | (q[4 * j + 1] << 8) | (q[4 * j + 2] << 16) | (q[4 * j + 3] << 24);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // 3 bits: 48 bits = three 16-bit halves (2-byte aligned)
    uint64_t v = 0;
#pragma unroll
    for (int i = 0; i < 16; i++) v |= (uint64_t)q[i] << (3 * i);
    uint16_t *d16 = reinterpret_cast<uint16_t *>(dst);
    d16[0] = (uint16_t)v;
    d16[1] = (uint16_t)(v >> 16);
    d16[2] = (uint16_t)(v >> 32);
  }
}

template <int BITS, bool HAD>
__global__ void __launch_bounds__(kThreads, 2) kvc_enc_ktile(const QuantParams P) {
  extern __shared__ float4 smem_f4[];
  float *Y = reinterpret_cast<float *>(smem_f4);                           // [128][128], swizzled
  uint8_t *stage = reinterpret_cast<uint8_t *>(Y + 128 * 128);              // [128][256] raw rows
  float *red = reinterpret_cast<float *>(stage + 128 * 256);               // [2][8][128]
  float *mu_s = red + 2 * 8 * 128;
  float *inv_s = mu_s + 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16 = P.g.bf16 != 0;
  const uint32_t H = P.g.H, T = P.g.T, n_sb = P.n_sb, G = P.group;
  const uint32_t n_tiles = P.g.L * H * n_sb;
  const int rg = tid >> 4, c8 = tid & 15;
  uint32_t flags = 0;

  uint32_t tile = blockIdx.x;
  if (tile < n_tiles) ktile_issue(P, tile, stage, rg, c8, flags);
  for (; tile < n_tiles; tile += gridDim.x) {
    const uint32_t sb = tile % n_sb, lh = tile / n_sb;
    const uint32_t t0 = sb * kSmoothBlock;
    const uint32_t nvalid = min((uint32_t)kSmoothBlock, T - t0);

    // ---- A: own staged rows -> registers; then start fetching the next tile
    cp_async_wait_all_q();
    float x[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const uint32_t r = rg + 16 * i;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (r < nvalid) w = *reinterpret_cast<const uint4 *>(stage + r * 256 + 16 * c8);
      unpack8(w, bf16, x[i]);
      if (!all_finite8(x[i])) flags |= KVC_FLAG_NONFINITE;
    }
    if (tile + gridDim.x < n_tiles) ktile_issue(P, tile + gridDim.x, stage, rg, c8, flags);

    if (P.smooth) {
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
      if (lane < 16) {
        reinterpret_cast<float4 *>(red + warp * 128 + 8 * c8)[0] = make_float4(mn[0], mn[1], mn[2], mn[3]);
        reinterpret_cast<float4 *>(red + warp * 128 + 8 * c8)[1] = make_float4(mn[4], mn[5], mn[6], mn[7]);
        reinterpret_cast<float4 *>(red + 1024 + warp * 128 + 8 * c8)[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
        reinterpret_cast<float4 *>(red + 1024 + warp * 128 + 8 * c8)[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
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
      const float4 m0 = reinterpret_cast<const float4 *>(mu_s + 8 * c8)[0];
      const float4 m1 = reinterpret_cast<const float4 *>(mu_s + 8 * c8)[1];
      const float4 s0 = reinterpret_cast<const float4 *>(inv_s + 8 * c8)[0];
      const float4 s1 = reinterpret_cast<const float4 *>(inv_s + 8 * c8)[1];
      const float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      const float iv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) x[i][j] = (rg + 16 * i < nvalid) ? __fmul_rn(__fsub_rn(x[i][j], m[j]), iv[j]) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int r = rg + 16 * i;
      float4 *row = reinterpret_cast<float4 *>(Y + r * 128);
      row[kchunk(2 * c8, r)] = make_float4(x[i][0], x[i][1], x[i][2], x[i][3]);
      row[kchunk(2 * c8 + 1, r)] = make_float4(x[i][4], x[i][5], x[i][6], x[i][7]);
    }
    __syncthreads();

    // ---- C: butterfly strides 1..16 along each row
    if (HAD) {
      const int part = lane & 3, rsub = lane >> 2;
      const uint32_t sbits = P.sign[part];
#pragma unroll 1
      for (int k = 0; k < 2; k++) {
        const int r = warp * 16 + k * 8 + rsub;
        float4 *row = reinterpret_cast<float4 *>(Y + r * 128) + 8 * part;
        const int rot = (part + 4 * (r & 1)) & 7;
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; q++) {
          const float4 a = row[(q + rot) & 7];
          v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        }
        apply_signs(v, sbits);
        fwht_in_thread(v);
#pragma unroll
        for (int q = 0; q < 8; q++) row[(q + rot) & 7] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      __syncthreads();
    }

    // ---- D: columns {cq, cq+32, cq+64, cq+96} x tokens 16*warp .. +15
    {
      const int cq = lane, rs = warp;
      float v[4][16];
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int r = 16 * rs + i;
#pragma unroll
        for (int k = 0; k < 4; k++) v[k][i] = Y[r * 128 + kcol(cq + 32 * k, r)];
      }
      if (HAD) {
        const float c = hadamard_scale();
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const float a0 = __fadd_rn(v[0][i], v[1][i]), a1 = __fsub_rn(v[0][i], v[1][i]);
          const float a2 = __fadd_rn(v[2][i], v[3][i]), a3 = __fsub_rn(v[2][i], v[3][i]);
          v[0][i] = __fmul_rn(__fadd_rn(a0, a2), c);
          v[2][i] = __fmul_rn(__fsub_rn(a0, a2), c);
          v[1][i] = __fmul_rn(__fadd_rn(a1, a3), c);
          v[3][i] = __fmul_rn(__fsub_rn(a1, a3), c);
        }
      }
      const int nv = (int)nvalid - 16 * rs;  // valid rows in this segment (may be <= 0)
      float mn[4], mx[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        mn[k] = __int_as_float(0x7f800000);
        mx[k] = __int_as_float(0xff800000);
#pragma unroll
        for (int i = 0; i < 16; i++)
          if (i < nv) {
            mn[k] = fminf(mn[k], v[k][i]);
            mx[k] = fmaxf(mx[k], v[k][i]);
          }
        red[rs * 128 + cq + 32 * k] = mn[k];
        red[1024 + rs * 128 + cq + 32 * k] = mx[k];
      }
      __syncthreads();
      const int spg = (int)(G >> 4);           // 16-token segments per group
      const int s0 = (rs / spg) * spg;         // first segment of this thread's group
      const uint32_t row0 = 16 * rs;
      const uint32_t tg = (t0 + (uint32_t)s0 * 16) / G;
      if (tg < P.n_tg) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int ch = cq + 32 * k;
          float a = red[s0 * 128 + ch], b = red[1024 + s0 * 128 + ch];
          for (int s = 1; s < spg; s++) {
            a = fminf(a, red[(s0 + s) * 128 + ch]);
            b = fmaxf(b, red[1024 + (s0 + s) * 128 + ch]);
          }
          float sc, z, rr;
          const uint32_t meta = quant_params<BITS>(a, b, sc, z, rr, flags);
          uint32_t q[16];
#pragma unroll
          for (int i = 0; i < 16; i++) q[i] = i < nv ? quant_code<BITS>(v[k][i], z, sc, rr) : 0u;
          const size_t g = ((size_t)lh * P.n_tg + tg) * kHeadDim + ch;
          store_codes16<BITS>(P.codes + g * (G * BITS / 8) + ((row0 % G) / 16) * (2 * BITS), q);
          if (row0 % G == 0) *reinterpret_cast<uint32_t *>(P.meta + g * 4) = meta;
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
static int resident_blocks(K kernel, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, smem) != cudaSuccess || n < 1) n = 1;
  return n;
}

template <typename K>
static int run(K kernel, bool tile, const QuantParams &p, int sm_count, void *stream, uint64_t work_units,
               size_t smem_override = 0) {
  const size_t smem = smem_override ? smem_override : (tile ? kTileSmem : 0);
  if (tile) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  const uint64_t want = tile ? work_units : (work_units + 7) / 8;  // tiles, or CTAs of 8 warps x 8 rows
  uint64_t blocks = (uint64_t)sm_count * resident_blocks(kernel, smem);
  if (want < blocks) blocks = want;
  if (blocks == 0) return 0;
  kernel<<<(unsigned)blocks, kThreads, smem, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

static bool use_tile(const QuantParams &p) { return p.smooth || p.axis == KVC_AXIS_OVER_TOKENS; }

template <int BITS>
static int dispatch(const QuantParams &p, bool had, bool enc, int sm, void *st, const char **name) {
  const bool tile = use_tile(p);
  const uint64_t units = tile ? (uint64_t)p.g.L * p.g.H * p.n_sb : ((uint64_t)p.g.L * p.g.T * p.g.H + 7) / 8;
  if (enc) {
    if (p.axis == KVC_AXIS_OVER_TOKENS) {
      *name = "kvc_enc_ktile";
      return had ? run(kvc_enc_ktile<BITS, true>, true, p, sm, st, units, kKtileSmem)
                 : run(kvc_enc_ktile<BITS, false>, true, p, sm, st, units, kKtileSmem);
    }
    if (tile) {
      *name = "kvc_enc_tile";
      return had ? run(kvc_enc_tile<BITS, true>, true, p, sm, st, units)
                 : run(kvc_enc_tile<BITS, false>, true, p, sm, st, units);
    }
    *name = "kvc_enc_rows";
    return had ? run(kvc_enc_rows<BITS, true>, false, p, sm, st, units)
               : run(kvc_enc_rows<BITS, false>, false, p, sm, st, units);
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
