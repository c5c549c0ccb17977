// kvc_quant.cu -- launches of the fused transform + quantize + pack (encode) and
// fused reconstruction (decode) kernels of kvc_quant_kernels.cuh: the format-v1
// instantiations here, format-v2 profiles (token delta, per-(layer, head) widths)
// handed to kvc_quant_delta.cu / kvc_quant_mixed.cu.
#include "kvc_quant_kernels.cuh"

namespace kvc {

static int launch(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, bool enc, int sm, int cap,
                  void *st, uint64_t *launches, const char **name) {
  int rc;
  if (p.mixed) {
    rc = widths ? launch_quant_mixed(p, maps, widths, enc, sm, cap, st, name) : (int)cudaErrorInvalidValue;
  } else if (p.delta) {
    rc = launch_quant_delta(p, maps, enc, sm, cap, st, name);
  } else {
    const NoWidths W = {0u};
    switch (p.bits) {
      case 2: rc = dispatch_v<2, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      case 3: rc = dispatch_v<3, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      case 4: rc = dispatch_v<4, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      default: rc = dispatch_v<8, false, false>(p, maps, W, enc, sm, cap, st, name); break;
    }
  }
  if (launches) ++*launches;
  return rc;
}

int launch_quantize(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, int sm_count, int max_per_sm,
                    void *stream, uint64_t *launches, const char **name) {
  return launch(p, maps, widths, true, sm_count, max_per_sm, stream, launches, name);
}

// ---------------------------------------------------------------------------
// Self-check of the quotient step of the encoders (qdiv2 / qsum2) against the
// correctly rounded division: block b takes the binary16 divisor with bits b + 1
// (every positive finite value), each thread 256 dividends from its own linear
// congruential sequence, in four kinds (uniform in [0, 256 s); within 4 ulps of
// k s and of (k + 1/2) s, k < 256, where the code decisions lie; any normal value
// below 2^17).  counts[0]: quotients that differ for t >= 1e-30 (below that the
// quotient underflows and its code is 0 either way), counts[1]: codes (rint of a
// quotient below 4096) that differ, counts[2]: dividends tested.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t qc_next(uint32_t &x) {
  x = x * 1664525u + 1013904223u;
  return x;
}

__device__ __forceinline__ float qc_dividend(uint32_t &x, int kind, float s) {
  const uint32_t k = qc_next(x) >> 24;
  if (kind == 0) return __fmul_rn(__fsub_rn(__uint_as_float(0x3f800000u | (qc_next(x) >> 9)), 1.0f), __fmul_rn(256.0f, s));
  if (kind == 3) return __uint_as_float(qc_next(x) % (0x47FFFFFFu - 0x00800000u) + 0x00800000u);
  const float c = __fmul_rn(kind == 1 ? (float)k + 0.5f : (float)k, s);
  return __uint_as_float(__float_as_uint(c) + (qc_next(x) % 9u) - 4u);  // below 0 or NaN: skipped
}

__global__ void __launch_bounds__(256) kvc_quotient_check(uint32_t seed, unsigned long long *counts) {
  const uint32_t sb = blockIdx.x + 1u;
  const float s = __half2float(__ushort_as_half((unsigned short)sb));
  const float r = __frcp_rn(s);
  const float2 r2 = bcast2(r), ns2 = bcast2(-s);
  uint32_t x = sb * 2654435761u ^ threadIdx.x * 40503u ^ seed * 0x9E3779B9u;
  unsigned long long nq = 0, nc = 0, nt = 0;
  for (int i = 0; i < 128; i++) {
    const float t0 = qc_dividend(x, (2 * i) & 3, s), t1 = qc_dividend(x, (2 * i + 1) & 3, s);
    const float2 d = qdiv2(make_float2(t0, t1), r2, ns2);
    const float2 u = qsum2(make_float2(t0, t1), make_float2(0.0f, 0.0f), r2, ns2);
    const float tt[2] = {t0, t1}, dd[2] = {d.x, d.y}, uu[2] = {u.x, u.y};
#pragma unroll
    for (int h = 0; h < 2; h++) {
      if (!(tt[h] >= 0.0f)) continue;
      nt++;
      const float a = __fdiv_rn(tt[h], s);
      if (tt[h] >= 1.0e-30f && __float_as_uint(a) != __float_as_uint(dd[h])) nq++;
      if (a < 4096.0f && (uint32_t)rintf(a) != (__float_as_uint(uu[h]) & 0xFFFFFu)) nc++;
    }
  }
  if (nq) atomicAdd(counts, nq);
  if (nc) atomicAdd(counts + 1, nc);
  atomicAdd(counts + 2, nt);
}

// The group scale's quotient: range_div<BITS>(w) against __fdiv_rn(w, 2^BITS - 1)
// for every non-negative binary32 bit pattern w (finite, infinite and NaN) and the
// four widths.  counts[3]: quotients that differ for finite w >= 1e-30; counts[4]:
// binary16 scales (rounded up) that differ, for any w; counts[5]: patterns tested.
template <int BITS>
__device__ __forceinline__ void rc_one(float w, unsigned long long &nq, unsigned long long &ns) {
  const float a = __fdiv_rn(w, (float)((1u << BITS) - 1u)), b = range_div<BITS>(w);
  if (w >= 1.0e-30f && fabsf(w) <= 3.402823466e38f && __float_as_uint(a) != __float_as_uint(b)) nq++;
  if (__half_as_ushort(__float2half_ru(a)) != __half_as_ushort(__float2half_ru(b))) ns++;
}

__global__ void __launch_bounds__(256) kvc_range_check(unsigned long long *counts) {
  unsigned long long nq = 0, ns = 0, nt = 0;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < 0x80000000u; u += stride) {
    const float w = __uint_as_float(u);
    rc_one<2>(w, nq, ns);
    rc_one<3>(w, nq, ns);
    rc_one<4>(w, nq, ns);
    rc_one<8>(w, nq, ns);
    nt++;
  }
  if (nq) atomicAdd(counts + 3, nq);
  if (ns) atomicAdd(counts + 4, ns);
  atomicAdd(counts + 5, nt);
}

int launch_quotient_check(uint32_t seed, unsigned long long *d_counts, void *stream) {
  kvc_quotient_check<<<0x7bff, 256, 0, (cudaStream_t)stream>>>(seed, d_counts);
  return (int)cudaGetLastError();
}

int launch_range_check(unsigned long long *d_counts, int sm_count, void *stream) {
  kvc_range_check<<<(unsigned)(sm_count > 0 ? sm_count * 8 : 1024), 256, 0, (cudaStream_t)stream>>>(d_counts);
  return (int)cudaGetLastError();
}

int launch_dequantize(const QuantParams &p, const WidthTable *widths, int sm_count, int max_per_sm, void *stream,
                      uint64_t *launches, const char **name) {
  return launch(p, nullptr, widths, false, sm_count, max_per_sm, stream, launches, name);
}

}  // namespace kvc
