// kvc_fused.cu -- the value encoder whose code chunks never pass through the
// payload: each CTA quantizes the rows of one lossless chunk of the value-code
// section into shared memory, runs the chunk's stages there and publishes it into
// the stream through the same decoupled look-back as the lossless encoder
// ("Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
// Serving", §3 design goal G1: closely coupled operations in one kernel; §4.1: the
// quantized output goes on to lossless encoding; §4.2: chunked stages and a
// device-resident stream).  The stream is byte for byte the one the unfused path
// writes: the chunk boundaries are the format's, so only profiles whose value-code
// section starts on a chunk boundary and whose chunks hold whole rows take it.
#include "kvc_lossless_dev.cuh"
#include "kvc_quant_kernels.cuh"

namespace kvc {

// Per CTA: tickets over the section's whole chunks, in order.  Chunk t's rows
// (a multiple of 128) are quantized by the 8 warps, 16 rows per warp step, into
// shared buffer t % 2; the stored form follows from the fast stage path (the size
// from the chunk as loaded, published at once for the successors' look-back; the
// transform only for a chunk that compresses).  Chunk t's own look-back, chunk
// table entry and the bulk copy into the stream run one chunk later, after chunk
// t + 1 is quantized, so that its predecessors have had a chunk's time to publish
// their sizes (taken right after it, the look-back waits on chunks still being
// quantized: measured slower).
// Rows past the last whole chunk go to the payload's code section, for the
// lossless launch that follows.
template <int BITS, bool HAD, bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
    kvc_enc_rows_lc(const QuantParams P, const LosslessParams L, const FastSpec F, uint32_t c0, uint32_t nfull) {
  static_assert(kThreads == FT, "the stage passes use every thread of the CTA");
  extern __shared__ uint4 smem_u4[];
  __shared__ uint32_t smask[2][32];
  __shared__ uint32_t s_t;
  const uint32_t cb = L.chunk_bytes, slot = cb + 64;
  uint8_t *const buf0 = reinterpret_cast<uint8_t *>(smem_u4);
  uint8_t *const buf1 = buf0 + slot;
  uint8_t *const A = buf1 + slot;                              // transform output
  uint32_t *const wsum = reinterpret_cast<uint32_t *>(A + slot);  // 64 words of scan scratch
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane & 1, rsub = lane >> 1;
  const uint32_t H = P.g.H, T = P.g.T;
  const uint32_t NR = P.g.L * T * H;
  constexpr uint32_t rec = 16 * BITS;  // code bytes of a row
  const uint32_t rpc = cb / rec;        // rows per chunk
  if (HAD && threadIdx.x < 64) {
    const int hh = threadIdx.x >> 5, j = threadIdx.x & 31;
    smask[hh][j] = pair_sign_mask(P.sign[2 * hh + (j >> 4)], (2 * j) & 31);
  }
  __syncthreads();
  uint32_t flags = 0;
  const uint32_t da = 128u % H, db = (128u / H) % T, dl = 128u / H / T;  // 128 rows on

  bool have_prev = false;  // a chunk quantized in the previous iteration, not yet in the stream
  uint32_t prev_c = 0, prev_size = 0;
  bool prev_raw = false;
  for (uint32_t it = 0;; it++) {
    if (threadIdx.x == 0) s_t = atomicAdd(L.ctrl + L.ticket_word, 1u);
    __syncthreads();
    const uint32_t t = s_t;
    uint8_t *const S = (it & 1u) ? buf1 : buf0;
    uint32_t c = 0, size = 0;
    bool raw = true;
    if (t < nfull) {
      // S last held chunk it - 2, whose copy was issued in the previous iteration
      if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncthreads();
      const uint32_t Rb = t * rpc;
      RowPos pos;
      pos.init(Rb + 16 * warp + rsub, H, T);
      for (uint32_t k = 0; k < rpc / 128; k++) {
        const uint32_t l = pos.l, tt = pos.b, h = pos.a;
        pos.advance(da, db, dl, H, T);
        const uint32_t R = (l * T + tt) * H + h;
        enc_row<BITS, HAD, BF16, false>(P, smask, half, true, l, tt, h, R, S + (size_t)(R - Rb) * rec, flags);
      }
      __syncthreads();
      c = c0 + t;
      uint32_t es;
      if (F.rze_w == 2) es = F.delta1 ? fast_size_bit8<2, true>(S, cb, wsum) : fast_size_bit8<2, false>(S, cb, wsum);
      else es = F.delta1 ? fast_size_bit8<1, true>(S, cb, wsum) : fast_size_bit8<1, false>(S, cb, wsum);
      if (threadIdx.x == 0) publish_size(L, c, align16u(es < cb ? es : cb));
      size = cb;
      raw = es >= cb;
      if (!raw) {
        fast_transform<true>(S, A, cb);
        uint32_t rs;
        if (F.rze_w == 2)
          rs = F.delta1 ? fast_delta_rze<2, true>(A, S, cb, wsum, L, c, false)
                        : fast_delta_rze<2, false>(A, S, cb, wsum, L, c, false);
        else
          rs = F.delta1 ? fast_delta_rze<1, true>(A, S, cb, wsum, L, c, false)
                        : fast_delta_rze<1, false>(A, S, cb, wsum, L, c, false);
        if (rs != es && threadIdx.x == 0)  // the two size computations must agree
          atomicOr(L.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CORRUPT);
        raw = rs >= cb;  // then nothing was written over S: it still holds the codes
        if (!raw) size = rs;
      }
      if (!raw && threadIdx.x < align16u(size) - size) S[size + threadIdx.x] = 0;
      // the bulk copy reads S through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
    }
    if (have_prev && warp == 0) {  // the previous chunk into the stream
      const uint32_t asz = align16u(prev_size);
      const uint64_t excl = prev_c ? lookback_excl(L, prev_c) : 0ull;
      if (lane == 0) {
        if (prev_c && (int64_t)prev_c != L.skip_ticket) st_word64(L.state + prev_c, kFlagIncl | (excl + asz));
        reinterpret_cast<uint32_t *>(L.stream + L.header_bytes)[prev_c] = prev_size | (prev_raw ? 0x80000000u : 0u);
        const uint64_t dst = L.data_start + excl;
        if (dst + asz > L.stream_cap) {
          atomicOr(L.ctrl + kCtrlFlags, (uint32_t)KVC_FLAG_CAPACITY);
        } else {
          uint8_t *const Sp = (it & 1u) ? buf0 : buf1;
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(L.stream + dst),
                       "r"(smem_u32(Sp)), "r"(asz)
                       : "memory");
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    if (t >= nfull) break;
    have_prev = true;
    prev_c = c;
    prev_size = size;
    prev_raw = raw;
  }

  // rows past the last whole chunk: codes into the payload's section
  const uint32_t r0 = nfull * rpc, n_left = (NR - r0 + 15) / 16;
  for (uint32_t j = blockIdx.x * (kThreads / 32) + warp; j < n_left; j += gridDim.x * (kThreads / 32)) {
    const uint32_t R = r0 + 16 * j + rsub;
    const bool valid = R < NR;
    RowPos pos;
    pos.init(valid ? R : r0, H, T);
    enc_row<BITS, HAD, BF16, false>(P, smask, half, valid, pos.l, pos.b, pos.a, valid ? R : r0,
                                    P.codes + (size_t)(valid ? R : r0) * rec, flags);
  }
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (flags) atomicOr(P.status, flags);
}

bool v_lossless_fusable(const QuantParams &v, const LosslessParams &lp, uint64_t codes_off, uint64_t codes_bytes,
                        uint32_t *c0, uint32_t *nfull) {
  FastSpec f;
  if (lp.n_stages == 0 || lp.generic_only || !lossless_fast_spec(lp, f) || !f.bit8) return false;
  if (v.axis != KVC_AXIS_OVER_CHANNELS || v.smooth || v.delta || v.mixed) return false;
  if (v.bits != 2 && v.bits != 4 && v.bits != 8) return false;
  const uint32_t rec = 16 * v.bits, cb = lp.chunk_bytes;
  if (cb % rec || (cb / rec) % 128 || codes_off % cb) return false;
  *c0 = (uint32_t)(codes_off / cb);
  *nfull = (uint32_t)(codes_bytes / cb);
  return *nfull > 0 && *c0 + *nfull < lp.n_chunks;
}

template <int BITS>
static int launch_lc(const QuantParams &v, const LosslessParams &lp, const FastSpec &f, uint32_t c0, uint32_t nfull,
                     int sm_count, void *stream) {
  const bool had = v.hadamard != 0, bf = v.g.bf16 != 0;
  auto k = had ? (bf ? kvc_enc_rows_lc<BITS, true, true> : kvc_enc_rows_lc<BITS, true, false>)
               : (bf ? kvc_enc_rows_lc<BITS, false, true> : kvc_enc_rows_lc<BITS, false, false>);
  const size_t smem = 3 * ((size_t)lp.chunk_bytes + 64) + 64 * 4;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem) != cudaSuccess || per_sm < 1) per_sm = 1;
  const uint64_t blocks = (uint64_t)sm_count * per_sm;
  k<<<(unsigned)blocks, kThreads, smem, (cudaStream_t)stream>>>(v, lp, f, c0, nfull);
  return (int)cudaGetLastError();
}

int launch_v_lossless(const QuantParams &v, const LosslessParams &lp, uint32_t c0, uint32_t nfull, int sm_count,
                      void *stream) {
  FastSpec f;
  if (!lossless_fast_spec(lp, f)) return (int)cudaErrorInvalidValue;
  switch (v.bits) {
    case 2: return launch_lc<2>(v, lp, f, c0, nfull, sm_count, stream);
    case 4: return launch_lc<4>(v, lp, f, c0, nfull, sm_count, stream);
    case 8: return launch_lc<8>(v, lp, f, c0, nfull, sm_count, stream);
    default: return (int)cudaErrorInvalidValue;
  }
}

}  // namespace kvc
