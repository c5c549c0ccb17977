/*
 * kvc_oracle.c -- plain, slow CPU oracle of the KV-cache compression data path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; the two are written independently from the same definitions.
 *
 * Sources (cited by page title and section):
 *   [KVServe]    "KVServe: Service-Aware KV Cache Compression for Communication-
 *                Efficient Disaggregated LLM Serving"
 *                  §5.1 Constructing the strategy space (BS = C(Q(T(X))), the
 *                  Delta / Hadamard / Affine transformers, the KIVI quantizer,
 *                  layer-/head-wise mixed precision),
 *                  §7.3 Accuracy and Compression Ratio (2-bit KIVI metadata limits
 *                  the ratio to about 5.33x; Qwen KV is not zero-centred).
 *   [FastKVComp] "Beyond Compression Ratio: High-Throughput KV Compression for
 *                Disaggregated LLM Serving"
 *                  §4.1 Fused Transform-Quantization (randomized Hadamard with
 *                  cached deterministic signs, quantization statistics, channel-wise
 *                  keys / token-wise values, min-max rule, all-layer output buffer;
 *                  reconstruction = dequantize, inverse Hadamard, normalization,
 *                  sign restoration),
 *                  §4.2 Searchable High-Throughput Lossless Backend (pipeline
 *                  TUPL8_1 -> BIT_8 -> RZE_2: tuple reordering, bit shuffling,
 *                  zero-oriented encoding; device bitstream + size scalar).
 *
 * The pages describe the steps in prose only.  Every choice they leave open is
 * fixed here as "format v1" (the stream layout, rounding of every fp32 step, the
 * smoothing statistic, the sign generator, the packing order and the byte formats
 * of the lossless stages); each such choice is marked READING below.  Format v2
 * adds two optional profile features (a stream that uses neither is a v1 stream,
 * byte for byte): per-(layer, head) code widths ([KVServe] §5.1 layer- and
 * head-wise mixed precision; [FastKVComp] §4.1 head-importance-aware mixed
 * precision) and the token-delta transformer ([KVServe] §5.1 "Delta", after
 * CacheGen).
 *
 * Arithmetic: IEEE binary32, round-to-nearest-even, one rounding per written
 * operation (build with -ffp-contract=off, no fast-math).  fmaf() is the fused
 * multiply-add of IEEE 754 (one rounding).  Conversions to and from binary16 and
 * bfloat16 are written below from the formats' definitions.
 *
 * OpenMP runs independent (layer, head) units and independent chunks on several
 * threads; it changes no arithmetic (every unit writes disjoint bytes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Status flags returned by the oracle (bit mask).                            */
/* ------------------------------------------------------------------------ */
#define KVO_FLAG_RANGE     1u  /* fp16 metadata (zero, scale or centre) overflowed; saturated */
#define KVO_FLAG_NONFINITE 2u  /* an input element was NaN or infinite */
#define KVO_FLAG_CORRUPT   4u  /* decode: stream header / table / chunk inconsistent */
#define KVO_FLAG_CAPACITY  8u  /* encode: output capacity too small */

/* Stage kinds of the lossless pipeline ([FastKVComp] §4.2). */
#define KVO_ST_TUPL  1
#define KVO_ST_BIT   2
#define KVO_ST_DELTA 3
#define KVO_ST_RZE   4

/* Quantization axis ([FastKVComp] §4.1: keys channel-wise, values token-wise). */
#define KVO_AXIS_OVER_TOKENS   0  /* a group = one channel over G consecutive tokens */
#define KVO_AXIS_OVER_CHANNELS 1  /* a group = one token over G consecutive channels */

#define KVO_SMOOTH_BLOCK 128u     /* READING: key smoothing statistics per 128-token block */
#define KVO_HEADER_BYTES 64u

typedef struct {
    uint32_t layers, tokens, kv_heads, head_dim;
    uint32_t dtype;        /* 1 = binary16, 2 = bfloat16 */
    uint32_t page_size;    /* tokens per page; used only when a block table is given */
    uint64_t token_stride; /* bytes between consecutive token rows inside a page */
    uint64_t page_stride;  /* bytes between consecutive physical pages */
} kvo_shape;

typedef struct {
    uint32_t smooth_keys, hadamard;
    uint32_t bits_k, bits_v, group_k, group_v, axis_k, axis_v;
    uint32_t n_stages;
    uint32_t stage_kind[4], stage_param[4];
    uint32_t chunk_bytes;
    uint64_t seed;
    uint32_t token_delta;        /* v2: anchor-token delta on K and V (see quantize_tensor) */
    uint32_t pad_;
    const uint8_t *bits_map_k;   /* v2: [layers][kv_heads] code widths of K, or NULL = bits_k everywhere */
    const uint8_t *bits_map_v;   /* v2: the same for V, or NULL = bits_v everywhere */
} kvo_profile;

typedef struct {
    uint64_t off[8], size[8]; /* S1 K codes, S2 K meta, S3 V codes, S4 V meta, S5 K centres, S6 K exponents,
                                 S7 K anchors, S8 V anchors */
    uint64_t payload_bytes;   /* Q: all sections, each 16-byte aligned */
    uint64_t n_chunks;
    uint64_t data_start;      /* first chunk byte in the stream (stages present) */
    uint64_t max_stream_bytes;
    uint64_t header_bytes;    /* 64, or 64 + the width map (v2) */
} kvo_layout;

#define KVO_DELTA_BLOCK 128u      /* READING: one anchor token per 128-token block */

/* Code width of (layer l, head h) of a tensor (0 = K, 1 = V). */
static uint32_t width_of(const kvo_profile *p, int tensor, uint32_t H, uint32_t l, uint32_t h)
{
    const uint8_t *m = tensor ? p->bits_map_v : p->bits_map_k;
    if (m) return m[(uint64_t)l * H + h];
    return tensor ? p->bits_v : p->bits_k;
}

static int has_maps(const kvo_profile *p) { return p->bits_map_k != NULL || p->bits_map_v != NULL; }

static uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t align16(uint64_t a) { return (a + 15) & ~(uint64_t)15; }

/* ------------------------------------------------------------------------ */
/* binary16 / bfloat16 <-> binary32, from the IEEE 754 format definitions.   */
/* A finite format with `man_bits` fraction bits, minimum normal exponent     */
/* `emin` and largest finite value `maxf`.  Rounding modes: 0 nearest-even,   */
/* 1 toward -inf, 2 toward +inf.  All intermediate doubles are exact.         */
/* ------------------------------------------------------------------------ */
static double round_to_format(double x, int man_bits, int emin, double maxf, int mode)
{
    if (isnan(x) || isinf(x)) return x;
    if (x == 0.0) return x;
    int neg = x < 0;
    double a = fabs(x);
    /* quantum: spacing of the format's values around a */
    int k;
    frexp(a, &k);              /* a = f * 2^k, f in [0.5, 1): floor(log2 a) = k - 1 */
    int e = k - 1;
    if (e < emin) e = emin;    /* subnormal range shares the quantum of the smallest binade */
    double q = ldexp(1.0, e - man_bits);
    double n = floor(a / q);   /* exact: a / q is a power-of-two scaling */
    double lo = n * q, hi = (n + 1.0) * q, rem = a - lo;
    double mag;
    int away; /* round magnitude away from zero? */
    if (rem == 0.0) {
        mag = lo;
        away = 0;
    } else if (mode == 0) {
        if (2.0 * rem < q) away = 0;
        else if (2.0 * rem > q) away = 1;
        else away = fmod(n, 2.0) != 0.0; /* tie: to the even neighbour */
        mag = away ? hi : lo;
    } else {
        /* toward -inf: a positive value truncates, a negative one grows */
        away = (mode == 1) ? neg : !neg;
        mag = away ? hi : lo;
    }
    if (mag > maxf) {
        /* overflow: infinity when rounding away from zero (or to nearest), else the largest finite */
        int to_inf = (mode == 0) ? 1 : away;
        mag = to_inf ? INFINITY : maxf;
    }
    return neg ? -mag : mag;
}

static const double F16_MAX = 65504.0;
static double bf16_max(void) { return ldexp(255.0, 120); } /* (2 - 2^-7) * 2^127 */

float kvo_f16_to_f32(uint16_t h)
{
    uint32_t s = h >> 15, ex = (h >> 10) & 31u, m = h & 1023u;
    double v;
    if (ex == 0) v = ldexp((double)m, -24);
    else if (ex == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024u), (int)ex - 25);
    return (float)(s ? -v : v);
}

uint16_t kvo_f32_to_f16(float x, int mode)
{
    if (isnan(x)) return 0x7e00;
    double r = round_to_format((double)x, 10, -14, F16_MAX, mode);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a)) return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) return sign | (uint16_t)(a / ldexp(1.0, -24));
    int k;
    double f = frexp(a, &k);                     /* a = f * 2^k */
    uint16_t ex = (uint16_t)(k - 1 + 15);
    uint16_t man = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(ex << 10) | man;
}

float kvo_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16; /* bfloat16 is the upper half of a binary32 */
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t kvo_f32_to_bf16(float x)
{
    if (isnan(x)) return 0x7fc0;
    double r = round_to_format((double)x, 7, -126, bf16_max(), 0);
    float f = (float)r; /* exact: every bfloat16 value is a binary32 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static float elem_to_f32(uint16_t bits, uint32_t dtype)
{
    return dtype == 1 ? kvo_f16_to_f32(bits) : kvo_bf16_to_f32(bits);
}

static uint16_t f32_to_elem(float x, uint32_t dtype)
{
    return dtype == 1 ? kvo_f32_to_f16(x, 0) : kvo_f32_to_bf16(x);
}

/* ------------------------------------------------------------------------ */
/* Randomized Hadamard transform ([FastKVComp] §4.1; [KVServe] §5.1).         */
/* READING: "randomized" = a diagonal of +-1 signs drawn once per profile from */
/* SplitMix64 (S. Vigna's published generator) seeded with the profile seed:   */
/* sign j is negative when the top bit of the j-th output is set.  One vector  */
/* serves every layer, head, K and V ("cached and reused").                    */
/* ------------------------------------------------------------------------ */
static uint64_t splitmix64_next(uint64_t *state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t kvo_splitmix64_output(uint64_t seed, uint32_t j)
{
    uint64_t st = seed, out = 0;
    for (uint32_t i = 0; i <= j; i++) out = splitmix64_next(&st);
    return out;
}

void kvo_signs(uint64_t seed, uint32_t D, float *sigma)
{
    uint64_t st = seed;
    for (uint32_t j = 0; j < D; j++) sigma[j] = (splitmix64_next(&st) >> 63) ? -1.0f : 1.0f;
}

/* READING: the Walsh-Hadamard butterfly in Sylvester (natural) order, strides
 * h = 1, 2, 4, ..., D/2 in that order; each butterfly (a, b) -> (a + b, a - b)
 * rounded to binary32.  The fixed stage order fixes every rounding. */
void kvo_fwht(float *v, uint32_t D)
{
    for (uint32_t h = 1; h < D; h <<= 1)
        for (uint32_t i = 0; i < D; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
}

/* READING: "normalization" = the factor 1/sqrt(D) rounded to binary32. */
float kvo_hadamard_scale(uint32_t D) { return (float)(1.0 / sqrt((double)D)); }

/* y = c * FWHT(sigma (.) x) */
void kvo_hadamard_forward(float *v, const float *sigma, uint32_t D)
{
    for (uint32_t j = 0; j < D; j++) v[j] = v[j] * sigma[j];
    kvo_fwht(v, D);
    float c = kvo_hadamard_scale(D);
    for (uint32_t j = 0; j < D; j++) v[j] = v[j] * c;
}

/* x = sigma (.) (c * FWHT(y)) -- inverse transform, normalization, sign restoration */
void kvo_hadamard_inverse(float *v, const float *sigma, uint32_t D)
{
    kvo_fwht(v, D);
    float c = kvo_hadamard_scale(D);
    for (uint32_t j = 0; j < D; j++) v[j] = v[j] * c;
    for (uint32_t j = 0; j < D; j++) v[j] = v[j] * sigma[j];
}

/* ------------------------------------------------------------------------ */
/* Per-channel key smoothing.  READING (the pages name an affine transformer, */
/* non-zero-centred keys and a "normalization" step but define none): per     */
/* (layer, head, 128-token block, channel) over the valid tokens:             */
/*   mu = binary16_rn( (mn + mx) * 0.5 )          (midrange, saturated)       */
/*   r  = max(|mx - mu|, |mn - mu|)                                           */
/*   e  = smallest integer with 2^e >= r (0 when r = 0), clamped [-126, 127]  */
/*   x' = (x - mu) * 2^-e                          (exact power-of-two scale) */
/* Decode: x = fma(x', 2^e, mu).                                              */
/* ------------------------------------------------------------------------ */
int kvo_ceil_log2(float r)
{
    if (!(r > 0.0f)) return 0;
    if (isinf(r)) return 127;
    int k;
    float f = frexpf(r, &k); /* r = f * 2^k, f in [0.5, 1) */
    int e = (f == 0.5f) ? k - 1 : k;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return e;
}

static uint16_t centre_f16(float mn, float mx, uint32_t *flags)
{
    float mid = (mn + mx) * 0.5f;
    uint16_t h = kvo_f32_to_f16(mid, 0);
    if ((h & 0x7fff) == 0x7c00) { /* overflowed to infinity: saturate */
        h = (h & 0x8000) | 0x7bff;
        *flags |= KVO_FLAG_RANGE;
    }
    return h;
}

/* ------------------------------------------------------------------------ */
/* Group-wise asymmetric min-max quantization ([FastKVComp] §4.1 "original    */
/* min-max quantization rule"; KIVI, [KVServe] §5.1, §7.3).                   */
/* READING: metadata = binary16 scale and zero per group (32 bits: the        */
/* 5.33x ceiling of 2-bit groups of 32 in [KVServe] §7.3).  Directed rounding */
/* keeps [mn, mx] inside [z, z + Q*s]:                                        */
/*   z = binary16_down(mn); s = binary16_up((mx - z) / Q), Q = 2^b - 1        */
/*   q = clamp(rint_even((y - z) / s), 0, Q)  (true binary32 division; q = 0  */
/*   when s = 0).  An infinite z or s saturates to +-65504 and flags RANGE.   */
/* Dequantization: y^ = fma(q, s, z).                                         */
/* ------------------------------------------------------------------------ */
void kvo_quantize_group(const float *y, uint32_t n, uint32_t bits,
                        uint16_t *s_out, uint16_t *z_out, uint8_t *codes, uint32_t *flags)
{
    float mn = y[0], mx = y[0];
    for (uint32_t i = 1; i < n; i++) {
        if (y[i] < mn) mn = y[i];
        if (y[i] > mx) mx = y[i];
    }
    /* READING: min and max are values; a zero extreme counts as +0 (adding +0
     * turns -0 into +0 and changes nothing else), so the result does not depend
     * on the order in which equal zeros of opposite sign are met. */
    mn = mn + 0.0f;
    mx = mx + 0.0f;
    uint32_t Q = (1u << bits) - 1u;
    uint16_t zh = kvo_f32_to_f16(mn, 1);
    if ((zh & 0x7fff) == 0x7c00) { zh = (zh & 0x8000) | 0x7bff; *flags |= KVO_FLAG_RANGE; }
    float z = kvo_f16_to_f32(zh);
    float w = mx - z;
    float v = w / (float)Q;
    uint16_t sh = kvo_f32_to_f16(v, 2);
    if ((sh & 0x7fff) == 0x7c00) { sh = (sh & 0x8000) | 0x7bff; *flags |= KVO_FLAG_RANGE; }
    float s = kvo_f16_to_f32(sh);
    for (uint32_t i = 0; i < n; i++) {
        uint32_t q = 0;
        if (s != 0.0f) {
            float t = y[i] - z;
            float d = t / s;
            float k = rintf(d);
            if (k >= (float)Q) q = Q;
            else if (k > 0.0f) q = (uint32_t)k;
            else q = 0; /* also NaN */
        }
        codes[i] = (uint8_t)q;
    }
    *s_out = sh;
    *z_out = zh;
}

/* READING: a group's G codes pack least-significant-bit first: bit j of code i
 * is bit (i*b + j) of the record, and record byte k holds record bits 8k..8k+7. */
void kvo_pack(const uint8_t *codes, uint32_t n, uint32_t bits, uint8_t *out)
{
    uint32_t nbytes = (n * bits + 7) / 8;
    memset(out, 0, nbytes);
    for (uint32_t i = 0; i < n; i++)
        for (uint32_t j = 0; j < bits; j++)
            if ((codes[i] >> j) & 1u) {
                uint32_t bit = i * bits + j;
                out[bit / 8] |= (uint8_t)(1u << (bit % 8));
            }
}

void kvo_unpack(const uint8_t *in, uint32_t n, uint32_t bits, uint8_t *codes)
{
    for (uint32_t i = 0; i < n; i++) {
        uint32_t c = 0;
        for (uint32_t j = 0; j < bits; j++) {
            uint32_t bit = i * bits + j;
            c |= (uint32_t)((in[bit / 8] >> (bit % 8)) & 1u) << j;
        }
        codes[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------------ */
/* Payload layout (READING; "preallocated all-layer output buffer",           */
/* [FastKVComp] §4.1).  Sections in order, each starting 16-byte aligned:     */
/*  S1 K codes, S2 K meta {scale, zero}, S3 V codes, S4 V meta,               */
/*  S5 K smoothing centres (binary16), S6 K smoothing exponents (int8),       */
/*  S7 K anchors, S8 V anchors (v2 token delta: element bits, 2 bytes).       */
/* Groups over tokens: records ordered [layer][head][token group][channel];   */
/* groups over channels: [layer][token][head][channel group].                 */
/* Smoothing and anchor planes: [layer][head][128-token block][channel].      */
/* ------------------------------------------------------------------------ */
static uint64_t n_groups(const kvo_shape *sh, uint32_t axis, uint32_t G)
{
    uint64_t L = sh->layers, T = sh->tokens, H = sh->kv_heads, D = sh->head_dim;
    if (axis == KVO_AXIS_OVER_TOKENS) return L * H * ceil_div(T, G) * D;
    return L * T * H * (D / G);
}

/* Code bytes of one (layer, head) of a tensor: T rows of D codes of its width
 * (groups over tokens: ceil(T/G) groups of G codes per channel). */
static uint64_t lh_code_bytes(const kvo_shape *sh, uint32_t axis, uint32_t G, uint32_t bits)
{
    uint64_t T = sh->tokens, D = sh->head_dim;
    if (axis == KVO_AXIS_OVER_TOKENS) return ceil_div(T, G) * D * G * bits / 8;
    return T * D * bits / 8;
}

/* READING (v2 layout with per-(layer, head) widths): groups over tokens keep
 * records [layer][head][token group][channel], the (layer, head) blocks back to
 * back, each with its own width; groups over channels keep records
 * [layer][token][head][channel group], a token's row holding its heads' records
 * back to back, each head with its own width.  With one width everywhere both
 * are the v1 layout. */
static uint64_t code_bytes(const kvo_profile *p, const kvo_shape *sh, int tensor)
{
    const uint32_t axis = tensor ? p->axis_v : p->axis_k, G = tensor ? p->group_v : p->group_k;
    uint64_t n = 0;
    for (uint32_t l = 0; l < sh->layers; l++)
        for (uint32_t h = 0; h < sh->kv_heads; h++)
            n += lh_code_bytes(sh, axis, G, width_of(p, tensor, sh->kv_heads, l, h));
    return n;
}

/* Bytes of the v2 width map that follows the 64-byte header: 2 bits per entry
 * (K entries l*H + h, then V entries), padded to 16 bytes. */
static uint64_t map_bytes(const kvo_profile *p, const kvo_shape *sh)
{
    if (!has_maps(p)) return 0;
    return align16(ceil_div(2 * (uint64_t)sh->layers * sh->kv_heads * 2, 8));
}

int kvo_layout_of(const kvo_profile *p, const kvo_shape *sh, kvo_layout *lay)
{
    memset(lay, 0, sizeof *lay);
    uint64_t gk = n_groups(sh, p->axis_k, p->group_k), gv = n_groups(sh, p->axis_v, p->group_v);
    uint64_t nsb = (uint64_t)sh->layers * sh->kv_heads * ceil_div(sh->tokens, KVO_SMOOTH_BLOCK) * sh->head_dim;
    uint64_t nab = (uint64_t)sh->layers * sh->kv_heads * ceil_div(sh->tokens, KVO_DELTA_BLOCK) * sh->head_dim;
    lay->size[0] = code_bytes(p, sh, 0);
    lay->size[1] = gk * 4;
    lay->size[2] = code_bytes(p, sh, 1);
    lay->size[3] = gv * 4;
    lay->size[4] = p->smooth_keys ? nsb * 2 : 0;
    lay->size[5] = p->smooth_keys ? nsb : 0;
    lay->size[6] = p->token_delta ? nab * 2 : 0;
    lay->size[7] = p->token_delta ? nab * 2 : 0;
    uint64_t o = 0;
    for (int i = 0; i < 8; i++) {
        lay->off[i] = o;
        o += align16(lay->size[i]);
    }
    lay->payload_bytes = o;
    lay->header_bytes = KVO_HEADER_BYTES + map_bytes(p, sh);
    if (p->n_stages == 0) {
        lay->n_chunks = 0;
        lay->data_start = lay->header_bytes;
        lay->max_stream_bytes = lay->header_bytes + o;
    } else {
        lay->n_chunks = ceil_div(o, p->chunk_bytes);
        lay->data_start = align16(lay->header_bytes + 4 * lay->n_chunks);
        lay->max_stream_bytes = lay->data_start + o; /* every chunk stored raw */
    }
    return 0;
}

/* Byte offset of (layer l, head h)'s code block (groups over tokens), or of
 * (layer l, token 0, head h)'s first record plus the layer's row length in
 * *row_bytes (groups over channels), inside the tensor's code section. */
static uint64_t code_base(const kvo_profile *p, const kvo_shape *sh, int tensor, uint32_t l, uint32_t h,
                          uint64_t *row_bytes)
{
    const uint32_t H = sh->kv_heads, D = sh->head_dim;
    const uint32_t axis = tensor ? p->axis_v : p->axis_k, G = tensor ? p->group_v : p->group_k;
    uint64_t off = 0;
    if (axis == KVO_AXIS_OVER_TOKENS) {
        for (uint32_t l2 = 0; l2 < sh->layers; l2++)
            for (uint32_t h2 = 0; h2 < H; h2++) {
                if (l2 == l && h2 == h) return off;
                off += lh_code_bytes(sh, axis, G, width_of(p, tensor, H, l2, h2));
            }
        return off;
    }
    for (uint32_t l2 = 0; l2 < l; l2++)
        for (uint32_t h2 = 0; h2 < H; h2++) off += lh_code_bytes(sh, axis, G, width_of(p, tensor, H, l2, h2));
    uint64_t row = 0, head = 0;
    for (uint32_t h2 = 0; h2 < H; h2++) {
        if (h2 == h) head = row;
        row += (uint64_t)D * width_of(p, tensor, H, l, h2) / 8;
    }
    *row_bytes = row;
    return off + head;
}

/* Row address of token t of layer `base` (contiguous or through a block table). */
static const uint16_t *row_ptr(const uint8_t *base, const kvo_shape *sh, const int32_t *block_table, uint64_t t)
{
    uint64_t off;
    if (block_table) {
        uint64_t page = (uint64_t)(uint32_t)block_table[t / sh->page_size];
        off = page * sh->page_stride + (t % sh->page_size) * sh->token_stride;
    } else {
        off = t * sh->token_stride;
    }
    return (const uint16_t *)(base + off);
}

static void put_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void put_u32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint32_t get_u32(const uint8_t *p) { uint32_t v = 0; for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i); return v; }
static void put_u64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint64_t get_u64(const uint8_t *p) { uint64_t v = 0; for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i); return v; }

/* Quantize one tensor (0 = K, 1 = V) of every layer into the payload Q.
 * Pipeline per (layer, head), in the order of BS = C(Q(T(X))) ([KVServe] §5.1):
 * smoothing (keys, optional) -> randomized Hadamard (optional) -> groups -> pack. */
static uint32_t quantize_tensor(const kvo_profile *p, const kvo_shape *sh, int tensor,
                                const uint8_t *const *bases, const int32_t *block_table,
                                const kvo_layout *lay, uint8_t *Q)
{
    const uint32_t L = sh->layers, T = sh->tokens, H = sh->kv_heads, D = sh->head_dim;
    const uint32_t G = tensor ? p->group_v : p->group_k;
    const uint32_t axis = tensor ? p->axis_v : p->axis_k;
    const int smooth = (tensor == 0) && p->smooth_keys;
    uint8_t *codes_sec = Q + lay->off[tensor ? 2 : 0];
    uint8_t *anchor_sec = Q + lay->off[tensor ? 7 : 6];
    uint8_t *meta_sec = Q + lay->off[tensor ? 3 : 1];
    uint16_t *mu_sec = (uint16_t *)(Q + lay->off[4]);
    int8_t *e_sec = (int8_t *)(Q + lay->off[5]);
    float sigma[1024];
    kvo_signs(p->seed, D, sigma);
    const uint64_t nTG = ceil_div(T, G), nSB = ceil_div(T, KVO_SMOOTH_BLOCK);
    uint32_t flags = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
    for (int64_t lh = 0; lh < (int64_t)L * H; lh++) {
        const uint32_t l = (uint32_t)(lh / H), h = (uint32_t)(lh % H);
        const uint32_t bits = width_of(p, tensor, H, l, h);
        const uint64_t rec = (uint64_t)G * bits / 8;
        uint64_t row_bytes = 0;
        const uint64_t cbase = code_base(p, sh, tensor, l, h, &row_bytes);
        float *X = (float *)malloc((size_t)T * D * sizeof(float));
        float *col = (float *)malloc((size_t)(T > 0 ? T : 1) * sizeof(float));
        uint8_t codes[128 * 8];
        uint8_t packed[1024];
        for (uint64_t t = 0; t < T; t++) {
            const uint16_t *r = row_ptr(bases[l], sh, block_table, t) + (uint64_t)h * D;
            for (uint32_t d = 0; d < D; d++) {
                float x = elem_to_f32(r[d], sh->dtype);
                if (!isfinite(x)) flags |= KVO_FLAG_NONFINITE;
                X[t * D + d] = x;
            }
        }
        /* transformer stage 0 (v2, optional): token delta ([KVServe] §5.1 "Delta",
         * after CacheGen).  READING: the first token of every 128-token block is
         * the block's anchor; every token of the block (the anchor included, which
         * becomes 0) is replaced by its fp32 difference from the anchor, channel by
         * channel; the anchor's element bits are kept in the payload. */
        if (p->token_delta) {
            const uint64_t nAB = ceil_div(T, KVO_DELTA_BLOCK);
            for (uint64_t ab = 0; ab < nAB; ab++) {
                uint64_t t0 = ab * KVO_DELTA_BLOCK, t1 = t0 + KVO_DELTA_BLOCK;
                if (t1 > T) t1 = T;
                const uint16_t *ar = row_ptr(bases[l], sh, block_table, t0) + (uint64_t)h * D;
                for (uint32_t c = 0; c < D; c++) {
                    uint64_t cell = (((uint64_t)l * H + h) * nAB + ab) * D + c;
                    put_u16(anchor_sec + 2 * cell, ar[c]);
                }
                float a[1024];
                for (uint32_t c = 0; c < D; c++) a[c] = X[t0 * D + c];
                for (uint64_t t = t0; t < t1; t++)
                    for (uint32_t c = 0; c < D; c++) X[t * D + c] = X[t * D + c] - a[c];
            }
        }
        /* transformer stage 1: per-channel key smoothing */
        if (smooth) {
            for (uint64_t sb = 0; sb < nSB; sb++) {
                uint64_t t0 = sb * KVO_SMOOTH_BLOCK, t1 = t0 + KVO_SMOOTH_BLOCK;
                if (t1 > T) t1 = T;
                for (uint32_t c = 0; c < D; c++) {
                    float mn = X[t0 * D + c], mx = mn;
                    for (uint64_t t = t0 + 1; t < t1; t++) {
                        float x = X[t * D + c];
                        if (x < mn) mn = x;
                        if (x > mx) mx = x;
                    }
                    mn = mn + 0.0f; /* a zero extreme counts as +0 (see kvo_quantize_group) */
                    mx = mx + 0.0f;
                    uint16_t muh = centre_f16(mn, mx, &flags);
                    float mu = kvo_f16_to_f32(muh);
                    float r1 = fabsf(mx - mu), r2 = fabsf(mn - mu);
                    float r = r1 > r2 ? r1 : r2;
                    int e = kvo_ceil_log2(r);
                    float inv = ldexpf(1.0f, -e);
                    for (uint64_t t = t0; t < t1; t++) X[t * D + c] = (X[t * D + c] - mu) * inv;
                    uint64_t cell = (((uint64_t)l * H + h) * nSB + sb) * D + c;
                    uint8_t *mp = (uint8_t *)(mu_sec + cell);
                    put_u16(mp, muh);
                    e_sec[cell] = (int8_t)e;
                }
            }
        }
        /* transformer stage 2: randomized Hadamard along head_dim */
        if (p->hadamard)
            for (uint64_t t = 0; t < T; t++) kvo_hadamard_forward(X + t * D, sigma, D);
        /* quantizer: groups, min-max rule, packing */
        if (axis == KVO_AXIS_OVER_TOKENS) {
            for (uint64_t tg = 0; tg < nTG; tg++) {
                uint64_t t0 = tg * G, n = (t0 + G <= T) ? G : T - t0;
                for (uint32_t c = 0; c < D; c++) {
                    uint16_t s, z;
                    for (uint64_t i = 0; i < n; i++) col[i] = X[(t0 + i) * D + c];
                    memset(codes, 0, G);
                    kvo_quantize_group(col, (uint32_t)n, bits, &s, &z, codes, &flags);
                    kvo_pack(codes, G, bits, packed); /* tail codes stay 0 */
                    uint64_t g = (((uint64_t)l * H + h) * nTG + tg) * D + c;
                    memcpy(codes_sec + cbase + (tg * D + c) * rec, packed, rec);
                    put_u16(meta_sec + g * 4, s);
                    put_u16(meta_sec + g * 4 + 2, z);
                }
            }
        } else {
            for (uint64_t t = 0; t < T; t++)
                for (uint32_t cg = 0; cg < D / G; cg++) {
                    uint16_t s, z;
                    kvo_quantize_group(X + t * D + (uint64_t)cg * G, G, bits, &s, &z, codes, &flags);
                    kvo_pack(codes, G, bits, packed);
                    uint64_t g = (((uint64_t)l * T + t) * H + h) * (D / G) + cg;
                    memcpy(codes_sec + cbase + t * row_bytes + cg * rec, packed, rec);
                    put_u16(meta_sec + g * 4, s);
                    put_u16(meta_sec + g * 4 + 2, z);
                }
        }
        free(col);
        free(X);
    }
    return flags;
}

/* Q = all sections; padding bytes are zero. */
uint32_t kvo_quantize(const kvo_profile *p, const kvo_shape *sh,
                      const uint8_t *const *k_bases, const uint8_t *const *v_bases,
                      const int32_t *block_table, uint8_t *Q)
{
    kvo_layout lay;
    kvo_layout_of(p, sh, &lay);
    memset(Q, 0, lay.payload_bytes);
    uint32_t flags = 0;
    flags |= quantize_tensor(p, sh, 0, k_bases, block_table, &lay, Q);
    flags |= quantize_tensor(p, sh, 1, v_bases, block_table, &lay, Q);
    return flags;
}

/* Reconstruction ([FastKVComp] §4.1 "Fused Reconstruction"): dequantize, inverse
 * Hadamard, normalization and sign restoration, then (keys) undo the smoothing,
 * then (v2) add the block's anchor back, then round to the element type and
 * write the row. */
static void dequantize_tensor(const kvo_profile *p, const kvo_shape *sh, int tensor, const uint8_t *Q,
                              const kvo_layout *lay, uint8_t *const *bases, const int32_t *block_table)
{
    const uint32_t L = sh->layers, T = sh->tokens, H = sh->kv_heads, D = sh->head_dim;
    const uint32_t G = tensor ? p->group_v : p->group_k;
    const uint32_t axis = tensor ? p->axis_v : p->axis_k;
    const int smooth = (tensor == 0) && p->smooth_keys;
    const uint8_t *codes_sec = Q + lay->off[tensor ? 2 : 0];
    const uint8_t *anchor_sec = Q + lay->off[tensor ? 7 : 6];
    const uint8_t *meta_sec = Q + lay->off[tensor ? 3 : 1];
    const uint8_t *mu_sec = Q + lay->off[4];
    const int8_t *e_sec = (const int8_t *)(Q + lay->off[5]);
    float sigma[1024];
    kvo_signs(p->seed, D, sigma);
    const uint64_t nTG = ceil_div(T, G), nSB = ceil_div(T, KVO_SMOOTH_BLOCK);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lh = 0; lh < (int64_t)L * H; lh++) {
        const uint32_t l = (uint32_t)(lh / H), h = (uint32_t)(lh % H);
        const uint32_t bits = width_of(p, tensor, H, l, h);
        const uint64_t rec = (uint64_t)G * bits / 8;
        uint64_t row_bytes = 0;
        const uint64_t cbase = code_base(p, sh, tensor, l, h, &row_bytes);
        float *X = (float *)malloc((size_t)T * D * sizeof(float));
        uint8_t codes[1024];
        if (axis == KVO_AXIS_OVER_TOKENS) {
            for (uint64_t tg = 0; tg < nTG; tg++) {
                uint64_t t0 = tg * G, n = (t0 + G <= T) ? G : T - t0;
                for (uint32_t c = 0; c < D; c++) {
                    uint64_t g = (((uint64_t)l * H + h) * nTG + tg) * D + c;
                    kvo_unpack(codes_sec + cbase + (tg * D + c) * rec, G, bits, codes);
                    float s = kvo_f16_to_f32(get_u16(meta_sec + g * 4));
                    float z = kvo_f16_to_f32(get_u16(meta_sec + g * 4 + 2));
                    for (uint64_t i = 0; i < n; i++) X[(t0 + i) * D + c] = fmaf((float)codes[i], s, z);
                }
            }
        } else {
            for (uint64_t t = 0; t < T; t++)
                for (uint32_t cg = 0; cg < D / G; cg++) {
                    uint64_t g = (((uint64_t)l * T + t) * H + h) * (D / G) + cg;
                    kvo_unpack(codes_sec + cbase + t * row_bytes + cg * rec, G, bits, codes);
                    float s = kvo_f16_to_f32(get_u16(meta_sec + g * 4));
                    float z = kvo_f16_to_f32(get_u16(meta_sec + g * 4 + 2));
                    for (uint32_t i = 0; i < G; i++) X[t * D + (uint64_t)cg * G + i] = fmaf((float)codes[i], s, z);
                }
        }
        if (p->hadamard)
            for (uint64_t t = 0; t < T; t++) kvo_hadamard_inverse(X + t * D, sigma, D);
        if (smooth) {
            for (uint64_t t = 0; t < T; t++) {
                uint64_t sb = t / KVO_SMOOTH_BLOCK;
                for (uint32_t c = 0; c < D; c++) {
                    uint64_t cell = (((uint64_t)l * H + h) * nSB + sb) * D + c;
                    float mu = kvo_f16_to_f32(get_u16(mu_sec + 2 * cell));
                    int e = e_sec[cell];
                    if (e < -126) e = -126;
                    float sc = ldexpf(1.0f, e);
                    X[t * D + c] = fmaf(X[t * D + c], sc, mu);
                }
            }
        }
        /* undo the token delta: add the block's anchor back in fp32 */
        if (p->token_delta) {
            const uint64_t nAB = ceil_div(T, KVO_DELTA_BLOCK);
            for (uint64_t t = 0; t < T; t++) {
                uint64_t ab = t / KVO_DELTA_BLOCK;
                for (uint32_t c = 0; c < D; c++) {
                    uint64_t cell = (((uint64_t)l * H + h) * nAB + ab) * D + c;
                    float a = elem_to_f32(get_u16(anchor_sec + 2 * cell), sh->dtype);
                    X[t * D + c] = X[t * D + c] + a;
                }
            }
        }
        for (uint64_t t = 0; t < T; t++) {
            uint16_t *r = (uint16_t *)row_ptr(bases[l], sh, block_table, t) + (uint64_t)h * D;
            for (uint32_t d = 0; d < D; d++) r[d] = f32_to_elem(X[t * D + d], sh->dtype);
        }
        free(X);
    }
}

void kvo_dequantize(const kvo_profile *p, const kvo_shape *sh, const uint8_t *Q,
                    uint8_t *const *k_bases, uint8_t *const *v_bases, const int32_t *block_table)
{
    kvo_layout lay;
    kvo_layout_of(p, sh, &lay);
    dequantize_tensor(p, sh, 0, Q, &lay, k_bases, block_table);
    dequantize_tensor(p, sh, 1, Q, &lay, v_bases, block_table);
}

/* ------------------------------------------------------------------------ */
/* Lossless stages ([FastKVComp] §4.2: tuple reordering, bit shuffling,       */
/* zero-oriented encoding; the workloads add a delta stage).  READING: the   */
/* byte formats of LC's stages are not on the pages; these are format v1's.   */
/* Every stage keeps a tail (the bytes past the last whole tuple/word) as is. */
/* ------------------------------------------------------------------------ */

/* TUPL_k: view n bytes as m = n/k tuples of k bytes; emit column j (byte j of
 * every tuple) for j = 0..k-1, then the tail. */
size_t kvo_tupl_encode(const uint8_t *in, size_t n, uint32_t k, uint8_t *out)
{
    size_t m = n / k;
    for (size_t j = 0; j < k; j++)
        for (size_t i = 0; i < m; i++) out[j * m + i] = in[i * k + j];
    memcpy(out + m * k, in + m * k, n - m * k);
    return n;
}

size_t kvo_tupl_decode(const uint8_t *in, size_t n, uint32_t k, uint8_t *out)
{
    size_t m = n / k;
    for (size_t j = 0; j < k; j++)
        for (size_t i = 0; i < m; i++) out[i * k + j] = in[j * m + i];
    memcpy(out + m * k, in + m * k, n - m * k);
    return n;
}

/* BIT_8: over the first n8 = 8*floor(n/8) bytes, plane p (p = 0..7, least
 * significant first) holds n8/8 bytes whose bit i (LSB first) is bit p of
 * input byte i; then the tail. */
size_t kvo_bit_encode(const uint8_t *in, size_t n, uint8_t *out)
{
    size_t n8 = n / 8 * 8, P = n8 / 8;
    memset(out, 0, n8);
    for (size_t i = 0; i < n8; i++)
        for (uint32_t p = 0; p < 8; p++)
            if ((in[i] >> p) & 1u) out[p * P + i / 8] |= (uint8_t)(1u << (i % 8));
    memcpy(out + n8, in + n8, n - n8);
    return n;
}

size_t kvo_bit_decode(const uint8_t *in, size_t n, uint8_t *out)
{
    size_t n8 = n / 8 * 8, P = n8 / 8;
    memset(out, 0, n8);
    for (size_t i = 0; i < n8; i++)
        for (uint32_t p = 0; p < 8; p++)
            if ((in[p * P + i / 8] >> (i % 8)) & 1u) out[i] |= (uint8_t)(1u << p);
    memcpy(out + n8, in + n8, n - n8);
    return n;
}

static uint64_t get_word(const uint8_t *p, uint32_t w)
{
    uint64_t v = 0;
    for (uint32_t i = 0; i < w; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

static void put_word(uint8_t *p, uint32_t w, uint64_t v)
{
    for (uint32_t i = 0; i < w; i++) p[i] = (uint8_t)(v >> (8 * i));
}

/* DELTA_w: little-endian w-byte words; word 0 kept, word i replaced by
 * word i - word (i-1) modulo 2^(8w); then the tail. */
size_t kvo_delta_encode(const uint8_t *in, size_t n, uint32_t w, uint8_t *out)
{
    size_t m = n / w;
    uint64_t mask = (w == 8) ? ~0ULL : ((1ULL << (8 * w)) - 1);
    for (size_t i = 0; i < m; i++) {
        uint64_t cur = get_word(in + i * w, w), prev = i ? get_word(in + (i - 1) * w, w) : 0;
        put_word(out + i * w, w, (cur - prev) & mask);
    }
    memcpy(out + m * w, in + m * w, n - m * w);
    return n;
}

size_t kvo_delta_decode(const uint8_t *in, size_t n, uint32_t w, uint8_t *out)
{
    size_t m = n / w;
    uint64_t mask = (w == 8) ? ~0ULL : ((1ULL << (8 * w)) - 1), acc = 0;
    for (size_t i = 0; i < m; i++) {
        acc = (acc + get_word(in + i * w, w)) & mask;
        put_word(out + i * w, w, acc);
    }
    memcpy(out + m * w, in + m * w, n - m * w);
    return n;
}

/* RZE_w: m = floor(n/w) words.  B = bitmap of nonzero words (ceil(m/8) bytes,
 * bit i LSB-first = word i nonzero); B2 = bitmap of the nonzero bytes of B
 * (ceil(|B|/8) bytes).  Output = B2, the nonzero bytes of B in order, the
 * nonzero words in order, the tail.  The decoder needs n. */
size_t kvo_rze_encode(const uint8_t *in, size_t n, uint32_t w, uint8_t *out)
{
    size_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8;
    uint8_t *B = (uint8_t *)calloc(nb ? nb : 1, 1);
    for (size_t i = 0; i < m; i++)
        if (get_word(in + i * w, w) != 0) B[i / 8] |= (uint8_t)(1u << (i % 8));
    memset(out, 0, nb2);
    size_t o = nb2;
    for (size_t j = 0; j < nb; j++)
        if (B[j]) {
            out[j / 8] |= (uint8_t)(1u << (j % 8));
            out[o++] = B[j];
        }
    for (size_t i = 0; i < m; i++)
        if ((B[i / 8] >> (i % 8)) & 1u) {
            memcpy(out + o, in + i * w, w);
            o += w;
        }
    memcpy(out + o, in + m * w, n - m * w);
    o += n - m * w;
    free(B);
    return o;
}

/* Returns 0 on success, -1 if `size` stored bytes do not decode to exactly n bytes. */
int kvo_rze_decode(const uint8_t *in, size_t size, size_t n, uint32_t w, uint8_t *out)
{
    size_t m = n / w, nb = (m + 7) / 8, nb2 = (nb + 7) / 8;
    if (size < nb2) return -1;
    uint8_t *B = (uint8_t *)calloc(nb ? nb : 1, 1);
    size_t o = nb2;
    for (size_t j = 0; j < nb; j++)
        if ((in[j / 8] >> (j % 8)) & 1u) {
            if (o >= size) { free(B); return -1; }
            B[j] = in[o++];
        }
    for (size_t i = 0; i < m; i++) {
        if ((B[i / 8] >> (i % 8)) & 1u) {
            if (o + w > size) { free(B); return -1; }
            memcpy(out + i * w, in + o, w);
            o += w;
        } else {
            memset(out + i * w, 0, w);
        }
    }
    free(B);
    if (o + (n - m * w) != size) return -1;
    memcpy(out + m * w, in + o, n - m * w);
    return 0;
}

/* Apply one stage (encode).  Output capacity: 2n + 64 bytes is enough for RZE. */
size_t kvo_stage_encode(uint32_t kind, uint32_t param, const uint8_t *in, size_t n, uint8_t *out)
{
    switch (kind) {
    case KVO_ST_TUPL: return kvo_tupl_encode(in, n, param, out);
    case KVO_ST_BIT: return kvo_bit_encode(in, n, out);
    case KVO_ST_DELTA: return kvo_delta_encode(in, n, param, out);
    case KVO_ST_RZE: return kvo_rze_encode(in, n, param, out);
    }
    return 0;
}

/* Encode one chunk of n raw bytes through the stage list.  Returns the stored
 * size; *raw = 1 when the chunk is stored verbatim (READING: when the encoded
 * form is not smaller than the raw bytes). */
size_t kvo_chunk_encode(const kvo_profile *p, const uint8_t *in, size_t n, uint8_t *out, int *raw)
{
    size_t cap = 2 * n + 64;
    uint8_t *a = (uint8_t *)malloc(cap), *b = (uint8_t *)malloc(cap);
    memcpy(a, in, n);
    size_t len = n;
    for (uint32_t s = 0; s < p->n_stages; s++) {
        len = kvo_stage_encode(p->stage_kind[s], p->stage_param[s], a, len, b);
        uint8_t *t = a; a = b; b = t;
    }
    if (len >= n) {
        memcpy(out, in, n);
        len = n;
        *raw = 1;
    } else {
        memcpy(out, a, len);
        *raw = 0;
    }
    free(a);
    free(b);
    return len;
}

/* Decode one stored chunk back to its n raw bytes; -1 when inconsistent. */
int kvo_chunk_decode(const kvo_profile *p, const uint8_t *in, size_t size, int raw, size_t n, uint8_t *out)
{
    if (raw) {
        if (size != n) return -1;
        memcpy(out, in, n);
        return 0;
    }
    if (size >= n) return -1;
    uint8_t *a = (uint8_t *)malloc(n + 16), *b = (uint8_t *)malloc(n + 16);
    int rc = 0;
    int s = (int)p->n_stages - 1;
    if (p->stage_kind[s] == KVO_ST_RZE) {
        rc = kvo_rze_decode(in, size, n, p->stage_param[s], a);
        s--;
    } else {
        if (size != n) rc = -1; /* length-preserving stages only */
        else memcpy(a, in, n);
    }
    for (; rc == 0 && s >= 0; s--) {
        uint32_t k = p->stage_kind[s], prm = p->stage_param[s];
        if (k == KVO_ST_TUPL) kvo_tupl_decode(a, n, prm, b);
        else if (k == KVO_ST_BIT) kvo_bit_decode(a, n, b);
        else if (k == KVO_ST_DELTA) kvo_delta_decode(a, n, prm, b);
        else { rc = -1; break; } /* RZE only as the last stage */
        uint8_t *t = a; a = b; b = t;
    }
    if (rc == 0) memcpy(out, a, n);
    free(a);
    free(b);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Stream container (READING; "GPU-resident compressed bitstream" and a      */
/* "compressed-size scalar", [FastKVComp] §4.2).                              */
/*  [0,64)   header (little-endian; see kvo_write_header)                    */
/*  [64,HB)  v2 width map (only with per-(layer, head) widths; HB = header    */
/*           bytes, written at header offset 6)                               */
/*  no stages: Q follows at byte HB.                                         */
/*  stages:   u32 table[n_chunks] at byte HB (bit 31 = stored raw, bits 0..30 */
/*            = stored size); chunk i starts at data_start + sum_{j<i}       */
/*            align16(size_j), data_start = align16(HB + 4 n_chunks);        */
/*            padding bytes are zero.                                        */
/* ------------------------------------------------------------------------ */
/* READING (v2): version 2 when the profile uses the token delta or width maps,
 * else 1.  Flags byte: bit 0 smoothing, bit 1 Hadamard, bit 2 token delta, bit 3
 * width map.  With a map the two width bytes are 0 and the map follows the 64
 * header bytes: entry i takes bits 2i, 2i+1 (least significant first) with the
 * code 0, 1, 2, 3 for widths 2, 3, 4, 8; K entries l*H + h come first, then V. */
static uint32_t width_code(uint32_t bits) { return bits == 2 ? 0u : bits == 3 ? 1u : bits == 4 ? 2u : 3u; }

void kvo_write_header(const kvo_profile *p, const kvo_shape *sh, const kvo_layout *lay, uint8_t *h)
{
    memset(h, 0, lay->header_bytes);
    const int v2 = p->token_delta || has_maps(p);
    h[0] = 'K'; h[1] = 'V'; h[2] = 'C'; h[3] = '1';
    put_u16(h + 4, v2 ? 2 : 1);        /* format version */
    put_u16(h + 6, (uint16_t)lay->header_bytes);
    put_u32(h + 8, sh->layers);
    put_u32(h + 12, sh->tokens);
    put_u16(h + 16, (uint16_t)sh->kv_heads);
    put_u16(h + 18, (uint16_t)sh->head_dim);
    h[20] = (uint8_t)sh->dtype;
    h[21] = (uint8_t)((p->smooth_keys ? 1 : 0) | (p->hadamard ? 2 : 0) | (p->token_delta ? 4 : 0) |
                      (has_maps(p) ? 8 : 0));
    h[22] = has_maps(p) ? 0 : (uint8_t)p->bits_k;
    h[23] = has_maps(p) ? 0 : (uint8_t)p->bits_v;
    if (has_maps(p)) {
        const uint64_t n = (uint64_t)sh->layers * sh->kv_heads;
        for (int tensor = 0; tensor < 2; tensor++)
            for (uint64_t i = 0; i < n; i++) {
                uint64_t e = tensor * n + i;
                uint32_t w = width_code(width_of(p, tensor, sh->kv_heads, (uint32_t)(i / sh->kv_heads),
                                                 (uint32_t)(i % sh->kv_heads)));
                h[KVO_HEADER_BYTES + e / 4] |= (uint8_t)(w << (2 * (e % 4)));
            }
    }
    put_u16(h + 24, (uint16_t)p->group_k);
    put_u16(h + 26, (uint16_t)p->group_v);
    h[28] = (uint8_t)p->axis_k;
    h[29] = (uint8_t)p->axis_v;
    h[30] = (uint8_t)p->n_stages;
    for (uint32_t s = 0; s < p->n_stages; s++) {
        h[32 + 2 * s] = (uint8_t)p->stage_kind[s];
        h[33 + 2 * s] = (uint8_t)p->stage_param[s];
    }
    put_u32(h + 40, p->n_stages ? p->chunk_bytes : 0);
    put_u32(h + 44, (uint32_t)lay->n_chunks);
    put_u64(h + 48, p->seed);
    put_u64(h + 56, lay->payload_bytes);
}

/* Lossless-encode Q into stream (after the header).  Returns the total stream size. */
uint64_t kvo_lossless_encode(const kvo_profile *p, const kvo_layout *lay, const uint8_t *Q, uint8_t *stream)
{
    const uint64_t HB = lay->header_bytes;
    if (p->n_stages == 0) {
        memcpy(stream + HB, Q, lay->payload_bytes);
        return HB + lay->payload_bytes;
    }
    const uint64_t nc = lay->n_chunks, cb = p->chunk_bytes, P = lay->payload_bytes;
    uint8_t *tmp = (uint8_t *)malloc(nc * cb + 16);
    uint32_t *sizes = (uint32_t *)malloc((nc ? nc : 1) * sizeof(uint32_t));
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < (int64_t)nc; i++) {
        uint64_t off = (uint64_t)i * cb, n = (off + cb <= P) ? cb : P - off;
        int raw;
        size_t sz = kvo_chunk_encode(p, Q + off, n, tmp + off, &raw);
        sizes[i] = (uint32_t)sz | (raw ? 0x80000000u : 0u);
    }
    uint64_t pos = lay->data_start;
    memset(stream + HB, 0, lay->data_start - HB);
    for (uint64_t i = 0; i < nc; i++) {
        put_u32(stream + HB + 4 * i, sizes[i]);
        uint64_t sz = sizes[i] & 0x7fffffffu;
        memcpy(stream + pos, tmp + i * cb, sz);
        memset(stream + pos + sz, 0, align16(sz) - sz);
        pos += align16(sz);
    }
    free(sizes);
    free(tmp);
    return pos;
}

/* Full encode: quantize, then header + lossless stream.  Returns flags; the
 * stream size goes to *stream_bytes.  cap = capacity of `stream`. */
uint32_t kvo_encode(const kvo_profile *p, const kvo_shape *sh,
                    const uint8_t *const *k_bases, const uint8_t *const *v_bases, const int32_t *block_table,
                    uint8_t *stream, uint64_t cap, uint64_t *stream_bytes)
{
    kvo_layout lay;
    kvo_layout_of(p, sh, &lay);
    *stream_bytes = 0;
    if (cap < lay.max_stream_bytes) return KVO_FLAG_CAPACITY;
    uint8_t *Q = (uint8_t *)malloc(lay.payload_bytes ? lay.payload_bytes : 1);
    uint32_t flags = kvo_quantize(p, sh, k_bases, v_bases, block_table, Q);
    kvo_write_header(p, sh, &lay, stream);
    *stream_bytes = kvo_lossless_encode(p, &lay, Q, stream);
    free(Q);
    return flags;
}

/* Decode: validate the header against the profile and shape, undo the lossless
 * stages into Q, then reconstruct.  Writes nothing to K/V when corrupt. */
uint32_t kvo_lossless_decode(const kvo_profile *p, const kvo_shape *sh, const uint8_t *stream, uint64_t stream_bytes,
                             uint8_t *Q)
{
    kvo_layout lay;
    kvo_layout_of(p, sh, &lay);
    const uint64_t HB = lay.header_bytes;
    uint8_t *want = (uint8_t *)malloc(HB);
    kvo_write_header(p, sh, &lay, want);
    int hdr_bad = stream_bytes < HB || memcmp(want, stream, HB) != 0;
    free(want);
    if (hdr_bad) return KVO_FLAG_CORRUPT;
    if (p->n_stages == 0) {
        if (stream_bytes < HB + lay.payload_bytes) return KVO_FLAG_CORRUPT;
        memcpy(Q, stream + HB, lay.payload_bytes);
        return 0;
    }
    const uint64_t nc = lay.n_chunks, cb = p->chunk_bytes, P = lay.payload_bytes;
    if (stream_bytes < lay.data_start) return KVO_FLAG_CORRUPT;
    uint64_t *offs = (uint64_t *)malloc((nc ? nc : 1) * sizeof(uint64_t));
    uint64_t pos = lay.data_start;
    int bad = 0;
    for (uint64_t i = 0; i < nc; i++) {
        uint32_t e = get_u32(stream + HB + 4 * i);
        uint64_t sz = e & 0x7fffffffu;
        offs[i] = pos;
        pos += align16(sz);
        if (pos > stream_bytes) bad = 1;
    }
    if (!bad) {
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
        for (int64_t i = 0; i < (int64_t)nc; i++) {
            uint32_t e = get_u32(stream + HB + 4 * i);
            uint64_t off = (uint64_t)i * cb, n = (off + cb <= P) ? cb : P - off;
            if (kvo_chunk_decode(p, stream + offs[i], e & 0x7fffffffu, (int)(e >> 31), n, Q + off) != 0) bad = 1;
        }
    }
    free(offs);
    return bad ? KVO_FLAG_CORRUPT : 0;
}

uint32_t kvo_decode(const kvo_profile *p, const kvo_shape *sh, const uint8_t *stream, uint64_t stream_bytes,
                    uint8_t *const *k_bases, uint8_t *const *v_bases, const int32_t *block_table)
{
    kvo_layout lay;
    kvo_layout_of(p, sh, &lay);
    uint8_t *Q = (uint8_t *)malloc(lay.payload_bytes ? lay.payload_bytes : 1);
    uint32_t flags = kvo_lossless_decode(p, sh, stream, stream_bytes, Q);
    if (!(flags & KVO_FLAG_CORRUPT)) kvo_dequantize(p, sh, Q, k_bases, v_bases, block_table);
    free(Q);
    return flags;
}

int kvo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
