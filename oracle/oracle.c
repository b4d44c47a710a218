/*
 * oracle.c -- plain, slow CPU oracle of the DeepSeek-V4.1 engram forward.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares
 * no code, header, table or helper with the CUDA path and includes nothing
 * from it.
 *
 * It follows the four stages of the CPU reference page
 * "metrale_model_arch/deepseek_v41_ref/engram.rs" in that page's order and
 * notation, with scalar loops and the precision the page fixes (i64 for the
 * hash, f32 for the projection and the gate).  The one departure, taken from
 * the GPU page "spark_model/layers/engram_v41.rs" (module doc, item 4), is
 * that the gate updates an FP32 highway: `bf16_out = 0` skips the final bf16
 * rounding of `gate_and_add`; `1` reproduces the CPU page exactly.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 * (-fopenmp optional).  Contraction must stay off: the pages round every f32
 * product and sum separately.  OpenMP only splits independent tokens or
 * output rows, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_E_CAPACITY -1 /* start_pos + T > max_seq */
#define ORC_E_TOKEN -2    /* input id outside token_map */
#define ORC_E_ROW -3      /* gathered row id outside the table */
#define ORC_E_PRIME -4    /* a prime <= 0 */

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the OpenMP loops (no effect without OpenMP). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* Number formats                                                       */
/* ------------------------------------------------------------------ */

static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* Round half to even, for |v| < 2^52. */
static double round_ties_even(double v) {
    double f = floor(v);
    double diff = v - f;
    if (diff > 0.5) return f + 1.0;
    if (diff < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* f32 -> bf16 bits, round to nearest, ties to even (the to_bf16_rne the CPU
 * page imports).  A NaN keeps its sign and becomes a quiet bf16 NaN. */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u = f2u(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float orc_bf16_to_f32(uint16_t b) { return u2f((uint32_t)b << 16); }

/* IEEE binary16 -> f32 (exact). */
float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    float v;
    if (e == 0) v = ldexpf((float)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexpf((float)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* e4m3fn decode (page "metrale_model_arch/deepseek_v41_ref/engram.rs", module
 * doc, item 2, and the doc of its e4m3 decoder).
 * exponent 15 with mantissa 7 is NaN; exponent 0 is subnormal m/8 * 2^-6;
 * otherwise (1 + m/8) * 2^(e-7); the sign is kept, so 0x80 is -0.0. */
float orc_e4m3_to_f32(uint8_t b) {
    float sign = (b & 0x80) ? -1.0f : 1.0f;
    int e = (b >> 3) & 0x0F;
    float m = (float)(b & 0x07);
    if (e == 15 && m == 7.0f) return NAN;
    if (e == 0) return sign * m / 8.0f * ldexpf(1.0f, -6);
    return sign * (1.0f + m / 8.0f) * ldexpf(1.0f, e - 7);
}

/* f32 -> e4m3fn, round to nearest even (the same page, the doc of its e4m3
 * encoder).  NaN -> 0x7F; |x| > 448 saturates to 0x7E; an f32 with
 * exponent field 0 (zero or f32 subnormal) -> signed zero; e4m3 subnormals
 * are RNE(|x| * 512); a mantissa that rounds up to 8 carries into the
 * exponent. */
uint8_t orc_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    float ax = fabsf(x);
    int exp_field = (int)((f2u(ax) >> 23) & 0xFF);
    if (exp_field == 0) return sign;
    double a = (double)ax;
    if (a > 448.0) return sign | 0x7E;
    int e = exp_field - 127;
    if (e < -6) return sign | (uint8_t)round_ties_even(a * 512.0);
    int mant = (int)round_ties_even((a * ldexp(1.0, -e) - 1.0) * 8.0);
    if (mant == 8) { e += 1; mant = 0; }
    return sign | (uint8_t)(((e + 7) << 3) | mant);
}

/* f32 -> e8m0 as a power of two (the same page, the doc of its e8m0 scale
 * encoder).  The nearest exponent; a mantissa of exactly one half
 * (x = 1.5 * 2^e) rounds up only when the biased exponent field is odd, so
 * the stored 8-bit code of a tie is even.  The sign is dropped. */
float orc_f32_to_e8m0(float x) {
    uint32_t bits = f2u(x);
    uint32_t e = (bits >> 23) & 0xFF;
    uint32_t m = bits & 0x7FFFFFu;
    if (m > 0x400000u || (m == 0x400000u && (e & 1u) == 1u)) e += 1;
    return u2f(e << 23);
}

/* e8m0 byte -> f32: the byte is a biased exponent, value 2^(code - 127);
 * code 255 is NaN (the byte f32_to_e8m0_rne's result stores: its exponent
 * field).  Code 0 is 2^-127, an f32 subnormal. */
float orc_e8m0_to_f32(uint8_t code) {
    if (code == 255) return NAN;
    return ldexpf(1.0f, (int)code - 127);
}

/* ------------------------------------------------------------------ */
/* Stage 1: the n-gram hash                                             */
/* ------------------------------------------------------------------ */

/* Two's-complement wrapping product: the exact product reduced mod 2^64,
 * read back as a signed value. */
static int64_t wrapping_mul(int64_t a, int64_t b) {
    return (int64_t)((uint64_t)a * (uint64_t)b);
}
static int64_t wrapping_add(int64_t a, int64_t b) {
    return (int64_t)((uint64_t)a + (uint64_t)b);
}

/* The Euclidean remainder of x by P > 0: the one r in [0, P) with
 * x - r divisible by P, taken from the exact 128-bit quotient. */
static int64_t euclid_mod(int64_t x, int64_t P) {
    __int128 r = (__int128)x % (__int128)P;   /* sign of x, |r| < P */
    if (r < 0) r += P;
    return (int64_t)r;
}

/* How many leading window slots of position p are real ids: the first shift
 * j (0 <= j < ng) that reaches before position 0 or lands on an unmapped
 * (-1) id, or ng if none does.  Slot j < cut holds cache[p - j]; slot
 * j >= cut holds the pad (a blocked slot blocks every larger shift). */
static int window_cut(const int64_t *seq_cache, int64_t p, int ng) {
    for (int j = 0; j < ng; ++j)
        if (j > p || seq_cache[p - j] == -1) return j;
    return ng;
}

/* The n-gram hash of the CPU reference page
 * "metrale_model_arch/deepseek_v41_ref/engram.rs" (module doc, item 1: the
 * compressed token map, the n-gram window with pad, the look-back cache
 * carried across the prefill/decode split, a multiplier per look-back slot,
 * the products XOR-combined, then % prime per (n-gram size, head) plus that
 * slot's offset), for a batch of sequences.  Written as equations:
 *
 *   cache[b][start_pos + s] = token_map[ids[b][s]]          (all s, first)
 *   w_j(p) = cache[b][p - j]   if j < cut(p),   pad_id otherwise
 *   for n-gram size g = 2 .. ng and head h, column c = (g - 2) H + h:
 *     X_g(p)        = XOR_{j = 0 .. g-1} ( w_j(p) *wrap mult[l][j] )
 *     id[b][s][l][c] = euclid_mod(X_g(p), primes[l][c]) + offsets[l][c]
 *
 *   token_map [vocab]          compressed id per token, -1 = unmapped
 *   pad_id                     token_map[pad token]
 *   mult    [L * ng]           multiplier of look-back slot j in layer l
 *   primes  [L * C]            prime of column c = (g - 2) H + h in layer l
 *   offsets [L * C]            row offset of that column in layer l's table
 *   cache   [B * max_seq]      compressed ids of every position seen (in/out)
 *   ids     [B * T]            input token ids at positions start_pos ..
 *   out     [B * T * L * C]    row ids
 *
 * Inputs are checked before the cache is touched. */
int orc_hash(const int64_t *token_map, int64_t vocab, int64_t pad_id,
             const int64_t *mult, const int64_t *primes, const int64_t *offsets,
             int L, int ng, int H, int64_t *cache, int B, int64_t max_seq,
             const int64_t *ids, int T, int64_t start_pos, int64_t *out) {
    const int C = (ng - 1) * H;
    if (ng < 2 || ng > 64) return ORC_E_CAPACITY;
    if (start_pos < 0 || start_pos + T > max_seq) return ORC_E_CAPACITY;
    for (int i = 0; i < L * C; ++i)
        if (primes[i] <= 0) return ORC_E_PRIME;
    for (int64_t i = 0; i < (int64_t)B * T; ++i)
        if (ids[i] < 0 || ids[i] >= vocab) return ORC_E_TOKEN;

    /* Every new position enters the cache before any window is formed. */
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < T; ++s)
            cache[(int64_t)b * max_seq + start_pos + s] = token_map[ids[(int64_t)b * T + s]];

    for (int b = 0; b < B; ++b) {
        const int64_t *seq_cache = cache + (int64_t)b * max_seq;
        for (int s = 0; s < T; ++s) {
            const int64_t p = start_pos + s;
            const int cut = window_cut(seq_cache, p, ng);
            for (int l = 0; l < L; ++l) {
                for (int g = 2; g <= ng; ++g) {
                    /* X_g: the g-slot window, each slot times its multiplier */
                    int64_t X = 0;
                    for (int j = 0; j < g; ++j) {
                        const int64_t w = j < cut ? seq_cache[p - j] : pad_id;
                        X ^= wrapping_mul(w, mult[(int64_t)l * ng + j]);
                    }
                    for (int h = 0; h < H; ++h) {
                        const int c = (g - 2) * H + h;
                        out[(((int64_t)b * T + s) * L + l) * C + c] =
                            wrapping_add(euclid_mod(X, primes[(int64_t)l * C + c]), offsets[(int64_t)l * C + c]);
                    }
                }
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Stage 2: table rows                                                  */
/* ------------------------------------------------------------------ */

/* Page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 2, for a table that
 * is already stored as e4m3 codes:
 *   row(id)[d] = bf16_rne( e4m3_to_f32(table[id][d]) * scales[id][d / blk] )
 * table [R, hd] u8, scales [R, hd / blk] f32, out [n, hd] bf16 bits. */
int orc_rows_fp8(const uint8_t *table, const float *scales, int64_t R, int hd, int blk,
                 const int64_t *ids, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= R) return ORC_E_ROW;
    const int nblk = hd / blk;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const int64_t id = ids[i];
        for (int d = 0; d < hd; ++d) {
            const float v = orc_e4m3_to_f32(table[id * hd + d]);
            const float s = scales[id * nblk + d / blk];
            out[i * hd + d] = orc_f32_to_bf16(v * s);
        }
    }
    return ORC_OK;
}

/* The fp8 rows with one-byte e8m0 scales (the 1-byte scale storage of
 * `f32_to_e8m0_rne` on the CPU reference page):
 *   row(id)[d] = bf16_rne( e4m3_to_f32(table[id][d]) * e8m0_to_f32(scales[id][d / blk]) )
 * scales [R, hd / blk] u8. */
int orc_rows_fp8_e8m0(const uint8_t *table, const uint8_t *scales, int64_t R, int hd, int blk,
                      const int64_t *ids, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= R) return ORC_E_ROW;
    const int nblk = hd / blk;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const int64_t id = ids[i];
        for (int d = 0; d < hd; ++d) {
            const float v = orc_e4m3_to_f32(table[id * hd + d]);
            const float s = orc_e8m0_to_f32(scales[id * nblk + d / blk]);
            out[i * hd + d] = orc_f32_to_bf16(v * s);
        }
    }
    return ORC_OK;
}

/* One 84-byte Q2_K block per 256-wide row (page "spark_model/layers/engram_v41.rs",
 * module doc, item 2), in the ggml super-block layout:
 *   bytes  0..15  scales[16]: low nibble = sub-block scale, high = sub-block min
 *   bytes 16..79  qs[64]: 2-bit quants, four per byte
 *   bytes 80..81  d    (binary16, little-endian)
 *   bytes 82..83  dmin (binary16, little-endian)
 * Value v in [0, 256): half = v / 128, w = v % 128, j = w / 32, l = w % 32,
 *   q  = (qs[32 * half + l] >> 2j) & 3,   sb = 8 * half + 2j + l / 16,
 *   y  = d * (scales[sb] & 15) * q - dmin * (scales[sb] >> 4),
 * then bf16 round-to-nearest-even.  out [n, 256] bf16 bits. */
int orc_rows_q2k(const uint8_t *blocks, int64_t R, const int64_t *ids, int64_t n,
                 uint16_t *out) {
    for (int64_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= R) return ORC_E_ROW;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const uint8_t *blk = blocks + ids[i] * 84;
        const uint8_t *sc = blk;
        const uint8_t *qs = blk + 16;
        const float d = orc_f16_to_f32((uint16_t)(blk[80] | (blk[81] << 8)));
        const float dmin = orc_f16_to_f32((uint16_t)(blk[82] | (blk[83] << 8)));
        for (int v = 0; v < 256; ++v) {
            const int half = v / 128, w = v % 128, j = w / 32, l = w % 32;
            const int q = (qs[32 * half + l] >> (2 * j)) & 3;
            const int s = sc[8 * half + 2 * j + l / 16];
            const float y = d * (float)(s & 15) * (float)q - dmin * (float)(s >> 4);
            out[i * 256 + v] = orc_f32_to_bf16(y);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Stage 3: the wkv projection                                          */
/* ------------------------------------------------------------------ */

/* Page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 3:
 *   y[r][o] = bf16_rne( sum_{i = 0 .. in-1} x[r][i] * w[o][i] ),
 * accumulated in f32 in index order.  x [rows, in] and w [out, in] are bf16
 * bits; y [rows, out] bf16 bits; acc (optional) receives the f32 sums before
 * rounding. */
void orc_linear_bf16(const uint16_t *x, int64_t rows, int64_t in_f, const uint16_t *w,
                     int64_t out_f, float *acc, uint16_t *y) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t o = 0; o < out_f; ++o) {
            const uint16_t *xr = x + r * in_f;
            const uint16_t *wr = w + o * in_f;
            float sum = 0.0f;
            for (int64_t i = 0; i < in_f; ++i)
                sum += orc_bf16_to_f32(xr[i]) * orc_bf16_to_f32(wr[i]);
            if (acc) acc[r * out_f + o] = sum;
            y[r * out_f + o] = orc_f32_to_bf16(sum);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Stage 4: the gate                                                    */
/* ------------------------------------------------------------------ */

/* Page "metrale_model_arch/deepseek_v41_ref/engram.rs", module doc, item 4, on
 * the FP32 highway:
 *   h  [T, hc, D] f32, updated in place
 *   kv [T, (hc + 1) * D] bf16 bits: key c = columns [c D, (c+1) D),
 *                                   value  = columns [hc D, (hc+1) D)
 *   q, k [hc, D] f32 (bf16 values); they enter only as their product.
 * Per (t, c), in f32 and index order:
 *   hh = sum h^2, kk = sum key^2, dot = sum (h * (q k)) * key
 *   s  = dot * (1/sqrt(hh/D + eps) * 1/sqrt(kk/D + eps)) * D^-1/2
 *   g  = copysign(sqrt(max(|s|, 1e-6)), s),  gate = 1 / (1 + exp(-g))
 *   h  = h + gate * value    (then bf16_rne when bf16_out != 0)
 * gate_out [T, hc] (optional) receives the gate values. */
void orc_gate(float *h, const uint16_t *kv, const float *q, const float *k, int64_t T,
              int hc, int D, float eps, int bf16_out, float *gate_out) {
    const int64_t kv_w = (int64_t)D * (hc + 1);
    const float inv_sqrt_dim = powf((float)D, -0.5f);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *value = kv + t * kv_w + (int64_t)hc * D;
        for (int c = 0; c < hc; ++c) {
            float *hr = h + (t * hc + c) * D;
            const uint16_t *key = kv + t * kv_w + (int64_t)c * D;
            float hh = 0.0f, kk = 0.0f, dot = 0.0f;
            for (int d = 0; d < D; ++d) {
                const float kd = orc_bf16_to_f32(key[d]);
                hh += hr[d] * hr[d];
                kk += kd * kd;
                dot += hr[d] * (q[c * D + d] * k[c * D + d]) * kd;
            }
            const float rstd = (1.0f / sqrtf(hh / (float)D + eps)) *
                               (1.0f / sqrtf(kk / (float)D + eps));
            const float s = dot * rstd * inv_sqrt_dim;
            const float g = copysignf(sqrtf(fmaxf(fabsf(s), 1e-6f)), s);
            const float gate = 1.0f / (1.0f + expf(-g));
            if (gate_out) gate_out[t * hc + c] = gate;
            for (int d = 0; d < D; ++d) {
                float o = hr[d] + gate * orc_bf16_to_f32(value[d]);
                if (bf16_out) o = orc_bf16_to_f32(orc_f32_to_bf16(o));
                hr[d] = o;
            }
        }
    }
}
