/*
 * q8_oracle.c -- plain, slow, single-threaded CPU oracle for the Q8_0 weight x q8_1
 * activation block-quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls
 * this file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load it (through oracle/__init__.py).  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Sources (docs.rs pages of the memra-engine crate):
 *   [accprobe]  memra-engine 0.124.1, src/bin/accprobe_bench.rs
 *               - synth_w_q8_0: a Q8_0 row is in_f/32 blocks of 34 bytes, an fp16 scale
 *                 at +0 (little endian) followed by 32 int8 quants;
 *               - f32_to_f16_bits: binary16 with round-to-nearest-even;
 *               - module doc: the MMQ floor applies the scales once per 32-wide k block.
 *   [census]    memra-engine 0.113.0, src/bin/decode_kernel_census.rs, fn q8:
 *               row_bytes = in_f/32*(32+2); q8_1 activation = one i8 per column plus a
 *               per-32-block f32 scale; bytes streamed = out_f*row_bytes.
 *   [f16_ffi]   memra-engine 0.81.0, src/memra_engine/f16_ffi.rs
 *               - module doc, numeric-config paragraph: int8 values are exact in fp16,
 *                 so the dequant rounds only the d*q products;
 *               - try_f16_gemm / f16_act / build_q8_f16 (W8A8 pilot): amax = max |v|;
 *                 if amax > 0 { d = amax/127; q = (v/d).round().clamp(-127, 127) }.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the quantizer divides by the f32 scale d = amax/127 with IEEE division and rounds
 *     half away from zero (Rust f32::round); a block whose d is 0 gets all-zero quants;
 *   - the Q8_0 weight quantizer divides by the f32 d and stores fp16(d) (round to
 *     nearest even);
 *   - the fold is y = sum over blocks, in ascending block order, of
 *     (f32(d_w) * d_a) * f32(D) with f32 rounding after every operation (y32), and the
 *     same sum with double products and accumulation (y64, the reference value).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off keeps every f32 multiply and add separately rounded.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define QK 32           /* values per block                                   */
#define Q8_0_BYTES 34   /* fp16 scale + 32 int8 quants, [accprobe] synth_w_q8_0 */

/* ------------------------------------------------------------------------------------ */
/* O0: IEEE-754 binary16 <-> binary32, written from the format definition.               */
/*   binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                  */
/*   normal    value = (1024 + f) * 2^(e - 25), e in 1..30                               */
/*   subnormal value = f * 2^-24                                                         */
/* ------------------------------------------------------------------------------------ */

float oracle_f16_to_f32(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexpf((float)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round-to-nearest, ties-to-even, with gradual underflow and overflow to infinity. */
uint16_t oracle_f32_to_f16(float x)
{
    uint32_t b;
    memcpy(&b, &x, sizeof b);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    uint32_t ebits = (b >> 23) & 0xffu;
    uint32_t frac = b & 0x7fffffu;

    if (ebits == 0xffu)                         /* inf / NaN */
        return frac ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7c00u);
    if (ebits == 0)                             /* f32 zero or subnormal: < 2^-126 */
        return sign;                            /* far below half of 2^-24        */

    /* |x| = sig * 2^(e - 23), sig in [2^23, 2^24) */
    int e = (int)ebits - 127;
    uint32_t sig = frac | 0x800000u;
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);      /* |x| >= 2^16 > max finite */

    /* Number of low bits of sig to drop: 13 for normal binary16 results; more when the
       result is subnormal (unit 2^-24). */
    int shift = (e >= -14) ? 13 : (-1 - e);
    if (shift > 24)
        return sign;                            /* |x| < 2^-25: rounds to zero */
    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1u;

    uint32_t enc;
    if (e >= -14)
        enc = ((uint32_t)(e + 14) << 10) + q;   /* q carries the implicit 1024; a carry
                                                   to 2048 bumps the exponent, and
                                                   0x7c00 is infinity */
    else
        enc = q;                                /* q == 1024 is the smallest normal */
    if (enc > 0x7c00u)
        enc = 0x7c00u;
    return (uint16_t)(sign | enc);
}

/* Array forms of the two conversions (one call instead of one per element). */
void oracle_f32_to_f16_array(const float *x, uint16_t *h, int64_t count)
{
    for (int64_t i = 0; i < count; i++)
        h[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f16_to_f32_array(const uint16_t *h, float *x, int64_t count)
{
    for (int64_t i = 0; i < count; i++)
        x[i] = oracle_f16_to_f32(h[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Per-block scalar quantization, [f16_ffi] W8A8 pilot:                                   */
/*   amax = max |v|;  d = amax / 127;  q = clamp(round_half_away(v / d), -127, 127).      */
/* Returns d; writes 32 quants.                                                          */
/* ------------------------------------------------------------------------------------ */
static float quantize_block(const float *v, int8_t *q)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; i++) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    for (int i = 0; i < QK; i++) {
        if (d == 0.0f) {
            q[i] = 0;
            continue;
        }
        float r = roundf(v[i] / d);
        if (r != r)          /* NaN (a NaN entry, or inf / inf): out of contract, quantized to 0 */
            r = 0.0f;
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        q[i] = (int8_t)r;
    }
    return d;
}

/* O2: q8_1 activation quantization, [census] fn q8 (one i8 per column plus a per-32-block
   f32 scale).  x is [m][k] row-major; xq is [m][k]; xd is [m][k/32]. */
void oracle_quantize_q8_1(const float *x, int8_t *xq, float *xd, int64_t m, int64_t k)
{
    int64_t nb = k / QK;
    for (int64_t t = 0; t < m; t++)
        for (int64_t b = 0; b < nb; b++)
            xd[t * nb + b] = quantize_block(x + t * k + b * QK, xq + t * k + b * QK);
}

/* O1: Q8_0 weight quantization (data preparation).  w is [n][k] row-major; out holds n
   rows of k/32 blocks of 34 bytes: fp16(d) little endian, then 32 int8 quants. */
void oracle_quantize_q8_0(const float *w, uint8_t *out, int64_t n, int64_t k)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < nb; b++) {
            uint8_t *blk = out + (r * nb + b) * Q8_0_BYTES;
            int8_t q[QK];
            float d = quantize_block(w + r * k + b * QK, q);
            uint16_t h = oracle_f32_to_f16(d);
            blk[0] = (uint8_t)(h & 0xff);
            blk[1] = (uint8_t)(h >> 8);
            memcpy(blk + 2, q, QK);
        }
}

static const uint8_t *block_ptr(const uint8_t *w, int64_t r, int64_t b, int64_t nb)
{
    return w + (r * nb + b) * Q8_0_BYTES;
}

static float block_scale(const uint8_t *blk)
{
    return oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
}

static int32_t block_dot(const uint8_t *blk, const int8_t *xq)
{
    const int8_t *wq = (const int8_t *)(blk + 2);
    int32_t s = 0;
    for (int i = 0; i < QK; i++)
        s += (int32_t)wq[i] * (int32_t)xq[i];
    return s;
}

/* O3: exact per-block integer dots D[t][j][b] = sum_i wq[r_j, 32b+i] * xq[t, 32b+i]
   for the selected weight rows r_j = rows[j] (all rows when rows == NULL). */
void oracle_block_dots(const uint8_t *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n,
                       int64_t k, const int64_t *rows, int64_t nrows)
{
    int64_t nb = k / QK;
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            for (int64_t b = 0; b < nb; b++)
                D[(t * nr + j) * nb + b] = block_dot(block_ptr(w, r, b, nb), xq + t * k + b * QK);
        }
}

/* O4: the fold.  For each token t and selected weight row r_j:
     y32[t][j] = sum_b (f32(d_w[r,b]) * d_a[t,b]) * f32(D)   (f32, ascending b)
     y64[t][j] = sum_b  d_w * d_a * D                          (double)
     S[t][j]   = sum_b |d_w * d_a * D|                         (double; error scale)
   Any output pointer may be NULL. */
void oracle_matmul(const uint8_t *w, const int8_t *xq, const float *xd, int64_t m, int64_t n,
                   int64_t k, const int64_t *rows, int64_t nrows, float *y32, double *y64,
                   double *S)
{
    int64_t nb = k / QK;
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            float acc32 = 0.0f;
            double acc64 = 0.0, abs64 = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *blk = block_ptr(w, r, b, nb);
                int32_t dot = block_dot(blk, xq + t * k + b * QK);
                float dw = block_scale(blk);
                float da = xd[t * nb + b];
                float s = dw * da;
                float term = s * (float)dot;
                acc32 = acc32 + term;
                double term64 = (double)dw * (double)da * (double)dot;
                acc64 += term64;
                abs64 += fabs(term64);
            }
            if (y32)
                y32[t * nr + j] = acc32;
            if (y64)
                y64[t * nr + j] = acc64;
            if (S)
                S[t * nr + j] = abs64;
        }
}

/* O5: Q8_0 -> fp16 row-major dequant, [f16_ffi] memra_q8_0_dequant_f16:
   w16[r][32b+i] = fp16_rn(f32(d_w) * q).  The f32 product of an 11-bit significand and
   a 7-bit integer is exact, so this is the correctly rounded fp16 of the exact product. */
void oracle_dequant_f16(const uint8_t *w, uint16_t *out, int64_t n, int64_t k)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = block_ptr(w, r, b, nb);
            float dw = block_scale(blk);
            const int8_t *wq = (const int8_t *)(blk + 2);
            for (int i = 0; i < QK; i++)
                out[r * k + b * QK + i] = oracle_f32_to_f16(dw * (float)wq[i]);
        }
}

/* O6: load-time repack of Q8_0 for the tensor-core GEMM (a layout change, no arithmetic
   beyond exact conversions): wq16[r][32b+i] = binary16(q) -- exact, |q| <= 127 -- and the
   scale plane wdt[b][r] = f32(d_w[r][b]), block-major with leading dimension ldn >= n
   (columns n..ldn-1 are left untouched). */
void oracle_repack_q8_0(const uint8_t *w, uint16_t *wq16, float *wdt, int64_t n, int64_t k,
                        int64_t ldn)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = block_ptr(w, r, b, nb);
            const int8_t *wq = (const int8_t *)(blk + 2);
            for (int i = 0; i < QK; i++)
                wq16[r * k + b * QK + i] = oracle_f32_to_f16((float)wq[i]);
            wdt[b * ldn + r] = block_scale(blk);
        }
}

/* ------------------------------------------------------------------------------------ */
/* O7: Q4_0 weights, [f16_ffi] memra_q4_0_dequant_f16 ("GGUF Q4_0 18B blocks -> row-major */
/* fp16 mirror").  The page names the GGUF format and its 18-byte block; the layout read  */
/* here is that format's: an fp16 scale d (little endian) at +0, then 16 bytes, element i */
/* (i < 16) in the low nibble of byte 2 + i and element i + 16 in its high nibble, value  */
/* d * (nibble - 8).                                                                      */
/* ------------------------------------------------------------------------------------ */
#define Q4_0_BYTES 18

static int q4_0_value(const uint8_t *blk, int i)
{
    uint8_t byte = blk[2 + (i & 15)];
    int nib = (i < 16) ? (byte & 0x0f) : (byte >> 4);
    return nib - 8;
}

static const uint8_t *q4_0_block_ptr(const uint8_t *w, int64_t r, int64_t b, int64_t nb)
{
    return w + (r * nb + b) * Q4_0_BYTES;
}

/* O7a: Q4_0 writer (data preparation; the pages give no quantizer for it): per block
   amax = max |v|, d = amax / 7 (f32), q = clamp(round_half_away(v / d), -8, 7), stored as
   the nibble q + 8 with fp16(d); a block whose d is 0 stores d = 0 and nibbles 8. */
void oracle_quantize_q4_0(const float *w, uint8_t *out, int64_t n, int64_t k)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < nb; b++) {
            const float *v = w + r * k + b * QK;
            uint8_t *blk = out + (r * nb + b) * Q4_0_BYTES;
            float amax = 0.0f;
            for (int i = 0; i < QK; i++) {
                float a = fabsf(v[i]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 7.0f;
            int nib[QK];
            for (int i = 0; i < QK; i++) {
                float q = 0.0f;
                if (d != 0.0f) {
                    q = roundf(v[i] / d);
                    if (q != q)
                        q = 0.0f;
                    if (q > 7.0f)
                        q = 7.0f;
                    if (q < -8.0f)
                        q = -8.0f;
                }
                nib[i] = (int)q + 8;
            }
            uint16_t h = oracle_f32_to_f16(d);
            blk[0] = (uint8_t)(h & 0xff);
            blk[1] = (uint8_t)(h >> 8);
            for (int i = 0; i < 16; i++)
                blk[2 + i] = (uint8_t)(nib[i] | (nib[i + 16] << 4));
        }
}

/* O7b: Q4_0 -> fp16 row-major dequant: w16[r][32b+i] = fp16_rn(f32(d) * (nibble - 8)).
   The f32 product of an 11-bit significand and an integer in [-8, 7] is exact. */
void oracle_dequant_q4_0_f16(const uint8_t *w, uint16_t *out, int64_t n, int64_t k)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < n; r++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = q4_0_block_ptr(w, r, b, nb);
            float dw = block_scale(blk);
            for (int i = 0; i < QK; i++)
                out[r * k + b * QK + i] = oracle_f32_to_f16(dw * (float)q4_0_value(blk, i));
        }
}

static int32_t q4_0_block_dot(const uint8_t *blk, const int8_t *xq)
{
    int32_t s = 0;
    for (int i = 0; i < QK; i++)
        s += (int32_t)q4_0_value(blk, i) * (int32_t)xq[i];
    return s;
}

/* O7c: exact block dots of Q4_0 weights with q8_1 quants, as O3. */
void oracle_block_dots_q4_0(const uint8_t *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n,
                            int64_t k, const int64_t *rows, int64_t nrows)
{
    int64_t nb = k / QK;
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            for (int64_t b = 0; b < nb; b++)
                D[(t * nr + j) * nb + b] = q4_0_block_dot(q4_0_block_ptr(w, r, b, nb), xq + t * k + b * QK);
        }
}

/* O7d: the fold of O4 over Q4_0 blocks (y32 in f32, ascending b; y64 and S in double). */
void oracle_matmul_q4_0(const uint8_t *w, const int8_t *xq, const float *xd, int64_t m, int64_t n,
                        int64_t k, const int64_t *rows, int64_t nrows, float *y32, double *y64,
                        double *S)
{
    int64_t nb = k / QK;
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            float acc32 = 0.0f;
            double acc64 = 0.0, abs64 = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *blk = q4_0_block_ptr(w, r, b, nb);
                int32_t dot = q4_0_block_dot(blk, xq + t * k + b * QK);
                float dw = block_scale(blk);
                float da = xd[t * nb + b];
                float s = dw * da;
                float term = s * (float)dot;
                acc32 = acc32 + term;
                double term64 = (double)dw * (double)da * (double)dot;
                acc64 += term64;
                abs64 += fabs(term64);
            }
            if (y32)
                y32[t * nr + j] = acc32;
            if (y64)
                y64[t * nr + j] = acc64;
            if (S)
                S[t * nr + j] = abs64;
        }
}

/* ------------------------------------------------------------------------------------ */
/* O8: K-quant superblocks, [f16_ffi] memra_q6_K_dequant_f16 / memra_q4_K_dequant_f16 /   */
/* memra_q5_K_dequant_f16 ("GGUF Q6_K 210B / Q4_K 144B / Q5_K 176B superblocks ->         */
/* row-major fp16 mirror").  The page names the GGUF formats and their superblock sizes;  */
/* the layouts read here are those formats' (256 weights per superblock):                 */
/*                                                                                        */
/* Q6_K (210 bytes): ql[128] at +0, qh[64] at +128, int8 scales[16] at +192, fp16 d at    */
/*   +208.  Weight e (0..255) lies in half h = e / 128, at p = e % 128 = 32 g + l (g 0..3, */
/*   l 0..31); its 6-bit code q = (low 4 bits: the low nibble (g < 2) or high nibble       */
/*   (g >= 2) of ql[64 h + 32 (g % 2) + l]) + 16 * ((qh[32 h + l] >> 2 g) & 3), and its    */
/*   value is d * scales[e / 16] * (q - 32).                                               */
/* Q4_K (144 bytes): fp16 d at +0, fp16 dmin at +2, 12 scale bytes at +4, qs[128] at +16.  */
/*   Sub-block j (0..7) of 32 weights has a 6-bit scale sc_j and a 6-bit min m_j:          */
/*   j < 4:  sc = s[j] & 63,  m = s[j + 4] & 63;                                           */
/*   j >= 4: sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4),                                */
/*           m  = (s[j + 4] >> 4) | ((s[j] >> 6) << 4).                                    */
/*   Weight e = 64 g + 32 u + l (g 0..3, u 0..1) is in sub-block j = 2 g + u, its 4-bit    */
/*   code q is the low (u = 0) or high (u = 1) nibble of qs[32 g + l], and its value is   */
/*   d * sc_j * q - dmin * m_j.                                                            */
/* Q5_K (176 bytes): as Q4_K with qh[32] at +16 and qs[128] at +48; the code gains a fifth */
/*   bit, q += 16 * ((qh[l] >> j) & 1).                                                    */
/*                                                                                        */
/* Readings (the pages are silent): the fp16 mirror is the correctly rounded binary16 of   */
/* each weight's exact value (as for Q8_0, where the f32 product is already exact); the    */
/* matmul with the q8_1 activation takes, per 32-wide activation block b, exact integers   */
/* -- Q6_K: E_b = sc_2i * sum_{first 16} (q - 32) xq + sc_2i+1 * sum_{last 16} (q - 32) xq */
/* (i = b % 8); Q4_K / Q5_K: D_b = sum q xq and X_b = sum xq -- and folds them with the    */
/* block's scales: y += d d_a E_b, or y += d_a (d sc_j D_b - dmin m_j X_b).                */
/* ------------------------------------------------------------------------------------ */
#define QK_K 256
#define Q6_K_BYTES 210
#define Q4_K_BYTES 144
#define Q5_K_BYTES 176

enum { KQ_Q6_K = 6, KQ_Q4_K = 4, KQ_Q5_K = 5 };

static int kq_bytes(int fmt)
{
    return fmt == KQ_Q6_K ? Q6_K_BYTES : fmt == KQ_Q4_K ? Q4_K_BYTES : Q5_K_BYTES;
}

static float f16_at(const uint8_t *p)
{
    return oracle_f16_to_f32((uint16_t)(p[0] | (p[1] << 8)));
}

/* The 6-bit scale and min of sub-block j of a Q4_K / Q5_K superblock (12 scale bytes s). */
static void k4_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* The unsigned code of weight e of a superblock (Q6_K: 0..63, Q4_K: 0..15, Q5_K: 0..31). */
static int kq_code(int fmt, const uint8_t *sb, int e)
{
    if (fmt == KQ_Q6_K) {
        int h = e / 128, p = e % 128, g = p / 32, l = p % 32;
        int byte = sb[64 * h + 32 * (g % 2) + l];
        int lo = (g < 2) ? (byte & 15) : (byte >> 4);
        int hi = (sb[128 + 32 * h + l] >> (2 * g)) & 3;
        return lo + 16 * hi;
    }
    int g = e / 64, u = (e / 32) % 2, l = e % 32;
    const uint8_t *qs = sb + (fmt == KQ_Q4_K ? 16 : 48);
    int byte = qs[32 * g + l];
    int q = u ? (byte >> 4) : (byte & 15);
    if (fmt == KQ_Q5_K)
        q += 16 * ((sb[16 + l] >> (2 * g + u)) & 1);
    return q;
}

/* The exact value of weight e of a superblock, in double (every such value is an integer
   multiple of 2^-24 below 2^28 in magnitude, so double holds it exactly). */
static double kq_value(int fmt, const uint8_t *sb, int e)
{
    int q = kq_code(fmt, sb, e);
    if (fmt == KQ_Q6_K) {
        int sc = (int)(int8_t)sb[192 + e / 16];
        return (double)f16_at(sb + 208) * (double)sc * (double)(q - 32);
    }
    int sc, m;
    k4_scale_min(sb + 4, e / 32, &sc, &m);
    return (double)f16_at(sb) * (double)sc * (double)q - (double)f16_at(sb + 2) * (double)m;
}

/* binary64 -> binary16, round to nearest even (gradual underflow, overflow to infinity),
   written from the two formats' definitions like oracle_f32_to_f16. */
uint16_t oracle_f64_to_f16(double x)
{
    uint64_t b;
    memcpy(&b, &x, sizeof b);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    uint32_t ebits = (uint32_t)((b >> 52) & 0x7ffu);
    uint64_t frac = b & 0xfffffffffffffull;
    if (ebits == 0x7ffu)
        return frac ? (uint16_t)(sign | 0x7e00u) : (uint16_t)(sign | 0x7c00u);
    if (ebits == 0)
        return sign;                                  /* zero or < 2^-1022 */
    int e = (int)ebits - 1023;                        /* |x| = sig * 2^(e - 52) */
    uint64_t sig = frac | (1ull << 52);
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);
    int shift = (e >= -14) ? 42 : (28 - e);           /* bits dropped: result unit 2^-24 below 2^-14 */
    if (shift > 53)
        return sign;                                  /* |x| < 2^-25 */
    uint64_t q = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1u;
    uint64_t enc = (e >= -14) ? ((uint64_t)(e + 14) << 10) + q : q;
    if (enc > 0x7c00u)
        enc = 0x7c00u;
    return (uint16_t)(sign | (uint16_t)enc);
}

/* O8a: K-quant -> fp16 row-major dequant: w16[r][e] = fp16_rn(exact value of weight e). */
void oracle_dequant_kq_f16(int fmt, const uint8_t *w, uint16_t *out, int64_t n, int64_t k)
{
    int64_t ns = k / QK_K, sbytes = kq_bytes(fmt);
    for (int64_t r = 0; r < n; r++)
        for (int64_t s = 0; s < ns; s++) {
            const uint8_t *sb = w + (r * ns + s) * sbytes;
            for (int e = 0; e < QK_K; e++)
                out[r * k + s * QK_K + e] = oracle_f64_to_f16(kq_value(fmt, sb, e));
        }
}

/* The exact integers of 32-wide activation block i (0..7) of a superblock: *E for Q6_K;
   *D = sum q xq and *X = sum xq for Q4_K / Q5_K. */
static void kq_block_ints(int fmt, const uint8_t *sb, int i, const int8_t *xq, int32_t *E, int32_t *D, int32_t *X)
{
    int32_t d0 = 0, d1 = 0, x = 0;
    for (int l = 0; l < QK; l++) {
        int e = 32 * i + l;
        int q = kq_code(fmt, sb, e);
        x += xq[l];
        if (fmt == KQ_Q6_K) {
            if (l < 16)
                d0 += (q - 32) * xq[l];
            else
                d1 += (q - 32) * xq[l];
        } else {
            d0 += q * xq[l];
        }
    }
    if (fmt == KQ_Q6_K) {
        *E = (int32_t)(int8_t)sb[192 + 2 * i] * d0 + (int32_t)(int8_t)sb[192 + 2 * i + 1] * d1;
        *D = 0;
    } else {
        *E = 0;
        *D = d0;
    }
    *X = x;
}

/* O8b: the exact per-block integers the fold consumes, [t][j][b] for the selected rows:
   Q6_K: E_b; Q4_K / Q5_K: D_b (X_b depends on the activation only). */
void oracle_block_dots_kq(int fmt, const uint8_t *w, const int8_t *xq, int32_t *out, int64_t m,
                          int64_t n, int64_t k, const int64_t *rows, int64_t nrows)
{
    int64_t ns = k / QK_K, nb = k / QK, sbytes = kq_bytes(fmt);
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *sb = w + (r * ns + b / 8) * sbytes;
                int32_t E, D, X;
                kq_block_ints(fmt, sb, (int)(b % 8), xq + t * k + b * QK, &E, &D, &X);
                out[(t * nr + j) * nb + b] = (fmt == KQ_Q6_K) ? E : D;
            }
        }
}

/* O8c: the fold over K-quant weights.  Per 32-wide block b (ascending):
     Q6_K:          term = d * d_a * E_b
     Q4_K / Q5_K:   term = d_a * (d * sc_j * D_b - dmin * m_j * X_b)
   y32: f32, each operation rounded, in the order written; y64: double; S: the sum over
   blocks of the magnitudes of the term's products (d d_a E, or |d_a d sc D| + |d_a dmin m X|). */
void oracle_matmul_kq(int fmt, const uint8_t *w, const int8_t *xq, const float *xd, int64_t m,
                      int64_t n, int64_t k, const int64_t *rows, int64_t nrows, float *y32,
                      double *y64, double *S)
{
    int64_t ns = k / QK_K, nb = k / QK, sbytes = kq_bytes(fmt);
    int64_t nr = rows ? nrows : n;
    for (int64_t t = 0; t < m; t++)
        for (int64_t j = 0; j < nr; j++) {
            int64_t r = rows ? rows[j] : j;
            float acc32 = 0.0f;
            double acc64 = 0.0, abs64 = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *sb = w + (r * ns + b / 8) * sbytes;
                int i = (int)(b % 8);
                int32_t E, D, X;
                kq_block_ints(fmt, sb, i, xq + t * k + b * QK, &E, &D, &X);
                float da = xd[t * nb + b];
                if (fmt == KQ_Q6_K) {
                    float d = f16_at(sb + 208);
                    float s = d * da;
                    acc32 = acc32 + s * (float)E;
                    double term = (double)d * (double)da * (double)E;
                    acc64 += term;
                    abs64 += fabs(term);
                } else {
                    int sc, mn;
                    k4_scale_min(sb + 4, i, &sc, &mn);
                    float d = f16_at(sb), dmin = f16_at(sb + 2);
                    float dsc = d * (float)sc, dmm = dmin * (float)mn;
                    float v = dsc * (float)D - dmm * (float)X;
                    acc32 = acc32 + da * v;
                    double p1 = (double)da * (double)d * (double)sc * (double)D;
                    double p2 = (double)da * (double)dmin * (double)mn * (double)X;
                    acc64 += p1 - p2;
                    abs64 += fabs(p1) + fabs(p2);
                }
            }
            if (y32)
                y32[t * nr + j] = acc32;
            if (y64)
                y64[t * nr + j] = acc64;
            if (S)
                S[t * nr + j] = abs64;
        }
}
