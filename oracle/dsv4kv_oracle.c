/*
 * dsv4kv oracle -- plain, slow, obviously-correct CPU reference of the
 * DeepSeek-V4.1 compressed-KV write (compress -> RMSNorm -> RoPE -> quantize
 * into a paged pool) and read (paged gather-dequant to bf16).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; every number in it is derived here from the definitions.
 *
 * Arithmetic is fp64 except where the method itself fixes fp32 (the
 * quantizer's decisions are taken on fp32 values, exactly as a store kernel
 * receives them; see orc_quantize_row).  Build with -ffp-contract=off and no
 * fast-math: rounding must be the one the C source spells out.
 *
 * Sources (web pages, cited by title and section):
 *  [P4]  sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels"
 *        -- Summary (KVLayout, PagedKV<layout, page_bits>::row, v41::store_row,
 *        c1/c2 compressors, V4.1 dequantizers) and the review of store_row_fp8
 *        (the ue8m0 closed form and clear_negative_zero).
 *  [P2]  sglang PR #46230 -- low_ratio_extend_offsets and the fused
 *        | kv | score | projection.
 *  [P3]  flashinfer_sparse.py -- compressed_block_size = block_size //
 *        compress_ratio and _compressed_topk_to_slots.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  row order codes-then-scales; FP4 low nibble = even dim; FP4 scale =
 *  e4m3(amax/6) with fp32 division; RoPE on interleaved pairs at position
 *  ratio*j; out_loc == 0 = not stored; id < 0 = zero row.
 *
 * Pins: every function here is checked by the CPU test-suite against
 * something other than itself (closed forms, torch/numpy library routines,
 * brute force, invariants).  No function is left "parity unpinned" except the
 * readings above that no page value fixes (FP4 nibble order and scale rule,
 * RoPE pair layout), which are self-consistent only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_D 512          /* latent width [P4 Summary: 448 nope + 64 rope] */
#define ORC_NOPE 448
#define ORC_ROPE 64

enum { ORC_V4 = 0, ORC_V41 = 1, ORC_V41_FP4 = 2 };

/* ------------------------------------------------------------------------ */
/* KVLayout row sizes [P4 Summary, KVLayout bullet]:                         */
/*   V4      = 448 fp8 nope + 64 bf16 rope (128 B) + ue8m0 scales -> 584 B   */
/*   V41     = 512 fp8 codes + one ue8m0 per 32 dims (16 B)       -> 528 B   */
/*   V41_FP4 = 512 e2m1 codes (256 B) + one e4m3 per 16 dims (32 B) -> 288 B */
/* ------------------------------------------------------------------------ */
int orc_row_bytes(int layout)
{
    switch (layout) {
    case ORC_V4:      return ORC_NOPE * 1 + ORC_ROPE * 2 + 8; /* 8 scale bytes: 584-448-128 */
    case ORC_V41:     return ORC_D * 1 + ORC_D / 32;
    case ORC_V41_FP4: return ORC_D / 2 + ORC_D / 16;
    default:          return -1;
    }
}

/* ------------------------------------------------------------------------ */
/* Number formats, from their definitions.                                  */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN and
 * there is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_value(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) mag = ldexp((double)m, -9);
    else         mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* FP4 E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal (m * 0.5).  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; no inf/NaN. */
double orc_e2m1_value(unsigned nib)
{
    unsigned s = (nib >> 3) & 1u, e = (nib >> 1) & 3u, m = nib & 1u;
    double mag;
    if (e == 0u) mag = 0.5 * (double)m;
    else         mag = ldexp(1.0 + (double)m / 2.0, (int)e - 1);
    return s ? -mag : mag;
}

/* Nearest representable magnitude by enumeration.  mags[0..n) ascending,
 * index == code.  Ties go to the even code (mantissa LSB 0): round-to-nearest-
 * even.  |a| beyond the largest finite value saturates ("satfinite").  The
 * two candidate distances are exact in fp64 (Sterbenz: adjacent codes are
 * within a factor two of each other, or one of them is zero). */
static unsigned nearest_code(double a, const double *mags, unsigned n)
{
    unsigned lo = 0, c;
    double dlo, dhi;
    if (a >= mags[n - 1]) return n - 1;
    for (c = 0; c < n; ++c)
        if (mags[c] <= a) lo = c;
    dlo = a - mags[lo];
    dhi = mags[lo + 1] - a;
    if (dlo < dhi) return lo;
    if (dhi < dlo) return lo + 1;
    return (lo & 1u) ? lo + 1 : lo;
}

/* Encode with sign; a result whose magnitude is zero is stored as +0
 * (clear_negative_zero [P4 review]). */
static unsigned encode_signed(double x, const double *mags, unsigned n, unsigned sign_bit)
{
    unsigned c = nearest_code(fabs(x), mags, n);
    if (c != 0u && x < 0.0) c |= sign_bit;
    return c;
}

static double E4M3_MAGS[127]; /* codes 0x00..0x7E, ascending */
static double E2M1_MAGS[8];
static int tables_ready = 0;

static void init_tables(void)
{
    unsigned c;
    if (tables_ready) return;
    for (c = 0; c < 127; ++c) E4M3_MAGS[c] = orc_e4m3_value(c);
    for (c = 0; c < 8; ++c)   E2M1_MAGS[c] = orc_e2m1_value(c);
    tables_ready = 1;
}

unsigned orc_e4m3_encode(double x)  /* RNE, satfinite, -0 -> +0 */
{
    init_tables();
    return encode_signed(x, E4M3_MAGS, 127u, 0x80u);
}

unsigned orc_e2m1_encode(double x)  /* RNE, satfinite, -0 -> +0 */
{
    init_tables();
    return encode_signed(x, E2M1_MAGS, 8u, 0x8u);
}

/* bf16 bits of x, round to nearest even, from the definition: 8 significant
 * bits, exponent range of fp32, subnormal step 2^-133, overflow -> inf. */
uint16_t orc_bf16_bits(double x)
{
    uint16_t sign;
    double a, step, v;
    int p, q;
    float vf;
    uint32_t b;
    if (isnan(x)) return 0x7FC0u;
    sign = signbit(x) ? 0x8000u : 0u;
    a = fabs(x);
    if (a == 0.0) return sign;
    (void)frexp(a, &p);             /* a in [2^(p-1), 2^p) */
    q = p - 1;
    if (q < -126) q = -126;         /* subnormals share the bottom binade's step */
    step = ldexp(1.0, q - 7);
    v = nearbyint(a / step) * step; /* default rounding mode: ties to even */
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    vf = (float)v;                  /* exact: v has <= 8 significant bits */
    memcpy(&b, &vf, 4);
    return (uint16_t)(sign | (b >> 16));
}

double orc_bf16_value(uint16_t bits)
{
    uint32_t b = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* ue8m0 scale byte of a V41 group [P4 review of store_row_fp8]:
 *     byte = 127 + ceil(log2(max(amax / 448, 1e-4)))
 * ceil(log2(.)) is monotone, so ceil(log2(max(u, v))) = max(ceil(log2 u),
 * ceil(log2 v)); ceil(log2(1e-4)) = -13.  ceil(log2(amax/448)) is the
 * smallest integer k with amax <= 448 * 2^k, found by exact fp64 comparison
 * (448 * 2^k is exact).  amax = 0 gives -inf, i.e. the -13 clamp. */
unsigned orc_ue8m0(float amax_f)
{
    double amax = (double)amax_f;
    int k, p;
    if (!(amax > 0.0)) return 127u - 13u;
    (void)frexp(amax, &p);
    k = p - 12;                               /* 448 * 2^(p-12) < 2^(p-3) < amax */
    while (ldexp(448.0, k) < amax) ++k;
    if (k < -13) k = -13;
    return (unsigned)(127 + k);
}

/* ------------------------------------------------------------------------ */
/* store_row: the single quantizer for the V4.1 rows [P4 Summary].           */
/* Input: the fp32 row the quantizer receives.  Output: row_bytes bytes,     */
/* codes first, then scales.                                                 */
/* ------------------------------------------------------------------------ */
int orc_quantize_row(int layout, const float *x, uint8_t *row)
{
    int g, d;
    if (layout == ORC_V41) {
        /* one ue8m0 byte per 32 dims; code = e4m3(x * 2^(127 - e)) */
        for (g = 0; g < ORC_D / 32; ++g) {
            float amax = 0.0f;
            unsigned e;
            for (d = 32 * g; d < 32 * g + 32; ++d)
                if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
            e = orc_ue8m0(amax);
            for (d = 32 * g; d < 32 * g + 32; ++d)
                row[d] = (uint8_t)orc_e4m3_encode(ldexp((double)x[d], 127 - (int)e));
            row[ORC_D + g] = (uint8_t)e;
        }
        return 0;
    }
    if (layout == ORC_V41_FP4) {
        /* one e4m3 scale per 16 dims: s = e4m3(amax / 6) (fp32 division);
         * code = e2m1(x / s) (fp32 division); s == 0 -> all codes 0.
         * Packing: dim 2i in the low nibble of byte i, 2i+1 in the high. */
        memset(row, 0, (size_t)orc_row_bytes(ORC_V41_FP4));
        for (g = 0; g < ORC_D / 16; ++g) {
            float amax = 0.0f, sdiv, sval;
            unsigned sc;
            for (d = 16 * g; d < 16 * g + 16; ++d)
                if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
            sdiv = amax / 6.0f;
            sc = orc_e4m3_encode((double)sdiv);
            sval = (float)orc_e4m3_value(sc);
            for (d = 16 * g; d < 16 * g + 16; ++d) {
                unsigned nib = 0u;
                if (sval != 0.0f) {
                    float q = x[d] / sval;
                    nib = orc_e2m1_encode((double)q);
                }
                row[d / 2] |= (uint8_t)(nib << (4 * (d & 1)));
            }
            row[ORC_D / 2 + g] = (uint8_t)sc;
        }
        return 0;
    }
    if (layout == ORC_V4) {
        /* V4 (reading of "448 fp8 nope + 64 bf16 rope + ue8m0 scales"):
         * bytes 0..447 e4m3 codes of dims 0..447 with one ue8m0 per 64 dims
         * (same closed form), bytes 448..575 the 64 rope dims as bf16 (RNE of
         * the fp32 value), bytes 576..582 the 7 scales, byte 583 zero. */
        for (g = 0; g < ORC_NOPE / 64; ++g) {
            float amax = 0.0f;
            unsigned e;
            for (d = 64 * g; d < 64 * g + 64; ++d)
                if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
            e = orc_ue8m0(amax);
            for (d = 64 * g; d < 64 * g + 64; ++d)
                row[d] = (uint8_t)orc_e4m3_encode(ldexp((double)x[d], 127 - (int)e));
            row[ORC_NOPE + 2 * ORC_ROPE + g] = (uint8_t)e;
        }
        for (d = ORC_NOPE; d < ORC_D; ++d) {
            uint16_t b = orc_bf16_bits((double)x[d]);
            row[ORC_NOPE + 2 * (d - ORC_NOPE)] = (uint8_t)(b & 0xFF);
            row[ORC_NOPE + 2 * (d - ORC_NOPE) + 1] = (uint8_t)(b >> 8);
        }
        row[ORC_NOPE + 2 * ORC_ROPE + 7] = 0;
        return 0;
    }
    return -2;
}

/* Dequantize one row to fp64 (exact: every product fits 8 significant bits). */
int orc_dequant_row(int layout, const uint8_t *row, double *out)
{
    int d;
    if (layout == ORC_V41) {
        for (d = 0; d < ORC_D; ++d) {
            unsigned e = row[ORC_D + d / 32];
            double scale = (e == 255u) ? NAN : ldexp(1.0, (int)e - 127);
            out[d] = orc_e4m3_value(row[d]) * scale;
        }
        return 0;
    }
    if (layout == ORC_V41_FP4) {
        for (d = 0; d < ORC_D; ++d) {
            unsigned nib = (row[d / 2] >> (4 * (d & 1))) & 15u;
            out[d] = orc_e2m1_value(nib) * orc_e4m3_value(row[ORC_D / 2 + d / 16]);
        }
        return 0;
    }
    if (layout == ORC_V4) {
        for (d = 0; d < ORC_NOPE; ++d) {
            unsigned e = row[ORC_NOPE + 2 * ORC_ROPE + d / 64];
            double scale = (e == 255u) ? NAN : ldexp(1.0, (int)e - 127);
            out[d] = orc_e4m3_value(row[d]) * scale;
        }
        for (d = ORC_NOPE; d < ORC_D; ++d)
            out[d] = orc_bf16_value((uint16_t)(row[ORC_NOPE + 2 * (d - ORC_NOPE)]
                                    | (row[ORC_NOPE + 2 * (d - ORC_NOPE) + 1] << 8)));
        return 0;
    }
    return -2;
}

/* ------------------------------------------------------------------------ */
/* PagedKV<layout, page_bits>::row [P4 Summary]: slot -> (page, in-page row) */
/* -> byte offset.  Pages are row_bytes << page_bits bytes, unpadded.        */
/* ------------------------------------------------------------------------ */
int64_t orc_row_offset(int layout, int page_bits, int64_t slot)
{
    int64_t rb = orc_row_bytes(layout);
    int64_t page = slot >> page_bits;
    int64_t off = slot & (((int64_t)1 << page_bits) - 1);
    return page * (rb << page_bits) + off * rb;
}

/* ------------------------------------------------------------------------ */
/* Write plan [P2 low_ratio_extend_offsets; P3 state = pos // ratio;        */
/* P4 c2 bullet: the ratio-2 decode compressor keeps a pair-state ring].    */
/* ext is int32 [2, n_slots]: ext[r] = first source row of request slot r,   */
/* ext[n_slots + r] = its count n_r of new tokens.  start_pos (NULL = all 0) */
/* gives the position p0 of the first new token; new token t (t < n_r) sits  */
/* at position p0 + t in source row first_r + t.                             */
/* Compressed row c pools the tokens at positions ratio*c .. ratio*c+ratio-1 */
/* and is produced by the step that holds its last token: ratio 1: c in      */
/* [p0, p0+n); ratio 2: c in [p0 >> 1, (p0 + n) >> 1) -- an odd trailing     */
/* token waits for the next step, and when p0 is odd the first pair's first  */
/* token (position p0 - 1) comes from the ring.  Output rows are numbered    */
/* request by request.  Per row k: req, j (= k - first row of the request),  */
/* c, pos = ratio*c, src = source row of the pair's first token (-1 when it  */
/* is in the ring), default slot page_table[r][c >> page_bits] << page_bits  */
/* | (c & mask) (-1 past the table).  Returns the total row count; fills the */
/* arrays for k < cap.                                                       */
/* ------------------------------------------------------------------------ */
int64_t orc_plan(int ratio, const int32_t *ext, int n_slots, const int32_t *start_pos,
                 const int32_t *page_table, int max_pages, int page_bits,
                 int64_t cap, int32_t *req, int32_t *jj, int64_t *cc, int64_t *src,
                 int64_t *pos, int64_t *slot)
{
    int64_t k = 0;
    int r;
    for (r = 0; r < n_slots; ++r) {
        int64_t n = ext[n_slots + r] > 0 ? ext[n_slots + r] : 0;
        int64_t p0 = start_pos ? start_pos[r] : 0;
        int64_t c_lo = ratio == 2 ? (p0 >> 1) : p0;
        int64_t c_hi = ratio == 2 ? ((p0 + n) >> 1) : p0 + n;
        int64_t c;
        if (n == 0) continue;
        for (c = c_lo; c < c_hi; ++c, ++k) {
            int64_t t0 = (int64_t)ratio * c;          /* position of the first token */
            if (k >= cap) continue;
            if (req) req[k] = r;
            if (jj) jj[k] = (int32_t)(c - c_lo);
            if (cc) cc[k] = c;
            if (src) src[k] = t0 >= p0 ? (int64_t)ext[r] + (t0 - p0) : -1;
            if (pos) pos[k] = t0;
            if (slot) {
                int64_t lp = c >> page_bits;
                slot[k] = (page_table && c >= 0 && lp < max_pages)
                    ? (((int64_t)page_table[(int64_t)r * max_pages + lp] << page_bits)
                       | (c & (((int64_t)1 << page_bits) - 1)))
                    : -1;
            }
        }
    }
    return k;
}

/* ------------------------------------------------------------------------ */
/* Fused compressor: pool -> RMSNorm -> RoPE -> store_row -> paged write     */
/* [P4 Summary, c1/c2 bullet; P2 fused | kv | score | projection].           */
/*                                                                           */
/* rows: bf16 bits, row k at rows + k*row_stride; kv in cols [0, 512).       */
/* score: bf16 bits [n_rows, score_stride], or NULL for the fused layout     */
/*        (score at rows + 512).  Unused for ratio 1.                        */
/* start_pos / ring: see orc_plan; ring is bf16 [n_slots, ring_size, 1024]   */
/*        (kv | score per entry), read for pairs whose first token is       */
/*        before the step and then updated (NULL: no ring; such a pair is a  */
/*        fault).                                                            */
/* norm_w: bf16 [512] or NULL (no RMSNorm).  freqs: fp32 [max_pos, 64]       */
/*        (cos, sin) per complex pair, or NULL (no RoPE).                    */
/* out_loc: int32 [n_out] slot per output row (0 = not stored), or NULL to   */
/*        use the plan's page-table slot.  Rows k >= total have no source.   */
/* which: NULL, or the output rows to compute (n_which of them, each in      */
/*        [0, n_out)); per-row outputs and prequant_in are then indexed by  */
/*        position in `which`.  Used to check sampled rows of large cases.  */
/* prequant_in: if non-NULL, the fp32 rows fed to the quantizer are these    */
/*        ("identical-input" mode) instead of this oracle's fp64 result      */
/*        rounded to fp32.                                                   */
/* Outputs (each nullable): pool bytes, prequant fp64/fp32 rows, bf16 latent */
/*        (post-norm, pre-RoPE).  Returns the total row count or < 0.        */
/* ------------------------------------------------------------------------ */
int64_t orc_compress_store(
    int layout, int ratio,
    const uint16_t *rows, int64_t n_rows, int64_t row_stride,
    const uint16_t *score, int64_t score_stride,
    const int32_t *ext, int n_slots, const int32_t *start_pos,
    uint16_t *ring, int ring_size,
    const int32_t *page_table, int max_pages, int page_bits,
    const uint16_t *norm_w, float eps,
    const float *freqs, int max_pos,
    const int32_t *out_loc, int64_t n_out,
    const int64_t *which, int64_t n_which,
    uint8_t *pool, int64_t pool_rows,
    const float *prequant_in,
    double *prequant_f64, float *prequant_f32, uint16_t *latent_out,
    int64_t *n_faults)
{
    int64_t total, k, o, faults = 0;
    int32_t *req, *jj;
    int64_t *src, *pslot, *pos, *cc;
    int rb = orc_row_bytes(layout);
    double x[ORC_D];
    float xf[ORC_D];
    uint8_t rowbuf[600];
    memset(rowbuf, 0, sizeof(rowbuf));

    if (ratio != 1 && ratio != 2) return -1;
    if (layout != ORC_V4 && layout != ORC_V41 && layout != ORC_V41_FP4) return -2;
    if (ring && (ratio != 2 || ring_size < 1)) return -1;
    for (o = 0; which && o < n_which; ++o)
        if (which[o] < 0 || which[o] >= n_out) return -1;
    total = orc_plan(ratio, ext, n_slots, start_pos, page_table, max_pages, page_bits,
                     0, NULL, NULL, NULL, NULL, NULL, NULL);
    req = (int32_t *)calloc((size_t)(total + 1), sizeof(int32_t));
    jj = (int32_t *)calloc((size_t)(total + 1), sizeof(int32_t));
    cc = (int64_t *)calloc((size_t)(total + 1), sizeof(int64_t));
    pos = (int64_t *)calloc((size_t)(total + 1), sizeof(int64_t));
    src = (int64_t *)calloc((size_t)(total + 1), sizeof(int64_t));
    pslot = (int64_t *)calloc((size_t)(total + 1), sizeof(int64_t));
    orc_plan(ratio, ext, n_slots, start_pos, page_table, max_pages, page_bits,
             total, req, jj, cc, src, pos, pslot);

    for (o = 0; o < (which ? n_which : n_out); ++o) {
        int d, t, bad = 0;
        int64_t slot;
        k = which ? which[o] : o;
        if (k >= total) { /* no source row: nothing computed or stored */
            if (prequant_f64) memset(prequant_f64 + o * ORC_D, 0, ORC_D * sizeof(double));
            if (prequant_f32) memset(prequant_f32 + o * ORC_D, 0, ORC_D * sizeof(float));
            if (latent_out) memset(latent_out + o * ORC_D, 0, ORC_D * sizeof(uint16_t));
            continue;
        }
        {   /* the pair's tokens: new rows, or (first token) the ring */
            int r = req[k];
            int64_t first_new = src[k] >= 0 ? src[k] : ext[r];    /* first new source row used */
            int64_t last_new = src[k] >= 0 ? src[k] + ratio - 1 : ext[r];
            if (first_new < 0 || last_new >= n_rows) bad = 1;
            if (src[k] < 0 && !ring) bad = 1;
        }
        if (pos[k] < 0) bad = 1;   /* no token precedes position 0 */
        if (freqs && pos[k] >= max_pos) bad = 1;
        slot = out_loc ? (int64_t)out_loc[k] : pslot[k];
        if (bad) { /* a row that cannot be computed: zero outputs, one fault */
            ++faults;
            if (prequant_f64) memset(prequant_f64 + o * ORC_D, 0, ORC_D * sizeof(double));
            if (prequant_f32) memset(prequant_f32 + o * ORC_D, 0, ORC_D * sizeof(float));
            if (latent_out) memset(latent_out + o * ORC_D, 0, ORC_D * sizeof(uint16_t));
            continue;
        }

        /* pool: ratio 1 passthrough; ratio 2 per-dim softmax of the pair's
         * scores weighting the pair's kv values */
        for (d = 0; d < ORC_D; ++d) {
            if (ratio == 1) {
                x[d] = orc_bf16_value(rows[src[k] * row_stride + d]);
            } else {
                double kv[2], sc[2], m, w[2], den = 0.0, num = 0.0;
                for (t = 0; t < 2; ++t) {
                    if (t == 0 && src[k] < 0) {   /* token pos[k] from the pair-state ring */
                        const uint16_t *e = ring + ((int64_t)req[k] * ring_size
                                                    + (cc[k] % ring_size)) * (2 * ORC_D);
                        kv[t] = orc_bf16_value(e[d]);
                        sc[t] = orc_bf16_value(e[ORC_D + d]);
                    } else {
                        int64_t rr = (src[k] >= 0 ? src[k] : ext[req[k]] - 1) + t;
                        kv[t] = orc_bf16_value(rows[rr * row_stride + d]);
                        sc[t] = score ? orc_bf16_value(score[rr * score_stride + d])
                                      : orc_bf16_value(rows[rr * row_stride + ORC_D + d]);
                    }
                }
                m = sc[0] > sc[1] ? sc[0] : sc[1];
                for (t = 0; t < 2; ++t) { w[t] = exp(sc[t] - m); den += w[t]; }
                for (t = 0; t < 2; ++t) num += (w[t] / den) * kv[t];
                x[d] = num;
            }
        }
        /* RMSNorm over all 512 dims: x / sqrt(mean(x^2) + eps) * w */
        if (norm_w) {
            double ss = 0.0, inv;
            for (d = 0; d < ORC_D; ++d) ss += x[d] * x[d];
            inv = 1.0 / sqrt(ss / ORC_D + (double)eps);
            for (d = 0; d < ORC_D; ++d) x[d] = x[d] * inv * orc_bf16_value(norm_w[d]);
        }
        if (latent_out)
            for (d = 0; d < ORC_D; ++d) latent_out[o * ORC_D + d] = orc_bf16_bits(x[d]);
        /* RoPE on the 64 rope dims, interleaved complex pairs
         * (448+2i, 449+2i) rotated by (cos, sin) = freqs[pos][2i], [2i+1] */
        if (freqs) {
            int i;
            for (i = 0; i < ORC_ROPE / 2; ++i) {
                double c = freqs[(int64_t)pos[k] * ORC_ROPE + 2 * i];
                double s = freqs[(int64_t)pos[k] * ORC_ROPE + 2 * i + 1];
                double a = x[ORC_NOPE + 2 * i], b = x[ORC_NOPE + 2 * i + 1];
                x[ORC_NOPE + 2 * i] = a * c - b * s;
                x[ORC_NOPE + 2 * i + 1] = a * s + b * c;
            }
        }
        for (d = 0; d < ORC_D; ++d) {
            xf[d] = prequant_in ? prequant_in[o * ORC_D + d] : (float)x[d];
            if (prequant_f64) prequant_f64[o * ORC_D + d] = x[d];
            if (prequant_f32) prequant_f32[o * ORC_D + d] = (float)x[d];
        }
        /* quantize and write; out_loc == 0 marks a row that is not stored;
         * a destination outside the pool (or past the page table) is one
         * fault, the row's other outputs stay written */
        if (slot == 0) continue;
        if (slot < 0 || slot >= pool_rows) { ++faults; continue; }
        orc_quantize_row(layout, xf, rowbuf);
        if (pool) memcpy(pool + orc_row_offset(layout, page_bits, slot), rowbuf, (size_t)rb);
    }
    /* the ring keeps each request's last ring_size even-position new tokens
     * (kv | score of position q at entry (q / 2) % ring_size), written after
     * every row of the step has read it; a token at a negative position has
     * no entry and, like a source row out of range, counts one fault */
    if (ring && !which) {
        int r;
        for (r = 0; r < n_slots; ++r) {
            int64_t n = ext[n_slots + r] > 0 ? ext[n_slots + r] : 0;
            int64_t p0 = start_pos ? start_pos[r] : 0;
            int64_t q = p0 + n - 2 * (int64_t)ring_size;
            if (q < p0) q = p0;
            for (; q < p0 + n; ++q) {
                int64_t row = (int64_t)ext[r] + (q - p0);
                uint16_t *e;
                int d;
                if (q & 1) continue;
                if (q < 0 || row < 0 || row >= n_rows) { ++faults; continue; }
                e = ring + ((int64_t)r * ring_size + ((q >> 1) % ring_size)) * (2 * ORC_D);
                for (d = 0; d < ORC_D; ++d) {
                    e[d] = rows[row * row_stride + d];
                    e[ORC_D + d] = score ? score[row * score_stride + d]
                                         : rows[row * row_stride + ORC_D + d];
                }
            }
        }
    }
    free(req); free(jj); free(pos); free(src); free(pslot); free(cc);
    if (n_faults) *n_faults = faults;
    return total;
}

/* ------------------------------------------------------------------------ */
/* Paged gather-dequant [P4 Summary, dequantize_k_cache_paged]:              */
/* out[i] = bf16(dequant(pool row ids[i])); ids[i] < 0 -> zero row;          */
/* ids[i] >= pool_rows -> zero row and one fault.  The pool is addressed as  */
/* a flat row array (pages are unpadded, so slot * row_bytes).               */
/* ------------------------------------------------------------------------ */
int64_t orc_dequant_gather(int layout, const uint8_t *pool, int64_t pool_rows,
                           const int32_t *ids, int64_t n, uint16_t *out)
{
    int64_t i, faults = 0;
    int rb = orc_row_bytes(layout);
    double v[ORC_D];
    if (layout != ORC_V4 && layout != ORC_V41 && layout != ORC_V41_FP4) return -2;
    for (i = 0; i < n; ++i) {
        int d;
        int64_t id = ids[i];
        if (id < 0 || id >= pool_rows) {
            if (id >= pool_rows) ++faults;
            memset(out + i * ORC_D, 0, ORC_D * sizeof(uint16_t));
            continue;
        }
        orc_dequant_row(layout, pool + id * rb, v);
        for (d = 0; d < ORC_D; ++d) out[i * ORC_D + d] = orc_bf16_bits(v[d]);
    }
    return faults;
}

/* ------------------------------------------------------------------------ */
/* Top-k compressed ids -> physical slots [P3 _compressed_topk_to_slots,    */
/* single-rank branch].  topk is int32 [n_tok, k], request-local compressed  */
/* ids (< 0 = empty).  slot = page_table[req][id >> page_bits] << page_bits   */
/* | (id & mask), or -1 for an empty entry, a page index past max_pages, or  */
/* an invalid token.  lens[t] = number of slots >= 0 in row t.               */
/* The slot is formed in 64-bit arithmetic.  A page entry < 0, or a slot     */
/* that int32 cannot hold, is not a page the pool has: slot -1 and one fault */
/* (the pages give physical page numbers only as non-negative int32 slots).  */
/* ------------------------------------------------------------------------ */
int64_t orc_topk_to_slots(const int32_t *topk, int64_t n_tok, int k,
                          const int32_t *token_to_req, const uint8_t *is_valid,
                          const int32_t *page_table, int n_req, int max_pages,
                          int page_bits, int32_t *slots, int32_t *lens)
{
    int64_t t, faults = 0;
    for (t = 0; t < n_tok; ++t) {
        int c, cnt = 0;
        int32_t r = token_to_req[t];
        int valid = is_valid ? (is_valid[t] != 0) : 1;
        if (r < 0 || r >= n_req) { valid = 0; ++faults; }
        for (c = 0; c < k; ++c) {
            int32_t id = topk[t * k + c];
            int32_t s = -1;
            if (valid && id >= 0) {
                int64_t lp = (int64_t)id >> page_bits;
                if (lp < max_pages) {
                    int64_t phys = page_table[(int64_t)r * max_pages + lp];
                    int64_t slot = phys * ((int64_t)1 << page_bits)
                                   + (id & ((1 << page_bits) - 1));
                    if (phys < 0 || slot > INT32_MAX)
                        ++faults;
                    else
                        s = (int32_t)slot;
                } else {
                    ++faults;
                }
            }
            slots[t * k + c] = s;
            if (s >= 0) ++cnt;
        }
        if (lens) lens[t] = cnt;
    }
    return faults;
}

/* ------------------------------------------------------------------------ */
/* Short-context ids [P4 test table: fill_all_compressed_indices; P3         */
/* "short-context bypass" of the indexer].  Every compressed row a token can  */
/* see is selected: out[t][j] = j for j < min(lens[t], k), -1 after; lens[t]  */
/* is the token's visible compressed length (a negative one counts as 0).    */
/* ------------------------------------------------------------------------ */
void orc_fill_all_indices(int64_t n_tok, int k, const int32_t *lens, int32_t *out)
{
    int64_t t;
    int j;
    for (t = 0; t < n_tok; ++t)
        for (j = 0; j < k; ++j)
            out[t * k + j] = j < lens[t] ? j : -1;
}

/* Vectorised helpers for the tests' exhaustive pins. */
void orc_ue8m0_many(const float *amax, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = (uint8_t)orc_ue8m0(amax[i]);
}

void orc_e4m3_encode_many(const double *x, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(x[i]);
}

void orc_e2m1_encode_many(const double *x, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(x[i]);
}

void orc_bf16_bits_many(const double *x, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_bf16_bits(x[i]);
}
