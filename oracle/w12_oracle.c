/*
 * w12_oracle.c -- plain, slow, scalar CPU oracle for the lossless W12 weight
 * format and for the skinny GEMM that reads it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; it includes nothing but the C standard library.
 *
 * Sources (the three pages about "SpecPilot: Autonomous Algorithm Discovery and
 * Systems Optimization for Speculative Decoding"):
 *   [F5a]  thelatestinai.com listing page, Figure 5(a) caption: every BF16
 *          weight becomes three 4-bit planes -- A = sign + top three mantissa
 *          bits, E = 4-bit exponent offset inside a 16-binade window per output
 *          channel, B = the low mantissa bits; A and E form the 8-bit view the
 *          Q pass reads; weights outside the window go to an exact escape list.
 *   [F7]   same page, Figure 7 caption: the Q pass reads the 8-bit view nested
 *          in each W12 record.
 *   [MF]   ai.info "AI summary" page, Main Findings, "W12 compression" and
 *          "W12 works beyond speculation": lossless, 12.01-12.02 bits/weight,
 *          escape fraction 7.3e-5.
 *   [KC3]  ai.info page, Key Contributions item 3: the Q pass is zero-copy.
 *
 * Readings of what the pages leave open:
 *   R1 window anchor: a channel's window is the 16 binades ending at the
 *      largest finite normal exponent of that channel (row n of W[N][K]);
 *      ebase = max(emax, 16) - 15, so ebase is in [1, 239];
 *   R2 E is counted from the bottom of the window (E = e - ebase);
 *   R3 zeros, subnormals, Inf, NaN and values below the window are escapes;
 *   R4 an escaped slot holds the placeholder A = s<<3, E = 0, B = 0;
 *   R5 record bit order: record12 = A<<8 | E<<4 | B, AE byte = A<<4 | E (the
 *      record's top byte), one AE byte per weight, row-major [N][K];
 *   R6 B plane: per row, one little-endian 32-bit word per group of 8 weights;
 *      nibble slot j (bits 4j..4j+3) holds B of weight 8g+2j for j < 4 and of
 *      weight 8g+2(j-4)+1 for j >= 4; slots past K hold 0;
 *   R7 escape list: tiles of 128 rows x 256 columns, tile t = (n/128)*ceil(K/256)
 *      + k/256; entry = (n%128)<<24 | (k%256)<<16 | bf16 bits, ascending within
 *      a tile; tile_ptr[T+1] is the exclusive prefix count;
 *   R8 blob: "W12\0", u32 version 1, u64 N, K, n_esc, T, then ebase[N], AE,
 *      B, tile_ptr, escapes; all integers little-endian;
 *   R9 Q8 view: the weight rebuilt from A and E alone, B taken as 0, no escape
 *      patch (zero-copy reading of the A+E byte, [KC3], [F7]);
 *   R10 GEMM reference: y[m][n] = sum_k x[m][k] * W[n][k] in double precision,
 *      summed in increasing k.
 *
 * Epilogues of the projections of a decode step (the pages time the
 * projections of a dense layer -- q, k, v, o, gate, up, down -- and leave the
 * work beside each GEMM open; these are the plainest readings):
 *   R11 BF16 output: an FP32 result rounded to the nearest BF16, ties to the
 *      even significand, values at or beyond the largest finite BF16 plus half
 *      an ulp to infinity (IEEE 754 round-to-nearest-even);
 *   R12 gated MLP: with the gate and up rows interleaved (row 2i = gate row i,
 *      row 2i+1 = up row i), h[m][i] = silu(y[m][2i]) * y[m][2i+1], where
 *      silu(g) = g / (1 + exp(-g)).
 *
 * Encoder option (the pages fix the max-anchored window, R1; this variant
 * trades the top outliers of heavy-tailed rows for fewer escapes):
 *   R13 count-maximising window: a row's window base is the b in [1, b1]
 *      (b1 = the R1 base) whose 16 binades [b, b+15] hold the most finite
 *      normal weights of the row, the largest such b on ties; weights above
 *      the window then escape too, and their slot holds the saturated
 *      placeholder A = s<<3 | 7, E = 15, B = 15 -- the window's largest
 *      magnitude with the weight's sign -- so that the 8-bit view reads them
 *      as the nearest value it can hold.  Decoding is unchanged.
 *
 * A separate low-bit copy for the Q pass (the pages keep an INT6/INT8 copy on
 * the smaller GPU, RTX PRO 6000 section; the plainest INT8 reading):
 *   R14 INT8 copy: per row n, scale[n] = amax / 127 in FP32, amax the largest
 *      |w| over the row's finite weights; q[n][k] = rint(w / scale[n]) in FP32
 *      (round half to even), clamped to [-127, 127]; Inf goes to +-127, NaN to
 *      0, and a row whose scale is 0 has q = 0.  The Q-pass product is
 *      y[m][n] = scale[n] * sum_k x[m][k] q[n][k].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_TILE_ROWS 128
#define ORC_TILE_COLS 256
#define ORC_HEADER_BYTES 40

/* ---- little helpers: plain byte-wise little-endian IO ------------------- */

static void put_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v);
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

static void put_u64(uint8_t *p, uint64_t v)
{
    int i;
    for (i = 0; i < 8; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}

static uint32_t get_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

static uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    int i;
    for (i = 0; i < 8; i++)
        v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* ---- the fields of one BF16 weight ------------------------------------- */

static int bf16_sign(uint16_t b) { return (b >> 15) & 1; }
static int bf16_exp(uint16_t b) { return (b >> 7) & 0xFF; }
static int bf16_mant(uint16_t b) { return b & 0x7F; }

/* A "finite normal" exponent is 1..254 (0 = zero/subnormal, 255 = Inf/NaN). */
static int is_finite_normal(uint16_t b)
{
    int e = bf16_exp(b);
    return e >= 1 && e <= 254;
}

int64_t orc_tile_rows(void) { return ORC_TILE_ROWS; }
int64_t orc_tile_cols(void) { return ORC_TILE_COLS; }

/* R6: bytes of one row of the B plane. */
int64_t orc_b_row_bytes(int64_t K)
{
    return 4 * ((K + 7) / 8);
}

/* R7: number of escape tiles. */
int64_t orc_num_tiles(int64_t N, int64_t K)
{
    int64_t tr = (N + ORC_TILE_ROWS - 1) / ORC_TILE_ROWS;
    int64_t tc = (K + ORC_TILE_COLS - 1) / ORC_TILE_COLS;
    return tr * tc;
}

/* R1: the window base of one row [F5a]. */
int orc_row_ebase(const uint16_t *row, int64_t K)
{
    int emax = 0;
    int64_t k;
    for (k = 0; k < K; k++) {
        if (is_finite_normal(row[k]) && bf16_exp(row[k]) > emax)
            emax = bf16_exp(row[k]);
    }
    if (emax < 16)
        emax = 16; /* also covers a row with no finite normal weight at all */
    return emax - 15;
}

/* R13: the count-maximising window base of one row. */
int orc_row_ebase_count_max(const uint16_t *row, int64_t K)
{
    int64_t count[256];
    int64_t best = -1, c;
    int b, e, best_b = 1, b1 = orc_row_ebase(row, K);
    int64_t k;
    for (e = 0; e < 256; e++)
        count[e] = 0;
    for (k = 0; k < K; k++)
        if (is_finite_normal(row[k]))
            count[bf16_exp(row[k])]++;
    for (b = 1; b <= b1; b++) {
        c = 0;
        for (e = b; e <= b + 15; e++)
            c += count[e];
        if (c >= best) { /* ">=": the largest base among equal counts */
            best = c;
            best_b = b;
        }
    }
    return best_b;
}

/* Window base of a row under the chosen rule (0: R1, 1: R13). */
static int row_base(const uint16_t *row, int64_t K, int count_max)
{
    return count_max ? orc_row_ebase_count_max(row, K) : orc_row_ebase(row, K);
}

/* R13: a finite normal weight above the window (never under R1). */
static int above_window(uint16_t b, int ebase)
{
    return is_finite_normal(b) && bf16_exp(b) > ebase + 15;
}

/* R1 + R3: does weight `b` of a row with window base `ebase` fit the window? */
static int in_window(uint16_t b, int ebase)
{
    int e = bf16_exp(b);
    return is_finite_normal(b) && e >= ebase && e <= ebase + 15;
}

/* The three 4-bit fields of one record [F5a], with R2 and R4. */
static int field_A(uint16_t b, int ebase)
{
    if (in_window(b, ebase))
        return (bf16_sign(b) << 3) | (bf16_mant(b) >> 4);
    if (above_window(b, ebase))
        return (bf16_sign(b) << 3) | 7; /* R13 saturated placeholder */
    return bf16_sign(b) << 3; /* R4 placeholder */
}

static int field_E(uint16_t b, int ebase)
{
    if (in_window(b, ebase))
        return bf16_exp(b) - ebase;
    if (above_window(b, ebase))
        return 15;
    return 0;
}

static int field_B(uint16_t b, int ebase)
{
    if (in_window(b, ebase))
        return bf16_mant(b) & 0xF;
    if (above_window(b, ebase))
        return 15;
    return 0;
}

/* R6: nibble slot that holds weight k8 (0..7) of its group of eight. */
static int b_slot_of(int k8)
{
    if (k8 % 2 == 0)
        return k8 / 2;         /* evens in slots 0..3 */
    return 4 + (k8 - 1) / 2;   /* odds in slots 4..7 */
}

static int64_t count_escapes(const uint16_t *w, int64_t N, int64_t K, int count_max)
{
    int64_t n, k, count = 0;
    for (n = 0; n < N; n++) {
        int ebase = row_base(w + n * K, K, count_max);
        for (k = 0; k < K; k++)
            if (!in_window(w[n * K + k], ebase))
                count++;
    }
    return count;
}

static int64_t encoded_size(const uint16_t *w, int64_t N, int64_t K, int count_max)
{
    int64_t T = orc_num_tiles(N, K);
    return ORC_HEADER_BYTES + N + N * K + N * orc_b_row_bytes(K) + 4 * (T + 1) +
           4 * count_escapes(w, N, K, count_max);
}

/* Size in bytes of the blob that orc_encode writes for this matrix. */
int64_t orc_encoded_size(const uint16_t *w, int64_t N, int64_t K)
{
    return encoded_size(w, N, K, 0);
}

/* The same for orc_encode_count_max. */
int64_t orc_encoded_size_count_max(const uint16_t *w, int64_t N, int64_t K)
{
    return encoded_size(w, N, K, 1);
}

/*
 * Encode W[N][K] (BF16 bit patterns, row-major) into a W12 blob (R8), with
 * the R1 window (count_max = 0) or the R13 one.  Returns the blob length, or
 * -1 if `cap` is too small / arguments are bad.
 */
static int64_t encode_with(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, int64_t cap,
                           int count_max)
{
    int64_t T, tiles_c, n_esc, len, n, k, t;
    int64_t off_ebase, off_ae, off_b, off_ptr, off_esc, brow;
    int *ebase;

    if (N < 0 || K < 0)
        return -1;
    len = encoded_size(w, N, K, count_max);
    if (len > cap)
        return -1;
    T = orc_num_tiles(N, K);
    tiles_c = (K + ORC_TILE_COLS - 1) / ORC_TILE_COLS;
    n_esc = count_escapes(w, N, K, count_max);
    brow = orc_b_row_bytes(K);

    off_ebase = ORC_HEADER_BYTES;
    off_ae = off_ebase + N;
    off_b = off_ae + N * K;
    off_ptr = off_b + N * brow;
    off_esc = off_ptr + 4 * (T + 1);

    memset(blob, 0, (size_t)len);
    memcpy(blob, "W12", 4); /* "W12\0" */
    put_u32(blob + 4, 1);
    put_u64(blob + 8, (uint64_t)N);
    put_u64(blob + 16, (uint64_t)K);
    put_u64(blob + 24, (uint64_t)n_esc);
    put_u64(blob + 32, (uint64_t)T);

    ebase = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    if (!ebase)
        return -1;

    /* per-channel window base (R1) */
    for (n = 0; n < N; n++) {
        ebase[n] = row_base(w + n * K, K, count_max);
        blob[off_ebase + n] = (uint8_t)ebase[n];
    }

    /* AE plane (R5) and B plane (R6), one weight at a time */
    for (n = 0; n < N; n++) {
        for (k = 0; k < K; k++) {
            uint16_t b = w[n * K + k];
            int A = field_A(b, ebase[n]);
            int E = field_E(b, ebase[n]);
            int B = field_B(b, ebase[n]);
            int64_t word_at = off_b + n * brow + 4 * (k / 8);
            uint32_t word = get_u32(blob + word_at);
            blob[off_ae + n * K + k] = (uint8_t)((A << 4) | E);
            word |= (uint32_t)B << (4 * b_slot_of((int)(k % 8)));
            put_u32(blob + word_at, word);
        }
    }

    /* escape list (R7): visit tiles in order, and inside a tile rows then
     * columns in increasing order, so each tile's entries come out sorted. */
    {
        int64_t written = 0;
        put_u32(blob + off_ptr, 0);
        for (t = 0; t < T; t++) {
            int64_t tr = t / tiles_c, tc = t % tiles_c;
            int64_t n0 = tr * ORC_TILE_ROWS, k0 = tc * ORC_TILE_COLS;
            for (n = n0; n < N && n < n0 + ORC_TILE_ROWS; n++) {
                for (k = k0; k < K && k < k0 + ORC_TILE_COLS; k++) {
                    uint16_t b = w[n * K + k];
                    if (!in_window(b, ebase[n])) {
                        uint32_t entry = ((uint32_t)(n - n0) << 24) |
                                         ((uint32_t)(k - k0) << 16) | b;
                        put_u32(blob + off_esc + 4 * written, entry);
                        written++;
                    }
                }
            }
            put_u32(blob + off_ptr + 4 * (t + 1), (uint32_t)written);
        }
    }
    free(ebase);
    return len;
}

int64_t orc_encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, int64_t cap)
{
    return encode_with(w, N, K, blob, cap, 0);
}

/* R13: the same blob layout with the count-maximising window. */
int64_t orc_encode_count_max(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, int64_t cap)
{
    return encode_with(w, N, K, blob, cap, 1);
}

/* Read the header: out[0..3] = N, K, n_esc, T.  Returns 0, or -1 if malformed. */
int orc_blob_header(const uint8_t *blob, int64_t len, int64_t *out)
{
    int64_t N, K, n_esc, T, want;
    if (len < ORC_HEADER_BYTES)
        return -1;
    if (memcmp(blob, "W12", 4) != 0 || get_u32(blob + 4) != 1)
        return -1;
    N = (int64_t)get_u64(blob + 8);
    K = (int64_t)get_u64(blob + 16);
    n_esc = (int64_t)get_u64(blob + 24);
    T = (int64_t)get_u64(blob + 32);
    if (N < 0 || K < 0 || T != orc_num_tiles(N, K))
        return -1;
    want = ORC_HEADER_BYTES + N + N * K + N * orc_b_row_bytes(K) + 4 * (T + 1) + 4 * n_esc;
    if (want != len)
        return -1;
    out[0] = N;
    out[1] = K;
    out[2] = n_esc;
    out[3] = T;
    return 0;
}

/*
 * Rebuild rows [n0, n1) of W from a blob.  with_b = 1: the lossless decode
 * (all three planes, then every escape written back).  with_b = 0: the Q8
 * view (R9): A and E only, no escape patch.  out holds (n1-n0) rows of K.
 */
static int decode_rows(const uint8_t *blob, int64_t len, int64_t n0, int64_t n1,
                       int with_b, uint16_t *out)
{
    int64_t hdr[4], N, K, T, brow, tiles_c, n, k, t;
    int64_t off_ebase, off_ae, off_b, off_ptr, off_esc;
    if (orc_blob_header(blob, len, hdr) != 0)
        return -1;
    N = hdr[0];
    K = hdr[1];
    T = hdr[3];
    if (n0 < 0 || n1 > N || n0 > n1)
        return -1;
    brow = orc_b_row_bytes(K);
    tiles_c = (K + ORC_TILE_COLS - 1) / ORC_TILE_COLS;
    off_ebase = ORC_HEADER_BYTES;
    off_ae = off_ebase + N;
    off_b = off_ae + N * K;
    off_ptr = off_b + N * brow;
    off_esc = off_ptr + 4 * (T + 1);

    for (n = n0; n < n1; n++) {
        int ebase = blob[off_ebase + n];
        for (k = 0; k < K; k++) {
            int ae = blob[off_ae + n * K + k];
            int A = ae >> 4, E = ae & 0xF, B = 0;
            uint32_t word;
            if (with_b) {
                word = get_u32(blob + off_b + n * brow + 4 * (k / 8));
                B = (int)((word >> (4 * b_slot_of((int)(k % 8)))) & 0xF);
            }
            /* sign | exponent | top three mantissa bits | low four */
            out[(n - n0) * K + k] = (uint16_t)(((A >> 3) << 15) | ((ebase + E) << 7) |
                                               ((A & 7) << 4) | B);
        }
    }
    if (!with_b)
        return 0;
    for (t = 0; t < T; t++) {
        int64_t tr = t / tiles_c, tc = t % tiles_c, i;
        uint32_t p0 = get_u32(blob + off_ptr + 4 * t);
        uint32_t p1 = get_u32(blob + off_ptr + 4 * (t + 1));
        for (i = p0; i < (int64_t)p1; i++) {
            uint32_t entry = get_u32(blob + off_esc + 4 * i);
            int64_t row = tr * ORC_TILE_ROWS + (entry >> 24);
            int64_t col = tc * ORC_TILE_COLS + ((entry >> 16) & 0xFF);
            if (row >= n0 && row < n1 && col < K)
                out[(row - n0) * K + col] = (uint16_t)(entry & 0xFFFF);
        }
    }
    return 0;
}

/* Lossless decode of the whole matrix [F5a], [MF]. */
int orc_decode(const uint8_t *blob, int64_t len, uint16_t *w_out)
{
    int64_t hdr[4];
    if (orc_blob_header(blob, len, hdr) != 0)
        return -1;
    return decode_rows(blob, len, 0, hdr[0], 1, w_out);
}

int orc_decode_rows(const uint8_t *blob, int64_t len, int64_t n0, int64_t n1, uint16_t *w_out)
{
    return decode_rows(blob, len, n0, n1, 1, w_out);
}

/* The 8-bit view the Q pass reads, rebuilt as BF16 [F5a], [F7], R9. */
int orc_decode_q8(const uint8_t *blob, int64_t len, uint16_t *w_out)
{
    int64_t hdr[4];
    if (orc_blob_header(blob, len, hdr) != 0)
        return -1;
    return decode_rows(blob, len, 0, hdr[0], 0, w_out);
}

/* ---- GEMM reference (R10) ----------------------------------------------- */

static double bf16_value(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * y[m][n] = sum_k x[m][k] * w[n][k] for rows n in [n0, n1); y is [M][N].
 * x is [M][K] BF16, w is [N][K] BF16 (already decoded).
 */
void orc_gemm_rows(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K,
                   int64_t n0, int64_t n1, double *y)
{
    int64_t m, n, k;
    for (m = 0; m < M; m++) {
        for (n = n0; n < n1; n++) {
            double acc = 0.0;
            for (k = 0; k < K; k++)
                acc += bf16_value(x[m * K + k]) * bf16_value(w[n * K + k]);
            y[m * N + n] = acc;
        }
    }
}

void orc_gemm(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, double *y)
{
    orc_gemm_rows(x, w, M, N, K, 0, N, y);
}

/* s[m][n] = sum_k |x[m][k] * w[n][k]|: the scale of the acceptance bound. */
void orc_abs_gemm(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K,
                  double *s)
{
    int64_t m, n, k;
    for (m = 0; m < M; m++) {
        for (n = 0; n < N; n++) {
            double acc = 0.0;
            for (k = 0; k < K; k++) {
                double p = bf16_value(x[m * K + k]) * bf16_value(w[n * K + k]);
                acc += p < 0 ? -p : p;
            }
            s[m * N + n] = acc;
        }
    }
}

/* ---- epilogues (R11, R12) ----------------------------------------------- */

static double f32_bits_value(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * R11: the BF16 nearest to v.  The two candidates are v's bit pattern cut to
 * 16 bits (toward zero) and the next BF16 away from zero; whichever is nearer
 * wins, and a tie goes to the one whose last significand bit is 0.  Past the
 * largest finite BF16 the next value away from zero is infinity, which counts
 * as 2^128 in the comparison (the unbounded-exponent rounding of IEEE 754).
 * A NaN gives a quiet NaN of the same sign.
 */
static uint16_t round_bf16_one(float v)
{
    uint32_t u, lo, hi;
    double a, dlo, dhi;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    lo = u & 0xFFFF0000u;
    if (lo == u)
        return (uint16_t)(u >> 16);
    hi = lo + 0x10000u;
    a = fabs((double)v);
    dlo = a - fabs(f32_bits_value(lo));
    dhi = ((hi & 0x7F800000u) == 0x7F800000u ? ldexp(1.0, 128) : fabs(f32_bits_value(hi))) - a;
    if (dlo < dhi)
        return (uint16_t)(lo >> 16);
    if (dhi < dlo)
        return (uint16_t)(hi >> 16);
    return (uint16_t)(((lo >> 16) & 1u) ? (hi >> 16) : (lo >> 16));
}

void orc_round_bf16(const float *v, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = round_bf16_one(v[i]);
}

/* R12: h[m][i] = silu(y[m][2i]) * y[m][2i+1] for y [M][N], N even; h [M][N/2]. */
void orc_silu_mul(const double *y, int64_t M, int64_t N, double *h)
{
    int64_t m, i;
    for (m = 0; m < M; m++) {
        for (i = 0; i < N / 2; i++) {
            double g = y[m * N + 2 * i], u = y[m * N + 2 * i + 1];
            h[m * (N / 2) + i] = g / (1.0 + exp(-g)) * u;
        }
    }
}

/* ---- INT8 copy for the Q pass (R14) ------------------------------------- */

static float bf16_float(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

void orc_i8_quantize(const uint16_t *w, int64_t N, int64_t K, int8_t *q, float *scale)
{
    int64_t n, k;
    for (n = 0; n < N; n++) {
        float amax = 0.0f, sc;
        for (k = 0; k < K; k++) {
            float v = bf16_float(w[n * K + k]);
            if (isfinite(v) && fabsf(v) > amax)
                amax = fabsf(v);
        }
        sc = amax / 127.0f;
        scale[n] = sc;
        for (k = 0; k < K; k++) {
            float v = bf16_float(w[n * K + k]), t;
            if (sc == 0.0f || isnan(v)) {
                q[n * K + k] = 0;
                continue;
            }
            t = rintf(v / sc);
            if (t > 127.0f)
                t = 127.0f;
            if (t < -127.0f)
                t = -127.0f;
            q[n * K + k] = (int8_t)t;
        }
    }
}

/* y[m][n] = sum_k x[m][k] * (q[n][k] * scale[n]) in double, k ascending. */
void orc_gemm_i8(const uint16_t *x, const int8_t *q, const float *scale, int64_t M, int64_t N, int64_t K,
                 double *y)
{
    int64_t m, n, k;
    for (m = 0; m < M; m++) {
        for (n = 0; n < N; n++) {
            double acc = 0.0;
            for (k = 0; k < K; k++)
                acc += bf16_value(x[m * K + k]) * ((double)q[n * K + k] * (double)scale[n]);
            y[m * N + n] = acc;
        }
    }
}

/* s[m][n] = sum_k |x[m][k] * q[n][k] * scale[n]|: the scale of the bound. */
void orc_abs_gemm_i8(const uint16_t *x, const int8_t *q, const float *scale, int64_t M, int64_t N, int64_t K,
                     double *s)
{
    int64_t m, n, k;
    for (m = 0; m < M; m++) {
        for (n = 0; n < N; n++) {
            double acc = 0.0;
            for (k = 0; k < K; k++)
                acc += fabs(bf16_value(x[m * K + k]) * ((double)q[n * K + k] * (double)scale[n]));
            s[m * N + n] = acc;
        }
    }
}
