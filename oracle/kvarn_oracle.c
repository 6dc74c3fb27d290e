/*
 * kvarn_oracle.c -- plain, slow CPU oracle for the KVarN KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Arithmetic is IEEE fp64 throughout, written as the plain definition of
 * each step, with no blocking, fusion or reordering.  Every integer decision
 * (an FP8/FP16 scale code, a quantisation code) is taken on the fp64 value
 * of its definition; the fp64 pre-rounding value of each code is reported
 * beside it so that a comparison can tell a decision that sits on a rounding
 * boundary from a wrong one.
 *
 * Sources (pages on the subject; titles as published):
 *  [P1] "KVarN: 2-Bit KV-Cache That Beats FP16 Throughput, and Where the
 *       Catch Lives", section "What KVarN does differently": Hadamard
 *       rotation along the channel dimension; Sinkhorn-like alternation of
 *       column and row standard-deviation normalisation in log space.
 *  [P2] "Huawei's KVarN puts KV-cache quantization inside vLLM's backend",
 *       section "What KVarN changes in vLLM's serving path" (preset
 *       kvarn_k4v2_g128: 4-bit keys, 2-bit values per 128-token tile, dual
 *       FP8 scales and FP16 zero-points) and section "The four-stage
 *       pipeline" (rotation, variance normalisation, asymmetric
 *       round-to-nearest, dequantisation at read time).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - H is the Sylvester-ordered 128-point Hadamard matrix / sqrt(128), no
 *    random sign flips; R = X H acts on the channels of each token row.
 *  - "standard deviation" = mean-centred population std (divide by n);
 *    columns are normalised before rows in each of the N iterations; a
 *    row/column whose std is at most 1e-6 of its root-mean-square (or is all
 *    zero) keeps its factor.
 *  - after N iterations the column log-factors v are centred (geometric mean
 *    1) and exp(v) is stored as the per-channel FP8 E4M3 scale g (round to
 *    nearest even, saturating; a zero result becomes 2^-9); the row factors
 *    are discarded.
 *  - per token: Y = R / g, zero-point b = FP16 round-down of min_c Y,
 *    step a = E4M3 round-up of (max_c Y - b) / L (floor 2^-9), L = 2^bits - 1.
 *  - code = clamp(rne((Y - b) / a), 0, L), ties to even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define D 128 /* head_dim: channels per token */
#define T 128 /* tokens per tile (one paged block) */

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448, smallest 2^-9. */
double ora_e4m3_decode(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);           /* subnormal: m * 2^-9 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value, ties to the even code, saturating to +-448. */
uint8_t ora_e4m3_encode_rne(double x)
{
    uint8_t sign = 0, best = 0;
    double ax = x, bestd = INFINITY;
    if (isnan(x)) return 0x7F;
    if (x < 0) { sign = 0x80; ax = -x; }
    if (ax >= 448.0) return sign | 0x7E;
    for (int c = 0; c <= 0x7E; c++) {
        double d = fabs(ora_e4m3_decode((uint8_t)c) - ax);
        if (d < bestd || (d == bestd && (c & 1) == 0)) { bestd = d; best = (uint8_t)c; }
    }
    return sign | best;
}

/* Smallest non-negative E4M3 value >= x (x >= 0), saturating at 448. */
uint8_t ora_e4m3_encode_ru(double x)
{
    if (!(x > 0)) return 0;
    if (x >= 448.0) return 0x7E;
    uint8_t c = ora_e4m3_encode_rne(x);
    if (ora_e4m3_decode(c) < x) c++;                 /* next code is the next value up */
    return c;
}

/* IEEE binary16. */
double ora_f16_decode(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/* fp64 value that is exactly an fp16 number -> its bits. */
static uint16_t f16_bits_of_exact(double v)
{
    uint16_t s = 0;
    if (v < 0 || (v == 0 && signbit(v))) { s = 0x8000; v = -v; }
    if (v == 0) return s;
    if (v < ldexp(1.0, -14)) return s | (uint16_t)(v / ldexp(1.0, -24));
    int e;
    double f = frexp(v, &e);                          /* v = f * 2^e, f in [0.5,1) */
    int be = e - 1 + 15;
    uint16_t m = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return s | (uint16_t)(be << 10) | m;
}

/* Spacing of the fp16 grid at |x| (x finite, |x| <= 65504). */
static double f16_ulp(double ax)
{
    if (ax < ldexp(1.0, -14)) return ldexp(1.0, -24);
    int e;
    frexp(ax, &e);
    return ldexp(1.0, e - 1 - 10);
}

/* Largest fp16 value <= x ("round down"), saturating to +-65504. */
uint16_t ora_f16_encode_rd(double x)
{
    if (x >= 65504.0) return 0x7BFF;
    if (x <= -65504.0) return 0xFBFF;
    double q = f16_ulp(fabs(x));
    double v = floor(x / q) * q;                      /* exact: q is a power of two */
    if (v < -65504.0) v = -65504.0;
    return f16_bits_of_exact(v);
}

/* Nearest fp16 value, ties to even, saturating to +-65504. */
uint16_t ora_f16_encode_rne(double x)
{
    if (x >= 65504.0) return 0x7BFF;
    if (x <= -65504.0) return 0xFBFF;
    double q = f16_ulp(fabs(x));
    double v = rint(x / q) * q;                       /* rint: ties to even */
    if (v > 65504.0) v = 65504.0;
    if (v < -65504.0) v = -65504.0;
    return f16_bits_of_exact(v);
}

double ora_bf16_decode(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Rotation [P1 "What KVarN does differently"; P2 "The four-stage      */
/* pipeline", first stage]                                             */
/* ------------------------------------------------------------------ */

/* H[i][j] = (-1)^popcount(i & j) / sqrt(128): Sylvester order, symmetric,
 * orthonormal, so H is its own inverse. */
void ora_hadamard_matrix(double *H)
{
    double s = 1.0 / sqrt((double)D);
    for (int i = 0; i < D; i++)
        for (int j = 0; j < D; j++)
            H[i * D + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -s : s;
}

/* Y = X H for a [rows][128] matrix X (rotation of every token row over its
 * channels; the same call with a rotated input undoes it). */
static double H_table[D * D];
static pthread_once_t H_once = PTHREAD_ONCE_INIT;
static void H_init(void) { ora_hadamard_matrix(H_table); }

void ora_rotate(const double *X, int rows, double *Y)
{
    const double *H = H_table;
    pthread_once(&H_once, H_init);
    for (int t = 0; t < rows; t++)
        for (int c = 0; c < D; c++) {
            double acc = 0.0;
            for (int k = 0; k < D; k++) acc += X[t * D + k] * H[k * D + c];
            Y[t * D + c] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* Sinkhorn-like variance normalisation [P1 "What KVarN does           */
/* differently", second step; P2 "The four-stage pipeline", "Iterative */
/* variance normalization"]                                            */
/* ------------------------------------------------------------------ */

/* Population std of n values (two-pass, mean-centred) and their rms. */
static void std_rms(const double *z, int n, double *sd, double *rms)
{
    double mean = 0.0, ss = 0.0, sq = 0.0;
    for (int i = 0; i < n; i++) mean += z[i];
    mean /= n;
    for (int i = 0; i < n; i++) { ss += (z[i] - mean) * (z[i] - mean); sq += z[i] * z[i]; }
    *sd = sqrt(ss / n);
    *rms = sqrt(sq / n);
}

static int degenerate(double sd, double rms) { return !(sd > 1e-6 * rms); }

/* Log-space alternating normalisation of R [T][D].  u[t] (rows = tokens)
 * and v[c] (columns = channels) start at 0; each iteration divides every
 * column of Z = R * exp(-u_t - v_c) by its std (v_c += ln sd_c), then every
 * row (u_t += ln sd_t).  On return v is NOT yet centred. */
void ora_sinkhorn(const double *R, int iters, double *u, double *v)
{
    double z[T > D ? T : D], eu[T], ev[D], sd, rms;
    for (int t = 0; t < T; t++) u[t] = 0.0;
    for (int c = 0; c < D; c++) v[c] = 0.0;
    for (int it = 0; it < iters; it++) {
        /* column step: std over the tokens of each channel */
        for (int t = 0; t < T; t++) eu[t] = exp(-u[t]);
        for (int c = 0; c < D; c++) {
            double evc = exp(-v[c]);
            for (int t = 0; t < T; t++) z[t] = R[t * D + c] * eu[t] * evc;
            std_rms(z, T, &sd, &rms);
            if (!degenerate(sd, rms)) v[c] += log(sd);
        }
        /* row step: std over the channels of each token */
        for (int c = 0; c < D; c++) ev[c] = exp(-v[c]);
        for (int t = 0; t < T; t++) {
            for (int c = 0; c < D; c++) z[c] = R[t * D + c] * eu[t] * ev[c];
            std_rms(z, D, &sd, &rms);
            if (!degenerate(sd, rms)) u[t] += log(sd);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Quantisation of one tile [P2 "What KVarN changes in vLLM's serving  */
/* path" (K4/V2, dual FP8 scales, FP16 zero-points) and "The four-stage */
/* pipeline" (asymmetric round-to-nearest)]                            */
/* ------------------------------------------------------------------ */

#define ORA_FLAG_CLAMPED 1   /* some code was clamped (range saturated) */
#define ORA_FLAG_STEP_SAT 2  /* a per-token step saturated at 448 */

/* X: [T][D] input tile (token rows), exact values of the 16-bit inputs.
 * levels: L = 15 (keys) or 3 (values).  Outputs: g8[D] and a8[T] E4M3
 * codes, b16[T] FP16 bits, code[T][D] (token-major), and optionally the fp64
 * pre-rounding value (Y - b) / a of every code (pre[T][D]), the rotated tile
 * (Rout[T][D]) and the centred column log-factors (vout[D]).  Returns flags. */
int ora_quantize_tile_ex(const double *X, int levels, int iters, int rotate,
                         uint8_t *g8, uint8_t *a8, uint16_t *b16, uint8_t *code,
                         double *pre, double *Rout, double *vout);
void ora_dequantize_record_ex(int kind, const uint8_t *rec, int rotate, double *Xhat);

int ora_quantize_tile(const double *X, int levels, int iters,
                      uint8_t *g8, uint8_t *a8, uint16_t *b16, uint8_t *code,
                      double *pre, double *Rout, double *vout)
{
    return ora_quantize_tile_ex(X, levels, iters, 1, g8, a8, b16, code, pre, Rout, vout);
}

/* The same steps with the rotation optional: rotate = 0 quantises X itself
 * (R = X).  With iters = 0 as well the tile gets plain per-token asymmetric
 * round-to-nearest under unit channel scales.  These are the ablations of the
 * per-token error study ("Huawei's KVarN puts KV-cache quantization inside
 * vLLM's backend", section "Why KV-cache quantization degrades under
 * autoregressive decoding": the largest 5% of per-token errors drive the
 * accuracy loss; section "The four-stage pipeline": rotation and variance
 * normalisation are the stages that shrink them). */
int ora_quantize_tile_ex(const double *X, int levels, int iters, int rotate,
                         uint8_t *g8, uint8_t *a8, uint16_t *b16, uint8_t *code,
                         double *pre, double *Rout, double *vout)
{
    static __thread double R[T * D];
    double u[T], v[D], gval[D], mv = 0.0;
    int flags = 0;

    if (rotate)
        ora_rotate(X, T, R);
    else
        memcpy(R, X, sizeof(double) * T * D);
    ora_sinkhorn(R, iters, u, v);

    /* gauge: geometric mean of the column factors = 1 */
    for (int c = 0; c < D; c++) mv += v[c];
    mv /= D;
    for (int c = 0; c < D; c++) {
        v[c] -= mv;
        uint8_t gc = ora_e4m3_encode_rne(exp(v[c]));
        if (gc == 0) gc = 0x01;                       /* never a zero scale */
        g8[c] = gc;
        gval[c] = ora_e4m3_decode(gc);
        if (vout) vout[c] = v[c];
    }

    for (int t = 0; t < T; t++) {
        double y[D], ymin = INFINITY, ymax = -INFINITY;
        for (int c = 0; c < D; c++) {
            y[c] = R[t * D + c] / gval[c];
            if (y[c] < ymin) ymin = y[c];
            if (y[c] > ymax) ymax = y[c];
        }
        /* zero-point: the largest FP16 value <= min Y; step: the smallest
         * E4M3 value >= (max Y - b) / L, so that b .. b + L a covers the row */
        uint16_t bt = ora_f16_encode_rd(ymin);
        double bval = ora_f16_decode(bt);
        double step = (ymax - bval) / levels;
        uint8_t at = ora_e4m3_encode_ru(step);
        if (at == 0) at = 0x01;                       /* floor 2^-9 */
        if (at == 0x7E && ora_e4m3_decode(0x7E) < step) flags |= ORA_FLAG_STEP_SAT;
        double aval = ora_e4m3_decode(at);
        b16[t] = bt;
        a8[t] = at;
        for (int c = 0; c < D; c++) {
            double x = (y[c] - bval) / aval;          /* position on the level grid */
            double r = rint(x);                       /* nearest level, ties to even */
            int k = (int)r;
            if (r < 0) { k = 0; flags |= ORA_FLAG_CLAMPED; }
            if (r > levels) { k = levels; flags |= ORA_FLAG_CLAMPED; }
            code[t * D + c] = (uint8_t)k;
            if (pre) pre[t * D + c] = x;
        }
    }
    if (Rout) memcpy(Rout, R, sizeof(double) * T * D);
    return flags;
}

enum { ORA_K4 = 0, ORA_V2 = 1, ORA_K2 = 2, ORA_V4 = 3 };

/* ------------------------------------------------------------------ */
/* Packed record layout (16-byte aligned, scales first)                */
/*   K (levels 15): g[128] E4M3 | a[128] E4M3 | b[128] FP16 LE |        */
/*                  codes[128 tokens][64 B], byte i of token t =       */
/*                  code[t][2i] | code[t][2i+1] << 4          = 8704 B */
/*   K2 (levels 3, the K2/V2 preset): same header | codes[128 tok]    */
/*                  [32 B], byte i of token t = sum_k code[t][4i+k]<<2k */
/*                                                            = 4608 B */
/*   V (levels 3):  same header | codes[128 channels][32 B]: channel c */
/*                  = 8 little-endian 32-bit words, word w holds tokens */
/*                  16w..16w+15, token 16w+u at bit u (u even) or bit   */
/*                  15+u (u odd)                              = 4608 B */
/*   V4 (levels 15, the K4/V4 preset): same header | codes[128 ch]    */
/*                  [64 B]: channel c = 16 LE 32-bit words, word w    */
/*                  holds tokens 8w..8w+7, token 8w+u at bit 2u (u     */
/*                  even) or 14+2u (u odd)                    = 8704 B */
/* ------------------------------------------------------------------ */

/* bit of token u (0..15) inside its 32-bit V word */
static int ora_v_bit(int u) { return (u & 1) ? 15 + u : u; }
/* bit of token u (0..7) inside its 32-bit V4 word: even tokens in the low
 * half-word, odd tokens in the high half-word, 4 bits each */
static int ora_v4_bit(int u) { return (u & 1) ? 14 + 2 * u : 2 * u; }

/* record kinds: ORA_K4 (4-bit keys), ORA_V2 (2-bit values), ORA_K2 (2-bit
 * keys), ORA_V4 (4-bit values) */
int ora_record_bytes(int kind) { return 512 + ((kind == ORA_K4 || kind == ORA_V4) ? D * T / 2 : D * T / 4); }
int ora_kind_levels(int kind) { return (kind == ORA_K4 || kind == ORA_V4) ? 15 : 3; }

void ora_pack_record(int kind, const uint8_t *g8, const uint8_t *a8, const uint16_t *b16,
                     const uint8_t *code, uint8_t *rec)
{
    memcpy(rec, g8, D);
    memcpy(rec + 128, a8, T);
    for (int t = 0; t < T; t++) { rec[256 + 2 * t] = (uint8_t)(b16[t] & 0xFF); rec[257 + 2 * t] = (uint8_t)(b16[t] >> 8); }
    uint8_t *p = rec + 512;
    if (kind == ORA_K4) {
        for (int t = 0; t < T; t++)
            for (int i = 0; i < D / 2; i++)
                p[t * 64 + i] = (uint8_t)(code[t * D + 2 * i] | (code[t * D + 2 * i + 1] << 4));
    } else if (kind == ORA_K2) {
        for (int t = 0; t < T; t++)
            for (int i = 0; i < D / 4; i++) {
                uint8_t byte = 0;
                for (int k = 0; k < 4; k++) byte |= (uint8_t)(code[t * D + 4 * i + k] << (2 * k));
                p[t * 32 + i] = byte;
            }
    } else if (kind == ORA_V4) {
        for (int c = 0; c < D; c++)
            for (int w = 0; w < T / 8; w++) {
                uint32_t word = 0;
                for (int u = 0; u < 8; u++)
                    word |= (uint32_t)code[(8 * w + u) * D + c] << ora_v4_bit(u);
                for (int k = 0; k < 4; k++) p[c * 64 + 4 * w + k] = (uint8_t)(word >> (8 * k));
            }
    } else {
        for (int c = 0; c < D; c++)
            for (int w = 0; w < T / 16; w++) {
                uint32_t word = 0;
                for (int u = 0; u < 16; u++)
                    word |= (uint32_t)code[(16 * w + u) * D + c] << ora_v_bit(u);
                for (int k = 0; k < 4; k++) p[c * 32 + 4 * w + k] = (uint8_t)(word >> (8 * k));
            }
    }
}

void ora_unpack_record(int kind, const uint8_t *rec, uint8_t *g8, uint8_t *a8, uint16_t *b16,
                       uint8_t *code)
{
    memcpy(g8, rec, D);
    memcpy(a8, rec + 128, T);
    for (int t = 0; t < T; t++) b16[t] = (uint16_t)(rec[256 + 2 * t] | (rec[257 + 2 * t] << 8));
    const uint8_t *p = rec + 512;
    for (int t = 0; t < T; t++)
        for (int c = 0; c < D; c++)
            code[t * D + c] = kind == ORA_K4 ? (uint8_t)((p[t * 64 + c / 2] >> (4 * (c & 1))) & 15)
                            : kind == ORA_K2 ? (uint8_t)((p[t * 32 + c / 4] >> (2 * (c & 3))) & 3)
                            : kind == ORA_V4 ? (uint8_t)((p[c * 64 + 4 * (t / 8) + ora_v4_bit(t % 8) / 8]
                                                          >> (ora_v4_bit(t % 8) % 8)) & 15)
                                             : (uint8_t)((p[c * 32 + 4 * (t / 16) + ora_v_bit(t % 16) / 8]
                                                          >> (ora_v_bit(t % 16) % 8)) & 3);
}

/* Dequantise one record [P2 "The four-stage pipeline", fourth stage]:
 * Rhat[t][c] = g_c (a_t code_tc + b_t), Xhat = Rhat H (unrotated). */
void ora_dequantize_record(int kind, const uint8_t *rec, double *Xhat)
{
    ora_dequantize_record_ex(kind, rec, 1, Xhat);
}

/* Dequantise without the inverse rotation when rotate = 0 (records made by
 * ora_quantize_tile_ex with rotate = 0). */
void ora_dequantize_record_ex(int kind, const uint8_t *rec, int rotate, double *Xhat)
{
    static __thread double Rh[T * D];
    uint8_t g8[D], a8[T], code[T * D];
    uint16_t b16[T];
    ora_unpack_record(kind, rec, g8, a8, b16, code);
    for (int t = 0; t < T; t++)
        for (int c = 0; c < D; c++)
            Rh[t * D + c] = ora_e4m3_decode(g8[c]) *
                            (ora_e4m3_decode(a8[t]) * code[t * D + c] + ora_f16_decode(b16[t]));
    if (rotate)
        ora_rotate(Rh, T, Xhat);
    else
        memcpy(Xhat, Rh, sizeof(double) * T * D);
}

/* ------------------------------------------------------------------ */
/* Decode attention                                                    */
/* ------------------------------------------------------------------ */

/* Plain softmax attention of G queries q[G][D] over n keys/values
 * K[n][D], V[n][D]: s = scale <q, k>, p = softmax(s), out = sum p v.
 * n == 0 gives out = 0. */
void ora_attention(const double *q, int G, const double *K, const double *V, int n,
                   double scale, double *out)
{
    double *s = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    for (int g = 0; g < G; g++) {
        double m = -INFINITY, l = 0.0;
        for (int i = 0; i < n; i++) {
            double acc = 0.0;
            for (int d = 0; d < D; d++) acc += q[g * D + d] * K[i * D + d];
            s[i] = scale * acc;
            if (s[i] > m) m = s[i];
        }
        for (int d = 0; d < D; d++) out[g * D + d] = 0.0;
        for (int i = 0; i < n; i++) {
            double p = exp(s[i] - m);
            l += p;
            for (int d = 0; d < D; d++) out[g * D + d] += p * V[i * D + d];
        }
        if (n > 0)
            for (int d = 0; d < D; d++) out[g * D + d] /= l;
    }
    free(s);
}

/* The same attention over packed tiles plus a raw tail, computed the way the
 * pages describe reading the cache [P2 "The four-stage pipeline": scales are
 * applied at read time]: the key rotation and per-channel key scales are
 * folded into the query, per-token scale/zero into the scores, per-channel
 * value scales into the accumulator, and one inverse rotation is applied to
 * the output.  krec/vrec: n_tiles records each (keys of kind kkind, values
 * of kind vkind); ktail/vtail: [n_tail][D]. */
void ora_attention_folded(const double *q, int G, const uint8_t *const *krec,
                          const uint8_t *const *vrec, int n_tiles, const double *ktail,
                          const double *vtail, int n_tail, double scale, int kkind, int vkind, double *out)
{
    int n = n_tiles * T + n_tail;
    double *s = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    double *qr = (double *)malloc(sizeof(double) * D), *acc_rot = (double *)malloc(sizeof(double) * D),
           *acc_raw = (double *)malloc(sizeof(double) * D), *orot = (double *)malloc(sizeof(double) * D);
    uint8_t g8[D], a8[T], code[T * D];
    uint16_t b16[T];
    for (int g = 0; g < G; g++) {
        ora_rotate(q + g * D, 1, qr);                 /* q' = (q H) * scale */
        for (int d = 0; d < D; d++) qr[d] *= scale;
        double m = -INFINITY;
        for (int tile = 0; tile < n_tiles; tile++) {
            ora_unpack_record(kkind, krec[tile], g8, a8, b16, code);
            double qg[D], S = 0.0;
            for (int c = 0; c < D; c++) { qg[c] = qr[c] * ora_e4m3_decode(g8[c]); S += qg[c]; }
            for (int t = 0; t < T; t++) {
                double dot = 0.0;
                for (int c = 0; c < D; c++) dot += qg[c] * code[t * D + c];
                double st = ora_e4m3_decode(a8[t]) * dot + ora_f16_decode(b16[t]) * S;
                s[tile * T + t] = st;
                if (st > m) m = st;
            }
        }
        for (int i = 0; i < n_tail; i++) {
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += q[g * D + d] * ktail[i * D + d];
            s[n_tiles * T + i] = scale * dot;
            if (s[n_tiles * T + i] > m) m = s[n_tiles * T + i];
        }
        double l = 0.0;
        for (int d = 0; d < D; d++) { acc_rot[d] = 0.0; acc_raw[d] = 0.0; }
        for (int tile = 0; tile < n_tiles; tile++) {
            ora_unpack_record(vkind, vrec[tile], g8, a8, b16, code);
            double pb = 0.0, pacc[D];
            for (int c = 0; c < D; c++) pacc[c] = 0.0;
            for (int t = 0; t < T; t++) {
                double p = exp(s[tile * T + t] - m);
                l += p;
                pb += p * ora_f16_decode(b16[t]);
                double pa = p * ora_e4m3_decode(a8[t]);
                for (int c = 0; c < D; c++) pacc[c] += pa * code[t * D + c];
            }
            for (int c = 0; c < D; c++) acc_rot[c] += ora_e4m3_decode(g8[c]) * (pacc[c] + pb);
        }
        for (int i = 0; i < n_tail; i++) {
            double p = exp(s[n_tiles * T + i] - m);
            l += p;
            for (int d = 0; d < D; d++) acc_raw[d] += p * vtail[i * D + d];
        }
        ora_rotate(acc_rot, 1, orot);                 /* one inverse rotation */
        for (int d = 0; d < D; d++) out[g * D + d] = n > 0 ? (orot[d] + acc_raw[d]) / l : 0.0;
    }
    free(s); free(qr); free(acc_rot); free(acc_raw); free(orot);
}

/* ------------------------------------------------------------------ */
/* Batch drivers (host threads over independent units)                 */
/* ------------------------------------------------------------------ */

/* Quantise n tiles.  src: 16-bit values (dtype 0 = fp16, 1 = bf16); tile i's
 * token row r starts at element first[i] + r * row_stride, channels
 * contiguous.  levels/iters as above.  rec: n records of
 * ora_record_bytes(kind) bytes, quantised to ora_kind_levels(kind) levels.
 * flags: n ints (may be NULL). */
typedef struct {
    const uint16_t *src; int dtype; const int64_t *first; int64_t row_stride;
    int n, kind, iters, nthreads, tid; uint8_t *rec; int *flags;
} qjob;

static void *quantize_worker(void *arg)
{
    qjob *j = (qjob *)arg;
    int L = ora_kind_levels(j->kind), rb = ora_record_bytes(j->kind);
    double *X = (double *)malloc(sizeof(double) * T * D);
    uint8_t g8[D], a8[T], *code = (uint8_t *)malloc(T * D);
    uint16_t b16[T];
    for (int i = j->tid; i < j->n; i += j->nthreads) {
        for (int t = 0; t < T; t++)
            for (int c = 0; c < D; c++) {
                uint16_t h = j->src[j->first[i] + (int64_t)t * j->row_stride + c];
                X[t * D + c] = j->dtype ? ora_bf16_decode(h) : ora_f16_decode(h);
            }
        int f = ora_quantize_tile(X, L, j->iters, g8, a8, b16, code, NULL, NULL, NULL);
        ora_pack_record(j->kind, g8, a8, b16, code, j->rec + (int64_t)i * rb);
        if (j->flags) j->flags[i] = f;
    }
    free(X); free(code);
    return NULL;
}

void ora_quantize_batch(const uint16_t *src, int dtype, const int64_t *first, int64_t row_stride,
                        int n, int kind, int iters, uint8_t *rec, int *flags, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    pthread_t th[256];
    qjob jobs[256];
    if (nthreads > 256) nthreads = 256;
    for (int k = 0; k < nthreads; k++) {
        jobs[k] = (qjob){src, dtype, first, row_stride, n, kind, iters, nthreads, k, rec, flags};
        pthread_create(&th[k], NULL, quantize_worker, &jobs[k]);
    }
    for (int k = 0; k < nthreads; k++) pthread_join(th[k], NULL);
}

/* The same batch with every field of each tile returned unpacked, for
 * comparisons: tile i's g8[i][128], a8[i][128], b16[i][128] and codes
 * code[i][128][128] (token-major), and where the pointers are not NULL the
 * pre-rounding values pre[i][128][128] and the rotated tile R[i][128][128]. */
typedef struct {
    const uint16_t *src; int dtype; const int64_t *first; int64_t row_stride;
    int n, levels, iters, nthreads, tid;
    uint8_t *g8, *a8; uint16_t *b16; uint8_t *code; double *pre, *R; int *flags;
} fjob;

static void *fields_worker(void *arg)
{
    fjob *j = (fjob *)arg;
    double *X = (double *)malloc(sizeof(double) * T * D);
    for (int i = j->tid; i < j->n; i += j->nthreads) {
        for (int t = 0; t < T; t++)
            for (int c = 0; c < D; c++) {
                uint16_t h = j->src[j->first[i] + (int64_t)t * j->row_stride + c];
                X[t * D + c] = j->dtype ? ora_bf16_decode(h) : ora_f16_decode(h);
            }
        int64_t o = (int64_t)i * T * D;
        int f = ora_quantize_tile(X, j->levels, j->iters, j->g8 + (int64_t)i * D, j->a8 + (int64_t)i * T,
                                  j->b16 + (int64_t)i * T, j->code + o, j->pre ? j->pre + o : NULL,
                                  j->R ? j->R + o : NULL, NULL);
        if (j->flags) j->flags[i] = f;
    }
    free(X);
    return NULL;
}

void ora_quantize_batch_fields(const uint16_t *src, int dtype, const int64_t *first, int64_t row_stride, int n,
                               int levels, int iters, uint8_t *g8, uint8_t *a8, uint16_t *b16, uint8_t *code,
                               double *pre, double *R, int *flags, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    fjob jobs[256];
    for (int k = 0; k < nthreads; k++) {
        jobs[k] = (fjob){src, dtype, first, row_stride, n, levels, iters, nthreads, k, g8, a8, b16, code, pre, R,
                         flags};
        pthread_create(&th[k], NULL, fields_worker, &jobs[k]);
    }
    for (int k = 0; k < nthreads; k++) pthread_join(th[k], NULL);
}

/* Decode attention for many independent units (one sequence x KV head
 * each): unit u has G queries q[u][G][D], n_tiles[u] packed K/V records
 * (pointers krec[off[u] + i], vrec[off[u] + i]) and n_tail[u] raw tail
 * tokens at ktail/vtail + u*T*D.  Uses the folded form. */
typedef struct {
    const double *q; int G; const uint8_t *const *krec, *const *vrec; const int64_t *off;
    const int32_t *n_tiles; const double *ktail, *vtail; const int32_t *n_tail; double scale;
    int kkind, vkind, n_units, nthreads, tid; double *out;
} ajob;

static void *attention_worker(void *arg)
{
    ajob *j = (ajob *)arg;
    for (int u = j->tid; u < j->n_units; u += j->nthreads)
        ora_attention_folded(j->q + (int64_t)u * j->G * D, j->G, j->krec + j->off[u], j->vrec + j->off[u],
                             j->n_tiles[u], j->ktail + (int64_t)u * T * D, j->vtail + (int64_t)u * T * D,
                             j->n_tail[u], j->scale, j->kkind, j->vkind, j->out + (int64_t)u * j->G * D);
    return NULL;
}

void ora_attention_batch(const double *q, int G, const uint8_t *const *krec, const uint8_t *const *vrec,
                         const int64_t *off, const int32_t *n_tiles, const double *ktail,
                         const double *vtail, const int32_t *n_tail, double scale, int kkind, int vkind,
                         int n_units, double *out, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    ajob jobs[256];
    for (int k = 0; k < nthreads; k++) {
        jobs[k] = (ajob){q, G, krec, vrec, off, n_tiles, ktail, vtail, n_tail, scale, kkind, vkind, n_units,
                         nthreads, k, out};
        pthread_create(&th[k], NULL, attention_worker, &jobs[k]);
    }
    for (int k = 0; k < nthreads; k++) pthread_join(th[k], NULL);
}
