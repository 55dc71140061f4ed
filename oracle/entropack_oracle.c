/*
 * Plain CPU oracle of the EntroPack codec (test infrastructure only; see
 * entropack_oracle.h for the passages followed and the pins).  Written for
 * clarity: scalar loops, fp64 where the format says fp64, no blocking and
 * no threads.  Build with -ffp-contract=off so that no expression is fused.
 */
#include "entropack_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { O_OK = 0, O_ERR_ARG = 1, O_ERR_SHAPE = 2, O_ERR_NONFINITE = 3, O_ERR_CORRUPT = 4, O_ERR_UNSUPPORTED = 5,
       O_ERR_NOMEM = 6 };
enum { O_C_BF16 = 0, O_C_FP16 = 1, O_C_FP8 = 2, O_C_INT8 = 3, O_C_FP32 = 4 };

/* ---------------------------------------------- lossless element split (§5)
   BF16 / FP16: coded byte = bits 14..7, raw byte = bit 15 | bits 6..0
   FP8 e4m3:    coded byte = the element, no raw byte
   FP32:        coded byte = bits 30..23 (the exponent), raw bytes =
                (bit 31 | bits 22..16), bits 15..8, bits 7..0 */
static int lossless_dtype_ok(int c) { return c == O_C_BF16 || c == O_C_FP16 || c == O_C_FP8 || c == O_C_FP32; }
static int elem_bytes(int c) { return c == O_C_FP8 ? 1 : (c == O_C_FP32 ? 4 : 2); }
static int raw_per_elem(int c) { return c == O_C_FP8 ? 0 : (c == O_C_FP32 ? 3 : 1); }

static uint8_t split_elem(int c, const uint8_t *x, uint8_t *raw) {
    if (c == O_C_FP8) return x[0];
    if (c == O_C_FP32) {
        uint32_t v = (uint32_t)x[0] | ((uint32_t)x[1] << 8) | ((uint32_t)x[2] << 16) | ((uint32_t)x[3] << 24);
        raw[0] = (uint8_t)(((v >> 24) & 0x80) | ((v >> 16) & 0x7F));
        raw[1] = (uint8_t)(v >> 8);
        raw[2] = (uint8_t)v;
        return (uint8_t)(v >> 23);
    }
    uint16_t v = (uint16_t)(x[0] | (x[1] << 8));
    raw[0] = (uint8_t)(((v >> 8) & 0x80) | (v & 0x7F));
    return (uint8_t)(v >> 7);
}

static void join_elem(int c, uint8_t e, const uint8_t *raw, uint8_t *x) {
    if (c == O_C_FP8) { x[0] = e; return; }
    if (c == O_C_FP32) {
        uint32_t v = ((uint32_t)(raw[0] & 0x80) << 24) | ((uint32_t)e << 23) | ((uint32_t)(raw[0] & 0x7F) << 16) |
                     ((uint32_t)raw[1] << 8) | raw[2];
        for (int i = 0; i < 4; i++) x[i] = (uint8_t)(v >> (8 * i));
        return;
    }
    uint16_t v = (uint16_t)(((raw[0] & 0x80) << 8) | ((uint16_t)e << 7) | (raw[0] & 0x7F));
    x[0] = (uint8_t)v;
    x[1] = (uint8_t)(v >> 8);
}

#define TILE_R 32
#define TILE_C 128
#define LANES 4
#define BLOCKS_PER_TILE 512
#define RANS_L 65536u
#define PROB_BITS 12
#define PROB_SCALE 4096u
#define N_CTX_LOSSY 5
#define CTX_UNIFORM 5 /* pseudo-context of the uniform escape bytes */
#define HEADER_BYTES 128
#define MAGIC 0x314B5045u
#define J_MIN (-640)
#define J_MAX 128
#define PEAK_BOUND 15000.0

/* ------------------------------------------------------------------ helpers */
static void put_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put_u32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put_u64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t *p) { uint32_t v = 0; for (int i = 3; i >= 0; i--) v = (v << 8) | p[i]; return v; }
static uint64_t get_u64(const uint8_t *p) { uint64_t v = 0; for (int i = 7; i >= 0; i--) v = (v << 8) | p[i]; return v; }
static uint64_t align16(uint64_t v) { return (v + 15u) & ~(uint64_t)15u; }
/* tile-grid dimensions: the matrix is padded with zeros to whole tiles */
static int64_t pad_rows(int64_t M) { return (M + TILE_R - 1) / TILE_R * TILE_R; }
static int64_t pad_cols(int64_t K) { return (K + TILE_C - 1) / TILE_C * TILE_C; }

/* zero-padded copy of w (M x K) as Mp x Kp; NULL when out of memory */
static uint16_t *padded_copy(const uint16_t *w, int64_t M, int64_t K, int64_t Mp, int64_t Kp) {
    uint16_t *wp = (uint16_t *)calloc((size_t)(Mp * Kp), sizeof(uint16_t));
    if (!wp) return NULL;
    for (int64_t r = 0; r < M; r++) memcpy(wp + r * Kp, w + r * K, (size_t)K * sizeof(uint16_t));
    return wp;
}

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* block b of a tile -> (row in tile, first column in tile) */
static void block_place(int b, int *row, int *col) {
    int slab = b / 128, rem = b % 128;
    *row = rem / 4;
    *col = 32 * slab + 8 * (rem % 4);
}

/* ------------------------------------------------- row scale and grid (§4.1) */
double oracle_row_rms(const uint16_t *w_row, int64_t K) {
    double s = 0.0;
    for (int64_t k = 0; k < K; k++) {
        double v = oracle_bf16_to_f64(w_row[k]);
        s += v * v;
    }
    return sqrt(s / (double)K);
}

double oracle_delta(int j) { return exp2((double)j / 64.0); }

double oracle_rn7(double v) {
    int e;
    double m = frexp(v, &e);
    return ldexp(rint(m * 128.0), e - 7);
}

double oracle_tr7(double v) {
    int e;
    double m = frexp(v, &e);
    return ldexp(floor(m * 128.0), e - 7);
}

static double row_step(double s_r, int j) {
    if (s_r == 0.0) return 0.0;
    double g = oracle_rn7(s_r * oracle_delta(j));
    if (g < ldexp(1.0, -120)) g = ldexp(1.0, -120);
    if (g > ldexp(1.0, 120)) g = ldexp(1.0, 120);
    return g;
}

/* ------------------------------------------------------ nearest E8 (§4.2) */
/* nearest point of D8 (integer vectors with even sum) to y */
static void d8_nearest(const double y[8], int64_t f[8]) {
    int64_t sum = 0;
    for (int i = 0; i < 8; i++) {
        f[i] = (int64_t)floor(y[i] + 0.5);
        sum += f[i];
    }
    if (sum & 1) {
        int worst = 0;
        double worst_d = -1.0;
        for (int i = 0; i < 8; i++) {
            double d = fabs(y[i] - (double)f[i]);
            if (d > worst_d) { worst_d = d; worst = i; }
        }
        if (y[worst] >= (double)f[worst]) f[worst] += 1; else f[worst] -= 1;
    }
}

void oracle_e8_nearest(const double x[8], int64_t a[8], int *coset) {
    int64_t A[8], B[8];
    double y[8], d0 = 0.0, d1 = 0.0;
    d8_nearest(x, A);
    for (int i = 0; i < 8; i++) y[i] = x[i] - 0.5;
    d8_nearest(y, B);
    for (int i = 0; i < 8; i++) {
        double e0 = x[i] - (double)A[i];
        double e1 = y[i] - (double)B[i];
        d0 += e0 * e0;
        d1 += e1 * e1;
    }
    *coset = (d1 < d0) ? 1 : 0;
    for (int i = 0; i < 8; i++) a[i] = *coset ? B[i] : A[i];
}

/* ------------------------------------------------------------ symbols (§4.3) */
/* Returns the number of escaped positions.  u[i] is the coded byte, ctx[i]
 * its context and payload[i] the int16 escape value of position i. */
int oracle_block_symbols(const int64_t a[8], int c, uint8_t u[8], uint8_t ctx[8], int32_t payload[8]) {
    int64_t v[8], lo[8], hi[8];
    int64_t sum7 = 0;
    for (int i = 0; i < 7; i++) sum7 += a[i];
    int64_t p = sum7 & 1;
    int64_t v7 = (a[7] - p) / 2; /* exact: a_7 and the other seven have the same parity */
    for (int i = 0; i < 7; i++) v[i] = 2 * a[i] + c;
    v[7] = 4 * v7 + c;
    ctx[0] = 0; lo[0] = -126; hi[0] = 127;
    for (int i = 1; i < 7; i++) { ctx[i] = (uint8_t)(1 + c); lo[i] = -127; hi[i] = 127; }
    ctx[7] = (uint8_t)(3 + c); lo[7] = -127; hi[7] = 125;
    int n_esc = 0;
    for (int i = 0; i < 8; i++) {
        payload[i] = 0;
        if (v[i] >= lo[i] && v[i] <= hi[i]) {
            u[i] = (uint8_t)(v[i] + 128);
        } else {
            u[i] = (uint8_t)(i == 0 ? c : 0);
            payload[i] = (int32_t)v[i];
            n_esc++;
        }
    }
    return n_esc;
}

/* ------------------------------------------------------- normaliser (§3) */
void oracle_normalize(const uint64_t counts[256], uint32_t freq[256]) {
    uint64_t N = 0;
    for (int u = 0; u < 256; u++) N += counts[u];
    for (int u = 0; u < 256; u++) freq[u] = 0;
    if (N == 0) return;
    int64_t S = 0;
    for (int u = 0; u < 256; u++) {
        if (counts[u] == 0) continue;
        uint64_t f = (uint64_t)(((unsigned __int128)PROB_SCALE * counts[u]) / N);
        freq[u] = (uint32_t)(f < 1 ? 1 : f);
        S += freq[u];
    }
    if (S < (int64_t)PROB_SCALE) {
        int best = -1;
        for (int u = 0; u < 256; u++)
            if (counts[u] > 0 && (best < 0 || counts[u] > counts[best])) best = u;
        freq[best] += (uint32_t)(PROB_SCALE - S);
    }
    while (S > (int64_t)PROB_SCALE) {
        int best = -1;
        for (int u = 0; u < 256; u++)
            if (freq[u] > 1 && (best < 0 || freq[u] > freq[best])) best = u;
        freq[best] -= 1;
        S -= 1;
    }
    for (int u = 0; u < 256; u++) {
        if (freq[u] == PROB_SCALE) {
            freq[u] = PROB_SCALE - 1;
            freq[(u + 1) & 255] = 1;
            break;
        }
    }
}

/* ----------------------------------------------------------------- rANS (§2) */
static void cum_of(const uint32_t *freq, uint32_t *cum) {
    uint32_t c = 0;
    for (int u = 0; u < 256; u++) { cum[u] = c; c += freq[u]; }
}

int oracle_rans_encode(const uint8_t *syms, const uint8_t *ctx, int64_t n, const uint32_t *freq_by_ctx,
                       uint32_t *state, uint16_t *words, int64_t max_words, int64_t *n_words) {
    uint32_t cum_by_ctx[8][256];
    for (int c = 0; c < 8; c++) cum_of(freq_by_ctx + 256 * c, cum_by_ctx[c]);
    uint32_t x = RANS_L;
    int64_t emitted = 0;
    for (int64_t i = n - 1; i >= 0; i--) {
        uint32_t f = freq_by_ctx[256 * ctx[i] + syms[i]];
        uint32_t cum = cum_by_ctx[ctx[i]][syms[i]];
        if (f == 0) return O_ERR_ARG;
        while ((uint64_t)x >= ((uint64_t)f << 20)) {
            if (emitted >= max_words) return O_ERR_NOMEM;
            words[emitted++] = (uint16_t)(x & 0xFFFF);
            x >>= 16;
        }
        x = (x / f) * PROB_SCALE + (x % f) + cum;
    }
    for (int64_t i = 0; i < emitted / 2; i++) { /* emission order -> decode order */
        uint16_t t = words[i];
        words[i] = words[emitted - 1 - i];
        words[emitted - 1 - i] = t;
    }
    *state = x;
    *n_words = emitted;
    return O_OK;
}

/* slot -> symbol table of one context built by a plain loop (-1 = no symbol) */
static void slot_table(const uint32_t *freq, int16_t *sym_of_slot) {
    for (int s = 0; s < (int)PROB_SCALE; s++) sym_of_slot[s] = -1;
    uint32_t c = 0;
    for (int u = 0; u < 256; u++) {
        for (uint32_t k = 0; k < freq[u] && c < PROB_SCALE; k++) sym_of_slot[c++] = (int16_t)u;
    }
}

typedef struct {
    const uint16_t *words;
    int64_t n_words, pos;
    uint32_t x;
    int bad;
} lane_dec;

static int lane_symbol(lane_dec *d, const uint32_t *freq, const uint32_t *cum, const int16_t *sym_of_slot) {
    uint32_t slot = d->x & (PROB_SCALE - 1);
    int s = sym_of_slot[slot];
    if (s < 0) { d->bad = 1; return 0; }
    d->x = freq[s] * (d->x >> PROB_BITS) + slot - cum[s];
    if (d->x < RANS_L) {
        if (d->pos >= d->n_words) { d->bad = 1; return s; }
        d->x = (d->x << 16) | d->words[d->pos++];
    }
    return s;
}

int oracle_rans_decode(const uint16_t *words, int64_t n_words, uint32_t state, const uint8_t *ctx, int64_t n,
                       const uint32_t *freq_by_ctx, uint8_t *syms_out) {
    int16_t tab[8][PROB_SCALE];
    uint32_t cum[8][256];
    for (int c = 0; c < 8; c++) {
        slot_table(freq_by_ctx + 256 * c, tab[c]);
        cum_of(freq_by_ctx + 256 * c, cum[c]);
    }
    lane_dec d = {words, n_words, 0, state, 0};
    for (int64_t i = 0; i < n; i++) {
        syms_out[i] = (uint8_t)lane_symbol(&d, freq_by_ctx + 256 * ctx[i], cum[ctx[i]], tab[ctx[i]]);
        if (d.bad) return O_ERR_CORRUPT;
    }
    return (d.x == RANS_L && d.pos == n_words) ? O_OK : O_ERR_CORRUPT;
}

/* ------------------------------------------------ conversions (§4.5) */
/* Round a finite double to the nearest value with p significand bits whose
 * exponent is at least emin (so subnormals are the multiples of
 * 2^(emin-p+1)); ties to even.  No upper bound is applied here. */
static double round_to_format(double v, int p, int emin) {
    if (v == 0.0 || !isfinite(v)) return v;
    int E;
    frexp(fabs(v), &E); /* |v| in [2^(E-1), 2^E) */
    int e = E - 1 < emin ? emin : E - 1;
    double quantum = ldexp(1.0, e - (p - 1));
    return copysign(rint(fabs(v) / quantum) * quantum, v);
}

/* bits of a finite value already representable in the format */
static uint32_t encode_bits(double r, int p, int emin, int ebits) {
    uint32_t sign = signbit(r) ? 1u : 0u;
    double a = fabs(r);
    uint32_t mbits = (uint32_t)(p - 1), expf = 0, man = 0;
    if (a == 0.0) {
        expf = 0; man = 0;
    } else {
        int E;
        frexp(a, &E);
        int e = E - 1;
        if (e < emin) { /* subnormal */
            expf = 0;
            man = (uint32_t)ldexp(a, -(emin - (int)mbits));
        } else {
            expf = (uint32_t)(e - emin + 1);
            man = (uint32_t)(ldexp(a, -(e - (int)mbits)) - ldexp(1.0, (int)mbits));
        }
    }
    return (sign << (ebits + mbits)) | (expf << mbits) | man;
}

uint16_t oracle_f32_to_bf16(float v) {
    if (isnan(v)) return 0x7FC0;
    double r = round_to_format((double)v, 8, -126);
    if (fabs(r) > 0x1.FEp127) return signbit(r) ? 0xFF80 : 0x7F80;
    if (isinf(r)) return signbit(r) ? 0xFF80 : 0x7F80;
    return (uint16_t)encode_bits(r, 8, -126, 8);
}

uint16_t oracle_f32_to_f16(float v) {
    if (isnan(v)) return 0x7E00;
    double r = round_to_format((double)v, 11, -14);
    if (isinf(r) || fabs(r) > 65504.0) return signbit(r) ? 0xFC00 : 0x7C00;
    return (uint16_t)encode_bits(r, 11, -14, 5);
}

uint8_t oracle_f32_to_e4m3_satfinite(float v) {
    if (isnan(v)) return 0x7F;
    double r = round_to_format((double)v, 4, -6);
    if (fabs(r) > 448.0) r = copysign(448.0, r);
    return (uint8_t)encode_bits(r, 4, -6, 4);
}

int8_t oracle_f32_to_int8(float v) {
    double r = rint((double)v);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

/* ---------------------------------------------------- quantisation pass */
typedef struct {
    int64_t M, K;   /* true shape */
    int64_t Mp, Kp; /* padded shape of the matrix the stats index (row stride Kp) */
    double *s;      /* row RMS over the K true columns (0 for padding rows) */
    double *peak;   /* row max |w| */
} rowstats;

/* wp: the zero-padded Mp x Kp matrix; statistics of row r use its K true columns */
static int row_stats(const uint16_t *wp, int64_t M, int64_t K, int64_t Mp, int64_t Kp, rowstats *rs) {
    rs->M = M; rs->K = K; rs->Mp = Mp; rs->Kp = Kp;
    rs->s = (double *)calloc((size_t)Mp, sizeof(double));
    rs->peak = (double *)calloc((size_t)Mp, sizeof(double));
    if (!rs->s || !rs->peak) return O_ERR_NOMEM;
    for (int64_t r = 0; r < M; r++) {
        rs->s[r] = oracle_row_rms(wp + r * Kp, K);
        double pk = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double v = fabs(oracle_bf16_to_f64(wp[r * Kp + k]));
            if (v > pk) pk = v;
        }
        rs->peak[r] = pk;
    }
    return O_OK;
}

static void free_stats(rowstats *rs) { free(rs->s); free(rs->peak); }

static int valid_j(const rowstats *rs, int j) {
    for (int64_t r = 0; r < rs->M; r++) {
        if (rs->s[r] == 0.0) continue;
        double g = (double)(float)row_step(rs->s[r], j);
        if (!(rs->peak[r] <= PEAK_BOUND * g)) return 0;
    }
    return 1;
}

static int smallest_valid_j(const rowstats *rs) {
    int lo = J_MIN, hi = J_MAX;
    if (valid_j(rs, lo)) return lo;
    while (hi - lo > 1) {
        int mid = lo + (hi - lo) / 2;
        if (valid_j(rs, mid)) hi = mid; else lo = mid;
    }
    return hi;
}

/* quantise block (r, col0..col0+7) with step g; writes a[8], coset */
static void quantise_block(const uint16_t *w, int64_t K, int64_t r, int64_t col0, double g, int64_t a[8], int *c) {
    if (g == 0.0) {
        for (int i = 0; i < 8; i++) a[i] = 0;
        *c = 0;
        return;
    }
    double x[8];
    for (int i = 0; i < 8; i++) x[i] = oracle_bf16_to_f64(w[r * K + col0 + i]) / g;
    oracle_e8_nearest(x, a, c);
}

static int64_t n_sample_rows(int64_t M, float sample_frac) {
    double want = ceil((double)sample_frac * (double)M);
    int64_t n = (int64_t)want;
    if (!(want >= 1.0)) n = 1;
    if (n > M) n = M;
    if (n < 1) n = 1;
    return n;
}

/* wp: the zero-padded matrix (row stride rs->Kp); only true rows and columns are sampled */
static double estimate_with_stats(const uint16_t *wp, const rowstats *rs, float sample_frac, int j) {
    int64_t M = rs->M, K = rs->K, Kp = rs->Kp;
    int64_t ns = n_sample_rows(M, sample_frac);
    uint64_t counts[N_CTX_LOSSY][256];
    memset(counts, 0, sizeof(counts));
    uint64_t n_esc = 0;
    for (int64_t i = 0; i < ns; i++) {
        int64_t r = (int64_t)(((unsigned __int128)i * (uint64_t)M) / (uint64_t)ns);
        double g = (double)(float)row_step(rs->s[r], j);
        for (int64_t col0 = 0; col0 < K; col0 += 8) {
            int64_t a[8];
            int c;
            uint8_t u[8], cx[8];
            int32_t pl[8];
            quantise_block(wp, Kp, r, col0, g, a, &c);
            n_esc += (uint64_t)oracle_block_symbols(a, c, u, cx, pl);
            for (int k = 0; k < 8; k++) counts[cx[k]][u[k]]++;
        }
    }
    double H = 0.0;
    for (int cx = 0; cx < N_CTX_LOSSY; cx++) {
        uint64_t N = 0;
        for (int u = 0; u < 256; u++) N += counts[cx][u];
        for (int u = 0; u < 256; u++)
            if (counts[cx][u] > 0) H += (double)counts[cx][u] * log2((double)N / (double)counts[cx][u]);
    }
    return (H + 16.0 * (double)n_esc) / (double)(ns * K);
}

double oracle_estimate_bpp(const uint16_t *w, int64_t M, int64_t K, float sample_frac, int j) {
    if (M <= 0 || K <= 0 || K % 8) return -1.0;
    int64_t Mp = pad_rows(M), Kp = pad_cols(K);
    uint16_t *wp = padded_copy(w, M, K, Mp, Kp);
    rowstats rs;
    double e = -1.0;
    if (wp && row_stats(wp, M, K, Mp, Kp, &rs) == O_OK) e = estimate_with_stats(wp, &rs, sample_frac, j);
    if (wp) free_stats(&rs);
    free(wp);
    return e;
}

static int select_with_stats(const uint16_t *w, const rowstats *rs, float target_bpp, float sample_frac, int *j_lo_out) {
    double T = (double)target_bpp;
    int j_lo = smallest_valid_j(rs);
    if (j_lo_out) *j_lo_out = j_lo;
    double e_lo = estimate_with_stats(w, rs, sample_frac, j_lo);
    if (e_lo <= T) return j_lo;
    double e_hi = estimate_with_stats(w, rs, sample_frac, J_MAX);
    if (e_hi > T) return J_MAX;
    int lo = j_lo, hi = J_MAX;
    while (hi - lo > 1) {
        int mid = lo + (hi - lo) / 2;
        double e = estimate_with_stats(w, rs, sample_frac, mid);
        if (e <= T) { hi = mid; e_hi = e; } else { lo = mid; e_lo = e; }
    }
    return (fabs(e_hi - T) <= fabs(e_lo - T)) ? hi : lo;
}

int oracle_select_j(const uint16_t *w, int64_t M, int64_t K, float target_bpp, float sample_frac, int *j_lo_out) {
    if (M <= 0 || K <= 0 || K % 8) return J_MAX + 1;
    int64_t Mp = pad_rows(M), Kp = pad_cols(K);
    uint16_t *wp = padded_copy(w, M, K, Mp, Kp);
    rowstats rs;
    int j = J_MAX + 1;
    if (wp && row_stats(wp, M, K, Mp, Kp, &rs) == O_OK) j = select_with_stats(wp, &rs, target_bpp, sample_frac, j_lo_out);
    if (wp) free_stats(&rs);
    free(wp);
    return j;
}

/* ------------------------------------------------------------ serialiser */
typedef struct {
    int mode, container, n_ctx;
    int64_t M, K, n_tiles;
    float target_bpp;
    int j;
    double delta;
    uint32_t n_sample;
    uint32_t freq[8][256];
    const float *rowmeta; /* g (| m | t) */
    int64_t rowmeta_floats;
    uint8_t **tile_bytes;
    uint64_t *tile_size;
} blob_parts;

static int serialise(const blob_parts *bp, uint8_t **blob, size_t *bytes) {
    uint64_t tables_off = HEADER_BYTES, tables_size = 0;
    for (int c = 0; c < bp->n_ctx; c++) {
        int lo = -1, hi = -1;
        for (int u = 0; u < 256; u++)
            if (bp->freq[c][u] > 0) { if (lo < 0) lo = u; hi = u; }
        tables_size += 4 + (lo < 0 ? 0 : 2 * (uint64_t)(hi - lo + 1));
    }
    uint64_t rowmeta_off = align16(tables_off + tables_size);
    uint64_t offsets_off = align16(rowmeta_off + 4 * (uint64_t)bp->rowmeta_floats);
    uint64_t payload_off = align16(offsets_off + 8 * (uint64_t)(bp->n_tiles + 1));
    uint64_t payload = 0;
    for (int64_t t = 0; t < bp->n_tiles; t++) payload += bp->tile_size[t];
    uint64_t total = payload_off + payload;
    uint8_t *b = (uint8_t *)calloc((size_t)total, 1);
    if (!b) return O_ERR_NOMEM;
    put_u32(b + 0, MAGIC);
    put_u16(b + 4, 1);
    b[6] = (uint8_t)bp->mode;
    b[7] = (uint8_t)bp->container;
    put_u64(b + 8, (uint64_t)bp->M);
    put_u64(b + 16, (uint64_t)bp->K);
    put_u64(b + 24, (uint64_t)bp->n_tiles);
    memcpy(b + 32, &bp->target_bpp, 4);
    put_u32(b + 36, (uint32_t)bp->j);
    memcpy(b + 40, &bp->delta, 8);
    put_u16(b + 48, TILE_R);
    put_u16(b + 50, TILE_C);
    b[52] = LANES;
    b[53] = (uint8_t)bp->n_ctx;
    put_u64(b + 56, tables_off);
    put_u64(b + 64, rowmeta_off);
    put_u64(b + 72, offsets_off);
    put_u64(b + 80, payload_off);
    put_u64(b + 88, total);
    put_u32(b + 96, bp->n_sample);
    uint8_t *p = b + tables_off;
    for (int c = 0; c < bp->n_ctx; c++) {
        int lo = -1, hi = -1;
        for (int u = 0; u < 256; u++)
            if (bp->freq[c][u] > 0) { if (lo < 0) lo = u; hi = u; }
        if (lo < 0) { put_u16(p, 0); put_u16(p + 2, 0); p += 4; continue; }
        put_u16(p, (uint16_t)lo);
        put_u16(p + 2, (uint16_t)(hi - lo + 1));
        p += 4;
        for (int u = lo; u <= hi; u++) { put_u16(p, (uint16_t)bp->freq[c][u]); p += 2; }
    }
    memcpy(b + rowmeta_off, bp->rowmeta, 4 * (size_t)bp->rowmeta_floats);
    uint64_t off = 0;
    for (int64_t t = 0; t < bp->n_tiles; t++) {
        put_u64(b + offsets_off + 8 * (uint64_t)t, off);
        memcpy(b + payload_off + off, bp->tile_bytes[t], (size_t)bp->tile_size[t]);
        off += bp->tile_size[t];
    }
    put_u64(b + offsets_off + 8 * (uint64_t)bp->n_tiles, off);
    *blob = b;
    *bytes = (size_t)total;
    return O_OK;
}

/* one tile's payload from its lanes' (raw?, states, words) */
static int pack_tile(const uint8_t *raw, uint64_t raw_len, const uint32_t state[4], uint16_t *const words[4],
                     const int64_t nw[4], uint8_t **out, uint64_t *size) {
    uint64_t n = (raw ? raw_len : 0) + 16 + 8;
    for (int l = 0; l < 4; l++) {
        if (nw[l] > 65535) return O_ERR_UNSUPPORTED;
        n += 2 * (uint64_t)nw[l];
    }
    n = align16(n);
    uint8_t *t = (uint8_t *)calloc((size_t)n, 1), *p = t;
    if (!t) return O_ERR_NOMEM;
    if (raw) { memcpy(p, raw, (size_t)raw_len); p += raw_len; }
    for (int l = 0; l < 4; l++) { put_u32(p, state[l]); p += 4; }
    for (int l = 0; l < 4; l++) { put_u16(p, (uint16_t)nw[l]); p += 2; }
    for (int l = 0; l < 4; l++)
        for (int64_t i = 0; i < nw[l]; i++) { put_u16(p, words[l][i]); p += 2; }
    *out = t;
    *size = n;
    return O_OK;
}

static void free_tiles(uint8_t **tb, int64_t n) {
    if (!tb) return;
    for (int64_t t = 0; t < n; t++) free(tb[t]);
    free(tb);
}

/* --------------------------------------------------------- lossy encoder */
#define J_SELECT (-100000) /* forced_j value that asks for the rate search */

static int encode_lossy(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int forced_j, int container,
                        float sample_frac, uint8_t **blob, size_t *bytes);

int oracle_encode(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int container, float sample_frac,
                  uint8_t **blob, size_t *bytes) {
    return encode_lossy(w, M, K, target_bpp, J_SELECT, container, sample_frac, blob, bytes);
}

int oracle_encode_at(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int j, int container,
                     float sample_frac, uint8_t **blob, size_t *bytes) {
    if (j < J_MIN || j > J_MAX) return O_ERR_ARG;
    return encode_lossy(w, M, K, target_bpp, j, container, sample_frac, blob, bytes);
}

int oracle_smallest_valid_j(const uint16_t *w, int64_t M, int64_t K) {
    if (!w || M <= 0 || K <= 0 || K % 8) return J_MAX + 1;
    int64_t Mp = pad_rows(M), Kp = pad_cols(K);
    uint16_t *wp = padded_copy(w, M, K, Mp, Kp);
    rowstats rs;
    int j = J_MAX + 1;
    if (wp && row_stats(wp, M, K, Mp, Kp, &rs) == O_OK) j = smallest_valid_j(&rs);
    if (wp) free_stats(&rs);
    free(wp);
    return j;
}

static int encode_lossy(const uint16_t *w, int64_t M, int64_t K, float target_bpp, int forced_j, int container,
                        float sample_frac, uint8_t **blob, size_t *bytes) {
    if (!w || !blob || !bytes) return O_ERR_ARG;
    if (M <= 0 || K <= 0 || K % 8) return O_ERR_SHAPE;
    if (container < O_C_BF16 || container > O_C_INT8) return O_ERR_ARG;
    if (!(target_bpp > 0.0f) || !isfinite(target_bpp) || !(sample_frac > 0.0f) || !isfinite(sample_frac)) return O_ERR_ARG;
    for (int64_t i = 0; i < M * K; i++)
        if ((w[i] & 0x7F80) == 0x7F80) return O_ERR_NONFINITE;

    /* from here on the matrix is the zero-padded Mp x Kp one; the true shape
       only enters the row statistics, the rate estimate and the header */
    const int64_t M_true = M, K_true = K;
    const uint16_t *w_true = w;
    M = pad_rows(M_true);
    K = pad_cols(K_true);
    uint16_t *wp = padded_copy(w_true, M_true, K_true, M, K);
    if (!wp) return O_ERR_NOMEM;
    w = wp;

    rowstats rs;
    int rc = row_stats(w, M_true, K_true, M, K, &rs);
    if (rc != O_OK) { free_stats(&rs); free(wp); return rc; }
    int j;
    if (forced_j == J_SELECT) {
        j = select_with_stats(w, &rs, target_bpp, sample_frac, NULL);
    } else {
        /* a resolution chosen by the caller must keep every row's peak in range */
        if (forced_j < smallest_valid_j(&rs)) { free_stats(&rs); free(wp); return O_ERR_ARG; }
        j = forced_j;
    }

    int64_t n_blocks = M * (K / 8);
    int32_t *val = (int32_t *)malloc((size_t)(M * K) * sizeof(int32_t)); /* v of every coordinate */
    uint8_t *sym = (uint8_t *)malloc((size_t)(M * K));                    /* coded byte u */
    uint8_t *cos_ = (uint8_t *)malloc((size_t)n_blocks);
    float *meta = (float *)malloc((size_t)M * 3 * sizeof(float));
    if (!val || !sym || !cos_ || !meta) { rc = O_ERR_NOMEM; goto done_early; }

    float *g = meta, *m = meta + M, *t = meta + 2 * M;
    uint64_t counts[N_CTX_LOSSY][256];
    memset(counts, 0, sizeof(counts));
    for (int64_t r = 0; r < M; r++) {
        g[r] = (float)row_step(rs.s[r], j);
        double Q = 0.0;
        for (int64_t col0 = 0; col0 < K; col0 += 8) {
            int64_t a[8];
            int c;
            uint8_t u[8], cx[8];
            int32_t pl[8];
            quantise_block(w, K, r, col0, (double)g[r], a, &c);
            oracle_block_symbols(a, c, u, cx, pl);
            cos_[(r * K + col0) / 8] = (uint8_t)c;
            for (int i = 0; i < 8; i++) {
                double q = fabs((double)a[i] + 0.5 * c);
                if (q > Q) Q = q;
                sym[r * K + col0 + i] = u[i];
                int esc = (i == 0) ? (u[i] <= 1) : (u[i] == 0);
                int64_t v = esc ? (int64_t)pl[i] : (int64_t)u[i] - 128;
                if (v < -32768 || v > 32767) { rc = O_ERR_UNSUPPORTED; goto done_early; }
                val[r * K + col0 + i] = (int32_t)v;
                counts[cx[i]][u[i]]++;
            }
        }
        if (container == O_C_FP8) m[r] = (float)(Q == 0.0 ? 1.0 : oracle_tr7(448.0 / Q));
        else if (container == O_C_INT8) m[r] = (float)(Q == 0.0 ? 1.0 : (2.0 * Q <= 127.0 ? 2.0 : oracle_tr7(127.0 / Q)));
        else m[r] = 1.0f;
        t[r] = (float)((double)g[r] / (double)m[r]);
    }

    blob_parts bp;
    memset(&bp, 0, sizeof(bp));
    bp.mode = 0; bp.container = container; bp.n_ctx = N_CTX_LOSSY;
    bp.M = M_true; bp.K = K_true; bp.n_tiles = (M / TILE_R) * (K / TILE_C);
    bp.target_bpp = target_bpp; bp.j = j; bp.delta = oracle_delta(j);
    bp.n_sample = (uint32_t)n_sample_rows(M_true, sample_frac);
    for (int c = 0; c < N_CTX_LOSSY; c++) oracle_normalize(counts[c], bp.freq[c]);
    for (int u = 0; u < 256; u++) bp.freq[CTX_UNIFORM][u] = 16;

    /* row metadata: g, then m and t for FP8/INT8 */
    float *rm = (float *)malloc((size_t)M * 3 * sizeof(float));
    if (!rm) { rc = O_ERR_NOMEM; goto done_early; }
    memcpy(rm, g, (size_t)M * sizeof(float));
    bp.rowmeta_floats = M;
    if (container == O_C_FP8 || container == O_C_INT8) {
        memcpy(rm + M, m, (size_t)M * sizeof(float));
        memcpy(rm + 2 * M, t, (size_t)M * sizeof(float));
        bp.rowmeta_floats = 3 * M;
    }
    bp.rowmeta = rm;

    bp.tile_bytes = (uint8_t **)calloc((size_t)bp.n_tiles, sizeof(uint8_t *));
    bp.tile_size = (uint64_t *)calloc((size_t)bp.n_tiles, sizeof(uint64_t));
    const int64_t max_syms = 128 * (8 + 16);
    uint8_t *ls = (uint8_t *)malloc(max_syms), *lc = (uint8_t *)malloc(max_syms);
    uint16_t *lw[4];
    for (int l = 0; l < 4; l++) lw[l] = (uint16_t *)malloc(sizeof(uint16_t) * max_syms);
    if (!bp.tile_bytes || !bp.tile_size || !ls || !lc || !lw[0] || !lw[1] || !lw[2] || !lw[3]) { rc = O_ERR_NOMEM; goto done; }
    int64_t tiles_per_row = K / TILE_C;
    for (int64_t tile = 0; tile < bp.n_tiles && rc == O_OK; tile++) {
        int64_t r0 = (tile / tiles_per_row) * TILE_R, c0 = (tile % tiles_per_row) * TILE_C;
        uint32_t state[4];
        int64_t nw[4];
        for (int l = 0; l < 4 && rc == O_OK; l++) {
            int64_t n = 0;
            for (int b = l; b < BLOCKS_PER_TILE; b += 4) {
                int br, bc;
                block_place(b, &br, &bc);
                int64_t r = r0 + br, col0 = c0 + bc;
                int c = cos_[(r * K + col0) / 8];
                for (int i = 0; i < 8; i++) {
                    ls[n] = sym[r * K + col0 + i];
                    lc[n] = (uint8_t)(i == 0 ? 0 : (i < 7 ? 1 + c : 3 + c));
                    n++;
                }
                for (int i = 0; i < 8; i++) {
                    uint8_t u = sym[r * K + col0 + i];
                    int esc = (i == 0) ? (u <= 1) : (u == 0);
                    if (!esc) continue;
                    uint16_t P = (uint16_t)(int16_t)val[r * K + col0 + i];
                    ls[n] = (uint8_t)(P >> 8); lc[n] = CTX_UNIFORM; n++;
                    ls[n] = (uint8_t)(P & 0xFF); lc[n] = CTX_UNIFORM; n++;
                }
            }
            rc = oracle_rans_encode(ls, lc, n, &bp.freq[0][0], &state[l], lw[l], max_syms, &nw[l]);
        }
        if (rc == O_OK) rc = pack_tile(NULL, 0, state, lw, nw, &bp.tile_bytes[tile], &bp.tile_size[tile]);
    }
    if (rc == O_OK) rc = serialise(&bp, blob, bytes);
done:
    free(ls); free(lc);
    for (int l = 0; l < 4; l++) free(lw[l]);
    free_tiles(bp.tile_bytes, bp.n_tiles);
    free(bp.tile_size);
    free(rm);
done_early:
    free(val); free(sym); free(cos_); free(meta);
    free_stats(&rs);
    free(wp);
    return rc;
}

/* ------------------------------------------------------ lossless encoder (§5) */
int oracle_encode_lossless_dtype(const void *w_in, int64_t M, int64_t K, int dtype, uint8_t **blob, size_t *bytes) {
    if (!w_in || !blob || !bytes) return O_ERR_ARG;
    if (!lossless_dtype_ok(dtype)) return O_ERR_ARG;
    if (M <= 0 || K <= 0 || K % 8) return O_ERR_SHAPE;
    const int eb = elem_bytes(dtype), rb = raw_per_elem(dtype);
    /* the zero-padded Mp x Kp matrix is coded; the header keeps the true shape */
    const int64_t M_true = M, K_true = K;
    M = pad_rows(M_true);
    K = pad_cols(K_true);
    uint8_t *w = (uint8_t *)calloc((size_t)(M * K), (size_t)eb);
    if (!w) return O_ERR_NOMEM;
    for (int64_t r = 0; r < M_true; r++)
        memcpy(w + (size_t)(r * K) * eb, (const uint8_t *)w_in + (size_t)(r * K_true) * eb, (size_t)K_true * eb);
    uint64_t counts[256];
    memset(counts, 0, sizeof(counts));
    uint8_t scratch[3];
    for (int64_t i = 0; i < M * K; i++) counts[split_elem(dtype, w + (size_t)i * eb, scratch)]++;
    blob_parts bp;
    memset(&bp, 0, sizeof(bp));
    bp.mode = 1; bp.container = dtype; bp.n_ctx = 1;
    bp.M = M_true; bp.K = K_true; bp.n_tiles = (M / TILE_R) * (K / TILE_C);
    oracle_normalize(counts, bp.freq[0]);
    float dummy = 0.0f;
    bp.rowmeta = &dummy;
    bp.rowmeta_floats = 0;
    bp.tile_bytes = (uint8_t **)calloc((size_t)bp.n_tiles, sizeof(uint8_t *));
    bp.tile_size = (uint64_t *)calloc((size_t)bp.n_tiles, sizeof(uint64_t));
    const uint64_t raw_len = (uint64_t)rb * 4096u;
    uint8_t *raw = (uint8_t *)malloc(raw_len ? raw_len : 1);
    uint8_t ls[1024], lc[1024];
    uint16_t *lw[4];
    int rc = O_OK;
    for (int l = 0; l < 4; l++) lw[l] = (uint16_t *)malloc(sizeof(uint16_t) * 1024);
    if (!raw || !bp.tile_bytes || !bp.tile_size || !lw[0] || !lw[1] || !lw[2] || !lw[3]) rc = O_ERR_NOMEM;
    memset(lc, 0, sizeof(lc));
    int64_t tiles_per_row = K / TILE_C;
    for (int64_t tile = 0; tile < bp.n_tiles && rc == O_OK; tile++) {
        int64_t r0 = (tile / tiles_per_row) * TILE_R, c0 = (tile % tiles_per_row) * TILE_C;
        /* raw bytes in block order: element i of block b at rb * (8 b + i) */
        for (int b = 0; b < BLOCKS_PER_TILE; b++) {
            int br, bc;
            block_place(b, &br, &bc);
            for (int i = 0; i < 8; i++)
                split_elem(dtype, w + (size_t)((r0 + br) * K + c0 + bc + i) * eb, raw + (size_t)rb * (8 * b + i));
        }
        uint32_t state[4];
        int64_t nw[4];
        for (int l = 0; l < 4 && rc == O_OK; l++) {
            int64_t n = 0;
            for (int b = l; b < BLOCKS_PER_TILE; b += 4) {
                int br, bc;
                block_place(b, &br, &bc);
                for (int i = 0; i < 8; i++)
                    ls[n++] = split_elem(dtype, w + (size_t)((r0 + br) * K + c0 + bc + i) * eb, scratch);
            }
            rc = oracle_rans_encode(ls, lc, n, &bp.freq[0][0], &state[l], lw[l], 1024, &nw[l]);
        }
        if (rc == O_OK) rc = pack_tile(rb ? raw : NULL, raw_len, state, lw, nw, &bp.tile_bytes[tile], &bp.tile_size[tile]);
    }
    if (rc == O_OK) rc = serialise(&bp, blob, bytes);
    for (int l = 0; l < 4; l++) free(lw[l]);
    free_tiles(bp.tile_bytes, bp.n_tiles);
    free(bp.tile_size);
    free(raw);
    free(w);
    return rc;
}

int oracle_encode_lossless(const uint16_t *w, int64_t M, int64_t K, uint8_t **blob, size_t *bytes) {
    return oracle_encode_lossless_dtype(w, M, K, O_C_BF16, blob, bytes);
}

void oracle_free(void *p) { free(p); }

/* ---------------------------------------------------------------- decoder */
typedef struct {
    int mode, container, n_ctx;
    int64_t M, K, n_tiles; /* true shape */
    int64_t Mp, Kp;        /* tile grid: the shape padded to whole tiles */
    uint64_t rowmeta_off, offsets_off, payload_off;
    uint32_t freq[8][256], cum[8][256];
    int16_t tab[8][PROB_SCALE];
} parsed;

static int parse(const uint8_t *b, size_t bytes, parsed *ps) {
    if (!b || bytes < HEADER_BYTES) return O_ERR_CORRUPT;
    if (get_u32(b) != MAGIC || get_u16(b + 4) != 1) return O_ERR_CORRUPT;
    ps->mode = b[6];
    ps->container = b[7];
    ps->M = (int64_t)get_u64(b + 8);
    ps->K = (int64_t)get_u64(b + 16);
    ps->n_tiles = (int64_t)get_u64(b + 24);
    if (ps->mode > 1 || (ps->mode == 0 && ps->container > 3) || (ps->mode == 1 && !lossless_dtype_ok(ps->container)))
        return O_ERR_CORRUPT;
    if (ps->M <= 0 || ps->K <= 0 || ps->K % 8) return O_ERR_CORRUPT;
    if (ps->M > ((int64_t)1 << 40) || ps->K > ((int64_t)1 << 40)) return O_ERR_CORRUPT;
    ps->Mp = pad_rows(ps->M);
    ps->Kp = pad_cols(ps->K);
    if (ps->n_tiles != (ps->Mp / TILE_R) * (ps->Kp / TILE_C)) return O_ERR_CORRUPT;
    if (get_u16(b + 48) != TILE_R || get_u16(b + 50) != TILE_C || b[52] != LANES) return O_ERR_CORRUPT;
    ps->n_ctx = b[53];
    if (ps->n_ctx != (ps->mode == 0 ? N_CTX_LOSSY : 1)) return O_ERR_CORRUPT;
    uint64_t tables_off = get_u64(b + 56);
    ps->rowmeta_off = get_u64(b + 64);
    ps->offsets_off = get_u64(b + 72);
    ps->payload_off = get_u64(b + 80);
    uint64_t total = get_u64(b + 88);
    if (total != bytes || tables_off != HEADER_BYTES) return O_ERR_CORRUPT;
    if (!(tables_off <= ps->rowmeta_off && ps->rowmeta_off <= ps->offsets_off && ps->offsets_off <= ps->payload_off &&
          ps->payload_off <= total))
        return O_ERR_CORRUPT;
    if ((ps->rowmeta_off | ps->offsets_off | ps->payload_off) & 15) return O_ERR_CORRUPT;
    memset(ps->freq, 0, sizeof(ps->freq));
    const uint8_t *p = b + tables_off, *end = b + ps->rowmeta_off;
    for (int c = 0; c < ps->n_ctx; c++) {
        if (p + 4 > end) return O_ERR_CORRUPT;
        int lo = get_u16(p), n = get_u16(p + 2);
        p += 4;
        if (lo + n > 256 || p + 2 * n > end) return O_ERR_CORRUPT;
        uint32_t s = 0;
        for (int i = 0; i < n; i++) { ps->freq[c][lo + i] = get_u16(p); s += get_u16(p); p += 2; }
        if (!(s == PROB_SCALE || (s == 0 && n == 0))) return O_ERR_CORRUPT;
    }
    if (ps->mode == 0)
        for (int u = 0; u < 256; u++) ps->freq[CTX_UNIFORM][u] = 16;
    uint64_t meta_floats = ps->mode == 1 ? 0 : (uint64_t)ps->Mp * ((ps->container >= O_C_FP8) ? 3 : 1);
    if (ps->rowmeta_off + 4 * meta_floats > ps->offsets_off) return O_ERR_CORRUPT;
    if (ps->offsets_off + 8 * (uint64_t)(ps->n_tiles + 1) > ps->payload_off) return O_ERR_CORRUPT;
    uint64_t prev = 0, min_tile = (ps->mode == 1 ? 4096u * (uint64_t)raw_per_elem(ps->container) : 0u) + 24u;
    for (int64_t t = 0; t <= ps->n_tiles; t++) {
        uint64_t o = get_u64(b + ps->offsets_off + 8 * (uint64_t)t);
        if (t == 0 && o != 0) return O_ERR_CORRUPT;
        if (o & 15) return O_ERR_CORRUPT;
        if (t > 0 && o < prev + min_tile) return O_ERR_CORRUPT;
        prev = o;
    }
    if (ps->payload_off + prev != total) return O_ERR_CORRUPT;
    for (int c = 0; c < 8; c++) {
        slot_table(ps->freq[c], ps->tab[c]);
        cum_of(ps->freq[c], ps->cum[c]);
    }
    return O_OK;
}

static float rowmeta_at(const uint8_t *b, const parsed *ps, int which, int64_t r) {
    float v;
    memcpy(&v, b + ps->rowmeta_off + 4 * ((uint64_t)which * (uint64_t)ps->Mp + (uint64_t)r), 4);
    return v;
}

/* decode one tile; writes container values (out) and/or symbol bytes (sym_out)
   for the blocks inside the true M x K matrix (padding blocks are decoded and
   checked, not written) */
static int decode_tile(const uint8_t *b, const parsed *ps, int64_t tile, void *out, uint8_t *sym_out, int32_t *k_out) {
    int64_t K = ps->K, tiles_per_row = ps->Kp / TILE_C;
    int64_t r0 = (tile / tiles_per_row) * TILE_R, c0 = (tile % tiles_per_row) * TILE_C;
    uint64_t t_off = get_u64(b + ps->offsets_off + 8 * (uint64_t)tile);
    uint64_t t_end = get_u64(b + ps->offsets_off + 8 * (uint64_t)(tile + 1));
    const uint8_t *tp = b + ps->payload_off + t_off;
    const uint8_t *raw = NULL;
    const int rb = ps->mode == 1 ? raw_per_elem(ps->container) : 0, eb = elem_bytes(ps->container);
    if (ps->mode == 1) { raw = tp; tp += 4096 * rb; }
    uint32_t state[4];
    int64_t nw[4];
    for (int l = 0; l < 4; l++) state[l] = get_u32(tp + 4 * l);
    for (int l = 0; l < 4; l++) nw[l] = get_u16(tp + 16 + 2 * l);
    const uint8_t *wp = tp + 24;
    uint64_t need = (uint64_t)(wp - (b + ps->payload_off + t_off)) + 2 * (uint64_t)(nw[0] + nw[1] + nw[2] + nw[3]);
    if (need > t_end - t_off) return O_ERR_CORRUPT;
    for (int l = 0; l < 4; l++) {
        /* words are little-endian u16: copy them into an aligned array */
        uint16_t *words = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(nw[l] + 1));
        if (!words) return O_ERR_NOMEM;
        for (int64_t i = 0; i < nw[l]; i++) words[i] = get_u16(wp + 2 * i);
        wp += 2 * nw[l];
        lane_dec d = {words, nw[l], 0, state[l], 0};
        for (int bb = l; bb < BLOCKS_PER_TILE; bb += 4) {
            int br, bc;
            block_place(bb, &br, &bc);
            int64_t r = r0 + br, col0 = c0 + bc;
            int inside = r < ps->M && col0 < ps->K;
            if (ps->mode == 1) {
                for (int i = 0; i < 8; i++) {
                    int e = lane_symbol(&d, ps->freq[0], ps->cum[0], ps->tab[0]);
                    if (sym_out && inside) sym_out[r * K + col0 + i] = (uint8_t)e;
                    if (out && inside)
                        join_elem(ps->container, (uint8_t)e, raw + (size_t)rb * (8 * bb + i),
                                  (uint8_t *)out + (size_t)(r * K + col0 + i) * eb);
                }
                continue;
            }
            /* lossy: s0, then s1..s6 under 1+c, s7 under 3+c, then escape payloads */
            int u[8];
            u[0] = lane_symbol(&d, ps->freq[0], ps->cum[0], ps->tab[0]);
            int c = u[0] & 1;
            for (int i = 1; i < 7; i++) u[i] = lane_symbol(&d, ps->freq[1 + c], ps->cum[1 + c], ps->tab[1 + c]);
            u[7] = lane_symbol(&d, ps->freq[3 + c], ps->cum[3 + c], ps->tab[3 + c]);
            int64_t v[8];
            for (int i = 0; i < 8; i++) {
                int esc = (i == 0) ? (u[i] <= 1) : (u[i] == 0);
                if (!esc) { v[i] = u[i] - 128; continue; }
                int hi = lane_symbol(&d, ps->freq[CTX_UNIFORM], ps->cum[CTX_UNIFORM], ps->tab[CTX_UNIFORM]);
                int lo = lane_symbol(&d, ps->freq[CTX_UNIFORM], ps->cum[CTX_UNIFORM], ps->tab[CTX_UNIFORM]);
                v[i] = (int16_t)(uint16_t)((hi << 8) | lo);
            }
            /* payload consistency: v_i = 2 a_i + c for i < 7, v_7 = 4 v7 + c */
            for (int i = 0; i < 7; i++)
                if (((v[i] - c) & 1) != 0) d.bad = 1;
            if (((v[7] - c) & 3) != 0) d.bad = 1;
            int64_t a[8], sum7 = 0;
            for (int i = 0; i < 7; i++) { a[i] = (v[i] - c) / 2; sum7 += a[i]; }
            int64_t p = sum7 & 1;
            a[7] = 2 * ((v[7] - c) / 4) + p;
            if (sym_out && inside)
                for (int i = 0; i < 8; i++) sym_out[r * K + col0 + i] = (uint8_t)u[i];
            if (k_out && inside)
                for (int i = 0; i < 8; i++) k_out[r * K + col0 + i] = (int32_t)(2 * a[i] + c);
            if (!out || !inside) continue;
            float g = rowmeta_at(b, ps, 0, r);
            float m = (ps->container >= O_C_FP8) ? rowmeta_at(b, ps, 1, r) : 1.0f;
            for (int i = 0; i < 8; i++) {
                double q = (double)a[i] + 0.5 * (double)c;
                int64_t idx = r * K + col0 + i;
                switch (ps->container) {
                case O_C_BF16: ((uint16_t *)out)[idx] = oracle_f32_to_bf16((float)((double)g * q)); break;
                case O_C_FP16: ((uint16_t *)out)[idx] = oracle_f32_to_f16((float)((double)g * q)); break;
                case O_C_FP8: ((uint8_t *)out)[idx] = oracle_f32_to_e4m3_satfinite((float)(q * (double)m)); break;
                default: ((int8_t *)out)[idx] = oracle_f32_to_int8((float)(q * (double)m)); break;
                }
            }
        }
        int ok = !d.bad && d.x == RANS_L && d.pos == d.n_words;
        free(words);
        if (!ok) return O_ERR_CORRUPT;
    }
    return O_OK;
}

int oracle_decode(const uint8_t *blob, size_t bytes, void *out, float *row_scale_out, int64_t t_lo, int64_t t_hi) {
    parsed *ps = (parsed *)malloc(sizeof(parsed));
    if (!ps) return O_ERR_NOMEM;
    int rc = parse(blob, bytes, ps);
    if (rc == O_OK && (t_lo < 0 || t_hi > ps->n_tiles || t_lo > t_hi)) rc = O_ERR_ARG;
    if (rc == O_OK && row_scale_out && t_lo == 0 && ps->mode == 0 && ps->container >= O_C_FP8)
        for (int64_t r = 0; r < ps->M; r++) row_scale_out[r] = rowmeta_at(blob, ps, 2, r);
    for (int64_t t = t_lo; t < t_hi && rc == O_OK; t++) rc = decode_tile(blob, ps, t, out, NULL, NULL);
    free(ps);
    return rc;
}

int oracle_decode_symbols(const uint8_t *blob, size_t bytes, uint8_t *sym_out, int64_t t_lo, int64_t t_hi) {
    parsed *ps = (parsed *)malloc(sizeof(parsed));
    if (!ps) return O_ERR_NOMEM;
    int rc = parse(blob, bytes, ps);
    if (rc == O_OK && (t_lo < 0 || t_hi > ps->n_tiles || t_lo > t_hi)) rc = O_ERR_ARG;
    for (int64_t t = t_lo; t < t_hi && rc == O_OK; t++) rc = decode_tile(blob, ps, t, NULL, sym_out, NULL);
    free(ps);
    return rc;
}

int oracle_decode_lattice(const uint8_t *blob, size_t bytes, int32_t *k_out, int64_t t_lo, int64_t t_hi) {
    parsed *ps = (parsed *)malloc(sizeof(parsed));
    if (!ps) return O_ERR_NOMEM;
    int rc = parse(blob, bytes, ps);
    if (rc == O_OK && ps->mode != 0) rc = O_ERR_ARG;
    if (rc == O_OK && (t_lo < 0 || t_hi > ps->n_tiles || t_lo > t_hi)) rc = O_ERR_ARG;
    for (int64_t t = t_lo; t < t_hi && rc == O_OK; t++) rc = decode_tile(blob, ps, t, NULL, NULL, k_out);
    free(ps);
    return rc;
}

/* batch conversions for the conversion pins: kind 0 bf16, 1 fp16, 2 e4m3, 3 int8 */
void oracle_convert_f32(int kind, int64_t n, const float *in, void *out) {
    for (int64_t i = 0; i < n; i++) {
        switch (kind) {
        case 0: ((uint16_t *)out)[i] = oracle_f32_to_bf16(in[i]); break;
        case 1: ((uint16_t *)out)[i] = oracle_f32_to_f16(in[i]); break;
        case 2: ((uint8_t *)out)[i] = oracle_f32_to_e4m3_satfinite(in[i]); break;
        default: ((int8_t *)out)[i] = oracle_f32_to_int8(in[i]); break;
        }
    }
}

/* ------------------------------------------------------------- fp64 GEMM */
void oracle_gemm_f64(const double *x, const double *w, double *y, int64_t T, int64_t N, int64_t K) {
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < N; n++) {
            double s = 0.0;
            for (int64_t k = 0; k < K; k++) s += x[t * K + k] * w[n * K + k];
            y[t * N + n] = s;
        }
}

/* ---------------------------------------- fixed-width 4-bit comparators
   The comparators of the evaluation ("EntroPack: Fast and Accurate
   Entropy-Coded Weight Compression at Arbitrary Bitrates", Abstract: lower
   relative L2 weight error than NF4 at a 4-bit target, with less storage;
   lower errors than fixed-width codes of about the same size).

   Both are block-absmax 4-bit codebook quantisers: a block of `block`
   consecutive weights stores its absolute maximum s as FP32 and one 4-bit
   code per weight (4 + 32 / block bits per weight).  The code of w is the
   nearest codebook level to w / s, both computed in FP32 (ties to the lower
   code); the reconstruction is BF16(level * s), one FP32 product rounded to
   nearest even.

   NF4 codebook (4-bit NormalFloat): quantiles of N(0, 1), scaled so that the
   extremes are +-1, with an exact zero; 8 non-negative levels at
   probabilities evenly spaced from 1/2 to 1 - d, and 7 negative levels at
   probabilities evenly spaced from 1/2 to 1 - d and mirrored, where
   d = (1/32 + 1/30) / 2 keeps the outermost quantile finite.
   INT4 codebook (symmetric absmax integer): the 15 levels k / 7, k = -7..7,
   and a 16th code equal to level 0 (never chosen: ties go to the lower code). */
static double normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

static double normal_quantile(double p) { /* bisection on the CDF to the last bit */
    double lo = -40.0, hi = 40.0;
    for (int i = 0; i < 200; i++) {
        double mid = 0.5 * (lo + hi);
        if (normal_cdf(mid) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

void oracle_nf4_levels(double cb[16]) {
    const double d = 0.5 * (1.0 / 32.0 + 1.0 / 30.0), top = 1.0 - d;
    double v[16];
    int n = 0;
    for (int i = 0; i < 7; i++) /* negative: 7 probabilities from 1 - d towards 1/2, step (1/2 - d) / 7 */
        v[n++] = -normal_quantile(top - (0.5 - d) * (double)i / 7.0);
    v[n++] = 0.0;
    for (int i = 0; i < 8; i++) /* positive: 8 probabilities from 1 - d towards 1/2, step (1/2 - d) / 8 */
        v[n++] = normal_quantile(top - (0.5 - d) * (double)i / 8.0);
    const double mx = normal_quantile(top);
    for (int i = 0; i < 16; i++) v[i] /= mx;
    for (int i = 1; i < 16; i++) /* ascending */
        for (int j = i; j > 0 && v[j] < v[j - 1]; j--) { double t = v[j]; v[j] = v[j - 1]; v[j - 1] = t; }
    for (int i = 0; i < 16; i++) cb[i] = v[i];
}

void oracle_int4_levels(double cb[16]) {
    for (int k = -7; k <= 7; k++) cb[k + 7] = (double)k / 7.0;
    cb[15] = 0.0;
}

/* quantise n BF16 weights with a 16-level codebook (FP32 copies of the levels
   are what the decisions and reconstructions use); codes[i] in 0..15,
   scales[n / block rounded up], recon[i] BF16 bits.  Returns bits per weight. */
double oracle_q4_roundtrip(const uint16_t *w, int64_t n, int64_t block, const double levels[16],
                           uint8_t *codes, float *scales, uint16_t *recon) {
    float cb[16];
    for (int k = 0; k < 16; k++) cb[k] = (float)levels[k];
    for (int64_t b0 = 0, bi = 0; b0 < n; b0 += block, bi++) {
        const int64_t b1 = b0 + block < n ? b0 + block : n;
        float s = 0.0f;
        for (int64_t i = b0; i < b1; i++) {
            float a = fabsf((float)oracle_bf16_to_f64(w[i]));
            if (a > s) s = a;
        }
        scales[bi] = s;
        for (int64_t i = b0; i < b1; i++) {
            const float x = s > 0.0f ? (float)oracle_bf16_to_f64(w[i]) / s : 0.0f;
            int best = 0;
            float bd = fabsf(x - cb[0]);
            for (int k = 1; k < 16; k++) {
                const float dk = fabsf(x - cb[k]);
                if (dk < bd) { bd = dk; best = k; }
            }
            codes[i] = (uint8_t)best;
            recon[i] = oracle_f32_to_bf16(cb[best] * s);
        }
    }
    return 4.0 + 32.0 / (double)block;
}

/* E4M3 value of a byte: bias 7, 3 mantissa bits, subnormals at exponent 0,
   S.1111.111 is NaN (never produced by the satfinite conversion) */
double oracle_e4m3_to_f64(uint8_t b) {
    const int e = (b >> 3) & 0xF, m = b & 7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, e - 7);
    if (e == 15 && m == 7) v = NAN;
    return (b & 0x80) ? -v : v;
}

/* FP8 comparator: per-row scale t = max|w| / 448 (FP32), w / t rounded to E4M3
   (satfinite), reconstruction BF16(e4m3 * t).  8 + 32 / K bits per weight.
   codes (M*K bytes) and scales (M floats) may be NULL. */
double oracle_fp8_row_roundtrip(const uint16_t *w, int64_t M, int64_t K, uint16_t *recon, uint8_t *codes,
                                float *scales) {
    for (int64_t r = 0; r < M; r++) {
        float s = 0.0f;
        for (int64_t c = 0; c < K; c++) {
            float a = fabsf((float)oracle_bf16_to_f64(w[r * K + c]));
            if (a > s) s = a;
        }
        const float t = s / 448.0f;
        if (scales) scales[r] = t;
        for (int64_t c = 0; c < K; c++) {
            const float x = t > 0.0f ? (float)oracle_bf16_to_f64(w[r * K + c]) / t : 0.0f;
            const uint8_t q = oracle_f32_to_e4m3_satfinite(x);
            if (codes) codes[r * K + c] = q;
            recon[r * K + c] = oracle_f32_to_bf16((float)oracle_e4m3_to_f64(q) * t);
        }
    }
    return 8.0 + 32.0 / (double)K;
}
