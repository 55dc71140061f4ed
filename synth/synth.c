/*
 * Seeded synthetic inputs shared by the CPU oracle, the GPU tests and the
 * benchmark.  Holds no arithmetic of the codec: it only draws numbers.
 *
 * Every draw is counter based, so any index range can be produced by any
 * thread and the result never depends on the thread count:
 *   u64(seed, stream, n) = mix(key(seed, stream) + (n + 1) * GAMMA)
 * where mix() is the SplitMix64 output function (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and
 * GAMMA = 0x9E3779B97F4A7C15.
 *
 * Normals come from the Box-Muller transform (one uniform pair gives two
 * normals; normal n uses pair n/2, cosine for even n, sine for odd n).
 * Student-t with nu = 5 is Z / sqrt(V/5) with V ~ chi^2(5) built as
 * -2 ln(U1 U2) + Z'^2 (chi^2(4) plus chi^2(1)).
 *
 * Outputs are BF16 bit patterns, rounded to nearest even from the double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * GAMMA + 0x632BE59BD9B4E019ULL) ^ mix64(stream + 0xD1B54A32D192ED03ULL);
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t n) {
    return mix64(stream_key(seed, stream) + (n + 1) * GAMMA);
}

/* uniform in the open interval (0, 1) */
static inline double u01(uint64_t key, uint64_t n) {
    uint64_t v = mix64(key + (n + 1) * GAMMA);
    return ((double)(v >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t n) {
    uint64_t m = n >> 1;
    double u1 = u01(key, 2 * m), u2 = u01(key, 2 * m + 1);
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925 * u2;
    return (n & 1) ? r * sin(t) : r * cos(t);
}

static inline uint16_t bf16_rne(double v) {
    float f = (float)v;
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u) return (uint16_t)(b >> 16) | ((b & 0xFFFF) ? 0x40 : 0);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

/* ---------------------------------------------------------------- threads */
typedef void (*range_fn)(void *ctx, uint64_t lo, uint64_t hi);
typedef struct { range_fn fn; void *ctx; uint64_t lo, hi; } job_t;
static void *job_run(void *p) { job_t *j = (job_t *)p; j->fn(j->ctx, j->lo, j->hi); return NULL; }

static void parallel_range(range_fn fn, void *ctx, uint64_t n, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n < (uint64_t)n_threads * 4096u) n_threads = 1;
    if (n_threads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    job_t jobs[256];
    for (int t = 0; t < n_threads; t++) {
        jobs[t].fn = fn; jobs[t].ctx = ctx;
        jobs[t].lo = n * (uint64_t)t / (uint64_t)n_threads;
        jobs[t].hi = n * (uint64_t)(t + 1) / (uint64_t)n_threads;
        pthread_create(&th[t], NULL, job_run, &jobs[t]);
    }
    for (int t = 0; t < n_threads; t++) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------- normal */
typedef struct { uint64_t key; double mean, std; uint16_t *out; } normal_ctx;
static void normal_range(void *p, uint64_t lo, uint64_t hi) {
    normal_ctx *c = (normal_ctx *)p;
    for (uint64_t i = lo; i < hi; i++) c->out[i] = bf16_rne(c->mean + c->std * normal_at(c->key, i));
}
/* n BF16 values ~ N(mean, std^2) */
void synth_normal_bf16(uint64_t seed, uint64_t n, double mean, double std, uint16_t *out, int n_threads) {
    normal_ctx c = {stream_key(seed, 1), mean, std, out};
    parallel_range(normal_range, &c, n, n_threads);
}

/* n doubles ~ N(0, 1) (used by tests that need real-valued draws) */
typedef struct { uint64_t key; double *out; } normal_f64_ctx;
static void normal_f64_range(void *p, uint64_t lo, uint64_t hi) {
    normal_f64_ctx *c = (normal_f64_ctx *)p;
    for (uint64_t i = lo; i < hi; i++) c->out[i] = normal_at(c->key, i);
}
void synth_normal_f64(uint64_t seed, uint64_t n, double *out, int n_threads) {
    normal_f64_ctx c = {stream_key(seed, 1), out};
    parallel_range(normal_f64_range, &c, n, n_threads);
}

/* n doubles uniform in (lo, hi) */
void synth_uniform_f64(uint64_t seed, uint64_t n, double lo, double hi, double *out) {
    uint64_t key = stream_key(seed, 7);
    for (uint64_t i = 0; i < n; i++) out[i] = lo + (hi - lo) * u01(key, i);
}

/* ------------------------------------------------------------- student-t */
typedef struct { uint64_t kz, ku; double scale; uint16_t *out; } t5_ctx;
static void t5_range(void *p, uint64_t lo, uint64_t hi) {
    t5_ctx *c = (t5_ctx *)p;
    for (uint64_t i = lo; i < hi; i++) {
        /* normals 2i and 2i+1 share one Box-Muller pair: compute it once */
        double r = sqrt(-2.0 * log(u01(c->kz, 2 * i))), th = 6.283185307179586476925 * u01(c->kz, 2 * i + 1);
        double z = r * cos(th), z2 = r * sin(th);
        double v = -2.0 * log(u01(c->ku, 2 * i) * u01(c->ku, 2 * i + 1)) + z2 * z2;
        c->out[i] = bf16_rne(c->scale * z / sqrt(v / 5.0));
    }
}
/* n BF16 values of a Student-t (nu = 5) scaled to standard deviation std */
void synth_student_t5_bf16(uint64_t seed, uint64_t n, double std, uint16_t *out, int n_threads) {
    t5_ctx c = {stream_key(seed, 2), stream_key(seed, 3), std / sqrt(5.0 / 3.0), out};
    parallel_range(t5_range, &c, n, n_threads);
}

/* ------------------------------------------------- rows with outliers */
typedef struct { uint64_t kz; uint64_t cols; const double *sigma; uint16_t *out; } rows_ctx;
static void rows_range(void *p, uint64_t lo, uint64_t hi) {
    rows_ctx *c = (rows_ctx *)p;
    for (uint64_t i = lo; i < hi; i++) c->out[i] = bf16_rne(c->sigma[i / c->cols] * normal_at(c->kz, i));
}
/*
 * rows x cols BF16 matrix: row r has standard deviation sigma_r drawn
 * log-uniform in [sig_lo, sig_hi]; entries Gaussian; then exactly
 * n_out = round(frac * rows * cols) distinct positions (drawn without
 * replacement) are set to +-k_sigma * sigma_r with a random sign.
 */
int synth_rows_outliers_bf16(uint64_t seed, uint64_t rows, uint64_t cols, double sig_lo, double sig_hi,
                             double frac, double k_sigma, uint16_t *out, int n_threads) {
    uint64_t n = rows * cols;
    double *sigma = (double *)malloc(rows * sizeof(double));
    if (!sigma) return -1;
    uint64_t ks = stream_key(seed, 4);
    double a = log(sig_lo), b = log(sig_hi);
    for (uint64_t r = 0; r < rows; r++) sigma[r] = exp(a + (b - a) * u01(ks, r));
    rows_ctx c = {stream_key(seed, 5), cols, sigma, out};
    parallel_range(rows_range, &c, n, n_threads);
    uint64_t n_out = (uint64_t)llround(frac * (double)n);
    uint8_t *used = (uint8_t *)calloc((n + 7) / 8, 1);
    if (!used) { free(sigma); return -1; }
    uint64_t kp = stream_key(seed, 6), draw = 0;
    for (uint64_t m = 0; m < n_out; m++) {
        uint64_t pos;
        do { pos = mix64(kp + (++draw) * GAMMA) % n; } while (used[pos >> 3] & (1u << (pos & 7)));
        used[pos >> 3] |= (uint8_t)(1u << (pos & 7));
        double sgn = (mix64(kp + (++draw) * GAMMA) & 1) ? 1.0 : -1.0;
        out[pos] = bf16_rne(sgn * k_sigma * sigma[pos / cols]);
    }
    free(used);
    free(sigma);
    return (int)0;
}

/*
 * Overwrite whole rows of a BF16 matrix with special values for the
 * lossless path: kind 0 = +0, 1 = -0, 2 = a repeated constant, 3 =
 * subnormals (exponent 0, random mantissa and sign), 4 = alternating
 * +-inf, 5 = NaNs with random payloads and signs, 6 = the largest
 * finite values of both signs.
 */
void synth_special_row_bf16(uint64_t seed, uint64_t cols, int kind, uint16_t *row) {
    uint64_t key = stream_key(seed, 8 + (uint64_t)kind);
    for (uint64_t k = 0; k < cols; k++) {
        uint64_t r = mix64(key + (k + 1) * GAMMA);
        uint16_t sgn = (uint16_t)((r >> 40) & 1) << 15;
        switch (kind) {
        case 0: row[k] = 0x0000; break;
        case 1: row[k] = 0x8000; break;
        case 2: row[k] = 0x3C4A; break;
        case 3: row[k] = sgn | (uint16_t)(1 + (r % 127)); break;
        case 4: row[k] = (k & 1) ? 0xFF80 : 0x7F80; break;
        case 5: row[k] = sgn | 0x7F80 | (uint16_t)(1 + (r % 127)); break;
        default: row[k] = sgn | 0x7F7F; break;
        }
    }
}
