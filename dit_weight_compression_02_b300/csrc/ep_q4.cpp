// Host side of the fixed-width comparators: the 4-bit codebook levels and
// block-absmax encoder, and the per-row-scaled FP8 E4M3 encoder.
//
// These are the formats EntroPack is measured against ("EntroPack: Fast and
// Accurate Entropy-Coded Weight Compression at Arbitrary Bitrates", Abstract:
// lower relative L2 weight error than NF4 at a 4-bit target, with less
// storage).  A block of `block` consecutive weights keeps its absolute maximum
// s as FP32 and a 4-bit code per weight: the nearest level to w / s, both in
// FP32, ties to the lower code.  The GPU reconstructs BF16(level * s).
//
// NF4 levels: the standard-normal quantiles at 7 negative and 8 positive
// evenly spaced probabilities between 1/2 and 1 - d, d = (1/32 + 1/30) / 2,
// plus an exact zero, divided by the outermost quantile so the extremes are
// +-1.  The quantile here is Newton's method on the normal CDF (std::erfc) in
// long double, started from 0 and iterated to a fixed point.
// INT4 levels: k / 7 for k = -7..7, and a 16th code equal to 0 that the
// nearest search never picks.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "entropack.h"

namespace {

long double phi_cdf(long double x) { return 0.5L * std::erfc(-x / std::sqrt(2.0L)); }

long double phi_pdf(long double x) {
    return std::exp(-0.5L * x * x) / std::sqrt(2.0L * 3.14159265358979323846264338327950288L);
}

long double normal_quantile(long double p) {
    long double x = 0.0L;
    for (int it = 0; it < 100; ++it) {
        const long double step = (phi_cdf(x) - p) / phi_pdf(x);
        x -= step;
        if (std::fabs(step) < 1e-18L * (1.0L + std::fabs(x))) break;
    }
    return x;
}

void nf4_levels(float out[16]) {
    const long double d = 0.5L * (1.0L / 32.0L + 1.0L / 30.0L);
    const long double hi = 1.0L - d, span = 0.5L - d;
    const long double top = normal_quantile(hi);
    long double v[16];
    // ascending: the 7 negative levels from the outermost inwards, zero, then
    // the 8 positive levels from the innermost outwards
    for (int i = 0; i < 7; ++i) v[i] = -normal_quantile(hi - span * (long double)i / 7.0L);
    v[7] = 0.0L;
    for (int i = 0; i < 8; ++i) v[15 - i] = normal_quantile(hi - span * (long double)i / 8.0L);
    for (int i = 0; i < 16; ++i) out[i] = (float)(double)(v[i] / top);
    out[0] = -1.0f;
    out[15] = 1.0f;
}

void int4_levels(float out[16]) {
    for (int k = -7; k <= 7; ++k) out[k + 7] = (float)((double)k / 7.0);
    out[15] = 0.0f;
}

float bf16_value(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// one block: scale and codes (nibble of element i at byte i / 2, low nibble first)
bool encode_block(const uint16_t* w, int64_t lo, int64_t hi, const float* lv, uint8_t* codes, float* scale) {
    float s = 0.0f;
    for (int64_t i = lo; i < hi; ++i) {
        const float a = std::fabs(bf16_value(w[i]));
        if (!std::isfinite(a)) return false;
        if (a > s) s = a;
    }
    *scale = s;
    for (int64_t i = lo; i < hi; ++i) {
        const float x = s > 0.0f ? bf16_value(w[i]) / s : 0.0f;
        int best = 0;
        float bd = std::fabs(x - lv[0]);
        for (int k = 1; k < 16; ++k) {
            const float dk = std::fabs(x - lv[k]);
            if (dk < bd) { bd = dk; best = k; }
        }
        uint8_t& byte = codes[i >> 1];
        byte = (i & 1) ? (uint8_t)((byte & 0x0F) | (best << 4)) : (uint8_t)((byte & 0xF0) | best);
    }
    return true;
}

// E4M3 (bias 7, 3 mantissa bits, subnormals below 2^-6, largest finite 448)
// of a finite float, rounded to nearest even and saturated to +-448
uint8_t e4m3_satfinite(float x) {
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    const float a = std::fabs(x);
    if (a >= 448.0f) return sign | 0x7E;
    if (a < 0.015625f) {  // below 2^-6: multiples of 2^-9, the byte is the multiple (8 = 2^-6)
        const float q = std::nearbyint(a * 512.0f);
        return sign | (uint8_t)q;
    }
    int e2 = 0;
    std::frexp(a, &e2);  // a = f * 2^e2, f in [0.5, 1): the exponent of a is e2 - 1
    const int e = e2 - 1;
    float q = std::nearbyint(std::ldexp(a, 3 - e));  // 8 .. 16 in steps of 2^(e - 3)
    int ee = e;
    if (q >= 16.0f) {
        q = 8.0f;
        ee += 1;
    }
    return sign | (uint8_t)(((ee + 7) << 3) | ((int)q - 8));
}

}  // namespace

extern "C" {

ep_status ep_q4_levels(int32_t kind, float* levels) {
    if (!levels) return EP_ERR_INVALID_ARG;
    if (kind == EP_Q4_NF4) nf4_levels(levels);
    else if (kind == EP_Q4_INT4) int4_levels(levels);
    else return EP_ERR_INVALID_ARG;
    return EP_OK;
}

ep_status ep_q4_encode(const uint16_t* w, int64_t n, int64_t block, const float* levels, uint8_t* codes, float* scales,
                       int32_t n_threads) {
    if (!w || !levels || !codes || !scales) return EP_ERR_INVALID_ARG;
    if (n <= 0 || (n & 1) || n > (int64_t(1) << 40)) return EP_ERR_SHAPE;
    if (block < 16 || block % 16 || block > (int64_t(1) << 30)) return EP_ERR_INVALID_ARG;
    for (int k = 0; k < 16; ++k)
        if (!std::isfinite(levels[k])) return EP_ERR_INVALID_ARG;
    const int64_t n_blocks = (n + block - 1) / block;
    int threads = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
    if (threads < 1) threads = 1;
    if ((int64_t)threads > n_blocks) threads = (int)n_blocks;
    std::vector<char> ok((size_t)threads, 1);
    auto work = [&](int t) {
        // contiguous block ranges; blocks hold an even number of elements, so no
        // two threads touch the same code byte
        const int64_t b0 = n_blocks * t / threads, b1 = n_blocks * (t + 1) / threads;
        for (int64_t b = b0; b < b1 && ok[(size_t)t]; ++b) {
            const int64_t lo = b * block, hi = lo + block < n ? lo + block : n;
            if (!encode_block(w, lo, hi, levels, codes, scales + b)) ok[(size_t)t] = 0;
        }
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < threads; ++t) pool.emplace_back(work, t);
    work(0);
    for (auto& th : pool) th.join();
    for (char c : ok)
        if (!c) return EP_ERR_NONFINITE;
    return EP_OK;
}

ep_status ep_fp8_row_encode(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* codes, float* scales,
                            int32_t n_threads) {
    if (!w || !codes || !scales) return EP_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || cols % 8 || rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
        return EP_ERR_SHAPE;
    int threads = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
    if (threads < 1) threads = 1;
    if ((int64_t)threads > rows) threads = (int)rows;
    std::vector<char> ok((size_t)threads, 1);
    auto work = [&](int t) {
        const int64_t r0 = rows * t / threads, r1 = rows * (t + 1) / threads;
        for (int64_t r = r0; r < r1; ++r) {
            const uint16_t* row = w + r * cols;
            float s = 0.0f;
            for (int64_t c = 0; c < cols; ++c) {
                const float a = std::fabs(bf16_value(row[c]));
                if (!std::isfinite(a)) {
                    ok[(size_t)t] = 0;
                    return;
                }
                if (a > s) s = a;
            }
            const float sc = s / 448.0f;
            scales[r] = sc;
            for (int64_t c = 0; c < cols; ++c)
                codes[r * cols + c] = e4m3_satfinite(sc > 0.0f ? bf16_value(row[c]) / sc : 0.0f);
        }
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < threads; ++t) pool.emplace_back(work, t);
    work(0);
    for (auto& th : pool) th.join();
    for (char c : ok)
        if (!c) return EP_ERR_NONFINITE;
    return EP_OK;
}

}  // extern "C"
