// Host encoder of the EntroPack stream (format version 1), multithreaded.
//
// Steps, in the order of the method ("EntroPack: Fast and Accurate
// Entropy-Coded Weight Compression at Arbitrary Bitrates", Abstract):
//   1. row normalisation: per-row RMS s_r, step g_r = RN7(s_r * Delta_j);
//   2. sampled storage estimate: entropy of the coded symbols on a strided row
//      sample, bisected over the log grid Delta_j = 2^(j/64) towards target_bpp;
//   3. E8 lattice quantisation of every 8-block of w / g_r (Conway-Sloane);
//   4. conditional model: (coset, a0) jointly, coordinates 1..6 given the
//      coset, the parity-reduced last coordinate given the coset;
//   5. 12-bit frequency tables over the whole tensor;
//   6. rANS in independently decodable 32 x 128 tiles, 4 interleaved lanes.
// Every floating-point step follows the exact operation order that stream
// format version 1 fixes, so that the bytes equal those of any other conforming encoder;
// the sources are compiled with -ffp-contract=off.
#include <algorithm>
#include <climits>
#include <map>
#include <memory>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "ep_format.hpp"

namespace ep {
namespace {

// ----------------------------------------------------------------- threads
template <typename F>
void parallel_for(int64_t n, int threads, F&& fn) {
    if (n <= 0) return;
    threads = (int)std::max<int64_t>(1, std::min<int64_t>(threads, n));
    if (threads == 1) {
        fn(0, n, 0);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(threads);
    for (int t = 0; t < threads; t++)
        pool.emplace_back([&, t] { fn(n * t / threads, n * (t + 1) / threads, t); });
    for (auto& th : pool) th.join();
}

inline double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// --------------------------------------------------------------- row steps
inline double delta_of(int j) { return std::exp2((double)j / 64.0); }

// round v > 0 to 7 significant bits: nearest-even (RN7) or toward zero (TR7)
inline double round7(double v, bool nearest) {
    int e = 0;
    double m = std::frexp(v, &e);
    double s = m * 128.0;
    return std::ldexp(nearest ? std::rint(s) : std::floor(s), e - 7);
}

inline double step_of(double s, int j) {
    if (s == 0.0) return 0.0;
    double g = round7(s * delta_of(j), true);
    const double lo = std::ldexp(1.0, -120), hi = std::ldexp(1.0, 120);
    return g < lo ? lo : (g > hi ? hi : g);
}

// ------------------------------------------------------------ E8 quantiser
// Closest point of the coset D8 + h (h = 0 or 1/2) to v: round each
// coordinate; if the integer sum is odd, re-round the worst coordinate the
// other way (Conway & Sloane's D_n decoder).  Returns the squared distance.
inline double nearest_d8(const double* v, double h, int64_t* out) {
    double y[8];
    int64_t sum = 0;
    for (int i = 0; i < 8; i++) {
        y[i] = v[i] - h;
        out[i] = (int64_t)std::floor(y[i] + 0.5);
        sum += out[i];
    }
    if (sum & 1) {
        int k = 0;
        double worst = -1.0;
        for (int i = 0; i < 8; i++) {
            double e = std::fabs(y[i] - (double)out[i]);
            if (e > worst) {
                worst = e;
                k = i;
            }
        }
        out[k] += (y[k] >= (double)out[k]) ? 1 : -1;
    }
    double d = 0.0;
    for (int i = 0; i < 8; i++) {
        double e = y[i] - (double)out[i];
        d += e * e;
    }
    return d;
}

// E8 = D8 u (D8 + 1/2); ties keep the integer coset.
inline int quantise_e8(const double* x, int64_t* a) {
    int64_t A[8], B[8];
    double d0 = nearest_d8(x, 0.0, A);
    double d1 = nearest_d8(x, 0.5, B);
    const bool half = d1 < d0;
    std::memcpy(a, half ? B : A, sizeof(A));
    return half ? 1 : 0;
}

// ----------------------------------------------------------------- symbols
struct BlockCode {
    uint8_t u[8];      // coded bytes
    int16_t esc[8];    // escape payloads (valid where escaped)
    uint8_t n_esc;
    uint8_t coset;
};

// symbol values: k_i = 2 a_i + c (i < 7), w = 4 v7 + c with v7 = (a7 - p) / 2
inline void code_block(const int64_t* a, int c, BlockCode* bc, bool* overflow) {
    int64_t par = 0;
    for (int i = 0; i < 7; i++) par += a[i];
    par &= 1;
    bc->coset = (uint8_t)c;
    bc->n_esc = 0;
    for (int i = 0; i < 8; i++) {
        int64_t v = (i < 7) ? 2 * a[i] + c : 4 * ((a[7] - par) / 2) + c;
        int64_t lo = (i == 0) ? -126 : -127;
        int64_t hi = (i == 7) ? 125 : 127;
        if (v >= lo && v <= hi) {
            bc->u[i] = (uint8_t)(v + 128);
            bc->esc[i] = 0;
        } else {
            if (v < -32768 || v > 32767) *overflow = true;
            bc->u[i] = (uint8_t)(i == 0 ? c : 0);
            bc->esc[i] = (int16_t)v;
            bc->n_esc++;
        }
    }
}

inline int context_of(int i, int c) { return i == 0 ? 0 : (i < 7 ? 1 + c : 3 + c); }

struct RowInfo {
    std::vector<double> rms, peak;
};

// ----------------------------------------------------- 12-bit normaliser
void normalise_counts(const uint64_t* n, uint32_t* f) {
    uint64_t total = 0;
    for (int u = 0; u < 256; u++) total += n[u];
    std::fill(f, f + 256, 0u);
    if (total == 0) return;
    int64_t sum = 0;
    for (int u = 0; u < 256; u++) {
        if (!n[u]) continue;
        uint64_t v = (uint64_t)(((unsigned __int128)kProbScale * n[u]) / total);
        f[u] = (uint32_t)std::max<uint64_t>(1, v);
        sum += f[u];
    }
    if (sum < (int64_t)kProbScale) {
        int top = -1;
        for (int u = 0; u < 256; u++)
            if (n[u] && (top < 0 || n[u] > n[top])) top = u;
        f[top] += (uint32_t)(kProbScale - sum);
    }
    while (sum > (int64_t)kProbScale) {
        int top = -1;
        for (int u = 0; u < 256; u++)
            if (f[u] > 1 && (top < 0 || f[u] > f[top])) top = u;
        f[top]--;
        sum--;
    }
    for (int u = 0; u < 256; u++)
        if (f[u] == kProbScale) {
            f[u] = kProbScale - 1;
            f[(u + 1) & 255] = 1;
            break;
        }
}

// --------------------------------------------------------------- rANS lane
struct SymTable {
    uint32_t f[8][256];
    uint32_t cum[8][256];
};

// Encode one lane (symbols given with their contexts, decode order).  Words
// come out in decode order; returns false if a symbol has f == 0.
bool rans_lane(const uint8_t* sym, const uint8_t* ctx, int n, const SymTable& T, uint32_t* state,
               std::vector<uint16_t>& words) {
    words.clear();
    uint32_t x = kRansL;
    for (int i = n - 1; i >= 0; i--) {
        const uint32_t f = T.f[ctx[i]][sym[i]];
        if (!f) return false;
        const uint64_t bound = (uint64_t)f << 20;
        while ((uint64_t)x >= bound) {
            words.push_back((uint16_t)x);
            x >>= 16;
        }
        x = (x / f) * kProbScale + (x % f) + T.cum[ctx[i]][sym[i]];
    }
    std::reverse(words.begin(), words.end());
    *state = x;
    return true;
}

// tile block b -> (row in tile, first column in tile)
inline void tile_block(int b, int* r, int* c) {
    const int slab = b >> 7, rem = b & 127;
    *r = rem >> 2;
    *c = 32 * slab + 8 * (rem & 3);
}

inline uint64_t up16(uint64_t v) { return (v + 15) & ~(uint64_t)15; }

// ------------------------------------------------------------ blob writer
struct TileBytes {
    std::vector<uint8_t> bytes;
};

struct Writer {
    int mode, container, n_ctx;
    int64_t rows, cols, n_tiles;
    float target_bpp;
    int j;
    uint32_t n_sample;
    const uint32_t (*freq)[256];
    const float* meta;
    uint64_t meta_floats;
};

ep_status write_blob(const Writer& W, std::vector<TileBytes>& tiles, int threads, uint8_t** blob, size_t* out_bytes) {
    uint64_t table_bytes = 0;
    int lo[8], hi[8];
    for (int c = 0; c < W.n_ctx; c++) {
        lo[c] = hi[c] = -1;
        for (int u = 0; u < 256; u++)
            if (W.freq[c][u]) {
                if (lo[c] < 0) lo[c] = u;
                hi[c] = u;
            }
        table_bytes += 4 + (lo[c] < 0 ? 0 : 2ull * (uint64_t)(hi[c] - lo[c] + 1));
    }
    const uint64_t tables_off = kHeaderBytes;
    const uint64_t rowmeta_off = up16(tables_off + table_bytes);
    const uint64_t offsets_off = up16(rowmeta_off + 4 * W.meta_floats);
    const uint64_t payload_off = up16(offsets_off + 8ull * (uint64_t)(W.n_tiles + 1));
    std::vector<uint64_t> off((size_t)W.n_tiles + 1, 0);
    for (int64_t t = 0; t < W.n_tiles; t++) off[t + 1] = off[t] + tiles[t].bytes.size();
    const uint64_t total = payload_off + off[W.n_tiles];
    uint8_t* b = (uint8_t*)std::calloc((size_t)total, 1);
    if (!b) return EP_ERR_NOMEM;
    auto w16 = [&](uint64_t o, uint16_t v) { std::memcpy(b + o, &v, 2); };
    auto w32 = [&](uint64_t o, uint32_t v) { std::memcpy(b + o, &v, 4); };
    auto w64 = [&](uint64_t o, uint64_t v) { std::memcpy(b + o, &v, 8); };
    w32(0, kMagic);
    w16(4, 1);
    b[6] = (uint8_t)W.mode;
    b[7] = (uint8_t)W.container;
    w64(8, (uint64_t)W.rows);
    w64(16, (uint64_t)W.cols);
    w64(24, (uint64_t)W.n_tiles);
    std::memcpy(b + 32, &W.target_bpp, 4);
    w32(36, (uint32_t)W.j);
    const double d = W.mode == 0 ? delta_of(W.j) : 0.0;
    std::memcpy(b + 40, &d, 8);
    w16(48, kTileRows);
    w16(50, kTileCols);
    b[52] = kLanes;
    b[53] = (uint8_t)W.n_ctx;
    w64(56, tables_off);
    w64(64, rowmeta_off);
    w64(72, offsets_off);
    w64(80, payload_off);
    w64(88, total);
    w32(96, W.n_sample);
    uint64_t p = tables_off;
    for (int c = 0; c < W.n_ctx; c++) {
        if (lo[c] < 0) {
            p += 4;  // lo = n = 0 (already zero)
            continue;
        }
        w16(p, (uint16_t)lo[c]);
        w16(p + 2, (uint16_t)(hi[c] - lo[c] + 1));
        p += 4;
        for (int u = lo[c]; u <= hi[c]; u++, p += 2) w16(p, (uint16_t)W.freq[c][u]);
    }
    if (W.meta_floats) std::memcpy(b + rowmeta_off, W.meta, 4 * W.meta_floats);
    for (int64_t t = 0; t <= W.n_tiles; t++) w64(offsets_off + 8ull * (uint64_t)t, off[t]);
    parallel_for(W.n_tiles, threads, [&](int64_t t0, int64_t t1, int) {
        for (int64_t t = t0; t < t1; t++)
            std::memcpy(b + payload_off + off[t], tiles[t].bytes.data(), tiles[t].bytes.size());
    });
    *blob = b;
    *out_bytes = (size_t)total;
    return EP_OK;
}

// tile payload from (raw?, lane states, lane words)
void pack_tile(const uint8_t* raw, size_t raw_len, const uint32_t* st, std::vector<uint16_t>* words,
               TileBytes& out) {
    uint64_t n = (raw ? raw_len : 0) + kTileHeaderBytes;
    for (int l = 0; l < kLanes; l++) n += 2 * words[l].size();
    out.bytes.assign(up16(n), 0);
    uint8_t* p = out.bytes.data();
    if (raw) {
        std::memcpy(p, raw, raw_len);
        p += raw_len;
    }
    for (int l = 0; l < kLanes; l++, p += 4) std::memcpy(p, &st[l], 4);
    for (int l = 0; l < kLanes; l++, p += 2) {
        uint16_t c = (uint16_t)words[l].size();
        std::memcpy(p, &c, 2);
    }
    for (int l = 0; l < kLanes; l++) {
        std::memcpy(p, words[l].data(), 2 * words[l].size());
        p += 2 * words[l].size();
    }
}

// ------------------------------------------------------------ lossy encode
class LossyEncoder {
   public:
    // w: the matrix padded with zeros to whole tiles (M x K, both multiples of
    // the tile); Mt x Kt: the true shape, which alone enters the row statistics,
    // the rate estimate and the header
    LossyEncoder(const uint16_t* w, int64_t M, int64_t K, int64_t Mt, int64_t Kt, const ep_params& p, int threads)
        : w_(w), M_(M), K_(K), Mt_(Mt), Kt_(Kt), p_(p), threads_(threads) {}

    static constexpr int kSelectJ = -100000;  // run(): choose j by the rate search

    // pieces of the rate search, used on their own by the model-level allocation
    void prepare() { row_stats(); }
    int smallest_admissible() const {
        int lo = kJMin, hi = kJMax;
        if (admissible(lo)) return lo;
        while (hi - lo > 1) {
            const int mid = lo + (hi - lo) / 2;
            (admissible(mid) ? hi : lo) = mid;
        }
        return hi;
    }
    double estimate_at(int j) const { return estimate(j); }

    ep_status run(uint8_t** blob, size_t* bytes, int forced_j = kSelectJ) {
        row_stats();
        int j;
        if (forced_j == kSelectJ) {
            j = choose_j();
        } else {
            if (forced_j > kJMax || forced_j < smallest_admissible()) return EP_ERR_INVALID_ARG;
            j = forced_j;
        }
        g_.assign((size_t)M_, 0.f);
        for (int64_t r = 0; r < M_; r++) g_[r] = (float)step_of(rows_.rms[r], j);
        ep_status st = quantise_all();
        if (st != EP_OK) return st;
        for (int c = 0; c < kLossyContexts; c++) normalise_counts(counts_[c], T_.f[c]);
        for (int u = 0; u < 256; u++) T_.f[kLossyContexts][u] = 16;  // uniform escape bytes
        for (int c = 0; c < 8; c++) {
            uint32_t acc = 0;
            for (int u = 0; u < 256; u++) {
                T_.cum[c][u] = acc;
                acc += T_.f[c][u];
            }
        }
        std::vector<TileBytes> tiles((size_t)(M_ / kTileRows) * (size_t)(K_ / kTileCols));
        st = encode_tiles(tiles);
        if (st != EP_OK) return st;
        std::vector<float> meta(g_.begin(), g_.end());
        if (p_.container == EP_C_FP8_E4M3 || p_.container == EP_C_INT8) {
            meta.insert(meta.end(), mult_.begin(), mult_.end());
            meta.insert(meta.end(), tscale_.begin(), tscale_.end());
        }
        Writer W{0, p_.container, kLossyContexts, Mt_, Kt_, (int64_t)tiles.size(), p_.target_bpp, j,
                 (uint32_t)sample_rows(), T_.f, meta.data(), (uint64_t)meta.size()};
        return write_blob(W, tiles, threads_, blob, bytes);
    }

   private:
    const uint16_t* w_;
    int64_t M_, K_;    // padded shape (row stride K_)
    int64_t Mt_, Kt_;  // true shape
    ep_params p_;
    int threads_;
    RowInfo rows_;
    std::vector<float> g_, mult_, tscale_;
    std::vector<BlockCode> codes_;  // one per 8-block, row-major
    uint64_t counts_[kLossyContexts][256] = {{0}};
    SymTable T_{};

    // RMS and peak of each true row over its true columns; padding rows stay 0
    void row_stats() {
        rows_.rms.assign((size_t)M_, 0.0);
        rows_.peak.assign((size_t)M_, 0.0);
        parallel_for(Mt_, threads_, [&](int64_t r0, int64_t r1, int) {
            for (int64_t r = r0; r < r1; r++) {
                const uint16_t* row = w_ + r * K_;
                double s = 0.0, pk = 0.0;
                for (int64_t k = 0; k < Kt_; k++) {
                    double v = bf16_value(row[k]);
                    s += v * v;
                    pk = std::max(pk, std::fabs(v));
                }
                rows_.rms[r] = std::sqrt(s / (double)Kt_);
                rows_.peak[r] = pk;
            }
        });
    }

    bool admissible(int j) const {
        for (int64_t r = 0; r < M_; r++) {
            if (rows_.rms[r] == 0.0) continue;
            const double g = (double)(float)step_of(rows_.rms[r], j);
            if (!(rows_.peak[r] <= kPeakBound * g)) return false;
        }
        return true;
    }

    int64_t sample_rows() const {
        const double want = std::ceil((double)p_.sample_frac * (double)Mt_);
        int64_t n = want >= 1.0 ? (int64_t)want : 1;
        return std::min<int64_t>(std::max<int64_t>(n, 1), Mt_);
    }

    // bits per parameter of the coded symbols on the row sample at index j
    double estimate(int j) const {
        const int64_t ns = sample_rows();
        const int T = threads_;
        std::vector<uint64_t> hist((size_t)T * kLossyContexts * 256, 0), esc((size_t)T, 0);
        parallel_for(ns, T, [&](int64_t i0, int64_t i1, int t) {
            uint64_t* H = hist.data() + (size_t)t * kLossyContexts * 256;
            for (int64_t i = i0; i < i1; i++) {
                const int64_t r = (int64_t)(((unsigned __int128)i * (uint64_t)Mt_) / (uint64_t)ns);
                const double g = (double)(float)step_of(rows_.rms[r], j);
                for (int64_t k0 = 0; k0 < Kt_; k0 += 8) {
                    BlockCode bc;
                    block(r, k0, g, &bc);
                    esc[t] += bc.n_esc;
                    for (int q = 0; q < 8; q++) H[context_of(q, bc.coset) * 256 + bc.u[q]]++;
                }
            }
        });
        double bits = 0.0;
        uint64_t n_esc = 0;
        for (int t = 0; t < T; t++) n_esc += esc[t];
        for (int c = 0; c < kLossyContexts; c++) {
            uint64_t cnt[256] = {0}, N = 0;
            for (int u = 0; u < 256; u++) {
                for (int t = 0; t < T; t++) cnt[u] += hist[((size_t)t * kLossyContexts + c) * 256 + u];
                N += cnt[u];
            }
            for (int u = 0; u < 256; u++)
                if (cnt[u]) bits += (double)cnt[u] * std::log2((double)N / (double)cnt[u]);
        }
        return (bits + 16.0 * (double)n_esc) / (double)(ns * Kt_);
    }

    int choose_j() const {
        int lo = smallest_admissible(), hi = kJMax;
        const double T = (double)p_.target_bpp;
        const int j_lo = lo;
        double e_lo = estimate(j_lo);
        if (e_lo <= T) return j_lo;
        hi = kJMax;
        double e_hi = estimate(hi);
        if (e_hi > T) return hi;
        while (hi - lo > 1) {
            const int mid = lo + (hi - lo) / 2;
            const double e = estimate(mid);
            if (e <= T) {
                hi = mid;
                e_hi = e;
            } else {
                lo = mid;
                e_lo = e;
            }
        }
        return std::fabs(e_hi - T) <= std::fabs(e_lo - T) ? hi : lo;
    }

    void block(int64_t r, int64_t k0, double g, BlockCode* bc) const {
        int64_t a[8] = {0};
        int c = 0;
        if (g != 0.0) {
            double x[8];
            const uint16_t* src = w_ + r * K_ + k0;
            for (int i = 0; i < 8; i++) x[i] = bf16_value(src[i]) / g;
            c = quantise_e8(x, a);
        }
        bool ovf = false;
        code_block(a, c, bc, &ovf);
    }

    ep_status quantise_all() {
        const int64_t bpr = K_ / 8;
        codes_.resize((size_t)(M_ * bpr));
        mult_.assign((size_t)M_, 1.f);
        tscale_.assign((size_t)M_, 0.f);
        const int T = threads_;
        std::vector<uint64_t> hist((size_t)T * kLossyContexts * 256, 0);
        std::atomic<bool> overflow{false};
        parallel_for(M_, T, [&](int64_t r0, int64_t r1, int t) {
            uint64_t* H = hist.data() + (size_t)t * kLossyContexts * 256;
            for (int64_t r = r0; r < r1; r++) {
                const double g = (double)g_[r];
                double qmax = 0.0;
                for (int64_t b = 0; b < bpr; b++) {
                    int64_t a[8] = {0};
                    int c = 0;
                    if (g != 0.0) {
                        double x[8];
                        const uint16_t* src = w_ + r * K_ + 8 * b;
                        for (int i = 0; i < 8; i++) x[i] = bf16_value(src[i]) / g;
                        c = quantise_e8(x, a);
                    }
                    for (int i = 0; i < 8; i++) qmax = std::max(qmax, std::fabs((double)a[i] + 0.5 * c));
                    BlockCode& bc = codes_[(size_t)(r * bpr + b)];
                    bool ovf = false;
                    code_block(a, c, &bc, &ovf);
                    if (ovf) overflow = true;
                    for (int q = 0; q < 8; q++) H[context_of(q, c) * 256 + bc.u[q]]++;
                }
                double m = 1.0;
                if (qmax > 0.0) {
                    if (p_.container == EP_C_FP8_E4M3) m = round7(448.0 / qmax, false);
                    if (p_.container == EP_C_INT8) m = (2.0 * qmax <= 127.0) ? 2.0 : round7(127.0 / qmax, false);
                }
                mult_[r] = (float)m;
                tscale_[r] = (float)((double)g_[r] / (double)mult_[r]);
            }
        });
        if (overflow) return EP_ERR_UNSUPPORTED;
        for (int t = 0; t < T; t++)
            for (int c = 0; c < kLossyContexts; c++)
                for (int u = 0; u < 256; u++) counts_[c][u] += hist[((size_t)t * kLossyContexts + c) * 256 + u];
        return EP_OK;
    }

    ep_status encode_tiles(std::vector<TileBytes>& tiles) {
        const int64_t tpr = K_ / kTileCols, bpr = K_ / 8;
        std::atomic<bool> bad{false};
        parallel_for((int64_t)tiles.size(), threads_, [&](int64_t t0, int64_t t1, int) {
            std::vector<uint8_t> sym, ctx;
            std::vector<uint16_t> words[kLanes];
            sym.reserve(kBlocksPerLane * 24);
            ctx.reserve(kBlocksPerLane * 24);
            for (int64_t t = t0; t < t1; t++) {
                const int64_t r0 = (t / tpr) * kTileRows, c0 = (t % tpr) * kTileCols;
                uint32_t st[kLanes];
                for (int l = 0; l < kLanes; l++) {
                    sym.clear();
                    ctx.clear();
                    for (int b = l; b < kBlocksPerTile; b += kLanes) {
                        int br, bc;
                        tile_block(b, &br, &bc);
                        const BlockCode& code = codes_[(size_t)((r0 + br) * bpr + (c0 + bc) / 8)];
                        for (int q = 0; q < 8; q++) {
                            sym.push_back(code.u[q]);
                            ctx.push_back((uint8_t)context_of(q, code.coset));
                        }
                        if (code.n_esc)
                            for (int q = 0; q < 8; q++) {
                                const bool e = q == 0 ? code.u[q] <= 1 : code.u[q] == 0;
                                if (!e) continue;
                                const uint16_t P = (uint16_t)code.esc[q];
                                sym.push_back((uint8_t)(P >> 8));
                                ctx.push_back(kLossyContexts);
                                sym.push_back((uint8_t)(P & 0xFF));
                                ctx.push_back(kLossyContexts);
                            }
                    }
                    if (!rans_lane(sym.data(), ctx.data(), (int)sym.size(), T_, &st[l], words[l]) ||
                        words[l].size() > 65535)
                        bad = true;
                }
                pack_tile(nullptr, 0, st, words, tiles[(size_t)t]);
            }
        });
        return bad ? EP_ERR_UNSUPPORTED : EP_OK;
    }
};

// --------------------------------------------------------- lossless encode
// Element split: the coded byte and the raw bytes of one element.
struct LosslessSplit {
    int container, eb, rb;  // element type, element bytes, raw bytes per element
    uint8_t code(const uint8_t* x, uint8_t* raw) const {
        if (container == EP_C_FP8_E4M3) return x[0];
        if (container == EP_C_FP32) {
            uint32_t v;
            std::memcpy(&v, x, 4);
            raw[0] = (uint8_t)(((v >> 24) & 0x80u) | ((v >> 16) & 0x7Fu));
            raw[1] = (uint8_t)(v >> 8);
            raw[2] = (uint8_t)v;
            return (uint8_t)(v >> 23);
        }
        uint16_t v;
        std::memcpy(&v, x, 2);
        raw[0] = (uint8_t)(((v >> 8) & 0x80u) | (v & 0x7Fu));
        return (uint8_t)(v >> 7);
    }
};

// w: the matrix padded to whole tiles (M x K elements of `container`);
// Mt x Kt: the true shape (header only)
ep_status encode_lossless(const uint8_t* w, int64_t M, int64_t K, int64_t Mt, int64_t Kt, int container,
                         int threads, uint8_t** blob, size_t* bytes) {
    const LosslessSplit sp{container, (int)container_bytes(container), lossless_raw_per_elem(container)};
    std::vector<uint64_t> hist((size_t)threads * 256, 0);
    parallel_for(M, threads, [&](int64_t r0, int64_t r1, int t) {
        uint64_t* H = hist.data() + (size_t)t * 256;
        uint8_t scratch[3];
        for (int64_t i = r0 * K; i < r1 * K; i++) H[sp.code(w + (size_t)i * sp.eb, scratch)]++;
    });
    uint64_t cnt[256] = {0};
    for (int t = 0; t < threads; t++)
        for (int u = 0; u < 256; u++) cnt[u] += hist[(size_t)t * 256 + u];
    SymTable T{};
    normalise_counts(cnt, T.f[0]);
    uint32_t acc = 0;
    for (int u = 0; u < 256; u++) {
        T.cum[0][u] = acc;
        acc += T.f[0][u];
    }
    const int64_t tpr = K / kTileCols, n_tiles = (M / kTileRows) * tpr;
    const size_t raw_len = (size_t)sp.rb * 4096;
    std::vector<TileBytes> tiles((size_t)n_tiles);
    parallel_for(n_tiles, threads, [&](int64_t t0, int64_t t1, int) {
        std::vector<uint8_t> raw(raw_len ? raw_len : 1);
        uint8_t sym[kBlocksPerLane * 8], ctx[kBlocksPerLane * 8] = {0}, scratch[3];
        std::vector<uint16_t> words[kLanes];
        for (int64_t t = t0; t < t1; t++) {
            const int64_t r0 = (t / tpr) * kTileRows, c0 = (t % tpr) * kTileCols;
            for (int b = 0; b < kBlocksPerTile; b++) {
                int br, bc;
                tile_block(b, &br, &bc);
                const uint8_t* src = w + (size_t)((r0 + br) * K + c0 + bc) * sp.eb;
                for (int q = 0; q < 8; q++) sp.code(src + (size_t)q * sp.eb, raw.data() + (size_t)sp.rb * (8 * b + q));
            }
            uint32_t st[kLanes];
            for (int l = 0; l < kLanes; l++) {
                int n = 0;
                for (int b = l; b < kBlocksPerTile; b += kLanes) {
                    int br, bc;
                    tile_block(b, &br, &bc);
                    const uint8_t* src = w + (size_t)((r0 + br) * K + c0 + bc) * sp.eb;
                    for (int q = 0; q < 8; q++) sym[n++] = sp.code(src + (size_t)q * sp.eb, scratch);
                }
                rans_lane(sym, ctx, n, T, &st[l], words[l]);
            }
            pack_tile(sp.rb ? raw.data() : nullptr, raw_len, st, words, tiles[(size_t)t]);
        }
    });
    Writer W{1, container, 1, Mt, Kt, n_tiles, 0.f, 0, 0u, T.f, nullptr, 0};
    return write_blob(W, tiles, threads, blob, bytes);
}

}  // namespace
}  // namespace ep

namespace {

bool any_nonfinite_bf16(const uint16_t* w, int64_t rows, int64_t cols, int threads) {
    std::atomic<bool> nonfinite{false};
    ep::parallel_for(rows, threads, [&](int64_t r0, int64_t r1, int) {
        for (int64_t i = r0 * cols; i < r1 * cols; i++)
            if ((w[i] & 0x7F80) == 0x7F80) {
                nonfinite = true;
                return;
            }
    });
    return nonfinite;
}

int thread_count(int32_t requested) {
    const int t = requested > 0 ? requested : (int)std::max(1u, std::thread::hardware_concurrency());
    return std::min(t, 256);
}

ep_status encode_impl(const void* w_in, int64_t rows, int64_t cols, const ep_params* p, int forced_j, uint8_t** blob,
                      size_t* blob_bytes) {
    const uint16_t* w = static_cast<const uint16_t*>(w_in);  // lossy input: BF16 bit patterns
    if (!w || !p || !blob || !blob_bytes) return EP_ERR_INVALID_ARG;
    *blob = nullptr;
    *blob_bytes = 0;
    if (rows <= 0 || cols <= 0 || cols % 8) return EP_ERR_SHAPE;
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 40)) return EP_ERR_SHAPE;
    if (p->mode != EP_MODE_LOSSY_E8 && p->mode != EP_MODE_LOSSLESS_TILEANS) return EP_ERR_INVALID_ARG;
    const int threads = thread_count(p->n_threads);
    try {
        // tiles cover the matrix padded with zeros to whole 32 x 128 tiles
        const int64_t Mp = (rows + ep::kTileRows - 1) / ep::kTileRows * ep::kTileRows;
        const int64_t Kp = (cols + ep::kTileCols - 1) / ep::kTileCols * ep::kTileCols;
        const bool lossless = p->mode == EP_MODE_LOSSLESS_TILEANS;
        if (lossless && !ep::lossless_container_ok(p->container)) return EP_ERR_INVALID_ARG;
        const size_t eb = lossless ? ep::container_bytes(p->container) : sizeof(uint16_t);
        std::vector<uint8_t> padded;
        const uint8_t* wp = static_cast<const uint8_t*>(w_in);
        if (Mp != rows || Kp != cols) {
            padded.assign((size_t)(Mp * Kp) * eb, 0);
            ep::parallel_for(rows, threads, [&](int64_t r0, int64_t r1, int) {
                for (int64_t r = r0; r < r1; r++)
                    std::memcpy(padded.data() + (size_t)(r * Kp) * eb, wp + (size_t)(r * cols) * eb, (size_t)cols * eb);
            });
            wp = padded.data();
        }
        if (lossless) return ep::encode_lossless(wp, Mp, Kp, rows, cols, p->container, threads, blob, blob_bytes);
        if (p->container < EP_C_BF16 || p->container > EP_C_INT8) return EP_ERR_INVALID_ARG;
        if (!(p->target_bpp > 0.f) || !std::isfinite(p->target_bpp)) return EP_ERR_INVALID_ARG;
        ep_params q = *p;
        if (!(q.sample_frac > 0.f) || !std::isfinite(q.sample_frac)) q.sample_frac = 0.05f;
        if (any_nonfinite_bf16(w, rows, cols, threads)) return EP_ERR_NONFINITE;
        ep::LossyEncoder enc(reinterpret_cast<const uint16_t*>(wp), Mp, Kp, rows, cols, q, threads);
        return enc.run(blob, blob_bytes, forced_j);
    } catch (const std::bad_alloc&) {
        return EP_ERR_NOMEM;
    }
}

}  // namespace

extern "C" ep_status ep_encode(const void* w_in, int64_t rows, int64_t cols, const ep_params* p, uint8_t** blob,
                               size_t* blob_bytes) {
    return encode_impl(w_in, rows, cols, p, ep::LossyEncoder::kSelectJ, blob, blob_bytes);
}

extern "C" ep_status ep_encode_at(const void* w, int64_t rows, int64_t cols, const ep_params* p, int32_t j,
                                  uint8_t** blob, size_t* blob_bytes) {
    if (!p || p->mode != EP_MODE_LOSSY_E8) return EP_ERR_INVALID_ARG;
    if (j < ep::kJMin || j > ep::kJMax) return EP_ERR_INVALID_ARG;
    return encode_impl(w, rows, cols, p, j, blob, blob_bytes);
}

extern "C" ep_status ep_estimate_bpp(const uint16_t* w, int64_t rows, int64_t cols, float sample_frac, int32_t j,
                                     int32_t n_threads, double* bpp, int32_t* j_min) {
    if (!w || !bpp) return EP_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || cols % 8 || rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 40))
        return EP_ERR_SHAPE;
    if (j < ep::kJMin || j > ep::kJMax) return EP_ERR_INVALID_ARG;
    const int threads = thread_count(n_threads);
    try {
        if (any_nonfinite_bf16(w, rows, cols, threads)) return EP_ERR_NONFINITE;
        ep_params q{};
        q.sample_frac = sample_frac > 0.f && std::isfinite(sample_frac) ? sample_frac : 0.05f;
        // the rate search reads only true rows and columns: no padding needed
        ep::LossyEncoder enc(w, rows, cols, rows, cols, q, threads);
        enc.prepare();
        *bpp = enc.estimate_at(j);
        if (j_min) *j_min = enc.smallest_admissible();
        return EP_OK;
    } catch (const std::bad_alloc&) {
        return EP_ERR_NOMEM;
    }
}

extern "C" ep_status ep_allocate_bits(const ep_layer_ref* layers, int64_t n_layers, float avg_bpp, float sample_frac,
                                      int32_t n_threads, int32_t* j_out, double* est_bpp_out, int32_t* t_out) {
    if (!layers || !j_out || n_layers <= 0) return EP_ERR_INVALID_ARG;
    if (!(avg_bpp > 0.f) || !std::isfinite(avg_bpp)) return EP_ERR_INVALID_ARG;
    for (int64_t l = 0; l < n_layers; l++) {
        const ep_layer_ref& L = layers[l];
        if (!L.w || !(L.sensitivity > 0.f) || !std::isfinite(L.sensitivity)) return EP_ERR_INVALID_ARG;
        if (L.rows <= 0 || L.cols <= 0 || L.cols % 8 || L.rows > ((int64_t)1 << 40) || L.cols > ((int64_t)1 << 40))
            return EP_ERR_SHAPE;
    }
    const int threads = thread_count(n_threads);
    try {
        ep_params q{};
        q.sample_frac = sample_frac > 0.f && std::isfinite(sample_frac) ? sample_frac : 0.05f;
        const size_t nl = (size_t)n_layers;
        std::vector<std::unique_ptr<ep::LossyEncoder>> enc(nl);
        std::vector<int> jmin(nl), off(nl);
        std::vector<std::map<int, double>> memo(nl);
        double n_total = 0.0;
        for (size_t l = 0; l < nl; l++) {
            const ep_layer_ref& L = layers[l];
            if (any_nonfinite_bf16(L.w, L.rows, L.cols, threads)) return EP_ERR_NONFINITE;
            enc[l].reset(new ep::LossyEncoder(L.w, L.rows, L.cols, L.rows, L.cols, q, threads));
            enc[l]->prepare();
            jmin[l] = enc[l]->smallest_admissible();
            // equal Lagrangian slopes: alpha * Delta^2 constant, Delta_j = 2^(j / 64)
            off[l] = (int)std::lround(32.0 * std::log2((double)L.sensitivity));
            n_total += (double)(L.rows * L.cols);
        }
        auto j_of = [&](size_t l, int t) { return std::min(std::max(t - off[l], jmin[l]), ep::kJMax); };
        auto est = [&](size_t l, int j) {
            auto it = memo[l].find(j);
            if (it != memo[l].end()) return it->second;
            const double e = enc[l]->estimate_at(j);
            memo[l][j] = e;
            return e;
        };
        auto total = [&](int t) {
            double e = 0.0;
            for (size_t l = 0; l < nl; l++) e += (double)(layers[l].rows * layers[l].cols) * est(l, j_of(l, t));
            return e;
        };
        const double budget = (double)avg_bpp * n_total;
        int t_lo = INT32_MAX, t_hi = INT32_MIN;
        for (size_t l = 0; l < nl; l++) {
            t_lo = std::min(t_lo, jmin[l] + off[l]);
            t_hi = std::max(t_hi, ep::kJMax + off[l]);
        }
        int t;
        if (total(t_lo) <= budget) {
            t = t_lo;
        } else if (total(t_hi) > budget) {
            t = t_hi;
        } else {
            int lo = t_lo, hi = t_hi;  // total(lo) > budget >= total(hi)
            while (hi - lo > 1) {
                const int mid = lo + (hi - lo) / 2;
                (total(mid) <= budget ? hi : lo) = mid;
            }
            t = hi;
        }
        for (size_t l = 0; l < nl; l++) {
            j_out[l] = j_of(l, t);
            if (est_bpp_out) est_bpp_out[l] = est(l, j_out[l]);
        }
        if (t_out) *t_out = t;
        return EP_OK;
    } catch (const std::bad_alloc&) {
        return EP_ERR_NOMEM;
    }
}
