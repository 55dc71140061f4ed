// Host-side stream parsing and validation, info queries and status strings.
// A stream is validated completely before any kernel is launched, so that a
// corrupt or truncated blob ends the call with a clear error instead of a
// half-converted tensor ("EntroPack PyTorch Guide", "Test saved artifacts and
// reloads before deployment": a partial failure ends in a clear error;
// "Diagnose compression failures in the correct order": the stored object must
// hold everything the decoder reads).
#include <cstdlib>
#include <cstring>
#include <new>

#include "ep_format.hpp"

namespace ep {
namespace {

template <typename T>
T rd(const uint8_t* p) {
    T v;
    std::memcpy(&v, p, sizeof(T));  // little-endian host (x86-64 / aarch64)
    return v;
}

}  // namespace

ep_status parse_and_validate(const uint8_t* b, size_t bytes, Layout* L) {
    if (!b || !L) return EP_ERR_INVALID_ARG;
    if (bytes < (size_t)kHeaderBytes) return EP_ERR_CORRUPT;
    if (rd<uint32_t>(b) != kMagic || rd<uint16_t>(b + 4) != 1) return EP_ERR_CORRUPT;
    L->mode = b[6];
    L->container = b[7];
    L->rows = (int64_t)rd<uint64_t>(b + 8);
    L->cols = (int64_t)rd<uint64_t>(b + 16);
    L->n_tiles = (int64_t)rd<uint64_t>(b + 24);
    L->target_bpp = rd<float>(b + 32);
    L->j = rd<int32_t>(b + 36);
    L->delta = rd<double>(b + 40);
    if (L->mode > 1 || (L->mode == 0 && L->container > 3) || (L->mode == 1 && !lossless_container_ok(L->container)))
        return EP_ERR_CORRUPT;
    if (L->rows <= 0 || L->cols <= 0 || L->cols % 8) return EP_ERR_CORRUPT;
    if (L->rows > (int64_t)1 << 40 || L->cols > (int64_t)1 << 40) return EP_ERR_CORRUPT;
    L->rows_p = (L->rows + kTileRows - 1) / kTileRows * kTileRows;
    L->cols_p = (L->cols + kTileCols - 1) / kTileCols * kTileCols;
    if (L->n_tiles != (L->rows_p / kTileRows) * (L->cols_p / kTileCols)) return EP_ERR_CORRUPT;
    if (rd<uint16_t>(b + 48) != kTileRows || rd<uint16_t>(b + 50) != kTileCols || b[52] != kLanes) return EP_ERR_CORRUPT;
    L->n_ctx = b[53];
    if (L->n_ctx != (L->mode == 0 ? kLossyContexts : 1)) return EP_ERR_CORRUPT;
    L->tables_off = rd<uint64_t>(b + 56);
    L->rowmeta_off = rd<uint64_t>(b + 64);
    L->offsets_off = rd<uint64_t>(b + 72);
    L->payload_off = rd<uint64_t>(b + 80);
    L->total = rd<uint64_t>(b + 88);
    L->n_sample_rows = rd<uint32_t>(b + 96);
    if (L->total != bytes || L->tables_off != (uint64_t)kHeaderBytes) return EP_ERR_CORRUPT;
    if (!(L->tables_off <= L->rowmeta_off && L->rowmeta_off <= L->offsets_off && L->offsets_off <= L->payload_off &&
          L->payload_off <= L->total))
        return EP_ERR_CORRUPT;
    if ((L->rowmeta_off | L->offsets_off | L->payload_off) & 15u) return EP_ERR_CORRUPT;

    // context tables
    std::memset(L->freq, 0, sizeof(L->freq));
    uint64_t p = L->tables_off;
    for (int c = 0; c < L->n_ctx; c++) {
        if (p + 4 > L->rowmeta_off) return EP_ERR_CORRUPT;
        L->ctx_off[c] = p;
        uint32_t lo = rd<uint16_t>(b + p), n = rd<uint16_t>(b + p + 2);
        p += 4;
        if (lo + n > 256 || p + 2ull * n > L->rowmeta_off) return EP_ERR_CORRUPT;
        uint32_t sum = 0;
        for (uint32_t i = 0; i < n; i++) {
            uint32_t f = rd<uint16_t>(b + p + 2ull * i);
            if (f > kProbScale - 1) return EP_ERR_CORRUPT;  // format keeps every f in 12 bits
            L->freq[c][lo + i] = f;
            sum += f;
        }
        p += 2ull * n;
        if (!(sum == kProbScale || (sum == 0 && n == 0))) return EP_ERR_CORRUPT;
    }

    // row metadata and tile offsets
    const uint64_t meta_floats =
        L->mode == 1 ? 0 : (uint64_t)L->rows_p * (L->container >= EP_C_FP8_E4M3 ? 3u : 1u);
    if (L->rowmeta_off + 4 * meta_floats > L->offsets_off) return EP_ERR_CORRUPT;
    if (L->offsets_off + 8ull * (uint64_t)(L->n_tiles + 1) > L->payload_off) return EP_ERR_CORRUPT;
    const uint64_t payload = L->total - L->payload_off;
    const uint64_t raw_bytes = L->mode == 1 ? 4096u * (uint64_t)lossless_raw_per_elem(L->container) : 0u;
    const uint64_t min_tile = raw_bytes + (uint64_t)kTileHeaderBytes;
    uint64_t prev = rd<uint64_t>(b + L->offsets_off);
    if (prev != 0) return EP_ERR_CORRUPT;
    for (int64_t t = 0; t < L->n_tiles; t++) {
        uint64_t nxt = rd<uint64_t>(b + L->offsets_off + 8ull * (uint64_t)(t + 1));
        if ((nxt & 15u) || nxt < prev + min_tile || nxt > payload) return EP_ERR_CORRUPT;
        const uint8_t* th = b + L->payload_off + prev + raw_bytes;
        uint64_t words = 0;
        for (int l = 0; l < kLanes; l++) words += rd<uint16_t>(th + 16 + 2 * l);
        if (min_tile + 2 * words > nxt - prev) return EP_ERR_CORRUPT;
        prev = nxt;
    }
    if (prev != payload) return EP_ERR_CORRUPT;
    return EP_OK;
}

}  // namespace ep

extern "C" {

int32_t ep_version(void) { return 1; }

const char* ep_status_string(ep_status s) {
    switch (s) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_SHAPE: return "unsupported shape (empty, or cols not a multiple of 8)";
        case EP_ERR_NONFINITE: return "non-finite input to a lossy encode";
        case EP_ERR_CORRUPT: return "corrupt stream";
        case EP_ERR_UNSUPPORTED: return "value range outside format version 1";
        case EP_ERR_NOMEM: return "out of host memory";
        case EP_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

void ep_free(void* p) { std::free(p); }

ep_status ep_query(const uint8_t* blob, size_t bytes, ep_info* out) {
    if (!out) return EP_ERR_INVALID_ARG;
    auto* L = new (std::nothrow) ep::Layout();
    if (!L) return EP_ERR_NOMEM;
    ep_status st = ep::parse_and_validate(blob, bytes, L);
    if (st == EP_OK) {
        out->rows = L->rows;
        out->cols = L->cols;
        out->n_tiles = L->n_tiles;
        out->mode = L->mode;
        out->container = L->container;
        out->target_bpp = L->target_bpp;
        out->j = L->j;
        out->delta = L->delta;
        out->total_bytes = L->total;
        out->n_sample_rows = L->n_sample_rows;
        out->actual_bpp = 8.0 * (double)L->total / ((double)L->rows * (double)L->cols);
        out->out_elem_bytes = ep::container_bytes(L->container);
        out->has_row_scale = (L->mode == 0 && L->container >= EP_C_FP8_E4M3) ? 1 : 0;
    }
    delete L;
    return st;
}

ep_status ep_actual_bpp(const uint8_t* blob, size_t bytes, double* bpp) {
    if (!bpp) return EP_ERR_INVALID_ARG;
    ep_info info;
    ep_status st = ep_query(blob, bytes, &info);
    if (st == EP_OK) *bpp = info.actual_bpp;
    return st;
}

// Validated stream handles: the layout parsed once, launched many times.
ep_status ep_stream_open(const uint8_t* h_blob, size_t bytes, ep_stream_handle** out) {
    if (!h_blob || !out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    ep_stream_handle* h = new (std::nothrow) ep_stream_handle;
    if (!h) return EP_ERR_NOMEM;
    const ep_status st = ep::parse_and_validate(h_blob, bytes, &h->L);
    if (st != EP_OK) {
        delete h;
        return st;
    }
    *out = h;
    return EP_OK;
}

void ep_stream_close(ep_stream_handle* h) { delete h; }

ep_status ep_decode_h(const ep_stream_handle* h, const void* d_blob, void* d_out, float* d_row_scale_out,
                      uint32_t* d_status, ep_stream_t stream) {
    if (!h) return EP_ERR_INVALID_ARG;
    return ep::decode_parsed(h->L, d_blob, d_out, d_row_scale_out, d_status, stream);
}

}  // extern "C"
