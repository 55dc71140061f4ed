// Internal constants and the parsed stream layout of format version 1
// (tile 32 x 128, 4 rANS lanes, 12-bit tables, 16-bit words; any shape with
// cols % 8 == 0, coded as the matrix padded with zeros to whole tiles).  Shared by
// the host encoder, the host validator and the CUDA launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include "entropack.h"

namespace ep {

constexpr int kTileRows = 32;
constexpr int kTileCols = 128;
constexpr int kLanes = 4;
constexpr int kBlocksPerTile = 512;  // 8-wide blocks per tile
constexpr int kBlocksPerLane = 128;
constexpr uint32_t kRansL = 1u << 16;
constexpr int kProbBits = 12;
constexpr uint32_t kProbScale = 1u << kProbBits;
constexpr int kLossyContexts = 5;  // joint (coset, a0); coords | coset; last | coset
constexpr int kHeaderBytes = 128;
constexpr uint32_t kMagic = 0x314B5045u;  // "EPK1"
constexpr int kJMin = -640;
constexpr int kJMax = 128;
constexpr double kPeakBound = 15000.0;
constexpr int kTileHeaderBytes = 24;   // 4 x u32 state + 4 x u16 word counts
constexpr int kRawBytesPerTile = 4096;  // lossless BF16/FP16: one sign+mantissa byte per element

// Lossless element split: raw bytes per element kept uncoded
// (BF16/FP16: 1, FP8: 0, FP32: 3) and element sizes in bytes.
inline int lossless_raw_per_elem(int container) {
    return container == EP_C_FP8_E4M3 ? 0 : (container == EP_C_FP32 ? 3 : 1);
}
inline bool lossless_container_ok(int c) {
    return c == EP_C_BF16 || c == EP_C_FP16 || c == EP_C_FP8_E4M3 || c == EP_C_FP32;
}

// Stream layout after host validation.  All offsets are byte offsets from the
// start of the blob.
struct Layout {
    int mode = 0, container = 0, n_ctx = 0;
    int64_t rows = 0, cols = 0, n_tiles = 0;  // true shape
    int64_t rows_p = 0, cols_p = 0;           // tile grid: the shape padded to whole tiles
    float target_bpp = 0.f;
    int32_t j = 0;
    double delta = 0.0;
    uint32_t n_sample_rows = 0;
    uint64_t tables_off = 0, rowmeta_off = 0, offsets_off = 0, payload_off = 0, total = 0;
    uint64_t ctx_off[8] = {0};  // offset of each context's (lo, n, freq[n]) record
    uint32_t freq[8][256] = {{0}};
};

// Parse and validate every field of a host copy (headers, tables, tile offsets,
// per-tile word counts).  Returns EP_OK or EP_ERR_CORRUPT / EP_ERR_INVALID_ARG.
ep_status parse_and_validate(const uint8_t* blob, size_t bytes, Layout* out);

// Enqueue the decode of a stream that parse_and_validate already accepted into
// L (ep_decode without a second host parse): d_blob holds the same bytes on
// the device; d_out and d_blob are 16-byte aligned; d_status is zeroed first.
ep_status decode_parsed(const Layout& L, const void* d_blob, void* d_out, float* d_row_scale, uint32_t* d_status,
                        ep_stream_t stream);

// Fused CompressedLinear (ep_fused.cu): Y = X W^T (+ b) with W decoded
// straight into shared memory, in passes of fused_tokens_per_pass(cols)
// tokens (0: the shape is not served).  L is a validated lossy BF16 stream;
// the caller has checked pointers and shapes.  d_status is zeroed first.
int64_t fused_tokens_per_pass(int64_t cols);
ep_status fused_linear_parsed(const Layout& L, const void* d_blob, const uint16_t* d_x, int64_t tokens,
                              uint16_t* d_y, const uint16_t* d_bias, uint32_t* d_status, ep_stream_t stream);

inline size_t container_bytes(int container) {
    return container == EP_C_FP32 ? 4 : (container >= EP_C_FP8_E4M3 ? 1 : 2);
}

}  // namespace ep

// the opaque handle of the C ABI: a parsed, validated stream layout
struct ep_stream_handle {
    ep::Layout L;
};
