// GPU decode of EntroPack streams on B300 (sm_103a): fused rANS symbol
// decoding, E8 reconstruction, row rescaling and container conversion
// ("EntroPack: Fast and Accurate Entropy-Coded Weight Compression at Arbitrary
// Bitrates", Abstract: the symbols are decoded and the weight values rebuilt
// in one pass on the GPU; containers BF16, FP16, FP8, INT8).
//
// Work decomposition.  A tile (32 x 128 weights) carries 4 independent rANS
// lanes; thread (tig, l) of a warp runs lane l of tile tig, so one warp
// decodes a group of 8 tiles, and a thread running NL lanes interleaves NL
// groups.  One persistent CTA per SM: 1024 threads of one lane each, or 640
// threads of two lanes each (1280 lanes), share one copy of the stream's slot
// tables in shared memory (one u32 per 12-bit slot); each lane stages its
// 16-bit words in a 64-byte shared-memory ring.
// A lane decodes its 128 blocks of 8 coordinates in the format's order; the
// four lanes of a tile write the four quarters of one 64-byte row segment, so
// every warp-wide 128-bit store covers whole 64-byte units of HBM (a half
// written unit costs a read-modify-write in the memory system).  Escapes
// (values beyond the direct byte range) are rare: the fast path is
// branch-free and a warp-uniform test sends a block with any escape through
// the slow path, which reads the escape payload's words from global memory.
//
// Slot entry: f << 20 | u << 12 | (slot - cum_u), with f the 12-bit frequency
// and u the symbol byte.  One LDS, one shift, one AND and one IMAD advance
// the state.  Reconstruction: for a coordinate u = 2q + 128, the float with
// bits (e & 0xFF000) | bits(1536.0f) has the value 1536 + u/2 = 1600 + q, so
// fma(F, g, -1600 g) is fp32(g * q) rounded once (1600 g is exact because
// the format's row steps and multipliers carry at most 7 significant bits).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "ep_format.hpp"

namespace ep {
namespace {

constexpr int kThreads = 1024;   // threads of a one-lane CTA
// threads of a CTA whose threads run NL lanes each: 1024 x 1 or 640 x 2 (two
// lanes per thread at 20 warps leave the compiler room to interleave them)
__host__ __device__ constexpr int cta_threads(int nl) { return nl == 1 ? kThreads : 640; }
constexpr int kSlabs = 4;        // K-slabs of a tile
constexpr int kSlabCols = 32;    // columns of a K-slab
constexpr int kTilesPerWarp = 8;
constexpr int kSlots = 4096;
constexpr uint32_t kMagicLo = 0x44C00000u;  // 1536.0f: bits 12..19 carry u, worth u/2
constexpr float kMagicLoQ = 1600.0f;        // 1536 + 128/2
constexpr uint32_t kMagicHi = 0x4AC00000u;  // 6291456.0f (spacing 0.5): escape path, any int16 payload
constexpr float kMagicHiQ = 6291520.0f;     // 6291456 + 128/2

// Kernel variants: lossy containers, then lossless streams of 16-bit elements
// (BF16 / FP16: coded bits 14..7, one raw byte), of FP8 elements (the whole
// byte coded) and of FP32 elements (coded exponent, three raw bytes).
enum Kind { K_BF16 = 0, K_FP16 = 1, K_FP8 = 2, K_INT8 = 3, K_LOSSLESS = 4, K_LOSSLESS8 = 5, K_LOSSLESS32 = 6 };

__host__ __device__ constexpr bool is_lossless(int kind) { return kind >= K_LOSSLESS; }
// raw (uncoded) bytes per element and per tile of a lossless kind
__host__ __device__ constexpr uint32_t raw_per_elem(int kind) {
    return kind == K_LOSSLESS ? 1u : (kind == K_LOSSLESS32 ? 3u : 0u);
}

struct DecodeArgs {
    const uint8_t* blob;
    const uint64_t* tile_off;
    const uint8_t* payload;
    uint64_t payload_bytes;
    const float* g;  // row steps
    const float* m;  // FP8/INT8 multipliers
    const float* t;  // FP8/INT8 output scales
    uint32_t ctx_off[8];
    int n_ctx;
    void* out;
    float* scale_out;
    uint8_t* sym_out;
    uint32_t* status;
    int64_t rows, cols, n_tiles;  // true shape (the output is rows x cols, row stride cols)
    int64_t tiles_per_row;        // tiles per row of the padded grid
};

// ---------------------------------------------------------------- tables
// Expand the stream's (lo, n, f[n]) records into 4096-entry slot tables.
// Scratch `fr` / `cu` (n_ctx x 256 u32 each) hold frequencies and cumulative
// frequencies.  Every thread fills slots s = tid, tid + blockDim, ... of each
// context by a binary search for the largest u with cum[u] <= s (that symbol
// has f > 0 and covers s); neighbouring lanes take the same search path, so
// the cum reads broadcast and the table stores are conflict-free.
__device__ void build_tables(const DecodeArgs& a, uint32_t* tab, uint32_t* fr, uint32_t* cu) {
    const int n_ctx = a.n_ctx;
    for (int i = threadIdx.x; i < n_ctx * 256; i += blockDim.x) fr[i] = 0;
    __syncthreads();
    for (int c = 0; c < n_ctx; c++) {
        const uint16_t* rec = reinterpret_cast<const uint16_t*>(a.blob + a.ctx_off[c]);
        // the host validated these records; a device copy that differs from the
        // host copy must still not write outside the table (it then fails the
        // lane end checks)
        const int lo = rec[0] < 256 ? rec[0] : 256;
        const int n = rec[1] < 256 - lo ? rec[1] : 256 - lo;
        for (int i = threadIdx.x; i < n; i += blockDim.x) fr[c * 256 + lo + i] = rec[2 + i] & 0xFFFu;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < n_ctx) {  // exclusive prefix sum of one context per warp
        uint32_t v[8], s = 0;
        for (int k = 0; k < 8; k++) {
            v[k] = fr[warp * 256 + lane * 8 + k];
            s += v[k];
        }
        uint32_t incl = s;
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        uint32_t run = incl - s;
        for (int k = 0; k < 8; k++) {
            cu[warp * 256 + lane * 8 + k] = run;
            run += v[k];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_ctx * kSlots; i += blockDim.x) {
        const int c = i / kSlots;
        const uint32_t s = (uint32_t)(i % kSlots);
        const uint32_t* C = cu + c * 256;
        int u = 0;  // C[0] = 0 <= s; the steps sum to 255, so u + step never passes 255
#pragma unroll
        for (int step = 128; step >= 1; step >>= 1)
            if (C[u + step] <= s) u += step;
        tab[i] = (fr[c * 256 + u] << 20) | ((uint32_t)u << 12) | ((s - C[u]) & 0xFFFu);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- rANS lane
// State x in [2^16, 2^32) before every symbol.  A lane's 16-bit words are
// staged in a private 64-byte ring in shared memory (4 chunks of 16 bytes,
// chunk c of the payload in slot c % 4), filled by cp.async before every
// pair of blocks (top_up).  Every symbol reads the word at the lane's position
// together with its slot-table entry, so the refill never waits on a load
// issued for an earlier symbol: the warp's register scoreboard would
// otherwise stall all 32 lanes on whichever lane refilled last.
constexpr uint32_t kRingChunks = 4;
constexpr uint32_t kRingBytesPerLane = kRingChunks * 16;

extern __shared__ __align__(128) uint32_t g_smem[];  // the decode CTA's dynamic shared memory

struct Lane {
    uint32_t x, next;
    uint32_t a, aend;       // payload byte offsets: next word, one past the lane's last word
    uint32_t issued, clast;  // next chunk to stage, last chunk of the lane (chunk = 16 bytes)
    uint32_t roff;           // byte offset of the lane's 64-byte ring in g_smem (a multiple of 64)
    uint32_t ring;           // shared-window address of the same ring (for cp.async)
    const uint8_t* pay;

    // the 16-bit word at payload offset o (even): slot (o / 16) % 4 of the ring
    __device__ __forceinline__ uint32_t word_at(uint32_t o) const {
        return reinterpret_cast<const uint16_t*>(g_smem)[(roff | (o & (kRingBytesPerLane - 2u))) >> 1];
    }

    __device__ __forceinline__ void stage_chunk() {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ring + ((issued % kRingChunks) << 4)),
                     "l"(pay + ((size_t)issued << 4))
                     : "memory");
        issued++;
    }
    // Start a lane at payload offset a0 with n words: stage its first chunks and wait for them.
    __device__ __forceinline__ void start(uint32_t a0, uint32_t n) {
        a = a0;
        aend = a0 + 2u * n;
        issued = a0 >> 4;
        clast = n ? ((aend - 1u) >> 4) : issued - 1u;  // empty lane: clast + 1 == issued, nothing to stage
        const uint32_t target = n ? min(issued + kRingChunks, clast + 1u) : issued;
        while (issued < target) stage_chunk();
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        next = word_at(a);
    }
    // Top-up point (see top_up below): stage at most two chunks for this lane
    // and report whether the coming reads are not yet known to be complete.
    // Top-ups run before every pair of blocks and again after any block that
    // took the escape path (whose payload words are read from global memory,
    // so the lane may have moved past chunks never staged).  Each top-up
    // commits one cp.async group; waiting for every group but the newest then
    // completes every chunk below `old`, the first chunk staged here.  Two
    // blocks without escapes read at most 16 words plus the one word read
    // ahead, payload bytes a .. a + 33, which lie in chunks cpos .. cpos + 2.
    __device__ __forceinline__ bool stage_pair() {
        const uint32_t cpos = a >> 4;
        issued = max(issued, cpos);  // chunks an escape payload skipped are never read
        const uint32_t old = issued;
        const uint32_t target = min(cpos + kRingChunks, clast + 1u);
        if (issued < target) stage_chunk();
        if (issued < target) stage_chunk();
        const uint32_t need = min(cpos + 2u, clast);
        return a < aend && need >= old;
    }
    // slow path: stage everything the ring can hold (the caller then waits for all)
    __device__ __forceinline__ void stage_all() {
        issued = max(issued, a >> 4);
        const uint32_t target = min((a >> 4) + kRingChunks, clast + 1u);
        while (issued < target) stage_chunk();
    }
    // x < 2^16: shift in the prefetched word, then read the following one.  Only
    // lanes that refilled touch shared memory; the new word is first used one
    // symbol later, by which time the load has landed.
    __device__ __forceinline__ void renorm() {
        if (x < kRansL) {
            x = (x << 16) | next;
            a += 2u;
            next = word_at(a);
        }
    }
    // one table symbol; returns the slot entry
    __device__ __forceinline__ uint32_t sym(const uint32_t* tab) {
        const uint32_t e = tab[x & (kProbScale - 1)];
        x = (e >> 20) * (x >> kProbBits) + (e & 0xFFFu);
        renorm();
        return e;
    }
    // one uniform byte (f = 16, cum = 16 * byte) of an escape payload; its
    // renormalisation words come straight from global memory, so the ring
    // need not hold them.  A lane that runs past its last word (a corrupt
    // stream) reads zeros and fails the lane end check.
    __device__ __forceinline__ uint32_t byte() {
        const uint32_t slot = x & (kProbScale - 1);
        x = 16u * (x >> kProbBits) + (slot & 15u);
        if (x < kRansL) {
            x = (x << 16) | next;
            a += 2u;
            next = a < aend ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(pay + a)) : 0u;
        }
        return slot >> 4;
    }
};

// Stage everything the NL lanes' rings can hold and wait for all of it.
template <int NL>
__device__ __forceinline__ void stage_all_wait(Lane (&ln)[NL]) {
#pragma unroll
    for (int i = 0; i < NL; i++) ln[i].stage_all();
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Top-up of the NL lanes a thread decodes, before every pair of blocks (and
// after a block with escapes): one cp.async group per top-up; if any lane of
// the warp might read a chunk that is not known to be complete, stage all and
// wait for everything (rare: lane starts and ends), otherwise wait for every
// group but the one just committed.
template <int NL>
__device__ __forceinline__ void top_up(Lane (&ln)[NL]) {
    bool urgent = false;
#pragma unroll
    for (int i = 0; i < NL; i++) urgent |= ln[i].stage_pair();
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (__any_sync(0xffffffffu, urgent)) {
        stage_all_wait<NL>(ln);
    } else {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
    }
}

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

__device__ __forceinline__ uint32_t sym_byte(uint32_t e) { return (e >> 12) & 0xFFu; }

__device__ __forceinline__ uint32_t pack2(float a, float b, int kind) {
    if (kind == K_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack4_fp8(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t i8(float v) {
    int i = __float2int_rn(v);
    i = max(-127, min(127, i));
    return (uint32_t)i & 0xFFu;
}

__device__ __forceinline__ uint32_t pack4_i8(float a, float b, float c, float d) {
    return i8(a) | (i8(b) << 8) | (i8(c) << 16) | (i8(d) << 24);
}

template <int KIND>
__device__ __forceinline__ void store_block(void* out, int64_t eoff, const float* y) {
    if (KIND == K_BF16 || KIND == K_FP16) {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + eoff) =
            make_uint4(pack2(y[0], y[1], KIND), pack2(y[2], y[3], KIND), pack2(y[4], y[5], KIND),
                       pack2(y[6], y[7], KIND));
    } else if (KIND == K_FP8) {
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) + eoff) =
            make_uint2(pack4_fp8(y[0], y[1], y[2], y[3]), pack4_fp8(y[4], y[5], y[6], y[7]));
    } else {
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) + eoff) =
            make_uint2(pack4_i8(y[0], y[1], y[2], y[3]), pack4_i8(y[4], y[5], y[6], y[7]));
    }
}

__device__ __forceinline__ void dump_syms(uint8_t* sym_out, int64_t eoff, const uint32_t* u) {
    uint2 s;
    s.x = u[0] | (u[1] << 8) | (u[2] << 16) | (u[3] << 24);
    s.y = u[4] | (u[5] << 8) | (u[6] << 16) | (u[7] << 24);
    *reinterpret_cast<uint2*>(sym_out + eoff) = s;
}

// ------------------------------------------------------------- one group
// A warp decodes NL tile groups at once: thread (tig, l) runs rANS lane l of
// tile tig of each group, interleaving the NL independent lanes so that one
// lane's table-load latency overlaps the other's arithmetic.  Every thread
// runs the same number of steps (inactive lanes decode from a dummy state and
// store nothing), so warp votes are always uniform.
template <int KIND>
struct LaneTile {
    bool active;
    const uint8_t* tb;  // tile payload (lossless: raw bytes first)
    int64_t base;       // output element offset of the lane's block in slab 0, tile row 0
    int32_t rows_left;  // true rows of the tile, capped at 32 (blocks in tile rows >= rows_left are padding)
    int64_t col0;       // the lane's first column in slab 0 (blocks at col0 + 32 slab >= cols are padding)
    const float* gr;    // row steps of the tile's rows: gr[row]
    const float* mr;    // FP8/INT8 multipliers: mr[row]
    float gnext;        // row step of the next block (prefetched one block ahead)

    // validate the tile, find the lane's words and start the lane
    __device__ __forceinline__ void setup(const DecodeArgs& a, int64_t grp, Lane& ln, uint32_t ring_off,
                                          uint32_t* status) {
        const int lane = threadIdx.x & 31, l = lane & 3, tig = lane >> 2;
        constexpr uint32_t kRaw = 4096u * raw_per_elem(KIND);
        constexpr uint32_t kHdr = kRaw + kTileHeaderBytes;
        const int64_t tile = grp * kTilesPerWarp + tig;
        active = grp >= 0 && tile < a.n_tiles;
        uint64_t o0 = 0, o1 = 0;
        if (active) {
            o0 = a.tile_off[tile];
            o1 = a.tile_off[tile + 1];
            if (o0 > o1 || o1 > a.payload_bytes || (o0 & 15u) || o1 - o0 < kHdr) {
                if (l == 0) flag(status, EP_STATUS_TILE_BOUNDS);
                active = false;
            }
        }
        tb = a.payload + (active ? o0 : 0);
        const uint8_t* th = tb + kRaw;
        ln.x = kRansL;
        ln.pay = a.payload;
        ln.roff = ring_off;
        ln.ring = (uint32_t)__cvta_generic_to_shared(g_smem) + ring_off;
        uint32_t a0 = 0, nwl = 0;
        if (active) {
            const uint2 nwv = *reinterpret_cast<const uint2*>(th + 16);
            const uint32_t nw[4] = {nwv.x & 0xFFFFu, nwv.x >> 16, nwv.y & 0xFFFFu, nwv.y >> 16};
            const uint32_t total = nw[0] + nw[1] + nw[2] + nw[3];
            uint32_t before = 0;
            for (int i = 0; i < 4; i++) before += (i < l) ? nw[i] : 0u;
            if (kHdr + 2ull * total > o1 - o0) {
                if (l == 0) flag(status, EP_STATUS_TILE_BOUNDS);
                active = false;
            } else {
                ln.x = reinterpret_cast<const uint32_t*>(th)[l];
                a0 = (uint32_t)(th + kTileHeaderBytes + 2u * before - a.payload);
                nwl = l == 0 ? nw[0] : (l == 1 ? nw[1] : (l == 2 ? nw[2] : nw[3]));
            }
        }
        ln.start(a0, nwl);
        const int64_t t = active ? tile : 0;
        const int64_t tr0 = (t / a.tiles_per_row) * kTileRows;
        const int64_t tc0 = (t % a.tiles_per_row) * kTileCols;
        // this lane's block of step j sits at tile row j % 32 and tile column
        // 32 (j / 32) + 8 l: the tile's four lanes write one 64-byte row segment
        const int64_t row0 = tr0;
        rows_left = (int32_t)min(a.rows - row0, (int64_t)kTileRows);
        col0 = tc0 + 8 * l;
        base = row0 * a.cols + col0;
        gr = a.g + row0;
        mr = a.m + row0;
        gnext = active ? __ldg(gr) : 0.f;
    }
};

// RAGGED: the stream's shape is not a whole number of tiles, so blocks in the
// padding must not be stored (the tile-aligned variant skips those checks).
template <int KIND, bool DUMP, int NL, bool RAGGED>
__device__ __forceinline__ void decode_group(const DecodeArgs& a, const uint32_t* tab, int64_t grp0,
                                             uint32_t* status, uint32_t ring_off) {
    // fields used inside the block loop, read once: the batched kernel's
    // descriptors live in global memory, which the output stores could alias
    void* const outp = a.out;
    uint8_t* const symp = a.sym_out;
    const int64_t step = a.cols;
    const int l = threadIdx.x & 3;
    Lane ln[NL];
    LaneTile<KIND> T[NL];
    bool esc_bad[NL];
#pragma unroll
    for (int i = 0; i < NL; i++) {
        T[i].setup(a, grp0 + i, ln[i], ring_off + kRingBytesPerLane * i, status);
        esc_bad[i] = false;
    }

    bool slow_prev = false;  // warp-uniform: the previous block took the escape path
    for (int slab = 0; slab < kSlabs; slab++) {
        int64_t eoff[NL];
        bool col_in[NL];  // the slab's block lies inside the true columns
#pragma unroll
        for (int i = 0; i < NL; i++) {
            eoff[i] = T[i].base + kSlabCols * slab;
            col_in[i] = T[i].active && (!RAGGED || T[i].col0 + kSlabCols * slab < a.cols);
        }
#pragma unroll 2
        for (int row = 0; row < kTileRows; row++) {
            const int j = slab * kTileRows + row;
            if ((row & 1) == 0 || slow_prev) top_up<NL>(ln);
            if constexpr (is_lossless(KIND)) {
                uint32_t e[NL][8];
#pragma unroll
                for (int k = 0; k < 8; k++)
#pragma unroll
                    for (int i = 0; i < NL; i++) e[i][k] = ln[i].sym(tab);
#pragma unroll
                for (int i = 0; i < NL; i++) {
                    const bool st = col_in[i] && (!RAGGED || row < T[i].rows_left);
                    // raw bytes of block 4 j + l start at raw_per_elem * 8 * (4 j + l)
                    const uint8_t* rp = T[i].tb + raw_per_elem(KIND) * 8 * (4 * j + l);
                    if constexpr (KIND == K_LOSSLESS) {
                        uint2 raw = make_uint2(0, 0);
                        if (T[i].active) raw = *reinterpret_cast<const uint2*>(rp);
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; h++) {
                            const uint32_t rw = (h < 2 ? raw.x : raw.y) >> (16 * (h & 1));
                            const uint32_t r0 = rw & 0xFFu, r1 = (rw >> 8) & 0xFFu;
                            const uint32_t v0 = ((r0 & 0x80u) << 8) | ((e[i][2 * h] >> 5) & 0x7F80u) | (r0 & 0x7Fu);
                            const uint32_t v1 =
                                ((r1 & 0x80u) << 8) | ((e[i][2 * h + 1] >> 5) & 0x7F80u) | (r1 & 0x7Fu);
                            w[h] = v0 | (v1 << 16);
                        }
                        if (st)
                            *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(outp) + eoff[i]) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                    } else if constexpr (KIND == K_LOSSLESS8) {
                        uint32_t u[8];
#pragma unroll
                        for (int k = 0; k < 8; k++) u[k] = sym_byte(e[i][k]);
                        if (st)
                            *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(outp) + eoff[i]) =
                                make_uint2(u[0] | (u[1] << 8) | (u[2] << 16) | (u[3] << 24),
                                           u[4] | (u[5] << 8) | (u[6] << 16) | (u[7] << 24));
                    } else {  // K_LOSSLESS32: 24 raw bytes per block, 3 per element
                        uint32_t r[6] = {0, 0, 0, 0, 0, 0};
                        if (T[i].active) {
                            const uint2* rq = reinterpret_cast<const uint2*>(rp);  // 24 * block: 8-byte aligned
                            const uint2 q0 = rq[0], q1 = rq[1], q2 = rq[2];
                            r[0] = q0.x; r[1] = q0.y; r[2] = q1.x; r[3] = q1.y; r[4] = q2.x; r[5] = q2.y;
                        }
                        uint32_t v[8];
#pragma unroll
                        for (int k = 0; k < 8; k++) {
                            // raw bytes 3k .. 3k + 2 of the block (little-endian in r[])
                            const uint32_t b0 = (r[(3 * k) >> 2] >> (8 * ((3 * k) & 3))) & 0xFFu;
                            const uint32_t b1 = (r[(3 * k + 1) >> 2] >> (8 * ((3 * k + 1) & 3))) & 0xFFu;
                            const uint32_t b2 = (r[(3 * k + 2) >> 2] >> (8 * ((3 * k + 2) & 3))) & 0xFFu;
                            v[k] = ((b0 & 0x80u) << 24) | (sym_byte(e[i][k]) << 23) | ((b0 & 0x7Fu) << 16) | (b1 << 8) | b2;
                        }
                        if (st) {
                            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(outp) + eoff[i]);
                            dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
                            dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
                        }
                    }
                    if (st) {
                        if (DUMP) {
                            uint32_t u[8];
#pragma unroll
                            for (int k = 0; k < 8; k++) u[k] = sym_byte(e[i][k]);
                            dump_syms(symp, eoff[i], u);
                        }
                    }
                    eoff[i] += step;
                }
            } else {
            float mult[NL];
#pragma unroll
            for (int i = 0; i < NL; i++) {
                mult[i] = T[i].gnext;  // prefetched one block ahead (the L1 beside the rings is small)
                T[i].gnext = (T[i].active && j + 1 < kBlocksPerLane) ? __ldg(T[i].gr + ((row + 1) & 31)) : 0.f;
                if (KIND == K_FP8 || KIND == K_INT8) mult[i] = T[i].active ? __ldg(T[i].mr + row) : 0.f;
            }
            uint32_t e[NL][8];
            const uint32_t* t1[NL];
#pragma unroll
            for (int i = 0; i < NL; i++) {
                e[i][0] = ln[i].sym(tab);
                t1[i] = tab + kSlots + ((e[i][0] >> 12) & 1u) * kSlots;  // context 1 + c
            }
#pragma unroll
            for (int k = 1; k < 7; k++)
#pragma unroll
                for (int i = 0; i < NL; i++) e[i][k] = ln[i].sym(t1[i]);
#pragma unroll
            for (int i = 0; i < NL; i++) e[i][7] = ln[i].sym(t1[i] + 2 * kSlots);  // context 3 + c
            bool esc[NL];
            bool any = false;
#pragma unroll
            for (int i = 0; i < NL; i++) {
                bool v = ((e[i][0] >> 13) & 0x7Fu) == 0;  // s0 byte 0 or 1
#pragma unroll
                for (int k = 1; k < 8; k++) v |= (e[i][k] & 0x000FF000u) == 0;  // byte 0
                esc[i] = v && T[i].active;
                any |= esc[i];
            }
            const bool slow = __any_sync(0xffffffffu, any);
            slow_prev = slow;
            // no copy may still be in flight into a ring slot that the next
            // top-up refills after the payload moved the lanes on
            if (slow) asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
            for (int i = 0; i < NL; i++) {
                float y[8];
                if (slow) {
                    const uint32_t c = (e[i][0] >> 12) & 1u;
                    int32_t B[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) B[k] = (int32_t)sym_byte(e[i][k]);
                    if (esc[i]) {
#pragma unroll
                        for (int k = 0; k < 8; k++) {
                            const bool is_esc = (k == 0) ? (B[0] <= 1) : (B[k] == 0);
                            if (!is_esc) continue;
                            const uint32_t hi = ln[i].byte();
                            const uint32_t lo = ln[i].byte();
                            const int32_t P = (int32_t)(int16_t)(uint16_t)((hi << 8) | lo);
                            const int32_t mask = (k == 7) ? 3 : 1;
                            if (((P - (int32_t)c) & mask) != 0) esc_bad[i] = true;
                            B[k] = P + 128;
                        }
                    }
                    const int32_t px = B[0] ^ B[1] ^ B[2] ^ B[3] ^ B[4] ^ B[5] ^ B[6];
                    B[7] += px & 2;
                    const float cst = -mult[i] * kMagicHiQ;  // exact: mult has <= 7 significant bits
#pragma unroll
                    for (int k = 0; k < 8; k++) y[k] = fmaf(__uint_as_float(kMagicHi + (uint32_t)B[k]), mult[i], cst);
                } else {
                    uint32_t F[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) F[k] = (e[i][k] & 0x000FF000u) | kMagicLo;
                    // parity of a_0..a_6 is bit 1 of the XOR of the symbol bytes (bit 13 of the entries)
                    const uint32_t px = e[i][0] ^ e[i][1] ^ e[i][2] ^ e[i][3] ^ e[i][4] ^ e[i][5] ^ e[i][6];
                    F[7] += px & 0x2000u;
                    const float cst = -mult[i] * kMagicLoQ;  // exact: mult has <= 7 significant bits
#pragma unroll
                    for (int k = 0; k < 8; k++) y[k] = fmaf(__uint_as_float(F[k]), mult[i], cst);
                }
                if (col_in[i] && (!RAGGED || row < T[i].rows_left)) {
                    store_block<KIND>(outp, eoff[i], y);
                    if (DUMP) {
                        uint32_t u[8];
#pragma unroll
                        for (int k = 0; k < 8; k++) u[k] = sym_byte(e[i][k]);
                        dump_syms(symp, eoff[i], u);
                    }
                }
                eoff[i] += step;
            }
            }  // lossy
        }
    }
#pragma unroll
    for (int i = 0; i < NL; i++) {
        if (T[i].active && (ln[i].x != kRansL || ln[i].a != ln[i].aend)) flag(status, EP_STATUS_LANE_END);
        if (esc_bad[i]) flag(status, EP_STATUS_ESCAPE);
    }
}

__device__ __forceinline__ void copy_row_scales(const DecodeArgs& a, int64_t first, int64_t stride) {
    if (a.scale_out)
        for (int64_t r = first; r < a.rows; r += stride) a.scale_out[r] = a.t[r];
}

// Shared-memory layout of a decode CTA (g_smem, 128-byte aligned): n_ctx slot
// tables (16 KB each), the n_ctx x 256 frequency and cumulative-frequency
// scratch of the table build, then one 64-byte word ring per lane.
__host__ __device__ constexpr size_t decode_smem_bytes(int n_ctx, int nl) {
    return (size_t)n_ctx * (kSlots + 512) * 4 + (size_t)cta_threads(nl) * nl * kRingBytesPerLane;
}

// byte offset of this thread's first ring in g_smem (a thread running NL
// lanes owns NL consecutive rings): after the tables and their build scratch
// of n_ctx contexts (18432 bytes each, a multiple of 128)
template <int NL>
__device__ __forceinline__ uint32_t lane_ring(int n_ctx) {
    return (uint32_t)n_ctx * (kSlots + 512) * 4 + kRingBytesPerLane * NL * threadIdx.x;
}

// Lanes per thread (NL): two interleaved lanes per thread (512 threads) give
// each warp more independent work and share the per-block overhead, which
// pays when there are more tile groups than warp slots (the batched kernel,
// large matrices); a single matrix of less than one wave of groups decodes
// faster with one lane per thread (1024 threads), since its time is one
// lane's serial latency.  The symbol-dump debug kernel always uses one.

// ------------------------------------------------------------ single stream
// Tile groups are dealt round-robin over the CTAs first (group g goes to CTA
// g % gridDim.x), so a small matrix still spreads over every SM.
template <int KIND, bool DUMP, int NL, bool RAGGED>
__global__ void __launch_bounds__(cta_threads(NL), 1) decode_kernel(const DecodeArgs a) {
    uint32_t* const smem = g_smem;
    uint32_t* tab = smem;                    // n_ctx x 4096
    uint32_t* fr = smem + a.n_ctx * kSlots;  // n_ctx x 256
    uint32_t* cu = fr + a.n_ctx * 256;       // n_ctx x 256
    build_tables(a, tab, fr, cu);
    if (KIND == K_FP8 || KIND == K_INT8)
        copy_row_scales(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
    // groups are taken NL at a time: warp job p decodes groups NL p .. NL p + NL - 1
    const int64_t n_groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
    const int64_t n_jobs = (n_groups + NL - 1) / NL;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t p = (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; p < n_jobs; p += stride)
        decode_group<KIND, DUMP, NL, RAGGED>(a, tab, p * NL, a.status, lane_ring<NL>(a.n_ctx));
}

// ----------------------------------------------------------------- batched
// Many streams (e.g. every linear layer of a model) in one persistent launch.
// Work unit = 32 tile groups (one per warp) of one stream; CTAs claim units in
// stream order from a global counter, rebuild their tables when the stream
// changes, and count finished units per stream.  With ring = R > 0, stream i
// may share its output buffer with stream i - R ("decode back to back into
// reused buffers"): a unit of stream i first waits (bounded) until every unit
// of stream i - R is finished.  Claims are made only by running CTAs and in
// stream order, so every awaited unit is held by a running CTA: no deadlock.
struct BatchCounters {
    unsigned long long claim;
    uint32_t pad[2];
    // followed by uint32_t done[n_items]
};

constexpr uint32_t kWaitSpins = 1u << 23;  // x ~256 ns sleep: about 2 s before giving up

constexpr int kBatchNL = 2;                              // lanes per thread in the batched kernel
constexpr int kBatchThreads = cta_threads(kBatchNL);    // 640: 20 warps
constexpr int kGroupsPerUnit = kBatchThreads / 32 * kBatchNL;  // 40 groups: one per warp and lane slot

template <int KIND, bool RAGGED>
__global__ void __launch_bounds__(kBatchThreads, 1)
    batch_kernel(const DecodeArgs* __restrict__ items, const int64_t* __restrict__ unit_start, int64_t n_items,
                 int32_t ring, BatchCounters* ctr, uint32_t* status) {
    uint32_t* const smem = g_smem;
    __shared__ int64_t s_unit, s_item;
    __shared__ int s_skip;
    uint32_t* done = reinterpret_cast<uint32_t*>(ctr + 1);
    const int64_t total = unit_start[n_items];
    int64_t cur = -1;
    for (;;) {
        if (threadIdx.x == 0) {
            const int64_t u = (int64_t)atomicAdd(&ctr->claim, 1ull);
            int64_t lo = 0, hi = n_items - 1;  // item with unit_start[item] <= u < unit_start[item + 1]
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (unit_start[mid] <= u) lo = mid; else hi = mid - 1;
            }
            s_unit = u;
            s_item = lo;
            s_skip = 0;
            if (u < total && ring > 0 && lo >= ring) {
                const int64_t prev = lo - ring;
                const uint32_t need = (uint32_t)(unit_start[prev + 1] - unit_start[prev]);
                uint32_t spins = 0;
                while (*reinterpret_cast<volatile uint32_t*>(done + prev) < need && spins < kWaitSpins) {
                    __nanosleep(256);
                    spins++;
                }
                if (spins >= kWaitSpins) {
                    atomicOr(status, EP_STATUS_WAIT_TIMEOUT);
                    s_skip = 1;
                }
                __threadfence();
            }
        }
        __syncthreads();
        const int64_t unit = s_unit, item = s_item;
        if (unit >= total) break;
        const DecodeArgs& a = items[item];
        uint32_t* tab = smem;
        if (item != cur) {
            build_tables(a, tab, smem + a.n_ctx * kSlots, smem + a.n_ctx * kSlots + a.n_ctx * 256);
            cur = item;
        }
        const int64_t grp = (unit - unit_start[item]) * kGroupsPerUnit + (threadIdx.x >> 5) * kBatchNL;
        const int64_t n_groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
        if (!s_skip && grp < n_groups)
            decode_group<KIND, false, kBatchNL, RAGGED>(a, tab, grp, status, lane_ring<kBatchNL>(kLossyContexts));
        if ((KIND == K_FP8 || KIND == K_INT8) && unit == unit_start[item])
            copy_row_scales(a, threadIdx.x, blockDim.x);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(done + item, 1u);
        }
    }
}

// ------------------------------------------------------------ launching
constexpr size_t kBatchSmem = decode_smem_bytes(kLossyContexts, kBatchNL);
constexpr size_t kMaxSmem = decode_smem_bytes(kLossyContexts, 1) > kBatchSmem ? decode_smem_bytes(kLossyContexts, 1) : kBatchSmem;

struct DeviceInfo {
    int sms = 0;
};

DeviceInfo device_info() {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return DeviceInfo{148};
    if (!cache[dev].sms) cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
    return cache[dev];
}

// cudaFuncSetAttribute applies to the calling thread's current device only:
// raise a kernel's dynamic shared-memory limit once per device (bit d of
// *done records device d; setting it twice is harmless).
ep_status raise_smem_limit(const void* kernel, std::atomic<uint64_t>* done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EP_ERR_CUDA;
    const uint64_t bit = 1ull << dev;
    if (done->load(std::memory_order_acquire) & bit) return EP_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess)
        return EP_ERR_CUDA;
    done->fetch_or(bit, std::memory_order_release);
    return EP_OK;
}

template <int KIND, bool DUMP, int NL, bool RAGGED>
ep_status launch_nl(const DecodeArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> done{0};
    if (raise_smem_limit(reinterpret_cast<const void*>(decode_kernel<KIND, DUMP, NL, RAGGED>), &done) != EP_OK)
        return EP_ERR_CUDA;
    const int64_t jobs = ((a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp + NL - 1) / NL;
    const int64_t cap = device_info().sms;
    const int grid = (int)(jobs < cap ? jobs : cap);
    decode_kernel<KIND, DUMP, NL, RAGGED><<<grid, cta_threads(NL), decode_smem_bytes(a.n_ctx, NL), stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

bool is_ragged(int64_t rows, int64_t cols) { return (rows % kTileRows) != 0 || (cols % kTileCols) != 0; }

template <int KIND, bool DUMP, bool RAGGED>
ep_status launch_r(const DecodeArgs& a, cudaStream_t stream) {
    const int64_t groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
    if (DUMP || groups <= (int64_t)device_info().sms * (kThreads / 32))
        return launch_nl<KIND, DUMP, 1, RAGGED>(a, stream);
    return launch_nl<KIND, DUMP, 2, RAGGED>(a, stream);
}

template <int KIND, bool DUMP>
ep_status launch(const DecodeArgs& a, cudaStream_t stream) {
    return is_ragged(a.rows, a.cols) ? launch_r<KIND, DUMP, true>(a, stream) : launch_r<KIND, DUMP, false>(a, stream);
}

constexpr size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }
constexpr size_t batch_units_off(int64_t n) { return up256(sizeof(DecodeArgs) * (size_t)n); }
constexpr size_t batch_ctr_off(int64_t n) { return up256(batch_units_off(n) + sizeof(int64_t) * (size_t)(n + 1)); }
constexpr size_t batch_bytes(int64_t n) {
    return up256(batch_ctr_off(n) + sizeof(BatchCounters) + sizeof(uint32_t) * (size_t)n);
}

size_t batch_layout(int64_t n, size_t* items_off, size_t* units_off, size_t* ctr_off) {
    *items_off = 0;
    *units_off = batch_units_off(n);
    *ctr_off = batch_ctr_off(n);
    return batch_bytes(n);
}

// kernel arguments of a stream already parsed and validated into L
ep_status fill_args_parsed(const Layout& L, const void* d_blob, void* d_out, float* d_scale, uint8_t* d_sym,
                           uint32_t* d_status, DecodeArgs* a) {
    if (!d_blob || !d_out) return EP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_blob) | reinterpret_cast<uintptr_t>(d_out)) & 15u) return EP_ERR_INVALID_ARG;
    if (d_sym && (reinterpret_cast<uintptr_t>(d_sym) & 7u)) return EP_ERR_INVALID_ARG;
    std::memset(a, 0, sizeof(*a));
    const uint8_t* db = static_cast<const uint8_t*>(d_blob);
    a->blob = db;
    a->tile_off = reinterpret_cast<const uint64_t*>(db + L.offsets_off);
    a->payload = db + L.payload_off;
    a->payload_bytes = L.total - L.payload_off;
    a->g = reinterpret_cast<const float*>(db + L.rowmeta_off);
    a->m = a->g + L.rows_p;  // row metadata covers the padded rows
    a->t = a->g + 2 * L.rows_p;
    for (int c = 0; c < L.n_ctx; c++) a->ctx_off[c] = (uint32_t)L.ctx_off[c];
    a->n_ctx = L.n_ctx;
    a->out = d_out;
    a->scale_out = d_scale;
    a->sym_out = d_sym;
    a->status = d_status;
    a->rows = L.rows;
    a->cols = L.cols;
    a->n_tiles = L.n_tiles;
    a->tiles_per_row = L.cols_p / kTileCols;
    return EP_OK;
}

ep_status fill_args(const uint8_t* h_blob, const void* d_blob, size_t bytes, void* d_out, float* d_scale,
                    uint8_t* d_sym, uint32_t* d_status, Layout& L, DecodeArgs* a) {
    if (!h_blob || !d_blob || !d_out) return EP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_blob) | reinterpret_cast<uintptr_t>(d_out)) & 15u) return EP_ERR_INVALID_ARG;
    if (d_sym && (reinterpret_cast<uintptr_t>(d_sym) & 7u)) return EP_ERR_INVALID_ARG;
    ep_status st = parse_and_validate(h_blob, bytes, &L);
    if (st != EP_OK) return st;
    return fill_args_parsed(L, d_blob, d_out, d_scale, d_sym, d_status, a);
}

int kind_of(const Layout& L) {
    if (L.mode != EP_MODE_LOSSLESS_TILEANS) return L.container;
    return L.container == EP_C_FP8_E4M3 ? K_LOSSLESS8 : (L.container == EP_C_FP32 ? K_LOSSLESS32 : K_LOSSLESS);
}

template <int KIND, bool RAGGED>
ep_status launch_batch_r(const ep_batch_plan* p, uint32_t* d_status, cudaStream_t stream) {
    static std::atomic<uint64_t> done{0};
    if (raise_smem_limit(reinterpret_cast<const void*>(batch_kernel<KIND, RAGGED>), &done) != EP_OK)
        return EP_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(p->d_workspace);
    const int64_t cap = device_info().sms;
    const int grid = (int)(p->total_units < cap ? p->total_units : cap);
    if (grid <= 0) return EP_OK;
    batch_kernel<KIND, RAGGED><<<grid, kBatchThreads, kBatchSmem, stream>>>(
        reinterpret_cast<const DecodeArgs*>(ws + p->items_off), reinterpret_cast<const int64_t*>(ws + p->units_off),
        p->n_items, p->ring, reinterpret_cast<BatchCounters*>(ws + p->counters_off), d_status);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

// plan->reserved != 0: some item's shape is not a whole number of tiles
template <int KIND>
ep_status launch_batch(const ep_batch_plan* p, uint32_t* d_status, cudaStream_t stream) {
    return p->reserved ? launch_batch_r<KIND, true>(p, d_status, stream) : launch_batch_r<KIND, false>(p, d_status, stream);
}

ep_status launch_parsed(const Layout& L, const DecodeArgs& a, bool dump, uint32_t* d_status, cudaStream_t stream) {
    if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), stream) != cudaSuccess) return EP_ERR_CUDA;
    switch (kind_of(L)) {
        case K_BF16: return dump ? launch<K_BF16, true>(a, stream) : launch<K_BF16, false>(a, stream);
        case K_FP16: return dump ? launch<K_FP16, true>(a, stream) : launch<K_FP16, false>(a, stream);
        case K_FP8: return dump ? launch<K_FP8, true>(a, stream) : launch<K_FP8, false>(a, stream);
        case K_INT8: return dump ? launch<K_INT8, true>(a, stream) : launch<K_INT8, false>(a, stream);
        case K_LOSSLESS8: return dump ? launch<K_LOSSLESS8, true>(a, stream) : launch<K_LOSSLESS8, false>(a, stream);
        case K_LOSSLESS32:
            return dump ? launch<K_LOSSLESS32, true>(a, stream) : launch<K_LOSSLESS32, false>(a, stream);
        default: return dump ? launch<K_LOSSLESS, true>(a, stream) : launch<K_LOSSLESS, false>(a, stream);
    }
}

ep_status decode_impl(const uint8_t* h_blob, const void* d_blob, size_t bytes, void* d_out, float* d_scale,
                      uint8_t* d_sym, uint32_t* d_status, cudaStream_t stream) {
    if (!d_status) return EP_ERR_INVALID_ARG;
    thread_local Layout L;
    DecodeArgs a;
    ep_status st = fill_args(h_blob, d_blob, bytes, d_out, d_scale, d_sym, d_status, L, &a);
    if (st != EP_OK) return st;
    return launch_parsed(L, a, d_sym != nullptr, d_status, stream);
}

}  // namespace

ep_status decode_parsed(const Layout& L, const void* d_blob, void* d_out, float* d_row_scale, uint32_t* d_status,
                        ep_stream_t stream) {
    if (!d_status) return EP_ERR_INVALID_ARG;
    DecodeArgs a;
    ep_status st = fill_args_parsed(L, d_blob, d_out, d_row_scale, nullptr, d_status, &a);
    if (st != EP_OK) return st;
    return launch_parsed(L, a, false, d_status, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace ep
extern "C" {

ep_status ep_decode(const uint8_t* h_blob, const void* d_blob, size_t bytes, void* d_out, float* d_row_scale_out,
                    uint32_t* d_status, ep_stream_t stream) {
    return ep::decode_impl(h_blob, d_blob, bytes, d_out, d_row_scale_out, nullptr, d_status,
                           reinterpret_cast<cudaStream_t>(stream));
}

ep_status ep_decode_symbols(const uint8_t* h_blob, const void* d_blob, size_t bytes, void* d_out,
                            float* d_row_scale_out, uint8_t* d_sym_out, uint32_t* d_status, ep_stream_t stream) {
    if (!d_sym_out) return EP_ERR_INVALID_ARG;
    return ep::decode_impl(h_blob, d_blob, bytes, d_out, d_row_scale_out, d_sym_out, d_status,
                           reinterpret_cast<cudaStream_t>(stream));
}

size_t ep_batch_workspace_bytes(int64_t n_items) {
    if (n_items <= 0) return 0;
    size_t a, b, c;
    return ep::batch_layout(n_items, &a, &b, &c);
}

ep_status ep_batch_prepare(const ep_batch_item* items, int64_t n_items, int32_t ring, void* d_workspace,
                           size_t workspace_bytes, ep_batch_plan* plan) {
    using namespace ep;
    if (!items || n_items <= 0 || !d_workspace || !plan || ring < 0) return EP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_workspace) & 255u) return EP_ERR_INVALID_ARG;
    size_t items_off, units_off, ctr_off;
    const size_t need = batch_layout(n_items, &items_off, &units_off, &ctr_off);
    if (workspace_bytes < need) return EP_ERR_INVALID_ARG;
    std::vector<DecodeArgs> args((size_t)n_items);
    std::vector<int64_t> units((size_t)n_items + 1, 0);
    Layout* L = new (std::nothrow) Layout();
    if (!L) return EP_ERR_NOMEM;
    int kind = -1, n_ctx = 0;
    bool ragged = false;
    ep_status st = EP_OK;
    for (int64_t i = 0; i < n_items && st == EP_OK; i++) {
        const ep_batch_item& it = items[i];
        // the batch kernel reports through the status word given to ep_batch_decode
        st = fill_args(it.h_blob, it.d_blob, it.bytes, it.d_out, it.d_row_scale_out, nullptr, nullptr, *L,
                       &args[(size_t)i]);
        if (st != EP_OK) break;
        const int k = kind_of(*L);
        if (kind >= 0 && k != kind) st = EP_ERR_INVALID_ARG;  // one container/mode per batch
        kind = k;
        n_ctx = std::max(n_ctx, L->n_ctx);
        ragged = ragged || is_ragged(L->rows, L->cols);
        const int64_t groups = (L->n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
        units[(size_t)i + 1] = units[(size_t)i] + (groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
    }
    delete L;
    if (st != EP_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    if (cudaMemcpy(ws + items_off, args.data(), sizeof(DecodeArgs) * args.size(), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(ws + units_off, units.data(), sizeof(int64_t) * units.size(), cudaMemcpyHostToDevice) !=
            cudaSuccess)
        return EP_ERR_CUDA;
    std::memset(plan, 0, sizeof(*plan));
    plan->n_items = n_items;
    plan->total_units = units[(size_t)n_items];
    plan->ring = ring;
    plan->kind = kind;
    plan->n_ctx = n_ctx;
    plan->reserved = ragged ? 1 : 0;
    plan->d_workspace = d_workspace;
    plan->workspace_bytes = workspace_bytes;
    plan->items_off = items_off;
    plan->units_off = units_off;
    plan->counters_off = ctr_off;
    return EP_OK;
}

ep_status ep_batch_decode(const ep_batch_plan* plan, uint32_t* d_status, ep_stream_t stream) {
    using namespace ep;
    if (!plan || !plan->d_workspace || !d_status || plan->n_items <= 0) return EP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(plan->d_workspace);
    const size_t ctr_bytes = sizeof(BatchCounters) + sizeof(uint32_t) * (size_t)plan->n_items;
    if (cudaMemsetAsync(ws + plan->counters_off, 0, ctr_bytes, s) != cudaSuccess) return EP_ERR_CUDA;
    if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), s) != cudaSuccess) return EP_ERR_CUDA;
    switch (plan->kind) {
        case K_BF16: return launch_batch<K_BF16>(plan, d_status, s);
        case K_FP16: return launch_batch<K_FP16>(plan, d_status, s);
        case K_FP8: return launch_batch<K_FP8>(plan, d_status, s);
        case K_INT8: return launch_batch<K_INT8>(plan, d_status, s);
        case K_LOSSLESS: return launch_batch<K_LOSSLESS>(plan, d_status, s);
        case K_LOSSLESS8: return launch_batch<K_LOSSLESS8>(plan, d_status, s);
        case K_LOSSLESS32: return launch_batch<K_LOSSLESS32>(plan, d_status, s);
    }
    return EP_ERR_INVALID_ARG;
}

ep_status ep_sync_status(const uint32_t* d_status, ep_stream_t stream) {
    if (!d_status) return EP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, d_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return EP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EP_ERR_CUDA;
    return h ? EP_ERR_CORRUPT : EP_OK;
}

}  // extern "C"

// ------------------------------------------------ allocation-free batched decode
// Some callers cannot allocate device memory at all: code that runs inside
// another framework's memory pool or allocator lock, plug-ins loaded into a
// host process that owns every allocation, or real-time paths where a
// cudaMalloc would synchronise the device.  ep_batch_decode_static serves
// them: the batch kernel's scratch (item descriptors, unit table, claim and
// completion counters) lives in the file-scope device array below instead of
// a caller workspace.  Every GPU that loads the library holds these bytes
// until the process exits.
namespace ep {
namespace {
constexpr int64_t kStaticMaxItems = EP_BATCH_STATIC_MAX_ITEMS;
constexpr size_t kStaticScratchBytes = batch_bytes(kStaticMaxItems);
}  // namespace
}  // namespace ep

static __device__ __align__(256) uint8_t g_ep_batch_scratch[ep::kStaticScratchBytes];

namespace ep {
namespace {

// Device address of g_ep_batch_scratch on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked up
// once per device (with that device current) and cached.
ep_status static_scratch_address(uint8_t** out) {
    static std::mutex mu;
    static uint8_t* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ep_batch_scratch) != cudaSuccess || !p) return EP_ERR_CUDA;
        cache[dev] = static_cast<uint8_t*>(p);
    }
    *out = cache[dev];
    return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" ep_status ep_batch_decode_static(const ep_batch_item* items, int64_t n_items, int32_t ring,
                                            uint32_t* d_status, ep_stream_t stream) {
    using namespace ep;
    if (!items || n_items <= 0 || ring < 0 || !d_status) return EP_ERR_INVALID_ARG;
    if (n_items > kStaticMaxItems) return EP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = nullptr;
    ep_status st = static_scratch_address(&ws);
    if (st != EP_OK) return st;
    const size_t units_off = batch_units_off(n_items), ctr_off = batch_ctr_off(n_items);
    // Host threads calling at the same time would interleave their copies
    // into the one array: hold the array from the first copy to the launch.
    // Each call's copies and kernel then follow one another on its stream;
    // calls on different streams can still overlap on the GPU (see the header).
    static std::mutex array_mu;
    std::lock_guard<std::mutex> hold(array_mu);

    // Validate every stream and stage the descriptors in fixed-size host
    // chunks on this thread's stack; each chunk goes to the device array with
    // one cudaMemcpyAsync from pageable memory, which returns once the bytes
    // are staged, so the stack buffer can be reused at once.
    thread_local Layout L;
    constexpr int64_t kChunk = 32;
    DecodeArgs chunk[kChunk];
    int64_t units[kChunk + 1];
    int64_t unit_total = 0;
    int kind = -1, n_ctx = 0;
    bool ragged = false;
    for (int64_t base = 0; base < n_items; base += kChunk) {
        const int64_t n = std::min<int64_t>(kChunk, n_items - base);
        for (int64_t i = 0; i < n; i++) {
            const ep_batch_item& it = items[base + i];
            st = fill_args(it.h_blob, it.d_blob, it.bytes, it.d_out, it.d_row_scale_out, nullptr, nullptr, L,
                           &chunk[i]);
            if (st != EP_OK) return st;
            const int k = kind_of(L);
            if (kind >= 0 && k != kind) return EP_ERR_INVALID_ARG;  // one container/mode per batch
            kind = k;
            n_ctx = std::max(n_ctx, L.n_ctx);
            ragged = ragged || is_ragged(L.rows, L.cols);
            units[i] = unit_total;
            const int64_t groups = (L.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
            unit_total += (groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
        }
        if (cudaMemcpyAsync(ws + sizeof(DecodeArgs) * (size_t)base, chunk, sizeof(DecodeArgs) * (size_t)n,
                            cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(ws + units_off + sizeof(int64_t) * (size_t)base, units, sizeof(int64_t) * (size_t)n,
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return EP_ERR_CUDA;
    }
    units[0] = unit_total;  // unit_start[n_items]
    if (cudaMemcpyAsync(ws + units_off + sizeof(int64_t) * (size_t)n_items, units, sizeof(int64_t),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return EP_ERR_CUDA;
    // the counters start at zero on every call; the previous call's values stay behind otherwise
    if (cudaMemsetAsync(ws + ctr_off, 0, sizeof(BatchCounters) + sizeof(uint32_t) * (size_t)n_items, s) !=
            cudaSuccess ||
        cudaMemsetAsync(d_status, 0, sizeof(uint32_t), s) != cudaSuccess)
        return EP_ERR_CUDA;
    ep_batch_plan plan;
    std::memset(&plan, 0, sizeof(plan));
    plan.n_items = n_items;
    plan.total_units = unit_total;
    plan.ring = ring;
    plan.kind = kind;
    plan.n_ctx = n_ctx;
    plan.reserved = ragged ? 1 : 0;
    plan.d_workspace = ws;
    plan.workspace_bytes = kStaticScratchBytes;
    plan.items_off = 0;
    plan.units_off = units_off;
    plan.counters_off = ctr_off;
    switch (kind) {
        case K_BF16: return launch_batch<K_BF16>(&plan, d_status, s);
        case K_FP16: return launch_batch<K_FP16>(&plan, d_status, s);
        case K_FP8: return launch_batch<K_FP8>(&plan, d_status, s);
        case K_INT8: return launch_batch<K_INT8>(&plan, d_status, s);
        case K_LOSSLESS: return launch_batch<K_LOSSLESS>(&plan, d_status, s);
        case K_LOSSLESS8: return launch_batch<K_LOSSLESS8>(&plan, d_status, s);
        case K_LOSSLESS32: return launch_batch<K_LOSSLESS32>(&plan, d_status, s);
    }
    return EP_ERR_INVALID_ARG;
}
