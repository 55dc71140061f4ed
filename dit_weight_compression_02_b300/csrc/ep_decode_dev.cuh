// Device-side building blocks of the EntroPack stream decode, shared by the
// decode kernels (ep_decode.cu) and the fused decode-and-multiply linear
// kernel (ep_fused.cu): the kernel argument block of one stream, the
// shared-memory slot tables, the rANS lane with its shared-memory word ring,
// container conversion and the per-tile lane set-up.  Stream format version
// 1 (tiles of 32 x 128, 4 lanes, 12-bit tables, 16-bit words).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_format.hpp"

namespace ep {

// Kernel arguments of one stream (device pointers into its blob, its shape).
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

// Fill the arguments of a stream already validated into L (d_out may be
// NULL for kernels that write elsewhere).
ep_status decode_args_of(const Layout& L, const void* d_blob, void* d_out, uint32_t* d_status, DecodeArgs* a);

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
    // symbol later, by which time the load has landed.  Written without a
    // branch (selects and a predicated load) so that the compiler can
    // schedule the symbol chain together with independent work around it.
    __device__ __forceinline__ void renorm() {
        const uint32_t r = x < kRansL;
        x = r ? ((x << 16) | next) : x;
        a += r << 1;
        const uint32_t addr = (uint32_t)__cvta_generic_to_shared(g_smem) + (roff | (a & (kRingBytesPerLane - 2u)));
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p ld.shared.u16 %0, [%1];\n\t}"
                     : "+r"(next) : "r"(addr), "r"(r));
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

// The escape path of one lane's block.  v[k] holds the coded byte of
// coordinate k in bits 12..19 (a slot entry or a spliced float); when `esc`,
// every escaped coordinate (s0 byte 0 or 1, s1..s7 byte 0) takes its int16
// payload from the lane's words, two uniform bytes each.  Writes
// y[k] = fp32(mult * q_k), rounded once (mult has at most 7 significant bits,
// so mult * 6291520 is exact), and flags a payload that contradicts the
// coset.
__device__ __forceinline__ void escape_block(Lane& ln, const uint32_t* v, bool esc, float mult, float* y,
                                             bool& esc_bad) {
    const uint32_t c = (v[0] >> 12) & 1u;
    int32_t B[8];
#pragma unroll
    for (int k = 0; k < 8; k++) B[k] = (int32_t)sym_byte(v[k]);
    if (esc) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const bool is_esc = (k == 0) ? (B[0] <= 1) : (B[k] == 0);
            if (!is_esc) continue;
            const uint32_t hi = ln.byte();
            const uint32_t lo = ln.byte();
            const int32_t P = (int32_t)(int16_t)(uint16_t)((hi << 8) | lo);
            const int32_t mask = (k == 7) ? 3 : 1;
            if (((P - (int32_t)c) & mask) != 0) esc_bad = true;
            B[k] = P + 128;
        }
    }
    const int32_t px = B[0] ^ B[1] ^ B[2] ^ B[3] ^ B[4] ^ B[5] ^ B[6];
    B[7] += px & 2;
    const float cst = -mult * kMagicHiQ;
#pragma unroll
    for (int k = 0; k < 8; k++) y[k] = fmaf(__uint_as_float(kMagicHi + (uint32_t)B[k]), mult, cst);
}

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

    // validate the tile, find the lane's words and start the lane: thread
    // (tig, l) of the warp takes lane l of tile 8 grp + tig
    __device__ __forceinline__ void setup(const DecodeArgs& a, int64_t grp, Lane& ln, uint32_t ring_off,
                                          uint32_t* status) {
        const int tig = (threadIdx.x & 31) >> 2;
        setup_at(a, grp * kTilesPerWarp + tig, grp >= 0, ln, ring_off, status);
    }
    // the same for lane threadIdx.x % 4 of a given tile (inactive when !want
    // or the tile is past the stream's last)
    __device__ __forceinline__ void setup_at(const DecodeArgs& a, int64_t tile, bool want, Lane& ln,
                                             uint32_t ring_off, uint32_t* status) {
        const int l = threadIdx.x & 3;
        constexpr uint32_t kRaw = 4096u * raw_per_elem(KIND);
        constexpr uint32_t kHdr = kRaw + kTileHeaderBytes;
        active = want && tile >= 0 && tile < a.n_tiles;
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

}  // namespace
}  // namespace ep
