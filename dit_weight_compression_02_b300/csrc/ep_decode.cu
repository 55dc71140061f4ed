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
// A single lossy matrix with fewer tile groups than one wave of warps is bound
// by one lane's chain of dependent symbols; it runs a software-pipelined block
// loop (decode_group_pipelined) in 512-thread CTAs.
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

#include "ep_decode_dev.cuh"
#include "ep_format.hpp"

namespace ep {
namespace {

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
                    escape_block(ln[i], e[i], esc[i], mult[i], y, esc_bad[i]);
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

// Latency-bound decode (a single matrix that fills fewer warps than the SMs
// hold): the block loop is software pipelined so that one lane's work of two
// neighbouring blocks overlaps.  While block j is checked for escapes,
// rebuilt and stored, the symbols of block j + 1 are already decoded from the
// state after block j's symbols, on the speculation that block j has no
// escape.  A block with an escape (rare) restores the lane state saved before
// the speculation, decodes its escape payload and decodes block j + 1 again.
// Lossy streams only; the bits produced are those of decode_group.
template <int KIND, bool DUMP, int NL, bool RAGGED>
__device__ __forceinline__ void decode_group_pipelined(const DecodeArgs& a, const uint32_t* tab, int64_t grp0,
                                                       uint32_t* status, uint32_t ring_off) {
    void* const outp = a.out;
    uint8_t* const symp = a.sym_out;
    const int64_t cols = a.cols;
    Lane ln[NL];
    LaneTile<KIND> T[NL];
    bool esc_bad[NL];
#pragma unroll
    for (int i = 0; i < NL; i++) {
        T[i].setup(a, grp0 + i, ln[i], ring_off + kRingBytesPerLane * i, status);
        esc_bad[i] = false;
    }
    // the 8 symbols of one block of every lane, as F = bits(1536 + u/2)
    auto block_syms = [&](uint32_t (&D)[NL][8]) {
        const uint32_t* t1[NL];
#pragma unroll
        for (int i = 0; i < NL; i++) {
            D[i][0] = (ln[i].sym(tab) & 0x000FF000u) | kMagicLo;
            t1[i] = tab + kSlots + ((D[i][0] >> 12) & 1u) * kSlots;  // context 1 + c
        }
#pragma unroll
        for (int k = 1; k < 7; k++)
#pragma unroll
            for (int i = 0; i < NL; i++) D[i][k] = (ln[i].sym(t1[i]) & 0x000FF000u) | kMagicLo;
#pragma unroll
        for (int i = 0; i < NL; i++) D[i][7] = (ln[i].sym(t1[i] + 2 * kSlots) & 0x000FF000u) | kMagicLo;
    };
    uint32_t F[NL][8];
    bool last_slow = false;
    top_up<NL>(ln);
    block_syms(F);
#pragma unroll 2
    for (int j = 0; j < kBlocksPerLane; j++) {
        const int slab = j >> 5, row = j & 31;
        float mult[NL];
#pragma unroll
        for (int i = 0; i < NL; i++)
            mult[i] = __ldg((KIND == K_FP8 || KIND == K_INT8 ? T[i].mr : T[i].gr) + row);
        // restore point: the lane state after block j's symbols
        uint32_t sx[NL], sa[NL], sn[NL];
#pragma unroll
        for (int i = 0; i < NL; i++) {
            sx[i] = ln[i].x;
            sa[i] = ln[i].a;
            sn[i] = ln[i].next;
        }
        const bool more = j + 1 < kBlocksPerLane;
        uint32_t G[NL][8];
        // unconditional, so that it shares a basic block with block j's
        // reconstruction below; after the last block it decodes past the
        // lane's end (ring reads only) and the state is restored after the loop
        if ((j & 1) == 1) top_up<NL>(ln);  // block j + 1 starts a pair
        block_syms(G);
        bool esc[NL];
        bool any = false;
        float y[NL][8];
#pragma unroll
        for (int i = 0; i < NL; i++) {
            bool v = ((F[i][0] >> 13) & 0x7Fu) == 0;  // s0 byte 0 or 1
#pragma unroll
            for (int k = 1; k < 8; k++) v |= (F[i][k] & 0x000FF000u) == 0;  // byte 0
            esc[i] = v && T[i].active;
            any |= esc[i];
            // the fast path's values, computed before the vote so that they
            // share a basic block with block j + 1's symbol chain
            const uint32_t px = F[i][0] ^ F[i][1] ^ F[i][2] ^ F[i][3] ^ F[i][4] ^ F[i][5] ^ F[i][6];
            const uint32_t f7 = F[i][7] + (px & 0x2000u);
            const float cst = -mult[i] * kMagicLoQ;  // exact: mult has <= 7 significant bits
#pragma unroll
            for (int k = 0; k < 7; k++) y[i][k] = fmaf(__uint_as_float(F[i][k]), mult[i], cst);
            y[i][7] = fmaf(__uint_as_float(f7), mult[i], cst);
        }
        if (__any_sync(0xffffffffu, any)) {
            // rare: undo the speculation, decode block j's escape payloads (from
            // global memory), then decode block j + 1 again from the new state
            asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
            for (int i = 0; i < NL; i++) {
                ln[i].x = sx[i];
                ln[i].a = sa[i];
                ln[i].next = sn[i];
                escape_block(ln[i], F[i], esc[i], mult[i], y[i], esc_bad[i]);
            }
            if (more) {
                top_up<NL>(ln);
                block_syms(G);
            } else {
                last_slow = true;  // the state is the lane's true end state
            }
        }
#pragma unroll
        for (int i = 0; i < NL; i++) {
            const bool st = T[i].active && (!RAGGED || (T[i].col0 + kSlabCols * slab < cols && row < T[i].rows_left));
            if (st) {
                const int64_t eoff = T[i].base + kSlabCols * slab + (int64_t)row * cols;
                store_block<KIND>(outp, eoff, y[i]);
                if (DUMP) {
                    uint32_t u[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) u[k] = sym_byte(F[i][k]);
                    dump_syms(symp, eoff, u);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < NL; i++)
#pragma unroll
            for (int k = 0; k < 8; k++) F[i][k] = G[i][k];
        if (!more && !last_slow)
#pragma unroll
            for (int i = 0; i < NL; i++) {  // undo the decode past the lane's end
                ln[i].x = sx[i];
                ln[i].a = sa[i];
                ln[i].next = sn[i];
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

// Latency-bound single matrices (lossy): one lane per thread, 512 threads, the
// pipelined block loop.
constexpr int kPipeThreads = 512;
// The pipelined kernel pays off while the SMs hold few warps; from about nine
// tile groups per SM on, the one-lane kernel's extra warps hide the latency as
// well (8192 x 8192: 2048 groups, measured 3-4 % faster on the one-lane kernel)
constexpr int kPipeGroupsPerSM = 9;

template <int KIND, bool DUMP, bool RAGGED>
__global__ void __launch_bounds__(kPipeThreads, 1) decode_kernel_pipe(const DecodeArgs a) {
    uint32_t* const smem = g_smem;
    uint32_t* tab = smem;
    uint32_t* fr = smem + a.n_ctx * kSlots;
    uint32_t* cu = fr + a.n_ctx * 256;
    build_tables(a, tab, fr, cu);
    if (KIND == K_FP8 || KIND == K_INT8)
        copy_row_scales(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
    const int64_t n_groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t p = (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; p < n_groups; p += stride)
        decode_group_pipelined<KIND, DUMP, 1, RAGGED>(a, tab, p, a.status, lane_ring<1>(a.n_ctx));
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
ep_status launch_pipe(const DecodeArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> done{0};
    if (raise_smem_limit(reinterpret_cast<const void*>(decode_kernel_pipe<KIND, DUMP, RAGGED>), &done) != EP_OK)
        return EP_ERR_CUDA;
    const int64_t groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
    const int64_t cap = device_info().sms;
    const int grid = (int)(groups < cap ? groups : cap);
    const size_t smem = (size_t)a.n_ctx * (kSlots + 512) * 4 + (size_t)kPipeThreads * kRingBytesPerLane;
    decode_kernel_pipe<KIND, DUMP, RAGGED><<<grid, kPipeThreads, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

template <int KIND, bool DUMP, bool RAGGED>
ep_status launch_r(const DecodeArgs& a, cudaStream_t stream) {
    const int64_t groups = (a.n_tiles + kTilesPerWarp - 1) / kTilesPerWarp;
    if constexpr (!is_lossless(KIND))
        if (groups <= (int64_t)device_info().sms * kPipeGroupsPerSM) return launch_pipe<KIND, DUMP, RAGGED>(a, stream);
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

ep_status decode_args_of(const Layout& L, const void* d_blob, void* d_out, uint32_t* d_status, DecodeArgs* a) {
    if (!d_blob || (reinterpret_cast<uintptr_t>(d_blob) & 15u)) return EP_ERR_INVALID_ARG;
    static char dummy[16] __attribute__((aligned(16)));  // never written: stands in for a missing output
    return fill_args_parsed(L, d_blob, d_out ? d_out : dummy, nullptr, nullptr, d_status, a);
}

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
