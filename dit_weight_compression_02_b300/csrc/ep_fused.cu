// Fused CompressedLinear for few tokens on B300 (sm_103a): the weight stream
// is decoded straight into the tcgen05 B operand in shared memory and
// multiplied with X without ever writing W to global memory ("EntroPack: Fast
// and Accurate Entropy-Coded Weight Compression at Arbitrary Bitrates",
// Abstract: symbol decoding and weight reconstruction run fused on the GPU
// and feed inference; "EntroPack PyTorch Guide", "Replace one linear layer
// before a whole model": CompressedLinear.from_linear).
//
// Y[T x N] = X[T x K] W[N x K]^T (+ b), BF16 in and out, fp32 accumulation.
//
// Work unit: R whole tile rows of W (32 R weight rows, all K).  Each of the
// unit's 4 R (K / 128) rANS lanes is one decode thread, so every tile of the
// unit decodes at once.  A tile's lanes emit one 32-column row segment per
// step and finish a K-slab (32 rows x 32 columns) every 32 steps; the unit
// therefore produces its weights half a K-slab at a time: rows 16 h' .. 16 h'
// + 15 of K-slab s for every tile (h = 2 s + h').  The decode threads write
// those rows, already BF16, into a shared-memory buffer laid out as the MMA's
// K-major B operand (64-byte swizzle; a 64-byte row holds one tile's 32 slab
// columns), then arrive on an mbarrier.  One thread issues tcgen05.mma (M =
// 128 tokens, N = 16 weight rows, K = 16) over the half slab, with X streamed
// by TMA in matching chunks (128 tokens x the tile's 32 slab columns, the same
// 64-byte swizzle), into TMEM accumulators: 32 columns per tile row and token
// tile.  When the MMAs have read the buffer a commit releases it
// for the next half slab.  After the unit's last half slab, four warps read
// the accumulators back (tcgen05.ld), add the bias, round to BF16 and store Y.
//
// Shared memory bounds the unit: the slot tables take 80 KB and one half
// slab takes 1 KB per tile, so R is the largest of 1..3 that fits (3 for a
// K = 3840 layer, whose 320 tile rows then take 107 CTAs: one wave).  TMEM (512 columns)
// bounds the tokens of one pass to 512 / (32 R) token tiles of 128; more
// tokens run as further passes, each decoding W again, so the kernel serves
// the few-token regime (a K = 3840 layer takes up to 640 tokens per pass).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "ep_decode_dev.cuh"
#include "ep_sm100.cuh"

namespace ep {
namespace {

using namespace sm100;

constexpr int kFM = 128;                         // tokens per MMA (M) and per token tile
constexpr int kFN = 16;                          // weight rows per MMA (N): half a K-slab's rows
constexpr int kHalves = 2 * kSlabs;              // half slabs per tile
constexpr uint32_t kWBlockBytes = kFN * 64;      // B operand of one (tile row, tile): 16 rows x 64 B
constexpr uint32_t kXStageBytes = kFM * 64;      // A operand chunk: 128 tokens x a tile's 32 slab columns
constexpr int kXStages = 4;
constexpr int kMaxUnitRows = 3;                  // tile rows per unit (R)
constexpr int kMaxTilesPerRow = 96;              // K / 128 limit: one tile row's half slab fills 96 KB
constexpr int kTmemCols = 512;
constexpr uint64_t kFusedWaitNs = 2000000000ull;  // 2 s per wait before a role gives up

struct FusedShape {
    int64_t T;          // tokens of this pass (<= 128 m_tiles)
    int64_t N, K;       // out_features, in_features (K % 128 == 0)
    int tc;             // tiles per tile row: K / 128
    int tr;             // tile rows: ceil(N / 32)
    int R;              // tile rows per unit
    int n_units;        // ceil(tr / R)
    int m_tiles;        // token tiles of 128
    int dec_threads;    // decode threads: max(4 R tc rounded up to a warp, 128)
    uint32_t tmem_cols; // accumulator columns allocated: a power of two >= 32 R m_tiles
};

// Shared-memory layout (byte offsets from g_smem): slot tables, one word
// ring per lane, then (1024-byte aligned in the shared window) the X stages
// and the half-slab W buffer, then the mbarriers and the TMEM address.  The
// table build's frequency scratch (n_ctx x 2 KB) borrows the X stages, which
// are idle then.
struct FusedSmem {
    uint32_t rings, xs, wb, bars, total;
};
constexpr uint32_t kFusedBarBytes = (2 * kXStages + 4) * 8 + 8;  // the mbarriers below and the TMEM address

__host__ __device__ inline FusedSmem fused_smem(int n_ctx, int n_lanes, int R, int tc, uint32_t base_mod1024) {
    FusedSmem m;
    m.rings = (uint32_t)n_ctx * kSlots * 4;
    const uint32_t end_rings = m.rings + (uint32_t)n_lanes * kRingBytesPerLane;
    // base_mod1024: the shared-window address of g_smem modulo 1024
    m.xs = ((end_rings + base_mod1024 + 1023u) & ~1023u) - base_mod1024;
    m.wb = m.xs + kXStages * kXStageBytes;
    m.bars = m.wb + (uint32_t)R * tc * kWBlockBytes;
    m.total = m.bars + kFusedBarBytes;
    return m;
}

// Bytes to allocate: the layout above for any alignment of g_smem.
__host__ inline uint32_t fused_smem_alloc(int n_ctx, int n_lanes, int R, int tc) {
    return (uint32_t)n_ctx * kSlots * 4 + (uint32_t)n_lanes * kRingBytesPerLane + 1023u + kXStages * kXStageBytes +
           (uint32_t)R * tc * kWBlockBytes + kFusedBarBytes;
}

// Shared-memory descriptor of a K-major operand in the 64-byte swizzle layout:
// rows of 32 bf16 (64 B), 8-row atoms of 512 B (stride 512 B), atoms on
// 512-byte boundaries; swizzle mode 4 = 64 B (bits 61-63), descriptor
// version 1 (bits 46-47).  Advancing K by 16 elements adds 32 B.
__device__ __forceinline__ uint64_t sw64_kmajor_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1u << 16) | ((uint64_t)(512u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)4u << 61);
}

__device__ __forceinline__ void fused_fail(volatile int* abort_flag, uint32_t* status) {
    *abort_flag = 1;
    atomicOr(status, EP_STATUS_WAIT_TIMEOUT);
}

__global__ void __launch_bounds__(1024, 1)
    fused_linear_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tx, uint16_t* __restrict__ y,
                        const uint16_t* __restrict__ bias, const FusedShape sh, uint32_t* status) {
    uint8_t* const sm = reinterpret_cast<uint8_t*>(g_smem);
    const int n_lanes = 4 * sh.R * sh.tc;  // lanes of a full unit, one decode thread each
    const FusedSmem L = fused_smem(a.n_ctx, n_lanes, sh.R, sh.tc, smem_addr(g_smem) & 1023u);
    uint32_t* tab = g_smem;
    uint8_t* xs = sm + L.xs;
    uint8_t* wb = sm + L.wb;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L.bars);
    uint64_t* xfull = bars;                 // [kXStages] X chunk landed
    uint64_t* xempty = bars + kXStages;     // [kXStages] X chunk consumed
    uint64_t* wfull = bars + 2 * kXStages;  // half slab written by every decode thread
    uint64_t* wempty = wfull + 1;           // half slab consumed by the MMAs
    uint64_t* dfull = wfull + 2;            // a unit's accumulators complete
    uint64_t* dempty = wfull + 3;           // a unit's accumulators read back
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wfull + 4);
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tma_warp = sh.dec_threads >> 5, mma_warp = tma_warp + 1;

    // slot tables of the stream (every thread takes part); the frequency
    // scratch sits in the X stages, which TMA fills only afterwards
    build_tables(a, tab, reinterpret_cast<uint32_t*>(xs), reinterpret_cast<uint32_t*>(xs) + a.n_ctx * 256);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kXStages; s++) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        mbar_init(wfull, sh.dec_threads);
        mbar_init(wempty, 1);
        mbar_init(dfull, 1);
        mbar_init(dempty, 128);
        fence_barrier_init();
        s_abort = 0;
        tma_prefetch_map(&tx);
    }
    if (warp == mma_warp) {
        tmem_alloc(tmem_slot, sh.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == tma_warp) {
        // ------------------------------------------------ X producer
        if (lane == 0) {
            uint32_t s = 0, ph = 0;
            for (int u = blockIdx.x; u < sh.n_units && !s_abort; u += gridDim.x)
                for (int h = 0; h < kHalves && !s_abort; h++)
                    for (int m = 0; m < sh.m_tiles && !s_abort; m++)
                        for (int t = 0; t < sh.tc; t++) {
                            if (!mbar_wait(&xempty[s], ph ^ 1u, globaltimer_ns() + kFusedWaitNs)) {
                                fused_fail(&s_abort, status);
                                break;
                            }
                            mbar_arrive_expect_tx(&xfull[s], kXStageBytes);
                            // columns 128 t + 32 slab .. + 31, tokens 128 m .. 128 m + 127
                            tma_load_2d(xs + s * kXStageBytes, &tx, &xfull[s], t * kTileCols + (h >> 1) * kSlabCols,
                                        m * kFM);
                            if (++s == kXStages) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
        }
    } else if (warp == mma_warp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kFM, kFN);
            uint32_t s = 0, ph = 0, hs = 0, units_done = 0;
            for (int u = blockIdx.x; u < sh.n_units && !s_abort; u += gridDim.x) {
                const int rows_u = min(sh.R, sh.tr - u * sh.R);
                // the previous unit's accumulators must have been read back
                if (units_done && !mbar_wait(dempty, (units_done - 1) & 1u, globaltimer_ns() + kFusedWaitNs)) {
                    fused_fail(&s_abort, status);
                    break;
                }
                tc_fence_after_sync();
                bool ok = true;
                for (int h = 0; h < kHalves && ok; h++, hs++) {
                    if (!mbar_wait(wfull, hs & 1u, globaltimer_ns() + kFusedWaitNs)) {
                        fused_fail(&s_abort, status);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    for (int m = 0; m < sh.m_tiles && ok; m++)
                        for (int t = 0; t < sh.tc; t++) {
                            if (!mbar_wait(&xfull[s], ph, globaltimer_ns() + kFusedWaitNs)) {
                                fused_fail(&s_abort, status);
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
                            const uint64_t da = sw64_kmajor_desc(smem_addr(xs + s * kXStageBytes));
                            for (int r = 0; r < rows_u; r++) {
                                const uint64_t db = sw64_kmajor_desc(smem_addr(wb + (r * sh.tc + t) * kWBlockBytes));
                                // accumulator columns of (token tile m, tile row r, half h & 1)
                                const uint32_t d = tmem + (uint32_t)((m * sh.R + r) * 32 + (h & 1) * kFN);
#pragma unroll
                                for (int k = 0; k < 2; k++)
                                    umma_bf16(d, da + 2u * k, db + 2u * k, idesc, (h >= 2 || t > 0 || k > 0) ? 1u : 0u);
                            }
                            umma_commit(&xempty[s]);
                            if (++s == kXStages) {
                                s = 0;
                                ph ^= 1u;
                            }
                        }
                    if (ok) umma_commit(wempty);  // the buffer is free once these MMAs have read it
                }
                if (!ok) break;
                umma_commit(dfull);
                units_done++;
            }
        }
    } else if (warp < tma_warp) {
        // ------------------------------------------------ decode threads (+ epilogue: warps 0..3)
        const int i = threadIdx.x;
        const int lanes_per_row = 4 * sh.tc;
        uint32_t hs = 0, units_done = 0;
        for (int u = blockIdx.x; u < sh.n_units && !s_abort; u += gridDim.x) {
            const int rows_u = min(sh.R, sh.tr - u * sh.R);
            const int r = i / lanes_per_row, t = (i >> 2) % sh.tc, l = i & 3;
            const bool mine = i < rows_u * lanes_per_row;
            Lane ln[1];
            LaneTile<K_BF16> T;
            // decode threads past the unit's lanes run an empty lane that
            // only reads (lane 0's ring)
            T.setup_at(a, (int64_t)(u * sh.R + r) * sh.tc + t, mine, ln[0],
                       L.rings + kRingBytesPerLane * (uint32_t)(i < n_lanes ? i : 0), status);
            bool esc_bad = false, slow_prev = false;
            // this lane's 16-byte slot in the B operand of (tile row r, tile t):
            // 16-byte column l of each 64-byte row, swizzled
            uint8_t* wrow = wb + (mine ? (r * sh.tc + t) * kWBlockBytes : 0);
            const uint32_t chunk = (uint32_t)l;
            bool ok = true;
            for (int h = 0; h < kHalves && ok; h++, hs++) {
                // the MMAs of the previous half slab must have read the buffer
                if (hs > 0 && !mbar_wait(wempty, (hs - 1) & 1u, globaltimer_ns() + kFusedWaitNs)) {
                    fused_fail(&s_abort, status);
                    ok = false;
                    break;
                }
                for (int rho = 0; rho < kFN; rho++) {
                    const int row = (h & 1) * kFN + rho;
                    if ((row & 1) == 0 || slow_prev) top_up<1>(ln);
                    const float g = __ldg(T.gr + row);
                    uint32_t e[8];
                    e[0] = ln[0].sym(tab);
                    const uint32_t* t1 = tab + kSlots + ((e[0] >> 12) & 1u) * kSlots;  // context 1 + c
#pragma unroll
                    for (int k = 1; k < 7; k++) e[k] = ln[0].sym(t1);
                    e[7] = ln[0].sym(t1 + 2 * kSlots);  // context 3 + c
                    bool esc = ((e[0] >> 13) & 0x7Fu) == 0;  // s0 byte 0 or 1
#pragma unroll
                    for (int k = 1; k < 8; k++) esc |= (e[k] & 0x000FF000u) == 0;
                    esc = esc && T.active;
                    const bool slow = __any_sync(0xffffffffu, esc);
                    slow_prev = slow;
                    float yv[8];
                    if (slow) {
                        asm volatile("cp.async.wait_group 0;" ::: "memory");
                        escape_block(ln[0], e, esc, g, yv, esc_bad);
                    } else {
                        uint32_t F[8];
#pragma unroll
                        for (int k = 0; k < 8; k++) F[k] = (e[k] & 0x000FF000u) | kMagicLo;
                        const uint32_t px = e[0] ^ e[1] ^ e[2] ^ e[3] ^ e[4] ^ e[5] ^ e[6];
                        F[7] += px & 0x2000u;
                        const float cst = -g * kMagicLoQ;
#pragma unroll
                        for (int k = 0; k < 8; k++) yv[k] = fmaf(__uint_as_float(F[k]), g, cst);
                    }
                    if (mine)
                        *reinterpret_cast<uint4*>(wrow + rho * 64 + ((chunk ^ (uint32_t)((rho >> 1) & 3)) << 4)) =
                            make_uint4(pack2(yv[0], yv[1], K_BF16), pack2(yv[2], yv[3], K_BF16),
                                       pack2(yv[4], yv[5], K_BF16), pack2(yv[6], yv[7], K_BF16));
                }
                fence_proxy_async_smem();  // the rows just written are read by tcgen05.mma
                mbar_arrive(wfull);
            }
            if (T.active && (ln[0].x != kRansL || ln[0].a != ln[0].aend)) flag(status, EP_STATUS_LANE_END);
            if (esc_bad) flag(status, EP_STATUS_ESCAPE);
            if (!ok) break;
            // ---------------------------------------- epilogue (warps 0..3)
            if (warp < 4) {
                if (!mbar_wait(dfull, units_done & 1u, globaltimer_ns() + kFusedWaitNs)) {
                    fused_fail(&s_abort, status);
                    break;
                }
                tc_fence_after_sync();
                for (int m = 0; m < sh.m_tiles; m++) {
                    const int64_t tok = (int64_t)m * kFM + warp * 32 + lane;
                    for (int rr = 0; rr < rows_u; rr++) {
                        uint32_t acc[32];
                        tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)((m * sh.R + rr) * 32), acc);
                        tmem_ld_wait();
                        const int64_t col = (int64_t)(u * sh.R + rr) * 32;  // first weight row of this tile row
                        if (tok < sh.T) {
                            uint16_t* dst = y + tok * sh.N + col;
#pragma unroll
                            for (int q = 0; q < 4; q++) {  // 8 weight rows each; N is a multiple of 8
                                if (col + 8 * q >= sh.N) break;
                                float v[8];
#pragma unroll
                                for (int e2 = 0; e2 < 8; e2++) v[e2] = __uint_as_float(acc[8 * q + e2]);
                                if (bias) {  // the bias joins the fp32 sum before the one rounding
                                    const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + col + 8 * q));
                                    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                                    for (int e2 = 0; e2 < 4; e2++) {
                                        v[2 * e2] += __uint_as_float(bw[e2] << 16);
                                        v[2 * e2 + 1] += __uint_as_float(bw[e2] & 0xFFFF0000u);
                                    }
                                }
                                *reinterpret_cast<uint4*>(dst + 8 * q) =
                                    make_uint4(pack2(v[0], v[1], K_BF16), pack2(v[2], v[3], K_BF16),
                                               pack2(v[4], v[5], K_BF16), pack2(v[6], v[7], K_BF16));
                            }
                        }
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(dempty);
            }
            units_done++;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == mma_warp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, sh.tmem_cols);
    }
}

// ------------------------------------------------------------ host side
// X [T x K] row-major BF16 read in boxes of 128 tokens x 32 columns, which
// land as 128 rows of 64 bytes, 64-byte swizzled (the swizzle span equals
// the box row, so the rows are packed).  Tokens past T read as zero.
bool make_x_map(CUtensorMap* map, const void* x, int64_t T, int64_t K) {
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kSlabCols, (cuuint32_t)kFM};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fused_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 148;
    return n > 0 ? n : 148;
}

// Dynamic shared memory one CTA may use on the current device.
uint32_t fused_smem_budget() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || optin <= 0)
        return 0;
    return (uint32_t)optin - 256u;  // room for the kernel's static shared memory
}

// Tile rows per unit for tc tiles per tile row: the most (up to 3) whose
// shared memory fits the budget; 0 when not even one does.
int fused_unit_rows(int tc, uint32_t budget) {
    if (tc <= 0 || tc > kMaxTilesPerRow) return 0;
    for (int R = kMaxUnitRows; R >= 1; R--)
        if (fused_smem_alloc(kLossyContexts, 4 * R * tc, R, tc) <= budget) return R;
    return 0;
}

}  // namespace

// Tokens one pass of the fused kernel covers for a layer of in_features K
// (0 when the fused kernel does not serve the shape: K % 128 != 0, or a
// tile row too long for shared memory).
int64_t fused_tokens_per_pass(int64_t K) {
    if (K <= 0 || K % 128) return 0;
    const int R = fused_unit_rows((int)std::min<int64_t>(K / 128, 1 << 20), fused_smem_budget());
    if (R == 0) return 0;
    return (int64_t)kFM * (kTmemCols / (32 * R));
}

// Y = X W^T (+ b) by the fused kernel, passes of fused_tokens_per_pass(K)
// tokens.  The stream is lossy BF16 and already validated into L; the caller
// has checked the shapes and pointers.
ep_status fused_linear_parsed(const Layout& L, const void* d_blob, const uint16_t* d_x, int64_t tokens,
                              uint16_t* d_y, const uint16_t* d_bias, uint32_t* d_status, ep_stream_t stream_h) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    const int64_t per_pass = fused_tokens_per_pass(L.cols);
    if (per_pass <= 0) return EP_ERR_UNSUPPORTED;
    DecodeArgs a;
    ep_status st = decode_args_of(L, d_blob, nullptr, d_status, &a);
    if (st != EP_OK) return st;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EP_ERR_CUDA;
    FusedShape sh;
    sh.N = L.rows;
    sh.K = L.cols;
    sh.tc = (int)(L.cols / 128);
    sh.tr = (int)((L.rows + 31) / 32);
    const uint32_t budget = fused_smem_budget();
    sh.R = fused_unit_rows(sh.tc, budget);
    if (sh.R == 0) return EP_ERR_UNSUPPORTED;
    sh.n_units = (sh.tr + sh.R - 1) / sh.R;
    sh.dec_threads = std::max(128, (4 * sh.R * sh.tc + 31) / 32 * 32);
    // the layout plus up to 16 KB of slack behind it (as much as the budget allows)
    const uint32_t smem = std::min(budget, fused_smem_alloc(a.n_ctx, 4 * sh.R * sh.tc, sh.R, sh.tc) + 16384u);
    if (!(attr_done.load() & (1ull << dev))) {
        if (cudaFuncSetAttribute(fused_linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget) !=
            cudaSuccess)
            return EP_ERR_CUDA;
        attr_done.fetch_or(1ull << dev);
    }
    const int grid = std::min(sh.n_units, fused_sms());
    if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), stream) != cudaSuccess) return EP_ERR_CUDA;
    for (int64_t t0 = 0; t0 < tokens; t0 += per_pass) {
        sh.T = std::min(per_pass, tokens - t0);
        sh.m_tiles = (int)((sh.T + kFM - 1) / kFM);
        uint32_t cols = 32;
        while (cols < (uint32_t)(32 * sh.R * sh.m_tiles)) cols <<= 1;
        sh.tmem_cols = cols;
        CUtensorMap tx;
        if (!make_x_map(&tx, d_x + t0 * L.cols, sh.T, L.cols)) return EP_ERR_CUDA;
        fused_linear_kernel<<<grid, sh.dec_threads + 64, smem, stream>>>(a, tx, d_y + t0 * L.rows, d_bias, sh,
                                                                        d_status);
        if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    }
    return EP_OK;
}

}  // namespace ep

extern "C" int64_t ep_fused_tokens_per_pass(int64_t cols) { return ep::fused_tokens_per_pass(cols); }
