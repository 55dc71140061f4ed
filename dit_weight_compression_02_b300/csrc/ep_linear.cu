// Linear layers on compressed weights for B300 (sm_103a): Y = X W^T with
// BF16 X [tokens x K], W [N x K] (N = out_features) and BF16 Y [tokens x N]
// ("EntroPack PyTorch Guide", "Replace one linear layer before a whole
// model": CompressedLinear.from_linear; the Abstract's fused decode feeding
// inference).
//
// The GEMM is a persistent, warp-specialised tcgen05 kernel:
//   warp 0       TMA producer: 128x64 tiles of X and 256x64 tiles of W into a
//                4-stage shared-memory ring (128-byte swizzle, K-major)
//   warp 1       allocates 512 TMEM columns and issues tcgen05.mma
//                (M = 128 tokens, N = 256 weight rows, K = 16 per instruction,
//                fp32 accumulators) into two alternating 256-column buffers
//   warps 2..5   epilogue: tcgen05.ld of the finished accumulator, plus the
//                optional bias in fp32, BF16 rounding, 16-byte stores of Y,
//                then release of the buffer,
//                so the epilogue of one tile overlaps the MMAs of the next
// Output tiles are visited in groups of 16 token tiles (see tile_coords), so
// the CTAs running at the same time share a few W row-slabs and the group's
// rows of X stay resident in the 126 MB L2.
//
// ep_compressed_linear decodes the weight stream with the decode kernel of
// ep_decode.cu into a caller-owned BF16 workspace (78.6 MB for a 10240 x
// 3840 layer, which also fits the L2) and runs the GEMM on it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "ep_format.hpp"
#include "ep_sm100.cuh"

namespace ep {
namespace {

using namespace sm100;

constexpr int BM = 128;  // tokens per tile (MMA M, TMEM lanes)
constexpr int BN = 256;  // weight rows per tile (MMA N, TMEM columns per accumulator)
constexpr int BK = 64;   // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int STAGES = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr size_t kGemmSmem = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before a role gives up

struct GemmShape {
    int64_t T, N, K;
    int tiles_m, tiles_n, kblocks;
};

// Tile order: token tiles in groups of kGroupM; inside a group the CTAs walk
// the weight slabs n, token tiles fastest.  A wave of 148 tiles then touches
// kGroupM X row-blocks (16 x 0.98 MB for K = 3840) and a few W slabs, so the
// group's X stays in L2 while W streams through once per group.
constexpr int kGroupM = 16;

__device__ __forceinline__ void tile_coords(int t, const GemmShape& sh, int& m, int& n) {
    const int per_group = kGroupM * sh.tiles_n;
    const int g = t / per_group, r = t % per_group;
    const int gm = min(kGroupM, sh.tiles_m - g * kGroupM);  // the last group may be short
    m = g * kGroupM + r % gm;
    n = r / gm;
}

__device__ __forceinline__ void gemm_fail(volatile int* abort_flag, uint32_t* status) {
    *abort_flag = 1;
    atomicOr(status, EP_STATUS_WAIT_TIMEOUT);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                     uint16_t* __restrict__ y, const uint16_t* __restrict__ bias, const GemmShape sh,
                     uint32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ volatile int s_abort;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        fence_barrier_init();
        s_abort = 0;
        tma_prefetch_map(&tx);
        tma_prefetch_map(&tw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int n_tiles = sh.tiles_m * sh.tiles_n;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t s = 0, ph = 0;
        for (int t = blockIdx.x; t < n_tiles && !s_abort; t += gridDim.x) {
            int m, n;
            tile_coords(t, sh, m, n);
            for (int kb = 0; kb < sh.kblocks; kb++) {
                if (!mbar_wait(&empty[s], ph ^ 1u, globaltimer_ns() + kWaitNs)) {
                    gemm_fail(&s_abort, status);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                tma_load_2d(sA + s * A_BYTES, &tx, &full[s], kb * BK, m * BM);
                tma_load_2d(sB + s * B_BYTES, &tw, &full[s], kb * BK, n * BN);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        uint32_t s = 0, ph = 0, acc = 0, aph = 0;
        for (int t = blockIdx.x; t < n_tiles && !s_abort; t += gridDim.x) {
            if (!mbar_wait(&tempty[acc], aph ^ 1u, globaltimer_ns() + kWaitNs)) {
                gemm_fail(&s_abort, status);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d = tmem + acc * BN;
            bool ok = true;
            for (int kb = 0; kb < sh.kblocks; kb++) {
                if (!mbar_wait(&full[s], ph, globaltimer_ns() + kWaitNs)) {
                    gemm_fail(&s_abort, status);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t da = sw128_kmajor_desc(smem_addr(sA + s * A_BYTES));
                const uint64_t db = sw128_kmajor_desc(smem_addr(sB + s * B_BYTES));
#pragma unroll
                for (int k = 0; k < BK / 16; k++)
                    umma_bf16(d, da + 2u * k, db + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
                umma_commit(&empty[s]);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(&tfull[acc]);
            acc ^= 1u;
            if (!acc) aph ^= 1u;
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // the TMEM lane quarter this warp may read
        uint32_t acc = 0, aph = 0;
        for (int t = blockIdx.x; t < n_tiles && !s_abort; t += gridDim.x) {
            int m, n;
            tile_coords(t, sh, m, n);
            if (!mbar_wait(&tfull[acc], aph, globaltimer_ns() + kWaitNs)) {
                gemm_fail(&s_abort, status);
                break;
            }
            tc_fence_after_sync();
            const int64_t row = (int64_t)m * BM + q * 32 + lane;
            uint16_t* yrow = y + row * sh.N;
#pragma unroll 1
            for (int c = 0; c < BN / 32; c++) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + acc * BN + c * 32, r);
                tmem_ld_wait();
                const int64_t col = (int64_t)n * BN + c * 32;
                if (row < sh.T && col < sh.N) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + col);
#pragma unroll
                    for (int i = 0; i < 4; i++) {  // 8 columns each; N is a multiple of 8
                        if (col + 8 * i >= sh.N) break;
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) v[e] = __uint_as_float(r[8 * i + e]);
                        if (bias) {  // Y = BF16(acc + b): the bias joins the fp32 sum before the one rounding
                            const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + col + 8 * i));
                            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                v[2 * e] += __uint_as_float(bw[e] << 16);
                                v[2 * e + 1] += __uint_as_float(bw[e] & 0xFFFF0000u);
                            }
                        }
                        uint32_t p[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                            p[e] = *reinterpret_cast<uint32_t*>(&h);
                        }
                        dst[i] = make_uint4(p[0], p[1], p[2], p[3]);
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&tempty[acc]);
            acc ^= 1u;
            if (!acc) aph ^= 1u;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side
// Row-major bf16 matrix [outer x inner] read in boxes of [box_outer x 64] with
// the 128-byte swizzle; out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return cache[dev] ? cache[dev] : 148;
}

ep_status gemm_launch(const uint16_t* d_x, const uint16_t* d_w, uint16_t* d_y, const uint16_t* d_bias, int64_t T,
                      int64_t N, int64_t K, uint32_t* d_status, cudaStream_t stream) {
    // the shared-memory limit is a per-device setting: raise it once per device
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EP_ERR_CUDA;
    if (!(attr_done.load(std::memory_order_acquire) & (1ull << dev))) {
        if (cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem) !=
            cudaSuccess)
            return EP_ERR_CUDA;
        attr_done.fetch_or(1ull << dev, std::memory_order_release);
    }
    CUtensorMap tx, tw;
    if (!make_map(&tx, d_x, (uint64_t)K, (uint64_t)T, BM) || !make_map(&tw, d_w, (uint64_t)K, (uint64_t)N, BN))
        return EP_ERR_CUDA;
    GemmShape sh;
    sh.T = T;
    sh.N = N;
    sh.K = K;
    sh.tiles_m = (int)((T + BM - 1) / BM);
    sh.tiles_n = (int)((N + BN - 1) / BN);
    sh.kblocks = (int)((K + BK - 1) / BK);
    const int tiles = sh.tiles_m * sh.tiles_n;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    gemm_bf16_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(tx, tw, d_y, d_bias, sh, d_status);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ep_status check_gemm_args(const void* d_x, const void* d_w, const void* d_y, const void* d_bias, int64_t T, int64_t N,
                          int64_t K, const uint32_t* d_status) {
    if (!d_x || !d_w || !d_y || !d_status) return EP_ERR_INVALID_ARG;
    if (!aligned16(d_x) || !aligned16(d_w) || !aligned16(d_y) || !aligned16(d_bias)) return EP_ERR_INVALID_ARG;
    if (T <= 0 || N <= 0 || K <= 0) return EP_ERR_SHAPE;
    if (N % 8 || K % 8) return EP_ERR_SHAPE;
    if (T > ((int64_t)1 << 31) - BM || N > ((int64_t)1 << 31) - BN || K > ((int64_t)1 << 31)) return EP_ERR_SHAPE;
    return EP_OK;
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// CompressedLinear on a stream already parsed and validated into L
ep_status compressed_linear_parsed(const Layout& L, const void* d_blob, const uint16_t* d_x, int64_t tokens,
                                   uint16_t* d_y, const uint16_t* d_bias, int32_t mode, void* d_ws, size_t ws_bytes,
                                   uint32_t* d_status, ep_stream_t stream) {
    ep_status st;
    if (L.mode != EP_MODE_LOSSY_E8 || L.container != EP_C_BF16) return EP_ERR_UNSUPPORTED;
    if (mode == EP_LINEAR_FUSED) {
        // W never leaves the chip: no workspace
        if (fused_tokens_per_pass(L.cols) <= 0) return EP_ERR_UNSUPPORTED;
        st = check_gemm_args(d_x, d_blob, d_y, d_bias, tokens, L.rows, L.cols, d_status);
        if (st != EP_OK) return st;
        return fused_linear_parsed(L, d_blob, d_x, tokens, d_y, d_bias, d_status, stream);
    }
    if (mode != EP_LINEAR_DECODE_THEN_GEMM) return EP_ERR_UNSUPPORTED;
    const size_t need = (size_t)L.rows * (size_t)L.cols * 2u;
    if (!d_ws || ws_bytes < need) return EP_ERR_INVALID_ARG;
    st = check_gemm_args(d_x, d_ws, d_y, d_bias, tokens, L.rows, L.cols, d_status);
    if (st != EP_OK) return st;
    // the decode zeroes the status word and writes W into the workspace; the
    // GEMM (same stream) reads it back, mostly from L2
    st = decode_parsed(L, d_blob, d_ws, nullptr, d_status, stream);
    if (st != EP_OK) return st;
    return gemm_launch(d_x, static_cast<const uint16_t*>(d_ws), d_y, d_bias, tokens, L.rows, L.cols, d_status,
                       reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace ep

extern "C" {

ep_status ep_linear_bf16(const uint16_t* d_x, const uint16_t* d_w, uint16_t* d_y, const uint16_t* d_bias,
                         int64_t tokens, int64_t rows, int64_t cols, uint32_t* d_status, ep_stream_t stream) {
    ep_status st = ep::check_gemm_args(d_x, d_w, d_y, d_bias, tokens, rows, cols, d_status);
    if (st != EP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), s) != cudaSuccess) return EP_ERR_CUDA;
    return ep::gemm_launch(d_x, d_w, d_y, d_bias, tokens, rows, cols, d_status, s);
}

ep_status ep_compressed_linear(const uint8_t* h_blob, const void* d_blob, size_t bytes, const uint16_t* d_x,
                               int64_t tokens, uint16_t* d_y, const uint16_t* d_bias, int32_t mode, void* d_ws,
                               size_t ws_bytes, uint32_t* d_status, ep_stream_t stream) {
    using namespace ep;
    if (!h_blob || !d_blob || !d_status) return EP_ERR_INVALID_ARG;
    thread_local Layout L;  // parsed and validated once per call
    ep_status st = parse_and_validate(h_blob, bytes, &L);
    if (st != EP_OK) return st;
    return compressed_linear_parsed(L, d_blob, d_x, tokens, d_y, d_bias, mode, d_ws, ws_bytes, d_status, stream);
}

ep_status ep_compressed_linear_h(const ep_stream_handle* h, const void* d_blob, const uint16_t* d_x, int64_t tokens,
                                 uint16_t* d_y, const uint16_t* d_bias, int32_t mode, void* d_ws, size_t ws_bytes,
                                 uint32_t* d_status, ep_stream_t stream) {
    if (!h || !d_blob || !d_status) return EP_ERR_INVALID_ARG;
    return ep::compressed_linear_parsed(h->L, d_blob, d_x, tokens, d_y, d_bias, mode, d_ws, ws_bytes, d_status,
                                        stream);
}

}  // extern "C"
