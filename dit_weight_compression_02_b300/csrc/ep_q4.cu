// GPU reconstruction of the fixed-width comparators.  NF4 / INT4:
// out[i] = BF16(levels[code_i] * scale[i / block]), one FP32 product rounded
// to nearest even.  The codes are packed two per byte, element 2j in the low
// nibble of byte j.
//
// The work is HBM-bound (0.5 B of codes + 4 / block B of scale read and 2 B
// written per weight): each thread turns 16 codes (one 8-byte load, one
// scale, since block % 16 == 0) into 32 output bytes with two 16-byte stores;
// a grid of whole waves strides over the groups.  A ragged tail (n % 16 != 0)
// is finished element by element by the thread that owns the last group.
// FP8 per row: out[r, c] = BF16(e4m3(code[r, c]) * scale[r]), 16 codes (one
// 16-byte load) to two 16-byte stores per thread.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "entropack.h"

namespace {

struct Levels {
    float v[16];
};

constexpr int kThreads = 256;
static_assert(kThreads == 256, "the FP8 kernel tabulates one E4M3 value per thread");

__global__ void __launch_bounds__(kThreads) q4_decode_kernel(const uint2* __restrict__ codes,
                                                             const float* __restrict__ scales, int64_t n,
                                                             int64_t block, Levels lv, uint4* __restrict__ out) {
    __shared__ float cb[16];
    if (threadIdx.x == 0) {  // constant indices: the levels stay in the parameter bank
#pragma unroll
        for (int k = 0; k < 16; ++k) cb[k] = lv.v[k];
    }
    __syncthreads();
    const int64_t full = n >> 4;  // whole groups of 16
    const int64_t groups = (n + 15) >> 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < groups; g += stride) {
        const int64_t e0 = g << 4;
        const float s = __ldg(scales + e0 / block);
        if (g < full) {
            const uint2 c = __ldg(codes + g);
            uint32_t packed[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t word = h ? c.y : c.x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t byte = (word >> (8 * j)) & 0xFFu;
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(cb[byte & 0xFu] * s, cb[byte >> 4] * s);
                    packed[h * 4 + j] = *reinterpret_cast<const uint32_t*>(&pr);
                }
            }
            out[2 * g] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            out[2 * g + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        } else {
            const uint8_t* cbytes = reinterpret_cast<const uint8_t*>(codes);
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
            for (int64_t i = e0; i < n; ++i) {
                const uint32_t byte = cbytes[i >> 1];
                const uint32_t code = (i & 1) ? (byte >> 4) : (byte & 0xFu);
                o[i] = __float2bfloat16_rn(cb[code] * __ldg(scales + i / block));
            }
        }
    }
}

// E4M3 byte -> float, exact: normal (8 + m) 2^(e - 10), subnormal m 2^-9
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
    return (b & 0x80u) ? -v : v;
}

// Per-row-scaled FP8 comparator: out[r, c] = BF16(e4m3(code[r, c]) * scale[r]).
// The CTA first tabulates the 256 E4M3 values in shared memory (kThreads ==
// 256).  One thread turns 16 codes (one 16-byte load) into two 16-byte stores; each
// half of 8 codes lies in one row (cols % 8 == 0) and takes that row's scale.
// With an odd number of 8-code groups the last one is done alone.
__device__ __forceinline__ uint4 fp8_group(const float* lut, uint32_t lo, uint32_t hi, float s) {
    uint32_t p[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint32_t word = h < 2 ? lo : hi;
        const uint32_t b0 = (word >> (16 * (h & 1))) & 0xFFu, b1 = (word >> (16 * (h & 1) + 8)) & 0xFFu;
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lut[b0] * s, lut[b1] * s);
        p[h] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

__global__ void __launch_bounds__(kThreads) fp8_row_decode_kernel(const uint8_t* __restrict__ codes,
                                                                  const float* __restrict__ scales, int64_t rows,
                                                                  int64_t cols, uint4* __restrict__ out) {
    __shared__ float lut[256];  // the value of every E4M3 byte
    lut[threadIdx.x] = e4m3_value(threadIdx.x);
    __syncthreads();
    const int64_t n8 = rows * cols / 8;  // 8-code groups
    const int64_t per_row = cols / 8;
    const int64_t n16 = n8 / 2;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const uint4* c16 = reinterpret_cast<const uint4*>(codes);
    const bool narrow = n8 < 0x7FFFFFFF;  // 32-bit row arithmetic suffices
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < n16; g += stride) {
        const uint4 c = __ldg(c16 + g);
        // row of the first half by one division; the second half is in that row or the next
        const int64_t r0 = narrow ? (int64_t)((uint32_t)(2 * g) / (uint32_t)per_row) : (2 * g) / per_row;
        const int64_t r1 = r0 + ((2 * g + 1) >= (r0 + 1) * per_row ? 1 : 0);
        const float s0 = __ldg(scales + r0);
        const float s1 = __ldg(scales + r1);
        out[2 * g] = fp8_group(lut, c.x, c.y, s0);
        out[2 * g + 1] = fp8_group(lut, c.z, c.w, s1);
    }
    if ((n8 & 1) && blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t g8 = n8 - 1;
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(codes) + g8);
        out[g8] = fp8_group(lut, c.x, c.y, __ldg(scales + g8 / per_row));
    }
}

int grid_for(int64_t work_items) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t per_wave = (int64_t)sms * (2048 / kThreads);
    int64_t grid = (work_items + kThreads - 1) / kThreads;
    if (grid > per_wave * 4) grid = per_wave * 4;
    return (int)grid;
}

}  // namespace

extern "C" ep_status ep_fp8_row_decode(const uint8_t* d_codes, const float* d_scales, int64_t rows, int64_t cols,
                                       uint16_t* d_out, ep_stream_t stream) {
    if (!d_codes || !d_scales || !d_out) return EP_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || cols % 8 || rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
        return EP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(d_codes) & 15) || (reinterpret_cast<uintptr_t>(d_scales) & 3) ||
        (reinterpret_cast<uintptr_t>(d_out) & 15))
        return EP_ERR_INVALID_ARG;
    fp8_row_decode_kernel<<<(unsigned)grid_for(rows * cols / 16 + 1), kThreads, 0, (cudaStream_t)stream>>>(
        d_codes, d_scales, rows, cols, reinterpret_cast<uint4*>(d_out));
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

extern "C" ep_status ep_q4_decode(const uint8_t* d_codes, const float* d_scales, int64_t n, int64_t block,
                                  const float* levels, uint16_t* d_out, ep_stream_t stream) {
    if (!d_codes || !d_scales || !levels || !d_out) return EP_ERR_INVALID_ARG;
    if (n <= 0 || (n & 1) || n > (int64_t(1) << 40)) return EP_ERR_SHAPE;
    if (block < 16 || block % 16 || block > (int64_t(1) << 30)) return EP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_codes) & 7) || (reinterpret_cast<uintptr_t>(d_scales) & 3) ||
        (reinterpret_cast<uintptr_t>(d_out) & 15))
        return EP_ERR_INVALID_ARG;
    Levels lv;
    for (int k = 0; k < 16; ++k) lv.v[k] = levels[k];
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t groups = (n + 15) >> 4;
    const int64_t per_wave = (int64_t)sms * (2048 / kThreads);
    int64_t grid = (groups + kThreads - 1) / kThreads;
    if (grid > per_wave * 4) grid = per_wave * 4;
    q4_decode_kernel<<<(unsigned)grid, kThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const uint2*>(d_codes), d_scales, n, block, lv, reinterpret_cast<uint4*>(d_out));
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
