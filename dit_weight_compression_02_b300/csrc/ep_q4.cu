// GPU reconstruction of the fixed-width 4-bit comparators (NF4 / INT4):
// out[i] = BF16(levels[code_i] * scale[i / block]), one FP32 product rounded
// to nearest even.  The codes are packed two per byte, element 2j in the low
// nibble of byte j.
//
// The work is HBM-bound (0.5 B of codes + 4 / block B of scale read and 2 B
// written per weight): each thread turns 16 codes (one 8-byte load, one
// scale, since block % 16 == 0) into 32 output bytes with two 16-byte stores;
// a grid of whole waves strides over the groups.  A ragged tail (n % 16 != 0)
// is finished element by element by the thread that owns the last group.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "entropack.h"

namespace {

struct Levels {
    float v[16];
};

constexpr int kThreads = 256;

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

}  // namespace

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
