// quant.cu -- the two bandwidth kernels of the path:
//   act_quant       ("DeepSeek-V3 Administrator & Developer Guide", §8.5.1 act_quant_kernel)
//   weight_dequant  (same guide, §8.5.2 weight_dequant_kernel; scale shape §6.3 item 2)
//
// Both stream HBM once with 16-byte vector accesses. act_quant: 8 threads own one 128-element
// block (16 bf16 = 32 bytes each), reduce |x| with 3 xor-shuffles inside the 8-lane group and
// write 16 e4m3 codes (16 bytes) each; lane 0 of the group writes the block's fp32 scale.
// act_quant issues the loads of two grid-stride steps before using either, so that enough
// bytes are in flight per SM to cover HBM latency (64 bytes per thread).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bs {

namespace {

// Grid-stride over groups of 16 elements; thread g handles x[16g .. 16g+15], which lie in
// block g/8 (blocks are contiguous because K % 128 == 0). Two steps per iteration: both
// groups' loads are issued first.
template <bool UE8M0>
__global__ void __launch_bounds__(256) act_quant_kernel(const uint4* __restrict__ x,
                                                        uint4* __restrict__ y,
                                                        float* __restrict__ s,
                                                        int64_t num_groups) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int lane = threadIdx.x & 31;
    // Every lane of a warp takes the same branches (num_groups is a multiple of 8 and the grid
    // covers whole warps; the tests below use the warp's first group), so the shuffles inside
    // quant_block16 are always full-warp. Inactive lanes quantise zeros and store nothing.
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         g - lane < num_groups; g += 2 * stride) {
        const int64_t g2 = g + stride;
        const bool a1 = g < num_groups, a2 = g2 < num_groups;
        uint32_t w1[8] = {}, w2[8] = {};
        if (a1) {
            const uint4 v0 = __ldcs(x + 2 * g), v1 = __ldcs(x + 2 * g + 1);
            w1[0] = v0.x; w1[1] = v0.y; w1[2] = v0.z; w1[3] = v0.w;
            w1[4] = v1.x; w1[5] = v1.y; w1[6] = v1.z; w1[7] = v1.w;
        }
        if (a2) {
            const uint4 v0 = __ldcs(x + 2 * g2), v1 = __ldcs(x + 2 * g2 + 1);
            w2[0] = v0.x; w2[1] = v0.y; w2[2] = v0.z; w2[3] = v0.w;
            w2[4] = v1.x; w2[5] = v1.y; w2[6] = v1.z; w2[7] = v1.w;
        }
        uint32_t out[4];
        float sc = quant_block16<UE8M0>(w1, out);
        if (a1) {
            __stcs(y + g, make_uint4(out[0], out[1], out[2], out[3]));
            if ((threadIdx.x & 7) == 0) s[g >> 3] = sc;
        }
        if (g2 - lane < num_groups) {
            sc = quant_block16<UE8M0>(w2, out);
            if (a2) {
                __stcs(y + g2, make_uint4(out[0], out[1], out[2], out[3]));
                if ((threadIdx.x & 7) == 0) s[g2 >> 3] = sc;
            }
        }
    }
}

// weight_dequant, vector path (K % 16 == 0): thread g converts 16 consecutive codes of one row.
__global__ void __launch_bounds__(256) weight_dequant_vec_kernel(const uint4* __restrict__ w,
                                                                 const float* __restrict__ s,
                                                                 uint4* __restrict__ y,
                                                                 int64_t N, int64_t K) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t groups_per_row = K >> 4;
    const int64_t kblocks = (K + 127) >> 7;
    const int64_t total = N * groups_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += stride) {
        const int64_t n = g / groups_per_row;
        const int64_t k = (g - n * groups_per_row) << 4;
        const float sc = __ldg(s + (n >> 7) * kblocks + (k >> 7));
        const uint4 v = __ldcs(w + g);
        const uint32_t words[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const __nv_fp8x2_storage_t pair =
                    static_cast<__nv_fp8x2_storage_t>((words[i] >> (16 * h)) & 0xFFFFu);
                const float2 f = __half22float2(
                    __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
                const __nv_bfloat162 b =
                    __floats2bfloat162_rn(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
                out[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
            }
        }
        __stcs(y + 2 * g, make_uint4(out[0], out[1], out[2], out[3]));
        __stcs(y + 2 * g + 1, make_uint4(out[4], out[5], out[6], out[7]));
    }
}

// weight_dequant, general path (any K): one element per thread.
__global__ void __launch_bounds__(256) weight_dequant_scalar_kernel(
    const uint8_t* __restrict__ w, const float* __restrict__ s, __nv_bfloat16* __restrict__ y,
    int64_t N, int64_t K) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t kblocks = (K + 127) >> 7;
    const int64_t total = N * K;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int64_t n = i / K;
        const int64_t k = i - n * K;
        const float sc = __ldg(s + (n >> 7) * kblocks + (k >> 7));
        const __half h = __half(__nv_cvt_fp8_to_halfraw(w[i], __NV_E4M3));
        y[i] = __float2bfloat16_rn(__fmul_rn(__half2float(h), sc));
    }
}

// Blocks of 256 threads for `threads` work items, at most `per_sm` per SM (grid-stride beyond).
int grid_for(int64_t threads, int num_sms, int per_sm) {
    const int64_t blocks = (threads + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K, bool ue8m0,
                             int num_sms, cudaStream_t stream) {
    // Up to 2^26 elements (8192 x 7168 and below), at most 8 blocks of 256 threads per SM
    // (two rounds of the four that fit at this kernel's 51 registers), striding over the
    // groups: measured 3-9 % faster from 2048 x 7168 to 8192 x 7168 than 32 per SM, whose
    // blocks retire and relaunch while the stream runs. Larger inputs keep 32 per SM (a
    // resident grid was measured slower at 4096 x 18432).
    const int64_t groups = M * K / 16;
    const int grid = grid_for(groups, num_sms, M * K <= (int64_t{1} << 26) ? 8 : 32);
    const uint4* xv = static_cast<const uint4*>(x);
    uint4* yv = static_cast<uint4*>(y);
    if (ue8m0) return launch_pdl(act_quant_kernel<true>, grid, 256, 0, stream, xv, yv, s, groups);
    return launch_pdl(act_quant_kernel<false>, grid, 256, 0, stream, xv, yv, s, groups);
}

cudaError_t launch_weight_dequant(const void* w, const float* s, void* y, int64_t N, int64_t K,
                                  cudaStream_t stream) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool vec = (K % 16 == 0) && (reinterpret_cast<uintptr_t>(w) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    if (vec)
        return launch_pdl(weight_dequant_vec_kernel, grid_for(N * K / 16, sms, 32), 256, 0,
                          stream, static_cast<const uint4*>(w), s, static_cast<uint4*>(y), N, K);
    return launch_pdl(weight_dequant_scalar_kernel, grid_for(N * K, sms, 32), 256, 0, stream,
                      static_cast<const uint8_t*>(w), s, static_cast<__nv_bfloat16*>(y), N, K);
}

}  // namespace fp8bs
