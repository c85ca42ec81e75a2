// linear_bf16.cu -- the bf16 path of linear() with FP8 weights: y = x . W'^T, where W' is the
// bf16 weight that weight_dequant would produce ("DeepSeek-V3 Administrator & Developer Guide",
// §6.3: with gemm_impl = "bf16" the FP8 weight is dequantised (§8.5.2) and a bf16 GEMM runs;
// the weight is dequantised per tile in shared memory instead of being written to and read back
// from HBM as bf16.
//
// Decode orientation (M <= 64): 128-row slabs of W take the MMA's M side, the MT rows of x its
// N side; one CTA per slab streams its e4m3 weight (half the bytes of bf16 weights).
//   warp 0          TMA producer of the deep ring: per K block the e4m3 weight tile (the HBM
//                   stream) and the bf16 rows of x (128-byte swizzle, two 64-wide halves)
//   warp 1          MMA issuer: 8 x tcgen05.mma kind::f16 (K = 16) per K block into one TMEM
//                   accumulator for the whole K loop (the block scale is inside W')
//   warps 2 .. 5    epilogue: the accumulator to bf16 y
//   warps 6 .. 13   dequantisers: per K block, e4m3 tile -> bf16 W' tile (fp32 product with
//                   the block scale, rounded to bf16: weight_dequant's arithmetic) written
//                   straight into TMEM with tcgen05.st (lane = weight row, 32-bit column =
//                   two consecutive K), where the MMA takes its A operand: a second, shallow
//                   ring of two 64-column slots. W' never touches shared memory, which the
//                   TMA stream, the dequantisers' reads and the MMA's reads of x already share.
// A slot of the deep ring is free once the dequantisers have read its weight tile and the MMA
// has read its rows of x.
#include "gemm_common.cuh"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fp8bs {

namespace {

template <int MT>
struct LinCfg {
    static constexpr int EPI_WARPS = 4;
    static constexpr int DQ_WARPS = 8;
    static constexpr int DQ0 = 2 + EPI_WARPS;            // first dequantiser warp
    static constexpr int THREADS = 32 * (2 + EPI_WARPS + DQ_WARPS);
    static constexpr int WQ_TILE = BM * BK;              // e4m3 weight tile (128 x 128)
    static constexpr int HALF = 64;                      // bf16 K elements per 128-byte row
    static constexpr int XB_TILE = MT * BK * 2;          // bf16 activation tile: two halves
    static constexpr int A_SLOT = WQ_TILE + XB_TILE;     // deep ring: weight codes + rows of x
    static constexpr int W_COL0 = 64;                    // TMEM: accumulator in 0 .. MT-1, then
    static constexpr int W_COLS = BK / 2;                // W' slots of 64 columns (bf16 pairs)
    static constexpr uint32_t TMEM_COLS = 256;
};

// Eight e4m3 codes (one 64-bit word) -> eight bf16 (four words): fp32(code) * scale, rounded to
// binary32 then to bf16 -- bit for bit what weight_dequant writes.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

__device__ __forceinline__ void dequant8(uint32_t lo, uint32_t hi, float sc, uint32_t* out) {
    const uint32_t w[2] = {lo, hi};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const __nv_fp8x2_storage_t pair =
                static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu);
            const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
            out[2 * i + h] = bf16x2(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
        }
    }
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile (8-row atoms
// of 1024 bytes: the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ int sw128(int r, int c) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

template <int MT>
__global__ void __launch_bounds__(LinCfg<MT>::THREADS, 1)
    linear_bf16_swap_kernel(const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ CUtensorMap tmX,
                            const float* __restrict__ w_s, void* y, const int M, const int N,
                            const int K, const int sa, const int sb, const int weights_constant) {
    using Cfg = LinCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sA = smem;                              // [sa][W e4m3 | x bf16]
    uint64_t* fullA = reinterpret_cast<uint64_t*>(sA + sa * Cfg::A_SLOT);
    uint64_t* emptyA = fullA + sa;
    uint64_t* deqB = emptyA + sa;
    uint64_t* emptyB = deqB + sb;
    uint64_t* tfull = emptyB + sb;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_kb = K / BK;
    const int n0 = blockIdx.x * BM;
    const int m0 = blockIdx.y * MT;
    const float* ws_row = w_s + static_cast<int64_t>(blockIdx.x) * num_kb;
    const int prefill = min(sa, num_kb);
    const uint64_t stream = l2_policy_evict_first();  // weights: read once
    const uint64_t keep = l2_policy_evict_last();     // x: read by every CTA

    if (threadIdx.x == 0) {
        for (int i = 0; i < sa; ++i) {
            mbar_init(&fullA[i], 1);
            mbar_init(&emptyA[i], Cfg::DQ_WARPS + 1);   // dequantisers + the MMA's commit
        }
        for (int i = 0; i < sb; ++i) {
            mbar_init(&deqB[i], Cfg::DQ_WARPS);
            mbar_init(&emptyB[i], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        // Weights the caller declared constant start streaming before earlier kernels finish.
        if (weights_constant)
            for (int kb = 0; kb < prefill; ++kb) {
                mbar_arrive_expect_tx(&fullA[kb], Cfg::A_SLOT);
                tma_load_2d_hint(sA + kb * Cfg::A_SLOT, &tmW, &fullA[kb], kb * BK, n0, stream);
            }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 1) tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            auto load_x = [&](int slot, int kb) {
                uint8_t* xs = sA + slot * Cfg::A_SLOT + Cfg::WQ_TILE;
                tma_load_2d_hint(xs, &tmX, &fullA[slot], kb * BK, m0, keep);
                tma_load_2d_hint(xs + MT * 128, &tmX, &fullA[slot], kb * BK + Cfg::HALF, m0, keep);
            };
            for (int kb = 0; kb < prefill; ++kb) {
                if (!weights_constant) {
                    mbar_arrive_expect_tx(&fullA[kb], Cfg::A_SLOT);
                    tma_load_2d_hint(sA + kb * Cfg::A_SLOT, &tmW, &fullA[kb], kb * BK, n0,
                                     stream);
                }
                load_x(kb, kb);
            }
            int stage = prefill % sa;
            uint32_t phase = prefill == sa ? 1u : 0u;
            int64_t issued = prefill;
            for (int kb = prefill; kb < num_kb; ++kb) {
                if (!mbar_wait(&emptyA[stage], phase ^ 1)) {
                    record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                    // drain what is in flight before leaving
                    const int64_t first = issued > sa ? issued - sa : 0;
                    for (int64_t i = first; i < issued; ++i)
                        if (!mbar_wait(&fullA[i % sa], static_cast<uint32_t>((i / sa) & 1),
                                       kDrainLimitNs))
                            record_error(FP8BS_DEVERR_DRAIN_WAIT);
                    break;
                }
                mbar_arrive_expect_tx(&fullA[stage], Cfg::A_SLOT);
                tma_load_2d_hint(sA + stage * Cfg::A_SLOT, &tmW, &fullA[stage], kb * BK, n0,
                                 stream);
                load_x(stage, kb);
                ++issued;
                if (++stage == sa) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, MT);
            int a = 0, b = 0;
            uint32_t pa = 0, pb = 0;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&deqB[b], pb) || !mbar_wait(&fullA[a], pa)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t w_tmem =
                    tmem_base + static_cast<uint32_t>(Cfg::W_COL0 + b * Cfg::W_COLS);
                const uint32_t x_addr = smem_addr(sA + a * Cfg::A_SLOT + Cfg::WQ_TILE);
#pragma unroll
                for (int j = 0; j < BK / 16; ++j) {
                    const uint32_t h = j / 4, o = (j % 4) * 32;   // 64-wide half, 16-wide step
                    mma_bf16_ta(tmem_base, w_tmem + 8 * j,
                                smem_desc_k_sw128(x_addr + h * (MT * 128) + o), idesc,
                                (kb > 0 || j > 0) ? 1u : 0u);
                }
                mma_commit(&emptyB[b]);
                mma_commit(&emptyA[a]);
                if (++b == sb) {
                    b = 0;
                    pb ^= 1;
                }
                if (++a == sa) {
                    a = 0;
                    pa ^= 1;
                }
            }
            mma_commit(tfull);
            mma_commit(drain);
            if (!mbar_wait(drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else if (warp >= Cfg::DQ0) {
        // Dequantisers: warp w handles the TMEM lane quarter w % 4 (weight rows 32 (w % 4) ..
        // +31, one per lane) and one 64-wide half of the K block; each lane converts the 64
        // codes of its row's half and stores them as 32 columns of bf16 pairs.
        const int quarter = warp & 3;
        const int khalf = (warp - Cfg::DQ0) >> 2;
        const int r = quarter * 32 + lane;
        int a = 0, b = 0;
        uint32_t pa = 0, pb = 0;
        for (int kb = 0; kb < num_kb; ++kb) {
            if (!warp_wait(&emptyB[b], pb ^ 1) || !warp_wait(&fullA[a], pa)) {
                if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                break;
            }
            tc_fence_after();
            const float sc = __ldg(ws_row + kb);
            const uint8_t* qslot = sA + a * Cfg::A_SLOT;
            uint32_t o[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(qslot + sw128(r, 4 * khalf + i));
                dequant8(v.x, v.y, sc, o + 8 * i);
                dequant8(v.z, v.w, sc, o + 8 * i + 4);
            }
            tmem_st_32cols(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(Cfg::W_COL0 + b * Cfg::W_COLS + 32 * khalf),
                           o);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&emptyA[a]);
                mbar_arrive(&deqB[b]);
            }
            if (++a == sa) {
                a = 0;
                pa ^= 1;
            }
            if (++b == sb) {
                b = 0;
                pb ^= 1;
            }
        }
    } else {
        // Epilogue: TMEM lane = output column n0 + 32 * quarter + lane, columns = rows of x.
        const int quarter = warp & 3;
        const int n = n0 + quarter * 32 + lane;
        if (warp_wait(tfull, 0)) {
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            float acc[MT];
            if constexpr (MT >= 32) {
#pragma unroll
                for (int c = 0; c < MT / 32; ++c) tmem_ld_32cols(taddr + 32 * c, acc + 32 * c);
#pragma unroll
                for (int c = 0; c < MT / 32; ++c) tmem_wait_ld_32(acc + 32 * c);
            } else {
                tmem_ld_16cols(taddr, acc);
                tmem_wait_ld_16(acc);
            }
            if (n < N) {
                __nv_bfloat16* yc = static_cast<__nv_bfloat16*>(y);
#pragma unroll
                for (int j = 0; j < MT; ++j)
                    if (m0 + j < M) yc[static_cast<int64_t>(m0 + j) * N + n] = __float2bfloat16_rn(acc[j]);
            }
        } else if (lane == 0) {
            record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int MT>
cudaError_t launch_lin(const CUtensorMap& tmW, const CUtensorMap& tmX, const float* w_s, void* y,
                       int M, int N, int K, int weights_constant, cudaStream_t stream) {
    using Cfg = LinCfg<MT>;
    // a shallow bf16 ring (two slots), the rest of shared memory for the e4m3 weight stream
    const int sb = 2;                              // W' slots in TMEM
    const int bar_bytes = 8 * (2 * kMaxStages + 2 * sb + 2) + 16;
    int sa = (kSmemLimit - 1024 - bar_bytes) / Cfg::A_SLOT;
    if (sa > kMaxStages) sa = kMaxStages;
    if (sa < 2) return cudaErrorInvalidValue;
    const int smem = 1024 + sa * Cfg::A_SLOT + bar_bytes;
    cudaError_t e = set_smem(linear_bf16_swap_kernel<MT>, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((N + BM - 1) / BM, (M + MT - 1) / MT);
    return launch_pdl(linear_bf16_swap_kernel<MT>, grid, Cfg::THREADS, smem, stream, tmW, tmX,
                      w_s, y, M, N, K, sa, sb, weights_constant);
}

}  // namespace

cudaError_t launch_linear_bf16_swap(const CUtensorMap& tmW, const CUtensorMap& tmX,
                                    const float* w_s, void* y, int M, int N, int K, int MT,
                                    int weights_constant, cudaStream_t stream) {
    switch (MT) {
        case 16: return launch_lin<16>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        case 32: return launch_lin<32>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        case 64: return launch_lin<64>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_linear(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
