// gemm_swapab.cu -- FP8 GEMM with fp32 block scales for few rows of A (decode, M <= 128):
// 128 rows of B take the MMA's M side and the MT (16, 32, 64 or 128) rows of A its N side, so
// the weight stream fills the tensor core's 128 lanes and every SM streams its own 128-row
// weight slab. The activation scales are staged in shared memory transposed, [kb][m]; the
// promotion warps fold each K block's TMEM partial into fp32 registers as in gemm_tn.cu.
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

template <int MT>
struct SwapCfg {
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int X_TILE = MT * BK;          // activation rows per stage
    static constexpr int STAGE = A_TILE + X_TILE;   // weight slab + activation rows
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * MT);
};

template <int MT>
__global__ void __launch_bounds__(SwapCfg<MT>::THREADS, 1)
    gemm_swapab_kernel(const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmA, const GemmArgs g,
                       const int stages) {
    using Cfg = SwapCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sW = smem;                                   // [stages][128 x 128] weights
    uint8_t* sX = smem + stages * A_TILE;                 // [stages][MT x 128] activations
    const int num_kb = g.K / BK;
    float* sAs = reinterpret_cast<float*>(sX + stages * Cfg::X_TILE);  // [num_kb][MT]
    float* sRaw = sAs + num_kb * MT;             // a_s rows m0 .. m0+MT-1 as stored: [MT][num_kb]
    float* sBs = sRaw + num_kb * MT;             // b_s row of this slab: [num_kb]
    const Ring ring = carve_ring(reinterpret_cast<uint8_t*>(sBs + ((num_kb + 3) & ~3)), stages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM;
    const int m0 = blockIdx.y * MT;

    // Prologue order: barriers; (weights declared constant: the whole weight ring, before
    // waiting for earlier kernels); wait; scales; TMEM; block sync; activations (and weights).
    const uint64_t keep = l2_policy_evict_last();    // activations: reused by every CTA
    const uint64_t stream = l2_policy_evict_first(); // weights: read once
    const int prefill = min(stages, num_kb);
    // The scales (a few hundred bytes: rows a_s[m0 .. m0+rows) and the slab's b_s row, both
    // contiguous) are requested by the promotion threads before the block synchronises, and the
    // weight stream only starts after it: the scales then return at unloaded latency instead of
    // queueing behind megabytes of weights.
    const int scale_rows = min(MT, g.M - m0);
    const float* as_rows = g.a_s + static_cast<int64_t>(m0) * num_kb;
    const float* bs_row = g.b_s + static_cast<int64_t>(blockIdx.x) * num_kb;
    if (threadIdx.x == 0) {
        init_ring(ring, stages, Cfg::EPI_WARPS);
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        // Weights the caller declared constant need not wait for the kernels before this one:
        // the ring starts filling while they finish.
        if (g.weights_constant) {
            for (int kb = 0; kb < prefill; ++kb) {
                mbar_arrive_expect_tx(&ring.full[kb], Cfg::STAGE);
                tma_load_2d_hint(sW + kb * A_TILE, &tmB, &ring.full[kb], kb * BK, n0, stream);
            }
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp >= 2) {
        const int t = threadIdx.x - 64;
        for (int i = t; i < scale_rows * num_kb; i += 32 * Cfg::EPI_WARPS)
            cp_async_4(sRaw + i, as_rows + i);
        for (int i = t; i < num_kb; i += 32 * Cfg::EPI_WARPS) cp_async_4(sBs + i, bs_row + i);
        cp_async_commit();
    }
    if (warp == 1) tmem_alloc(ring.tmem_holder, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;
    if (threadIdx.x == 0) {
        // fill the whole ring at once
        for (int kb = 0; kb < prefill; ++kb) {
            if (!g.weights_constant) {
                mbar_arrive_expect_tx(&ring.full[kb], Cfg::STAGE);
                tma_load_2d_hint(sW + kb * A_TILE, &tmB, &ring.full[kb], kb * BK, n0, stream);
            }
            tma_load_2d_hint(sX + kb * Cfg::X_TILE, &tmA, &ring.full[kb], kb * BK, m0, keep);
        }
    }

    if (warp == 0) {
        if (lane == 0) {
            int stage = prefill % stages;
            uint32_t phase = prefill == stages ? 1u : 0u;
            int64_t issued = prefill;
            bool ok = true;
            for (int kb = prefill; kb < num_kb; ++kb) {
                if (!mbar_wait(&ring.empty[stage], phase ^ 1)) {
                    record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&ring.full[stage], Cfg::STAGE);
                tma_load_2d_hint(sW + stage * A_TILE, &tmB, &ring.full[stage], kb * BK, n0, stream);
                tma_load_2d_hint(sX + stage * Cfg::X_TILE, &tmA, &ring.full[stage], kb * BK, m0,
                                 keep);
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) drain_tma(ring, stages, issued);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, MT);
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(&ring.tempty[buf], tphase ^ 1) ||
                    !mbar_wait(&ring.full[stage], phase)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t w_addr = smem_addr(sW + stage * A_TILE);
                const uint32_t x_addr = smem_addr(sX + stage * Cfg::X_TILE);
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * MT);
#pragma unroll
                for (int j = 0; j < BK / MMA_K; ++j)
                    mma_f8(d_tmem, smem_desc_k_sw128(w_addr + j * MMA_K),
                           smem_desc_k_sw128(x_addr + j * MMA_K), idesc, j > 0 ? 1u : 0u);
                mma_commit(&ring.empty[stage]);
                mma_commit(&ring.tfull[buf]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
                buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            mma_commit(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else {
        // Combined scales a_s[m, kb] * b_s[slab, kb] of this CTA's MT rows, transposed to
        // [kb][m] (zero past row M). Only the promotion warps need them, so the producer and
        // the MMA issuer start streaming while they are staged; reads are coalesced along kb.
        // Combined scales sAs[kb][m] = a_s[m0+m, kb] * b_s[slab, kb] (zero past row M), from the
        // rows copied at kernel start.
        cp_async_wait_all();
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::EPI_WARPS) : "memory");
        const int valid = scale_rows * num_kb;
        for (int i = threadIdx.x - 64; i < MT * num_kb; i += 32 * Cfg::EPI_WARPS) {
            const int j = i / num_kb, kb = i - j * num_kb;
            sAs[kb * MT + j] = i < valid ? sRaw[i] * sBs[kb] : 0.0f;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::EPI_WARPS) : "memory");
        const int quarter = warp & 3;
        const int n = n0 + quarter * 32 + lane;      // output column owned by this thread
        float acc[MT];
#pragma unroll
        for (int i = 0; i < MT; ++i) acc[i] = 0.0f;
        int buf = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
            if (!warp_wait(&ring.tfull[buf], tphase)) {
                if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * MT);
            const float* as_kb = sAs + kb * MT;
            if constexpr (MT >= 32) {
                // Chunks of 32 columns, the next load in flight while one is folded in.
                constexpr int NCH = MT / 32;
                float va[32], vb[32];
                tmem_ld_32cols(taddr, va);
                tmem_wait_ld_32(va);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float* cur = (c & 1) ? vb : va;
                    float* nxt = (c & 1) ? va : vb;
                    if (c + 1 < NCH) tmem_ld_32cols(taddr + 32 * (c + 1), nxt);
                    if (c + 1 == NCH) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ring.tempty[buf]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(as_kb + c * 32 + i);
                        fma2_into(acc + c * 32 + i, cur[i + 0], cur[i + 1], a4.x, a4.y);
                        fma2_into(acc + c * 32 + i + 2, cur[i + 2], cur[i + 3], a4.z, a4.w);
                    }
                    if (c + 1 < NCH) tmem_wait_ld_32(nxt);
                }
            } else {
                float v[16];
                tmem_ld_16cols(taddr, v);
                tmem_wait_ld_16(v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ring.tempty[buf]);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(as_kb + i);
                    fma2_into(acc + i, v[i + 0], v[i + 1], a4.x, a4.y);
                    fma2_into(acc + i + 2, v[i + 2], v[i + 3], a4.z, a4.w);
                }
            }
            buf ^= 1;
            if (buf == 0) tphase ^= 1;
        }
        if (ok && n < g.N) {
            __nv_bfloat16* c = static_cast<__nv_bfloat16*>(g.c);
#pragma unroll
            for (int j = 0; j < MT; ++j)
                if (m0 + j < g.M) c[static_cast<int64_t>(m0 + j) * g.N + n] = __float2bfloat16_rn(acc[j]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int MT>
cudaError_t launch_swap(const CUtensorMap& tmB, const CUtensorMap& tmA, const GemmArgs& g,
                        cudaStream_t stream) {
    using Cfg = SwapCfg<MT>;
    const int num_kb = g.K / BK;
    // scale staging: transposed [num_kb][MT], raw rows [MT][num_kb], b_s row, one barrier
    const int scale_bytes = 2 * num_kb * MT * 4 + ((num_kb + 3) & ~3) * 4 + 16;
    const int fixed = 1024 + scale_bytes + ring_bytes(kMaxStages);
    int stages = (kSmemLimit - fixed) / Cfg::STAGE;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;   // K too large for the scale staging
    const int smem = 1024 + stages * Cfg::STAGE + scale_bytes + ring_bytes(stages);
    cudaError_t e = set_smem(gemm_swapab_kernel<MT>, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((g.N + BM - 1) / BM, (g.M + MT - 1) / MT);
    return launch_pdl(gemm_swapab_kernel<MT>, grid, Cfg::THREADS, smem, stream, tmB, tmA, g,
                      stages);
}

}  // namespace

cudaError_t launch_gemm_swapab(const CUtensorMap& tmB, const CUtensorMap& tmA,
                               const GemmArgs& g, int MT, cudaStream_t stream) {
    switch (MT) {
        case 16: return launch_swap<16>(tmB, tmA, g, stream);
        case 32: return launch_swap<32>(tmB, tmA, g, stream);
        case 64: return launch_swap<64>(tmB, tmA, g, stream);
        case 128: return launch_swap<128>(tmB, tmA, g, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_swapab(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
