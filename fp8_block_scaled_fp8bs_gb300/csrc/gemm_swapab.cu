// gemm_swapab.cu -- FP8 GEMM with fp32 block scales for few rows of A (decode, M <= 128):
// 128 rows of B take the MMA's M side and the MT (16, 32, 64 or 128) rows of A its N side, so
// the weight stream fills the tensor core's 128 lanes and every SM streams its own 128-row
// weight slab. Two MMA issuers take the K blocks in turn, each into its own pair of TMEM
// buffers, and the promotion warps fold each K block's partial into fp32 registers with the
// combined scale a_s[m, kb] * b_s[slab, kb], as in gemm_tn.cu.
//
// Split K (quantised input only): when the slabs alone would leave most SMs idle (N = 2048 or
// 576 at decode: 16 or 5 slabs on 152 SMs), S CTAs, launched as one thread-block cluster, share
// each slab: CTA r streams K blocks [r*num_kb/S, (r+1)*num_kb/S) of it, and the S partial sums
// of the C rows are added in rank order (K order) through distributed shared memory before the
// bf16 store -- no workspace and no flags, and the additions happen in a fixed order.
//
// Two ways in for the activations:
//   quantised (fp8bs_gemm): TMA brings e4m3 rows of A; their scales are staged in shared memory
//       transposed to [kb][m] before the main loop.
//   bf16 (fp8bs_act_quant_gemm, FUSED; at most 16 rows): before its main loop every CTA reads
//       x (bf16) and quantises all of it with act_quant's arithmetic ("DeepSeek-V3 Administrator
//       & Developer Guide", §8.5.1) into a resident e4m3 operand -- one 16-row tile per K block
//       in the layout TMA would have written (128-byte swizzle) -- and its block scales, while
//       the weight ring fills. No kernel and no grid-wide synchronisation stands between the
//       previous layer and this GEMM; the CTAs of the first weight slab also write y and s.
//       (Quantising each K block as its stage arrived, with a proxy fence per block, ran at
//       ~1030 clk per K block against ~700 for the weight stream.)
#include "gemm_common.cuh"
#include "quant_math.cuh"

namespace fp8bs {

namespace {

template <int MT, bool FUSED>
struct SwapCfg {
    static_assert(!FUSED || MT == 16, "in-kernel quantisation: 16-row tiles");
    static constexpr int EPI_WARPS = 4;
    static constexpr int Q_WARPS = FUSED ? 4 : 0;   // quantiser warps, after the promotion warps
    static constexpr int Q_WARP0 = 2 + EPI_WARPS;
    static constexpr int S_WARPS = FUSED ? 0 : 1;   // scale warp (quantised input), same place
    // MMA issuers: warp 1 and the last warp take the K blocks in turn, each into its own pair of
    // TMEM buffers. One thread issuing alone spends ~70 clk per tcgen05 instruction, 4 MMAs and
    // 2 commits per K block: that, not the weight stream, had set the pace (N = 18432, M = 1:
    // 22.7 us, 20.7 us with the MMAs left out; N = 7168, K = 18432: 28.3 against 22.6 us).
    static constexpr int ISSUERS = 2;
    static constexpr int ISSUER2 = 2 + EPI_WARPS + Q_WARPS + S_WARPS;
    static constexpr int NBUF = 2 * ISSUERS;        // TMEM partial buffers (K block kb: kb % 4)
    static constexpr int THREADS = 64 + 32 * (EPI_WARPS + Q_WARPS + S_WARPS + ISSUERS - 1);
    static constexpr int X_TILE = MT * BK;          // e4m3 activation rows of one K block
    // A stage: a weight tile and (quantised input) the activation tile; FUSED keeps the
    // activations resident instead.
    static constexpr int STAGE = A_TILE + (FUSED ? 0 : X_TILE);
    static constexpr int TX_BYTES = STAGE;          // bytes TMA brings per stage
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(NBUF * MT);
    static constexpr int BAR_BYTES = 2 * NBUF * 8;  // tfull[NBUF], tempty[NBUF] after the ring
};

// Shared-memory bytes after the stages, for a CTA that takes nkb K blocks: (FUSED) the
// resident e4m3 activation tiles [nkb][MT x 128], then the transposed scales [nkb][MT], then
// (quantised input) the raw a_s rows [MT][nkb], and the b_s row.
template <int MT, bool FUSED>
__host__ __device__ constexpr int swap_scale_bytes(int nkb) {
    return (FUSED ? nkb * MT * BK : 0) + nkb * MT * 4 + (FUSED ? 0 : nkb * MT * 4) +
           ((nkb + 3) & ~3) * 4 + 16;
}

// Bounded spin until *p >= target.
__device__ __forceinline__ bool spin_until_at_least(const int* p, int target) {
    const volatile int* v = p;
    if (*v >= target) return true;
    const uint64_t t0 = global_timer_ns();
    while (*v < target)
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// Split-K exchange: CTA q of the cluster adds up rows [q*wm, (q+1)*wm) of C, wm a multiple of
// 4 (so that four consecutive rows travel as one float4); its receive area (at the start of the
// stage memory, free once every CTA of the cluster has finished its K loop) holds S slots of
// 128 columns x wm rows, column-major with a row pitch of p4 float4 (p4 odd: the float4 stores
// of eight consecutive columns fall in distinct bank groups).
__host__ __device__ constexpr int swap_rows_per_rank(int rows, int S) {
    return ((rows + S - 1) / S + 3) / 4 * 4;
}
__host__ __device__ constexpr int swap_pitch4(int wm) { return (wm / 4) | 1; }
__host__ __device__ constexpr int swap_recv_bytes(int MT, int S) {
    return S * BM * swap_pitch4(swap_rows_per_rank(MT, S)) * 16;
}

// PLAIN: one group starting at row 0, no split, not `early` (every fused launch, and the usual
// decode GEMM). Its instantiation has none of the split exchange, group lookup or per-group row
// count: compiled with them, the same launches of the decode step ran ~1.4 % slower (N = 18432,
// K = 7168, M = 1..64: 23.16 against 22.84 us at M = 1, 25.92 against 25.31 us at M = 64).
template <int MT, bool FUSED, bool PLAIN>
__global__ void __launch_bounds__(SwapCfg<MT, FUSED>::THREADS, 1)
    gemm_swapab_kernel(const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmA, const GemmArgs g,
                       const __grid_constant__ GroupTable gt, const int stages,
                       const FusedQuant fq, const int ksplit, const int early_arg) {
    static_assert(PLAIN || !FUSED, "fused launches are plain");
    using Cfg = SwapCfg<MT, FUSED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sW = smem;                                   // [stages][128 x 128] weights
    // [stages][MT x 128] e4m3 activations, or (FUSED) [num_kb][MT x 128] resident
    uint8_t* sX = smem + stages * A_TILE;
    const int num_kb = g.K / BK;
    // This CTA's slab and K blocks kb_lo .. kb_lo + nkb - 1 (all of them unless split).
    const int S = PLAIN ? 1 : ksplit;
    const bool early = !PLAIN && early_arg != 0;
    const int slab = blockIdx.x / S;
    const int kb_lo = (blockIdx.x - slab * S) * num_kb / S;
    const int nkb = (blockIdx.x - slab * S + 1) * num_kb / S - kb_lo;
    float* sAs = reinterpret_cast<float*>(sX + (FUSED ? num_kb : stages) * Cfg::X_TILE);
    float* sRaw = sAs + nkb * MT;      // a_s rows m0 .. m0+MT-1, this CTA's K blocks: [MT][nkb]
    float* sBs = sRaw + (FUSED ? 0 : nkb * MT);          // b_s row of this slab: [nkb]
    uint8_t* ring_mem = reinterpret_cast<uint8_t*>(sBs + ((nkb + 3) & ~3));
    const Ring ring = carve_ring(ring_mem, stages);
    // The partial buffers' barriers (the ring's own two pairs serve one issuer only).
    uint64_t* tfull = reinterpret_cast<uint64_t*>(ring_mem + ring_bytes(stages));
    uint64_t* tempty = tfull + Cfg::NBUF;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = slab * BM;
    // Group and rows of this CTA: blockIdx.y counts the MT-row tiles of all groups, group by
    // group; group grp owns rows row_off[grp] .. row_off[grp+1]-1 of A, a_s and C, rows
    // grp*N .. of the stacked B and scale rows grp*ceil(N/128) .. of the stacked b_s.
    int grp = 0;
    if constexpr (!PLAIN)
        while (static_cast<int>(blockIdx.y) >= gt.tile_off[grp + 1]) ++grp;
    const int m0 = PLAIN ? static_cast<int>(blockIdx.y) * MT
                         : gt.row_off[grp] + (static_cast<int>(blockIdx.y) - gt.tile_off[grp]) * MT;
    const int b_row = grp * g.N + n0;                    // row of the stacked B

    // Prologue order: barriers; (weights declared constant: the whole weight ring, before
    // waiting for earlier kernels); wait; scales; TMEM; block sync; activations (and weights).
    const uint64_t keep = l2_policy_evict_last();    // activations: reused by every CTA
    const uint64_t stream = l2_policy_evict_first(); // weights: read once
    const int prefill = min(stages, nkb);
    // The scales (a few hundred bytes: rows a_s[m0 .. m0+rows) and the slab's b_s row, both
    // contiguous) are requested by the promotion threads before the block synchronises, and the
    // weight stream only starts after it: the scales then return at unloaded latency instead of
    // queueing behind megabytes of weights.
    const int scale_rows = min(MT, (PLAIN ? g.M : gt.row_off[grp + 1]) - m0);
    const float* as_rows = g.a_s + static_cast<int64_t>(m0) * num_kb;
    const float* bs_row =
        g.b_s + (static_cast<int64_t>(grp) * ((g.N + BM - 1) / BM) + slab) * num_kb + kb_lo;
    // Quantised input: the scale warp counts here the K blocks of sAs it has filled.
    int* sScaleDone = reinterpret_cast<int*>(ring.tmem_holder + 1);
    if (threadIdx.x == 0) {
        // each issuer commits its final drain (the ring's own tfull / tempty go unused)
        init_ring(ring, stages, Cfg::EPI_WARPS, 1, Cfg::ISSUERS);
        for (int b = 0; b < Cfg::NBUF; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        fence_barrier_init();
        *sScaleDone = 0;
        if constexpr (!FUSED) tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        // Weights the caller declared constant need not wait for the kernels before this one:
        // the ring starts filling while they finish.
        if (g.weights_constant) {
            for (int i = 0; i < prefill; ++i) {
                mbar_arrive_expect_tx(&ring.full[i], Cfg::TX_BYTES);
                tma_load_2d_hint(sW + i * A_TILE, &tmB, &ring.full[i], (kb_lo + i) * BK, b_row,
                                 stream);
            }
        }
    }
    // `early`: this launch reads nothing the kernel just before it writes (the second of two
    // launches over disjoint groups), so it starts its work at once and waits for that kernel
    // only before exiting -- its own completion then still implies the other's.
    if (!early) grid_dependency_wait();
    grid_launch_dependents();
    if (FUSED && warp >= 2 && warp < 2 + Cfg::EPI_WARPS) {
        const int t = threadIdx.x - 64;
        for (int i = t; i < num_kb; i += 32 * Cfg::EPI_WARPS) cp_async_4(sBs + i, bs_row + i);
        cp_async_commit();
    }
    if constexpr (FUSED) {
        // Every warp quantises x whole. Task t: row t / num_kb, K block t % num_kb; eight lanes
        // per task, lane l taking elements 16 (l % 8) .. +15 of the block (quant_block16's
        // layout), four tasks per warp at a time, and each lane loads BATCH tasks before it
        // quantises any. Loop bounds are warp-uniform: quant_block16 shuffles across the warp.
        constexpr int NW = Cfg::THREADS / 32;
        constexpr int BATCH = 4;
        const int sub = lane >> 3;
        const int chunk = lane & 7;
        const int rows = scale_rows;
        const int tasks = rows * num_kb;
        const bool writer = blockIdx.x == 0;              // first slab: also write y and s
        for (int base = warp * 4; base < tasks; base += NW * 4 * BATCH) {
            uint32_t w[BATCH][8];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int t = base + b * NW * 4 + sub;
                uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
                if (t < tasks) {
                    const int row = t / num_kb;
                    const int kb = t - row * num_kb;
                    const uint4* src =
                        fq.x + ((static_cast<int64_t>(m0 + row) * g.K + kb * BK + chunk * 16) >> 3);
                    v0 = __ldg(src);
                    v1 = __ldg(src + 1);
                }
                w[b][0] = v0.x; w[b][1] = v0.y; w[b][2] = v0.z; w[b][3] = v0.w;
                w[b][4] = v1.x; w[b][5] = v1.y; w[b][6] = v1.z; w[b][7] = v1.w;
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                if (base + b * NW * 4 >= tasks) break;
                const int t = base + b * NW * 4 + sub;
                uint32_t out[4];
                const float sc = fq.ue8m0 ? quant_block16<true>(w[b], out)
                                          : quant_block16<false>(w[b], out);
                if (t < tasks) {
                    const int row = t / num_kb;
                    const int kb = t - row * num_kb;
                    const uint4 q = make_uint4(out[0], out[1], out[2], out[3]);
                    *reinterpret_cast<uint4*>(sX + kb * Cfg::X_TILE + (row >> 3) * 1024 +
                                              (row & 7) * 128 + ((chunk ^ (row & 7)) << 4)) = q;
                    if (chunk == 0) sAs[kb * MT + row] = sc;
                    if (writer) {
                        const int64_t grow = m0 + row;
                        fq.y[(grow * g.K + kb * BK + chunk * 16) >> 4] = q;
                        if (chunk == 0) fq.s[grow * num_kb + kb] = sc;
                    }
                }
            }
        }
        // Rows past M: zero codes and zero scales in every K block.
        for (int i = threadIdx.x; i < (MT - rows) * num_kb * 8; i += Cfg::THREADS) {
            const int row = rows + i / (num_kb * 8);
            const int rem = i - (row - rows) * num_kb * 8;
            const int kb = rem >> 3;
            const int ch = rem & 7;
            *reinterpret_cast<uint4*>(sX + kb * Cfg::X_TILE + (row >> 3) * 1024 + (row & 7) * 128 +
                                      ((ch ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            if (ch == 0) sAs[kb * MT + row] = 0.0f;
        }
        // The tiles are read next by the tensor core (async proxy), after the block barrier.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (!FUSED && warp == Cfg::Q_WARP0) {
        if (S == 1) {
            // The rows are one contiguous run of scale_rows * num_kb floats: 16-byte copies
            // when its start and length allow (sRaw is 16-byte aligned), else 4-byte ones.
            const int count = scale_rows * num_kb;
            if ((reinterpret_cast<uintptr_t>(as_rows) & 15) == 0 && (count & 3) == 0) {
                for (int i = 4 * lane; i < count; i += 4 * 32) cp_async_16(sRaw + i, as_rows + i);
            } else {
                for (int i = lane; i < count; i += 32) cp_async_4(sRaw + i, as_rows + i);
            }
        } else if ((reinterpret_cast<uintptr_t>(as_rows) & 15) == 0 &&
                   ((num_kb | kb_lo | nkb) & 3) == 0) {
            // This CTA's K blocks of each row, 16 bytes at a time (every segment aligned).
            for (int i = 4 * lane; i < scale_rows * nkb; i += 4 * 32) {
                const int j = i / nkb;
                cp_async_16(sRaw + i,
                            as_rows + static_cast<int64_t>(j) * num_kb + kb_lo + i - j * nkb);
            }
        } else {
            // This CTA's K blocks of each row.
            for (int i = lane; i < scale_rows * nkb; i += 32) {
                const int j = i / nkb;
                cp_async_4(sRaw + i, as_rows + static_cast<int64_t>(j) * num_kb + kb_lo + i - j * nkb);
            }
        }
        for (int i = lane; i < nkb; i += 32) cp_async_4(sBs + i, bs_row + i);
        cp_async_commit();
    }
    if (warp == 1) tmem_alloc(ring.tmem_holder, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;
    // Activations on the first stages (quantised input; FUSED holds them already).
    if (threadIdx.x == 0) {
        // fill the whole ring at once
        for (int i = 0; i < prefill; ++i) {
            const int kb = kb_lo + i;
            if (!g.weights_constant) {
                mbar_arrive_expect_tx(&ring.full[i], Cfg::TX_BYTES);
                tma_load_2d_hint(sW + i * A_TILE, &tmB, &ring.full[i], kb * BK, b_row, stream);
            }
            if constexpr (!FUSED)
                tma_load_2d_hint(sX + i * Cfg::X_TILE, &tmA, &ring.full[i], kb * BK, m0, keep);
        }
    }

    if (warp == 0) {
        if (lane == 0) {
            int stage = prefill % stages;
            uint32_t phase = prefill == stages ? 1u : 0u;
            int64_t issued = prefill;
            bool ok = true;
            for (int kb = kb_lo + prefill; kb < kb_lo + nkb; ++kb) {
                if (!mbar_wait(&ring.empty[stage], phase ^ 1)) {
                    record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&ring.full[stage], Cfg::TX_BYTES);
                tma_load_2d_hint(sW + stage * A_TILE, &tmB, &ring.full[stage], kb * BK, b_row,
                                 stream);
                if constexpr (!FUSED)
                    tma_load_2d_hint(sX + stage * Cfg::X_TILE, &tmA, &ring.full[stage], kb * BK,
                                     m0, keep);
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) drain_tma(ring, stages, issued);
        }
    } else if (warp == 1 || warp == Cfg::ISSUER2) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, MT);
            const int me = warp == 1 ? 0 : 1;         // this issuer's K blocks: kb % 2 == me
            int stage = 0;
            uint32_t phase = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                if ((kb & 1) != me) {                   // the other issuer's K block
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    continue;
                }
                const int buf = kb & (Cfg::NBUF - 1);
                const uint32_t tphase = static_cast<uint32_t>(kb / Cfg::NBUF) & 1u;
                if (!mbar_wait(&tempty[buf], tphase ^ 1) || !mbar_wait(&ring.full[stage], phase)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t w_addr = smem_addr(sW + stage * A_TILE);
                const uint32_t x_addr = smem_addr(sX + (FUSED ? kb : stage) * Cfg::X_TILE);
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * MT);
#pragma unroll
                for (int j = 0; j < BK / MMA_K; ++j)
                    mma_f8(d_tmem, smem_desc_k_sw128(w_addr + j * MMA_K),
                           smem_desc_k_sw128(x_addr + j * MMA_K), idesc, j > 0 ? 1u : 0u);
                mma_commit(&ring.empty[stage]);
                mma_commit(&tfull[buf]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            mma_commit(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else if (!FUSED && warp == Cfg::Q_WARP0) {
        // Scale warp: combined scales sAs[kb][m] = a_s[m0+m, kb] * b_s[slab, kb] (zero past row
        // M), transposed from the copied rows so that the promotion reads them as float4 along
        // m, one K block at a time and published as it goes: the promotion of block 0 need not
        // wait for the whole table.
        cp_async_wait_all();
        __syncwarp();
        for (int kb = 0; kb < nkb; ++kb) {
            const float sb = sBs[kb];
#pragma unroll
            for (int j = lane; j < MT; j += 32)
                sAs[kb * MT + j] = j < scale_rows ? sRaw[j * nkb + kb] * sb : 0.0f;
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                *reinterpret_cast<volatile int*>(sScaleDone) = kb + 1;
            }
        }
    } else if (FUSED && warp >= Cfg::Q_WARP0) {
        // Quantiser warps: their part was the prologue.
    } else {
        // Promotion warps.
        if constexpr (FUSED) {
            cp_async_wait_all();
            asm volatile("bar.sync 1, %0;" ::"n"(32 * Cfg::EPI_WARPS) : "memory");
        }
        const int quarter = warp & 3;
        const int n = n0 + quarter * 32 + lane;      // output column owned by this thread
        float acc[MT];
#pragma unroll
        for (int i = 0; i < MT; ++i) acc[i] = 0.0f;
        int buf = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            if (!warp_wait(&tfull[buf], tphase)) {
                if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                ok = false;
                break;
            }
            // FUSED: this block's a_s (quantised in the prologue) times b_s; otherwise the
            // staged products.
            float sb = 1.0f;
            if constexpr (!FUSED) {
                if (!spin_until_at_least(sScaleDone, kb + 1)) {
                    if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                    ok = false;
                    break;
                }
                __threadfence_block();
            }
            if constexpr (FUSED) sb = sBs[kb];
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * MT);
            const float* as_kb = sAs + kb * MT;
            auto scales4 = [&](int i) {
                float4 a4 = *reinterpret_cast<const float4*>(as_kb + i);
                if constexpr (FUSED) {   // rows past M: zero, as when staged
                    a4.x = i < scale_rows ? a4.x * sb : 0.0f;
                    a4.y = i + 1 < scale_rows ? a4.y * sb : 0.0f;
                    a4.z = i + 2 < scale_rows ? a4.z * sb : 0.0f;
                    a4.w = i + 3 < scale_rows ? a4.w * sb : 0.0f;
                }
                return a4;
            };
            if constexpr (MT >= 32) {
                // Chunks of 32 columns, the next load in flight while one is folded in; only
                // the chunks that hold rows of this CTA (a group of a grouped launch may have
                // fewer rows than MT).
                constexpr int NCH = MT / 32;
                const int nch = PLAIN ? NCH : (scale_rows + 31) >> 5;
                float va[32], vb[32];
                tmem_ld_32cols(taddr, va);
                if (!PLAIN && NCH == 2 && nch == 2) {
                    // General launches at MT = 64 (split K, grouped): both chunks in flight
                    // together, one round trip, the buffer back, then both folded in. (The
                    // N = 7168, K = 18432 down-projection at M = 64, split two ways: 34.4 ->
                    // 32.7 us. The plain launch measured no better this way.)
                    tmem_ld_32cols(taddr + 32, vb);
                    tmem_wait_ld_32(va);
                    tmem_wait_ld_32(vb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[buf]);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float* cur = c ? vb : va;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 a4 = scales4(c * 32 + i);
                            fma2_into(acc + c * 32 + i, cur[i + 0], cur[i + 1], a4.x, a4.y);
                            fma2_into(acc + c * 32 + i + 2, cur[i + 2], cur[i + 3], a4.z, a4.w);
                        }
                    }
                    if (++buf == Cfg::NBUF) {
                        buf = 0;
                        tphase ^= 1;
                    }
                    continue;
                }
                tmem_wait_ld_32(va);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (c < nch) {
                        float* cur = (c & 1) ? vb : va;
                        float* nxt = (c & 1) ? va : vb;
                        if (c + 1 < nch) tmem_ld_32cols(taddr + 32 * (c + 1), nxt);
                        if (c + 1 == nch) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[buf]);
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 a4 = scales4(c * 32 + i);
                            fma2_into(acc + c * 32 + i, cur[i + 0], cur[i + 1], a4.x, a4.y);
                            fma2_into(acc + c * 32 + i + 2, cur[i + 2], cur[i + 3], a4.z, a4.w);
                        }
                        if (c + 1 < nch) tmem_wait_ld_32(nxt);
                    }
                }
            } else {
                float v[16];
                tmem_ld_16cols(taddr, v);
                tmem_wait_ld_16(v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 a4 = scales4(i);
                    fma2_into(acc + i, v[i + 0], v[i + 1], a4.x, a4.y);
                    fma2_into(acc + i + 2, v[i + 2], v[i + 3], a4.z, a4.w);
                }
            }
            if (++buf == Cfg::NBUF) {
                buf = 0;
                tphase ^= 1;
            }
        }
        if (S == 1) {
            if (ok && n < g.N) {
                __nv_bfloat16* c = static_cast<__nv_bfloat16*>(g.c);
#pragma unroll
                for (int j = 0; j < MT; ++j)
                    if (j < scale_rows)
                        c[static_cast<int64_t>(m0 + j) * g.N + n] = __float2bfloat16_rn(acc[j]);
            }
        } else {
            // Split K: rows j .. j+3 of C (j < scale_rows, j % 4 == 0) are added up by CTA
            // j / wm of the cluster, which receives this CTA's partial of them as one float4
            // in slot `rank` of its receive area (rows past M hold zeros).
            const int t = quarter * 32 + lane;
            const int wm = swap_rows_per_rank(scale_rows, S);
            const int p4 = swap_pitch4(wm);
            const int rank = static_cast<int>(cluster_ctarank());
            const uint32_t recv = smem_addr(smem);
            cluster_sync();               // every CTA of the cluster is done with its stages
            if (ok) {
#pragma unroll
                for (int j = 0; j < MT; j += 4) {
                    if (j < scale_rows) {
                        const int q = j / wm;
                        const uint32_t off = static_cast<uint32_t>(
                            ((rank * BM + t) * p4 + (j - q * wm) / 4) * 16);
                        st_shared_cluster_f4(mapa_shared(recv + off, static_cast<uint32_t>(q)),
                                             make_float4(acc[j], acc[j + 1], acc[j + 2],
                                                         acc[j + 3]));
                    }
                }
            }
            cluster_sync();               // every partial has landed
            const float4* rv = reinterpret_cast<const float4*>(smem);
            const int j0 = rank * wm;
            const int j_end = min(scale_rows, j0 + wm);
            for (int j = j0; ok && j < j_end; j += 4) {
                float v[4];
                for (int r = 0; r < S; ++r) {
                    const float4 p = rv[(r * BM + t) * p4 + (j - j0) / 4];
                    v[0] = r == 0 ? p.x : v[0] + p.x;
                    v[1] = r == 0 ? p.y : v[1] + p.y;
                    v[2] = r == 0 ? p.z : v[2] + p.z;
                    v[3] = r == 0 ? p.w : v[3] + p.w;
                }
                if (n < g.N) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (j + i < j_end)
                            static_cast<__nv_bfloat16*>(g.c)[static_cast<int64_t>(m0 + j + i) *
                                                                 g.N + n] =
                                __float2bfloat16_rn(v[i]);
                }
            }
        }
    }
    // The other warps take part in the two cluster barriers of the split-K exchange.
    const bool promotion_warp = warp >= 2 && warp < 2 + Cfg::EPI_WARPS;
    if (S > 1 && !promotion_warp) {
        cluster_sync();
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    if (early && threadIdx.x == 0) grid_dependency_wait();
}

// Stages and dynamic shared-memory bytes of a launch whose CTAs take nkb K blocks each.
template <int MT, bool FUSED>
bool swap_smem(int nkb, int* stages_out, int* smem_out) {
    using Cfg = SwapCfg<MT, FUSED>;
    const int scale_bytes = swap_scale_bytes<MT, FUSED>(nkb);
    const int fixed = 1024 + scale_bytes + ring_bytes(kMaxStages) + Cfg::BAR_BYTES;
    int stages = (kSmemLimit - fixed) / Cfg::STAGE;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return false;   // K too large for the scale staging (FUSED: the activations)
    *stages_out = stages;
    *smem_out = 1024 + stages * Cfg::STAGE + scale_bytes + ring_bytes(stages) + Cfg::BAR_BYTES;
    return true;
}

// Fewest K blocks per CTA worth a split of the K loop.
constexpr int kMinSplitKb = 4;

// CTAs per slab for a launch over `row_tiles` MT-row tiles: the largest S (up to kMaxSplit) for
// which every CTA of the grid is resident at once, as whole clusters, with at least kMinSplitKb
// K blocks each; 1 for no split; 0 if the kernel cannot take this K (the activation scales do
// not fit).
// The instantiation a launch runs: the plain one, or (not fused) the general one.
template <int MT, bool FUSED>
auto swap_kernel(bool plain) {
    if constexpr (FUSED)
        return gemm_swapab_kernel<MT, true, true>;
    else
        return plain ? gemm_swapab_kernel<MT, false, true> : gemm_swapab_kernel<MT, false, false>;
}

template <int MT, bool FUSED>
int plan_swap(int row_tiles, int N, int K, int num_sms) {
    using Cfg = SwapCfg<MT, FUSED>;
    auto kernel = swap_kernel<MT, FUSED>(false);      // split launches run the general one
    const int num_kb = K / BK;
    const int slabs = (N + BM - 1) / BM;
    if (set_smem(kernel, kSmemLimit) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    for (int c = FUSED ? 1 : kMaxSplit; c > 1; --c) {
        int st = 0, sm = 0;
        if (static_cast<int64_t>(slabs) * row_tiles * c > num_sms || num_kb / c < kMinSplitKb ||
            !swap_smem<MT, FUSED>((num_kb + c - 1) / c, &st, &sm) ||
            swap_recv_bytes(MT, c) > st * Cfg::STAGE)
            continue;
        if (max_active_clusters(reinterpret_cast<const void*>(kernel), Cfg::THREADS, sm, c) <
            static_cast<int64_t>(slabs) * row_tiles)
            continue;
        return c;
    }
    int st = 0, sm = 0;
    return swap_smem<MT, FUSED>(num_kb, &st, &sm) ? 1 : 0;
}

template <int MT, bool FUSED>
cudaError_t launch_swap(const CUtensorMap& tmB, const CUtensorMap& tmA, const GemmArgs& g,
                        const GroupTable& gt, const FusedQuant& fq, int S, bool early,
                        cudaStream_t stream) {
    using Cfg = SwapCfg<MT, FUSED>;
    const bool plain = S == 1 && gt.num_groups == 1 && gt.row_off[0] == 0 && !early;
    auto kernel = swap_kernel<MT, FUSED>(plain);
    cudaError_t e = set_smem(kernel, kSmemLimit);
    if (e != cudaSuccess) return e;
    const int num_kb = g.K / BK;
    int stages = 0, smem = 0;
    if (S < 1 || (FUSED && !plain) ||
        !swap_smem<MT, FUSED>((num_kb + S - 1) / S, &stages, &smem))
        return cudaErrorInvalidValue;
    if (S > 1 && swap_recv_bytes(MT, S) > stages * Cfg::STAGE) return cudaErrorInvalidValue;
    const int row_tiles = gt.tile_off[gt.num_groups];
    if (row_tiles == 0) return cudaSuccess;
    const dim3 grid(((g.N + BM - 1) / BM) * S, row_tiles);
    return launch_pdl_cluster(kernel, grid, Cfg::THREADS, smem, stream, S, false, tmB, tmA, g, gt,
                              stages, fq, S, early ? 1 : 0);
}

template <int MT>
bool check_swap(int K, int S) {
    int st = 0, sm = 0;
    const int num_kb = K / BK;
    if (S < 1 || S > num_kb || !swap_smem<MT, false>((num_kb + S - 1) / S, &st, &sm)) return false;
    return S == 1 || swap_recv_bytes(MT, S) <= st * SwapCfg<MT, false>::STAGE;
}

}  // namespace

bool check_gemm_swapab(int MT, int K, int ksplit) {
    switch (MT) {
        case 16: return check_swap<16>(K, ksplit);
        case 32: return check_swap<32>(K, ksplit);
        case 64: return check_swap<64>(K, ksplit);
        case 128: return check_swap<128>(K, ksplit);
        default: return false;
    }
}

int plan_gemm_swapab(int MT, bool fused, int row_tiles, int N, int K, int num_sms) {
    if (fused) return MT == 16 ? plan_swap<16, true>(row_tiles, N, K, num_sms) : 0;
    switch (MT) {
        case 16: return plan_swap<16, false>(row_tiles, N, K, num_sms);
        case 32: return plan_swap<32, false>(row_tiles, N, K, num_sms);
        case 64: return plan_swap<64, false>(row_tiles, N, K, num_sms);
        case 128: return plan_swap<128, false>(row_tiles, N, K, num_sms);
        default: return 0;
    }
}

void fill_row_tiles(GroupTable* gt, const int64_t* row_off, int groups, int MT) {
    gt->num_groups = groups;
    gt->row_off[0] = static_cast<int>(row_off[0]);
    gt->tile_off[0] = 0;
    for (int i = 0; i < groups; ++i) {
        const int rows = static_cast<int>(row_off[i + 1] - row_off[i]);
        gt->row_off[i + 1] = static_cast<int>(row_off[i + 1]);
        gt->tile_off[i + 1] = gt->tile_off[i] + (rows + MT - 1) / MT;
    }
}

cudaError_t launch_gemm_swapab(const CUtensorMap& tmB, const CUtensorMap& tmA,
                               const GemmArgs& g, const GroupTable& gt, int MT,
                               const FusedQuant& fq, int ksplit, bool early,
                               cudaStream_t stream) {
    if (fq.x)
        return MT == 16 ? launch_swap<16, true>(tmB, tmA, g, gt, fq, ksplit, early, stream)
                        : cudaErrorInvalidValue;
    switch (MT) {
        case 16: return launch_swap<16, false>(tmB, tmA, g, gt, fq, ksplit, early, stream);
        case 32: return launch_swap<32, false>(tmB, tmA, g, gt, fq, ksplit, early, stream);
        case 64: return launch_swap<64, false>(tmB, tmA, g, gt, fq, ksplit, early, stream);
        case 128: return launch_swap<128, false>(tmB, tmA, g, gt, fq, ksplit, early, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_swapab(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
