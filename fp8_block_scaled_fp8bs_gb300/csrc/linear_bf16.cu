// linear_bf16.cu -- the bf16 path of linear() with FP8 weights: y = x . W'^T, where W' is the
// bf16 weight that weight_dequant would produce ("DeepSeek-V3 Administrator & Developer Guide",
// §6.3: with gemm_impl = "bf16" the FP8 weight is dequantised (§8.5.2) and a bf16 GEMM runs).
// Here the weight is dequantised tile by tile on chip instead of being written to and read back
// from HBM as bf16.
//
// 128-row slabs of W take the MMA's M side, MT (16, 32, 64 or 128) rows of x its N side; each
// CTA streams the e4m3 codes of one slab (half the bytes of the bf16 weight) against XT tiles
// of x (XT = 2 for M > 128: each dequantised K block then feeds two 128-row tiles, halving the
// dequantisation per FLOP). CTAs that share a slab are adjacent in launch order, so for
// M > 128 a slab is read from HBM about once and the other tiles of x find it in L2.
//   warp 0          weight producer: per K block the e4m3 tile (the HBM stream) into the
//                   weight ring; a slot is free as soon as the dequantisers have read it
//   warp 1 + ISSUERS (lane 0) x producer: the bf16 rows of x (128-byte swizzle, 64-wide K
//                   halves) into the x ring; a slot is free once the MMAs reading it are done.
//                   It is an epilogue warp, idle until the end of the K loop.
//   warps 1 .. ISSUERS  MMA issuers (lane 0). XT = 1: K block kb to issuer kb % ISSUERS (four
//                   at MT <= 64, two at MT = 128); XT = 2: issuer t takes tile t of x for
//                   every K block. Per K block 8 x tcgen05.mma kind::f16 (K = 16) into the
//                   issuer's own TMEM accumulator for the whole K loop (the block scale is
//                   inside W'). One thread issuing alone is held to about one small MMA per
//                   60-80 clk and stalls at its next barrier wait until the tensor core has
//                   caught up. With two issuers the decode rows still ran 32 us against 26 us
//                   with the MMAs left out (M = 1, N = 18432, K = 7168), hence four there.
//   warps 2 .. 5    epilogue: the accumulators to bf16 y (summed for XT = 1)
//   warps 6 .. 21   dequantisers, two groups of eight taking K blocks in turn (a warp's barrier
//                   waits and arrivals cost a few hundred clk per K block, which the other
//                   group overlaps): e4m3 tile -> bf16 W' tile (fp32 product with
//                   the block scale, rounded to bf16: weight_dequant's arithmetic) written
//                   straight into TMEM with tcgen05.st (lane = weight row, 32-bit column =
//                   two consecutive K), where the MMA takes its A operand: a third ring, of
//                   four 64-column TMEM slots. W' never touches shared memory, which the
//                   TMA streams, the dequantisers' reads and the MMA's reads of x share.
// Separate weight and x rings let the weight ring run ahead of the MMAs (its slots recycle at
// dequantisation) and, with two tiles of x, let the x ring work in K halves so that four slots
// fit.
#include "gemm_common.cuh"

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fp8bs {

namespace {

template <int MT, int XT>
struct LinCfg {
    static_assert(XT == 1 || (XT == 2 && MT == 128), "two x tiles only with 128 rows each");
    static constexpr int EPI_WARPS = 4;
    static constexpr int DQ_GROUP = 8;                   // dequantiser warps per K block
    static constexpr int DQ_GROUPS = 2;                  // groups, taking K blocks in turn
    static constexpr int DQ_WARPS = DQ_GROUP * DQ_GROUPS;
    static constexpr int DQ0 = 2 + EPI_WARPS;            // first dequantiser warp
    // MMA issuers: warps 1 .. ISSUERS. Four where four accumulators fit beside the W' slots in
    // TMEM (one tile of x, MT <= 64), else two.
    static constexpr int ISSUERS = (XT == 1 && MT <= 64) ? 4 : 2;
    static constexpr int X_PRODUCER = 1 + ISSUERS;       // an epilogue warp, idle until the end
    static constexpr int THREADS = 32 * (2 + EPI_WARPS + DQ_WARPS);
    static constexpr int W_TILE = BM * BK;               // e4m3 weight tile (128 x 128)
    static constexpr int HALF = 64;                      // bf16 K elements per 128-byte row
    static constexpr int XH_TILE = MT * 128;             // one tile of x, one 64-wide K half
    // x ring slot: XT tiles x HPS K halves. Two tiles (large M): one K half per slot, so that
    // four slots fit beside the weight ring; one tile: a whole K block per slot, so that an
    // issuer waits once per K block (each wait after issued MMAs costs it a drain).
    static constexpr int HPS = XT == 2 ? 1 : 2;
    static constexpr int X_SLOT = XT * HPS * XH_TILE;
    static constexpr int SX = (XT == 2 || MT >= 128) ? 4 : 8;   // x ring slots
    static constexpr int BAR_BYTES = 8 * (2 * kMaxStages + 2 * SX + 2 * 4 + 2) + 16;
    static constexpr int SW_FIT = (kSmemLimit - 1024 - BAR_BYTES - SX * X_SLOT) / W_TILE;
    static constexpr int SW = SW_FIT > kMaxStages ? kMaxStages : SW_FIT;   // weight ring slots
    static_assert(SW >= 2, "shared memory");
    static constexpr int ACC_COLS = MT > 64 ? MT : 64;   // TMEM: accumulator i at ACC_COLS i,
    static constexpr int W_COL0 = ISSUERS * ACC_COLS;    // then the W' slots of 64 columns
    static constexpr int W_COLS = BK / 2;                // (bf16 pairs)
    static constexpr int SB = 4;                         // W' slots
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(W_COL0 + SB * W_COLS <= static_cast<int>(TMEM_COLS), "TMEM columns");
    static_assert(X_PRODUCER >= 2 && X_PRODUCER < 2 + EPI_WARPS, "x producer: an epilogue warp");
    static constexpr int MMA_PER_KB = XT;                // issuer commits per K block
    static constexpr int SMEM = 1024 + SW * W_TILE + SX * X_SLOT + BAR_BYTES;
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
            // both products in one packed multiply (each rounded to nearest as __fmul_rn)
            const float2 p = __fmul2_rn(f, make_float2(sc, sc));
            out[2 * i + h] = bf16x2(p.x, p.y);
        }
    }
}

// `CW` (16 or 32) consecutive TMEM columns of this warp's lane quarter into registers.
template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
    if constexpr (CW == 32) {
        tmem_ld_32cols(taddr, v);
        tmem_wait_ld_32(v);
    } else {
        tmem_ld_16cols(taddr, v);
        tmem_wait_ld_16(v);
    }
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile (8-row atoms
// of 1024 bytes: the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ int sw128(int r, int c) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

template <int MT, int XT>
__global__ void __launch_bounds__(LinCfg<MT, XT>::THREADS, 1)
    linear_bf16_swap_kernel(const __grid_constant__ CUtensorMap tmW,
                            const __grid_constant__ CUtensorMap tmX,
                            const float* __restrict__ w_s, void* y, const int M, const int N,
                            const int K, const int weights_constant, const int tiles_per_phase) {
    using Cfg = LinCfg<MT, XT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sW = smem;                                   // [SW][W e4m3 tile]
    uint8_t* sX = sW + Cfg::SW * Cfg::W_TILE;             // [SX][XT tiles x one K half of x]
    uint64_t* fullW = reinterpret_cast<uint64_t*>(sX + Cfg::SX * Cfg::X_SLOT);
    uint64_t* emptyW = fullW + Cfg::SW;
    uint64_t* fullX = emptyW + Cfg::SW;
    uint64_t* emptyX = fullX + Cfg::SX;
    uint64_t* deqB = emptyX + Cfg::SX;
    uint64_t* emptyB = deqB + Cfg::SB;
    uint64_t* tfull = emptyB + Cfg::SB;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_kb = K / BK;
    // CTA -> (weight slab, tile of x): the tiles of x go in phases of tiles_per_phase, and
    // within a phase the CTAs of one slab are adjacent (the slab is read from HBM about once per
    // phase, the phase's tiles of x stay in L2 while every slab passes them).
    const int m_tiles = (M + MT * XT - 1) / (MT * XT);
    const int slabs = (N + BM - 1) / BM;
    const int phase = static_cast<int>(blockIdx.x) / (slabs * tiles_per_phase);
    const int in_phase = static_cast<int>(blockIdx.x) - phase * slabs * tiles_per_phase;
    const int phase_tiles = min(tiles_per_phase, m_tiles - phase * tiles_per_phase);
    const int slab = in_phase / phase_tiles;
    const int n0 = slab * BM;
    const int m0 = (phase * tiles_per_phase + in_phase - slab * phase_tiles) * MT * XT;
    const float* ws_row = w_s + static_cast<int64_t>(slab) * num_kb;
    const int w_prefill = min(Cfg::SW, num_kb);
    // weights: read once, or (several tiles of x) by the neighbouring CTAs too
    const uint64_t stream = m_tiles > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
    const uint64_t keep = l2_policy_evict_last();     // x: read by every CTA

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::SW; ++i) {
            mbar_init(&fullW[i], 1);
            mbar_init(&emptyW[i], Cfg::DQ_GROUP);        // the dequantisers have read the codes
        }
        for (int i = 0; i < Cfg::SX; ++i) {
            mbar_init(&fullX[i], 1);
            mbar_init(&emptyX[i], Cfg::MMA_PER_KB);      // the MMAs reading it are done
        }
        for (int i = 0; i < Cfg::SB; ++i) {
            mbar_init(&deqB[i], Cfg::DQ_GROUP);
            mbar_init(&emptyB[i], Cfg::MMA_PER_KB);
        }
        mbar_init(tfull, Cfg::ISSUERS);
        mbar_init(drain, Cfg::ISSUERS);
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        // Weights the caller declared constant start streaming before earlier kernels finish.
        if (weights_constant)
            for (int kb = 0; kb < w_prefill; ++kb) {
                mbar_arrive_expect_tx(&fullW[kb], Cfg::W_TILE);
                tma_load_2d_hint(sW + kb * Cfg::W_TILE, &tmW, &fullW[kb], kb * BK, n0, stream);
            }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 1) tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp >= 1 && warp <= Cfg::ISSUERS && lane == 0) {
        // MMA issuer me. XT = 1: K blocks me, me + 2, ... into accumulator me; XT = 2: every K
        // block against tile me of x, into accumulator me. Per K block: wait for its W' slot,
        // then per 64-wide K half for the x slot, 4 MMAs (K = 16), release the x slot; after
        // both halves release the W' slot.
        constexpr uint32_t idesc = idesc_bf16_f32(BM, MT);
        const int me = warp - 1;
        const uint32_t acc = tmem_base + static_cast<uint32_t>(me * Cfg::ACC_COLS);
        constexpr int STEP = XT == 2 ? 1 : Cfg::ISSUERS;
        const int first = XT == 2 ? 0 : me;
        const int x_off = (XT == 2 ? me : 0) * Cfg::XH_TILE;
        bool ok = true;
        for (int kb = first; ok && kb < num_kb; kb += STEP) {
            const int b = kb % Cfg::SB;
            if (!mbar_wait(&deqB[b], static_cast<uint32_t>((kb / Cfg::SB) & 1))) {
                record_error(FP8BS_DEVERR_MMA_WAIT);
                break;
            }
            const uint32_t w_tmem = tmem_base + static_cast<uint32_t>(Cfg::W_COL0 + b * Cfg::W_COLS);
#pragma unroll
            for (int p = 0; p < 2 / Cfg::HPS; ++p) {
                const int q = (2 / Cfg::HPS) * kb + p;    // x slot sequence number
                const int xs = q % Cfg::SX;
                // One tile: the first dequantiser warp of the K block waited for this slot
                // before signalling deqB, so the issuer need not wait again.
                if (XT == 2 && !mbar_wait(&fullX[xs], static_cast<uint32_t>((q / Cfg::SX) & 1))) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t x_addr = smem_addr(sX + xs * Cfg::X_SLOT + x_off);
#pragma unroll
                for (int j = 0; j < 4 * Cfg::HPS; ++j) {
                    const int h = p * Cfg::HPS + j / 4;   // K half of the block
                    mma_bf16_ta(acc, w_tmem + 8 * (4 * h + j % 4),
                                smem_desc_k_sw128(x_addr + (j / 4) * Cfg::XH_TILE + 32 * (j % 4)),
                                idesc, (kb > first || h > 0 || j % 4 > 0) ? 1u : 0u);
                }
                mma_commit(&emptyX[xs]);
            }
            mma_commit(&emptyB[b]);
        }
        mma_commit(tfull);
        mma_commit(drain);
        if (!mbar_wait(drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
    }
    if (warp == Cfg::X_PRODUCER && lane == 0) {
        // x producer: per slot, the XT tiles' HPS 64-wide K halves (128-byte swizzled rows).
        const int slots = (2 / Cfg::HPS) * num_kb;
        int issued = 0;
        for (int q = 0; q < slots; ++q) {
            const int xs = q % Cfg::SX;
            if (q >= Cfg::SX &&
                !mbar_wait(&emptyX[xs], static_cast<uint32_t>(((q / Cfg::SX) & 1) ^ 1))) {
                record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                for (int i = issued > Cfg::SX ? issued - Cfg::SX : 0; i < issued; ++i)
                    if (!mbar_wait(&fullX[i % Cfg::SX], static_cast<uint32_t>((i / Cfg::SX) & 1),
                                   kDrainLimitNs))
                        record_error(FP8BS_DEVERR_DRAIN_WAIT);
                break;
            }
            mbar_arrive_expect_tx(&fullX[xs], Cfg::X_SLOT);
#pragma unroll
            for (int t = 0; t < XT; ++t)
#pragma unroll
                for (int h = 0; h < Cfg::HPS; ++h)
                    tma_load_2d_hint(sX + xs * Cfg::X_SLOT + (t * Cfg::HPS + h) * Cfg::XH_TILE,
                                     &tmX, &fullX[xs], (q * Cfg::HPS + h) * Cfg::HALF,
                                     m0 + t * MT, keep);
            ++issued;
        }
    }
    __syncwarp();

    if (warp == 0) {
        if (lane == 0) {
            // weight producer: the e4m3 tile of each K block
            if (!weights_constant)
                for (int kb = 0; kb < w_prefill; ++kb) {
                    mbar_arrive_expect_tx(&fullW[kb], Cfg::W_TILE);
                    tma_load_2d_hint(sW + kb * Cfg::W_TILE, &tmW, &fullW[kb], kb * BK, n0,
                                     stream);
                }
            int issued = w_prefill;
            for (int kb = w_prefill; kb < num_kb; ++kb) {
                const int ws = kb % Cfg::SW;
                if (!mbar_wait(&emptyW[ws], static_cast<uint32_t>(((kb / Cfg::SW) & 1) ^ 1))) {
                    record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                    for (int i = issued > Cfg::SW ? issued - Cfg::SW : 0; i < issued; ++i)
                        if (!mbar_wait(&fullW[i % Cfg::SW],
                                       static_cast<uint32_t>((i / Cfg::SW) & 1), kDrainLimitNs))
                            record_error(FP8BS_DEVERR_DRAIN_WAIT);
                    break;
                }
                mbar_arrive_expect_tx(&fullW[ws], Cfg::W_TILE);
                tma_load_2d_hint(sW + ws * Cfg::W_TILE, &tmW, &fullW[ws], kb * BK, n0, stream);
                ++issued;
            }
        }
    } else if (warp >= Cfg::DQ0) {
        // Dequantisers: group g takes the K blocks kb with kb % 2 == g. Warp w handles the TMEM
        // lane quarter w % 4 (weight rows 32 (w % 4) .. +31, one per lane) and one 64-wide half
        // of the K block; each lane reads the 64 codes of its row's half, hands the weight slot
        // back, and stores them dequantised as 32 columns of bf16 pairs.
        const int group = (warp - Cfg::DQ0) / Cfg::DQ_GROUP;
        const int quarter = warp & 3;
        const int khalf = ((warp - Cfg::DQ0) >> 2) & 1;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(Cfg::W_COL0 + 32 * khalf);
        float sc_next = group < num_kb ? __ldg(ws_row + group) : 0.f;
        for (int kb = group; kb < num_kb; kb += Cfg::DQ_GROUPS) {
            const int b = kb % Cfg::SB, ws = kb % Cfg::SW;
            const float sc = sc_next;                   // the block scale, fetched one step early
            if (kb + Cfg::DQ_GROUPS < num_kb) sc_next = __ldg(ws_row + kb + Cfg::DQ_GROUPS);
            if (!warp_wait(&fullW[ws], static_cast<uint32_t>((kb / Cfg::SW) & 1))) {
                if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                break;
            }
            const uint8_t* wslot = sW + ws * Cfg::W_TILE;
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = *reinterpret_cast<const uint4*>(wslot + sw128(r, 4 * khalf + i));
            __syncwarp();
            if (lane == 0) mbar_arrive(&emptyW[ws]);
            if (!warp_wait(&emptyB[b], static_cast<uint32_t>(((kb / Cfg::SB) & 1) ^ 1))) {
                if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                break;
            }
            tc_fence_after();
            uint32_t o[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dequant8(v[i].x, v[i].y, sc, o + 8 * i);
                dequant8(v[i].z, v[i].w, sc, o + 8 * i + 4);
            }
            tmem_st_32cols(lane_base + static_cast<uint32_t>(b * Cfg::W_COLS), o);
            tmem_wait_st();
            tc_fence_before();
            if (XT == 1 && (warp - Cfg::DQ0) % Cfg::DQ_GROUP == 0 &&
                !warp_wait(&fullX[kb % Cfg::SX], static_cast<uint32_t>((kb / Cfg::SX) & 1))) {
                if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&deqB[b]);
        }
    } else if (warp >= 2) {
        // Epilogue: TMEM lane = output column n0 + 32 * quarter + lane, columns = rows of x;
        // y = acc 0 + acc 1 in fp32 (accumulator i holds the K blocks kb with kb % 2 == i).
        const int quarter = warp & 3;
        const int n = n0 + quarter * 32 + lane;
        if (warp_wait(tfull, 0)) {
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            // XT = 1: the written accumulators are summed; XT = 2: accumulator t is tile t
            const int used = XT == 2 ? 1 : min(num_kb, Cfg::ISSUERS);
            constexpr int CW = MT < 32 ? MT : 32;          // columns (rows of x) per chunk
            __nv_bfloat16* yc = static_cast<__nv_bfloat16*>(y);
#pragma unroll 1
            for (int c = 0; c < XT * MT / CW; ++c) {
                // chunk c: columns CW c .. of accumulator c / (MT / CW) (XT = 2), rows of x
                // m0 + CW c ..
                float acc[CW];
                tmem_ld_cols<CW>(taddr + (XT == 2 ? (c / (MT / CW)) * Cfg::ACC_COLS +
                                                        (c % (MT / CW)) * CW
                                                  : CW * c),
                                 acc);
                for (int i = 1; i < used; ++i) {
                    float t[CW];
                    tmem_ld_cols<CW>(taddr + i * Cfg::ACC_COLS + CW * c, t);
#pragma unroll
                    for (int j = 0; j < CW; ++j) acc[j] += t[j];
                }
                if (n < N) {
                    // Streaming stores (evict-first in L2): y is written once, and at large M
                    // the tiles of x, loaded evict-last, are what every later slab needs from L2.
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        const int m = m0 + CW * c + j;
                        if (m < M) {
                            const __nv_bfloat16 v = __float2bfloat16_rn(acc[j]);
                            __stcs(reinterpret_cast<unsigned short*>(yc) +
                                       static_cast<int64_t>(m) * N + n,
                                   *reinterpret_cast<const unsigned short*>(&v));
                        }
                    }
                }
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

template <int MT, int XT>
cudaError_t launch_lin(const CUtensorMap& tmW, const CUtensorMap& tmX, const float* w_s, void* y,
                       int M, int N, int K, int weights_constant, cudaStream_t stream) {
    using Cfg = LinCfg<MT, XT>;
    cudaError_t e = set_smem(linear_bf16_swap_kernel<MT, XT>, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t m_tiles = (M + MT * XT - 1) / (MT * XT);
    const int64_t ctas = static_cast<int64_t>((N + BM - 1) / BM) * m_tiles;
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    // Tiles of x per phase: as many as fill a quarter of L2 (bf16 rows, MT x XT x K each), at
    // least one. With every tile at once (4096 x 7168 rows, 16 tiles, 58.7 MB) the tiles were
    // re-read from HBM by every wave of slabs: 0.74 GB read against 0.19 GB of x and codes.
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const int64_t tile_bytes = static_cast<int64_t>(MT) * XT * K * 2;
    const int64_t fit = tile_bytes > 0 ? (static_cast<int64_t>(l2) / 4) / tile_bytes : m_tiles;
    const int tiles_per_phase =
        static_cast<int>(fit < 1 ? 1 : fit > m_tiles ? m_tiles : fit);
    const dim3 grid(static_cast<unsigned>(ctas));
    return launch_pdl(linear_bf16_swap_kernel<MT, XT>, grid, Cfg::THREADS, Cfg::SMEM, stream, tmW,
                      tmX, w_s, y, M, N, K, weights_constant, tiles_per_phase);
}

}  // namespace

cudaError_t launch_linear_bf16_swap(const CUtensorMap& tmW, const CUtensorMap& tmX,
                                    const float* w_s, void* y, int M, int N, int K, int MT,
                                    int weights_constant, cudaStream_t stream) {
    switch (MT) {
        case 16: return launch_lin<16, 1>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        case 32: return launch_lin<32, 1>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        case 64: return launch_lin<64, 1>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        case 128:
            // beyond one 128-row tile of x, each CTA takes two
            if (M > 128)
                return launch_lin<128, 2>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
            return launch_lin<128, 1>(tmW, tmX, w_s, y, M, N, K, weights_constant, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_linear(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
