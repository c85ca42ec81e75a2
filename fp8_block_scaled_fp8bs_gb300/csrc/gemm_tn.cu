// gemm_tn.cu -- FP8 GEMM with fp32 block scales, normal orientation (M > 128): tiles of 128
// rows of A (the MMA's M side) by BN = 64, 128 or 256 columns of B, persistent over tiles and
// over the groups of a grouped launch.
//
//   promotion warps   tcgen05.ld each K block's fp32 partial from one of two TMEM buffers in
//                     32-column chunks (the next chunk's load in flight while the current one
//                     is folded in), release the buffer, and fold it into fp32 registers with
//                     the block's scale a_s[m,kb] * b_s[n/128,kb]; after the last block, bf16
//                     and store. The two buffers let the tensor cores compute block kb+1
//                     while block kb is promoted.
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

// Scales of four consecutive K blocks starting at block k (k a multiple of 4): one 16-byte
// load when the row is 16-byte aligned and holds whole groups of four, else scalar loads.
__device__ __forceinline__ float4 load_scales4(const float* row, int k, int n, bool vec) {
    if (vec && k + 4 <= n) return __ldg(reinterpret_cast<const float4*>(row + k));
    float4 r;
    r.x = k < n ? __ldg(row + k) : 0.0f;
    r.y = k + 1 < n ? __ldg(row + k + 1) : 0.0f;
    r.z = k + 2 < n ? __ldg(row + k + 2) : 0.0f;
    r.w = k + 3 < n ? __ldg(row + k + 3) : 0.0f;
    return r;
}

__device__ __forceinline__ float pick4(const float4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Tile = 128 rows of A x BN columns of B (BN = 64, 128 or 256). Warp layout (whole
// warpgroups, so that register budgets can be moved between them):
//   warps 0 .. 7     promotion/epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 and the
//                    columns (BN/2)*(w/4) .. +BN/2-1 of the tile
//   warp 8           TMA producer
//   warp 9           MMA issuer (also allocates and frees TMEM)
//   warps 10, 11     idle (they complete the last warpgroup)
// The block has 384 threads, so each thread starts with 168 registers. With BN = 256 (128
// accumulator columns per thread) the control warpgroup gives registers back (kCtlRegs) and
// the promotion warpgroups take them (kEpiRegs): 4*32*kCtlRegs + 8*32*kEpiRegs <= 384*168
// keeps the split inside the block's launch allocation, so setmaxnreg.inc never waits.
template <int BN>
struct TnCfg {
    static constexpr int EPI_WARPS = 8;
    static constexpr int CW = BN / 2;                         // columns per promotion thread
    static constexpr int THREADS = 32 * EPI_WARPS + 128;
    static constexpr int B_TILE = BN * BK;
    static constexpr int STAGE = A_TILE + B_TILE;
    static constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * BN);
    static constexpr bool SPLIT_REGS = (BN == 256);
    static constexpr uint32_t kCtlRegs = 40;
    static constexpr uint32_t kEpiRegs = 232;
    static_assert(!SPLIT_REGS || 4 * 32 * kCtlRegs + 8 * 32 * kEpiRegs <= 384 * 168,
                  "register split exceeds the launch allocation");
};

template <int BN>
__global__ void __launch_bounds__(TnCfg<BN>::THREADS, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs g, const __grid_constant__ GroupTable gt, const int stages) {
    using Cfg = TnCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + stages * A_TILE;
    const Ring ring = carve_ring(sB + stages * Cfg::B_TILE, stages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_kb = g.K / BK;
    const int n_tiles = (g.N + BN - 1) / BN;
    const int num_tiles = gt.tile_off[gt.num_groups];
    constexpr int PRODUCER = Cfg::EPI_WARPS;
    constexpr int ISSUER = Cfg::EPI_WARPS + 1;

    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        init_ring(ring, stages, Cfg::EPI_WARPS);
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == ISSUER) tmem_alloc(ring.tmem_holder, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;

    if (warp >= Cfg::EPI_WARPS) {
        if constexpr (Cfg::SPLIT_REGS) regs_dec<Cfg::kCtlRegs>();
        if (warp == PRODUCER && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
                const int b_row = t.g * g.N + t.n0;      // row of the stacked B
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&ring.empty[stage], phase ^ 1)) {
                        record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ring.full[stage], Cfg::STAGE);
                    tma_load_2d(sA + stage * A_TILE, &tmA, &ring.full[stage], kb * BK, t.m0);
                    tma_load_2d(sB + stage * Cfg::B_TILE, &tmB, &ring.full[stage], kb * BK, b_row);
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) drain_tma(ring, stages, issued);
        } else if (warp == ISSUER && lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&ring.tempty[buf], tphase ^ 1) ||
                        !mbar_wait(&ring.full[stage], phase)) {
                        record_error(FP8BS_DEVERR_MMA_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * A_TILE);
                    const uint32_t b_addr = smem_addr(sB + stage * Cfg::B_TILE);
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
                    for (int j = 0; j < BK / MMA_K; ++j)
                        mma_f8(d_tmem, smem_desc_k_sw128(a_addr + j * MMA_K),
                               smem_desc_k_sw128(b_addr + j * MMA_K), idesc, j > 0 ? 1u : 0u);
                    mma_commit(&ring.empty[stage]);
                    mma_commit(&ring.tfull[buf]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    buf ^= 1;
                    if (buf == 0) tphase ^= 1;
                }
            }
            // Make sure nothing this thread issued is still running before TMEM is freed.
            mma_commit(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else {
        if constexpr (Cfg::SPLIT_REGS) regs_inc<Cfg::kEpiRegs>();
        // Promotion / epilogue warps.
        const int quarter = warp & 3;
        const int col0 = (warp >> 2) * Cfg::CW;
        const int row_in_tile = quarter * 32 + lane;
        const int nb_count = (g.N + 127) / 128;
        const bool vec_scales = (num_kb % 4 == 0) &&
                                ((reinterpret_cast<uintptr_t>(g.a_s) & 15u) == 0) &&
                                ((reinterpret_cast<uintptr_t>(g.b_s) & 15u) == 0);
        int buf = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            const int n0 = t.n0;
            const int row = t.m0 + row_in_tile;
            const int nb = min((n0 + col0) / 128, nb_count - 1);
            const float* as_row = g.a_s + static_cast<int64_t>(min(row, g.M - 1)) * num_kb;
            const float* bs_row =
                g.b_s + (static_cast<int64_t>(t.g) * nb_count + nb) * num_kb;
            float acc[Cfg::CW];
#pragma unroll
            for (int i = 0; i < Cfg::CW; ++i) acc[i] = 0.0f;
            // Scales in groups of four K blocks, the next group in flight.
            float4 a_cur = load_scales4(as_row, 0, num_kb, vec_scales);
            float4 b_cur = load_scales4(bs_row, 0, num_kb, vec_scales);
            float4 a_nxt = load_scales4(as_row, 4, num_kb, vec_scales);
            float4 b_nxt = load_scales4(bs_row, 4, num_kb, vec_scales);
            for (int kb = 0; kb < num_kb; ++kb) {
                const int j = kb & 3;
                const float sc = pick4(a_cur, j) * pick4(b_cur, j);
                if (j == 3) {
                    a_cur = a_nxt;
                    b_cur = b_nxt;
                    a_nxt = load_scales4(as_row, kb + 5, num_kb, vec_scales);
                    b_nxt = load_scales4(bs_row, kb + 5, num_kb, vec_scales);
                }
                if (!warp_wait(&ring.tfull[buf], tphase)) {
                    if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + col0);
                // Four chunks of 32 columns: the load of chunk c+1 is in flight while chunk c is
                // folded in; the buffer is handed back as soon as the last chunk has landed.
                float va[32], vb[32];
                tmem_ld_32cols(taddr, va);
                tmem_wait_ld_32(va);
#pragma unroll
                for (int c = 0; c < Cfg::CW / 32; ++c) {
                    float* cur = (c & 1) ? vb : va;
                    float* nxt = (c & 1) ? va : vb;
                    if (c + 1 < Cfg::CW / 32) tmem_ld_32cols(taddr + 32 * (c + 1), nxt);
                    if (c + 1 == Cfg::CW / 32) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ring.tempty[buf]);
                    }
                    // Packed fp32x2 FMAs (round-to-nearest per component): half the issue slots.
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 r = __ffma2_rn(make_float2(cur[i], cur[i + 1]), make_float2(sc, sc),
                                                    make_float2(acc[c * 32 + i], acc[c * 32 + i + 1]));
                        acc[c * 32 + i] = r.x;
                        acc[c * 32 + i + 1] = r.y;
                    }
                    if (c + 1 < Cfg::CW / 32) tmem_wait_ld_32(nxt);
                }
                buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            if (!ok) break;
            if (row < t.row_end) {
                __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(g.c) +
                                      static_cast<int64_t>(row) * g.N + n0 + col0;
                const int valid = min(Cfg::CW, g.N - (n0 + col0));
                if ((g.N & 7) == 0) {
#pragma unroll
                    for (int j = 0; j < Cfg::CW / 8; ++j) {
                        if (8 * j < valid) {
                            uint4 o;
                            o.x = pack_bf16x2(acc[8 * j + 0], acc[8 * j + 1]);
                            o.y = pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]);
                            o.z = pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]);
                            o.w = pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]);
                            *reinterpret_cast<uint4*>(crow + 8 * j) = o;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < Cfg::CW; ++j)
                        if (j < valid) crow[j] = __float2bfloat16_rn(acc[j]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == ISSUER) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int BN>
cudaError_t launch_tn(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                      const GroupTable& gt, int num_sms, cudaStream_t stream) {
    using Cfg = TnCfg<BN>;
    int stages = (kSmemLimit - 1024 - ring_bytes(kMaxStages)) / Cfg::STAGE;
    if (stages > kMaxStages) stages = kMaxStages;
    const int smem = 1024 + stages * Cfg::STAGE + ring_bytes(stages);
    cudaError_t e = set_smem(gemm_tn_kernel<BN>, smem);
    if (e != cudaSuccess) return e;
    const int tiles = gt.tile_off[gt.num_groups];
    if (tiles == 0) return cudaSuccess;
    const int grid = tiles < num_sms ? tiles : num_sms;
    return launch_pdl(gemm_tn_kernel<BN>, grid, Cfg::THREADS, smem, stream, tmA, tmB, g, gt,
                      stages);
}

}  // namespace

int pick_tile_n(int64_t m_tiles_total, int64_t N, int num_sms) {
    if (m_tiles_total * ((N + 255) / 256) >= num_sms) return 256;
    if (m_tiles_total * ((N + 127) / 128) * 5 >= num_sms * 4) return 128;
    return 64;
}

void fill_group_table(GroupTable* gt, const int64_t* row_off, int groups, int N, int bn) {
    const int n_tiles = (N + bn - 1) / bn;
    gt->num_groups = groups;
    gt->row_off[0] = static_cast<int>(row_off[0]);
    gt->tile_off[0] = 0;
    for (int i = 0; i < groups; ++i) {
        const int rows = static_cast<int>(row_off[i + 1] - row_off[i]);
        gt->row_off[i + 1] = static_cast<int>(row_off[i + 1]);
        gt->tile_off[i + 1] = gt->tile_off[i] + ((rows + BM - 1) / BM) * n_tiles;
    }
}

cudaError_t launch_gemm_tn(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           const GroupTable& gt, int BN, int num_sms, cudaStream_t stream) {
    switch (BN) {
        case 64: return launch_tn<64>(tmA, tmB, g, gt, num_sms, stream);
        case 128: return launch_tn<128>(tmA, tmB, g, gt, num_sms, stream);
        case 256: return launch_tn<256>(tmA, tmB, g, gt, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_tn(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
