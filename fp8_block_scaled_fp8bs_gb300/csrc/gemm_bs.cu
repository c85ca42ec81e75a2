// gemm_bs.cu -- FP8 GEMM with ue8m0 (power-of-two) block scales on the block-scaled MMA.
//
// When every scale is a power of two (ue8m0 scales: "DeepSeek-V3 User Guide", FAQ "What is
// scale_fmt: ue8m0?"), the scale of a 128-wide K block can be applied by the tensor core
// itself: tcgen05.mma kind::mxf8f6f4 with block scaling multiplies each 32-wide K slice of a row
// of A by 2^sfa and of a row of B by 2^sfb, both ue8m0 exponents read from TMEM. Giving the
// four slices of block kb the exponents of a_s[m,kb] and b_s[n/128,kb] makes the MMA compute
// sum_kb a_s * b_s * P_kb exactly as §8.5.3 defines it (a power-of-two factor is exact in
// fp32), and the accumulator then stays in TMEM for the whole K loop: no promotion pass.
//
// Warp layout (320 threads):
//   warps 0 .. 3   scale-factor writers: per K block, tcgen05.st the exponents of the tile's
//                  128 rows of a_s and of its b_s block into the stage's TMEM scale slot
//   warps 4 .. 7   epilogue: read the finished accumulator, round to bf16, store
//   warp 8         TMA producer
//   warp 9         MMA issuer (allocates and frees TMEM)
// TMEM: two BN-column accumulators, then per stage 8 columns of scale factors (4 for A, 4 for
// B). A stage's full barrier completes when its TMA bytes have landed AND the four scale-factor
// warps have written its slot; the MMA's commit to the stage's empty barrier frees both.
//
// Scale-factor placement. Tiles are BN <= 128 columns wide and start on a multiple of BN, so
// the tile lies inside one 128-row block of B and its B exponent is one value: every lane,
// column and byte of the B slot holds it. For A, lane L of the slot's four columns holds
//   L < 32:  column j = exponent of tile row L + 32 j
//   L >= 32: every column = exponent of tile row L
// with the same byte in all four bytes of a word. This serves row m whether the tensor core
// takes it from lane m column 0, from lane m column m/32, or from lane m%32 column m/32.
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

template <int BN>
struct BsCfg {
    static_assert(BN == 64 || BN == 128, "the B exponent must be uniform over a tile");
    static constexpr int SF_WARPS = 4;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 32 * (SF_WARPS + EPI_WARPS + 2);
    static constexpr int B_TILE = BN * BK;
    static constexpr int STAGE = A_TILE + B_TILE;
    static constexpr int SF_COLS = 8;                 // per stage: A in 0..3, B in 4..7
    static constexpr int SF_COL0 = 2 * BN;            // after the two accumulators
};

template <int BN>
__host__ __device__ constexpr uint32_t bs_tmem_cols(int stages) {
    return tmem_cols_for(static_cast<uint32_t>(2 * BN + stages * BsCfg<BN>::SF_COLS));
}

// Biased exponent of a scale that must be 2^e with -126 <= e <= 127: for such a value the
// binary32 exponent field is the ue8m0 code of the same number. `ok` is cleared otherwise.
__device__ __forceinline__ uint32_t ue8m0_code(float v, bool& ok) {
    const uint32_t bits = __float_as_uint(v);
    const uint32_t e = (bits >> 23) & 0xFFu;
    ok = ok && (bits & 0x807FFFFFu) == 0 && e != 0 && e != 0xFFu;
    return e;
}

__device__ __forceinline__ uint32_t splat4(uint32_t byte) { return byte * 0x01010101u; }

// Exponents of a_s[row, kb] for the rows this scale-factor lane writes (4 rows in warp 0,
// the lane's own row elsewhere) and of b_s[nb, kb], raw fp32; kb past the end loads nothing.
__device__ __forceinline__ void load_sf(float* va, float& vb, const float* const* as_r,
                                        const float* bs_row, int kb, int num_kb, bool four) {
    if (kb >= num_kb) return;
    if (four) {
#pragma unroll
        for (int j = 0; j < 4; ++j) va[j] = __ldg(as_r[j] + kb);
    } else {
        const float v = __ldg(as_r[0] + kb);
#pragma unroll
        for (int j = 0; j < 4; ++j) va[j] = v;
    }
    vb = __ldg(bs_row + kb);
}

template <int BN>
__global__ void __launch_bounds__(BsCfg<BN>::THREADS, 1)
    gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs g, const __grid_constant__ GroupTable gt, const int stages) {
    using Cfg = BsCfg<BN>;
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
    constexpr int PRODUCER = Cfg::SF_WARPS + Cfg::EPI_WARPS;
    constexpr int ISSUER = PRODUCER + 1;
    const uint32_t tmem_cols = bs_tmem_cols<BN>(stages);

    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        init_ring(ring, stages, Cfg::EPI_WARPS, 1 + Cfg::SF_WARPS);
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == ISSUER) tmem_alloc(ring.tmem_holder, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;

    if (warp == PRODUCER) {
        if (lane == 0) {
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
        }
    } else if (warp == ISSUER) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_block_scaled(BM, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&ring.tempty[buf], tphase ^ 1)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&ring.full[stage], phase)) {
                        record_error(FP8BS_DEVERR_MMA_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * A_TILE);
                    const uint32_t b_addr = smem_addr(sB + stage * Cfg::B_TILE);
                    const uint32_t sfa =
                        tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
#pragma unroll
                    for (int j = 0; j < BK / MMA_K; ++j)
                        mma_f8_block_scaled(d_tmem, smem_desc_k_sw128(a_addr + j * MMA_K),
                                            smem_desc_k_sw128(b_addr + j * MMA_K), idesc, sfa,
                                            sfa + 4, (kb > 0 || j > 0) ? 1u : 0u);
                    mma_commit(&ring.empty[stage]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&ring.tfull[buf]);
                buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            // Make sure nothing this thread issued is still running before TMEM is freed.
            mma_commit(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else if (warp < Cfg::SF_WARPS) {
        // Scale-factor writers: warp w owns TMEM lanes 32w .. 32w+31 of every slot.
        constexpr int P = 8;                      // K blocks of scales in flight per lane
        const int nb_count = (g.N + 127) / 128;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const bool four = (warp == 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true, pow2 = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            // Rows past the group's end (clamped into A) are computed but never stored.
            const float* as_r[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = t.m0 + (four ? lane + 32 * j : warp * 32 + lane);
                as_r[j] = g.a_s + static_cast<int64_t>(min(row, g.M - 1)) * num_kb;
            }
            const float* bs_row =
                g.b_s + (static_cast<int64_t>(t.g) * nb_count + t.n0 / 128) * num_kb;
            float va[P][4], vb[P];
#pragma unroll
            for (int i = 0; i < P; ++i) load_sf(va[i], vb[i], as_r, bs_row, i, num_kb, four);
            for (int kb0 = 0; ok && kb0 < num_kb; kb0 += P) {
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    const int kb = kb0 + i;
                    if (kb >= num_kb) break;
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) w[j] = splat4(ue8m0_code(va[i][j], pow2));
                    const uint32_t wb = splat4(ue8m0_code(vb[i], pow2));
                    load_sf(va[i], vb[i], as_r, bs_row, kb + P, num_kb, four);
                    if (!warp_wait(&ring.empty[stage], phase ^ 1)) {
                        if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + lane_base +
                                           static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
                    tmem_st_4cols(taddr, w[0], w[1], w[2], w[3]);
                    tmem_st_4cols(taddr + 4, wb, wb, wb, wb);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ring.full[stage]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
        if (!__all_sync(0xffffffffu, pow2) && lane == 0) record_error(FP8BS_DEVERR_SCALE_NOT_POW2);
    } else {
        // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. tile rows of the same numbers.
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        int buf = 0;
        uint32_t tphase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            if (!warp_wait(&ring.tfull[buf], tphase)) {
                if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * BN);
            float acc[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld_32cols(taddr + 32 * c, acc + 32 * c);
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_wait_ld_32(acc + 32 * c);
            // The accumulator is in registers: hand the buffer back before storing.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.tempty[buf]);
            buf ^= 1;
            if (buf == 0) tphase ^= 1;
            const int row = t.m0 + row_in_tile;
            if (row < t.row_end) {
                __nv_bfloat16* crow =
                    static_cast<__nv_bfloat16*>(g.c) + static_cast<int64_t>(row) * g.N + t.n0;
                store_row_bf16<BN>(crow, acc, min(BN, g.N - t.n0), (g.N & 7) == 0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == ISSUER) tmem_dealloc(tmem_base, tmem_cols);
}

template <int BN>
cudaError_t launch_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                      const GroupTable& gt, int num_sms, cudaStream_t stream) {
    using Cfg = BsCfg<BN>;
    int stages = (kSmemLimit - 1024 - ring_bytes(kMaxStages)) / Cfg::STAGE;
    if (stages > kMaxStages) stages = kMaxStages;
    static_assert(bs_tmem_cols<BN>(kMaxStages) <= 512, "TMEM holds 512 columns");
    const int smem = 1024 + stages * Cfg::STAGE + ring_bytes(stages);
    cudaError_t e = set_smem(gemm_bs_kernel<BN>, smem);
    if (e != cudaSuccess) return e;
    const int tiles = gt.tile_off[gt.num_groups];
    if (tiles == 0) return cudaSuccess;
    const int grid = tiles < num_sms ? tiles : num_sms;
    return launch_pdl(gemm_bs_kernel<BN>, grid, Cfg::THREADS, smem, stream, tmA, tmB, g, gt,
                      stages);
}

}  // namespace

int pick_tile_n_bs(int64_t m_tiles_total, int64_t N, int num_sms) {
    return m_tiles_total * ((N + 127) / 128) * 5 >= num_sms * 4 ? 128 : 64;
}

cudaError_t launch_gemm_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           const GroupTable& gt, int BN, int num_sms, cudaStream_t stream) {
    switch (BN) {
        case 64: return launch_bs<64>(tmA, tmB, g, gt, num_sms, stream);
        case 128: return launch_bs<128>(tmA, tmB, g, gt, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_error_bs(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
