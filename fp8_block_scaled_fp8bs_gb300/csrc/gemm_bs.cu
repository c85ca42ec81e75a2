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
// Warp layout (320 threads; 352 at BN = 64):
//   warps 0 .. 3   scale-factor writers: per K block, tcgen05.st the exponents of the tile's
//                  128 rows of a_s and of its b_s block into the stage's TMEM scale slot
//   warps 4 .. 7   epilogue: read the finished accumulator, round to bf16, store
//   warp 8         TMA producer
//   warp 9         MMA issuer (allocates and frees TMEM)
//   warp 10        BN = 64 and 192: a second MMA issuer. The two take a tile's K blocks in
//                  turn, each into its own accumulator; the epilogue adds the two. One thread
//                  issuing alone advances one K block per ~650-770 clk at these widths,
//                  more than the MMAs take (MLA N = 576: 22.2 us with one issuer, 17.9-18.3 us
//                  with two; N = 1536 at 192: 26.6 and 23.2 us).
// TMEM: accumulator buffers of BN columns per issuer (two, or one at BN > 128), then per stage
// 8 or 12 columns of scale factors (4 for A, 4 or 8 for B). A stage's full barrier completes
// when its TMA bytes have landed AND the four scale-factor warps have written its slot; the
// MMA's commit to the stage's empty barrier frees both.
//
// Scale-factor placement. The tensor core takes the exponent of row m of A from lane m,
// column m/32 of the A slot, and the exponent of row n of B (for output rows of lane quarter q)
// from lane 32q + n%32, column n/32 of the B slot -- measured on GB300 by giving every lane,
// column and byte of the slots a distinct exponent. Lane L writes the exponent of tile row L
// into all four columns of the A slot. Tiles start on a multiple of BN: a 64- or 128-wide tile
// lies inside one 128-row block of B, whose exponent is written to every lane and column of a
// 4-column B slot; a 256-wide tile spans two blocks, whose exponents fill columns 0-3 and 4-7
// of an 8-column B slot. Every byte of a word holds the same exponent.
//
// Work schedule. Data-parallel: CTA c computes tiles c, c + gridDim.x, ... whole. Stream-K
// (when a workspace is given and the tiles alone would leave SMs idle): the tiles x K blocks
// units are cut into gridDim.x equal contiguous ranges and CTA c works through its range tile
// by tile, so a tile's K loop may be shared by consecutive CTAs. Only a CTA's first piece can
// start inside a tile; that CTA writes its fp32 partial to its own workspace slot and counts it
// in the flag of the tile's owner, the CTA holding the tile's first K blocks (the last piece of
// its own range). The owner waits for its flag, adds the partials in K order -- a fixed order,
// so results do not depend on timing -- resets the flag and stores. It only waits on CTAs
// after it, each of which writes its partial before anything else, and every CTA of the grid
// is resident (one per SM), so the wait always ends.
#include <atomic>

#include "gemm_common.cuh"

namespace fp8bs {

namespace {

template <int BN>
struct BsCfg {
    static_assert(BN == 64 || BN == 128 || BN == 192 || BN == 256, "tile width");
    static constexpr int SF_WARPS = 4;
    static constexpr int EPI_WARPS = 4;
    // MMA issuers: two at BN = 64 and 192, taking a tile's K blocks in turn into accumulators
    // of their own (one thread issuing alone advances one K block per ~650-770 clk at these
    // widths whatever N is; the MLA q projection, 128 tiles of 192, went from 26.6 to 23.2 us).
    // A third at 64 changed nothing (MLA kv projection 17.7 us either way). 128 keeps one (two
    // buffers of two accumulators would not fit in TMEM, and one buffer loses the epilogue
    // overlap its many-round shapes need); 256 has no room for a second.
    static constexpr int ISSUERS = (BN <= 64 || BN == 192) ? 2 : 1;
    static constexpr int THREADS = 32 * (SF_WARPS + EPI_WARPS + 1 + ISSUERS);
    static constexpr int B_TILE = BN * BK;
    static constexpr int STAGE = A_TILE + B_TILE;
    // Scale-factor columns per stage: A in 0..3, then B: 4 columns (one 128-row block of B
    // per tile, BN <= 128) or 8 (BN = 192 or 256: the tile spans two blocks of B; column c of
    // the slot covers tile rows 32c .. 32c+31).
    static constexpr int SF_B_COLS = BN > 128 ? 8 : 4;
    static constexpr int SF_COLS = 4 + SF_B_COLS;
    // Accumulators: two buffers of ISSUERS x BN columns (the epilogue of one tile overlaps the
    // next), or one where two would leave no TMEM for the scale factors (BN = 256, and 192
    // with its two issuers).
    static constexpr int NBUF = BN > 128 ? 1 : 2;
    static constexpr int ACC = ISSUERS * BN;          // TMEM columns of one buffer
    static constexpr int SF_COL0 = NBUF * ACC;
    static constexpr int PART = BM * BN * 4;          // one fp32 partial tile (stream-K)
    // Shared-memory scratch of the epilogue's coalesced stores of whole 192- and 256-wide tiles,
    // 4 KB per epilogue warp. Narrower tiles store rows directly: at BN = 128 the stages fill
    // shared memory, and at BN = 64 a lane's 128-byte row is one whole line anyway (the MLA kv
    // projection measured 17.5 us direct, 19.0 us through the scratch).
    static constexpr int SCRATCH = BN > 128 ? EPI_WARPS * 4096 : 0;
};

template <int BN>
__host__ __device__ constexpr uint32_t bs_tmem_cols(int stages) {
    return tmem_cols_for(
        static_cast<uint32_t>(BsCfg<BN>::NBUF * BsCfg<BN>::ACC + stages * BsCfg<BN>::SF_COLS));
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

// Hand a TMEM accumulator back to the MMA issuer once this warp's loads of it have completed.
__device__ __forceinline__ void release_tmem(uint64_t* tempty, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tempty);
}

// With several MMA issuers (issuer i's accumulator BN columns after issuer 0's): add to v the
// 32 columns at `taddr` of the accumulators of issuers 1 .. nacc-1, in issuer order.
template <int BN, int ISSUERS>
__device__ __forceinline__ void add_issuer_accs(uint32_t taddr, int nacc, float* v) {
#pragma unroll
    for (int i = 1; i < ISSUERS; ++i) {
        if (i < nacc) {
            float t[32];
            tmem_ld_32cols(taddr + static_cast<uint32_t>(i * BN), t);
            tmem_wait_ld_32(t);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] += t[k];
        }
    }
}

// PLAIN: whole tiles only (no stream-K workspace, no split K). Its instantiation compiles the
// schedule with those fixed, which drops the stream-K and split-K paths: the MLA projections
// (whole tiles) ran ~4 % faster that way (N = 576: 18.35 -> 17.6 us; N = 1536: 23.2 -> 22.3 us).
template <int BN, bool PLAIN>
__global__ void __launch_bounds__(BsCfg<BN>::THREADS, 1)
    gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs g, const __grid_constant__ GroupTable gt, const int stages,
                   const StreamK sk_arg) {
    StreamK sk = sk_arg;
    if constexpr (PLAIN) {
        sk.parts = nullptr;
        sk.flags = nullptr;
        sk.ksplit = 1;
        sk.dp_tiles = 0;
    }
    using Cfg = BsCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + stages * A_TILE;
    const bool stream_k = sk.parts != nullptr;
    // The epilogue's store scratch (after the stages). Stream-K only: the first contributor's
    // partial of the tile this CTA owns, copied in while the owner's own piece still runs
    // (1024-byte aligned), and the barrier counting its bytes (after the ring).
    uint8_t* sScratch = sB + stages * Cfg::B_TILE;
    float4* sPart = reinterpret_cast<float4*>(sScratch + Cfg::SCRATCH);
    const Ring ring = carve_ring(sScratch + Cfg::SCRATCH + (stream_k ? Cfg::PART : 0), stages);
    uint64_t* part_bar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ring.full) +
                                                     ring_bytes(stages));

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
        // every issuer commits each finished buffer and its final drain
        init_ring(ring, stages, Cfg::EPI_WARPS, 1 + Cfg::SF_WARPS, Cfg::ISSUERS);
        if (stream_k) {
            mbar_init(part_bar, 1);
            fence_barrier_init();
        }
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == ISSUER) tmem_alloc(ring.tmem_holder, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;

    Sched sched = sched_begin(sk, num_tiles, num_kb);
    int tile, kb0, kb1;
    const bool split = sk.ksplit > 1;
    bool exchanged = false;      // split K: this thread has been through the exchange

    if (warp == PRODUCER) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            while (ok && sched_next(sched, num_kb, tile, kb0, kb1)) {
                const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
                const int b_row = t.g * g.N + t.n0;      // row of the stacked B
                for (int kb = kb0; kb < kb1; ++kb) {
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
    } else if (warp >= ISSUER && warp < ISSUER + Cfg::ISSUERS) {
        if (lane == 0) {
            const int me = warp - ISSUER;
            constexpr uint32_t idesc = idesc_e4m3_block_scaled(BM, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            while (ok && sched_next(sched, num_kb, tile, kb0, kb1)) {
                if (!mbar_wait(&ring.tempty[buf], tphase ^ 1)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem =
                    tmem_base + static_cast<uint32_t>(buf * Cfg::ACC + me * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if ((kb - kb0) % Cfg::ISSUERS != me) {     // the other issuer's K block
                        if (++stage == stages) {
                            stage = 0;
                            phase ^= 1;
                        }
                        continue;
                    }
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
                                            sfa + 4,
                                            (kb - kb0 >= Cfg::ISSUERS || j > 0) ? 1u : 0u);
                    mma_commit(&ring.empty[stage]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&ring.tfull[buf]);
                if (Cfg::NBUF == 2) buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            // Make sure nothing this thread issued is still running before TMEM is freed.
            mma_commit(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else if (warp < Cfg::SF_WARPS) {
        // Scale-factor writers: warp w owns TMEM lanes 32w .. 32w+31 of every slot, i.e. tile
        // rows 32w .. 32w+31.
        constexpr int P = 8;                      // K blocks of scales in flight per lane
        const int nb_count = (g.N + 127) / 128;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true, pow2 = true;
        while (ok && sched_next(sched, num_kb, tile, kb0, kb1)) {
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            // Rows past the group's end (clamped into A) are computed but never stored.
            const int row = min(t.m0 + warp * 32 + lane, g.M - 1);
            const float* as_row = g.a_s + static_cast<int64_t>(row) * num_kb;
            const float* bs_row =
                g.b_s + (static_cast<int64_t>(t.g) * nb_count + t.n0 / 128) * num_kb;
            // BN = 192 or 256: the tile's second 128-row block of B (the first again past N)
            const float* bs_row2 = BN > 128 && t.n0 / 128 + 1 < nb_count ? bs_row + num_kb : bs_row;
            // A 192-wide tile starting at an odd multiple of 64 meets its second block of B at
            // tile row 64 (column 2 of the slot), otherwise at row 128 (column 4).
            const bool b_shift = BN > 128 && (t.n0 & 127) != 0;
            float va[P], vb[P], vb2[P];
#pragma unroll
            for (int i = 0; i < P; ++i) {
                if (kb0 + i < kb1) {
                    va[i] = __ldg(as_row + kb0 + i);
                    vb[i] = __ldg(bs_row + kb0 + i);
                    if constexpr (BN > 128) vb2[i] = __ldg(bs_row2 + kb0 + i);
                }
            }
            for (int kbp = kb0; ok && kbp < kb1; kbp += P) {
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    const int kb = kbp + i;
                    if (kb >= kb1) break;
                    const uint32_t wa = splat4(ue8m0_code(va[i], pow2));
                    const uint32_t wb = splat4(ue8m0_code(vb[i], pow2));
                    uint32_t wb2 = 0;
                    if constexpr (BN > 128) wb2 = splat4(ue8m0_code(vb2[i], pow2));
                    if (!warp_wait(&ring.empty[stage], phase ^ 1)) {
                        if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + lane_base +
                                           static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
                    tmem_st_4cols(taddr, wa, wa, wa, wa);
                    if constexpr (BN > 128) {
                        const uint32_t wx = b_shift ? wb2 : wb;
                        tmem_st_4cols(taddr + 4, wb, wb, wx, wx);
                        tmem_st_4cols(taddr + 8, wb2, wb2, wb2, wb2);
                    } else {
                        tmem_st_4cols(taddr + 4, wb, wb, wb, wb);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ring.full[stage]);
                    // The scales of kb + P, requested only now: a release (the arrive) would
                    // otherwise wait for them to return from memory.
                    if (kb + P < kb1) {
                        va[i] = __ldg(as_row + kb + P);
                        vb[i] = __ldg(bs_row + kb + P);
                        if constexpr (BN > 128) vb2[i] = __ldg(bs_row2 + kb + P);
                    }
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
        const int epi_thread = row_in_tile;        // 0 .. 127
        int buf = 0;
        uint32_t tphase = 0, part_phase = 0;
        bool ok = true;
        while (ok && sched_next(sched, num_kb, tile, kb0, kb1)) {
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            const bool owner = !split && kb0 == 0 && kb1 < num_kb;
            int parts = 0;
            bool got = true;
            if (owner) {
                // The tile continues in the next CTAs, each of which starts with its piece of
                // it. While this CTA's own piece is still on the tensor cores, thread 0 waits
                // for their partials and copies the first into shared memory; the outcome
                // reaches the other epilogue threads through the word after the TMEM address.
                parts = sk_contributors(sk, tile, num_tiles, num_kb);
                volatile uint32_t* outcome = ring.tmem_holder + 1;
                if (epi_thread == 0) {
                    got = flag_wait(sk.flags + blockIdx.x, parts);
                    if (got) {
                        sk.flags[blockIdx.x] = 0;        // ready for the next call
                        fence_proxy_async_global();
                        const float4* src = sk.parts + static_cast<int64_t>(blockIdx.x + 1) *
                                                           (BN / 4) * BM;
                        constexpr uint32_t kBytes = BM * BN * sizeof(float);
                        mbar_arrive_expect_tx(part_bar, kBytes);
                        for (int q = 0; q < 4; ++q)
                            bulk_load(sPart + q * (kBytes / 64), src + q * (kBytes / 64),
                                      kBytes / 4, part_bar);
                    } else {
                        record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                    }
                    *outcome = got ? 1u : 0u;
                }
                epilogue_bar<128>();
                got = *outcome != 0;
            }
            if (!warp_wait(&ring.tfull[buf], tphase)) {
                if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * Cfg::ACC);
            // Issuer i's accumulator (i x BN columns on) holds K blocks kb0 + i, kb0 + i +
            // ISSUERS, ...: the first nacc issuers received some.
            const int nacc = min(Cfg::ISSUERS, kb1 - kb0);
            if (split) {
                // Split K: once every CTA of the cluster is past its K loop (its stage memory
                // free), send each slice of the accumulator to the CTA that adds that slice up;
                // then add up this CTA's slice and store it.
                const SplitTile sp = split_tile(BN, sk.ksplit, smem);
                cluster_sync();
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld_32cols(taddr + 32 * c, v);
                    tmem_wait_ld_32(v);
                    add_issuer_accs<BN, Cfg::ISSUERS>(taddr + 32 * c, nacc, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        split_push4(sp, row_in_tile, 32 * c + 4 * j,
                                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                }
                release_tmem(&ring.tempty[buf], lane);
                cluster_sync();
                split_reduce_store<128>(sp, reinterpret_cast<const float4*>(smem), epi_thread, BN,
                                        t, g);
                exchanged = true;
                break;
            }
            const int row = t.m0 + row_in_tile;
            const bool store = row < t.row_end;
            __nv_bfloat16* crow =
                static_cast<__nv_bfloat16*>(g.c) + static_cast<int64_t>(row) * g.N + t.n0;
            const int valid = min(BN, g.N - t.n0);
            const bool vec = (g.N & 7) == 0;
            uint8_t* scratch = Cfg::SCRATCH > 0 ? sScratch + quarter * 4096 : nullptr;
            const WarpRows wr{static_cast<__nv_bfloat16*>(g.c), g.N, t.m0 + quarter * 32,
                              t.row_end, t.n0};

            if (kb0 == 0 && kb1 == num_kb) {
                if constexpr (BN > 128) {
                    // A whole 192- or 256-wide tile: the row into registers as bf16 pairs, the
                    // buffer back (at BN = 256 the only one: the next tile's MMAs wait for it),
                    // then store. Storing between the loads held the buffer ~9K clk per tile.
                    static_assert(BN <= 128 || Cfg::ISSUERS <= 2, "the wide epilogue adds two");
                    drain_row_bf16<BN>(taddr, crow, store, valid, vec, nacc > 1, scratch, wr, lane,
                                       [&] { release_tmem(&ring.tempty[buf], lane); });
                } else {
                    // A whole tile: the accumulator into registers, the buffer back, then store.
                    float acc[BN];
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) tmem_ld_32cols(taddr + 32 * c, acc + 32 * c);
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) tmem_wait_ld_32(acc + 32 * c);
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        add_issuer_accs<BN, Cfg::ISSUERS>(taddr + 32 * c, nacc, acc + 32 * c);
                    release_tmem(&ring.tempty[buf], lane);
                    if (Cfg::SCRATCH > 0 && vec) {
                        uint32_t pk[BN / 2];
#pragma unroll
                        for (int i = 0; i < BN / 2; ++i) pk[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
                        store_rows_coalesced<BN>(scratch, pk, wr, lane);
                    } else if (store) {
                        store_row_bf16<BN>(crow, acc, valid, vec);
                    }
                }
            } else if (kb0 > 0) {
                // A piece that does not start its tile: publish the partial in this CTA's slot,
                // 32 columns at a time, and count it in the flag of the tile's owner.
                float4* slot = sk.parts + static_cast<int64_t>(blockIdx.x) * (BN / 4) * BM;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld_32cols(taddr + 32 * c, v);
                    tmem_wait_ld_32(v);
                    add_issuer_accs<BN, Cfg::ISSUERS>(taddr + 32 * c, nacc, v);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(slot + (8 * c + q) * BM + row_in_tile,
                               make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
                }
                release_tmem(&ring.tempty[buf], lane);
                epilogue_bar<128>();
                if (epi_thread == 0) {
                    __threadfence();
                    flag_add_release(sk.flags + sk_tile_owner(sk, tile, num_tiles, num_kb), 1);
                }
            } else {
                // The tile's first piece: per 32 columns, add the partials of the pieces that
                // continue it in K order (the first from shared memory) and store.
                const bool have = got && mbar_wait(part_bar, part_phase);
                part_phase ^= 1;
                if (got && !have && lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld_32cols(taddr + 32 * c, v);
                    tmem_wait_ld_32(v);
                    add_issuer_accs<BN, Cfg::ISSUERS>(taddr + 32 * c, nacc, v);
                    if (have) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 p = sPart[(8 * c + q) * BM + row_in_tile];
                            v[4 * q] += p.x;
                            v[4 * q + 1] += p.y;
                            v[4 * q + 2] += p.z;
                            v[4 * q + 3] += p.w;
                        }
#pragma unroll 1
                        for (int j = 2; j <= parts; ++j) {
                            const float4* slot =
                                sk.parts + static_cast<int64_t>(blockIdx.x + j) * (BN / 4) * BM;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 p = __ldcg(slot + (8 * c + q) * BM + row_in_tile);
                                v[4 * q] += p.x;
                                v[4 * q + 1] += p.y;
                                v[4 * q + 2] += p.z;
                                v[4 * q + 3] += p.w;
                            }
                        }
                    }
                    if (store && have) store_row_bf16<32>(crow + 32 * c, v, valid - 32 * c, vec);
                }
                release_tmem(&ring.tempty[buf], lane);
                if (!have) ok = false;
            }
            if (Cfg::NBUF == 2) buf ^= 1;
            if (buf == 0) tphase ^= 1;
        }
    }

    // Split K: every thread takes part in the exchange's two cluster barriers (the epilogue
    // warps above, unless a wait ran out before them).
    if (split && !exchanged) {
        cluster_sync();
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == ISSUER) tmem_dealloc(tmem_base, tmem_cols);
}

// ================================================================ CTA pairs
//
// The same GEMM on CTA pairs (cta_group::2): a cluster of two CTAs on neighbouring SMs computes
// a 256 x BN tile. CTA r (cluster rank r) loads rows 128r .. 128r+127 of the A tile and rows
// (BN/2)r .. (BN/2)(r+1)-1 of the B tile into its own shared memory, writes the scale factors
// of its 128 rows of A and of all BN rows of B into its own TMEM, and receives its 128 rows of
// the accumulator in its own TMEM; the even CTA issues the MMAs for both. Per SM this halves
// the bytes of B that TMA writes to and the tensor cores read from shared memory in each K
// block -- the one-CTA kernel moves 2 x (16 KB + BN x 128 B) per K block through one SM's
// shared memory, more than it delivers at the MMA rate.
//   - Both CTAs' TMA bytes complete the even CTA's `full` barrier of the stage; the even CTA's
//     MMA commits arrive on the `empty` and `tfull` barriers of both CTAs at once; both CTAs'
//     epilogue warps release a TMEM buffer on the even CTA's `tempty` barrier.
//   - Scale factors travel in chunks of CHUNK K blocks through a ring of SLOTS TMEM slots per
//     CTA: both CTAs' scale-factor warps fill a slot and arrive on the even CTA's `sf_full`,
//     the MMA commit after the chunk's last K block frees it in both CTAs (`sf_empty`), and
//     the writers run up to SLOTS - 1 chunks ahead of the MMAs. A hand-over between the SMs
//     per K block (the one-CTA kernel's scheme) measured 2.3 x slower than the same pipeline
//     without scale factors; per chunk it is paid once per CTA per CHUNK K blocks.
//   - Whole tiles, one group; tiles ordered 256-row blocks fastest.
template <int BN>
struct PairCfg {
    static_assert(BN == 128 || BN == 192 || BN == 256, "pair tile width");
    static constexpr int SF_WARPS = 4;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 32 * (SF_WARPS + EPI_WARPS + 2);
    static constexpr int B_HALF = (BN / 2) * BK;            // this CTA's half of the B tile
    static constexpr int STAGE = A_TILE + B_HALF;
    static constexpr int CHUNK = 8;                          // K blocks per scale-factor slot
    static constexpr int SLOTS = 2;
    static constexpr int SF_A = 4 * CHUNK;                   // A: 4 columns per K block
    static constexpr int SF_SLOT = SF_A + 8 * CHUNK;         // then B: 8 columns per K block
    static constexpr int NBUF = BN > 128 ? 1 : 2;
    static constexpr int SF_COL0 = NBUF * BN;
};

template <int BN>
__host__ __device__ constexpr int pair_stages() {
    return (kSmemLimit - 1024 - ring_bytes(kMaxStages) - 64) / PairCfg<BN>::STAGE > kMaxStages
               ? kMaxStages
               : (kSmemLimit - 1024 - ring_bytes(kMaxStages) - 64) / PairCfg<BN>::STAGE;
}

template <int BN>
__host__ __device__ constexpr int pair_smem() {
    return 1024 + pair_stages<BN>() * PairCfg<BN>::STAGE + ring_bytes(pair_stages<BN>()) + 64;
}

template <int BN>
__host__ __device__ constexpr uint32_t pair_tmem_cols() {
    return tmem_cols_for(
        static_cast<uint32_t>(PairCfg<BN>::SF_COL0 + PairCfg<BN>::SLOTS * PairCfg<BN>::SF_SLOT));
}

template <int BN>
__global__ void __launch_bounds__(PairCfg<BN>::THREADS, 1)
    gemm_bs_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
    using Cfg = PairCfg<BN>;
    constexpr int stages = pair_stages<BN>();
    constexpr uint32_t tmem_cols = pair_tmem_cols<BN>();
    static_assert(tmem_cols <= 512, "TMEM holds 512 columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + stages * A_TILE;
    const Ring ring = carve_ring(sB + stages * Cfg::B_HALF, stages);
    // Scale-factor slots: [SLOTS] filled (even CTA: both CTAs' writers), [SLOTS] free.
    uint64_t* sf_full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ring.full) +
                                                    ring_bytes(stages));
    uint64_t* sf_empty = sf_full + Cfg::SLOTS;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int num_kb = g.K / BK;
    const int m_pairs = (g.M + 2 * BM - 1) / (2 * BM);
    const int num_tiles = m_pairs * ((g.N + BN - 1) / BN);
    const int nb_count = (g.N + 127) / 128;
    constexpr int PRODUCER = Cfg::SF_WARPS + Cfg::EPI_WARPS;
    constexpr int ISSUER = PRODUCER + 1;

    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        // full: the leader's producer (and both CTAs' TMA bytes); tempty: the epilogue warps of
        // both CTAs; sf_full: the scale-factor warps of both CTAs.
        init_ring(ring, stages, 2 * Cfg::EPI_WARPS, 1);
        for (int i = 0; i < Cfg::SLOTS; ++i) {
            mbar_init(&sf_full[i], 2 * Cfg::SF_WARPS);
            mbar_init(&sf_empty[i], 1);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == ISSUER) tmem_alloc_pair(ring.tmem_holder, tmem_cols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // both CTAs' barriers are initialised before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = *ring.tmem_holder;

    if (warp == PRODUCER) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                // This CTA's rows of A and of B; a box that would start past the end of the
                // matrix (ragged last tiles) is loaded in range instead: the rows it feeds are
                // never stored, and the byte count stays the same.
                const int m0 = min((tile % m_pairs) * (2 * BM) + static_cast<int>(rank) * BM,
                                   g.M - 1);
                const int nb0 = min((tile / m_pairs) * BN + static_cast<int>(rank) * (BN / 2),
                                    g.N - 1);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&ring.empty[stage], phase ^ 1)) {
                        record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&ring.full[stage], 2 * Cfg::STAGE);
                    const uint32_t full0 = mapa_shared(smem_addr(&ring.full[stage]), 0);
                    tma_load_2d_pair(sA + stage * A_TILE, &tmA, full0, kb * BK, m0);
                    tma_load_2d_pair(sB + stage * Cfg::B_HALF, &tmB, full0, kb * BK, nb0);
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    drain_tma(ring, stages, issued);
                } else {
                    // This CTA's copies complete on the leader's barriers: give copies still in
                    // flight time to land before the CTA may exit.
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
    } else if (warp == ISSUER) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_e4m3_block_scaled(2 * BM, BN);
            int stage = 0, buf = 0, slot = 0;
            uint32_t phase = 0, tphase = 0, sphase = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                if (!mbar_wait_cluster(&ring.tempty[buf], tphase ^ 1)) {
                    record_error(FP8BS_DEVERR_MMA_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    const int j = kb % Cfg::CHUNK;
                    if ((j == 0 && !mbar_wait_cluster(&sf_full[slot], sphase)) ||
                        !mbar_wait(&ring.full[stage], phase)) {
                        record_error(FP8BS_DEVERR_MMA_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * A_TILE);
                    const uint32_t b_addr = smem_addr(sB + stage * Cfg::B_HALF);
                    const uint32_t sf = tmem_base +
                                        static_cast<uint32_t>(Cfg::SF_COL0 + slot * Cfg::SF_SLOT);
#pragma unroll
                    for (int jj = 0; jj < BK / MMA_K; ++jj)
                        mma_f8_block_scaled_pair(d_tmem, smem_desc_k_sw128(a_addr + jj * MMA_K),
                                                 smem_desc_k_sw128(b_addr + jj * MMA_K), idesc,
                                                 sf + 4 * j, sf + Cfg::SF_A + 8 * j,
                                                 (kb > 0 || jj > 0) ? 1u : 0u);
                    mma_commit_pair(&ring.empty[stage]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (j == Cfg::CHUNK - 1 || kb == num_kb - 1) {
                        mma_commit_pair(&sf_empty[slot]);     // the slot is free in both CTAs
                        if (++slot == Cfg::SLOTS) {
                            slot = 0;
                            sphase ^= 1;
                        }
                    }
                }
                if (!ok) break;
                mma_commit_pair(&ring.tfull[buf]);
                if (Cfg::NBUF == 2) buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            // Make sure nothing issued is still running before TMEM is freed.
            mma_commit_pair(ring.drain);
            if (!mbar_wait(ring.drain, 0, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
        }
    } else if (warp < Cfg::SF_WARPS) {
        // Scale-factor writers: warp w owns TMEM lanes 32w .. 32w+31 of this CTA's slots, i.e.
        // rows 32w .. 32w+31 of its 128 rows of the tile; every lane writes the exponents of
        // all BN rows of B (the tensor core of each CTA reads them from its own TMEM). Per K
        // block j of a chunk: A exponent in columns 4j .. 4j+3; B in SF_A + 8j .. +7, column c
        // for tile rows 32c .. 32c+31 (the second 128-row block of B from column 2 or 4 on).
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t sf_full0 = mapa_shared(smem_addr(sf_full), 0);
        int slot = 0;
        uint32_t sphase = 0;
        bool ok = true, pow2 = true;
        for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
            const int m0 = (tile % m_pairs) * (2 * BM) + static_cast<int>(rank) * BM;
            const int n0 = (tile / m_pairs) * BN;
            const int row = min(m0 + warp * 32 + lane, g.M - 1);
            const float* as_row = g.a_s + static_cast<int64_t>(row) * num_kb;
            const float* bs_row = g.b_s + static_cast<int64_t>(n0 / 128) * num_kb;
            const float* bs_row2 = BN > 128 && n0 / 128 + 1 < nb_count ? bs_row + num_kb : bs_row;
            const bool b_shift = BN > 128 && (n0 & 127) != 0;
            for (int kc = 0; kc < num_kb; kc += Cfg::CHUNK) {
                uint32_t wa[Cfg::CHUNK], wb[Cfg::CHUNK], wb2[Cfg::CHUNK];
#pragma unroll
                for (int i = 0; i < Cfg::CHUNK; ++i) {
                    wa[i] = wb[i] = wb2[i] = 0;
                    if (kc + i < num_kb) {
                        wa[i] = splat4(ue8m0_code(__ldg(as_row + kc + i), pow2));
                        wb[i] = splat4(ue8m0_code(__ldg(bs_row + kc + i), pow2));
                        wb2[i] = BN > 128 ? splat4(ue8m0_code(__ldg(bs_row2 + kc + i), pow2))
                                          : wb[i];
                    }
                }
                if (!warp_wait(&sf_empty[slot], sphase ^ 1)) {
                    if (lane == 0) record_error(FP8BS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + lane_base +
                                       static_cast<uint32_t>(Cfg::SF_COL0 + slot * Cfg::SF_SLOT);
                static_assert(Cfg::CHUNK == 8, "one 32-column A store, two 32-column B stores");
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < Cfg::CHUNK; ++i)
                    v[4 * i] = v[4 * i + 1] = v[4 * i + 2] = v[4 * i + 3] = wa[i];
                tmem_st_32cols(taddr, v);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int k = 4 * h + i;
                        const uint32_t wx = b_shift ? wb2[k] : wb[k];
                        v[8 * i + 0] = wb[k];
                        v[8 * i + 1] = wb[k];
                        v[8 * i + 2] = wx;
                        v[8 * i + 3] = wx;
                        v[8 * i + 4] = v[8 * i + 5] = v[8 * i + 6] = v[8 * i + 7] = wb2[k];
                    }
                    tmem_st_32cols(taddr + Cfg::SF_A + 32 * h, v);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(sf_full0 + static_cast<uint32_t>(slot * 8));
                if (++slot == Cfg::SLOTS) {
                    slot = 0;
                    sphase ^= 1;
                }
            }
        }
        if (!__all_sync(0xffffffffu, pow2) && lane == 0) record_error(FP8BS_DEVERR_SCALE_NOT_POW2);
    } else if (warp < Cfg::SF_WARPS + Cfg::EPI_WARPS) {
        // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (this CTA's rows of the same
        // numbers) and hands the buffer back to the leader once it has read it all.
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const bool vec = (g.N & 7) == 0;
        int buf = 0;
        uint32_t tphase = 0;
        for (int tile = pair; tile < num_tiles; tile += num_pairs) {
            const int m0 = (tile % m_pairs) * (2 * BM) + static_cast<int>(rank) * BM;
            const int n0 = (tile / m_pairs) * BN;
            if (!warp_wait(&ring.tfull[buf], tphase)) {
                if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * BN);
            const int row = m0 + row_in_tile;
            const bool store = row < g.M;
            __nv_bfloat16* crow =
                static_cast<__nv_bfloat16*>(g.c) + static_cast<int64_t>(row) * g.N + n0;
            const int valid = min(BN, g.N - n0);
            drain_row_bf16<BN>(taddr, crow, store, valid, vec, false, nullptr, WarpRows{}, lane, [&] {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(&ring.tempty[buf]), 0));
            });
            if (Cfg::NBUF == 2) buf ^= 1;
            if (buf == 0) tphase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();      // no CTA leaves while the other may still signal it or use its TMEM
    tc_fence_after();
    if (warp == ISSUER) tmem_dealloc_pair(tmem_base, tmem_cols);
}

template <int BN>
cudaError_t launch_bs_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           int pairs, cudaStream_t stream) {
    using Cfg = PairCfg<BN>;
    cudaError_t e = set_smem(gemm_bs_pair_kernel<BN>, pair_smem<BN>());
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(gemm_bs_pair_kernel<BN>, dim3(2 * pairs), Cfg::THREADS,
                              pair_smem<BN>(), stream, 2, false, tmA, tmB, g);
}

template <int BN>
int pair_clusters() {
    if (set_smem(gemm_bs_pair_kernel<BN>, pair_smem<BN>()) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return max_active_clusters(reinterpret_cast<const void*>(gemm_bs_pair_kernel<BN>),
                               PairCfg<BN>::THREADS, pair_smem<BN>(), 2);
}

// Stages and dynamic shared memory: with a stream-K workspace one partial tile (and its
// barrier) is kept in shared memory, at two stages' cost.
template <int BN>
constexpr int bs_stages(bool stream_k) {
    return (kSmemLimit - 1024 - ring_bytes(kMaxStages) - BsCfg<BN>::SCRATCH -
            (stream_k ? BsCfg<BN>::PART + 16 : 0)) / BsCfg<BN>::STAGE > kMaxStages
               ? kMaxStages
               : (kSmemLimit - 1024 - ring_bytes(kMaxStages) - BsCfg<BN>::SCRATCH -
                  (stream_k ? BsCfg<BN>::PART + 16 : 0)) / BsCfg<BN>::STAGE;
}

template <int BN>
constexpr int bs_smem(bool stream_k) {
    return 1024 + bs_stages<BN>(stream_k) * BsCfg<BN>::STAGE + BsCfg<BN>::SCRATCH +
           (stream_k ? BsCfg<BN>::PART + 16 : 0) + ring_bytes(bs_stages<BN>(stream_k));
}

template <int BN>
cudaError_t launch_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                      const GroupTable& gt, int num_sms, const StreamKArgs& ska,
                      cudaStream_t stream) {
    using Cfg = BsCfg<BN>;
    // A partial tile wider than 128 would not fit in shared memory: those widths run whole
    // tiles or split K in a cluster.
    if (BN > 128 && ska.workspace) return cudaErrorInvalidValue;
    static_assert(bs_tmem_cols<BN>(kMaxStages) <= 512, "TMEM holds 512 columns");
    const bool stream_k = ska.workspace != nullptr && ska.ksplit <= 1;
    const int stages = bs_stages<BN>(stream_k);
    const int smem = bs_smem<BN>(stream_k);
    if (ska.ksplit > 1 && split_recv_bytes(BN, ska.ksplit) > stages * Cfg::STAGE)
        return cudaErrorInvalidValue;
    const bool plain = !stream_k && ska.ksplit <= 1;
    auto kernel = plain ? gemm_bs_kernel<BN, true> : gemm_bs_kernel<BN, false>;
    cudaError_t e = set_smem(kernel, kSmemLimit);
    if (e != cudaSuccess) return e;
    const int tiles = gt.tile_off[gt.num_groups];
    if (tiles == 0) return cudaSuccess;
    StreamK sk = {nullptr, nullptr, 0, 1};
    const int grid = stream_k_grid(ska, tiles, g.K / BK, num_sms, &sk);
    e = launch_pdl_cluster(kernel, grid, Cfg::THREADS, smem, stream, sk.ksplit, stream_k, tmA, tmB,
                           g, gt, stages, sk);
    if (e == cudaSuccess || !stream_k) return e;
    // The runtime could not place every CTA of the stream-K grid at once (fewer SMs available
    // to this context than the plan assumed): whole tiles instead, which need no co-residency.
    cudaGetLastError();
    const StreamK whole = {nullptr, nullptr, 0, 1};
    e = set_smem(gemm_bs_kernel<BN, true>, kSmemLimit);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(gemm_bs_kernel<BN, true>, tiles < num_sms ? tiles : num_sms,
                              Cfg::THREADS, bs_smem<BN>(false), stream, 1, false, tmA, tmB, g,
                              gt, bs_stages<BN>(false), whole);
}

template <int BN>
int split_clusters_bs(int S) {
    using Cfg = BsCfg<BN>;
    if (split_recv_bytes(BN, S) > bs_stages<BN>(false) * Cfg::STAGE) return 0;
    if (set_smem(gemm_bs_kernel<BN, false>, kSmemLimit) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return max_active_clusters(reinterpret_cast<const void*>(gemm_bs_kernel<BN, false>), Cfg::THREADS,
                               bs_smem<BN>(false), S);
}

}  // namespace

// Tile width by rounds of tiles over the SMs times the measured time of one K block at that
// width relative to 128 (256: 134; 192 with its two MMA issuers: 104, from the prefill
// up-projection at 192 (353 us, 21 rounds) against 256 (346 us, 16 rounds); 64, also with two
// issuers: 76, from the MLA kv projection): wider tiles carry fewer operand bytes per MAC but
// leave more SMs idle when tiles are few.
int pick_tile_n_bs(int64_t m_tiles_total, int64_t N, int num_sms) {
    static const int kWidth[4] = {256, 192, 64, 128};
    static const int kCost[4] = {134, 104, 76, 100};
    int best = 128;
    int64_t best_cost = INT64_MAX;
    for (int i = 0; i < 4; ++i) {
        const int64_t tiles = m_tiles_total * ((N + kWidth[i] - 1) / kWidth[i]);
        const int64_t cost = (tiles + num_sms - 1) / num_sms * kCost[i];
        if (cost < best_cost) {
            best_cost = cost;
            best = kWidth[i];
        }
    }
    return best;
}

cudaError_t launch_gemm_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           const GroupTable& gt, int BN, int num_sms, const StreamKArgs& ska,
                           cudaStream_t stream) {
    switch (BN) {
        case 64: return launch_bs<64>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 128: return launch_bs<128>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 192: return launch_bs<192>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 256: return launch_bs<256>(tmA, tmB, g, gt, num_sms, ska, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_bs_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const GemmArgs& g, int BN, int pairs, cudaStream_t stream) {
    switch (BN) {
        case 128: return launch_bs_pair<128>(tmA, tmB, g, pairs, stream);
        case 192: return launch_bs_pair<192>(tmA, tmB, g, pairs, stream);
        case 256: return launch_bs_pair<256>(tmA, tmB, g, pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

int max_pair_clusters_bs(int BN) {
    switch (BN) {
        case 128: return pair_clusters<128>();
        case 192: return pair_clusters<192>();
        case 256: return pair_clusters<256>();
        default: return 0;
    }
}

int max_split_clusters_bs(int BN, int S) {
    switch (BN) {
        case 64: return split_clusters_bs<64>(S);
        case 128: return split_clusters_bs<128>(S);
        case 192: return split_clusters_bs<192>(S);
        case 256: return split_clusters_bs<256>(S);
        default: return 0;
    }
}

// A stream-K workspace that needs no allocation: a file-scope device array, zero at module
// load (every call that completes leaves its counters at zero again), big enough for devices
// with up to kStaticWsSms SMs. Its address is looked up once per device, on the first call made
// with that device current, and kept for the life of the process.
constexpr int kStaticWsSms = 160;
constexpr size_t kStaticWsBytes = stream_k_workspace(kStaticWsSms);
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];
constexpr int kMaxDevices = 64;
static std::atomic<void*> g_static_ws_addr[kMaxDevices];

cudaError_t bs_static_workspace(int num_sms, void** ws, size_t* bytes) {
    if (num_sms > kStaticWsSms || stream_k_workspace(num_sms) > kStaticWsBytes)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_static_ws_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess) return e;
        g_static_ws_addr[dev].store(p, std::memory_order_release);
    }
    *ws = p;
    *bytes = kStaticWsBytes;
    return cudaSuccess;
}

// Zero the counters of the static workspace on the current device, if a call has used it: a
// call abandoned after a device wait error may have left a counter that no later call would
// bring back to zero. Enqueued on `stream`; nothing to do before the first use.
cudaError_t reset_static_workspace_counters(cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
    void* p = g_static_ws_addr[dev].load(std::memory_order_acquire);
    if (!p) return cudaSuccess;
    return cudaMemsetAsync(p, 0, stream_k_flag_bytes(kStaticWsSms), stream);
}

cudaError_t read_error_bs(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
