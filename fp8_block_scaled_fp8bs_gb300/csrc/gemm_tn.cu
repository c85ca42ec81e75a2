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
//
// Split K (StreamK::ksplit = S > 1, when the tiles alone would leave most SMs idle, e.g. one
// MoE expert's few hundred rows): S CTAs, one thread-block cluster per tile, each promote one
// K range of the tile into registers, then add the S partials slice by slice through
// distributed shared memory in rank order (gemm_common.cuh, split_reduce_store).
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

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
    static constexpr int NCH = CW / 32;                       // 32-column TMEM chunks per thread
    // Up to two chunks fit in registers next to the accumulator: they are loaded together
    // and the buffer is handed back after one TMEM round trip. With three or four the chunks
    // are loaded one after another, each while the previous one is folded in.
    static constexpr bool LOAD_ALL = NCH <= 2;
    // With BN = 192 a thread's 96 columns may span two 128-row blocks of B (at a chunk edge).
    static constexpr bool TWO_B = (BN % 128) != 0 && CW > 64;
    static constexpr bool SPLIT_REGS = (BN >= 192);
    static constexpr uint32_t kCtlRegs = 40;
    static constexpr uint32_t kEpiRegs = 232;
    static_assert(!SPLIT_REGS || 4 * 32 * kCtlRegs + 8 * 32 * kEpiRegs <= 384 * 168,
                  "register split exceeds the launch allocation");
};

template <int BN>
__global__ void __launch_bounds__(TnCfg<BN>::THREADS, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs g, const __grid_constant__ GroupTable gt, const int stages,
                   const StreamK sk) {
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

    Sched sched = sched_begin(sk, num_tiles, num_kb);
    int tile, kb0, kb1;
    bool exchanged = false;      // split K: this thread has been through the exchange

    if (warp >= Cfg::EPI_WARPS) {
        if constexpr (Cfg::SPLIT_REGS) regs_dec<Cfg::kCtlRegs>();
        if (warp == PRODUCER && lane == 0) {
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
        } else if (warp == ISSUER && lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            while (ok && sched_next(sched, num_kb, tile, kb0, kb1)) {
                for (int kb = kb0; kb < kb1; ++kb) {
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
        constexpr int EPI_THREADS = 32 * Cfg::EPI_WARPS;
        int buf = 0;
        uint32_t tphase = 0;
        // Pieces are recomputed from their index (piece_at), so that only the index and the K
        // end stay live through the K loop: these warps are at their register limit.
        bool ok = true;
        const bool split = sk.ksplit > 1;
        for (int p = 0; ok; ++p) {
            int tile, kb0, kb1;
            if (!piece_at(sk, p, num_tiles, num_kb, tile, kb0, kb1)) break;
            const TileCoord t = decode_tile<BN>(gt, tile, n_tiles);
            const int n0 = t.n0;
            const int row = t.m0 + row_in_tile;
            const int nb = min((n0 + col0) / 128, nb_count - 1);
            const int nb2 = min((n0 + col0 + Cfg::CW - 1) / 128, nb_count - 1);
            const float* as_row = g.a_s + static_cast<int64_t>(min(row, g.M - 1)) * num_kb;
            const float* bs_row =
                g.b_s + (static_cast<int64_t>(t.g) * nb_count + nb) * num_kb;
            const float* bs_row2 =
                g.b_s + (static_cast<int64_t>(t.g) * nb_count + nb2) * num_kb;
            // This thread's float4s of a partial tile in a stream-K slot: columns col0 .. col0+CW-1
            // of row row_in_tile, at [col / 4][row].
            const int part_base = (col0 / 4) * BM + row_in_tile;
            float acc[Cfg::CW];
#pragma unroll
            for (int i = 0; i < Cfg::CW; ++i) acc[i] = 0.0f;
            if (!split && kb0 == 0 && kb1 < num_kb) {
                // This CTA owns a shared tile: the pieces after its own are computed first by
                // the next CTAs (their ranges are at least a tile long, so they are done by
                // now); start from the sum of their partials.
                const int parts = sk_contributors(sk, tile, num_tiles, num_kb);
                volatile uint32_t* outcome = ring.tmem_holder + 1;
                if (threadIdx.x == 0) {
                    const bool got = flag_wait(sk.flags + blockIdx.x, parts);
                    if (got) {
                        sk.flags[blockIdx.x] = 0;        // ready for the next call
                    } else {
                        record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                    }
                    *outcome = got ? 1u : 0u;
                }
                epilogue_bar<EPI_THREADS>();
                if (*outcome == 0) {
                    ok = false;
                    break;
                }
                // The first partial goes straight into the (zero) accumulator; any further ones
                // (a tile shared by three or more CTAs) are added 8 float4 at a time.
                const float4* slot1 = sk.parts + static_cast<int64_t>(blockIdx.x + 1) * (BN / 4) * BM;
#pragma unroll
                for (int i = 0; i < Cfg::CW / 4; ++i) {
                    const float4 p = __ldcg(slot1 + part_base + i * BM);
                    acc[4 * i] = p.x;
                    acc[4 * i + 1] = p.y;
                    acc[4 * i + 2] = p.z;
                    acc[4 * i + 3] = p.w;
                }
#pragma unroll 1
                for (int j = 2; j <= parts; ++j) {
                    const float4* slot = sk.parts + static_cast<int64_t>(blockIdx.x + j) * (BN / 4) * BM;
#pragma unroll
                    for (int i0 = 0; i0 < Cfg::CW / 4; i0 += 8) {
                        float4 p[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) p[i] = __ldcg(slot + part_base + (i0 + i) * BM);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            acc[4 * (i0 + i)] += p[i].x;
                            acc[4 * (i0 + i) + 1] += p[i].y;
                            acc[4 * (i0 + i) + 2] += p[i].z;
                            acc[4 * (i0 + i) + 3] += p[i].w;
                        }
                        asm volatile("" ::: "memory");   // keep the next chunk's loads here
                    }
                }
            }
            // Scales of K blocks kb and kb+1 in registers, kb+2 requested as kb is consumed (the
            // scale arrays stay in L2; two blocks of MMA time hide the load).
            float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f, sbb0 = 0.f, sbb1 = 0.f;
            sa0 = __ldg(as_row + kb0);
            sb0 = __ldg(bs_row + kb0);
            if constexpr (Cfg::TWO_B) sbb0 = __ldg(bs_row2 + kb0);
            if (kb0 + 1 < kb1) {
                sa1 = __ldg(as_row + kb0 + 1);
                sb1 = __ldg(bs_row + kb0 + 1);
                if constexpr (Cfg::TWO_B) sbb1 = __ldg(bs_row2 + kb0 + 1);
            }
            for (int kb = kb0; kb < kb1; ++kb) {
                const float sc = sa0 * sb0;
                const float sc2 = Cfg::TWO_B ? sa0 * sbb0 : sc;
                sa0 = sa1;
                sb0 = sb1;
                sbb0 = sbb1;
                if (kb + 2 < kb1) {
                    sa1 = __ldg(as_row + kb + 2);
                    sb1 = __ldg(bs_row + kb + 2);
                    if constexpr (Cfg::TWO_B) sbb1 = __ldg(bs_row2 + kb + 2);
                }
                if (!warp_wait(&ring.tfull[buf], tphase)) {
                    if (lane == 0) record_error(FP8BS_DEVERR_EPILOGUE_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + col0);
                if constexpr (Cfg::LOAD_ALL) {
                    // All chunks in flight at once; the buffer goes back after one round trip.
                    float v[Cfg::CW];
#pragma unroll
                    for (int c = 0; c < Cfg::NCH; ++c) tmem_ld_32cols(taddr + 32 * c, v + 32 * c);
#pragma unroll
                    for (int c = 0; c < Cfg::NCH; ++c) tmem_wait_ld_32(v + 32 * c);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ring.tempty[buf]);
#pragma unroll
                    for (int c = 0; c < Cfg::NCH; ++c) {
                        // the chunk's 128-row block of B: the thread's first, or the next one
                        const float s_c =
                            Cfg::TWO_B && min((n0 + col0 + 32 * c) / 128, nb_count - 1) != nb
                                ? sc2
                                : sc;
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            fma2_into(acc + 32 * c + i, v[32 * c + i], v[32 * c + i + 1], s_c, s_c);
                    }
                } else {
                    // Three or four chunks through two 32-column register buffers: chunks 0 and
                    // 1 are loaded together; chunk 0 is folded in while chunk 2 loads into its
                    // registers, chunk 1 while chunk 3 loads; the buffer goes back once the last
                    // chunk has landed, after two round trips, and the rest is folded in after.
                    static_assert(Cfg::NCH == 3 || Cfg::NCH == 4, "two register buffers");
                    auto scale_of = [&](int c) {
                        return Cfg::TWO_B && min((n0 + col0 + 32 * c) / 128, nb_count - 1) != nb
                                   ? sc2
                                   : sc;
                    };
                    auto fold = [&](int c, const float* v) {
                        const float s_c = scale_of(c);
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            fma2_into(acc + 32 * c + i, v[i], v[i + 1], s_c, s_c);
                    };
                    float va[32], vb[32];
                    tmem_ld_32cols(taddr, va);
                    tmem_ld_32cols(taddr + 32, vb);
                    tmem_wait_ld_32(va);
                    tmem_wait_ld_32(vb);
                    fold(0, va);
                    tmem_ld_32cols(taddr + 64, va);
                    fold(1, vb);
                    if constexpr (Cfg::NCH == 4) tmem_ld_32cols(taddr + 96, vb);
                    tmem_wait_ld_32(va);
                    if constexpr (Cfg::NCH == 4) tmem_wait_ld_32(vb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ring.tempty[buf]);
                    fold(2, va);
                    if constexpr (Cfg::NCH == 4) fold(3, vb);
                }
                buf ^= 1;
                if (buf == 0) tphase ^= 1;
            }
            if (!ok) break;
            if (split) {
                // Split K: once every CTA of the cluster is past its K loop (its stage memory
                // free), send each slice of this partial to the CTA that adds it up; then add
                // up this CTA's slice and store it.
                const SplitTile sp = split_tile(BN, sk.ksplit, smem);
                cluster_sync();
#pragma unroll
                for (int i = 0; i < Cfg::CW / 4; ++i)
                    split_push4(sp, row_in_tile, col0 + 4 * i,
                                make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2],
                                            acc[4 * i + 3]));
                cluster_sync();
                split_reduce_store<EPI_THREADS>(sp, reinterpret_cast<const float4*>(smem),
                                                threadIdx.x, BN, t, g);
                exchanged = true;
                break;
            }
            if (kb0 > 0) {
                // A piece that does not start its tile: publish the partial in this CTA's slot
                // and count it in the flag of the tile's owner.
                float4* slot = sk.parts + static_cast<int64_t>(blockIdx.x) * (BN / 4) * BM;
#pragma unroll
                for (int i = 0; i < Cfg::CW / 4; ++i)
                    __stcg(slot + part_base + i * BM,
                           make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]));
                epilogue_bar<EPI_THREADS>();
                if (threadIdx.x == 0) {
                    __threadfence();
                    flag_add_release(sk.flags + sk_tile_owner(sk, tile, num_tiles, num_kb), 1);
                }
                continue;
            }
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

    // Split K: every thread takes part in the exchange's two cluster barriers (the promotion
    // warps above, unless a wait ran out before them).
    if (sk.ksplit > 1 && !exchanged) {
        cluster_sync();
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == ISSUER) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int BN>
constexpr int tn_stages() {
    return (kSmemLimit - 1024 - ring_bytes(kMaxStages)) / TnCfg<BN>::STAGE > kMaxStages
               ? kMaxStages
               : (kSmemLimit - 1024 - ring_bytes(kMaxStages)) / TnCfg<BN>::STAGE;
}

template <int BN>
constexpr int tn_smem() {
    return 1024 + tn_stages<BN>() * TnCfg<BN>::STAGE + ring_bytes(tn_stages<BN>());
}

template <int BN>
cudaError_t launch_tn(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                      const GroupTable& gt, int num_sms, const StreamKArgs& ska,
                      cudaStream_t stream) {
    using Cfg = TnCfg<BN>;
    constexpr int stages = tn_stages<BN>();
    constexpr int smem = tn_smem<BN>();
    if (ska.ksplit > 1 && split_recv_bytes(BN, ska.ksplit) > stages * Cfg::STAGE)
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem(gemm_tn_kernel<BN>, smem);
    if (e != cudaSuccess) return e;
    const int tiles = gt.tile_off[gt.num_groups];
    if (tiles == 0) return cudaSuccess;
    StreamK sk = {nullptr, nullptr, 0, 1};
    const int grid = stream_k_grid(ska, tiles, g.K / BK, num_sms, &sk);
    const bool stream_k = sk.parts != nullptr;
    e = launch_pdl_cluster(gemm_tn_kernel<BN>, grid, Cfg::THREADS, smem, stream, sk.ksplit,
                           stream_k, tmA, tmB, g, gt, stages, sk);
    if (e == cudaSuccess || !stream_k) return e;
    // The runtime could not place every CTA of the stream-K grid at once (fewer SMs available
    // to this context than the plan assumed): whole tiles instead, which need no co-residency.
    cudaGetLastError();
    const StreamK whole = {nullptr, nullptr, 0, 1};
    return launch_pdl_cluster(gemm_tn_kernel<BN>, tiles < num_sms ? tiles : num_sms,
                              Cfg::THREADS, smem, stream, 1, false, tmA, tmB, g, gt, stages,
                              whole);
}

template <int BN>
int split_clusters_tn(int S) {
    using Cfg = TnCfg<BN>;
    if (split_recv_bytes(BN, S) > tn_stages<BN>() * Cfg::STAGE) return 0;
    if (set_smem(gemm_tn_kernel<BN>, tn_smem<BN>()) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return max_active_clusters(reinterpret_cast<const void*>(gemm_tn_kernel<BN>), Cfg::THREADS,
                               tn_smem<BN>(), S);
}

}  // namespace

// Relative time of one K block of a 128 x BN tile, measured on GB300 at prefill shapes (745,
// 960 and 1050 clk for BN = 128, 192 and 256); BN = 64 from the N = 64 MMA rate.
int pick_tile_n(int64_t m_tiles_total, int64_t N, int num_sms) {
    static const int kWidth[4] = {256, 192, 128, 64};
    static const int kCost[4] = {141, 129, 100, 80};
    int best = 256;
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
                           const GroupTable& gt, int BN, int num_sms, const StreamKArgs& ska,
                           cudaStream_t stream) {
    switch (BN) {
        case 64: return launch_tn<64>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 128: return launch_tn<128>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 192: return launch_tn<192>(tmA, tmB, g, gt, num_sms, ska, stream);
        case 256: return launch_tn<256>(tmA, tmB, g, gt, num_sms, ska, stream);
        default: return cudaErrorInvalidValue;
    }
}

int max_split_clusters_tn(int BN, int S) {
    switch (BN) {
        case 64: return split_clusters_tn<64>(S);
        case 128: return split_clusters_tn<128>(S);
        case 192: return split_clusters_tn<192>(S);
        case 256: return split_clusters_tn<256>(S);
        default: return 0;
    }
}

cudaError_t read_error_tn(unsigned int* out, bool clear, cudaStream_t stream) {
    return read_tu_error(out, clear, stream);
}

}  // namespace fp8bs
