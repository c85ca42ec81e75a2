// gemm.cu -- block-scaled FP8 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes C[M,N] (bf16) = sum_kb a_s[m,kb] * b_s[n/128,kb] * P_kb[m,n], where P_kb is the
// fp32 product of the 128-wide K block kb of A (e4m3 [M,K]) and B (e4m3 [N,K]) --
// "DeepSeek-V3 Administrator & Developer Guide", §8.5.3 fp8_gemm_kernel.
//
// Structure (one CTA per SM, warp-specialised):
//   TMA producer warp   streams 128-byte-wide K slices of A and B into a ring of shared-memory
//                       stages (128-byte swizzle), completion counted on mbarriers.
//   MMA issuer warp     for each K block, 4 x tcgen05.mma (K = 32 each) into one of two TMEM
//                       buffers, then tcgen05.commit to free the stage and publish the buffer.
//   promotion warps     tcgen05.ld the block's fp32 partial from TMEM in 32-column chunks (the
//                       next chunk's load in flight while the current one is folded in),
//                       release the buffer, and fold it into fp32 registers with the block's
//                       scale a_s[m,kb] * b_s[n/128,kb]. After the last block: bf16 and store.
// The two TMEM buffers let the tensor cores compute block kb+1 while block kb is promoted.
//
// Two orientations share this scheme:
//   gemm_tn_kernel      128 rows of A x BN columns of B per tile, persistent over tiles.
//   gemm_swapab_kernel  for few rows of A (decode): 128 rows of B take the MMA's M side and
//                       the MT rows of A its N side, so the weight stream fills the tensor
//                       core's 128 lanes and every SM streams its own 128-row weight slab.
//
// Every wait is bounded (ptx.cuh); a wait that runs out records a bit in the device error
// word, the CTA stops issuing, drains its in-flight TMA copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "../../include/fp8bs.h"

namespace fp8bs {

__device__ unsigned int g_device_error = 0;

namespace {

constexpr int BM = 128;       // tile rows on the MMA's M side = TMEM lanes
constexpr int BK = 128;       // K block: one scale block, one 128-byte swizzle row of e4m3
constexpr int MMA_K = 32;     // K per tcgen05.mma for 8-bit operands
constexpr int A_TILE = BM * BK;  // bytes of one 128 x 128 e4m3 tile

__device__ __forceinline__ void record_error(unsigned bit) { atomicOr(&g_device_error, bit); }

__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t used) {
    uint32_t c = 32;
    while (c < used) c <<= 1;
    return c;
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait: every lane waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// acc[0..1] += (v0, v1) * (s0, s1) as one packed fp32x2 FMA (round-to-nearest per component).
__device__ __forceinline__ void fma2_into(float* acc, float v0, float v1, float s0, float s1) {
    const float2 r = __ffma2_rn(make_float2(v0, v1), make_float2(s0, s1), make_float2(acc[0], acc[1]));
    acc[0] = r.x;
    acc[1] = r.y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Shared-memory bookkeeping common to both kernels.
struct Ring {
    uint64_t* full;    // [stages] TMA bytes landed
    uint64_t* empty;   // [stages] MMAs reading the stage are done
    uint64_t* tfull;   // [2] TMEM buffer holds a finished partial
    uint64_t* tempty;  // [2] TMEM buffer has been read out
    uint64_t* drain;   // [1] all MMAs issued by the CTA are done
    uint32_t* tmem_holder;
};

__device__ __forceinline__ Ring carve_ring(uint8_t* p, int stages) {
    Ring r;
    r.full = reinterpret_cast<uint64_t*>(p);
    r.empty = r.full + stages;
    r.tfull = r.empty + stages;
    r.tempty = r.tfull + 2;
    r.drain = r.tempty + 2;
    r.tmem_holder = reinterpret_cast<uint32_t*>(r.drain + 1);
    return r;
}

constexpr int ring_bytes(int stages) { return (2 * stages + 5) * 8 + 16; }

// full[s] completes on `full_count` arrivals plus the stage's TMA bytes (the producer's
// arrive.expect_tx is one arrival; the block-scaled kernel adds its scale-factor warps).
__device__ __forceinline__ void init_ring(const Ring& r, int stages, uint32_t epi_warps,
                                          uint32_t full_count = 1) {
    for (int s = 0; s < stages; ++s) {
        mbar_init(&r.full[s], full_count);
        mbar_init(&r.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
        mbar_init(&r.tfull[b], 1);
        mbar_init(&r.tempty[b], epi_warps);
    }
    mbar_init(r.drain, 1);
    fence_barrier_init();
}

// After an abort, wait (briefly) for the TMA copies this producer issued but that no consumer
// saw land, so that no copy is still writing shared memory when the CTA exits.
__device__ __forceinline__ void drain_tma(const Ring& r, int stages, int64_t issued) {
    const int64_t first = issued > stages ? issued - stages : 0;
    for (int64_t i = first; i < issued; ++i) {
        const int s = static_cast<int>(i % stages);
        const uint32_t ph = static_cast<uint32_t>((i / stages) & 1);
        if (!mbar_wait(&r.full[s], ph, kDrainLimitNs)) record_error(FP8BS_DEVERR_DRAIN_WAIT);
    }
}

// ================================================================ normal orientation

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

template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Coordinates of one output tile: group, first row (global), first column, end of the group's
// rows. Tiles are numbered group by group, m tiles fastest within a group.
struct TileCoord {
    int g, m0, n0, row_end;
};

template <int BN>
__device__ __forceinline__ TileCoord decode_tile(const GroupTable& gt, int tile, int n_tiles) {
    int grp = 0;
    while (tile >= gt.tile_off[grp + 1]) ++grp;   // groups without tiles are skipped
    const int local = tile - gt.tile_off[grp];
    const int m_tiles = (gt.tile_off[grp + 1] - gt.tile_off[grp]) / n_tiles;
    TileCoord t;
    t.g = grp;
    t.m0 = gt.row_off[grp] + (local % m_tiles) * BM;
    t.n0 = (local / m_tiles) * BN;
    t.row_end = gt.row_off[grp + 1];
    return t;
}

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

// ================================================================ block-scaled orientation
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
// Round `CW` fp32 values to bf16 and store the first `valid` of them at `crow` (one row of C):
// 16-byte stores when the row pitch keeps them aligned (N % 8 == 0), else element stores.
template <int CW>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* crow, const float* acc, int valid,
                                               bool vec) {
    if (vec) {
#pragma unroll
        for (int j = 0; j < CW / 8; ++j) {
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
        for (int j = 0; j < CW; ++j)
            if (j < valid) crow[j] = __float2bfloat16_rn(acc[j]);
    }
}


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

// ================================================================ swapped orientation

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

// ================================================================ diagnostics

__global__ void probe_wait_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        // Nothing ever arrives on `bar`: the wait must run out and report.
        if (!mbar_wait(&bar, 0, timeout_ns)) record_error(FP8BS_DEVERR_PROBE);
    }
}

constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxStages = 8;

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

cudaError_t launch_probe_wait(uint64_t timeout_ns, cudaStream_t stream) {
    probe_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError();
}

cudaError_t read_device_error(unsigned int* out, bool clear, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    if (clear) {
        static const unsigned int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaStreamSynchronize(stream);
}

}  // namespace fp8bs
