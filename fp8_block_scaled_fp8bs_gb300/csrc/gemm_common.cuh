// gemm_common.cuh -- pieces shared by the GEMM kernels (gemm_tn.cu, gemm_bs.cu, gemm_swapab.cu):
// tile constants, the shared-memory ring of TMA stages with its mbarriers, tile decoding for
// grouped launches, the bf16 row store and the device error word.
//
// Every GEMM kernel computes C[M,N] (bf16) = sum_kb a_s[m,kb] * b_s[n/128,kb] * P_kb[m,n],
// where P_kb is the product of the 128-wide K block kb of A (e4m3 [M,K]) and B (e4m3 [N,K]) --
// "DeepSeek-V3 Administrator & Developer Guide", §8.5.3 fp8_gemm_kernel -- with the same
// warp-specialised scheme (one CTA per SM):
//   TMA producer warp   streams 128-byte-wide K slices of A and B into a ring of shared-memory
//                       stages (128-byte swizzle), completion counted on mbarriers;
//   MMA issuer warp     per K block, 4 x tcgen05.mma (K = 32 each) into TMEM, then
//                       tcgen05.commit to free the stage;
//   epilogue warps      tcgen05.ld the fp32 accumulator from TMEM, round to bf16 and store.
// The kernels differ in where the block scales are applied (CUDA-core promotion of each K
// block's partial in gemm_tn.cu and gemm_swapab.cu; the tensor core itself, from ue8m0 scale
// factors in TMEM, in gemm_bs.cu) and in the orientation of the MMA.
//
// Every wait is bounded (ptx.cuh); a wait that runs out records a bit in the device error
// word, the CTA stops issuing, drains its in-flight TMA copies and MMAs, frees TMEM and exits.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "../../include/fp8bs.h"

namespace fp8bs {
namespace {

// Each translation unit that includes this header has its own error word (internal linkage);
// read_device_error in diag.cu combines the words of all of them.
__device__ unsigned int g_device_error = 0;

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
// tfull[b] and drain complete on one commit from each of `issuers` MMA-issuing threads. (Each
// barrier is initialised once: re-initialising a live mbarrier is undefined.)
__device__ __forceinline__ void init_ring(const Ring& r, int stages, uint32_t epi_warps,
                                          uint32_t full_count = 1, uint32_t issuers = 1) {
    for (int s = 0; s < stages; ++s) {
        mbar_init(&r.full[s], full_count);
        mbar_init(&r.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
        mbar_init(&r.tfull[b], issuers);
        mbar_init(&r.tempty[b], epi_warps);
    }
    mbar_init(r.drain, issuers);
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

// Read BN accumulator columns of this thread's TMEM lane as packed bf16 pairs (the rounding of
// store_row_bf16; column 2i in the low half of pk[i]), 16 columns per load (the packed row
// takes BN/2 registers); with `two`, the sum of two accumulators BN columns apart (two MMA
// issuers). Holding the row in registers lets the epilogue hand a single accumulator buffer
// back before its global stores, which are scattered over 32 rows per warp instruction and
// take several times as long as the loads.
template <int BN>
__device__ __forceinline__ void tmem_row_bf16(uint32_t taddr, uint32_t* pk, bool two) {
#pragma unroll
    for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld_16cols(taddr + 16 * c, v);
        tmem_wait_ld_16(v);
        if (two) {
            float u[16];
            tmem_ld_16cols(taddr + BN + 16 * c, u);
            tmem_wait_ld_16(u);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += u[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) pk[8 * c + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
}

// store_row_bf16's 16-byte stores (N % 8 == 0) for a row packed by tmem_row_bf16.
template <int CW>
__device__ __forceinline__ void store_row_packed(__nv_bfloat16* crow, const uint32_t* pk,
                                                 int valid) {
#pragma unroll
    for (int j = 0; j < CW / 8; ++j)
        if (8 * j < valid)
            *reinterpret_cast<uint4*>(crow + 8 * j) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

// Where a warp's 32 output rows go: rows row0 .. row0+31 of C (leading dimension N) from column
// n0, rows at or past row_end not stored.
struct WarpRows {
    __nv_bfloat16* c;
    int64_t N;
    int row0, row_end, n0;
};

// The 16-byte stores of a warp's 32 rows (lane l holds CW columns of row l as packed bf16 pairs)
// through a shared-memory scratch of the warp (32 x CH x 2 bytes), CH = 64 or 32 columns at a
// time: each lane writes its row's piece of the chunk (16-byte piece k of row r at position
// k ^ (r & 7), or k ^ ((r >> 1) & 3) for 64-byte rows, so that the eight lanes of a shared-memory
// phase hit distinct banks), then CH/8 lanes store each row's piece, 32/(CH/8) rows per
// instruction. Row-per-lane stores touch 32 rows per instruction: measured on GB300 they held
// the memory pipeline long enough to cost ~15 % of the ue8m0 prefill GEMM (385 against 329 us
// with the stores left out).
template <int CW, int CH = 64>
__device__ __forceinline__ void store_rows_coalesced(uint8_t* scratch, const uint32_t* pk,
                                                     const WarpRows& w, int lane) {
    static_assert(CH == 32 || CH == 64, "chunk width");
    static_assert(CW % CH == 0, "whole chunks");
    constexpr int KCH = CH / 8;           // 16-byte pieces per row of a chunk
    constexpr int RPI = 32 / KCH;         // rows per store instruction
    const auto pos = [](int r, int k) { return CH == 64 ? (k ^ (r & 7)) : (k ^ ((r >> 1) & 3)); };
    const int sub = lane % KCH;
#pragma unroll
    for (int q = 0; q < CW / CH; ++q) {
#pragma unroll
        for (int k = 0; k < KCH; ++k) {
            const uint32_t* src = pk + (CH / 2) * q + 4 * k;
            *reinterpret_cast<uint4*>(scratch + lane * (2 * CH) + pos(lane, k) * 16) =
                make_uint4(src[0], src[1], src[2], src[3]);
        }
        __syncwarp();
        const int col = w.n0 + CH * q + 8 * sub;
#pragma unroll
        for (int i = 0; i < KCH; ++i) {
            const int r = RPI * i + lane / KCH;
            const uint4 v =
                *reinterpret_cast<const uint4*>(scratch + r * (2 * CH) + pos(r, sub) * 16);
            if (w.row0 + r < w.row_end && col < w.N)
                *reinterpret_cast<uint4*>(w.c + static_cast<int64_t>(w.row0 + r) * w.N + col) = v;
        }
        __syncwarp();
    }
}

// The epilogue of a whole BN-column tile from one TMEM buffer (with `two`, the sum of the two
// issuers' accumulators): with 16-byte stores, the row into registers, `release` (the buffer
// back to the MMA issuer), then the stores (through the warp's scratch when it has one);
// otherwise (element stores, N % 8 != 0) 32 columns at a time with the next chunk's load in
// flight and `release` after the last load.
template <int BN, typename Release>
__device__ __forceinline__ void drain_row_bf16(uint32_t taddr, __nv_bfloat16* crow, bool store,
                                               int valid, bool vec, bool two, uint8_t* scratch,
                                               const WarpRows& w, int lane, Release release) {
    if (vec) {
        uint32_t pk[BN / 2];
        tmem_row_bf16<BN>(taddr, pk, two);
        release();
        if (scratch != nullptr)
            store_rows_coalesced<BN>(scratch, pk, w, lane);
        else if (store)
            store_row_packed<BN>(crow, pk, valid);
        return;
    }
    if (two) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
            float v[32], u[32];
            tmem_ld_32cols(taddr + 32 * c, v);
            tmem_ld_32cols(taddr + BN + 32 * c, u);
            tmem_wait_ld_32(v);
            tmem_wait_ld_32(u);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += u[i];
            if (c + 1 == BN / 32) release();
            if (store) store_row_bf16<32>(crow + 32 * c, v, valid - 32 * c, false);
        }
        return;
    }
    float va[32], vb[32];
    tmem_ld_32cols(taddr, va);
    tmem_wait_ld_32(va);
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
        float* cur = (c & 1) ? vb : va;
        float* nxt = (c & 1) ? va : vb;
        if (c + 1 < BN / 32) tmem_ld_32cols(taddr + 32 * (c + 1), nxt);
        if (c + 1 == BN / 32) release();
        if (store) store_row_bf16<32>(crow + 32 * c, cur, valid - 32 * c, false);
        if (c + 1 < BN / 32) tmem_wait_ld_32(nxt);
    }
}

constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxStages = 8;

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// ------------------------------------------------------------------ work schedule (stream-K)
//
// A CTA works through pieces (tile, first K block, end K block). Data-parallel tiles come
// first: CTA c takes tiles c, c + gridDim.x, ... below `dp_tiles`, each whole. The remaining
// tiles x K blocks "units" are cut into gridDim.x equal contiguous ranges, one per CTA, which
// each CTA works through tile by tile, so a tile's K loop may be shared by consecutive CTAs.
// Only a CTA's first shared piece can start inside a tile. That CTA writes its fp32 partial to
// its own workspace slot and counts it in the flag of the tile's owner, the CTA holding the
// tile's first K blocks (the last piece of its own range), which adds the partials in a fixed
// order -- results do not depend on timing -- resets its flag and stores the tile. The owner
// only waits on CTAs after it, each of which writes its partial before its other pieces, and
// every CTA of the grid is resident (one per SM), so the wait always ends.
struct StreamK {
    int* flags;       // [gridDim.x] partials published for the tile each CTA owns
    float4* parts;    // [gridDim.x][BN/4][128]: a CTA's partial, float4 of columns x rows
    int dp_tiles;     // tiles computed whole before the shared ones (a multiple of gridDim.x)
    int ksplit;       // > 1: split K inside a cluster (no workspace; see split_k_range)
};

struct Sched {
    int tile;           // next data-parallel tile
    int dp_tiles;
    int u, u_end;       // shared units (fewer than 2^31): cursor and end of this CTA's range
    int kb_lo, kb_hi;   // K blocks of a data-parallel tile (all of them unless split)
};

// ------------------------------------------------------------------ split K inside a cluster
//
// With StreamK::ksplit = S > 1 the grid holds S CTAs per output tile, launched as clusters of S
// consecutive CTAs: CTA r of cluster t computes K blocks [r*num_kb/S, (r+1)*num_kb/S) of tile
// t into fp32. The S partials are then added through distributed shared memory -- the columns
// of the tile are cut into S slices of W (a multiple of 8) and CTA q adds slice q of every
// partial in rank order, i.e. in K order -- and stored as bf16. No workspace, no flags, no
// waiting on other CTAs beyond two cluster barriers, and a fixed order of additions.
__device__ __forceinline__ void split_k_range(int num_kb, int S, int& tile, int& kb0, int& kb1) {
    tile = blockIdx.x / S;
    const int r = blockIdx.x - tile * S;
    kb0 = r * num_kb / S;
    kb1 = (r + 1) * num_kb / S;
}

__host__ __device__ constexpr int split_slice(int bn, int S) { return ((bn + S - 1) / S + 7) / 8 * 8; }

// Bytes of the receive area of a split tile: S slots of W columns x 128 rows of fp32.
__host__ __device__ constexpr int split_recv_bytes(int bn, int S) {
    return S * split_slice(bn, S) * BM * 4;
}

struct SplitTile {
    int S, rank, W;
    uint32_t recv;   // shared-window address of the receive area (the same in every CTA)
};

__device__ __forceinline__ SplitTile split_tile(int bn, int S, const void* recv) {
    SplitTile sp;
    sp.S = S;
    sp.rank = static_cast<int>(cluster_ctarank());
    sp.W = split_slice(bn, S);
    sp.recv = smem_addr(recv);
    return sp;
}

// Send columns col .. col+3 (col % 4 == 0) of row `row` of this CTA's partial to the CTA that
// adds up their slice: slot `rank` of its receive area, stored as float4 [W/4][128] per slot.
__device__ __forceinline__ void split_push4(const SplitTile& sp, int row, int col, float4 v) {
    const int q = col / sp.W;
    const uint32_t off =
        static_cast<uint32_t>(((sp.rank * sp.W + col - q * sp.W) / 4 * BM + row) * 16);
    st_shared_cluster_f4(mapa_shared(sp.recv + off, static_cast<uint32_t>(q)), v);
}

// This CTA's slice of the tile: the S partials added in rank order, rounded to bf16 and stored
// (rows past row_end and columns past N are skipped). `tid` counts the calling threads.
template <int THREADS>
__device__ __forceinline__ void split_reduce_store(const SplitTile& sp, const float4* recv,
                                                   int tid, int bn, const TileCoord& t,
                                                   const GemmArgs& g) {
    const int c_lo = sp.rank * sp.W;
    const int c_hi = min(bn, c_lo + sp.W);
    const int items = c_hi > c_lo ? (c_hi - c_lo) / 8 * BM : 0;
    const bool vec = (g.N & 7) == 0;
    for (int i = tid; i < items; i += THREADS) {
        const int row = i % BM;
        const int grp = i / BM;
        float v[8];
        for (int r = 0; r < sp.S; ++r) {
            const float4* slot = recv + (r * sp.W / 4 + 2 * grp) * BM + row;
            const float4 p0 = slot[0];
            const float4 p1 = slot[BM];
            if (r == 0) {
                v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
                v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
            } else {
                v[0] += p0.x; v[1] += p0.y; v[2] += p0.z; v[3] += p0.w;
                v[4] += p1.x; v[5] += p1.y; v[6] += p1.z; v[7] += p1.w;
            }
        }
        const int grow = t.m0 + row;
        const int col = t.n0 + c_lo + 8 * grp;
        if (grow < t.row_end && col < g.N) {
            __nv_bfloat16* crow =
                static_cast<__nv_bfloat16*>(g.c) + static_cast<int64_t>(grow) * g.N + col;
            store_row_bf16<8>(crow, v, g.N - col, vec);
        }
    }
}

// Start of CTA `cta`'s range of the `units` shared units.
__device__ __forceinline__ int64_t sk_range_start(int cta, int64_t units) {
    return static_cast<int64_t>(cta) * units / gridDim.x;
}

// The CTA whose range holds shared unit x: the largest c with floor(c * units / grid) <= x.
__device__ __forceinline__ int sk_owner(int64_t x, int64_t units) {
    return static_cast<int>(((x + 1) * gridDim.x - 1) / units);
}

__device__ __forceinline__ int64_t sk_units(const StreamK& sk, int num_tiles, int num_kb) {
    return sk.parts ? static_cast<int64_t>(num_tiles - sk.dp_tiles) * num_kb : 0;
}

__device__ __forceinline__ Sched sched_begin(const StreamK& sk, int num_tiles, int num_kb) {
    Sched s;
    s.tile = blockIdx.x;
    s.dp_tiles = sk.parts ? sk.dp_tiles : num_tiles;
    const int64_t units = sk_units(sk, num_tiles, num_kb);
    s.u = sk.parts ? static_cast<int>(sk_range_start(blockIdx.x, units)) : 0;
    s.u_end = sk.parts ? static_cast<int>(sk_range_start(blockIdx.x + 1, units)) : 0;
    s.kb_lo = 0;
    s.kb_hi = num_kb;
    if (sk.ksplit > 1) {            // one piece: this CTA's K range of its cluster's tile
        split_k_range(num_kb, sk.ksplit, s.tile, s.kb_lo, s.kb_hi);
        s.dp_tiles = s.tile + 1;
    }
    return s;
}

__device__ __forceinline__ bool sched_next(Sched& s, int num_kb, int& tile, int& kb0, int& kb1) {
    if (s.tile < s.dp_tiles) {
        tile = s.tile;
        kb0 = s.kb_lo;
        kb1 = s.kb_hi;
        s.tile += gridDim.x;
        return true;
    }
    if (s.u >= s.u_end) return false;
    const int rel = s.u / num_kb;
    tile = s.dp_tiles + rel;
    kb0 = s.u - rel * num_kb;
    const int left = s.u_end - s.u;
    kb1 = left < num_kb - kb0 ? kb0 + left : num_kb;
    s.u += kb1 - kb0;
    return true;
}

// Piece p of this CTA's sequence (the same sequence as sched_next), computed from p alone.
__device__ __forceinline__ bool piece_at(const StreamK& sk, int p, int num_tiles, int num_kb,
                                         int& tile, int& kb0, int& kb1) {
    if (sk.ksplit > 1) {
        if (p > 0) return false;
        split_k_range(num_kb, sk.ksplit, tile, kb0, kb1);
        return true;
    }
    const int dp_tiles = sk.parts ? sk.dp_tiles : num_tiles;
    const int n_dp = blockIdx.x < dp_tiles ? (dp_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (p < n_dp) {
        tile = blockIdx.x + p * gridDim.x;
        kb0 = 0;
        kb1 = num_kb;
        return true;
    }
    if (!sk.parts) return false;
    const int64_t units = sk_units(sk, num_tiles, num_kb);
    const int u0 = static_cast<int>(sk_range_start(blockIdx.x, units));
    const int u_end = static_cast<int>(sk_range_start(blockIdx.x + 1, units));
    const int q = p - n_dp;
    const int rel = u0 / num_kb + q;
    const int start = q == 0 ? u0 : rel * num_kb;
    if (start >= u_end) return false;
    tile = dp_tiles + rel;
    kb0 = start - rel * num_kb;
    kb1 = min(num_kb, u_end - rel * num_kb);
    return true;
}

// Number of CTAs after this one whose ranges start inside shared tile `tile` (this CTA owns
// it: its range holds the tile's first K block).
__device__ __forceinline__ int sk_contributors(const StreamK& sk, int tile, int num_tiles,
                                               int num_kb) {
    const int64_t units = sk_units(sk, num_tiles, num_kb);
    const int64_t tile_end = static_cast<int64_t>(tile - sk.dp_tiles + 1) * num_kb;
    int n = 0;
    for (int j = blockIdx.x + 1; j < static_cast<int>(gridDim.x) &&
                                 sk_range_start(j, units) < tile_end; ++j)
        ++n;
    return n;
}

// The owner of shared tile `tile`.
__device__ __forceinline__ int sk_tile_owner(const StreamK& sk, int tile, int num_tiles,
                                             int num_kb) {
    return sk_owner(static_cast<int64_t>(tile - sk.dp_tiles) * num_kb,
                    sk_units(sk, num_tiles, num_kb));
}

__device__ __forceinline__ void flag_add_release(int* flag, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(flag), "r"(v) : "memory");
}

__device__ __forceinline__ int flag_load_acquire(const int* flag) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return v;
}

// Wait (bounded) until *flag == target.
__device__ __forceinline__ bool flag_wait(const int* flag, int target) {
    if (flag_load_acquire(flag) == target) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (flag_load_acquire(flag) == target) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Named barrier 1 among `threads` threads (the epilogue warps of a kernel).
template <int threads>
__device__ __forceinline__ void epilogue_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(threads) : "memory");
}

// Host: grid size and kernel parameter for a stream-K or split-K plan (see StreamKArgs in
// kernels.h).
inline int stream_k_grid(const StreamKArgs& ska, int tiles, int num_kb, int num_sms,
                         StreamK* sk) {
    sk->ksplit = 1;
    if (ska.ksplit > 1) {
        sk->ksplit = ska.ksplit;
        return tiles * ska.ksplit;
    }
    if (!ska.workspace) return tiles < num_sms ? tiles : num_sms;
    const int64_t units = static_cast<int64_t>(tiles - ska.dp_tiles) * num_kb;
    const int grid = ska.dp_tiles > 0 || units >= num_sms ? num_sms : static_cast<int>(units);
    sk->flags = static_cast<int*>(ska.workspace);
    sk->parts = reinterpret_cast<float4*>(static_cast<char*>(ska.workspace) +
                                          stream_k_flag_bytes(num_sms));
    sk->dp_tiles = ska.dp_tiles;
    return grid;
}

// Read (and, if `clear`, reset) this translation unit's error word; enqueued on `stream`.
inline cudaError_t read_tu_error(unsigned int* out, bool clear, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_error, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess || !clear) return e;
    static const unsigned int zero = 0;
    return cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned int), 0,
                                   cudaMemcpyHostToDevice, stream);
}

}  // namespace
}  // namespace fp8bs
