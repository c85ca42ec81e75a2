// api.cu -- the C ABI (include/fp8bs.h): argument checks, device checks, TMA tensor-map
// encoding and the choice of GEMM kernel. Nothing here allocates memory or synchronises.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fp8bs.h"
#include "kernels.h"

namespace fp8bs {

int max_active_clusters(const void* kernel, int threads, int smem, int cluster_x) {
    struct Entry {
        const void* kernel;
        int threads, smem, cluster_x, dev, n;
    };
    static std::mutex mu;
    static Entry cache[128];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& c = cache[i];
            if (c.kernel == kernel && c.threads == threads && c.smem == smem &&
                c.cluster_x == cluster_x && c.dev == dev)
                return c.n;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster_x));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (used < 128) cache[used++] = Entry{kernel, threads, smem, cluster_x, dev, n};
    return n;
}

}  // namespace fp8bs

namespace {

using fp8bs::GemmArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// The kernels are built for sm_103a only; arch-specific code runs on compute capability 10.3.
int check_device(int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return FP8BS_ERR_UNSUPPORTED_DEVICE;
    return FP8BS_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up through the runtime so that the library does not
// link libcuda directly (it then loads on machines without a driver).
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            p = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 2-D map over a row-major e4m3 matrix [rows, K] with boxes of {128 bytes, box_rows} and
// 128-byte swizzling (the tcgen05 K-major SW128 layout). Rows past the end read as zero.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Over a row-major bf16 matrix [rows, K], box {64 elements (128 bytes), box_rows}, 128-byte
// swizzle: the K-major layout of a bf16 MMA operand, one 64-wide half of a K block per box.
bool make_map_bf16_sw128(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                         int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA; }

// Stream-K plans (see StreamKArgs in kernels.h). Whole tiles for all but the last one to two
// waves, the rest shared; used when the busiest SM's K blocks (plus the hand-over of a partial)
// drop clearly below the data-parallel schedule's ceil(tiles / SMs) whole tiles.
fp8bs::StreamKArgs no_stream_k() { return fp8bs::StreamKArgs{nullptr, 0, 1}; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The kernels count shared units (tiles x K blocks) in 32 bits.
bool units_fit(int64_t tiles, int64_t num_kb) { return tiles * num_kb < INT32_MAX; }

int dp_tiles_before_sharing(int64_t tiles, int sms) {
    return tiles < 2 * sms ? 0 : static_cast<int>((tiles / sms - 1) * sms);
}

// fp32 scales (promotion kernel): the owner adds the other pieces' partials before its own
// piece, which needs every CTA's range to span at least one tile (>= SMs tiles shared).
fp8bs::StreamKArgs plan_stream_k_tn(int64_t tiles, int64_t num_kb, int sms, void* workspace) {
    if (!workspace || tiles < sms || num_kb < 2 || !units_fit(tiles, num_kb)) return no_stream_k();
    const int dp = dp_tiles_before_sharing(tiles, sms);
    const int64_t cost_dp = ceil_div(tiles, sms) * num_kb;
    const int64_t cost_sk = dp / sms * num_kb + ceil_div((tiles - dp) * num_kb, sms) + 2;
    if (cost_sk * 100 >= cost_dp * 97) return no_stream_k();
    return fp8bs::StreamKArgs{workspace, dp, 1};
}

// Relative time of one K block of a 128 x bn tile in the split schedule below (the tile-width
// models of the two kernels; the block-scaled kernel's 64-wide tiles have two MMA issuers:
// 18.3 us for the MLA kv projection as 144 such tiles against 24.1 us as 80 tiles 128 wide,
// both one round). The block-scaled 192-wide tile keeps 117 here although its two issuers make
// whole tiles cheaper (104 in pick_tile_n_bs): split two ways, the MLA kv projection measured
// 18.75 us against 17.6 us as whole 64-wide tiles, which 104 would not predict.
int64_t width_cost(bool block_scaled, int bn) {
    switch (bn) {
        case 256: return block_scaled ? 134 : 141;
        case 192: return block_scaled ? 117 : 129;
        case 128: return 100;
        default: return block_scaled ? 76 : 80;
    }
}

// Split K inside a cluster (StreamKArgs::ksplit) when the tiles are few: the tile width and
// split with the lowest modelled time -- a CTA's share of the K blocks plus five K blocks for
// the exchange of partials, at the width's K-block cost --
// provided every cluster of the grid can be resident at once. Taken only if it beats
// `cost_plain` (the whole-tile schedule) by 10 %; otherwise ksplit = 1. Measured on GB300: one
// MoE expert's 300 rows (N=2048, K=7168, fp32 scales) take 29.8 us as 24 whole 256-wide tiles
// and 16.7-17.4 us split four ways; the MLA kv projection (M=2048, N=576) is fastest as 144
// whole 64-wide tiles (18.3 us against 19.7 us as 48 192-wide tiles split two ways).
struct SplitPlan {
    int bn;
    int ksplit;
};

SplitPlan plan_split(bool block_scaled, int64_t m_tiles, int64_t N, int64_t num_kb, int sms,
                     int64_t cost_plain) {
    static const int kWidths[4] = {64, 128, 192, 256};    // on a tie the narrower
    SplitPlan best = {0, 1};
    int64_t best_cost = cost_plain * 9 / 10;
    for (int bn : kWidths) {
        const int64_t tiles = m_tiles * ceil_div(N, bn);
        for (int S = fp8bs::kMaxSplit; S > 1; --S) {
            if (tiles * S > sms || num_kb / S < 2) continue;
            const int64_t cost = (ceil_div(num_kb, S) + 5) * width_cost(block_scaled, bn);
            if (cost >= best_cost) continue;
            const int fit = block_scaled ? fp8bs::max_split_clusters_bs(bn, S)
                                         : fp8bs::max_split_clusters_tn(bn, S);
            if (fit < tiles) continue;
            best = SplitPlan{bn, S};
            best_cost = cost;
        }
    }
    return best;
}

// ue8m0 scales (block-scaled kernel, 128-column tiles when shared). Measured: with ranges
// shorter than a tile (fewer tiles than SMs) the hand-over of partials at the end costs more
// than the balance gains (MLA N = 576: 24.0 us shared against 22.4 us whole), so tiles are only
// shared when there are at least as many as SMs.
fp8bs::StreamKArgs plan_stream_k_bs(int64_t m_tiles, int64_t N, int64_t num_kb, int sms,
                                    void* workspace) {
    if (!workspace || num_kb < 2) return no_stream_k();
    const int bn_dp = fp8bs::pick_tile_n_bs(m_tiles, N, sms);
    // whole tiles at bn_dp against shared 128-wide tiles, in 128-wide K-block times
    const int64_t cost_dp =
        ceil_div(m_tiles * ceil_div(N, bn_dp), sms) * num_kb * width_cost(true, bn_dp) / 100;
    const int64_t tiles = m_tiles * ceil_div(N, 128);
    if (tiles < sms || !units_fit(tiles, num_kb)) return no_stream_k();
    const int dp = dp_tiles_before_sharing(tiles, sms);
    const int64_t cost_sk = dp / sms * num_kb + ceil_div((tiles - dp) * num_kb, sms) + 4;
    if (cost_sk * 10 >= cost_dp * 9) return no_stream_k();
    return fp8bs::StreamKArgs{workspace, dp, 1};
}

// The kernel and launch configuration for a GEMM of this shape (fp8bs_gemm_plan reports it).
struct GemmPlan {
    int kind;                  // FP8BS_KERNEL_*
    int tile;                  // MT (swapped) or BN (normal orientation)
    fp8bs::StreamKArgs ska;    // stream-K workspace or split K (normal orientation)
    int ksplit;                // CTAs per tile sharing its K loop in a cluster (1: none)
    int pairs;                 // CTA pairs launched (FP8BS_KERNEL_BLOCK_SCALED_PAIR)
};

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, bool block_scaled, void* workspace,
                   int sms) {
    GemmPlan p;
    p.ska = no_stream_k();
    p.ksplit = 1;
    p.pairs = 0;
    if (M <= 128) {
        // Few rows of A (decode): weights on the MMA's M side, one 128-row slab per CTA (or
        // per cluster, with the K loop split).
        const int MT = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
        const int S = fp8bs::plan_gemm_swapab(MT, false, static_cast<int>((M + MT - 1) / MT),
                                              static_cast<int>(N), static_cast<int>(K), sms);
        if (S > 0) {
            p.kind = FP8BS_KERNEL_SWAPPED;
            p.tile = MT;
            p.ksplit = S;
            return p;
        }
        // K too long to stage the activation scales: the normal kernel below.
    }
    const int64_t m_tiles = (M + 127) / 128;
    int BN;
    if (block_scaled) {
        p.ska = plan_stream_k_bs(m_tiles, N, K / 128, sms, workspace);
        BN = p.ska.workspace ? 128 : fp8bs::pick_tile_n_bs(m_tiles, N, sms);
        // The CTA-pair kernel is not chosen here: measured on GB300 it runs 9-12 % slower than
        // the one-CTA kernel (prefill up 412 against 378 us, the MLA q projection 30.5 against
        // 27.2 us); fp8bs_gemm_config can select it.
    } else {
        BN = fp8bs::pick_tile_n(m_tiles, N, sms);
        p.ska = plan_stream_k_tn(m_tiles * ceil_div(N, BN), K / 128, sms, workspace);
    }
    if (!p.ska.workspace) {
        // Few tiles: split their K loops between the CTAs of a cluster, if that pays.
        const int64_t cost_plain =
            ceil_div(m_tiles * ceil_div(N, BN), sms) * (K / 128) * width_cost(block_scaled, BN);
        const SplitPlan sp = plan_split(block_scaled, m_tiles, N, K / 128, sms, cost_plain);
        if (sp.ksplit > 1) {
            BN = sp.bn;
            p.ska = fp8bs::StreamKArgs{nullptr, 0, sp.ksplit};
            p.ksplit = sp.ksplit;
        }
    }
    p.kind = block_scaled ? FP8BS_KERNEL_BLOCK_SCALED : FP8BS_KERNEL_PROMOTED;
    p.tile = BN;
    return p;
}

// A caller-given configuration (fp8bs_gemm_config): kernel, tile and K split, checked against
// what the kernels support for this shape. false: not supported.
bool config_plan(const int cfg[3], int64_t M, int64_t N, int64_t K, bool block_scaled,
                 void* workspace, int sms, GemmPlan* p) {
    const int kind = cfg[0], tile = cfg[1], ks = cfg[2];
    const int64_t num_kb = K / 128;
    p->kind = kind;
    p->tile = tile;
    p->ska = no_stream_k();
    p->ksplit = 1;
    p->pairs = 0;
    if (ks < 0 || ks > fp8bs::kMaxSplit || ks > num_kb) return false;
    switch (kind) {
        case FP8BS_KERNEL_SWAPPED:
            if ((tile != 16 && tile != 32 && tile != 64 && tile != 128) || M > tile || ks == 0)
                return false;
            p->ksplit = ks;
            return fp8bs::check_gemm_swapab(tile, static_cast<int>(K), ks);
        case FP8BS_KERNEL_PROMOTED:
        case FP8BS_KERNEL_BLOCK_SCALED: {
            const bool bs = kind == FP8BS_KERNEL_BLOCK_SCALED;
            if (bs && !block_scaled) return false;
            if (tile != 64 && tile != 128 && tile != 192 && tile != 256) return false;
            const int64_t tiles = ceil_div(M, 128) * ceil_div(N, tile);
            if (ks == 0) {      // stream-K over the workspace
                if (!workspace || (bs && tile != 128) || tiles < sms || num_kb < 2 ||
                    !units_fit(tiles, num_kb))
                    return false;
                p->ska = fp8bs::StreamKArgs{workspace, dp_tiles_before_sharing(tiles, sms), 1};
                return true;
            }
            if (ks > 1) {
                const int fit = bs ? fp8bs::max_split_clusters_bs(tile, ks)
                                   : fp8bs::max_split_clusters_tn(tile, ks);
                if (fit < 1 || tiles * ks > INT32_MAX) return false;
                p->ska = fp8bs::StreamKArgs{nullptr, 0, ks};
                p->ksplit = ks;
            }
            return true;
        }
        case FP8BS_KERNEL_BLOCK_SCALED_PAIR: {
            if (!block_scaled || ks != 1) return false;
            if (tile != 128 && tile != 192 && tile != 256) return false;
            const int64_t tiles = ceil_div(M, 256) * ceil_div(N, tile);
            const int64_t cap = std::min<int64_t>(sms / 2, fp8bs::max_pair_clusters_bs(tile));
            if (cap < 1) return false;
            p->pairs = static_cast<int>(std::min<int64_t>(tiles, cap));
            return true;
        }
        default:
            return false;
    }
}

// fp8bs_gemm_ex, fp8bs_gemm_ws and fp8bs_gemm_config: checks, then the kernel for the shape
// (or the caller's configuration `cfg`, if given; see fp8bs.h).
int gemm_impl(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
              int64_t M, int64_t N, int64_t K, int scale_fmt, unsigned int flags,
              void* workspace, size_t workspace_bytes, void* stream, const int* cfg = nullptr) {
    if ((flags & ~FP8BS_GEMM_WEIGHTS_CONSTANT) != 0) return FP8BS_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || K % FP8BS_BLOCK != 0) return FP8BS_ERR_INVALID_ARG;
    if (scale_fmt != FP8BS_SCALE_FP32 && scale_fmt != FP8BS_SCALE_UE8M0)
        return FP8BS_ERR_INVALID_ARG;
    // The kernels index with 32-bit row/column coordinates (TMA coordinates are 32-bit).
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BS_OK;
    if (!c) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(c)) return FP8BS_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        int sms = 0;
        if (int e = check_device(&sms)) return e;
        return status_of(cudaMemsetAsync(c, 0, static_cast<size_t>(M * N) * 2, st));
    }
    if (!a || !a_s || !b || !b_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned4(a_s) || !aligned4(b_s))
        return FP8BS_ERR_MISALIGNED;
    int sms = 0;
    if (int e = check_device(&sms)) return e;
    if (workspace) {
        if (!aligned16(workspace)) return FP8BS_ERR_MISALIGNED;
        if (workspace_bytes < fp8bs::stream_k_workspace(sms)) return FP8BS_ERR_INVALID_ARG;
    }

    GemmArgs g;
    g.a_s = a_s;
    g.b_s = b_s;
    g.c = c;
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.weights_constant = (flags & FP8BS_GEMM_WEIGHTS_CONSTANT) ? 1 : 0;

    const bool block_scaled = scale_fmt == FP8BS_SCALE_UE8M0;
    GemmPlan p;
    if (cfg) {
        if (!config_plan(cfg, M, N, K, block_scaled, workspace, sms, &p))
            return FP8BS_ERR_INVALID_ARG;
    } else {
        p = plan_gemm(M, N, K, block_scaled, workspace, sms);
    }
    CUtensorMap tmA, tmB;
    if (p.kind == FP8BS_KERNEL_SWAPPED) {
        if (!make_map(&tmB, b, N, K, 128) || !make_map(&tmA, a, M, K, p.tile))
            return FP8BS_ERR_CUDA;
        const int64_t rows[2] = {0, M};
        fp8bs::GroupTable gt;
        fp8bs::fill_row_tiles(&gt, rows, 1, p.tile);
        return status_of(fp8bs::launch_gemm_swapab(tmB, tmA, g, gt, p.tile, fp8bs::FusedQuant{},
                                                   p.ksplit, false, st));
    }
    if (p.kind == FP8BS_KERNEL_BLOCK_SCALED_PAIR) {
        if (!make_map(&tmA, a, M, K, 128) || !make_map(&tmB, b, N, K, p.tile / 2))
            return FP8BS_ERR_CUDA;
        return status_of(fp8bs::launch_gemm_bs_pair(tmA, tmB, g, p.tile, p.pairs, st));
    }
    if (!make_map(&tmA, a, M, K, 128) || !make_map(&tmB, b, N, K, p.tile)) return FP8BS_ERR_CUDA;
    const int64_t rows[2] = {0, M};
    fp8bs::GroupTable gt;
    fp8bs::fill_group_table(&gt, rows, 1, static_cast<int>(N), p.tile);
    if (p.kind == FP8BS_KERNEL_BLOCK_SCALED)
        return status_of(fp8bs::launch_gemm_bs(tmA, tmB, g, gt, p.tile, sms, p.ska, st));
    return status_of(fp8bs::launch_gemm_tn(tmA, tmB, g, gt, p.tile, sms, p.ska, st));
}

}  // namespace

extern "C" {

const char* fp8bs_status_string(int status) {
    switch (status) {
        case FP8BS_OK: return "ok";
        case FP8BS_ERR_INVALID_ARG: return "invalid argument";
        case FP8BS_ERR_MISALIGNED: return "pointer not aligned";
        case FP8BS_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        case FP8BS_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int fp8bs_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K, int scale_fmt,
                    void* stream) {
    if (M < 0 || K < 0 || K % FP8BS_BLOCK != 0) return FP8BS_ERR_INVALID_ARG;
    if (scale_fmt != FP8BS_SCALE_FP32 && scale_fmt != FP8BS_SCALE_UE8M0)
        return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || K == 0) return FP8BS_OK;
    if (!x || !y || !s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned4(s)) return FP8BS_ERR_MISALIGNED;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return status_of(fp8bs::launch_act_quant(x, y, s, M, K, scale_fmt == FP8BS_SCALE_UE8M0, sms,
                                             static_cast<cudaStream_t>(stream)));
}

int fp8bs_weight_dequant(const void* w, const float* s, void* y, int64_t N, int64_t K,
                         void* stream) {
    if (N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return FP8BS_OK;
    if (!w || !s || !y) return FP8BS_ERR_INVALID_ARG;
    if (!aligned4(s) || (reinterpret_cast<uintptr_t>(y) & 1u)) return FP8BS_ERR_MISALIGNED;
    if (K % 16 == 0 && (!aligned16(w) || !aligned16(y))) return FP8BS_ERR_MISALIGNED;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return status_of(
        fp8bs::launch_weight_dequant(w, s, y, N, K, static_cast<cudaStream_t>(stream)));
}

int fp8bs_gemm(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
               int64_t M, int64_t N, int64_t K, int scale_fmt, void* stream) {
    return fp8bs_gemm_ex(a, a_s, b, b_s, c, M, N, K, scale_fmt, 0u, stream);
}

int fp8bs_gemm_ex(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
                  int64_t M, int64_t N, int64_t K, int scale_fmt, unsigned int flags,
                  void* stream) {
    return gemm_impl(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, nullptr, 0, stream);
}

int fp8bs_gemm_ws(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
                  int64_t M, int64_t N, int64_t K, int scale_fmt, unsigned int flags,
                  void* workspace, size_t workspace_bytes, void* stream) {
    return gemm_impl(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, workspace, workspace_bytes,
                     stream);
}

int fp8bs_act_quant_gemm(const void* x, void* y, float* s, const void* b, const float* b_s,
                         void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                         unsigned int flags, void* workspace, size_t workspace_bytes,
                         void* stream) {
    if ((flags & ~(FP8BS_GEMM_WEIGHTS_CONSTANT | FP8BS_GEMM_QUANT_IN_KERNEL)) != 0)
        return FP8BS_ERR_INVALID_ARG;
    const bool in_kernel = (flags & FP8BS_GEMM_QUANT_IN_KERNEL) != 0;
    flags &= ~FP8BS_GEMM_QUANT_IN_KERNEL;
    if (M < 0 || N < 0 || K < 0 || K % FP8BS_BLOCK != 0) return FP8BS_ERR_INVALID_ARG;
    if (scale_fmt != FP8BS_SCALE_FP32 && scale_fmt != FP8BS_SCALE_UE8M0)
        return FP8BS_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BS_OK;
    if (!c) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(c)) return FP8BS_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int sms = 0;
    if (K == 0) {
        if (int e = check_device(&sms)) return e;
        return status_of(cudaMemsetAsync(c, 0, static_cast<size_t>(M * N) * 2, st));
    }
    if (!x || !y || !s || !b || !b_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned4(s) || !aligned16(b) || !aligned4(b_s))
        return FP8BS_ERR_MISALIGNED;
    if (int e = check_device(&sms)) return e;
    if (workspace) {
        if (!aligned16(workspace)) return FP8BS_ERR_MISALIGNED;
        if (workspace_bytes < fp8bs::stream_k_workspace(sms)) return FP8BS_ERR_INVALID_ARG;
    }
    const bool ue8m0 = scale_fmt == FP8BS_SCALE_UE8M0;
    if (in_kernel && M <= 16) {
        // One launch: every CTA of the decode GEMM quantises x (at most 16 rows) before its
        // main loop.
        const int MT = 16;
        GemmArgs g;
        g.a_s = s;
        g.b_s = b_s;
        g.c = c;
        g.M = static_cast<int>(M);
        g.N = static_cast<int>(N);
        g.K = static_cast<int>(K);
        g.weights_constant = (flags & FP8BS_GEMM_WEIGHTS_CONSTANT) ? 1 : 0;
        fp8bs::FusedQuant fq;
        fq.x = static_cast<const uint4*>(x);
        fq.y = static_cast<uint4*>(y);
        fq.s = s;
        fq.ue8m0 = ue8m0 ? 1 : 0;
        // Only where the separate GEMM would not split its K loop either: the one kernel
        // promotes every K block in order, and C must equal that of the separate calls.
        const int row_tiles = (g.M + MT - 1) / MT;
        if (fp8bs::plan_gemm_swapab(MT, false, row_tiles, g.N, g.K, sms) == 1 &&
            fp8bs::plan_gemm_swapab(MT, true, row_tiles, g.N, g.K, sms) == 1) {
            // x is read directly (no tensor map): tmB stands in for the unused map of A.
            CUtensorMap tmB;
            if (!make_map(&tmB, b, N, K, 128)) return FP8BS_ERR_CUDA;
            const int64_t rows[2] = {0, M};
            fp8bs::GroupTable gt;
            fp8bs::fill_row_tiles(&gt, rows, 1, MT);
            return status_of(fp8bs::launch_gemm_swapab(tmB, tmB, g, gt, MT, fq, 1, false, st));
        }
        // K too long to stage the scales, or a split K loop: two launches below.
    }
    // Two launches: act_quant, then the GEMM on its output.
    if (int st2 = status_of(fp8bs::launch_act_quant(x, y, s, M, K, ue8m0, sms, st))) return st2;
    return gemm_impl(y, s, b, b_s, c, M, N, K, scale_fmt, flags, workspace, workspace_bytes,
                     stream);
}

int fp8bs_linear_bf16(const void* x, const void* w, const float* w_s, void* y, int64_t M,
                      int64_t N, int64_t K, unsigned int flags, void* stream) {
    if ((flags & ~FP8BS_GEMM_WEIGHTS_CONSTANT) != 0) return FP8BS_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || K % FP8BS_BLOCK != 0) return FP8BS_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BS_OK;
    if (!y) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(y)) return FP8BS_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int sms = 0;
    if (K == 0) {
        if (int e = check_device(&sms)) return e;
        return status_of(cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * 2, st));
    }
    if (!x || !w || !w_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned4(w_s)) return FP8BS_ERR_MISALIGNED;
    if (int e = check_device(&sms)) return e;
    const int MT = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    CUtensorMap tmW, tmX;
    if (!make_map(&tmW, w, N, K, 128) || !make_map_bf16_sw128(&tmX, x, M, K, MT))
        return FP8BS_ERR_CUDA;
    return status_of(fp8bs::launch_linear_bf16_swap(
        tmW, tmX, w_s, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), MT,
        (flags & FP8BS_GEMM_WEIGHTS_CONSTANT) ? 1 : 0, st));
}

int fp8bs_gemm_noalloc(const void* a, const float* a_s, const void* b, const float* b_s,
                       void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                       unsigned int flags, void* stream) {
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    void* ws = nullptr;
    size_t bytes = 0;
    const cudaError_t e = fp8bs::bs_static_workspace(sms, &ws, &bytes);
    if (e == cudaErrorInvalidValue) return FP8BS_ERR_UNSUPPORTED_DEVICE;
    if (e != cudaSuccess) return FP8BS_ERR_CUDA;
    return gemm_impl(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, ws, bytes, stream);
}

int fp8bs_gemm_config(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
                      int64_t M, int64_t N, int64_t K, int scale_fmt, unsigned int flags,
                      int kernel, int tile, int ksplit, void* workspace, size_t workspace_bytes,
                      void* stream) {
    const int cfg[3] = {kernel, tile, ksplit};
    return gemm_impl(a, a_s, b, b_s, c, M, N, K, scale_fmt, flags, workspace, workspace_bytes,
                     stream, cfg);
}

int fp8bs_gemm_plan(int64_t M, int64_t N, int64_t K, int scale_fmt, int with_workspace,
                    int* kernel, int* tile, int* ksplit, int* stream_k) {
    if (!kernel || !tile || !ksplit || !stream_k) return FP8BS_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % FP8BS_BLOCK != 0) return FP8BS_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (scale_fmt != FP8BS_SCALE_FP32 && scale_fmt != FP8BS_SCALE_UE8M0)
        return FP8BS_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    // Any non-null pointer stands for a workspace here: the plan only asks whether one is given.
    static char marker;
    const GemmPlan p = plan_gemm(M, N, K, scale_fmt == FP8BS_SCALE_UE8M0,
                                 with_workspace ? &marker : nullptr, sms);
    *kernel = p.kind;
    *tile = p.tile;
    *ksplit = p.ksplit;
    *stream_k = p.ska.workspace != nullptr ? 1 : 0;
    return FP8BS_OK;
}

int fp8bs_gemm_workspace_size(size_t* bytes) {
    if (!bytes) return FP8BS_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    *bytes = fp8bs::stream_k_workspace(sms);
    return FP8BS_OK;
}

int fp8bs_gemm_grouped(const void* a, const float* a_s, const void* b, const float* b_s, void* c,
                       const int64_t* row_offsets, int64_t groups, int64_t N, int64_t K,
                       int scale_fmt, void* stream) {
    if (groups < 0 || groups > fp8bs::kMaxGroups || N < 0 || K < 0 || K % FP8BS_BLOCK != 0)
        return FP8BS_ERR_INVALID_ARG;
    if (scale_fmt != FP8BS_SCALE_FP32 && scale_fmt != FP8BS_SCALE_UE8M0)
        return FP8BS_ERR_INVALID_ARG;
    if (groups == 0 || N == 0) return FP8BS_OK;
    if (!row_offsets || row_offsets[0] != 0) return FP8BS_ERR_INVALID_ARG;
    for (int64_t i = 0; i < groups; ++i)
        if (row_offsets[i + 1] < row_offsets[i]) return FP8BS_ERR_INVALID_ARG;
    const int64_t M = row_offsets[groups];
    if (M > INT32_MAX || N * groups > INT32_MAX || K > INT32_MAX) return FP8BS_ERR_INVALID_ARG;
    if (M == 0) return FP8BS_OK;
    if (!c) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(c)) return FP8BS_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        int sms = 0;
        if (int e = check_device(&sms)) return e;
        return status_of(cudaMemsetAsync(c, 0, static_cast<size_t>(M * N) * 2, st));
    }
    if (!a || !a_s || !b || !b_s) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned4(a_s) || !aligned4(b_s))
        return FP8BS_ERR_MISALIGNED;
    int sms = 0;
    if (int e = check_device(&sms)) return e;

    GemmArgs g;
    g.a_s = a_s;
    g.b_s = b_s;
    g.c = c;
    g.M = static_cast<int>(M);
    g.N = static_cast<int>(N);
    g.K = static_cast<int>(K);
    g.weights_constant = 0;
    // Groups of at most 64 rows run in the swapped orientation (their weights on the MMA's M
    // side, their few rows on its N side, as at decode), the others as 128-row tiles. With both
    // kinds, the small groups' launch follows the other one without waiting for it (the two
    // write disjoint rows of C): its CTAs take the SMs the first launch's last round leaves
    // idle. The small groups' launch takes one CTA per 128-row weight slab of each group: where
    // that is a little more than one wave (10 MoE experts x 16 slabs on 152 SMs took 48 us for
    // 147 MB of weights), its largest groups join the tiles instead, provided they add no round
    // to the tile launch.
    const bool block_scaled = scale_fmt == FP8BS_SCALE_UE8M0;
    const int64_t slabs = ceil_div(N, 128);
    auto tile_rounds = [&](int64_t m_tiles) {
        if (m_tiles == 0) return static_cast<int64_t>(0);
        const int bn = block_scaled ? fp8bs::pick_tile_n_bs(m_tiles, N, sms)
                                    : fp8bs::pick_tile_n(m_tiles, N, sms);
        return ceil_div(m_tiles * ceil_div(N, bn), sms);
    };
    int64_t cand[fp8bs::kMaxGroups];               // groups of 1 .. 64 rows, fewest rows first
    int64_t n_cand = 0, m_big = 0;
    for (int64_t i = 0; i < groups; ++i) {
        const int64_t rows = row_offsets[i + 1] - row_offsets[i];
        if (rows > 0 && rows <= 64)
            cand[n_cand++] = i;
        else
            m_big += (rows + 127) / 128;
    }
    std::stable_sort(cand, cand + n_cand, [&](int64_t x, int64_t y) {
        return row_offsets[x + 1] - row_offsets[x] < row_offsets[y + 1] - row_offsets[y];
    });
    int64_t keep = n_cand;
    if (m_big > 0 && keep * slabs > sms && keep * slabs < 2 * static_cast<int64_t>(sms)) {
        const int64_t fit = sms / slabs;
        if (tile_rounds(m_big + (keep - fit)) <= tile_rounds(m_big)) keep = fit;
    }
    int64_t small_max = 0;
    for (int64_t j = 0; j < keep; ++j)
        small_max = std::max(small_max, row_offsets[cand[j] + 1] - row_offsets[cand[j]]);
    const int64_t small_count = keep;
    const int MT = small_max <= 16 ? 16 : small_max <= 32 ? 32 : 64;
    int S = 0;
    if (small_count > 0)      // 0: K too long for the swapped kernel, every group as tiles
        S = fp8bs::plan_gemm_swapab(MT, false, static_cast<int>(small_count), g.N, g.K, sms);
    bool small[fp8bs::kMaxGroups] = {};
    if (S > 0)
        for (int64_t j = 0; j < keep; ++j) small[cand[j]] = true;
    auto is_small = [&](int64_t i) { return small[i]; };

    int64_t m_tiles_total = 0;
    for (int64_t i = 0; i < groups; ++i) {
        const int64_t rows = row_offsets[i + 1] - row_offsets[i];
        if (!is_small(i)) m_tiles_total += (rows + 127) / 128;
    }
    bool launched = false;
    if (m_tiles_total > 0) {
        // The group table keeps every group's rows; the small groups contribute no tiles.
        const int BN = block_scaled ? fp8bs::pick_tile_n_bs(m_tiles_total, N, sms)
                                    : fp8bs::pick_tile_n(m_tiles_total, N, sms);
        const int n_tiles = static_cast<int>(ceil_div(N, BN));
        fp8bs::GroupTable gt;
        gt.num_groups = static_cast<int>(groups);
        gt.row_off[0] = 0;
        gt.tile_off[0] = 0;
        for (int64_t i = 0; i < groups; ++i) {
            const int64_t rows = row_offsets[i + 1] - row_offsets[i];
            gt.row_off[i + 1] = static_cast<int>(row_offsets[i + 1]);
            gt.tile_off[i + 1] =
                gt.tile_off[i] + (is_small(i) ? 0 : static_cast<int>((rows + 127) / 128)) * n_tiles;
        }
        CUtensorMap tmA, tmB;
        if (!make_map(&tmA, a, M, K, 128) || !make_map(&tmB, b, N * groups, K, BN))
            return FP8BS_ERR_CUDA;
        const cudaError_t e =
            block_scaled ? fp8bs::launch_gemm_bs(tmA, tmB, g, gt, BN, sms, no_stream_k(), st)
                         : fp8bs::launch_gemm_tn(tmA, tmB, g, gt, BN, sms, no_stream_k(), st);
        if (e != cudaSuccess) return FP8BS_ERR_CUDA;
        launched = true;
    }
    if (small_count > 0 && S > 0) {
        fp8bs::GroupTable gt;
        gt.num_groups = static_cast<int>(groups);
        gt.row_off[0] = 0;
        gt.tile_off[0] = 0;
        for (int64_t i = 0; i < groups; ++i) {
            gt.row_off[i + 1] = static_cast<int>(row_offsets[i + 1]);
            gt.tile_off[i + 1] =
                gt.tile_off[i] + (is_small(i) ? 1 : 0);
        }
        CUtensorMap tmA, tmB;
        if (!make_map(&tmB, b, N * groups, K, 128) || !make_map(&tmA, a, M, K, MT))
            return FP8BS_ERR_CUDA;
        return status_of(fp8bs::launch_gemm_swapab(tmB, tmA, g, gt, MT, fp8bs::FusedQuant{}, S,
                                                   launched, st));
    }
    return FP8BS_OK;
}

int fp8bs_device_error(unsigned int* out, int clear, void* stream) {
    if (!out) return FP8BS_ERR_INVALID_ARG;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return status_of(fp8bs::read_device_error(out, clear != 0, static_cast<cudaStream_t>(stream)));
}

int fp8bs_probe_occupy(int ctas, uint64_t duration_ns, void* stream) {
    if (ctas < 1 || ctas > 1024) return FP8BS_ERR_INVALID_ARG;
    if (duration_ns > 5000000000ull) duration_ns = 5000000000ull;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return status_of(fp8bs::launch_probe_occupy(ctas, duration_ns,
                                                static_cast<cudaStream_t>(stream)));
}

int fp8bs_probe_wait_timeout(uint64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000000ull) timeout_ns = 1000000ull;
    if (timeout_ns > 2000000000ull) timeout_ns = 2000000000ull;
    int sms = 0;
    if (int st = check_device(&sms)) return st;
    return status_of(fp8bs::launch_probe_wait(timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
