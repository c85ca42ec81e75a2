// kernels.h -- internal launchers behind the C ABI (include/fp8bs.h). Arguments are already
// validated by the caller; each launcher only enqueues work on `stream` and returns the
// launch status.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8bs {

// Launch with programmatic stream serialisation (see grid_dependency_wait in ptx.cuh): the
// launch may begin while the previous kernel on the stream is finishing.
// With cluster_x > 1 the grid is launched as clusters of cluster_x consecutive CTAs along x
// (grid.x must be a multiple of it). With `cooperative` the launch is a cooperative one: the
// runtime places every CTA of the grid at once (or refuses the launch), which the stream-K
// schedule relies on -- a tile's owner waits for partials from CTAs with larger indices.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster_x, bool cooperative,
                               Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n++].val.programmaticStreamSerializationAllowed = 1;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n++].val.clusterDim.z = 1;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n++].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    return launch_pdl_cluster(kernel, grid, block, smem, stream, 1, false,
                              static_cast<Args&&>(args)...);
}

// Split K inside a cluster: at most this many CTAs share a tile (the portable cluster size).
constexpr int kMaxSplit = 8;

// How many clusters of `cluster_x` CTAs of `kernel` (with `threads` threads and `smem` bytes of
// dynamic shared memory, already allowed by cudaFuncSetAttribute) can be resident at once on
// the current device; 0 if the query fails. Cached per (kernel, cluster size, smem, device).
int max_active_clusters(const void* kernel, int threads, int smem, int cluster_x);

cudaError_t launch_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K, bool ue8m0,
                             int num_sms, cudaStream_t stream);

cudaError_t launch_weight_dequant(const void* w, const float* s, void* y, int64_t N, int64_t K,
                                  cudaStream_t stream);

// Tensor maps are encoded by the caller (they need the driver entry point).
struct GemmArgs {
    const float* a_s;   // [M, K/128]
    const float* b_s;   // [ceil(N/128), K/128] per group
    void* c;            // bf16 [M, N]
    int M, N, K;        // M: all rows (of every group); N, K: per group
    int weights_constant;  // B and b_s may be read before earlier kernels on the stream finish
};

// Row groups of a grouped GEMM. Group i owns rows row_off[i] .. row_off[i+1]-1 of A, a_s and
// C, rows i*N .. i*N+N-1 of the stacked B, and scale rows i*ceil(N/128) .. of the stacked b_s.
// tile_off[i] is the first linear tile of group i (its m tiles times the n tiles of N). A plain
// GEMM is one group.
constexpr int kMaxGroups = 256;
struct GroupTable {
    int num_groups;
    int row_off[kMaxGroups + 1];
    int tile_off[kMaxGroups + 1];
};

// Tiles of 128 rows and `bn` columns for the given group row offsets (host-side helper).
void fill_group_table(GroupTable* gt, const int64_t* row_off, int groups, int N, int bn);

// Stream-K schedule of the normal-orientation kernels: a workspace (null: every tile computed
// whole by one CTA) and the number of tiles computed whole before the rest are shared (a
// multiple of the grid, which is then the SM count; 0 shares every tile). See gemm_common.cuh.
struct StreamKArgs {
    void* workspace;
    int dp_tiles;
    int ksplit;       // > 1: no workspace; ksplit CTAs (one cluster) share each tile's K loop
};

// Workspace layout: one int counter per SM (rounded up to 256 bytes), then one 128 x 256 fp32
// partial tile per SM -- the same for every problem size. It starts zero-filled and every call
// that completes leaves the counters at zero.
constexpr size_t stream_k_flag_bytes(int num_sms) {
    return (static_cast<size_t>(num_sms) * sizeof(int) + 255) / 256 * 256;
}
constexpr size_t stream_k_workspace(int num_sms) {
    return stream_k_flag_bytes(num_sms) + static_cast<size_t>(num_sms) * 128 * 256 * sizeof(float);
}

// Tile width for the normal orientation with fp32 scales: the one of 256, 192, 128 and 64
// columns that minimises rounds of tiles x measured time per tile.
int pick_tile_n(int64_t m_tiles_total, int64_t N, int num_sms);

// Normal orientation: 128-row tiles of A on the MMA's M side, BN (64, 128, 192 or 256)
// columns of B on its N side. tmA: box {128, 128} over A [rows, K]; tmB: box {128, BN} over B
// [groups*N, K].
cudaError_t launch_gemm_tn(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           const GroupTable& gt, int BN, int num_sms, const StreamKArgs& ska,
                           cudaStream_t stream);

// Clusters of S CTAs of the normal-orientation kernel at tile width BN (fp32 scales: _tn;
// ue8m0: _bs) that can be resident at once for a split-K launch; 0 if that split does not fit.
int max_split_clusters_tn(int BN, int S);
int max_split_clusters_bs(int BN, int S);

// Block-scaled orientation, for scales that are all powers of two (FP8BS_SCALE_UE8M0): the
// tensor core applies a_s and b_s as ue8m0 exponents per K block; tiles of 128 rows x BN
// (64 or 128; 128 when K loops are shared) columns, same maps and group table as
// launch_gemm_tn.
int pick_tile_n_bs(int64_t m_tiles_total, int64_t N, int num_sms);
cudaError_t launch_gemm_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g,
                           const GroupTable& gt, int BN, int num_sms, const StreamKArgs& ska,
                           cudaStream_t stream);
// Block-scaled GEMM on CTA pairs (cta_group::2): tiles of 256 rows of A x BN (128, 192 or 256)
// columns of B, each computed by a cluster of two CTAs; one group, whole tiles, `pairs`
// clusters persistent over the tiles. tmA: box {128, 128} over A; tmB: box {128, BN/2} over B.
// max_pair_clusters_bs: how many such clusters can be resident at once (0: query failed).
cudaError_t launch_gemm_bs_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const GemmArgs& g, int BN, int pairs, cudaStream_t stream);
int max_pair_clusters_bs(int BN);

// The library's static stream-K workspace on the current device (no allocation); fails with
// cudaErrorInvalidValue on a device with more SMs than it covers.
cudaError_t bs_static_workspace(int num_sms, void** ws, size_t* bytes);
// Zero the static workspace's counters on the current device (enqueued on `stream`).
cudaError_t reset_static_workspace_counters(cudaStream_t stream);

// Activations quantised inside the decode GEMM launch (MT <= 64): x bf16 [M, K] -> y e4m3,
// s fp32 (as act_quant writes them); every CTA quantises the rows of each K block it reads,
// those of the first weight slab also write y and s. x == nullptr: plain GEMM.
struct FusedQuant {
    const uint4* x;
    uint4* y;
    float* s;
    int ue8m0;
};

// Swapped orientation for few rows of A: 128-row slabs of B on the MMA's M side, MT rows of A
// on its N side. tmB: box {128, 128} over B [N,K]; tmA: box {128, MT} over A [M,K] (with
// FusedQuant: a bf16 map over x, box {128, MT}, no swizzle).
// Groups: the launch covers the MT-row tiles of every group of `gt` (tile_off counts row
// tiles, see fill_row_tiles); group i's rows take the stacked B's rows i*N .. and b_s's scale
// rows i*ceil(N/128) .. (a plain GEMM is one group). ksplit > 1 (quantised input only): the K
// loop of each 128-row slab is split between the ksplit CTAs of a cluster, whose fp32 partials
// are added in rank order through distributed shared memory. early: the launch reads nothing
// the kernel before it on the stream writes, so it starts at once and waits for that kernel
// only before it exits. plan_gemm_swapab gives the split for `row_tiles` tiles (1: none; 0:
// this kernel cannot take K, whose activation scales would not fit in shared memory).
int plan_gemm_swapab(int MT, bool fused, int row_tiles, int N, int K, int num_sms);
// Whether the quantised-input kernel can run with MT rows, this K and a split of ksplit.
bool check_gemm_swapab(int MT, int K, int ksplit);
void fill_row_tiles(GroupTable* gt, const int64_t* row_off, int groups, int MT);
cudaError_t launch_gemm_swapab(const CUtensorMap& tmB, const CUtensorMap& tmA,
                               const GemmArgs& g, const GroupTable& gt, int MT,
                               const FusedQuant& fq, int ksplit, bool early,
                               cudaStream_t stream);

// bf16 path, decode orientation (M <= 64, MT = 16, 32 or 64): y bf16 [M, N] = x . W'^T with W'
// the bf16 dequantisation of the e4m3 weight (128 x 128 block scales w_s). tmW: box {128, 128}
// over W [N, K] (128-byte swizzle); tmX: bf16 map over x [M, K], box {64, MT}, 128-byte swizzle.
cudaError_t launch_linear_bf16_swap(const CUtensorMap& tmW, const CUtensorMap& tmX,
                                    const float* w_s, void* y, int M, int N, int K, int MT,
                                    int weights_constant, cudaStream_t stream);

// Diagnostic kernel: one wait on a barrier nothing signals (see fp8bs_probe_wait_timeout).
cudaError_t launch_probe_wait(uint64_t timeout_ns, cudaStream_t stream);

// Diagnostic kernel: `ctas` CTAs that each take a whole SM (most of its shared memory) and
// return after `duration_ns` (see fp8bs_probe_occupy).
cudaError_t launch_probe_occupy(int ctas, uint64_t duration_ns, cudaStream_t stream);

// The device error word of the library (read/clear; synchronises `stream`): the OR of the
// words of the kernel files, each read (and cleared) by its own function below.
cudaError_t read_device_error(unsigned int* out, bool clear, cudaStream_t stream);
cudaError_t read_error_tn(unsigned int* out, bool clear, cudaStream_t stream);
cudaError_t read_error_bs(unsigned int* out, bool clear, cudaStream_t stream);
cudaError_t read_error_swapab(unsigned int* out, bool clear, cudaStream_t stream);
cudaError_t read_error_linear(unsigned int* out, bool clear, cudaStream_t stream);

}  // namespace fp8bs
