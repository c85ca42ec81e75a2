/*
 * fp8bs.h -- C ABI of the FP8 block-scaled linear-layer library for NVIDIA GB300 (sm_103a).
 *
 * The library implements the three FP8 operations of the DeepSeek-V3 inference demo's linear
 * path, as the pages describe them:
 *   - act_quant       "DeepSeek-V3 Administrator & Developer Guide", §8.5.1 act_quant_kernel;
 *                     ue8m0 scales: "DeepSeek-V3 User Guide", FAQ "What is scale_fmt: ue8m0?".
 *   - weight_dequant  "DeepSeek-V3 Administrator & Developer Guide", §8.5.2 weight_dequant_kernel
 *                     (scale shape from §6.3 The FP8 path, item 2).
 *   - fp8_gemm        "DeepSeek-V3 Administrator & Developer Guide", §8.5.3 fp8_gemm_kernel;
 *                     used by linear() when gemm_impl == "fp8" (§6.3 item 3).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer into memory the caller owns; the library allocates and
 *     frees nothing and keeps no per-call state, so calls from several host threads are safe.
 *     Exceptions, marked "host memory allowed" below: act_quant's input x and the bf16 output
 *     of the GEMMs and of the bf16 path may also point into pinned (page-locked) host memory,
 *     as cudaHostAlloc, cudaMallocHost or cudaHostRegister provide it. The kernels then read or
 *     write it in place over the host link (NVLink-C2C on GB300), with no staging copy; the
 *     bytes still cross the link once. Those kernels access x and C with plain loads and
 *     stores, never with the tensor memory accelerator, which only reads device memory.
 *   - Matrices are row-major and contiguous. bf16 is the 16-bit brain float; e4m3 is
 *     float8_e4m3fn (1 byte, largest magnitude 448, no infinity).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is only enqueued:
 *     no call synchronises the host. Errors that happen while a kernel runs surface at the
 *     caller's next synchronisation (or through fp8bs_device_error for bounded waits).
 *   - Arguments are checked before anything is launched; a failed check launches nothing and
 *     returns a nonzero fp8bs_status. A size of zero (M, N or K where allowed) is a no-op that
 *     returns FP8BS_OK (fp8bs_gemm with K == 0 writes zeros).
 *   - Inputs and outputs must not overlap.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols stay visible when the library is built with -fvisibility=hidden. */
#if defined(__GNUC__)
#define FP8BS_API __attribute__((visibility("default")))
#else
#define FP8BS_API
#endif

/* Quantisation block along K (1 x 128 for activations, 128 x 128 for weights). */
#define FP8BS_BLOCK 128

typedef enum {
    FP8BS_SCALE_FP32 = 0,  /* s = max(amax, 1e-4) / 448, one IEEE binary32 division */
    FP8BS_SCALE_UE8M0 = 1  /* s as above, then rounded up to the nearest power of two */
} fp8bs_scale_fmt;

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1,        /* null pointer, negative size, K % 128 != 0, bad enum */
    FP8BS_ERR_MISALIGNED = 2,         /* a pointer is not 16-byte aligned */
    FP8BS_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    FP8BS_ERR_CUDA = 4                /* a CUDA runtime call or launch failed */
} fp8bs_status;

/*
 * fp8bs_act_quant -- quantise bf16 activations to e4m3 with one fp32 scale per 1x128 block.
 * ("DeepSeek-V3 Administrator & Developer Guide", §8.5.1.)
 *
 *   x  [in]  bf16 [M, K], 16-byte aligned; host memory allowed.
 *   y  [out] e4m3 [M, K], 16-byte aligned.
 *   s  [out] fp32 [M, K/128], 4-byte aligned: s[m, b] is the scale of x[m, 128b : 128b+128].
 *   M >= 0, K >= 0 with K % 128 == 0.
 *   scale_fmt: FP8BS_SCALE_FP32 or FP8BS_SCALE_UE8M0.
 *
 * Per block: amax = max |x|; s = max(amax, 1e-4f) / 448.0f (IEEE binary32 division);
 * for UE8M0, s = 2^ceil(log2 s) exactly; y = x / s (IEEE binary32 division), converted to
 * e4m3 with round-to-nearest-even and saturation at +-448. Results are bit-exact.
 */
FP8BS_API int fp8bs_act_quant(const void* x, void* y, float* s, int64_t M, int64_t K,
                              int scale_fmt, void* stream);

/*
 * fp8bs_weight_dequant -- expand e4m3 weights with 128x128 block scales to bf16.
 * ("DeepSeek-V3 Administrator & Developer Guide", §8.5.2 and §6.3 item 2.)
 *
 *   w  [in]  e4m3 [N, K].
 *   s  [in]  fp32 [ceil(N/128), ceil(K/128)], 4-byte aligned: one scale per 128x128 block;
 *            a partial edge block uses its own single scale.
 *   y  [out] bf16 [N, K].
 *   N >= 0, K >= 0 (any values). w and y must be 16-byte aligned when K % 16 == 0
 *   (the vectorised path); otherwise only element alignment is needed.
 *
 * y[n, k] = bf16_rne(fp32(w[n, k]) * s[n/128, k/128]) with the product rounded to binary32
 * first. Results are bit-exact.
 */
FP8BS_API int fp8bs_weight_dequant(const void* w, const float* s, void* y, int64_t N,
                                   int64_t K, void* stream);

/*
 * fp8bs_gemm -- block-scaled FP8 GEMM C = A . B^T with bf16 output.
 * ("DeepSeek-V3 Administrator & Developer Guide", §8.5.3.)
 *
 *   a    [in]  e4m3 [M, K], 16-byte aligned (typically the act_quant output).
 *   a_s  [in]  fp32 [M, K/128], 4-byte aligned (per row, per 128-wide K block).
 *   b    [in]  e4m3 [N, K], 16-byte aligned (a Linear weight, out x in).
 *   b_s  [in]  fp32 [ceil(N/128), K/128], 4-byte aligned (per 128x128 block of b).
 *   c    [out] bf16 [M, N], 16-byte aligned; host memory allowed.
 *   M >= 0, N >= 0, K >= 0 with K % 128 == 0.
 *   scale_fmt: FP8BS_SCALE_FP32: a_s and b_s are any positive finite fp32 values.
 *              FP8BS_SCALE_UE8M0: the caller promises that every a_s and b_s value is a power
 *              of two 2^e with -126 <= e <= 127 (the V3.1 ue8m0 scales; act_quant with
 *              FP8BS_SCALE_UE8M0 produces such a_s). For M > 128 the tensor cores then apply
 *              the scales themselves (block-scaled MMA with ue8m0 scale factors). A scale that
 *              breaks the promise sets FP8BS_DEVERR_SCALE_NOT_POW2 and makes C undefined.
 *
 * C[m, n] = sum_kb a_s[m, kb] * b_s[n/128, kb] * sum_{k in block kb} a[m, k] * b[n, k]:
 * each block's partial product is formed on the tensor cores in fp32, scaled and accumulated
 * in fp32, and the sum is rounded once to bf16. Accuracy: |C - C_exact| <=
 * 2^-7 |C_exact| + 1e-3 rms(C_exact) elementwise on the documented workloads.
 */
FP8BS_API int fp8bs_gemm(const void* a, const float* a_s, const void* b, const float* b_s,
                         void* c, int64_t M, int64_t N, int64_t K, int scale_fmt, void* stream);

/*
 * fp8bs_gemm_ex -- fp8bs_gemm with flags (fp8bs_gemm is fp8bs_gemm_ex with flags == 0).
 *
 *   flags: 0 or FP8BS_GEMM_WEIGHTS_CONSTANT. With FP8BS_GEMM_WEIGHTS_CONSTANT the caller
 *   promises that b and b_s are not written by any work enqueued earlier on `stream` (model
 *   weights during inference): the kernel may then start reading them before the kernel
 *   ahead of it on the stream has finished (the act_quant that produces `a`, typically),
 *   which hides the start of the weight stream behind it. Unknown flag bits are rejected.
 *
 * Every kernel of this library is launched with programmatic stream serialisation: it may
 * begin while the kernel before it finishes, and waits for that kernel before reading anything
 * it could have written (all inputs, or all but b and b_s with the flag above).
 */
#define FP8BS_GEMM_WEIGHTS_CONSTANT 0x1u
/* fp8bs_act_quant_gemm only: quantise the activations inside the GEMM kernel (M <= 16). */
#define FP8BS_GEMM_QUANT_IN_KERNEL 0x2u
FP8BS_API int fp8bs_gemm_ex(const void* a, const float* a_s, const void* b, const float* b_s,
                            void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                            unsigned int flags, void* stream);

/*
 * fp8bs_gemm_ws -- fp8bs_gemm_ex with a device workspace, which lets the library share the K
 * loop of an output tile between SMs (stream-K) when the tiles do not fill the SMs evenly
 * (M > 128, at least as many tiles as SMs, e.g. the prefill up-projection with fp32 scales);
 * otherwise the call runs as fp8bs_gemm_ex. The partial sums of a shared tile are added in a
 * fixed order, so results do not depend on timing. A stream-K grid is launched cooperatively
 * (the runtime places all its CTAs at once); where the runtime cannot, the call computes whole
 * tiles instead. ("DeepSeek-V3 Administrator & Developer Guide", §8.5.3, computed as in
 * fp8bs_gemm; the pages' kernel has no split of K.) Every call, with or without a workspace,
 * may also split a tile's K loop between the CTAs of a thread-block cluster when the tiles are
 * few (fp8bs_gemm_plan shows the choice); that needs no workspace.
 *
 *   workspace        device memory of at least fp8bs_gemm_workspace_size bytes, 16-byte
 *                    aligned, owned by the caller. It must hold zeros before its first use;
 *                    every call that completes without a device error leaves it that way (after
 *                    a device error, fill it with zeros again). Calls that may run at the same
 *                    time (on different streams) need different workspaces. NULL: no splitting.
 *   workspace_bytes  its size in bytes; a non-NULL workspace smaller than
 *                    fp8bs_gemm_workspace_size returns FP8BS_ERR_INVALID_ARG.
 *   other arguments  as in fp8bs_gemm_ex.
 */
FP8BS_API int fp8bs_gemm_ws(const void* a, const float* a_s, const void* b, const float* b_s,
                            void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                            unsigned int flags, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * fp8bs_gemm_plan -- which kernel, tile and schedule fp8bs_gemm_ws (or fp8bs_gemm_ex, when
 * with_workspace == 0) would launch for these sizes on the current device. Launches nothing.
 * The pages' fp8_gemm picks its configuration by autotuning ("DeepSeek-V3 Administrator &
 * Developer Guide", §8.5.3 and §6.5); this library picks it from the shape, and this call shows
 * the pick.
 *
 *   M, N, K > 0 with K % 128 == 0; scale_fmt as in fp8bs_gemm.
 *   kernel   [out] FP8BS_KERNEL_SWAPPED (M <= 128: 128-row weight slabs on the MMA's M side),
 *                  FP8BS_KERNEL_PROMOTED (fp32 scales applied by CUDA cores per K block),
 *                  FP8BS_KERNEL_BLOCK_SCALED (ue8m0 scales applied by the tensor cores) or
 *                  FP8BS_KERNEL_BLOCK_SCALED_PAIR (the same on pairs of SMs, 256-row tiles).
 *   tile     [out] rows of A per CTA (swapped) or columns of B per tile (otherwise).
 *   ksplit   [out] CTAs of one thread-block cluster that share each tile's K loop (1: none).
 *   stream_k [out] 1 if tiles share K loops through the workspace (stream-K), else 0.
 */
#define FP8BS_KERNEL_SWAPPED 0
#define FP8BS_KERNEL_PROMOTED 1
#define FP8BS_KERNEL_BLOCK_SCALED 2
#define FP8BS_KERNEL_BLOCK_SCALED_PAIR 3
FP8BS_API int fp8bs_gemm_plan(int64_t M, int64_t N, int64_t K, int scale_fmt, int with_workspace,
                              int* kernel, int* tile, int* ksplit, int* stream_k);

/*
 * fp8bs_gemm_config -- fp8bs_gemm_ws with the launch configuration given by the caller, in the
 * vocabulary of fp8bs_gemm_plan, instead of chosen from the shape: for callers that tune their
 * own shapes (the pages' fp8_gemm autotunes over tile configurations, "DeepSeek-V3
 * Administrator & Developer Guide", §6.5 and §8.5.3) and for tests that cover every kernel
 * schedule. Results and accuracy as in fp8bs_gemm.
 *
 *   kernel  FP8BS_KERNEL_SWAPPED      tile = rows of A per CTA, 16, 32, 64 or 128, and >= M.
 *           FP8BS_KERNEL_PROMOTED     tile = 64, 128, 192 or 256 columns (any scale_fmt).
 *           FP8BS_KERNEL_BLOCK_SCALED tile = 64, 128, 192 or 256 (scale_fmt UE8M0).
 *           FP8BS_KERNEL_BLOCK_SCALED_PAIR  tile = 128, 192 or 256 (UE8M0, ksplit 1).
 *   ksplit  1: whole tiles; 2 .. 8 (and at most K/128): each tile's K loop split between that
 *           many CTAs of a cluster; 0 (normal orientation only; tile 128 for BLOCK_SCALED):
 *           stream-K over `workspace`, which is then required, for shapes with at least as
 *           many tiles as SMs.
 *   Other arguments as in fp8bs_gemm_ws. A configuration the kernels do not support for the
 *   shape returns FP8BS_ERR_INVALID_ARG and launches nothing.
 */
FP8BS_API int fp8bs_gemm_config(const void* a, const float* a_s, const void* b, const float* b_s,
                                void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                                unsigned int flags, int kernel, int tile, int ksplit,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * fp8bs_gemm_workspace_size -- bytes of workspace fp8bs_gemm_ws uses on the current device: the
 * same for every problem size (one 128 x 256 fp32 partial tile and one counter per SM, about
 * 20 MB on 152 SMs).
 *   bytes [out] host pointer receiving the size.
 */
FP8BS_API int fp8bs_gemm_workspace_size(size_t* bytes);

/*
 * fp8bs_act_quant_gemm -- act_quant followed by the block-scaled GEMM on its output, the two
 * steps of linear() on the FP8 path ("DeepSeek-V3 Administrator & Developer Guide", §6.3
 * item 3: act_quant, then fp8_gemm; §8.5.1 and §8.5.3), as one call. By default two kernels
 * run back to back (the GEMM starts while act_quant finishes and, with
 * FP8BS_GEMM_WEIGHTS_CONSTANT, streams its weights meanwhile). With
 * FP8BS_GEMM_QUANT_IN_KERNEL and M <= 16 one kernel does both: before its main loop every CTA
 * of the GEMM reads x and quantises it whole, as act_quant would, into shared memory (while
 * its weight stages fill), and the CTAs of the first 128 columns also write y and s. The two
 * launches run instead where the separate GEMM would split each weight slab's K loop between
 * several CTAs (few slabs, see fp8bs_gemm_plan) or where the quantised x (16 x K bytes) does
 * not fit in shared memory beside two weight stages (K up to 11264). On GB300 at decode
 * sizes the single kernel measured no faster than the two (N = 18432, K = 7168: 25.7 against
 * 25.1 us at M = 1, 30.7 against 25.4 us at M = 8: every CTA quantises all of x), so it is not
 * the default.
 *
 *   x      [in]  bf16 [M, K], 16-byte aligned; host memory allowed (also with
 *          FP8BS_GEMM_QUANT_IN_KERNEL, where the GEMM's CTAs read it).
 *   y      [out] e4m3 [M, K], 16-byte aligned: the quantised activations, as fp8bs_act_quant.
 *   s      [out] fp32 [M, K/128], 4-byte aligned: their scales, as fp8bs_act_quant.
 *   b, b_s, c, M, N, K, scale_fmt, flags  as in fp8bs_gemm_ex (a = y, a_s = s); scale_fmt
 *          also selects act_quant's scale format.
 *   workspace, workspace_bytes  as in fp8bs_gemm_ws, for the GEMM of the two-launch case
 *          (NULL: no split K loops).
 *
 * y, s and c are bit for bit those of fp8bs_act_quant then fp8bs_gemm_ws on the same stream.
 */
FP8BS_API int fp8bs_act_quant_gemm(const void* x, void* y, float* s, const void* b,
                                   const float* b_s, void* c, int64_t M, int64_t N, int64_t K,
                                   int scale_fmt, unsigned int flags, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * fp8bs_linear_bf16 -- the bf16 path of linear() with an FP8 weight: y = x . W'^T, where W' is
 * the bf16 weight fp8bs_weight_dequant would produce from w and w_s ("DeepSeek-V3
 * Administrator & Developer Guide", §6.3: with gemm_impl = "bf16", weight_dequant (§8.5.2)
 * then a bf16 GEMM). W' is formed tile by tile on chip (in tensor memory), never in HBM;
 * products are accumulated in fp32 on the tensor cores and y is rounded once to bf16. Any M:
 * each CTA pairs one 128-row slab of w with up to 128 rows of x, or two tiles of 128 rows
 * when M > 128.
 *
 *   x    [in]  bf16 [M, K], 16-byte aligned.
 *   w    [in]  e4m3 [N, K], 16-byte aligned.
 *   w_s  [in]  fp32 [ceil(N/128), K/128], 4-byte aligned.
 *   y    [out] bf16 [M, N], 16-byte aligned; host memory allowed.
 *   M >= 0, N >= 0, K >= 0 with K % 128 == 0.
 *   flags: 0 or FP8BS_GEMM_WEIGHTS_CONSTANT (as in fp8bs_gemm_ex).
 *
 * Accuracy: |y - y_exact| <= 2^-7 |y_exact| + 1e-3 rms(y_exact) elementwise, y_exact the
 * product of x with W' in exact arithmetic.
 */
FP8BS_API int fp8bs_linear_bf16(const void* x, const void* w, const float* w_s, void* y,
                                int64_t M, int64_t N, int64_t K, unsigned int flags,
                                void* stream);

/*
 * fp8bs_gemm_noalloc -- fp8bs_gemm_ws on a workspace that the library keeps in a static device
 * array (about 21 MB per device, sized for up to 160 SMs and reserved when the library's device
 * code is loaded): no memory is allocated by the caller or by the library at any time. The pages have no
 * counterpart of this entry point: their fp8_gemm neither splits K nor uses scratch memory.
 *
 *   Arguments, results and accuracy as in fp8bs_gemm_ws.
 *   Calls on one device share the one workspace: they must not run at the same time (issue
 *   them on one stream, or order them). After a call that recorded a device wait error, clear
 *   the error with fp8bs_device_error(clear != 0), which also zeroes the workspace's counters,
 *   before the next call. The workspace's address is looked up on the first call made with
 *   each device current and kept for the life of the process (a device reset invalidates it).
 *   A device with more than 160 SMs (more than the static workspace covers) returns
 *   FP8BS_ERR_UNSUPPORTED_DEVICE without launching anything.
 */
FP8BS_API int fp8bs_gemm_noalloc(const void* a, const float* a_s, const void* b, const float* b_s,
                                 void* c, int64_t M, int64_t N, int64_t K, int scale_fmt,
                                 unsigned int flags, void* stream);

/*
 * fp8bs_gemm_grouped -- several independent block-scaled GEMMs in one launch, one per group of
 * rows of A: the MoE expert loop of "DeepSeek-V3 Administrator & Developer Guide", §6.4 MoE
 * expert routing (each local expert runs its Linear on the tokens routed to it), with every
 * expert's GEMM as in §8.5.3.
 *
 *   a           [in]  e4m3 [T, K], 16-byte aligned: the rows of all groups, group i's rows
 *                     row_offsets[i] .. row_offsets[i+1]-1 (tokens gathered by expert).
 *   a_s         [in]  fp32 [T, K/128], 4-byte aligned.
 *   b           [in]  e4m3 [groups, N, K] (the experts' weights stacked), 16-byte aligned.
 *   b_s         [in]  fp32 [groups, ceil(N/128), K/128], 4-byte aligned.
 *   c           [out] bf16 [T, N], 16-byte aligned (host memory allowed): row r of group
 *                     i is A[r] . B[i]^T.
 *   row_offsets [in]  HOST array of groups+1 non-decreasing row offsets, row_offsets[0] == 0,
 *                     T = row_offsets[groups]; empty groups are allowed.
 *   groups      0 .. 256.  N >= 0, K >= 0 with K % 128 == 0.  scale_fmt as in fp8bs_gemm
 *               (with FP8BS_SCALE_UE8M0 every group runs on the block-scaled MMA).
 *
 * Results and accuracy are those of fp8bs_gemm on each group's rows. Groups of at most 64
 * rows are computed in the swapped orientation (their weights on the MMA's M side, as for
 * decode-sized M); the others as 128-row tiles. With both kinds the call enqueues two kernels,
 * and the second starts without waiting for the first (they write disjoint rows of c) but
 * completes only after it, so work enqueued after the call sees all of c.
 */
FP8BS_API int fp8bs_gemm_grouped(const void* a, const float* a_s, const void* b, const float* b_s,
                                 void* c, const int64_t* row_offsets, int64_t groups, int64_t N,
                                 int64_t K, int scale_fmt, void* stream);

/* Human-readable name of an fp8bs_status value (a static string; never NULL). */
FP8BS_API const char* fp8bs_status_string(int status);

/*
 * fp8bs_device_error -- read (and, if `clear` != 0, reset) the library's device error word
 * on the current device. Every wait inside the library's kernels is bounded in time; a wait
 * that runs out sets a bit here (see FP8BS_DEVERR_*), abandons the kernel's remaining work
 * (its output is then undefined) and lets the kernel exit cleanly. Synchronises `stream`.
 * With `clear`, the counters of fp8bs_gemm_noalloc's static workspace on this device are also
 * zeroed (a call abandoned after a wait error may leave them nonzero).
 *   out [out] host pointer receiving the word (0 = no error since the last clear).
 */
FP8BS_API int fp8bs_device_error(unsigned int* out, int clear, void* stream);

#define FP8BS_DEVERR_PRODUCER_WAIT 0x1u  /* TMA producer waited too long for a free stage */
#define FP8BS_DEVERR_MMA_WAIT 0x2u       /* MMA issuer waited too long for data or TMEM */
#define FP8BS_DEVERR_EPILOGUE_WAIT 0x4u  /* promotion/epilogue waited too long for TMEM */
#define FP8BS_DEVERR_DRAIN_WAIT 0x8u     /* in-flight copies did not drain after an abort */
#define FP8BS_DEVERR_SCALE_NOT_POW2 0x10u /* FP8BS_SCALE_UE8M0 GEMM met a scale that is not 2^e */
#define FP8BS_DEVERR_PROBE 0x100u        /* set by fp8bs_probe_wait_timeout */

/*
 * fp8bs_probe_wait_timeout -- diagnostic: launch one block that waits on a shared-memory
 * barrier that nothing signals, with the given limit in nanoseconds (clamped to 1 ms..2 s).
 * The wait runs out and sets FP8BS_DEVERR_PROBE in the device error word, exercising the
 * same bounded-wait path the GEMM kernels use. Enqueued only; read the word with
 * fp8bs_device_error.
 */
FP8BS_API int fp8bs_probe_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * fp8bs_probe_occupy -- diagnostic: launch `ctas` (1 .. 1024) CTAs that each hold one SM (they
 * claim most of its shared memory) and return after duration_ns (at most 5 s). Enqueued only.
 * With it a caller can run a GEMM while another stream holds some of the SMs: a stream-K
 * launch (fp8bs_gemm_ws) is a cooperative launch whose CTAs the runtime places all at once, so
 * its tiles' owners never wait on contributors that have no SM.
 */
FP8BS_API int fp8bs_probe_occupy(int ctas, uint64_t duration_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
