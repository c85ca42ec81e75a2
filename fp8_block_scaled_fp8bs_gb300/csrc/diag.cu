// diag.cu -- the bounded-wait probe (fp8bs_probe_wait_timeout) and the device error word that
// combines the words of every kernel file (fp8bs_device_error).
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

__global__ void probe_wait_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        // Nothing ever arrives on `bar`: the wait must run out and report.
        if (!mbar_wait(&bar, 0, timeout_ns)) record_error(FP8BS_DEVERR_PROBE);
    }
}

// Holds its SM (it claims most of the SM's shared memory) until duration_ns have passed.
__global__ void probe_occupy_kernel(uint64_t duration_ns) {
    extern __shared__ uint8_t held[];
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        volatile uint8_t* p = held;
        while (global_timer_ns() - t0 < duration_ns) p[0] = 1;
    }
}

constexpr int kOccupySmem = 200 * 1024;

}  // namespace

cudaError_t launch_probe_occupy(int ctas, uint64_t duration_ns, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(probe_occupy_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kOccupySmem);
    if (e != cudaSuccess) return e;
    probe_occupy_kernel<<<ctas, 32, kOccupySmem, stream>>>(duration_ns);
    return cudaGetLastError();
}

cudaError_t launch_probe_wait(uint64_t timeout_ns, cudaStream_t stream) {
    probe_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError();
}

cudaError_t read_device_error(unsigned int* out, bool clear, cudaStream_t stream) {
    unsigned int words[5] = {0, 0, 0, 0, 0};
    cudaError_t e = read_tu_error(&words[0], clear, stream);
    if (e == cudaSuccess) e = read_error_tn(&words[1], clear, stream);
    if (e == cudaSuccess) e = read_error_bs(&words[2], clear, stream);
    if (e == cudaSuccess) e = read_error_swapab(&words[3], clear, stream);
    if (e == cudaSuccess) e = read_error_linear(&words[4], clear, stream);
    if (e == cudaSuccess && clear) e = reset_static_workspace_counters(stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    *out = words[0] | words[1] | words[2] | words[3] | words[4];
    return e;
}

}  // namespace fp8bs
