// quant_math.cuh -- the per-element arithmetic of act_quant ("DeepSeek-V3 Administrator &
// Developer Guide", §8.5.1 act_quant_kernel), shared by the standalone kernel (quant.cu) and
// the decode GEMM that quantises its own activations (gemm_swapab.cu), so that both produce the
// same codes and scales bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace fp8bs {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Quotient x / s rounded to nearest binary32, from r = RN(1/s): q0 = RN(x r) is within one ulp
// of x/s, the remainder x - q0 s is exact in one fused multiply-add, and one more fused
// multiply-add with r lands on RN(x/s). This is Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; also in Muller et al., "Handbook of Floating-Point Arithmetic"). For the
// values that occur here (x and amax bf16, s = RN(max(amax, 1e-4) / 448)) the identity is
// checked exhaustively on the host by the test suite.
// The correction step adds +0 to a zero quotient, which would turn x = -0 into +0; the sign
// of x is put back (for x != 0 the quotient already carries it, as s > 0).
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
    const float q0 = __fmul_rn(x, r);
    const float rem = __fmaf_rn(-q0, s, x);
    const float q = __fmaf_rn(rem, r, q0);
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Sixteen bf16 values (packed two per word) of one 128-element block, held by one of eight
// consecutive lanes that own the block: the block's amax is reduced with shuffles (every lane
// of the warp must call this), and the lane's 16 e4m3 codes (packed four per word) and the
// block's scale are returned.
template <bool UE8M0>
__device__ __forceinline__ float quant_block16(const uint32_t (&w)[8], uint32_t (&out)[4]) {
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    // s = max(amax, 1e-4) / 448 with one IEEE division.
    float sc = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
    if (UE8M0) {
        // 2^ceil(log2 s): s is a positive normal number; if any mantissa bit is set, clear the
        // mantissa and add one to the exponent.
        uint32_t bits = __float_as_uint(sc);
        if (bits & 0x007FFFFFu) bits = (bits & 0xFF800000u) + 0x00800000u;
        sc = __uint_as_float(bits);
    }
    const float r = __frcp_rn(sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = pack_e4m3x2(div_by_scale(f[4 * i], sc, r),
                                        div_by_scale(f[4 * i + 1], sc, r));
        const uint32_t hi = pack_e4m3x2(div_by_scale(f[4 * i + 2], sc, r),
                                        div_by_scale(f[4 * i + 3], sc, r));
        out[i] = lo | (hi << 16);
    }
    return sc;
}

}  // namespace
}  // namespace fp8bs
