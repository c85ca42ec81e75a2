/*
 * oracle.h -- plain, single-threaded CPU oracle for the FP8 block-scaled linear path
 * (act_quant, weight_dequant, fp8_gemm) described for the DeepSeek-V3 inference demo.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or call this
 * code: it exists so that tests, the smoke check and the benchmark's CPU-baseline leg can
 * check the CUDA library against an implementation that shares no code with it.
 *
 * Sources (page title, section):
 *   "DeepSeek-V3 Administrator & Developer Guide", §8.5.1 act_quant_kernel,
 *     §8.5.2 weight_dequant_kernel, §8.5.3 fp8_gemm_kernel, §6.3 The FP8 path;
 *   "DeepSeek-V3 User Guide", FAQ "What is scale_fmt: ue8m0?", and troubleshooting
 *     "Last dimension size must be divisible by block_size";
 *   codevetter "deepseek-ai/DeepSeek-V3" overview, System map (FP8 quantization data flow).
 *
 * Every floating-point result is formed in binary64 and rounded once where the method
 * rounds (to binary32, bf16 or e4m3). All layouts are row-major and contiguous.
 */
#ifndef FP8BS_ORACLE_H
#define FP8BS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_BLOCK 128          /* quantisation block along K (1x128 act, 128x128 weight) */
#define ORACLE_SCALE_FP32 0       /* s = max(amax, 1e-4) / 448 */
#define ORACLE_SCALE_UE8M0 1      /* s rounded up to a power of two */

/* e4m3fn codec: value of a code (NaN for 0x7F/0xFF) and the RNE, saturating encoder. */
double oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e4m3_encode(float v);

/* bf16 <-> binary32 (bf16 passed as its 16-bit pattern). */
float oracle_bf16_to_float(uint16_t h);
uint16_t oracle_bf16_rne(float f);

/* One IEEE binary32 division a/b (correctly rounded), formed in binary64. */
float oracle_f32_div(float a, float b);

/* act_quant: x bf16 [M,K] -> y e4m3 codes [M,K], s fp32 [M,K/128]. K % 128 == 0. */
void oracle_act_quant(const uint16_t* x, uint8_t* y, float* s, int64_t M, int64_t K,
                      int scale_fmt);

/* weight_dequant: w e4m3 [N,K], s fp32 [ceil(N/128), ceil(K/128)] -> y bf16 [N,K]. */
void oracle_weight_dequant(const uint8_t* w, const float* s, uint16_t* y, int64_t N,
                           int64_t K);

/* fp8_gemm: C[M,N] = sum_kb a_s[m,kb] b_s[n/128,kb] sum_{k in kb} A[m,k] B[n,k], in binary64.
   a e4m3 [M,K], a_s fp32 [M,K/128], b e4m3 [N,K], b_s fp32 [ceil(N/128),K/128]. */
void oracle_gemm(const uint8_t* a, const float* a_s, const uint8_t* b, const float* b_s,
                 double* c, int64_t M, int64_t N, int64_t K);

/* The same sum for `count` chosen output elements (rows mi[i], columns ni[i]). */
void oracle_gemm_at(const uint8_t* a, const float* a_s, const uint8_t* b, const float* b_s,
                    const int64_t* mi, const int64_t* ni, int64_t count, double* out,
                    int64_t M, int64_t N, int64_t K);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_ORACLE_H */
