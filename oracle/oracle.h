/*
 * oracle.h — plain, slow CPU reference for the block-quantized GEMV and the
 * sparse MoE layer.  TEST INFRASTRUCTURE ONLY: the parity tests, the smoke
 * check and the benchmark's CPU baseline call it; the library never does.
 * It shares no code, header, table or constant with the CUDA library: every
 * format constant below is restated here on purpose.
 *
 * Everything is computed from the plain definitions, in double, and rounded
 * to the output type once.  Sources (the pages name the formats and the MoE
 * structure; the byte layouts are the GGUF/llama.cpp reading):
 *   [Titan Engine, §激进量化策略]  Q4_K weights
 *   [Titan Engine, §MoE 专家流式加载]  sparse activation, 2 of 8 experts
 *   [KTransformers, §支持的量化格式]  Q4_K_M / Q6_K / Q8_0
 *   [NTransformer (Show HN), §量化支持]  Q8_0 / Q4_K_M / Q6_K
 *   [KTransformers, §支持的量化格式]  Q4_0 / Q5_K / Q2_K / Q3_K (the other GGUF
 *                                    blocks the page lists)
 *   [Titan Engine, §激进量化策略 / §模型格式支持]  NVIDIA FP4 (Blackwell's
 *       native 4-bit float): E2M1 values with E4M3 scales per 16 weights
 *
 * All functions return 0 on success, -1 on a bad argument.
 */
#ifndef DQ_ORACLE_H
#define DQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* format ids and activation dtype ids, same numbering as the public ABI but
 * declared independently */
enum { OR_Q4_K = 1, OR_Q6_K = 2, OR_Q8_0 = 3, OR_Q4_0 = 4, OR_Q5_K = 5, OR_NVFP4 = 6,
       OR_Q2_K = 7, OR_Q3_K = 8 };
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* weights per block / bytes per block */
int or_geometry(int fmt, int* qk, int* bytes);

/* decode n weights (whole blocks) to fp32 */
int or_dequant(int fmt, const uint8_t* blocks, int64_t n, float* out);

/* activation element -> double (exact) for the three dtypes */
int or_act_to_f64(int dtype, const void* x, int64_t n, double* out);

/* y[b][r] for the rows in `rows` (or all N rows if rows == NULL):
 * y = sum_k W[row][k] * x[b][k] in double, rounded to fp32 once.
 * y is [batch][nrows] (nrows = N when rows == NULL). nthreads >= 1. */
int or_qgemv(int fmt, const uint8_t* W, int64_t N, int64_t K, const void* x,
             int xdt, int batch, const int64_t* rows, int64_t nrows, float* y,
             int nthreads);

/* logits[t][e] = sum_h Wr[e][h] * x[t][h], in double */
int or_router_logits(const float* Wr, int E, int H, const void* x, int xdt,
                     int T, double* logits, int nthreads);

/* top-k by a full stable sort on (-logit, index); gates = softmax over the
 * selected logits (== full softmax renormalised over the selection) */
int or_topk(const double* logits, int T, int E, int k, int32_t* idx,
            double* gate);

/* stable counting permute of the T*k pairs p = t*k + slot by expert */
int or_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
               int32_t* offsets, int32_t* sorted);

/* silu(g) = g / (1 + exp(-g)) in double */
double or_silu(double g);

/* FFN of one expert on one activation vector (double in, double out):
 * out[H] = Wd * (silu(Wg v) * (Wu v)); Wg, Wu are [F][H], Wd is [H][F]. */
int or_expert_ffn(int fmt, const uint8_t* Wg, const uint8_t* Wu,
                  const uint8_t* Wd, int H, int F, const double* v,
                  double* out);

/* The whole MoE layer for the tokens listed in `tokens` (all T if NULL):
 *   y[i][H] (fp32, rounded once) for token tokens[i];
 *   idx[T][k], gate[T][k], logits[T][E] for all T tokens (nullable).
 * Expert matrices are stacked [E][rows][blocks] as in the public ABI. */
int or_moe_forward(int fmt, int E, int k, int H, int F, int n_shared,
                   const float* Wr, const uint8_t* w_gate,
                   const uint8_t* w_up, const uint8_t* w_down,
                   const uint8_t* sh_gate, const uint8_t* sh_up,
                   const uint8_t* sh_down, const void* x, int xdt, int T,
                   const int32_t* tokens, int ntokens, float* y, int32_t* idx,
                   double* gate, double* logits, int nthreads);

#ifdef __cplusplus
}
#endif

#endif
