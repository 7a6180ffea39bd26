/*
 * dqmoe.h — C ABI of the block-quantized GEMV / sparse-MoE library for one
 * GB300 GPU (sm_103a).
 *
 * What is computed.  Three offloading inference engines describe the same
 * data-parallel decode hot path: weight matrices stored as llama.cpp-style
 * quantized super-blocks (Q4_K, Q6_K, Q8_0) multiplied by activations, and a
 * sparse mixture-of-experts layer that activates a few experts per token.
 *   - Titan Engine: trillion-parameter inference on consumer hardware
 *     (zingnex.cn), sections "MoE 专家流式加载" (only 2 of 8 experts are
 *     active per forward pass) and "激进量化策略" (Q4_K weights).
 *   - KTransformers (news.fishai.com.cn/news/2715575), section "支持的量化格式"
 *     (Q4_K_M, Q6_K, Q8_0) and "技术原理" (sparse MoE matrices, CUDA Graph:
 *     one graph launch per decode step).
 *   - NTransformer, Show HN: Llama 3.1 70B on a single RTX 3090
 *     (hn.213312.xyz/article/47104667), section "量化支持" (Q4_0/Q8_0/Q4_K_M/
 *     Q5_K/Q6_K/F16/F32) and "核心性能" (decode speed follows resident bytes).
 * The pages name the formats but print no byte layout.  This library reads
 * them as the GGUF/llama.cpp layouts spelled out below (byte for byte).
 *
 * Conventions shared by every entry point.
 *   - Every pointer argument named "device" is a CUDA device pointer owned by
 *     the caller; the library never frees it and never keeps it after the call
 *     returns (calls are asynchronous on `stream`; the caller keeps buffers
 *     alive until the stream has passed the call).
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.  No entry point synchronises the stream or the device (except
 *     dq_moe_forward_streamed and dq_device_status, which say so), and no
 *     entry point allocates device memory: scratch is passed in by the
 *     caller.  The one exception is the library's own fixed scratch array of
 *     DQ_NOALLOC_SCRATCH_BYTES that dq_moe_forward_noalloc uses: it is
 *     resident on every GPU that loads the library, whether or not that entry
 *     point is called.
 *   - Return value: DQ_OK (0) or a negative dq_status.  Arguments are checked
 *     before anything is launched: on an argument error nothing is enqueued.
 *     DQ_ERR_CUDA means a launch reported an error (cudaGetLastError); the
 *     stream state is then whatever CUDA left it in.
 *   - No C++ exception crosses this boundary.  Kernels never trap: a device-
 *     side wait that runs past its time limit records DQ_ERR_DEVICE_TIMEOUT in
 *     a device status word (see dq_device_status) and returns.
 *
 * Layouts.
 *   - Quantized matrix W with N rows and K columns: row n is the K/QK blocks
 *     of that row, consecutive, starting at byte n * row_bytes where
 *     row_bytes = (K/QK) * block_bytes.  Rows are consecutive.  W must be
 *     16-byte aligned and row_bytes a multiple of 16 (true for every shape
 *     with K a multiple of 256 for Q4_K, Q8_0, Q4_0, Q5_K and NVFP4, of 1024
 *     for Q2_K, of 2048 for Q6_K and Q3_K).
 *   - Activations x: [batch][K] row-major in x_dtype.  Outputs y: [batch][N]
 *     row-major, always fp32 (MoE activations reach ~1e7, beyond fp16).
 */
#ifndef DQMOE_H
#define DQMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Block formats.                                                           */
/*                                                                          */
/* Q4_K super-block, 256 weights in 144 bytes:                              */
/*   bytes 0-1   d     fp16 super-block scale                               */
/*   bytes 2-3   dmin  fp16 super-block min scale                           */
/*   bytes 4-15  12 bytes holding eight 6-bit (sc_j, m_j) pairs, j = 0..7:  */
/*               j<4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63                 */
/*               j>=4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4)          */
/*                     m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)          */
/*   bytes 16-143 qs[128]: four 32-byte groups c = 0..3; byte l of group c  */
/*               holds weight 64c+l in its low nibble (sub-block 2c) and    */
/*               weight 64c+32+l in its high nibble (sub-block 2c+1).       */
/*   weight i of sub-block j: w = d*sc_j*q - dmin*m_j, q in [0,15].         */
/* Q6_K super-block, 256 weights in 210 bytes:                              */
/*   bytes 0-127 ql[128], 128-191 qh[64], 192-207 int8 scales[16],          */
/*   208-209 fp16 d.  Half h (0,1) uses ql[64h..], qh[32h..]; for l=0..31:  */
/*     weight 128h+l    : low nibble of ql[64h+l],    qh bits 0-1          */
/*     weight 128h+l+32 : low nibble of ql[64h+l+32], qh bits 2-3          */
/*     weight 128h+l+64 : high nibble of ql[64h+l],   qh bits 4-5          */
/*     weight 128h+l+96 : high nibble of ql[64h+l+32],qh bits 6-7          */
/*   (qh byte is qh[32h+l], its two bits are the high bits of the 6-bit q). */
/*   weight i: w = d * scales[i/16] * (q - 32), q in [0,63].                */
/* Q8_0 block, 32 weights in 34 bytes: fp16 d, int8 qs[32]; w = d*q.        */
/* Q4_0 block, 32 weights in 18 bytes: fp16 d, qs[16]; byte j holds weight j */
/*   in its low nibble and weight j+16 in its high nibble; w = d*(q - 8).   */
/* Q5_K super-block, 256 weights in 176 bytes:                              */
/*   bytes 0-15 as Q4_K (d, dmin, the 12 scale/min bytes), bytes 16-47      */
/*   qh[32], bytes 48-175 qs[128] as Q4_K's.  Weight 64c+l (c = 0..3,       */
/*   l = 0..31) takes the low nibble of qs[32c+l] plus bit 2c of qh[l] as   */
/*   bit 4; weight 64c+32+l the high nibble plus bit 2c+1.  q in [0,31];    */
/*   w = d*sc_j*q - dmin*m_j as Q4_K.  Both are the other GGUF blocks the   */
/*   [KTransformers, §支持的量化格式] list names beside Q4_K, Q6_K, Q8_0;    */
/*   dq_dequant and dq_qgemv take them, the MoE layer does not.             */
/* Q2_K super-block, 256 weights in 84 bytes:                               */
/*   bytes 0-15  scales[16]: low nibble = scale sc_j, high nibble = min m_j */
/*               of the sixteen 16-weight sub-blocks j                      */
/*   bytes 16-79 qs[64] of 2-bit quants, bytes 80-81 fp16 d, 82-83 fp16 dmin */
/*   weight 128h+32r+l (h = 0,1; r = 0..3; l = 0..31): bits 2r..2r+1 of     */
/*   qs[32h+l]; sub-block j = weight/16; w = d*sc_j*q - dmin*m_j, q in 0..3. */
/* Q3_K super-block, 256 weights in 110 bytes:                              */
/*   bytes 0-31 hmask[32], 32-95 qs[64] (2-bit low quants as Q2_K's),       */
/*   96-107 twelve bytes of sixteen 6-bit scales, 108-109 fp16 d.           */
/*   weight 128h+32r+l: low = bits 2r..2r+1 of qs[32h+l], high bit = bit    */
/*   4h+r of hmask[l]; q = low - 4 when the high bit is clear, else low     */
/*   (q in -4..3).  Scale j: bits 0-3 = nibble j/8 of byte j%8, bits 4-5 =  */
/*   bits 2(j/4)..2(j/4)+1 of byte 8 + j%4; w = d*(s_j - 32)*q.  Q2_K and   */
/*   Q3_K are the low-bit blocks of the [KTransformers, §支持的量化格式] list  */
/*   (Q2_K_L, Q2_K_XS, Q3_K_M mixes); dq_dequant and dq_qgemv take them, the */
/*   MoE layer does not.                                                    */
/* NVFP4 super-block, 256 weights in 144 bytes (the pages name NVIDIA's FP4 */
/*   as Blackwell's native 4-bit float, [Titan Engine, §激进量化策略], and    */
/*   print no layout; this is the library's):                               */
/*   bytes 0-15   E4M3 scales of the sixteen 16-weight blocks               */
/*   bytes 16-143 E2M1 codes, weight 2i in the low nibble of byte 16+i,     */
/*                weight 2i+1 in its high nibble                            */
/*   w = e2m1(code) * e4m3(scale[i/16]); a per-tensor scale, where a model  */
/*   has one, is the caller's (it commutes with the product).  NaN scale    */
/*   bytes are out of contract.  dq_dequant, dq_qgemv and MoE experts.      */
/* ------------------------------------------------------------------------ */
typedef enum { DQ_Q4_K = 1, DQ_Q6_K = 2, DQ_Q8_0 = 3, DQ_Q4_0 = 4, DQ_Q5_K = 5,
               DQ_NVFP4 = 6, DQ_Q2_K = 7, DQ_Q3_K = 8 } dq_fmt;

/* Activation element types accepted by the entry points. */
typedef enum { DQ_F32 = 0, DQ_F16 = 1, DQ_BF16 = 2 } dq_dtype;

typedef enum {
  DQ_OK = 0,
  DQ_ERR_ARG = -1,          /* null pointer, bad size, K not a multiple of QK, batch out of range */
  DQ_ERR_ALIGN = -2,        /* a pointer or a row stride is not 16-byte aligned */
  DQ_ERR_UNSUPPORTED = -3,  /* format / dtype / shape this build does not handle */
  DQ_ERR_WORKSPACE = -4,    /* workspace pointer null or smaller than dq_moe_workspace_size */
  DQ_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  DQ_ERR_DEVICE_TIMEOUT = -6 /* a kernel's bounded wait ran out (read via dq_device_status) */
} dq_status;

#define DQ_QK_K 256         /* weights per Q4_K / Q6_K super-block */
#define DQ_QK8_0 32         /* weights per Q8_0 block */
#define DQ_Q4_K_BYTES 144
#define DQ_Q6_K_BYTES 210
#define DQ_Q8_0_BYTES 34
#define DQ_QK4_0 32         /* weights per Q4_0 block */
#define DQ_Q4_0_BYTES 18
#define DQ_Q5_K_BYTES 176
#define DQ_NVFP4_BYTES 144  /* per 256-weight super-block */
#define DQ_Q2_K_BYTES 84
#define DQ_Q3_K_BYTES 110
#define DQ_MAX_BATCH 8      /* activation columns per dq_qgemv call */

/* Weights per block and bytes per block of `fmt`.  Host-only, no CUDA.
 * Returns DQ_ERR_ARG for an unknown format or null outputs. */
int dq_block_geometry(int fmt, int* weights_per_block, int* bytes_per_block);

/* dq_dequant — decode `n_weights` weights (a whole number of blocks) of format
 * `fmt` into fp32.  Step "block decode" of the path; exposed so the decoded
 * values can be compared bit for bit (every closed form above is exact in
 * fp32 up to the final rounding of the Q4_K subtraction).
 *   blocks : device, n_weights/QK consecutive blocks, 2-byte aligned (the
 *            Q6_K/Q8_0/Q4_0/Q3_K blocks are 210/34/18/110 B).
 *   out    : device fp32 [n_weights], 4-byte aligned.
 * Errors: DQ_ERR_ARG (null, n_weights <= 0 or not a multiple of QK),
 *         DQ_ERR_ALIGN, DQ_ERR_CUDA. */
int dq_dequant(int fmt, const void* blocks, int64_t n_weights, float* out,
               void* stream);

/* dq_qgemv — y[b][n] = sum_k W[n][k] * x[b][k] for b < batch, fp32 accumulate,
 * W decoded inside the kernel (never materialised).  The decode linear of the
 * engines above ([NTransformer, §核心性能]: decode rate is set by the bytes of
 * the resident quantized weights; [Titan Engine, §性能表现]).
 *   W      : device, N rows of K/QK blocks (layout above), 16-byte aligned.
 *   x      : device [batch][K] of x_dtype, 16-byte aligned.
 *   y      : device fp32 [batch][N], 4-byte aligned; fully overwritten.
 *   batch  : 1..DQ_MAX_BATCH.
 * fp16/bf16 activations run on the tensor-core path (weights decoded to fp16
 * in registers); fp32 activations run on an fp32 CUDA-core path (decode and
 * products in fp32).
 * Range of the 16-bit path: Q4_K, Q5_K, Q6_K, Q2_K and Q3_K rows, and Q8_0
 * at batch 1, are decoded in per-row or per-sub-block power-of-two units and
 * take any finite fp16 d and dmin.  Q8_0 and Q4_0 at batch 2..8 and NVFP4
 * decode to absolute fp16 weights: every decoded weight |w| must stay below
 * 65504 (Q8_0: |d| < 515; Q4_0: |d| < 8187; NVFP4 always holds, |w| <= 2688).
 * Beyond that the output is inf or NaN; the call cannot detect it. 
 * Errors: DQ_ERR_ARG (null, N/K <= 0, K % 256 != 0 — every format is
 *         streamed in 256-weight units —, batch outside 1..8),
 *         DQ_ERR_ALIGN (W, x not 16-B aligned, y not 4-B aligned; rows must
 *         stay 16-B aligned: Q2_K needs K % 1024 == 0 (84-byte blocks), Q6_K
 *         and Q3_K K % 2048 == 0 (210- and 110-byte blocks)),
 *         DQ_ERR_UNSUPPORTED (N > 65535*64), DQ_ERR_CUDA. */
int dq_qgemv(int fmt, const void* W, int64_t N, int64_t K, const void* x,
             int x_dtype, int batch, float* y, void* stream);

/* dq_qgemv with the K split chosen by the caller (tuning and tests): the 16-bit
 * activation path splits the K/256 super-blocks of every 64-row tile over a
 * thread-block cluster of `ksplit` CTAs (1..8, clamped to K/256) and sums the
 * partial results through distributed shared memory in a fixed order.
 * ksplit = 0 lets the library choose (what dq_qgemv does).  Ignored for fp32
 * activations.  Errors: as dq_qgemv, plus DQ_ERR_ARG for ksplit outside 0..8. */
int dq_qgemv_ksplit(int fmt, const void* W, int64_t N, int64_t K, const void* x,
                    int x_dtype, int batch, float* y, int ksplit, void* stream);

/* Flags of dq_qgemv_ex. */
#define DQ_QGEMV_WEIGHTS_EARLY 1u
/* dq_qgemv_ex — dq_qgemv with the K split (0 = library's choice, as
 * dq_qgemv_ksplit) and flags.
 *   DQ_QGEMV_WEIGHTS_EARLY: the caller guarantees that W is not written by
 *     the kernel issued just before this call on `stream` (weights are
 *     loaded once and stay read-only, as in decode).  The kernel then starts
 *     streaming its first weight stages while that kernel is still finishing
 *     (programmatic dependent launch), hiding the start-up latency of a chain
 *     of GEMVs.  x and y are still ordered after the previous kernel.
 *     Ignored for fp32 activations.
 * Every kernel of this library is launched as a programmatic dependent
 * launch: it may be scheduled while the previous kernel in the stream drains,
 * and waits for that kernel's completion before it reads any input other than
 * W under DQ_QGEMV_WEIGHTS_EARLY, or writes any output.
 * Errors: as dq_qgemv_ksplit, plus DQ_ERR_ARG for unknown flag bits. */
int dq_qgemv_ex(int fmt, const void* W, int64_t N, int64_t K, const void* x,
                int x_dtype, int batch, float* y, int ksplit, unsigned flags,
                void* stream);

/* ------------------------------------------------------------------------ */
/* Sparse MoE layer.                                                         */
/*   logits[t][e] = sum_h router_W[e][h] * x[t][h]            (fp32)         */
/*   sel(t)       = the top_k largest logits, lowest index first on ties     */
/*   gate[t][i]   = exp(l_i - l_max) / sum_{j in sel} exp(l_j - l_max)       */
/*                  (softmax over all E, renormalised over the selection)    */
/*   FFN_e(v)     = W_down_e * ( silu(W_gate_e v) (.) (W_up_e v) ),          */
/*                  silu(g) = g / (1 + exp(-g))                              */
/*   y[t]         = sum_i gate[t][i] * FFN_{sel_i}(x_t) + sum_s FFN_shared_s(x_t) */
/* [Titan Engine, §MoE 专家流式加载] (activate 2 of 8 experts per forward);  */
/* [KTransformers, §技术原理] (sparse MoE matrices).  The pages give no      */
/* router or FFN formula: softmax top-k renormalised with SwiGLU experts is */
/* the Mixtral / DeepSeek-V3 (plain softmax routing) reading.                */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t E;          /* routed experts, 1..256 */
  int32_t top_k;      /* experts per token, 1..min(E, 8) */
  int32_t hidden;     /* H: length of x rows, rows of W_down */
  int32_t ffn;        /* F: rows of W_gate / W_up, columns of W_down */
  int32_t n_shared;   /* always-on shared experts, 0..4, weight 1 each */
  int32_t fmt;        /* dq_fmt of every expert matrix: DQ_Q4_K, DQ_Q6_K,
                         DQ_Q8_0 or DQ_NVFP4 (others: DQ_ERR_UNSUPPORTED).
                         Range: experts with more than 32 tokens in a call
                         (the tensor-core GEMM) and Q8_0 experts on any path
                         decode to absolute fp16 weights, which must stay
                         below 65504 in magnitude (Q4_K: 945|d| + 63|dmin|,
                         Q6_K: 32|d||s|, Q8_0: 127|d|); beyond that the
                         output is inf or NaN, undetected. */
  const float* router_W; /* device fp32 [E][H] */
  const void* w_gate; /* device, E stacked [F rows][H/QK blocks] matrices */
  const void* w_up;   /* device, E stacked [F][H/QK] */
  const void* w_down; /* device, E stacked [H rows][F/QK blocks] */
  const void* sh_gate; /* device, n_shared stacked [F][H/QK]; NULL if n_shared == 0 */
  const void* sh_up;   /* device, n_shared stacked [F][H/QK] */
  const void* sh_down; /* device, n_shared stacked [H][F/QK] */
} dq_moe_desc;

/* Bytes of scratch dq_moe_forward needs for T tokens (host-only, no CUDA).
 * Errors: DQ_ERR_ARG on a malformed descriptor or T <= 0,
 *         DQ_ERR_UNSUPPORTED on shapes outside the limits above. */
int dq_moe_workspace_size(const dq_moe_desc* desc, int T, size_t* bytes);

/* dq_moe_router — steps "router" and "top-k + gates" alone.
 *   router_W : device fp32 [E][H];  x : device [T][H] of x_dtype; H % 32 == 0.
 *   logits   : device fp32 [T][E], required: the logits are summed there
 *              before the selection reads them (this entry point takes no
 *              workspace).
 *   topk_idx : device int32 [T][top_k], slot order = descending logit,
 *              lowest expert index first among equal logits.
 *   topk_gate: device fp32 [T][top_k], renormalised softmax weights.
 * Errors: DQ_ERR_ARG (a null pointer, H % 32 != 0, sizes <= 0, top_k > E),
 *         DQ_ERR_ALIGN (router_W, x, logits, topk_idx or topk_gate not 4-byte
 *         aligned), DQ_ERR_UNSUPPORTED (E > 256, top_k > 8 or T > 65536),
 *         DQ_ERR_CUDA. */
int dq_moe_router(const float* router_W, int E, int H, const void* x,
                  int x_dtype, int T, int top_k, float* logits,
                  int32_t* topk_idx, float* topk_gate, void* stream);

/* dq_moe_permute — step "token -> expert permute" alone.  The T*top_k
 * (token, slot) pairs p = t*top_k + slot are ordered by (expert, p):
 *   offsets : device int32 [E+1], offsets[e] = number of pairs routed to
 *             experts < e (exclusive prefix sum of the per-expert counts).
 *   sorted  : device int32 [T*top_k], the pair ids p in that order (stable).
 * Errors: DQ_ERR_ARG, DQ_ERR_UNSUPPORTED (E > 256, T*top_k > 65536),
 *         DQ_ERR_CUDA.  Expert ids outside [0, E) are out of contract. */
int dq_moe_permute(const int32_t* topk_idx, int T, int top_k, int E,
                   int32_t* offsets, int32_t* sorted, void* stream);

/* dq_moe_forward — the whole layer for T tokens (router, top-k, permute,
 * grouped gate/up with SwiGLU, grouped down, weighted combine + shared).
 *   x        : device [T][H] of x_dtype, 16-byte aligned; x_dtype DQ_F16 or
 *              DQ_BF16.  The experts multiply 16-bit tensor-core operands,
 *              which cannot meet the 1e-5 relative bar fp32 activations are
 *              held to, so DQ_F32 is refused (DQ_ERR_UNSUPPORTED); a caller
 *              with fp32 activations rounds them to bf16 first.
 *   y        : device fp32 [T][H], 16-byte aligned, fully overwritten.
 *   ws       : device scratch of at least dq_moe_workspace_size bytes,
 *              256-byte aligned; contents on entry are ignored.
 *   topk_idx, topk_gate, logits : optional device outputs as in
 *              dq_moe_router (NULL to skip).
 * The launches go on `stream` with no host synchronisation, so the layer is
 * capturable in one CUDA graph ([KTransformers, §技术原理]: one graph call
 * per decode step).  When experts with one token sit beside experts with
 * more (T > 1 and at most E/2 picks), the kernels of the larger groups run
 * on a second stream of the library's (highest priority), forked from
 * `stream` and joined back into it before the layer's last kernel, so the
 * call is ordered on `stream` exactly as one stream would be; the results do
 * not depend on it.  That stream (one per device and caller stream) is
 * created by the first such call made outside stream capture and kept until
 * the process exits; such a call captured on a stream that has not run one
 * outside capture stays on `stream`.
 * Errors: DQ_ERR_ARG, DQ_ERR_ALIGN (x, y not 16-byte aligned, ws not 256-byte
 *         aligned, an optional output not 4-byte aligned), DQ_ERR_UNSUPPORTED
 *         (also fp32 x), DQ_ERR_WORKSPACE, DQ_ERR_CUDA. */
int dq_moe_forward(const dq_moe_desc* desc, const void* x, int x_dtype, int T,
                   float* y, void* ws, size_t ws_bytes, int32_t* topk_idx,
                   float* topk_gate, float* logits, void* stream);

/* dq_moe_forward_noalloc — dq_moe_forward for callers that cannot allocate
 * device memory, so cannot provide the `ws` scratch buffer: code running
 * under a host framework that owns all device memory and gives no workspace
 * hook (plugins, custom-op shims), or decode loops that must not allocate on
 * the hot path.  The inference engines this library follows have no
 * counterpart; it exists for such callers only.
 * Scratch comes from one fixed array of DQ_NOALLOC_SCRATCH_BYTES (32 MiB)
 * inside the library: every GPU that loads the library keeps that much
 * device memory until the process exits.  No call allocates or frees memory,
 * and none creates the second stream dq_moe_forward may use: every launch
 * goes on `stream`.
 * The first call on a device (with that device current) looks up the array's
 * device address once (cudaGetSymbolAddress); make that first call before any
 * stream capture: a first call made while `stream` is capturing is refused
 * with DQ_ERR_UNSUPPORTED before anything is looked up or enqueued.  All calls on a device share the one array and each call
 * overwrites it, so calls that may overlap on the GPU (different streams
 * without ordering) race: order them.  Nothing needs to be zero on entry.
 * Arguments and outputs as dq_moe_forward (without ws / ws_bytes).
 * Errors: as dq_moe_forward; DQ_ERR_WORKSPACE when
 * dq_moe_workspace_size(desc, T) exceeds DQ_NOALLOC_SCRATCH_BYTES (decode-
 * sized T fits: e.g. 8 tokens of the 256-expert layer, 16 of the 8-expert one);
 * DQ_ERR_UNSUPPORTED for a first call on a device under stream capture;
 * DQ_ERR_CUDA if the array's address cannot be obtained. */
#define DQ_NOALLOC_SCRATCH_BYTES (32u << 20)
int dq_moe_forward_noalloc(const dq_moe_desc* desc, const void* x, int x_dtype, int T,
                           float* y, int32_t* topk_idx, float* topk_gate, float* logits,
                           void* stream);

/* ------------------------------------------------------------------------ */
/* Expert streaming: the routed experts in page-locked host memory, a device */
/* cache of expert slots ([Titan Engine, §MoE 专家流式加载]: experts loaded   */
/* on demand, an LRU cache of hot experts, asynchronous loads hiding the     */
/* transfer; [NTransformer, §核心技术] SLEP: a double-buffered pipeline that  */
/* overlaps transfers with GPU compute).                                     */
/*                                                                          */
/* Each dq_moe_forward_streamed call runs the router and top-k on `stream`,  */
/* reads the routing back (one host synchronisation of `stream`), keeps the  */
/* cache least-recently-used, copies the missing experts on `copy_stream` in */
/* up to phases-1 chunks (one cudaMemcpyAsync per matrix), and runs the      */
/* grouped expert kernels chunk by chunk on `stream`, each after its chunk's */
/* copies: the cached experts (and the shared ones) first, with no wait.     */
/* It keeps every expert on the grouped mma.sync kernel (dq_moe_forward runs */
/* one-token experts on the block-diagonal kernel and experts with more than */
/* 32 tokens on the tensor-core GEMM), so the two agree within the layer's   */
/* tolerance, not bit for bit.  Not capturable in a CUDA graph (the host     */
/* reads the routing).  A cache is used by one host thread at a time.        */
/* ------------------------------------------------------------------------ */
typedef struct dq_expert_cache dq_expert_cache;

/* dq_expert_cache_create
 *   host_experts : a descriptor as for dq_moe_forward, except that w_gate,
 *                  w_up and w_down point to page-locked host memory holding
 *                  all E experts (same stacked layout; 16-byte aligned);
 *                  router_W and the shared experts are device memory.
 *   slots        : experts the device cache holds, at least
 *                  min(E, max_tokens * top_k).
 *   slot_gate, slot_up : device, slots * ffn rows each (one expert's
 *                  gate / up matrix per slot); slot_down: slots * hidden
 *                  rows.  16-byte aligned, owned by the caller, kept until
 *                  the cache is destroyed.
 *   max_tokens   : the largest T of a call (1..65536).
 *   phases       : 1..8 copy/compute chunks per call (1: all copies first).
 *   *cache       : receives the handle.
 * Allocates host memory (page-locked staging, events), no device memory.
 * Errors: DQ_ERR_ARG (including host expert memory that is not page-locked),
 *         DQ_ERR_ALIGN, DQ_ERR_UNSUPPORTED, DQ_ERR_CUDA. */
int dq_expert_cache_create(const dq_moe_desc* host_experts, int slots, void* slot_gate,
                           void* slot_up, void* slot_down, int max_tokens, int phases,
                           dq_expert_cache** cache);

/* Bytes of device scratch dq_moe_forward_streamed needs for T tokens. */
int dq_expert_cache_workspace_size(const dq_expert_cache* cache, int T, size_t* bytes);

/* dq_moe_forward_streamed — the layer for T <= max_tokens tokens.
 *   x, y, x_dtype, ws, ws_bytes : as dq_moe_forward (ws of at least
 *                  dq_expert_cache_workspace_size bytes, 256-byte aligned).
 *   stream       : compute stream; copy_stream: the copies (a different
 *                  stream; NULL is the legacy default stream).
 * Returns once the work is enqueued (after the routing read-back).
 * Errors: DQ_ERR_ARG, DQ_ERR_ALIGN, DQ_ERR_UNSUPPORTED (fp32 x, as
 *         dq_moe_forward), DQ_ERR_WORKSPACE, DQ_ERR_CUDA. */
int dq_moe_forward_streamed(dq_expert_cache* cache, const void* x, int x_dtype, int T, float* y,
                            void* ws, size_t ws_bytes, void* stream, void* copy_stream);

/* Cumulative counts: experts found in the cache, experts copied, bytes copied. */
int dq_expert_cache_stats(const dq_expert_cache* cache, long long* hits, long long* misses,
                          long long* bytes_copied);

/* Releases the host resources of the cache (not the caller's slot buffers). */
int dq_expert_cache_destroy(dq_expert_cache* cache);

/* dq_stage — copy `bytes` from src to dst with a kernel launched like every
 * other kernel of this library (programmatic dependent launch on `stream`):
 * for moving a decode step's activations in from page-locked host memory and
 * its outputs back out without leaving the chain of launches, so that the
 * GEMV after the copy is scheduled while the copy drains (a copy-engine copy
 * between two kernels ends that chain).  The pages do not describe this call;
 * it serves the host-buffer decode loop ([KTransformers, §技术原理]: one
 * graph launch per decode step) and the benchmark's end-to-end measurement.
 *   dst, src : device memory or page-locked (mapped) host memory the GPU can
 *              address, 16-byte aligned, not overlapping.
 *   bytes    : a positive multiple of 16.
 * The copy waits for the kernel before it on `stream` (its source may be that
 * kernel's output) and is asynchronous like every call.
 * Errors: DQ_ERR_ARG (null pointer, bytes <= 0, overlapping ranges),
 *         DQ_ERR_ALIGN (pointers or size not 16-byte multiples), DQ_ERR_CUDA. */
int dq_stage(void* dst, const void* src, int64_t bytes, void* stream);

/* Human-readable name of a dq_status value (static string, never NULL). */
const char* dq_status_string(int status);

/* Reads and clears the device status word of the current device: DQ_OK, or
 * DQ_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait since the last
 * read.  Synchronous (waits for the device).  Errors: DQ_ERR_ARG, DQ_ERR_CUDA. */
int dq_device_status(int* status);

#ifdef __cplusplus
}
#endif

#endif /* DQMOE_H */
