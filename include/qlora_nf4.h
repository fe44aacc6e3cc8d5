/*
 * qlora_nf4.h -- C ABI of the B300 (sm_103a) QLoRA NF4 library.
 *
 * The hot path of QLoRA over NF4 4-bit weights, as the method's pages state it:
 *
 *   nf4_quantize / nf4_dequantize
 *       Blockwise NF4: every 64 consecutive elements share one absmax; each
 *       element is divided by it and replaced by the index of the nearest of
 *       16 normal-quantile levels with an exact zero; two indices are packed
 *       per byte; the absmax constants are quantised a second time ("double
 *       quantisation").  Sources: "QLoRA technical analysis" (xdnf.cn) §2.1
 *       (absmax normalisation and argmin search), "QLoRA paper summary"
 *       (blog.csdn.net, QLoRA论文概述: NF4 from normal quantiles, double
 *       quantisation), "PEFT course notes" (demo.tomabc.com) §4.2.
 *
 *   qlora_linear_fwd
 *       Y = X deq(Q)^T + (alpha/r) (X A^T) B^T with W in R^{d x k},
 *       B in R^{d x r}, A in R^{r x k} ("PEFT course notes" §2.2: h = Wx + BAx;
 *       "PEFT quantization guide" (huggingface docs, 量化): bf16 compute dtype).
 *
 *   qlora_linear_bwd_dx
 *       dX = dY deq(Q) + (alpha/r) (dY B) A: the gradient flowing through the
 *       frozen 4-bit weight into the inputs ("QLoRA paper summary", abstract).
 *
 *   qlora_linear_bwd_lora
 *       dA = (alpha/r) (dY B)^T X and dB = (alpha/r) dY^T (X A^T): the
 *       gradients that reach the trainable adapter ("QLoRA paper summary",
 *       abstract: back-propagation through the frozen 4-bit weight into LoRA).
 *
 *   qlora_linear_fwd_f32 / qlora_linear_bwd_dx_f32
 *       the layer with fp32 compute dtype (bnb_4bit_compute_dtype = float32:
 *       "LoftQ explainer" §3.2 and its troubleshooting table).
 *
 *   loftq_init
 *       T alternations of Q_t = NF4(W - s B A) and a rank-r approximation of
 *       W - deq(Q_t) ("LoftQ explainer" (mhpn.cn) §2.2 objective, §2.3 algorithm).
 *
 *   loftq_replace_lora
 *       one LoftQ step that keeps the caller's quantised weight and only
 *       replaces the adapter ("PEFT quantization guide", replace_lora_weights_loftq).
 *
 *   nf4_merge_lora
 *       merge (or unmerge) an adapter into the quantised weight: dequantise,
 *       add (subtract) s B A, quantise again ("PEFT quantization guide",
 *       merging adapters into quantised weights).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: the caller owns every buffer.  Pointers documented "device" must
 *   be device (or managed) memory on the current CUDA device and 16-byte
 *   aligned; pointers documented "host" are ordinary host memory.  The library
 *   allocates no device memory; scratch space is the caller's workspace `ws`
 *   of at least qn_workspace_bytes(...) bytes (device, 256-byte aligned).
 *   The first 256 KiB of a workspace are a zero area (semaphores and
 *   accumulators for grid-wide hand-offs): zero them once when the
 *   workspace is allocated; every call leaves them zero again when its
 *   kernels finish.  qn_workspace_bytes() includes them.
 * - Layout: matrices are row-major.  W (d x k) element (i, j) is at i*k + j;
 *   its flat element index e = i*k + j is what the 64-element blocks run over.
 * - bf16 buffers are passed as `uint16_t *` holding IEEE bfloat16 bit patterns.
 * - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *   call only enqueues work on it and returns, except loftq_init, which
 *   synchronises the stream once per alternation to report residuals.
 * - Errors: argument errors return before anything is enqueued and leave
 *   outputs untouched.  A failed launch returns QN_ECUDA.  Kernels never trap:
 *   a bounded wait that expires records QN_ETIMEOUT in a device status word
 *   that qn_device_status() reads.  qn_last_error() gives a message for the
 *   calling thread's last non-OK status.
 */
#ifndef QLORA_NF4_H
#define QLORA_NF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QN_ABI_VERSION 2

typedef enum {
  QN_OK = 0,
  QN_EINVAL = 1,       /* null pointer, bad enum, non-finite alpha ...        */
  QN_ESHAPE = 2,       /* sizes out of range or inconsistent                  */
  QN_EALIGN = 3,       /* pointer not 16-byte aligned                          */
  QN_ENOMEM = 4,       /* workspace smaller than qn_workspace_bytes()          */
  QN_ECUDA = 5,        /* a CUDA runtime call or kernel launch failed          */
  QN_ETIMEOUT = 6,     /* a bounded device-side wait expired                   */
  QN_EUNSUPPORTED = 7  /* valid request this build does not implement          */
} qn_status;

typedef enum { QN_F32 = 0, QN_BF16 = 1 } qn_dtype;

typedef enum {
  QN_OP_QUANTIZE = 0,
  QN_OP_DEQUANTIZE = 1,
  QN_OP_LINEAR_FWD = 2,
  QN_OP_LINEAR_BWD_DX = 3,
  QN_OP_LOFTQ = 4,            /* loftq_init and loftq_replace_lora */
  QN_OP_LINEAR_BWD_LORA = 5,
  QN_OP_LINEAR_F32 = 6,       /* qlora_linear_fwd_f32 and qlora_linear_bwd_dx_f32 */
  QN_OP_MERGE = 7
} qn_op;

/*
 * Quantised state of one tensor of n = d*k elements (all pointers device,
 * caller-owned).  Block size 64 and double-quantisation group 256 are the only
 * supported values.
 *   codes        uint8[ceil(n/2)]  element 2q in the low nibble of byte q,
 *                                  element 2q+1 in the high nibble; an unused
 *                                  high nibble (odd n) is 0.
 *   absmax       fp32[nblk]        exact block absmax, nblk = ceil(n/64).
 *                                  Always written by nf4_quantize; read by the
 *                                  dequantiser only when dq == 0.
 *   absmax_q     int8[nblk]        (dq) int8 code of absmax - mean.
 *   absmax_scale fp32[ngrp]        (dq) per-256-block scale, ngrp = ceil(nblk/256).
 *   absmax_mean  fp32[1]           (dq) exact mean of absmax rounded to fp32.
 */
typedef struct {
  int64_t d;
  int64_t k;
  int32_t block;     /* must be 64                     */
  int32_t dq;        /* 1 = double-quantised constants */
  int32_t dq_block;  /* must be 256                    */
  int32_t reserved;
  uint8_t *codes;
  float *absmax;
  int8_t *absmax_q;
  float *absmax_scale;
  float *absmax_mean;
} qn_nf4;

/* ABI version of the loaded library (QN_ABI_VERSION at build time). */
int qn_abi_version(void);

/* Message for the calling thread's last non-OK status ("" if none). */
const char *qn_last_error(void);

/*
 * Host copies of the constant tables the kernels use: the 16 NF4 levels
 * (ascending) and the 15 fp32 decision thresholds t_i, where t_i is the
 * largest fp32 not above the exact midpoint (c_i + c_{i+1}) / 2, so that
 * code(v) = #{ i : v > t_i } is the nearest level with ties to the lower
 * index.  Either pointer may be NULL.
 */
void qn_nf4_tables(float codebook[16], float thresholds[15]);

/*
 * Workspace bytes the call `op` needs for the given sizes (0 if none).
 * M: rows of X / dY; d, k: W is d x k; r: LoRA rank (LoftQ: sized for the
 * largest r + oversample it accepts).
 */
size_t qn_workspace_bytes(qn_op op, int64_t M, int64_t d, int64_t k, int32_t r);

/*
 * nf4_quantize -- blockwise NF4 quantisation of W (d x k, flat n = d*k).
 *   W      device, n elements of dtype wdt (QN_F32 or QN_BF16).
 *   Q      host struct; Q->d, Q->k, Q->block (64), Q->dq, Q->dq_block (256)
 *          and its device output pointers must be set (absmax_q, absmax_scale,
 *          absmax_mean may be NULL when dq == 0).
 *   ws     device workspace of ws_bytes >= qn_workspace_bytes(QN_OP_QUANTIZE,..)
 * Per block j: m_j = max |x|; codes = nearest level of fp32(x / m_j) (IEEE
 * division; a block with m_j = 0 gets code 7, the exact zero).  With dq:
 * mu = nearest fp32 to the exact mean of all m_j; per group g of 256 blocks
 * sigma_g = fp32(max_j |fp32(m_j - mu)| / 127) and
 * q_j = clamp(rint_half_even(fp32(fp32(m_j - mu) / sigma_g)), -127, 127)
 * (q_j = 0 when sigma_g = 0).  Results are bit-identical for any launch shape.
 */
qn_status nf4_quantize(const void *W, qn_dtype wdt, const qn_nf4 *Q,
                       void *ws, size_t ws_bytes, void *stream);

/*
 * nf4_dequantize -- W'[e] = fp32(c[code_e] * m'_{block(e)}), written as fp32
 * or rounded to bf16 (nearest even).  m' = fp32(fp32(q_j * sigma_g) + mu) when
 * Q->dq, else the exact absmax.  Wout: device, n elements of dtype odt.
 */
qn_status nf4_dequantize(const qn_nf4 *Q, void *Wout, qn_dtype odt, void *stream);

/*
 * qlora_linear_fwd -- Y = X deq(Q)^T + (alpha/r) (X A^T) B^T.
 *   Q     quantised weight, d x k with k % 64 == 0.
 *   X     device bf16 [M x k];  A device bf16 [r x k];  B device bf16 [d x r].
 *   Y     device bf16 [M x d] (written).
 *   1 <= M, 1 <= r <= 256.  Accumulation is fp32.  The tensor-core paths
 *   multiply the NF4 levels (or bf16(deq(Q)) for M > 16) by bf16 X; the
 *   adapter term keeps about 16 significant bits of u = s X A^T.
 *   Paths: M <= 8 with M * k <= 16384 (and the per-CTA limits of that
 *   kernel) -- one persistent kernel; other M <= 16 -- the few-token
 *   kernels; M > 16 and r <= 64 -- the tcgen05 GEMM, whose workspace also
 *   holds the bf16 hi/lo split of u (M x 128) and the fp32 block constants
 *   of W (d x 2*ceil(k/128)).  ws: qn_workspace_bytes(QN_OP_LINEAR_FWD).
 *   Stream order: the M <= 16 kernels are launched as programmatic
 *   dependents of the kernel before them (they start early and wait for it
 *   with griddepcontrol.wait before reading any operand), so the call may
 *   directly follow the kernel that writes X, Q, A or B.
 *   The persistent kernel hands u between its CTAs through the workspace
 *   counters; if that hand-off times out (all CTAs could not be resident,
 *   e.g. other work filled the GPU for seconds) Y is wrong and the next
 *   qn_device_status() returns QN_ETIMEOUT: results are valid once
 *   qn_device_status() has returned QN_OK.
 */
qn_status qlora_linear_fwd(const qn_nf4 *Q, const uint16_t *X, int64_t M,
                           const uint16_t *A, const uint16_t *B, int32_t r,
                           float alpha, uint16_t *Y,
                           void *ws, size_t ws_bytes, void *stream);

/*
 * qlora_linear_fwd_group -- several projections of one input in one call:
 *   Y[g] = X deq(Q[g])^T + (alpha[g]/r[g]) (X A[g]^T) B[g]^T,  g < n,
 * the layer of "PEFT course notes" §2.2 applied to a shared activation (the
 * query/key/value or gate/up projections of a transformer block).
 *   n      1..8 projections; Q, A, B, r, alpha, Y are host arrays of n entries
 *          (each as in qlora_linear_fwd); every Q[g] has the same k.
 *   X      device bf16 [M x k], shared.
 *   ws     qn_workspace_bytes(QN_OP_LINEAR_FWD, M, sum of d, k, sum of r).
 * With M <= 16 (and k <= 16384) the group runs as one launch sequence whose
 * memory round trips overlap across projections; otherwise it is the n
 * single calls in order.  Results equal those of n qlora_linear_fwd calls
 * up to fp32 summation order.
 */
qn_status qlora_linear_fwd_group(int32_t n, const qn_nf4 *const *Q, const uint16_t *X, int64_t M,
                                 const uint16_t *const *A, const uint16_t *const *B, const int32_t *r,
                                 const float *alpha, uint16_t *const *Y,
                                 void *ws, size_t ws_bytes, void *stream);

/*
 * qlora_linear_bwd_dx -- dX = dY deq(Q) + (alpha/r) (dY B) A.
 *   dY device bf16 [M x d]; A, B as in the forward; dX device bf16 [M x k].
 *   Same size rules and workspace query (QN_OP_LINEAR_BWD_DX); for M > 16,
 *   r <= 64 and d % 8 == 0 the workspace also holds bf16 W^T (k x d), the
 *   bf16 hi/lo split of v = (alpha/r) dY B (M x 128) and [A^T | A^T]
 *   (k x 128 bf16) for the tensor-core GEMM.
 */
qn_status qlora_linear_bwd_dx(const qn_nf4 *Q, const uint16_t *dY, int64_t M,
                              const uint16_t *A, const uint16_t *B, int32_t r,
                              float alpha, uint16_t *dX,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * loftq_init -- LoftQ initialisation of one fp32 matrix W (d x k, device).
 *   For t = 1..T: Q_t = NF4(W - s B_{t-1} A_{t-1}) (B_0 A_0 = 0, s = alpha/r);
 *   R_t = W - deq(Q_t); the rank-r part of R_t by randomised subspace
 *   iteration (oversample columns, power_iters passes, Gaussian test matrix
 *   from `seed`); B_t = U_r sqrt(S_r)/sqrt(s), A_t = sqrt(S_r) V_r^T/sqrt(s).
 *   Outputs: Q (as nf4_quantize, holding Q_T; Q_0 = NF4(W) when T == 0),
 *   A device fp32 [r x k], B device fp32 [d x r],
 *   resid host fp64[T+1]: resid[t] = ||W - deq(Q_t) - s B_t A_t||_F, with
 *   resid[0] the plain QLoRA residual ||W - deq(NF4(W))||_F.
 *   1 <= r, r + oversample <= 96, 0 <= T <= 64, d, k multiples of 64 and >= r + oversample.
 *   Block size 64 and the DQ setting are taken from Q (Q->dq); the rank-r
 *   step is always the randomised one.
 */
qn_status loftq_init(const float *W, int64_t d, int64_t k, int32_t r, float alpha,
                     int32_t T, uint64_t seed, int32_t oversample, int32_t power_iters,
                     const qn_nf4 *Q, float *A, float *B, double *resid,
                     void *ws, size_t ws_bytes, void *stream);

/*
 * loftq_replace_lora -- one LoftQ step against the caller's quantised weight.
 *   W     device fp32 [Q->d x Q->k], the unquantised reference weight.
 *   Q     the quantised weight (input only: it is not requantised).
 *   A, B  device fp32 [r x k], [d x r] (written): B A s is the rank-r
 *         approximation of R = W - deq(Q) (randomised subspace iteration as
 *         in loftq_init, with `seed`, `oversample`, `power_iters`);
 *         B = U_r sqrt(S_r)/sqrt(s), A = sqrt(S_r) V_r^T/sqrt(s), s = alpha/r.
 *   resid host fp64[2]: ||R||_F and ||R - s B A||_F.
 *   Sizes, limits and workspace as loftq_init (qn_workspace_bytes(QN_OP_LOFTQ)).
 */
qn_status loftq_replace_lora(const float *W, const qn_nf4 *Q, int32_t r, float alpha, uint64_t seed,
                             int32_t oversample, int32_t power_iters, float *A, float *B, double *resid,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * qlora_linear_bwd_lora -- gradients of the adapter factors for dL/dY = dY:
 *   dA = s (dY B)^T X   (r x k),   dB = s dY^T (X A^T)   (d x r),   s = alpha/r.
 *   X  device bf16 [M x k];  dY device bf16 [M x d];  A bf16 [r x k];  B bf16 [d x r].
 *   dA, dB device fp32 (written).  1 <= M, d, k;  1 <= r <= 256.
 *   The token contractions run on the tensor cores with X A^T and dY B kept
 *   as bf16 hi + lo (about 16 significant bits), fp32 accumulation, and a
 *   fixed summation order (results do not depend on the launch).
 *   ws: qn_workspace_bytes(QN_OP_LINEAR_BWD_LORA, M, d, k, r).
 */
qn_status qlora_linear_bwd_lora(const uint16_t *X, const uint16_t *dY, int64_t M, int64_t d, int64_t k,
                                const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                                float *dA, float *dB, void *ws, size_t ws_bytes, void *stream);

/*
 * qlora_linear_fwd_f32 / qlora_linear_bwd_dx_f32 -- the layer with fp32
 * compute dtype: X, A, B, Y (dY, dX) are device fp32 with the shapes of
 * qlora_linear_fwd / qlora_linear_bwd_dx, and the weight enters as its exact
 * fp32 dequantisation (the value nf4_dequantize writes).  fp32 FMA on the
 * CUDA cores, fp32 accumulation.  Size rules as the bf16 calls; ws:
 * qn_workspace_bytes(QN_OP_LINEAR_F32, M, d, k, r) (the M x r projection).
 */
qn_status qlora_linear_fwd_f32(const qn_nf4 *Q, const float *X, int64_t M, const float *A, const float *B,
                               int32_t r, float alpha, float *Y, void *ws, size_t ws_bytes, void *stream);
qn_status qlora_linear_bwd_dx_f32(const qn_nf4 *Q, const float *dY, int64_t M, const float *A, const float *B,
                                  int32_t r, float alpha, float *dX, void *ws, size_t ws_bytes, void *stream);

/*
 * nf4_merge_lora -- Qout = NF4(deq(Q) + sign * s * B A), s = alpha / r;
 * sign = +1 merges the adapter, -1 unmerges it.  Because the result is
 * quantised again, unmerge(merge(Q)) is not Q in general.
 *   Q     input quantised weight, d x k with k % 64 == 0.
 *   A, B  device bf16 [r x k], [d x r], 1 <= r <= 256.
 *   Qout  output state with Q's shape (its own dq setting); Qout == Q
 *         (the same buffers) merges in place.
 *   The adapter product is summed in fp32 in ascending rank order (each
 *   bf16 x bf16 term is exact), t = fp32(s * sum), w = fp32(deq +- t), then
 *   quantised exactly as nf4_quantize does (bit-identical to quantising
 *   that fp32 tensor).  ws: qn_workspace_bytes(QN_OP_MERGE) (needed when
 *   Qout->dq).
 */
qn_status nf4_merge_lora(const qn_nf4 *Q, const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                         int32_t sign, const qn_nf4 *Qout, void *ws, size_t ws_bytes, void *stream);

/*
 * nf4_quantize_noalloc -- nf4_quantize without a caller workspace.  The
 * method's pages have no counterpart to this entry point: it exists for
 * callers that cannot call cudaMalloc (code running while another allocator
 * owns the free device memory, or loops that cannot afford the device-wide
 * synchronisation an allocation implies).  Arguments, results and errors are
 * those of nf4_quantize; the 2.25 KiB of scratch the double-quantisation mean
 * needs is a static device array inside the library, which every GPU that
 * loads the library keeps until the process exits.
 *   - The first call on each device looks up that array's device address
 *     (cudaGetSymbolAddress) with the device current; make that first call
 *     before any stream capture.
 *   - The call clears the scratch itself on `stream` before using it.
 *   - All calls share the one array: calls that overlap on the GPU (on
 *     different streams, or from different host threads) race and may
 *     return wrong constants.  Serialise them.
 *   - Tensors above 2^40 elements are rejected with QN_ESHAPE.
 *   - No device memory is allocated or freed.
 */
qn_status nf4_quantize_noalloc(const void *W, qn_dtype wdt, const qn_nf4 *Q, void *stream);

/*
 * Synchronises `stream`, then reads and clears the device status word that
 * bounded waits write.  Returns QN_OK, QN_ETIMEOUT, or QN_ECUDA.
 */
qn_status qn_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_NF4_H */
