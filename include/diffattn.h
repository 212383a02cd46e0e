/*
 * diffattn.h -- C ABI of the differential-attention forward for NVIDIA GB300
 * (sm_103a).
 *
 * The operation (paperleet "Differential Transformer Attention", Formula and
 * conventions; aifetchly "Differential Transformer: Canceling LLM Attention
 * Noise", section 1):
 *
 *     A_b = softmax(Q_b K_b^T / sqrt(D) + M)      b = 1, 2, softmax over keys
 *     O   = (A_1 - lambda * A_2) V
 *
 * with Q1, K1, Q2, K2 of shape [B, H, T, D], V and O of shape [B, H, T, 2D],
 * and M the optional causal mask: 0 where key j <= query i, -inf where
 * j > i, applied to both branches.  The scalar lambda comes from four
 * parameter vectors (aifetchly, section 3; paperleet, Formula and conventions):
 *
 *     lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
 *
 * It is not restricted to [0, 1].  Per-head normalisation, its fixed
 * (1 - lambda_init) multiplier and the projections are not part of this
 * operation.
 *
 * Conventions shared by every entry point:
 *   - Return value: DIFFATTN_OK (0) on success, a negative DIFFATTN_ERR_* code
 *     otherwise.  No exception, signal or abort crosses the ABI.
 *   - Ownership: the caller owns every buffer.  The library never allocates
 *     device memory per call and never frees caller memory.  Inputs are const
 *     and are never written.
 *   - Asynchrony: device work is enqueued on the caller's stream (a
 *     cudaStream_t; NULL means the legacy default stream).  No entry point
 *     synchronises the stream except diffattn_get_device_error.
 *   - Argument checks happen on the host before any CUDA call; a call that
 *     fails them touches neither the GPU nor any buffer.
 *   - Thread safety: entry points may be called from several host threads.
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle, binary-compatible with cudaStream_t. */
typedef struct CUstream_st *diffattn_stream_t;

/* Return codes. */
#define DIFFATTN_OK               0
#define DIFFATTN_ERR_INVALID     -1  /* bad shape, stride, pointer, dtype or non-finite scalar */
#define DIFFATTN_ERR_UNSUPPORTED -2  /* a valid request this build has no kernel for */
#define DIFFATTN_ERR_CUDA        -3  /* a CUDA runtime or driver call failed (incl. launch) */
#define DIFFATTN_ERR_TIMEOUT     -4  /* a kernel's bounded wait ran out (see get_device_error) */

/* Element types of Q1, K1, Q2, K2, V and O (all six share one type). */
#define DIFFATTN_BF16 0   /* bfloat16 storage, fp32 accumulation, bf16 output */
#define DIFFATTN_F32  1   /* float32 storage and arithmetic */

/* Kernel identifiers returned by diffattn_select_kernel. */
#define DIFFATTN_KERNEL_TCGEN05 1  /* tensor-core kernel: bf16, value width 128, D == 64 or 128 */
#define DIFFATTN_KERNEL_SIMT    2  /* CUDA-core kernel: any supported shape */

/*
 * Shape and layout of one call.
 *
 * B, H, T, D: batch, (query) heads, sequence length and Q/K width; all >= 1.
 * D <= 128.
 * Dv: width of V and O.  0 means 2*D, the operation's own shape (paperleet,
 * Formula and conventions: V and O are [B, H, T, 2D]).  Any other value
 * 1 .. 256 is the head shape of DIFF V2 and similar layouts (the
 * aiengineeringfromscratch lesson, "V1 contre V2": the head dimension stays that
 * of the baseline, so V is as wide as Q and K, Dv = D).  The field is last in
 * the struct, so a zero-initialised descriptor keeps the 2*D shape.
 * dtype: DIFFATTN_BF16 or DIFFATTN_F32.
 * kv_group: query heads per key/value head (grouped key/value heads, the
 * layout of DIFF V2: aiengineeringfromscratch lesson, "V1 contre V2" and its
 * GQA exercise).  0 or 1: Q1, Q2, K1, K2, V and O all have H heads.  g > 1:
 * H must be a multiple of g; Q1, Q2 and O have H heads, K1, K2 and V have
 * H / g heads, and query head h reads key/value head h / g (integer
 * division).  The two branches may also share one key tensor (pass the same
 * pointer and strides as K1 and K2); the tensor-core kernel then loads each
 * key tile once for both branches.
 * *_stride: element strides of the B, H and T dimensions of each tensor
 * ([0] = B, [1] = H, [2] = T).  The innermost (D or 2D) dimension is always
 * contiguous (stride 1).  Strides must be >= 0; a stride of 0 is allowed on B
 * and H (broadcast).  Distinct tensors may alias each other, except that O
 * must not overlap any input.
 */
typedef struct {
    int64_t B, H, T, D;
    int32_t dtype;
    int32_t kv_group;          /* query heads per key/value head; 0 or 1 = none */
    int64_t q1_stride[3];
    int64_t k1_stride[3];
    int64_t q2_stride[3];
    int64_t k2_stride[3];
    int64_t v_stride[3];
    int64_t o_stride[3];
    int64_t Dv;                /* V and O width; 0 = 2 * D */
} diffattn_desc;

/*
 * diffattn_lambda -- lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init.
 *
 * lq1, lk1, lq2, lk2: device pointers to n contiguous float32 values each
 * (the lambda parameter vectors, paperleet: "equal nonempty parameter vectors
 * [D_lambda]").  n >= 1.
 * lambda_init: the layer's initial value, e.g. 0.8 - 0.6 exp(-0.3 (l - 1)).
 * lambda_out: device pointer to one float32; receives lambda, computed with
 * float64 dot products and exponentials and rounded once to float32.
 * Launches one small kernel on `stream`.  Errors: DIFFATTN_ERR_INVALID for a
 * NULL pointer, n < 1 or a non-finite lambda_init; DIFFATTN_ERR_CUDA if the
 * launch fails.
 */
int diffattn_lambda(const float *lq1, const float *lk1, const float *lq2,
                    const float *lk2, int64_t n, double lambda_init,
                    float *lambda_out, diffattn_stream_t stream);

/*
 * diffattn_lambda_backward -- gradients of lambda = exp(lq1 . lk1) -
 * exp(lq2 . lk2) + lambda_init with respect to the four vectors, given
 * dlambda = dL/dlambda (paperleet "Differential Transformer Attention",
 * Return requirements: differential_lambda passes gradients to all four
 * parameter vectors).  With e_b = exp(lq_b . lk_b):
 *
 *     dlq1 = dlambda e1 lk1    dlk1 = dlambda e1 lq1
 *     dlq2 = -dlambda e2 lk2   dlk2 = -dlambda e2 lq2
 *
 * lq1, lk1, lq2, lk2: device pointers to n contiguous float32 values each;
 * dlambda: device pointer to one float32 (for example diffattn_bwd's output);
 * dlq1, dlk1, dlq2, dlk2: device pointers to n float32 values each,
 * overwritten.  Dot products and exponentials in float64.  One launch on
 * `stream`.  Errors: DIFFATTN_ERR_INVALID for a NULL pointer or n < 1;
 * DIFFATTN_ERR_CUDA if the launch fails.
 */
int diffattn_lambda_backward(const float *lq1, const float *lk1, const float *lq2,
                             const float *lk2, int64_t n, const float *dlambda,
                             float *dlq1, float *dlk1, float *dlq2, float *dlk2,
                             diffattn_stream_t stream);

/*
 * diffattn_workspace_bytes -- size of the optional scheduler workspace that
 * diffattn_fwd accepts (a few bytes; the value is stable for a given library
 * version).
 */
size_t diffattn_workspace_bytes(void);

/*
 * diffattn_fwd -- O = (A_1 - lambda A_2) V.
 *
 * desc: shape, dtype and strides (host pointer, read during the call only).
 * q1, k1, q2, k2, v: device pointers to the inputs, laid out as desc says.
 * lambda: the coefficient, used when lambda_dev is NULL; must be finite.
 * lambda_dev: optional device pointer to one float32 holding lambda (for
 * example the output of diffattn_lambda); when non-NULL it overrides `lambda`
 * and is read by the kernel, so no host synchronisation is needed.
 * causal: non-zero applies the causal mask to both branches.
 * out: device pointer to O, [B, H, T, Dv] with desc->o_stride, same dtype as
 * the inputs (bf16 results are rounded to nearest even from fp32).
 * workspace, workspace_bytes: optional device scratch of at least
 * diffattn_workspace_bytes() bytes, 4-byte aligned, owned by the caller.  With
 * it the tensor-core kernel hands out work items dynamically (a CTA claims its
 * next item when it needs one), which balances the load when SMs run at
 * different speeds; without it (NULL) items are assigned statically.  The
 * workspace must hold zeros before its first use; every call leaves it zeroed
 * when its kernel finishes.  Calls that may run at the same time on the GPU
 * (different streams) must use different workspaces.  The result does not
 * depend on the schedule.
 * stream: the CUDA stream to launch on.
 *
 * The tensor-core kernel runs when dtype is bf16, the value width is 128 with
 * D == 64 (Dv = 2D) or D == 128 (Dv = D), every base pointer is 16-byte
 * aligned and every stride is a multiple of 8 elements; any other valid
 * request runs on the CUDA-core kernel.  One kernel launch per call.
 * Errors: DIFFATTN_ERR_INVALID (NULL pointers, sizes < 1, D > 128, Dv < 0 or
 * > 256, unknown dtype, negative strides, negative kv_group or one that does
 * not divide H,
 * non-finite lambda, a
 * workspace smaller than diffattn_workspace_bytes() or not 4-byte aligned);
 * DIFFATTN_ERR_CUDA (tensor-map encoding or launch failure).
 */
int diffattn_fwd(const diffattn_desc *desc, const void *q1, const void *k1,
                 const void *q2, const void *k2, const void *v, float lambda,
                 const float *lambda_dev, int causal, void *out, void *workspace,
                 size_t workspace_bytes, diffattn_stream_t stream);

/* Per-head normalisation applied by diffattn_fwd_ex. */
#define DIFFATTN_NORM_NONE  0   /* no normalisation */
#define DIFFATTN_NORM_RMS   1   /* x / sqrt(mean(x^2) + eps) */
#define DIFFATTN_NORM_GROUP 2   /* (x - mean(x)) / sqrt(var(x) + eps), var the mean squared deviation */

/*
 * Output epilogue of diffattn_fwd_ex: for every (b, h, t) row x of O (the
 * head's Dv output channels; Dv = 2D unless the descriptor says otherwise),
 *
 *     y = out_scale * (norm(x) * weight[h] + bias[h])
 *
 * which is the step that follows the operation in the Differential
 * Transformer: a per-head normalisation (called GroupNorm by aifetchly, section
 * 4, and by the ultralytics glossary, RMSNorm for DIFF V1 by the
 * aiengineeringfromscratch lesson), then the fixed multiplier (1 - lambda_init).
 *
 * norm: DIFFATTN_NORM_*.  eps: > 0 when norm != NONE (e.g. 1e-5).
 * weight, bias: optional device pointers to [H, Dv] float32 per-channel
 * affine parameters (NULL = 1 and 0).  out_scale: finite multiplier applied
 * last (e.g. 1 - lambda_init; 1 for none).
 */
typedef struct {
    int32_t norm;
    float eps;
    const float *weight;
    const float *bias;
    float out_scale;
    int32_t reserved;   /* must be 0 */
} diffattn_epilogue;

/*
 * diffattn_fwd_ex -- diffattn_fwd followed by the output epilogue `epi`
 * (host pointer, read during the call only; NULL = none), fused into the
 * same kernel.  Arguments and errors as diffattn_fwd, plus
 * DIFFATTN_ERR_INVALID for an unknown norm, a non-positive or non-finite eps
 * with a norm, a non-finite out_scale or a non-zero reserved field.
 */
int diffattn_fwd_ex(const diffattn_desc *desc, const void *q1, const void *k1,
                    const void *q2, const void *k2, const void *v, float lambda,
                    const float *lambda_dev, int causal, const diffattn_epilogue *epi,
                    void *out, void *workspace, size_t workspace_bytes,
                    diffattn_stream_t stream);

/*
 * diffattn_fwd_host -- diffattn_fwd with the inputs and the output in host
 * memory: copies the inputs in, runs the forward and copies O out, as a
 * pipeline over chunks of whole key/value heads (the copy of chunk c + 1 and
 * the copy back of chunk c - 1 overlap the forward of chunk c).  The result
 * is the same as diffattn_fwd's.
 *
 * q1_host, k1_host, q2_host, k2_host, v_host: host pointers to the inputs;
 * out_host: host pointer that receives O.  Page-locked (pinned) host memory
 * lets the copies run asynchronously; pageable memory also works, with copies
 * that block the calling thread.  q1 .. v, out: device buffers of the full
 * sizes, owned by the caller, that the call fills and uses (the same as
 * diffattn_fwd's inputs and output).  Every tensor, on the host and on the
 * device, must be dense in the [B, H, T, *] order desc describes (K1, K2 and V
 * with H / kv_group heads).  The copies start after the work already queued on
 * `stream`, and the call's last copy is ordered before later work on
 * `stream`; synchronise the stream before reading out_host.  The library keeps
 * two copy streams and a few events per device for this call, created on
 * first use; calls from several host threads are enqueued one at a time.
 * Other arguments and errors as diffattn_fwd, plus DIFFATTN_ERR_INVALID for a
 * NULL host pointer or a tensor that is not dense.  No counterpart on the
 * pages: a library convenience for callers whose data starts and ends on the
 * host.
 */
int diffattn_fwd_host(const diffattn_desc *desc, const void *q1_host, const void *k1_host,
                      const void *q2_host, const void *k2_host, const void *v_host,
                      float lambda, const float *lambda_dev, int causal, void *out_host,
                      void *q1, void *k1, void *q2, void *k2, void *v, void *out,
                      void *workspace, size_t workspace_bytes, diffattn_stream_t stream);

/*
 * diffattn_fwd_train -- diffattn_fwd that also keeps what the backward needs
 * (the forward of a training step): besides O it writes
 *
 *     out2 = A_2 V                  [B, H, T, Dv], desc->o_stride, inputs' dtype
 *     lse  = log sum_j exp(S_b)     [B, H, T, 2] float32, dense, natural log,
 *                                   S_b = Q_b K_b^T / sqrt(D) + M, b = 1, 2
 *
 * (with O = A_1 V - lambda A_2 V, the pair (O, out2) gives each branch's
 * output).  No output epilogue.  Other arguments, kernel choice and errors as
 * diffattn_fwd, plus DIFFATTN_ERR_INVALID for a NULL out2 or lse.  out2 must
 * not overlap any input or O.
 */
int diffattn_fwd_train(const diffattn_desc *desc, const void *q1, const void *k1,
                       const void *q2, const void *k2, const void *v, float lambda,
                       const float *lambda_dev, int causal, void *out, void *out2, float *lse,
                       void *workspace, size_t workspace_bytes, diffattn_stream_t stream);

/*
 * diffattn_bwd_workspace_bytes -- bytes of device workspace diffattn_bwd needs
 * for this descriptor (four float32 row statistics per query row, plus 512
 * bytes of partial sums), or 0 for a NULL descriptor or sizes < 1.
 */
size_t diffattn_bwd_workspace_bytes(const diffattn_desc *desc);

/*
 * diffattn_bwd -- gradients of the operation: given dout = dL/dO, writes
 * dL/dQ1, dL/dK1, dL/dQ2, dL/dK2, dL/dV and dL/dlambda (paperleet
 * "Differential Transformer Attention", Return requirements: gradients flow
 * through both Q/K branches, the value and the coefficient).  With
 * W = A_1 - lambda A_2:
 *
 *     dV = W^T dO        dlambda = -sum(dO * (A_2 V))
 *     dS_b = A_b * (dA_b - rowsum(dA_b * A_b)),  dA_1 = dO V^T, dA_2 = -lambda dO V^T
 *     dQ_b = dS_b K_b / sqrt(D)      dK_b = dS_b^T Q_b / sqrt(D)
 *
 * The gradients of the four lambda vectors follow from dlambda through
 * diffattn_lambda_backward.  With kv_group > 1, dK1, dK2 and dV of a key/value head sum the
 * contributions of every query head that reads it.
 *
 * desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal: as diffattn_fwd (the
 * forward's inputs).  dout: device pointer, [B, H, T, Dv] with desc->o_stride,
 * same dtype as the inputs.  dq1, dq2: device pointers to dense [B, H, T, D];
 * dk1, dk2: dense [B, H / kv_group, T, D]; dv: dense [B, H / kv_group, T, Dv];
 * all of the inputs' dtype, all overwritten; they must not overlap each other
 * or any input.  dlambda: device pointer to one float32, overwritten.
 * workspace: device memory of at least diffattn_bwd_workspace_bytes(desc)
 * bytes, 16-byte aligned, owned by the caller; its contents need no
 * initialisation.
 *
 * Kernels: with bf16, D = 64 and V = 2D, 16-byte aligned bases (inputs, dout
 * and the gradients) and strides that are multiples of 8 elements, on the
 * tensor cores (bf16 operands, fp32 accumulation): the forward kernel in
 * row-statistics mode, then a dQ kernel and a dK/dV kernel.  Anything else
 * valid (other D, other value widths such as the DIFF V2 head's Dv = D, fp32)
 * runs on the CUDA cores in fp32 arithmetic.  Either way five launches on
 * `stream` (row statistics, dQ, dK/dV, and two for dlambda), no atomics, so
 * the result is reproducible bit for bit.
 * Errors: DIFFATTN_ERR_INVALID (as diffattn_fwd, plus a NULL gradient pointer,
 * a missing, small or misaligned workspace); DIFFATTN_ERR_CUDA (launch
 * failure).
 */
int diffattn_bwd(const diffattn_desc *desc, const void *q1, const void *k1,
                 const void *q2, const void *k2, const void *v, float lambda,
                 const float *lambda_dev, int causal, const void *dout, void *dq1,
                 void *dk1, void *dq2, void *dk2, void *dv, float *dlambda,
                 void *workspace, size_t workspace_bytes, diffattn_stream_t stream);

/*
 * diffattn_bwd_saved -- diffattn_bwd from the results diffattn_fwd_train kept:
 * out (O), out2 (A_2 V) and lse, with the same desc, inputs, lambda and mask.
 * The row statistics then come from one elementwise pass over dO, O and out2
 * instead of a recomputation of the forward: Dd_2 = dO . out2 and
 * Dd_1 = dO . (O + lambda out2).  out, out2 and dout share desc->o_stride.
 * Other arguments, kernels and errors as diffattn_bwd, plus
 * DIFFATTN_ERR_INVALID for a NULL out, out2 or lse.
 */
int diffattn_bwd_saved(const diffattn_desc *desc, const void *q1, const void *k1,
                       const void *q2, const void *k2, const void *v, float lambda,
                       const float *lambda_dev, int causal, const void *out,
                       const void *out2, const float *lse, const void *dout, void *dq1,
                       void *dk1, void *dq2, void *dk2, void *dv, float *dlambda,
                       void *workspace, size_t workspace_bytes, diffattn_stream_t stream);

/*
 * Queries over a key/value cache: Tq new queries against Tk cached keys (one
 * decode step for small Tq, a chunk of a prefill for larger Tq).
 * Q1, Q2: [B, H, Tq, D]; K1, K2: [B, H_kv, Tk, D]; V: [B, H_kv, Tk, Dv]; O:
 * [B, H, Tq, Dv], with H_kv = H / kv_group (kv_group as in diffattn_desc; 0
 * or 1 = H_kv = H) and Dv as in diffattn_desc (last field; 0 = 2D).  Strides
 * as in diffattn_desc ([0] = B, [1] = H or H_kv, [2] = the sequence
 * dimension), innermost stride 1.
 */
typedef struct {
    int64_t B, H, Tq, Tk, D;
    int32_t dtype;
    int32_t kv_group;          /* query heads per key/value head; 0 or 1 = none */
    int64_t q1_stride[3];
    int64_t k1_stride[3];
    int64_t q2_stride[3];
    int64_t k2_stride[3];
    int64_t v_stride[3];
    int64_t o_stride[3];
    int64_t Dv;                /* V and O width; 0 = 2 * D */
} diffattn_kv_desc;

/*
 * diffattn_decode_workspace_bytes -- bytes of device workspace diffattn_decode
 * needs for this descriptor (partial results of the key-range splits; 16 bytes,
 * unused, when the call runs on the forward kernels), or 0 if the descriptor
 * is invalid or unsupported.
 */
size_t diffattn_decode_workspace_bytes(const diffattn_kv_desc *desc);

/*
 * diffattn_decode -- O = (softmax(Q1 K1^T / sqrt(D) + M) - lambda
 * softmax(Q2 K2^T / sqrt(D) + M)) V for Tq queries over Tk cached keys, then
 * the optional epilogue `epi` (as in diffattn_fwd_ex; NULL = none).
 *
 * causal: non-zero places query i at position Tk - Tq + i and masks keys
 * j > Tk - Tq + i in both branches (requires Tk >= Tq); zero lets every query
 * see every key.
 * workspace: device memory of at least diffattn_decode_workspace_bytes(desc)
 * bytes, 16-byte aligned, owned by the caller; its contents need no
 * initialisation and are overwritten.  Calls that may run at the same time on
 * the GPU must use different workspaces.
 * Other arguments as diffattn_fwd.
 *
 * Kernels.  Split-key decode: dtype bf16 or fp32, D in {32, 64, 128}, Dv =
 * 2D, Tq <= 8 (D <= 64) or Tq <= 4 (D = 128), K1, K2 and V with 16-byte
 * aligned base pointers and strides that are multiples of 16 bytes.  Two
 * kernel launches per call (the key-range splits, then their combination).
 * Work is bound by reading K1, K2 and V once: one CTA serves up to 8 query
 * rows (4 for D = 128) of the query heads that share a key/value head, so with
 * kv_group = g the cache of a key/value head is read ceil(g * Tq / 8) times
 * (ceil(g * Tq / 4) for D = 128), not g * ceil(Tq / 8) times.
 * Units of up to 16 query rows on the tensor cores: bf16 with value width
 * 128 and either D = 64 with more than 8 query rows per key/value head
 * (g * Tq > 8, Tq <= 16), or the DIFF V2 head D = Dv = 128 with Tq <= 16
 * (aiengineeringfromscratch lesson, "V1 contre V2").  The workspace is sized
 * for the split-key decode on the tensor cores (the cache of a key/value head
 * read ceil(g * Tq / 16) times), which runs when Q1, Q2, K1, K2 and V have
 * 16-byte aligned bases and strides with the cache rows dense along the
 * sequence, and at D = 128 K1 and K2 are one tensor (same pointer and
 * strides).  Otherwise the call runs, at D = 64 with Tq <= 8, the split-key
 * layout of up to 8-row units on the CUDA cores (the workspace has room for
 * it; it needs aligned K1, K2 and V), else the forward kernels.
 * Any other request (more query rows, another D or Dv) runs as one launch of
 * the forward kernels with the queries placed at the end of the key sequence:
 * on the tensor cores when diffattn_fwd would choose them for this shape and
 * layout (bf16, value width 128, D = 64 or 128, aligned), else on the CUDA
 * cores; the workspace is then not used.
 * Errors: DIFFATTN_ERR_INVALID (NULL pointers, sizes < 1, D > 128, Dv < 0 or
 * > 256, Tk < Tq with the causal mask, unknown dtype, negative strides,
 * negative kv_group or one that does not divide H, non-finite lambda, bad
 * epilogue, missing, small or misaligned workspace); DIFFATTN_ERR_UNSUPPORTED
 * (a split-key decode other than the V2 head's with unaligned K1, K2 or V,
 * or sizes beyond the int32
 * index range); DIFFATTN_ERR_CUDA (launch failure).
 */
int diffattn_decode(const diffattn_kv_desc *desc, const void *q1, const void *k1,
                    const void *q2, const void *k2, const void *v, float lambda,
                    const float *lambda_dev, int causal, const diffattn_epilogue *epi,
                    void *out, void *workspace, size_t workspace_bytes,
                    diffattn_stream_t stream);

/*
 * diffattn_decode_noalloc -- diffattn_decode for callers that cannot allocate
 * device memory when they run the decode step (an inference runtime or plug-in
 * host that owns every buffer and passes only inputs and outputs, a process
 * held to a fixed device-memory budget, or a latency-critical loop that must
 * not call the allocator, which may synchronise the device).  There is no
 * counterpart on the pages; this is a library convenience.
 *
 * Same arguments as diffattn_decode without the workspace: the partial results
 * of the key-range splits go to a scratch buffer of 8 MiB (8388608 bytes) that
 * is part of the library; every GPU that loads the library holds one such
 * buffer until the process exits.  The call allocates nothing.  The first call
 * on a device (and the first after a device reset, or from another context)
 * looks up the buffer's device address, with that device current; under CUDA's
 * lazy module loading that first call is also where the driver loads the
 * buffer's module and commits its 8 MiB, which may synchronise the device.
 * Make that first call at set-up, before capturing any stream and outside any
 * latency-critical region.
 * Every call shares the one buffer: calls that run on the GPU at the same time
 * race and corrupt each other's results.  Calls enqueued one after another on
 * one stream do not: each call's kernels finish before the next call's start.
 * The buffer needs no clearing; each call writes everything it reads.
 * Errors: every check of diffattn_decode other than the workspace's comes
 * first and gives the same code; then DIFFATTN_ERR_UNSUPPORTED when the problem
 * needs more than 8 MiB of partial results (diffattn_decode_workspace_bytes
 * reports the need; use diffattn_decode with a workspace instead).
 */
int diffattn_decode_noalloc(const diffattn_kv_desc *desc, const void *q1,
                            const void *k1, const void *q2, const void *k2,
                            const void *v, float lambda, const float *lambda_dev,
                            int causal, const diffattn_epilogue *epi, void *out,
                            diffattn_stream_t stream);

/*
 * diffattn_select_kernel -- which kernel diffattn_fwd would launch for this
 * descriptor and these pointers (DIFFATTN_KERNEL_*), or a negative error code
 * if the arguments are invalid.  Host only; touches no GPU state.
 */
int diffattn_select_kernel(const diffattn_desc *desc, const void *q1,
                           const void *k1, const void *q2, const void *k2,
                           const void *v, const void *out);

/*
 * diffattn_get_device_error -- synchronise `stream`, then report whether any
 * kernel of this library on the current device ran out of a bounded wait
 * since the previous call (DIFFATTN_ERR_TIMEOUT), and clear that record.
 * Every wait inside the kernels has an iteration and time limit; on expiry
 * the kernel records the failure, stops issuing work, releases what it holds
 * and returns, leaving the CUDA context usable.  Returns DIFFATTN_OK when no
 * wait ran out, DIFFATTN_ERR_CUDA if the synchronisation itself fails.
 */
int diffattn_get_device_error(diffattn_stream_t stream);

/*
 * diffattn_selftest_timeout -- test hook for the failure path above; the
 * pages have no counterpart.  Enqueues on `stream` a one-thread kernel that
 * waits, with the same bounded wait the library's kernels use, on a barrier
 * that nothing ever completes.  The wait gives up after its time limit (about
 * two seconds), records DIFFATTN_ERR_TIMEOUT in the device status word and the
 * kernel returns normally; a following diffattn_get_device_error reports the
 * timeout and clears it, and the CUDA context stays usable.  Returns
 * DIFFATTN_OK once enqueued, DIFFATTN_ERR_CUDA if the launch fails.  Touches
 * no caller memory.
 */
int diffattn_selftest_timeout(diffattn_stream_t stream);

/* Human-readable text for a return code (static storage, never NULL). */
const char *diffattn_strerror(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
int diffattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
