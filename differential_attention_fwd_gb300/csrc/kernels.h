// kernels.h -- internal interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "diffattn.h"

namespace diffattn {

// Output epilogue applied after O = O1/l1 - lambda O2/l2 (the same values as
// DIFFATTN_NORM_* in the public header).
enum : int { kNormNone = 0, kNormRms = 1, kNormGroup = 2 };

// Parameters of the tensor-core kernel (bf16; D = 64 or 128, value width 128).
// Queries and keys may be sequences of different lengths: query row i sits at
// position i + kv_off of the key sequence (kv_off = Tk - Tq for queries at the
// end of a key/value cache, 0 when queries and keys are one sequence), and the
// causal mask hides keys j > i + kv_off.
struct TcParams {
    int B, H, T;            // T: query rows (Tq)
    int Tk;                 // keys
    int kv_off;             // causal offset of query row 0 in the key sequence (>= 0)
    int nq;                 // number of 128-row query tiles along T
    int nk;                 // number of 64-row key tiles along Tk
    int total_items;        // B * H * nq
    int group;              // heads per scheduling group (L2 locality)
    int causal;
    float scale_log2;       // log2(e) / sqrt(D)
    float lambda;           // used when lambda_dev == nullptr
    const float* lambda_dev;
    __nv_bfloat16* out;
    int64_t o_sB, o_sH, o_sT;
    uint32_t* status;       // device status word
    uint32_t* sched;        // 2 words: item counter, finished CTAs (nullptr: static schedule)
    int norm;               // kNorm*
    float norm_eps;
    const float* norm_weight;   // [H, 2D] or nullptr
    const float* norm_bias;     // [H, 2D] or nullptr
    float out_scale;            // applied last
    int kv_group;               // query heads per key/value head (>= 1)
    int k_shared;               // K1 and K2 are one tensor: load each key tile once
    // Row-statistics mode (the first pass of the backward): when stats is set,
    // the epilogue writes, per query row, the negated log2-sum-exp of each
    // branch's scaled scores and the negated Dd_b = dO . (A_b V) to
    // stats[(b*H + h)*T + t][0..3] (-lse_1, -lse_2, -Dd_1, -Dd_2) instead of
    // writing O.
    float* stats;
    const __nv_bfloat16* dout;
    int64_t do_sB, do_sH, do_sT;
    // Training outputs (when out2 is set): A_2 V with the output's strides, and
    // the natural-log log-sum-exp of each branch's scaled scores, lse[(b*H + h)*T
    // + t][branch].
    __nv_bfloat16* out2;
    float* lse;
};

// Parameters of the CUDA-core kernel (any D <= 128, value width Dv <= 256,
// fp32 or bf16).  T query rows over Tk keys; query row i sees keys
// j <= i + kv_off under the causal mask.
struct SimtParams {
    int B, H, T, D;
    int Tk, kv_off, Dv;
    int causal;
    float scale;            // 1 / sqrt(D)
    float lambda;
    const float* lambda_dev;
    const void* q1; const void* k1; const void* q2; const void* k2; const void* v;
    void* out;
    int64_t s_q1[3], s_k1[3], s_q2[3], s_k2[3], s_v[3], s_o[3];
    int norm;
    float norm_eps;
    const float* norm_weight;
    const float* norm_bias;
    float out_scale;
    int kv_group;           // query head h reads key/value head h / kv_group
    void* out2;             // training outputs (optional): A_2 V with the output's strides,
    float* lse;             // and the natural-log log-sum-exp of each branch, [B, H, T, 2]
};

// Parameters of the decode kernels (Tq queries over Tk cached keys).
struct DecodeParams {
    int B, H, Tq, Tk, D;
    int kv_group;           // query heads per key/value head (>= 1)
    int Hk;                 // key/value heads, H / kv_group
    int row_chunks;         // CTAs along the kv_group * Tq query rows of a key/value head
    int dense_kv;           // K1, K2 and V rows contiguous along the sequence (async staging)
    int tc_ok;              // the tensor-core first pass may run: bf16, D = 64 (V = 2D) or
                            // D = 128 with V = D and one key tensor, dense K/V rows,
                            // Q rows 16-byte aligned
    int tc_only;            // units of up to 16 rows (the DIFF V2 head, or bf16 D = 64 with
                            // more than 8 rows per key/value head): the tensor-core first
                            // pass and the combine pass of value width 128 only
    int k_shared;           // K1 and K2 are one tensor
    uint32_t* status;       // device status word (bounded waits of the tensor-core pass)
    const CUtensorMap* tc_maps;   // host memory: K1, K2 and V tensor maps (128-row boxes) for
                                  // the tensor-core pass's launch; never read on the device
    int causal;
    int bf16;               // element type: 1 bf16, 0 fp32
    int tq_bucket;          // query rows per CTA: 1, 2, 4, 8 (or 16 on the tensor-core pass)
    int splits;             // key-range splits per unit (b, key/value head, row chunk)
    int total_items;        // units * splits
    int split_len;          // keys per split (multiple of 256)
    float scale_log2;       // log2(e) / sqrt(D)
    float lambda;
    const float* lambda_dev;
    const void* q1; const void* k1; const void* q2; const void* k2; const void* v;
    void* out;
    int64_t s_q1[3], s_k1[3], s_q2[3], s_k2[3], s_v[3], s_o[3];
    float* work;            // partial results, decode_work_floats(...) floats
    int tc_tpu;             // tensor-core pass: key tiles per unit,
    int tc_grid;            //   CTAs (each streams a contiguous range of the
    int64_t tc_total;       //   units' tiles), tiles of all units
    int norm;
    float norm_eps;
    const float* norm_weight;
    const float* norm_bias;
    float out_scale;
};

// Parameters of the backward (CUDA-core kernels, any D <= 128, value width Dv
// <= 256).  Inputs use the descriptor's strides; dout uses the output strides;
// the gradients are dense: dq [B, H, T, D], dk [B, Hk, T, D], dv [B, Hk, T, Dv].
struct BwdParams {
    int B, H, Hk, kv_group, T, D;
    int Dv;
    int causal;
    float scale;            // 1 / sqrt(D)
    float lambda;
    const float* lambda_dev;
    const void* q1; const void* k1; const void* q2; const void* k2; const void* v;
    const void* dout;
    void* dq1; void* dk1; void* dq2; void* dk2; void* dv;
    int64_t s_q1[3], s_k1[3], s_q2[3], s_k2[3], s_v[3], s_do[3];
    float* stats;           // [B, H, T, 4]: log-sum-exp of each branch, Dd_1, Dd_2,
                            // then 128 floats of dlambda partial sums
    float* dlambda;         // one float
};

// Parameters of the tensor-core backward (bf16, D = 64).  Gradients are dense
// like BwdParams'; stats holds the forward kernel's row statistics (log2 units).
struct BwdTcParams {
    int B, H, Hk, kv_group, T;
    int nq128, nk64, nk128;     // 128-row and 64-row tiles along T
    int causal;
    float scale;                // 1 / sqrt(D)
    float scale_log2;           // log2(e) / sqrt(D)
    float lambda;
    const float* lambda_dev;
    uint32_t* status;
    const float* stats;
    void* dq1; void* dq2; void* dk1; void* dk2; void* dv;
};

// Row statistics for the backward from the forward's saved results: O (the
// output), O2 = A_2 V and the natural-log log-sum-exp of each branch.  Dd_2 =
// dO . O2 and Dd_1 = dO . (O + lambda O2).  log2_negated selects the layout
// the tensor-core kernels read (-lse_1 log2(e), -lse_2 log2(e), -Dd_1, -Dd_2)
// instead of the CUDA-core one (lse_1, lse_2, Dd_1, Dd_2).
struct PrepParams {
    int B, H, T, Dv;
    int bf16;
    int log2_negated;
    float lambda;
    const float* lambda_dev;
    const void* out; const void* out2; const void* dout;
    int64_t s_o[3];         // shared by out, out2 and dout
    const float* lse;       // [B, H, T, 2]
    float* stats;           // [B, H, T, 4]
};

// Decode helpers: query-row bucket (rows rounded up to 1, 2, 4 or 8; 0 if
// there are more rows than one CTA of width D takes), and the number of
// workspace floats for `units` CTAs along the heads and query rows.
int decode_tq_bucket(int rows, int D);
int decode_max_rows(int D);
size_t decode_work_floats(int64_t units, int splits, int tq_bucket, int64_t D);

// Each returns 0 on success, -1 if the launch failed.
int launch_decode(const DecodeParams& p, cudaStream_t stream);
// The tensor-core first pass of the decode (decode_tc.cu): D = 64 with 4, 8 or
// 16 query rows per unit, D = 128 (value width 128, one key tensor) with 1 to 16.  It sets p's tc_* fields and p->splits (partial slots per
// unit) for its launch; the caller launches the combine pass with that p.
int launch_decode_tc_first_pass(DecodeParams* p, cudaStream_t stream);
// Workspace floats the tensor-core pass may need (its slots per unit on any
// GPU of up to 1024 SMs).
size_t decode_tc_work_floats(int64_t units, int64_t Tk, int tq_bucket);
// head_dim: the Q/K width, 64 or 128 (the value width is 128 either way).
int launch_fwd_tc(const CUtensorMap* maps /*q1,k1,q2,k2,v,out*/, const TcParams& p, int head_dim,
                  int grid, cudaStream_t stream);
int launch_bwd_tc(const CUtensorMap* maps /*dq: q1,k1,q2,k2,v,do; dkdv: the same*/,
                  const BwdTcParams& p, int num_sms, cudaStream_t stream);
// dlambda = sign * (sum over rows of stats[row][3]) (sign -1 when the rows hold
// Dd_2, +1 when they hold -Dd_2); the 128 floats after the rows' statistics
// hold the per-block partial sums.
int launch_bwd_dlambda(const float* stats, int64_t rows, float sign, float* out,
                       cudaStream_t stream);
int launch_bwd_prep(const PrepParams& p, cudaStream_t stream);
// The CUDA-core backward without its statistics pass (the statistics are in
// p.stats already).
int launch_bwd_simt_grads_f32(const BwdParams& p, cudaStream_t stream);
int launch_bwd_simt_grads_bf16(const BwdParams& p, cudaStream_t stream);
int launch_bwd_simt_f32(const BwdParams& p, cudaStream_t stream);
int launch_bwd_simt_bf16(const BwdParams& p, cudaStream_t stream);
int launch_fwd_simt_f32(const SimtParams& p, cudaStream_t stream);
int launch_fwd_simt_bf16(const SimtParams& p, cudaStream_t stream);
int launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                  int64_t n, double lambda_init, float* out, cudaStream_t stream);
int launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                      int64_t n, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                      float* dlk2, cudaStream_t stream);

// Host helpers of the C-ABI layer (api.cu).
// Unique ID of the calling thread's current CUDA context, 0 if none.
unsigned long long current_context();
// Every argument check diffattn_decode makes except those of its workspace;
// on success *work_bytes receives the workspace the call needs.
int decode_check(const diffattn_kv_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                 const diffattn_epilogue* epi, const void* out, size_t* work_bytes);

// One-thread kernel whose bounded wait on a barrier nothing completes runs
// out and records the timeout in `status` (the failure path, tested without a
// fault).
int launch_selftest_timeout(uint32_t* status, cudaStream_t stream);

}  // namespace diffattn
