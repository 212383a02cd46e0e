// bwd_simt.cu -- backward of the differential-attention forward on the CUDA
// cores (any D <= 128, any value width Dv <= 256, fp32 or bf16 storage, fp32
// arithmetic).
//
// Given dO = dL/dO for O = (A_1 - lambda A_2) V (paperleet "Differential
// Transformer Attention", Return requirements: gradients through both Q/K
// branches, the value and the coefficient), with W = A_1 - lambda A_2:
//   dV = W^T dO,   dW = dO V^T,   dlambda = -sum(dO * (A_2 V))
//   dS_1 = A_1 * (dW - Dd_1),          Dd_1 = rowsum(dO * (A_1 V))
//   dS_2 = -lambda A_2 * (dW - Dd_2),  Dd_2 = rowsum(dO * (A_2 V))
//   dQ_b = dS_b K_b / sqrt(D),   dK_b = dS_b^T Q_b / sqrt(D)
// (rowsum(dA_b * A_b) for the softmax backward is Dd_1 for branch 1 and
// -lambda Dd_2 for branch 2, since dA_1 = dW and dA_2 = -lambda dW.)
//
// Kernels:
//   stats   one warp per query row: a forward pass per branch that keeps the
//           row's log-sum-exp and Dd_b (the branch output dotted with dO);
//   prep    instead of stats, when the forward saved O, A_2 V and the
//           log-sum-exp: Dd_b from those, one warp per row;
//   dq      one warp per query row: recomputes A_b from the log-sum-exp, forms
//           dS_b one key per lane and accumulates dQ_b;
//   dkdv    one warp per key row of a key/value head: walks the visible query
//           rows of every query head that reads it, accumulates dK_1, dK_2
//           and dV;
//   dlambda -sum of Dd_2 over all rows, in a fixed order (two small launches).
#include "kernels.h"

#include <cmath>

namespace diffattn {
namespace bwd {

constexpr int WARPS = 4;
constexpr int MAX_D = 128;
constexpr int MAX_DV = 2 * MAX_D;
constexpr int OPL = MAX_DV / 32;   // value columns per lane
constexpr int QPL = MAX_D / 32;    // Q/K columns per lane

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Query row i of query head (b, h), as a warp's work item.
struct Row {
    int b, h, hk, i;
};
__device__ __forceinline__ bool row_of(const BwdParams& p, Row& r) {
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t bh = blockIdx.x / rows_per_head;
    r.b = (int)(bh / p.H);
    r.h = (int)(bh - (int64_t)r.b * p.H);
    r.hk = r.h / p.kv_group;
    r.i = (int)((blockIdx.x - bh * rows_per_head) * WARPS + (threadIdx.x >> 5));
    return r.i < p.T;
}

// ------------------------------------------------------------------ stats
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) bwd_stats_kernel(const BwdParams p) {
    __shared__ float qs[WARPS][2][MAX_D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Row r;
    if (!row_of(p, r)) return;
    const T* q1 = static_cast<const T*>(p.q1) + r.b * p.s_q1[0] + r.h * p.s_q1[1] + (int64_t)r.i * p.s_q1[2];
    const T* q2 = static_cast<const T*>(p.q2) + r.b * p.s_q2[0] + r.h * p.s_q2[1] + (int64_t)r.i * p.s_q2[2];
    const T* k1 = static_cast<const T*>(p.k1) + r.b * p.s_k1[0] + r.hk * p.s_k1[1];
    const T* k2 = static_cast<const T*>(p.k2) + r.b * p.s_k2[0] + r.hk * p.s_k2[1];
    const T* v = static_cast<const T*>(p.v) + r.b * p.s_v[0] + r.hk * p.s_v[1];
    const T* dout = static_cast<const T*>(p.dout) + r.b * p.s_do[0] + r.h * p.s_do[1] + (int64_t)r.i * p.s_do[2];
    const int D = p.D, Dv = p.Dv;
    for (int d = lane; d < D; d += 32) {
        qs[warp][0][d] = ld(q1, d);
        qs[warp][1][d] = ld(q2, d);
    }
    __syncwarp();
    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float o1[OPL], o2[OPL];
#pragma unroll
    for (int c = 0; c < OPL; ++c) o1[c] = o2[c] = 0.f;
    const int kend = p.causal ? r.i + 1 : p.T;
    for (int k0 = 0; k0 < kend; k0 += 32) {
        const int key = k0 + lane;
        const bool valid = key < kend;
        float s1 = -INFINITY, s2 = -INFINITY;
        if (valid) {
            float d1 = 0.f, d2 = 0.f;
            for (int d = 0; d < D; ++d) {
                d1 = fmaf(qs[warp][0][d], ld(k1, (int64_t)key * p.s_k1[2] + d), d1);
                d2 = fmaf(qs[warp][1][d], ld(k2, (int64_t)key * p.s_k2[2] + d), d2);
            }
            s1 = d1 * p.scale;
            s2 = d2 * p.scale;
        }
        const float n1 = fmaxf(m1, warp_max(s1)), n2 = fmaxf(m2, warp_max(s2));
        const float a1 = expf(m1 - n1), a2 = expf(m2 - n2);
        const float p1 = valid ? expf(s1 - n1) : 0.f, p2 = valid ? expf(s2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(p1);
        l2 = l2 * a2 + warp_sum(p2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int c = 0; c < OPL; ++c) {
            o1[c] *= a1;
            o2[c] *= a2;
        }
        const int nk = min(32, kend - k0);
        for (int t = 0; t < nk; ++t) {
            const float w1 = __shfl_sync(0xffffffffu, p1, t), w2 = __shfl_sync(0xffffffffu, p2, t);
            const int64_t vr = (int64_t)(k0 + t) * p.s_v[2];
#pragma unroll
            for (int c = 0; c < OPL; ++c) {
                const int col = lane + 32 * c;
                if (col < Dv) {
                    const float x = ld(v, vr + col);
                    o1[c] = fmaf(w1, x, o1[c]);
                    o2[c] = fmaf(w2, x, o2[c]);
                }
            }
        }
    }
    float dd1 = 0.f, dd2 = 0.f;
#pragma unroll
    for (int c = 0; c < OPL; ++c) {
        const int col = lane + 32 * c;
        if (col < Dv) {
            const float g = ld(dout, col);
            dd1 = fmaf(g, o1[c], dd1);
            dd2 = fmaf(g, o2[c], dd2);
        }
    }
    dd1 = warp_sum(dd1) / l1;
    dd2 = warp_sum(dd2) / l2;
    if (lane == 0) {
        float* s = p.stats + (((int64_t)r.b * p.H + r.h) * p.T + r.i) * 4;
        s[0] = m1 + logf(l1);
        s[1] = m2 + logf(l2);
        s[2] = dd1;
        s[3] = dd2;
    }
}

// ------------------------------------------------------------------ dQ
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) bwd_dq_kernel(const BwdParams p) {
    __shared__ float qs[WARPS][2][MAX_D];
    __shared__ float gs[WARPS][MAX_DV];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Row r;
    if (!row_of(p, r)) return;
    const int64_t row = ((int64_t)r.b * p.H + r.h) * p.T + r.i;
    const T* q1 = static_cast<const T*>(p.q1) + r.b * p.s_q1[0] + r.h * p.s_q1[1] + (int64_t)r.i * p.s_q1[2];
    const T* q2 = static_cast<const T*>(p.q2) + r.b * p.s_q2[0] + r.h * p.s_q2[1] + (int64_t)r.i * p.s_q2[2];
    const T* k1 = static_cast<const T*>(p.k1) + r.b * p.s_k1[0] + r.hk * p.s_k1[1];
    const T* k2 = static_cast<const T*>(p.k2) + r.b * p.s_k2[0] + r.hk * p.s_k2[1];
    const T* v = static_cast<const T*>(p.v) + r.b * p.s_v[0] + r.hk * p.s_v[1];
    const T* dout = static_cast<const T*>(p.dout) + r.b * p.s_do[0] + r.h * p.s_do[1] + (int64_t)r.i * p.s_do[2];
    const int D = p.D, Dv = p.Dv;
    for (int d = lane; d < D; d += 32) {
        qs[warp][0][d] = ld(q1, d);
        qs[warp][1][d] = ld(q2, d);
    }
    for (int c = lane; c < Dv; c += 32) gs[warp][c] = ld(dout, c);
    __syncwarp();
    const float lse1 = p.stats[row * 4 + 0], lse2 = p.stats[row * 4 + 1];
    const float dd1 = p.stats[row * 4 + 2], dd2 = p.stats[row * 4 + 3];
    const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
    float g1[QPL], g2[QPL];
#pragma unroll
    for (int c = 0; c < QPL; ++c) g1[c] = g2[c] = 0.f;
    const int kend = p.causal ? r.i + 1 : p.T;
    for (int k0 = 0; k0 < kend; k0 += 32) {
        const int key = k0 + lane;
        float ds1 = 0.f, ds2 = 0.f;
        if (key < kend) {
            float d1 = 0.f, d2 = 0.f, dw = 0.f;
            for (int d = 0; d < D; ++d) {
                d1 = fmaf(qs[warp][0][d], ld(k1, (int64_t)key * p.s_k1[2] + d), d1);
                d2 = fmaf(qs[warp][1][d], ld(k2, (int64_t)key * p.s_k2[2] + d), d2);
            }
            for (int c = 0; c < Dv; ++c) dw = fmaf(gs[warp][c], ld(v, (int64_t)key * p.s_v[2] + c), dw);
            const float a1 = expf(d1 * p.scale - lse1), a2 = expf(d2 * p.scale - lse2);
            ds1 = a1 * (dw - dd1);
            ds2 = -lam * a2 * (dw - dd2);
        }
        const int nk = min(32, kend - k0);
        for (int t = 0; t < nk; ++t) {
            const float w1 = __shfl_sync(0xffffffffu, ds1, t), w2 = __shfl_sync(0xffffffffu, ds2, t);
#pragma unroll
            for (int c = 0; c < QPL; ++c) {
                const int col = lane + 32 * c;
                if (col < D) {
                    g1[c] = fmaf(w1, ld(k1, (int64_t)(k0 + t) * p.s_k1[2] + col), g1[c]);
                    g2[c] = fmaf(w2, ld(k2, (int64_t)(k0 + t) * p.s_k2[2] + col), g2[c]);
                }
            }
        }
    }
    T* dq1 = static_cast<T*>(p.dq1) + row * D;
    T* dq2 = static_cast<T*>(p.dq2) + row * D;
#pragma unroll
    for (int c = 0; c < QPL; ++c) {
        const int col = lane + 32 * c;
        if (col < D) {
            st(dq1, col, g1[c] * p.scale);
            st(dq2, col, g2[c] * p.scale);
        }
    }
}

// ------------------------------------------------------------------ dK, dV
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) bwd_dkdv_kernel(const BwdParams p) {
    __shared__ float ks[WARPS][2][MAX_D];
    __shared__ float vs[WARPS][MAX_DV];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t bhk = blockIdx.x / rows_per_head;
    const int b = (int)(bhk / p.Hk);
    const int hk = (int)(bhk - (int64_t)b * p.Hk);
    const int j = (int)((blockIdx.x - bhk * rows_per_head) * WARPS + warp);
    if (j >= p.T) return;
    const T* k1 = static_cast<const T*>(p.k1) + b * p.s_k1[0] + hk * p.s_k1[1] + (int64_t)j * p.s_k1[2];
    const T* k2 = static_cast<const T*>(p.k2) + b * p.s_k2[0] + hk * p.s_k2[1] + (int64_t)j * p.s_k2[2];
    const T* v = static_cast<const T*>(p.v) + b * p.s_v[0] + hk * p.s_v[1] + (int64_t)j * p.s_v[2];
    const int D = p.D, Dv = p.Dv;
    for (int d = lane; d < D; d += 32) {
        ks[warp][0][d] = ld(k1, d);
        ks[warp][1][d] = ld(k2, d);
    }
    for (int c = lane; c < Dv; c += 32) vs[warp][c] = ld(v, c);
    __syncwarp();
    const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
    float gk1[QPL], gk2[QPL], gv[OPL];
#pragma unroll
    for (int c = 0; c < QPL; ++c) gk1[c] = gk2[c] = 0.f;
#pragma unroll
    for (int c = 0; c < OPL; ++c) gv[c] = 0.f;
    const int i_begin = p.causal ? j : 0;
    for (int h = hk * p.kv_group; h < (hk + 1) * p.kv_group; ++h) {
        const T* q1 = static_cast<const T*>(p.q1) + b * p.s_q1[0] + h * p.s_q1[1];
        const T* q2 = static_cast<const T*>(p.q2) + b * p.s_q2[0] + h * p.s_q2[1];
        const T* dout = static_cast<const T*>(p.dout) + b * p.s_do[0] + h * p.s_do[1];
        const float* stats = p.stats + ((int64_t)b * p.H + h) * p.T * 4;
        for (int i0 = i_begin; i0 < p.T; i0 += 32) {
            const int i = i0 + lane;
            float w = 0.f, ds1 = 0.f, ds2 = 0.f;
            if (i < p.T) {
                float d1 = 0.f, d2 = 0.f, dw = 0.f;
                for (int d = 0; d < D; ++d) {
                    d1 = fmaf(ld(q1, (int64_t)i * p.s_q1[2] + d), ks[warp][0][d], d1);
                    d2 = fmaf(ld(q2, (int64_t)i * p.s_q2[2] + d), ks[warp][1][d], d2);
                }
                for (int c = 0; c < Dv; ++c) dw = fmaf(ld(dout, (int64_t)i * p.s_do[2] + c), vs[warp][c], dw);
                const float* s = stats + (int64_t)i * 4;
                const float a1 = expf(d1 * p.scale - s[0]), a2 = expf(d2 * p.scale - s[1]);
                w = a1 - lam * a2;
                ds1 = a1 * (dw - s[2]);
                ds2 = -lam * a2 * (dw - s[3]);
            }
            const int ni = min(32, p.T - i0);
            for (int t = 0; t < ni; ++t) {
                const float wt = __shfl_sync(0xffffffffu, w, t);
                const float s1 = __shfl_sync(0xffffffffu, ds1, t), s2 = __shfl_sync(0xffffffffu, ds2, t);
                const int64_t it = i0 + t;
#pragma unroll
                for (int c = 0; c < OPL; ++c) {
                    const int col = lane + 32 * c;
                    if (col < Dv) gv[c] = fmaf(wt, ld(dout, it * p.s_do[2] + col), gv[c]);
                }
#pragma unroll
                for (int c = 0; c < QPL; ++c) {
                    const int col = lane + 32 * c;
                    if (col < D) {
                        gk1[c] = fmaf(s1, ld(q1, it * p.s_q1[2] + col), gk1[c]);
                        gk2[c] = fmaf(s2, ld(q2, it * p.s_q2[2] + col), gk2[c]);
                    }
                }
            }
        }
    }
    const int64_t krow = ((int64_t)b * p.Hk + hk) * p.T + j;
    T* dk1 = static_cast<T*>(p.dk1) + krow * D;
    T* dk2 = static_cast<T*>(p.dk2) + krow * D;
    T* dv = static_cast<T*>(p.dv) + krow * Dv;
#pragma unroll
    for (int c = 0; c < QPL; ++c) {
        const int col = lane + 32 * c;
        if (col < D) {
            st(dk1, col, gk1[c] * p.scale);
            st(dk2, col, gk2[c] * p.scale);
        }
    }
#pragma unroll
    for (int c = 0; c < OPL; ++c) {
        const int col = lane + 32 * c;
        if (col < Dv) st(dv, col, gv[c]);
    }
}

// ------------------------------------------------------------------ dlambda
// dlambda = -sum over all rows of Dd_2, summed in a fixed order so that the
// result is reproducible: block i sums its contiguous share of the rows
// (threads take fixed strided subsets, then a fixed tree), then one block sums
// the per-block partials in block order.
constexpr int DLAMBDA_BLOCKS = 128;

__global__ void __launch_bounds__(256) bwd_dlambda_partial_kernel(const float* stats, int64_t rows,
                                                                  float* partials) {
    __shared__ float part[8];
    const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per;
    const int64_t r1 = min(rows, r0 + per);
    float s = 0.f;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) s += stats[r * 4 + 3];
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += part[w];
        partials[blockIdx.x] = t;
    }
}

__global__ void __launch_bounds__(32) bwd_dlambda_final_kernel(const float* partials, int n,
                                                               float sign, float* out) {
    float s = 0.f;
    for (int i = threadIdx.x; i < n; i += 32) s += partials[i];
    s = warp_sum(s);
    if (threadIdx.x == 0) *out = sign * s;
}

int launch_dlambda(const float* stats, int64_t rows, float* partials, float sign, float* out,
                   cudaStream_t stream) {
    bwd_dlambda_partial_kernel<<<DLAMBDA_BLOCKS, 256, 0, stream>>>(stats, rows, partials);
    if (cudaGetLastError() != cudaSuccess) return -1;
    bwd_dlambda_final_kernel<<<1, 32, 0, stream>>>(partials, DLAMBDA_BLOCKS, sign, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------------ prep
// Row statistics from the forward's saved results (one warp per row):
// Dd_2 = dO . O2, Dd_1 = dO . (O + lambda O2), since O = O1 - lambda O2.
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) bwd_prep_kernel(const PrepParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int64_t rows = (int64_t)p.B * p.H * p.T;
    if (row >= rows) return;
    const int64_t bh = row / p.T;
    const int t = (int)(row - bh * p.T);
    const int b = (int)(bh / p.H);
    const int h = (int)(bh - (int64_t)b * p.H);
    const int64_t off = b * p.s_o[0] + h * p.s_o[1] + (int64_t)t * p.s_o[2];
    const T* o = static_cast<const T*>(p.out) + off;
    const T* o2 = static_cast<const T*>(p.out2) + off;
    const T* g = static_cast<const T*>(p.dout) + off;
    float d0 = 0.f, d2 = 0.f;
    for (int c = lane; c < p.Dv; c += 32) {
        const float gc = ld(g, c);
        d0 = fmaf(gc, ld(o, c), d0);
        d2 = fmaf(gc, ld(o2, c), d2);
    }
    d0 = warp_sum(d0);
    d2 = warp_sum(d2);
    if (lane == 0) {
        const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
        const float dd1 = fmaf(lam, d2, d0);
        const float lse1 = p.lse[row * 2], lse2 = p.lse[row * 2 + 1];
        float* st = p.stats + row * 4;
        if (p.log2_negated) {
            st[0] = -lse1 * 1.4426950408889634f;
            st[1] = -lse2 * 1.4426950408889634f;
            st[2] = -dd1;
            st[3] = -d2;
        } else {
            st[0] = lse1;
            st[1] = lse2;
            st[2] = dd1;
            st[3] = d2;
        }
    }
}

template <typename T>
int launch_grads(const BwdParams& p, cudaStream_t stream) {
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t qblocks = rows_per_head * p.B * p.H;
    const int64_t kblocks = rows_per_head * p.B * p.Hk;
    if (qblocks > 0x7fffffffLL) return -1;
    bwd_dq_kernel<T><<<(unsigned)qblocks, WARPS * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    bwd_dkdv_kernel<T><<<(unsigned)kblocks, WARPS * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    const int64_t rows = (int64_t)p.B * p.H * p.T;
    return launch_dlambda(p.stats, rows, p.stats + rows * 4, -1.0f, p.dlambda, stream);
}

template <typename T>
int launch(const BwdParams& p, cudaStream_t stream) {
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t qblocks = rows_per_head * p.B * p.H;
    const int64_t kblocks = rows_per_head * p.B * p.Hk;
    if (qblocks > 0x7fffffffLL) return -1;
    bwd_stats_kernel<T><<<(unsigned)qblocks, WARPS * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    bwd_dq_kernel<T><<<(unsigned)qblocks, WARPS * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    bwd_dkdv_kernel<T><<<(unsigned)kblocks, WARPS * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    const int64_t rows = (int64_t)p.B * p.H * p.T;
    return launch_dlambda(p.stats, rows, p.stats + rows * 4, -1.0f, p.dlambda, stream);
}

}  // namespace bwd

int launch_bwd_dlambda(const float* stats, int64_t rows, float sign, float* out,
                       cudaStream_t stream) {
    return bwd::launch_dlambda(stats, rows, const_cast<float*>(stats) + rows * 4, sign, out,
                               stream);
}

int launch_bwd_prep(const PrepParams& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.H * p.T;
    const int64_t blocks = (rows + bwd::WARPS - 1) / bwd::WARPS;
    if (blocks > 0x7fffffffLL) return -1;
    if (p.bf16)
        bwd::bwd_prep_kernel<__nv_bfloat16><<<(unsigned)blocks, bwd::WARPS * 32, 0, stream>>>(p);
    else
        bwd::bwd_prep_kernel<float><<<(unsigned)blocks, bwd::WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
int launch_bwd_simt_grads_f32(const BwdParams& p, cudaStream_t stream) {
    return bwd::launch_grads<float>(p, stream);
}
int launch_bwd_simt_grads_bf16(const BwdParams& p, cudaStream_t stream) {
    return bwd::launch_grads<__nv_bfloat16>(p, stream);
}
int launch_bwd_simt_f32(const BwdParams& p, cudaStream_t stream) { return bwd::launch<float>(p, stream); }
int launch_bwd_simt_bf16(const BwdParams& p, cudaStream_t stream) {
    return bwd::launch<__nv_bfloat16>(p, stream);
}

}  // namespace diffattn
