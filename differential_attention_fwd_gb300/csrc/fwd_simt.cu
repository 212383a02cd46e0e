// fwd_simt.cu -- differential-attention forward on the CUDA cores.
//
// O = (softmax(Q1 K1^T / sqrt(D) + M) - lambda softmax(Q2 K2^T / sqrt(D) + M)) V
// (paperleet "Differential Transformer Attention", Formula and conventions).
//
// The general path: fp32 inputs (exact fp32 arithmetic, expf), and bf16
// inputs of any shape the tensor-core kernel does not take (D != 64,
// unaligned strides, a value width other than the tensor-core kernel's).  One
// warp owns one query row.  Keys are visited in chunks of 32, one key per lane
// for the two dot products; each branch keeps a streaming-softmax state
// (running max, running sum) and its own output accumulator, each lane holding
// the output columns lane, lane+32, ...  Masked keys (causal: key > query +
// kv_off) are skipped.  With grouped key/value heads, query head h reads
// key/value head h / kv_group.
#include "kernels.h"

#include <cmath>

namespace diffattn {
namespace simt {

constexpr int WARPS = 4;          // query rows per block
constexpr int MAX_D = 128;
constexpr int MAX_DV = 256;
constexpr int OPL = MAX_DV / 32;  // output columns per lane

__device__ __forceinline__ float load(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store(__nv_bfloat16* p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

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

template <typename T>
__global__ void __launch_bounds__(WARPS * 32)
diffattn_fwd_simt_kernel(const SimtParams p) {
    __shared__ float qs[WARPS][2][MAX_D];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t blk = blockIdx.x;
    const int64_t bh = blk / rows_per_head;
    const int b = (int)(bh / p.H);
    const int h = (int)(bh - (int64_t)b * p.H);
    const int i = (int)((blk - bh * rows_per_head) * WARPS + warp);
    if (i >= p.T) return;   // whole warp leaves together

    const T* q1 = static_cast<const T*>(p.q1) + b * p.s_q1[0] + h * p.s_q1[1];
    const int hk = h / p.kv_group;   // key/value head of this query head
    const T* k1 = static_cast<const T*>(p.k1) + b * p.s_k1[0] + hk * p.s_k1[1];
    const T* q2 = static_cast<const T*>(p.q2) + b * p.s_q2[0] + h * p.s_q2[1];
    const T* k2 = static_cast<const T*>(p.k2) + b * p.s_k2[0] + hk * p.s_k2[1];
    const T* v = static_cast<const T*>(p.v) + b * p.s_v[0] + hk * p.s_v[1];
    T* out = static_cast<T*>(p.out) + b * p.s_o[0] + h * p.s_o[1] + (int64_t)i * p.s_o[2];
    const int D = p.D;
    const int Dv = p.Dv;

    for (int d = lane; d < D; d += 32) {
        qs[warp][0][d] = load(q1, (int64_t)i * p.s_q1[2] + d);
        qs[warp][1][d] = load(q2, (int64_t)i * p.s_q2[2] + d);
    }
    __syncwarp();

    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float o1[OPL], o2[OPL];
#pragma unroll
    for (int r = 0; r < OPL; ++r) o1[r] = o2[r] = 0.f;

    // keys [0, kend) are visible; the causal offset keeps kend >= 1
    const int kend = p.causal ? min(i + p.kv_off + 1, p.Tk) : p.Tk;
    for (int k0 = 0; k0 < kend; k0 += 32) {
        const int key = k0 + lane;
        const bool valid = key < kend;
        float s1 = -INFINITY, s2 = -INFINITY;
        if (valid) {
            float d1 = 0.f, d2 = 0.f;
            const int64_t r1 = (int64_t)key * p.s_k1[2];
            const int64_t r2 = (int64_t)key * p.s_k2[2];
            for (int d = 0; d < D; ++d) {
                d1 = fmaf(qs[warp][0][d], load(k1, r1 + d), d1);
                d2 = fmaf(qs[warp][1][d], load(k2, r2 + d), d2);
            }
            s1 = d1 * p.scale;
            s2 = d2 * p.scale;
        }
        // chunk k0 always holds at least one visible key (k0 < kend)
        const float n1 = fmaxf(m1, warp_max(s1));
        const float n2 = fmaxf(m2, warp_max(s2));
        const float a1 = expf(m1 - n1);
        const float a2 = expf(m2 - n2);
        const float p1 = valid ? expf(s1 - n1) : 0.f;
        const float p2 = valid ? expf(s2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(p1);
        l2 = l2 * a2 + warp_sum(p2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int r = 0; r < OPL; ++r) {
            o1[r] *= a1;
            o2[r] *= a2;
        }
        const int nk = min(32, kend - k0);
        for (int t = 0; t < nk; ++t) {
            const float w1 = __shfl_sync(0xffffffffu, p1, t);
            const float w2 = __shfl_sync(0xffffffffu, p2, t);
            const int64_t vr = (int64_t)(k0 + t) * p.s_v[2];
#pragma unroll
            for (int r = 0; r < OPL; ++r) {
                const int c = lane + 32 * r;
                if (c < Dv) {
                    const float vv = load(v, vr + c);
                    o1[r] = fmaf(w1, vv, o1[r]);
                    o2[r] = fmaf(w2, vv, o2[r]);
                }
            }
        }
    }
    const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
    const float inv1 = 1.0f / l1;
    const float inv2 = 1.0f / l2;
    if (p.out2) {
        // training outputs: A_2 V and the natural-log log-sum-exp of each branch
        T* o2row = static_cast<T*>(p.out2) + b * p.s_o[0] + h * p.s_o[1] + (int64_t)i * p.s_o[2];
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const int c = lane + 32 * k;
            if (c < Dv) store(o2row, c, __fmul_rn(o2[k], inv2));
        }
        if (lane == 0) {
            float* lse = p.lse + (((int64_t)b * p.H + h) * p.T + i) * 2;
            lse[0] = m1 + logf(l1);
            lse[1] = m2 + logf(l2);
        }
    }
    float r[OPL];
#pragma unroll
    for (int k = 0; k < OPL; ++k) {
        const float a = __fmul_rn(o1[k], inv1);
        const float bb = __fmul_rn(o2[k], inv2);
        r[k] = __fsub_rn(a, __fmul_rn(lam, bb));
    }
    if (p.norm != kNormNone) {
        // per-head normalisation over the row's 2D channels (spread over lanes)
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const int c = lane + 32 * k;
            if (c < Dv) part += (p.norm == kNormRms) ? r[k] * r[k] : r[k];
        }
        const float tot = warp_sum(part);
        float mu = 0.f, rinv;
        if (p.norm == kNormRms) {
            rinv = rsqrtf(tot / Dv + p.norm_eps);
        } else {
            mu = tot / Dv;
            float dev = 0.f;
#pragma unroll
            for (int k = 0; k < OPL; ++k) {
                const int c = lane + 32 * k;
                if (c < Dv) dev += (r[k] - mu) * (r[k] - mu);
            }
            rinv = rsqrtf(warp_sum(dev) / Dv + p.norm_eps);
        }
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const int c = lane + 32 * k;
            if (c < Dv) {
                float y = (r[k] - mu) * rinv;
                if (p.norm_weight) y *= __ldg(p.norm_weight + h * Dv + c);
                if (p.norm_bias) y += __ldg(p.norm_bias + h * Dv + c);
                r[k] = y;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < OPL; ++k) {
        const int c = lane + 32 * k;
        if (c < Dv) store(out, c, p.out_scale == 1.0f ? r[k] : r[k] * p.out_scale);
    }
}

template <typename T>
int launch(const SimtParams& p, cudaStream_t stream) {
    const int64_t rows_per_head = (p.T + WARPS - 1) / WARPS;
    const int64_t blocks = rows_per_head * p.B * p.H;
    if (blocks > 0x7fffffffLL) return -1;
    diffattn_fwd_simt_kernel<T><<<(unsigned)blocks, WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace simt

int launch_fwd_simt_f32(const SimtParams& p, cudaStream_t stream) {
    return simt::launch<float>(p, stream);
}
int launch_fwd_simt_bf16(const SimtParams& p, cudaStream_t stream) {
    return simt::launch<__nv_bfloat16>(p, stream);
}

}  // namespace diffattn
