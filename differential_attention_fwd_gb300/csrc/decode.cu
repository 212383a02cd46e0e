// decode.cu -- differential attention for a few queries over a long key/value
// cache (decode), O = (softmax(Q1 K1^T / sqrt(D) + M) - lambda softmax(Q2 K2^T /
// sqrt(D) + M)) V with Tq new queries and Tk cached keys (paperleet
// "Differential Transformer Attention", Formula and conventions; the
// aiengineeringfromscratch lesson notes that the value cache is the decode
// cost to watch).  With the causal mask, query i sits at position
// Tk - Tq + i and sees keys j <= Tk - Tq + i.
//
// The work is bound by reading K1, K2 and V once (256 bytes per key and head
// for D = 64 in bf16), so it runs on the CUDA cores with coalesced loads and
// splits the keys of every head across CTAs:
//   pass 1 (partial): for each work item (b, key/value head, row chunk, split)
//     a CTA walks the item's key range in chunks of 256 keys (the grid is one
//     wave of persistent CTAs that take the items in turn): every thread scores one key against all
//     query rows of the CTA in both branches,
//     the block keeps an online softmax per (query, branch) in log2 units, and
//     every warp accumulates P V for its share of the keys, lanes spread over
//     the output columns.  The split's (max, sum, unnormalised O) go to the
//     workspace.
//   pass 2 (combine): one block per (b, h, query) merges the splits, forms
//     O1 / l1 - lambda O2 / l2 and applies the optional output epilogue.
// Query rows: the kv_group query heads that share a key/value head (grouped
// key/value heads, the DIFF V2 layout) contribute kv_group * Tq rows, row
// (i, q) = i * Tq + q for the group's i-th head; they are cut into row_chunks
// chunks of tq_bucket rows, so one pass over a head's cache serves up to
// tq_bucket rows of several heads.
#include "kernels.h"

#include <cmath>

namespace diffattn {
namespace dec {

constexpr int CHUNK = 256;     // keys per chunk = threads per block
constexpr int WARPS = CHUNK / 32;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16-byte vector of T unpacked to floats
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float* p, float* x) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* x) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// DPL consecutive output columns of a value row in one naturally aligned load
template <typename T, int DPL>
__device__ __forceinline__ void load_cols(const T* p, float* x) {
    if constexpr (sizeof(T) == 2 && DPL == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(w << 16);
        x[1] = __uint_as_float(w & 0xffff0000u);
    } else if constexpr (sizeof(T) == 2 && DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(w.x << 16); x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16); x[3] = __uint_as_float(w.y & 0xffff0000u);
    } else if constexpr (sizeof(T) == 2 && DPL == 8) {
        Vec<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(p), x);
    } else if constexpr (sizeof(T) == 4 && DPL == 2) {
        const float2 w = *reinterpret_cast<const float2*>(p);
        x[0] = w.x; x[1] = w.y;
    } else {
#pragma unroll
        for (int i = 0; i < DPL; i += 4) Vec<float>::load(reinterpret_cast<const float*>(p) + i, x + i);
    }
}

__device__ __forceinline__ float block_max_partial(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// exp2 that maps (-inf) - (-inf) to 0 weight instead of NaN
__device__ __forceinline__ float ex2_masked(float s, float m) {
    return (s == -INFINITY) ? 0.f : exp2f(s - m);
}

template <typename T, int D, int TQ>
__global__ void __launch_bounds__(CHUNK)
decode_partial_kernel(const DecodeParams p) {
    constexpr int DV = 2 * D;
    constexpr int DPL = DV / 32;                  // output columns per lane
    constexpr int NV = Vec<T>::N;
    extern __shared__ float sm[];
    float* qs = sm;                               // [TQ][2][D]
    float* sc = qs + TQ * 2 * D;                  // [CHUNK][TQ][2] scores, then weights
    float* red = sc + CHUNK * TQ * 2;             // [WARPS][TQ][2] partial max / sums
    float* stat = red + WARPS * TQ * 2;           // [TQ][2]: running max, running sum, scale
    float* alpha = stat + TQ * 2 * 2;             // [TQ][2]
    float* acc_red = alpha + TQ * 2;              // [WARPS][TQ][2][DV] (final reduction)

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    __shared__ int last_key[TQ];
    // Persistent: the grid holds as many CTAs as fit on the GPU at once, and
    // CTA c takes work items c, c + grid, ...; items are (unit, key split)
    // pairs of equal length, so no CTA has more than one item more than another.
    for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
    __syncthreads();    // the previous item's shared-memory reads are done
    const int split = item % p.splits;
    const int unit = item / p.splits;              // (b, key/value head, row chunk)
    const int rc = unit % p.row_chunks;
    const int bhk = unit / p.row_chunks;
    const int b = bhk / p.Hk;
    const int hk = bhk - b * p.Hk;
    const int k_begin = split * p.split_len;
    const int k_end = min(p.Tk, k_begin + p.split_len);
    const int n_rows = p.kv_group * p.Tq;          // query rows of this key/value head

    const T* k1 = static_cast<const T*>(p.k1) + b * p.s_k1[0] + hk * p.s_k1[1];
    const T* k2 = static_cast<const T*>(p.k2) + b * p.s_k2[0] + hk * p.s_k2[1];
    const T* v = static_cast<const T*>(p.v) + b * p.s_v[0] + hk * p.s_v[1];

    // query rows (rows past the group's last are zero and never written back)
    for (int i = tid; i < TQ * 2 * D; i += CHUNK) {
        const int r = i / (2 * D), br = (i / D) & 1, d = i % D;
        const int row = rc * TQ + r;
        float x = 0.f;
        if (row < n_rows) {
            const int h = hk * p.kv_group + row / p.Tq;
            const int q = row % p.Tq;
            x = br ? to_f(static_cast<const T*>(p.q2)[b * p.s_q2[0] + h * p.s_q2[1] + (int64_t)q * p.s_q2[2] + d])
                   : to_f(static_cast<const T*>(p.q1)[b * p.s_q1[0] + h * p.s_q1[1] + (int64_t)q * p.s_q1[2] + d]);
        }
        qs[i] = x;
    }

    if (tid < TQ * 2) {
        stat[2 * tid] = -INFINITY;   // running max (log2 units)
        stat[2 * tid + 1] = 0.f;     // running sum
    }
    // last visible key of each row; causal: row (i, q) sits at position Tk - Tq + q
    if (tid < TQ) last_key[tid] = p.causal ? p.Tk - p.Tq + (rc * TQ + tid) % p.Tq : p.Tk;
    float acc[TQ][2][DPL];
#pragma unroll
    for (int q = 0; q < TQ; ++q)
#pragma unroll
        for (int br = 0; br < 2; ++br)
#pragma unroll
            for (int c = 0; c < DPL; ++c) acc[q][br][c] = 0.f;
    __syncthreads();

    for (int c0 = k_begin; c0 < k_end; c0 += CHUNK) {
        // ---- scores: one key per thread, all queries, both branches
        const int key = c0 + tid;
        float s[TQ][2];
#pragma unroll
        for (int q = 0; q < TQ; ++q) s[q][0] = s[q][1] = 0.f;
        if (key < k_end) {
            const T* r1 = k1 + (int64_t)key * p.s_k1[2];
            const T* r2 = k2 + (int64_t)key * p.s_k2[2];
#pragma unroll
            for (int d0 = 0; d0 < D; d0 += NV) {
                float x1[NV], x2[NV];
                Vec<T>::load(r1 + d0, x1);
                Vec<T>::load(r2 + d0, x2);
#pragma unroll
                for (int q = 0; q < TQ; ++q)
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        s[q][0] = fmaf(qs[(q * 2 + 0) * D + d0 + e], x1[e], s[q][0]);
                        s[q][1] = fmaf(qs[(q * 2 + 1) * D + d0 + e], x2[e], s[q][1]);
                    }
            }
        }
#pragma unroll
        for (int q = 0; q < TQ; ++q) {
            const bool vis = key < k_end && key <= last_key[q];
#pragma unroll
            for (int br = 0; br < 2; ++br) {
                const float x = vis ? s[q][br] * p.scale_log2 : -INFINITY;
                s[q][br] = x;
                sc[(tid * TQ + q) * 2 + br] = x;
                const float wm = block_max_partial(x);
                if (lane == 0) red[(warp * TQ + q) * 2 + br] = wm;
            }
        }
        __syncthreads();
        // ---- new running max and the rescale factor, per (query, branch)
        if (tid < TQ * 2) {
            float cm = -INFINITY;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) cm = fmaxf(cm, red[w * TQ * 2 + tid]);
            const float m_old = stat[2 * tid];
            const float m_new = fmaxf(m_old, cm);
            alpha[tid] = (m_old == m_new) ? 1.f : exp2f(m_old - m_new);
            stat[2 * tid] = m_new;
        }
        __syncthreads();
        // ---- weights and their sums
#pragma unroll
        for (int q = 0; q < TQ; ++q)
#pragma unroll
            for (int br = 0; br < 2; ++br) {
                const float w = ex2_masked(s[q][br], stat[2 * (q * 2 + br)]);
                sc[(tid * TQ + q) * 2 + br] = w;
                const float ws = warp_sum(w);
                if (lane == 0) red[(warp * TQ + q) * 2 + br] = ws;
            }
        __syncthreads();
        if (tid < TQ * 2) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) sum += red[w * TQ * 2 + tid];
            stat[2 * tid + 1] = stat[2 * tid + 1] * alpha[tid] + sum;
        }
        // ---- O += P V: warp w takes keys w, w + 8, ...; lane takes DPL columns
#pragma unroll
        for (int q = 0; q < TQ; ++q)
#pragma unroll
            for (int br = 0; br < 2; ++br) {
                const float a = alpha[q * 2 + br];
#pragma unroll
                for (int c = 0; c < DPL; ++c) acc[q][br][c] *= a;
            }
        const int nk = min(CHUNK, k_end - c0);
        int t = warp;
        // UNROLL value rows in flight per warp before they are used
        constexpr int UNROLL = (TQ * DPL <= 16) ? 8 : 4;
        for (; t + (UNROLL - 1) * WARPS < nk; t += UNROLL * WARPS) {
            float x[UNROLL][DPL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                load_cols<T, DPL>(v + (int64_t)(c0 + t + u * WARPS) * p.s_v[2] + lane * DPL, x[u]);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
#pragma unroll
                for (int q = 0; q < TQ; ++q)
#pragma unroll
                    for (int br = 0; br < 2; ++br) {
                        const float w = sc[((t + u * WARPS) * TQ + q) * 2 + br];
#pragma unroll
                        for (int c = 0; c < DPL; ++c) acc[q][br][c] = fmaf(w, x[u][c], acc[q][br][c]);
                    }
        }
        for (; t < nk; t += WARPS) {
            float x[DPL];
            load_cols<T, DPL>(v + (int64_t)(c0 + t) * p.s_v[2] + lane * DPL, x);
#pragma unroll
            for (int q = 0; q < TQ; ++q)
#pragma unroll
                for (int br = 0; br < 2; ++br) {
                    const float w = sc[(t * TQ + q) * 2 + br];
#pragma unroll
                    for (int c = 0; c < DPL; ++c) acc[q][br][c] = fmaf(w, x[c], acc[q][br][c]);
                }
        }
        __syncthreads();
    }

    // ---- reduce the warps' accumulators and write the split's partial result
#pragma unroll
    for (int q = 0; q < TQ; ++q)
#pragma unroll
        for (int br = 0; br < 2; ++br)
#pragma unroll
            for (int c = 0; c < DPL; ++c)
                acc_red[((warp * TQ + q) * 2 + br) * DV + lane * DPL + c] = acc[q][br][c];
    __syncthreads();
    float* part = p.work + ((int64_t)unit * p.splits + split) * TQ * (4 + 2 * DV);
    for (int i = tid; i < TQ * 2 * DV; i += CHUNK) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) sum += acc_red[w * TQ * 2 * DV + i];
        const int q = i / (2 * DV);
        const int rest = i - q * 2 * DV;
        part[q * (4 + 2 * DV) + 4 + rest] = sum;
    }
    if (tid < TQ * 2) {
        const int q = tid >> 1, br = tid & 1;
        part[q * (4 + 2 * DV) + 2 * br] = stat[2 * tid];
        part[q * (4 + 2 * DV) + 2 * br + 1] = stat[2 * tid + 1];
    }
    }   // work items
}

// One block per (b, h, query), one thread per output column.
template <typename T, int D, int TQ>
__global__ void __launch_bounds__(2 * D)
decode_combine_kernel(const DecodeParams p) {
    constexpr int DV = 2 * D;
    __shared__ float red[DV / 32];
    const int c = threadIdx.x;
    const int q = blockIdx.x % p.Tq;
    const int bh = blockIdx.x / p.Tq;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    // where the partial kernel kept this (head, query) row
    const int hk = h / p.kv_group;
    const int row = (h - hk * p.kv_group) * p.Tq + q;
    const int unit = (b * p.Hk + hk) * p.row_chunks + row / TQ;
    const float* part = p.work + (int64_t)unit * p.splits * TQ * (4 + 2 * DV) + (row % TQ) * (4 + 2 * DV);
    const int64_t sstride = (int64_t)TQ * (4 + 2 * DV);
    float val[2];
#pragma unroll
    for (int br = 0; br < 2; ++br) {
        float M = -INFINITY;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, part[s * sstride + 2 * br]);
        float L = 0.f, O = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float w = ex2_masked(part[s * sstride + 2 * br], M);
            L = fmaf(part[s * sstride + 2 * br + 1], w, L);
            O = fmaf(part[s * sstride + 4 + br * DV + c], w, O);
        }
        val[br] = O / L;
    }
    const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
    float r = __fsub_rn(val[0], __fmul_rn(lam, val[1]));
    if (p.norm != kNormNone) {
        auto block_sum = [&](float x) {
            x = warp_sum(x);
            __syncthreads();
            if ((c & 31) == 0) red[c >> 5] = x;
            __syncthreads();
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < DV / 32; ++w) t += red[w];
            return t;
        };
        float mu = 0.f, rinv;
        if (p.norm == kNormRms) {
            rinv = rsqrtf(block_sum(r * r) / DV + p.norm_eps);
        } else {
            mu = block_sum(r) / DV;
            rinv = rsqrtf(block_sum((r - mu) * (r - mu)) / DV + p.norm_eps);
        }
        r = (r - mu) * rinv;
        if (p.norm_weight) r *= __ldg(p.norm_weight + h * DV + c);
        if (p.norm_bias) r += __ldg(p.norm_bias + h * DV + c);
    }
    r *= p.out_scale;
    T* out = static_cast<T*>(p.out) + b * p.s_o[0] + h * p.s_o[1] + (int64_t)q * p.s_o[2];
    if constexpr (sizeof(T) == 4) {
        out[c] = r;
    } else {
        out[c] = __float2bfloat16_rn(r);
    }
}

template <typename T, int D, int TQ>
int launch_tq(const DecodeParams& p, cudaStream_t stream) {
    constexpr int DV = 2 * D;
    const size_t smem = sizeof(float) * (TQ * 2 * D + CHUNK * TQ * 2 + WARPS * TQ * 2 + TQ * 4 +
                                         TQ * 2 + WARPS * TQ * 2 * DV);
    if (cudaFuncSetAttribute(decode_partial_kernel<T, D, TQ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    // one wave of CTAs, as many as are resident at once
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_partial_kernel<T, D, TQ>, CHUNK,
                                                      smem) != cudaSuccess)
        return -1;
    const int64_t slots = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(p.total_items < slots ? p.total_items : slots);
    decode_partial_kernel<T, D, TQ><<<grid, CHUNK, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    decode_combine_kernel<T, D, TQ><<<p.B * p.H * p.Tq, DV, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T, int D>
int launch_d(const DecodeParams& p, cudaStream_t stream) {
    if (p.tq_bucket == 1) return launch_tq<T, D, 1>(p, stream);
    if (p.tq_bucket == 2) return launch_tq<T, D, 2>(p, stream);
    if (p.tq_bucket == 4) return launch_tq<T, D, 4>(p, stream);
    if constexpr (D <= 64) {
        if (p.tq_bucket == 8) return launch_tq<T, D, 8>(p, stream);
    }
    return -1;
}

template <typename T>
int launch_t(const DecodeParams& p, cudaStream_t stream) {
    if (p.D == 32) return launch_d<T, 32>(p, stream);
    if (p.D == 64) return launch_d<T, 64>(p, stream);
    if (p.D == 128) return launch_d<T, 128>(p, stream);
    return -1;
}

}  // namespace dec

int decode_max_rows(int D) { return D <= 64 ? 8 : 4; }

int decode_tq_bucket(int rows, int D) {
    const int cap = decode_max_rows(D);
    for (int t = 1; t <= cap; t *= 2)
        if (rows <= t) return t;
    return 0;
}

size_t decode_work_floats(int64_t units, int splits, int tq_bucket, int64_t D) {
    return (size_t)units * splits * tq_bucket * (4 + 4 * D);
}

int launch_decode(const DecodeParams& p, cudaStream_t stream) {
    return p.bf16 ? dec::launch_t<__nv_bfloat16>(p, stream) : dec::launch_t<float>(p, stream);
}

}  // namespace diffattn
