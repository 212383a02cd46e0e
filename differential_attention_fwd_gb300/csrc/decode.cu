// decode.cu -- differential attention for a few queries over a long key/value
// cache (decode), O = (softmax(Q1 K1^T / sqrt(D) + M) - lambda softmax(Q2 K2^T /
// sqrt(D) + M)) V with Tq new queries and Tk cached keys (paperleet
// "Differential Transformer Attention", Formula and conventions; the
// aiengineeringfromscratch lesson notes that the value cache is the decode
// cost to watch).  With the causal mask, query i sits at position
// Tk - Tq + i and sees keys j <= Tk - Tq + i.
//
// The work is bound by reading K1, K2 and V once (512 bytes per key and head
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
// For bf16, D = 64 and dense cache rows, pass 1 has two faster forms: the
// staged kernel below (cp.async ring) for one or two query rows per CTA, and
// for four to sixteen rows the tensor-core pass in decode_tc.cu (units of 16
// rows, and the DIFF V2 head D = 128, run on that pass only).
// Query rows: the kv_group query heads that share a key/value head (grouped
// key/value heads, the DIFF V2 layout) contribute kv_group * Tq rows, row
// (i, q) = i * Tq + q for the group's i-th head; they are cut into row_chunks
// chunks of tq_bucket rows, so one pass over a head's cache serves up to
// tq_bucket rows of several heads.
#include "kernels.h"
#include "ptx.cuh"
#include "pdl.cuh"

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
    pdl_launch_dependents();
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

// One block per (b, h, query), one thread per output column.  Launched as a
// programmatic dependent of the first pass: its blocks may become resident
// while the first pass runs and start reading as soon as it completes.
template <typename T, int D, int TQ>
__global__ void __launch_bounds__(2 * D)
decode_combine_kernel(const DecodeParams p) {
    constexpr int DV = 2 * D;
    __shared__ float red[DV / 32];
    pdl_wait();
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
    // both branches per split, so that each loop's loads are in flight together
    float M[2] = {-INFINITY, -INFINITY};
#pragma unroll 8
    for (int s = 0; s < p.splits; ++s) {
        M[0] = fmaxf(M[0], part[s * sstride]);
        M[1] = fmaxf(M[1], part[s * sstride + 2]);
    }
    float L[2] = {0.f, 0.f}, O[2] = {0.f, 0.f};
#pragma unroll 8
    for (int s = 0; s < p.splits; ++s) {
        const float* ps = part + s * sstride;
#pragma unroll
        for (int br = 0; br < 2; ++br) {
            const float w = ex2_masked(ps[2 * br], M[br]);
            L[br] = fmaf(ps[2 * br + 1], w, L[br]);
            O[br] = fmaf(ps[4 + br * DV + c], w, O[br]);
        }
    }
    const float val[2] = {O[0] / L[0], O[1] / L[1]};
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

// ---------------------------------------------------------------------------
// First pass with asynchronous staging (bf16, D = 64, key and value rows dense
// along the sequence): every thread of the CTA copies its share of a chunk of
// 64 keys (K1, K2 and V rows) into a ring of shared-memory stages with
// cp.async, two chunks ahead of the chunk being computed and across the CTA's
// work items, so the compute never waits on HBM latency; two CTAs share an SM,
// so one computes while the other waits at a barrier.  K rows are
// stored with their 16-byte pieces XOR-swizzled by (row mod 8), so that the
// thread-per-key reads of a warp (32 rows, one piece each) hit distinct banks.
// Per chunk: thread (key, branch) scores its key against the TQ query rows of
// its branch; the block forms the online-softmax statistics; warp w
// accumulates P V for keys w, w + 8, ... with the lanes over the columns.  The
// partial results have the layout the combine pass reads.
namespace as {

constexpr int CH = 64;                  // keys per chunk
constexpr int THREADS = 2 * CH;         // 2 branches x CH keys
constexpr int WARPS = THREADS / 32;
constexpr int WPB = WARPS / 2;          // warps per branch
constexpr int HDIM = 64;
constexpr int DV = 2 * HDIM;
constexpr int KROW = HDIM * 2;          // bytes of one bf16 key row (128)
constexpr int VROW = DV * 2;            // bytes of one bf16 value row (256)
constexpr int STAGE = CH * (2 * KROW + VROW);   // 32 KB
constexpr int NST = 2;                  // stages: one chunk in flight ahead (three CTAs fit
                                        // an SM: at Tq = 1 over 8192 keys 0.84 of the copy
                                        // bandwidth, against 0.74 with three stages and two CTAs)

template <int TQ>
constexpr size_t smem_bytes() {
    return (size_t)NST * STAGE +
           sizeof(float) * (TQ * 2 * HDIM + CH * TQ * 2 + WARPS * TQ * 2 + TQ * 4 + TQ * 2 +
                            WARPS * TQ * 2 * DV) + 16 * TQ + 128;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The CTA's sequence of chunks: item it (the CTA's k-th), chunk c of it.
struct Cursor {
    int item = 0, c = 0, n = 0;        // n: chunks of the item; item >= total when done
    int k_begin = 0, k_end = 0;
    __device__ void set(const DecodeParams& p, int it) {
        item = it;
        c = 0;
        if (it < p.total_items) {
            const int split = it % p.splits;
            k_begin = split * p.split_len;
            k_end = min(p.Tk, k_begin + p.split_len);
            n = (k_end - k_begin + CH - 1) / CH;
        } else {
            n = 0;
        }
    }
    __device__ bool done(const DecodeParams& p) const { return item >= p.total_items; }
    __device__ void next(const DecodeParams& p) {
        if (++c >= n) set(p, item + gridDim.x);
    }
};

template <int TQ>
__global__ void __launch_bounds__(THREADS, 3) decode_async_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* stages = smem_raw;                                    // [NST][K1 | K2 | V]
    float* qs = reinterpret_cast<float*>(smem_raw + NST * STAGE);  // [TQ][2][HDIM]
    float* sc = qs + TQ * 2 * HDIM;                                // [CH][TQ][2]
    float* red = sc + CH * TQ * 2;                                 // [WARPS][TQ]: per-branch partials
    float* stat = red + WARPS * TQ * 2;                            // [TQ][2]: max, sum
    float* alpha = stat + TQ * 4;                                  // [TQ][2]
    float* acc_red = alpha + TQ * 2;                               // [WARPS][TQ][2][DV]
    int* last_key = reinterpret_cast<int*>(acc_red + WARPS * TQ * 2 * DV);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kk = tid & (CH - 1);          // this thread's key within the chunk
    pdl_launch_dependents();
    const int br = tid / CH;                // and its branch
    const __nv_bfloat16* K1 = static_cast<const __nv_bfloat16*>(p.k1);
    const __nv_bfloat16* K2 = static_cast<const __nv_bfloat16*>(p.k2);
    const __nv_bfloat16* Vv = static_cast<const __nv_bfloat16*>(p.v);

    // copy chunk `cur` into stage st: K rows as 8 swizzled 16-byte pieces,
    // V rows as 16 plain pieces; rows past the item's keys are zero-filled
    auto issue = [&](const Cursor& cur, int st) {
        const int unit = cur.item / p.splits;
        const int bhk = unit / p.row_chunks;
        const int b = bhk / p.Hk, hk = bhk - b * p.Hk;
        const int key0 = cur.k_begin + cur.c * CH;
        const char* k1 = reinterpret_cast<const char*>(K1 + b * p.s_k1[0] + hk * p.s_k1[1]);
        const char* k2 = reinterpret_cast<const char*>(K2 + b * p.s_k2[0] + hk * p.s_k2[1]);
        const char* vv = reinterpret_cast<const char*>(Vv + b * p.s_v[0] + hk * p.s_v[1]);
        uint8_t* base = stages + st * STAGE;
#pragma unroll
        for (int i = 0; i < CH * 8 / THREADS; ++i) {        // K pieces: 8 per row
            const int id = tid + i * THREADS;
            const int r = id >> 3, j = id & 7;
            const int key = key0 + r;
            const bool ok = key < cur.k_end;
            const int64_t off = (int64_t)(ok ? key : 0) * KROW + j * 16;
            const int dst = r * KROW + ((j ^ (r & 7)) << 4);
            cp_async16(base + dst, k1 + off, ok);
            cp_async16(base + CH * KROW + dst, k2 + off, ok);
        }
#pragma unroll
        for (int i = 0; i < CH * 16 / THREADS; ++i) {       // V pieces: 16 per row
            const int id = tid + i * THREADS;
            const int r = id >> 4, j = id & 15;
            const int key = key0 + r;
            const bool ok = key < cur.k_end;
            cp_async16(base + 2 * CH * KROW + r * VROW + j * 16,
                       vv + (int64_t)(ok ? key : 0) * VROW + j * 16, ok);
        }
    };

    Cursor icur, ccur;                 // issue and compute positions
    icur.set(p, blockIdx.x);
    ccur = icur;
#pragma unroll
    for (int s0 = 0; s0 < NST - 1; ++s0) {
        if (!icur.done(p)) {
            issue(icur, s0);
            icur.next(p);
        }
        cp_async_commit();
    }
    float acc[TQ][2][4];
    int st = 0;                        // stage of the chunk being computed
    int ist = NST - 1;                 // stage the next issue goes to
    while (!ccur.done(p)) {
        if (!icur.done(p)) {
            issue(icur, ist);
            icur.next(p);
        }
        cp_async_commit();
        if (++ist == NST) ist = 0;
        cp_async_wait<NST - 1>();
        __syncthreads();
        const int unit = ccur.item / p.splits;
        const int rc = unit % p.row_chunks;
        const int n_rows = p.kv_group * p.Tq;
        if (ccur.c == 0) {
            // a new item: its query rows, statistics and accumulators
            const int bhk = unit / p.row_chunks;
            const int b = bhk / p.Hk, hk = bhk - b * p.Hk;
            for (int i = tid; i < TQ * 2 * HDIM; i += THREADS) {
                const int r = i / (2 * HDIM), qb = (i / HDIM) & 1, d = i % HDIM;
                const int row = rc * TQ + r;
                float x = 0.f;
                if (row < n_rows) {
                    const int h = hk * p.kv_group + row / p.Tq;
                    const int q = row % p.Tq;
                    x = qb ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.q2)[
                                 b * p.s_q2[0] + h * p.s_q2[1] + (int64_t)q * p.s_q2[2] + d])
                           : __bfloat162float(static_cast<const __nv_bfloat16*>(p.q1)[
                                 b * p.s_q1[0] + h * p.s_q1[1] + (int64_t)q * p.s_q1[2] + d]);
                }
                qs[i] = x;
            }
            if (tid < TQ * 2) {
                stat[2 * tid] = -INFINITY;
                stat[2 * tid + 1] = 0.f;
            }
            if (tid < TQ) last_key[tid] = p.causal ? p.Tk - p.Tq + (rc * TQ + tid) % p.Tq : p.Tk;
#pragma unroll
            for (int q = 0; q < TQ; ++q)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[q][b2][c] = 0.f;
            __syncthreads();
        }
        const uint8_t* stg = stages + st * STAGE;
        const int key = ccur.k_begin + ccur.c * CH + kk;
        // ---- scores: this thread's key against the TQ rows of its branch
        float s[TQ];
#pragma unroll
        for (int q = 0; q < TQ; ++q) s[q] = 0.f;
        {
            const uint8_t* krow = stg + br * CH * KROW + kk * KROW;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float x[8];
                Vec<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(krow + ((j ^ (kk & 7)) << 4)), x);
#pragma unroll
                for (int q = 0; q < TQ; ++q)
#pragma unroll
                    for (int e = 0; e < 8; ++e) s[q] = fmaf(qs[(q * 2 + br) * HDIM + j * 8 + e], x[e], s[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < TQ; ++q) {
            const bool vis = key < ccur.k_end && key <= last_key[q];
            s[q] = vis ? s[q] * p.scale_log2 : -INFINITY;
            const float wm = block_max_partial(s[q]);
            if (lane == 0) red[warp * TQ + q] = wm;
        }
        __syncthreads();
        // ---- new running max and rescale factor per (row, branch): the first
        // WPB warps hold branch 1, the others branch 2
        if (tid < TQ * 2) {
            const int q = tid >> 1, b2 = tid & 1;
            float cm = -INFINITY;
#pragma unroll
            for (int w = 0; w < WPB; ++w) cm = fmaxf(cm, red[(b2 * WPB + w) * TQ + q]);
            const float m_old = stat[2 * tid];
            const float m_new = fmaxf(m_old, cm);
            alpha[tid] = (m_old == m_new) ? 1.f : exp2f(m_old - m_new);
            stat[2 * tid] = m_new;
        }
        __syncthreads();
        // ---- weights and their sums
#pragma unroll
        for (int q = 0; q < TQ; ++q) {
            const float w = ex2_masked(s[q], stat[2 * (q * 2 + br)]);
            sc[(kk * TQ + q) * 2 + br] = w;
            const float ws = warp_sum(w);
            if (lane == 0) red[warp * TQ + q] = ws;
        }
        __syncthreads();
        if (tid < TQ * 2) {
            const int q = tid >> 1, b2 = tid & 1;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < WPB; ++w) sum += red[(b2 * WPB + w) * TQ + q];
            stat[2 * tid + 1] = stat[2 * tid + 1] * alpha[tid] + sum;
        }
        // ---- O += P V: warp w takes keys w, w + WARPS, ...; lane takes 4 columns
#pragma unroll
        for (int q = 0; q < TQ; ++q)
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
                const float a = alpha[q * 2 + b2];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[q][b2][c] *= a;
            }
        {
            const uint8_t* vrows = stg + 2 * CH * KROW + lane * 8;
#pragma unroll 4
            for (int t = warp; t < CH; t += WARPS) {
                float x[4];
                load_cols<__nv_bfloat16, 4>(reinterpret_cast<const __nv_bfloat16*>(vrows + t * VROW), x);
#pragma unroll
                for (int q = 0; q < TQ; ++q)
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2) {
                        const float w = sc[(t * TQ + q) * 2 + b2];
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[q][b2][c] = fmaf(w, x[c], acc[q][b2][c]);
                    }
            }
        }
        if (ccur.c == ccur.n - 1) {
            // ---- the item's last chunk: reduce the warps' accumulators and
            // write the split's partial result
#pragma unroll
            for (int q = 0; q < TQ; ++q)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc_red[((warp * TQ + q) * 2 + b2) * DV + lane * 4 + c] = acc[q][b2][c];
            __syncthreads();
            const int split = ccur.item % p.splits;
            float* part = p.work + ((int64_t)unit * p.splits + split) * TQ * (4 + 2 * DV);
            for (int i = tid; i < TQ * 2 * DV; i += THREADS) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < WARPS; ++w) sum += acc_red[w * TQ * 2 * DV + i];
                const int q = i / (2 * DV);
                part[q * (4 + 2 * DV) + 4 + (i - q * 2 * DV)] = sum;
            }
            if (tid < TQ * 2) {
                const int q = tid >> 1, b2 = tid & 1;
                part[q * (4 + 2 * DV) + 2 * b2] = stat[2 * tid];
                part[q * (4 + 2 * DV) + 2 * b2 + 1] = stat[2 * tid + 1];
            }
        }
        __syncthreads();   // the stage and the shared statistics are free again
        if (++st == NST) st = 0;
        ccur.next(p);
    }
    cp_async_wait<0>();
}

}  // namespace as

// The combine pass as a programmatic dependent of the first pass just
// launched on `stream` (which signals at its start that it may launch).
template <typename T, int D, int TQ>
int launch_combine(const DecodeParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.H * p.Tq));
    cfg.blockDim = dim3(2 * D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<T, D, TQ>, p) == cudaSuccess ? 0 : -1;
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
    // the staged first pass for up to two query rows per CTA (at Tq = 1 over
    // an 8192-key cache: 0.73 of the copy bandwidth against 0.63); with more
    // rows its per-chunk arithmetic outweighs the hidden latency, and the
    // per-thread-load pass above runs faster
    if constexpr (sizeof(T) == 2 && D == as::HDIM && TQ <= 2) {
        if (p.dense_kv) {
            constexpr size_t sm2 = as::smem_bytes<TQ>();
            if (cudaFuncSetAttribute(as::decode_async_kernel<TQ>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2) != cudaSuccess)
                return -1;
            int per_sm2 = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, as::decode_async_kernel<TQ>,
                                                              as::THREADS, sm2) != cudaSuccess)
                return -1;
            const int64_t slots2 = (int64_t)sms * (per_sm2 > 0 ? per_sm2 : 1);
            const int g2 = (int)(p.total_items < slots2 ? p.total_items : slots2);
            as::decode_async_kernel<TQ><<<g2, as::THREADS, sm2, stream>>>(p);
            if (cudaGetLastError() != cudaSuccess) return -1;
            return launch_combine<T, D, TQ>(p, stream);
        }
    }
    // four or eight query rows per CTA: the tensor-core first pass
    if constexpr (sizeof(T) == 2 && D == 64 && TQ >= 4) {
        if (p.tc_ok) {
            DecodeParams q = p;             // the pass's own split of the keys
            if (launch_decode_tc_first_pass(&q, stream) != 0) return -1;
            return launch_combine<T, D, TQ>(q, stream);
        }
    }
    decode_partial_kernel<T, D, TQ><<<grid, CHUNK, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    return launch_combine<T, D, TQ>(p, stream);
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

// Units of up to 16 rows on the tensor cores only (the DIFF V2 head, D = 128,
// or D = 64 with more than 8 rows per key/value head; value width 128 either
// way): the tensor-core first pass, then the combine pass of value width 128
// (its instance for D = 64).
template <int TQ>
int launch_tc_only_tq(const DecodeParams& p, cudaStream_t stream) {
    DecodeParams q = p;
    if (launch_decode_tc_first_pass(&q, stream) != 0) return -1;
    return launch_combine<__nv_bfloat16, 64, TQ>(q, stream);
}

int launch_tc_only(const DecodeParams& p, cudaStream_t stream) {
    if (!p.tc_ok || !p.bf16 || (p.D != 64 && p.D != 128)) return -1;
    if (p.tq_bucket == 1) return launch_tc_only_tq<1>(p, stream);
    if (p.tq_bucket == 2) return launch_tc_only_tq<2>(p, stream);
    if (p.tq_bucket == 4) return launch_tc_only_tq<4>(p, stream);
    if (p.tq_bucket == 8) return launch_tc_only_tq<8>(p, stream);
    if (p.tq_bucket == 16) return launch_tc_only_tq<16>(p, stream);
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
    if (p.tc_only) return dec::launch_tc_only(p, stream);
    return p.bf16 ? dec::launch_t<__nv_bfloat16>(p, stream) : dec::launch_t<float>(p, stream);
}

}  // namespace diffattn
