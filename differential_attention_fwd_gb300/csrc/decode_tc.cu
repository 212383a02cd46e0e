// decode_tc.cu -- the first pass of the decode (a few queries over a long
// key/value cache) on the tensor cores, for query rows that share a key/value
// head: bf16, value width 128, dense cache rows, up to 16 rows per unit (the
// MMA's N: the query heads of a grouped key/value head, DIFF V2's layout, or
// several new queries).  Two head shapes: D = 64 (V = 2D) with 4, 8 or 16 rows
// per unit, and the DIFF V2 head D = 128 (V = D; aiengineeringfromscratch
// lesson, "V1 contre V2") with 1 to 16, whose two branches share one key tensor
// (one key tile per stage serves both score products).  It writes split
// partials in the layout of the CUDA-core first pass in decode.cu for a value
// width of 128, which the combine pass there merges.
//
// Work: a unit is (b, key/value head, row chunk); its keys form tpu tiles of
// 128.  The units' tiles are laid end to end and every CTA streams one
// contiguous range of them (equal lengths to within a tile), in segments cut
// at unit boundaries; each segment leaves one partial result, in the slot
// given by its CTA's place among the unit's CTAs, and the CTA with a unit's
// last segment marks the unit's unused slots empty.
//
// Per segment, per tile of 128 keys: TMA brings K1, K2 (or the one shared key
// tile, in 64-column panels at D = 128) and V into shared memory in the
// 128-byte swizzled layout of the MMA operands, two tiles ahead
// (keys past the segment's end are loaded but get zero weight; past the
// cache's end they read as zero).  Then
//   S_b^T = K_b Q_b^T        (tcgen05, M = 128 keys in TMEM lanes, N = 16 rows,
//                             the rows past the unit's TQ are zero)
// each thread (one key) takes its scores for every row, P = 2^(S * scale - m)
// against the running row max m, and writes P^T as bf16 to shared memory;
//   [O_1^T O_2^T] += V^T [P_1^T P_2^T]
//                            (tcgen05, A = V^T read MN-major from the staged V
//                             tile, M = 128 output columns, N = 32: both
//                             branches' rows share the value operand).
// Row maxima are formed only when some probability would exceed 2^8 (always
// on a segment's first tile), and then O and the row sums are rescaled: the
// lazy rescale of the tensor-core forward.  Each thread keeps per-row partial
// sums; they are reduced at the segment's end, when O^T is read out of TMEM (one
// output column per thread) into the segment's partial result.
//
// Three single threads issue the asynchronous work, so that no one of them
// serialises the tile: thread 0 issues the score products (and issues the
// next tile's right after the current P^T is in shared memory, so they run
// under the PV products), lane 0 of warp 2 issues the PV products, and lane 0
// of warp 1 issues the TMA loads.  Each commits to its own barriers; the
// final barrier counts both MMA issuers' commits.
#include "kernels.h"
#include "ptx.cuh"
#include "pdl.cuh"

#include <cmath>

namespace diffattn {
namespace dtc {

constexpr int KT = 128;                 // keys per tile = threads = TMEM lanes
constexpr int THREADS = KT;
constexpr int DV = 128;                 // value width
constexpr int NR = 16;                  // MMA N: query rows per unit, padded
constexpr int K_PANEL = KT * 128;       // 16 KB: 128 keys x 64 columns (the swizzle span)
constexpr int Q_PANEL = NR * 128;       // 2 KB: 16 rows x 64 columns
constexpr int V_HALF = KT * 128;        // 16 KB: 64 value columns of 128 keys
constexpr int P_SUB = 2 * NR * 128;     // 4 KB: 32 rows (P_1^T, then P_2^T) x 64 keys
constexpr int P_BUF = 2 * P_SUB;        // two 64-key halves

// Shared memory for Q/K width HD, KS = one key tile shared by both branches
// (offsets from a 1024-byte aligned base).  A stage holds the key tile(s) as
// HD / 64 panels each, then the two 64-column halves of V: 64 KB for D = 64
// with two key tensors and for D = 128 with one.  The NST = 3 stages start at
// offset 0 (two tiles in flight ahead of the one computed).  D = 128 with two
// key tensors would need 96 KB stages, two of which leave no tile in flight
// while one is computed; that shape runs on the forward kernels.
template <int HD, bool KS>
struct Cfg {
    static_assert((HD == 64 && !KS) || (HD == 128 && KS), "Q/K width and key sharing");
    static constexpr int PANELS = HD / 64;
    static constexpr int K_BYTES = KT * HD * 2;          // one branch's key tile
    static constexpr int NK = KS ? 1 : 2;                // key tiles per stage
    static constexpr int STAGE = NK * K_BYTES + 2 * V_HALF;
    static constexpr int NST = 3;
    static_assert(STAGE == 64 * 1024, "stage size");
    static constexpr int Q_BYTES = NR * HD * 2;          // per branch
    static constexpr int OFF_P = NST * STAGE;            // P^T: [2 buffers][branch][64-key half]
    static constexpr int OFF_Q = OFF_P + 2 * P_BUF;      // [branch]
    static constexpr int OFF_RED = OFF_Q + 2 * Q_BYTES;  // float [4 warps][2][NR]
    static constexpr int OFF_BAR = OFF_RED + 4 * 2 * NR * 4;   // S_FULL, PV_DONE[2], FINAL, FULL[NST]
    static constexpr int NUM_BARS = 4 + NST;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;    // TMEM base address, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

constexpr uint32_t TMEM_COLS = 128;
constexpr uint32_t TM_S = 0;            // S1^T at 0, S2^T at 16
constexpr uint32_t TM_O = 32;           // O1^T at 32, O2^T at 48
constexpr uint32_t IDESC_S = idesc_bf16_f32(KT, NR, 0, 0);   // K (K-major) x Q^T (K-major), K = 16 per product
// both branches in one product: N = 32 rows of [P_1^T; P_2^T] into O_1^T, O_2^T
constexpr uint32_t IDESC_PV = idesc_bf16_f32(DV, 2 * NR, 1, 0);  // V^T (MN-major) x P^T (K-major)

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Offset of the 16-byte chunk c of row r in a 128-byte swizzled row layout
// (8-row atoms of 1024 bytes): chunk c sits at c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// The CTA's tiles.  The units' key tiles are laid end to end (unit-major,
// tpu = ceil(Tk / KT) tiles per unit, `total` in all); CTA c takes the
// contiguous range [bound(c), bound(c + 1)), bound(c) = c * total / grid, so
// every CTA streams the same number of tiles to within one.  The range is cut
// into segments at unit boundaries: a segment is one unit's tiles in this
// range, with its own row state and its own partial result.
__device__ __forceinline__ int64_t tile_bound(const DecodeParams& p, int c) {
    return (int64_t)c * p.tc_total / p.tc_grid;
}

// The first CTA whose range holds tiles of `unit`: the slot of a segment of
// `unit` is its CTA's index minus this.
__device__ __forceinline__ int first_cta(const DecodeParams& p, int unit) {
    const int64_t t0 = (int64_t)unit * p.tc_tpu;
    int c = (int)(t0 * p.tc_grid / p.tc_total);     // bound(c) <= t0
    while (c + 1 < p.tc_grid && tile_bound(p, c + 1) <= t0) ++c;
    return c;
}

struct Cursor {
    int64_t t = 0, t_end = 0;               // first tile of the segment; end of the CTA's range
    int unit = 0, c = 0, n = 0, k_begin = 0, k_end = 0;
    __device__ void start(const DecodeParams& p, int64_t tt) {
        t = tt;
        c = 0;
        if (t < t_end) {
            unit = (int)(t / p.tc_tpu);
            const int tile0 = (int)(t - (int64_t)unit * p.tc_tpu);
            const int64_t seg_end = min(t_end, (int64_t)(unit + 1) * p.tc_tpu);
            n = (int)(seg_end - t);
            k_begin = tile0 * KT;
            k_end = min(p.Tk, (tile0 + n) * KT);
        } else {
            n = 0;
        }
    }
    __device__ bool done() const { return t >= t_end; }
    // the segment ends where its unit does (it holds the unit's last tiles)
    __device__ bool unit_last(const DecodeParams& p) const {
        return t + n == (int64_t)(unit + 1) * p.tc_tpu;
    }
    __device__ void next(const DecodeParams& p) {
        if (++c >= n) start(p, t + n);
    }
};

// Stage tile `cur` into shared memory at `dst` with TMA box loads of 128
// rows x 64 columns (the panels of K1, of K2 unless the keys are shared, and
// the two 64-column halves of V), completion counted on `full`.
template <int HD, bool KS>
__device__ __forceinline__ void stage_tile(const DecodeParams& p, const Cursor& cur, uint8_t* dst,
                                           uint64_t* full, const CUtensorMap* k1, const CUtensorMap* k2,
                                           const CUtensorMap* v) {
    using C = Cfg<HD, KS>;
    const int bhk = cur.unit / p.row_chunks;
    const int b = bhk / p.Hk, hk = bhk - b * p.Hk;
    const int key0 = cur.k_begin + cur.c * KT;
    mbar_arrive_expect_tx(full, C::STAGE);
#pragma unroll
    for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_4d(dst + pn * K_PANEL, k1, full, pn * 64, key0, hk, b);
        if (!KS) tma_load_4d(dst + C::K_BYTES + pn * K_PANEL, k2, full, pn * 64, key0, hk, b);
    }
    tma_load_4d(dst + C::NK * C::K_BYTES, v, full, 0, key0, hk, b);
    tma_load_4d(dst + C::NK * C::K_BYTES + V_HALF, v, full, 64, key0, hk, b);
}

template <int TQ, int HD, bool KS>
__global__ void __launch_bounds__(THREADS, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
                 const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    static_assert(TQ >= 1 && TQ <= NR, "rows per unit");
    using C = Cfg<HD, KS>;
    constexpr int STAGE = C::STAGE, NST = C::NST, K_BYTES = C::K_BYTES, Q_BYTES = C::Q_BYTES;
    constexpr int OFF_P = C::OFF_P, OFF_Q = C::OFF_Q, OFF_RED = C::OFF_RED, OFF_BAR = C::OFF_BAR;
    constexpr int NUM_BARS = C::NUM_BARS, OFF_MISC = C::OFF_MISC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // S_FULL, PV_DONE[2], FINAL, FULL[NST]
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 4);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);          // [4 warps][2][NR]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const AbortState ab{abort_flag, p.status};
    pdl_launch_dependents();                // the combine pass may take its places now

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) mbar_init(&bars[i], i == 3 ? 2 : 1);   // FINAL: both MMA issuers
        *abort_flag = 0;
        fence_mbar_init();
    }
    // P^T and Q rows past the unit's TQ stay zero for the whole kernel
    for (int i = tid; i < (2 * P_BUF + 2 * Q_BYTES) / 16; i += THREADS)
        reinterpret_cast<uint4*>(smem + OFF_P)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(tmem_ptr, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_ptr;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;

    Cursor icur, ccur;                      // issue (producer) and compute positions
    icur.t_end = tile_bound(p, blockIdx.x + 1);
    icur.start(p, tile_bound(p, blockIdx.x));
    ccur = icur;
    uint32_t issued = 0;                    // tiles staged so far (the producer thread)
    constexpr int PRODUCER = 32;            // lane 0 of warp 1 issues the TMA loads
    constexpr int PV_ISSUER = 64;           // lane 0 of warp 2 issues the PV products
    if (tid == PRODUCER) {
        tma_prefetch_desc(&tm_k1);
        tma_prefetch_desc(&tm_k2);
        tma_prefetch_desc(&tm_v);
        for (int s0 = 0; s0 < NST - 1 && !icur.done(); ++s0) {
            stage_tile<HD, KS>(p, icur, smem + s0 * STAGE, &bars[4 + s0], &tm_k1, &tm_k2, &tm_v);
            icur.next(p);
            ++issued;
        }
    }

    float m[2][TQ], l[2][TQ];               // running row max (log2 units), this thread's row sums
    int last_key[TQ];
    uint32_t sph = 0;                       // S_FULL phase
    bool s_issued = false;                  // thread 0: the tile's score product is already issued
    auto issue_scores = [&](uint32_t t, int stage) -> bool {
        if (!mbar_wait(&bars[4 + stage], (t / NST) & 1u, ab)) return false;
        tc_fence_after();
#pragma unroll
        for (int br = 0; br < 2; ++br) {
            const uint64_t ka = sdesc_sw128(sbase + stage * STAGE + (KS ? 0 : br) * K_BYTES, 16, 1024);
            const uint64_t qb = sdesc_sw128(sbase + OFF_Q + br * Q_BYTES, 16, 1024);
            // HD / 16 products of depth 16, four per 64-column panel
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const int pn = kk >> 2, ks = kk & 3;
                mma_ss(tmem + TM_S + br * NR, ka + pn * (K_PANEL >> 4) + 2 * ks,
                       qb + pn * (Q_PANEL >> 4) + 2 * ks, IDESC_S, kk > 0);
            }
        }
        mma_commit(&bars[0]);
        return true;
    };
    uint32_t g = 0;                         // tiles computed so far (all segments): P buffer g & 1
    int st = 0;                             // stage of the tile being computed
    bool ok = true;
    while (!ccur.done()) {
        const int unit = ccur.unit;
        if (ccur.c == 0) {
            // a new segment: its unit's query rows (swizzled K-major rows), row state
            const int rc = unit % p.row_chunks;
            const int bhk = unit / p.row_chunks;
            const int b = bhk / p.Hk, hk = bhk - b * p.Hk;
            const int n_rows = p.kv_group * p.Tq;
            constexpr int QCH = HD / 8;          // 16-byte chunks of a query row
            for (int i = tid; i < TQ * 2 * QCH; i += THREADS) {
                const int r = i / (2 * QCH), br = (i / QCH) & 1, c = i % QCH;
                const int row = rc * TQ + r;
                uint4 x = make_uint4(0, 0, 0, 0);
                if (row < n_rows) {
                    const int h = hk * p.kv_group + row / p.Tq;
                    const int q = row % p.Tq;
                    const __nv_bfloat16* src = br
                        ? static_cast<const __nv_bfloat16*>(p.q2) + b * p.s_q2[0] + h * p.s_q2[1] + (int64_t)q * p.s_q2[2]
                        : static_cast<const __nv_bfloat16*>(p.q1) + b * p.s_q1[0] + h * p.s_q1[1] + (int64_t)q * p.s_q1[2];
                    x = *reinterpret_cast<const uint4*>(src + c * 8);
                }
                *reinterpret_cast<uint4*>(smem + OFF_Q + br * Q_BYTES + (c >> 3) * Q_PANEL + sw128(r, c & 7)) = x;
            }
            fence_proxy_async_smem();
#pragma unroll
            for (int r = 0; r < TQ; ++r) {
                m[0][r] = m[1][r] = -INFINITY;
                l[0][r] = l[1][r] = 0.f;
                last_key[r] = p.causal ? p.Tk - p.Tq + (rc * TQ + r) % p.Tq : p.Tk;
            }
        }
        if (!__syncthreads_and(ok)) { ok = false; break; }   // the query rows are in shared memory
        if (tid == 0 && !s_issued) ok = issue_scores(g, st);
        s_issued = false;
        ok = __syncthreads_and(ok) && mbar_wait_warp(&bars[0], sph, ab);
        sph ^= 1;
        tc_fence_after();
        uint32_t u[2][NR];
        ld16(lane_base + TM_S, u[0]);
        ld16(lane_base + TM_S + NR, u[1]);
        tmem_wait_ld();
        const int key = ccur.k_begin + ccur.c * KT + tid;
        float s[2][TQ], pr[2][TQ];
        bool big = false;
#pragma unroll
        for (int r = 0; r < TQ; ++r) {
            const bool vis = key < ccur.k_end && key <= last_key[r];
#pragma unroll
            for (int br = 0; br < 2; ++br) {
                s[br][r] = vis ? __uint_as_float(u[br][r]) * sl2 : -INFINITY;
                pr[br][r] = vis ? ex2_approx(s[br][r] - m[br][r]) : 0.f;
                big |= !(pr[br][r] <= 256.0f);
            }
        }
        // S^T is in registers (the next score product may overwrite it);
        // block-wide: abort (bit 1) or a row whose probabilities exceed 2^8 (bit 0)
        tc_fence_before();
        const int vote = __syncthreads_or((ok ? 0 : 2) | (big ? 1 : 0));
        if (vote & 2) { ok = false; break; }
        if (vote & 1) {
            // exact tile row maxima (warp, then the four warps), new running
            // maxima, and the rescale of this thread's sums and of O^T
#pragma unroll
            for (int br = 0; br < 2; ++br)
#pragma unroll
                for (int r = 0; r < TQ; ++r) {
                    float v = s[br][r];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) red[(warp * 2 + br) * NR + r] = v;
                }
            __syncthreads();
            float alpha[2][TQ];
#pragma unroll
            for (int br = 0; br < 2; ++br)
#pragma unroll
                for (int r = 0; r < TQ; ++r) {
                    const float tmax = fmaxf(fmaxf(red[(0 + br) * NR + r], red[(2 + br) * NR + r]),
                                             fmaxf(red[(4 + br) * NR + r], red[(6 + br) * NR + r]));
                    const float mn = fmaxf(m[br][r], tmax);
                    alpha[br][r] = (mn == -INFINITY) ? 1.f : ex2_approx(m[br][r] - mn);
                    m[br][r] = mn;
                    l[br][r] *= alpha[br][r];
                    pr[br][r] = (s[br][r] == -INFINITY) ? 0.f : ex2_approx(s[br][r] - mn);
                }
            if (ccur.c > 0) {
                // O^T holds this segment's earlier tiles: rescale its columns
                // (one per row) once the previous PV product has completed
                ok = mbar_wait_warp(&bars[1 + ((g - 1) & 1u)], ((g - 1) >> 1) & 1u, ab);
                tc_fence_after();
#pragma unroll
                for (int br = 0; br < 2; ++br) {
                    uint32_t o[NR];
                    ld16(lane_base + TM_O + br * NR, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < TQ; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[br][r]);
                    tmem_st16(lane_base + TM_O + br * NR, o);
                }
                tmem_wait_st();
                tc_fence_before();
            }
            if (!__syncthreads_and(ok)) { ok = false; break; }
        }
        // P^T to P buffer g & 1, free once the PV product of tile g - 2 has
        // read it (the ((g >> 1) - 1)-th completion of that buffer's barrier);
        // thread tid writes column tid of every row, bf16
        const uint32_t pb = g & 1u;
        if (g >= 2) ok = mbar_wait_warp(&bars[1 + pb], ((g >> 1) & 1u) ^ 1u, ab);
        {
            const int kc = tid & 63;
            uint8_t* pbase = smem + OFF_P + pb * P_BUF + (tid >> 6) * P_SUB;   // this key's half
#pragma unroll
            for (int br = 0; br < 2; ++br)
#pragma unroll
                for (int r = 0; r < TQ; ++r) {
                    *reinterpret_cast<__nv_bfloat16*>(pbase + sw128(br * NR + r, kc >> 3) + (kc & 7) * 2) =
                        __float2bfloat16_rn(pr[br][r]);
                    l[br][r] += pr[br][r];
                }
        }
        fence_proxy_async_smem();
        if (!__syncthreads_and(ok)) { ok = false; break; }
        if (tid == PV_ISSUER) {
            // [O_1^T O_2^T] += V^T [P_1^T P_2^T]: A = the staged V tile
            // (MN-major, the two 64-column halves V_HALF apart), B = the 32
            // rows of P^T in two 64-key halves
            tc_fence_after();
            const uint64_t va = sdesc_sw128(sbase + st * STAGE + C::NK * K_BYTES, V_HALF, 1024);
            const uint64_t pd = sdesc_sw128(sbase + OFF_P + pb * P_BUF, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk)
                mma_ss(tmem + TM_O, va + 128 * kk, pd + (kk >> 2) * (P_SUB >> 4) + 2 * (kk & 3),
                       IDESC_PV, (ccur.c > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars[1 + pb]);
        }
        if (tid == 0) {
            if (ccur.c + 1 < ccur.n) {      // the next tile's scores, same segment
                ok = issue_scores(g + 1, (st + 1) % NST);
                s_issued = ok;
            }
        }
        if (ccur.c == ccur.n - 1) {
            // ---- the segment's last tile: O^T (column tid) and the row sums
            // into the segment's partial result slot
            ok = mbar_wait_warp(&bars[1 + pb], (g >> 1) & 1u, ab);
            tc_fence_after();
            uint32_t o[2][NR];
            ld16(lane_base + TM_O, o[0]);
            ld16(lane_base + TM_O + NR, o[1]);
            tmem_wait_ld();
            tc_fence_before();
#pragma unroll
            for (int br = 0; br < 2; ++br)
#pragma unroll
                for (int r = 0; r < TQ; ++r) {
                    float v = l[br][r];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == 0) red[(warp * 2 + br) * NR + r] = v;
                }
            if (!__syncthreads_and(ok)) { ok = false; break; }
            const int slot = (int)blockIdx.x - first_cta(p, unit);
            float* part = p.work + ((int64_t)unit * p.splits + slot) * TQ * (4 + 2 * DV);
#pragma unroll
            for (int r = 0; r < TQ; ++r) {
                part[r * (4 + 2 * DV) + 4 + tid] = __uint_as_float(o[0][r]);
                part[r * (4 + 2 * DV) + 4 + DV + tid] = __uint_as_float(o[1][r]);
            }
#pragma unroll
            for (int br = 0; br < 2; ++br)
#pragma unroll
                for (int r = 0; r < TQ; ++r)
                    if (tid == r * 2 + br) {
                        part[r * (4 + 2 * DV) + 2 * br] = m[br][r];
                        part[r * (4 + 2 * DV) + 2 * br + 1] =
                            red[(0 + br) * NR + r] + red[(2 + br) * NR + r] + red[(4 + br) * NR + r] +
                            red[(6 + br) * NR + r];
                    }
            if (ccur.unit_last(p)) {
                // the unit's slots past its last segment saw no keys:
                // row max -inf, sum 0, O 0 (they weigh nothing in the merge)
                float* empty = part + TQ * (4 + 2 * DV);
                const int nf = (p.splits - 1 - slot) * TQ * (4 + 2 * DV);
                for (int i = tid; i < nf; i += THREADS) {
                    const int col = i % (4 + 2 * DV);
                    empty[i] = (col == 0 || col == 2) ? -INFINITY : 0.f;
                }
            }
        }
        // ---- prefetch (the producer thread): tile g + NST - 1 into the stage of tile
        // g - 1, once the PV product of tile g - 1 has read its values
        if (tid == PRODUCER && !icur.done()) {
            if (g >= 1) ok = mbar_wait(&bars[1 + ((g - 1) & 1u)], ((g - 1) >> 1) & 1u, ab);
            const int ist = (st + NST - 1) % NST;
            if (ok) {
                stage_tile<HD, KS>(p, icur, smem + ist * STAGE, &bars[4 + ist], &tm_k1, &tm_k2, &tm_v);
                icur.next(p);
                ++issued;
            }
        }
        ++g;
        if (++st == NST) st = 0;
        ccur.next(p);
        if (!__syncthreads_and(ok)) { ok = false; break; }
    }

    // Teardown: no copy or MMA of this CTA may still be in flight.
    if (tid == PRODUCER) {
        for (uint32_t t = g; t < issued; ++t)       // loads staged but not consumed (abort)
            mbar_wait_teardown(&bars[4 + t % NST], (t / NST) & 1u, 200ull * 1000ull * 1000ull);
    }
    if (tid == 0 || tid == PV_ISSUER) mma_commit(&bars[3]);
    if (tid == 0) {
        mbar_wait_teardown(&bars[3], 0, 200ull * 1000ull * 1000ull);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

template <int TQ, int HD, bool KS>
int launch_first_pass_tq(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t stream) {
    constexpr int smem = Cfg<HD, KS>::SMEM_BYTES;
    if (cudaFuncSetAttribute(decode_tc_kernel<TQ, HD, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return -1;
    decode_tc_kernel<TQ, HD, KS><<<p.tc_grid, THREADS, smem, stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int HD, bool KS>
int launch_first_pass_hd(const DecodeParams& p, cudaStream_t stream) {
    if (p.tq_bucket == 4) return launch_first_pass_tq<4, HD, KS>(p, p.tc_maps, stream);
    if (p.tq_bucket == 8) return launch_first_pass_tq<8, HD, KS>(p, p.tc_maps, stream);
    if (p.tq_bucket == 16) return launch_first_pass_tq<16, HD, KS>(p, p.tc_maps, stream);
    if constexpr (HD == 128) {
        if (p.tq_bucket == 1) return launch_first_pass_tq<1, HD, KS>(p, p.tc_maps, stream);
        if (p.tq_bucket == 2) return launch_first_pass_tq<2, HD, KS>(p, p.tc_maps, stream);
    }
    return -1;
}

// Segments of one unit at most: every CTA range holds at least
// floor(total / grid) tiles, so tpu consecutive tiles meet at most
// ceil((tpu - 1) / that) + 1 ranges (and never more than tpu).
int64_t tc_slots(int64_t total, int64_t tpu, int64_t grid) {
    const int64_t per = total / grid;
    const int64_t s = (tpu - 1 + per - 1) / per + 1;
    return s < tpu ? s : tpu;
}

constexpr int64_t kMaxGrid = 1024;

}  // namespace dtc

size_t decode_tc_work_floats(int64_t units, int64_t Tk, int tq_bucket) {
    const int64_t tpu = (Tk + dtc::KT - 1) / dtc::KT;
    const int64_t total = units * tpu;
    const int64_t grid = total < dtc::kMaxGrid ? total : dtc::kMaxGrid;
    return (size_t)(units * dtc::tc_slots(total, tpu, grid) * tq_bucket * (4 + 2 * dtc::DV));
}

int launch_decode_tc_first_pass(DecodeParams* p, cudaStream_t stream) {
    if (!p->tc_maps) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    const int64_t units = (int64_t)p->B * p->Hk * p->row_chunks;
    const int64_t tpu = (p->Tk + dtc::KT - 1) / dtc::KT;
    const int64_t total = units * tpu;
    int64_t grid = total < sms ? total : sms;
    if (grid > dtc::kMaxGrid) grid = dtc::kMaxGrid;
    p->tc_tpu = (int)tpu;
    p->tc_total = total;
    p->tc_grid = (int)grid;
    p->splits = (int)dtc::tc_slots(total, tpu, grid);   // partial slots per unit
    if (p->D == 64) return dtc::launch_first_pass_hd<64, false>(*p, stream);
    if (p->D == 128 && p->k_shared) return dtc::launch_first_pass_hd<128, true>(*p, stream);
    return -1;
}

}  // namespace diffattn
