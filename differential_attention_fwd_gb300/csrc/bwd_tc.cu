// bwd_tc.cu -- backward of the differential-attention forward on the sm_103a
// tensor cores (bf16, D = 64, V width 128).
//
// Given dO = dL/dO for O = (A_1 - lambda A_2) V (paperleet "Differential
// Transformer Attention", Return requirements: gradients through both Q/K
// branches, the value and the coefficient), and the row statistics of the
// first pass (the forward kernel in statistics mode: lse_b, the log2-sum-exp
// of branch b's scaled scores, and Dd_b = dO . (A_b V) per query row, both
// stored negated so that the kernels below add them):
//
//   A_b  = 2^(S_b * log2(e) / sqrt(D) - lse_b)          S_b = Q_b K_b^T
//   dP   = dO V^T
//   dS_1 = A_1 * (dP - Dd_1)        dS_2 = -lambda A_2 * (dP - Dd_2)
//   dQ_b = dS_b K_b / sqrt(D)       dK_b = dS_b^T Q_b / sqrt(D)
//   dV   = (A_1 - lambda A_2)^T dO
//
// Two kernels, both persistent (one CTA per SM) with a TMA producer warp, one
// MMA-issuing thread and two warpgroups that turn scores into gradients of the
// scores in tensor memory (TMEM):
//
// dq kernel: work item (b, h, 128-query tile); TMEM lanes are query rows.
//   The item's dO is copied into TMEM once (warpgroup 0), as the A operand of
//   dP = dO V^T.  Per 64-key tile j: S_1 and S_2 (M128 N64 MMAs from shared
//   memory) into one of two TMEM buffers, dP into its single buffer (the
//   elementwise warps read it at the start of their tile and release it);
//   warpgroup b forms dS_b from S_b and dP and writes it back over S_b as
//   bf16; then dQ_b += dS_b K_b (A from TMEM, K_b read MN-major from the same
//   shared-memory tile the score product read K-major).  The score buffers
//   alternate so that tile j+1's products overlap tile j's elementwise work.
//
// dkdv kernel: work item (b, key/value head, 128-key tile); TMEM lanes are key
//   rows.  For every query head of the group and every 64-query tile:
//   S_1^T = K_1 Q_1^T, S_2^T, dP^T = V dO^T; the two warpgroups split the 64
//   query columns, form dS_1^T, dS_2^T and W^T = A_1^T - lambda A_2^T and write
//   them as bf16 operands (W^T and dS_1^T to the spare TMEM columns, dS_2^T
//   to shared memory); then dV += W^T dO, dK_b += dS_b^T Q_b.  The item's accumulators (dV, dK_1, dK_2: 256
//   columns) leave room for one set of score buffers (192 columns); the
//   warpgroups copy a tile's scores to registers and release the buffers at
//   once, so the next tile's score products run during this tile's
//   elementwise work.
//
// Causal masking: key j is visible to query i iff j <= i; key tiles above the
// diagonal are skipped and crossing tiles are masked element by element
// (masked entries have A_b = 0, hence dS_b = 0 and no contribution to dV).
// Every mbarrier wait is bounded (see ptx.cuh); on expiry the kernel records
// DIFFATTN_ERR_TIMEOUT in the status word, drains and frees TMEM.
#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"

#include <cmath>

namespace diffattn {
namespace bwdtc {

constexpr int HD = 64;             // Q/K width D
constexpr int VD = 128;            // V/O width 2D
constexpr int NUM_THREADS = 384;
constexpr uint32_t REGS_WORK = 200;
constexpr uint32_t REGS_OTHER = 104;
static_assert(256 * REGS_WORK + 128 * REGS_OTHER <= NUM_THREADS * 168, "register split");

// Wait profiles (only in the separate build compiled with
// -DDIFFATTN_WAIT_PROFILE; the regular build has none of it): a role's
// issuing thread (lane 0 of each elementwise warp) counts SM cycles by what it
// waits for or works on, in N kinds, and adds them to a [3 roles][N] array of
// its kernel when the CTA ends.
#ifdef DIFFATTN_WAIT_PROFILE
template <int N>
struct ProfT {
    unsigned long long c[N] = {};
    long long t0 = 0;
    __device__ __forceinline__ void start() { t0 = clock64(); }
    template <class F>
    __device__ __forceinline__ bool timed(int kind, F&& f) {
        const long long a = clock64();
        const bool r = f();
        c[kind] += (unsigned long long)(clock64() - a);
        return r;
    }
    __device__ __forceinline__ void flush(unsigned long long (*g)[N], int role, bool reporter) {
        c[0] = (unsigned long long)(clock64() - t0);
        if (reporter)
            for (int i = 0; i < N; ++i) atomicAdd(&g[role][i], c[i]);
    }
};
#define BP_WAIT(pf, kind, expr) (pf).timed((kind), [&]() -> bool { return (expr); })
#define BP_MARK(var) long long var = clock64()
#define BP_ADD(pf, kind, since) ((pf).c[kind] += (unsigned long long)(clock64() - (since)))
#define BP_RESET(var) (var = clock64())
#define BP_COUNT(pf, kind) ((pf).c[kind] += 1)
#define BP_FLUSH(pf, g, role, rep) (pf).flush((g), (role), (rep))
#else
template <int N>
struct ProfT {
    __device__ __forceinline__ void start() {}
};
#define BP_WAIT(pf, kind, expr) (expr)
#define BP_MARK(var) ((void)0)
#define BP_ADD(pf, kind, since) ((void)0)
#define BP_RESET(var) ((void)0)
#define BP_COUNT(pf, kind) ((void)0)
#define BP_FLUSH(pf, g, role, rep) ((void)0)
#endif

// The CTA's k-th work item in a boustrophedon order over the item list.
__device__ __forceinline__ int item_index(int k, int cta, int grid) {
    const int base = k * grid;
    return base + ((k & 1) ? (grid - 1 - cta) : cta);
}

// ===========================================================================
// dq kernel
// ===========================================================================
namespace dq {

constexpr int BM = 128;            // query rows per item (TMEM lanes)
constexpr int BN = 64;             // keys per tile
constexpr int KSTAGES = 4;         // (K1, K2) ring
constexpr int VSTAGES = 3;         // V ring
constexpr uint32_t Q_BYTES = BM * HD * 2;          // 16 KB
constexpr uint32_t DO_HALF = BM * 64 * 2;          // 16 KB per 64-column half
constexpr uint32_t K_BYTES = BN * HD * 2;          // 8 KB
constexpr uint32_t V_HALF = BN * 64 * 2;           // 8 KB
constexpr uint32_t V_BYTES = 2 * V_HALF;

constexpr uint32_t OFF_Q1 = 0;
constexpr uint32_t OFF_Q2 = OFF_Q1 + Q_BYTES;
constexpr uint32_t OFF_DO = OFF_Q2 + Q_BYTES;                  // two halves
constexpr uint32_t OFF_K = OFF_DO + 2 * DO_HALF;                // stage s: K1 +0, K2 +K_BYTES
constexpr uint32_t OFF_V = OFF_K + KSTAGES * 2 * K_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + VSTAGES * V_BYTES;
constexpr int BAR_Q_FULL = 0;
constexpr int BAR_Q_EMPTY = 1;
constexpr int BAR_K_FULL = 2;
constexpr int BAR_K_EMPTY = BAR_K_FULL + KSTAGES;
constexpr int BAR_V_FULL = BAR_K_EMPTY + KSTAGES;
constexpr int BAR_V_EMPTY = BAR_V_FULL + VSTAGES;
constexpr int BAR_S_FULL = BAR_V_EMPTY + VSTAGES;     // [buffer]
constexpr int BAR_DS_FULL = BAR_S_FULL + 2;           // [buffer], 8 warps
constexpr int BAR_DQ_FULL = BAR_DS_FULL + 2;
constexpr int BAR_DQ_EMPTY = BAR_DQ_FULL + 1;         // 8 warps
constexpr int BAR_FINAL = BAR_DQ_EMPTY + 1;
constexpr int BAR_DP_FREE = BAR_FINAL + 1;            // 8 warps: a tile's dP read out of TMEM
constexpr int BAR_DO_READY = BAR_DP_FREE + 1;         // 4 warps: the item's dO copied into TMEM
constexpr int BAR_DO_FREE = BAR_DO_READY + 1;         // MMA: the item's last dP product done
constexpr int NUM_BARS = BAR_DO_FREE + 1;
constexpr uint32_t OFF_TMEM_PTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_PTR + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM: buffer b at b*128: S1 +0, S2 +64 (dS_1, dS_2 written over them);
// dP at 256 (one buffer: the elementwise warps read it at the start of their
// tile, so the next tile's dP may follow at once); the item's dO at 320 as the
// A operand of dP = dO V^T (64 columns: bf16 pairs, dO being fixed for the
// item, so the products read only V from shared memory); dQ1 at 384, dQ2 at 448.
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_DP = 256;
constexpr uint32_t TM_DO = 320;
constexpr uint32_t TM_DQ = 384;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);     // Q x K^T, dO x V^T
constexpr uint32_t IDESC_DQ = idesc_bf16_f32(BM, HD, 0, 1);    // dS (TMEM) x K (MN-major)

// Wait profile of this kernel (g_prof[role][kind], see ProfT).  Roles: 0 the
// TMA producer, 1 the MMA-issuing thread, 2 the eight elementwise warps.
// Kinds: 0 the role's cycles from start to end; the producer's waits for the
// Q/dO slot (1), a K stage (2) and a V stage (3) to be released; the MMA
// thread's waits for Q/dO and the item's dO in TMEM (4), K (5), V (6), the dS
// operands and the previous tile's dP read out (7), and the dQ accumulators to
// be read out (8); the elementwise warps' waits for the scores
// (9), their TMEM read of S_b and dP (10), arithmetic (11), the dS store into
// TMEM with its fences (12), the wait for the dQ accumulators (13) and the
// epilogue (14); tile (15) and item (16) counts.
enum : int {
    kQTotal = 0, kQQEmpty = 1, kQKEmpty = 2, kQVEmpty = 3, kQQFull = 4, kQKFull = 5, kQVFull = 6,
    kQDsFull = 7, kQDqEmpty = 8, kQSFull = 9, kQRead = 10, kQMath = 11, kQStore = 12,
    kQDqFull = 13, kQEpilogue = 14, kQTiles = 15, kQItems = 16, kQKinds = 17
};
#ifdef DIFFATTN_WAIT_PROFILE
__device__ unsigned long long g_prof[3][kQKinds];
#endif
using Prof = ProfT<kQKinds>;

struct Item {
    int b, h, qt, n_kv;
};
__device__ __forceinline__ Item decode_item(int idx, const BwdTcParams& p) {
    // longest first: the last query tiles of every head, then the ones before
    const int BH = p.B * p.H;
    const int r = idx / BH;
    const int bh = idx - r * BH;
    Item it;
    it.qt = p.causal ? (p.nq128 - 1 - r) : r;
    it.b = bh / p.H;
    it.h = bh - it.b * p.H;
    it.n_kv = p.causal ? min(2 * it.qt + 2, p.nk64) : p.nk64;
    return it;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q1,
                       const __grid_constant__ CUtensorMap tm_k1,
                       const __grid_constant__ CUtensorMap tm_q2,
                       const __grid_constant__ CUtensorMap tm_k2,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const BwdTcParams p) {
    // The dK/dV kernel that follows reads nothing this kernel writes: it may
    // take each SM as soon as this kernel's CTA there has finished.
    pdl_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_PTR);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
    const uint32_t warp = warp_id();
    const uint32_t lane = threadIdx.x & 31;
    const AbortState ab{abort_flag, p.status};
    const int total = p.B * p.H * p.nq128;

    if (threadIdx.x == 0) {
        mbar_init(&bars[BAR_Q_FULL], 1);
        mbar_init(&bars[BAR_Q_EMPTY], 1);
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(&bars[BAR_K_FULL + s], 1);
            mbar_init(&bars[BAR_K_EMPTY + s], 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            mbar_init(&bars[BAR_V_FULL + s], 1);
            mbar_init(&bars[BAR_V_EMPTY + s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[BAR_S_FULL + i], 1);
            mbar_init(&bars[BAR_DS_FULL + i], 8);
        }
        mbar_init(&bars[BAR_DQ_FULL], 1);
        mbar_init(&bars[BAR_DQ_EMPTY], 8);
        mbar_init(&bars[BAR_FINAL], 1);
        mbar_init(&bars[BAR_DP_FREE], 8);
        mbar_init(&bars[BAR_DO_READY], 4);
        mbar_init(&bars[BAR_DO_FREE], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_ptr, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;
    const int grid = gridDim.x, cta = blockIdx.x;

    if (warp >= 8) {
        regs_dec<REGS_OTHER>();
        if (warp == 8) {
            // ------------------------------------------------------ producer
            if (elect_one()) {
                Prof pf;
                pf.start();
                uint32_t kst = 0, kph = 0, vst = 0, vph = 0, qph = 0;
                uint32_t armed_q = 0, armed_k[KSTAGES] = {}, armed_v[VSTAGES] = {};
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int idx = item_index(k, cta, grid);
                    if (idx >= total) break;
                    const Item it = decode_item(idx, p);
                    const int hk = it.h / p.kv_group;
                    if (k > 0) {
                        if (!(ok = BP_WAIT(pf, kQQEmpty, mbar_wait(&bars[BAR_Q_EMPTY], qph, ab)))) break;
                        qph ^= 1;
                    }
                    mbar_arrive_expect_tx(&bars[BAR_Q_FULL], 2 * Q_BYTES + 2 * DO_HALF);
                    tma_load_4d(smem + OFF_Q1, &tm_q1, &bars[BAR_Q_FULL], 0, it.qt * BM, it.h, it.b);
                    tma_load_4d(smem + OFF_Q2, &tm_q2, &bars[BAR_Q_FULL], 0, it.qt * BM, it.h, it.b);
                    tma_load_4d(smem + OFF_DO, &tm_do, &bars[BAR_Q_FULL], 0, it.qt * BM, it.h, it.b);
                    tma_load_4d(smem + OFF_DO + DO_HALF, &tm_do, &bars[BAR_Q_FULL], 64, it.qt * BM,
                                it.h, it.b);
                    ++armed_q;
                    for (int j = 0; j < it.n_kv; ++j) {
                        if (!(ok = BP_WAIT(pf, kQKEmpty, mbar_wait(&bars[BAR_K_EMPTY + kst], kph ^ 1, ab)))) break;
                        uint8_t* kd = smem + OFF_K + kst * 2 * K_BYTES;
                        mbar_arrive_expect_tx(&bars[BAR_K_FULL + kst], 2 * K_BYTES);
                        tma_load_4d(kd, &tm_k1, &bars[BAR_K_FULL + kst], 0, j * BN, hk, it.b);
                        tma_load_4d(kd + K_BYTES, &tm_k2, &bars[BAR_K_FULL + kst], 0, j * BN, hk, it.b);
                        ++armed_k[kst];
                        if (++kst == KSTAGES) { kst = 0; kph ^= 1; }
                        if (!(ok = BP_WAIT(pf, kQVEmpty, mbar_wait(&bars[BAR_V_EMPTY + vst], vph ^ 1, ab)))) break;
                        uint8_t* vd = smem + OFF_V + vst * V_BYTES;
                        mbar_arrive_expect_tx(&bars[BAR_V_FULL + vst], V_BYTES);
                        tma_load_4d(vd, &tm_v, &bars[BAR_V_FULL + vst], 0, j * BN, hk, it.b);
                        tma_load_4d(vd + V_HALF, &tm_v, &bars[BAR_V_FULL + vst], 64, j * BN, hk, it.b);
                        ++armed_v[vst];
                        if (++vst == VSTAGES) { vst = 0; vph ^= 1; }
                    }
                }
                const uint64_t lim = 200ull * 1000ull * 1000ull;
                if (armed_q) mbar_wait_teardown(&bars[BAR_Q_FULL], (armed_q - 1) & 1, lim);
                for (int s = 0; s < KSTAGES; ++s)
                    if (armed_k[s]) mbar_wait_teardown(&bars[BAR_K_FULL + s], (armed_k[s] - 1) & 1, lim);
                for (int s = 0; s < VSTAGES; ++s)
                    if (armed_v[s]) mbar_wait_teardown(&bars[BAR_V_FULL + s], (armed_v[s] - 1) & 1, lim);
                BP_FLUSH(pf, g_prof, 0, true);
            }
            __syncwarp();
        } else if (warp == 9) {
            // ------------------------------------------------------ MMA issue
            if (elect_one()) {
                Prof pf;
                pf.start();
                const uint64_t q1d = sdesc_sw128(smem_u32(smem + OFF_Q1), 16, 1024);
                const uint64_t q2d = sdesc_sw128(smem_u32(smem + OFF_Q2), 16, 1024);
                const uint64_t kkd = sdesc_sw128(smem_u32(smem + OFF_K), 16, 1024);        // K-major
                const uint64_t kmd = sdesc_sw128(smem_u32(smem + OFF_K), K_BYTES, 1024);   // MN-major
                const uint64_t vd = sdesc_sw128(smem_u32(smem + OFF_V), 16, 1024);
                uint32_t kc = 0;            // key tiles consumed so far (K ring position)
                uint32_t vst = 0, vph = 0, qph = 0, dqph = 0, dsph = 0;
                bool ok = true;
                // S_1, S_2 of key tile kt into buffer buf, then dP into its buffer
                // once the elementwise warps have read tile kt - 1's and, for an
                // item's first tile, the item's dO is in TMEM (item number ki);
                // an item's last dP releases the dO columns
                auto issue_s = [&](uint32_t kt, int buf, int ki, bool first_tile, bool last_tile) -> bool {
                    const uint32_t ks = kt % KSTAGES;
                    if (!BP_WAIT(pf, kQKFull, mbar_wait(&bars[BAR_K_FULL + ks], (kt / KSTAGES) & 1u, ab)))
                        return false;
                    if (!BP_WAIT(pf, kQVFull, mbar_wait(&bars[BAR_V_FULL + vst], vph, ab))) return false;
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * 128;
                    const uint64_t k1 = kkd + ((ks * 2 * K_BYTES) >> 4);
                    const uint64_t k2 = k1 + (K_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        mma_ss(d, q1d + 2 * kk, k1 + 2 * kk, IDESC_S, kk > 0);
                        mma_ss(d + 64, q2d + 2 * kk, k2 + 2 * kk, IDESC_S, kk > 0);
                    }
                    if (kt > 0 && !BP_WAIT(pf, kQDsFull, mbar_wait(&bars[BAR_DP_FREE], (kt - 1) & 1u, ab)))
                        return false;
                    if (first_tile &&
                        !BP_WAIT(pf, kQQFull, mbar_wait(&bars[BAR_DO_READY], (uint32_t)ki & 1u, ab)))
                        return false;
                    tc_fence_after();
                    const uint64_t v0 = vd + ((vst * V_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < VD / 16; ++kk) {
                        const uint32_t voff = (kk >> 2) * (V_HALF >> 4) + 2 * (kk & 3);
                        mma_ts(tmem_base + TM_DP, tmem_base + TM_DO + kk * 8, v0 + voff, IDESC_S, kk > 0);
                    }
                    mma_commit(&bars[BAR_S_FULL + buf]);
                    mma_commit(&bars[BAR_V_EMPTY + vst]);
                    if (last_tile) mma_commit(&bars[BAR_DO_FREE]);
                    if (++vst == VSTAGES) { vst = 0; vph ^= 1; }
                    return true;
                };
                bool first = true;
                for (int k = 0; ok; ++k) {
                    const int idx = item_index(k, cta, grid);
                    if (idx >= total) break;
                    const Item it = decode_item(idx, p);
                    const int n = it.n_kv;
                    if (!(ok = BP_WAIT(pf, kQQFull, mbar_wait(&bars[BAR_Q_FULL], qph, ab)))) break;
                    qph ^= 1;
                    for (int t = 0; t < 2 && t < n && ok; ++t) ok = issue_s(kc + t, t, k, t == 0, t == n - 1);
                    if (!ok) break;
                    if (n <= 2) mma_commit(&bars[BAR_Q_EMPTY]);
                    for (int j = 0; j < n; ++j) {
                        const int buf = j & 1;
                        if (!(ok = BP_WAIT(pf, kQDsFull, mbar_wait(&bars[BAR_DS_FULL + buf], (dsph >> buf) & 1u, ab))))
                            break;
                        dsph ^= 1u << buf;
                        if (j == 0 && !first) {
                            if (!(ok = BP_WAIT(pf, kQDqEmpty, mbar_wait(&bars[BAR_DQ_EMPTY], dqph, ab)))) break;
                            dqph ^= 1;
                        }
                        tc_fence_after();
                        const uint32_t ks = (kc + j) % KSTAGES;
                        const uint64_t k1 = kmd + ((ks * 2 * K_BYTES) >> 4);
                        const uint64_t k2 = k1 + (K_BYTES >> 4);
                        const uint32_t a = tmem_base + buf * 128;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            mma_ts(tmem_base + TM_DQ, a + kk * 8, k1 + 128 * kk, IDESC_DQ,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                            mma_ts(tmem_base + TM_DQ + 64, a + 64 + kk * 8, k2 + 128 * kk, IDESC_DQ,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars[BAR_K_EMPTY + ks]);
                        if (j + 2 < n) {
                            if (!(ok = issue_s(kc + j + 2, buf, k, false, j + 3 == n))) break;
                            if (j + 3 == n) mma_commit(&bars[BAR_Q_EMPTY]);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bars[BAR_DQ_FULL]);
                    kc += n;
                    first = false;
                }
                mma_commit(&bars[BAR_FINAL]);
                mbar_wait_teardown(&bars[BAR_FINAL], 0, 200ull * 1000ull * 1000ull);
                BP_FLUSH(pf, g_prof, 1, true);
            }
            __syncwarp();
        }
    } else {
        regs_inc<REGS_WORK>();
        // ------------------------------------------- dS and the dQ epilogue
        Prof pf;
        pf.start();
        const int br = warp >> 2;
        const uint32_t quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem_base + ((quad * 32u) << 16);
        const float sl2 = p.scale_log2;
        const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
        const float coef = br ? -lam : 1.0f;
        uint32_t sph = 0, dqph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, cta, grid);
            if (idx >= total) break;
            const Item it = decode_item(idx, p);
            const int q = it.qt * BM + row;
            const bool live = q < p.T;
            float nlse = 0.f, ndd = 0.f;    // -lse_b and -Dd_b of this row
            if (live) {
                const float4 st = *reinterpret_cast<const float4*>(
                    p.stats + (((int64_t)it.b * p.H + it.h) * p.T + q) * 4);
                nlse = br ? st.y : st.x;
                ndd = br ? st.w : st.z;
            }
            if (br == 0) {
                // the item's dO rows into TMEM (the dP products' A operand), once
                // its TMA load has landed and the previous item's last dP is done
                if (!(ok = mbar_wait_warp(&bars[BAR_Q_FULL], (uint32_t)k & 1u, ab))) break;
                if (k > 0 && !(ok = mbar_wait_warp(&bars[BAR_DO_FREE], (uint32_t)(k - 1) & 1u, ab))) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // 64 columns: row `row` of the 128-byte swizzled half, chunk c at c ^ (row % 8)
                    const uint8_t* src = smem + OFF_DO + h * DO_HALF + row * 128;
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) * 16));
                        w[4 * c] = x.x;
                        w[4 * c + 1] = x.y;
                        w[4 * c + 2] = x.z;
                        w[4 * c + 3] = x.w;
                    }
                    tmem_st32(lane_base + TM_DO + 32 * h, w);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_DO_READY]);
            }
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t nlse2 = f2_pack(nlse, nlse);
            const uint64_t coef2 = f2_pack(coef, coef);
            const uint64_t cndd2 = f2_pack(coef * ndd, coef * ndd);
            for (int j = 0; j < it.n_kv; ++j) {
                const int buf = j & 1;
                const uint32_t tS = lane_base + buf * 128 + br * 64;
                const uint32_t tP = lane_base + TM_DP;
                if (!(ok = BP_WAIT(pf, kQSFull, mbar_wait_warp(&bars[BAR_S_FULL + buf], (sph >> buf) & 1u, ab))))
                    break;
                BP_MARK(tp);
                sph ^= 1u << buf;
                tc_fence_after();
                uint32_t s[64], dp[64];
                tmem_ld32(tS, &s[0]);
                tmem_ld32(tS + 32, &s[32]);
                tmem_ld32(tP, &dp[0]);
                tmem_ld32(tP + 32, &dp[32]);
                tmem_wait_ld();
                // dP is in registers: the next tile's dP may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_DP_FREE]);
                BP_ADD(pf, kQRead, tp);
                BP_RESET(tp);
                const int kv0 = j * BN;
                // only tiles that cross the diagonal or the end of the sequence
                // need a mask (the decision is the same for the whole CTA)
                const bool edge = (p.causal && kv0 + BN - 1 > it.qt * BM) || kv0 + BN > p.T;
                uint32_t pk[32];
                if (edge) {
                    // keys kv0 + c with c > lim are masked (future, or past T)
                    int lim = p.causal ? q - kv0 : 63;
                    if (p.T - 1 - kv0 < lim) lim = p.T - 1 - kv0;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const uint64_t x = f2_fma(f2_from_bits(s[2 * c], s[2 * c + 1]), sl2x2, nlse2);
                        const float a0 = (2 * c > lim) ? 0.f : ex2_approx(f2_lo(x));
                        const float a1 = (2 * c + 1 > lim) ? 0.f : ex2_approx(f2_hi(x));
                        const uint64_t y = f2_fma(f2_from_bits(dp[2 * c], dp[2 * c + 1]), coef2, cndd2);
                        const uint64_t z = f2_mul(f2_pack(a0, a1), y);
                        pk[c] = pack_bf16x2(f2_lo(z), f2_hi(z));
                    }
                } else {
                    // in three phases, in place in the score registers, so that
                    // each is a run of independent operations: the exponents, the
                    // exponentials, then dS_b = coef * A_b * (dP - Dd_b)
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const uint64_t x = f2_fma(f2_from_bits(s[2 * c], s[2 * c + 1]), sl2x2, nlse2);
                        s[2 * c] = static_cast<uint32_t>(x);
                        s[2 * c + 1] = static_cast<uint32_t>(x >> 32);
                    }
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = __float_as_uint(ex2_approx(__uint_as_float(s[c])));
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const uint64_t y = f2_fma(f2_from_bits(dp[2 * c], dp[2 * c + 1]), coef2, cndd2);
                        const uint64_t z = f2_mul(f2_from_bits(s[2 * c], s[2 * c + 1]), y);
                        pk[c] = pack_bf16x2(f2_lo(z), f2_hi(z));
                    }
                }
                BP_ADD(pf, kQMath, tp);
                BP_RESET(tp);
                tmem_st32(tS, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_DS_FULL + buf]);
                BP_ADD(pf, kQStore, tp);
                BP_COUNT(pf, kQTiles);
            }
            if (!ok) break;
            BP_COUNT(pf, kQItems);
            // dQ_b = scale * (dS_b K_b): this warpgroup's 64 columns
            if (!(ok = BP_WAIT(pf, kQDqFull, mbar_wait_warp(&bars[BAR_DQ_FULL], dqph, ab)))) break;
            BP_MARK(te);
            dqph ^= 1;
            tc_fence_after();
            uint32_t g[64];
            tmem_ld32(lane_base + TM_DQ + br * 64, &g[0]);
            tmem_ld32(lane_base + TM_DQ + br * 64 + 32, &g[32]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BAR_DQ_EMPTY]);
            if (live) {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(br ? p.dq2 : p.dq1) +
                                     (((int64_t)it.b * p.H + it.h) * p.T + q) * HD;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 8 * i;
                    *reinterpret_cast<uint4*>(dst + c) = make_uint4(
                        pack_bf16x2(__uint_as_float(g[c]) * p.scale, __uint_as_float(g[c + 1]) * p.scale),
                        pack_bf16x2(__uint_as_float(g[c + 2]) * p.scale, __uint_as_float(g[c + 3]) * p.scale),
                        pack_bf16x2(__uint_as_float(g[c + 4]) * p.scale, __uint_as_float(g[c + 5]) * p.scale),
                        pack_bf16x2(__uint_as_float(g[c + 6]) * p.scale, __uint_as_float(g[c + 7]) * p.scale));
                }
            }
            BP_ADD(pf, kQEpilogue, te);
        }
        BP_FLUSH(pf, g_prof, 2, lane == 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace dq

// ===========================================================================
// dkdv kernel
// ===========================================================================
namespace dkdv {

// Wait profile of this kernel (g_prof[role][kind], see ProfT).  Roles: 0 the TMA producer, 1 the MMA-issuing thread, 2 the eight
// elementwise warps.  Kinds: 0 the role's cycles from start to end; the
// producer's waits for the K/V slot (1) and for a query stage (2) to be
// released; the MMA thread's waits for K/V (3), for the scores to be read out
// (4), for a query stage (5), for the bf16 operands (6) and for the
// accumulators to be read out (7); the elementwise warps' waits for the
// scores (8), their handling of the row statistics (9: scratch writes and the
// next tile's load), their TMEM read of the
// scores (10), arithmetic (11), wait for the previous tile's gradient
// products (12), operand stores (13), wait for the accumulators (14) and the
// epilogue (15); the tile (16) and item (17) counts.
enum : int {
    kPTotal = 0, kPKvEmpty = 1, kPQEmpty = 2, kPKvFull = 3, kPSFree = 4, kPQFull = 5,
    kPDsFull = 6, kPAccEmpty = 7, kPSFull = 8, kPStats = 9, kPRead = 10, kPMath = 11,
    kPPkFree = 12, kPStore = 13, kPAccFull = 14, kPEpilogue = 15, kPTiles = 16, kPItems = 17,
    kPKinds = 18
};
#ifdef DIFFATTN_WAIT_PROFILE
__device__ unsigned long long g_prof[3][kPKinds];
#endif
using Prof = ProfT<kPKinds>;

constexpr int BM = 128;            // key rows per item (TMEM lanes)
constexpr int BN = 64;             // query rows per tile
constexpr int QSTAGES = 4;         // (Q1, Q2, dO) ring
constexpr uint32_t K_BYTES = BM * HD * 2;          // 16 KB
constexpr uint32_t V_HALF = BM * 64 * 2;           // 16 KB
constexpr uint32_t Q_BYTES = BN * HD * 2;          // 8 KB
constexpr uint32_t DO_HALF = BN * 64 * 2;          // 8 KB
constexpr uint32_t QSTAGE_BYTES = 2 * Q_BYTES + 2 * DO_HALF;   // 32 KB
constexpr uint32_t QS_Q1 = 0, QS_Q2 = Q_BYTES, QS_DO = 2 * Q_BYTES;

constexpr uint32_t OFF_K1 = 0;
constexpr uint32_t OFF_K2 = OFF_K1 + K_BYTES;
constexpr uint32_t OFF_V = OFF_K2 + K_BYTES;                       // two halves
constexpr uint32_t OFF_QS = OFF_V + 2 * V_HALF;                    // stages (1024-aligned)
constexpr uint32_t QSTAGE_STRIDE = (QSTAGE_BYTES + 1023) & ~1023u;
// bf16 operand written to shared memory by the elementwise warps: dS_2^T
// [128 keys x 64 queries], K-major with 128-byte swizzling (W^T and dS_1^T go
// to tensor memory)
constexpr uint32_t PK_BYTES = BM * BN * 2;                         // 16 KB
constexpr uint32_t OFF_PK = OFF_QS + QSTAGES * QSTAGE_STRIDE;
// per elementwise warp: the row statistics of its 32 query columns, by
// quantity (-lse_1, -lse_2, -Dd_1, -Dd_2: 4 x 32 floats)
constexpr uint32_t SCR_BYTES = 8 * 4 * 32 * 4;                     // 4 KB
constexpr uint32_t OFF_SCR = OFF_PK + PK_BYTES;
constexpr uint32_t OFF_BAR = OFF_SCR + SCR_BYTES;
constexpr int BAR_KV_FULL = 0;
constexpr int BAR_KV_EMPTY = 1;
constexpr int BAR_Q_FULL = 2;
constexpr int BAR_Q_EMPTY = BAR_Q_FULL + QSTAGES;
constexpr int BAR_S_FULL = BAR_Q_EMPTY + QSTAGES;
constexpr int BAR_S_FREE = BAR_S_FULL + 1;            // 8 warps: scores read from TMEM
constexpr int BAR_DS_FULL = BAR_S_FREE + 1;           // 8 warps: bf16 operands in smem
constexpr int BAR_PK_FREE = BAR_DS_FULL + 1;          // MMA: the operands have been read
constexpr int BAR_ACC_FULL = BAR_PK_FREE + 1;
constexpr int BAR_ACC_EMPTY = BAR_ACC_FULL + 1;       // 8 warps
constexpr int BAR_FINAL = BAR_ACC_EMPTY + 1;
constexpr int NUM_BARS = BAR_FINAL + 1;
constexpr uint32_t OFF_TMEM_PTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_PTR + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM: S1^T [0,64), S2^T [64,128), dP^T [128,192); dV [192,320), dK1
// [320,384), dK2 [384,448); the bf16 operands W^T [448,480) and dS1^T
// [480,512) (32 columns each: two queries per column).
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S1 = 0, TM_S2 = 64, TM_DP = 128, TM_DV = 192, TM_DK1 = 320, TM_DK2 = 384;
constexpr uint32_t TM_W = 448, TM_DS1 = 480;
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);     // K x Q^T, V x dO^T
constexpr uint32_t IDESC_DV = idesc_bf16_f32(BM, VD, 0, 1);    // W^T (TMEM) x dO (MN-major)
constexpr uint32_t IDESC_DK = idesc_bf16_f32(BM, HD, 0, 1);    // dS^T x Q (MN-major)

struct Item {
    int b, hk, kt;
    int qt0;        // first 64-row query tile that sees a key of the tile
    int per_head;   // query tiles per head
};
__device__ __forceinline__ Item decode_item(int idx, const BwdTcParams& p) {
    // longest first: causal key tiles near the start see the most queries
    const int BHk = p.B * p.Hk;
    const int r = idx / BHk;
    const int bhk = idx - r * BHk;
    Item it;
    it.kt = r;
    it.b = bhk / p.Hk;
    it.hk = bhk - it.b * p.Hk;
    it.qt0 = p.causal ? 2 * r : 0;
    it.per_head = p.nk64 - it.qt0;     // 64-row query tiles [qt0, nk64)
    return it;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q1,
                         const __grid_constant__ CUtensorMap tm_k1,
                         const __grid_constant__ CUtensorMap tm_q2,
                         const __grid_constant__ CUtensorMap tm_k2,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const BwdTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + OFF_TMEM_PTR);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
    const uint32_t warp = warp_id();
    const uint32_t lane = threadIdx.x & 31;
    const AbortState ab{abort_flag, p.status};
    const int total = p.B * p.Hk * p.nk128;
    const int g = p.kv_group;

    if (threadIdx.x == 0) {
        mbar_init(&bars[BAR_KV_FULL], 1);
        mbar_init(&bars[BAR_KV_EMPTY], 1);
        for (int s = 0; s < QSTAGES; ++s) {
            mbar_init(&bars[BAR_Q_FULL + s], 1);
            mbar_init(&bars[BAR_Q_EMPTY + s], 1);
        }
        mbar_init(&bars[BAR_S_FULL], 1);
        mbar_init(&bars[BAR_S_FREE], 8);
        mbar_init(&bars[BAR_DS_FULL], 8);
        mbar_init(&bars[BAR_PK_FREE], 1);
        mbar_init(&bars[BAR_ACC_FULL], 1);
        mbar_init(&bars[BAR_ACC_EMPTY], 8);
        mbar_init(&bars[BAR_FINAL], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_ptr, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;
    const int grid = gridDim.x, cta = blockIdx.x;

    if (warp >= 8) {
        regs_dec<REGS_OTHER>();
        if (warp == 8) {
            // ------------------------------------------------------ producer
            if (elect_one()) {
                Prof pf;
                pf.start();
                uint32_t qs = 0, qph = 0, kvph = 0;
                uint32_t armed_kv = 0, armed_q[QSTAGES] = {};
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int idx = item_index(k, cta, grid);
                    if (idx >= total) break;
                    const Item it = decode_item(idx, p);
                    if (k > 0) {
                        if (!(ok = BP_WAIT(pf, kPKvEmpty, mbar_wait(&bars[BAR_KV_EMPTY], kvph, ab)))) break;
                        kvph ^= 1;
                    }
                    const int k0 = it.kt * BM;
                    mbar_arrive_expect_tx(&bars[BAR_KV_FULL], 2 * K_BYTES + 2 * V_HALF);
                    tma_load_4d(smem + OFF_K1, &tm_k1, &bars[BAR_KV_FULL], 0, k0, it.hk, it.b);
                    tma_load_4d(smem + OFF_K2, &tm_k2, &bars[BAR_KV_FULL], 0, k0, it.hk, it.b);
                    tma_load_4d(smem + OFF_V, &tm_v, &bars[BAR_KV_FULL], 0, k0, it.hk, it.b);
                    tma_load_4d(smem + OFF_V + V_HALF, &tm_v, &bars[BAR_KV_FULL], 64, k0, it.hk, it.b);
                    ++armed_kv;
                    for (int t = 0; t < g * it.per_head && ok; ++t) {
                        const int h = it.hk * g + t / it.per_head;
                        const int qt = it.qt0 + t % it.per_head;
                        if (!(ok = BP_WAIT(pf, kPQEmpty, mbar_wait(&bars[BAR_Q_EMPTY + qs], qph ^ 1, ab)))) break;
                        uint8_t* st = smem + OFF_QS + qs * QSTAGE_STRIDE;
                        const int q0 = qt * BN;
                        mbar_arrive_expect_tx(&bars[BAR_Q_FULL + qs], QSTAGE_BYTES);
                        tma_load_4d(st + QS_Q1, &tm_q1, &bars[BAR_Q_FULL + qs], 0, q0, h, it.b);
                        tma_load_4d(st + QS_Q2, &tm_q2, &bars[BAR_Q_FULL + qs], 0, q0, h, it.b);
                        tma_load_4d(st + QS_DO, &tm_do, &bars[BAR_Q_FULL + qs], 0, q0, h, it.b);
                        tma_load_4d(st + QS_DO + DO_HALF, &tm_do, &bars[BAR_Q_FULL + qs], 64, q0, h, it.b);
                        ++armed_q[qs];
                        if (++qs == QSTAGES) { qs = 0; qph ^= 1; }
                    }
                }
                const uint64_t lim = 200ull * 1000ull * 1000ull;
                if (armed_kv) mbar_wait_teardown(&bars[BAR_KV_FULL], (armed_kv - 1) & 1, lim);
                for (int s = 0; s < QSTAGES; ++s)
                    if (armed_q[s]) mbar_wait_teardown(&bars[BAR_Q_FULL + s], (armed_q[s] - 1) & 1, lim);
                BP_FLUSH(pf, g_prof, 0, true);
            }
            __syncwarp();
        } else if (warp == 9) {
            // ------------------------------------------------------ MMA issue
            if (elect_one()) {
                Prof pf;
                pf.start();
                const uint64_t k1d = sdesc_sw128(smem_u32(smem + OFF_K1), 16, 1024);
                const uint64_t k2d = sdesc_sw128(smem_u32(smem + OFF_K2), 16, 1024);
                const uint64_t vd = sdesc_sw128(smem_u32(smem + OFF_V), 16, 1024);
                const uint64_t qk = sdesc_sw128(smem_u32(smem + OFF_QS), 16, 1024);       // K-major
                const uint64_t qm = sdesc_sw128(smem_u32(smem + OFF_QS), DO_HALF, 1024);  // MN-major
                const uint64_t pkd = sdesc_sw128(smem_u32(smem + OFF_PK), 16, 1024);      // K-major
                uint32_t kvph = 0, accph = 0, dsph = 0;
                uint32_t tiles = 0;       // query tiles whose scores were issued (whole launch)
                uint32_t done = 0;        // query tiles whose dV/dK products were issued
                bool ok = true, first = true;
                // S_1^T, S_2^T, dP^T of the next query tile (stage tiles % QSTAGES);
                // the previous tile's scores must have been read out of TMEM.
                auto issue_s = [&]() -> bool {
                    const uint32_t qs = tiles % QSTAGES;
                    if (tiles > 0 && !BP_WAIT(pf, kPSFree, mbar_wait(&bars[BAR_S_FREE], (tiles - 1) & 1u, ab)))
                        return false;
                    if (!BP_WAIT(pf, kPQFull, mbar_wait(&bars[BAR_Q_FULL + qs], (tiles / QSTAGES) & 1u, ab)))
                        return false;
                    tc_fence_after();
                    const uint64_t sb = (qs * QSTAGE_STRIDE) >> 4;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        mma_ss(tmem_base + TM_S1, k1d + 2 * kk, qk + sb + (QS_Q1 >> 4) + 2 * kk,
                               IDESC_S, kk > 0);
                        mma_ss(tmem_base + TM_S2, k2d + 2 * kk, qk + sb + (QS_Q2 >> 4) + 2 * kk,
                               IDESC_S, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < VD / 16; ++kk) {
                        const uint32_t aoff = (kk >> 2) * (V_HALF >> 4) + 2 * (kk & 3);
                        const uint32_t boff = (QS_DO >> 4) + (kk >> 2) * (DO_HALF >> 4) + 2 * (kk & 3);
                        mma_ss(tmem_base + TM_DP, vd + aoff, qk + sb + boff, IDESC_S, kk > 0);
                    }
                    mma_commit(&bars[BAR_S_FULL]);
                    ++tiles;
                    return true;
                };
                for (int k = 0; ok; ++k) {
                    const int idx = item_index(k, cta, grid);
                    if (idx >= total) break;
                    const Item it = decode_item(idx, p);
                    const int n = g * it.per_head;
                    if (!(ok = BP_WAIT(pf, kPKvFull, mbar_wait(&bars[BAR_KV_FULL], kvph, ab)))) break;
                    kvph ^= 1;
                    if (!(ok = issue_s())) break;
                    if (n == 1) mma_commit(&bars[BAR_KV_EMPTY]);
                    for (int t = 0; t < n; ++t) {
                        // the next tile's scores overlap this tile's elementwise work
                        if (t + 1 < n) {
                            if (!(ok = issue_s())) break;
                            if (t + 2 == n) mma_commit(&bars[BAR_KV_EMPTY]);
                        }
                        if (!(ok = BP_WAIT(pf, kPDsFull, mbar_wait(&bars[BAR_DS_FULL], dsph, ab)))) break;
                        dsph ^= 1;
                        if (t == 0 && !first) {
                            if (!(ok = BP_WAIT(pf, kPAccEmpty, mbar_wait(&bars[BAR_ACC_EMPTY], accph, ab)))) break;
                            accph ^= 1;
                        }
                        tc_fence_after();
                        const uint32_t qs = done % QSTAGES;
                        const uint64_t sb = (qs * QSTAGE_STRIDE) >> 4;
                        // dV += W^T dO, dK_1 += dS_1^T Q_1 (A operands from TMEM),
                        // dK_2 += dS_2^T Q_2 (A operand from shared memory)
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                            mma_ts(tmem_base + TM_DV, tmem_base + TM_W + kk * 8,
                                   qm + sb + (QS_DO >> 4) + 128 * kk, IDESC_DV, acc);
                            mma_ts(tmem_base + TM_DK1, tmem_base + TM_DS1 + kk * 8,
                                   qm + sb + (QS_Q1 >> 4) + 128 * kk, IDESC_DK, acc);
                            mma_ss(tmem_base + TM_DK2, pkd + 2 * kk,
                                   qm + sb + (QS_Q2 >> 4) + 128 * kk, IDESC_DK, acc);
                        }
                        mma_commit(&bars[BAR_PK_FREE]);
                        mma_commit(&bars[BAR_Q_EMPTY + qs]);
                        ++done;
                    }
                    if (!ok) break;
                    mma_commit(&bars[BAR_ACC_FULL]);
                    first = false;
                }
                mma_commit(&bars[BAR_FINAL]);
                mbar_wait_teardown(&bars[BAR_FINAL], 0, 200ull * 1000ull * 1000ull);
                BP_FLUSH(pf, g_prof, 1, true);
            }
            __syncwarp();
        }
    } else {
        regs_inc<REGS_WORK>();
        // ---------------------------------- dS^T, W^T and the dK/dV epilogue
        Prof pf;
        pf.start();
        const int half = warp >> 2;          // query columns [32*half, 32*half + 32)
        const uint32_t quad = warp & 3;
        const int row = quad * 32 + lane;    // key row within the tile
        const uint32_t lane_base = tmem_base + ((quad * 32u) << 16);
        const float sl2 = p.scale_log2;
        const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
        uint32_t accph = 0, qc = 0;   // qc: query tiles consumed (whole launch)
        bool ok = true;
        // Row statistics (-lse_1, -lse_2, -Dd_1, -Dd_2) of the warp's 32 query
        // columns: lane l loads column l's from global memory one tile ahead
        // (zeros past T) and, when the tile starts, writes them to the warp's
        // scratch by quantity, so that the packed f32x2 arithmetic reads the
        // values of a column pair with one load and the tile's products wait
        // on no copy of them.
        float* scr = reinterpret_cast<float*>(smem + OFF_SCR) + warp * 128;
        const int col = 32 * half + (int)lane;
        auto stats_of = [&](int b, int h, int qt) -> float4 {
            const int q = qt * BN + col;
            if (q >= p.T) return make_float4(0.f, 0.f, 0.f, 0.f);
            return __ldg(reinterpret_cast<const float4*>(p.stats) + (((int64_t)b * p.H + h) * p.T + q));
        };
        float4 nst = make_float4(0.f, 0.f, 0.f, 0.f);     // the next tile's statistics
        if (item_index(0, cta, grid) < total) {
            const Item it0 = decode_item(item_index(0, cta, grid), p);
            nst = stats_of(it0.b, it0.hk * g, it0.qt0);
        }
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, cta, grid);
            if (idx >= total) break;
            const Item it = decode_item(idx, p);
            const int key = it.kt * BM + row;
            const int n = g * it.per_head;
            int h = it.hk * g, qt = it.qt0;  // the tile's query head and 64-row query tile
            for (int t = 0; t < n; ++t, ++qc) {
                int h1 = h, qt1 = qt + 1;    // the next tile's
                if (qt1 == p.nk64) {
                    qt1 = it.qt0;
                    ++h1;
                }
                BP_MARK(tp);
                __syncwarp();               // the previous tile's reads of the scratch are done
                scr[lane] = nst.x;
                scr[32 + lane] = nst.y;
                scr[64 + lane] = nst.z;
                scr[96 + lane] = nst.w;
                __syncwarp();
                if (t + 1 < n) {
                    nst = stats_of(it.b, h1, qt1);
                } else {
                    const int nidx = item_index(k + 1, cta, grid);
                    if (nidx < total) {
                        const Item nit = decode_item(nidx, p);
                        nst = stats_of(nit.b, nit.hk * g, nit.qt0);
                    }
                }
                BP_ADD(pf, kPStats, tp);
                if (!(ok = BP_WAIT(pf, kPSFull, mbar_wait_warp(&bars[BAR_S_FULL], qc & 1u, ab)))) break;
                BP_RESET(tp);
                tc_fence_after();
                const uint32_t c0 = 32 * half;
                uint32_t s1[32], s2[32], dp[32];
                tmem_ld32(lane_base + TM_S1 + c0, s1);
                tmem_ld32(lane_base + TM_S2 + c0, s2);
                tmem_ld32(lane_base + TM_DP + c0, dp);
                tmem_wait_ld();
                // the scores are in registers: the next tile's products may overwrite them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_S_FREE]);
                BP_ADD(pf, kPRead, tp);
                BP_RESET(tp);
                // query qt*64 + c0 + c sees this key iff key <= query (and query < T);
                // statistics are stored negated: (-lse_1, -lse_2, -Dd_1, -Dd_2)
                const int qbase = qt * BN + (int)c0;
                uint32_t w1[16], w2[16], w3[16];
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t nlam2 = f2_pack(-lam, -lam);
                // only warps whose 32 queries meet the diagonal or the end of the
                // sequence need a mask (the decision is the same for the whole warp)
                const bool edge = (p.causal && qbase < it.kt * BM + BM - 1) || qbase + 32 > p.T;
                if (edge) {
                    const int first_vis = p.causal ? key - qbase : 0;   // columns c >= first_vis are visible
                    const int qlim = p.T - qbase;                         // columns c < qlim exist
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float4 sa = make_float4(scr[c], scr[32 + c], scr[64 + c], scr[96 + c]);
                        const float4 sb = make_float4(scr[c + 1], scr[33 + c], scr[65 + c], scr[97 + c]);
                        const bool v0 = c >= first_vis && c < qlim;
                        const bool v1 = c + 1 >= first_vis && c + 1 < qlim;
                        const float a10 = v0 ? ex2_approx(fmaf(__uint_as_float(s1[c]), sl2, sa.x)) : 0.f;
                        const float a11 = v1 ? ex2_approx(fmaf(__uint_as_float(s1[c + 1]), sl2, sb.x)) : 0.f;
                        const float a20 = v0 ? ex2_approx(fmaf(__uint_as_float(s2[c]), sl2, sa.y)) : 0.f;
                        const float a21 = v1 ? ex2_approx(fmaf(__uint_as_float(s2[c + 1]), sl2, sb.y)) : 0.f;
                        const float p0 = __uint_as_float(dp[c]), p1 = __uint_as_float(dp[c + 1]);
                        // statistics of queries at or past T are not loaded: select, never
                        // multiply, so that whatever the buffer holds cannot reach the sums
                        const float d10 = v0 ? a10 * (p0 + sa.z) : 0.f;
                        const float d11 = v1 ? a11 * (p1 + sb.z) : 0.f;
                        const float d20 = v0 ? -lam * a20 * (p0 + sa.w) : 0.f;
                        const float d21 = v1 ? -lam * a21 * (p1 + sb.w) : 0.f;
                        w1[c / 2] = pack_bf16x2(d10, d11);
                        w2[c / 2] = pack_bf16x2(d20, d21);
                        w3[c / 2] = pack_bf16x2(a10 - lam * a20, a11 - lam * a21);
                    }
                } else {
                    // In three phases over all 32 columns, in place in the score
                    // registers, so that every phase is a run of independent
                    // operations: the exponents, the exponentials (A_1, A_2), then
                    // dS_1, dS_2 and W.  Columns c .. c + 3 take one load of each
                    // statistic (two column pairs).
                    const float4* pl = reinterpret_cast<const float4*>(scr);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 l1 = pl[c / 4], l2 = pl[8 + c / 4];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int cc = c + 2 * hh;
                            const uint64_t L1 = hh ? f2_pack(l1.z, l1.w) : f2_pack(l1.x, l1.y);
                            const uint64_t L2 = hh ? f2_pack(l2.z, l2.w) : f2_pack(l2.x, l2.y);
                            const uint64_t x1 = f2_fma(f2_from_bits(s1[cc], s1[cc + 1]), sl2x2, L1);
                            const uint64_t x2 = f2_fma(f2_from_bits(s2[cc], s2[cc + 1]), sl2x2, L2);
                            s1[cc] = static_cast<uint32_t>(x1);
                            s1[cc + 1] = static_cast<uint32_t>(x1 >> 32);
                            s2[cc] = static_cast<uint32_t>(x2);
                            s2[cc + 1] = static_cast<uint32_t>(x2 >> 32);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        s1[c] = __float_as_uint(ex2_approx(__uint_as_float(s1[c])));
                        s2[c] = __float_as_uint(ex2_approx(__uint_as_float(s2[c])));
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 e1 = pl[16 + c / 4], e2 = pl[24 + c / 4];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int cc = c + 2 * hh;
                            const uint64_t E1 = hh ? f2_pack(e1.z, e1.w) : f2_pack(e1.x, e1.y);
                            const uint64_t E2 = hh ? f2_pack(e2.z, e2.w) : f2_pack(e2.x, e2.y);
                            const uint64_t a1 = f2_from_bits(s1[cc], s1[cc + 1]);
                            const uint64_t a2n = f2_mul(f2_from_bits(s2[cc], s2[cc + 1]), nlam2);
                            const uint64_t dp2 = f2_from_bits(dp[cc], dp[cc + 1]);
                            const uint64_t d1 = f2_mul(a1, f2_add(dp2, E1));
                            const uint64_t d2 = f2_mul(a2n, f2_add(dp2, E2));
                            const uint64_t w = f2_add(a1, a2n);
                            w1[cc / 2] = pack_bf16x2(f2_lo(d1), f2_hi(d1));
                            w2[cc / 2] = pack_bf16x2(f2_lo(d2), f2_hi(d2));
                            w3[cc / 2] = pack_bf16x2(f2_lo(w), f2_hi(w));
                        }
                    }
                }
                BP_ADD(pf, kPMath, tp);
                // the previous tile's dV/dK products must have read the operands
                if (qc > 0 && !(ok = BP_WAIT(pf, kPPkFree, mbar_wait_warp(&bars[BAR_PK_FREE], (qc - 1) & 1u, ab))))
                    break;
                BP_RESET(tp);
                // W^T and dS_1^T to TMEM: queries [c0, c0 + 32) are packed columns
                // [16*half, 16*half + 16) of their regions
                tmem_st16(lane_base + TM_W + 16 * half, w3);
                tmem_st16(lane_base + TM_DS1 + 16 * half, w1);
                // dS_2^T to shared memory: row `row`, queries [c0, c0 + 32) = 16-byte
                // chunks 4*half .. 4*half + 3, swizzled by the row's position within
                // its 8-row group
                uint8_t* prow = smem + OFF_PK + row * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = (uint32_t)(((4 * half + i) ^ (row & 7)) * 16);
                    *reinterpret_cast<uint4*>(prow + off) =
                        make_uint4(w2[4 * i], w2[4 * i + 1], w2[4 * i + 2], w2[4 * i + 3]);
                }
                fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_DS_FULL]);
                BP_ADD(pf, kPStore, tp);
                BP_COUNT(pf, kPTiles);
                h = h1;
                qt = qt1;
            }
            if (!ok) break;
            BP_COUNT(pf, kPItems);
            // epilogue: warpgroup 0 writes dV columns 0-63 and dK_1, warpgroup
            // 1 dV columns 64-127 and dK_2
            if (!(ok = BP_WAIT(pf, kPAccFull, mbar_wait_warp(&bars[BAR_ACC_FULL], accph, ab)))) break;
            BP_MARK(te);
            accph ^= 1;
            tc_fence_after();
            uint32_t gv[64], gk[64];
            tmem_ld32(lane_base + TM_DV + 64 * half, &gv[0]);
            tmem_ld32(lane_base + TM_DV + 64 * half + 32, &gv[32]);
            tmem_ld32(lane_base + (half ? TM_DK2 : TM_DK1), &gk[0]);
            tmem_ld32(lane_base + (half ? TM_DK2 : TM_DK1) + 32, &gk[32]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BAR_ACC_EMPTY]);
            if (key < p.T) {
                const int64_t krow = ((int64_t)it.b * p.Hk + it.hk) * p.T + key;
                __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(p.dv) + krow * VD + 64 * half;
                __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(half ? p.dk2 : p.dk1) + krow * HD;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 8 * i;
                    *reinterpret_cast<uint4*>(dv + c) = make_uint4(
                        pack_bf16x2(__uint_as_float(gv[c]), __uint_as_float(gv[c + 1])),
                        pack_bf16x2(__uint_as_float(gv[c + 2]), __uint_as_float(gv[c + 3])),
                        pack_bf16x2(__uint_as_float(gv[c + 4]), __uint_as_float(gv[c + 5])),
                        pack_bf16x2(__uint_as_float(gv[c + 6]), __uint_as_float(gv[c + 7])));
                    *reinterpret_cast<uint4*>(dk + c) = make_uint4(
                        pack_bf16x2(__uint_as_float(gk[c]) * p.scale, __uint_as_float(gk[c + 1]) * p.scale),
                        pack_bf16x2(__uint_as_float(gk[c + 2]) * p.scale, __uint_as_float(gk[c + 3]) * p.scale),
                        pack_bf16x2(__uint_as_float(gk[c + 4]) * p.scale, __uint_as_float(gk[c + 5]) * p.scale),
                        pack_bf16x2(__uint_as_float(gk[c + 6]) * p.scale, __uint_as_float(gk[c + 7]) * p.scale));
                }
            }
            BP_ADD(pf, kPEpilogue, te);
        }
        BP_FLUSH(pf, g_prof, 2, lane == 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace dkdv

}  // namespace bwdtc

#ifdef DIFFATTN_WAIT_PROFILE
// The backward kernels' wait-profile counters accumulated since the last call,
// copied to `out` and cleared: the dK/dV kernel's [3 roles][18 kinds], then,
// when `n` has room, the dQ kernel's [3][17].  Only in the build with
// -DDIFFATTN_WAIT_PROFILE.
extern "C" int diffattn_bwd_wait_profile(unsigned long long* out, int n) {
    constexpr int kN = 3 * bwdtc::dkdv::kPKinds;
    constexpr int kQ = 3 * bwdtc::dq::kQKinds;
    if (!out || n < kN) return -1;
    static unsigned long long zero[kN > kQ ? kN : kQ] = {};
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(out, bwdtc::dkdv::g_prof, kN * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMemcpyToSymbol(bwdtc::dkdv::g_prof, zero, kN * sizeof(unsigned long long)) != cudaSuccess)
        return -3;
    if (n >= kN + kQ &&
        (cudaMemcpyFromSymbol(out + kN, bwdtc::dq::g_prof, kQ * sizeof(unsigned long long)) != cudaSuccess ||
         cudaMemcpyToSymbol(bwdtc::dq::g_prof, zero, kQ * sizeof(unsigned long long)) != cudaSuccess))
        return -3;
    return 0;
}
#endif

int launch_bwd_tc(const CUtensorMap* maps, const BwdTcParams& p, int num_sms, cudaStream_t stream) {
    using namespace bwdtc;
    if (cudaFuncSetAttribute(dq::diffattn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dq::SMEM_BYTES) != cudaSuccess)
        return -1;
    if (cudaFuncSetAttribute(dkdv::diffattn_bwd_dkdv_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dkdv::SMEM_BYTES) != cudaSuccess)
        return -1;
    const int dq_items = p.B * p.H * p.nq128;
    const int kv_items = p.B * p.Hk * p.nk128;
    dq::diffattn_bwd_dq_kernel<<<dq_items < num_sms ? dq_items : num_sms, NUM_THREADS,
                                 dq::SMEM_BYTES, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                           maps[4], maps[5], p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // The dK/dV kernel depends on the row statistics (complete before the dQ
    // kernel started), not on dQ: it is launched as a programmatic dependent of
    // the dQ kernel, so its CTAs fill the SMs the dQ kernel's tail leaves idle.
    // One CTA of either kernel takes a whole SM's registers, so they never
    // share an SM (nor its tensor memory).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kv_items < num_sms ? kv_items : num_sms);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = dkdv::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dkdv::diffattn_bwd_dkdv_kernel, maps[6], maps[7], maps[8], maps[9],
                              maps[10], maps[11], p) == cudaSuccess
               ? 0
               : -1;
}

}  // namespace diffattn
