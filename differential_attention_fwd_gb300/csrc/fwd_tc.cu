// fwd_tc.cu -- differential-attention forward on the sm_103a tensor cores.
//
// Computes O = (softmax(Q1 K1^T / sqrt(D) + M) - lambda softmax(Q2 K2^T / sqrt(D) + M)) V
// (paperleet "Differential Transformer Attention", Formula and conventions;
// aifetchly "Differential Transformer...", section 1) for bf16 inputs with
// V width 128 and Q/K width D = 64 (the operation's own shape, V = 2D) or
// D = 128 (the DIFF V2 head of the aiengineeringfromscratch lesson, "V1 contre
// V2": the head dimension stays that of the baseline, so V is as wide as Q and
// K), fp32 accumulation, bf16 output.
//
// Queries and keys may be sequences of different lengths (queries over a
// key/value cache): query row i sits at key position i + kv_off, and the
// causal mask hides keys j > i + kv_off.
//
// One CTA per SM (persistent).  A work item is (batch b, head h, 128-query
// tile).  Per item the CTA loads Q1/Q2 once and streams (K1, K2) and V tiles
// of 64 keys through TMA rings in shared memory.  Both score products
// S_b = Q_b K_b^T run as tcgen05 MMAs into tensor memory (TMEM), each branch
// with two S buffers so that the MMA of tile j+1 overlaps the softmax of tile
// j.  Each branch keeps its own streaming-softmax row state (max and sum) in
// the registers of its own warpgroup, one query row per thread; the
// probabilities P_b are written back over S_b in TMEM as bf16 and feed the
// O_b += P_b V MMAs, both reading the same V tile from shared memory.  The
// epilogue writes O_1 / l_1 - lambda O_2 / l_2.
//
// Warp roles (384 threads = 3 warpgroups):
//   warps 0-3   softmax + epilogue, branch 1 (TMEM lanes 0-127)
//   warps 4-7   softmax + epilogue, branch 2
//   warp  8     TMA producer
//   warp  9     TMEM allocation; MMA issue for branch 1
//   warp  10    MMA issue for branch 2
//   warp  11    idle (it completes the third warpgroup)
// One MMA-issuing thread per branch, so each branch's PV and next score
// product go to the tensor core as soon as that branch's P is ready.
// Registers: launched at 168 per thread (384 x 168 = 64512); the third
// warpgroup gives registers back (104 per thread) and the two softmax
// warpgroups take them (200 per thread): 256 x 200 + 128 x 104 = 64512.
// TMEM columns: S1 buffers [0,64) [64,128), S2 buffers [128,192) [192,256),
// O1 [256,384), O2 [384,512) (the same at D = 64 and D = 128: only the depth of
// the score products changes).
//
// Shared memory holds Q and K rows as 64-column panels of 128 bytes per row
// (the 128-byte swizzle span): one panel at D = 64, two at D = 128.  The key
// ring has 5 stages of (K1, K2) at D = 64; at D = 128 it has 2 such stages, or
// 4 stages of one shared key tile when the branches share their keys.
//
// Tensor-core order per branch b (its own issuing thread, executed in order):
//   S_b(0), S_b(1), then for each tile j: PV_b(j), S_b(j+2) into the buffer
//   PV_b(j) has just read P_b(j) from.  Shared resources (a K or V stage, the
//   Q tile, O) are released when both branches' commits have arrived.
//
// Grouped key/value heads: query head h reads the K1, K2 and V tiles of
// key/value head h / kv_group.  When K1 and K2 are one tensor (the two
// branches share their keys), each key tile is loaded once and both score
// products read it from the same shared-memory stage.
//
// Causal masking (both branches): KV tiles above the diagonal are never
// loaded; tiles that cross the diagonal mask key > query with -inf before the
// row max.
//
// Streaming softmax: the running max m is kept in log2 units of the scaled
// scores.  O and l are rescaled only when a tile's row max exceeds m by more
// than 8 (a factor 256), so P stays <= 256 and the rescale (a TMEM
// read-modify-write of the O row) is rare.  This lazy rescaling is the
// conditional-rescale idea of FlashAttention-4; the final O / l is exact
// whichever m was used.
#include "ptx.cuh"
#include "kernels.h"

namespace diffattn {
namespace tc {

constexpr int BM = 128;            // query rows per tile (= TMEM lanes)
constexpr int BN = 64;             // keys per KV tile
constexpr int VD = 128;            // V/O width
constexpr int KSTAGES = 5;         // key ring stages allocated (barriers)
constexpr int NUM_THREADS = 384;
constexpr uint32_t REGS_SOFTMAX = 200;
constexpr uint32_t REGS_OTHER = 104;
static_assert(256 * REGS_SOFTMAX + 128 * REGS_OTHER <= NUM_THREADS * 168, "register split");

constexpr uint32_t Q_PANEL = BM * 64 * 2;        // 16 KB: 128 query rows x 64 columns
constexpr uint32_t K_PANEL = BN * 64 * 2;        // 8 KB: 64 key rows x 64 columns
constexpr uint32_t V_HALF_BYTES = BN * 64 * 2;   // 8 KB per 64-column half
constexpr uint32_t V_BYTES = 2 * V_HALF_BYTES;   // 16 KB
constexpr uint32_t OUT_BYTES = BM * VD * 2;      // 32 KB

// Shared-memory layout for Q/K width HD (offsets from a 1024-byte aligned
// base).  Q1, Q2: PANELS panels each; the key ring: K_RING bytes; the value
// ring: VSTAGES stages (cols 0-63 at +0, 64-127 at +V_HALF_BYTES); the output
// staging: [branch][warp] 32 rows x 128 bytes.
template <int HD>
struct Cfg {
    static_assert(HD == 64 || HD == 128, "Q/K width");
    static constexpr int PANELS = HD / 64;
    static constexpr uint32_t Q_BYTES = BM * HD * 2;       // per branch
    static constexpr uint32_t K_BYTES = BN * HD * 2;       // one branch's key tile
    static constexpr uint32_t K_RING = HD == 64 ? KSTAGES * 2 * K_BYTES : 4 * K_BYTES;
    static constexpr int VSTAGES = HD == 64 ? 4 : 3;
    static constexpr uint32_t OFF_Q1 = 0;
    static constexpr uint32_t OFF_Q2 = OFF_Q1 + Q_BYTES;
    static constexpr uint32_t OFF_K = OFF_Q2 + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + K_RING;
    static constexpr uint32_t OFF_OUT = OFF_V + VSTAGES * V_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_OUT + OUT_BYTES;
    // key ring: stages and the byte stride between them (one key tile per
    // branch, or one shared by both)
    __device__ __forceinline__ static int kstages(bool shared) {
        return HD == 64 ? KSTAGES : (shared ? 4 : 2);
    }
    __device__ __forceinline__ static uint32_t kstride(bool shared) {
        return (HD == 128 && shared) ? K_BYTES : 2 * K_BYTES;
    }
};
constexpr int VSTAGES_MAX = 4;
// barriers
constexpr int BAR_Q_FULL = 0;
constexpr int BAR_Q_EMPTY = 1;
constexpr int BAR_K_FULL = 2;
constexpr int BAR_K_EMPTY = BAR_K_FULL + KSTAGES;
constexpr int BAR_V_FULL = BAR_K_EMPTY + KSTAGES;
constexpr int BAR_V_EMPTY = BAR_V_FULL + VSTAGES_MAX;
constexpr int BAR_S_FULL = BAR_V_EMPTY + VSTAGES_MAX;  // [branch][buffer]
constexpr int BAR_P_FULL = BAR_S_FULL + 4;             // [branch][buffer]
constexpr int BAR_PV_DONE = BAR_P_FULL + 4;            // [branch]
constexpr int BAR_O_FULL = BAR_PV_DONE + 2;
constexpr int BAR_O_EMPTY = BAR_O_FULL + 1;
constexpr int BAR_L_READY = BAR_O_EMPTY + 1;           // 1/l of both branches in smem
constexpr int BAR_FINAL = BAR_L_READY + 1;              // [branch]
constexpr int ITEM_RING = 8;                            // published work items in flight
constexpr int BAR_ITEM_FULL = BAR_FINAL + 2;            // [ITEM_RING] producer -> consumers
constexpr int BAR_ITEM_EMPTY = BAR_ITEM_FULL + ITEM_RING;  // [ITEM_RING] 10 consumer warps
constexpr int NUM_ITEM_CONSUMERS = 10;                  // 2 MMA warps + 8 softmax warps
constexpr int BAR_NORM_A = BAR_ITEM_EMPTY + ITEM_RING;  // per-row partial sums of both halves
constexpr int BAR_NORM_B = BAR_NORM_A + 1;              // per-row partial squared deviations
constexpr int NUM_BARS = BAR_NORM_B + 1;
// small state after the barriers (offsets from OFF_BAR)
constexpr uint32_t REL_TMEM_PTR = NUM_BARS * 8;
constexpr uint32_t REL_ABORT = REL_TMEM_PTR + 4;
constexpr uint32_t REL_INVL = (REL_ABORT + 4 + 15) & ~15u;     // float [2][128]
constexpr uint32_t REL_RING = REL_INVL + 2 * BM * 4;             // int [ITEM_RING]
constexpr uint32_t REL_STAT = REL_RING + ITEM_RING * 4;          // float [2 stats][2 halves][128]
constexpr uint32_t REL_END = REL_STAT + 2 * 2 * BM * 4;
template <int HD>
constexpr uint32_t smem_bytes() { return Cfg<HD>::OFF_BAR + REL_END + 1024; }   // + alignment slack

static_assert(smem_bytes<64>() <= 232448 && smem_bytes<128>() <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 256;                                   // O1 at 256, O2 at 384
constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);   // Q (K-major) x K^T (K-major), K = 16 per product
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, VD, 0, 1);  // P (TMEM) x V (MN-major)

__device__ __forceinline__ uint32_t tm_s(int br, int buf) { return br * 128 + buf * 64; }

struct Item {
    int qt, b, h, n_kv;
};

// The CTA's k-th work item in a boustrophedon order over the item list, so
// that with causal items sorted longest-first every CTA gets a similar total.
__device__ __forceinline__ int item_index(int k, int cta, int grid) {
    const int base = k * grid;
    return base + ((k & 1) ? (grid - 1 - cta) : cta);
}

// Item list: heads are taken in groups of p.group heads (a group's K1/K2/V
// fits comfortably in L2, so the CTAs working at the same time share it);
// within a group, items run longest first (causal: last query tile first),
// then head by head.
__device__ __forceinline__ Item decode_item(int idx, const TcParams& p) {
    const int BH = p.B * p.H;
    const int per_group = p.group * p.nq;
    const int g = idx / per_group;
    const int g0 = g * p.group;
    const int gsize = min(p.group, BH - g0);
    const int w = idx - g * per_group;
    const int r = w / gsize;
    const int bh = g0 + (w - r * gsize);
    Item it;
    it.qt = p.causal ? (p.nq - 1 - r) : r;
    it.b = bh / p.H;
    it.h = bh - it.b * p.H;
    // 64-key tiles: all of them, or (causal) those holding a key <= the
    // position of the tile's last query.
    it.n_kv = p.causal ? min((it.qt * BM + BM - 1 + p.kv_off) / BN + 1, p.nk) : p.nk;
    return it;
}

// Work items are published by the producer thread into a small ring in shared
// memory; every consumer warp reads the same sequence.  With a scheduler
// counter (p.sched != nullptr) each CTA claims its next item from a global
// counter when it needs one, so SMs that run slower simply take fewer items;
// without one, CTA c takes the static boustrophedon sequence.  -1 ends the
// sequence.
struct ItemRing {
    uint64_t* bars;
    volatile int* slots;
    const AbortState* ab;
    // consumer side, single thread (the MMA-issuing thread of its warp)
    __device__ __forceinline__ bool get_one(int k, int& idx) const {
        const int s = k % ITEM_RING;
        if (!mbar_wait(&bars[BAR_ITEM_FULL + s], (uint32_t)(k / ITEM_RING) & 1u, *ab)) return false;
        idx = slots[s];
        mbar_arrive(&bars[BAR_ITEM_EMPTY + s]);
        return true;
    }
    // consumer side, whole warp (all lanes call; lane 0 arrives for the warp)
    __device__ __forceinline__ bool get(int k, int& idx) const {
        const int s = k % ITEM_RING;
        if (!mbar_wait_warp(&bars[BAR_ITEM_FULL + s], (uint32_t)(k / ITEM_RING) & 1u, *ab)) return false;
        idx = slots[s];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&bars[BAR_ITEM_EMPTY + s]);
        return true;
    }
};

// Wait profile (only in a separate build of the library compiled with
// -DDIFFATTN_WAIT_PROFILE; the regular build has none of it): each role's
// issuing thread (lane 0 of each softmax warp) counts the SM cycles it spends
// in mbarrier waits, by what completes the barrier, and adds them to
// g_wait_prof[role][kind] when the CTA ends.  Roles: 0 the TMA producer, 1 the
// two MMA-issuing threads, 2 the eight softmax warps.  Kinds: 0 the role's
// cycles from start to end; waits on TMA loads: 1 Q full, 2 K full, 3 V full;
// waits on tensor-core work: 4 at an item's start (the first S full; the
// producer's Q slot released by the item's last score product), 5 within an
// item (later S full, PV done; K and V stages released by MMA commits), 6 the
// item's last products before the epilogue (O full); 7 waits on other warps
// (P full, O read out, the item ring, the epilogue's exchanges).  For the key
// tiles the MMA threads also record the lead of each wait, the cycles from the
// tile's TMA issue to the start of the wait (8: sum, 9: count), and for the
// waits longer than 64 cycles the cycles from issue to landing (10: sum, 11:
// count); and, right after each key-tile wait, the time of a second wait on the
// same (now complete) phase: the floor of a wait that finds its data there
// (12: sum).  Each CTA also stamps the global timer at its start and end
// (g_cta_span), which shows the spread of the CTAs' finishing times.  The
// softmax warps also time their work outside waits: an item's first tile (13),
// its other tiles (14), each from the score wait to the P hand-off, and the
// epilogue from the O wait to the output store (15); with the tile and item
// counts (16, 17); and the epilogue's steps: O read out of TMEM (18), the
// exchange of 1/l with the other warpgroup (19), the arithmetic (20), the
// wait for the staging buffer (21) and the staging writes with the store (22).
enum : int {
    kWaitTotal = 0, kWaitQ = 1, kWaitK = 2, kWaitV = 3, kWaitItemStart = 4, kWaitTensor = 5,
    kWaitEpilogue = 6, kWaitPeer = 7, kLeadSum = 8, kLeadCount = 9, kLateSum = 10,
    kLateCount = 11, kFloorSum = 12, kFirstTileBusy = 13, kTileBusy = 14, kEpilogueBusy = 15,
    kTileCount = 16, kItemCount = 17, kEpiLoad = 18, kEpiSync = 19, kEpiMath = 20,
    kEpiStageWait = 21, kEpiStore = 22, kWaitKinds = 23
};
#ifdef DIFFATTN_WAIT_PROFILE
constexpr int kSpanCtas = 1024;
__device__ unsigned long long g_wait_prof[3][kWaitKinds];
__device__ unsigned long long g_cta_span[kSpanCtas][2];
struct WaitProf {
    unsigned long long c[kWaitKinds] = {};
    long long t0 = 0;
    __device__ __forceinline__ void start() { t0 = clock64(); }
    template <class F>
    __device__ __forceinline__ bool timed(int kind, F&& f) {
        const long long a = clock64();
        const bool r = f();
        c[kind] += (unsigned long long)(clock64() - a);
        return r;
    }
    // a key-tile wait: its lead after the TMA issue stamped in `issued`
    template <class F>
    __device__ __forceinline__ bool key_wait(long long issued, F&& f) {
        const long long a = clock64();
        const bool r = f();
        const long long b = clock64();
        c[kWaitK] += (unsigned long long)(b - a);
        c[kLeadSum] += (unsigned long long)(a > issued ? a - issued : 0);
        c[kLeadCount] += 1;
        if (b - a > 64) {
            c[kLateSum] += (unsigned long long)(b - issued);
            c[kLateCount] += 1;
        }
        const long long f0 = clock64();
        f();                                   // the same phase again: complete
        c[kFloorSum] += (unsigned long long)(clock64() - f0);
        return r;
    }
    __device__ __forceinline__ void flush(int role, bool reporter) {
        c[kWaitTotal] = (unsigned long long)(clock64() - t0);
        if (reporter)
            for (int i = 0; i < kWaitKinds; ++i) atomicAdd(&g_wait_prof[role][i], c[i]);
    }
};
#define TIMED_WAIT(wp, kind, expr) (wp).timed((kind), [&]() -> bool { return (expr); })
#define KEY_WAIT(wp, stage, expr) (wp).key_wait(kissue[stage], [&]() -> bool { return (expr); })
#define STAMP_KEY_ISSUE(stage) (kissue[stage] = clock64())
#define PROF_MARK(var) const long long var = clock64()
#define PROF_ADD(wp, kind, since) ((wp).c[kind] += (unsigned long long)(clock64() - (since)))
#define PROF_COUNT(wp, kind) ((wp).c[kind] += 1)
#else
struct WaitProf {
    __device__ __forceinline__ void start() {}
    __device__ __forceinline__ void flush(int, bool) {}
};
#define TIMED_WAIT(wp, kind, expr) (expr)
#define KEY_WAIT(wp, stage, expr) (expr)
#define STAMP_KEY_ISSUE(stage) ((void)0)
#define PROF_MARK(var) ((void)0)
#define PROF_ADD(wp, kind, since) ((void)0)
#define PROF_COUNT(wp, kind) ((void)0)
#endif

// Row max of one thread's 64 scores (four independent chains of
// three-input maxima).
__device__ __forceinline__ float tile_row_max(const float (&s)[64]) {
    float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
    for (int c = 4; c < 60; c += 8) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
    }
    mx0 = fmax3(mx0, s[60], s[61]);
    mx1 = fmax3(mx1, s[62], s[63]);
    return fmax3(mx0, mx1, fmaxf(mx2, mx3));
}

// P = 2^(s * scale_log2 - m) for one thread's 64 scores, two columns per
// packed operation: P rounded to bf16 pairs into pk, and the sum of the
// unrounded P returned.
__device__ __forceinline__ float tile_exp2(const float (&s)[64], float sl2, float m, uint32_t (&pk)[32]) {
    const uint64_t scale2 = f2_pack(sl2, sl2);
    const uint64_t negm2 = f2_pack(-m, -m);
    uint64_t rsum[4] = {0, 0, 0, 0};     // four short addition chains
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const uint64_t x = f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), scale2, negm2);
        const float p0 = ex2_approx(f2_lo(x));
        const float p1 = ex2_approx(f2_hi(x));
        rsum[c & 3] = f2_add(rsum[c & 3], f2_pack(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
    }
    const uint64_t r = f2_add(f2_add(rsum[0], rsum[1]), f2_add(rsum[2], rsum[3]));
    return f2_lo(r) + f2_hi(r);
}

template <int HD>
__global__ void __launch_bounds__(NUM_THREADS, 1)
diffattn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q1,
                       const __grid_constant__ CUtensorMap tm_k1,
                       const __grid_constant__ CUtensorMap tm_q2,
                       const __grid_constant__ CUtensorMap tm_k2,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const TcParams p) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + REL_TMEM_PTR);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + REL_ABORT);
    float* inv_l = reinterpret_cast<float*>(smem + C::OFF_BAR + REL_INVL);
#ifdef DIFFATTN_WAIT_PROFILE
    __shared__ volatile long long kissue[KSTAGES];    // TMA issue time of each key stage
#endif
    const bool k_shared = p.k_shared != 0;
    const int kstages = C::kstages(k_shared);
    const uint32_t kstride = C::kstride(k_shared);

    const uint32_t warp = warp_id();
    const uint32_t lane = threadIdx.x & 31;
    const AbortState ab{abort_flag, p.status};
#ifdef DIFFATTN_WAIT_PROFILE
    if (threadIdx.x == 0 && blockIdx.x < kSpanCtas) g_cta_span[blockIdx.x][0] = globaltimer_ns();
#endif

    if (threadIdx.x == 0) {
        mbar_init(&bars[BAR_Q_FULL], 1);
        mbar_init(&bars[BAR_Q_EMPTY], 2);
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(&bars[BAR_K_FULL + s], 1);
            mbar_init(&bars[BAR_K_EMPTY + s], 2);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            mbar_init(&bars[BAR_V_FULL + s], 1);
            mbar_init(&bars[BAR_V_EMPTY + s], 2);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars[BAR_S_FULL + i], 1);
            mbar_init(&bars[BAR_P_FULL + i], 4);
        }
        mbar_init(&bars[BAR_PV_DONE + 0], 1);
        mbar_init(&bars[BAR_PV_DONE + 1], 1);
        mbar_init(&bars[BAR_O_FULL], 2);
        mbar_init(&bars[BAR_O_EMPTY], 8);
        mbar_init(&bars[BAR_L_READY], 8);
        mbar_init(&bars[BAR_FINAL + 0], 1);
        mbar_init(&bars[BAR_FINAL + 1], 1);
        for (int i = 0; i < ITEM_RING; ++i) {
            mbar_init(&bars[BAR_ITEM_FULL + i], 1);
            mbar_init(&bars[BAR_ITEM_EMPTY + i], NUM_ITEM_CONSUMERS);
        }
        mbar_init(&bars[BAR_NORM_A], 8);
        mbar_init(&bars[BAR_NORM_B], 8);
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

    const int grid = gridDim.x;
    const int cta = blockIdx.x;
    const ItemRing ring{bars, reinterpret_cast<volatile int*>(smem + C::OFF_BAR + REL_RING), &ab};

    if (warp >= 8) {
      regs_dec<REGS_OTHER>();
      if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (elect_one()) {
            tma_prefetch_desc(&tm_q1);
            tma_prefetch_desc(&tm_k1);
            tma_prefetch_desc(&tm_q2);
            tma_prefetch_desc(&tm_k2);
            tma_prefetch_desc(&tm_v);
            WaitProf wp;
            wp.start();
            uint32_t kst = 0, kph = 0, vst = 0, vph = 0, qph = 0;
            uint32_t armed_q = 0, armed_k[KSTAGES] = {}, armed_v[VSTAGES_MAX] = {};
            bool ok = true;
            bool first = true;
            // Item claimed for the current position of the sequence; the next
            // one is claimed once every load of this one has been issued (the
            // producer runs a ring ahead of the compute, so the claim's latency
            // stays hidden, and a CTA holds no claimed item it will not reach
            // soon: +0.5-0.7 % against claiming right after publishing).
            int sk = 0;    // static sequence position
            auto claim = [&]() -> int {
                if (p.sched) {
                    const int idx = (int)atomicAdd(p.sched, 1u);
                    return idx < p.total_items ? idx : -1;
                }
                for (; sk * grid < p.total_items; ++sk) {
                    const int idx = item_index(sk, cta, grid);
                    if (idx < p.total_items) { ++sk; return idx; }
                }
                return -1;
            };
            int idx = claim();
            for (int k = 0; ok; ++k) {
                // publish item k (or the end of the sequence) to the consumers
                const int slot = k % ITEM_RING;
                if (k >= ITEM_RING) {
                    if (!(ok = TIMED_WAIT(wp, kWaitPeer, mbar_wait(&bars[BAR_ITEM_EMPTY + slot],
                                                                   (uint32_t)(k / ITEM_RING - 1) & 1u, ab))))
                        break;
                }
                ring.slots[slot] = idx;
                mbar_arrive(&bars[BAR_ITEM_FULL + slot]);
                if (idx < 0) break;
                const Item it = decode_item(idx, p);
                if (!first) {
                    if (!(ok = TIMED_WAIT(wp, kWaitItemStart, mbar_wait(&bars[BAR_Q_EMPTY], qph, ab)))) break;
                    qph ^= 1;
                }
                first = false;
                mbar_arrive_expect_tx(&bars[BAR_Q_FULL], 2 * C::Q_BYTES);
#pragma unroll
                for (int pn = 0; pn < C::PANELS; ++pn) {
                    tma_load_4d(smem + C::OFF_Q1 + pn * Q_PANEL, &tm_q1, &bars[BAR_Q_FULL], pn * 64,
                                it.qt * BM, it.h, it.b);
                    tma_load_4d(smem + C::OFF_Q2 + pn * Q_PANEL, &tm_q2, &bars[BAR_Q_FULL], pn * 64,
                                it.qt * BM, it.h, it.b);
                }
                ++armed_q;
                const int hk = it.h / p.kv_group;     // key/value head of this query head
                for (int j = 0; j < it.n_kv; ++j) {
                    if (!(ok = TIMED_WAIT(wp, kWaitTensor, mbar_wait(&bars[BAR_K_EMPTY + kst], kph ^ 1, ab))))
                        break;
                    uint8_t* kdst = smem + C::OFF_K + kst * kstride;
                    // one key tile for both branches when they share their keys
                    mbar_arrive_expect_tx(&bars[BAR_K_FULL + kst], (k_shared ? 1 : 2) * C::K_BYTES);
#pragma unroll
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        tma_load_4d(kdst + pn * K_PANEL, &tm_k1, &bars[BAR_K_FULL + kst], pn * 64, j * BN,
                                    hk, it.b);
                        if (!k_shared)
                            tma_load_4d(kdst + C::K_BYTES + pn * K_PANEL, &tm_k2, &bars[BAR_K_FULL + kst],
                                        pn * 64, j * BN, hk, it.b);
                    }
                    STAMP_KEY_ISSUE(kst);
                    ++armed_k[kst];
                    if (++kst == (uint32_t)kstages) { kst = 0; kph ^= 1; }

                    if (!(ok = TIMED_WAIT(wp, kWaitTensor, mbar_wait(&bars[BAR_V_EMPTY + vst], vph ^ 1, ab))))
                        break;
                    uint8_t* vdst = smem + C::OFF_V + vst * V_BYTES;
                    mbar_arrive_expect_tx(&bars[BAR_V_FULL + vst], V_BYTES);
                    tma_load_4d(vdst, &tm_v, &bars[BAR_V_FULL + vst], 0, j * BN, hk, it.b);
                    tma_load_4d(vdst + V_HALF_BYTES, &tm_v, &bars[BAR_V_FULL + vst], 64, j * BN, hk, it.b);
                    ++armed_v[vst];
                    if (++vst == (uint32_t)C::VSTAGES) { vst = 0; vph ^= 1; }
                }
                idx = claim();
            }
            // Never leave a copy in flight into shared memory we are about to
            // give back: wait (bounded) for the last armed phase of every ring.
            const uint64_t lim = 200ull * 1000ull * 1000ull;
            if (armed_q) mbar_wait_teardown(&bars[BAR_Q_FULL], (armed_q - 1) & 1, lim);
            for (int s = 0; s < KSTAGES; ++s)
                if (armed_k[s]) mbar_wait_teardown(&bars[BAR_K_FULL + s], (armed_k[s] - 1) & 1, lim);
            for (int s = 0; s < C::VSTAGES; ++s)
                if (armed_v[s]) mbar_wait_teardown(&bars[BAR_V_FULL + s], (armed_v[s] - 1) & 1, lim);
            wp.flush(0, true);
        }
        __syncwarp();
      } else if (warp == 9 || warp == 10) {
        // ----------------------------------------- MMA issue, one warp per branch
        const int br = warp - 9;
        if (elect_one()) {
            // Descriptors for stage 0 and K-step 0; other stages and K-steps
            // differ only in the start-address field (address >> 4, which
            // stays below 2^14 for every shared-memory address).
            const uint64_t qdesc = sdesc_sw128(smem_u32(smem + (br ? C::OFF_Q2 : C::OFF_Q1)), 16, 1024);
            const uint64_t kdesc =
                sdesc_sw128(smem_u32(smem + C::OFF_K + (k_shared ? 0 : br) * C::K_BYTES), 16, 1024);
            const uint64_t vdesc = sdesc_sw128(smem_u32(smem + C::OFF_V), V_HALF_BYTES, 1024);
            const uint32_t d_o = tmem_base + TM_O + br * 128;
            WaitProf wp;
            wp.start();
            uint32_t kst = 0, kph = 0, vst = 0, vph = 0, qph = 0, oeph = 0;
            uint32_t pph = 0;     // bit buffer: phase of P_FULL[br][buffer]
            bool ok = true;

            // S_b = Q_b K_b^T: HD / 16 products of depth 16, four per 64-column
            // panel (a step of 32 bytes inside the swizzle span)
            auto issue_s = [&](uint32_t stage, int buf) {
                const uint32_t d = tmem_base + tm_s(br, buf);
                const uint64_t kd = kdesc + ((stage * kstride) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t pn = kk >> 2, ks = kk & 3;
                    mma_ss(d, qdesc + pn * (Q_PANEL >> 4) + 2 * ks, kd + pn * (K_PANEL >> 4) + 2 * ks,
                           IDESC_S, kk > 0);
                }
            };
            auto issue_pv = [&](uint32_t stage, int buf, bool acc) {
                const uint32_t pa = tmem_base + tm_s(br, buf);
                const uint64_t vd = vdesc + ((stage * V_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(d_o, pa + kk * 8, vd + 128 * kk, IDESC_PV, (acc || kk > 0) ? 1u : 0u);
            };

            bool first = true;
            for (int k = 0; ok; ++k) {
                int idx = -1;
                if (!(ok = TIMED_WAIT(wp, kWaitPeer, ring.get_one(k, idx))) || idx < 0) break;
                const Item it = decode_item(idx, p);
                const int n = it.n_kv;
                if (!(ok = TIMED_WAIT(wp, kWaitQ, mbar_wait(&bars[BAR_Q_FULL], qph, ab)))) break;
                qph ^= 1;
                // S_b(0), S_b(1) into buffers 0 and 1
                for (int t = 0; t < 2 && t < n; ++t) {
                    if (!(ok = KEY_WAIT(wp, kst, mbar_wait(&bars[BAR_K_FULL + kst], kph, ab)))) break;
                    tc_fence_after();
                    issue_s(kst, t);
                    mma_commit(&bars[BAR_S_FULL + 2 * br + t]);
                    mma_commit(&bars[BAR_K_EMPTY + kst]);
                    if (++kst == (uint32_t)kstages) { kst = 0; kph ^= 1; }
                }
                if (!ok) break;
                if (n <= 2) mma_commit(&bars[BAR_Q_EMPTY]);

                for (int j = 0; j < n; ++j) {
                    const int buf = j & 1;
                    // The tiles PV_b(j) and S_b(j+2) read were loaded long
                    // before P_b(j) is ready (the rings run far ahead), so
                    // their barriers are checked first: once P_b(j) arrives,
                    // both products issue with no other wait in between.
                    if (!(ok = TIMED_WAIT(wp, kWaitV, mbar_wait(&bars[BAR_V_FULL + vst], vph, ab)))) break;
                    if (j + 2 < n &&
                        !(ok = KEY_WAIT(wp, kst, mbar_wait(&bars[BAR_K_FULL + kst], kph, ab))))
                        break;
                    if (j == 0 && !first) {
                        if (!(ok = TIMED_WAIT(wp, kWaitPeer, mbar_wait(&bars[BAR_O_EMPTY], oeph, ab)))) break;
                        oeph ^= 1;
                    }
                    // O_b += P_b(j) V(j)
                    if (!(ok = TIMED_WAIT(wp, kWaitPeer,
                                          mbar_wait(&bars[BAR_P_FULL + 2 * br + buf], (pph >> buf) & 1u, ab))))
                        break;
                    pph ^= 1u << buf;
                    tc_fence_after();
                    issue_pv(vst, buf, j > 0);
                    mma_commit(&bars[BAR_PV_DONE + br]);
                    mma_commit(&bars[BAR_V_EMPTY + vst]);
                    if (++vst == (uint32_t)C::VSTAGES) { vst = 0; vph ^= 1; }
                    // S_b(j+2) into the buffer P_b(j) was just read from
                    if (j + 2 < n) {
                        issue_s(kst, buf);
                        mma_commit(&bars[BAR_S_FULL + 2 * br + buf]);
                        mma_commit(&bars[BAR_K_EMPTY + kst]);
                        if (++kst == (uint32_t)kstages) { kst = 0; kph ^= 1; }
                        if (j + 3 == n) mma_commit(&bars[BAR_Q_EMPTY]);
                    }
                }
                if (!ok) break;
                mma_commit(&bars[BAR_O_FULL]);
                first = false;
            }
            // Every MMA this thread issued must have finished before TMEM is freed.
            mma_commit(&bars[BAR_FINAL + br]);
            mbar_wait_teardown(&bars[BAR_FINAL + br], 0, 200ull * 1000ull * 1000ull);
            wp.flush(1, true);
        }
        __syncwarp();
      }
    } else {
        regs_inc<REGS_SOFTMAX>();
        // ------------------------------------------------- softmax + epilogue
        const int br = warp >> 2;            // branch
        const uint32_t quad = warp & 3;      // TMEM lane quadrant
        const int row = quad * 32 + lane;    // query row within the tile
        const uint32_t lane_base = tmem_base + ((quad * 32u) << 16);
        const uint32_t tO = lane_base + TM_O + br * 128;
        const float sl2 = p.scale_log2;
        const float lam = p.lambda_dev ? __ldg(p.lambda_dev) : p.lambda;
        uint32_t sph = 0;          // bit buf: phase of S_FULL[br][buf]
        uint32_t ofph = 0, lph = 0, naph = 0, nbph = 0;
        float* stat = reinterpret_cast<float*>(smem + C::OFF_BAR + REL_STAT);
        uint32_t pv_count = 0;     // PV_b products issued for earlier items
        bool ok = true;

        WaitProf wp;
        wp.start();
        int idx = -1;
        Item next{};
        ok = TIMED_WAIT(wp, kWaitPeer, ring.get(0, idx));
        if (ok && idx >= 0) next = decode_item(idx, p);
        for (int k = 0; ok && idx >= 0; ++k) {
            const Item it = next;
            const int q = it.qt * BM + row;
            float m_run = -INFINITY;
            float l = 0.f;

            for (int j = 0; j < it.n_kv; ++j) {
                const int buf = j & 1;
                const uint32_t tS = lane_base + tm_s(br, buf);
                if (!(ok = TIMED_WAIT(wp, j == 0 ? kWaitItemStart : kWaitTensor,
                                      mbar_wait_warp(&bars[BAR_S_FULL + 2 * br + buf], (sph >> buf) & 1u, ab))))
                    break;
                PROF_MARK(tile_t0);
                sph ^= 1u << buf;
                tc_fence_after();
                uint32_t u[64];
                tmem_ld32(tS + 0, &u[0]);
                tmem_ld32(tS + 32, &u[32]);
                tmem_wait_ld();
                float s[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);

                const int kv0 = j * BN;
                if (p.causal) {
                    if (kv0 + BN - 1 > it.qt * BM + p.kv_off) {   // the tile crosses the diagonal
                        const int lim = q + p.kv_off - kv0;        // keys kv0 + c with c > lim are in the future
#pragma unroll
                        for (int c = 0; c < 64; ++c) s[c] = (c > lim) ? -INFINITY : s[c];
                    }
                } else if (kv0 + BN > p.Tk) {
                    const int lim = p.Tk - kv0;           // keys at or beyond Tk do not exist
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = (c >= lim) ? -INFINITY : s[c];
                }
                // Lazy rescale: the running max moves only when a row's tile
                // max exceeds it by more than 8 (log2 units), i.e. when some
                // P of the row would exceed 2^8.  Such a row's tile sum then
                // exceeds 2^8 as well, so the exponentials are first taken
                // against the running max and the row max (a reduction on the
                // critical path) is formed only when some row's sum exceeds
                // 2^8; the decision equals the one the row max alone would
                // give.  The first tile of an item sets the running max.  The
                // decision is warp-uniform: the O rescale below is a
                // warp-collective TMEM access.
                float alpha = 1.0f;
                bool rescale = false;
                if (j == 0) m_run = tile_row_max(s) * sl2;
                uint32_t pk[32];
                float tsum = tile_exp2(s, sl2, m_run, pk);
                // P goes to TMEM at once; the sum check overlaps the store,
                // and a rescale (rare) stores the recomputed P over it.
                tmem_st32(tS, &pk[0]);
                if (j > 0 && __any_sync(0xffffffffu, !(tsum <= 256.0f))) {
                    const float mxs = tile_row_max(s) * sl2;
                    if (__any_sync(0xffffffffu, mxs > m_run + 8.0f)) {
                        const float m_new = fmaxf(m_run, mxs);
                        alpha = ex2_approx(m_run - m_new);
                        l *= alpha;
                        m_run = m_new;
                        rescale = true;
                        tsum = tile_exp2(s, sl2, m_run, pk);
                        tmem_wait_st();
                        tmem_st32(tS, &pk[0]);
                    }
                }
                if (rescale) {
                    // O_b row *= alpha, once PV_b(j-1) has completed (S_b(j)
                    // completing already implies PV_b(j-2) has).
                    if (!(ok = TIMED_WAIT(wp, kWaitTensor,
                                          mbar_wait_warp(&bars[BAR_PV_DONE + br], (pv_count + j - 1) & 1u, ab))))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(tO + c4 * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + c4 * 32, o);
                    }
                }
                tmem_wait_st();
                l += tsum;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_P_FULL + 2 * br + buf]);
                PROF_ADD(wp, j == 0 ? kFirstTileBusy : kTileBusy, tile_t0);
                PROF_COUNT(wp, kTileCount);
            }
            if (!ok) break;
            PROF_COUNT(wp, kItemCount);
            pv_count += it.n_kv;
            // The next item is fetched and decoded here, while the item's last
            // PV products complete, rather than after the epilogue.
            if (!(ok = TIMED_WAIT(wp, kWaitPeer, ring.get(k + 1, idx)))) break;
            if (idx >= 0) next = decode_item(idx, p);

            // ---------------------------------------------------- epilogue
            if (!(ok = TIMED_WAIT(wp, kWaitEpilogue, mbar_wait_warp(&bars[BAR_O_FULL], ofph, ab)))) break;
            PROF_MARK(epi_t0);
            ofph ^= 1;
            tc_fence_after();
            if (p.stats) {
                // Row statistics for the backward: this branch's log2-sum-exp
                // and Dd_b = dO . (O_b / l_b), 32 columns at a time.
                const bool live = q < p.T;
                const __nv_bfloat16* g = p.dout + it.b * p.do_sB + it.h * p.do_sH +
                                         (int64_t)(live ? q : 0) * p.do_sT;
                float dd = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o[32];
                    tmem_ld32(tO + c4 * 32, o);
                    uint4 gv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        gv[i] = live ? *reinterpret_cast<const uint4*>(g + c4 * 32 + 8 * i)
                                     : make_uint4(0, 0, 0, 0);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t w[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            dd = fmaf(__uint_as_float(o[8 * i + 2 * e]), __uint_as_float(w[e] << 16), dd);
                            dd = fmaf(__uint_as_float(o[8 * i + 2 * e + 1]),
                                      __uint_as_float(w[e] & 0xffff0000u), dd);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_O_EMPTY]);
                if (live) {
                    // stored negated: the consumers add them
                    float* st = p.stats + (((int64_t)it.b * p.H + it.h) * p.T + q) * 4;
                    st[br] = -(m_run + log2f(l));
                    st[2 + br] = -(dd / l);
                }
                continue;
            }
            inv_l[br * BM + row] = 1.0f / l;
            const int c0 = br * 64;          // this warpgroup writes output columns [c0, c0+64)
            uint32_t o1[64], o2[64];
            tmem_ld32(lane_base + TM_O + c0, &o1[0]);
            tmem_ld32(lane_base + TM_O + c0 + 32, &o1[32]);
            tmem_ld32(lane_base + TM_O + 128 + c0, &o2[0]);
            tmem_ld32(lane_base + TM_O + 128 + c0 + 32, &o2[32]);
            tmem_wait_ld();
            PROF_ADD(wp, kEpiLoad, epi_t0);
            PROF_MARK(sync_t0);
            // O is in registers: the next item's PV may overwrite TMEM.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[BAR_O_EMPTY]);
                mbar_arrive(&bars[BAR_L_READY]);
            }
            if (!(ok = TIMED_WAIT(wp, kWaitPeer, mbar_wait_warp(&bars[BAR_L_READY], lph, ab)))) break;
            lph ^= 1;
            PROF_ADD(wp, kEpiSync, sync_t0);
            PROF_MARK(math_t0);
            const float inv1 = inv_l[row];
            const float inv2 = inv_l[BM + row];
            if (p.out2 && q < p.T) {
                // training outputs: A_2 V for this thread's 64 columns, and this
                // branch's log-sum-exp (natural log) of the scaled scores
                __nv_bfloat16* o2row = p.out2 + it.b * p.o_sB + it.h * p.o_sH + (int64_t)q * p.o_sT + c0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 8 * i;
                    *reinterpret_cast<uint4*>(o2row + c) = make_uint4(
                        pack_bf16x2(__uint_as_float(o2[c]) * inv2, __uint_as_float(o2[c + 1]) * inv2),
                        pack_bf16x2(__uint_as_float(o2[c + 2]) * inv2, __uint_as_float(o2[c + 3]) * inv2),
                        pack_bf16x2(__uint_as_float(o2[c + 4]) * inv2, __uint_as_float(o2[c + 5]) * inv2),
                        pack_bf16x2(__uint_as_float(o2[c + 6]) * inv2, __uint_as_float(o2[c + 7]) * inv2));
                }
                p.lse[(((int64_t)it.b * p.H + it.h) * p.T + q) * 2 + br] =
                    (m_run + log2f(l)) * 0.6931471805599453f;
            }
            // O = O1 / l1 - lambda O2 / l2 for this thread's 64 columns: a = O1 / l1
            // and b = O2 / l2 rounded, then a - lambda b in one fused step
            // (identical branches at lambda = 1 give a = b, hence exactly 0)
            float r[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float a = __fmul_rn(__uint_as_float(o1[c]), inv1);
                const float bb = __fmul_rn(__uint_as_float(o2[c]), inv2);
                r[c] = __fmaf_rn(bb, -lam, a);
            }
            if (p.norm != kNormNone) {
                // Per-head normalisation over the row's 2D = 128 channels; the
                // two warpgroups hold 64 channels each and exchange partial
                // sums through shared memory.
                float part = 0.f;
                if (p.norm == kNormRms) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) part = fmaf(r[c], r[c], part);
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) part += r[c];
                }
                stat[br * BM + row] = part;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[BAR_NORM_A]);
                if (!(ok = TIMED_WAIT(wp, kWaitPeer, mbar_wait_warp(&bars[BAR_NORM_A], naph, ab)))) break;
                naph ^= 1;
                const float tot = stat[row] + stat[BM + row];
                float mu = 0.f, rinv;
                if (p.norm == kNormRms) {
                    rinv = rsqrtf(tot * (1.0f / VD) + p.norm_eps);
                } else {
                    mu = tot * (1.0f / VD);
                    float dev = 0.f;
#pragma unroll
                    for (int c = 0; c < 64; ++c) dev = fmaf(r[c] - mu, r[c] - mu, dev);
                    stat[2 * BM + br * BM + row] = dev;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[BAR_NORM_B]);
                    if (!(ok = TIMED_WAIT(wp, kWaitPeer, mbar_wait_warp(&bars[BAR_NORM_B], nbph, ab)))) break;
                    nbph ^= 1;
                    const float var = (stat[2 * BM + row] + stat[3 * BM + row]) * (1.0f / VD);
                    rinv = rsqrtf(var + p.norm_eps);
                }
                const float* wrow = p.norm_weight ? p.norm_weight + it.h * VD + c0 : nullptr;
                const float* brow = p.norm_bias ? p.norm_bias + it.h * VD + c0 : nullptr;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    float y = (r[c] - mu) * rinv;
                    if (wrow) y *= __ldg(wrow + c);
                    if (brow) y += __ldg(brow + c);
                    r[c] = y * p.out_scale;
                }
            } else if (p.out_scale != 1.0f) {
#pragma unroll
                for (int c = 0; c < 64; ++c) r[c] *= p.out_scale;
            }
            // Stage this warp's 32 rows x 64 columns in shared memory (128-byte
            // swizzled rows, as the output tensor map expects) and write them
            // with one TMA store; rows at or past T are clipped by the TMA unit.
            uint8_t* stage = smem + C::OFF_OUT + br * (OUT_BYTES / 2) + quad * 4096;
            PROF_ADD(wp, kEpiMath, math_t0);
            PROF_MARK(stage_t0);
            if (lane == 0) bulk_wait_read_all();     // the previous store has read the buffer
            __syncwarp();
            PROF_ADD(wp, kEpiStageWait, stage_t0);
            PROF_MARK(store_t0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = 8 * i;
                *reinterpret_cast<uint4*>(stage + lane * 128 + ((i ^ (lane & 7)) * 16)) =
                    make_uint4(pack_bf16x2(r[c], r[c + 1]), pack_bf16x2(r[c + 2], r[c + 3]),
                               pack_bf16x2(r[c + 4], r[c + 5]), pack_bf16x2(r[c + 6], r[c + 7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_4d(&tm_o, stage, c0, it.qt * BM + (int)quad * 32, it.h, it.b);
                bulk_commit();
            }
            PROF_ADD(wp, kEpiStore, store_t0);
            PROF_ADD(wp, kEpilogueBusy, epi_t0);
        }
        // Every output store must be complete before the CTA exits.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        wp.flush(2, lane == 0);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
#ifdef DIFFATTN_WAIT_PROFILE
    if (threadIdx.x == 0 && blockIdx.x < kSpanCtas) g_cta_span[blockIdx.x][1] = globaltimer_ns();
#endif
    if (warp == 9) tmem_dealloc(tmem_base, TMEM_COLS);
    // The last CTA to finish returns the scheduler counter to zero for the
    // next launch that uses it.
    if (p.sched && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

}  // namespace tc

namespace {
template <int HD>
int launch_hd(const CUtensorMap* maps, const TcParams& p, int grid, cudaStream_t stream) {
    constexpr uint32_t smem = tc::smem_bytes<HD>();
    cudaError_t e = cudaFuncSetAttribute(tc::diffattn_fwd_tc_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -1;
    tc::diffattn_fwd_tc_kernel<HD><<<grid, tc::NUM_THREADS, smem, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
}  // namespace

#ifdef DIFFATTN_WAIT_PROFILE
// The wait profile of the launches since the previous call ([3 roles][23
// kinds], see WaitProf), copied to `out` and cleared; then the start and end
// global-timer stamps of the last launch's CTAs ([1024][2], zero past the
// grid).  Only in the build with -DDIFFATTN_WAIT_PROFILE.
extern "C" int diffattn_wait_profile(unsigned long long* out, int n) {
    constexpr int kN = 3 * tc::kWaitKinds;
    constexpr int kS = 2 * tc::kSpanCtas;
    if (!out || n < kN + kS) return -1;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(out, tc::g_wait_prof, kN * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMemcpyFromSymbol(out + kN, tc::g_cta_span, kS * sizeof(unsigned long long)) != cudaSuccess)
        return -3;
    static unsigned long long zero[kN + kS] = {};
    return cudaMemcpyToSymbol(tc::g_wait_prof, zero, kN * sizeof(unsigned long long)) == cudaSuccess &&
                   cudaMemcpyToSymbol(tc::g_cta_span, zero, kS * sizeof(unsigned long long)) ==
                       cudaSuccess
               ? 0
               : -3;
}
#endif

int launch_fwd_tc(const CUtensorMap* maps, const TcParams& p, int head_dim, int grid,
                  cudaStream_t stream) {
    static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
    if (head_dim == 64) return launch_hd<64>(maps, p, grid, stream);
    if (head_dim == 128) return launch_hd<128>(maps, p, grid, stream);
    return -1;
}

}  // namespace diffattn
