// api.cu -- the C ABI declared in include/diffattn.h: argument checks, kernel
// selection, TMA tensor-map encoding and launches on the caller's stream.
#include "diffattn.h"
#include "kernels.h"

#include <cmath>
#include <cstdint>
#include <mutex>

namespace diffattn {

// The library's device status word (one per device, module scope).  Kernels
// OR status bits into it; diffattn_get_device_error reads and clears it.
__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
static_assert(DIFFATTN_NORM_NONE == kNormNone && DIFFATTN_NORM_RMS == kNormRms &&
                  DIFFATTN_NORM_GROUP == kNormGroup, "norm codes");
// Scheduler workspace: an item counter and a finished-CTA counter (2 words),
// rounded up to leave room.
constexpr size_t kWorkspaceBytes = 64;

struct DeviceState {
    bool ready = false;
    unsigned long long ctx = 0;   // ID of the context the addresses below belong to
    int num_sms = 0;
    uint32_t* status = nullptr;   // device address of g_status_word
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

// A unique identifier of the calling thread's current CUDA context (the
// driver's context ID, never reused within the process, so a context created
// again after a device reset gets a new one), 0 if there is no current context
// or the driver entry points cannot be found.
unsigned long long current_context() {
    using CtxGetCurrentFn = CUresult (*)(CUcontext*);
    using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static CtxGetCurrentFn get_current = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetCurrentFn>(nullptr);
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    static CtxGetIdFn get_id = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetIdFn>(nullptr);
        return reinterpret_cast<CtxGetIdFn>(f);
    }();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
        get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

namespace {

int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DIFFATTN_ERR_CUDA;
    const unsigned long long ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& st = g_devices[dev];
    // A device reset or another current context loads the library's module
    // again, possibly at other addresses: look them up again then.  (No
    // current context yet: the lookup below makes the primary one current.)
    if (!st.ready || ctx == 0 || st.ctx != ctx) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DIFFATTN_ERR_CUDA;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return DIFFATTN_ERR_CUDA;
        st.num_sms = sms;
        st.status = static_cast<uint32_t*>(addr);
        st.ctx = current_context();
        st.ready = true;
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return DIFFATTN_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = &st;
    return DIFFATTN_OK;
}

bool strides_nonneg(const int64_t s[3]) { return s[0] >= 0 && s[1] >= 0 && s[2] >= 0; }

// Query heads per key/value head: 0 and 1 both mean one each.
int64_t group_of(int32_t kv_group) { return kv_group > 1 ? kv_group : 1; }

// K1 and K2 are the same tensor (same base and the same strides on every
// dimension that is stepped).
bool same_tensor(const void* a, const int64_t sa[3], const void* b, const int64_t sb[3],
                 int64_t B, int64_t Hk, int64_t T) {
    return a == b && (B == 1 || sa[0] == sb[0]) && (Hk == 1 || sa[1] == sb[1]) &&
           (T == 1 || sa[2] == sb[2]);
}

// Value width of a descriptor: 0 means 2D (the operation's own shape).
int64_t value_width(int64_t Dv, int64_t D) { return Dv == 0 ? 2 * D : Dv; }

int validate(const diffattn_desc* d, const void* q1, const void* k1, const void* q2,
             const void* k2, const void* v, const void* out) {
    if (!d || !q1 || !k1 || !q2 || !k2 || !v || !out) return DIFFATTN_ERR_INVALID;
    if (d->B < 1 || d->H < 1 || d->T < 1 || d->D < 1 || d->D > 128) return DIFFATTN_ERR_INVALID;
    if (d->Dv < 0 || value_width(d->Dv, d->D) > 256) return DIFFATTN_ERR_INVALID;
    if (d->dtype != DIFFATTN_BF16 && d->dtype != DIFFATTN_F32) return DIFFATTN_ERR_INVALID;
    if (d->kv_group < 0 || d->H % group_of(d->kv_group) != 0) return DIFFATTN_ERR_INVALID;
    if (!strides_nonneg(d->q1_stride) || !strides_nonneg(d->k1_stride) ||
        !strides_nonneg(d->q2_stride) || !strides_nonneg(d->k2_stride) ||
        !strides_nonneg(d->v_stride) || !strides_nonneg(d->o_stride))
        return DIFFATTN_ERR_INVALID;
    // Index arithmetic limits of the kernels (int32 rows, tiles and items).
    if (d->T > INT32_MAX - 128 || d->B > INT32_MAX || d->H > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
    const int64_t nq = (d->T + 127) / 128;
    if (d->B * d->H > INT32_MAX / nq) return DIFFATTN_ERR_UNSUPPORTED;
    return DIFFATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Heads per scheduling group of the tensor-core forward, for L2 locality: the
// CTAs working at the same time share the K1, K2 and V of one group
// (kv_bytes per key and key/value head: 512 in bf16 at D = 64 -- K1 128, K2
// 128, V 256).
// Causal items have unequal lengths and run longest first within a group;
// groups of about 64 MiB of keys and values with at least four items per CTA
// keep both the L2 hit rate and the balance (at B2 H16 T8192 that is 16 heads
// and 1024 items, ~2% faster than one group of all heads; at B1 H16 T32768,
// 4 heads, ~3% faster).  Non-causal items are all equally long; their groups
// take at most ~48 MiB with an item for every SM.
int head_group(int64_t BH, int64_t Tk, int64_t kv_bytes, int nq, int causal, int num_sms) {
    const int64_t head_bytes = Tk * kv_bytes;
    const int64_t budget = causal ? (64ll << 20) : (48ll << 20);
    int64_t g = budget / (head_bytes > 0 ? head_bytes : 1);
    const int64_t min_g = causal ? (4ll * num_sms + nq - 1) / nq : ((int64_t)num_sms + nq - 1) / nq;
    if (g < min_g) g = min_g;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    return (int)g;
}

// A stride qualifies for the tensor-core path if its dimension has size 1
// (never stepped) or it is a positive multiple of 8 elements (16 bytes).
bool tc_stride_ok(int64_t stride, int64_t size) {
    return size == 1 || (stride > 0 && stride % 8 == 0 && stride < (int64_t(1) << 38));
}
bool tc_strides_ok(const int64_t s[3], int64_t B, int64_t heads, int64_t T) {
    return tc_stride_ok(s[0], B) && tc_stride_ok(s[1], heads) && tc_stride_ok(s[2], T);
}

// Shapes the tensor-core kernel takes: bf16, value width 128, Q/K width 64 (the
// operation's V = 2D) or 128 (the DIFF V2 head, V as wide as Q and K).
bool tc_shape(int32_t dtype, int64_t D, int64_t Dv) {
    return dtype == DIFFATTN_BF16 && Dv == 128 && (D == 64 || D == 128);
}

// The tensor-core kernel for Tq query rows over Tk keys (queries and the
// output with Tq rows, K1, K2 and V with Tk rows).
bool tc_ok(int32_t dtype, int64_t B, int64_t H, int64_t Hk, int64_t Tq, int64_t Tk, int64_t D,
           int64_t Dv, const int64_t* sq1, const int64_t* sk1, const int64_t* sq2,
           const int64_t* sk2, const int64_t* sv, const int64_t* so, const void* q1,
           const void* k1, const void* q2, const void* k2, const void* v, const void* out) {
    return tc_shape(dtype, D, Dv) && aligned16(q1) && aligned16(k1) && aligned16(q2) &&
           aligned16(k2) && aligned16(v) && aligned16(out) && tc_strides_ok(sq1, B, H, Tq) &&
           tc_strides_ok(sk1, B, Hk, Tk) && tc_strides_ok(sq2, B, H, Tq) &&
           tc_strides_ok(sk2, B, Hk, Tk) && tc_strides_ok(sv, B, Hk, Tk) &&
           tc_strides_ok(so, B, H, Tq);
}

int select(const diffattn_desc* d, const void* q1, const void* k1, const void* q2,
           const void* k2, const void* v, const void* out) {
    const int64_t hk = d->H / group_of(d->kv_group);
    return tc_ok(d->dtype, d->B, d->H, hk, d->T, d->T, d->D, value_width(d->Dv, d->D), d->q1_stride,
                 d->k1_stride, d->q2_stride, d->k2_stride, d->v_stride, d->o_stride, q1, k1, q2,
                 k2, v, out)
               ? DIFFATTN_KERNEL_TCGEN05
               : DIFFATTN_KERNEL_SIMT;
}

// 4-D bf16 tensor map {inner, T, heads, B} with a {box_inner, box_rows, 1, 1}
// box and 128-byte swizzling; rows past T read as zeros.
int encode_map_t(CUtensorMap* m, const void* base, int64_t inner, int64_t B, int64_t T,
                 int64_t heads, const int64_t s[3], uint32_t box_inner, uint32_t box_rows) {
    int64_t sT = s[2], sH = s[1], sB = s[0];
    // A size-1 dimension is never stepped; give it a stride the encoder accepts.
    if (T == 1) sT = inner;
    if (heads == 1) sH = sT * T;
    if (B == 1) sB = sH * heads;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)T, (cuuint64_t)heads,
                                (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)sT * 2, (cuuint64_t)sH * 2, (cuuint64_t)sB * 2};
    const cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

int encode_map(CUtensorMap* m, const void* base, int64_t inner, const diffattn_desc* d,
               int64_t heads, const int64_t s[3], uint32_t box_inner, uint32_t box_rows) {
    return encode_map_t(m, base, inner, d->B, d->T, heads, s, box_inner, box_rows);
}

void copy3(int64_t dst[3], const int64_t src[3]) {
    dst[0] = src[0];
    dst[1] = src[1];
    dst[2] = src[2];
}

// Checks of a decode descriptor that need no pointers; fills the key-range
// split plan.
struct DecodePlan {
    int tq_bucket = 0, splits = 0, split_len = 0;
    int kv_group = 1, Hk = 0, row_chunks = 0;
    size_t work_bytes = 0;
    // The queries go through the forward kernels instead (more query rows than
    // the split-key decode takes, or a value width other than 2D).
    bool forward = false;
    // The tensor-core split-key decode in units of up to 16 query rows, or the
    // forward kernels when the call's layout does not allow it: the DIFF V2
    // head (bf16, D = 128, value width 128, up to 16 queries; it needs one key
    // tensor for both branches), and bf16 D = 64 with more than 8 query rows
    // per key/value head (up to 16 queries).  Dense 16-byte aligned rows.
    bool tc_only = false;
    // For a tensor-core plan at D = 64: the split-key layout of up to 8-row
    // units that a call runs on the CUDA cores when its layout does not allow
    // the tensor-core pass (the workspace has room for both).
    bool fb_valid = false;
    int fb_tq_bucket = 0, fb_splits = 0, fb_split_len = 0, fb_row_chunks = 0;
};

// Query rows per unit of the tensor-core decode (1, 2, 4, 8 or 16).
int tc_bucket(int64_t rows) {
    for (int t = 1; t <= 16; t *= 2)
        if (rows <= t) return t;
    return 16;
}

// Bytes a call asks for when it runs on the forward kernels: none are used,
// but the workspace contract (a non-zero size for a valid request) holds.
constexpr size_t kForwardPathWorkBytes = 16;

// The split-key layout of a decode with up to `cap` rows per unit (the
// descriptor already checked; Tq <= cap, value width 2D).
int plan_split_key(const diffattn_kv_desc* d, int cap, DecodePlan* plan) {
    // The query rows of the heads that share a key/value head (g * Tq of
    // them) go in as few CTAs as the row capacity allows, evenly filled.
    const int64_t g = group_of(d->kv_group);
    const int64_t rows = g * d->Tq;
    const int64_t row_chunks = (rows + cap - 1) / cap;
    const int tqb = decode_tq_bucket((int)((rows + row_chunks - 1) / row_chunks), (int)d->D);
    if (tqb == 0) return DIFFATTN_ERR_UNSUPPORTED;
    const int64_t Hk = d->H / g;
    const int64_t units = d->B * Hk * row_chunks;
    if (units > (1ll << 24) || d->B * d->H > (1ll << 24)) return DIFFATTN_ERR_UNSUPPORTED;
    // The CUDA-core first passes split every unit's keys into ~4096 work
    // items for the whole call, with at least 256 keys (one chunk) per split:
    // their persistent grids then end at most one short item apart across
    // CTAs.  The tensor-core pass cuts the keys itself, at launch; for the
    // shapes it may take (four or eight rows, bf16, D = 64) the CUDA-core
    // layout, used only when it cannot run, keeps ~1024 items, so that the
    // workspace is about the size the tensor-core pass needs.
    const int64_t chunks = (d->Tk + 255) / 256;
    const int64_t target = (tqb >= 4 && d->dtype == DIFFATTN_BF16 && d->D == 64) ? 1024 : 4096;
    int64_t splits = (target + units - 1) / units;
    if (splits > chunks) splits = chunks;
    if (splits < 1) splits = 1;
    const int64_t split_len = ((chunks + splits - 1) / splits) * 256;
    splits = (d->Tk + split_len - 1) / split_len;
    if (units * splits > INT32_MAX || d->B * d->H * d->Tq > INT32_MAX) return DIFFATTN_ERR_UNSUPPORTED;
    plan->tq_bucket = tqb;
    plan->splits = (int)splits;
    plan->split_len = (int)split_len;
    plan->kv_group = (int)g;
    plan->Hk = (int)Hk;
    plan->row_chunks = (int)row_chunks;
    size_t floats = decode_work_floats(units, (int)splits, tqb, d->D);
    if (tqb >= 4 && d->dtype == DIFFATTN_BF16 && d->D == 64) {
        // the tensor-core pass cuts the keys its own way (contiguous tile
        // ranges per CTA); room for whichever first pass the call takes
        const size_t tc = decode_tc_work_floats(units, d->Tk, tqb);
        if (tc > floats) floats = tc;
    }
    plan->work_bytes = floats * sizeof(float);
    return DIFFATTN_OK;
}

int plan_decode(const diffattn_kv_desc* d, int causal, DecodePlan* plan) {
    if (!d) return DIFFATTN_ERR_INVALID;
    if (d->B < 1 || d->H < 1 || d->Tq < 1 || d->Tk < 1 || d->D < 1) return DIFFATTN_ERR_INVALID;
    if (d->dtype != DIFFATTN_BF16 && d->dtype != DIFFATTN_F32) return DIFFATTN_ERR_INVALID;
    if (d->kv_group < 0 || d->H % group_of(d->kv_group) != 0) return DIFFATTN_ERR_INVALID;
    if (d->Dv < 0 || d->D > 128 || value_width(d->Dv, d->D) > 256) return DIFFATTN_ERR_INVALID;
    if (!strides_nonneg(d->q1_stride) || !strides_nonneg(d->k1_stride) ||
        !strides_nonneg(d->q2_stride) || !strides_nonneg(d->k2_stride) ||
        !strides_nonneg(d->v_stride) || !strides_nonneg(d->o_stride))
        return DIFFATTN_ERR_INVALID;
    if (causal && d->Tk < d->Tq) return DIFFATTN_ERR_INVALID;
    if (d->Tk > INT32_MAX / 2 || d->Tq > INT32_MAX / 2 || d->H > (1 << 24))
        return DIFFATTN_ERR_UNSUPPORTED;
    const int cap = (d->D == 32 || d->D == 64 || d->D == 128) ? decode_max_rows((int)d->D) : 0;
    const bool bf16_vw128 = d->dtype == DIFFATTN_BF16 && value_width(d->Dv, d->D) == 128;
    const int64_t rows_per_kv = group_of(d->kv_group) * d->Tq;
    if (bf16_vw128 && d->Tq <= 16 && (d->D == 128 || (d->D == 64 && rows_per_kv > 8))) {
        // rows of the heads that share a key/value head, 16 per unit at most,
        // evenly filled
        const int64_t g = group_of(d->kv_group);
        const int64_t rows = rows_per_kv;
        const int64_t row_chunks = (rows + 15) / 16;
        const int64_t Hk = d->H / g;
        const int64_t units = d->B * Hk * row_chunks;
        if (units > (1ll << 24) || d->B * d->H > (1ll << 24) || d->B * d->H * d->Tq > INT32_MAX)
            return DIFFATTN_ERR_UNSUPPORTED;
        plan->tc_only = true;
        plan->tq_bucket = tc_bucket((rows + row_chunks - 1) / row_chunks);
        plan->splits = 1;                   // the tensor-core pass sets its own
        plan->split_len = (int)(((d->Tk + 255) / 256) * 256);
        plan->kv_group = (int)g;
        plan->Hk = (int)Hk;
        plan->row_chunks = (int)row_chunks;
        plan->work_bytes = decode_tc_work_floats(units, d->Tk, plan->tq_bucket) * sizeof(float);
        if (d->D == 64 && d->Tq <= cap) {
            DecodePlan fb;
            const int rc = plan_split_key(d, cap, &fb);
            if (rc != DIFFATTN_OK) return rc;
            plan->fb_valid = true;
            plan->fb_tq_bucket = fb.tq_bucket;
            plan->fb_splits = fb.splits;
            plan->fb_split_len = fb.split_len;
            plan->fb_row_chunks = fb.row_chunks;
            if (fb.work_bytes > plan->work_bytes) plan->work_bytes = fb.work_bytes;
        }
        return DIFFATTN_OK;
    }
    if (d->Tq > cap || value_width(d->Dv, d->D) != 2 * d->D) {
        // queries over the cache on the forward kernels (chunked prefill)
        const int64_t nq = (d->Tq + 127) / 128;
        if (d->B * d->H > INT32_MAX / nq) return DIFFATTN_ERR_UNSUPPORTED;
        plan->forward = true;
        plan->kv_group = (int)group_of(d->kv_group);
        plan->Hk = (int)(d->H / plan->kv_group);
        plan->work_bytes = kForwardPathWorkBytes;
        return DIFFATTN_OK;
    }
    return plan_split_key(d, cap, plan);
}

bool kv_aligned(const void* p, const int64_t s[3], size_t esize) {
    return aligned16(p) && (s[0] * (int64_t)esize) % 16 == 0 && (s[1] * (int64_t)esize) % 16 == 0 &&
           (s[2] * (int64_t)esize) % 16 == 0;
}

int forward_impl(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                 const diffattn_epilogue* epi, void* out, void* out2, float* lse,
                 void* workspace, size_t workspace_bytes, diffattn_stream_t stream);
int backward_impl(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                  const void* k2, const void* v, float lambda, const float* lambda_dev,
                  int causal, const void* out, const void* out2, const float* lse,
                  const void* dout, void* dq1, void* dk1, void* dq2, void* dk2, void* dv,
                  float* dlambda, void* workspace, size_t workspace_bytes,
                  diffattn_stream_t stream);

}  // namespace
}  // namespace diffattn

using namespace diffattn;

extern "C" {

int diffattn_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                    int64_t n, double lambda_init, float* lambda_out, diffattn_stream_t stream) {
    if (!lq1 || !lk1 || !lq2 || !lk2 || !lambda_out || n < 1 || !std::isfinite(lambda_init))
        return DIFFATTN_ERR_INVALID;
    return launch_lambda(lq1, lk1, lq2, lk2, n, lambda_init, lambda_out,
                         reinterpret_cast<cudaStream_t>(stream)) == 0
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

int diffattn_lambda_backward(const float* lq1, const float* lk1, const float* lq2,
                             const float* lk2, int64_t n, const float* dlambda, float* dlq1,
                             float* dlk1, float* dlq2, float* dlk2, diffattn_stream_t stream) {
    if (!lq1 || !lk1 || !lq2 || !lk2 || !dlambda || !dlq1 || !dlk1 || !dlq2 || !dlk2 || n < 1)
        return DIFFATTN_ERR_INVALID;
    return launch_lambda_bwd(lq1, lk1, lq2, lk2, n, dlambda, dlq1, dlk1, dlq2, dlk2,
                             reinterpret_cast<cudaStream_t>(stream)) == 0
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

int diffattn_select_kernel(const diffattn_desc* desc, const void* q1, const void* k1,
                           const void* q2, const void* k2, const void* v, const void* out) {
    const int rc = validate(desc, q1, k1, q2, k2, v, out);
    if (rc != DIFFATTN_OK) return rc;
    return select(desc, q1, k1, q2, k2, v, out);
}

size_t diffattn_workspace_bytes(void) { return kWorkspaceBytes; }

int diffattn_fwd(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev,
                 int causal, void* out, void* workspace, size_t workspace_bytes,
                 diffattn_stream_t stream) {
    return diffattn_fwd_ex(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, nullptr, out,
                           workspace, workspace_bytes, stream);
}

int diffattn_fwd_ex(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                    const void* k2, const void* v, float lambda, const float* lambda_dev,
                    int causal, const diffattn_epilogue* epi, void* out, void* workspace,
                    size_t workspace_bytes, diffattn_stream_t stream) {
    return forward_impl(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out, nullptr,
                        nullptr, workspace, workspace_bytes, stream);
}

int diffattn_fwd_train(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                       const void* k2, const void* v, float lambda, const float* lambda_dev,
                       int causal, void* out, void* out2, float* lse, void* workspace,
                       size_t workspace_bytes, diffattn_stream_t stream) {
    if (!out2 || !lse) return DIFFATTN_ERR_INVALID;
    return forward_impl(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, nullptr, out, out2,
                        lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace diffattn {
namespace {

// Shape and layout of one forward launch: Tq query rows over Tk keys, query
// row i at key position i + kv_off (causal mask: keys j > i + kv_off hidden).
struct FwdShape {
    int64_t B, H, Hk, Tq, Tk, D, Dv, kv_off;
    int32_t dtype;
    const int64_t *sq1, *sk1, *sq2, *sk2, *sv, *so;
};

int check_epilogue(const diffattn_epilogue* epi, diffattn_epilogue* e) {
    *e = diffattn_epilogue{DIFFATTN_NORM_NONE, 0.f, nullptr, nullptr, 1.0f, 0};
    if (!epi) return DIFFATTN_OK;
    *e = *epi;
    if (e->reserved != 0 || e->norm < DIFFATTN_NORM_NONE || e->norm > DIFFATTN_NORM_GROUP ||
        !std::isfinite(e->out_scale) ||
        (e->norm != DIFFATTN_NORM_NONE && !(std::isfinite(e->eps) && e->eps > 0.f)))
        return DIFFATTN_ERR_INVALID;
    return DIFFATTN_OK;
}

// One forward launch (arguments already checked): the tensor-core kernel when
// the shape, pointers and strides allow it, else the CUDA-core kernel.
int launch_forward(const FwdShape& f, const void* q1, const void* k1, const void* q2,
                   const void* k2, const void* v, float lambda, const float* lambda_dev,
                   int causal, const diffattn_epilogue& e, void* out, void* out2, float* lse,
                   void* workspace, cudaStream_t st) {
    DeviceState* dev = nullptr;
    int rc = device_state(&dev);
    if (rc != DIFFATTN_OK) return rc;
    const int64_t g = f.H / f.Hk;
    if (tc_ok(f.dtype, f.B, f.H, f.Hk, f.Tq, f.Tk, f.D, f.Dv, f.sq1, f.sk1, f.sq2, f.sk2, f.sv, f.so,
              q1, k1, q2, k2, v, out) &&
        (!out2 || aligned16(out2))) {
        CUtensorMap maps[6];
        // Q tiles are 128 query rows; K and V tiles are 64 key rows; every box
        // is 64 elements (128 bytes) wide, the 128-byte swizzle span (Q and K
        // rows of width 128 take two boxes).  O is stored by each warp in
        // 32-row x 64-column boxes.  K1, K2 and V have H / kv_group heads.
        if (encode_map_t(&maps[0], q1, f.D, f.B, f.Tq, f.H, f.sq1, 64, 128) != DIFFATTN_OK ||
            encode_map_t(&maps[1], k1, f.D, f.B, f.Tk, f.Hk, f.sk1, 64, 64) != DIFFATTN_OK ||
            encode_map_t(&maps[2], q2, f.D, f.B, f.Tq, f.H, f.sq2, 64, 128) != DIFFATTN_OK ||
            encode_map_t(&maps[3], k2, f.D, f.B, f.Tk, f.Hk, f.sk2, 64, 64) != DIFFATTN_OK ||
            encode_map_t(&maps[4], v, 128, f.B, f.Tk, f.Hk, f.sv, 64, 64) != DIFFATTN_OK ||
            encode_map_t(&maps[5], out, 128, f.B, f.Tq, f.H, f.so, 64, 32) != DIFFATTN_OK)
            return DIFFATTN_ERR_CUDA;
        const bool k_shared = same_tensor(k1, f.sk1, k2, f.sk2, f.B, f.Hk, f.Tk);
        TcParams p{};
        p.B = (int)f.B;
        p.H = (int)f.H;
        p.T = (int)f.Tq;
        p.Tk = (int)f.Tk;
        p.kv_off = causal ? (int)f.kv_off : 0;
        p.nq = (int)((f.Tq + 127) / 128);
        p.nk = (int)((f.Tk + 63) / 64);
        p.total_items = (int)(f.B * f.H * p.nq);
        // key/value bytes per key and key/value head, for the L2 grouping
        const int64_t kv_bytes = ((k_shared ? 1 : 2) * f.D + f.Dv) * 2;
        p.group = head_group(f.B * f.H, f.Tk, kv_bytes, p.nq, causal, dev->num_sms);
        p.causal = causal ? 1 : 0;
        p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)f.D));
        p.lambda = lambda;
        p.lambda_dev = lambda_dev;
        p.out = static_cast<__nv_bfloat16*>(out);
        p.o_sB = f.so[0];
        p.o_sH = f.so[1];
        p.o_sT = f.so[2];
        p.status = dev->status;
        p.sched = static_cast<uint32_t*>(workspace);
        p.norm = e.norm;
        p.norm_eps = e.eps;
        p.norm_weight = e.weight;
        p.norm_bias = e.bias;
        p.out_scale = e.out_scale;
        p.kv_group = (int)g;
        p.k_shared = k_shared ? 1 : 0;
        p.out2 = static_cast<__nv_bfloat16*>(out2);
        p.lse = lse;
        const int grid = p.total_items < dev->num_sms ? p.total_items : dev->num_sms;
        return launch_fwd_tc(maps, p, (int)f.D, grid, st) == 0 ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
    }

    SimtParams p{};
    p.B = (int)f.B;
    p.H = (int)f.H;
    p.T = (int)f.Tq;
    p.D = (int)f.D;
    p.Tk = (int)f.Tk;
    p.kv_off = causal ? (int)f.kv_off : 0;
    p.Dv = (int)f.Dv;
    p.causal = causal ? 1 : 0;
    p.scale = (float)(1.0 / std::sqrt((double)f.D));
    p.lambda = lambda;
    p.lambda_dev = lambda_dev;
    p.q1 = q1;
    p.k1 = k1;
    p.q2 = q2;
    p.k2 = k2;
    p.v = v;
    p.out = out;
    copy3(p.s_q1, f.sq1);
    copy3(p.s_k1, f.sk1);
    copy3(p.s_q2, f.sq2);
    copy3(p.s_k2, f.sk2);
    copy3(p.s_v, f.sv);
    copy3(p.s_o, f.so);
    p.norm = e.norm;
    p.norm_eps = e.eps;
    p.norm_weight = e.weight;
    p.norm_bias = e.bias;
    p.out_scale = e.out_scale;
    p.kv_group = (int)g;
    p.out2 = out2;
    p.lse = lse;
    rc = (f.dtype == DIFFATTN_F32) ? launch_fwd_simt_f32(p, st) : launch_fwd_simt_bf16(p, st);
    return rc == 0 ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

// The forward, optionally with the training outputs (out2 = A_2 V with the
// output's strides, lse = [B, H, T, 2] natural-log log-sum-exp per branch).
int forward_impl(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                 const diffattn_epilogue* epi, void* out, void* out2, float* lse,
                 void* workspace, size_t workspace_bytes, diffattn_stream_t stream) {
    int rc = validate(desc, q1, k1, q2, k2, v, out);
    if (rc != DIFFATTN_OK) return rc;
    diffattn_epilogue e;
    rc = check_epilogue(epi, &e);
    if (rc != DIFFATTN_OK) return rc;
    if (!lambda_dev && !std::isfinite(lambda)) return DIFFATTN_ERR_INVALID;
    if (workspace && (workspace_bytes < kWorkspaceBytes ||
                      (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0))
        return DIFFATTN_ERR_INVALID;
    const diffattn_desc& d = *desc;
    const FwdShape f{d.B, d.H, d.H / group_of(d.kv_group), d.T, d.T, d.D, value_width(d.Dv, d.D), 0,
                     d.dtype, d.q1_stride, d.k1_stride, d.q2_stride, d.k2_stride, d.v_stride,
                     d.o_stride};
    return launch_forward(f, q1, k1, q2, k2, v, lambda, lambda_dev, causal, e, out, out2, lse,
                          workspace, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace diffattn

extern "C" {

size_t diffattn_bwd_workspace_bytes(const diffattn_desc* desc) {
    if (!desc || desc->B < 1 || desc->H < 1 || desc->T < 1) return 0;
    // row statistics (4 floats per query row), then 128 floats of partial sums
    return (size_t)desc->B * desc->H * desc->T * 4 * sizeof(float) + 128 * sizeof(float);
}

int diffattn_bwd(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                 const void* dout, void* dq1, void* dk1, void* dq2, void* dk2, void* dv,
                 float* dlambda, void* workspace, size_t workspace_bytes,
                 diffattn_stream_t stream) {
    return backward_impl(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, nullptr, nullptr,
                         nullptr, dout, dq1, dk1, dq2, dk2, dv, dlambda, workspace,
                         workspace_bytes, stream);
}

int diffattn_bwd_saved(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                       const void* k2, const void* v, float lambda, const float* lambda_dev,
                       int causal, const void* out, const void* out2, const float* lse,
                       const void* dout, void* dq1, void* dk1, void* dq2, void* dk2, void* dv,
                       float* dlambda, void* workspace, size_t workspace_bytes,
                       diffattn_stream_t stream) {
    if (!out || !out2 || !lse) return DIFFATTN_ERR_INVALID;
    return backward_impl(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, out, out2, lse,
                         dout, dq1, dk1, dq2, dk2, dv, dlambda, workspace, workspace_bytes,
                         stream);
}

}  // extern "C"

namespace diffattn {
namespace {

// The backward.  With the forward's saved results (out, out2 = A_2 V and the
// log-sum-exp, all non-NULL) the row statistics come from one elementwise
// pass over them; without, from a recomputation of the forward.
int backward_impl(const diffattn_desc* desc, const void* q1, const void* k1, const void* q2,
                  const void* k2, const void* v, float lambda, const float* lambda_dev,
                  int causal, const void* out, const void* out2, const float* lse,
                  const void* dout, void* dq1, void* dk1, void* dq2, void* dk2, void* dv,
                  float* dlambda, void* workspace, size_t workspace_bytes,
                  diffattn_stream_t stream) {
    const bool saved = out != nullptr;
    int rc = validate(desc, q1, k1, q2, k2, v, dout);
    if (rc != DIFFATTN_OK) return rc;
    const int64_t dv_width = value_width(desc->Dv, desc->D);
    if (!dq1 || !dk1 || !dq2 || !dk2 || !dv || !dlambda) return DIFFATTN_ERR_INVALID;
    if (!lambda_dev && !std::isfinite(lambda)) return DIFFATTN_ERR_INVALID;
    const size_t need = diffattn_bwd_workspace_bytes(desc);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return DIFFATTN_ERR_INVALID;
    const diffattn_desc& d = *desc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the tensor-core backward takes the operation's own shape at D = 64
    if (d.D == 64 && dv_width == 128 && select(desc, q1, k1, q2, k2, v, dout) == DIFFATTN_KERNEL_TCGEN05 && aligned16(dq1) &&
        aligned16(dk1) && aligned16(dq2) && aligned16(dk2) && aligned16(dv)) {
        DeviceState* dev = nullptr;
        rc = device_state(&dev);
        if (rc != DIFFATTN_OK) return rc;
        const int64_t g = group_of(d.kv_group);
        const int64_t hk = d.H / g;
        float* stats = static_cast<float*>(workspace);
        if (saved) {
            // Pass 1: the row statistics from the forward's saved results.
            PrepParams pp{};
            pp.B = (int)d.B;
            pp.H = (int)d.H;
            pp.T = (int)d.T;
            pp.Dv = (int)(2 * d.D);
            pp.bf16 = 1;
            pp.log2_negated = 1;
            pp.lambda = lambda;
            pp.lambda_dev = lambda_dev;
            pp.out = out;
            pp.out2 = out2;
            pp.dout = dout;
            copy3(pp.s_o, d.o_stride);
            pp.lse = lse;
            pp.stats = stats;
            if (launch_bwd_prep(pp, st) != 0) return DIFFATTN_ERR_CUDA;
        } else {
        // Pass 1: the forward kernel in row-statistics mode.
        CUtensorMap fmaps[6];
        if (encode_map(&fmaps[0], q1, 64, &d, d.H, d.q1_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&fmaps[1], k1, 64, &d, hk, d.k1_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&fmaps[2], q2, 64, &d, d.H, d.q2_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&fmaps[3], k2, 64, &d, hk, d.k2_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&fmaps[4], v, 128, &d, hk, d.v_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&fmaps[5], dout, 128, &d, d.H, d.o_stride, 64, 32) != DIFFATTN_OK)
            return DIFFATTN_ERR_CUDA;
        TcParams f{};
        f.B = (int)d.B;
        f.H = (int)d.H;
        f.T = (int)d.T;
        f.Tk = (int)d.T;
        f.kv_off = 0;
        f.nq = (int)((d.T + 127) / 128);
        f.nk = (int)((d.T + 63) / 64);
        f.total_items = (int)(d.B * d.H * f.nq);
        f.group = head_group(d.B * d.H, d.T, 512, f.nq, causal, dev->num_sms);
        f.causal = causal ? 1 : 0;
        f.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.D));
        f.lambda = 0.f;
        f.lambda_dev = nullptr;
        f.out = nullptr;
        f.o_sB = f.o_sH = f.o_sT = 0;
        f.status = dev->status;
        f.sched = nullptr;
        f.norm = kNormNone;
        f.norm_eps = 0.f;
        f.norm_weight = f.norm_bias = nullptr;
        f.out_scale = 1.0f;
        f.kv_group = (int)g;
        f.k_shared = same_tensor(k1, d.k1_stride, k2, d.k2_stride, d.B, hk, d.T) ? 1 : 0;
        f.stats = static_cast<float*>(workspace);
        f.dout = static_cast<const __nv_bfloat16*>(dout);
        f.do_sB = d.o_stride[0];
        f.do_sH = d.o_stride[1];
        f.do_sT = d.o_stride[2];
        const int fgrid = f.total_items < dev->num_sms ? f.total_items : dev->num_sms;
        if (launch_fwd_tc(fmaps, f, 64, fgrid, st) != 0) return DIFFATTN_ERR_CUDA;
        }
        // Pass 2: dQ, then dK and dV, on the tensor cores.
        CUtensorMap maps[12];
        if (encode_map(&maps[0], q1, 64, &d, d.H, d.q1_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[1], k1, 64, &d, hk, d.k1_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&maps[2], q2, 64, &d, d.H, d.q2_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[3], k2, 64, &d, hk, d.k2_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&maps[4], v, 128, &d, hk, d.v_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&maps[5], dout, 128, &d, d.H, d.o_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[6], q1, 64, &d, d.H, d.q1_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&maps[7], k1, 64, &d, hk, d.k1_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[8], q2, 64, &d, d.H, d.q2_stride, 64, 64) != DIFFATTN_OK ||
            encode_map(&maps[9], k2, 64, &d, hk, d.k2_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[10], v, 128, &d, hk, d.v_stride, 64, 128) != DIFFATTN_OK ||
            encode_map(&maps[11], dout, 128, &d, d.H, d.o_stride, 64, 64) != DIFFATTN_OK)
            return DIFFATTN_ERR_CUDA;
        BwdTcParams b{};
        b.B = (int)d.B;
        b.H = (int)d.H;
        b.Hk = (int)hk;
        b.kv_group = (int)g;
        b.T = (int)d.T;
        b.nq128 = (int)((d.T + 127) / 128);
        b.nk64 = (int)((d.T + 63) / 64);
        b.nk128 = (int)((d.T + 127) / 128);
        b.causal = causal ? 1 : 0;
        b.scale = (float)(1.0 / std::sqrt((double)d.D));
        b.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.D));
        b.lambda = lambda;
        b.lambda_dev = lambda_dev;
        b.status = dev->status;
        b.stats = stats;
        b.dq1 = dq1;
        b.dq2 = dq2;
        b.dk1 = dk1;
        b.dk2 = dk2;
        b.dv = dv;
        if (launch_bwd_tc(maps, b, dev->num_sms, st) != 0) return DIFFATTN_ERR_CUDA;
        // the statistics hold -Dd_2, so dlambda = -sum(Dd_2) is their plain sum
        return launch_bwd_dlambda(stats, d.B * d.H * d.T, 1.0f, dlambda, st) == 0
                   ? DIFFATTN_OK
                   : DIFFATTN_ERR_CUDA;
    }
    BwdParams p{};
    p.B = (int)d.B;
    p.H = (int)d.H;
    p.kv_group = (int)group_of(d.kv_group);
    p.Hk = (int)(d.H / p.kv_group);
    p.T = (int)d.T;
    p.D = (int)d.D;
    p.Dv = (int)dv_width;
    p.causal = causal ? 1 : 0;
    p.scale = (float)(1.0 / std::sqrt((double)d.D));
    p.lambda = lambda;
    p.lambda_dev = lambda_dev;
    p.q1 = q1;
    p.k1 = k1;
    p.q2 = q2;
    p.k2 = k2;
    p.v = v;
    p.dout = dout;
    p.dq1 = dq1;
    p.dk1 = dk1;
    p.dq2 = dq2;
    p.dk2 = dk2;
    p.dv = dv;
    copy3(p.s_q1, d.q1_stride);
    copy3(p.s_k1, d.k1_stride);
    copy3(p.s_q2, d.q2_stride);
    copy3(p.s_k2, d.k2_stride);
    copy3(p.s_v, d.v_stride);
    copy3(p.s_do, d.o_stride);
    p.stats = static_cast<float*>(workspace);
    p.dlambda = dlambda;
    if (saved) {
        PrepParams pp{};
        pp.B = (int)d.B;
        pp.H = (int)d.H;
        pp.T = (int)d.T;
        pp.Dv = (int)dv_width;
        pp.bf16 = d.dtype == DIFFATTN_BF16 ? 1 : 0;
        pp.log2_negated = 0;
        pp.lambda = lambda;
        pp.lambda_dev = lambda_dev;
        pp.out = out;
        pp.out2 = out2;
        pp.dout = dout;
        copy3(pp.s_o, d.o_stride);
        pp.lse = lse;
        pp.stats = p.stats;
        if (launch_bwd_prep(pp, st) != 0) return DIFFATTN_ERR_CUDA;
        rc = (d.dtype == DIFFATTN_F32) ? launch_bwd_simt_grads_f32(p, st)
                                       : launch_bwd_simt_grads_bf16(p, st);
    } else {
        rc = (d.dtype == DIFFATTN_F32) ? launch_bwd_simt_f32(p, st) : launch_bwd_simt_bf16(p, st);
    }
    return rc == 0 ? DIFFATTN_OK : DIFFATTN_ERR_CUDA;
}

}  // namespace
}  // namespace diffattn

extern "C" {



size_t diffattn_decode_workspace_bytes(const diffattn_kv_desc* desc) {
    DecodePlan plan;
    // The plan does not depend on the mask; check the shape with it off.
    if (plan_decode(desc, 0, &plan) != DIFFATTN_OK) return 0;
    return plan.work_bytes;
}

}  // extern "C"

namespace diffattn {
namespace {

// Every check of a decode call except those of its workspace: pointers, the
// descriptor (and the split plan it gives), lambda, the epilogue and the
// alignment of the cache.
int decode_args(const diffattn_kv_desc* desc, const void* q1, const void* k1, const void* q2,
                const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                const diffattn_epilogue* epi, const void* out, DecodePlan* plan,
                diffattn_epilogue* e) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !out) return DIFFATTN_ERR_INVALID;
    int rc = plan_decode(desc, causal, plan);
    if (rc != DIFFATTN_OK) return rc;
    if (!lambda_dev && !std::isfinite(lambda)) return DIFFATTN_ERR_INVALID;
    rc = check_epilogue(epi, e);
    if (rc != DIFFATTN_OK) return rc;
    // the forward kernels take any alignment (and so does the tensor-core
    // decode of up to 16 rows, which falls back to them)
    if (plan->forward || plan->tc_only) return DIFFATTN_OK;
    const size_t esize = desc->dtype == DIFFATTN_BF16 ? 2 : 4;
    if (!kv_aligned(k1, desc->k1_stride, esize) || !kv_aligned(k2, desc->k2_stride, esize) ||
        !kv_aligned(v, desc->v_stride, esize))
        return DIFFATTN_ERR_UNSUPPORTED;
    return DIFFATTN_OK;
}

}  // namespace

int decode_check(const diffattn_kv_desc* desc, const void* q1, const void* k1, const void* q2,
                 const void* k2, const void* v, float lambda, const float* lambda_dev, int causal,
                 const diffattn_epilogue* epi, const void* out, size_t* work_bytes) {
    DecodePlan plan;
    diffattn_epilogue e;
    const int rc = decode_args(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out, &plan, &e);
    if (rc == DIFFATTN_OK) *work_bytes = plan.work_bytes;
    return rc;
}

}  // namespace diffattn

extern "C" {

int diffattn_decode(const diffattn_kv_desc* desc, const void* q1, const void* k1, const void* q2,
                    const void* k2, const void* v, float lambda, const float* lambda_dev,
                    int causal, const diffattn_epilogue* epi, void* out, void* workspace,
                    size_t workspace_bytes, diffattn_stream_t stream) {
    DecodePlan plan;
    diffattn_epilogue e;
    int rc = decode_args(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out, &plan, &e);
    if (rc != DIFFATTN_OK) return rc;
    if (!workspace || workspace_bytes < plan.work_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return DIFFATTN_ERR_INVALID;
    const diffattn_kv_desc& d = *desc;
    const size_t esize = d.dtype == DIFFATTN_BF16 ? 2 : 4;
    const int64_t dv = value_width(d.Dv, d.D);
    const int64_t hk = d.H / group_of(d.kv_group);
    const bool k_shared = same_tensor(k1, d.k1_stride, k2, d.k2_stride, d.B, hk, d.Tk);
    const bool dense_kv = d.k1_stride[2] == d.D && d.k2_stride[2] == d.D && d.v_stride[2] == dv;
    // the tensor-core decode of up to 16 rows needs dense, aligned rows of the
    // cache and of the queries, and at D = 128 one key tensor for both branches
    const bool tc_call = plan.tc_only && (d.D == 64 || k_shared) && dense_kv &&
                         kv_aligned(k1, d.k1_stride, esize) && kv_aligned(k2, d.k2_stride, esize) &&
                         kv_aligned(v, d.v_stride, esize) && kv_aligned(q1, d.q1_stride, esize) &&
                         kv_aligned(q2, d.q2_stride, esize);
    auto run_forward = [&]() {
        // Tq query rows at the end of the Tk-key sequence: query i at key
        // position Tk - Tq + i; one forward launch with the static schedule
        const FwdShape f{d.B, d.H, plan.Hk, d.Tq, d.Tk, d.D, dv, d.Tk - d.Tq,
                         d.dtype, d.q1_stride, d.k1_stride, d.q2_stride, d.k2_stride, d.v_stride,
                         d.o_stride};
        return launch_forward(f, q1, k1, q2, k2, v, lambda, lambda_dev, causal, e, out, nullptr,
                              nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
    };
    if (plan.forward) return run_forward();
    if (plan.tc_only && !tc_call) {
        // at D = 64 the split-key layout of up to 8-row units on the CUDA cores
        // (which needs aligned K1, K2 and V); else the forward kernels
        if (!plan.fb_valid || !kv_aligned(k1, d.k1_stride, esize) || !kv_aligned(k2, d.k2_stride, esize) ||
            !kv_aligned(v, d.v_stride, esize))
            return run_forward();
        plan.tc_only = false;
        plan.tq_bucket = plan.fb_tq_bucket;
        plan.splits = plan.fb_splits;
        plan.split_len = plan.fb_split_len;
        plan.row_chunks = plan.fb_row_chunks;
    }
    DecodeParams p{};
    p.B = (int)d.B;
    p.H = (int)d.H;
    p.Tq = (int)d.Tq;
    p.Tk = (int)d.Tk;
    p.D = (int)d.D;
    p.causal = causal ? 1 : 0;
    p.bf16 = d.dtype == DIFFATTN_BF16 ? 1 : 0;
    p.kv_group = plan.kv_group;
    p.Hk = plan.Hk;
    p.row_chunks = plan.row_chunks;
    p.dense_kv = dense_kv ? 1 : 0;
    p.tc_only = plan.tc_only ? 1 : 0;
    p.k_shared = k_shared ? 1 : 0;
    p.tc_ok = plan.tc_only || (p.dense_kv && d.dtype == DIFFATTN_BF16 && d.D == 64 &&
                          kv_aligned(q1, d.q1_stride, esize) && kv_aligned(q2, d.q2_stride, esize))
                  ? 1 : 0;
    p.tq_bucket = plan.tq_bucket;
    p.splits = plan.splits;
    p.total_items = (int)((int64_t)plan.Hk * d.B * plan.row_chunks * plan.splits);
    p.split_len = plan.split_len;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d.D));
    p.lambda = lambda;
    p.lambda_dev = lambda_dev;
    p.q1 = q1;
    p.k1 = k1;
    p.q2 = q2;
    p.k2 = k2;
    p.v = v;
    p.out = out;
    copy3(p.s_q1, d.q1_stride);
    copy3(p.s_k1, d.k1_stride);
    copy3(p.s_q2, d.q2_stride);
    copy3(p.s_k2, d.k2_stride);
    copy3(p.s_v, d.v_stride);
    copy3(p.s_o, d.o_stride);
    p.work = static_cast<float*>(workspace);
    CUtensorMap kv_maps[3];
    if (p.tc_ok) {
        DeviceState* dev = nullptr;
        rc = device_state(&dev);
        if (rc != DIFFATTN_OK) return rc;
        p.status = dev->status;
        // the cache as 4-D {inner, Tk, heads, B} maps with 128-key boxes; if
        // the encoder refuses them, the CUDA-core pass runs instead
        diffattn_desc md{};
        md.B = d.B;
        md.T = d.Tk;
        if (encode_map(&kv_maps[0], k1, d.D, &md, hk, d.k1_stride, 64, 128) == DIFFATTN_OK &&
            encode_map(&kv_maps[1], k2, d.D, &md, hk, d.k2_stride, 64, 128) == DIFFATTN_OK &&
            encode_map(&kv_maps[2], v, dv, &md, hk, d.v_stride, 64, 128) == DIFFATTN_OK)
            p.tc_maps = kv_maps;
        else if (plan.tc_only)
            return run_forward();
        else
            p.tc_ok = 0;
    }
    p.norm = e.norm;
    p.norm_eps = e.eps;
    p.norm_weight = e.weight;
    p.norm_bias = e.bias;
    p.out_scale = e.out_scale;
    return launch_decode(p, reinterpret_cast<cudaStream_t>(stream)) == 0 ? DIFFATTN_OK
                                                                       : DIFFATTN_ERR_CUDA;
}

}  // extern "C"

namespace diffattn {
namespace {

// Streams and events of the host-buffer forward, created once per device.
constexpr int kHostChunksMax = 8;
struct HostPipe {
    bool ready = false;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t start = nullptr, in[kHostChunksMax] = {}, done[kHostChunksMax] = {},
                out[kHostChunksMax] = {};
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mutex;      // held while a call enqueues (the events are reused)

int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DIFFATTN_ERR_CUDA;
    HostPipe& hp = g_pipes[dev];
    if (!hp.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.copy_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.copy_out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, ef) != cudaSuccess)
            return DIFFATTN_ERR_CUDA;
        for (int i = 0; i < kHostChunksMax; ++i)
            if (cudaEventCreateWithFlags(&hp.in[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.out[i], ef) != cudaSuccess)
                return DIFFATTN_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return DIFFATTN_OK;
}

// Dense element strides of a [B, heads, T, inner] tensor.
bool dense(const int64_t s[3], const diffattn_desc& d, int64_t heads, int64_t inner) {
    return (d.T == 1 || s[2] == inner) && (heads == 1 || s[1] == d.T * inner) &&
           (d.B == 1 || s[0] == heads * d.T * inner);
}

}  // namespace
}  // namespace diffattn

extern "C" {

int diffattn_fwd_host(const diffattn_desc* desc, const void* q1_host, const void* k1_host,
                      const void* q2_host, const void* k2_host, const void* v_host, float lambda,
                      const float* lambda_dev, int causal, void* out_host, void* q1, void* k1,
                      void* q2, void* k2, void* v, void* out, void* workspace,
                      size_t workspace_bytes, diffattn_stream_t stream) {
    int rc = validate(desc, q1, k1, q2, k2, v, out);
    if (rc != DIFFATTN_OK) return rc;
    if (!q1_host || !k1_host || !q2_host || !k2_host || !v_host || !out_host)
        return DIFFATTN_ERR_INVALID;
    if (!lambda_dev && !std::isfinite(lambda)) return DIFFATTN_ERR_INVALID;
    const diffattn_desc& d = *desc;
    const int64_t g = group_of(d.kv_group);
    const int64_t hk = d.H / g;
    const int64_t dv = value_width(d.Dv, d.D);
    if (!dense(d.q1_stride, d, d.H, d.D) || !dense(d.q2_stride, d, d.H, d.D) ||
        !dense(d.k1_stride, d, hk, d.D) || !dense(d.k2_stride, d, hk, d.D) ||
        !dense(d.v_stride, d, hk, dv) || !dense(d.o_stride, d, d.H, dv))
        return DIFFATTN_ERR_INVALID;
    DeviceState* dev = nullptr;
    rc = device_state(&dev);
    if (rc != DIFFATTN_OK) return rc;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* hp = nullptr;
    rc = host_pipe(&hp);
    if (rc != DIFFATTN_OK) return rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = d.dtype == DIFFATTN_BF16 ? 2 : 4;
    // Chunks of whole key/value heads (with their g query heads: in the dense
    // layout both are contiguous byte ranges), each with at least two work
    // items per SM for the forward, at most kHostChunksMax.  The call then takes
    // about the input copies' time plus one chunk's forward and output copy.
    const int64_t units = d.B * hk;
    const int64_t items_per_unit = g * ((d.T + 127) / 128);
    int64_t chunks = units * items_per_unit / (2ll * dev->num_sms);
    if (chunks > kHostChunksMax) chunks = kHostChunksMax;
    if (chunks > units) chunks = units;
    if (chunks < 1) chunks = 1;
    const bool k_same = k1_host == k2_host && k1 == k2;
    const int64_t qrow = d.T * d.D * (int64_t)es;        // bytes of one query head of Q1 / Q2
    const int64_t orow = d.T * dv * (int64_t)es;         // of O and of V per head
    auto copy = [&](void* dst, const void* src, int64_t off, int64_t bytes, cudaMemcpyKind kind,
                    cudaStream_t s) {
        return cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off,
                               (size_t)bytes, kind, s) == cudaSuccess;
    };
    // the copies start after the work already on the caller's stream
    if (cudaEventRecord(hp->start, st) != cudaSuccess ||
        cudaStreamWaitEvent(hp->copy_in, hp->start, 0) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t u0 = units * c / chunks, u1 = units * (c + 1) / chunks;
        const int64_t nq = (u1 - u0) * g;                  // query heads in the chunk
        const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
        if (!copy(q1, q1_host, u0 * g * qrow, nq * qrow, h2d, hp->copy_in) ||
            !copy(q2, q2_host, u0 * g * qrow, nq * qrow, h2d, hp->copy_in) ||
            !copy(k1, k1_host, u0 * qrow, (u1 - u0) * qrow, h2d, hp->copy_in) ||
            (!k_same && !copy(k2, k2_host, u0 * qrow, (u1 - u0) * qrow, h2d, hp->copy_in)) ||
            !copy(v, v_host, u0 * orow, (u1 - u0) * orow, h2d, hp->copy_in) ||
            cudaEventRecord(hp->in[c], hp->copy_in) != cudaSuccess ||
            cudaStreamWaitEvent(st, hp->in[c], 0) != cudaSuccess)
            return DIFFATTN_ERR_CUDA;
        // the chunk as a problem of its own: B = 1, its query heads as H
        diffattn_desc cd = d;
        cd.B = 1;
        cd.H = nq;
        for (int64_t* sd : {cd.q1_stride, cd.q2_stride, cd.k1_stride, cd.k2_stride, cd.v_stride,
                            cd.o_stride})
            sd[0] = 0;
        rc = forward_impl(&cd, static_cast<char*>(q1) + u0 * g * qrow,
                          static_cast<char*>(k1) + u0 * qrow, static_cast<char*>(q2) + u0 * g * qrow,
                          static_cast<char*>(k2) + u0 * qrow, static_cast<char*>(v) + u0 * orow,
                          lambda, lambda_dev, causal, nullptr,
                          static_cast<char*>(out) + u0 * g * orow, nullptr, nullptr, workspace,
                          workspace_bytes, stream);
        if (rc != DIFFATTN_OK) return rc;
        if (cudaEventRecord(hp->done[c], st) != cudaSuccess ||
            cudaStreamWaitEvent(hp->copy_out, hp->done[c], 0) != cudaSuccess ||
            !copy(out_host, out, u0 * g * orow, nq * orow, cudaMemcpyDeviceToHost, hp->copy_out) ||
            cudaEventRecord(hp->out[c], hp->copy_out) != cudaSuccess)
            return DIFFATTN_ERR_CUDA;
    }
    // the call is complete on the caller's stream once the last output copy is
    return cudaStreamWaitEvent(st, hp->out[chunks - 1], 0) == cudaSuccess ? DIFFATTN_OK
                                                                           : DIFFATTN_ERR_CUDA;
}

int diffattn_selftest_timeout(diffattn_stream_t stream) {
    DeviceState* dev = nullptr;
    const int rc = device_state(&dev);
    if (rc != DIFFATTN_OK) return rc;
    return launch_selftest_timeout(dev->status, reinterpret_cast<cudaStream_t>(stream)) == 0
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

int diffattn_get_device_error(diffattn_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    DeviceState* dev = nullptr;
    int rc = device_state(&dev);
    if (rc != DIFFATTN_OK) return rc;
    uint32_t word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    if (word == 0) return DIFFATTN_OK;
    if (cudaMemset(dev->status, 0, sizeof(word)) != cudaSuccess) return DIFFATTN_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DIFFATTN_ERR_CUDA;
    return DIFFATTN_ERR_TIMEOUT;
}

const char* diffattn_strerror(int code) {
    switch (code) {
        case DIFFATTN_OK: return "success";
        case DIFFATTN_ERR_INVALID: return "invalid argument";
        case DIFFATTN_ERR_UNSUPPORTED: return "unsupported request";
        case DIFFATTN_ERR_CUDA: return "CUDA error";
        case DIFFATTN_ERR_TIMEOUT: return "a kernel wait ran out of time";
        default: return "unknown error code";
    }
}

int diffattn_version(void) { return 200; }

}  // extern "C"
