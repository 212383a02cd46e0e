// noalloc.cu -- decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode step: an inference runtime or plug-in host that owns every device
// buffer and hands the kernel only its inputs and outputs, a process held to
// a fixed device-memory budget, or a latency-critical loop that must not pay
// for an allocator call (cudaMalloc may synchronise the device).  For them,
// diffattn_decode_noalloc keeps the split-KV partial results in a buffer that
// is part of the loaded library itself, so a call allocates nothing.
//
// The buffer is a file-scope device array of kNoAllocScratchBytes.  Every GPU
// that loads the library holds one copy of it until the process exits.  Every
// call uses the same array: two calls that run on the GPU at the same time
// (different streams, or host threads) overwrite each other's partial results.
// Nothing in it needs to start at zero: each call writes every slot it reads.
#include "diffattn.h"
#include "kernels.h"

#include <cmath>
#include <cstdint>
#include <mutex>

namespace diffattn {
namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct Scratch {
    unsigned long long ctx = 0;   // ID of the context the address belongs to
    float* ptr = nullptr;
};
Scratch g_scratch[kMaxDevices];

// Device address of the scratch array in the current context.  The array's
// name is a host-side stand-in in host code; the address comes from the
// runtime, once per device and context, with that device current.  A device
// reset or another current context (which load the module again, possibly
// elsewhere) make the next call look it up again.
int scratch_for_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DIFFATTN_ERR_CUDA;
    const unsigned long long ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mutex);
    Scratch& s = g_scratch[dev];
    if (!s.ptr || ctx == 0 || s.ctx != ctx) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return DIFFATTN_ERR_CUDA;
        s.ptr = static_cast<float*>(ptr);
        s.ctx = current_context();
    }
    *out = s.ptr;
    return DIFFATTN_OK;
}

}  // namespace
}  // namespace diffattn

extern "C" {

int diffattn_decode_noalloc(const diffattn_kv_desc* desc, const void* q1, const void* k1,
                            const void* q2, const void* k2, const void* v, float lambda,
                            const float* lambda_dev, int causal, const diffattn_epilogue* epi,
                            void* out, diffattn_stream_t stream) {
    // the checks of diffattn_decode first, so errors come in the same order
    size_t need = 0;
    int rc = diffattn::decode_check(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out,
                                    &need);
    if (rc != DIFFATTN_OK) return rc;
    // then the one limit of this entry point: the partial results must fit
    if (need > diffattn::kNoAllocScratchBytes) return DIFFATTN_ERR_UNSUPPORTED;
    float* scratch = nullptr;
    rc = diffattn::scratch_for_current_device(&scratch);
    if (rc != DIFFATTN_OK) return rc;
    return diffattn_decode(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out, scratch,
                           diffattn::kNoAllocScratchBytes, stream);
}

}  // extern "C"
