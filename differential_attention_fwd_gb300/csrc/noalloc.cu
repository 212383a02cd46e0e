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
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  The array's
// name is a host-side stand-in in host code; the address comes from the
// runtime, once per device, with that device current.
int scratch_for_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DIFFATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return DIFFATTN_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float*>(ptr);
    }
    *out = g_scratch_ptr[dev];
    return DIFFATTN_OK;
}

}  // namespace
}  // namespace diffattn

extern "C" {

int diffattn_decode_noalloc(const diffattn_kv_desc* desc, const void* q1, const void* k1,
                            const void* q2, const void* k2, const void* v, float lambda,
                            const float* lambda_dev, int causal, const diffattn_epilogue* epi,
                            void* out, diffattn_stream_t stream) {
    const size_t need = diffattn_decode_workspace_bytes(desc);
    if (need == 0) {
        // invalid or unsupported descriptor: let the regular entry point say which
        return diffattn_decode(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out,
                               nullptr, 0, stream);
    }
    // more partial results than the static buffer holds
    if (need > diffattn::kNoAllocScratchBytes) return DIFFATTN_ERR_UNSUPPORTED;
    float* scratch = nullptr;
    const int rc = diffattn::scratch_for_current_device(&scratch);
    if (rc != DIFFATTN_OK) return rc;
    return diffattn_decode(desc, q1, k1, q2, k2, v, lambda, lambda_dev, causal, epi, out, scratch,
                           diffattn::kNoAllocScratchBytes, stream);
}

}  // extern "C"
