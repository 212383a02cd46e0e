// unit_throughput.cu -- throughput of the instructions the attention kernels'
// elementwise warps use (ex2.approx.f32, ex2.approx.bf16x2, fma.rn.f32x2,
// cvt.rn.bf16x2.f32, scalar fmul) and of mixes of them, on one CTA of 512
// threads per SM (or 256, two warps per SM sub-partition as in the kernels)
// with eight independent dependency chains per thread, timed with clock64 per
// CTA.  Not part of the library: a measurement that
// tells which unit bounds a warp's arithmetic.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o unit_throughput unit_throughput.cu
//   ./unit_throughput
//
// Each line reports, per SM, the thread-level operations of the loop body per
// clock: one "operation" is one pass over a chain, which is one instruction of
// the named kind (plus the cheap helper noted in brackets).  Every write goes
// to an index below the grid's size; no thread waits on another.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

namespace {

constexpr int kIters = 2048;
constexpr int kChains = 8;
constexpr int kThreads = 512;

__device__ __forceinline__ float ex2_f32(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
    uint32_t y;
    asm volatile("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm volatile("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// MODE: 0 ex2 (+fadd), 1 ex2.bf16x2 (+xor), 2 fma.f32x2, 3 cvt (+fadd, or),
// 4 fmul (+xor), 5 ex2 (+fadd) with two fma.f32x2, 6 ex2 (+fadd) with a cvt
// (+xor), 7 ex2 alone, 8 fma.f32x2 with a cvt (+xor), 9 ex2 of arguments in
// [-16, -1] (+ffma), 10 the pattern of a softmax column pair: an fma.f32x2
// forming two exponents, two ex2, an add.f32x2 into a running sum and a cvt
// of the pair (+xor, and two 64-bit logic operations that keep the chain in
// range), 11 the same pattern without the logic operations: the pair's 2^x
// feed the next exponents directly (+xor only).
template <int MODE, int NT>
__global__ void __launch_bounds__(NT, 1) probe(unsigned long long* cycles, float* sink) {
    float x[kChains];
    uint32_t xb[kChains];
    uint64_t x2[kChains];
    for (int i = 0; i < kChains; ++i) {
        x[i] = -0.5f - 0.01f * (threadIdx.x & 7) - 0.001f * i;      // 2^x stays in (0, 1)
        xb[i] = 0xBF00BF00u + i;
        x2[i] = (static_cast<uint64_t>(__float_as_uint(x[i])) << 32) | __float_as_uint(0.5f * x[i]);
    }
    const uint64_t m = (static_cast<uint64_t>(__float_as_uint(0.999f)) << 32) | __float_as_uint(0.999f);
    const uint64_t a = (static_cast<uint64_t>(__float_as_uint(-1e-4f)) << 32) | __float_as_uint(-1e-4f);
    const uint64_t h = (static_cast<uint64_t>(__float_as_uint(-1.0f)) << 32) | __float_as_uint(-1.0f);
    const uint64_t z = 0;
    uint64_t rs[kChains];
    for (int i = 0; i < kChains; ++i) {
        rs[i] = 0;
        if (MODE == 11) x2[i] = (static_cast<uint64_t>(__float_as_uint(0.7f)) << 32) | __float_as_uint(0.6f);
    }
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            if (MODE == 0) x[i] = ex2_f32(x[i]) - 1.5f;
            if (MODE == 1) xb[i] = ex2_bf16x2(xb[i]) ^ 0x80008000u;
            if (MODE == 2) x2[i] = fma_f32x2(x2[i], m, a);
            if (MODE == 3) x[i] = __uint_as_float(cvt_bf16x2(x[i], x[i] + 1.f) | 0xBF000000u);
            if (MODE == 4) x[i] = -__uint_as_float(__float_as_uint(x[i]) ^ 0x1u) * 1.0001f;
            if (MODE == 5) {
                x[i] = ex2_f32(x[i]) - 1.5f;
                x2[i] = fma_f32x2(x2[i], m, a);
                x2[(i + 4) % kChains] = fma_f32x2(x2[(i + 4) % kChains], m, a);
            }
            if (MODE == 6) {
                x[i] = ex2_f32(x[i]) - 1.5f;
                xb[i] = cvt_bf16x2(x[(i + 1) % kChains], x[(i + 2) % kChains]) ^ xb[i];
            }
            if (MODE == 7) x[i] = ex2_f32(x[i]);
            if (MODE == 8) {
                x2[i] = fma_f32x2(x2[i], m, a);
                xb[i] = cvt_bf16x2(__uint_as_float(static_cast<uint32_t>(x2[(i + 3) % kChains])), 1.f) ^ xb[i];
            }
            if (MODE == 9) x[i] = fmaf(ex2_f32(x[i]), -15.0f, -1.0f);
            if (MODE == 11) {
                const uint64_t e = fma_f32x2(x2[i], h, z);     // exponents in [-1, -0.25]
                const float p0 = ex2_f32(__uint_as_float(static_cast<uint32_t>(e)));
                const float p1 = ex2_f32(__uint_as_float(static_cast<uint32_t>(e >> 32)));
                const uint64_t pp = (static_cast<uint64_t>(__float_as_uint(p1)) << 32) | __float_as_uint(p0);
                asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(rs[i]) : "l"(pp));
                xb[i] ^= cvt_bf16x2(p0, p1);
                x2[i] = pp;                                       // in [0.5, 1)
            }
            if (MODE == 10) {
                // exponents of a column pair, their 2^x, the running sum, the bf16 pair
                const uint64_t e = fma_f32x2(x2[i], m, a);
                const float p0 = ex2_f32(__uint_as_float(static_cast<uint32_t>(e)));
                const float p1 = ex2_f32(__uint_as_float(static_cast<uint32_t>(e >> 32)));
                const uint64_t pp = (static_cast<uint64_t>(__float_as_uint(p1)) << 32) | __float_as_uint(p0);
                uint64_t sum;
                asm volatile("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(pp), "l"(x2[(i + 1) % kChains]));
                xb[i] ^= cvt_bf16x2(p0, p1);
                x2[i] = (sum & 0x807FFFFF807FFFFFull) | 0x3F0000003F000000ull;   // back to [-1, 1)
            }
        }
    }
    const long long t1 = clock64();
    __syncthreads();
    if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
    float s = 0.f;
    for (int i = 0; i < kChains; ++i)
        s += x[i] + __uint_as_float(xb[i]) + __uint_as_float(static_cast<uint32_t>(x2[i])) +
             __uint_as_float(static_cast<uint32_t>(rs[i]));
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;     // keeps the chains live
}

template <int MODE, int NT = kThreads>
int run(int sms, unsigned long long* cycles, float* sink, const char* name) {
    static_assert(NT <= kThreads, "sink size");
    for (int rep = 0; rep < 2; ++rep) probe<MODE, NT><<<sms, NT>>>(cycles, sink);
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    static unsigned long long h[4096];
    if (cudaMemcpy(h, cycles, sms * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess)
        return -1;
    double mean = 0;
    for (int i = 0; i < sms; ++i) mean += static_cast<double>(h[i]);
    mean /= sms;
    const double ops = static_cast<double>(NT) * kIters * kChains;
    std::printf("%-28s %9.0f cycles  %6.2f operations/clock/SM\n", name, mean, ops / mean);
    return 0;
}

}  // namespace

int main() {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 1 ||
        sms > 4096)
        return 1;
    unsigned long long* cycles = nullptr;
    float* sink = nullptr;
    if (cudaMalloc(&cycles, sms * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&sink, static_cast<size_t>(sms) * kThreads * sizeof(float)) != cudaSuccess)
        return 1;
    int rc = 0;
    rc |= run<0>(sms, cycles, sink, "ex2.f32 (+fadd)");
    rc |= run<1>(sms, cycles, sink, "ex2.bf16x2 (+xor)");
    rc |= run<2>(sms, cycles, sink, "fma.f32x2");
    rc |= run<3>(sms, cycles, sink, "cvt.bf16x2 (+fadd, or)");
    rc |= run<4>(sms, cycles, sink, "fmul (+xor)");
    rc |= run<5>(sms, cycles, sink, "ex2 (+fadd) + 2 fma.f32x2");
    rc |= run<6>(sms, cycles, sink, "ex2 (+fadd) + cvt (+xor)");
    rc |= run<7>(sms, cycles, sink, "ex2 alone");
    rc |= run<8>(sms, cycles, sink, "fma.f32x2 + cvt (+xor)");
    rc |= run<9>(sms, cycles, sink, "ex2 of [-16, -1] (+ffma)");
    rc |= run<10>(sms, cycles, sink, "softmax pair: fma2 2ex2 add2 cvt");
    rc |= run<11>(sms, cycles, sink, "softmax pair, no logic ops");
    rc |= run<11, 256>(sms, cycles, sink, "same, 256 threads");
    rc |= run<7, 256>(sms, cycles, sink, "ex2 alone, 256 threads");
    rc |= run<10, 256>(sms, cycles, sink, "softmax pair, 256 threads");
    cudaFree(cycles);
    cudaFree(sink);
    return rc == 0 ? 0 : 1;
}
