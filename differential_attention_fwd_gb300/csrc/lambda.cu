// lambda.cu -- the scalar re-parameterisation
//   lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
// (aifetchly "Differential Transformer...", section 3; paperleet
// "Differential Transformer Attention", Formula and conventions).
// One warp: float64 dot products, float64 exponentials, one rounding to fp32.
#include "kernels.h"

namespace diffattn {

__global__ void __launch_bounds__(32)
diffattn_lambda_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                       const float* __restrict__ lq2, const float* __restrict__ lk2, int64_t n,
                       double lambda_init, float* __restrict__ out) {
    double d1 = 0.0, d2 = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += 32) {
        d1 = fma((double)lq1[i], (double)lk1[i], d1);
        d2 = fma((double)lq2[i], (double)lk2[i], d2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        d1 += __shfl_xor_sync(0xffffffffu, d1, o);
        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
    }
    if (threadIdx.x == 0) *out = (float)(exp(d1) - exp(d2) + lambda_init);
}

// Backward: with e_b = exp(lq_b . lk_b) and g = dL/dlambda,
//   dL/dlq1 = g e1 lk1, dL/dlk1 = g e1 lq1, dL/dlq2 = -g e2 lk2, dL/dlk2 = -g e2 lq2.
// One block: the dot products in float64 by the first warp, then every thread
// writes its share of the four gradient vectors.
__global__ void __launch_bounds__(256)
diffattn_lambda_bwd_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                           const float* __restrict__ lq2, const float* __restrict__ lk2, int64_t n,
                           const float* __restrict__ dlambda, float* __restrict__ dlq1,
                           float* __restrict__ dlk1, float* __restrict__ dlq2,
                           float* __restrict__ dlk2) {
    __shared__ double coef[2];
    if (threadIdx.x < 32) {
        double d1 = 0.0, d2 = 0.0;
        for (int64_t i = threadIdx.x; i < n; i += 32) {
            d1 = fma((double)lq1[i], (double)lk1[i], d1);
            d2 = fma((double)lq2[i], (double)lk2[i], d2);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            d1 += __shfl_xor_sync(0xffffffffu, d1, o);
            d2 += __shfl_xor_sync(0xffffffffu, d2, o);
        }
        if (threadIdx.x == 0) {
            const double g = (double)*dlambda;
            coef[0] = g * exp(d1);
            coef[1] = -g * exp(d2);
        }
    }
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        dlq1[i] = (float)(coef[0] * lk1[i]);
        dlk1[i] = (float)(coef[0] * lq1[i]);
        dlq2[i] = (float)(coef[1] * lk2[i]);
        dlk2[i] = (float)(coef[1] * lq2[i]);
    }
}

int launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                      int64_t n, const float* dlambda, float* dlq1, float* dlk1, float* dlq2,
                      float* dlk2, cudaStream_t stream) {
    diffattn_lambda_bwd_kernel<<<1, 256, 0, stream>>>(lq1, lk1, lq2, lk2, n, dlambda, dlq1, dlk1,
                                                      dlq2, dlk2);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                  int64_t n, double lambda_init, float* out, cudaStream_t stream) {
    diffattn_lambda_kernel<<<1, 32, 0, stream>>>(lq1, lk1, lq2, lk2, n, lambda_init, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace diffattn
