// gq_fused.cu -- the pieces of the fused entry points (gq_mul_mat_rmsnorm,
// gq_mul_mat_swiglu) for shapes the fused decode kernel does not take: a per-token
// RMSNorm of X ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
// section 4.1) ahead of the plain product, and Swish(gate) * up (section 4.4) after two
// plain products. At decode (N <= 2) both steps run inside the streaming kernel instead
// (gq_gemv.cu, kFuse).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kNormThreads = 256;

// One CTA per token: Xhat[n][k] = X[n][k] * inv * gamma[k], inv = 1 / sqrt(mean_k x^2 + eps).
// The sum of squares runs in a fixed order (thread strides, a fixed shuffle tree, the warps
// in order), so the result does not depend on timing.
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_x_kernel(const float* __restrict__ X, const float* __restrict__ gamma, float eps,
                 int64_t K, float* __restrict__ Xhat) {
    __shared__ float part[kNormThreads / 32];
    const float* x = X + static_cast<int64_t>(blockIdx.x) * K;
    float* y = Xhat + static_cast<int64_t>(blockIdx.x) * K;
    float ss = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += kNormThreads) ss = fmaf(x[k], x[k], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float total = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) total += part[w];
    const float inv = 1.0f / sqrtf(total / static_cast<float>(K) + eps);
    for (int64_t k = threadIdx.x; k < K; k += kNormThreads) y[k] = x[k] * inv * gamma[k];
}

// H = Swish(G) * U elementwise, Swish(z) = z / (1 + e^-z).
__global__ void __launch_bounds__(256)
swiglu_kernel(const float* __restrict__ G, const float* __restrict__ U, float* __restrict__ H,
              int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const float g = G[i];
        H[i] = g / (1.0f + expf(-g)) * U[i];
    }
}

}  // namespace

cudaError_t launch_rmsnorm_x(const float* X, const float* gamma, float eps, int64_t N,
                             int64_t K, float* Xhat, cudaStream_t s) {
    if (N <= 0 || K <= 0) return cudaSuccess;
    if (N > 2147483647) return cudaErrorInvalidValue;
    rmsnorm_x_kernel<<<static_cast<unsigned>(N), kNormThreads, 0, s>>>(X, gamma, eps, K, Xhat);
    return cudaGetLastError();
}

cudaError_t launch_swiglu(const float* G, const float* U, float* H, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    // grid-stride: 16 blocks of 256 threads per SM at most
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, int64_t(info->sm_count) * 16);
    swiglu_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(G, U, H, n);
    return cudaGetLastError();
}

}  // namespace gq
