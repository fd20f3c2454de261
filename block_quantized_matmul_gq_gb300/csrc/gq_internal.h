// gq_internal.h -- host-side interface between the C ABI (gq_capi.cu) and the kernel
// translation units. Not installed; callers use include/gq.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gq.h"

namespace gq {

constexpr int kQ4Bytes = 18;    // fp16 scale + 16 bytes of nibble codes
constexpr int kQ8Bytes = 34;    // fp16 scale + 32 int8 codes
constexpr int kQ4KBytes = 144;  // Q4_K super-block: fp16 d, fp16 dmin, 12 scale bytes, 128 code bytes
constexpr int kQ4KWeights = 256;

inline int block_bytes_of(gq_type t) {
    switch (t) {
        case GQ_TYPE_Q4_0: return kQ4Bytes;
        case GQ_TYPE_Q8_0: return kQ8Bytes;
        case GQ_TYPE_Q4_K: return kQ4KBytes;
    }
    return 0;
}

// Weights per block: 32, or 256 for a Q4_K super-block; 0 for an unknown type.
inline int block_weights_of(gq_type t) {
    return t == GQ_TYPE_Q4_K ? kQ4KWeights : (block_bytes_of(t) ? 32 : 0);
}

// One validated, non-empty mul_mat problem (K > 0, M > 0) as the launchers see it.
struct MatProblem {
    const uint8_t* W;
    const float* X;
    float* Y;
    int64_t M;
    int64_t K;
    // Fused forms (CUDA-core decode only): RMSNorm of X ahead of the product when gamma is
    // set; Swish(X W^T) * (X W2^T) into Y when W2 (the up matrix) is set.
    const uint8_t* W2 = nullptr;
    const float* gamma = nullptr;
    float eps = 0.0f;
};

// Per-device facts, looked up once per device.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
    unsigned* status = nullptr;   // device address of this device's status word
};
cudaError_t current_device_info(DeviceInfo** out);

// n_blocks blocks of block_weights_of(t) weights each, consecutive in W and in out.
cudaError_t launch_quantize(gq_type t, const float* W, int64_t n_blocks, uint8_t* out,
                            cudaStream_t s);
cudaError_t launch_dequantize(gq_type t, const uint8_t* blocks, int64_t n_elems, float* out,
                              cudaStream_t s);

// Y = X . What^T for every problem on the decode (CUDA-core, streaming) kernels; all
// share type t and N tokens.
cudaError_t launch_mul_mat(gq_type t, const MatProblem* probs, int count, int64_t N,
                           cudaStream_t s);

// Fused decode forms on the CUDA-core decode kernel (see MatProblem::gamma, ::W2): whether
// the streaming kernel takes this shape, and the launch (any N, in passes of up to 4).
bool fused_decode_eligible(gq_type t, const MatProblem& p);
cudaError_t launch_mul_mat_fused(gq_type t, const MatProblem& p, int64_t N, cudaStream_t s);

// Composite pieces of the fused entry points (gq_fused.cu): Xhat = RMSNorm(X) per token
// (N x K), and H = Swish(G) * U elementwise (n floats).
cudaError_t launch_rmsnorm_x(const float* X, const float* gamma, float eps, int64_t N,
                             int64_t K, float* Xhat, cudaStream_t s);
cudaError_t launch_swiglu(const float* G, const float* U, float* H, int64_t n, cudaStream_t s);

// Quantized-activation mul_mat (X quantized per 32-block like Q8_0, integer block sums):
// the streaming decode kernel with Q8_0 activation records, up to 4 tokens per pass over
// the weights. Needs K % 256 == 0, 16-byte aligned W and X, and records that fit shared
// memory (q8x_eligible).
bool q8x_eligible(gq_type t, const MatProblem& p);
cudaError_t launch_mul_mat_q8x(gq_type t, const MatProblem* probs, int count, int64_t N,
                               cudaStream_t s);

// Prefill path: tcgen05 tensor-core GEMM. Its workspace (256-byte aligned) is the bf16
// copy of X: gemm_x_bytes(K, N) == gemm_workspace_bytes(K, N) bytes.
constexpr int64_t kGemmMinTokens = 65;
int64_t gemm_x_bytes(int64_t K, int64_t N);
int64_t gemm_workspace_bytes(int64_t K, int64_t N);
bool gemm_eligible(gq_type t, const MatProblem& p, int64_t N);
cudaError_t launch_gemm(gq_type t, const MatProblem& p, int64_t N, void* workspace,
                        int64_t workspace_bytes, cudaStream_t s);

// Decode on tensor cores for kGemvTcMinTokens..kGemvTcMaxTokens tokens (K % 256 == 0):
// grouped like launch_mul_mat. Needs gemv_tc_workspace_bytes of workspace (pre-arranged
// bf16 X tiles, 16 / 32 / 64 token rows per problem; Q4_K up to 16 tokens also the X block
// sums, 1 KB per 256 k), 256-byte aligned.
constexpr int64_t kGemvTcMinTokens = 3;
constexpr int64_t kGemvTcMaxTokens = 64;
bool gemv_tc_eligible(gq_type t, const MatProblem& p, int64_t N);
int64_t gemv_tc_workspace_bytes(gq_type t, const MatProblem* probs, int count, int64_t N);
cudaError_t launch_gemv_tc(gq_type t, const MatProblem* probs, int count, int64_t N,
                           void* workspace, cudaStream_t s);

}  // namespace gq
