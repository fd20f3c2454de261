// gq_noalloc.cu -- gq_mul_mat_noalloc: mul_mat that never allocates device memory.
//
// Some callers cannot call cudaMalloc (or anything that does) at the point where they
// multiply: engines that reserve all device memory up front in their own arena and forbid
// later allocation, and real-time loops with a fixed memory budget where an allocation
// could stall or fail mid-run. gq_mul_mat may allocate
// (its tensor-core path grows a library-owned workspace); this entry point instead uses a
// fixed array compiled into the library as that workspace.
//
// The array below is a file-scope __device__ variable of this module. A GPU holds it
// (kNoAllocScratchBytes) from the module's first use on that device (CUDA's default lazy
// module loading), or from context creation when modules load eagerly
// (CUDA_MODULE_LOADING=EAGER), until the process exits. Host code must not
// use its name as a pointer: on the host it is only a stand-in. Its device address is
// looked up once per device with cudaGetSymbolAddress, with that device current, and
// passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// Fixed workspace of the tensor-core paths. Prefill keeps a bf16 copy of X there, N * K * 2
// bytes, so it covers N * K <= 32 Mi elements (e.g. 2048 tokens x K = 11008, or 4096 x
// 8192); the tensor-core decode needs at most 64 * K * 2 + 16 MiB + 4 KiB.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up on the first call
// per device (the "set-up"); later calls reuse it. The cache is never refreshed: after
// cudaDeviceReset the module loads again at another address, so libgq must not be used
// on a device again once the process has reset it.
cudaError_t noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

bool aligned_to(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace gq

extern "C" gq_status gq_mul_mat_noalloc(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                                        const float* X, int64_t N, float* Y, void* stream) {
    // Same argument contract as gq_mul_mat.
    if (gq::block_bytes_of(t) == 0) return GQ_ERR_TYPE;
    const int64_t max_dim = (int64_t(1) << 31) - 1, max_elems = int64_t(1) << 40;
    if (M < 0 || K < 0 || N < 0 || K % gq::block_weights_of(t) != 0) return GQ_ERR_SHAPE;
    if (M > max_dim || K > max_dim || N > max_dim) return GQ_ERR_SHAPE;
    if (M * K > max_elems || N * K > max_elems || N * M > max_elems) return GQ_ERR_SHAPE;
    if (M == 0 || N == 0) return GQ_OK;
    if (!Y) return GQ_ERR_NULL;
    if (K > 0 && (!W_blocks || !X)) return GQ_ERR_NULL;
    if (!gq::aligned_to(Y, 4)) return GQ_ERR_ALIGN;
    if (K > 0 && (!gq::aligned_to(W_blocks, 16) || !gq::aligned_to(X, 4))) return GQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemsetAsync(Y, 0, sizeof(float) * N * M, s) == cudaSuccess ? GQ_OK
                                                                            : GQ_ERR_CUDA;
    const gq::MatProblem p{static_cast<const uint8_t*>(W_blocks), X, Y, M, K};
    const int64_t cap = static_cast<int64_t>(gq::kNoAllocScratchBytes);
    // Tensor-core decode (3..64 tokens): its bf16 X tiles, partial sums and split-tile
    // counters fit the array for any K up to ~390k; x_tiles_kernel rewrites the tiles and
    // zeroes the counters at the start of every call. Past that size, the CUDA-core decode
    // kernels, which need no workspace.
    if (gq::gemv_tc_eligible(t, p, N)) {
        if (gq::gemv_tc_workspace_bytes(t, &p, 1, N) > cap)
            return gq::launch_mul_mat(t, &p, 1, N, s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
        void* scratch = nullptr;
        if (gq::noalloc_scratch(&scratch) != cudaSuccess) return GQ_ERR_CUDA;
        return gq::launch_gemv_tc(t, &p, 1, N, scratch, s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
    }
    if (!gq::gemm_eligible(t, p, N))   // CUDA-core decode: needs no workspace at all
        return gq::launch_mul_mat(t, &p, 1, N, s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
    if (gq::gemm_x_bytes(K, N) > cap) return GQ_ERR_SHAPE;   // N * K beyond the fixed array
    void* scratch = nullptr;
    if (gq::noalloc_scratch(&scratch) != cudaSuccess) return GQ_ERR_CUDA;
    return gq::launch_gemm(t, p, N, scratch, cap, s) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}
