// gq_capi.cu -- the extern "C" entry points of include/gq.h: host-side argument checks,
// dispatch to the kernels, and the per-device status word that kernels set when a
// bounded wait runs out.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {

// Set by kernels (atomicOr) when a device-side wait gives up; read and cleared by
// gq_get_last_error. Host code reaches it only through cudaGetSymbolAddress.
__device__ unsigned g_status_word;

cudaError_t current_device_info(DeviceInfo** out) {
    static std::mutex mu;
    static DeviceInfo infos[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = infos[dev];
    if (d.device < 0) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&d.max_smem_optin,
                                       cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        void* p = nullptr;
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return e;
        d.status = static_cast<unsigned*>(p);
        d.device = dev;
    }
    *out = &d;
    return cudaSuccess;
}

}  // namespace gq

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxElems = int64_t(1) << 40;

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

bool known_type(gq_type t) { return gq::block_bytes_of(t) != 0; }

gq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GQ_OK : GQ_ERR_CUDA; }

// Shapes: non-negative, K a multiple of the type's block (32 weights; 256 for Q4_K), every
// dimension and product in range. The type must be known.
gq_status check_shape(gq_type t, int64_t M, int64_t K, int64_t N) {
    if (M < 0 || K < 0 || N < 0 || K % gq::block_weights_of(t) != 0) return GQ_ERR_SHAPE;
    if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return GQ_ERR_SHAPE;
    if (M * K > kMaxElems || N * K > kMaxElems || N * M > kMaxElems) return GQ_ERR_SHAPE;
    return GQ_OK;
}

gq_status quantize_impl(gq_type t, const float* W, int64_t M, int64_t K, void* out,
                        void* stream) {
    gq_status st = check_shape(t, M, K, 0);
    if (st != GQ_OK) return st;
    if (M == 0 || K == 0) return GQ_OK;
    if (!W || !out) return GQ_ERR_NULL;
    if (!aligned(W, 4) || !aligned(out, 16)) return GQ_ERR_ALIGN;
    return from_cuda(gq::launch_quantize(t, W, M * (K / gq::block_weights_of(t)),
                                         static_cast<uint8_t*>(out),
                                         static_cast<cudaStream_t>(stream)));
}

// Validates one problem; sets *empty when there is nothing to launch for it.
gq_status check_problem(const void* W, gq_type t, int64_t M, int64_t K, const float* X,
                        int64_t N, const float* Y, bool* empty) {
    if (!known_type(t)) return GQ_ERR_TYPE;
    gq_status st = check_shape(t, M, K, N);
    if (st != GQ_OK) return st;
    *empty = (M == 0 || N == 0);
    if (*empty) return GQ_OK;
    if (!Y) return GQ_ERR_NULL;
    if (K > 0 && (!W || !X)) return GQ_ERR_NULL;
    if (!aligned(Y, 4)) return GQ_ERR_ALIGN;
    if (K > 0 && (!aligned(W, 16) || !aligned(X, 4))) return GQ_ERR_ALIGN;
    return GQ_OK;
}

// Library-owned workspace of the prefill path, one buffer per (device, stream), grown on
// demand. Growing waits for the stream's queued work (which may still read the old buffer)
// and is refused while the stream is being captured into a graph.
cudaError_t internal_workspace(cudaStream_t s, size_t bytes, void** out) {
    static std::mutex mu;
    static std::map<std::pair<int, void*>, std::pair<void*, size_t>> buffers;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto& entry = buffers[std::make_pair(dev, static_cast<void*>(s))];
    if (entry.second >= bytes) {
        *out = entry.first;
        return cudaSuccess;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return e;
    if (cap != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (entry.first) cudaFree(entry.first);
    entry = {nullptr, 0};
    void* p = nullptr;
    e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) return e;
    entry = {p, bytes};
    *out = p;
    return cudaSuccess;
}

// Runs one validated, non-empty problem (K > 0): tensor cores when the shape qualifies,
// else the decode kernels. `ws` may be NULL (library workspace is used then).
gq_status run_one(gq_type t, const gq::MatProblem& p, int64_t N, void* ws, size_t ws_bytes,
                  cudaStream_t s) {
    if (gq::gemv_tc_eligible(t, p, N)) {
        const size_t need = static_cast<size_t>(gq::gemv_tc_workspace_bytes(t, &p, 1, N));
        void* w = ws;
        if (w == nullptr) {
            if (internal_workspace(s, need, &w) != cudaSuccess) return GQ_ERR_CUDA;
        } else if (ws_bytes < need || !aligned(ws, 256)) {
            return ws_bytes < need ? GQ_ERR_SHAPE : GQ_ERR_ALIGN;
        }
        return from_cuda(gq::launch_gemv_tc(t, &p, 1, N, w, s));
    }
    if (gq::gemm_eligible(t, p, N)) {
        const size_t need = static_cast<size_t>(gq::gemm_workspace_bytes(p.K, N));
        void* w = ws;
        if (w == nullptr) {
            if (internal_workspace(s, need, &w) != cudaSuccess) return GQ_ERR_CUDA;
            ws_bytes = need;
        } else if (ws_bytes < need || !aligned(ws, 256)) {
            return ws_bytes < need ? GQ_ERR_SHAPE : GQ_ERR_ALIGN;
        }
        return from_cuda(gq::launch_gemm(t, p, N, w, static_cast<int64_t>(ws_bytes), s));
    }
    return from_cuda(gq::launch_mul_mat(t, &p, 1, N, s));
}

}  // namespace

extern "C" {

int32_t gq_abi_version(void) { return GQ_ABI_VERSION; }

size_t gq_block_bytes(gq_type t) { return static_cast<size_t>(gq::block_bytes_of(t)); }

size_t gq_row_bytes(gq_type t, int64_t K) {
    const int bb = gq::block_bytes_of(t);
    if (bb == 0 || K < 0 || K % gq::block_weights_of(t) != 0) return 0;
    return static_cast<size_t>(K / gq::block_weights_of(t)) * static_cast<size_t>(bb);
}

gq_status gq_quantize_q4_0(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream) {
    return quantize_impl(GQ_TYPE_Q4_0, W, M, K, W_blocks, stream);
}

gq_status gq_quantize_q8_0(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream) {
    return quantize_impl(GQ_TYPE_Q8_0, W, M, K, W_blocks, stream);
}

gq_status gq_quantize_q4_k(const float* W, int64_t M, int64_t K, void* W_blocks,
                           void* stream) {
    return quantize_impl(GQ_TYPE_Q4_K, W, M, K, W_blocks, stream);
}

gq_status gq_dequantize(const void* W_blocks, gq_type t, int64_t M, int64_t K, float* W_out,
                        void* stream) {
    if (!known_type(t)) return GQ_ERR_TYPE;
    gq_status st = check_shape(t, M, K, 0);
    if (st != GQ_OK) return st;
    if (M == 0 || K == 0) return GQ_OK;
    if (!W_blocks || !W_out) return GQ_ERR_NULL;
    if (!aligned(W_blocks, 16) || !aligned(W_out, 4)) return GQ_ERR_ALIGN;
    return from_cuda(gq::launch_dequantize(t, static_cast<const uint8_t*>(W_blocks), M * K,
                                           W_out, static_cast<cudaStream_t>(stream)));
}

gq_status gq_mul_mat(const void* W_blocks, gq_type t, int64_t M, int64_t K, const float* X,
                     int64_t N, float* Y, void* stream) {
    bool empty = false;
    gq_status st = check_problem(W_blocks, t, M, K, X, N, Y, &empty);
    if (st != GQ_OK || empty) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(Y, 0, sizeof(float) * N * M, s));
    gq::MatProblem p{static_cast<const uint8_t*>(W_blocks), X, Y, M, K};
    return run_one(t, p, N, nullptr, 0, s);
}

size_t gq_mul_mat_workspace_size(gq_type t, int64_t M, int64_t K, int64_t N) {
    if (!known_type(t) || check_shape(t, M, K, N) != GQ_OK || M == 0 || N == 0 || K == 0)
        return 0;
    gq::MatProblem p{reinterpret_cast<const uint8_t*>(uintptr_t(256)),
                     reinterpret_cast<const float*>(uintptr_t(256)), nullptr, M, K};
    if (gq::gemv_tc_eligible(t, p, N))
        return static_cast<size_t>(gq::gemv_tc_workspace_bytes(t, &p, 1, N));
    return gq::gemm_eligible(t, p, N) ? static_cast<size_t>(gq::gemm_workspace_bytes(K, N)) : 0;
}

gq_status gq_mul_mat_ws(const void* W_blocks, gq_type t, int64_t M, int64_t K, const float* X,
                        int64_t N, float* Y, void* workspace, size_t workspace_bytes,
                        void* stream) {
    bool empty = false;
    gq_status st = check_problem(W_blocks, t, M, K, X, N, Y, &empty);
    if (st != GQ_OK || empty) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(Y, 0, sizeof(float) * N * M, s));
    gq::MatProblem p{static_cast<const uint8_t*>(W_blocks), X, Y, M, K};
    if ((gq::gemm_eligible(t, p, N) || gq::gemv_tc_eligible(t, p, N)) && workspace == nullptr)
        return GQ_ERR_NULL;
    return run_one(t, p, N, workspace, workspace_bytes, s);
}

}  // extern "C"

namespace {

// Validated problems of a batched call, split by path. `run` holds the non-empty K > 0
// problems; K == 0 ones are zeroed on the stream here.
struct BatchPlan {
    gq::MatProblem gemm[GQ_MAX_BATCH], tc[GQ_MAX_BATCH], cc[GQ_MAX_BATCH];
    int n_gemm = 0, n_tc = 0, n_cc = 0;
    size_t ws_bytes = 0;   // max(largest GEMM workspace, sum of tensor-core decode tiles)
};

gq_status plan_batch(const gq_mul_mat_problem* problems, int32_t count, gq_type t, int64_t N,
                     BatchPlan* plan, cudaStream_t s, bool zero_k0) {
    if (count < 0 || count > GQ_MAX_BATCH) return GQ_ERR_SHAPE;
    if (!known_type(t)) return GQ_ERR_TYPE;
    if (count == 0) return GQ_OK;
    if (!problems) return GQ_ERR_NULL;
    for (int i = 0; i < count; ++i) {
        const gq_mul_mat_problem& p = problems[i];
        bool empty = false;
        gq_status st = check_problem(p.W_blocks, t, p.M, p.K, p.X, N, p.Y, &empty);
        if (st != GQ_OK) return st;
    }
    size_t gemm_max = 0;
    for (int i = 0; i < count; ++i) {
        const gq_mul_mat_problem& p = problems[i];
        if (p.M == 0 || N == 0) continue;
        if (p.K == 0) {
            if (zero_k0 && cudaMemsetAsync(p.Y, 0, sizeof(float) * N * p.M, s) != cudaSuccess)
                return GQ_ERR_CUDA;
            continue;
        }
        const gq::MatProblem mp{static_cast<const uint8_t*>(p.W_blocks), p.X, p.Y, p.M, p.K};
        if (gq::gemm_eligible(t, mp, N)) {
            plan->gemm[plan->n_gemm++] = mp;
            gemm_max = std::max(gemm_max, static_cast<size_t>(gq::gemm_workspace_bytes(p.K, N)));
        } else if (gq::gemv_tc_eligible(t, mp, N)) {
            plan->tc[plan->n_tc++] = mp;
        } else {
            plan->cc[plan->n_cc++] = mp;
        }
    }
    const size_t tc_sum =
        plan->n_tc ? static_cast<size_t>(gq::gemv_tc_workspace_bytes(t, plan->tc, plan->n_tc, N)) : 0;
    plan->ws_bytes = std::max(gemm_max, tc_sum);
    return GQ_OK;
}

// GEMM problems run one after another, then one grouped tensor-core decode launch, then
// one CUDA-core decode launch; all on `s`, all sharing workspace `ws` in stream order.
gq_status run_batch(gq_type t, int64_t N, BatchPlan* plan, void* ws, size_t ws_bytes,
                    cudaStream_t s) {
    if (plan->ws_bytes > 0) {
        if (ws == nullptr) {
            if (internal_workspace(s, plan->ws_bytes, &ws) != cudaSuccess) return GQ_ERR_CUDA;
            ws_bytes = plan->ws_bytes;
        } else if (ws_bytes < plan->ws_bytes || !aligned(ws, 256)) {
            return ws_bytes < plan->ws_bytes ? GQ_ERR_SHAPE : GQ_ERR_ALIGN;
        }
    }
    for (int i = 0; i < plan->n_gemm; ++i) {
        gq_status st = from_cuda(
            gq::launch_gemm(t, plan->gemm[i], N, ws, static_cast<int64_t>(ws_bytes), s));
        if (st != GQ_OK) return st;
    }
    if (plan->n_tc > 0) {
        gq_status st = from_cuda(gq::launch_gemv_tc(t, plan->tc, plan->n_tc, N, ws, s));
        if (st != GQ_OK) return st;
    }
    if (plan->n_cc > 0) return from_cuda(gq::launch_mul_mat(t, plan->cc, plan->n_cc, N, s));
    return GQ_OK;
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

// Checks one quantized-activation problem; on success *run tells whether it has work
// (M, N, K all > 0). K == 0 problems get Y zeroed on the stream when `zero_k0`.
gq_status check_q8x(const void* W, gq_type t, int64_t M, int64_t K, const float* X, int64_t N,
                    float* Y, cudaStream_t s, bool zero_k0, bool* run) {
    bool empty = false;
    *run = false;
    if (t == GQ_TYPE_Q4_K) return GQ_ERR_TYPE;   // Q8_0 activation blocks pair with 32-weight blocks
    gq_status st = check_problem(W, t, M, K, X, N, Y, &empty);
    if (st != GQ_OK || empty) return st;
    if (K == 0) {
        if (zero_k0 && cudaMemsetAsync(Y, 0, sizeof(float) * N * M, s) != cudaSuccess)
            return GQ_ERR_CUDA;
        return GQ_OK;
    }
    if (!aligned(X, 16)) return GQ_ERR_ALIGN;
    const gq::MatProblem p{static_cast<const uint8_t*>(W), X, Y, M, K};
    if (K % 256 != 0 || !gq::q8x_eligible(t, p)) return GQ_ERR_SHAPE;
    *run = true;
    return GQ_OK;
}

}  // namespace

extern "C" {

gq_status gq_mul_mat_rmsnorm(const void* W_blocks, gq_type t, int64_t M, int64_t K,
                             const float* X, const float* gamma, float eps, int64_t N,
                             float* Y, void* stream) {
    bool empty = false;
    gq_status st = check_problem(W_blocks, t, M, K, X, N, Y, &empty);
    if (st != GQ_OK) return st;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return GQ_ERR_SHAPE;
    if (empty) return GQ_OK;
    if (K == 0) return GQ_ERR_SHAPE;   // the mean over no elements is undefined
    if (!gamma) return GQ_ERR_NULL;
    if (!aligned(gamma, 4)) return GQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gq::MatProblem p{static_cast<const uint8_t*>(W_blocks), X, Y, M, K};
    p.gamma = gamma;
    p.eps = eps;
    if (N <= 2 && gq::fused_decode_eligible(t, p))   // normalized inside the decode kernel
        return from_cuda(gq::launch_mul_mat_fused(t, p, N, s));
    // Otherwise: Xhat = RMSNorm(X) into library workspace, then the plain product on it.
    const size_t xb = (static_cast<size_t>(N * K) * 4 + 255) / 256 * 256;
    const size_t down = gq_mul_mat_workspace_size(t, M, K, N);
    void* w = nullptr;
    if (internal_workspace(s, xb + down, &w) != cudaSuccess) return GQ_ERR_CUDA;
    float* xhat = static_cast<float*>(w);
    cudaError_t e = gq::launch_rmsnorm_x(X, gamma, eps, N, K, xhat, s);
    if (e != cudaSuccess) return GQ_ERR_CUDA;
    const gq::MatProblem q{static_cast<const uint8_t*>(W_blocks), xhat, Y, M, K};
    return run_one(t, q, N, static_cast<uint8_t*>(w) + xb, down, s);
}

gq_status gq_mul_mat_swiglu(const void* W_gate, const void* W_up, gq_type t, int64_t M,
                            int64_t K, const float* X, int64_t N, float* H, void* stream) {
    bool empty = false;
    gq_status st = check_problem(W_gate, t, M, K, X, N, H, &empty);
    if (st != GQ_OK || empty) return st;
    if (K > 0 && !W_up) return GQ_ERR_NULL;
    if (K > 0 && !aligned(W_up, 16)) return GQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(H, 0, sizeof(float) * N * M, s));   // Swish(0) * 0
    gq::MatProblem p{static_cast<const uint8_t*>(W_gate), X, H, M, K};
    p.W2 = static_cast<const uint8_t*>(W_up);
    if (N <= 2 && gq::fused_decode_eligible(t, p))   // gate/up row pairs in the decode kernel
        return from_cuda(gq::launch_mul_mat_fused(t, p, N, s));
    // Otherwise: G and U into library workspace by two plain products, then Swish(G) * U.
    const size_t yb = (static_cast<size_t>(N * M) * 4 + 255) / 256 * 256;
    const size_t down = gq_mul_mat_workspace_size(t, M, K, N);
    void* w = nullptr;
    if (internal_workspace(s, 2 * yb + down, &w) != cudaSuccess) return GQ_ERR_CUDA;
    float* G = static_cast<float*>(w);
    float* U = reinterpret_cast<float*>(static_cast<uint8_t*>(w) + yb);
    void* dws = static_cast<uint8_t*>(w) + 2 * yb;
    const gq::MatProblem pg{static_cast<const uint8_t*>(W_gate), X, G, M, K};
    const gq::MatProblem pu{static_cast<const uint8_t*>(W_up), X, U, M, K};
    st = run_one(t, pg, N, dws, down, s);
    if (st == GQ_OK) st = run_one(t, pu, N, dws, down, s);
    if (st != GQ_OK) return st;
    return from_cuda(gq::launch_swiglu(G, U, H, N * M, s));
}

gq_status gq_mul_mat_q8x(const void* W_blocks, gq_type t, int64_t M, int64_t K, const float* X,
                         int64_t N, float* Y, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool run = false;
    gq_status st = check_q8x(W_blocks, t, M, K, X, N, Y, s, true, &run);
    if (st != GQ_OK || !run) return st;
    const gq::MatProblem p{static_cast<const uint8_t*>(W_blocks), X, Y, M, K};
    return from_cuda(gq::launch_mul_mat_q8x(t, &p, 1, N, s));
}

gq_status gq_mul_mat_q8x_batched(const gq_mul_mat_problem* problems, int32_t count, gq_type t,
                                 int64_t N, void* stream) {
    if (count < 0 || count > GQ_MAX_BATCH) return GQ_ERR_SHAPE;
    if (!known_type(t) || t == GQ_TYPE_Q4_K) return GQ_ERR_TYPE;
    if (count == 0) return GQ_OK;
    if (!problems) return GQ_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool run = false;
    for (int i = 0; i < count; ++i) {   // every argument check before any work is queued
        const gq_mul_mat_problem& p = problems[i];
        gq_status st = check_q8x(p.W_blocks, t, p.M, p.K, p.X, N, p.Y, s, false, &run);
        if (st != GQ_OK) return st;
    }
    gq::MatProblem runs[GQ_MAX_BATCH];
    int n = 0;
    for (int i = 0; i < count; ++i) {
        const gq_mul_mat_problem& p = problems[i];
        gq_status st = check_q8x(p.W_blocks, t, p.M, p.K, p.X, N, p.Y, s, true, &run);
        if (st != GQ_OK) return st;
        if (run) runs[n++] = {static_cast<const uint8_t*>(p.W_blocks), p.X, p.Y, p.M, p.K};
    }
    if (n == 0) return GQ_OK;
    return from_cuda(gq::launch_mul_mat_q8x(t, runs, n, N, s));
}

gq_status gq_mul_mat_batched(const gq_mul_mat_problem* problems, int32_t count, gq_type t,
                             int64_t N, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    BatchPlan plan;
    gq_status st = plan_batch(problems, count, t, N, &plan, s, true);
    if (st != GQ_OK) return st;
    return run_batch(t, N, &plan, nullptr, 0, s);
}

size_t gq_mul_mat_batched_workspace_size(const gq_mul_mat_problem* problems, int32_t count,
                                         gq_type t, int64_t N) {
    BatchPlan plan;
    if (plan_batch(problems, count, t, N, &plan, nullptr, false) != GQ_OK) return 0;
    return plan.ws_bytes;
}

gq_status gq_mul_mat_batched_ws(const gq_mul_mat_problem* problems, int32_t count, gq_type t,
                                int64_t N, void* workspace, size_t workspace_bytes,
                                void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    BatchPlan plan;
    gq_status st = plan_batch(problems, count, t, N, &plan, s, true);
    if (st != GQ_OK) return st;
    if (plan.ws_bytes > 0 && workspace == nullptr) return GQ_ERR_NULL;
    return run_batch(t, N, &plan, workspace, workspace_bytes, s);
}

gq_status gq_get_last_error(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GQ_ERR_CUDA;
    gq::DeviceInfo* info = nullptr;
    if (gq::current_device_info(&info) != cudaSuccess) return GQ_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, info->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GQ_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(info->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return GQ_ERR_CUDA;
        return GQ_ERR_TIMEOUT;
    }
    return GQ_OK;
}

const char* gq_status_string(gq_status s) {
    switch (s) {
        case GQ_OK: return "ok";
        case GQ_ERR_NULL: return "a required pointer is NULL";
        case GQ_ERR_SHAPE:
            return "invalid shape (negative, K not a multiple of the block, too large)";
        case GQ_ERR_TYPE: return "unknown block type, or one this entry point does not take";
        case GQ_ERR_ALIGN: return "misaligned pointer (blocks need 16 bytes, fp32 arrays 4)";
        case GQ_ERR_CUDA: return "CUDA runtime error";
        case GQ_ERR_TIMEOUT: return "a device-side wait ran out of time";
        case GQ_ERR_FORMAT: return "not a GGUF file, or a malformed or truncated one";
        case GQ_ERR_IO: return "the file could not be opened or mapped";
    }
    return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Self-test of the bounded-wait machinery: one thread waits on an mbarrier that nothing
// ever arrives on, with the given limit, through the same mbar_wait / report_status the
// streaming and tensor-core kernels use. The kernel returns normally; the host sees
// GQ_ERR_TIMEOUT from gq_get_last_error and the context stays usable.
// ---------------------------------------------------------------------------------------
namespace gq {
namespace {
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, unsigned* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t a = smem_addr(&bar);
    mbar_init(a, 1);
    fence_mbar_init();
    if (!mbar_wait(a, 0, limit_ns)) report_status(status, kStatusTimeout);
}
}  // namespace
}  // namespace gq

extern "C" gq_status gq_selftest_wait_timeout(int64_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 10000000) return GQ_ERR_SHAPE;
    gq::DeviceInfo* info = nullptr;
    if (gq::current_device_info(&info) != cudaSuccess) return GQ_ERR_CUDA;
    gq::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(limit_us) * 1000ull, info->status);
    return from_cuda(cudaGetLastError());
}
