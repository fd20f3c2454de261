// gq_gemv_tc.cu -- decode mul_mat for 5..64 tokens on the tensor cores:
//     Y[n][m] = sum_k What[m][k] * X[n][k]
//
// Small-batch decode still streams every weight once, so it stays bound by memory
// bandwidth ("A Complete Guide to llama.cpp and Customization with C++", section 2.1;
// "No Python! Building an AI Inference Engine Exclusively in C++", section 9), but with
// more than a few tokens the multiply-adds no longer fit the CUDA cores at HBM speed. Here
// the dequantized weights ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using
// C++", section 6.2) go through tcgen05.mma instead: M = 128 weight rows, N = kNPad tokens
// (16, 32 or 64; extra tokens are zero), K = 16 per instruction, fp32 in TMEM.
//
// Work is split like the CUDA-core decode kernel: all problems of a launch form one row
// sequence and each persistent CTA (one per SM) takes a contiguous, row-aligned share of
// equal bytes, walked as 128-row tiles over the whole of K:
//   warp 0       producer: the tile rows' raw blocks for one 256-k super-step (one 1-D
//                bulk copy per row, 144 / 272 bytes), and per 64-k stage the stage's
//                bf16 X tile (one 1-D bulk copy: X was pre-arranged into swizzled
//                kNPad x 64 tiles by x_tiles_kernel).
//   warp 1       TMEM owner and MMA issuer (one thread); two accumulators of kNPad columns
//                so a tile's epilogue overlaps the next tile's stream.
//   warps 2..9   dequantize rows to 128-byte-swizzled bf16 (shared with the prefill GEMM).
//   warps 10..13 epilogue: TMEM -> registers -> Y (one TMEM lane quadrant each).
// All waits are bounded: a CTA that gives up records a timeout in the status word, lets
// its copies and MMAs land, frees its TMEM and leaves.
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "gq_dequant.cuh"
#include "gq_device.cuh"
#include "gq_internal.h"
#include "gq_umma.cuh"

namespace gq {
namespace {

using namespace dq;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kSuperK = 256;
constexpr int kDequantWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * (kDequantWarps + kEpiWarps);   // 448
constexpr int kStages = 4;
constexpr int kRawStages = 3;
constexpr unsigned long long kDrainNs = 100000000ull;

template <int kType, int kNPad>
struct TcLayout {
    static constexpr int kA = kBM * kBK * 2;                // 16 KB
    static constexpr int kB = kNPad * kBK * 2;              // 2 / 4 / 8 KB
    static constexpr int kRawRow = RawFmt<kType>::kRow;     // 144 / 272
    static constexpr int kRaw = kBM * kRawRow;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kA;
    static constexpr int kOffRaw = kOffB + kStages * kB;
    static constexpr int kOffBar = kOffRaw + kRawStages * kRaw;
    // a_full[S], b_full[S], empty[S], raw_full[R], raw_empty[R], acc_full[2], acc_empty[2],
    // mma_done
    static constexpr int kNumBars = 3 * kStages + 2 * kRawStages + 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr int kTmemCols = 2 * kNPad < 32 ? 32 : 2 * kNPad;
    static_assert(kA % 1024 == 0 && kB % 1024 == 0 && kRaw % 1024 == 0, "1 KB aligned stages");
};

struct TcProb {
    const uint8_t* W;
    const float* X;       // n_tok x K fp32 activations
    const uint8_t* Xt;    // pre-arranged bf16 X tiles: K/64 tiles of kNPad x 128 bytes
    float* Y;
    int64_t M;
    int64_t row_bytes;
    int64_t byte_begin;
    int32_t K;
    int32_t pad_;
};

template <int kMaxProbs>
struct TcParams {
    int32_t count;
    int32_t n_tok;
    int64_t total_bytes;
    unsigned* status;
    TcProb p[kMaxProbs];
};

// First row (problem p, row r) whose first byte is at or after `byte`; (count, 0) = end.
template <int kMaxProbs>
__device__ void tc_row_at_byte(const TcParams<kMaxProbs>& P, int64_t byte, int& p, int64_t& r) {
    p = 0;
    while (p + 1 < P.count && P.p[p + 1].byte_begin <= byte) ++p;
    const int64_t off = byte - P.p[p].byte_begin;
    r = off <= 0 ? 0 : (off + P.p[p].row_bytes - 1) / P.p[p].row_bytes;
    if (r >= P.p[p].M) {
        ++p;
        r = 0;
    }
}

// Walk of one CTA's share, one 256-k super-step at a time: problem p, tile rows
// [row0, row0 + rows), super-step j of nsuper. Every role walks the same sequence.
struct TcWalk {
    int p;
    int64_t row0, re;     // tile start, end of this problem's part of the share
    int rows;
    int j, nsuper;
    bool valid;
};

template <int kMaxProbs>
__device__ void tc_walk_open(const TcParams<kMaxProbs>& P, TcWalk& w, int p, int64_t rb,
                             int p_end, int64_t r_end) {
    for (; p < P.count && p <= p_end; ++p, rb = 0) {
        const int64_t re = (p == p_end) ? r_end : P.p[p].M;
        if (re > rb) {
            w.p = p;
            w.row0 = rb;
            w.re = re;
            w.rows = static_cast<int>(min(static_cast<int64_t>(kBM), re - rb));
            w.j = 0;
            w.nsuper = P.p[p].K / kSuperK;
            w.valid = true;
            return;
        }
    }
    w.valid = false;
}

template <int kMaxProbs>
__device__ void tc_walk_next(const TcParams<kMaxProbs>& P, TcWalk& w, int p_end, int64_t r_end) {
    if (++w.j < w.nsuper) return;
    w.j = 0;
    w.row0 += kBM;
    if (w.row0 < w.re) {
        w.rows = static_cast<int>(min(static_cast<int64_t>(kBM), w.re - w.row0));
        return;
    }
    tc_walk_open(P, w, w.p + 1, 0, p_end, r_end);
}

template <int kType, int kNPad, int kMaxProbs>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ TcParams<kMaxProbs> P) {
    using L = TcLayout<kType, kNPad>;
    constexpr int S = kStages;
    constexpr int R = kRawStages;
    constexpr int kRawWords = L::kRawRow / 4;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t sA = base_addr + L::kOffA;
    const uint32_t sB = base_addr + L::kOffB;
    const uint32_t sRaw = base_addr + L::kOffRaw;
    const uint32_t bar0 = base_addr + L::kOffBar;
    auto a_full = [&](int s) { return bar0 + 8u * s; };
    auto b_full = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto raw_full = [&](int r) { return bar0 + 8u * (3 * S + r); };
    auto raw_empty = [&](int r) { return bar0 + 8u * (3 * S + R + r); };
    auto acc_full = [&](int b) { return bar0 + 8u * (3 * S + 2 * R + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 * R + 2 + b); };
    const uint32_t mma_done = bar0 + 8u * (3 * S + 2 * R + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(a_full(s), 32 * kDequantWarps);
            mbar_init(b_full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), 32 * kDequantWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 32 * kEpiWarps);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int p0, p1;
    int64_t r0, r1;
    tc_row_at_byte(P, P.total_bytes * blockIdx.x / gridDim.x, p0, r0);
    tc_row_at_byte(P, P.total_bytes * (blockIdx.x + 1) / gridDim.x, p1, r1);
    TcWalk w;
    tc_walk_open(P, w, p0, r0, p1, r1);

    if (warp == 0) {
        // ---------------- producer (whole warp; lane 0 arms the barriers) ----------------
        int raw_n = 0, ks = 0;
        bool ok = true;
        for (; w.valid && ok; tc_walk_next(P, w, p1, r1)) {
            const TcProb& pr = P.p[w.p];
            const int r = raw_n % R;
            if (!mbar_wait(raw_empty(r), ((raw_n / R) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(raw_full(r), L::kRawRow * w.rows);
            __syncwarp();
            const uint8_t* src = pr.W + w.row0 * pr.row_bytes + static_cast<int64_t>(w.j) * L::kRawRow;
            for (int row = lane; row < w.rows; row += 32)
                bulk_g2s_evict_first(sRaw + r * L::kRaw + row * L::kRawRow, src + row * pr.row_bytes,
                                     L::kRawRow, raw_full(r));
            ++raw_n;
            for (int q = 0; q < kSuperK / kBK; ++q, ++ks) {
                const int s = ks % S;
                if (!mbar_wait(empty(s), ((ks / S) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(b_full(s), L::kB);
                    bulk_g2s(sB + s * L::kB, pr.Xt + static_cast<int64_t>(4 * w.j + q) * L::kB,
                             L::kB, b_full(s));
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
        if (lane == 0) {
            for (int i = max(0, ks - S); i < ks; ++i)
                mbar_wait(b_full(i % S), (i / S) & 1, kDrainNs);
            for (int i = max(0, raw_n - R); i < raw_n; ++i)
                mbar_wait(raw_full(i % R), (i / R) & 1, kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kNPad);
            int ks = 0, tile = 0;
            bool ok = true;
            for (; w.valid && ok; tc_walk_next(P, w, p1, r1)) {
                const int b = tile & 1;
                if (w.j == 0) {
                    if (!mbar_wait(acc_empty(b), ((tile >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                for (int q = 0; q < kSuperK / kBK; ++q, ++ks) {
                    const int s = ks % S;
                    const uint32_t ph = (ks / S) & 1;
                    if (!mbar_wait(a_full(s), ph) || !mbar_wait(b_full(s), ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc = sw128_kmajor_desc(sA + s * L::kA + kk * 32);
                        const uint64_t bdesc = sw128_kmajor_desc(sB + s * L::kB + kk * 32);
                        umma_bf16(tmem + b * kNPad, adesc, bdesc, idesc,
                                  (w.j | q | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty(s));
                }
                if (ok && w.j == w.nsuper - 1) {
                    umma_commit(acc_full(b));
                    ++tile;
                }
            }
            // Completes when every MMA issued has finished (also after a timeout), so the
            // TMEM release below never races an MMA in flight.
            umma_commit(mma_done);
            if (!ok) report_status(P.status, kStatusTimeout);
        }
    } else if (warp < 2 + kDequantWarps) {
        // ---------------- dequantize ----------------
        const int dw = warp - 2;
        const int quad = dw & 3;
        const int half = dw >> 2;
        const int row = quad * 32 + lane;
        int raw_n = 0, ks = 0;
        bool ok = true;
        uint32_t raw[kRawWords];
        for (; w.valid && ok; tc_walk_next(P, w, p1, r1)) {
            const int r = raw_n % R;
            if (!mbar_wait(raw_full(r), (raw_n / R) & 1)) {
                ok = false;
                break;
            }
            const bool live = row < w.rows;
            if (live) {
                const uint8_t* src = base + L::kOffRaw + r * L::kRaw + row * L::kRawRow;
#pragma unroll
                for (int i = 0; i < kRawWords / 4; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
                    raw[4 * i] = v.x;
                    raw[4 * i + 1] = v.y;
                    raw[4 * i + 2] = v.z;
                    raw[4 * i + 3] = v.w;
                }
            }
            mbar_arrive(raw_empty(r));
            ++raw_n;
#pragma unroll
            for (int q = 0; q < 4; ++q, ++ks) {
                const int s = ks % S;
                if (!mbar_wait(empty(s), ((ks / S) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                uint8_t* arow = base + L::kOffA + s * L::kA + row * 128;
                if (!live) {
                    // rows past the end of the part: zero operands (their outputs are dropped)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(arow + (((4 * half + c) ^ (row & 7)) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                } else if (half == 0) {
                    if (q == 0) dequant_store<kType, 0, 0>(raw, arow, row);
                    if (q == 1) dequant_store<kType, 1, 0>(raw, arow, row);
                    if (q == 2) dequant_store<kType, 2, 0>(raw, arow, row);
                    if (q == 3) dequant_store<kType, 3, 0>(raw, arow, row);
                } else {
                    if (q == 0) dequant_store<kType, 0, 1>(raw, arow, row);
                    if (q == 1) dequant_store<kType, 1, 1>(raw, arow, row);
                    if (q == 2) dequant_store<kType, 2, 1>(raw, arow, row);
                    if (q == 3) dequant_store<kType, 3, 1>(raw, arow, row);
                }
                fence_proxy_async_smem();
                mbar_arrive(a_full(s));
            }
        }
        if (!ok) report_status(P.status, kStatusTimeout);
    } else {
        // ---------------- epilogue ----------------
        // A warp may only touch the TMEM lanes of its own quadrant: 32 * (warp % 4) + i.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t tlane = static_cast<uint32_t>(quad * 32) << 16;
        int tile = 0;
        bool ok = true;
        for (; w.valid && ok; tc_walk_next(P, w, p1, r1)) {
            if (w.j != w.nsuper - 1) continue;   // act once per tile
            const int b = tile & 1;
            if (!mbar_wait(acc_full(b), (tile >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const TcProb& pr = P.p[w.p];
#pragma unroll
            for (int c = 0; c < kNPad; c += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + tlane + b * kNPad + c, v);
                if (row < w.rows) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int n = c + jj;
                        if (n < P.n_tok) pr.Y[n * pr.M + w.row0 + row] = __uint_as_float(v[jj]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(b));
            ++tile;
        }
        if (!ok) report_status(P.status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) mbar_wait(mma_done, 0, kDrainNs);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// X (n_tok x K fp32, rows of K) -> kNPad x 64 bf16 tiles per 64-k stage, each row 128 bytes
// with 16-byte chunk c stored at c ^ (row % 8); tokens >= n_tok are zero.
// grid.y = problem; each thread writes one 16-byte chunk.
template <int kNPad, int kMaxProbs>
__global__ void __launch_bounds__(256)
x_tiles_kernel(const __grid_constant__ TcParams<kMaxProbs> P) {
    const int p = blockIdx.y;
    const int K = P.p[p].K;
    const float* X = P.p[p].X;
    uint8_t* out = const_cast<uint8_t*>(P.p[p].Xt);
    const int64_t chunks = static_cast<int64_t>(K / kBK) * kNPad * 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < chunks;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i & 7);
        const int n = static_cast<int>((i >> 3) % kNPad);
        const int64_t ks = (i >> 3) / kNPad;
        float v[8];
        if (n < P.n_tok) {
            const float* x = X + static_cast<int64_t>(n) * K + ks * kBK + 8 * c;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = x[e];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
        }
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            packed[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(out + ks * (kNPad * 128) + n * 128 + ((c ^ (n & 7)) << 4)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

template <typename KernelT>
cudaError_t ensure_smem(KernelT kernel, int device, int64_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int64_t> set_bytes;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), device);
    auto it = set_bytes.find(key);
    if (it != set_bytes.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e == cudaSuccess) set_bytes[key] = bytes;
    return e;
}

int npad_for(int64_t N) { return N <= 16 ? 16 : (N <= 32 ? 32 : 64); }

template <int kType, int kNPad, int kMaxProbs>
cudaError_t launch_tc_t(const MatProblem* probs, int count, int64_t N, uint8_t* ws,
                        const DeviceInfo* info, cudaStream_t s) {
    using L = TcLayout<kType, kNPad>;
    TcParams<kMaxProbs> P{};
    P.count = count;
    P.n_tok = static_cast<int32_t>(N);
    P.status = info->status;
    int64_t bytes = 0, ws_off = 0;
    int64_t max_chunks = 0;
    for (int i = 0; i < count; ++i) {
        TcProb& g = P.p[i];
        g.W = probs[i].W;
        g.X = probs[i].X;
        g.Xt = ws + ws_off;
        g.Y = probs[i].Y;
        g.M = probs[i].M;
        g.K = static_cast<int32_t>(probs[i].K);
        g.row_bytes = (probs[i].K / 32) * RawFmt<kType>::kBB;
        g.byte_begin = bytes;
        bytes += g.M * g.row_bytes;
        ws_off += static_cast<int64_t>(kNPad) * probs[i].K * 2;
        max_chunks = std::max<int64_t>(max_chunks, probs[i].K / kBK * kNPad * 8);
    }
    P.total_bytes = bytes;
    const unsigned gx = static_cast<unsigned>(std::min<int64_t>((max_chunks + 255) / 256, 64));
    x_tiles_kernel<kNPad, kMaxProbs><<<dim3(gx, count), 256, 0, s>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kernel = gemv_tc_kernel<kType, kNPad, kMaxProbs>;
    e = ensure_smem(kernel, info->device, L::kAlloc);
    if (e != cudaSuccess) return e;
    int64_t grid = (bytes + 65535) / 65536;
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, info->sm_count));
    kernel<<<static_cast<int>(grid), kThreads, L::kAlloc, s>>>(P);
    return cudaGetLastError();
}

template <int kType, int kMaxProbs>
cudaError_t launch_tc_np(const MatProblem* probs, int count, int64_t N, uint8_t* ws,
                         const DeviceInfo* info, cudaStream_t s) {
    switch (npad_for(N)) {
        case 16: return launch_tc_t<kType, 16, kMaxProbs>(probs, count, N, ws, info, s);
        case 32: return launch_tc_t<kType, 32, kMaxProbs>(probs, count, N, ws, info, s);
        default: return launch_tc_t<kType, 64, kMaxProbs>(probs, count, N, ws, info, s);
    }
}

}  // namespace

bool gemv_tc_eligible(const MatProblem& p, int64_t N) {
    if (N < kGemvTcMinTokens || N > kGemvTcMaxTokens) return false;
    if (p.K % kSuperK != 0 || p.K > (int64_t(1) << 24) || p.M <= 0) return false;
    return reinterpret_cast<uintptr_t>(p.W) % 16 == 0 && reinterpret_cast<uintptr_t>(p.X) % 4 == 0;
}

int64_t gemv_tc_workspace_bytes(const MatProblem* probs, int count, int64_t N) {
    int64_t b = 0;
    for (int i = 0; i < count; ++i) b += static_cast<int64_t>(npad_for(N)) * probs[i].K * 2;
    return b;
}

cudaError_t launch_gemv_tc(gq_type t, const MatProblem* probs, int count, int64_t N,
                           void* workspace, cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (count == 1) {
        return t == GQ_TYPE_Q4_0 ? launch_tc_np<GQ_TYPE_Q4_0, 1>(probs, count, N, ws, info, s)
                                 : launch_tc_np<GQ_TYPE_Q8_0, 1>(probs, count, N, ws, info, s);
    }
    if (count <= 16) {
        return t == GQ_TYPE_Q4_0 ? launch_tc_np<GQ_TYPE_Q4_0, 16>(probs, count, N, ws, info, s)
                                 : launch_tc_np<GQ_TYPE_Q8_0, 16>(probs, count, N, ws, info, s);
    }
    return t == GQ_TYPE_Q4_0 ? launch_tc_np<GQ_TYPE_Q4_0, GQ_MAX_BATCH>(probs, count, N, ws, info, s)
                             : launch_tc_np<GQ_TYPE_Q8_0, GQ_MAX_BATCH>(probs, count, N, ws, info, s);
}

}  // namespace gq
