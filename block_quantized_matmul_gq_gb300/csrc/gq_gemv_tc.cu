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
// sequence and each persistent CTA (one per SM) takes a contiguous share of about equal
// bytes, cut at 128-row tile boundaries, walked tile by tile over the whole of K:
//   warp 0       producer: per 256-k super-step one "raw stage" holding the tile's raw
//                blocks (one 2-D TMA copy through the problem's tensor map: 128 rows x
//                144 / 272 bytes) and the super-step's bf16 X (one 1-D bulk copy of four
//                kNPad x 64 tiles; X was pre-arranged into swizzled tiles by x_tiles_kernel).
//                The ring of raw stages is as deep as shared memory allows, because the
//                weight bytes in flight per SM decide the bandwidth; a stage is free again
//                once the dequantize warps have read its rows and the MMAs have read its X.
//   warp 1       TMEM owner and MMA issuer (one thread); two accumulators of kNPad columns
//                so a tile's epilogue overlaps the next tile's stream.
//   warps 2..9   dequantize rows to 128-byte-swizzled bf16 (shared with the prefill GEMM).
//   warps 10..13 epilogue: TMEM -> registers -> Y (one TMEM lane quadrant each).
// All waits are bounded: a CTA that gives up records a timeout in the status word, lets
// its copies and MMAs land, frees its TMEM and leaves.
#include <cuda.h>   // CUtensorMap and its enums (header only; no libcuda link)
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "gq_dequant.cuh"
#include "gq_device.cuh"
#include "gq_internal.h"
#include "gq_umma.cuh"

namespace gq {
namespace {

using namespace dq;

constexpr int kBM = 128;
constexpr int kBK = 64;                   // width of one pre-arranged X tile
constexpr int kSuperK = 256;              // k per raw stage
constexpr int kHalfK = 128;               // k per A slot (one dequantize group's half)
constexpr int kDequantWarps = 8;          // two groups of four warps (all 128 rows each)
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * (kDequantWarps + kEpiWarps);   // 448
constexpr int kGroupSlots = 3;            // A slots in TMEM per dequantize group
constexpr int kAccCols = 128;             // TMEM columns [0, 128): two accumulators
constexpr int kSlotCols = kHalfK / 2;     // 64 columns: 128 bf16 per lane
constexpr int kTmemCols = 512;            // accumulators + 2 x 3 A slots
constexpr int kSmemLimit = 232448;        // opt-in dynamic shared memory per CTA
constexpr unsigned long long kDrainNs = 100000000ull;
static_assert(kAccCols + 2 * kGroupSlots * kSlotCols <= kTmemCols, "TMEM budget");

template <int kType, int kNPad>
struct TcLayout {
    static constexpr int kB = kNPad * kBK * 2;              // one 64-k X tile: 2 / 4 / 8 KB
    static constexpr int kRawRow = RawFmt<kType>::kRow;     // 144 / 272
    static constexpr int kRaw = kBM * kRawRow;              // 18 / 34 KB of raw blocks
    static constexpr int kStage = kRaw + 4 * kB;            // raw blocks + the super-step's X
    static constexpr int kOffRaw = 0;
    static constexpr int kFixed = 1024 + 256;               // alignment slack, barriers, slot
    static constexpr int kRawFit = (kSmemLimit - kFixed) / kStage;
    static constexpr int kRawStages = kRawFit > 8 ? 8 : kRawFit;
    static constexpr int kOffBar = kOffRaw + kRawStages * kStage;
    // raw_full[R], raw_empty[R], a_full[2][G], a_empty[2][G], acc_full[2], acc_empty[2],
    // mma_done
    static constexpr int kNumBars = 2 * kRawStages + 4 * kGroupSlots + 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kB % 1024 == 0 && kRaw % 1024 == 0, "1 KB aligned tiles");
    static_assert(kRawStages >= 2 && kAlloc <= kSmemLimit, "shared memory budget");
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

// Largest number of problems one launch takes: the tensor maps and the problem table
// travel as kernel parameters (128 x (128 + 64) bytes here).
constexpr int kMaxLaunchProbs = 128;

template <int kMaxProbs>
struct TcParams {
    CUtensorMap maps[kMaxProbs];   // raw weight bytes per problem: rows x row bytes
    int32_t count;
    int32_t n_tok;
    int64_t total_bytes;
    unsigned* status;
    TcProb p[kMaxProbs];
};

// First tile start (problem p, row r, r a multiple of 128) at or after byte `byte` of the
// launch's row sequence; (count, 0) = end.
template <int kMaxProbs>
__device__ void tc_row_at_byte(const TcParams<kMaxProbs>& P, int64_t byte, int& p, int64_t& r) {
    p = 0;
    while (p + 1 < P.count && P.p[p + 1].byte_begin <= byte) ++p;
    const int64_t off = byte - P.p[p].byte_begin;
    const int64_t tile_bytes = P.p[p].row_bytes * kBM;
    r = off <= 0 ? 0 : (off + tile_bytes - 1) / tile_bytes * kBM;
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

// One dequantize group's half of a row's raw super-step (kWords 32-bit words) from shared
// memory. The half starts 16-byte aligned (kG = 0) or 8 bytes past (kG = 1): one 8-byte
// load at the unaligned end, 16-byte loads for the rest, which a quarter warp serves
// without bank conflicts at the 144 / 272-byte row pitch.
template <int kG, int kWords>
__device__ __forceinline__ void load_half_row(const uint8_t* src, uint32_t (&raw)[kWords]) {
    constexpr int w8 = kG == 0 ? kWords - 2 : 0;
    constexpr int w16 = kG == 0 ? 0 : 2;
    const uint2 e = *reinterpret_cast<const uint2*>(src + 4 * w8);
    raw[w8] = e.x;
    raw[w8 + 1] = e.y;
#pragma unroll
    for (int i = 0; i < (kWords - 2) / 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 4 * w16 + 16 * i);
        raw[w16 + 4 * i] = v.x;
        raw[w16 + 4 * i + 1] = v.y;
        raw[w16 + 4 * i + 2] = v.z;
        raw[w16 + 4 * i + 3] = v.w;
    }
}

template <int kType, int kNPad, int kMaxProbs>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ TcParams<kMaxProbs> P) {
    using L = TcLayout<kType, kNPad>;
    constexpr int R = L::kRawStages;
    constexpr int G = kGroupSlots;
    constexpr int kHalfWords = L::kRawRow / 8;   // one group's half of a row: 18 / 34 words
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t sRaw = base_addr + L::kOffRaw;   // stage r: raw at r * kStage, X after it
    const uint32_t bar0 = base_addr + L::kOffBar;
    auto raw_full = [&](int r) { return bar0 + 8u * r; };
    auto raw_empty = [&](int r) { return bar0 + 8u * (R + r); };
    auto a_full = [&](int g, int i) { return bar0 + 8u * (2 * R + g * G + i); };
    auto a_empty = [&](int g, int i) { return bar0 + 8u * (2 * R + 2 * G + g * G + i); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * R + 4 * G + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (2 * R + 4 * G + 2 + b); };
    const uint32_t mma_done = bar0 + 8u * (2 * R + 4 * G + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(raw_full(r), 1);
            // every dequantize thread once its half row is in registers, and the MMA
            // issuer's commit once the super-step's MMAs (the readers of its X) completed
            mbar_init(raw_empty(r), 32 * kDequantWarps + 1);
        }
        for (int g = 0; g < 2; ++g)
            for (int i = 0; i < G; ++i) {
                mbar_init(a_full(g, i), 32 * kDequantWarps / 2);
                mbar_init(a_empty(g, i), 1);
            }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 32 * kEpiWarps);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
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
        int raw_n = 0;
        bool ok = true;
        for (; w.valid; tc_walk_next(P, w, p1, r1), ++raw_n) {
            const int r = raw_n % R;
            if (!mbar_wait(raw_empty(r), ((raw_n / R) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = sRaw + r * L::kStage;
                mbar_arrive_expect_tx(raw_full(r), L::kStage);
                // Whole 128-row box; rows past the matrix end are filled with zeros.
                tma_load_2d(dst, &P.maps[w.p], w.j * (L::kRawRow / RawFmt<kType>::kElem),
                            static_cast<int>(w.row0), raw_full(r));
                bulk_g2s(dst + L::kRaw, P.p[w.p].Xt + static_cast<int64_t>(w.j) * 4 * L::kB,
                         4 * L::kB, raw_full(r));
            }
            __syncwarp();
        }
        if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
        if (lane == 0) {
            for (int i = max(0, raw_n - R); i < raw_n; ++i)
                mbar_wait(raw_full(i % R), (i / R) & 1, kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kNPad);
            int tile = 0, raw_n = 0;
            bool ok = true;
            for (; w.valid && ok; tc_walk_next(P, w, p1, r1), ++raw_n) {
                const int b = tile & 1;
                if (w.j == 0) {
                    if (!mbar_wait(acc_empty(b), ((tile >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const int r = raw_n % R;
                if (!mbar_wait(raw_full(r), (raw_n / R) & 1)) {   // the super-step's X landed
                    ok = false;
                    break;
                }
                const uint32_t sX = sRaw + r * L::kStage + L::kRaw;
                const int gi = raw_n % G;
                for (int g = 0; g < 2; ++g) {
                    if (!mbar_wait(a_full(g, gi), (raw_n / G) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_col = tmem + kAccCols + (g * G + gi) * kSlotCols;
#pragma unroll
                    for (int kk = 0; kk < kHalfK / 16; ++kk) {
                        // k = 128 g + 16 kk: X tile 2 g + kk / 4, 32 bytes per 16 k inside it
                        const uint64_t bdesc =
                            sw128_kmajor_desc(sX + (2 * g + kk / 4) * L::kB + (kk % 4) * 32);
                        umma_bf16_tmem_a(tmem + b * kNPad, a_col + kk * 8, bdesc, idesc,
                                         (w.j | g | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(a_empty(g, gi));
                }
                if (!ok) break;
                umma_commit(raw_empty(r));
                if (w.j == w.nsuper - 1) {
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
        // Group g (warps 2..5 or 6..9) takes k [128 g, 128 g + 128) of every super-step for
        // all 128 rows; each warp its TMEM lane quadrant 32 * (warp % 4) + i, one row per
        // thread, written to the group's A slot with tcgen05.st.
        const int g = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kAccCols;
        int raw_n = 0;
        bool ok = true;
        uint32_t raw[kHalfWords];
        for (; w.valid && ok; tc_walk_next(P, w, p1, r1), ++raw_n) {
            const int r = raw_n % R;
            if (!mbar_wait(raw_full(r), (raw_n / R) & 1)) {
                ok = false;
                break;
            }
            // Every row of the box is loaded; rows past the matrix end arrive as zeros and
            // dequantize to zero operands (their outputs are dropped).
            {
                const uint8_t* src = base + L::kOffRaw + r * L::kStage + row * L::kRawRow +
                                     g * (L::kRawRow / 2);
                if (g == 0)
                    load_half_row<0>(src, raw);
                else
                    load_half_row<1>(src, raw);
                uint32_t dep = 0;
#pragma unroll
                for (int i = 0; i < kHalfWords; ++i) dep ^= raw[i];
                release_to_async_proxy(dep);
            }
            mbar_arrive(raw_empty(r));
            const int gi = raw_n % G;
            if (!mbar_wait(a_empty(g, gi), ((raw_n / G) & 1) ^ 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_slot = a_lane + (g * G + gi) * kSlotCols;
            {
                uint32_t packed[16];
                dequant_block<kType, 0>(raw, packed);
                tmem_st16(a_slot, packed);
            }
            {
                uint32_t packed[16];
                dequant_block<kType, 1>(raw, packed);
                tmem_st16(a_slot + 16, packed);
            }
            {
                uint32_t packed[16];
                dequant_block<kType, 2>(raw, packed);
                tmem_st16(a_slot + 32, packed);
            }
            {
                uint32_t packed[16];
                dequant_block<kType, 3>(raw, packed);
                tmem_st16(a_slot + 48, packed);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(a_full(g, gi));
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
        tmem_dealloc(tmem, kTmemCols);
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

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map over a weight matrix's raw block bytes (rows x row bytes, 128-row x 256-k
// boxes). Weights do not move between decode steps, so maps are cached by
// (address, rows, K, type); the cache is bounded and simply cleared when full.
template <int kType>
cudaError_t weight_map(const uint8_t* W, int64_t M, int64_t K, CUtensorMap* out) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int64_t, int64_t>, CUtensorMap> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(static_cast<const void*>(W), M, K);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    constexpr int kElem = RawFmt<kType>::kElem;
    const int64_t row_bytes = (K / 32) * RawFmt<kType>::kBB;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / kElem), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(RawFmt<kType>::kRow / kElem),
                               static_cast<cuuint32_t>(kBM)};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap m{};
    CUresult r = enc(&m, kElem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                     2, const_cast<uint8_t*>(W), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (cache.size() >= 4096) cache.clear();
    cache.emplace(key, m);
    *out = m;
    return cudaSuccess;
}

int npad_for(int64_t N) { return N <= 16 ? 16 : (N <= 32 ? 32 : 64); }

template <int kType, int kNPad, int kMaxProbs>
cudaError_t launch_tc_t(const MatProblem* probs, int count, int64_t N, uint8_t* ws,
                        const DeviceInfo* info, cudaStream_t s) {
    using L = TcLayout<kType, kNPad>;
    static_assert(sizeof(TcParams<kMaxProbs>) <= 32000, "kernel parameter space");
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
        cudaError_t e = weight_map<kType>(probs[i].W, probs[i].M, probs[i].K, &P.maps[i]);
        if (e != cudaSuccess) return e;
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

template <int kType>
cudaError_t launch_tc_type(const MatProblem* probs, int count, int64_t N, uint8_t* ws,
                           const DeviceInfo* info, cudaStream_t s) {
    if (count == 1) return launch_tc_np<kType, 1>(probs, count, N, ws, info, s);
    if (count <= 16) return launch_tc_np<kType, 16>(probs, count, N, ws, info, s);
    return launch_tc_np<kType, kMaxLaunchProbs>(probs, count, N, ws, info, s);
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
    // Launches of at most kMaxLaunchProbs problems; their X tiles sit one after another.
    for (int i0 = 0; i0 < count; i0 += kMaxLaunchProbs) {
        const int n = std::min(kMaxLaunchProbs, count - i0);
        e = t == GQ_TYPE_Q4_0 ? launch_tc_type<GQ_TYPE_Q4_0>(probs + i0, n, N, ws, info, s)
                              : launch_tc_type<GQ_TYPE_Q8_0>(probs + i0, n, N, ws, info, s);
        if (e != cudaSuccess) return e;
        ws += gemv_tc_workspace_bytes(probs + i0, n, N);
    }
    return cudaSuccess;
}

}  // namespace gq
