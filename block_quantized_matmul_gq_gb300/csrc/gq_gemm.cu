// gq_gemm.cu -- prefill mul_mat on the 5th-generation tensor cores:
//     Y[n][m] = sum_k What[m][k] * X[n][k]        (Y = X . What^T, fp32 out)
//
// At prefill the product is a dense contraction ("No Python! Building an AI Inference
// Engine Exclusively in C++", section 6: over 90% of inference compute is GEMM), so it
// runs on tcgen05 tensor cores with bf16 operands and fp32 accumulation in TMEM. The
// weights stay block-quantized in HBM and are dequantized inside the kernel right after
// they are loaded ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
// section 6.2; "No Python! ...", section 9).
//
// One CTA computes a 128 (weight rows) x kBN (tokens) tile of Y^T over all of K:
//   warp 0      TMA producer: raw weight blocks (2-D tensor map over the block bytes,
//               one 256-k "super-step" = 8 blocks per row per copy) and bf16 X tiles
//               (64 k x kBN tokens, 128-byte swizzle) into rings of shared-memory stages.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M=128, N=kBN, K=16),
//               four per 64-k stage, and commits each stage back to the producers. (The
//               512-token kernel has a second issuing warp, warp 10: one per token half.)
//   warps 2..9  dequantize: a thread owns one row and one of the two blocks of every 64-k
//               stage; it turns the block into 32 bf16 values, each (c - 8) * d (or c * d)
//               computed exactly in fp32 (packed f32x2 arithmetic) and rounded once to
//               bf16, and stores them in the 128-byte-swizzled K-major layout the MMA
//               reads. A Q4_K super-step is one super-block (144 bytes, as 8 Q4_0 blocks);
//               its "blocks" are the eight sub-blocks, each d sc q - dmin m. After the K loop the same warps read the accumulator out of TMEM
//               (tcgen05.ld; warp w owns lanes 32*(w%4).., half the token columns) and
//               write Y.
// Shapes whose 256-token tiles fill two or more waves use 512-token tiles instead
// (gemm_wide_kernel): each dequantized A stage feeds two N = 256 MMAs.
// With fewer tiles than half the SMs, a tile is shared by a cluster of 2 or 4 CTAs along
// grid z, each taking a contiguous share of K; each parks its fp32 partial in its own
// shared memory and, after a cluster barrier, sums a quarter (or half) of the tile's token
// columns over the cluster through distributed shared memory, in rank order, into Y.
// X is converted to bf16 once per call by x_to_bf16_kernel into caller- or library-owned
// workspace (N x K bf16), which the tensor map reads.
// All waits are bounded; a CTA that gives up sets the device status word, lets its own
// copies and MMAs land, frees its TMEM and leaves.
#include <cuda.h>            // CUtensorMap and its enums (header only; no libcuda link)
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

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // k per MMA stage: 128 bytes of bf16 = one swizzle row
constexpr int kSuperK = 256;      // k per raw-weight copy: 8 blocks per row
constexpr int kDequantWarps = 8;  // two per SM sub-partition
constexpr int kThreads = 64 + 32 * kDequantWarps;   // producer, MMA, dequant/epilogue
constexpr unsigned long long kDrainNs = 100000000ull;   // 100 ms

template <int kType, int kBN>
struct Layout {
    // The dequant warps copy a raw super-step into registers as soon as it lands, so one
    // raw stage already gives the next copy four MMA stages of lead; Q4_0 and Q4_K (144-byte
    // raw rows) then fit four 48 KB operand stages. Q8_0 (272-byte raw rows) keeps two raw
    // stages and three operand stages.
    static constexpr int kRawStages = kType != GQ_TYPE_Q8_0 ? 1 : 2;   // Q4_K rows are Q4_0's size
    static constexpr int kStages = kBN >= 128 ? (kType != GQ_TYPE_Q8_0 ? 4 : 3) : 6;
    static constexpr int kA = kBM * kBK * 2;
    static constexpr int kB = kBN * kBK * 2;
    static constexpr int kRaw = kBM * RawFmt<kType>::kRow;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kA;
    static constexpr int kOffRaw = kOffB + kStages * kB;
    static constexpr int kOffBar = kOffRaw + kRawStages * kRaw;
    static constexpr int kNumBars = 2 * kStages + 2 * kRawStages + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;   // room to align the base to 1024
    static constexpr int kTmemCols = kBN < 32 ? 32 : kBN;
    static_assert(kB % 1024 == 0 && kA % 1024 == 0 && kRaw % 1024 == 0, "1 KB aligned stages");
    // A split-K CTA parks its fp32 partial tile in the operand stages.
    static_assert(kBM * kBN * 4 <= kOffRaw, "partial tile fits the operand stages");
};

// Up to 64 accumulator columns [taddr, taddr + 64) of the warp's 32 lanes into v, as x16
// loads issued together and waited for once (a load's latency is paid per batch, not per
// 16 columns). Loads only the 16-column groups that start below `avail` (warp-uniform).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64], int avail) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (16 * q < avail) tmem_ld16_async(taddr + 16 * q, v + 16 * q);
    tmem_ld_wait();
}

// Stage q (0..3) of a super-step for dequantize half h: block 2q + h of the thread's row,
// from the raw super-step in registers, into the row's 128-byte swizzled A line.
template <int kType>
__device__ __forceinline__ void dequant_stage(int q, int h, const uint32_t* raw, uint8_t* arow,
                                              int row) {
    if (h == 0) {
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
}

template <int kType, int kBN, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
            int M, int N, int K, float* __restrict__ Y, unsigned* status) {
    using L = Layout<kType, kBN>;
    constexpr int S = L::kStages;
    constexpr int kRawWords = RawFmt<kType>::kRow / 4;
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
    // barrier order: full[S], empty[S], raw_full[R], raw_empty[R], acc_full. Stage s is
    // "full" when its dequantized A (every dequantize thread arrives) and its X tile (the
    // producer's arrival with the copy's bytes) are both in place: one wait for the MMAs.
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    auto raw_full = [&](int r) { return bar0 + 8u * (2 * S + r); };
    auto raw_empty = [&](int r) { return bar0 + 8u * (2 * S + L::kRawStages + r); };
    const uint32_t acc_full = bar0 + 8u * (2 * S + 2 * L::kRawStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);

    const int m0 = blockIdx.x * kBM;
    const int n0 = blockIdx.y * kBN;
    // Split K: the gridDim.z CTAs of a cluster share the tile, CTA z taking super-steps
    // [j0, j0 + nsuper) of the whole K (every CTA gets at least one).
    const int nsuper_all = K / kSuperK;
    const int j0 = kSplit ? nsuper_all * static_cast<int>(blockIdx.z) / static_cast<int>(gridDim.z) : 0;
    const int nsuper =
        kSplit ? nsuper_all * static_cast<int>(blockIdx.z + 1) / static_cast<int>(gridDim.z) - j0
               : nsuper_all;
    const int nk = kSplit ? nsuper * (kSuperK / kBK) : K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 32 * kDequantWarps + 1);
            mbar_init(empty(s), 1);
        }
        for (int r = 0; r < L::kRawStages; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), 32 * kDequantWarps);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    __syncwarp();   // lane 0 of warp 0 initialized the barriers alone: the warp arrives whole
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tensormap(&tmap_w);
            prefetch_tensormap(&tmap_x);
            int raw_issued = 0, b_issued = 0;
            bool ok = true;
            for (int ks = 0; ks < nk && ok; ++ks) {
                // Raw weights run one super-step ahead of the k-stages that use them.
                const int want = min(ks / 4 + 2, nsuper);
                while (raw_issued < want) {
                    const int j = raw_issued, r = j % L::kRawStages;
                    if (!mbar_wait(raw_empty(r), ((j / L::kRawStages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(raw_full(r), L::kRaw);
                    tma_load_2d(sRaw + r * L::kRaw, &tmap_w,
                                (j0 + j) * (RawFmt<kType>::kRow / RawFmt<kType>::kElem), m0,
                                raw_full(r));
                    ++raw_issued;
                }
                if (!ok) break;
                const int s = ks % S;
                if (!mbar_wait(empty(s), ((ks / S) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                if (ks == 0) griddep_wait();   // the bf16 X of this call is complete
                mbar_arrive_expect_tx(full(s), L::kB);
                tma_load_2d(sB + s * L::kB, &tmap_x, (j0 * (kSuperK / kBK) + ks) * kBK, n0, full(s));
                ++b_issued;
            }
            if (!ok) report_status(status, kStatusTimeout);
            // Every copy this thread issued must land before the CTA's memory is released.
            for (int i = max(0, b_issued - S); i < b_issued; ++i)
                mbar_wait(full(i % S), (i / S) & 1, kDrainNs);
            for (int j = max(0, raw_issued - L::kRawStages); j < raw_issued; ++j)
                mbar_wait(raw_full(j % L::kRawStages), (j / L::kRawStages) & 1, kDrainNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
            bool ok = true;
            for (int ks = 0; ks < nk; ++ks) {
                const int s = ks % S;
                const uint32_t ph = (ks / S) & 1;
                if (!mbar_wait(full(s), ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t adesc = sw128_kmajor_desc(sA + s * L::kA + kk * 32);
                    const uint64_t bdesc = sw128_kmajor_desc(sB + s * L::kB + kk * 32);
                    umma_bf16(tmem, adesc, bdesc, idesc, (ks | kk) != 0 ? 1u : 0u);
                }
                umma_commit(empty(s));   // stage s is free once these MMAs have read it
            }
            umma_commit(acc_full);       // accumulator complete (also after a timeout)
            if (!ok) report_status(status, kStatusTimeout);
        }
    } else {
        // ---------------- dequantize, then epilogue ----------------
        // Eight warps: warp w takes TMEM lane quadrant w % 4 (tile rows 32*(w%4)..), and
        // half h = (w - 2) / 4: block 2q + h of every 64-k stage q, then token columns
        // [h*kBN/2, (h+1)*kBN/2) in the epilogue.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        bool ok = true;
        for (int j = 0; j < nsuper && ok; ++j) {
            const int r = j % L::kRawStages;
            if (!mbar_wait(raw_full(r), (j / L::kRawStages) & 1)) {
                ok = false;
                break;
            }
            uint32_t raw[kRawWords];
            const uint8_t* src = base + L::kOffRaw + r * L::kRaw + row * RawFmt<kType>::kRow;
#pragma unroll
            for (int i = 0; i < kRawWords / 4; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
                raw[4 * i] = v.x;
                raw[4 * i + 1] = v.y;
                raw[4 * i + 2] = v.z;
                raw[4 * i + 3] = v.w;
            }
            {
                // one word of each 16-byte load: all loads complete before the fence
                uint32_t dep = 0;
#pragma unroll
                for (int i = 0; i < kRawWords / 4; ++i) dep ^= raw[4 * i];
                release_to_async_proxy(dep);
            }
            mbar_arrive(raw_empty(r));
            // kRound 64-k stages per round: the waits, the proxy fence and the arrivals of
            // a round are paid once. Two per round pays for Q8_0, whose dequantization is
            // longer (measured: 7B lm_head at N = 2048 568 -> 533 us); Q4_0 lost with it
            // (398 -> 426 us), its four stages then refilling only in pairs.
            constexpr int kRound = kType == GQ_TYPE_Q8_0 ? 2 : 1;
#pragma unroll
            for (int q = 0; q < 4; q += kRound) {
                const int ks = 4 * j + q;
                bool free = true;
#pragma unroll
                for (int i = 0; i < kRound; ++i)
                    free = free && mbar_wait(empty((ks + i) % S), (((ks + i) / S) & 1) ^ 1);
                if (!free) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int i = 0; i < kRound; ++i)
                    dequant_stage<kType>(q + i, half, raw,
                                         base + L::kOffA + ((ks + i) % S) * L::kA + row * 128, row);
                fence_proxy_async_smem();
#pragma unroll
                for (int i = 0; i < kRound; ++i) mbar_arrive(full((ks + i) % S));
            }
        }
        if (!ok) report_status(status, kStatusTimeout);
        // Epilogue: accumulator rows are TMEM lanes, token columns are TMEM columns.
        const bool done = mbar_wait(acc_full, 0);
        tc_fence_after();
        if constexpr (kSplit) {
            if (!done) report_status(status, kStatusTimeout);
            // Split K: this CTA's partial tile goes to its own shared memory, the operand
            // stages being free once every MMA has completed: part[column][row] fp32.
            float* part = reinterpret_cast<float*>(base + L::kOffA);
            if (done) {
                const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16);
                const int c_begin = half * (kBN / 2);
                for (int c = c_begin; c < c_begin + kBN / 2; c += 64) {
                    uint32_t v[64];
                    tmem_ld64(tbase + c, v, c_begin + kBN / 2 - c);
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj)
                        if (c + jj < c_begin + kBN / 2) part[(c + jj) * kBM + row] = __uint_as_float(v[jj]);
                }
            }
        } else if (done && ok) {
            const int m = m0 + row;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            const int c_begin = half * (kBN / 2);
            const int c_end = min(c_begin + kBN / 2, N - n0);
            for (int c = c_begin; c < c_end; c += 64) {
                uint32_t v[64];
                tmem_ld64(tbase + c, v, c_end - c);
                if (m < M) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) {
                        const int n = n0 + c + jj;
                        if (c + jj < c_end && n < N)
                            Y[static_cast<int64_t>(n) * M + m] = __uint_as_float(v[jj]);
                    }
                }
            }
        } else if (!done) {
            report_status(status, kStatusTimeout);
        }
    }
    if constexpr (kSplit) {
        // Every CTA of the cluster has its partial in shared memory. CTA r then sums token
        // columns [r C / Z, (r + 1) C / Z) over the cluster's CTAs in rank order (the same
        // order whoever finishes first) and writes them to Y; a second barrier keeps every
        // CTA's shared memory alive until all reads of it are done. All threads take part
        // in both barriers; the CTAs of a cluster are co-scheduled, so neither waits on
        // work that cannot run.
        __syncwarp();
        cluster_sync();
        if (warp >= 2) {
            const int Z = static_cast<int>(gridDim.z);
            const int rank = static_cast<int>(cluster_ctarank());
            const int c_lo = kBN * rank / Z, c_hi = kBN * (rank + 1) / Z;
            const uint32_t part = smem_addr(base + L::kOffA);
            const int t = threadIdx.x - 64;                      // 0..255
            const bool vec = (M % 4 == 0) && (reinterpret_cast<uintptr_t>(Y) % 16 == 0);
            for (int idx = t; idx < (c_hi - c_lo) * (kBM / 4); idx += 32 * kDequantWarps) {
                const int c = c_lo + idx / (kBM / 4);
                const int r4 = 4 * (idx % (kBM / 4));
                const uint32_t off = static_cast<uint32_t>((c * kBM + r4) * 4);
                float4 acc = ld_shared_cluster_f4(map_shared_rank(part + off, 0));
                for (int z = 1; z < Z; ++z) {
                    const float4 v = ld_shared_cluster_f4(map_shared_rank(part + off, z));
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                const int n = n0 + c, m = m0 + r4;
                if (n >= N || m >= M) continue;
                float* y = Y + static_cast<int64_t>(n) * M + m;
                if (vec) {
                    *reinterpret_cast<float4*>(y) = acc;
                } else {
                    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                    for (int i = 0; i < 4 && m + i < M; ++i) y[i] = a[i];
                }
            }
        }
        cluster_sync();
    }
    // Warps 0 and 1 ran their loops on lane 0 alone: each warp reconverges before the
    // barrier, so that it counts whole warps and the TMEM is freed only after every
    // epilogue read.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------
// Wide tile: 128 weight rows x 512 tokens per CTA. Each dequantized A stage feeds two
// MMAs of N = 256 (token halves h = 0, 1, accumulators in TMEM columns [256 h, 256 h +
// 256)), so the A path -- dequantization, swizzled stores, proxy fence, waits -- is paid
// once per 2 x 256 tokens. The X tiles of the two halves are separate 32 KB units in a
// ring of their own; the A stages have theirs.
// ---------------------------------------------------------------------------------------
template <int kType>
struct WideLayout {
    static constexpr int kHalfN = 256;
    static constexpr int kRawStages = kType != GQ_TYPE_Q8_0 ? 1 : 2;
    static constexpr int kAStages = 2;
    static constexpr int kUnits = kType != GQ_TYPE_Q8_0 ? 5 : 3;
    static constexpr int kA = kBM * kBK * 2;
    static constexpr int kU = kHalfN * kBK * 2;
    static constexpr int kRaw = kBM * RawFmt<kType>::kRow;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kAStages * kA;
    static constexpr int kOffRaw = kOffB + kUnits * kU;
    static constexpr int kOffBar = kOffRaw + kRawStages * kRaw;
    static constexpr int kNumBars = 2 * kAStages + 2 * kUnits + 2 * kRawStages + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr int kTmemCols = 512;
    // Two MMA issuers, one per token half (warps 1 and kIssuer2Warp, on different SM
    // sub-partitions), share every A stage and take alternate X units: the per-stage
    // waits, issues and loop of one thread are split between two. Both have consumed
    // stage ks - 2 when stage ks's A is ready, so an issuer waiting on unit 2 ks + h finds
    // that unit slot's previous fill (2 ks + h - kUnits) consumed, and its parity test
    // exact, when kUnits >= 4. With 3 units (Q8_0) an issuer could wait on a slot whose
    // previous fill, the other issuer's, has not landed, and its parity test would see
    // the phase two back: Q8_0 keeps one issuer.
    static constexpr int kIssuers = kUnits >= 4 ? 2 : 1;
    static constexpr int kIssuer2Warp = 2 + kDequantWarps;   // 10
    static constexpr int kThreads = kIssuers == 2 ? 32 * (kIssuer2Warp + 1) : 64 + 32 * kDequantWarps;
    static_assert(kU % 1024 == 0 && kA % 1024 == 0 && kRaw % 1024 == 0, "1 KB aligned stages");
    static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
};

template <int kType>
__global__ void __launch_bounds__(WideLayout<kType>::kThreads, 1)
gemm_wide_kernel(const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_x, int M, int N, int K,
                 float* __restrict__ Y, unsigned* status) {
    using L = WideLayout<kType>;
    constexpr int SA = L::kAStages, SU = L::kUnits, R = L::kRawStages;
    constexpr int kRawWords = RawFmt<kType>::kRow / 4;
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
    // barrier order: a_full[SA], a_empty[SA], u_full[SU], u_empty[SU], raw_full[R],
    // raw_empty[R], acc_full
    auto a_full = [&](int s) { return bar0 + 8u * s; };
    auto a_empty = [&](int s) { return bar0 + 8u * (SA + s); };
    auto u_full = [&](int u) { return bar0 + 8u * (2 * SA + u); };
    auto u_empty = [&](int u) { return bar0 + 8u * (2 * SA + SU + u); };
    auto raw_full = [&](int r) { return bar0 + 8u * (2 * SA + 2 * SU + r); };
    auto raw_empty = [&](int r) { return bar0 + 8u * (2 * SA + 2 * SU + R + r); };
    const uint32_t acc_full = bar0 + 8u * (2 * SA + 2 * SU + 2 * R);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);

    const int m0 = blockIdx.x * kBM;
    const int n0 = blockIdx.y * (2 * L::kHalfN);
    const int nsuper = K / kSuperK;
    const int nk = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(a_full(s), 32 * kDequantWarps);
            mbar_init(a_empty(s), L::kIssuers);   // every issuer's MMAs read the stage
        }
        for (int u = 0; u < SU; ++u) {
            mbar_init(u_full(u), 1);
            mbar_init(u_empty(u), 1);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), 32 * kDequantWarps);
        }
        mbar_init(acc_full, L::kIssuers);   // one commit per MMA issuer
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    __syncwarp();   // lane 0 of warp 0 initialized the barriers alone: the warp arrives whole
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tensormap(&tmap_w);
            prefetch_tensormap(&tmap_x);
            int raw_issued = 0, u_issued = 0;
            bool ok = true;
            for (int ks = 0; ks < nk && ok; ++ks) {
                const int want = min(ks / 4 + 2, nsuper);
                while (raw_issued < want) {
                    const int j = raw_issued, r = j % R;
                    if (!mbar_wait(raw_empty(r), ((j / R) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(raw_full(r), L::kRaw);
                    tma_load_2d(sRaw + r * L::kRaw, &tmap_w,
                                j * (RawFmt<kType>::kRow / RawFmt<kType>::kElem), m0, raw_full(r));
                    ++raw_issued;
                }
                if (!ok) break;
                if (ks == 0) griddep_wait();   // the bf16 X of this call is complete
                for (int h = 0; h < 2; ++h) {
                    const int ub = 2 * ks + h, u = ub % SU;
                    if (!mbar_wait(u_empty(u), ((ub / SU) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(u_full(u), L::kU);
                    tma_load_2d(sB + u * L::kU, &tmap_x, ks * kBK, n0 + h * L::kHalfN, u_full(u));
                    ++u_issued;
                }
            }
            if (!ok) report_status(status, kStatusTimeout);
            // Every copy this thread issued must land before the CTA's memory is released.
            for (int i = max(0, u_issued - SU); i < u_issued; ++i)
                mbar_wait(u_full(i % SU), (i / SU) & 1, kDrainNs);
            for (int j = max(0, raw_issued - R); j < raw_issued; ++j)
                mbar_wait(raw_full(j % R), (j / R) & 1, kDrainNs);
        }
    } else if (warp == 1 || (L::kIssuers == 2 && warp == L::kIssuer2Warp)) {
        // ---------------- MMA issuers ----------------
        // Issuer h0 issues the MMAs of token half h0 (accumulator columns [256 h0,
        // 256 h0 + 256)) for every A stage; a single issuer takes both halves.
        constexpr int I = L::kIssuers;
        const int h0 = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, L::kHalfN);
            bool ok = true;
            for (int ks = 0; ks < nk && ok; ++ks) {
                const int sa = ks % SA;
                if (!mbar_wait(a_full(sa), (ks / SA) & 1)) {
                    ok = false;
                    break;
                }
                for (int h = h0; h < 2; h += I) {
                    const int ub = 2 * ks + h, u = ub % SU;
                    if (!mbar_wait(u_full(u), (ub / SU) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc = sw128_kmajor_desc(sA + sa * L::kA + kk * 32);
                        const uint64_t bdesc = sw128_kmajor_desc(sB + u * L::kU + kk * 32);
                        umma_bf16(tmem + h * L::kHalfN, adesc, bdesc, idesc,
                                  (ks | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(u_empty(u));   // X unit u is free once these MMAs have read it
                }
                umma_commit(a_empty(sa));      // and A stage sa once every issuer's have
            }
            umma_commit(acc_full);             // accumulators complete (also after a timeout)
            if (!ok) report_status(status, kStatusTimeout);
        }
    } else {
        // ---------------- dequantize, then epilogue ----------------
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        bool ok = true;
        for (int j = 0; j < nsuper && ok; ++j) {
            const int r = j % R;
            if (!mbar_wait(raw_full(r), (j / R) & 1)) {
                ok = false;
                break;
            }
            uint32_t raw[kRawWords];
            const uint8_t* src = base + L::kOffRaw + r * L::kRaw + row * RawFmt<kType>::kRow;
#pragma unroll
            for (int i = 0; i < kRawWords / 4; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
                raw[4 * i] = v.x;
                raw[4 * i + 1] = v.y;
                raw[4 * i + 2] = v.z;
                raw[4 * i + 3] = v.w;
            }
            {
                uint32_t dep = 0;
#pragma unroll
                for (int i = 0; i < kRawWords / 4; ++i) dep ^= raw[4 * i];
                release_to_async_proxy(dep);
            }
            mbar_arrive(raw_empty(r));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ks = 4 * j + q, sa = ks % SA;
                if (!mbar_wait(a_empty(sa), ((ks / SA) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                dequant_stage<kType>(q, half, raw, base + L::kOffA + sa * L::kA + row * 128, row);
                fence_proxy_async_smem();
                mbar_arrive(a_full(sa));
            }
        }
        if (!ok) report_status(status, kStatusTimeout);
        // Epilogue: warp (quad, half) writes token half `half` of its 32 rows.
        const bool done = mbar_wait(acc_full, 0);
        tc_fence_after();
        if (done && ok) {
            const int m = m0 + row;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            const int c_begin = half * L::kHalfN;
            const int c_end = min(c_begin + L::kHalfN, N - n0);
            for (int c = c_begin; c < c_end; c += 64) {
                uint32_t v[64];
                tmem_ld64(tbase + c, v, c_end - c);
                if (m < M) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) {
                        const int n = n0 + c + jj;
                        if (c + jj < c_end && n < N)
                            Y[static_cast<int64_t>(n) * M + m] = __uint_as_float(v[jj]);
                    }
                }
            }
        } else if (!done) {
            report_status(status, kStatusTimeout);
        }
    }
    __syncwarp();   // whole warps at the barrier (warps 0, 1 and 10 ran lane 0 alone)
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// X (fp32, n elements) -> bf16, round to nearest even. Each thread keeps kXUnroll
// 16-byte loads in flight. The kSide instance runs on a few blocks per SM with the
// max-shared carveout, so that the GEMM after it (a programmatic dependent) finds room on
// every SM and runs its prologue, first weight copies and dequantization beside the
// conversion; it is used for small X, where that start-up is a large part of the call.
constexpr int kXUnroll = 4;
constexpr int kXSideBlocksPerSm = 2;
constexpr int64_t kXSideMaxElems = int64_t(1) << 22;   // 16 MB of fp32 X
template <bool kSide>
__global__ void __launch_bounds__(256)
x_to_bf16_kernel(const float* __restrict__ X, int64_t n, __nv_bfloat16* __restrict__ out) {
    // The GEMM launched after this kernel may start its prologue and weight copies now; it
    // waits for this grid's completion before it reads the bf16 X.
    griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(X) & 15) == 0) {
        const int64_t n4 = n / 4;
        for (int64_t i = i0; i < n4; i += stride * kXUnroll) {
            float4 v[kXUnroll];
#pragma unroll
            for (int u = 0; u < kXUnroll; ++u)
                if (i + u * stride < n4) v[u] = reinterpret_cast<const float4*>(X)[i + u * stride];
#pragma unroll
            for (int u = 0; u < kXUnroll; ++u) {
                if (i + u * stride >= n4) break;
                __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + 4 * (i + u * stride));
                o[0] = __floats2bfloat162_rn(v[u].x, v[u].y);
                o[1] = __floats2bfloat162_rn(v[u].z, v[u].w);
            }
        }
        for (int64_t i = 4 * n4 + i0; i < n; i += stride) out[i] = __float2bfloat16_rn(X[i]);
    } else {
        for (int64_t i = i0; i < n; i += stride) out[i] = __float2bfloat16_rn(X[i]);
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
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

template <typename KernelT>
cudaError_t ensure_max_shared_carveout(KernelT kernel, int device) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, bool> done;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), device);
    if (done.count(key)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess) done[key] = true;
    return e;
}

// Split-K ways for a GEMM of `tiles` output tiles and `nsuper` 256-k super-steps. With
// fewer tiles than half the SMs, each tile is shared by a cluster of Z CTAs (Z = 2 or 4)
// that split K and sum their partials through distributed shared memory; Z is the largest
// that keeps every cluster resident at once (cudaOccupancyMaxActiveClusters, cached).
template <typename KernelT>
int split_k_ways(KernelT kernel, int smem_bytes, const DeviceInfo* info, int64_t tiles,
                 int64_t nsuper) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int>, int> max_clusters;
    for (int Z = 4; Z >= 2; Z /= 2) {
        if (tiles * Z > info->sm_count || nsuper < Z) continue;
        int active = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            const auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), info->device, Z);
            auto it = max_clusters.find(key);
            if (it != max_clusters.end()) {
                active = it->second;
            } else {
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3(1, 1, static_cast<unsigned>(Z));
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 1;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = static_cast<unsigned>(Z);
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    active = 0;
                }
                max_clusters[key] = active;
            }
        }
        if (tiles <= active) return Z;
    }
    return 1;
}

// Wide (512-token) tiles where their waves, each twice the work, are no more than the
// 256-token waves: then they save half the per-CTA fill, and Q8_0 also the cost of its
// longer dequantization. Measured (A/B, one box): TinyLLaMA lm_head N = 512 69.3 -> 61.2 us,
// LLaMA-7B attn N = 2048 60.8 -> 55.3 us, down 155.4 -> 152.1 us, lm_head Q4_0 399 -> 399 us
// and Q8_0 533 -> 492 us; gate_up (3 wide waves against 4.5 narrow ones) 148 -> 161 us,
// which this rule keeps narrow.
bool use_wide(int64_t mt, int64_t N, int sms) {
    if (N <= 256) return false;
    const int64_t w256 = (mt * ((N + 255) / 256) + sms - 1) / sms;
    const int64_t w512 = (mt * ((N + 511) / 512) + sms - 1) / sms;
    return 2 * w512 <= w256;
}

template <int kType>
cudaError_t launch_wide(CUtensorMap tw, CUtensorMap tx, const MatProblem& p, int64_t N,
                        int64_t mt, const DeviceInfo* info, cudaStream_t s) {
    using WL = WideLayout<kType>;
    auto kernel = gemm_wide_kernel<kType>;
    cudaError_t e = ensure_smem(kernel, info->device, WL::kAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(mt), static_cast<unsigned>((N + 511) / 512));
    cfg.blockDim = dim3(WL::kThreads);
    cfg.dynamicSmemBytes = WL::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int M = static_cast<int>(p.M), n = static_cast<int>(N), K = static_cast<int>(p.K);
    float* Y = p.Y;
    unsigned* status = info->status;
    void* args[] = {&tw, &tx, &M, &n, &K, &Y, &status};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
}

template <int kType, int kBN>
cudaError_t launch_gemm_t(const MatProblem& p, int64_t N, const __nv_bfloat16* xb,
                          const DeviceInfo* info, cudaStream_t s) {
    using L = Layout<kType, kBN>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t row_bytes = (p.K / kSuperK) * RawFmt<kType>::kRow;
    CUtensorMap tw{}, tx{};
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / RawFmt<kType>::kElem),
                                    static_cast<cuuint64_t>(p.M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(RawFmt<kType>::kRow / RawFmt<kType>::kElem),
                                   static_cast<cuuint32_t>(kBM)};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&tw, kType != GQ_TYPE_Q8_0 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                         2, const_cast<uint8_t*>(p.W), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K * 2)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBN)};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(xb),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    auto kernel = gemm_kernel<kType, kBN, false>;
    auto split_kernel = gemm_kernel<kType, kBN, true>;
    cudaError_t e = ensure_smem(kernel, info->device, L::kAlloc);
    if (e == cudaSuccess) e = ensure_smem(split_kernel, info->device, L::kAlloc);
    if (e != cudaSuccess) return e;
    const int64_t mt = (p.M + kBM - 1) / kBM, nt = (N + kBN - 1) / kBN;
    const int Z = split_k_ways(split_kernel, L::kAlloc, info, mt * nt, p.K / kSuperK);
    if (kBN == 256 && Z == 1 && use_wide(mt, N, info->sm_count))
        return launch_wide<kType>(tw, tx, p, N, mt, info, s);
    // A programmatic dependent of x_to_bf16_kernel: barrier setup, TMEM allocation, the
    // first weight copies and their dequantization overlap the conversion of X; the
    // producer waits for it (griddepcontrol.wait) before its first X tile copy. Nothing
    // else this kernel touches is written by x_to_bf16_kernel, and that kernel itself is
    // an ordinary launch, so everything earlier in the stream has completed.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(mt), static_cast<unsigned>(nt), static_cast<unsigned>(Z));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(Z);
    cfg.attrs = attr;
    cfg.numAttrs = Z == 1 ? 1 : 2;
    int M = static_cast<int>(p.M), n = static_cast<int>(N), K = static_cast<int>(p.K);
    float* Y = p.Y;
    unsigned* status = info->status;
    void* args[] = {&tw, &tx, &M, &n, &K, &Y, &status};
    return cudaLaunchKernelExC(
        &cfg, reinterpret_cast<const void*>(Z == 1 ? kernel : split_kernel), args);
}

}  // namespace

int64_t gemm_x_bytes(int64_t K, int64_t N) { return (N * K * 2 + 255) / 256 * 256; }

int64_t gemm_workspace_bytes(int64_t K, int64_t N) { return gemm_x_bytes(K, N); }

bool gemm_eligible(gq_type t, const MatProblem& p, int64_t N) {
    if (block_bytes_of(t) == 0) return false;
    if (N < kGemmMinTokens || p.K % kSuperK != 0 || p.M <= 0) return false;
    if (p.M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 24) || p.K > (int64_t(1) << 24))
        return false;
    return reinterpret_cast<uintptr_t>(p.W) % 16 == 0;
}

cudaError_t launch_gemm(gq_type t, const MatProblem& p, int64_t N, void* workspace,
                        int64_t workspace_bytes, cudaStream_t s) {
    (void)workspace_bytes;   // the bf16 copy of X is all this kernel needs
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    __nv_bfloat16* xb = static_cast<__nv_bfloat16*>(workspace);
    const int64_t n = N * p.K;
    const int64_t blocks = (n / 4 + 256 * kXUnroll - 1) / (256 * kXUnroll) + 1;
    if (n <= kXSideMaxElems) {
        // The instance's carveout: an SM set up for it alone would hold little shared
        // memory, and a GEMM CTA could not join it there until the SM drained.
        e = ensure_max_shared_carveout(x_to_bf16_kernel<true>, info->device);
        if (e != cudaSuccess) return e;
        const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(info->sm_count) * kXSideBlocksPerSm));
        x_to_bf16_kernel<true><<<grid, 256, 0, s>>>(p.X, n, xb);
    } else {
        const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(info->sm_count) * 8));
        x_to_bf16_kernel<false><<<grid, 256, 0, s>>>(p.X, n, xb);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (t == GQ_TYPE_Q4_0) return launch_gemm_t<GQ_TYPE_Q4_0, 256>(p, N, xb, info, s);
    if (t == GQ_TYPE_Q4_K) return launch_gemm_t<GQ_TYPE_Q4_K, 256>(p, N, xb, info, s);
    return launch_gemm_t<GQ_TYPE_Q8_0, 256>(p, N, xb, info, s);
}

}  // namespace gq
