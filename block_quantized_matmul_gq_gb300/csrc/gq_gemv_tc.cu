// gq_gemv_tc.cu -- decode mul_mat for 3..64 tokens on the tensor cores:
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
//   warps 1..4   MMA issuers, one per SM sub-partition: issuer q owns the 64-k quarter q
//                of every super-step (a single issuing thread cannot keep the tensor core
//                busy with N <= 64 MMAs), its own accumulator per set, and afterwards the
//                tile epilogue for its TMEM lane quadrant (the four accumulators added in
//                a fixed order).
//   warps 5..12  dequantize, two groups of four (one per 128-k half of every super-step),
//                one row per thread, written to the group's A slot in TMEM (tcgen05.st).
// Scaled form (Q4_0, up to 16 tokens): the A slots hold the exact codes c - 8, each 32-k
// block's MMAs write the block's own accumulator, and the dequantize warps add
// d_blk * acc_blk to a per-row fp32 sum one super-step behind the MMAs; the two groups'
// halves of a tile meet in shared memory and group 0 writes Y. The weights are never
// rounded. Other forms dequantize to bf16 ((c - 8) * d or c * d, rounded once; Q4_K
// sub-blocks d sc q - dmin m, rounded once in fp32 and once to bf16: a 256-k super-step is
// one 144-byte super-block, and group g takes its sub-blocks 4g .. 4g + 3).
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
constexpr int kQuarters = kSuperK / kBK;  // 64-k quarters of a super-step
constexpr int kMmaWarps = kQuarters;      // warps 1..4: one MMA issuer per quarter
constexpr int kDequantWarps = 8;          // two groups of four warps (all 128 rows each)
constexpr int kFirstDequantWarp = 1 + kMmaWarps;
constexpr int kThreads = 32 * (1 + kMmaWarps + kDequantWarps);   // 416
constexpr int kSlotCols = kHalfK / 2;     // 64 columns: 128 bf16 per lane
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 232448;        // opt-in dynamic shared memory per CTA
constexpr unsigned long long kDrainNs = 100000000ull;

template <int kType, int kNPad>
struct TcLayout {
    // TMEM: kAccBufs sets of four accumulators (one per quarter) of kNPad columns, then
    // two groups x kGroupSlots A slots of 64 columns. Two sets let a tile's epilogue
    // overlap the next tile's MMAs; at 64 tokens only one set fits next to the A slots.
    // Scaled form (Q4_0 and Q4_K, up to 16 tokens): A holds the exact codes (c - 8, or the
    // Q4_K q) and every 32-k block has its own accumulator, two buffers of a super-step's
    // eight (256 columns); the dequantize warps apply the block scales in fp32 (Q4_K: and
    // the mins, against the per-token block sums of X that follow each super-step's X
    // tiles, kSums).
    static constexpr bool kScaled = (kType == GQ_TYPE_Q4_0 || kType == GQ_TYPE_Q4_K) && kNPad == 16;
    static constexpr bool kSums = kScaled && kType == GQ_TYPE_Q4_K;
    static constexpr int kAccBufs = kNPad <= 32 ? 2 : 1;
    static constexpr int kUnitCols = (kSuperK / 32) * kNPad;   // scaled: a super-step's blocks
    static constexpr int kAccCols =
        kScaled ? 2 * kUnitCols : kAccBufs * kQuarters * kNPad;   // 256 / 256 / 256
    static constexpr int kGroupSlots = (kTmemCols - kAccCols) / (2 * kSlotCols);   // 3 / 2 / 2
    static_assert(kGroupSlots >= 2, "TMEM budget");
    static constexpr int kB = kNPad * kBK * 2;              // one 64-k X tile: 2 / 4 / 8 KB
    static constexpr int kRawRow = RawFmt<kType>::kRow;     // 144 / 272
    static constexpr int kRaw = kBM * kRawRow;              // 18 / 34 KB of raw blocks
    // X of a super-step: four tiles, then with kSums the 8 x kNPad fp32 block sums (512 B,
    // in a 1 KB slot that keeps the stages 1 KB aligned). kXCopy bytes are copied.
    static constexpr int kXCopy = 4 * kB + (kSums ? 8 * kNPad * 4 : 0);
    static constexpr int kXSlot = 4 * kB + (kSums ? 1024 : 0);
    static constexpr int kStage = kRaw + kXSlot;            // raw blocks + the super-step's X
    static constexpr int kStageTx = kRaw + kXCopy;          // bytes a stage's copies deliver
    static constexpr int kOffRaw = 0;
    // Scaled: the two dequantize groups' halves of a tile's y meet in shared memory, one
    // buffer (tiles are at least 8 super-steps apart), 128 rows x kNPad (+1 against bank
    // conflicts) fp32.
    static constexpr int kYStride = kNPad + 1;
    static constexpr int kYBytes = kScaled ? kBM * kYStride * 4 : 0;
    static constexpr int kFixed = 1024 + 512 + kYBytes;     // alignment slack, barriers, slot
    static constexpr int kRawFit = (kSmemLimit - kFixed) / kStage;
    static constexpr int kRawStages = kRawFit > 8 ? 8 : kRawFit;
    static constexpr int kOffBar = kOffRaw + kRawStages * kStage;
    // raw_full[R], raw_empty[R], a_full[2][G], a_empty[2][G], acc_full[B], acc_empty[B],
    // mma_done, and in the scaled form y_full, y_free
    static constexpr int kNumBars =
        2 * kRawStages + 4 * kGroupSlots + 2 * kAccBufs + 1 + (kScaled ? 2 : 0);
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffY = kOffMisc + 16;
    static constexpr int kBytes = kOffY + kYBytes;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kB % 1024 == 0 && kRaw % 1024 == 0, "1 KB aligned tiles");
    static_assert(kRawStages >= 2 && kAlloc <= kSmemLimit, "shared memory budget");
    static_assert(kNumBars * 8 + 16 <= kFixed - 1024 - kYBytes, "barrier space");
};

struct TcProb {
    const uint8_t* W;
    const float* X;       // n_tok x K fp32 activations
    const uint8_t* Xt;    // pre-arranged bf16 X tiles: K/64 tiles of kNPad x 128 bytes
    float* Y;
    int64_t M;
    int64_t row_bytes;
    int64_t unit_begin;   // index of the problem's first work unit in the launch
    int32_t K;
    int32_t nsuper;       // super-steps per tile: K / 256
};

// Largest number of problems one launch takes: the tensor maps and the problem table
// travel as kernel parameters (160 x (128 + 64) bytes here, under the 32 KB limit; a
// whole TinyLLaMA decode step, 155 matrices, is one launch).
constexpr int kMaxLaunchProbs = 160;
// Largest grid: the split-tile partial sums are sized for it.
constexpr int kMaxTcGrid = 256;

template <int kMaxProbs>
struct TcParams {
    CUtensorMap maps[kMaxProbs];   // raw weight bytes per problem: rows x row bytes
    int32_t count;
    int32_t n_tok;
    int64_t total_units;   // work units (one 128-row tile x one 256-k super-step) in all
    float* part;           // per CTA two 128 x kNPad partial-sum tiles of split tiles
    int* counters;         // per CTA boundary and TMEM lane quadrant: partials delivered
    unsigned* status;
    TcProb p[kMaxProbs];
};

// The work of a launch is a sequence of units, problem by problem, tile by tile, super-step
// by super-step; every unit moves and multiplies the same bytes, so CTA c takes units
// [U c / grid, U (c + 1) / grid): shares differ by at most one unit. A tile whose units
// fall to two or more CTAs is "split": each of them leaves a partial sum, and the last to
// deliver adds them all in CTA order (tc_finish_split). Every role of a CTA walks the same
// sequence.
struct TcWalk {
    int p;                // problem
    int64_t row0;         // first row of the tile
    int rows;             // rows of the tile that exist (<= 128)
    int j;                // current super-step of the tile
    int jbeg, jend;       // this share's super-steps of the tile: [jbeg, jend)
    int nsuper;
    int64_t u, u_end;     // current unit, end of the share
    bool valid;
};

// The problem that unit u belongs to: the last p with unit_begin <= u (binary search: the
// table lives in kernel-parameter space, where each probe can miss the constant cache).
template <int kMaxProbs>
__device__ int tc_problem_of(const TcParams<kMaxProbs>& P, int64_t u) {
    int lo = 0, hi = P.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].unit_begin <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

template <int kMaxProbs>
__device__ void tc_walk_tile(const TcParams<kMaxProbs>& P, TcWalk& w, int p, int64_t u) {
    const int64_t off = u - P.p[p].unit_begin;
    w.p = p;
    w.nsuper = P.p[p].nsuper;
    w.row0 = off / w.nsuper * kBM;
    w.rows = static_cast<int>(min(static_cast<int64_t>(kBM), P.p[p].M - w.row0));
    w.j = w.jbeg = static_cast<int>(off % w.nsuper);
    w.jend = static_cast<int>(min(static_cast<int64_t>(w.nsuper), w.jbeg + (w.u_end - u)));
    w.u = u;
}

template <int kMaxProbs>
__device__ void tc_walk_open(const TcParams<kMaxProbs>& P, TcWalk& w, int64_t u0, int64_t u1) {
    w.u_end = u1;
    w.valid = u0 < u1;
    if (w.valid) tc_walk_tile(P, w, tc_problem_of(P, u0), u0);
}

template <int kMaxProbs>
__device__ void tc_walk_next(const TcParams<kMaxProbs>& P, TcWalk& w) {
    ++w.u;
    if (++w.j < w.jend) return;
    if (w.u >= w.u_end) {
        w.valid = false;
        return;
    }
    const int p = (w.row0 + kBM < P.p[w.p].M) ? w.p : w.p + 1;   // next tile or problem
    tc_walk_tile(P, w, p, w.u);
}

// One dequantize group's half of a row's raw super-step (kWords 32-bit words) from shared
// memory. The half starts 16-byte aligned (kG = 0) or 8 bytes past (kG = 1): one 8-byte
// load at the unaligned end, 16-byte loads for the rest, which a quarter warp serves
// without bank conflicts at the 144 / 272-byte row pitch.
// One word of each shared load of load_half_row<kG>, combined: depending on it makes every
// load complete before what follows (the proxy fence that lets the stage be refilled).
template <int kG, int kWords>
__device__ __forceinline__ uint32_t half_row_dep(const uint32_t (&raw)[kWords]) {
    constexpr int w8 = kG == 0 ? kWords - 2 : 0;
    constexpr int w16 = kG == 0 ? 0 : 2;
    uint32_t d = raw[w8];
#pragma unroll
    for (int i = 0; i < (kWords - 2) / 4; ++i) d ^= raw[w16 + 4 * i];
    return d;
}

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

// A split tile (problem p, rows [row0, row0 + rows)): this CTA's warp for TMEM lane quadrant
// `quad` has written its 32 rows of partial sum to slot `slot` (0: the share starts inside
// the tile, 1: it ends inside). The contributors are CTA c - 1 (slot 1) and CTAs c ..
// c_end - 1 (slot 0), c the first CTA boundary inside the tile. Each contributor's warp
// counts itself in; the last one adds the partials in that CTA order (so the sum does not
// depend on who finishes last), writes Y and resets the counter for the next launch.
// Nothing waits for another CTA.
template <int kNPad, int kMaxProbs>
__device__ void tc_finish_split(const TcParams<kMaxProbs>& P, int p, int64_t row0, int rows,
                                int slot, int quad, int lane) {
    const TcProb& pr = P.p[p];
    const int64_t U = P.total_units;
    const int G = gridDim.x;
    const int64_t tile_u0 = pr.unit_begin + row0 / kBM * pr.nsuper;
    const int64_t tile_u1 = tile_u0 + pr.nsuper;
    int c = static_cast<int>(blockIdx.x) + slot;   // a boundary inside the tile
    while (c > 1 && U * (c - 1) / G > tile_u0) --c;
    int c_end = c + 1;
    while (c_end < G && U * c_end / G < tile_u1) ++c_end;
    int* counter = P.counters + c * 4 + quad;
    __threadfence();   // this lane's partial rows, before the count below
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(counter, 1) == c_end - c;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    const int row = quad * 32 + lane;
    if (row < rows) {
        // all loads of a contributor are issued before its adds, and all stores come last
        const int64_t tile_elems = static_cast<int64_t>(kNPad) * kBM;
        float y[kNPad];
        const float* first = P.part + (static_cast<int64_t>(c - 1) * 2 + 1) * tile_elems + row;
#pragma unroll
        for (int n = 0; n < kNPad; ++n) y[n] = __ldcg(first + n * kBM);
        for (int cc = c; cc < c_end; ++cc) {
            const float* src = P.part + static_cast<int64_t>(cc) * 2 * tile_elems + row;
            float v[kNPad];
#pragma unroll
            for (int n = 0; n < kNPad; ++n) v[n] = __ldcg(src + n * kBM);
#pragma unroll
            for (int n = 0; n < kNPad; ++n) y[n] += v[n];
        }
        float* Y = pr.Y + row0 + row;
#pragma unroll
        for (int n = 0; n < kNPad; ++n)
            if (n < P.n_tok) Y[n * pr.M] = y[n];
    }
    __syncwarp();
    if (lane == 0) *counter = 0;
}

// Waits on an mbarrier phase with every lane of the warp; true only if all lanes saw it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// MMA issuer warp of the scaled form (warps 1..4; issuer q owns the 64-k quarter q of
// every super-step, i.e. blocks 2q and 2q + 1). A holds the exact codes c - 8 and each
// block's two MMAs (K = 16) write the block's own accumulator, in the super-step's buffer
// (two buffers by super-step parity): acc_blk = sum over the block of (c - 8) * x. The
// dequantize warps apply the block scales (tc_dequant_scaled).
template <int kType, int kNPad, int kMaxProbs>
__device__ void tc_issue_scaled(const TcParams<kMaxProbs>& P, TcWalk& w, uint32_t tmem,
                                uint32_t sRaw, uint32_t bar0) {
    using L = TcLayout<kType, kNPad>;
    static_assert(L::kScaled, "scaled form");
    constexpr int R = L::kRawStages;
    constexpr int G = L::kGroupSlots;
    constexpr int B = L::kAccBufs;
    auto raw_full = [&](int r) { return bar0 + 8u * r; };
    auto raw_empty = [&](int r) { return bar0 + 8u * (R + r); };
    auto a_full = [&](int g, int i) { return bar0 + 8u * (2 * R + g * G + i); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * R + 4 * G + b); };
    const uint32_t mma_done = bar0 + 8u * (2 * R + 4 * G + 2 * B);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q = warp - 1;
    const int g = q >> 1;   // dequantize group that fills quarter q
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kNPad);
    int raw_n = 0;
    bool ok = true;
    for (; w.valid && ok; tc_walk_next(P, w), ++raw_n) {
        const int b = raw_n & 1;
        const int r = raw_n % R;
        const int gi = raw_n % G;
        // Buffer b's columns of blocks 2q, 2q + 1 were last read by group g scaling
        // super-step n - 2, which it did before storing the codes that a_full(g) announces.
        if (!warp_wait(raw_full(r), (raw_n / R) & 1) ||            // the super-step's X landed
            !warp_wait(a_full(g, gi), (raw_n / G) & 1)) {          // quarter q's codes stored
            ok = false;
            break;
        }
        tc_fence_after();
        if (lane == 0) {
            const uint32_t sX = sRaw + r * L::kStage + L::kRaw + q * L::kB;
            const uint32_t a_col =
                tmem + L::kAccCols + (g * G + gi) * kSlotCols + (q & 1) * (kBK / 2);
            const uint32_t d0 = tmem + static_cast<uint32_t>(b * L::kUnitCols + 2 * q * kNPad);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)   // blocks 2q (kk 0, 1) and 2q + 1 (kk 2, 3)
                umma_bf16_tmem_a(d0 + (kk >> 1) * kNPad, a_col + kk * 8,
                                 sw128_kmajor_desc(sX + kk * 32), idesc,
                                 static_cast<uint32_t>(kk & 1));
            // No commit for the A slot: the dequantize warps reuse it only after they have
            // waited for acc_full of the super-step two back, whose MMAs read it.
            umma_commit(raw_empty(r));
            umma_commit(acc_full(b));
        }
        __syncwarp();
    }
    // Completes when every MMA this thread issued has finished (also after a timeout), so
    // the TMEM release never races an MMA in flight.
    if (lane == 0) umma_commit(mma_done);
    if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
}

// Dequantize warp of the scaled form (warps 5..12; group g takes blocks 4g .. 4g + 3 of
// every super-step for all 128 rows, one row per thread). Per super-step it stores the
// codes c - 8 of its half row in the group's A slot, then, one super-step behind the MMAs,
// adds d_blk * acc_blk of its four blocks to its fp32 y (blocks and super-steps in order).
// Q4_K: the blocks are sub-blocks 4g .. 4g + 3, the codes q, and each adds
// D acc - M xsum with D = d sc and M = dmin m (exact) and xsum the block's sum of the bf16
// X, per token, which the super-step's stage holds after its X tiles; the stage is
// released only after that scaling.
// At a tile's end group 1 hands its y to group 0 through shared memory; group 0 writes
// y0 + y1 to Y, or to this CTA's partial slot of a split tile.
template <int kType, int kNPad, int kMaxProbs>
__device__ void tc_dequant_scaled(const TcParams<kMaxProbs>& P, TcWalk& w, uint32_t tmem,
                                  const uint8_t* base, uint32_t bar0) {
    using L = TcLayout<kType, kNPad>;
    static_assert(L::kScaled, "scaled form");
    constexpr int R = L::kRawStages;
    constexpr int G = L::kGroupSlots;
    constexpr int B = L::kAccBufs;
    constexpr bool kQ4K = kType == GQ_TYPE_Q4_K;
    // Q4_0: a half row of 72 bytes; Q4_K: the 16 header bytes and the group's two quarters
    constexpr int kHalfWords = kQ4K ? 20 : L::kRawRow / 8;
    constexpr int kHalfBlocks = 4;
    auto raw_full = [&](int r) { return bar0 + 8u * r; };
    auto raw_empty = [&](int r) { return bar0 + 8u * (R + r); };
    auto a_full = [&](int g, int i) { return bar0 + 8u * (2 * R + g * G + i); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * R + 4 * G + b); };
    const uint32_t mma_done = bar0 + 8u * (2 * R + 4 * G + 2 * B);
    const uint32_t y_full = mma_done + 8u;
    const uint32_t y_free = mma_done + 16u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = (warp - kFirstDequantWarp) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t a_lane = tmem + tlane + L::kAccCols;
    float* ybuf = reinterpret_cast<float*>(const_cast<uint8_t*>(base) + L::kOffY);

    float y[kNPad];
#pragma unroll
    for (int t = 0; t < kNPad; ++t) y[t] = 0.0f;
    float dprev[kHalfBlocks];
    float mprev[kHalfBlocks];         // Q4_K: the blocks' M = dmin m
    int prev_n = -1;                  // super-step whose scaling is due
    bool prev_last = false;           // ... and it ends its tile
    int prev_p = 0, prev_rows = 0, prev_slot = -1;
    int64_t prev_row0 = 0;
    int head_p = -1, head_rows = 0;
    int64_t head_row0 = 0;
    int tile_n = 0;                   // tiles finished by this CTA

    auto scale = [&](int n, const float (&d)[kHalfBlocks], const float (&m)[kHalfBlocks]) -> bool {
        const int b = n & 1;
        if (!warp_wait(acc_full(b), (n >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t acc =
            tmem + tlane + static_cast<uint32_t>(b * L::kUnitCols + g * kHalfBlocks * kNPad);
        uint32_t v[kHalfBlocks][16];   // all four blocks' accumulators behind one wait
#pragma unroll
        for (int blk = 0; blk < kHalfBlocks; ++blk) tmem_ld16_async(acc + blk * kNPad, v[blk]);
        tmem_ld_wait();
        if constexpr (kQ4K) {
            // the block sums of super-step n, in its stage after the X tiles (the stage is
            // released below, once they have been read)
            const int rn = n % R;
            const float4* xs = reinterpret_cast<const float4*>(
                base + L::kOffRaw + rn * L::kStage + L::kRaw + 4 * L::kB +
                (g * kHalfBlocks) * kNPad * 4);
            uint32_t dep = 0;
#pragma unroll
            for (int blk = 0; blk < kHalfBlocks; ++blk) {
#pragma unroll
                for (int t4 = 0; t4 < kNPad / 4; ++t4) {
                    const float4 s4 = xs[blk * (kNPad / 4) + t4];
                    const int t = 4 * t4;
                    fma2_bcast(y[t], y[t + 1], d[blk], __uint_as_float(v[blk][t]),
                               __uint_as_float(v[blk][t + 1]));
                    fma2_bcast(y[t + 2], y[t + 3], d[blk], __uint_as_float(v[blk][t + 2]),
                               __uint_as_float(v[blk][t + 3]));
                    fma2_bcast(y[t], y[t + 1], -m[blk], s4.x, s4.y);
                    fma2_bcast(y[t + 2], y[t + 3], -m[blk], s4.z, s4.w);
                    dep ^= __float_as_uint(s4.x);
                }
            }
            release_to_async_proxy(dep);
            mbar_arrive(raw_empty(rn));
        } else {
#pragma unroll
            for (int blk = 0; blk < kHalfBlocks; ++blk) {
#pragma unroll
                for (int t = 0; t < kNPad; t += 2)   // y = fma(d, acc, y) on two tokens at once
                    fma2_bcast(y[t], y[t + 1], d[blk], __uint_as_float(v[blk][t]),
                               __uint_as_float(v[blk][t + 1]));
            }
        }
        return true;
    };
    auto finish_tile = [&](int p, int64_t row0, int rows, int slot) -> bool {
        const uint32_t ph = tile_n & 1;
        float* yb = ybuf + row * L::kYStride;
        ++tile_n;
        if (g == 1) {
            if (!mbar_wait(y_free, ph ^ 1)) return false;   // group 0 read the last tile's
#pragma unroll
            for (int t = 0; t < kNPad; ++t) yb[t] = y[t];
            mbar_arrive(y_full);   // release: the stores above before group 0's reads
#pragma unroll
            for (int t = 0; t < kNPad; ++t) y[t] = 0.0f;
            return true;
        }
        if (!mbar_wait(y_full, ph)) return false;
#pragma unroll
        for (int t = 0; t < kNPad; ++t) y[t] += yb[t];
        mbar_arrive(y_free);
        const TcProb& pr = P.p[p];
        float* part = P.part + (static_cast<int64_t>(blockIdx.x) * 2 + max(slot, 0)) *
                                   (kNPad * kBM);
        if (row < rows) {
#pragma unroll
            for (int t = 0; t < kNPad; ++t) {
                if (t >= P.n_tok) continue;
                if (slot < 0)
                    pr.Y[t * pr.M + row0 + row] = y[t];
                else
                    part[t * kBM + row] = y[t];
            }
        }
#pragma unroll
        for (int t = 0; t < kNPad; ++t) y[t] = 0.0f;
        if (slot == 1) {
            tc_finish_split<kNPad>(P, p, row0, rows, 1, quad, lane);
        } else if (slot == 0) {   // the share's first tile: finished after the last one
            head_p = p;
            head_row0 = row0;
            head_rows = rows;
        }
        return true;
    };

    int raw_n = 0;
    bool ok = true;
    uint32_t raw[kHalfWords];
    for (; w.valid && ok; tc_walk_next(P, w), ++raw_n) {
        const int r = raw_n % R;
        if (!mbar_wait(raw_full(r), (raw_n / R) & 1)) {
            ok = false;
            break;
        }
        float dcur[kHalfBlocks];
        float mcur[kHalfBlocks];
        if constexpr (kQ4K) {
            // header and quarters 2g, 2g + 1 (sub-blocks 4g .. 4g + 3); the stage is released
            // after the scaling of this super-step, which reads its block sums
            const uint8_t* rowp = base + L::kOffRaw + r * L::kStage + row * L::kRawRow;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(
                    rowp + (i == 0 ? 0 : 16 + 64 * g + 16 * (i - 1)));
                raw[4 * i] = v.x;
                raw[4 * i + 1] = v.y;
                raw[4 * i + 2] = v.z;
                raw[4 * i + 3] = v.w;
            }
            const uint4 hd = make_uint4(raw[0], raw[1], raw[2], raw[3]);
            uint32_t sc01, m01, sc23, m23;
            q4k_scales(hd, 2 * g, sc01, m01);
            q4k_scales(hd, 2 * g + 1, sc23, m23);
            const float dd = half_bits_to_float(raw[0] & 0xFFFFu);
            const float dm = half_bits_to_float(raw[0] >> 16);
            const uint32_t scs[4] = {sc01 & 0xFFu, sc01 >> 8, sc23 & 0xFFu, sc23 >> 8};
            const uint32_t ms[4] = {m01 & 0xFFu, m01 >> 8, m23 & 0xFFu, m23 >> 8};
#pragma unroll
            for (int blk = 0; blk < kHalfBlocks; ++blk) {
                dcur[blk] = __fmul_rn(dd, static_cast<float>(scs[blk]));
                mcur[blk] = __fmul_rn(dm, static_cast<float>(ms[blk]));
            }
        } else {
            const uint8_t* src =
                base + L::kOffRaw + r * L::kStage + row * L::kRawRow + g * (L::kRawRow / 2);
            uint32_t dep;
            if (g == 0) {
                load_half_row<0>(src, raw);
                dep = half_row_dep<0>(raw);
            } else {
                load_half_row<1>(src, raw);
                dep = half_row_dep<1>(raw);
            }
            release_to_async_proxy(dep);
            mbar_arrive(raw_empty(r));
#pragma unroll
            for (int blk = 0; blk < kHalfBlocks; ++blk) {
                dcur[blk] = half_bits_to_float(u16_at(raw, blk * kQ4Bytes));
                mcur[blk] = 0.0f;
            }
        }
        // The A slot of super-step n was last read by the MMAs of n - G (G = 2), which this
        // thread saw complete when it waited for acc_full(n - 2) while scaling it.
        static_assert(G == 2, "slot reuse follows the accumulator buffers");
        const int gi = raw_n % G;
        tc_fence_after();
        const uint32_t a_slot = a_lane + (g * G + gi) * kSlotCols;
        if constexpr (kQ4K) {
            uint32_t packed[16];
            q4k_codes<0>(raw + 4, packed);
            tmem_st16(a_slot, packed);
            q4k_codes<1>(raw + 4, packed);
            tmem_st16(a_slot + 16, packed);
            q4k_codes<0>(raw + 12, packed);
            tmem_st16(a_slot + 32, packed);
            q4k_codes<1>(raw + 12, packed);
            tmem_st16(a_slot + 48, packed);
        } else {
            {
                uint32_t packed[16];
                q4_codes_at<0 * kQ4Bytes>(raw, packed);
                tmem_st16(a_slot, packed);
            }
            {
                uint32_t packed[16];
                q4_codes_at<1 * kQ4Bytes>(raw, packed);
                tmem_st16(a_slot + 16, packed);
            }
            {
                uint32_t packed[16];
                q4_codes_at<2 * kQ4Bytes>(raw, packed);
                tmem_st16(a_slot + 32, packed);
            }
            {
                uint32_t packed[16];
                q4_codes_at<3 * kQ4Bytes>(raw, packed);
                tmem_st16(a_slot + 48, packed);
            }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(a_full(g, gi));
        if (prev_n >= 0) {
            if (!scale(prev_n, dprev, mprev) ||
                (prev_last && !finish_tile(prev_p, prev_row0, prev_rows, prev_slot))) {
                ok = false;
                break;
            }
        }
        prev_n = raw_n;
#pragma unroll
        for (int blk = 0; blk < kHalfBlocks; ++blk) {
            dprev[blk] = dcur[blk];
            mprev[blk] = mcur[blk];
        }
        prev_last = w.j == w.jend - 1;
        if (prev_last) {
            // a tile cut by this share's start (jbeg > 0) is partial slot 0, one cut by its
            // end slot 1
            prev_p = w.p;
            prev_row0 = w.row0;
            prev_rows = w.rows;
            prev_slot = w.jbeg > 0 ? 0 : (w.jend < w.nsuper ? 1 : -1);
        }
    }
    if (ok && prev_n >= 0) {
        ok = scale(prev_n, dprev, mprev);
        if (ok && prev_last) ok = finish_tile(prev_p, prev_row0, prev_rows, prev_slot);
    }
    if (ok && head_p >= 0) tc_finish_split<kNPad>(P, head_p, head_row0, head_rows, 0, quad, lane);
    tmem_st_wait();   // no TMEM store of this thread may be in flight when TMEM is freed
    if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
}

template <int kType, int kNPad, int kMaxProbs>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ TcParams<kMaxProbs> P) {
    using L = TcLayout<kType, kNPad>;
    constexpr int R = L::kRawStages;
    constexpr int G = L::kGroupSlots;
    constexpr int B = L::kAccBufs;
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
    auto acc_empty = [&](int b) { return bar0 + 8u * (2 * R + 4 * G + B + b); };
    const uint32_t mma_done = bar0 + 8u * (2 * R + 4 * G + 2 * B);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(raw_full(r), 1);
            // every dequantize thread once its half row is in registers, and each MMA
            // issuer's commit once its quarter's MMAs (the readers of its X) completed
            mbar_init(raw_empty(r), 32 * kDequantWarps + kMmaWarps);
        }
        for (int g = 0; g < 2; ++g)
            for (int i = 0; i < G; ++i) {
                mbar_init(a_full(g, i), 32 * kDequantWarps / 2);
                mbar_init(a_empty(g, i), 2);   // the two issuers of the group's quarters
            }
        for (int b = 0; b < B; ++b) {
            mbar_init(acc_full(b), kMmaWarps);
            // read out by the issuer warps, or in the scaled form by the dequantize warps
            mbar_init(acc_empty(b), 32 * (L::kScaled ? kDequantWarps : kMmaWarps));
        }
        mbar_init(mma_done, kMmaWarps);
        if constexpr (L::kScaled) {
            for (int i = 0; i < 2; ++i) mbar_init(mma_done + 8u * (1 + i), 32 * kDequantWarps / 2);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    __syncwarp();   // whole warps at the barrier (roles run on single lanes)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The next kernel of the stream may take SMs as this grid's CTAs leave.
    griddep_launch_dependents();

    TcWalk w;
    tc_walk_open(P, w, P.total_units * blockIdx.x / gridDim.x,
                 P.total_units * (blockIdx.x + 1) / gridDim.x);

    if (warp == 0) {
        // ---------------- producer (whole warp; lane 0 arms the barriers) ----------------
        // The weights of the first R super-steps go out before the previous kernel of the
        // stream has completed (they are read-only during the call; the dequantize warps
        // may already work on them); the X tiles, written by that kernel, after it.
        int n_pre = 0;
        {
            TcWalk pre = w;
            for (; pre.valid && n_pre < R; tc_walk_next(P, pre), ++n_pre) {
                if (lane == 0) {
                    const uint32_t dst = sRaw + n_pre * L::kStage;
                    mbar_arrive_expect_tx(raw_full(n_pre), L::kStageTx);   // raw + X bytes
                    // Whole 128-row box; rows past the matrix end are filled with zeros.
                    tma_load_2d(dst, &P.maps[pre.p], pre.j * (L::kRawRow / RawFmt<kType>::kElem),
                                static_cast<int>(pre.row0), raw_full(n_pre));
                }
            }
        }
        griddep_wait();
        int raw_n = 0;
        bool ok = true;
        for (; w.valid; tc_walk_next(P, w), ++raw_n) {
            const int r = raw_n % R;
            if (raw_n >= n_pre && !mbar_wait(raw_empty(r), ((raw_n / R) & 1) ^ 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = sRaw + r * L::kStage;
                if (raw_n >= n_pre) {
                    mbar_arrive_expect_tx(raw_full(r), L::kStageTx);
                    tma_load_2d(dst, &P.maps[w.p], w.j * (L::kRawRow / RawFmt<kType>::kElem),
                                static_cast<int>(w.row0), raw_full(r));
                }
                bulk_g2s(dst + L::kRaw, P.p[w.p].Xt + static_cast<int64_t>(w.j) * L::kXSlot,
                         L::kXCopy, raw_full(r));
            }
            __syncwarp();
        }
        if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
        if (lane == 0) {
            for (int i = max(0, raw_n - R); i < raw_n; ++i)
                mbar_wait(raw_full(i % R), (i / R) & 1, kDrainNs);
        }
    } else if (warp < kFirstDequantWarp) {
        // ---------------- MMA issuers, then epilogue ----------------
        // Issuer q (warps 1..4) owns the 64-k quarter q of every super-step and its own
        // accumulator per set, so the four issue in parallel (a single issuing thread
        // cannot keep the tensor core busy with N <= 64 MMAs). The four accumulators of
        // a tile are added in a fixed order by the same warps afterwards, each warp for
        // the TMEM lane quadrant it may access (warp % 4); with two sets this epilogue
        // runs after the next tile's first MMAs have been queued.
        griddep_wait();   // X tiles, Y, partial sums and counters of the previous kernel
        if constexpr (L::kScaled) {
            tc_issue_scaled<kType, kNPad, kMaxProbs>(P, w, tmem, sRaw, bar0);
        } else {
            const int q = warp - 1;
            const int g = q >> 1;                      // dequantize group that fills quarter q
            const int quad = warp & 3;
            const uint32_t tlane = static_cast<uint32_t>(quad * 32) << 16;
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kNPad);
            int tile = 0, raw_n = 0;
            bool ok = true;
            // epilogue of a finished tile; `slot` < 0: the whole tile, write Y; else a split
            // tile's partial sum, written to partial slot `slot` of this CTA
            int pend_p = -1, pend_rows = 0, pend_tile = 0, pend_slot = -1;
            int64_t pend_row0 = 0;
            int head_p = -1, head_rows = 0;
            int64_t head_row0 = 0;
            auto epilogue = [&](int p, int64_t row0, int rows, int t, int slot) -> bool {
                const int b = t % B;
                if (!warp_wait(acc_full(b), (t / B) & 1)) return false;
                tc_fence_after();
                const TcProb& pr = P.p[p];
                const int row = quad * 32 + lane;
                float* part = P.part + (static_cast<int64_t>(blockIdx.x) * 2 + max(slot, 0)) *
                                           (kNPad * kBM);
                const uint32_t acc = tmem + tlane + static_cast<uint32_t>(b * kQuarters * kNPad);
#pragma unroll
                for (int c = 0; c < kNPad; c += 16) {
                    // y = (acc0 + acc1) + (acc2 + acc3), the same order for every element
                    float y[16];
                    {
                        uint32_t v0[16], v1[16];
                        tmem_ld16(acc + 0 * kNPad + c, v0);
                        tmem_ld16(acc + 1 * kNPad + c, v1);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            y[jj] = __uint_as_float(v0[jj]) + __uint_as_float(v1[jj]);
                    }
                    {
                        uint32_t v2[16], v3[16];
                        tmem_ld16(acc + 2 * kNPad + c, v2);
                        tmem_ld16(acc + 3 * kNPad + c, v3);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            y[jj] += __uint_as_float(v2[jj]) + __uint_as_float(v3[jj]);
                    }
                    if (row < rows) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int n = c + jj;
                            if (n >= P.n_tok) continue;
                            if (slot < 0)
                                pr.Y[n * pr.M + row0 + row] = y[jj];
                            else
                                part[n * kBM + row] = y[jj];
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty(b));
                if (slot == 1) {
                    tc_finish_split<kNPad>(P, p, row0, rows, 1, quad, lane);
                } else if (slot == 0) {   // the share's first tile: finished after the last one
                    head_p = p;
                    head_row0 = row0;
                    head_rows = rows;
                }
                return true;
            };
            for (; w.valid && ok; tc_walk_next(P, w), ++raw_n) {
                const int b = tile % B;
                if (w.j == w.jbeg) {   // a new tile: its accumulator set must have been read out
                    if (!warp_wait(acc_empty(b), ((tile / B) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const int r = raw_n % R;
                const int gi = raw_n % G;
                if (!warp_wait(raw_full(r), (raw_n / R) & 1) ||      // the super-step's X landed
                    !warp_wait(a_full(g, gi), (raw_n / G) & 1)) {    // quarter q dequantized
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sX = sRaw + r * L::kStage + L::kRaw + q * L::kB;
                    const uint32_t a_col =
                        tmem + L::kAccCols + (g * G + gi) * kSlotCols + (q & 1) * (kBK / 2);
                    const uint32_t d = tmem + static_cast<uint32_t>((b * kQuarters + q) * kNPad);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_bf16_tmem_a(d, a_col + kk * 8, sw128_kmajor_desc(sX + kk * 32), idesc,
                                         (w.j != w.jbeg || kk != 0) ? 1u : 0u);
                    umma_commit(a_empty(g, gi));
                    umma_commit(raw_empty(r));
                    if (w.j == w.jend - 1) umma_commit(acc_full(b));
                }
                __syncwarp();
                if (B == 2 && w.j == w.jbeg && pend_p >= 0) {
                    if (!epilogue(pend_p, pend_row0, pend_rows, pend_tile, pend_slot)) {
                        ok = false;
                        break;
                    }
                    pend_p = -1;
                }
                if (w.j == w.jend - 1) {
                    // a tile cut by this share's start (jbeg > 0) is partial slot 0, one cut by
                    // its end slot 1
                    const int slot = w.jbeg > 0 ? 0 : (w.jend < w.nsuper ? 1 : -1);
                    if (B == 1) {
                        if (!epilogue(w.p, w.row0, w.rows, tile, slot)) {
                            ok = false;
                            break;
                        }
                    } else {
                        pend_p = w.p;
                        pend_row0 = w.row0;
                        pend_rows = w.rows;
                        pend_tile = tile;
                        pend_slot = slot;
                    }
                    ++tile;
                }
            }
            if (ok && pend_p >= 0) ok = epilogue(pend_p, pend_row0, pend_rows, pend_tile, pend_slot);
            if (ok && head_p >= 0) tc_finish_split<kNPad>(P, head_p, head_row0, head_rows, 0, quad, lane);
            // Completes when every MMA this thread issued has finished (also after a timeout),
            // so the TMEM release below never races an MMA in flight.
            if (lane == 0) umma_commit(mma_done);
            if (!ok && lane == 0) report_status(P.status, kStatusTimeout);
        }
    } else {
        if constexpr (L::kScaled) {
            tc_dequant_scaled<kType, kNPad, kMaxProbs>(P, w, tmem, base, bar0);
        } else {
            // ---------------- dequantize ----------------
            // Group g (warps 5..8 or 9..12) takes k [128 g, 128 g + 128) of every super-step
            // for all 128 rows; each warp its TMEM lane quadrant 32 * (warp % 4) + i, one row
            // per thread, written to the group's A slot with tcgen05.st.
            const int g = (warp - kFirstDequantWarp) >> 2;
            const int quad = warp & 3;
            const int row = quad * 32 + lane;
            const uint32_t a_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + L::kAccCols;
            int raw_n = 0;
            bool ok = true;
            // Q4_K: the 16 header bytes and 64 code bytes of the group's two quarters
            uint32_t raw[kType == GQ_TYPE_Q4_K ? 20 : kHalfWords];
            for (; w.valid && ok; tc_walk_next(P, w), ++raw_n) {
                const int r = raw_n % R;
                if (!mbar_wait(raw_full(r), (raw_n / R) & 1)) {
                    ok = false;
                    break;
                }
                // Every row of the box is loaded; rows past the matrix end arrive as zeros and
                // dequantize to zero operands (their outputs are dropped).
                if constexpr (kType == GQ_TYPE_Q4_K) {
                    // the super-block's 16 header bytes and the code bytes of its quarters
                    // 2g and 2g + 1 (sub-blocks 4g .. 4g + 3): raw[0..3], raw[4..19]
                    const uint8_t* rowp = base + L::kOffRaw + r * L::kStage + row * L::kRawRow;
                    uint32_t dep = 0;
#pragma unroll
                    for (int i = 0; i < 5; ++i) {
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            rowp + (i == 0 ? 0 : 16 + 64 * g + 16 * (i - 1)));
                        raw[4 * i] = v.x;
                        raw[4 * i + 1] = v.y;
                        raw[4 * i + 2] = v.z;
                        raw[4 * i + 3] = v.w;
                        dep ^= v.x;
                    }
                    release_to_async_proxy(dep);
                } else {
                    const uint8_t* src = base + L::kOffRaw + r * L::kStage + row * L::kRawRow +
                                         g * (L::kRawRow / 2);
                    uint32_t dep;
                    if (g == 0) {
                        load_half_row<0>(src, raw);
                        dep = half_row_dep<0>(raw);
                    } else {
                        load_half_row<1>(src, raw);
                        dep = half_row_dep<1>(raw);
                    }
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
                if constexpr (kType == GQ_TYPE_Q4_K) {
                    const uint4 hd = make_uint4(raw[0], raw[1], raw[2], raw[3]);
                    uint32_t packed[16];
                    dequant_q4k_sub<0>(hd, 2 * g, raw + 4, packed);
                    tmem_st16(a_slot, packed);
                    dequant_q4k_sub<1>(hd, 2 * g, raw + 4, packed);
                    tmem_st16(a_slot + 16, packed);
                    dequant_q4k_sub<0>(hd, 2 * g + 1, raw + 12, packed);
                    tmem_st16(a_slot + 32, packed);
                    dequant_q4k_sub<1>(hd, 2 * g + 1, raw + 12, packed);
                    tmem_st16(a_slot + 48, packed);
                } else {
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
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(a_full(g, gi));
            }
            if (!ok) report_status(P.status, kStatusTimeout);
        }
    }
    __syncwarp();   // whole warps at the barrier (roles run on single lanes)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) mbar_wait(mma_done, 0, kDrainNs);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Arguments of x_tiles_kernel: every tensor-core decode problem of a call.
struct XtProb {
    const float* X;
    uint8_t* Xt;
    int64_t K;
    int32_t block_begin;   // first block of x_tiles_kernel that works on this problem
    int32_t x_aligned;     // X is 16-byte aligned: vector loads
};
constexpr int kXtChunksPerBlock = 1024;   // 4 per thread (256 threads)
// A launch that would have fewer blocks than SMs takes 256 chunks per block (one per
// thread) instead: more blocks, each one load latency long.
constexpr int kXtChunksPerBlockSmall = 256;
struct XtParams {
    int32_t count;
    int32_t n_tok;
    int* counters;
    int32_t n_counters;
    int32_t sums;        // append each super-step's 8 x kNPad block sums (Q4_K scaled form)
    int32_t chunks_per_block;   // kXtChunksPerBlock or kXtChunksPerBlockSmall
    XtProb p[GQ_MAX_BATCH];
};

// Bytes of one super-step's X in the workspace (and in a stage): four kNPad x 64 bf16
// tiles, and with block sums a 1 KB slot holding 8 x kNPad fp32 sums.
__host__ __device__ constexpr int64_t xt_superstep_bytes(int npad, bool sums) {
    return int64_t(4) * npad * kBK * 2 + (sums ? 1024 : 0);
}

// X (n_tok x K fp32, rows of K) -> kNPad x 64 bf16 tiles per 64-k stage, each row 128 bytes
// with 16-byte chunk c stored at c ^ (row % 8); tokens >= n_tok are zero. Four tiles form a
// super-step's slot (xt_superstep_bytes); with P.sums the slot also holds, for each of its
// eight 32-k blocks b and token n, the fp32 sum of the block's bf16 values at float
// index b * kNPad + n after the tiles (four threads' chunks, added by a fixed shuffle
// tree). One launch for all problems: each problem gets a run of blocks, each block 1024
// of its 16-byte output chunks. Block 0 also clears the split-tile counters of the decode
// kernels that follow.
template <int kNPad>
__global__ void __launch_bounds__(256)
x_tiles_kernel(const __grid_constant__ XtParams P) {
    // The tensor-core kernel after this one may start filling its weight rings already;
    // the tiles and counters may still be in use by the previous kernel of the stream.
    griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < P.n_counters; i += blockDim.x) P.counters[i] = 0;
    int lo = 0, hi = P.count - 1;   // the problem of this block: last block_begin <= block
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].block_begin <= static_cast<int>(blockIdx.x))
            lo = mid;
        else
            hi = mid - 1;
    }
    const XtProb& pr = P.p[lo];
    const int64_t chunks = pr.K / kBK * kNPad * 8;
    const int64_t first = static_cast<int64_t>(blockIdx.x - pr.block_begin) * P.chunks_per_block;
    const int64_t last = min(chunks, first + P.chunks_per_block);
    // Every chunk of the thread is loaded before any is converted, so that all of them are
    // in flight at once: a launch for few problems (a handful of blocks) is then one load
    // latency long, not kXtPerThread of them.
    constexpr int kXtPerThread = kXtChunksPerBlock / 256;
    float v[kXtPerThread][8];
#pragma unroll
    for (int i = 0; i < kXtPerThread; ++i) {
        const int64_t li = first + threadIdx.x + 256 * i;
        const int c = static_cast<int>(li & 7);
        const int n = static_cast<int>((li >> 3) % kNPad);
        const int64_t ks = (li >> 3) / kNPad;
        if (li < last && n < P.n_tok) {
            const float* x = pr.X + n * pr.K + ks * kBK + 8 * c;
            if (pr.x_aligned) {
                const float4 a = *reinterpret_cast<const float4*>(x);
                const float4 b = *reinterpret_cast<const float4*>(x + 4);
                v[i][0] = a.x; v[i][1] = a.y; v[i][2] = a.z; v[i][3] = a.w;
                v[i][4] = b.x; v[i][5] = b.y; v[i][6] = b.z; v[i][7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = x[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = 0.0f;
        }
    }
#pragma unroll
    for (int i = 0; i < kXtPerThread; ++i) {
        const int64_t li = first + threadIdx.x + 256 * i;
        if (li >= last) break;   // block-uniform: chunk counts are multiples of 512
        const int c = static_cast<int>(li & 7);
        const int n = static_cast<int>((li >> 3) % kNPad);
        const int64_t ks = (li >> 3) / kNPad;
        uint32_t packed[4];
        float part = 0.0f;   // this chunk's share of its block sum (the bf16 values)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[i][2 * e], v[i][2 * e + 1]);
            packed[e] = *reinterpret_cast<const uint32_t*>(&b);
            part += __low2float(b) + __high2float(b);
        }
        uint8_t* slot = pr.Xt + (ks >> 2) * xt_superstep_bytes(kNPad, P.sums != 0);
        *reinterpret_cast<uint4*>(slot + (ks & 3) * (kNPad * 128) + n * 128 + ((c ^ (n & 7)) << 4)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        if (P.sums) {   // uniform across the block: the same for every problem of a launch
            // chunks c = 4h .. 4h + 3 of one token row are threads li .. li + 3 (li % 4 ==
            // 0 at c = 4h): block 2 (ks % 4) + h of the super-step
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
            if ((c & 3) == 0) {
                const int blk = 2 * static_cast<int>(ks & 3) + (c >> 2);
                reinterpret_cast<float*>(slot + 4 * kNPad * 128)[blk * kNPad + n] = part;
            }
        }
    }
}

// A launch with the programmatic-stream-serialization attribute: the kernel may be
// scheduled before the previous kernel of the stream has completed, and orders itself
// after it with griddepcontrol.wait.
cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
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
    const int64_t row_bytes = (K / kSuperK) * RawFmt<kType>::kRow;
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

// Start of the workspace: two 128 x kNPad fp32 partial-sum tiles per CTA, then the
// split-tile counters (one per CTA boundary and lane quadrant), then the X tiles.
int64_t tc_part_bytes(int npad) { return int64_t(2) * kMaxTcGrid * kBM * npad * 4; }
constexpr int kCounters = kMaxTcGrid * 4;
constexpr int64_t kCounterBytes = kCounters * 4;   // 4 KB, keeps the X tiles 256-aligned

template <int kNPad>
cudaError_t launch_x_tiles(const MatProblem* probs, int count, int64_t N, uint8_t* part,
                           uint8_t* xt, bool sums, const DeviceInfo* info, cudaStream_t s) {
    XtParams P{};
    P.count = count;
    P.n_tok = static_cast<int32_t>(N);
    P.counters = reinterpret_cast<int*>(part + tc_part_bytes(kNPad));
    P.n_counters = kCounters;
    P.sums = sums ? 1 : 0;
    int64_t big = 0;
    for (int i = 0; i < count; ++i)
        big += (probs[i].K / kBK * kNPad * 8 + kXtChunksPerBlock - 1) / kXtChunksPerBlock;
    const int cpb = big < info->sm_count ? kXtChunksPerBlockSmall : kXtChunksPerBlock;
    P.chunks_per_block = cpb;
    int64_t blocks = 0, off = 0;
    for (int i = 0; i < count; ++i) {
        P.p[i].X = probs[i].X;
        P.p[i].Xt = xt + off;
        P.p[i].K = probs[i].K;
        P.p[i].block_begin = static_cast<int32_t>(blocks);
        P.p[i].x_aligned = reinterpret_cast<uintptr_t>(probs[i].X) % 16 == 0 && probs[i].K % 4 == 0;
        blocks += (probs[i].K / kBK * kNPad * 8 + cpb - 1) / cpb;
        off += probs[i].K / kSuperK * xt_superstep_bytes(kNPad, sums);
    }
    void* args[] = {&P};
    return launch_pdl(reinterpret_cast<const void*>(x_tiles_kernel<kNPad>),
                      dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, args);
}

template <int kType, int kNPad, int kMaxProbs>
cudaError_t launch_tc_t(const MatProblem* probs, int count, int64_t N, uint8_t* part,
                        uint8_t* xt, const DeviceInfo* info, cudaStream_t s) {
    using L = TcLayout<kType, kNPad>;
    static_assert(sizeof(TcParams<kMaxProbs>) <= 32000, "kernel parameter space");
    TcParams<kMaxProbs> P{};
    P.count = count;
    P.n_tok = static_cast<int32_t>(N);
    P.status = info->status;
    P.part = reinterpret_cast<float*>(part);
    P.counters = reinterpret_cast<int*>(part + tc_part_bytes(kNPad));
    int64_t units = 0, xt_off = 0;
    for (int i = 0; i < count; ++i) {
        TcProb& g = P.p[i];
        g.W = probs[i].W;
        g.X = probs[i].X;
        g.Xt = xt + xt_off;
        g.Y = probs[i].Y;
        g.M = probs[i].M;
        g.K = static_cast<int32_t>(probs[i].K);
        g.row_bytes = (probs[i].K / kSuperK) * RawFmt<kType>::kRow;
        g.nsuper = static_cast<int32_t>(probs[i].K / kSuperK);
        g.unit_begin = units;
        units += (g.M + kBM - 1) / kBM * g.nsuper;
        xt_off += probs[i].K / kSuperK * xt_superstep_bytes(kNPad, L::kSums);
        cudaError_t e = weight_map<kType>(probs[i].W, probs[i].M, probs[i].K, &P.maps[i]);
        if (e != cudaSuccess) return e;
    }
    P.total_units = units;
    auto kernel = gemv_tc_kernel<kType, kNPad, kMaxProbs>;
    cudaError_t e = ensure_smem(kernel, info->device, L::kAlloc);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>({units, info->sm_count, kMaxTcGrid})));
    void* args[] = {&P};
    return launch_pdl(reinterpret_cast<const void*>(kernel), dim3(static_cast<unsigned>(grid)),
                      dim3(kThreads), static_cast<size_t>(L::kAlloc), s, args);
}

template <int kType, int kMaxProbs>
cudaError_t launch_tc_np(const MatProblem* probs, int count, int64_t N, uint8_t* part,
                         uint8_t* xt, const DeviceInfo* info, cudaStream_t s) {
    switch (npad_for(N)) {
        case 16: return launch_tc_t<kType, 16, kMaxProbs>(probs, count, N, part, xt, info, s);
        case 32: return launch_tc_t<kType, 32, kMaxProbs>(probs, count, N, part, xt, info, s);
        default: return launch_tc_t<kType, 64, kMaxProbs>(probs, count, N, part, xt, info, s);
    }
}

template <int kType>
cudaError_t launch_tc_type(const MatProblem* probs, int count, int64_t N, uint8_t* part,
                           uint8_t* xt, const DeviceInfo* info, cudaStream_t s) {
    if (count == 1) return launch_tc_np<kType, 1>(probs, count, N, part, xt, info, s);
    if (count <= 16) return launch_tc_np<kType, 16>(probs, count, N, part, xt, info, s);
    return launch_tc_np<kType, kMaxLaunchProbs>(probs, count, N, part, xt, info, s);
}

}  // namespace

bool gemv_tc_eligible(gq_type t, const MatProblem& p, int64_t N) {
    if (block_bytes_of(t) == 0) return false;
    if (N < kGemvTcMinTokens || N > kGemvTcMaxTokens) return false;
    if (p.K % kSuperK != 0 || p.K > (int64_t(1) << 24) || p.M <= 0) return false;
    return reinterpret_cast<uintptr_t>(p.W) % 16 == 0 && reinterpret_cast<uintptr_t>(p.X) % 4 == 0;
}

// Whether the X slots of this call carry the block sums: the scaled form of Q4_K.
bool tc_sums(gq_type t, int64_t N) { return t == GQ_TYPE_Q4_K && npad_for(N) == 16; }

int64_t gemv_tc_workspace_bytes(gq_type t, const MatProblem* probs, int count, int64_t N) {
    const int npad = npad_for(N);
    int64_t b = tc_part_bytes(npad) + kCounterBytes;
    for (int i = 0; i < count; ++i)
        b += probs[i].K / kSuperK * xt_superstep_bytes(npad, tc_sums(t, N));
    return b;
}

cudaError_t launch_gemv_tc(gq_type t, const MatProblem* probs, int count, int64_t N,
                           void* workspace, cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    // Workspace: the partial sums (reused by every launch, in stream order), then the X
    // tiles of all problems one after another. Launches take at most kMaxLaunchProbs.
    uint8_t* part = static_cast<uint8_t*>(workspace);
    uint8_t* xt = part + tc_part_bytes(npad_for(N)) + kCounterBytes;
    const bool sums = tc_sums(t, N);
    switch (npad_for(N)) {
        case 16: e = launch_x_tiles<16>(probs, count, N, part, xt, sums, info, s); break;
        case 32: e = launch_x_tiles<32>(probs, count, N, part, xt, false, info, s); break;
        default: e = launch_x_tiles<64>(probs, count, N, part, xt, false, info, s); break;
    }
    if (e != cudaSuccess) return e;
    for (int i0 = 0; i0 < count; i0 += kMaxLaunchProbs) {
        const int n = std::min(kMaxLaunchProbs, count - i0);
        e = t == GQ_TYPE_Q4_0   ? launch_tc_type<GQ_TYPE_Q4_0>(probs + i0, n, N, part, xt, info, s)
            : t == GQ_TYPE_Q4_K ? launch_tc_type<GQ_TYPE_Q4_K>(probs + i0, n, N, part, xt, info, s)
                                : launch_tc_type<GQ_TYPE_Q8_0>(probs + i0, n, N, part, xt, info, s);
        if (e != cudaSuccess) return e;
        for (int i = i0; i < i0 + n; ++i)
            xt += probs[i].K / kSuperK * xt_superstep_bytes(npad_for(N), sums);
    }
    return cudaSuccess;
}

}  // namespace gq
