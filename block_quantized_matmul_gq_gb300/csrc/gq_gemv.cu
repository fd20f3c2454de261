// gq_gemv.cu -- decode-side mul_mat (few tokens): Y[n][m] = sum_k What[m][k] * X[n][k].
//
// At decode the product is a matrix-vector product that streams every weight once
// ("A Complete Guide to llama.cpp and Customization with C++", section 2.1) and is
// bound by memory bandwidth; the weights are dequantized right after they are loaded
// ("No Python! Building an AI Inference Engine Exclusively in C++", section 9;
// "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++", section 6.2:
// load, unpack with masks and shifts, scale, multiply-accumulate).
//
// GB300 design (not the pages' CPU/SIMD one):
//  * One persistent CTA per SM. All problems of a launch form one sequence of rows; each
//    CTA takes a contiguous, row-aligned share of equal estimated time (bytes plus a fixed
//    cost per ring stage), so small matrices (GQA k/v projections) ride along with large
//    ones and no CTA idles on a tail. The host computes the shares and passes them in the
//    kernel parameters: searching the problem table on the device cost every CTA one
//    dependent parameter load per earlier problem before its first copy (0.18 us per
//    problem of the launch, measured).
//  * Inside a CTA, each warp owns tiles of 4 rows and walks their K columns in column
//    groups of eight "chunks" (a chunk is 8 Q4_0 blocks = 144 B = 256 weights, or 4 Q8_0
//    blocks = 136 B = 128 weights), one ring stage per group. Every warp streams its own
//    tiles through a private ring of shared-memory stages filled by 1-D bulk copies (TMA
//    cp.async.bulk, L2 evict-first) issued by one lane -- a single copy when the stage
//    holds whole rows (K <= 2048 for Q4_0), else one per row -- completing on a per-warp
//    mbarrier; warps never wait for each other inside a problem. Rows are whole chunks
//    (K % 256 == 0), so copies are 16-byte aligned.
//  * Lanes and data. Q4_0: lane l takes block pair l (36 bytes) of the column group in all
//    four rows of the tile, so it reads the pair's activations from shared memory once
//    per tile, not once per row (with a lane per row and chunk, every 16-byte activation
//    load cost four shared-memory wavefronts, one per quarter warp, and the wavefronts
//    ran at 59 % of the pipe's peak). Q8_0 and the quantized-activation form: lane l
//    takes chunk l % 8 of row l / 8.
//  * Activations: at each problem boundary the CTA converts X into 16-bit block fixed
//    point in shared memory (one power-of-two scale 2^e per chunk), so the inner product
//    of a 32-weight block is EXACT integer arithmetic with dp2a (two 16x8-bit products
//    per instruction):
//        S = sum_i (16 (c_i - 8)) * x16_i       (Q4_0; codes become signed bytes 16(c-8))
//        S = sum_i c_i * x16_i                  (Q8_0)
//    then acc += d * float(S) and, per chunk, partial = acc * 2^(e - 15). The only
//    approximation is x16 = rint(x * 2^(15 - e)), 2^(e - 1) <= max |x| < 2^e, clamped to
//    +-32767: per element the rounding errs by at most 2^(e - 16) <= max |x| 2^-15 (the
//    clamp, where it acts, by at most |x| / 32767.5), so per chunk ||x - xhat||_2 <=
//    ||x_chunk|| (1 / 2048 + 1 / 32767.5), and by Cauchy-Schwarz |error| <= 0.52 of the
//    bound 1e-3 ||x|| ||What||, whatever the inputs.
//  * Q4_K super-blocks (the published GGUF Q4_K layout) stream in the geometry of Q4_0:
//    a chunk is one 144-byte super-block, and lane l takes quarter l % 4 (sub-blocks 2g,
//    2g + 1) of super-block l / 4 in all four rows of the tile; per row the sub-block sums
//    S_j = sum q x16 and X_j = sum x16 are exact integers, combined as
//    d (sc S + sc' S') - dmin (m X + m' X') in fp32 (quarter_dot_q4k).
//  * A lane keeps its running sums in registers across all columns; at the tile's end
//    the lanes' sums of each row are added with shuffles in a fixed order (Q4_0: a
//    transposed reduction of the four rows; otherwise the eight lanes of a row). When a
//    CTA's part of a problem has fewer 4-row tiles than warps, each tile's columns are
//    split between warps and the per-warp sums are added in a fixed order in shared
//    memory: deterministic, no atomics.
//  * Waits are bounded: a stage that never arrives sets the device status word; the CTA
//    leaves at the next problem boundary after draining its own copies.
//  * Fused forms of the same kernel: RMSNorm of X folded into the activation preparation
//    (per-token 1 / rms in a fixed-order reduction, times gamma, before the fixed-point
//    conversion), and gate/up row pairs (row 2m from the gate matrix, 2m + 1 from the up
//    matrix, adjacent lanes' sums combined into Swish(g) * u), so the SwiGLU output is
//    written once and the intermediate products never reach HBM ("Development Guide for
//    Small AI Models (TinyLLaMA, etc.) Using C++", sections 4.1 and 4.4).
// Shapes the streaming kernel does not take (K % 256 != 0, unaligned X, very large K)
// run on gemv_generic_kernel: one warp per row, plain loads, fp32 FMA.
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// Build-time tuning: warps per CTA and ring depth per warp (for <= 3 tokens / 4 tokens).
#ifndef GQ_GEMV_WARPS
#define GQ_GEMV_WARPS 16
#endif
#ifndef GQ_GEMV_STAGES
#define GQ_GEMV_STAGES 2
#endif
#ifndef GQ_GEMV_STAGES_N4
#define GQ_GEMV_STAGES_N4 2
#endif
constexpr int kWarps = GQ_GEMV_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kLanesPerRow = 8;               // one chunk per lane, 8 chunks per row per stage
constexpr int kTileRows = 32 / kLanesPerRow;   // 4 rows per warp tile
constexpr int kMaxTok = 4;                     // tokens per pass of the weight stream
// The same with Q8_0-quantized activations: their records are smaller, but more tokens per
// pass measured no faster (the per-token block sums bind from 4 tokens on: 212 us for 4,
// 431 us for 8 on the TinyLLaMA step).
constexpr int kMaxTokQ8x = 4;
// Ring depth per warp: deeper while the x16 buffer is small (<= 3 tokens).
template <int kNT>
__host__ __device__ constexpr int ring_stages() {
    return kNT <= 3 ? GQ_GEMV_STAGES : GQ_GEMV_STAGES_N4;
}

template <int kType>
struct Fmt;
template <>
struct Fmt<GQ_TYPE_Q4_0> {
    static constexpr int kBB = kQ4Bytes;
    static constexpr int kWeights = 32;
    static constexpr int kBlocksPerChunk = 8;
    static constexpr int kCodeShift = 4;   // dp2a sums come out as 16 * sum (c - 8) x16
};
template <>
struct Fmt<GQ_TYPE_Q8_0> {
    static constexpr int kBB = kQ8Bytes;
    static constexpr int kWeights = 32;
    static constexpr int kBlocksPerChunk = 4;
    static constexpr int kCodeShift = 0;
};
template <>
struct Fmt<GQ_TYPE_Q4_K> {   // a chunk is one super-block
    static constexpr int kBB = kQ4KBytes;
    static constexpr int kWeights = kQ4KWeights;
    static constexpr int kBlocksPerChunk = 1;
    static constexpr int kCodeShift = 0;
};

template <int kType>
struct Geo {
    static constexpr int kBB = Fmt<kType>::kBB;
    static constexpr int kBPC = Fmt<kType>::kBlocksPerChunk;
    static constexpr int kChunkBytes = kBB * kBPC;                 // 144 or 136
    static constexpr int kChunkWords = kChunkBytes / 4;            // 36 or 34
    static constexpr int kWPC = Fmt<kType>::kWeights * kBPC;       // weights per chunk: 256 / 128
    static constexpr int kRowStride = kLanesPerRow * kChunkBytes;  // 1152 or 1088 in a stage
    // One stage of one warp: 4 rows x 8 chunks, padded to 128-byte multiples.
    static constexpr int kStageBytes = (kTileRows * kRowStride + 127) / 128 * 128;
    // x16 record of one chunk for one token.
    //  Q4_0: four 144-byte pair records, one per pair of blocks (64 elements): their 64
    //   int16, one int bias per block (-128 * sum of the block's x16, the code offset 8
    //   folded in), then two float factors whose product is the chunk's power-of-two
    //   scale. A lane reads one pair record (pair_dot_q4); records 9 units of 16 bytes
    //   apart put the 8 lanes of a quarter warp in 8 different groups of 4 banks.
    //  Q4_K: the same four records, one per quarter of the super-block (sub-blocks 2g and
    //   2g + 1); the two ints are the plain sums of the sub-blocks' x16 (for the mins).
    //  Q8_0: kWPC int16, then the two scale factors; record stride 68 words (4 mod 32),
    //   so the 8 columns a warp reads sit in 8 different groups of 4 banks.
    static constexpr int kScaleOff = kWPC * 2;                     // Q8_0
    static constexpr int kXRec = kType == GQ_TYPE_Q8_0 ? kScaleOff + 16 : 4 * 144;  // 272 / 576
};

// Q4_0 pair record and Q4_K quarter record (see Geo): 64 int16 x16, two ints (Q4_0: biases;
// Q4_K: sub-block sums), two float scale factors.
struct Q4Pair {
    static constexpr int kRec = 144;
    static constexpr int kBiasOff = 128;
    static constexpr int kScaleOff = 136;
};
static_assert(Geo<GQ_TYPE_Q4_0>::kXRec == 4 * Q4Pair::kRec, "four pair records per chunk");
static_assert(Geo<GQ_TYPE_Q4_K>::kXRec == 4 * Q4Pair::kRec, "four quarter records per chunk");
static_assert(Geo<GQ_TYPE_Q4_K>::kChunkBytes == Geo<GQ_TYPE_Q4_0>::kChunkBytes &&
                  Geo<GQ_TYPE_Q4_K>::kChunkWords == Geo<GQ_TYPE_Q4_0>::kChunkWords,
              "Q4_K streams in the stage geometry of Q4_0");

struct GemvProb {
    const uint8_t* W;
    const float* X;
    float* Y;
    int64_t M;
    int64_t row_bytes;
    int64_t row_cost;     // balancing weight of one row (see kGroupCost)
    int64_t cost_begin;   // weight of all earlier problems
    int32_t C;            // chunks per row
    int32_t K;
    // Fused forms. gamma != NULL: X is RMS-normalized per token (x / sqrt(mean x^2 + eps)
    // * gamma) as it is prepared. W2 != NULL: gate/up pairs -- the row sequence has M =
    // 2 M_h rows, row 2m from W (gate m) and row 2m + 1 from W2 (up m), and Y (rows of
    // M_h) receives Swish(gate) * up.
    const uint8_t* W2;
    const float* gamma;
    float eps;
    int32_t pad_;
};

// Largest grid of the streaming kernel: the CTA shares travel as a table of kMaxGrid + 1
// cuts in the kernel parameters.
constexpr int kMaxGrid = 256;

template <int kMaxProbs>
struct GemvParams {
    // CTA c streams from row cut_r[c] of problem cut_p[c] up to (not including) row
    // cut_r[c + 1] of problem cut_p[c + 1]; (count, 0) is the end. Computed on the host:
    // finding them on the device meant a scan of the problem table, one dependent
    // parameter load per problem, before the CTA's first copy.
    int64_t cut_r[kMaxGrid + 1];
    int32_t cut_p[kMaxGrid + 1];
    int32_t count;
    int32_t n_tok;        // valid tokens of this pass, 1..kMaxTok
    int32_t max_c;        // largest C: the x buffer holds kNT * max_c records
    int32_t pad_;
    int64_t total_bytes;
    int64_t total_cost;
    unsigned* status;
    GemvProb p[kMaxProbs];
};

// CTA shares balance an estimate of time rather than bytes: a row weighs its bytes plus
// kGroupCost for each column group (one ring stage per 4-row tile), the part of a stage's
// cost that does not scale with its bytes (waits, refill, shuffles; a partly filled last
// group costs the same as a full one). 576 was the best of 0 / 576 / 1152 / 2304 / 4608
// measured on the TinyLLaMA and LLaMA-7B sets (Q4_0 and Q8_0, N = 1 and 2).
constexpr int64_t kGroupCost = 576;
// Balancing weight of a problem boundary inside a CTA's share: the CTA prepares that
// problem's activations and synchronizes its warps before streaming it (~2 us per extra
// problem in a clock-stamped trace of the TinyLLaMA and LLaMA-7B steps, where the CTAs
// with four or five problems finished up to 12 us after those with one). Long rows (more
// than one column group, one copy per row per stage) were slower per byte than their
// weight said, the longest the most (LLaMA-7B down_proj, K = 11008: +19 %).
//   Q8_0: kSegCost per boundary, kRowCopyCost more per column group of a long row.
//   Q4_0 / Q4_K: kSegCost4 per boundary, and per column group of a row with g groups
//   kLongRowCost4 * (g - 2) more (fitted to the per-CTA end times: TinyLLaMA K = 5632 and
//   LLaMA-7B K = 11008 rows). Q8_0 rows have twice the chunks at the same K, and this form
//   overweighted its K = 5632 rows (N = 2: 182.6 -> 190.7 us), so Q8_0 keeps the flat one.
constexpr int64_t kSegCost = 65536;
constexpr int64_t kRowCopyCost = 256;
constexpr int64_t kSegCost4 = 131072;
constexpr int64_t kLongRowCost4 = 143;

// First row (problem p, row r) whose weight begins at or after `cost`; (count, 0) = end.
// Host side: the cuts of the CTA shares (GemvParams::cut_p / cut_r). Costs increase with
// the cut, so the search starts at the previous cut's problem `p`.
template <int kMaxProbs>
void row_at_cost(const GemvParams<kMaxProbs>& P, int64_t cost, int& p, int64_t& r) {
    p = std::min(p, P.count - 1);
    while (p + 1 < P.count && P.p[p + 1].cost_begin <= cost) ++p;
    const int64_t off = cost - P.p[p].cost_begin;
    r = off <= 0 ? 0 : (off + P.p[p].row_cost - 1) / P.p[p].row_cost;
    if (P.p[p].W2 != nullptr) r = (r + 1) & ~int64_t(1);   // gate/up pairs stay together
    if (r >= P.p[p].M) {
        ++p;
        r = 0;
    }
}

// A CTA's share is a list of segments: one problem each, a row range [rb, re).
struct Segment {
    int p;
    int64_t rb, re;
    bool valid;
};

template <int kMaxProbs>
__device__ Segment find_segment(const GemvParams<kMaxProbs>& P, int p, int64_t rb, int p_end,
                                int64_t r_end) {
    for (; p < P.count && p <= p_end; ++p, rb = 0) {
        const int64_t re = (p == p_end) ? r_end : P.p[p].M;
        if (re > rb) return Segment{p, rb, re, true};
    }
    return Segment{0, 0, 0, false};
}

// How a segment is cut into work items: 4-row tiles whose K runs in column groups of 8
// chunks (one stage each); when there are fewer tiles than warps, each tile's column
// groups split into `ksplit` ranges so every warp works.
struct SegPlan {
    int ntiles, ncs, ksplit, items;
};

__device__ __forceinline__ SegPlan plan_segment(int64_t rows, int C) {
    SegPlan s;
    s.ntiles = static_cast<int>((rows + kTileRows - 1) / kTileRows);
    s.ncs = (C + kLanesPerRow - 1) / kLanesPerRow;
    s.ksplit = s.ntiles >= kWarps ? 1 : max(1, min(s.ncs, kWarps / s.ntiles));
    s.items = s.ntiles * s.ksplit;
    return s;
}

// Column-group range [cs_begin, cs_end) of k-group kg.
__device__ __forceinline__ void kgroup_range(const SegPlan& sp, int kg, int& cb, int& ce) {
    cb = kg * sp.ncs / sp.ksplit;
    ce = (kg + 1) * sp.ncs / sp.ksplit;
}

// One warp's walk through its stages: segment -> its items (item = warp, warp + kWarps,
// ...) -> column pairs of the item. Uniform across the lanes of the warp.
struct WarpCursor {
    Segment seg;
    SegPlan plan;
    int item, tile;
    int cs, ce;           // current column group and end of the item's range
    bool valid;
};

// Tile and column-group range of the cursor's item. No division when ksplit == 1, the
// common case (every stage of a K <= 2048 Q4_0 problem is its own item).
__device__ __forceinline__ void item_bounds(const SegPlan& sp, int item, int& tile, int& cb,
                                            int& ce) {
    if (sp.ksplit == 1) {
        tile = item;
        cb = 0;
        ce = sp.ncs;
    } else {
        tile = item / sp.ksplit;
        kgroup_range(sp, item - tile * sp.ksplit, cb, ce);
    }
}

template <int kMaxProbs>
__device__ void cursor_item(const GemvParams<kMaxProbs>& P, WarpCursor& c) {
    item_bounds(c.plan, c.item, c.tile, c.cs, c.ce);
}

template <int kMaxProbs>
__device__ void cursor_enter(const GemvParams<kMaxProbs>& P, WarpCursor& c, Segment seg,
                             int warp, int p_end, int64_t r_end) {
    while (seg.valid) {
        const SegPlan sp = plan_segment(seg.re - seg.rb, P.p[seg.p].C);
        if (warp < sp.items) {
            c.seg = seg;
            c.plan = sp;
            c.item = warp;
            c.valid = true;
            cursor_item(P, c);
            return;
        }
        seg = find_segment(P, seg.p + 1, 0, p_end, r_end);
    }
    c.valid = false;
}

template <int kMaxProbs>
__device__ void cursor_advance(const GemvParams<kMaxProbs>& P, WarpCursor& c, int warp,
                               int p_end, int64_t r_end) {
    if (++c.cs < c.ce) return;
    c.item += kWarps;
    if (c.item < c.plan.items) {
        cursor_item(P, c);
        return;
    }
    cursor_enter(P, c, find_segment(P, c.seg.p + 1, 0, p_end, r_end), warp, p_end, r_end);
}

__device__ __forceinline__ uint32_t word_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? __funnelshift_r(r[w], r[w + 1], 16) : r[w];
}

__device__ __forceinline__ uint32_t u16_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? (r[w] >> 16) : (r[w] & 0xFFFFu);
}

// Swish(z) = z / (1 + e^-z) ("Development Guide for Small AI Models (TinyLLaMA, etc.)
// Using C++", section 4.4).
__device__ __forceinline__ float swish(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// RMSNorm scale of each token of the problem ("Development Guide for Small AI Models
// (TinyLLaMA, etc.) Using C++", section 4.1): inv[t] = 1 / sqrt(mean_k x^2 + eps). The sum
// of squares runs in a fixed order (thread strides, a fixed shuffle tree, then the warps
// in order through `scratch`, kWarps * kNT floats), so it does not depend on timing. All
// threads of the CTA call it.
template <int kNT>
__device__ void rms_scales(const GemvProb& pr, int n_tok, float* scratch, float (&inv)[kNT]) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        float ss = 0.0f;
        if (t < n_tok) {
            const float* x = pr.X + static_cast<int64_t>(t) * pr.K;
            for (int k = threadIdx.x; k < pr.K; k += kThreads) ss = fmaf(x[k], x[k], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        if (lane == 0) scratch[warp * kNT + t] = ss;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        float ss = 0.0f;
        for (int w = 0; w < kWarps; ++w) ss += scratch[w * kNT + t];
        inv[t] = 1.0f / sqrtf(ss / static_cast<float>(pr.K) + pr.eps);
    }
    __syncthreads();   // scratch is the k-split buffer of the segment that follows
}

// X (n_tok x K fp32) -> x16 records, one per (token, chunk column). Warp per record.
// With kNorm (pr.gamma set), each x is first RMS-normalized: x * inv_rms[t] * gamma[k].
template <int kType, int kNT, bool kNorm>
__device__ void prepare_x(const GemvProb& pr, int n_tok, int max_c, uint8_t* xbuf,
                          float* scratch) {
    using G = Geo<kType>;
    constexpr int kPerLane = G::kWPC / 32;   // 8 (Q4_0, Q4_K) or 4 (Q8_0) elements
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int C = pr.C;
    float inv[kNT];
    if constexpr (kNorm) rms_scales<kNT>(pr, n_tok, scratch, inv);
    for (int idx = warp; idx < kNT * C; idx += kWarps) {
        const int t = idx / C;
        const int col = idx - t * C;
        uint8_t* rec = xbuf + (t * max_c + col) * G::kXRec;
        float v[kPerLane];
        if (t < n_tok) {
            const float4* src = reinterpret_cast<const float4*>(
                pr.X + static_cast<int64_t>(t) * pr.K + col * G::kWPC + lane * kPerLane);
#pragma unroll
            for (int i = 0; i < kPerLane / 4; ++i) {
                const float4 f = __ldg(src + i);
                v[4 * i] = f.x;
                v[4 * i + 1] = f.y;
                v[4 * i + 2] = f.z;
                v[4 * i + 3] = f.w;
            }
            if constexpr (kNorm) {
                float inv_t = inv[0];   // inv[t], kept in registers
#pragma unroll
                for (int tt = 1; tt < kNT; ++tt)
                    if (tt == t) inv_t = inv[tt];
                const float4* gsrc =
                    reinterpret_cast<const float4*>(pr.gamma + col * G::kWPC + lane * kPerLane);
#pragma unroll
                for (int i = 0; i < kPerLane / 4; ++i) {
                    const float4 gm = __ldg(gsrc + i);
                    v[4 * i] = v[4 * i] * inv_t * gm.x;
                    v[4 * i + 1] = v[4 * i + 1] * inv_t * gm.y;
                    v[4 * i + 2] = v[4 * i + 2] * inv_t * gm.z;
                    v[4 * i + 3] = v[4 * i + 3] * inv_t * gm.w;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = warp_max(amax);
        int e = 0;
        frexpf(amax, &e);   // amax = f * 2^e, f in [0.5, 1); e = 0 for amax = 0
        // x16 = rint(x * 2^(15 - e)): an exact power-of-two scaling, then one rounding.
        // 2^(15-e) as two normal floats (e spans -148..128 for finite inputs).
        const int sh = 15 - e, sh_a = sh / 2;
        const float f_a = __int_as_float((sh_a + 127) << 23);
        const float f_b = __int_as_float((sh - sh_a + 127) << 23);
        uint32_t packed[kPerLane / 2];
        int lane_sum = 0;
#pragma unroll
        for (int i = 0; i < kPerLane / 2; ++i) {
            const int a = max(-32767, min(32767, __float2int_rn((v[2 * i] * f_a) * f_b)));
            const int b = max(-32767, min(32767, __float2int_rn((v[2 * i + 1] * f_a) * f_b)));
            lane_sum += a + b;
            packed[i] = (static_cast<uint32_t>(a) & 0xFFFFu) | (static_cast<uint32_t>(b) << 16);
        }
        // Partial sums come out scaled by 2^(15 - e + kCodeShift); undo with two power-of-two
        // factors, each a normal float.
        const int u = e - 15 - Fmt<kType>::kCodeShift, u_a = u / 2;
        const float sc0 = __int_as_float((u_a + 127) << 23);
        const float sc1 = __int_as_float((u - u_a + 127) << 23);
        if constexpr (kPerLane == 8) {
            // Q4_0: lane l holds elements 8l..8l+7, i.e. block l / 4 of pair l / 8.
            // Q4_K: the same elements are part of sub-block l / 4 of quarter l / 8.
            uint8_t* prec = rec + (lane >> 3) * Q4Pair::kRec;
            *reinterpret_cast<uint4*>(prec + (lane & 7) * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            // block j covers lanes 4j..4j+3 (32 elements): Q4_0 bias = -128 * their sum,
            // Q4_K sub-block sum = their sum
            lane_sum += __shfl_xor_sync(0xFFFFFFFFu, lane_sum, 1);
            lane_sum += __shfl_xor_sync(0xFFFFFFFFu, lane_sum, 2);
            if ((lane & 3) == 0)
                *reinterpret_cast<int*>(prec + Q4Pair::kBiasOff + 4 * ((lane >> 2) & 1)) =
                    kType == GQ_TYPE_Q4_0 ? -128 * lane_sum : lane_sum;
            if ((lane & 7) == 0)
                *reinterpret_cast<float2*>(prec + Q4Pair::kScaleOff) = make_float2(sc0, sc1);
        } else {
            *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(packed[0], packed[1]);
            if (lane == 0)
                *reinterpret_cast<float2*>(rec + G::kScaleOff) = make_float2(sc0, sc1);
        }
    }
}

__device__ __forceinline__ int dp2a_lo_su(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp2a_hi_su(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------------------
// Quantized activations ("A Complete Guide to llama.cpp and Customization with C++",
// section 2.2: x_i ~= Delta_x q_x,i, and a block's dot product Delta Delta_x sum q q_x is
// a pure integer operation). Every 32-element block of x is quantized like a Q8_0 weight
// block: Delta = max |x| / 127 (IEEE division), q_x = round(x / Delta) (halves away from
// zero) clamped to [-127, 127], Delta_x = the fp16 value of Delta. Per block the integer
// sum S = sum q_i q_x,i comes from dp4a (four 8-bit products per instruction), and
// y += (Delta_w * Delta_x) * S: the scale product is exact in fp32 (11 + 11 bits), S is
// exact (|S| <= 127 * 127 * 32 < 2^24), one rounding per block.
// Record of one chunk for one token: kWPC int8 codes, then Delta_x per block (float),
// then for Q4_0 the sum of the block's codes (int; folds in the weights' -8 offset).
// Strides of 84 / 36 words (20 / 4 mod 32) put the 8 columns a warp reads in different
// bank groups.
// ---------------------------------------------------------------------------------------
template <int kType>
struct Q8xRec {
    using G = Geo<kType>;
    static constexpr int kScaleOff = G::kWPC;
    static constexpr int kSumOff = kScaleOff + 4 * G::kBPC;
    static constexpr int kUsed = kSumOff + (kType == GQ_TYPE_Q4_0 ? 4 * G::kBPC : 0);
    static constexpr int kXRec = kType == GQ_TYPE_Q4_0 ? 336 : 144;
    static_assert(kUsed <= kXRec && kXRec % 16 == 0, "record layout");
};

// Bytes of one chunk's activation record: x16 fixed point (kXM = 0) or Q8_0 codes (1).
template <int kType, int kXM>
__host__ __device__ constexpr int xrec_bytes() {
    if constexpr (kXM != 0)
        return Q8xRec<kType>::kXRec;
    else
        return Geo<kType>::kXRec;
}

__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int kType, int kNT>
__device__ void prepare_x_q8x(const GemvProb& pr, int n_tok, int max_c, uint8_t* xbuf) {
    using G = Geo<kType>;
    using R = Q8xRec<kType>;
    constexpr int kPerLane = G::kWPC / 32;         // 8 (Q4_0 chunk) or 4 (Q8_0 chunk)
    constexpr int kLanesPerBlock = 32 / kPerLane;  // lanes that share one 32-element block
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int C = pr.C;
    for (int idx = warp; idx < kNT * C; idx += kWarps) {
        const int t = idx / C;
        const int col = idx - t * C;
        uint8_t* rec = xbuf + (t * max_c + col) * R::kXRec;
        float v[kPerLane];
        if (t < n_tok) {
            const float4* src = reinterpret_cast<const float4*>(
                pr.X + static_cast<int64_t>(t) * pr.K + col * G::kWPC + lane * kPerLane);
#pragma unroll
            for (int i = 0; i < kPerLane / 4; ++i) {
                const float4 f = __ldg(src + i);
                v[4 * i] = f.x;
                v[4 * i + 1] = f.y;
                v[4 * i + 2] = f.z;
                v[4 * i + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) v[i] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int o = 1; o < kLanesPerBlock; o <<= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float d = amax / 127.0f;
        uint32_t packed[kPerLane / 4];
        int sum = 0;
#pragma unroll
        for (int w = 0; w < kPerLane / 4; ++w) {
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int c = 0;
                if (d != 0.0f) c = max(-127, min(127, static_cast<int>(roundf(v[4 * w + i] / d))));
                sum += c;
                word |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * i);
            }
            packed[w] = word;
        }
        if constexpr (kPerLane == 8)
            *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(packed[0], packed[1]);
        else
            *reinterpret_cast<uint32_t*>(rec + lane * 4) = packed[0];
#pragma unroll
        for (int o = 1; o < kLanesPerBlock; o <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane % kLanesPerBlock == 0) {
            const int j = lane / kLanesPerBlock;
            reinterpret_cast<float*>(rec + R::kScaleOff)[j] = __half2float(__float2half_rn(d));
            if constexpr (kType == GQ_TYPE_Q4_0) reinterpret_cast<int*>(rec + R::kSumOff)[j] = sum;
        }
    }
}

// One chunk against every token's Q8_0 record: out[t] += sum over the chunk's blocks of
// (Delta_w * Delta_x) * S.
template <int kType, int kNT>
__device__ __forceinline__ void chunk_dot_q8x(const uint8_t* raw, const uint8_t* xrec0,
                                              int rec_stride, float (&out)[kNT]) {
    using G = Geo<kType>;
    using R = Q8xRec<kType>;
    uint32_t r[G::kChunkWords];
    if constexpr (kType == GQ_TYPE_Q4_0) {
#pragma unroll
        for (int i = 0; i < G::kChunkWords / 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(raw + 16 * i);
            r[4 * i] = v.x;
            r[4 * i + 1] = v.y;
            r[4 * i + 2] = v.z;
            r[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < G::kChunkWords / 2; ++i) {
            const uint2 v = *reinterpret_cast<const uint2*>(raw + 8 * i);
            r[2 * i] = v.x;
            r[2 * i + 1] = v.y;
        }
    }
#pragma unroll
    for (int j = 0; j < G::kBPC; ++j) {
        const int base = j * G::kBB;
        const float dw = half_bits_to_float(u16_at(r, base));
        uint32_t q[8];
        if constexpr (kType == GQ_TYPE_Q4_0) {
            // unsigned codes c: elements 4i..4i+3 in the low nibbles, 16+4i.. in the high
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = word_at(r, base + 2 + 4 * i);
                q[i] = w & 0x0F0F0F0Fu;
                q[4 + i] = (w >> 4) & 0x0F0F0F0Fu;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = word_at(r, base + 2 + 4 * i);
        }
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            const uint8_t* rec = xrec0 + t * rec_stride;
            const int4 x0 = *reinterpret_cast<const int4*>(rec + 32 * j);
            const int4 x1 = *reinterpret_cast<const int4*>(rec + 32 * j + 16);
            const int xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            int S;
            if constexpr (kType == GQ_TYPE_Q4_0) {
                S = -8 * reinterpret_cast<const int*>(rec + R::kSumOff)[j];   // sum (c - 8) q_x
#pragma unroll
                for (int i = 0; i < 8; ++i) S = dp4a_us(q[i], xs[i], S);
            } else {
                S = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) S = __dp4a(static_cast<int>(q[i]), xs[i], S);
            }
            const float dx = reinterpret_cast<const float*>(rec + R::kScaleOff)[j];
            out[t] = fmaf(dw * dx, static_cast<float>(S), out[t]);
        }
    }
}

// Q8_0: one chunk (4 blocks) of one row against every token's x16 record:
// out[t] += chunk partial (scaled by 2^e).
template <int kNT>
__device__ __forceinline__ void chunk_dot_q8(const uint8_t* raw, const uint8_t* xrec0,
                                             int rec_stride, float (&out)[kNT]) {
    using G = Geo<GQ_TYPE_Q8_0>;
    uint32_t r[G::kChunkWords];
#pragma unroll
    for (int i = 0; i < G::kChunkWords / 2; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(raw + 8 * i);
        r[2 * i] = v.x;
        r[2 * i + 1] = v.y;
    }
    float acc[kNT];
#pragma unroll
    for (int t = 0; t < kNT; ++t) acc[t] = 0.0f;
#pragma unroll
    for (int j = 0; j < G::kBPC; ++j) {
        const int base = j * G::kBB;
        const float d = half_bits_to_float(u16_at(r, base));
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = word_at(r, base + 2 + 4 * i);
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            const uint4* xw = reinterpret_cast<const uint4*>(xrec0 + t * rec_stride + 64 * j);
            int s0 = 0, s1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 xv = xw[i];
                s0 = __dp2a_lo(static_cast<int>(xv.x), static_cast<int>(q[2 * i]), s0);
                s0 = __dp2a_hi(static_cast<int>(xv.y), static_cast<int>(q[2 * i]), s0);
                s1 = __dp2a_lo(static_cast<int>(xv.z), static_cast<int>(q[2 * i + 1]), s1);
                s1 = __dp2a_hi(static_cast<int>(xv.w), static_cast<int>(q[2 * i + 1]), s1);
            }
            acc[t] = fmaf(d, static_cast<float>(s0 + s1), acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        const float2 sc = *reinterpret_cast<const float2*>(xrec0 + t * rec_stride + G::kScaleOff);
        out[t] = fmaf(acc[t] * sc.x, sc.y, out[t]);
    }
}

// Q4_0 activations of one lane for one pair of blocks (64 elements), one token: the x16
// values, the two blocks' biases and the chunk's two scale factors, read from the pair
// record (Geo<GQ_TYPE_Q4_0>).
struct PairX {
    uint4 x[2][4];
    int bias[2];
    float2 sc;
};

__device__ __forceinline__ void load_pair_x(const uint8_t* rec, PairX& X) {
    using G = Geo<GQ_TYPE_Q4_0>;
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int i = 0; i < 4; ++i) X.x[b][i] = *reinterpret_cast<const uint4*>(rec + 64 * b + 16 * i);
    const int4 tail = *reinterpret_cast<const int4*>(rec + Q4Pair::kBiasOff);
    X.bias[0] = tail.x;
    X.bias[1] = tail.y;
    X.sc = make_float2(__int_as_float(tail.z), __int_as_float(tail.w));
}

// 16 * sum over one Q4_0 block of (c - 8) x16, from its code words split into lo bytes c
// (elements 4i..4i+3) and hi bytes 16c (elements 16+4i..):
//     16 * sum_lo c x + sum_hi (16 c) x + bias,   bias = -128 * sum x
// in four dp2a chains of four (asm is opaque to the compiler, which keeps each chain's
// order; independent chains give the scheduler work to interleave).
__device__ __forceinline__ int q4_block_dot(const uint4& x0, const uint4& x1, const uint4& x2,
                                            const uint4& x3, int bias, const uint32_t (&lo)[4],
                                            const uint32_t (&hi)[4]) {
    int sl0 = 0, sl1 = 0, sh1 = 0, sh0 = bias;
    sl0 = dp2a_lo_su(static_cast<int>(x0.x), lo[0], sl0);
    sl1 = dp2a_lo_su(static_cast<int>(x0.z), lo[1], sl1);
    sh0 = dp2a_lo_su(static_cast<int>(x2.x), hi[0], sh0);
    sh1 = dp2a_lo_su(static_cast<int>(x2.z), hi[1], sh1);
    sl0 = dp2a_hi_su(static_cast<int>(x0.y), lo[0], sl0);
    sl1 = dp2a_hi_su(static_cast<int>(x0.w), lo[1], sl1);
    sh0 = dp2a_hi_su(static_cast<int>(x2.y), hi[0], sh0);
    sh1 = dp2a_hi_su(static_cast<int>(x2.w), hi[1], sh1);
    sl0 = dp2a_lo_su(static_cast<int>(x1.x), lo[2], sl0);
    sl1 = dp2a_lo_su(static_cast<int>(x1.z), lo[3], sl1);
    sh0 = dp2a_lo_su(static_cast<int>(x3.x), hi[2], sh0);
    sh1 = dp2a_lo_su(static_cast<int>(x3.z), hi[3], sh1);
    sl0 = dp2a_hi_su(static_cast<int>(x1.y), lo[2], sl0);
    sl1 = dp2a_hi_su(static_cast<int>(x1.w), lo[3], sl1);
    sh0 = dp2a_hi_su(static_cast<int>(x3.y), hi[2], sh0);
    sh1 = dp2a_hi_su(static_cast<int>(x3.w), hi[3], sh1);
    return 16 * (sl0 + sl1) + (sh0 + sh1);
}

// Block b (0 or 1) of a lane's pair in one row: bytes 18b .. 18b + 17 of the pair's 36,
// held by the five words from byte 16b (block 0: scale in the low half of word 0, codes
// from byte 2; block 1: scale in the high half of word 0, codes in words 1..4).
__device__ __forceinline__ float q4_pair_block(const uint8_t* row_pair, int b, uint32_t (&lo)[4],
                                               uint32_t (&hi)[4]) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row_pair + 16 * b);
    uint32_t v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) v[i] = w[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q = b == 0 ? __funnelshift_r(v[i], v[i + 1], 16) : v[i + 1];
        lo[i] = q & 0x0F0F0F0Fu;
        hi[i] = q & 0xF0F0F0F0u;
    }
    return half_bits_to_float(b == 0 ? (v[0] & 0xFFFFu) : (v[0] >> 16));
}

// Q4_0: one pair of blocks (36 bytes, 64 weights) of each of the tile's `rows` rows against
// every token's pair record: out[r][t] += the pair's partial (scaled by 2^e). The lane
// reads the pair's activations once for all four rows of the tile (at one token all of
// them up front, at more tokens one block at a time), not once per row.
template <int kNT>
__device__ __forceinline__ void pair_dot_q4(const uint8_t* raw, int rs, int rows,
                                            const uint8_t* xp, int rec_stride,
                                            float (&out)[kTileRows][kNT]) {
    using G = Geo<GQ_TYPE_Q4_0>;
    PairX X;
    if constexpr (kNT == 1) load_pair_x(xp, X);
    float acc[kTileRows][kNT];
#pragma unroll
    for (int r = 0; r < kTileRows; ++r)
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[r][t] = 0.0f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        uint4 xv[kNT][4];
        int bias[kNT];
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            if constexpr (kNT == 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) xv[t][i] = X.x[b][i];
                bias[t] = X.bias[b];
            } else {
                const uint8_t* x = xp + t * rec_stride + 64 * b;
#pragma unroll
                for (int i = 0; i < 4; ++i) xv[t][i] = *reinterpret_cast<const uint4*>(x + 16 * i);
                bias[t] = *reinterpret_cast<const int*>(xp + t * rec_stride + Q4Pair::kBiasOff + 4 * b);
            }
        }
#pragma unroll
        for (int r = 0; r < kTileRows; ++r) {
            if (r >= rows) break;   // uniform across the warp
            uint32_t lo[4], hi[4];
            const float d = q4_pair_block(raw + r * rs, b, lo, hi);
#pragma unroll
            for (int t = 0; t < kNT; ++t)
                acc[r][t] = fmaf(d, static_cast<float>(q4_block_dot(xv[t][0], xv[t][1], xv[t][2],
                                                                    xv[t][3], bias[t], lo, hi)),
                                 acc[r][t]);
        }
    }
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        const float2 sc = kNT == 1 ? X.sc
                                   : *reinterpret_cast<const float2*>(xp + t * rec_stride +
                                                                      Q4Pair::kScaleOff);
#pragma unroll
        for (int r = 0; r < kTileRows; ++r) out[r][t] = fmaf(acc[r][t] * sc.x, sc.y, out[r][t]);
    }
}

// sum over one 32-element sub-block of q x16: x holds the sub-block's 32 int16 (word w =
// elements 2w, 2w + 1), q[i] the codes of elements 4i .. 4i + 3 as bytes. The high-nibble
// sub-block passes its codes as 16 q (the bytes masked, not shifted) and gets 16 S back,
// exact in int32 (|16 S| <= 240 * 32767 * 32 < 2^31), so an arithmetic shift by 4 returns
// S exactly. Four independent dp2a chains.
__device__ __forceinline__ int q4k_sub_dot(const uint4 (&x)[4], const uint32_t (&q)[8]) {
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    s0 = dp2a_lo_su(static_cast<int>(x[0].x), q[0], s0);
    s1 = dp2a_lo_su(static_cast<int>(x[0].z), q[1], s1);
    s2 = dp2a_lo_su(static_cast<int>(x[1].x), q[2], s2);
    s3 = dp2a_lo_su(static_cast<int>(x[1].z), q[3], s3);
    s0 = dp2a_hi_su(static_cast<int>(x[0].y), q[0], s0);
    s1 = dp2a_hi_su(static_cast<int>(x[0].w), q[1], s1);
    s2 = dp2a_hi_su(static_cast<int>(x[1].y), q[2], s2);
    s3 = dp2a_hi_su(static_cast<int>(x[1].w), q[3], s3);
    s0 = dp2a_lo_su(static_cast<int>(x[2].x), q[4], s0);
    s1 = dp2a_lo_su(static_cast<int>(x[2].z), q[5], s1);
    s2 = dp2a_lo_su(static_cast<int>(x[3].x), q[6], s2);
    s3 = dp2a_lo_su(static_cast<int>(x[3].z), q[7], s3);
    s0 = dp2a_hi_su(static_cast<int>(x[2].y), q[4], s0);
    s1 = dp2a_hi_su(static_cast<int>(x[2].w), q[5], s1);
    s2 = dp2a_hi_su(static_cast<int>(x[3].y), q[6], s2);
    s3 = dp2a_hi_su(static_cast<int>(x[3].w), q[7], s3);
    return (s0 + s1) + (s2 + s3);
}

// Q4_K: quarter g (sub-blocks 2g and 2g + 1, 64 weights) of one super-block in each of the
// tile's `rows` rows (sb = the super-block in row 0, rows rs bytes apart) against every
// token's quarter record: out[r][t] += the quarter's partial (scaled by 2^e), with
//     partial = d (sc_2g S_2g + sc_2g+1 S_2g+1) - dmin (m_2g X_2g + m_2g+1 X_2g+1),
// S_j = sum q x16 and X_j = sum x16 over sub-block j (both sums exact in int32: at most
// 63 * 2 * 15 * 32767 * 32 < 2^31 and 63 * 2 * 32767 * 32). Up to two tokens, the records
// are read once for all rows and each row's bytes once; at more tokens one sub-block at a
// time, and each row's codes once per sub-block.
template <int kNT>
__device__ __forceinline__ void quarter_dot_q4k(const uint8_t* sb, int g, int rs, int rows,
                                                const uint8_t* xp, int rec_stride,
                                                float (&out)[kTileRows][kNT]) {
    float acc[kTileRows][kNT];
#pragma unroll
    for (int r = 0; r < kTileRows; ++r)
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[r][t] = 0.0f;
    if constexpr (kNT <= 2) {
        PairX X[kNT];
#pragma unroll
        for (int t = 0; t < kNT; ++t) load_pair_x(xp + t * rec_stride, X[t]);
#pragma unroll
        for (int r = 0; r < kTileRows; ++r) {
            if (r >= rows) break;   // uniform across the warp
            const uint8_t* row = sb + r * rs;
            const uint4 hd = *reinterpret_cast<const uint4*>(row);
            const uint4 c0 = *reinterpret_cast<const uint4*>(row + 16 + 32 * g);
            const uint4 c1 = *reinterpret_cast<const uint4*>(row + 32 + 32 * g);
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t lo[8], hi[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo[i] = cw[i] & 0x0F0F0F0Fu;
                hi[i] = cw[i] & 0xF0F0F0F0u;   // 16 q: one instruction, no shift
            }
            uint32_t sc, m;
            q4k_scales(hd, g, sc, m);
            const float d = half_bits_to_float(hd.x & 0xFFFFu);
            const float dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                const int S0 = q4k_sub_dot(X[t].x[0], lo);
                const int S1 = q4k_sub_dot(X[t].x[1], hi) >> 4;   // 16 S1 exactly
                const int T = static_cast<int>(sc & 0xFFu) * S0 + static_cast<int>(sc >> 8) * S1;
                const int U = static_cast<int>(m & 0xFFu) * X[t].bias[0] +
                              static_cast<int>(m >> 8) * X[t].bias[1];
                acc[r][t] = fmaf(-dmin, static_cast<float>(U),
                                 fmaf(d, static_cast<float>(T), acc[r][t]));
            }
        }
#pragma unroll
        for (int t = 0; t < kNT; ++t)
#pragma unroll
            for (int r = 0; r < kTileRows; ++r)
                out[r][t] = fmaf(acc[r][t] * X[t].sc.x, X[t].sc.y, out[r][t]);
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 xv[kNT][4];
            int xs[kNT];
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                const uint8_t* x = xp + t * rec_stride + 64 * h;
#pragma unroll
                for (int i = 0; i < 4; ++i) xv[t][i] = *reinterpret_cast<const uint4*>(x + 16 * i);
                xs[t] = *reinterpret_cast<const int*>(xp + t * rec_stride + Q4Pair::kBiasOff + 4 * h);
            }
#pragma unroll
            for (int r = 0; r < kTileRows; ++r) {
                if (r >= rows) break;   // uniform across the warp
                const uint8_t* row = sb + r * rs;
                const uint4 hd = *reinterpret_cast<const uint4*>(row);
                const uint4 c0 = *reinterpret_cast<const uint4*>(row + 16 + 32 * g);
                const uint4 c1 = *reinterpret_cast<const uint4*>(row + 32 + 32 * g);
                const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint32_t q[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) q[i] = cw[i] & (h ? 0xF0F0F0F0u : 0x0F0F0F0Fu);
                uint32_t sc, m;
                q4k_scales(hd, g, sc, m);
                const int scj = static_cast<int>((sc >> (8 * h)) & 0xFFu);
                const int mj = static_cast<int>((m >> (8 * h)) & 0xFFu);
                const float d = half_bits_to_float(hd.x & 0xFFFFu);
                const float dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    const int S = q4k_sub_dot(xv[t], q) >> (4 * h);   // h = 1: 16 S exactly
                    acc[r][t] = fmaf(-dmin, static_cast<float>(mj * xs[t]),
                                     fmaf(d, static_cast<float>(scj * S), acc[r][t]));
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            const float2 sc = *reinterpret_cast<const float2*>(xp + t * rec_stride + Q4Pair::kScaleOff);
#pragma unroll
            for (int r = 0; r < kTileRows; ++r) out[r][t] = fmaf(acc[r][t] * sc.x, sc.y, out[r][t]);
        }
    }
}

// Sums each row of a 4-row tile over the 32 lanes (lane l holds v[r] for row r) in a fixed
// order, and leaves row r's total in lanes 8r .. 8r + 7 -- the lanes that own row r in the
// row-per-8-lanes layout -- with six shuffles: two exchanges halve the rows a lane carries
// (xor 16: rows 0-1 / 2-3; xor 8: one row each), three more add within groups of eight.
__device__ __forceinline__ float tile_row_sums(const float (&v)[kTileRows], int lane) {
    const bool up16 = lane & 16, up8 = lane & 8;
    float k0 = up16 ? v[2] : v[0], k1 = up16 ? v[3] : v[1];
    const float s0 = up16 ? v[0] : v[2], s1 = up16 ? v[1] : v[3];
    k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
    k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
    float k = up8 ? k1 : k0;
    k += __shfl_xor_sync(0xFFFFFFFFu, up8 ? k0 : k1, 8);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) k += __shfl_xor_sync(0xFFFFFFFFu, k, o);
    return k;
}

// kXM selects the activation form: 0 = 16-bit block fixed point (exact mul_mat within a
// proven bound), 1 = Q8_0-quantized activations (the quantized-activation product).
template <int kType, int kNT, int kMaxProbs, int kXM, int kFuse>
__global__ void __launch_bounds__(kThreads, 1)
gemv_stream_kernel(const __grid_constant__ GemvParams<kMaxProbs> P) {
    // kFuse: 0 plain, 1 RMSNorm of X in the preparation, 2 gate/up row pairs (Swish * up)
    constexpr bool kPair = kFuse == 2;
    constexpr bool kNorm = kFuse == 1;
    // Q4_0 and Q4_K with x16: a lane takes 64 weights (a block pair, a super-block quarter)
    // in every row of the tile.
    constexpr bool kPairMap = kType != GQ_TYPE_Q8_0 && kXM == 0;
    using G = Geo<kType>;
    constexpr int kRec = xrec_bytes<kType, kXM>();
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int S = ring_stages<kNT>();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * S * G::kStageBytes;                    // this warp's stages
    uint8_t* xbuf = smem + kWarps * S * G::kStageBytes;
    const int rec_stride = P.max_c * kRec;
    // Partial row sums of k-split items: [item < kWarps][row][token].
    float* red = reinterpret_cast<float*>(xbuf + kNT * rec_stride);
    uint64_t* bars = reinterpret_cast<uint64_t*>(red + kWarps * kTileRows * kNT) + warp * S;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_addr(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    // The next mul_mat of the stream may start on SMs this grid leaves and fill its rings.
    griddep_launch_dependents();

    // This CTA's rows: from the first row starting at or after byte c*T/G to the first
    // row starting at or after byte (c+1)*T/G.
    const int p0 = P.cut_p[blockIdx.x], p1 = P.cut_p[blockIdx.x + 1];
    const int64_t r0 = P.cut_r[blockIdx.x], r1 = P.cut_r[blockIdx.x + 1];
    const Segment first = find_segment(P, p0, r0, p1, r1);

    // Producer side of this warp's ring: the cursor's tile rows, one column group (up to 8
    // chunks) each. When a column group is a whole row, the tile's rows are contiguous in
    // memory and one copy fills the stage; otherwise one copy per row.
    WarpCursor prod;
    cursor_enter(P, prod, first, warp, p1, r1);
    int issued = 0;
    auto issue = [&](int s) {
        const GemvProb& pr = P.p[prod.seg.p];
        const int64_t row0 = prod.seg.rb + static_cast<int64_t>(prod.tile) * kTileRows;
        const int rows = static_cast<int>(min(static_cast<int64_t>(kTileRows), prod.seg.re - row0));
        const int c0 = kLanesPerRow * prod.cs;
        const int nc = min(kLanesPerRow, pr.C - c0);
        const uint32_t row_copy = static_cast<uint32_t>(nc * G::kChunkBytes);
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t dst = smem_addr(ring + s * G::kStageBytes);
        const uint8_t* src = pr.W + row0 * pr.row_bytes + static_cast<int64_t>(c0) * G::kChunkBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, row_copy * rows);
            if constexpr (kPair) {
                // row 2m + h of the sequence is row m of the gate (h = 0) or up (h = 1) matrix
                for (int r = 0; r < rows; ++r) {
                    const int64_t q = row0 + r;
                    const uint8_t* base_w = (q & 1) ? pr.W2 : pr.W;
                    bulk_g2s_evict_first(dst + r * G::kRowStride,
                                         base_w + (q >> 1) * pr.row_bytes +
                                             static_cast<int64_t>(c0) * G::kChunkBytes,
                                         row_copy, bar);
                }
            } else if (pr.C <= kLanesPerRow) {
                bulk_g2s_evict_first(dst, src, row_copy * rows, bar);
            } else {
                for (int r = 0; r < rows; ++r)
                    bulk_g2s_evict_first(dst + r * G::kRowStride, src + r * pr.row_bytes,
                                         row_copy, bar);
            }
        }
        cursor_advance(P, prod, warp, p1, r1);
        ++issued;
    };
    for (int s = 0; s < S && prod.valid; ++s) issue(s);
    // Only the weights, which no kernel of the call sequence writes, are read above; X and
    // Y may belong to the previous kernel of the stream, so everything after waits for it.
    griddep_wait();

    // Consumer side: all warps walk the CTA's segments together (x16 is per problem);
    // inside a segment each warp works through its own tiles.
    const int lc = lane % kLanesPerRow;   // which chunk of the column group this lane takes
    const int rrow = lane / kLanesPerRow; // which row of the tile
    int consumed = 0;
    bool timed_out = false;
    for (Segment seg = first; seg.valid; seg = find_segment(P, seg.p + 1, 0, p1, r1)) {
        if (__syncthreads_or(timed_out)) break;   // previous segment done everywhere
        const GemvProb& pr = P.p[seg.p];
        if constexpr (kXM == 0)
            prepare_x<kType, kNT, kNorm>(pr, P.n_tok, P.max_c, xbuf, red);
        else
            prepare_x_q8x<kType, kNT>(pr, P.n_tok, P.max_c, xbuf);
        __syncthreads();
        const SegPlan sp = plan_segment(seg.re - seg.rb, pr.C);
        for (int item = warp; item < sp.items && !timed_out; item += kWarps) {
            int tile, cb, ce;
            item_bounds(sp, item, tile, cb, ce);
            const int64_t row0 = seg.rb + static_cast<int64_t>(tile) * kTileRows;
            const int rows = static_cast<int>(min(static_cast<int64_t>(kTileRows), seg.re - row0));
            float acc[kNT];
#pragma unroll
            for (int t = 0; t < kNT; ++t) acc[t] = 0.0f;
            // Q4_0 with x16: lane l takes block pair l of the column group in every row of
            // the tile (acc4[r][t]); Q4_K: quarter l % 4 of super-block l / 4 in every row;
            // otherwise lane l takes chunk lc of row rrow (acc[t]).
            float acc4[kTileRows][kNT];
#pragma unroll
            for (int r = 0; r < kTileRows; ++r)
#pragma unroll
                for (int t = 0; t < kNT; ++t) acc4[r][t] = 0.0f;
            for (int cs = cb; cs < ce; ++cs) {
                const int s = consumed % S;
                if (!mbar_wait(smem_addr(&bars[s]), (consumed / S) & 1)) {
                    timed_out = true;
                    break;
                }
                // Whole-row stages hold rows at their global stride; others at kRowStride.
                const int rs = (!kPair && pr.C <= kLanesPerRow) ? static_cast<int>(pr.row_bytes)
                                                                 : G::kRowStride;
                const uint8_t* stage = ring + s * G::kStageBytes;
                uint32_t dep;   // depends on every shared load of the stage by this lane
                if constexpr (kPairMap) {
                    const int col = kLanesPerRow * cs + (lane >> 2);
                    if (col < pr.C) {
                        if constexpr (kType == GQ_TYPE_Q4_0)
                            pair_dot_q4<kNT>(stage + lane * (G::kChunkBytes / 4), rs, rows,
                                             xbuf + col * kRec + (lane & 3) * Q4Pair::kRec,
                                             rec_stride, acc4);
                        else
                            quarter_dot_q4k<kNT>(stage + (lane >> 2) * G::kChunkBytes, lane & 3,
                                                 rs, rows,
                                                 xbuf + col * kRec + (lane & 3) * Q4Pair::kRec,
                                                 rec_stride, acc4);
                    }
                    dep = __float_as_uint(acc4[0][0]) ^ __float_as_uint(acc4[1][0]) ^
                          __float_as_uint(acc4[2][0]) ^ __float_as_uint(acc4[3][0]);
                } else {
                    const int col = kLanesPerRow * cs + lc;
                    if (rrow < rows && col < pr.C) {
                        const uint8_t* raw = stage + rrow * rs + lc * G::kChunkBytes;
                        if constexpr (kXM == 0)
                            chunk_dot_q8<kNT>(raw, xbuf + col * kRec, rec_stride, acc);
                        else
                            chunk_dot_q8x<kType, kNT>(raw, xbuf + col * kRec, rec_stride, acc);
                    }
                    dep = __float_as_uint(acc[0]);
                }
                release_warp_to_async_proxy(dep);   // lane 0 refills it
                ++consumed;
                if (prod.valid) issue(s);   // refill the stage just read
            }
            if (timed_out) break;
            if constexpr (kPairMap) {
                // row rrow's sum lands in lanes 8 rrow .. 8 rrow + 7, as below
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    float v[kTileRows];
#pragma unroll
                    for (int r = 0; r < kTileRows; ++r) v[r] = acc4[r][t];
                    acc[t] = tile_row_sums(v, lane);
                }
            } else {
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
#pragma unroll
                    for (int o = 1; o < kLanesPerRow; o <<= 1)
                        acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
                }
            }
            if constexpr (kPair) {
                // The up row's sums sit kLanesPerRow lanes above the gate row's.
                float up[kNT];
#pragma unroll
                for (int t = 0; t < kNT; ++t)
                    up[t] = __shfl_down_sync(0xFFFFFFFFu, acc[t], kLanesPerRow);
                if (sp.ksplit == 1 && lc == 0 && (rrow & 1) == 0 && rrow < rows) {
                    const int64_t mh = pr.M >> 1;
#pragma unroll
                    for (int t = 0; t < kNT; ++t)
                        if (t < P.n_tok) pr.Y[t * mh + ((row0 + rrow) >> 1)] = swish(acc[t]) * up[t];
                }
            }
            if (lc == 0 && rrow < rows) {
                if (sp.ksplit == 1) {
                    if constexpr (!kPair) {
#pragma unroll
                        for (int t = 0; t < kNT; ++t)
                            if (t < P.n_tok) pr.Y[t * pr.M + row0 + rrow] = acc[t];
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) red[(item * kTileRows + rrow) * kNT + t] = acc[t];
                }
            }
        }
        if (sp.ksplit > 1) {
            // Sum the k-groups of each row in group order (deterministic).
            if (__syncthreads_or(timed_out)) break;
            if constexpr (kPair) {
                // one output per (gate, up) row pair: Swish(gate) * up
                const int n_out = sp.ntiles * (kTileRows / 2) * kNT;
                for (int idx = threadIdx.x; idx < n_out; idx += kThreads) {
                    const int t = idx % kNT;
                    const int rr = 2 * ((idx / kNT) % (kTileRows / 2));
                    const int tile = idx / (kNT * (kTileRows / 2));
                    const int64_t row = seg.rb + static_cast<int64_t>(tile) * kTileRows + rr;
                    if (row >= seg.re || t >= P.n_tok) continue;
                    float g = 0.0f, u = 0.0f;
                    for (int kg = 0; kg < sp.ksplit; ++kg) {
                        g += red[((tile * sp.ksplit + kg) * kTileRows + rr) * kNT + t];
                        u += red[((tile * sp.ksplit + kg) * kTileRows + rr + 1) * kNT + t];
                    }
                    pr.Y[t * (pr.M >> 1) + (row >> 1)] = swish(g) * u;
                }
            } else {
                const int n_out = sp.ntiles * kTileRows * kNT;
                for (int idx = threadIdx.x; idx < n_out; idx += kThreads) {
                    const int t = idx % kNT;
                    const int rr = (idx / kNT) % kTileRows;
                    const int tile = idx / (kNT * kTileRows);
                    const int64_t row = seg.rb + static_cast<int64_t>(tile) * kTileRows + rr;
                    if (row >= seg.re || t >= P.n_tok) continue;
                    float v = 0.0f;
                    for (int kg = 0; kg < sp.ksplit; ++kg)
                        v += red[((tile * sp.ksplit + kg) * kTileRows + rr) * kNT + t];
                    pr.Y[t * pr.M + row] = v;
                }
            }
        }
    }
    if (timed_out && lane == 0) report_status(P.status, kStatusTimeout);
    // Copies still in flight (only after a timeout) must land before the CTA exits.
    for (int i = consumed; i < issued; ++i)
        mbar_wait(smem_addr(&bars[i % S]), (i / S) & 1, 100000000ull);
}

// Any K % 32 == 0: one warp per row, lanes over blocks, fp32 FMA, xor-shuffle reduction
// (fixed order, so deterministic). Up to kMaxTok tokens per pass.
template <int kType>
__global__ void __launch_bounds__(256)
gemv_generic_kernel(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                    const float* __restrict__ X, int n_tok, float* __restrict__ Y) {
    constexpr int kBB = Fmt<kType>::kBB;
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         row < M; row += warps) {
        float acc[kMaxTok] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int64_t b = lane; b < nb; b += 32) {
            const unsigned short* blk =
                reinterpret_cast<const unsigned short*>(W + (row * nb + b) * kBB);
            const float d = half_bits_to_float(__ldg(blk));
            float w[32];
            if constexpr (kType == GQ_TYPE_Q4_0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t v = __ldg(blk + 1 + j);
                    w[2 * j] = static_cast<float>(static_cast<int>(v & 15) - 8) * d;
                    w[2 * j + 16] = static_cast<float>(static_cast<int>((v >> 4) & 15) - 8) * d;
                    w[2 * j + 1] = static_cast<float>(static_cast<int>((v >> 8) & 15) - 8) * d;
                    w[2 * j + 17] = static_cast<float>(static_cast<int>((v >> 12) & 15) - 8) * d;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t v = __ldg(blk + 1 + j);
                    w[2 * j] = static_cast<float>(static_cast<int8_t>(v & 0xFF)) * d;
                    w[2 * j + 1] = static_cast<float>(static_cast<int8_t>(v >> 8)) * d;
                }
            }
            for (int t = 0; t < n_tok; ++t) {
                const float* x = X + t * K + b * 32;
                float a = acc[t];
#pragma unroll
                for (int i = 0; i < 32; ++i) a = fmaf(w[i], __ldg(x + i), a);
                acc[t] = a;
            }
        }
        for (int t = 0; t < n_tok; ++t) {
            float a = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            if (lane == 0) Y[t * M + row] = a;
        }
    }
}

// Q4_K, any K % 256 == 0: one warp per row, lanes over 32-weight sub-blocks, each weight
// D_j q - M_j in fp32 (as gq_dequantize computes it), fp32 FMA, xor-shuffle reduction.
__global__ void __launch_bounds__(256)
gemv_generic_q4k_kernel(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                        const float* __restrict__ X, int n_tok, float* __restrict__ Y) {
    const int lane = threadIdx.x & 31;
    const int64_t nsub = K / 32;
    const int64_t row_bytes = (K / kQ4KWeights) * kQ4KBytes;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         row < M; row += warps) {
        float acc[kMaxTok] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int64_t b = lane; b < nsub; b += 32) {
            const uint8_t* sb = W + row * row_bytes + (b >> 3) * kQ4KBytes;
            const int j = static_cast<int>(b & 7);
            const uint4 hd = __ldg(reinterpret_cast<const uint4*>(sb));
            uint32_t sc2, m2;
            q4k_scales(hd, j >> 1, sc2, m2);
            const int h = j & 1;
            const float D = __fmul_rn(half_bits_to_float(hd.x & 0xFFFFu),
                                      static_cast<float>((sc2 >> (8 * h)) & 0xFFu));
            const float Mj = __fmul_rn(half_bits_to_float(hd.x >> 16),
                                       static_cast<float>((m2 >> (8 * h)) & 0xFFu));
            const uint4* cp = reinterpret_cast<const uint4*>(sb + 16 + 32 * (j >> 1));
            const uint4 c0 = __ldg(cp), c1 = __ldg(cp + 1);
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            float w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t q = (cw[i] >> (8 * k + 4 * h)) & 15u;
                    w[4 * i + k] = __fsub_rn(__fmul_rn(D, static_cast<float>(q)), Mj);
                }
            for (int t = 0; t < n_tok; ++t) {
                const float* x = X + t * K + b * 32;
                float a = acc[t];
#pragma unroll
                for (int i = 0; i < 32; ++i) a = fmaf(w[i], __ldg(x + i), a);
                acc[t] = a;
            }
        }
        for (int t = 0; t < n_tok; ++t) {
            float a = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            if (lane == 0) Y[t * M + row] = a;
        }
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
template <int kType, int kXM = 0>
int64_t stream_smem_bytes(int n_tok_template, int max_c) {
    using G = Geo<kType>;
    const int stages = n_tok_template <= 3 ? GQ_GEMV_STAGES : GQ_GEMV_STAGES_N4;
    return static_cast<int64_t>(kWarps) * stages * G::kStageBytes +
           static_cast<int64_t>(n_tok_template) * max_c * xrec_bytes<kType, kXM>() +
           static_cast<int64_t>(kWarps) * kTileRows * n_tok_template * 4 +
           static_cast<int64_t>(kWarps) * stages * 8;
}

// cudaFuncSetAttribute once per (kernel, device) for the largest size asked so far.
// Keyed by the kernel's address: instantiations share a function type.
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

template <int kType, int kNT, int kMaxProbs, int kXM, int kFuse>
cudaError_t launch_stream_t(GemvParams<kMaxProbs>& P, const DeviceInfo* info, cudaStream_t s) {
    auto kernel = gemv_stream_kernel<kType, kNT, kMaxProbs, kXM, kFuse>;
    const int64_t smem = stream_smem_bytes<kType, kXM>(kNT, P.max_c);
    if (smem > info->max_smem_optin) return cudaErrorInvalidValue;   // see stream_eligible
    cudaError_t e = ensure_smem(kernel, info->device, smem);
    if (e != cudaSuccess) return e;
    // Enough CTAs that each streams at least ~32 KB, at most one per SM.
    int64_t grid = (P.total_bytes + 32767) / 32768;
    grid = std::max<int64_t>(1, std::min<int64_t>({grid, int64_t(info->sm_count), int64_t(kMaxGrid)}));
    // Each CTA's share: from the first row starting at or after cost c T / G to the first
    // row starting at or after cost (c + 1) T / G.
    int p = 0;
    for (int64_t c = 0; c <= grid; ++c) {
        int64_t r = 0;
        int q = p;
        row_at_cost(P, P.total_cost * c / grid, q, r);
        P.cut_p[c] = q;
        P.cut_r[c] = r;
        p = std::min(q, P.count - 1);
    }
    // Programmatic dependent launch: this grid's CTAs may start filling their weight rings
    // while the previous kernel of the stream finishes (the kernel waits for it before it
    // touches X or Y).
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&P};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
}

template <int kType, int kMaxProbs, int kXM, int kFuse>
cudaError_t launch_stream_nt(GemvParams<kMaxProbs>& P, const DeviceInfo* info, cudaStream_t s) {
    switch (P.n_tok) {
        case 1: return launch_stream_t<kType, 1, kMaxProbs, kXM, kFuse>(P, info, s);
        case 2: return launch_stream_t<kType, 2, kMaxProbs, kXM, kFuse>(P, info, s);
        case 3: return launch_stream_t<kType, 3, kMaxProbs, kXM, kFuse>(P, info, s);
        default: return launch_stream_t<kType, 4, kMaxProbs, kXM, kFuse>(P, info, s);
    }
}

// Weights and bytes of one chunk (one ring-stage column) of a block type.
int chunk_weights(gq_type t) {
    return t == GQ_TYPE_Q4_0 ? Geo<GQ_TYPE_Q4_0>::kWPC
                             : (t == GQ_TYPE_Q8_0 ? Geo<GQ_TYPE_Q8_0>::kWPC : Geo<GQ_TYPE_Q4_K>::kWPC);
}
int chunk_bytes(gq_type t) {
    return t == GQ_TYPE_Q4_0 ? Geo<GQ_TYPE_Q4_0>::kChunkBytes
                             : (t == GQ_TYPE_Q8_0 ? Geo<GQ_TYPE_Q8_0>::kChunkBytes
                                                  : Geo<GQ_TYPE_Q4_K>::kChunkBytes);
}

template <int kMaxProbs, int kXM = 0, int kFuse = 0>
cudaError_t launch_stream(gq_type t, const MatProblem* probs, int count, int64_t tok0,
                          int n_tok, const DeviceInfo* info, cudaStream_t s) {
    GemvParams<kMaxProbs> P{};
    P.count = count;
    P.n_tok = n_tok;
    P.status = info->status;
    const int wpc = chunk_weights(t);
    const int cb = chunk_bytes(t);
    int64_t bytes = 0, cost = 0;
    int max_c = 1;
    for (int i = 0; i < count; ++i) {
        GemvProb& g = P.p[i];
        g.W = probs[i].W;
        g.X = probs[i].X + tok0 * probs[i].K;
        g.Y = probs[i].Y + tok0 * probs[i].M;
        g.W2 = probs[i].W2;
        g.gamma = probs[i].gamma;
        g.eps = probs[i].eps;
        g.M = kFuse == 2 ? 2 * probs[i].M : probs[i].M;   // gate/up pairs: two rows per output
        g.K = static_cast<int32_t>(probs[i].K);
        g.C = static_cast<int32_t>(probs[i].K / wpc);
        g.row_bytes = static_cast<int64_t>(g.C) * cb;
        const int64_t groups = (g.C + kLanesPerRow - 1) / kLanesPerRow;
        g.row_cost = g.row_bytes +
                     (t == GQ_TYPE_Q8_0
                          ? (kGroupCost + (g.C > kLanesPerRow ? kRowCopyCost : 0)) * groups
                          : (kGroupCost + kLongRowCost4 * std::max<int64_t>(0, groups - 2)) * groups);
        if (i > 0) cost += t == GQ_TYPE_Q8_0 ? kSegCost : kSegCost4;
        g.cost_begin = cost;
        bytes += g.M * g.row_bytes;
        cost += g.M * g.row_cost;
        max_c = std::max(max_c, g.C);
    }
    P.total_bytes = bytes;
    P.total_cost = cost;
    P.max_c = max_c;
    if (t == GQ_TYPE_Q4_0) return launch_stream_nt<GQ_TYPE_Q4_0, kMaxProbs, kXM, kFuse>(P, info, s);
    if (t == GQ_TYPE_Q8_0) return launch_stream_nt<GQ_TYPE_Q8_0, kMaxProbs, kXM, kFuse>(P, info, s);
    // Q4_K: plain products only (the callers route its other forms elsewhere)
    if constexpr (kXM == 0 && kFuse == 0)
        return launch_stream_nt<GQ_TYPE_Q4_K, kMaxProbs, kXM, kFuse>(P, info, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_generic(gq_type t, const MatProblem& p, int64_t tok0, int n_tok,
                           const DeviceInfo* info, cudaStream_t s) {
    const int64_t blocks = (p.M + 7) / 8;
    const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(info->sm_count) * 8));
    const float* X = p.X + tok0 * p.K;
    float* Y = p.Y + tok0 * p.M;
    if (t == GQ_TYPE_Q4_0)
        gemv_generic_kernel<GQ_TYPE_Q4_0><<<grid, 256, 0, s>>>(p.W, p.M, p.K, X, n_tok, Y);
    else if (t == GQ_TYPE_Q8_0)
        gemv_generic_kernel<GQ_TYPE_Q8_0><<<grid, 256, 0, s>>>(p.W, p.M, p.K, X, n_tok, Y);
    else
        gemv_generic_q4k_kernel<<<grid, 256, 0, s>>>(p.W, p.M, p.K, X, n_tok, Y);
    return cudaGetLastError();
}

// Shapes and pointers the streaming kernel takes at all (any token count).
bool stream_shape_ok(const MatProblem& p) {
    if (p.K % 256 != 0 || p.K > (int64_t(1) << 24)) return false;
    if (reinterpret_cast<uintptr_t>(p.X) % 16 != 0) return false;
    return reinterpret_cast<uintptr_t>(p.W) % 16 == 0;
}

// Whether the shared-memory plan for `n_tok` tokens of this problem fits the device.
template <int kXM = 0>
bool stream_fits(gq_type t, const MatProblem& p, int n_tok, const DeviceInfo* info) {
    const int c = static_cast<int>(p.K / chunk_weights(t));
    const int64_t smem = t == GQ_TYPE_Q4_0   ? stream_smem_bytes<GQ_TYPE_Q4_0, kXM>(n_tok, c)
                         : t == GQ_TYPE_Q8_0 ? stream_smem_bytes<GQ_TYPE_Q8_0, kXM>(n_tok, c)
                                             : stream_smem_bytes<GQ_TYPE_Q4_K, 0>(n_tok, c);
    return smem <= info->max_smem_optin;
}

}  // namespace

cudaError_t launch_mul_mat(gq_type t, const MatProblem* probs, int count, int64_t N,
                           cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    MatProblem fast[GQ_MAX_BATCH];
    int64_t step = 0;
    for (int64_t tok0 = 0; tok0 < N; tok0 += step) {
        // Tokens in this pass: as many as the x16 buffers of the streamable problems allow
        // (up to kMaxTok); a problem that does not fit even one token goes to the generic
        // kernel.
        int n_tok = static_cast<int>(std::min<int64_t>(kMaxTok, N - tok0));
        for (; n_tok > 1; --n_tok) {
            bool all_fit = true;
            for (int i = 0; i < count && all_fit; ++i)
                if (stream_shape_ok(probs[i]) && stream_fits(t, probs[i], 1, info))
                    all_fit = stream_fits(t, probs[i], n_tok, info);
            if (all_fit) break;
        }
        step = n_tok;
        int n_fast = 0;
        for (int i = 0; i < count; ++i) {
            if (stream_shape_ok(probs[i]) && stream_fits(t, probs[i], n_tok, info)) {
                fast[n_fast++] = probs[i];
            } else {
                e = launch_generic(t, probs[i], tok0, n_tok, info, s);
                if (e != cudaSuccess) return e;
            }
        }
        if (n_fast == 0) continue;
        if (n_fast == 1)
            e = launch_stream<1>(t, fast, n_fast, tok0, n_tok, info, s);
        else if (n_fast <= 16)
            e = launch_stream<16>(t, fast, n_fast, tok0, n_tok, info, s);
        else
            e = launch_stream<GQ_MAX_BATCH>(t, fast, n_fast, tok0, n_tok, info, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool q8x_eligible(gq_type t, const MatProblem& p) {
    DeviceInfo* info = nullptr;
    if (current_device_info(&info) != cudaSuccess) return false;
    return stream_shape_ok(p) && stream_fits<1>(t, p, 1, info);
}

cudaError_t launch_mul_mat_q8x(gq_type t, const MatProblem* probs, int count, int64_t N,
                               cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    int64_t step = 0;
    for (int64_t tok0 = 0; tok0 < N; tok0 += step) {
        // As many tokens per pass (<= kMaxTokQ8x) as every problem's records allow.
        int n_tok = static_cast<int>(std::min<int64_t>(kMaxTokQ8x, N - tok0));
        for (; n_tok > 1; --n_tok) {
            bool all_fit = true;
            for (int i = 0; i < count && all_fit; ++i) all_fit = stream_fits<1>(t, probs[i], n_tok, info);
            if (all_fit) break;
        }
        step = n_tok;
        if (count == 1)
            e = launch_stream<1, 1>(t, probs, count, tok0, n_tok, info, s);
        else
            e = launch_stream<GQ_MAX_BATCH, 1>(t, probs, count, tok0, n_tok, info, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gq

namespace gq {

// Fused forms on the CUDA-core decode kernel: RMSNorm of X in the activation preparation
// (p.gamma) and the gate/up pair with Swish(gate) * up written directly (p.W2). Shapes the
// streaming kernel takes only; the caller composes the other shapes from plain kernels.
bool fused_decode_eligible(gq_type t, const MatProblem& p) {
    if (t != GQ_TYPE_Q4_0 && t != GQ_TYPE_Q8_0) return false;   // Q4_K: composite forms
    DeviceInfo* info = nullptr;
    if (current_device_info(&info) != cudaSuccess) return false;
    if (p.gamma && reinterpret_cast<uintptr_t>(p.gamma) % 16 != 0) return false;   // float4
    if (p.W2 && reinterpret_cast<uintptr_t>(p.W2) % 16 != 0) return false;         // bulk copies
    return stream_shape_ok(p) && stream_fits(t, p, 1, info);
}

cudaError_t launch_mul_mat_fused(gq_type t, const MatProblem& p, int64_t N, cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    int64_t step = 0;
    for (int64_t tok0 = 0; tok0 < N; tok0 += step) {
        int n_tok = static_cast<int>(std::min<int64_t>(kMaxTok, N - tok0));
        while (n_tok > 1 && !stream_fits(t, p, n_tok, info)) --n_tok;
        step = n_tok;
        e = p.W2 ? launch_stream<1, 0, 2>(t, &p, 1, tok0, n_tok, info, s)
                 : launch_stream<1, 0, 1>(t, &p, 1, tok0, n_tok, info, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gq
