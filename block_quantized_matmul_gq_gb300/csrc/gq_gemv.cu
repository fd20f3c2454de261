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
//    CTA takes a contiguous, row-aligned share of equal bytes, so small matrices (GQA
//    k/v projections) ride along with large ones and no CTA idles on a tail.
//  * Thread 0 streams that share through a 3-stage ring of 1-D bulk copies (TMA,
//    cp.async.bulk) with an L2 evict-first hint; 256 threads consume it. A stage holds
//    256 "chunks": 8 Q4_0 blocks (144 B, 256 weights) or 4 Q8_0 blocks (136 B, 128
//    weights), one chunk per thread. Rows are whole chunks (K % 256 == 0), so every
//    copy is 16-byte aligned.
//  * Activations: each CTA converts the problem's X into 16-bit block fixed point in
//    shared memory (one power-of-two scale 2^e per chunk of 256 / 128 elements), so that
//    the inner product of a 32-weight block is EXACT integer arithmetic:
//        S = sum_i (16 (c_i - 8)) * x16_i       (Q4_0; codes become signed bytes 16(c-8))
//        S = sum_i c_i * x16_i                  (Q8_0)
//    with dp2a (two 16x8-bit products per instruction). Then acc += d * float(S) and, per
//    chunk, partial = acc * 2^e. The only approximation is x16 = rint(x / 2^e) with
//    |x16| <= 32767, i.e. |error| <= sqrt(256) / 65534 * ||x|| ||What|| = 2.4e-4 of the
//    bound 1e-3 ||x|| ||What|| (Cauchy-Schwarz per chunk), whatever the inputs.
//  * Row sums: per-chunk partials go to shared memory and one thread per row adds them in
//    k order (a carry links rows that straddle stages), so results are deterministic.
//  * Waits are bounded: a stage that never arrives sets the device status word and the
//    CTA leaves after draining its own copies.
// Shapes the fast kernel does not take (K % 256 != 0, unaligned X, very large K) run on
// gemv_generic_kernel: one warp per row, plain loads, fp32 FMA.
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kMaxTok = 4;   // tokens per pass of the weight stream

template <int kType>
struct Fmt;
template <>
struct Fmt<GQ_TYPE_Q4_0> {
    static constexpr int kBB = kQ4Bytes;
    static constexpr int kBlocksPerChunk = 8;
    static constexpr int kCodeShift = 4;   // codes enter dp2a as 16 * (c - 8)
};
template <>
struct Fmt<GQ_TYPE_Q8_0> {
    static constexpr int kBB = kQ8Bytes;
    static constexpr int kBlocksPerChunk = 4;
    static constexpr int kCodeShift = 0;
};

template <int kType>
struct Geo {
    static constexpr int kBB = Fmt<kType>::kBB;
    static constexpr int kBPC = Fmt<kType>::kBlocksPerChunk;
    static constexpr int kChunkBytes = kBB * kBPC;                 // 144 or 136
    static constexpr int kChunkWords = kChunkBytes / 4;            // 36 or 34
    static constexpr int kWPC = 32 * kBPC;                         // weights per chunk
    static constexpr int kStageBytes = kThreads * kChunkBytes;
    // x16 record of one chunk for one token: kWPC int16, then the int exponent, padded
    // to a 16-byte multiple whose word count is 4 mod 32 (bank-conflict-free reads).
    static constexpr int kXRec = kWPC * 2 + 16;                    // 528 or 272
};

struct GemvProb {
    const uint8_t* W;
    const float* X;
    float* Y;
    int64_t M;
    int64_t row_bytes;
    int64_t byte_begin;   // bytes of all earlier problems
    int32_t C;            // chunks per row
    int32_t K;
};

template <int kMaxProbs>
struct GemvParams {
    int32_t count;
    int32_t n_tok;        // valid tokens of this pass, 1..kMaxTok
    int32_t max_c;        // largest C: x buffer holds n_tok * max_c records
    int32_t pad_;
    int64_t total_bytes;
    unsigned* status;
    GemvProb p[kMaxProbs];
};

// First row (problem p, row r) whose first byte is at or after `byte`; (count, 0) = end.
template <int kMaxProbs>
__device__ void row_at_byte(const GemvParams<kMaxProbs>& P, int64_t byte, int& p, int64_t& r) {
    p = 0;
    while (p + 1 < P.count && P.p[p + 1].byte_begin <= byte) ++p;
    const int64_t off = byte - P.p[p].byte_begin;
    r = off <= 0 ? 0 : (off + P.p[p].row_bytes - 1) / P.p[p].row_bytes;
    if (r >= P.p[p].M) {
        ++p;
        r = 0;
    }
}

// Walks this CTA's share as a sequence of stages: (problem, segment rows, chunk offset).
struct Cursor {
    int p;
    int64_t r_begin, r_end;   // rows of the current segment (one problem)
    int64_t chunk, n_chunks;  // chunk offset of the current stage within the segment
    bool valid;
};

template <int kMaxProbs>
__device__ void open_segment(const GemvParams<kMaxProbs>& P, Cursor& c, int p, int64_t rb,
                             int p_end, int64_t r_end) {
    for (; p < P.count && p <= p_end; ++p, rb = 0) {
        const int64_t re = (p == p_end) ? r_end : P.p[p].M;
        if (re > rb) {
            c.p = p;
            c.r_begin = rb;
            c.r_end = re;
            c.chunk = 0;
            c.n_chunks = (re - rb) * P.p[p].C;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}

template <int kMaxProbs>
__device__ void advance(const GemvParams<kMaxProbs>& P, Cursor& c, int p_end, int64_t r_end) {
    c.chunk += kThreads;
    if (c.chunk >= c.n_chunks) open_segment(P, c, c.p + 1, 0, p_end, r_end);
}

__device__ __forceinline__ uint32_t word_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? __funnelshift_r(r[w], r[w + 1], 16) : r[w];
}

__device__ __forceinline__ uint32_t u16_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? (r[w] >> 16) : (r[w] & 0xFFFFu);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// X (n_tok x K fp32) -> x16 records, one per (token, chunk column). Warp per record.
template <int kType, int kNT>
__device__ void prepare_x(const GemvProb& pr, int n_tok, int max_c, uint8_t* xbuf) {
    using G = Geo<kType>;
    constexpr int kPerLane = G::kWPC / 32;   // 8 (Q4_0) or 4 (Q8_0) elements
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int C = pr.C;
    for (int idx = warp; idx < kNT * C; idx += kThreads / 32) {
        const int t = idx / C;
        const int col = idx - t * C;
        uint8_t* rec = xbuf + (static_cast<int64_t>(t) * max_c + col) * G::kXRec;
        float v[kPerLane];
        if (t < n_tok) {
            const float4* src = reinterpret_cast<const float4*>(
                pr.X + static_cast<int64_t>(t) * pr.K + static_cast<int64_t>(col) * G::kWPC +
                lane * kPerLane);
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
        amax = warp_max(amax);
        int e = 0;
        frexpf(amax, &e);   // amax = f * 2^e, f in [0.5, 1); e = 0 for amax = 0
        uint32_t packed[kPerLane / 2];
#pragma unroll
        for (int i = 0; i < kPerLane / 2; ++i) {
            const int a = max(-32767, min(32767, __float2int_rn(ldexpf(v[2 * i], 15 - e))));
            const int b = max(-32767, min(32767, __float2int_rn(ldexpf(v[2 * i + 1], 15 - e))));
            packed[i] = (static_cast<uint32_t>(a) & 0xFFFFu) | (static_cast<uint32_t>(b) << 16);
        }
        if constexpr (kPerLane == 8) {
            *reinterpret_cast<uint4*>(rec + lane * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        } else {
            *reinterpret_cast<uint2*>(rec + lane * 8) = make_uint2(packed[0], packed[1]);
        }
        if (lane == 0)
            *reinterpret_cast<int*>(rec + G::kWPC * 2) = e - 15 - Fmt<kType>::kCodeShift;
    }
}

// One chunk for every token: returns per-token partial sums (already scaled by 2^e).
template <int kType, int kNT>
__device__ __forceinline__ void chunk_dot(const uint8_t* raw, const uint8_t* xrec0,
                                          int rec_stride, float (&out)[kNT]) {
    using G = Geo<kType>;
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
    float acc[kNT];
#pragma unroll
    for (int t = 0; t < kNT; ++t) acc[t] = 0.0f;

#pragma unroll
    for (int j = 0; j < G::kBPC; ++j) {
        const int base = j * G::kBB;
        const float d = half_bits_to_float(u16_at(r, base));
        if constexpr (kType == GQ_TYPE_Q4_0) {
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t q = word_at(r, base + 2 + 4 * i);
                lo[i] = ((q << 4) & 0xF0F0F0F0u) ^ 0x80808080u;   // bytes 16*(c-8), elems 4i..
                hi[i] = (q & 0xF0F0F0F0u) ^ 0x80808080u;          // elems 16+4i..
            }
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                const uint4* xw = reinterpret_cast<const uint4*>(xrec0 + t * rec_stride + 64 * j);
                const uint4 x0 = xw[0], x1 = xw[1], x2 = xw[2], x3 = xw[3];
                int s0 = 0, s1 = 0;
                s0 = __dp2a_lo(static_cast<int>(x0.x), static_cast<int>(lo[0]), s0);
                s0 = __dp2a_hi(static_cast<int>(x0.y), static_cast<int>(lo[0]), s0);
                s1 = __dp2a_lo(static_cast<int>(x0.z), static_cast<int>(lo[1]), s1);
                s1 = __dp2a_hi(static_cast<int>(x0.w), static_cast<int>(lo[1]), s1);
                s0 = __dp2a_lo(static_cast<int>(x1.x), static_cast<int>(lo[2]), s0);
                s0 = __dp2a_hi(static_cast<int>(x1.y), static_cast<int>(lo[2]), s0);
                s1 = __dp2a_lo(static_cast<int>(x1.z), static_cast<int>(lo[3]), s1);
                s1 = __dp2a_hi(static_cast<int>(x1.w), static_cast<int>(lo[3]), s1);
                s0 = __dp2a_lo(static_cast<int>(x2.x), static_cast<int>(hi[0]), s0);
                s0 = __dp2a_hi(static_cast<int>(x2.y), static_cast<int>(hi[0]), s0);
                s1 = __dp2a_lo(static_cast<int>(x2.z), static_cast<int>(hi[1]), s1);
                s1 = __dp2a_hi(static_cast<int>(x2.w), static_cast<int>(hi[1]), s1);
                s0 = __dp2a_lo(static_cast<int>(x3.x), static_cast<int>(hi[2]), s0);
                s0 = __dp2a_hi(static_cast<int>(x3.y), static_cast<int>(hi[2]), s0);
                s1 = __dp2a_lo(static_cast<int>(x3.z), static_cast<int>(hi[3]), s1);
                s1 = __dp2a_hi(static_cast<int>(x3.w), static_cast<int>(hi[3]), s1);
                acc[t] = fmaf(d, static_cast<float>(s0 + s1), acc[t]);
            }
        } else {
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
    }
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        const int e = *reinterpret_cast<const int*>(xrec0 + t * rec_stride + G::kWPC * 2);
        out[t] = ldexpf(acc[t], e);
    }
}

template <int kType, int kNT, int kMaxProbs>
__global__ void __launch_bounds__(kThreads, 1)
gemv_stream_kernel(const __grid_constant__ GemvParams<kMaxProbs> P) {
    using G = Geo<kType>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* raw = smem;
    uint8_t* xbuf = raw + kStages * G::kStageBytes;
    const int64_t xbytes = static_cast<int64_t>(kNT) * P.max_c * G::kXRec;
    float* partial = reinterpret_cast<float*>(xbuf + xbytes);     // [2][kThreads][kNT]
    float* carry = partial + 2 * kThreads * kNT;                  // [2][kNT]
    uint64_t* bars = reinterpret_cast<uint64_t*>(carry + 2 * kNT + 2);   // 8-byte aligned

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    // This CTA's rows: from the first row starting at or after byte c*T/G to the first
    // row starting at or after byte (c+1)*T/G.
    int p0, p1;
    int64_t r0, r1;
    row_at_byte(P, P.total_bytes * blockIdx.x / gridDim.x, p0, r0);
    row_at_byte(P, P.total_bytes * (blockIdx.x + 1) / gridDim.x, p1, r1);

    Cursor prod, cons;
    open_segment(P, prod, p0, r0, p1, r1);
    cons = prod;

    int issued = 0;
    auto issue = [&](int s) {
        const GemvProb& pr = P.p[prod.p];
        const int cnt = static_cast<int>(min(static_cast<int64_t>(kThreads), prod.n_chunks - prod.chunk));
        const uint32_t bytes = static_cast<uint32_t>(cnt) * G::kChunkBytes;
        const uint8_t* src =
            pr.W + prod.r_begin * pr.row_bytes + prod.chunk * G::kChunkBytes;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_evict_first(smem_addr(raw + s * G::kStageBytes), src, bytes, bar);
        advance(P, prod, p1, r1);
        ++issued;
    };
    if (tid == 0)
        for (int s = 0; s < kStages && prod.valid; ++s) issue(s);

    int stage = 0;
    int cur_prob = -1;
    bool failed = false;
    const int rec_stride = P.max_c * G::kXRec;
    while (cons.valid) {
        const GemvProb& pr = P.p[cons.p];
        if (cons.p != cur_prob) {
            prepare_x<kType, kNT>(pr, P.n_tok, P.max_c, xbuf);
            __syncthreads();
            cur_prob = cons.p;
        }
        const int s = stage % kStages;
        const int cnt = static_cast<int>(min(static_cast<int64_t>(kThreads), cons.n_chunks - cons.chunk));
        const bool ok = mbar_wait(smem_addr(&bars[s]), (stage / kStages) & 1);
        float part[kNT];
#pragma unroll
        for (int t = 0; t < kNT; ++t) part[t] = 0.0f;
        if (ok && tid < cnt) {
            const int64_t g = cons.chunk + tid;            // chunk index within segment
            const int col = static_cast<int>(g % pr.C);
            chunk_dot<kType, kNT>(raw + s * G::kStageBytes + tid * G::kChunkBytes,
                                  xbuf + col * G::kXRec, rec_stride, part);
        }
        float* pbuf = partial + (stage & 1) * kThreads * kNT;
#pragma unroll
        for (int t = 0; t < kNT; ++t) pbuf[tid * kNT + t] = part[t];
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        // Row sums in k order; a row cut by the stage end carries into the next stage.
        {
            const int64_t s0 = cons.chunk;
            const int64_t C = pr.C;
            const int64_t r_first = s0 / C;
            const int nrows = static_cast<int>((s0 + cnt - 1) / C - r_first + 1);
            const float* cin = carry + ((stage + 1) & 1) * kNT;
            float* cout = carry + (stage & 1) * kNT;
            for (int rr = tid; rr < nrows; rr += kThreads) {
                const int64_t r = r_first + rr;
                const int64_t cb = max(s0, r * C);
                const int64_t ce = min(s0 + cnt, (r + 1) * C);
                float acc[kNT];
#pragma unroll
                for (int t = 0; t < kNT; ++t) acc[t] = cb > r * C ? cin[t] : 0.0f;
                for (int64_t c = cb; c < ce; ++c) {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) acc[t] += pbuf[(c - s0) * kNT + t];
                }
                if (ce == (r + 1) * C) {
                    const int64_t row = cons.r_begin + r;
#pragma unroll
                    for (int t = 0; t < kNT; ++t)
                        if (t < P.n_tok) pr.Y[t * pr.M + row] = acc[t];
                } else {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) cout[t] = acc[t];
                }
            }
        }
        if (tid == 0 && prod.valid) issue(s);
        advance(P, cons, p1, r1);
        ++stage;
    }
    if (failed && tid == 0) {
        report_status(P.status, kStatusTimeout);
        // Let copies already in flight land before this CTA's shared memory is released.
        for (int st = stage; st < issued; ++st)
            mbar_wait(smem_addr(&bars[st % kStages]), (st / kStages) & 1, 100000000ull);
    }
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

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
template <int kType>
int64_t stream_smem_bytes(int n_tok_template, int max_c) {
    using G = Geo<kType>;
    return static_cast<int64_t>(kStages) * G::kStageBytes +
           static_cast<int64_t>(n_tok_template) * max_c * G::kXRec +
           (2 * kThreads * n_tok_template + 2 * n_tok_template + 2) * 4 + kStages * 8 + 8;
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

template <int kType, int kNT, int kMaxProbs>
cudaError_t launch_stream_t(const GemvParams<kMaxProbs>& P, const DeviceInfo* info,
                            cudaStream_t s) {
    auto kernel = gemv_stream_kernel<kType, kNT, kMaxProbs>;
    const int64_t smem = stream_smem_bytes<kType>(kNT, P.max_c);
    cudaError_t e = ensure_smem(kernel, info->device, smem);
    if (e != cudaSuccess) return e;
    // Enough CTAs that each streams at least ~32 KB, at most one per SM.
    int64_t grid = (P.total_bytes + 32767) / 32768;
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, info->sm_count));
    kernel<<<static_cast<int>(grid), kThreads, static_cast<size_t>(smem), s>>>(P);
    return cudaGetLastError();
}

template <int kType, int kMaxProbs>
cudaError_t launch_stream_nt(const GemvParams<kMaxProbs>& P, const DeviceInfo* info,
                             cudaStream_t s) {
    switch (P.n_tok) {
        case 1: return launch_stream_t<kType, 1, kMaxProbs>(P, info, s);
        case 2: return launch_stream_t<kType, 2, kMaxProbs>(P, info, s);
        case 3: return launch_stream_t<kType, 3, kMaxProbs>(P, info, s);
        default: return launch_stream_t<kType, 4, kMaxProbs>(P, info, s);
    }
}

template <int kMaxProbs>
cudaError_t launch_stream(gq_type t, const MatProblem* probs, int count, int64_t tok0,
                          int n_tok, const DeviceInfo* info, cudaStream_t s) {
    GemvParams<kMaxProbs> P{};
    P.count = count;
    P.n_tok = n_tok;
    P.status = info->status;
    const int wpc = t == GQ_TYPE_Q4_0 ? Geo<GQ_TYPE_Q4_0>::kWPC : Geo<GQ_TYPE_Q8_0>::kWPC;
    const int cb = t == GQ_TYPE_Q4_0 ? Geo<GQ_TYPE_Q4_0>::kChunkBytes
                                     : Geo<GQ_TYPE_Q8_0>::kChunkBytes;
    int64_t bytes = 0;
    int max_c = 1;
    for (int i = 0; i < count; ++i) {
        GemvProb& g = P.p[i];
        g.W = probs[i].W;
        g.X = probs[i].X + tok0 * probs[i].K;
        g.Y = probs[i].Y + tok0 * probs[i].M;
        g.M = probs[i].M;
        g.K = static_cast<int32_t>(probs[i].K);
        g.C = static_cast<int32_t>(probs[i].K / wpc);
        g.row_bytes = static_cast<int64_t>(g.C) * cb;
        g.byte_begin = bytes;
        bytes += g.M * g.row_bytes;
        max_c = std::max(max_c, g.C);
    }
    P.total_bytes = bytes;
    P.max_c = max_c;
    if (t == GQ_TYPE_Q4_0) return launch_stream_nt<GQ_TYPE_Q4_0, kMaxProbs>(P, info, s);
    return launch_stream_nt<GQ_TYPE_Q8_0, kMaxProbs>(P, info, s);
}

cudaError_t launch_generic(gq_type t, const MatProblem& p, int64_t tok0, int n_tok,
                           const DeviceInfo* info, cudaStream_t s) {
    const int64_t blocks = (p.M + 7) / 8;
    const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(info->sm_count) * 8));
    const float* X = p.X + tok0 * p.K;
    float* Y = p.Y + tok0 * p.M;
    if (t == GQ_TYPE_Q4_0)
        gemv_generic_kernel<GQ_TYPE_Q4_0><<<grid, 256, 0, s>>>(p.W, p.M, p.K, X, n_tok, Y);
    else
        gemv_generic_kernel<GQ_TYPE_Q8_0><<<grid, 256, 0, s>>>(p.W, p.M, p.K, X, n_tok, Y);
    return cudaGetLastError();
}

bool stream_eligible(gq_type t, const MatProblem& p, const DeviceInfo* info) {
    if (p.K % 256 != 0 || p.K > (int64_t(1) << 30)) return false;
    if (reinterpret_cast<uintptr_t>(p.X) % 16 != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.W) % 16 != 0) return false;
    const int64_t c = p.K / (t == GQ_TYPE_Q4_0 ? 256 : 128);
    const int64_t smem = t == GQ_TYPE_Q4_0 ? stream_smem_bytes<GQ_TYPE_Q4_0>(kMaxTok, c)
                                           : stream_smem_bytes<GQ_TYPE_Q8_0>(kMaxTok, c);
    return smem <= info->max_smem_optin;
}

}  // namespace

cudaError_t launch_mul_mat(gq_type t, const MatProblem* probs, int count, int64_t N,
                           cudaStream_t s) {
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    MatProblem fast[GQ_MAX_BATCH];
    int n_fast = 0;
    for (int64_t tok0 = 0; tok0 < N; tok0 += kMaxTok) {
        const int n_tok = static_cast<int>(std::min<int64_t>(kMaxTok, N - tok0));
        n_fast = 0;
        for (int i = 0; i < count; ++i) {
            if (stream_eligible(t, probs[i], info)) {
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

}  // namespace gq
