// gq_quant.cu -- quantize (fp32 -> Q4_0 / Q8_0 blocks) and dequantize kernels.
//
// Quantization follows "A Complete Guide to llama.cpp and Customization with C++",
// section 2.2 (w_i ~= Delta * q_i, Delta = max|w_i| / 7, q_i in [-8, 7]) with the Q4_0
// block of "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
// section 6.1 (fp16 scale + 32 4-bit codes). It must be bit-exact, so it uses IEEE
// division (this file is built without fast-math), roundf (halves away from zero) and
// __float2half_rn (round to nearest even, subnormals kept).
//
// Because W is row-major and K is a multiple of the block, block b covers the consecutive
// floats W[wb .. wb + w - 1] (w = 32 weights, 256 for a Q4_K super-block) of the flattened
// matrix, and its bytes start at b * block_bytes. One warp quantizes one block per step:
// lane i owns element i (32-weight blocks) or elements 8i .. 8i + 7 (Q4_K).
//
// Q4_K super-blocks follow the published GGUF Q4_K layout (the pages name the format
// without one: "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
// section 6): fp16 d and dmin, twelve bytes of packed 6-bit sub-block scales sc_j and mins
// m_j, then 128 bytes of 4-bit codes (byte 32 g + l: weight 64 g + l in the low nibble,
// 64 g + 32 + l in the high one), What = d sc_j q - dmin m_j. The quantizer is this
// library's own: per 32-weight sub-block lo = min(0, min w), hi = max w, step =
// (hi - lo) / 15, min = -lo; d = max step / 63, dmin = max min / 63; sc_j = roundf(step_j
// / d), m_j = roundf(min_j / dmin) in [0, 63]; codes roundf((w + M_j) / D_j) in [0, 15]
// against D_j = fp16(d) sc_j, M_j = fp16(dmin) m_j. Bit-exact for finite inputs.
#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_q4_0_kernel(const float* __restrict__ W, int64_t n_blocks, uint8_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + threadIdx.x / 32;
         b < n_blocks; b += warps) {
        const float w = W[b * 32 + lane];
        const float amax = warp_max(fabsf(w));
        const float d = amax / 7.0f;
        int code = 8;
        if (d != 0.0f) code = min(15, max(0, static_cast<int>(roundf(w / d)) + 8));
        const int code_hi = __shfl_down_sync(0xFFFFFFFFu, code, 16);   // element lane+16
        uint8_t* blk = out + b * kQ4Bytes;
        if (lane == 0)
            *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(__float2half_rn(d));
        if (lane < 16) blk[2 + lane] = static_cast<uint8_t>(code | (code_hi << 4));
    }
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_0_kernel(const float* __restrict__ W, int64_t n_blocks, uint8_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + threadIdx.x / 32;
         b < n_blocks; b += warps) {
        const float w = W[b * 32 + lane];
        const float amax = warp_max(fabsf(w));
        const float d = amax / 127.0f;
        int code = 0;
        if (d != 0.0f) code = min(127, max(-127, static_cast<int>(roundf(w / d))));
        uint8_t* blk = out + b * kQ8Bytes;
        if (lane == 0)
            *reinterpret_cast<unsigned short*>(blk) = __half_as_ushort(__float2half_rn(d));
        blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(code));
    }
}

// Q4_K, one warp per super-block. Lane l holds elements 8l .. 8l + 7, i.e. part of
// sub-block l / 4; sub-block extremes come from the four lanes of the sub-block, the
// super-block's largest step and min from all eight sub-blocks.
__global__ void __launch_bounds__(kQuantThreads)
quantize_q4_k_kernel(const float* __restrict__ W, int64_t n_sb, uint8_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + threadIdx.x / 32;
         b < n_sb; b += warps) {
        const float* src = W + b * kQ4KWeights + 8 * lane;   // W is only 4-byte aligned
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = src[i];
        float lo = v[0], hi = v[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            lo = fminf(lo, v[i]);
            hi = fmaxf(hi, v[i]);
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
        }
        lo = fminf(lo, 0.0f);
        const float step = (hi - lo) / 15.0f;
        const float mn = 0.0f - lo;
        float smax = step, mmax = mn;   // both >= 0
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, o));
            mmax = fmaxf(mmax, __shfl_xor_sync(0xFFFFFFFFu, mmax, o));
        }
        // The largest positive value, else +0 (a -0 here would store d or dmin as -0).
        if (!(smax > 0.0f)) smax = 0.0f;
        if (!(mmax > 0.0f)) mmax = 0.0f;
        const float d = smax / 63.0f;
        const float dmin = mmax / 63.0f;
        const __half dh = __float2half_rn(d);
        const __half dminh = __float2half_rn(dmin);
        int sc = 0, m = 0;
        if (d != 0.0f) sc = min(63, max(0, static_cast<int>(roundf(step / d))));
        if (dmin != 0.0f) m = min(63, max(0, static_cast<int>(roundf(mn / dmin))));
        // the dequantization's own D_j and M_j (both products exact)
        const float D = __fmul_rn(__half2float(dh), static_cast<float>(sc));
        const float M = __fmul_rn(__half2float(dminh), static_cast<float>(m));
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = 0;
            if (D != 0.0f) q = min(15, max(0, static_cast<int>(roundf(__fadd_rn(v[i], M) / D))));
            packed[i >> 2] |= static_cast<uint32_t>(q) << (8 * (i & 3));
        }
        // Lane l with l % 8 < 4 holds the low nibbles of bytes 32 (l / 8) + 8 (l % 8) + i;
        // lane l + 4 holds the high nibbles of the same bytes.
        const uint32_t up0 = __shfl_down_sync(0xFFFFFFFFu, packed[0], 4);
        const uint32_t up1 = __shfl_down_sync(0xFFFFFFFFu, packed[1], 4);
        // All eight sub-blocks' scales and mins, for the header.
        int scs[8], ms[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            scs[j] = __shfl_sync(0xFFFFFFFFu, sc, 4 * j);
            ms[j] = __shfl_sync(0xFFFFFFFFu, m, 4 * j);
        }
        uint8_t* blk = out + b * kQ4KBytes;
        if ((lane & 7) < 4)
            *reinterpret_cast<uint2*>(blk + 16 + 32 * (lane >> 3) + 8 * (lane & 7)) =
                make_uint2(packed[0] | (up0 << 4), packed[1] | (up1 << 4));
        if (lane == 0) {
            uint32_t sw[3] = {0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t s0 = (scs[j] & 63) | ((scs[j + 4] >> 4) << 6);
                const uint32_t s1 = (ms[j] & 63) | ((ms[j + 4] >> 4) << 6);
                const uint32_t s2 = (scs[j + 4] & 15) | ((ms[j + 4] & 15) << 4);
                sw[0] |= s0 << (8 * j);
                sw[1] |= s1 << (8 * j);
                sw[2] |= s2 << (8 * j);
            }
            const uint32_t h = static_cast<uint32_t>(__half_as_ushort(dh)) |
                               (static_cast<uint32_t>(__half_as_ushort(dminh)) << 16);
            *reinterpret_cast<uint4*>(blk) = make_uint4(h, sw[0], sw[1], sw[2]);
        }
    }
}

// One thread per output element: What = (c - 8) * d or c * d, exact in fp32.
template <int kType>
__global__ void __launch_bounds__(256)
dequantize_kernel(const uint8_t* __restrict__ blocks, int64_t n_elems, float* __restrict__ out) {
    constexpr int kBB = kType == GQ_TYPE_Q4_0 ? kQ4Bytes : kQ8Bytes;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_elems;
         e += stride) {
        const uint8_t* blk = blocks + (e >> 5) * kBB;
        const int i = static_cast<int>(e & 31);
        const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(blk));
        float w;
        if (kType == GQ_TYPE_Q4_0) {
            const int byte = blk[2 + (i & 15)];
            const int code = i < 16 ? (byte & 15) : (byte >> 4);
            w = static_cast<float>(code - 8) * d;
        } else {
            w = static_cast<float>(static_cast<int8_t>(blk[2 + i])) * d;
        }
        out[e] = w;
    }
}

// Q4_K, one thread per output element: What = D_j q - M_j, D_j = d sc_j and M_j = dmin m_j
// exact in fp32, D_j q exact, one rounding at the subtraction.
__global__ void __launch_bounds__(256)
dequantize_q4_k_kernel(const uint8_t* __restrict__ blocks, int64_t n_elems,
                       float* __restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_elems;
         e += stride) {
        const uint8_t* sb = blocks + (e >> 8) * kQ4KBytes;
        const int o = static_cast<int>(e & 255);
        const int j = o >> 5, l = o & 31;
        const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb));
        const float dmin = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb + 2));
        const uint8_t* sc6 = sb + 4;
        int sc, m;
        if (j < 4) {
            sc = sc6[j] & 63;
            m = sc6[j + 4] & 63;
        } else {
            sc = (sc6[j + 4] & 15) | ((sc6[j - 4] >> 6) << 4);
            m = (sc6[j + 4] >> 4) | ((sc6[j] >> 6) << 4);
        }
        const int byte = sb[16 + 32 * (j >> 1) + l];
        const int q = (j & 1) ? (byte >> 4) : (byte & 15);
        const float D = __fmul_rn(d, static_cast<float>(sc));
        const float M = __fmul_rn(dmin, static_cast<float>(m));
        out[e] = __fsub_rn(__fmul_rn(D, static_cast<float>(q)), M);
    }
}

int grid_for(int64_t work_items, int per_block, const DeviceInfo* info) {
    const int64_t want = (work_items + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(info->sm_count) * 16;
    return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_quantize(gq_type t, const float* W, int64_t n_blocks, uint8_t* out,
                            cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(n_blocks, kQuantThreads / 32, info);
    if (t == GQ_TYPE_Q4_0)
        quantize_q4_0_kernel<<<grid, kQuantThreads, 0, s>>>(W, n_blocks, out);
    else if (t == GQ_TYPE_Q8_0)
        quantize_q8_0_kernel<<<grid, kQuantThreads, 0, s>>>(W, n_blocks, out);
    else
        quantize_q4_k_kernel<<<grid, kQuantThreads, 0, s>>>(W, n_blocks, out);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(gq_type t, const uint8_t* blocks, int64_t n_elems, float* out,
                              cudaStream_t s) {
    if (n_elems == 0) return cudaSuccess;
    DeviceInfo* info = nullptr;
    cudaError_t e = current_device_info(&info);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(n_elems, 256, info);
    if (t == GQ_TYPE_Q4_0)
        dequantize_kernel<GQ_TYPE_Q4_0><<<grid, 256, 0, s>>>(blocks, n_elems, out);
    else if (t == GQ_TYPE_Q8_0)
        dequantize_kernel<GQ_TYPE_Q8_0><<<grid, 256, 0, s>>>(blocks, n_elems, out);
    else
        dequantize_q4_k_kernel<<<grid, 256, 0, s>>>(blocks, n_elems, out);
    return cudaGetLastError();
}

}  // namespace gq
