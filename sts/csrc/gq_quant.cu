// gq_quant.cu -- quantize (fp32 -> Q4_0 / Q8_0 blocks) and dequantize kernels.
//
// Quantization follows "A Complete Guide to llama.cpp and Customization with C++",
// section 2.2 (w_i ~= Delta * q_i, Delta = max|w_i| / 7, q_i in [-8, 7]) with the Q4_0
// block of "Development Guide for Small AI Models (TinyLLaMA, etc.) Using C++",
// section 6.1 (fp16 scale + 32 4-bit codes). It must be bit-exact, so it uses IEEE
// division (this file is built without fast-math), roundf (halves away from zero) and
// __float2half_rn (round to nearest even, subnormals kept).
//
// Because W is row-major and K is a multiple of 32, block b covers the 32 consecutive
// floats W[32b .. 32b+31] of the flattened matrix, and its bytes start at b * block_bytes.
// One warp quantizes one block per step: lane i owns element i.
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
    else
        quantize_q8_0_kernel<<<grid, kQuantThreads, 0, s>>>(W, n_blocks, out);
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
    else
        dequantize_kernel<GQ_TYPE_Q8_0><<<grid, 256, 0, s>>>(blocks, n_elems, out);
    return cudaGetLastError();
}

}  // namespace gq
