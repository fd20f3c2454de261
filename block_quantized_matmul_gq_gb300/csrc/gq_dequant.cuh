// gq_dequant.cuh -- block dequantization to bf16 operand tiles for the tensor-core
// kernels (prefill GEMM and tensor-core decode): raw Q4_0 / Q8_0 bytes in registers ->
// (c - 8) * d or c * d, exact in fp32, rounded once to bf16, stored as 16-byte chunks of a
// 128-byte-swizzled K-major row ("Development Guide for Small AI Models (TinyLLaMA, etc.)
// Using C++", section 6.2: unpack with masks and shifts, then scale). Q4_K sub-blocks
// (published GGUF Q4_K layout) become d sc q - dmin m, rounded once in fp32 exactly as
// gq_dequantize writes it, then once more to bf16.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace dq {

template <int kType>
struct RawFmt;
template <>
struct RawFmt<GQ_TYPE_Q4_0> {
    static constexpr int kBB = kQ4Bytes;
    static constexpr int kRow = 8 * kQ4Bytes;   // 144 bytes per row per super-step
    static constexpr int kElem = 1;             // tensor-map element size (uint8)
};
template <>
struct RawFmt<GQ_TYPE_Q8_0> {
    static constexpr int kBB = kQ8Bytes;
    static constexpr int kRow = 8 * kQ8Bytes;   // 272 bytes
    static constexpr int kElem = 2;             // uint16 elements keep the box <= 256
};
template <>
struct RawFmt<GQ_TYPE_Q4_K> {
    static constexpr int kBB = kQ4KBytes;       // the super-step is one super-block
    static constexpr int kRow = kQ4KBytes;      // 144 bytes, as Q4_0
    static constexpr int kElem = 1;
};

__device__ __forceinline__ uint32_t word_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? __funnelshift_r(r[w], r[w + 1], 16) : r[w];
}

__device__ __forceinline__ uint32_t u16_at(const uint32_t* r, int byte_off) {
    const int w = byte_off >> 2;
    return (byte_off & 3) ? (r[w] >> 16) : (r[w] & 0xFFFFu);
}

// Byte k (0..3) of `word` as the float 2^23 + byte: the byte lands in the low mantissa.
template <int k>
__device__ __forceinline__ float byte_as_float(uint32_t word) {
    return __int_as_float(static_cast<int>(__byte_perm(word, 0x4B000000u, 0x7540u | k)));
}

// (a - b) * c on two fp32 lanes at once (Blackwell packed fp32), round to nearest.
__device__ __forceinline__ float2 sub_mul2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 a, b, c, t;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "sub.rn.f32x2 t, a, b;\n\tmul.rn.f32x2 t, t, c;\n\t"
        "mov.b64 {%0, %1}, t;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// (y0, y1) = fma(d, (a0, a1), (y0, y1)) on two fp32 lanes at once (Blackwell packed fp32):
// each lane rounded once, exactly like fmaf.
__device__ __forceinline__ void fma2_bcast(float& y0, float& y1, float d, float a0, float a1) {
    asm("{\n\t.reg .b64 y, a, dd;\n\t"
        "mov.b64 y, {%0, %1};\n\tmov.b64 a, {%2, %3};\n\tmov.b64 dd, {%4, %4};\n\t"
        "fma.rn.f32x2 y, dd, a, y;\n\t"
        "mov.b64 {%0, %1}, y;\n\t}"
        : "+f"(y0), "+f"(y1)
        : "f"(a0), "f"(a1), "f"(d));
}

// Dequantizes the block that starts at byte kOff of the raw bytes in r (kOff even) into
// 32 bf16 values packed in pairs: out[i] = elements 2i (low half) and 2i+1 (high half).
// Each value is the exact (c - 8) * d (Q4_0) or c * d (Q8_0) (at most 8 + 11 significant
// bits) rounded once to bf16.
template <int kType, int kOff>
__device__ __forceinline__ void dequant_block_at(const uint32_t* r, uint32_t (&out)[16]) {
    static_assert(kOff % 2 == 0, "blocks start on 2-byte boundaries");
    constexpr int base = kOff;
    const float d = half_bits_to_float(u16_at(r, base));
    if constexpr (kType == GQ_TYPE_Q4_0) {
        // In bf16x2 arithmetic, two elements per instruction. A nibble byte c placed under
        // the bf16 bit pattern 0x43 is the exact value 128 + c; subtracting 136 gives the
        // exact c - 8. The scale splits exactly into d = d_hi + d_lo (d_hi = bf16(d); d has
        // 11 significant bits, so the remainder has at most 4 and is a bf16 value), the
        // product (c - 8) * d_lo is exact in bf16, and fma(c - 8, d_hi, (c - 8) * d_lo)
        // rounds the exact (c - 8) * d once: the same bf16 as rounding it from fp32.
        const __nv_bfloat16 dh = __float2bfloat16_rn(d);
        const __nv_bfloat16 dl = __float2bfloat16_rn(d - __bfloat162float(dh));
        const __nv_bfloat162 dh2 = __halves2bfloat162(dh, dh);
        const __nv_bfloat162 dl2 = __halves2bfloat162(dl, dl);
        const __nv_bfloat162 off = __float2bfloat162_rn(136.0f);
        auto pair = [&](uint32_t bytes4, uint32_t sel) {
            const uint32_t v = __byte_perm(bytes4, 0x43434343u, sel);   // (128 + c, 128 + c')
            const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
            const __nv_bfloat162 a = __hfma2(q, dh2, __hmul2(q, dl2));
            return *reinterpret_cast<const uint32_t*>(&a);
        };
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w = word_at(r, base + 2 + 4 * i);
            const uint32_t lo = w & 0x0F0F0F0Fu;           // elements 4i..4i+3
            const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;    // elements 16+4i..
            out[2 * i] = pair(lo, 0x4140u);
            out[2 * i + 1] = pair(lo, 0x4342u);
            out[8 + 2 * i] = pair(hi, 0x4140u);
            out[8 + 2 * i + 1] = pair(hi, 0x4342u);
        }
    } else {
        // fp32: each code byte under the pattern of 2^23 is 2^23 + c + 128 exactly; the
        // exact c * d (packed f32x2) is rounded once to bf16.
        const float2 dd = make_float2(d, d);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = word_at(r, base + 2 + 4 * i) ^ 0x80808080u;   // c + 128
            v[4 * i + 0] = byte_as_float<0>(w);
            v[4 * i + 1] = byte_as_float<1>(w);
            v[4 * i + 2] = byte_as_float<2>(w);
            v[4 * i + 3] = byte_as_float<3>(w);
        }
        const float2 off = make_float2(8388736.0f, 8388736.0f);   // 2^23 + 128
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 p = sub_mul2(make_float2(v[2 * i], v[2 * i + 1]), off, dd);
            const __nv_bfloat162 b = __floats2bfloat162_rn(p.x, p.y);
            out[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
}

// (a - b) * c + e on two fp32 lanes at once (Blackwell packed fp32): the subtraction is
// exact where it is used (2^23 + q - 2^23), the fma rounds once.
__device__ __forceinline__ float2 sub_fma2(float2 a, float2 b, float2 c, float2 e) {
    float2 r;
    asm("{\n\t.reg .b64 a, b, c, e, t;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "mov.b64 e, {%8, %9};\n\t"
        "sub.rn.f32x2 t, a, b;\n\tfma.rn.f32x2 t, t, c, e;\n\t"
        "mov.b64 {%0, %1}, t;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(e.x), "f"(e.y));
    return r;
}

// Q4_K sub-block 2 quarter + h of a super-block: hd = its 16 header bytes (fp16 d and
// dmin, the packed 6-bit scales and mins), cw[0..7] = the quarter's 32 code bytes (word i:
// elements 4i .. 4i + 3 of the sub-block, in nibble h of each byte). Each value is
// fma(q, D, -M) with D = d sc and M = dmin m (both exact), i.e. d sc q - dmin m rounded
// once in fp32, then rounded to bf16; out[i] = elements 2i, 2i + 1.
template <int h>
__device__ __forceinline__ void dequant_q4k_sub(const uint4& hd, int quarter, const uint32_t* cw,
                                                uint32_t (&out)[16]) {
    uint32_t sc2, m2;
    q4k_scales(hd, quarter, sc2, m2);
    const float D = __fmul_rn(half_bits_to_float(hd.x & 0xFFFFu),
                              static_cast<float>((sc2 >> (8 * h)) & 0xFFu));
    const float Mn = -__fmul_rn(half_bits_to_float(hd.x >> 16),
                                static_cast<float>((m2 >> (8 * h)) & 0xFFu));
    const float2 dd = make_float2(D, D), mm = make_float2(Mn, Mn);
    const float2 off = make_float2(8388608.0f, 8388608.0f);   // 2^23
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = (cw[i] >> (4 * h)) & 0x0F0F0F0Fu;
        const float2 p0 = sub_fma2(make_float2(byte_as_float<0>(w), byte_as_float<1>(w)), off, dd, mm);
        const float2 p1 = sub_fma2(make_float2(byte_as_float<2>(w), byte_as_float<3>(w)), off, dd, mm);
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(p0.x, p0.y);
        const __nv_bfloat162 b1 = __floats2bfloat162_rn(p1.x, p1.y);
        out[2 * i] = *reinterpret_cast<const uint32_t*>(&b0);
        out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&b1);
    }
}

// Q4_K sub-block j (0..7) of the super-block whose 144 bytes are in r (header words
// r[0..3], quarter q's code words r[4 + 8q .. 4 + 8q + 7]).
template <int j>
__device__ __forceinline__ void dequant_subblock_q4k(const uint32_t* r, uint32_t (&out)[16]) {
    dequant_q4k_sub<j & 1>(make_uint4(r[0], r[1], r[2], r[3]), j >> 1, r + 4 + 8 * (j >> 1), out);
}

// Codes only: the 32 exact integers c - 8 of the Q4_0 block that starts at byte kOff of r,
// as bf16 pairs in the order of dequant_block_at (out[i] = elements 2i, 2i + 1). The
// block's scale is applied to the product afterwards, in fp32.
template <int kOff>
__device__ __forceinline__ void q4_codes_at(const uint32_t* r, uint32_t (&out)[16]) {
    static_assert(kOff % 2 == 0, "blocks start on 2-byte boundaries");
    const __nv_bfloat162 off = __float2bfloat162_rn(136.0f);
    auto pair = [&](uint32_t bytes4, uint32_t sel) {
        const uint32_t v = __byte_perm(bytes4, 0x43434343u, sel);   // (128 + c, 128 + c')
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
        return *reinterpret_cast<const uint32_t*>(&q);
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = word_at(r, kOff + 2 + 4 * i);
        const uint32_t lo = w & 0x0F0F0F0Fu;
        const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
        out[2 * i] = pair(lo, 0x4140u);
        out[2 * i + 1] = pair(lo, 0x4342u);
        out[8 + 2 * i] = pair(hi, 0x4140u);
        out[8 + 2 * i + 1] = pair(hi, 0x4342u);
    }
}

// Codes only, Q4_K: the 32 exact codes q (0..15) of one sub-block as bf16 pairs in the
// order of dequant_q4k_sub (out[i] = elements 2i, 2i + 1); cw[0..7] are the quarter's code
// words, nibble h. The scales and mins are applied to the product afterwards, in fp32.
template <int h>
__device__ __forceinline__ void q4k_codes(const uint32_t* cw, uint32_t (&out)[16]) {
    const __nv_bfloat162 off = __float2bfloat162_rn(128.0f);
    auto pair = [&](uint32_t bytes4, uint32_t sel) {
        const uint32_t v = __byte_perm(bytes4, 0x43434343u, sel);   // (128 + q, 128 + q')
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
        return *reinterpret_cast<const uint32_t*>(&q);
    };
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = (cw[i] >> (4 * h)) & 0x0F0F0F0Fu;   // elements 4i .. 4i + 3
        out[2 * i] = pair(w, 0x4140u);
        out[2 * i + 1] = pair(w, 0x4342u);
    }
}

// Block `blk` (0..7) of a row's super-step (Q4_K: sub-block blk of its super-block), raw
// bytes in r from the super-step's start.
template <int kType, int blk>
__device__ __forceinline__ void dequant_block(const uint32_t* r, uint32_t (&out)[16]) {
    if constexpr (kType == GQ_TYPE_Q4_K)
        dequant_subblock_q4k<blk>(r, out);
    else
        dequant_block_at<kType, blk * RawFmt<kType>::kBB>(r, out);
}

// Block 2q + h of the super-step, as four 16-byte chunks of the A row (elements
// 32h .. 32h + 31 of the 64-k stage), stored at chunk (4h + c) ^ (row % 8), each with one
// 128-bit shared store (measured 0.5-1.5 % faster on the LLaMA-7B prefill shapes than
// the plain vector assignment).
template <int kType, int q, int h>
__device__ __forceinline__ void dequant_store(const uint32_t* r, uint8_t* arow, int row) {
    uint32_t packed[16];
    dequant_block<kType, 2 * q + h>(r, packed);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::
                     "r"(smem_addr(arow + (((4 * h + c) ^ (row & 7)) << 4))),
                     "r"(packed[4 * c]), "r"(packed[4 * c + 1]), "r"(packed[4 * c + 2]),
                     "r"(packed[4 * c + 3]) : "memory");
}

}  // namespace dq
}  // namespace gq
