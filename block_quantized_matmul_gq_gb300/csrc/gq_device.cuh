// gq_device.cuh -- device-side building blocks shared by the libgq kernels (sm_103a):
// shared-memory mbarriers, 1-D bulk (TMA) copies global -> shared, bounded waits and the
// per-device status word. Inline PTX only; no CUTLASS/CuTe.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gq {

// Status bits written to the per-device status word by kernels that gave up waiting.
constexpr unsigned kStatusTimeout = 1u;

// A wait on an mbarrier that lasts longer than this is treated as a hang: the kernel
// records kStatusTimeout and leaves. Legitimate waits last microseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

// Programmatic dependent launch. launch_dependents lets the next kernel of the stream
// (launched with the programmatic-serialization attribute) be scheduled once every CTA
// of this grid has executed it; its CTAs then take SMs as this grid's CTAs leave.
// griddep_wait blocks until every prerequisite grid has completed and its memory
// operations are visible. Both are no-ops in a grid launched without the attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies) and the CTA.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Like mbar_try_wait, but a thread whose phase is not complete is suspended for up to
// `hint_ns` (or until the phase completes) instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier to complete; false if it has not after `limit`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
        if (global_ns() - t0 > limit) return false;
    }
}

// 1-D bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same, with an L2 eviction hint: streamed-once data (weights at decode) goes first.
__device__ __forceinline__ void bulk_g2s_evict_first(uint32_t dst, const void* src,
                                                     uint32_t bytes, uint32_t bar) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Before a shared-memory buffer that this thread has just read with ordinary loads is
// handed back for an async-proxy write (a bulk / TMA copy): waits for the loaded values
// (the dummy register depends on all of them) and orders the generic-proxy reads before
// later async-proxy accesses.
__device__ __forceinline__ void release_to_async_proxy(uint32_t depends_on_loads) {
    asm volatile("" ::"r"(depends_on_loads) : "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The same hand-back when the whole warp has read the buffer and lane 0 issues the refill:
// each lane waits for its own loads, the warp synchronises (ordering every lane's reads
// before lane 0's next instructions), and lane 0 alone fences the generic proxy against
// the async proxy that its copy writes through. Call with all lanes of the warp.
__device__ __forceinline__ void release_warp_to_async_proxy(uint32_t depends_on_loads) {
    asm volatile("" ::"r"(depends_on_loads) : "memory");
    __syncwarp();
    if ((threadIdx.x & 31) == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void report_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

// fp16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Q4_K. The 6-bit scales sc and mins m of sub-blocks 2g and 2g + 1 of a super-block
// whose 16 header bytes are hd (fp16 d | fp16 dmin << 16, then scale bytes s[0..11]), as
// two 8-bit lanes of a word: bits 0..7 for sub-block 2g, 8..15 for 2g + 1. The published
// packing: j < 4: sc_j = s[j] & 63, m_j = s[j + 4] & 63; j >= 4: sc_j = (s[j + 4] & 15) |
// (s[j - 4] >> 6) << 4, m_j = (s[j + 4] >> 4) | (s[j] >> 6) << 4. Sub-blocks 2g, 2g + 1
// take bytes 2 (g & 1) and 2 (g & 1) + 1 of each group of four scale bytes.
__device__ __forceinline__ void q4k_scales(const uint4& hd, int g, uint32_t& sc, uint32_t& m) {
    const int sh = 16 * (g & 1);
    const uint32_t a = (hd.y >> sh) & 0xFFFFu;   // s[j'] pair
    const uint32_t b = (hd.z >> sh) & 0xFFFFu;   // s[4 + j'] pair
    const uint32_t c = (hd.w >> sh) & 0xFFFFu;   // s[8 + j'] pair
    if (g < 2) {
        sc = a & 0x3F3Fu;
        m = b & 0x3F3Fu;
    } else {
        sc = (c & 0x0F0Fu) | ((a >> 2) & 0x3030u);
        m = ((c >> 4) & 0x0F0Fu) | ((b >> 2) & 0x3030u);
    }
}

}  // namespace gq
