// ep_device.cuh -- device helpers shared by the dispatch / combine kernels:
// inline-PTX wrappers for mbarriers and bulk asynchronous copies (the TMA
// engine's non-tensor form), bf16 bit handling and a bounded wait.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ep {

// Bits of the caller's device error word (same values as EP_ERRF_* in ep.h).
constexpr uint32_t kErrBadExpert = 1u;
constexpr uint32_t kErrCapacity = 2u;
constexpr uint32_t kErrTimeout = 4u;
constexpr uint32_t kErrBadSlot = 8u;

// Upper bound on any single wait inside a kernel.  A correct run waits
// microseconds; reaching this sets kErrTimeout and the kernel returns.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Raises the bytes the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete, at most kWaitLimitNs.
// Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// ------------------------------------------------------ bulk async copies

// global -> shared, completion counted in bytes on `bar`.
// Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's committed groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------ programmatic dependent launch

// Lets the next kernel of the stream (launched with programmatic stream
// serialization) start its prologue once every CTA of this grid got here.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the previous grid of the stream has completed and its memory
// is visible.  Returns at once when there is no such grid.  Every global
// read or write that may touch that grid's data comes after this.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------- bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// x / d rounded to nearest even, from rd = RN32(1 / d): q0 = RN(x * rd), the
// residual r = x - q0 * d (exact, one fused multiply-add), then RN(q0 + r * rd).
// This is Markstein's quotient correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Develop. 34(1), 1990): with rd the correctly rounded reciprocal and q0 within
// one ulp of x / d, the corrected quotient is the correctly rounded one as long
// as nothing underflows.  It is used only with d a block scale (a normal number
// in [2^-23, 2^120]) or 448, and x a bf16 value no larger in magnitude than
// the amax the scale came from: there the scale and every e4m3 code equal
// those of the IEEE quotient, for every bf16 amax and every such x (checked
// exhaustively against __fdiv_rn on the GPU, and the method against C's
// division on the CPU).  The sign comes from x, so that -0 stays -0.
__device__ __forceinline__ float quotient_rn(float x, float d, float rd) {
    const float q0 = __fmul_rn(x, rd);
    const float r = __fmaf_rn(-q0, d, x);
    return copysignf(__fmaf_rn(r, rd, q0), x);
}

// RN32(1 / 448), the reciprocal block_scale works with.
__device__ __forceinline__ float recip_448() { return __frcp_rn(448.0f); }

// Scale of a 128-channel block: v = RN32(max(amax, 1e-4) / 448); with UE8M0
// scales, the smallest power of two >= v (exact: bump the exponent unless the
// mantissa is zero; v is a positive normal number here).  r448 = recip_448().
__device__ __forceinline__ float block_scale(float amax, bool ue8m0, float r448) {
    float v = quotient_rn(fmaxf(amax, 1e-4f), 448.0f, r448);
    if (ue8m0) {
        uint32_t b = __float_as_uint(v);
        if (b & 0x007fffffu) b = (b & 0x7f800000u) + 0x00800000u;
        v = __uint_as_float(b);
    }
    return v;
}

// Biased exponent byte of a power-of-two scale (UE8M0: value 2^(e - 127)).
__device__ __forceinline__ uint8_t ue8m0_byte(float pow2) { return (uint8_t)(__float_as_uint(pow2) >> 23); }

// Two floats -> packed e4m3x2 (round to nearest even, saturate to +-448),
// `lo` in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Quantises up to four 128-channel blocks per warp, eight lanes per block:
// lanes 8g..8g+7 take block b0 + g (if below b_end), 16 consecutive bf16
// channels each from in_st + block * 256, find the block's amax in three
// shuffles within the eight lanes, and write their 16 e4m3 codes to
// code_st + block * 128.  Every lane of the warp must call it (the shuffles).
// Returns the block's scale in .sc; .first is set on the lane that should
// store it (lane 8g, live block), .b is the block.
struct BlockScale {
    float sc;
    int b;
    bool first;
};

__device__ __forceinline__ BlockScale quantize_blocks_8lanes(const unsigned char* in_st, unsigned char* code_st, int b0,
                                                            int b_end, bool ue8m0, float r448) {
    const int lane = threadIdx.x & 31;
    const int b = b0 + (lane >> 3), sub = lane & 7;
    const bool live = b < b_end;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
    if (live) {
        v0 = *reinterpret_cast<const uint4*>(in_st + b * 256 + sub * 32);
        v1 = *reinterpret_cast<const uint4*>(in_st + b * 256 + sub * 32 + 16);
    }
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float xv[16];
    float m = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        xv[2 * q] = bf16_lo(wv[q]);
        xv[2 * q + 1] = bf16_hi(wv[q]);
        m = fmaxf(m, fmaxf(fabsf(xv[2 * q]), fabsf(xv[2 * q + 1])));
    }
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    const float sc = block_scale(m, ue8m0, r448);
    const float rs = __frcp_rn(sc);
    uint32_t code[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo = pack_e4m3x2(quotient_rn(xv[4 * q], sc, rs), quotient_rn(xv[4 * q + 1], sc, rs));
        const uint32_t hi = pack_e4m3x2(quotient_rn(xv[4 * q + 2], sc, rs), quotient_rn(xv[4 * q + 3], sc, rs));
        code[q] = lo | (hi << 16);
    }
    if (live) *reinterpret_cast<uint4*>(code_st + b * 128 + sub * 16) = make_uint4(code[0], code[1], code[2], code[3]);
    return BlockScale{sc, b, live && sub == 0};
}

}  // namespace ep
