// combine.cu -- weighted top-k reduce of expert outputs back to token order
// (ep_combine): out[t] = bf16( sum_j w[t,j] * y[slot_of[t,j]] ), fp32
// accumulation in increasing j, one rounding to bf16.
//
// Combine is the reverse of dispatch and is measured beside it in "Pipeline
// direct NVLink dispatch with triple-buffered prefetch" (DeepEP PR #693),
// Validation table.  It reads k rows per token and writes one, so it is a
// gather bound by HBM reads.  The gather is done by the TMA engine: for a
// unit (token t, slice of its row) a producer warp issues one bulk copy per
// valid slot, y[slot_of[t,j]] slice -> shared stage row j, completing on the
// stage's "full" mbarrier.  A ring of NS stages keeps up to NS units in flight
// per CTA -- far more bytes than registers could hold -- while consumer warps
// sum the k staged rows in fp32 (8 output channels per thread per step: 16
// bytes of bf16 or 8 fp8 codes in), store the bf16 result with 16-byte
// coalesced stores and hand the stage back through its "empty" mbarrier.
// Batches whose units all fit on the GPU at once take one unit per CTA
// instead (combine_unit_kernel).  No tensor cores: there is no contraction,
// only k multiply-adds per output element.
#include "ep_device.cuh"
#include "ep_kernels.h"

// Pipeline shape (compile-time; the defaults are the tuned values).
#ifndef EP_COMBINE_STAGES
#define EP_COMBINE_STAGES 3
#endif
#ifndef EP_COMBINE_STAGE_BYTES
#define EP_COMBINE_STAGE_BYTES 16384
#endif
// Units the slice size aims at, per SM (bf16 and fp8 expert outputs).
// Measured on the 128-token batches: bf16 rows of 1024 channels combine in
// 2.0 us back to back as 512 units against 2.4 us as 1024; fp8 rows of 7168
// in 5.1 us as 896 units against 5.8 us as 512.
#ifndef EP_COMBINE_UNITS_PER_SM
#define EP_COMBINE_UNITS_PER_SM 2
#endif
#ifndef EP_COMBINE_FP8_UNITS_PER_SM
#define EP_COMBINE_FP8_UNITS_PER_SM 4
#endif
#ifndef EP_COMBINE_CONSUMER_WARPS
#define EP_COMBINE_CONSUMER_WARPS 4
#endif
// Consumer warps of the ring over fp8 expert outputs (more arithmetic per
// byte: every code is widened and multiplied by its block scale).
#ifndef EP_COMBINE_FP8_CONSUMER_WARPS
#define EP_COMBINE_FP8_CONSUMER_WARPS 4
#endif
// Consumer warps of the one-unit-per-CTA kernel (decode-sized batches).
// Measured: 8 against 4 took the decode combine from 5.4-6.6 to 5.4 us back
// to back and the decode step (fused dispatch + combine) from 11.3-11.8 to
// 9.4 us; 6, 12 and 16 were slower.  The ring keeps 4 (8 there cost 3-6% on
// the large workloads).
#ifndef EP_COMBINE_UNIT_CONSUMER_WARPS
#define EP_COMBINE_UNIT_CONSUMER_WARPS 8
#endif

namespace ep {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Shared-memory layout of a ring of NS stages: 2*NS mbarriers, NS x 32
// weights, NS valid-row masks, each region rounded up to 128 bytes, then the
// stages.
__host__ __device__ constexpr uint32_t round128(uint32_t b) { return (b + 127u) / 128u * 128u; }
__host__ __device__ constexpr uint32_t weights_offset(int ns) { return round128(16u * ns); }
__host__ __device__ constexpr uint32_t mask_offset(int ns) { return weights_offset(ns) + 128u * ns; }
__host__ __device__ constexpr uint32_t scales_offset(int ns) { return round128(mask_offset(ns) + 4u * ns); }
constexpr int kMaxSliceBlocks = 16;   // fp8: 128-channel blocks per slice at most
// fp8 expert outputs also stage the block scales of every row: [NS][32][16] f32.
__host__ __device__ constexpr uint32_t stages_offset(int ns, bool fp8) {
    return fp8 ? scales_offset(ns) + 32u * kMaxSliceBlocks * 4u * ns : scales_offset(ns);
}
constexpr int kConsumerWarps = EP_COMBINE_CONSUMER_WARPS;
// the ring's consumer warps and threads per CTA, by payload
__host__ __device__ constexpr int ring_consumer_warps(bool fp8) {
    return fp8 ? EP_COMBINE_FP8_CONSUMER_WARPS : kConsumerWarps;
}
__host__ __device__ constexpr int ring_threads(bool fp8) { return 32 * (1 + ring_consumer_warps(fp8)); }
constexpr int kStages = EP_COMBINE_STAGES;
constexpr uint32_t kStageBytesMax = EP_COMBINE_STAGE_BYTES;   // k rows x slice bytes per stage
// Stage of the one-unit kernel (all k rows of one unit; no ring).  Measured
// on the 128-token batch of 7168 channels: 16 KB stages (896 units) combine
// in 4.3 us back to back, 32 KB (512 units) in 4.8-4.9 us, 64 KB (256) in 5.8.
#ifndef EP_COMBINE_UNIT_STAGE_BYTES
#define EP_COMBINE_UNIT_STAGE_BYTES EP_COMBINE_STAGE_BYTES
#endif
constexpr uint32_t kUnitStageBytesMax = EP_COMBINE_UNIT_STAGE_BYTES;

struct Args {
    const unsigned char* y;
    const float* topk_w;
    const int32_t* slot_of;
    unsigned char* out;
    uint32_t* err_flags;
    int64_t R;               // rows of y
    int64_t units;           // T * slices
    int64_t row_bytes;       // H * 2
    int slices;              // units per token row
    int k;
    uint32_t slice_bytes;    // multiple of 16 (bf16) or of 128 (fp8)
    uint32_t stage_bytes;    // k * slice_bytes (rows of one stage are slice_bytes apart)
    const void* ys;          // fp8 only: scales [R, H/128], f32 or UE8M0 bytes
    int nb;                  // H / 128
    int ue8m0;
    int slice_blocks;        // fp8: 128-channel blocks per slice
};

// e4m3 code pair (low byte first) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

// Value of a UE8M0 exponent byte: 2^(e - 127) (e = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t e) {
    return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// Two fp32 lanes in one 64-bit register (an accumulator pair).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint32_t pack_pair_bf16x2(uint64_t pair) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(pair));
    return pack_bf16x2(lo, hi);
}

// acc += w * v on each lane of a pair: an IEEE product rounded to nearest,
// then an IEEE sum rounded to nearest (__fmul_rn / __fadd_rn, which are never
// contracted).  The packed two-wide mul.rn.f32x2 + add.rn.f32x2 of sm_100
// were used first: the compiled code gave exactly the results of
// fma.rn.f32x2 (one rounding instead of two), and 7 of the tiny workload's
// 131072 outputs then differed from the definition by one bf16 ulp.
__device__ __forceinline__ uint64_t madd_pair(uint64_t acc, float w, float vlo, float vhi) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc));
    return f32x2(__fadd_rn(lo, __fmul_rn(w, vlo)), __fadd_rn(hi, __fmul_rn(w, vhi)));
}

// Both lanes of a pair multiplied, rounded to nearest (mul.rn.f32x2).  Used
// only where the product feeds another multiply or add_pair: packed multiply
// followed by a packed add was compiled into a fused multiply-add.
__device__ __forceinline__ uint64_t mul_pair(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// acc + p on each lane, as two separately rounded fp32 adds.
__device__ __forceinline__ uint64_t add_pair(uint64_t acc, uint64_t p) {
    float al, ah, pl, ph;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(al), "=f"(ah) : "l"(acc));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(pl), "=f"(ph) : "l"(p));
    return f32x2(__fadd_rn(al, pl), __fadd_rn(ah, ph));
}

// Accumulates w * (value(code) * s) for 8 fp8 codes, as 4 lane pairs: the
// two products packed two-wide, the sum per lane.
__device__ __forceinline__ void accumulate_fp8(uint64_t (&acc)[4], float w, float s, const uint2& v) {
    const uint32_t words[2] = {v.x, v.y};
    const uint64_t s2 = f32x2(s, s), w2 = f32x2(w, w);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const float2 a = e4m3x2_to_float2((uint16_t)(words[q] & 0xffffu));
        const float2 b = e4m3x2_to_float2((uint16_t)(words[q] >> 16));
        acc[2 * q] = add_pair(acc[2 * q], mul_pair(mul_pair(f32x2(a.x, a.y), s2), w2));
        acc[2 * q + 1] = add_pair(acc[2 * q + 1], mul_pair(mul_pair(f32x2(b.x, b.y), s2), w2));
    }
}

// Accumulates w * y for 8 bf16 values, as 4 lane pairs.
__device__ __forceinline__ void accumulate(uint64_t (&acc)[4], float w, const uint4& v) {
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = madd_pair(acc[q], w, bf16_lo(words[q]), bf16_hi(words[q]));
}

// Warp 0 produces (indices, weights, bulk copies into a ring of NS stages);
// warps 1..kConsumerWarps consume (sum, convert, store) and hand each stage
// back through its "empty" mbarrier, so index loads and copies of later units
// overlap the arithmetic of earlier ones.
template <int NS, bool FP8>
__global__ void __launch_bounds__(ring_threads(FP8)) combine_kernel(const Args a) {
    constexpr int kCW = ring_consumer_warps(FP8);
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);                     // [NS] data landed
    uint64_t* empty = full + NS;                                            // [NS] stage free again
    float* w_s = reinterpret_cast<float*>(smem + weights_offset(NS));       // [NS][32] weights, 0 if no row
    uint32_t* mask_s = reinterpret_cast<uint32_t*>(smem + mask_offset(NS)); // [NS] valid-row bits
    float* sc_s = reinterpret_cast<float*>(smem + scales_offset(NS));      // fp8: [NS][32][16] block scales
    unsigned char* stages = smem + stages_offset(NS, FP8);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t first = blockIdx.x;
    pdl_launch_dependents();
    if (first >= a.units) return;
    const int64_t n_mine = (a.units - 1 - first) / gridDim.x + 1;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------------ producer
        // The slot and weight of unit i+1 are loaded while unit i is issued;
        // with fp8 expert outputs the slots run two units ahead and the block
        // scales of unit i+1 are loaded (from its slot, back by then) while
        // unit i is issued, so no load latency sits between two units.
        auto load_index = [&](int64_t i, int32_t& slot, float& w) {
            const int64_t t = (first + i * gridDim.x) / a.slices;
            slot = -1;
            w = 0.f;
            if (lane < a.k) {
                slot = __ldg(a.slot_of + t * a.k + lane);
                w = a.topk_w != nullptr ? __ldg(a.topk_w + t * a.k + lane) : 1.0f;
            }
        };
        auto load_scales = [&](int64_t i, int32_t slot, float (&sc)[kMaxSliceBlocks]) {
            if (!a.ue8m0 || slot < 0 || slot >= a.R) return;   // f32 scales go by cp.async below
            const int sl = (int)((first + i * gridDim.x) % a.slices);
            const int64_t s0 = (int64_t)slot * a.nb + (int64_t)sl * a.slice_blocks;
#pragma unroll
            for (int b = 0; b < kMaxSliceBlocks; ++b) {
                if (b < a.slice_blocks) {
                    sc[b] = a.ue8m0 ? ue8m0_value(__ldg(static_cast<const uint8_t*>(a.ys) + s0 + b))
                                    : __ldg(static_cast<const float*>(a.ys) + s0 + b);
                }
            }
        };
        int32_t next_slot, next2_slot = -1;
        float next_w, next2_w = 0.f;
        float sc_cur[kMaxSliceBlocks], sc_next[kMaxSliceBlocks];
        load_index(0, next_slot, next_w);
        if (FP8) {
            if (1 < n_mine) load_index(1, next2_slot, next2_w);
            load_scales(0, next_slot, sc_next);
        }
        int64_t i = 0;
        for (; i < n_mine; ++i) {
            const int64_t u = first + i * gridDim.x;
            const int64_t t = u / a.slices;
            const int sl = (int)(u - t * a.slices);
            const int s = (int)(i % NS);
            int32_t slot = next_slot;
            float w = next_w;
            if (FP8) {
#pragma unroll
                for (int b = 0; b < kMaxSliceBlocks; ++b) sc_cur[b] = sc_next[b];
                next_slot = next2_slot;
                next_w = next2_w;
                if (i + 2 < n_mine) load_index(i + 2, next2_slot, next2_w);
                if (i + 1 < n_mine) load_scales(i + 1, next_slot, sc_next);
            } else if (i + 1 < n_mine) {
                load_index(i + 1, next_slot, next_w);
            }
            if (slot < -1 || slot >= a.R) {
                if (sl == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrBadSlot);
                slot = -1;
            }
            if (slot < 0) w = 0.f;
            const uint32_t valid = __ballot_sync(kFull, slot >= 0);
            if (i >= NS) {   // wait until the consumers released this stage's previous unit
                ok = __all_sync(kFull, mbar_wait(&empty[s], (uint32_t)(((i / NS) - 1) & 1)));
                if (!ok) break;
            }
            // The row copies need only the slots: arm the stage's byte count
            // and start them first; the weights (and fp8 scales) follow, and
            // the one arrive that completes the phase publishes them.
            if (lane == 0) mbar_expect_tx(&full[s], (uint32_t)__popc(valid) * a.slice_bytes);
            __syncwarp();
            if (slot >= 0) {
                bulk_load(stages + (size_t)s * a.stage_bytes + (size_t)lane * a.slice_bytes,
                          a.y + (int64_t)slot * a.row_bytes + (int64_t)sl * a.slice_bytes, a.slice_bytes,
                          &full[s]);
            }
            if (lane < a.k) w_s[s * 32 + lane] = w;
            if (lane == 0) mask_s[s] = valid;
            if (FP8 && slot >= 0) {
                float* dst = sc_s + (s * 32 + lane) * kMaxSliceBlocks;
                if (a.ue8m0) {
#pragma unroll
                    for (int b = 0; b < kMaxSliceBlocks; ++b) {
                        if (b < a.slice_blocks) dst[b] = sc_cur[b];
                    }
                } else {
                    // f32 scales: 4-byte asynchronous copies straight into the
                    // stage, tracked by the stage's "full" barrier (the
                    // arrive below raises its pending count until they land),
                    // so the producer never waits on them
                    const float* src = static_cast<const float*>(a.ys) + (int64_t)slot * a.nb +
                                       (int64_t)sl * a.slice_blocks;
                    for (int b = 0; b < a.slice_blocks; ++b) {
                        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst + b)), "l"(src + b)
                                     : "memory");
                    }
                    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(&full[s])) : "memory");
                }
            }
            __syncwarp();   // every lane's arrive-on above precedes lane 0's arrive
            if (lane == 0) mbar_arrive(&full[s]);
        }
        if (!ok) {
            // Copies already issued target this CTA's shared memory: let them
            // land (each wait bounded) before the CTA exits.
            if (lane == 0) {
                for (int64_t r = (i > NS ? i - NS : 0); r < i; ++r) {
                    (void)mbar_wait(&full[r % NS], (uint32_t)((r / NS) & 1));
                }
                if (a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ctid = tid - 32;
    const int chunks = (int)(a.slice_bytes / 16);
    for (int64_t i = 0; i < n_mine; ++i) {
        const int64_t u = first + i * gridDim.x;
        const int64_t t = u / a.slices;
        const int sl = (int)(u - t * a.slices);
        const int s = (int)(i % NS);
        ok = __all_sync(kFull, mbar_wait(&full[s], (uint32_t)((i / NS) & 1)));
        if (!ok) break;
        const uint32_t valid = mask_s[s];
        const unsigned char* st = stages + (size_t)s * a.stage_bytes;
        if (FP8) {
            // 8 channels per step (twice the threads of 16): 8 code bytes in,
            // 16 bf16 bytes out.  A thread takes two steps, kCW*32 apart, in
            // one pass over the rows: two independent chains of products and
            // adds to overlap (every code costs a widening and two multiplies).
            unsigned char* dst = a.out + (t * a.row_bytes + (int64_t)sl * a.slice_bytes) * 2;
            const int steps = 2 * chunks, stride = kCW * 32;
            for (int ch = ctid; ch < steps; ch += 2 * stride) {
                const int ch2 = ch + stride;
                const bool two = ch2 < steps;
                const int blk = ch / 16, blk2 = ch2 / 16;
                uint64_t acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};   // +0.0f in both lanes
                for (int j = 0; j < a.k; ++j) {
                    if (valid & (1u << j)) {
                        const unsigned char* row = st + (size_t)j * a.slice_bytes;
                        const float* scj = sc_s + (s * 32 + j) * kMaxSliceBlocks;
                        const float w = w_s[s * 32 + j];
                        const uint2 v = *reinterpret_cast<const uint2*>(row + ch * 8);
                        const uint2 v2 = two ? *reinterpret_cast<const uint2*>(row + ch2 * 8) : make_uint2(0, 0);
                        accumulate_fp8(acc, w, scj[blk], v);
                        if (two) accumulate_fp8(acc2, w, scj[blk2], v2);
                    }
                }
                uint4 o;
                o.x = pack_pair_bf16x2(acc[0]);
                o.y = pack_pair_bf16x2(acc[1]);
                o.z = pack_pair_bf16x2(acc[2]);
                o.w = pack_pair_bf16x2(acc[3]);
                *reinterpret_cast<uint4*>(dst + ch * 16) = o;
                if (two) {
                    o.x = pack_pair_bf16x2(acc2[0]);
                    o.y = pack_pair_bf16x2(acc2[1]);
                    o.z = pack_pair_bf16x2(acc2[2]);
                    o.w = pack_pair_bf16x2(acc2[3]);
                    *reinterpret_cast<uint4*>(dst + ch2 * 16) = o;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            continue;
        }
        unsigned char* dst = a.out + t * a.row_bytes + (int64_t)sl * a.slice_bytes;
        for (int ch = ctid; ch < chunks; ch += kCW * 32) {
            uint64_t acc[4] = {0, 0, 0, 0};   // +0.0f in both lanes
            for (int j = 0; j < a.k; ++j) {
                if (valid & (1u << j)) {
                    const uint4 v = *reinterpret_cast<const uint4*>(st + (size_t)j * a.slice_bytes + ch * 16);
                    const float w = w_s[s * 32 + j];
                    accumulate(acc, w, v);
                }
            }
            uint4 o;
            o.x = pack_pair_bf16x2(acc[0]);
            o.y = pack_pair_bf16x2(acc[1]);
            o.z = pack_pair_bf16x2(acc[2]);
            o.w = pack_pair_bf16x2(acc[3]);
            *reinterpret_cast<uint4*>(dst + ch * 16) = o;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok && lane == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
}

// One unit per CTA, for batches whose units all fit on the GPU at once.  Each
// row of the unit has its own "full" mbarrier: lane j of the producer warp
// issues the bulk copy of row j as soon as its own slot is back (no warp-wide
// step in between), and the consumers accumulate row j as soon as it has
// landed, in increasing j, so that the sum overlaps the later rows' arrival.
// The consumer warps read the slots (for the valid-row mask) and the weights
// themselves, so that nothing but the rows passes through the producer.  With
// fp8 expert outputs the producer lane also stages its row's block scales
// (after starting the copy) and then arrives, which publishes them with the
// row.
constexpr uint32_t kUnitBarBytes = 32u * 8u;                       // full[32]
constexpr int kUnitConsumerWarps = EP_COMBINE_UNIT_CONSUMER_WARPS;
constexpr int kUnitThreads = 32 * (1 + kUnitConsumerWarps);
constexpr uint32_t kUnitWOffset = kUnitBarBytes;                   // [kUnitConsumerWarps][32] weights
constexpr uint32_t kUnitScaleOffset = round128(kUnitWOffset + 128u * kUnitConsumerWarps);   // fp8: [32][16] f32
__host__ __device__ constexpr uint32_t unit_stage_offset(bool fp8) {
    return fp8 ? round128(kUnitScaleOffset + 32u * kMaxSliceBlocks * 4u) : kUnitScaleOffset;
}

// As many CTAs per SM as the threads allow (7 of 288 threads): a decode-sized
// batch needs every unit resident at once (896 units, 5.9 per SM), and at 40
// registers a thread only 5 CTAs fit, which sends the batch to the ring
// (measured 7.4 against 4.3 us back to back).
template <bool FP8>
__global__ void __launch_bounds__(kUnitThreads, 2048 / kUnitThreads) combine_unit_kernel(const Args a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    float* w_s = reinterpret_cast<float*>(smem + kUnitWOffset);
    float* sc_s = reinterpret_cast<float*>(smem + kUnitScaleOffset);
    unsigned char* stage = smem + unit_stage_offset(FP8);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t u = blockIdx.x;
    const int64_t t = u / a.slices;
    const int sl = (int)(u - t * a.slices);
    pdl_launch_dependents();
    if (tid == 0) {
        for (int j = 0; j < a.k; ++j) mbar_init(&full[j], 1);
        fence_mbar_init();
        // Before the wait on the previous kernel: pull this token's slots and
        // weights towards L2 (no effect on what the loads after the wait
        // return; the L2 is the point of coherence).
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.slot_of + t * a.k) : "memory");
        if (a.topk_w != nullptr) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.topk_w + t * a.k) : "memory");
    }
    __syncthreads();
    if (warp == 1 && lane < a.k) {
        // Still before the wait: pull this unit's row slices towards L2, at
        // the slots as they read now.  Only an address hint (checked to lie
        // inside y): if the previous kernel rewrites the slots or y, the loads
        // after the wait still read the new values, and the prefetch is
        // wasted.  Relaxed gpu-scope loads keep the hint out of L1.
        int32_t s;
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(s) : "l"(a.slot_of + t * a.k + lane) : "memory");
        if (s >= 0 && s < a.R)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                         ::"l"(a.y + (int64_t)s * a.row_bytes + (int64_t)sl * a.slice_bytes), "r"(a.slice_bytes)
                         : "memory");
    }
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane < a.k) {
            const int32_t slot = __ldg(a.slot_of + t * a.k + lane);
            if (slot >= 0 && slot < a.R) {
                unsigned char* dst = stage + (size_t)lane * a.slice_bytes;
                const unsigned char* src = a.y + (int64_t)slot * a.row_bytes + (int64_t)sl * a.slice_bytes;
                if (FP8) {
                    mbar_expect_tx(&full[lane], a.slice_bytes);
                    bulk_load(dst, src, a.slice_bytes, &full[lane]);
                    const int64_t s0 = (int64_t)slot * a.nb + (int64_t)sl * a.slice_blocks;
                    float* sd = sc_s + lane * kMaxSliceBlocks;
                    for (int b = 0; b < a.slice_blocks; ++b) {
                        sd[b] = a.ue8m0 ? ue8m0_value(__ldg(static_cast<const uint8_t*>(a.ys) + s0 + b))
                                        : __ldg(static_cast<const float*>(a.ys) + s0 + b);
                    }
                    mbar_arrive(&full[lane]);   // publishes the scales; the phase ends once the row has landed too
                } else {
                    mbar_arrive_expect_tx(&full[lane], a.slice_bytes);
                    bulk_load(dst, src, a.slice_bytes, &full[lane]);
                }
                // the copy targets this CTA's shared memory: stay until it
                // has landed (bounded), whatever the consumers do
                (void)mbar_wait(&full[lane], 0);
            } else if (slot != -1 && sl == 0 && a.err_flags != nullptr) {
                atomicOr(a.err_flags, kErrBadSlot);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1;
    bool valid = false;
    if (lane < a.k) {
        const int32_t slot = __ldg(a.slot_of + t * a.k + lane);
        valid = slot >= 0 && slot < a.R;
        const float w = a.topk_w != nullptr ? __ldg(a.topk_w + t * a.k + lane) : 1.0f;
        w_s[cw * 32 + lane] = valid ? w : 0.f;
    }
    const uint32_t vmask = __ballot_sync(kFull, valid);
    __syncwarp();
    const int ctid = tid - 32;
    const int chunks = (int)(a.slice_bytes / 16);
    // fp8: steps of 8 codes (8 code bytes in, 16 bf16 bytes out), twice as
    // many as the 16-byte steps of bf16
    const int steps = FP8 ? 2 * chunks : chunks;
    for (int ch = ctid; ch < steps; ch += kUnitConsumerWarps * 32) {
        if (FP8) {
            const int blk = ch / 16;
            uint64_t acc[4] = {0, 0, 0, 0};   // +0.0f in both lanes
            for (int j = 0; j < a.k; ++j) {
                if (!((vmask >> j) & 1u)) continue;
                if (!mbar_wait(&full[j], 0)) {
                    if (a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
                    return;
                }
                const uint2 v = *reinterpret_cast<const uint2*>(stage + (size_t)j * a.slice_bytes + ch * 8);
                accumulate_fp8(acc, w_s[cw * 32 + j], sc_s[j * kMaxSliceBlocks + blk], v);
            }
            unsigned char* dst = a.out + (t * a.row_bytes + (int64_t)sl * a.slice_bytes) * 2 + ch * 16;
            uint4 o;
            o.x = pack_pair_bf16x2(acc[0]);
            o.y = pack_pair_bf16x2(acc[1]);
            o.z = pack_pair_bf16x2(acc[2]);
            o.w = pack_pair_bf16x2(acc[3]);
            *reinterpret_cast<uint4*>(dst) = o;
        } else {
            uint64_t acc[4] = {0, 0, 0, 0};   // +0.0f in both lanes
            for (int j = 0; j < a.k; ++j) {
                if (!((vmask >> j) & 1u)) continue;
                if (!mbar_wait(&full[j], 0)) {
                    if (a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
                    return;
                }
                const uint4 v = *reinterpret_cast<const uint4*>(stage + (size_t)j * a.slice_bytes + ch * 16);
                accumulate(acc, w_s[cw * 32 + j], v);
            }
            unsigned char* dst = a.out + t * a.row_bytes + (int64_t)sl * a.slice_bytes + ch * 16;
            uint4 o;
            o.x = pack_pair_bf16x2(acc[0]);
            o.y = pack_pair_bf16x2(acc[1]);
            o.z = pack_pair_bf16x2(acc[2]);
            o.w = pack_pair_bf16x2(acc[3]);
            *reinterpret_cast<uint4*>(dst) = o;
        }
    }
}

// Number of slices a row of n granules is cut into: the smallest divisor d of
// n whose slices hold at most max_per granules and give T*d >= want units;
// slices never drop below min_per granules once one size fits.
int pick_slices(int64_t T, int64_t n, int64_t max_per, int64_t min_per, int64_t want) {
    int best = 0;
    for (int64_t d = 1; d <= n; ++d) {
        if (n % d) continue;
        const int64_t per = n / d;
        if (per > max_per) continue;
        if (best && per < min_per) break;
        best = (int)d;
        if (T * d >= want) break;
    }
    return best ? best : (int)n;
}


// Cuts each row into slices for stages of at most stage_max bytes (k rows):
// the fewest slices that give about units_per_sm units per SM.
void set_slices(Args& a, const CombineParams& p, int num_sms, uint32_t stage_max) {
    if (p.fp8) {
        // whole 128-channel blocks (their scales are staged too), at most
        // kMaxSliceBlocks of them
        int64_t max_blocks = (int64_t)(stage_max / 128) / p.k;
        if (max_blocks > kMaxSliceBlocks) max_blocks = kMaxSliceBlocks;
        a.slices = pick_slices(p.T, a.nb, max_blocks > 0 ? max_blocks : 1, 1,
                               (int64_t)EP_COMBINE_FP8_UNITS_PER_SM * num_sms);
        a.slice_blocks = a.nb / a.slices;
        a.slice_bytes = (uint32_t)a.slice_blocks * 128u;
    } else {
        // 16-byte granules, at least 256 bytes a slice once one size fits
        const int64_t vec16 = a.row_bytes / 16;
        const int64_t max_per = (int64_t)(stage_max / 16) / p.k;
        a.slices = pick_slices(p.T, vec16, max_per > 0 ? max_per : 1, 16, (int64_t)EP_COMBINE_UNITS_PER_SM * num_sms);
        a.slice_bytes = (uint32_t)(a.row_bytes / a.slices);
    }
    a.stage_bytes = a.slice_bytes * (uint32_t)p.k;
    a.units = (int64_t)p.T * a.slices;
}

// If one CTA per unit fits on the GPU at once (small batches), launches
// exactly that (combine_unit_kernel): every unit starts immediately.
// Otherwise a persistent grid of kStages-deep rings, over slices cut for the
// ring's stage size.
template <bool FP8>
cudaError_t launch_combine_t(Args& a, const CombineParams& p, int num_sms, cudaStream_t stream) {
    set_slices(a, p, num_sms, kUnitStageBytesMax);
    size_t smem = unit_stage_offset(FP8) + (size_t)a.stage_bytes;
    cudaError_t err = cudaFuncSetAttribute(combine_unit_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_unit_kernel<FP8>, kUnitThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm >= 1 && a.units <= (int64_t)num_sms * per_sm) {
        return launch_kernel(true, combine_unit_kernel<FP8>, dim3((unsigned)a.units), dim3(kUnitThreads), smem, stream,
                             a);
    }
    set_slices(a, p, num_sms, kStageBytesMax);
    smem = stages_offset(kStages, FP8) + (size_t)kStages * a.stage_bytes;
    err = cudaFuncSetAttribute(combine_kernel<kStages, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<kStages, FP8>, ring_threads(FP8), smem);
    if (err != cudaSuccess) return err;
    const int64_t ctas = (int64_t)num_sms * (per_sm < 1 ? 1 : per_sm);
    const int64_t grid = ctas < a.units ? ctas : a.units;
    return launch_kernel(false, combine_kernel<kStages, FP8>, dim3((unsigned)grid), dim3(ring_threads(FP8)), smem,
                         stream, a);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int num_sms, cudaStream_t stream) {
    if (p.T == 0) return cudaSuccess;
    Args a{};
    a.y = static_cast<const unsigned char*>(p.y);
    a.topk_w = p.topk_w;
    a.slot_of = p.slot_of;
    a.out = static_cast<unsigned char*>(p.out);
    a.err_flags = p.err_flags;
    a.R = p.R;
    a.k = p.k;
    a.nb = p.H / 128;
    if (p.fp8) {
        a.ys = p.y_scales;
        a.ue8m0 = p.ue8m0;
        a.row_bytes = p.H;
        return launch_combine_t<true>(a, p, num_sms, stream);
    }
    a.row_bytes = (int64_t)p.H * 2;
    return launch_combine_t<false>(a, p, num_sms, stream);
}

}  // namespace ep
