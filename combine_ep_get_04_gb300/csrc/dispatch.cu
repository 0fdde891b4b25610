// dispatch.cu -- copy each token's hidden row to every receive row it is
// routed to (ep_dispatch), as a bf16 bit copy or with a fused per-128-channel
// amax / FP8 e4m3 cast.
//
// Prior art: "Pipeline direct NVLink dispatch with triple-buffered prefetch"
// (DeepEP PR #693), Summary: each dispatch warp stages tokens through shared
// memory with the TMA engine; three buffers hold the token whose stores are
// still in flight, the token being sent and the token being prefetched, and
// the oldest buffer is recycled once at most one store group is outstanding.
// Here the destination is this GPU's own HBM, so the same pipeline becomes:
//   bulk copy global->shared of the next unit (mbarrier completion) while the
//   k bulk copies shared->global of earlier units drain (bulk groups).
// A unit is a token row, or a slice of it when there are few tokens, so the
// grid covers every SM.  When there are more units than one resident wave of
// CTAs, each CTA takes one unit (bf16) or six (fp8) and the overlap of loads
// and stores comes from the several CTAs resident on each SM; the ring inside
// a CTA serves the CTAs that take several units.  Each row of x is read from
// HBM once and written k times; no thread touches the payload on the bf16
// path.
#include "ep_device.cuh"
#include "ep_kernels.h"
#include "ring_schedule.h"

// Units each CTA takes when there are more units than one resident wave of
// CTAs holds (0: a persistent grid of one wave, every CTA looping over an
// equal share).  The SMs do not get equal shares of memory bandwidth (per-CTA
// end times of one persistent bf16 dispatch ranged from 50 to 83 us on the
// prefill workload and from 81 to 201 us on the group-limited one, by SM), so
// a persistent grid ends on its slowest SMs; a grid of short CTAs lets the
// block scheduler give more of them to the SMs that free up first.  Tuned:
// bf16 one unit per CTA (prefill 88.5 -> 80.3 us, group-limited 202 -> 179
// us), fp8 six (its CTAs of fourteen warps cost more to start; skewed 98.8 ->
// 96.8 us with eight quantiser warps).
#ifndef EP_BF16_UNITS_PER_CTA
#define EP_BF16_UNITS_PER_CTA 1
#endif
#ifndef EP_FP8_UNITS_PER_CTA
#define EP_FP8_UNITS_PER_CTA 6
#endif

// Pipeline shape (compile-time; the defaults are the tuned values).
#ifndef EP_BF16_STAGES
#define EP_BF16_STAGES 4
#endif
#ifndef EP_BF16_LOOKAHEAD
#define EP_BF16_LOOKAHEAD 2
#endif
#ifndef EP_BF16_SLICE_GRANULES
#define EP_BF16_SLICE_GRANULES 1024   // 16-byte granules per bf16 unit at most
#endif
#ifndef EP_FP8_STAGES
#define EP_FP8_STAGES 4
#endif
#ifndef EP_FP8_OUT_STAGES
#define EP_FP8_OUT_STAGES 3
#endif
#ifndef EP_FP8_QUANT_WARPS
#define EP_FP8_QUANT_WARPS 12
#endif
#ifndef EP_FP8_SLICE_BLOCKS
#define EP_FP8_SLICE_BLOCKS 64        // 128-channel blocks per fp8 unit at most
#endif

namespace ep {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Shared-memory header holding a kernel's mbarriers (8 bytes each), rounded
// up to 128 bytes so that the stages after it stay 128-byte aligned.
__host__ __device__ constexpr uint32_t header_bytes(int n_barriers) { return (uint32_t)((n_barriers * 8 + 127) / 128 * 128); }

struct Bf16Args {
    const unsigned char* x;
    const int32_t* slot_of;
    const float* topk_w;
    unsigned char* recv;
    float* recv_w;
    uint32_t* err_flags;
    int64_t R;             // receive rows
    int64_t units;         // T * slices
    int64_t row_bytes;     // H * 2
    int slices;            // units per token row
    int k;
    uint32_t slice_bytes;  // row_bytes / slices, multiple of 16
    uint32_t stage_stride; // slice_bytes rounded up to 128
};

// One warp per CTA.  Lane 0 issues the loads; lane j issues the store of copy j.
template <int NS, int LA>
__global__ void __launch_bounds__(32) dispatch_bf16_kernel(const Bf16Args a) {
    static_assert(LA >= 1 && LA <= NS - 1, "lookahead must leave a stage for the stores");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* stages = smem + header_bytes(NS);
    const int lane = threadIdx.x;
    const int64_t first = blockIdx.x;
    pdl_launch_dependents();
    if (first >= a.units) return;
    const int64_t n_mine = (a.units - 1 - first) / gridDim.x + 1;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        // Before the wait on the previous kernel (the layout, which x does
        // not depend on): pull the slices of x the first loads will read
        // towards L2, so that their DRAM latency overlaps that kernel.  A
        // prefetch changes nothing the loads after the wait return (the L2
        // is the point of coherence).  Measured: layout + dispatch 1.1-1.3 us
        // shorter back to back on the prefill and group-limited workloads.
        for (int64_t i = 0; i < ring_prologue_loads(n_mine, LA); ++i) {
            const int64_t u = first + i * gridDim.x;
            const int64_t t = u / a.slices;
            const int sl = (int)(u - t * a.slices);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.x + t * a.row_bytes +
                                                                           (int64_t)sl * a.slice_bytes),
                         "r"(a.slice_bytes)
                         : "memory");
        }
    }
    __syncwarp();
    pdl_wait();

    auto issue_load = [&](int64_t i) {
        const int64_t u = first + i * gridDim.x;
        const int64_t t = u / a.slices;
        const int sl = (int)(u - t * a.slices);
        const int s = (int)(i % NS);
        mbar_arrive_expect_tx(&bars[s], a.slice_bytes);
        bulk_load(stages + (size_t)s * a.stage_stride,
                  a.x + t * a.row_bytes + (int64_t)sl * a.slice_bytes, a.slice_bytes, &bars[s]);
    };

    if (lane == 0) {
        for (int64_t i = 0; i < ring_prologue_loads(n_mine, LA); ++i) issue_load(i);
    }

    // Lane j holds the slot (and weight) of copy j of the next unit, loaded
    // one unit ahead.
    auto load_index = [&](int64_t i, int32_t& slot, float& w) {
        const int64_t t = (first + i * gridDim.x) / a.slices;
        slot = -1;
        w = 0.f;
        if (lane < a.k) {
            slot = __ldg(a.slot_of + t * a.k + lane);
            if (a.recv_w != nullptr) w = __ldg(a.topk_w + t * a.k + lane);
        }
    };
    int32_t next_slot;
    float next_w;
    load_index(0, next_slot, next_w);

    bool ok = true;
    int64_t i = 0;
    for (; i < n_mine; ++i) {
        const int64_t u = first + i * gridDim.x;
        const int64_t t = u / a.slices;
        const int sl = (int)(u - t * a.slices);
        const int s = (int)(i % NS);
        // Stage (i+LA)%NS was last read by the stores of unit i+LA-NS; at most
        // NS-LA-1 younger store groups may still be reading their stages.
        if (ring_issues_ahead(i, n_mine, LA)) {
            bulk_wait_read<NS - LA - 1>();
            __syncwarp();
            if (lane == 0) issue_load(i + LA);
        }
        int32_t slot = next_slot;
        const float w = next_w;
        if (i + 1 < n_mine) load_index(i + 1, next_slot, next_w);
        if (slot < -1 || slot >= a.R) {
            if (sl == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrBadSlot);
            slot = -1;
        }
        ok = __all_sync(kFull, mbar_wait(&bars[s], (uint32_t)((i / NS) & 1)));
        if (!ok) break;
        if (slot >= 0) {
            bulk_store(a.recv + (int64_t)slot * a.row_bytes + (int64_t)sl * a.slice_bytes,
                       stages + (size_t)s * a.stage_stride, a.slice_bytes);
            if (a.recv_w != nullptr && sl == 0) a.recv_w[slot] = w;
        }
        bulk_commit();
    }
    bulk_wait_all();
    if (!ok) {
        // Loads still in flight target this CTA's shared memory: those of
        // units i .. i+LA (unit i+LA was issued before the wait on unit i gave
        // up).  Let them land (each wait bounded) before the CTA exits.
        if (lane == 0) {
            for (int64_t r = i; r < ring_issued_end(i, n_mine, LA); ++r) {
                (void)mbar_wait(&bars[r % NS], (uint32_t)((r / NS) & 1));
            }
            if (a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
        }
    }
}

struct Fp8Args {
    const unsigned char* x;
    const int32_t* slot_of;
    const float* topk_w;
    unsigned char* recv;     // e4m3 [R, H]
    void* recv_s;            // [R, H/128] f32, or u8 exponents with ue8m0
    float* recv_w;
    uint32_t* err_flags;
    int64_t R;               // receive rows
    int64_t units;           // T * slices
    int H;
    int nb;                  // H / 128
    int slices;
    int nblk;                // 128-channel blocks per unit
    int k;
    int scale_bulk;          // scales stored with a bulk copy (16-byte granular)
    int ue8m0;               // power-of-two scales, stored as exponent bytes
    uint32_t in_stride;      // bytes per input stage (nblk*256, multiple of 128)
    uint32_t out_stride;     // bytes per output stage: nblk*128 q + nblk*4 scales, rounded to 128
};

constexpr int kFp8QuantWarps = EP_FP8_QUANT_WARPS;
constexpr int kFp8Threads = (2 + kFp8QuantWarps) * 32;   // producer, storer, quantisers
constexpr int kFp8OutStages = EP_FP8_OUT_STAGES;

// Warp-specialised: warp 0 (lane 0) fills a ring of NS input stages with bulk
// copies of x; warps 2.. quantise a unit from its input stage into one of NSO
// output stages (codes, then scales) and arrive on that stage's "full"
// barrier; warp 1 issues the k bulk stores of each finished output stage (lane
// j: copy j) and hands a stage back once its stores have read it.  No
// block-wide barrier inside the loop.
template <int NS, int NSO>
__global__ void __launch_bounds__(kFp8Threads) dispatch_fp8_kernel(const Fp8Args a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* in_full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* in_empty = in_full + NS;
    uint64_t* out_full = in_empty + NS;
    uint64_t* out_empty = out_full + NSO;
    unsigned char* in_st = smem + header_bytes(2 * NS + 2 * NSO);
    unsigned char* out_st = in_st + (size_t)NS * a.in_stride;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t first = blockIdx.x;
    pdl_launch_dependents();
    if (first >= a.units) return;
    const int64_t n_mine = (a.units - 1 - first) / gridDim.x + 1;
    const uint32_t in_bytes = (uint32_t)a.nblk * 256u;
    const uint32_t q_bytes = (uint32_t)a.nblk * 128u;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            mbar_init(&in_full[s], 1);
            mbar_init(&in_empty[s], kFp8QuantWarps);
        }
#pragma unroll
        for (int o = 0; o < NSO; ++o) {
            mbar_init(&out_full[o], kFp8QuantWarps);
            mbar_init(&out_empty[o], 1);
        }
        fence_mbar_init();
        // Before the wait on the previous kernel (the layout, which x does
        // not depend on): pull the x slices of this CTA's first units
        // towards L2.  A prefetch changes nothing the loads after the wait
        // return (the L2 is the point of coherence).
        for (int64_t i = 0; i < n_mine && i < NS; ++i) {
            const int64_t u = first + i * gridDim.x;
            const int64_t t = u / a.slices;
            const int sl = (int)(u - t * a.slices);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.x + (t * a.H + (int64_t)sl * a.nblk * 128) * 2),
                         "r"(in_bytes)
                         : "memory");
        }
    }
    __syncthreads();
    pdl_wait();

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            int64_t i = 0;
            for (; i < n_mine; ++i) {
                const int s = (int)(i % NS);
                if (i >= NS && !mbar_wait(&in_empty[s], (uint32_t)(((i / NS) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const int64_t u = first + i * gridDim.x;
                const int64_t t = u / a.slices;
                const int sl = (int)(u - t * a.slices);
                mbar_arrive_expect_tx(&in_full[s], in_bytes);
                bulk_load(in_st + (size_t)s * a.in_stride, a.x + (t * a.H + (int64_t)sl * a.nblk * 128) * 2,
                          in_bytes, &in_full[s]);
            }
            if (!ok) {
                // copies already issued target this CTA's shared memory: let
                // them land (each wait bounded) before the CTA exits
                for (int64_t r = (i > NS ? i - NS : 0); r < i; ++r) {
                    (void)mbar_wait(&in_full[r % NS], (uint32_t)((r / NS) & 1));
                }
                if (a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
            }
        }
        return;
    }

    if (warp == 1) {
        // -------------------------------------------------------- storer
        // Lane j holds the slot (and weight) of copy j, loaded one unit ahead.
        auto load_index = [&](int64_t i, int32_t& slot, float& w) {
            const int64_t t = (first + i * gridDim.x) / a.slices;
            slot = -1;
            w = 0.f;
            if (lane < a.k) {
                slot = __ldg(a.slot_of + t * a.k + lane);
                if (a.recv_w != nullptr) w = __ldg(a.topk_w + t * a.k + lane);
            }
        };
        int32_t next_slot;
        float next_w;
        load_index(0, next_slot, next_w);
        for (int64_t i = 0; i < n_mine; ++i) {
            const int o = (int)(i % NSO);
            const int64_t u = first + i * gridDim.x;
            const int64_t t = u / a.slices;
            const int sl = (int)(u - t * a.slices);
            int32_t slot = next_slot;
            const float w = next_w;
            if (i + 1 < n_mine) load_index(i + 1, next_slot, next_w);
            if (slot < -1 || slot >= a.R) {
                if (sl == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrBadSlot);
                slot = -1;
            }
            ok = __all_sync(kFull, mbar_wait(&out_full[o], (uint32_t)((i / NSO) & 1)));
            if (!ok) break;
            const unsigned char* ob = out_st + (size_t)o * a.out_stride;
            const float* oscale = reinterpret_cast<const float*>(ob + q_bytes);
            if (slot >= 0) {
                bulk_store(a.recv + (int64_t)slot * a.H + (int64_t)sl * a.nblk * 128, ob, q_bytes);
                const int64_t s0 = (int64_t)slot * a.nb + (int64_t)sl * a.nblk;
                if (a.ue8m0) {
                    uint8_t* edst = static_cast<uint8_t*>(a.recv_s) + s0;
                    for (int b = 0; b < a.nblk; ++b) edst[b] = ob[q_bytes + b];
                } else if (a.scale_bulk) {
                    bulk_store(static_cast<float*>(a.recv_s) + s0, oscale, (uint32_t)a.nblk * 4u);
                } else {
                    float* sdst = static_cast<float*>(a.recv_s) + s0;
                    for (int b = 0; b < a.nblk; ++b) sdst[b] = oscale[b];
                }
                if (a.recv_w != nullptr && sl == 0) a.recv_w[slot] = w;
            }
            bulk_commit();
            if (i >= 1) {   // the stores of unit i-1 have read their stage: hand it back
                bulk_wait_read<1>();
                __syncwarp();
                if (lane == 0) mbar_arrive(&out_empty[(i - 1) % NSO]);
            }
        }
        bulk_wait_all();
        if (!ok && lane == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
        return;
    }

    // ------------------------------------------------------------ quantisers
    const int qw = warp - 2;
    const float r448 = recip_448();
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = (int)(i % NS);
        const int o = (int)(i % NSO);
        ok = __all_sync(kFull, mbar_wait(&in_full[s], (uint32_t)((i / NS) & 1)));
        if (ok && i >= NSO) ok = __all_sync(kFull, mbar_wait(&out_empty[o], (uint32_t)(((i / NSO) - 1) & 1)));
        if (!ok) break;
        const unsigned char* ib = in_st + (size_t)s * a.in_stride;
        unsigned char* ob = out_st + (size_t)o * a.out_stride;
        float* oscale = reinterpret_cast<float*>(ob + q_bytes);
        // four blocks per warp, eight lanes per block
        for (int b0 = qw * 4; b0 < a.nblk; b0 += 4 * kFp8QuantWarps) {
            const BlockScale r = quantize_blocks_8lanes(ib, ob, b0, a.nblk, a.ue8m0 != 0, r448);
            if (r.first) {
                if (a.ue8m0) {
                    ob[q_bytes + r.b] = ue8m0_byte(r.sc);
                } else {
                    oscale[r.b] = r.sc;
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&in_empty[s]);
            mbar_arrive(&out_full[o]);
        }
    }
    if (!ok && lane == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
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

}  // namespace

constexpr int kBf16Stages = EP_BF16_STAGES;
constexpr int kBf16Lookahead = EP_BF16_LOOKAHEAD;
constexpr int kFp8Stages = EP_FP8_STAGES;

cudaError_t launch_dispatch_bf16(const DispatchParams& p, int num_sms, cudaStream_t stream) {
    if (p.T == 0) return cudaSuccess;
    Bf16Args a{};
    a.x = static_cast<const unsigned char*>(p.x);
    a.slot_of = p.slot_of;
    a.topk_w = p.topk_w;
    a.recv = static_cast<unsigned char*>(p.recv);
    a.recv_w = p.recv_w;
    a.err_flags = p.err_flags;
    a.R = p.R;
    a.row_bytes = (int64_t)p.H * 2;
    a.k = p.k;
    // Units of at most 16 KB, at least 1 KB, enough of them for ~4 per SM.
    const int64_t vec16 = a.row_bytes / 16;
    a.slices = pick_slices(p.T, vec16, EP_BF16_SLICE_GRANULES, 64, 4LL * num_sms);
    a.slice_bytes = (uint32_t)(a.row_bytes / a.slices);
    a.stage_stride = (a.slice_bytes + 127u) & ~127u;
    a.units = (int64_t)p.T * a.slices;
    const size_t smem = header_bytes(kBf16Stages) + (size_t)kBf16Stages * a.stage_stride;
    auto kern = dispatch_bf16_kernel<kBf16Stages, kBf16Lookahead>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)num_sms * per_sm;
    if (grid > a.units) grid = a.units;
    if (EP_BF16_UNITS_PER_CTA > 0) {
        const int64_t upc = EP_BF16_UNITS_PER_CTA > 0 ? EP_BF16_UNITS_PER_CTA : 1;
        const int64_t g2 = (a.units + upc - 1) / upc;
        if (g2 > grid) grid = g2;
    }
    return launch_kernel(grid >= a.units, kern, dim3((unsigned)grid), dim3(32), smem, stream, a);
}

cudaError_t launch_dispatch_fp8(const DispatchParams& p, int num_sms, cudaStream_t stream) {
    if (p.T == 0) return cudaSuccess;
    Fp8Args a{};
    a.x = static_cast<const unsigned char*>(p.x);
    a.slot_of = p.slot_of;
    a.topk_w = p.topk_w;
    a.recv = static_cast<unsigned char*>(p.recv);
    a.recv_s = p.recv_scales;
    a.ue8m0 = p.ue8m0;
    a.recv_w = p.recv_w;
    a.err_flags = p.err_flags;
    a.R = p.R;
    a.H = p.H;
    a.nb = p.H / 128;
    a.k = p.k;
    // Units of at most 64 blocks (16 KB of bf16), enough for ~4 per SM.
    a.slices = pick_slices(p.T, a.nb, EP_FP8_SLICE_BLOCKS, 2, 4LL * num_sms);
    a.nblk = a.nb / a.slices;
    a.scale_bulk = (a.nb % 4 == 0) && (a.nblk % 4 == 0);
    a.in_stride = (uint32_t)a.nblk * 256u;
    a.out_stride = ((uint32_t)a.nblk * 132u + 127u) & ~127u;
    a.units = (int64_t)p.T * a.slices;
    const size_t smem = header_bytes(2 * kFp8Stages + 2 * kFp8OutStages) + (size_t)kFp8Stages * a.in_stride +
                        (size_t)kFp8OutStages * a.out_stride;
    auto kern = dispatch_fp8_kernel<kFp8Stages, kFp8OutStages>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFp8Threads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)num_sms * per_sm;
    if (grid > a.units) grid = a.units;
    if (EP_FP8_UNITS_PER_CTA > 0) {
        const int64_t upc = EP_FP8_UNITS_PER_CTA > 0 ? EP_FP8_UNITS_PER_CTA : 1;
        const int64_t g2 = (a.units + upc - 1) / upc;
        if (g2 > grid) grid = g2;
    }
    // Programmatic serialization even for the persistent grid: its CTAs
    // start (and prefetch x) while the layout finishes.  Measured on the
    // skewed workload: layout + dispatch 2 us shorter back to back.
    return launch_kernel(true, kern, dim3((unsigned)grid), dim3(kFp8Threads), smem, stream, a);
}

}  // namespace ep
