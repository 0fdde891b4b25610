// layout_dispatch.cu -- ep_layout_dispatch: the layout and the dispatch of a
// small batch in one launch.
//
// The v1 low-latency path of the pages avoided a separate notify pre-sync
// ("Why did DeepEP v2 drop the double-buffer design...", question: the
// low_latency path skipped the notify kernels), and small decode batches are
// where a launch matters ("Why does DeepEP LL kernel use double
// send/recv/signal buffers?", last answer: the optimisation targets high TPS).
// On one GPU the counterpart is to fold the layout into the dispatch kernel:
// each CTA owns one unit (a token row or a slice of it, about one unit per
// SM), starts the bulk copy of its slice of x, and while that is in flight
// reads all routing ids (N <= kFusedMaxN) and finds the receive rows of its
// token's k copies from two counts per copy (t, j) of expert e: the valid ids
// of smaller experts (the packed offset of e) and the ids before (t, j) equal
// to e (the rank) -- the same deterministic source order as ep_get_layout.
// One extra CTA builds the full histogram and scan for counts and offsets.
// Each CTA then writes its share of the layout outputs and copies (bf16) or
// quantises (fp8) the slice into the k receive rows with bulk stores.
#include "ep.h"
#include "ep_device.cuh"
#include "ep_kernels.h"

// Units (CTAs) per SM the slice size aims at (compile-time; tuned value).
#ifndef EP_FUSED_UNITS_PER_SM
#define EP_FUSED_UNITS_PER_SM 1
#endif

namespace ep {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarpsF = 8;
constexpr int kThreadsF = kWarpsF * 32;
constexpr int kIdsPerThread = (int)(kFusedMaxN / kThreadsF);   // every id of the batch, in registers

struct FusedArgs {
    const int32_t* topk_idx;
    const unsigned char* x;
    const float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* part_counts;
    int32_t* part_offsets;
    int32_t* slot_of;
    int32_t* src_token;
    int32_t* src_k;
    unsigned char* recv;
    void* recv_s;            // f32 scales, or u8 exponents with ue8m0
    float* recv_w;
    uint32_t* err_flags;
    int T, H, E, k, P, mode, cap, N, R;
    int slices;              // units per token row
    int fp8;
    int ue8m0;               // power-of-two scales stored as exponent bytes
    int nb;                  // H / 128 (fp8)
    int nblk;                // 128-channel blocks per unit (fp8)
    int scale_bulk;          // scale rows stored with a bulk copy
    uint32_t in_bytes;       // bf16 bytes of one unit
    uint32_t in_stride;      // in_bytes rounded up to 128
};

// One CTA per unit u = (t, sl).
__global__ void __launch_bounds__(kThreadsF) layout_dispatch_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* tok_e = reinterpret_cast<int32_t*>(smem + 16);      // [32] experts of this token
    int32_t* rank_s = tok_e + 32;                                 // [32] rank of each copy
    int32_t* slot_s = rank_s + 32;                                // [32] receive row of each copy
    int32_t* wsum_s = slot_s + 32;                                // [8]
    int32_t* misc_s = wsum_s + 8;                                 // [0] valid ids, [1] flags, [2] scan total
    int32_t* cnt_s = misc_s + 8;                                  // [E]
    int32_t* off_s = cnt_s + a.E;                                 // [E]
    unsigned char* in_st = smem + ((16 + (32 * 3 + 16) * 4 + 8 * a.E + 127) & ~127);
    unsigned char* out_st = in_st + a.in_stride;                  // fp8 codes, then scales

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    // CTAs 0..units-1 each own one unit; the last CTA builds the histogram.
    const int units = (int)gridDim.x - 1;
    const bool hist_cta = (int)blockIdx.x == units;
    const int u = hist_cta ? 0 : (int)blockIdx.x;
    const int t = u / a.slices;
    const int sl = u - t * a.slices;
    const int tk0 = t * a.k;

    pdl_launch_dependents();
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    pdl_wait();
    if (tid == 0 && !hist_cta) {   // the slice of x does not depend on the layout: start it first
        mbar_arrive_expect_tx(bar, a.in_bytes);
        bulk_load(in_st, a.x + (int64_t)t * a.H * 2 + (int64_t)sl * a.in_bytes, a.in_bytes, bar);
    }
    // All loads of routing ids are issued at once, before anything waits.
    int ids[kIdsPerThread];
#pragma unroll
    for (int q = 0; q < kIdsPerThread; ++q) {
        const int n = q * kThreadsF + tid;
        ids[q] = n < a.N ? __ldg(a.topk_idx + n) : -1;
    }
    int my_tok_e = -2;                                // never equal to an id
    if (tid < a.k && !hist_cta) {
        my_tok_e = __ldg(a.topk_idx + tk0 + tid);
        if (my_tok_e < -1 || my_tok_e >= a.E) my_tok_e = -1;
    }
    if (tid == 0) {
        misc_s[0] = 0;
        misc_s[1] = 0;
    }
    for (int e = tid; e < a.E; e += kThreadsF) cnt_s[e] = 0;
    if (tid < 32) {
        rank_s[tid] = 0;
        tok_e[tid] = my_tok_e;
    }
    __syncthreads();
    if (hist_cta) {
        // counts, offsets and partition sums of all experts; bad ids
        bool bad = false;
#pragma unroll
        for (int q = 0; q < kIdsPerThread; ++q) {
            if (q * kThreadsF >= a.N) break;
            int e = ids[q];
            if (e < -1 || e >= a.E) {
                bad = true;
                e = -1;
            }
            const uint32_t peers = __match_any_sync(kFull, e);
            if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt_s[e], __popc(peers));
        }
        if (bad) atomicOr(&misc_s[1], (int)kErrBadExpert);
        __syncthreads();
        int32_t v[4], sum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = 4 * tid + q;
            v[q] = e < a.E ? cnt_s[e] : 0;
            sum += v[q];
        }
        int32_t incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) wsum_s[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int32_t ws = lane < kWarpsF ? wsum_s[lane] : 0;
            int32_t wincl = ws;
#pragma unroll
            for (int d = 1; d < kWarpsF; d <<= 1) {
                const int32_t o = __shfl_up_sync(kFull, wincl, d);
                if (lane >= d) wincl += o;
            }
            if (lane < kWarpsF) wsum_s[lane] = wincl - ws;
            if (lane == kWarpsF - 1) misc_s[2] = wincl;
        }
        __syncthreads();
        int32_t run = wsum_s[warp] + incl - sum;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = 4 * tid + q;
            if (e < a.E) off_s[e] = run;
            run += v[q];
        }
        __syncthreads();
        const int32_t total = misc_s[2];
        for (int e = tid; e < a.E; e += kThreadsF) {
            a.counts[e] = cnt_s[e];
            a.offsets[e] = off_s[e];
        }
        if (tid == 0) a.offsets[a.E] = total;
        const int per = a.E / a.P;
        for (int q = tid; q < a.P; q += kThreadsF) {
            const int e0 = q * per, e1 = e0 + per - 1;
            a.part_counts[q] = off_s[e1] + cnt_s[e1] - off_s[e0];
            a.part_offsets[q] = off_s[e0];
        }
        if (tid == 0) a.part_offsets[a.P] = total;
        __syncthreads();
        if (tid == 0 && a.err_flags != nullptr && misc_s[1]) atomicOr(a.err_flags, (uint32_t)misc_s[1]);
        return;
    }

    // Slot of copy j of this token, from two counts over all ids:
    //   lt_j = valid ids with a smaller expert than e_j (= offsets[e_j]),
    //   eq_j = ids before (t, j) with expert e_j      (= rank of the copy),
    // packed as lt << 16 | eq (both <= kFusedMaxN) and summed over the CTA.
    for (int j = 0; j < a.k; ++j) {
        const int ej = tok_e[j];
        int c = 0;
#pragma unroll
        for (int q = 0; q < kIdsPerThread; ++q) {
            if (q * kThreadsF >= a.N) break;
            const int e = ids[q];
            const int n = q * kThreadsF + tid;
            c += (e >= 0 && e < ej) ? 0x10000 : 0;
            c += (e == ej && n < tk0 + j) ? 1 : 0;
        }
        c = __reduce_add_sync(kFull, c);
        if (lane == 0 && c) atomicAdd(&rank_s[j], c);
    }
    // Counts this CTA needs to mark rows that hold no copy: per expert it
    // covers (capacity), or the number of valid ids (packed).
    if (a.mode == 0) {
        int c = 0;
#pragma unroll
        for (int q = 0; q < kIdsPerThread; ++q) {
            if (q * kThreadsF >= a.N) break;
            c += (ids[q] >= 0 && ids[q] < a.E) ? 1 : 0;
        }
        c = __reduce_add_sync(kFull, c);
        if (lane == 0 && c) atomicAdd(&misc_s[0], c);
    } else {
        for (int e = u; e < a.E; e += units) {
            int c = 0;
#pragma unroll
            for (int q = 0; q < kIdsPerThread; ++q) {
                if (q * kThreadsF >= a.N) break;
                c += ids[q] == e ? 1 : 0;
            }
            c = __reduce_add_sync(kFull, c);
            if (lane == 0 && c) atomicAdd(&cnt_s[e], c);
        }
    }
    __syncthreads();

    // Receive rows of this token's copies.
    if (tid < a.k) {
        const int e = tok_e[tid];
        int32_t slot = -1;
        if (e >= 0) {
            const int32_t lt = rank_s[tid] >> 16, rank = rank_s[tid] & 0xffff;
            if (a.mode == 0) {
                slot = lt + rank;
            } else if (rank < a.cap) {
                slot = e * a.cap + rank;
            } else if (sl == 0) {
                atomicOr(&misc_s[1], (int)kErrCapacity);
            }
        }
        slot_s[tid] = slot;
        if (sl == 0) {
            a.slot_of[tk0 + tid] = slot;
            if (slot >= 0) {
                a.src_token[slot] = t;
                a.src_k[slot] = tid;
                if (a.recv_w != nullptr) a.recv_w[slot] = __ldg(a.topk_w + tk0 + tid);
            }
        }
    }

    // Rows that hold no copy get src_token = src_k = -1.
    if (a.mode == 0) {
        const int total = misc_s[0];
        for (int r = total + u * kThreadsF + tid; r < a.R; r += units * kThreadsF) {
            a.src_token[r] = -1;
            a.src_k[r] = -1;
        }
    } else {
        for (int e = u; e < a.E; e += units) {
            const int row0 = e * a.cap;
            for (int r = min(cnt_s[e], a.cap) + tid; r < a.cap; r += kThreadsF) {
                a.src_token[row0 + r] = -1;
                a.src_k[row0 + r] = -1;
            }
        }
    }
    __syncthreads();

    // Copy or quantise the slice into the k receive rows.
    const bool ok = __syncthreads_and(mbar_wait(bar, 0)) != 0;
    if (ok) {
        if (!a.fp8) {
            if (warp == 0) {
                const int32_t slot = lane < a.k ? slot_s[lane] : -1;
                if (slot >= 0) {
                    bulk_store(a.recv + (int64_t)slot * a.H * 2 + (int64_t)sl * a.in_bytes, in_st, a.in_bytes);
                }
                bulk_commit();
                bulk_wait_all();
            }
        } else {
            const uint32_t q_bytes = (uint32_t)a.nblk * 128u;
            float* oscale = reinterpret_cast<float*>(out_st + q_bytes);
            for (int b = warp; b < a.nblk; b += kWarpsF) {
                const uint2 v = *reinterpret_cast<const uint2*>(in_st + b * 256 + lane * 8);
                const float x0 = bf16_lo(v.x), x1 = bf16_hi(v.x), x2 = bf16_lo(v.y), x3 = bf16_hi(v.y);
                float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, d));
                const float sc = block_scale(m, a.ue8m0 != 0);
                const uint32_t q01 = pack_e4m3x2(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
                const uint32_t q23 = pack_e4m3x2(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
                *reinterpret_cast<uint32_t*>(out_st + b * 128 + lane * 4) = q01 | (q23 << 16);
                if (lane == 0) {
                    if (a.ue8m0) {
                        out_st[q_bytes + b] = ue8m0_byte(sc);
                    } else {
                        oscale[b] = sc;
                    }
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (warp == 0) {
                const int32_t slot = lane < a.k ? slot_s[lane] : -1;
                if (slot >= 0) {
                    bulk_store(a.recv + (int64_t)slot * a.H + (int64_t)sl * a.nblk * 128, out_st, q_bytes);
                    const int64_t s0 = (int64_t)slot * a.nb + (int64_t)sl * a.nblk;
                    if (a.ue8m0) {
                        uint8_t* edst = static_cast<uint8_t*>(a.recv_s) + s0;
                        for (int b = 0; b < a.nblk; ++b) edst[b] = out_st[q_bytes + b];
                    } else if (a.scale_bulk) {
                        bulk_store(static_cast<float*>(a.recv_s) + s0, oscale, (uint32_t)a.nblk * 4u);
                    } else {
                        float* sdst = static_cast<float*>(a.recv_s) + s0;
                        for (int b = 0; b < a.nblk; ++b) sdst[b] = oscale[b];
                    }
                }
                bulk_commit();
                bulk_wait_all();
            }
        }
    } else if (tid == 0) {
        atomicOr(&misc_s[1], (int)kErrTimeout);
    }
    __syncthreads();
    if (tid == 0 && a.err_flags != nullptr && misc_s[1]) atomicOr(a.err_flags, (uint32_t)misc_s[1]);
}

int pick_divisor(int64_t T, int64_t n, int64_t max_per, int64_t min_per, int64_t want) {
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

bool fused_layout_dispatch_fits(int64_t N, int64_t T, int E) {
    return N <= kFusedMaxN && T <= kFusedMaxT && E <= 1024;
}

cudaError_t launch_layout_dispatch(const FusedLaunch& f, int num_sms, cudaStream_t stream) {
    FusedArgs a{};
    a.topk_idx = f.topk_idx;
    a.x = static_cast<const unsigned char*>(f.x);
    a.topk_w = f.topk_w;
    a.counts = f.counts;
    a.offsets = f.offsets;
    a.part_counts = f.part_counts;
    a.part_offsets = f.part_offsets;
    a.slot_of = f.slot_of;
    a.src_token = f.src_token;
    a.src_k = f.src_k;
    a.recv = static_cast<unsigned char*>(f.recv);
    a.recv_s = f.recv_scales;
    a.recv_w = f.recv_w;
    a.err_flags = f.err_flags;
    a.T = f.T;
    a.H = f.H;
    a.E = f.E;
    a.k = f.k;
    a.P = f.P;
    a.mode = f.mode;
    a.cap = f.cap;
    a.N = f.T * f.k;
    a.R = (int)f.R;
    a.fp8 = f.fp8;
    a.ue8m0 = f.ue8m0;
    if (f.fp8) {
        a.nb = f.H / 128;
        a.slices = pick_divisor(f.T, a.nb, 64, 2, (int64_t)EP_FUSED_UNITS_PER_SM * num_sms);
        a.nblk = a.nb / a.slices;
        a.scale_bulk = (a.nb % 4 == 0) && (a.nblk % 4 == 0);
        a.in_bytes = (uint32_t)a.nblk * 256u;
    } else {
        const int64_t vec16 = (int64_t)f.H * 2 / 16;
        a.slices = pick_divisor(f.T, vec16, 1024, 64, (int64_t)EP_FUSED_UNITS_PER_SM * num_sms);
        a.in_bytes = (uint32_t)(vec16 / a.slices * 16);
    }
    a.in_stride = (a.in_bytes + 127u) & ~127u;
    const size_t head = (16 + (32 * 3 + 16) * 4 + 8 * (size_t)f.E + 127) & ~(size_t)127;
    const size_t out_bytes = f.fp8 ? (((size_t)a.nblk * 132 + 127) & ~(size_t)127) : 0;
    const size_t smem = head + a.in_stride + out_bytes;
    cudaError_t err = cudaFuncSetAttribute(layout_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t units = (int64_t)f.T * a.slices;
    return launch_kernel(true, layout_dispatch_kernel, dim3((unsigned)(units + 1)), dim3(kThreadsF), smem, stream, a);
}

}  // namespace ep
