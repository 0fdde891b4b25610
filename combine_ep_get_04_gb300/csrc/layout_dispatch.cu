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
// Each CTA then writes its share of the layout outputs and copies the slice
// into the k receive rows (bf16: bulk stores issued from k warps at once) or
// quantises it (fp8: each warp stores the codes and scale of its 128-channel
// blocks from registers straight into the k rows).
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
constexpr int kWarpsF = 16;
constexpr int kThreadsF = kWarpsF * 32;
constexpr int kIdsPerThread = (int)(kFusedMaxN / kThreadsF);   // every id of the batch, in registers
constexpr int kExpPerThread = 1024 / kThreadsF;                // experts per thread in the scan (E <= 1024)
constexpr int kCopyChunk = 8;                                  // copies counted together (k <= 32)

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
    uint32_t in_bytes;       // bf16 bytes of one unit
};

// Shared memory: the mbarrier, then these int32 arrays, then the x slice.
__host__ __device__ constexpr uint32_t fused_head_bytes(int E) {
    return (16u + (32u + 32u + 32u * kWarpsF + 8u) * 4u + 8u * (uint32_t)E + 127u) & ~127u;
}

// One CTA per unit u = (t, sl).
__global__ void __launch_bounds__(kThreadsF) layout_dispatch_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* tok_e = reinterpret_cast<int32_t*>(smem + 16);      // [32] experts of this token
    int32_t* slot_s = tok_e + 32;                                 // [32] receive row of each copy
    int32_t* part_s = slot_s + 32;                                // [kWarpsF][32] per-warp counts per copy
    int32_t* misc_s = part_s + 32 * kWarpsF;                      // [0] valid ids, [1] flags, [2] scan total
    int32_t* cnt_s = misc_s + 8;                                  // [E]
    int32_t* off_s = cnt_s + a.E;                                 // [E]
    unsigned char* in_st = smem + fused_head_bytes(a.E);

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
    if (tid < 32) tok_e[tid] = my_tok_e;
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
        int32_t v[kExpPerThread], sum = 0;
#pragma unroll
        for (int q = 0; q < kExpPerThread; ++q) {
            const int e = kExpPerThread * tid + q;
            v[q] = e < a.E ? cnt_s[e] : 0;
            sum += v[q];
        }
        int32_t incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) part_s[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int32_t ws = lane < kWarpsF ? part_s[lane] : 0;
            int32_t wincl = ws;
#pragma unroll
            for (int d = 1; d < kWarpsF; d <<= 1) {
                const int32_t o = __shfl_up_sync(kFull, wincl, d);
                if (lane >= d) wincl += o;
            }
            if (lane < kWarpsF) part_s[lane] = wincl - ws;
            if (lane == kWarpsF - 1) misc_s[2] = wincl;
        }
        __syncthreads();
        int32_t run = part_s[warp] + incl - sum;
#pragma unroll
        for (int q = 0; q < kExpPerThread; ++q) {
            const int e = kExpPerThread * tid + q;
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
    // packed as lt << 16 | eq (both <= kFusedMaxN).  Eight copies are counted
    // together (independent sums), reduced per warp and kept per warp; the
    // warps' partial counts are added after the barrier.
    for (int j0 = 0; j0 < a.k; j0 += kCopyChunk) {
        int ej[kCopyChunk], c[kCopyChunk];
#pragma unroll
        for (int jj = 0; jj < kCopyChunk; ++jj) {
            ej[jj] = j0 + jj < a.k ? tok_e[j0 + jj] : -2;
            c[jj] = 0;
        }
#pragma unroll
        for (int q = 0; q < kIdsPerThread; ++q) {
            if (q * kThreadsF >= a.N) break;
            const int e = ids[q];
            const int n = q * kThreadsF + tid;
#pragma unroll
            for (int jj = 0; jj < kCopyChunk; ++jj) {
                c[jj] += (e >= 0 && e < ej[jj]) ? 0x10000 : 0;
                c[jj] += (e == ej[jj] && n < tk0 + j0 + jj) ? 1 : 0;
            }
        }
#pragma unroll
        for (int jj = 0; jj < kCopyChunk; ++jj) {
            const int r = __reduce_add_sync(kFull, c[jj]);
            if (lane == 0 && j0 + jj < 32) part_s[warp * 32 + j0 + jj] = r;
        }
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
            int32_t packed = 0;
#pragma unroll
            for (int w = 0; w < kWarpsF; ++w) packed += part_s[w * 32 + tid];
            const int32_t lt = packed >> 16, rank = packed & 0xffff;
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

    // Copy or quantise the slice into the k receive rows (the barrier also
    // publishes slot_s).
    const bool ok = __syncthreads_and(mbar_wait(bar, 0)) != 0;
    if (ok) {
        if (!a.fp8) {
            // copy j is issued by lane 0 of warp j % kWarpsF: up to kWarpsF bulk stores start together
            if (lane == 0) {
                for (int j = warp; j < a.k; j += kWarpsF) {
                    const int32_t slot = slot_s[j];
                    if (slot >= 0) {
                        bulk_store(a.recv + (int64_t)slot * a.H * 2 + (int64_t)sl * a.in_bytes, in_st, a.in_bytes);
                    }
                }
                bulk_commit();
                bulk_wait_read<0>();   // the slice stays in shared memory until every copy has read it
            }
        } else {
            // Warp per 128-channel block: amax, scale, codes; lane l holds the
            // codes of channels 4l..4l+3 and stores them (and lane j < k the
            // block's scale) into every copy's row.
            const float r448 = recip_448();
            const int64_t col0 = (int64_t)sl * a.nblk * 128;
            const int64_t s_col0 = (int64_t)sl * a.nblk;
            for (int b = warp; b < a.nblk; b += kWarpsF) {
                const uint2 v = *reinterpret_cast<const uint2*>(in_st + b * 256 + lane * 8);
                const float x0 = bf16_lo(v.x), x1 = bf16_hi(v.x), x2 = bf16_lo(v.y), x3 = bf16_hi(v.y);
                float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, d));
                const float sc = block_scale(m, a.ue8m0 != 0, r448);
                const float rs = __frcp_rn(sc);
                const uint32_t q01 = pack_e4m3x2(quotient_rn(x0, sc, rs), quotient_rn(x1, sc, rs));
                const uint32_t q23 = pack_e4m3x2(quotient_rn(x2, sc, rs), quotient_rn(x3, sc, rs));
                const uint32_t codes = q01 | (q23 << 16);
                const int64_t col = col0 + b * 128 + lane * 4;
                for (int j = 0; j < a.k; ++j) {
                    const int32_t slot = slot_s[j];
                    if (slot >= 0) *reinterpret_cast<uint32_t*>(a.recv + (int64_t)slot * a.H + col) = codes;
                }
                if (lane < a.k) {
                    const int32_t slot = slot_s[lane];
                    if (slot >= 0) {
                        const int64_t si = (int64_t)slot * a.nb + s_col0 + b;
                        if (a.ue8m0) {
                            static_cast<uint8_t*>(a.recv_s)[si] = ue8m0_byte(sc);
                        } else {
                            static_cast<float*>(a.recv_s)[si] = sc;
                        }
                    }
                }
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
        a.in_bytes = (uint32_t)a.nblk * 256u;
    } else {
        const int64_t vec16 = (int64_t)f.H * 2 / 16;
        a.slices = pick_divisor(f.T, vec16, 1024, 64, (int64_t)EP_FUSED_UNITS_PER_SM * num_sms);
        a.in_bytes = (uint32_t)(vec16 / a.slices * 16);
    }
    const size_t smem = fused_head_bytes(f.E) + ((a.in_bytes + 127u) & ~127u);
    cudaError_t err = cudaFuncSetAttribute(layout_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t units = (int64_t)f.T * a.slices;
    return launch_kernel(true, layout_dispatch_kernel, dim3((unsigned)(units + 1)), dim3(kThreadsF), smem, stream, a);
}

}  // namespace ep
