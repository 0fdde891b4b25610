// layout_dispatch.cu -- ep_layout_dispatch: the layout and the dispatch of a
// small batch in one launch.
//
// The v1 low-latency path of the pages avoided a separate notify pre-sync
// ("Why did DeepEP v2 drop the double-buffer design...", question: the
// low_latency path skipped the notify kernels), and small decode batches are
// where a launch matters ("Why does DeepEP LL kernel use double
// send/recv/signal buffers?", last answer: the optimisation targets high TPS).
// On one GPU the counterpart is to fold the layout into the dispatch kernel.
//
// Two kinds of CTA share the launch:
//  - unit CTAs, one per unit (a token row, or a slice of it when there are
//    few tokens; at most about one unit per SM).  Each starts the bulk copy of
//    its slice of x, reads all routing ids (N <= kFusedMaxN) into registers as
//    16-bit halves, two per word, and counts, for each copy (t, j) of its
//    token with expert e_j, the ids before the token equal to e_j and (packed
//    layout) the valid ids below e_j, both halves of a word compared at once
//    in SIMD-within-a-register arithmetic.  Rank = the first count plus the
//    token's own earlier copies of e_j; the receive row follows as in
//    ep_get_layout (same deterministic source order).  It then copies the
//    slice into its token's k receive rows with bulk stores issued from k
//    warps at once -- straight from the staged x slice (bf16), or from a
//    shared output stage that the warps fill with the codes and scales of
//    their 128-channel blocks (fp8).
//  - aux CTAs, a few, each building the full expert histogram: the first
//    writes counts, offsets and the partition sums; all of them share the
//    marking of receive rows that hold no copy (src_token = src_k = -1).
#include "ep.h"
#include "ep_device.cuh"
#include "ep_kernels.h"

// Units (CTAs) per SM the slice size aims at, at most (compile-time; tuned
// value).
#ifndef EP_FUSED_UNITS_PER_SM
#define EP_FUSED_UNITS_PER_SM 1
#endif
// Bytes of unused-row marking (src_token + src_k) per aux CTA the launch aims at.
#ifndef EP_FUSED_FILL_BYTES_PER_AUX
#define EP_FUSED_FILL_BYTES_PER_AUX 32768
#endif
#ifndef EP_FUSED_MAX_AUX
#define EP_FUSED_MAX_AUX 16
#endif

namespace ep {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarpsF = 16;
constexpr int kThreadsF = kWarpsF * 32;
constexpr int kIdsPerThread = (int)(kFusedMaxN / kThreadsF);   // every id of the batch, in registers
constexpr int kWordsPerThread = kIdsPerThread / 2;             // two 16-bit ids per word
constexpr int kExpPerThread = 1024 / kThreadsF;                // experts per thread in the scan (E <= 1024)
constexpr int kMaxTargets = 2 * 32;                            // counts a unit CTA takes: k, or 2k (packed)
constexpr int kMaxGroups = kMaxTargets / 4;                    // four 8-bit counts per word
constexpr uint32_t kHalfTop = 0x80008000u;                     // bit 15 of each half
constexpr uint32_t kHalfLow = 0x7fff7fffu;
constexpr uint32_t kNoId = 0xffffu;                            // half of a masked, bad or missing id
// fp8 units are quantised and stored in chunks of kChunkBlocks 128-channel
// blocks, one chunk per group of kChunkWarps warps (eight lanes per block),
// warps 1.. (warp 0 computes the receive rows meanwhile).
constexpr int kChunkWarps = 3;
constexpr int kChunkBlocks = 4 * kChunkWarps;
constexpr int kChunks = (kWarpsF - 1) / kChunkWarps;
constexpr int kFusedMaxBlocks = kChunks * kChunkBlocks;        // 128-channel blocks per fp8 unit at most
constexpr int kHeadBars = 8;                                   // x_full[kChunks], slots_ready
static_assert(kChunks + 1 <= kHeadBars, "mbarriers of the unit CTA");

static_assert(kIdsPerThread % 2 == 0, "ids are packed two per word");
static_assert(kIdsPerThread * 32 <= 255, "a warp's count per target must fit in 8 bits");

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
    int units;               // unit CTAs (blockIdx < units); the rest are aux CTAs
    int slices;              // units per token row
    int fp8;
    int ue8m0;               // power-of-two scales stored as exponent bytes
    int nb;                  // H / 128 (fp8)
    int nblk;                // 128-channel blocks per unit (fp8)
    uint32_t in_bytes;       // bf16 bytes of one unit
};

// Shared memory: the mbarriers, the small int32 arrays below, the aux CTAs'
// per-expert arrays, then (unit CTA) the x slice and the fp8 output stage.
__host__ __device__ constexpr uint32_t fused_head_bytes(int E) {
    return (8u * kHeadBars + (32u + kMaxGroups * kWarpsF + 32u + 8u) * 4u + 8u * (uint32_t)E + 127u) & ~127u;
}

// Bit 15 of each 16-bit half of w set where that half equals the half of b2
// (b2 = b in both halves, b < 0x8000): y = w ^ b2 is zero in a matching half;
// adding 0x7fff to its low 15 bits sets bit 15 unless they are all zero, and
// the half's own bit 15 is or-ed in.  No carry crosses a half.
__device__ __forceinline__ uint32_t halves_equal(uint32_t w, uint32_t b2) {
    const uint32_t y = w ^ b2;
    const uint32_t z = (y & kHalfLow) + kHalfLow;
    return ~(z | y) & kHalfTop;
}

// Bit 15 of each half of w set where that half is a valid id (< 0x8000) below
// b, given bm2 = b - 1 in both halves (b >= 1): (0x8000 + b - 1) - a stays in
// [0, 0xffff] for a < 0x8000, so no borrow crosses a half, and its bit 15 is
// set exactly when a <= b - 1.  Invalid halves (0xffff) are masked by ~w.
__device__ __forceinline__ uint32_t halves_below(uint32_t w, uint32_t bm2) {
    return ((bm2 | kHalfTop) - (w & kHalfLow)) & ~w & kHalfTop;
}

// Field f (8 bits) of a packed count word.
__device__ __forceinline__ uint32_t count_field(uint32_t v, int f) { return (v >> (8 * f)) & 0xffu; }

// Unit CTAs first (one per unit u = (t, sl)), then the aux CTAs.
__global__ void __launch_bounds__(kThreadsF) layout_dispatch_kernel(const FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* x_full = reinterpret_cast<uint64_t*>(smem);          // [kChunks] x slice (chunk) landed
    uint64_t* slots_ready = x_full + kChunks;                       // slot_s written
    int32_t* slot_s = reinterpret_cast<int32_t*>(smem + 8 * kHeadBars);   // [32] receive row of each copy
    uint32_t* part_s = reinterpret_cast<uint32_t*>(slot_s + 32);  // [kMaxGroups][kWarpsF] packed per-warp counts
    int32_t* wsum_s = reinterpret_cast<int32_t*>(part_s + kMaxGroups * kWarpsF);   // [32] aux: scan partials
    int32_t* misc_s = wsum_s + 32;                                // aux: [0] flags, [1] scan total
    int32_t* cnt_s = misc_s + 8;                                  // aux: [E]
    int32_t* off_s = cnt_s + a.E;                                 // aux: [E]
    unsigned char* in_st = smem + fused_head_bytes(a.E);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool aux = (int)blockIdx.x >= a.units;

    pdl_launch_dependents();
    if (aux) {
        // ---------------------------------------------------------- aux CTA
        const int ai = (int)blockIdx.x - a.units;
        const int n_aux = (int)gridDim.x - a.units;
        if (tid == 0) misc_s[0] = 0;
        for (int e = tid; e < a.E; e += kThreadsF) cnt_s[e] = 0;
        __syncthreads();
        pdl_wait();
        // histogram of all ids (warp-aggregated shared-memory adds); bad ids
        bool bad = false;
#pragma unroll
        for (int q = 0; q < kIdsPerThread; ++q) {
            if (q * kThreadsF >= a.N) break;
            const int n = q * kThreadsF + tid;
            int e = n < a.N ? __ldg(a.topk_idx + n) : -1;
            if (e < -1 || e >= a.E) {
                bad = true;
                e = -1;
            }
            const uint32_t peers = __match_any_sync(kFull, e);
            if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt_s[e], __popc(peers));
        }
        if (bad && ai == 0) atomicOr(&misc_s[0], (int)kErrBadExpert);
        __syncthreads();
        // exclusive scan over experts
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
            if (lane == kWarpsF - 1) misc_s[1] = wincl;
        }
        __syncthreads();
        const int32_t total = misc_s[1];
        if (ai == 0) {
            int32_t run = wsum_s[warp] + incl - sum;
#pragma unroll
            for (int q = 0; q < kExpPerThread; ++q) {
                const int e = kExpPerThread * tid + q;
                if (e < a.E) off_s[e] = run;
                run += v[q];
            }
            __syncthreads();
            for (int e = tid; e < a.E; e += kThreadsF) {
                a.counts[e] = cnt_s[e];
                a.offsets[e] = off_s[e];
            }
            if (tid == 0) a.offsets[a.E] = total;
            const int per = a.E / a.P;
            for (int p = tid; p < a.P; p += kThreadsF) {
                const int e0 = p * per, e1 = e0 + per - 1;
                a.part_counts[p] = off_s[e1] + cnt_s[e1] - off_s[e0];
                a.part_offsets[p] = off_s[e0];
            }
            if (tid == 0) a.part_offsets[a.P] = total;
            if (tid == 0 && a.err_flags != nullptr && misc_s[0]) atomicOr(a.err_flags, (uint32_t)misc_s[0]);
        }
        // Rows that hold no copy get src_token = src_k = -1: packed, rows
        // [total, R); capacity, rows [min(count, cap), cap) of each expert.
        // The aux CTAs take interleaved shares.
        if (a.mode == 0) {
            for (int r = total + ai * kThreadsF + tid; r < a.R; r += n_aux * kThreadsF) {
                a.src_token[r] = -1;
                a.src_k[r] = -1;
            }
        } else {
            // warp per expert (experts ai, ai + n_aux, ... of this aux CTA), lanes over its rows
            for (int e = ai + warp * n_aux; e < a.E; e += kWarpsF * n_aux) {
                const int64_t row0 = (int64_t)e * a.cap;
                for (int r = cnt_s[e] + lane; r < a.cap; r += 32) {
                    a.src_token[row0 + r] = -1;
                    a.src_k[row0 + r] = -1;
                }
            }
        }
        return;
    }

    // -------------------------------------------------------------- unit CTA
    const int u = (int)blockIdx.x;
    const int t = u / a.slices;
    const int sl = u - t * a.slices;
    const int tk0 = t * a.k;
    // bf16: the x slice in one bulk copy; fp8: one per chunk of blocks
    const int n_chunks = a.fp8 ? (a.nblk + kChunkBlocks - 1) / kChunkBlocks : 1;
    if (tid == 0) {
        for (int c = 0; c < n_chunks; ++c) mbar_init(&x_full[c], 1);
        mbar_init(slots_ready, 1);
        fence_mbar_init();
        // Before the wait on the previous kernel: pull this CTA's x slice
        // and (below) the routing ids towards L2, so that their DRAM (and
        // page-table) latency overlaps that kernel's tail.  A prefetch has no
        // effect on what the loads after the wait return: the L2 is the point
        // of coherence, and writes of the previous kernel land there.
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.x + (int64_t)t * a.H * 2 + (int64_t)sl * a.in_bytes),
                     "r"(a.in_bytes)
                     : "memory");
    }
    for (int q = tid; q * 32 < a.N; q += kThreadsF) {   // one 128-byte line each
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.topk_idx + q * 32) : "memory");
    }
    pdl_wait();
    if (tid == 0) {   // the slice of x does not depend on the layout: start it first
        const unsigned char* xs = a.x + (int64_t)t * a.H * 2 + (int64_t)sl * a.in_bytes;
        if (!a.fp8) {
            mbar_arrive_expect_tx(&x_full[0], a.in_bytes);
            bulk_load(in_st, xs, a.in_bytes, &x_full[0]);
        } else {
            for (int c = 0; c < n_chunks; ++c) {
                const uint32_t nbc = (uint32_t)min(kChunkBlocks, a.nblk - c * kChunkBlocks);
                mbar_arrive_expect_tx(&x_full[c], nbc * 256u);
                bulk_load(in_st + c * kChunkBlocks * 256, xs + c * kChunkBlocks * 256, nbc * 256u, &x_full[c]);
            }
        }
    }
    // Every routing id, loaded at once, as 16-bit halves (id n = q*kThreadsF +
    // tid in half q % 2 of word q / 2); before[] marks the halves of ids
    // before this token.  Masked, bad and missing ids become 0xffff.
    uint32_t word[kWordsPerThread], before[kWordsPerThread];
#pragma unroll
    for (int w = 0; w < kWordsPerThread; ++w) {
        word[w] = 0;
        before[w] = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = (2 * w + h) * kThreadsF + tid;
            const int e = n < a.N ? __ldg(a.topk_idx + n) : -1;
            const uint32_t half = (e >= 0 && e < a.E) ? (uint32_t)e : kNoId;
            word[w] |= half << (16 * h);
            before[w] |= (n < tk0 ? 0x8000u : 0u) << (16 * h);
        }
    }
    // The token's experts: lane j of every warp holds e_j (-1 if masked or bad).
    int ej = -2 - lane;                               // lanes >= k: never equal to an id
    if (lane < a.k) {
        ej = __ldg(a.topk_idx + tk0 + lane);
        if (ej < -1 || ej >= a.E) ej = -1;
    }
    // Per-warp counts, four 8-bit counts per word: in group j / 4, the ids
    // before the token equal to e_j; with the packed layout, in group
    // g_below + j / 4, the valid ids below e_j (offsets[e_j]).  Fields of
    // copies beyond k or with e_j < 0 hold counts nobody reads.
    const bool two_words = a.N > 2 * kThreadsF;                   // words beyond N hold no id
    const int g_below = (a.k + 3) / 4;
    for (int j0 = 0; j0 < a.k; j0 += 4) {
        uint32_t acc = 0;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const uint32_t b = (uint32_t)max(__shfl_sync(kFull, ej, (j0 + f) & 31), 0) * 0x00010001u;
            uint32_t c = __popc(halves_equal(word[0], b) & before[0]);
            if (two_words) c += __popc(halves_equal(word[1], b) & before[1]);
            acc |= c << (8 * f);
        }
        acc = __reduce_add_sync(kFull, acc);
        if (lane == 0) part_s[(j0 / 4) * kWarpsF + warp] = acc;
    }
    if (a.mode == 0) {
        for (int j0 = 0; j0 < a.k; j0 += 4) {
            uint32_t acc = 0;
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const int e = __shfl_sync(kFull, ej, (j0 + f) & 31);
                uint32_t c = 0;
                if (e > 0) {
                    const uint32_t bm = (uint32_t)(e - 1) * 0x00010001u;
                    c = __popc(halves_below(word[0], bm));
                    if (two_words) c += __popc(halves_below(word[1], bm));
                }
                acc |= c << (8 * f);
            }
            acc = __reduce_add_sync(kFull, acc);
            if (lane == 0) part_s[(g_below + j0 / 4) * kWarpsF + warp] = acc;
        }
    }
    __syncthreads();

    // Warp 0 turns the counts into the receive rows of this token's copies
    // (lane j = copy j) and publishes them through slots_ready, while the
    // other warps quantise.
    if (warp == 0) {
        const uint32_t peers = __match_any_sync(kFull, ej);
        int32_t slot = -1;
        if (lane < a.k && ej >= 0) {
            int32_t rank = __popc(peers & lanemask_lt());   // the token's own earlier copies of e_j
#pragma unroll
            for (int w = 0; w < kWarpsF; ++w) rank += (int32_t)count_field(part_s[(lane / 4) * kWarpsF + w], lane % 4);
            if (a.mode == 0) {
                const int gb = (a.k + 3) / 4 + lane / 4;
                int32_t lt = 0;
#pragma unroll
                for (int w = 0; w < kWarpsF; ++w) lt += (int32_t)count_field(part_s[gb * kWarpsF + w], lane % 4);
                slot = lt + rank;
            } else if (rank < a.cap) {
                slot = ej * a.cap + rank;
            } else if (sl == 0 && a.err_flags != nullptr) {
                atomicOr(a.err_flags, kErrCapacity);
            }
        }
        slot_s[lane] = slot;
        __syncwarp();
        if (lane == 0) mbar_arrive(slots_ready);
        if (sl == 0 && lane < a.k) {
            a.slot_of[tk0 + lane] = slot;
            if (slot >= 0) {
                a.src_token[slot] = t;
                a.src_k[slot] = lane;
                if (a.recv_w != nullptr) a.recv_w[slot] = __ldg(a.topk_w + tk0 + lane);
            }
        }
    }

    bool ok = true;
    if (!a.fp8) {
        // bf16: copy j is written by lane 0 of warp j % kWarpsF, straight from
        // the staged slice, up to kWarpsF copies at once
        if (lane == 0 && warp < a.k) {
            ok = mbar_wait(slots_ready, 0) && mbar_wait(&x_full[0], 0);
            if (ok) {
                for (int j = warp; j < a.k; j += kWarpsF) {
                    const int32_t slot = slot_s[j];
                    if (slot >= 0) {
                        bulk_store(a.recv + (int64_t)slot * a.H * 2 + (int64_t)sl * a.in_bytes, in_st, a.in_bytes);
                    }
                }
                bulk_commit();
                bulk_wait_read<0>();   // the slice stays in shared memory until every copy has read it
            }
        }
    } else if (warp > 0 && (warp - 1) / kChunkWarps < n_chunks) {
        // fp8: the warps of chunk c quantise its blocks into the shared output
        // stage [codes nblk*128 | f32 scales] as soon as that part of x has
        // landed (eight lanes per block, 16 channels each, the block's amax in
        // three shuffles), then the group's first lane writes the chunk into
        // the k rows with bulk stores -- so the stores of early chunks overlap
        // the quantisation of later ones.  (SIMT stores of the codes from
        // registers reached only ~17 GB/s per SM here: the rows are scattered
        // over the capacity buffer, one line per store.)
        const int c = (warp - 1) / kChunkWarps;
        const int wi = (warp - 1) - c * kChunkWarps;
        const int b_end = min(a.nblk, (c + 1) * kChunkBlocks);
        unsigned char* out_st = in_st + ((a.in_bytes + 127u) & ~127u);
        float* scale_st = reinterpret_cast<float*>(out_st + (uint32_t)a.nblk * 128u);
        ok = __all_sync(kFull, mbar_wait(&x_full[c], 0));
        if (ok) {
            const BlockScale r = quantize_blocks_8lanes(in_st, out_st, c * kChunkBlocks + wi * 4, b_end, a.ue8m0 != 0,
                                                        recip_448());
            if (r.first) scale_st[r.b] = r.sc;
            fence_proxy_async_smem();
        }
        // the chunk's warps have all written (or all given up)
        asm volatile("bar.sync %0, %1;" ::"r"(1 + c), "r"(kChunkWarps * 32) : "memory");
        const int b0 = c * kChunkBlocks, nbc = b_end - b0;
        const int64_t s_col0 = (int64_t)sl * a.nblk + b0;
        const bool scale_bulk = !a.ue8m0 && a.nb % 4 == 0 && a.nblk % 4 == 0;
        if (ok) ok = mbar_wait(slots_ready, 0);
        if (ok && wi == 0 && lane == 0) {
            for (int j = 0; j < a.k; ++j) {
                const int32_t slot = slot_s[j];
                if (slot < 0) continue;
                bulk_store(a.recv + (int64_t)slot * a.H + s_col0 * 128, out_st + b0 * 128, (uint32_t)nbc * 128u);
                if (scale_bulk) {
                    bulk_store(static_cast<float*>(a.recv_s) + (int64_t)slot * a.nb + s_col0, scale_st + b0,
                               (uint32_t)nbc * 4u);
                }
            }
            bulk_commit();
        }
        if (ok && !scale_bulk) {
            for (int q = wi * 32 + lane; q < a.k * nbc; q += kChunkWarps * 32) {
                const int j = q / nbc, bb = q - j * nbc;
                const int32_t slot = slot_s[j];
                if (slot < 0) continue;
                const int64_t si = (int64_t)slot * a.nb + s_col0 + bb;
                if (a.ue8m0) {
                    static_cast<uint8_t*>(a.recv_s)[si] = ue8m0_byte(scale_st[b0 + bb]);
                } else {
                    static_cast<float*>(a.recv_s)[si] = scale_st[b0 + bb];
                }
            }
        }
        if (ok && wi == 0 && lane == 0) bulk_wait_read<0>();   // the stage stays until every copy has read it
    }
    if (!ok && a.err_flags != nullptr) atomicOr(a.err_flags, kErrTimeout);
    if (tid == 0) {
        // no copy into this CTA's shared memory may be left in flight at exit
        for (int c = 0; c < n_chunks; ++c) (void)mbar_wait(&x_full[c], 0);
    }
}

// Slices a row of n granules is cut into for the fused launch: the most
// slices (a divisor d of n, slices of at most max_per and at least min_per
// granules) with T*d <= want units; at least the fewest that fit max_per.
int pick_fused_slices(int64_t T, int64_t n, int64_t max_per, int64_t min_per, int64_t want) {
    int best = 0;
    for (int64_t d = 1; d <= n; ++d) {
        if (n % d) continue;
        const int64_t per = n / d;
        if (per > max_per) continue;
        if (best == 0) {
            best = (int)d;
            continue;
        }
        if (per < min_per || T * d > want) break;
        best = (int)d;
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
    const int64_t want = (int64_t)EP_FUSED_UNITS_PER_SM * num_sms;
    if (f.fp8) {
        a.nb = f.H / 128;
        a.slices = pick_fused_slices(f.T, a.nb, kFusedMaxBlocks, 2, want);
        a.nblk = a.nb / a.slices;
        a.in_bytes = (uint32_t)a.nblk * 256u;
    } else {
        const int64_t vec16 = (int64_t)f.H * 2 / 16;
        a.slices = pick_fused_slices(f.T, vec16, 1024, 64, want);
        a.in_bytes = (uint32_t)(vec16 / a.slices * 16);
    }
    a.units = f.T * a.slices;
    // aux CTAs: enough that each marks about EP_FUSED_FILL_BYTES_PER_AUX bytes
    // of unused rows (capacity layout; the packed layout has at most the
    // masked copies to mark)
    int n_aux = 1;
    if (f.mode != 0) {
        const int64_t fill = (int64_t)f.R * 8;
        n_aux = (int)((fill + EP_FUSED_FILL_BYTES_PER_AUX - 1) / EP_FUSED_FILL_BYTES_PER_AUX);
        if (n_aux > EP_FUSED_MAX_AUX) n_aux = EP_FUSED_MAX_AUX;
    }
    if (f.mode != 0 && n_aux > f.E) n_aux = f.E;   // every capacity-mode aux CTA marks at least one expert
    if (n_aux < 1) n_aux = 1;
    // shared memory: head, the x slice, and (fp8) the output stage: codes + f32 scales
    size_t smem = fused_head_bytes(f.E) + ((a.in_bytes + 127u) & ~127u);
    if (f.fp8) smem += ((uint32_t)a.nblk * 132u + 127u) & ~127u;
    // More than half of an SM's shared memory, so that at most one CTA of
    // this kernel is resident per SM: the next launch of this kernel (started
    // early, programmatic serialization) then takes each SM as its CTA there
    // finishes, instead of stacking several early CTAs on the SMs this grid
    // left idle (measured on the decode workload: 3.8-4.4 us back to back
    // with the reservation, 7.5-8 us without).
    int dev = 0, smem_sm = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (err != cudaSuccess) return err;
    if (smem < (size_t)smem_sm / 2 + 1024) smem = (size_t)smem_sm / 2 + 1024;
    err = cudaFuncSetAttribute(layout_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(true, layout_dispatch_kernel, dim3((unsigned)(a.units + n_aux)), dim3(kThreadsF), smem,
                         stream, a);
}

}  // namespace ep
