// layout.cu -- top-k routing -> per-expert counts, prefix offsets, partition
// sums, slot map and source maps (ep_get_layout).
//
// Counts per expert follow the quoted low-latency dispatch excerpt on
// "Redundant atomics in internode_ll" (a token count per expert; partition =
// expert / experts-per-partition).  The slot order keeps source order inside
// each expert ("Reasons for not calling NVSHMEM public APIs?": data for one
// expert stays in order), which makes the layout deterministic: the rank of
// copy (t, j) inside expert e is the number of copies (t', j') < (t, j) of e.
//
// Design (no global atomics on the order, no spin-waits):
//  * The flattened ids are cut into chunks of kChunk entries, one CTA each.
//  * Every CTA needs, per expert, the copies before its chunk (its base) and
//    the total over all chunks (for the offsets).  Small inputs: each CTA
//    counts them itself from topk_idx (one launch, no workspace).  Large
//    inputs: a histogram kernel writes per-chunk counts [C][E] to the
//    workspace and the rank kernel sums the column of each expert.
//  * Inside a chunk, each warp of 32 consecutive entries ranks equal ids with
//    __match_any_sync; a [32 warps][E] table of per-warp counts, scanned down
//    each expert's column, gives the rank of every entry in the chunk.
#include "ep_device.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kThreads = 1024;          // one entry per thread per round
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int load_id(const int32_t* __restrict__ idx, int64_t n, int64_t end,
                                       int E, bool& bad) {
    if (n >= end) return -1;
    int e = __ldg(idx + n);
    if (e < -1 || e >= E) {
        bad = true;
        return -1;
    }
    return e;
}

// Adds the ids of entries [begin, end) to cnt[] (warp-aggregated shared atomics).
__device__ __forceinline__ void count_range(const int32_t* __restrict__ idx, int64_t begin,
                                            int64_t end, int E, int32_t* cnt) {
    const int lane = threadIdx.x & 31;
    for (int64_t base = begin; base < end; base += kThreads) {
        bool bad = false;
        const int e = load_id(idx, base + threadIdx.x, end, E, bad);
        const uint32_t peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[e], __popc(peers));
    }
}

}  // namespace

// Per-chunk expert histogram: hist[c*E + e] = copies of e in chunk c.
__global__ void __launch_bounds__(kThreads) layout_hist_kernel(const int32_t* __restrict__ idx,
                                                               int64_t N, int E, int64_t chunk,
                                                               int32_t* __restrict__ hist) {
    extern __shared__ int32_t cnt_s[];
    for (int e = threadIdx.x; e < E; e += kThreads) cnt_s[e] = 0;
    __syncthreads();
    const int64_t begin = blockIdx.x * chunk;
    const int64_t end = min(N, begin + chunk);
    count_range(idx, begin, end, E, cnt_s);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) hist[blockIdx.x * (int64_t)E + e] = cnt_s[e];
}

// Rank kernel.  grid.x >= number of chunks C; CTAs with blockIdx.x >= C only
// help to mark unused receive rows.
__global__ void __launch_bounds__(kThreads) layout_rank_kernel(LayoutParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int32_t* base_s = reinterpret_cast<int32_t*>(smem_raw);    // [E] copies before this round
    int32_t* cnt_s = base_s + p.E;                               // [E] totals
    int32_t* off_s = cnt_s + p.E;                                // [E] exclusive offsets
    int32_t* wsum_s = off_s + p.E;                               // [32] scan scratch
    uint16_t* tab = reinterpret_cast<uint16_t*>(wsum_s + 32);    // [kWarps][E]
    __shared__ int bad_s;
    __shared__ int dropped_s;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int E = p.E;
    const int c = blockIdx.x;
    const int64_t chunk_begin = (int64_t)c * p.chunk;
    const int64_t chunk_end = min(p.N, chunk_begin + p.chunk);
    const bool ranks_chunk = c < p.num_chunks;

    if (tid == 0) { bad_s = 0; dropped_s = 0; }

    // 1. Per-expert totals and the copies before this chunk.
    if (p.hist != nullptr) {
        for (int e = tid; e < E; e += kThreads) {
            int32_t before = 0, total = 0;
            for (int cc = 0; cc < p.num_chunks; ++cc) {
                const int32_t h = p.hist[cc * (int64_t)E + e];
                total += h;
                if (cc < c) before += h;
            }
            base_s[e] = before;
            cnt_s[e] = total;
        }
    } else {
        for (int e = tid; e < E; e += kThreads) { base_s[e] = 0; cnt_s[e] = 0; }
        __syncthreads();
        const int64_t split = ranks_chunk ? chunk_begin : p.N;
        count_range(p.topk_idx, 0, split, E, base_s);
        __syncthreads();
        for (int e = tid; e < E; e += kThreads) cnt_s[e] = base_s[e];
        __syncthreads();
        count_range(p.topk_idx, split, p.N, E, cnt_s);
    }
    __syncthreads();

    // 2. Exclusive scan of the totals over experts (E <= kThreads).
    {
        const int32_t v = tid < E ? cnt_s[tid] : 0;
        int32_t incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) wsum_s[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t ws = wsum_s[lane];
            int32_t wincl = ws;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(kFull, wincl, d);
                if (lane >= d) wincl += o;
            }
            wsum_s[lane] = wincl - ws;   // exclusive prefix of warp sums
        }
        __syncthreads();
        if (tid < E) off_s[tid] = wsum_s[warp] + incl - v;
    }
    __syncthreads();
    const int32_t total = off_s[E - 1] + cnt_s[E - 1];

    if (c == 0) {
        for (int e = tid; e < E; e += kThreads) {
            p.counts[e] = cnt_s[e];
            p.offsets[e] = off_s[e];
        }
        if (tid == 0) p.offsets[E] = total;
        const int per = E / p.P;
        for (int q = tid; q < p.P; q += kThreads) {
            const int e0 = q * per, e1 = e0 + per - 1;
            p.part_counts[q] = off_s[e1] + cnt_s[e1] - off_s[e0];
            p.part_offsets[q] = off_s[e0];
        }
        if (tid == 0) p.part_offsets[p.P] = total;
    }

    // 3. Rank the entries of this chunk, one round of kThreads entries at a time.
    if (ranks_chunk) {
        for (int i = tid; i < kWarps * E; i += kThreads) tab[i] = 0;
        __syncthreads();
        for (int64_t rb = chunk_begin; rb < chunk_end; rb += kThreads) {
            const int64_t n = rb + tid;
            bool bad = false;
            const int e = load_id(p.topk_idx, n, chunk_end, E, bad);
            if (bad) bad_s = 1;
            const uint32_t peers = __match_any_sync(kFull, e);
            const int in_warp = __popc(peers & lanemask_lt());
            if (e >= 0 && lane == __ffs(peers) - 1) tab[warp * E + e] = (uint16_t)__popc(peers);
            __syncthreads();
            int32_t round_total = 0;
            for (int x = tid; x < E; x += kThreads) {   // scan each expert's column
                int32_t run = 0;
#pragma unroll 8
                for (int w = 0; w < kWarps; ++w) {
                    const int32_t cw = tab[w * E + x];
                    tab[w * E + x] = (uint16_t)run;
                    run += cw;
                }
                round_total = run;
            }
            __syncthreads();
            if (n < chunk_end) {
                int32_t slot = -1;
                if (e >= 0) {
                    const int32_t rank = base_s[e] + tab[warp * E + e] + in_warp;
                    if (p.mode == 0) {
                        slot = off_s[e] + rank;
                    } else if (rank < p.cap) {
                        slot = e * p.cap + rank;
                    } else {
                        dropped_s = 1;
                    }
                }
                p.slot_of[n] = slot;
                if (slot >= 0) {
                    const int32_t t = (int32_t)(n / p.k);
                    p.src_token[slot] = t;
                    p.src_k[slot] = (int32_t)(n - (int64_t)t * p.k);
                }
            }
            __syncthreads();
            for (int x = tid; x < E; x += kThreads) {
                base_s[x] += round_total;
#pragma unroll 8
                for (int w = 0; w < kWarps; ++w) tab[w * E + x] = 0;
            }
            __syncthreads();
        }
    }

    // 4. Rows that hold no copy get src_token = src_k = -1.
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    if (p.mode == 0) {
        for (int64_t r = total + (int64_t)c * kThreads + tid; r < p.R; r += stride) {
            p.src_token[r] = -1;
            p.src_k[r] = -1;
        }
    } else {
        for (int64_t r = (int64_t)c * kThreads + tid; r < p.R; r += stride) {
            const int e = (int)(r / p.cap);
            if ((int32_t)(r - (int64_t)e * p.cap) >= cnt_s[e]) {
                p.src_token[r] = -1;
                p.src_k[r] = -1;
            }
        }
    }

    __syncthreads();
    if (tid == 0 && p.err_flags != nullptr) {
        uint32_t f = (bad_s ? kErrBadExpert : 0u) | (dropped_s ? kErrCapacity : 0u);
        if (f) atomicOr(p.err_flags, f);
    }
}

// ------------------------------------------------------------------ host

int64_t layout_num_chunks(int64_t N) { return N <= 0 ? 1 : (N + kLayoutChunk - 1) / kLayoutChunk; }

bool layout_uses_workspace(int64_t N) { return N > kLayoutSmallN; }

size_t layout_workspace_bytes(int64_t N, int E) {
    return layout_uses_workspace(N) ? (size_t)layout_num_chunks(N) * (size_t)E * sizeof(int32_t) : 0;
}

size_t layout_rank_smem_bytes(int E) {
    return (size_t)3 * E * sizeof(int32_t) + 32 * sizeof(int32_t) + (size_t)kWarps * E * sizeof(uint16_t);
}

cudaError_t launch_layout(const LayoutParams& p_in, int num_sms, cudaStream_t stream) {
    LayoutParams p = p_in;
    p.chunk = kLayoutChunk;
    p.num_chunks = (int)layout_num_chunks(p.N);
    const size_t smem = layout_rank_smem_bytes(p.E);
    cudaError_t err = cudaFuncSetAttribute(layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    if (p.hist != nullptr) {
        layout_hist_kernel<<<p.num_chunks, kThreads, p.E * sizeof(int32_t), stream>>>(p.topk_idx, p.N, p.E,
                                                                                     p.chunk, p.hist);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    // Extra CTAs only mark unused rows; keep about 8K rows per CTA.
    int64_t fill_ctas = (p.R + 8191) / 8192;
    int64_t grid = p.num_chunks;
    if (fill_ctas > grid) grid = fill_ctas < num_sms ? fill_ctas : num_sms;
    if (grid < p.num_chunks) grid = p.num_chunks;
    layout_rank_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
