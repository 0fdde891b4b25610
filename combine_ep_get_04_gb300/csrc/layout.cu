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
//  * The flattened ids are cut into chunks of 1024 entries, one CTA each, one
//    entry per thread.
//  * Every CTA needs, per expert, the copies before its chunk (its base) and
//    the total over all chunks (for the offsets).  Small inputs: each CTA
//    counts them itself from topk_idx (one launch, no workspace).  Large
//    inputs: a histogram kernel writes per-chunk counts [C][E] to the
//    workspace and the rank kernel sums each expert's column, several threads
//    per column with independent loads in flight.
//  * Inside a chunk, each warp of 32 consecutive entries ranks equal ids with
//    __match_any_sync; a [32 warps][E] table of per-warp counts, scanned down
//    each expert's column, gives the rank of every entry.  Ids are loaded once
//    and matched once.
//  * Receive rows that hold no copy are marked -1 per expert range (no
//    division per row).
// All index arithmetic is 32-bit: the host rejects T*k or R >= 2^31.
#include "ep_device.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kThreads = 1024;          // one entry per thread
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxRounds = (int)(kLayoutSmallN / kThreads);
static_assert(kLayoutChunk == kThreads, "one chunk entry per thread");

}  // namespace

// Per-chunk expert histogram: hist[c*E + e] = copies of e in chunk c (one
// entry per thread, warp-aggregated shared atomics).
__global__ void __launch_bounds__(kThreads) layout_hist_kernel(const int32_t* __restrict__ idx, int N, int E,
                                                               int32_t* __restrict__ hist) {
    extern __shared__ int32_t cnt_s[];
    pdl_launch_dependents();
    for (int e = threadIdx.x; e < E; e += kThreads) cnt_s[e] = 0;
    pdl_wait();
    const int n = blockIdx.x * kThreads + threadIdx.x;
    int e = -1;
    if (n < N) {
        e = __ldg(idx + n);
        if (e < -1 || e >= E) e = -1;
    }
    __syncthreads();
    const uint32_t peers = __match_any_sync(kFull, e);
    if (e >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&cnt_s[e], __popc(peers));
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += kThreads) hist[blockIdx.x * E + x] = cnt_s[x];
}

// Rank kernel.  grid.x >= number of chunks C (one chunk of kThreads entries
// per ranking CTA); CTAs with blockIdx.x >= C only help to mark unused rows.
__global__ void __launch_bounds__(kThreads) layout_rank_kernel(LayoutParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int32_t* base_s = reinterpret_cast<int32_t*>(smem_raw);    // [E] copies before this chunk
    int32_t* cnt_s = base_s + p.E;                               // [E] totals
    int32_t* off_s = cnt_s + p.E;                                // [E] exclusive offsets
    int32_t* wsum_s = off_s + p.E;                               // [32] scan scratch
    uint16_t* tab = reinterpret_cast<uint16_t*>(wsum_s + 32);    // [kWarps][E]
    __shared__ int flags_s;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int E = p.E;
    const int c = blockIdx.x;
    const int N = (int)p.N;
    const bool ranks_chunk = c < p.num_chunks;

    pdl_launch_dependents();
    if (tid == 0) flags_s = 0;
    for (int e = tid; e < E; e += kThreads) { base_s[e] = 0; cnt_s[e] = 0; }
    if (ranks_chunk) {
        for (int i = tid; i < kWarps * E; i += kThreads) tab[i] = 0;
    }
    __syncthreads();
    pdl_wait();

    // 1. This thread's entry of the chunk (my_e, its rank inside the warp),
    //    the per-warp counts of the chunk (tab), the totals and the copies
    //    before the chunk.
    int my_e = -1, my_in_warp = 0;
    bool bad = false;
    const int my_n = c * kThreads + tid;
    if (p.hist == nullptr) {
        // Small input (N <= kLayoutSmallN): every CTA reads all ids, round u
        // covering entries [u*kThreads, (u+1)*kThreads).
        int e[kMaxRounds];
#pragma unroll
        for (int u = 0; u < kMaxRounds; ++u) {
            const int n = u * kThreads + tid;
            e[u] = -1;
            if (n < N) {
                e[u] = __ldg(p.topk_idx + n);
                if (e[u] < -1 || e[u] >= E) {
                    if (u == c) bad = true;
                    e[u] = -1;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kMaxRounds; ++u) {
            if (u * kThreads >= N) break;
            const uint32_t peers = __match_any_sync(kFull, e[u]);
            if (e[u] >= 0 && lane == __ffs(peers) - 1) {
                const int cnt = __popc(peers);
                atomicAdd(&cnt_s[e[u]], cnt);
                if (u < c) atomicAdd(&base_s[e[u]], cnt);
                if (u == c) tab[warp * E + e[u]] = (uint16_t)cnt;
            }
            if (u == c) {
                my_e = e[u];
                my_in_warp = __popc(peers & lanemask_lt());
            }
        }
    } else {
        // This thread's entry is loaded first; it is used only after the
        // column sums below, so both latencies overlap.
        if (ranks_chunk && my_n < N) my_e = __ldg(p.topk_idx + my_n);
        // tpe threads per expert column of the histogram, each summing every
        // tpe-th chunk with eight independent loads in flight.  Consecutive
        // threads take consecutive experts of one chunk, so each warp load
        // reads one or two whole lines of the table every CTA reads.
        const int tpe = max(1, kThreads / E);
        const int e = tid % E, sub = tid / E;
        if (sub < tpe) {
            int32_t before = 0, total = 0;
            int cc = sub;
            for (; cc + 7 * tpe < p.num_chunks; cc += 8 * tpe) {
                int32_t h[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) h[u] = __ldg(p.hist + (cc + u * tpe) * E + e);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    total += h[u];
                    if (cc + u * tpe < c) before += h[u];
                }
            }
            for (; cc < p.num_chunks; cc += tpe) {
                const int32_t h = __ldg(p.hist + cc * E + e);
                total += h;
                if (cc < c) before += h;
            }
            if (before) atomicAdd(&base_s[e], before);
            if (total) atomicAdd(&cnt_s[e], total);
        }
        if (ranks_chunk) {
            if (my_e < -1 || my_e >= E) {
                bad = true;
                my_e = -1;
            }
            const uint32_t peers = __match_any_sync(kFull, my_e);
            my_in_warp = __popc(peers & lanemask_lt());
            if (my_e >= 0 && lane == __ffs(peers) - 1) tab[warp * E + my_e] = (uint16_t)__popc(peers);
        }
    }
    if (bad) atomicOr(&flags_s, (int)kErrBadExpert);
    __syncthreads();

    // 2. Exclusive scan of the totals over experts (E <= kThreads), and the
    //    exclusive scan of the per-warp counts down each expert's column.
    const int32_t v = tid < E ? cnt_s[tid] : 0;
    int32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) wsum_s[warp] = incl;
    if (ranks_chunk && tid < E) {   // eight independent loads at a time
        int32_t run = 0;
#pragma unroll
        for (int w0 = 0; w0 < kWarps; w0 += 8) {
            int32_t col[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) col[w] = tab[(w0 + w) * E + tid];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                tab[(w0 + w) * E + tid] = (uint16_t)run;
                run += col[w];
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        const int32_t ws = wsum_s[lane];
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
    __syncthreads();
    const int32_t total = off_s[E - 1] + cnt_s[E - 1];

    // 3. Outputs.
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

    if (ranks_chunk && my_n < N) {
        int32_t slot = -1;
        if (my_e >= 0) {
            const int32_t rank = base_s[my_e] + tab[warp * E + my_e] + my_in_warp;
            if (p.mode == 0) {
                slot = off_s[my_e] + rank;
            } else if (rank < p.cap) {
                slot = my_e * p.cap + rank;
            } else {
                atomicOr(&flags_s, (int)kErrCapacity);
            }
        }
        p.slot_of[my_n] = slot;
        if (slot >= 0) {
            const int t = my_n / p.k;
            p.src_token[slot] = t;
            p.src_k[slot] = my_n - t * p.k;
        }
    }

    // Rows that hold no copy get src_token = src_k = -1 (disjoint from the
    // rows written above, so no ordering is needed).
    {
        const int gw = c * kWarps + warp;             // this warp's index in the grid
        const int nw = gridDim.x * kWarps;
        if (p.mode == 0) {
            for (int r = total + gw * 32 + lane; r < (int)p.R; r += nw * 32) {
                p.src_token[r] = -1;
                p.src_k[r] = -1;
            }
        } else {
            for (int e = gw; e < E; e += nw) {
                const int row0 = e * p.cap;
                for (int r = min(cnt_s[e], p.cap) + lane; r < p.cap; r += 32) {
                    p.src_token[row0 + r] = -1;
                    p.src_k[row0 + r] = -1;
                }
            }
        }
    }

    __syncthreads();
    if (tid == 0 && p.err_flags != nullptr && flags_s) atomicOr(p.err_flags, (uint32_t)flags_s);
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
        err = launch_kernel(false, layout_hist_kernel, dim3(p.num_chunks), dim3(kThreads), p.E * sizeof(int32_t), stream,
                         p.topk_idx, (int)p.N, p.E, p.hist);
        if (err != cudaSuccess) return err;
    }
    // In capacity mode the unused rows are marked per expert; spread that over
    // up to 8 CTAs (about 8K rows each) beyond the ranking ones.
    const int64_t unused_rows = p.mode == 0 ? 0 : p.R;
    int64_t grid = p.num_chunks;
    const int64_t fill_ctas = (unused_rows + 8191) / 8192;
    if (fill_ctas > grid) grid = fill_ctas < 8 ? fill_ctas : 8;
    if (grid < p.num_chunks) grid = p.num_chunks;
    (void)num_sms;
    // The rank kernel is latency-sized (about one CTA per 1024 ids): let it
    // start while the histogram kernel (or the caller's previous kernel)
    // finishes.  Behind the histogram kernel it reserves more than half of
    // an SM's shared memory, so that its early-started CTAs take one SM each
    // instead of stacking two on the SMs that free up first (measured on the
    // group-limited workload: layout + dispatch 185.5 -> 183.4 us back to
    // back).
    size_t smem_launch = smem;
    if (p.hist != nullptr) {
        int dev = 0, smem_sm = 0;
        err = cudaGetDevice(&dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (err != cudaSuccess) return err;
        if (smem_launch < (size_t)smem_sm / 2 + 1024) smem_launch = (size_t)smem_sm / 2 + 1024;
        err = cudaFuncSetAttribute(layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_launch);
        if (err != cudaSuccess) return err;
    }
    return launch_kernel(true, layout_rank_kernel, dim3((unsigned)grid), dim3(kThreads), smem_launch, stream, p);
}

}  // namespace ep
