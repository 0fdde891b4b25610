// combine_src.cu -- the combine addressed from the expert side
// (ep_combine_src): the caller holds, per row of the expert-major buffer, the
// pair (token, top-k position) the row was dispatched from and the row's own
// weight -- the routing information that travels with each token in
// "Pipeline direct NVLink dispatch with triple-buffered prefetch" (Summary).
//
// The reduce must stay a gather in increasing j per token (the fp32 sum order
// of ep_combine), so the token-side map is rebuilt first: one kernel fills it
// with -1, then one thread per row scatters slot[t, j] = r and w[t, j] =
// row_w[r].  Pairs no row holds stay -1 and add nothing.  The gather itself is
// the TMA-staged combine kernel, reading y in place.  The inversion moves
// R * 12 bytes in and T * k * 8 out, small beside the k rows per token the
// gather reads.  The three kernels launch with programmatic serialization, so
// each one's launch overlaps the previous one's tail.
#include "ep_device.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    invert_src_kernel(const int32_t* __restrict__ src_token, const int32_t* __restrict__ src_k,
                      const float* __restrict__ row_w, int64_t R, int T, int k, int32_t* __restrict__ slot,
                      float* __restrict__ w, uint32_t* err_flags) {
    pdl_launch_dependents();
    pdl_wait();   // the map was filled by the previous kernel
    bool bad = false;
    for (int64_t r = (int64_t)blockIdx.x * kThreads + threadIdx.x; r < R; r += (int64_t)gridDim.x * kThreads) {
        const int32_t t = __ldg(src_token + r);
        if (t == -1) continue;
        const int32_t j = __ldg(src_k + r);
        if (t < 0 || t >= T || j < 0 || j >= k) {
            bad = true;
            continue;
        }
        const int64_t c = (int64_t)t * k + j;
        slot[c] = (int32_t)r;
        if (row_w != nullptr) w[c] = __ldg(row_w + r);
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && err_flags != nullptr)
        atomicOr(err_flags, kErrBadSlot);
}

// slot[i] = -1 for i < n (the pairs no row claims keep it).
__global__ void __launch_bounds__(kThreads) fill_map_kernel(int32_t* __restrict__ slot, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();   // the previous kernel of the stream may still read the map
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) slot[i] = -1;
}

}  // namespace

size_t combine_src_map_bytes(int64_t T, int k) { return ((size_t)T * k * 4 + 255) / 256 * 256; }

cudaError_t launch_combine_src(const CombineSrcParams& p, int num_sms, cudaStream_t stream) {
    if (p.base.T == 0) return cudaSuccess;
    int32_t* slot = static_cast<int32_t*>(p.workspace);
    float* w = reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + combine_src_map_bytes(p.base.T, p.base.k));
    const int64_t n = (int64_t)p.base.T * p.base.k;
    const int64_t cap = (int64_t)num_sms * 8;
    int64_t fill_blocks = (n + kThreads - 1) / kThreads;
    if (fill_blocks > cap) fill_blocks = cap;
    cudaError_t err = launch_kernel(true, fill_map_kernel, dim3((unsigned)fill_blocks), dim3(kThreads), 0, stream,
                                    slot, n);
    if (err != cudaSuccess) return err;
    if (p.base.R > 0) {
        int64_t blocks = (p.base.R + kThreads - 1) / kThreads;
        if (blocks > cap) blocks = cap;
        err = launch_kernel(true, invert_src_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p.src_token,
                            p.src_k, p.row_w, p.base.R, p.base.T, p.base.k, slot, w, p.base.err_flags);
        if (err != cudaSuccess) return err;
    }
    CombineParams c = p.base;
    c.slot_of = slot;
    c.topk_w = p.row_w != nullptr ? w : nullptr;
    return launch_combine(c, num_sms, stream);
}

}  // namespace ep
