// combine_src.cu -- the combine addressed from the expert side
// (ep_combine_src): the caller holds, per row of the expert-major buffer, the
// pair (token, top-k position) the row was dispatched from and the row's own
// weight -- the routing information that travels with each token in
// "Pipeline direct NVLink dispatch with triple-buffered prefetch" (Summary).
//
// The reduce must stay a gather in increasing j per token (the fp32 sum order
// of ep_combine), so the token-side map is rebuilt first: the workspace is
// filled with -1, then one thread per row scatters slot[t, j] = r and
// w[t, j] = row_w[r].  Pairs no row holds stay -1 and add nothing.  The
// gather itself is the TMA-staged combine kernel, reading y in place.  The
// inversion moves R * 12 bytes in and T * k * 8 out, small beside the k rows
// per token the gather reads.
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

}  // namespace

size_t combine_src_map_bytes(int64_t T, int k) { return ((size_t)T * k * 4 + 255) / 256 * 256; }

cudaError_t launch_combine_src(const CombineSrcParams& p, int num_sms, cudaStream_t stream) {
    if (p.base.T == 0) return cudaSuccess;
    int32_t* slot = static_cast<int32_t*>(p.workspace);
    float* w = reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + combine_src_map_bytes(p.base.T, p.base.k));
    cudaError_t err = cudaMemsetAsync(slot, 0xff, (size_t)p.base.T * p.base.k * sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
    if (p.base.R > 0) {
        int64_t blocks = (p.base.R + kThreads - 1) / kThreads;
        const int64_t cap = (int64_t)num_sms * 8;
        if (blocks > cap) blocks = cap;
        err = launch_kernel(false, invert_src_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p.src_token,
                            p.src_k, p.row_w, p.base.R, p.base.T, p.base.k, slot, w, p.base.err_flags);
        if (err != cudaSuccess) return err;
    }
    CombineParams c = p.base;
    c.slot_of = slot;
    c.topk_w = p.row_w != nullptr ? w : nullptr;
    return launch_combine(c, num_sms, stream);
}

}  // namespace ep
