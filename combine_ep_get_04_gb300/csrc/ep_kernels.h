// ep_kernels.h -- host-side launchers of the dispatch / combine kernels and
// their parameter blocks (internal to the library; the public C ABI is
// include/ep.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ep {

// Launches `kern`; with pdl, under programmatic stream serialization: it may
// begin while the previous kernel of the stream finishes, and waits
// (pdl_wait) before it writes global memory or reads what that kernel may
// write (before the wait it only prefetches into L2, and reads such memory
// only as an address hint for a prefetch).  Used for latency-sized grids
// (about one unit of work per CTA), where the launch gap is a large share of
// the time; large persistent grids launch normally.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Sets the text ep_last_error() returns on the calling thread.
void record_last_error(const char* msg);

// ----------------------------------------------------------------- layout

constexpr int64_t kLayoutChunk = 1024;   // entries ranked by one CTA
constexpr int64_t kLayoutSmallN = 4096;  // up to this many entries: one launch, no workspace

struct LayoutParams {
    const int32_t* topk_idx;
    int32_t* counts;
    int32_t* offsets;
    int32_t* part_counts;
    int32_t* part_offsets;
    int32_t* slot_of;
    int32_t* src_token;
    int32_t* src_k;
    int32_t* hist;        // [num_chunks][E] workspace, or nullptr for the one-launch path
    uint32_t* err_flags;  // may be nullptr
    int64_t N;            // T * k
    int64_t R;            // receive rows
    int64_t chunk;        // set by launch_layout
    int num_chunks;       // set by launch_layout
    int E, P, k, mode, cap;
};

int64_t layout_num_chunks(int64_t N);
bool layout_uses_workspace(int64_t N);
size_t layout_workspace_bytes(int64_t N, int E);
size_t layout_rank_smem_bytes(int E);
cudaError_t launch_layout(const LayoutParams& p, int num_sms, cudaStream_t stream);

// --------------------------------------------------------------- dispatch

struct DispatchParams {
    const void* x;          // bf16 [T, H]
    const float* topk_w;    // [T, k] or nullptr
    const int32_t* slot_of; // [T, k]
    void* recv;             // bf16 or e4m3 [R, H]
    void* recv_scales;      // [R, H/128] f32, or u8 exponents with ue8m0 (fp8)
    float* recv_w;          // [R] or nullptr
    uint32_t* err_flags;    // may be nullptr
    int64_t R;              // receive rows
    int T, H, k;
    int ue8m0;              // power-of-two scales stored as exponent bytes
};

cudaError_t launch_dispatch_bf16(const DispatchParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_dispatch_fp8(const DispatchParams& p, int num_sms, cudaStream_t stream);

// ------------------------------------------------ layout + dispatch fused

constexpr int64_t kFusedMaxN = 2048;   // routing entries: every CTA counts them all
constexpr int64_t kFusedMaxT = 2048;

struct FusedLaunch {
    const int32_t* topk_idx;
    const void* x;
    const float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* part_counts;
    int32_t* part_offsets;
    int32_t* slot_of;
    int32_t* src_token;
    int32_t* src_k;
    void* recv;
    void* recv_scales;
    float* recv_w;
    uint32_t* err_flags;
    int64_t R;
    int T, H, E, k, P, mode, cap, fp8, ue8m0;
};

bool fused_layout_dispatch_fits(int64_t N, int64_t T, int E);
cudaError_t launch_layout_dispatch(const FusedLaunch& f, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- combine

struct CombineParams {
    const void* y;          // bf16 [R, H], or e4m3 [R, H] with fp8
    const void* y_scales;   // fp8: [R, H/128] f32, or u8 exponents with ue8m0
    int fp8, ue8m0;
    const float* topk_w;    // [T, k]
    const int32_t* slot_of; // [T, k]
    void* out;              // bf16 [T, H]
    uint32_t* err_flags;    // may be nullptr
    int64_t R;              // rows of y
    int T, H, k;
};

cudaError_t launch_combine(const CombineParams& p, int num_sms, cudaStream_t stream);

// The combine addressed by the expert-side maps: base carries y, scales,
// out, err_flags and the shape (its slot_of / topk_w are ignored).
struct CombineSrcParams {
    CombineParams base;
    const float* row_w;       // [R] or nullptr (unweighted)
    const int32_t* src_token; // [R], -1 = no copy
    const int32_t* src_k;     // [R]
    void* workspace;          // combine_src_workspace_bytes(T, k) bytes
};

// Bytes of one [T, k] map rounded up to 256; the workspace holds two.
size_t combine_src_map_bytes(int64_t T, int k);
inline size_t combine_src_workspace_bytes(int64_t T, int k) { return 2 * combine_src_map_bytes(T, k); }

cudaError_t launch_combine_src(const CombineSrcParams& p, int num_sms, cudaStream_t stream);

}  // namespace ep
