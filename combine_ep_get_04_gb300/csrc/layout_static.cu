// layout_static.cu -- ep_get_layout_static: the layout computation with its
// scratch memory taken from a fixed array compiled into this library instead
// of a workspace the caller allocates.
//
// Why: some callers cannot allocate device memory at the point where they
// compute the layout -- for example code that works inside a fixed memory
// budget handed to it by a host framework, or a latency-critical path where a
// device allocation could stall the device.  This entry point lets them run
// the layout with only the input and output buffers they already own.
//
// Scratch: the per-chunk expert histogram (chunks of 1024 routing entries x E
// experts, 4 bytes each) lives in the file-scope array below.  Every GPU that
// loads this library holds it until the process exits.  Its device address is
// looked up once per device context, on the first call made while that
// context is current, and cached under the context's process-unique id: a
// context created later on the same device (after cudaDeviceReset, say)
// reloads the module, possibly at another address, and gets a fresh lookup.
// All calls share the array and it keeps the last call's contents;
// every entry a call reads is first written by the same call, so nothing has
// to be cleared.  Calls whose work overlaps on the GPU (different streams, or
// several host threads on one device) race on the array and must be ordered
// by the caller.
#include <cstdio>
#include <mutex>

#include <cuda.h>

#include "ep.h"
#include "ep_kernels.h"

namespace {

// 1 MiB: histogram rows for up to 262144 (chunk, expert) pairs, e.g. 2^20
// routing entries with 256 experts.
constexpr size_t kStaticScratchBytes = 1u << 20;

static __device__ __align__(256) int32_t g_layout_scratch[kStaticScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchEntry {
    unsigned long long ctx_id;   // 0: nothing cached
    int32_t* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

ep_status_t static_fail(ep_status_t st, const char* msg) {
    ep::record_last_error(msg);
    return st;
}

// Process-unique id of the calling thread's current context (cuCtxGetId,
// reached through the runtime's driver entry points, so that nothing links
// the driver library directly); 0 if there is no current context or the
// driver cannot tell, in which case nothing is cached.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_layout_scratch in the current device's current
// context: the cached one if it was looked up in this same context, else a
// fresh cudaGetSymbolAddress (checked), cached under the context's id.
ep_status_t scratch_for_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_fail(EP_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return static_fail(EP_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const unsigned long long id = current_context_id();
    if (id != 0 && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].ptr;
        return EP_OK;
    }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_layout_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
        g_scratch[dev] = ScratchEntry{};
        return static_fail(EP_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                         : "cudaGetSymbolAddress returned NULL");
    }
    // the lookup makes the device's primary context current if none was
    g_scratch[dev] = ScratchEntry{current_context_id(), static_cast<int32_t*>(ptr)};
    *out = static_cast<int32_t*>(ptr);
    return EP_OK;
}

}  // namespace

extern "C" {

ep_status_t ep_get_layout_static(const ep_shape_t* shape, const int32_t* topk_idx, int32_t* counts,
                                 int32_t* offsets, int32_t* part_counts, int32_t* part_offsets,
                                 int32_t* slot_of, int32_t* src_token, int32_t* src_k, uint32_t* err_flags,
                                 ep_stream_t stream) {
    const size_t need = ep_layout_workspace_bytes(shape);
    if (need == (size_t)-1) {
        // the shape is invalid: let the regular entry point report why
        return ep_get_layout(shape, topk_idx, counts, offsets, part_counts, part_offsets, slot_of, src_token,
                             src_k, nullptr, 0, err_flags, stream);
    }
    if (need > kStaticScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "this shape needs %zu bytes of layout scratch; the built-in array holds %zu "
                 "(use ep_get_layout with a caller-owned workspace)", need, kStaticScratchBytes);
        return static_fail(EP_ERR_UNSUPPORTED, msg);
    }
    int32_t* scratch = nullptr;
    if (need > 0) {
        const ep_status_t st = scratch_for_current_device(&scratch);
        if (st != EP_OK) return st;
    }
    return ep_get_layout(shape, topk_idx, counts, offsets, part_counts, part_offsets, slot_of, src_token, src_k,
                         scratch, need, err_flags, stream);
}

}  // extern "C"
