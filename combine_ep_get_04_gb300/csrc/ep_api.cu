// ep_api.cu -- the C ABI declared in include/ep.h: host-side argument checks,
// launch-shape choice and error reporting.  Every step of the work runs in
// the kernels of layout.cu, dispatch.cu and combine.cu on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "ep.h"
#include "ep_kernels.h"

namespace {

thread_local std::string g_last_error;

ep_status_t fail(ep_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ep_status_t ok() { return EP_OK; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the shape; returns EP_OK or a failure with the reason recorded.
ep_status_t check_shape(const ep_shape_t* s) {
    if (s == nullptr) return fail(EP_ERR_INVALID_ARG, "shape is NULL");
    if (s->T < 0) return fail(EP_ERR_INVALID_ARG, "T = %d < 0", s->T);
    if (s->H <= 0 || s->H % 8 != 0) return fail(EP_ERR_INVALID_ARG, "H = %d must be a positive multiple of 8", s->H);
    if (s->E < 1) return fail(EP_ERR_INVALID_ARG, "E = %d < 1", s->E);
    if (s->E > EP_MAX_EXPERTS) return fail(EP_ERR_UNSUPPORTED, "E = %d > %d", s->E, EP_MAX_EXPERTS);
    if (s->k < 1 || s->k > s->E) return fail(EP_ERR_INVALID_ARG, "k = %d must be in [1, E = %d]", s->k, s->E);
    if (s->k > EP_MAX_TOPK) return fail(EP_ERR_UNSUPPORTED, "k = %d > %d", s->k, EP_MAX_TOPK);
    if (s->num_partitions < 1 || s->E % s->num_partitions != 0)
        return fail(EP_ERR_INVALID_ARG, "num_partitions = %d must divide E = %d", s->num_partitions, s->E);
    if (s->mode != EP_LAYOUT_PACKED && s->mode != EP_LAYOUT_CAPACITY)
        return fail(EP_ERR_INVALID_ARG, "mode = %d is not a layout mode", s->mode);
    if (s->mode == EP_LAYOUT_CAPACITY && s->capacity < 1)
        return fail(EP_ERR_INVALID_ARG, "capacity = %d < 1 in capacity mode", s->capacity);
    const int64_t N = (int64_t)s->T * s->k;
    const int64_t R = s->mode == EP_LAYOUT_PACKED ? N : (int64_t)s->E * s->capacity;
    if (N > INT32_MAX || R > INT32_MAX)
        return fail(EP_ERR_UNSUPPORTED, "T*k = %lld or R = %lld exceeds 2^31-1", (long long)N, (long long)R);
    return ok();
}

int64_t rows_of(const ep_shape_t* s) {
    return s->mode == EP_LAYOUT_PACKED ? (int64_t)s->T * s->k : (int64_t)s->E * s->capacity;
}

// The current device must be an sm_103 part (the only code this library holds).
ep_status_t device_info(int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(EP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(EP_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3)
        return fail(EP_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library holds sm_103a code only", dev, major,
                    minor);
    return ok();
}

ep_status_t launched(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(EP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

namespace ep {
void record_last_error(const char* msg) { g_last_error = msg; }
}  // namespace ep

extern "C" {

int32_t ep_abi_version(void) { return 101; }

const char* ep_status_string(ep_status_t st) {
    switch (st) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_UNSUPPORTED: return "unsupported";
        case EP_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char* ep_status_str(ep_status_t st) { return ep_status_string(st); }

const char* ep_last_error(void) { return g_last_error.c_str(); }

int64_t ep_recv_rows(const ep_shape_t* shape) {
    if (check_shape(shape) != EP_OK) return -1;
    return rows_of(shape);
}

size_t ep_layout_workspace_bytes(const ep_shape_t* shape) {
    if (check_shape(shape) != EP_OK) return (size_t)-1;
    return ep::layout_workspace_bytes((int64_t)shape->T * shape->k, shape->E);
}

ep_status_t ep_get_layout(const ep_shape_t* shape, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                          int32_t* part_counts, int32_t* part_offsets, int32_t* slot_of, int32_t* src_token,
                          int32_t* src_k, void* workspace, size_t workspace_bytes, uint32_t* err_flags,
                          ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    const int64_t N = (int64_t)shape->T * shape->k;
    const int64_t R = rows_of(shape);
    if (N > 0 && (topk_idx == nullptr || slot_of == nullptr))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / slot_of is NULL");
    if (counts == nullptr || offsets == nullptr || part_counts == nullptr || part_offsets == nullptr)
        return fail(EP_ERR_INVALID_ARG, "counts / offsets / part_counts / part_offsets is NULL");
    if (R > 0 && (src_token == nullptr || src_k == nullptr))
        return fail(EP_ERR_INVALID_ARG, "src_token / src_k is NULL");
    const size_t need = ep::layout_workspace_bytes(N, shape->E);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(EP_ERR_INVALID_ARG, "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 3u))
        return fail(EP_ERR_INVALID_ARG, "workspace is not 4-byte aligned");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::LayoutParams p{};
    p.topk_idx = topk_idx;
    p.counts = counts;
    p.offsets = offsets;
    p.part_counts = part_counts;
    p.part_offsets = part_offsets;
    p.slot_of = slot_of;
    p.src_token = src_token;
    p.src_k = src_k;
    p.hist = need > 0 ? static_cast<int32_t*>(workspace) : nullptr;
    p.err_flags = err_flags;
    p.N = N;
    p.R = R;
    p.E = shape->E;
    p.P = shape->num_partitions;
    p.k = shape->k;
    p.mode = shape->mode;
    p.cap = shape->capacity;
    return launched(ep::launch_layout(p, num_sms, reinterpret_cast<cudaStream_t>(stream)), "layout launch");
}

ep_status_t ep_dispatch(const ep_shape_t* shape, const void* x, const float* topk_w, const int32_t* slot_of,
                        int32_t payload, void* recv, void* recv_scales, float* recv_w, uint32_t* err_flags,
                        ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    if (payload != EP_PAYLOAD_BF16 && payload != EP_PAYLOAD_FP8_E4M3 && payload != EP_PAYLOAD_FP8_E4M3_UE8M0)
        return fail(EP_ERR_INVALID_ARG, "payload = %d is not a payload format", payload);
    const bool fp8 = payload != EP_PAYLOAD_BF16;
    const bool ue8m0 = payload == EP_PAYLOAD_FP8_E4M3_UE8M0;
    if (fp8 && shape->H % 128 != 0) return fail(EP_ERR_INVALID_ARG, "fp8 payload needs H %% 128 == 0 (H = %d)", shape->H);
    if (shape->T == 0) return ok();
    if (x == nullptr || slot_of == nullptr || recv == nullptr)
        return fail(EP_ERR_INVALID_ARG, "x / slot_of / recv is NULL");
    if (!aligned16(x) || !aligned16(recv)) return fail(EP_ERR_INVALID_ARG, "x and recv must be 16-byte aligned");
    if (fp8 && (recv_scales == nullptr || (!ue8m0 && !aligned16(recv_scales))))
        return fail(EP_ERR_INVALID_ARG, "fp8 payload needs recv_scales (16-byte aligned for f32 scales)");
    if (recv_w != nullptr && topk_w == nullptr) return fail(EP_ERR_INVALID_ARG, "recv_w needs topk_w");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::DispatchParams p{};
    p.x = x;
    p.topk_w = topk_w;
    p.slot_of = slot_of;
    p.recv = recv;
    p.recv_scales = recv_scales;
    p.ue8m0 = ue8m0 ? 1 : 0;
    p.recv_w = recv_w;
    p.err_flags = err_flags;
    p.R = rows_of(shape);
    p.T = shape->T;
    p.H = shape->H;
    p.k = shape->k;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return launched(fp8 ? ep::launch_dispatch_fp8(p, num_sms, s) : ep::launch_dispatch_bf16(p, num_sms, s),
                    "dispatch launch");
}

ep_status_t ep_layout_dispatch(const ep_shape_t* shape, const int32_t* topk_idx, const void* x,
                               const float* topk_w, int32_t payload, int32_t* counts, int32_t* offsets,
                               int32_t* part_counts, int32_t* part_offsets, int32_t* slot_of, int32_t* src_token,
                               int32_t* src_k, void* recv, void* recv_scales, float* recv_w, void* workspace,
                               size_t workspace_bytes, uint32_t* err_flags, ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    const int64_t N = (int64_t)shape->T * shape->k;
    if (!ep::fused_layout_dispatch_fits(N, shape->T, shape->E) || shape->T == 0) {
        st = ep_get_layout(shape, topk_idx, counts, offsets, part_counts, part_offsets, slot_of, src_token, src_k,
                           workspace, workspace_bytes, err_flags, stream);
        if (st != EP_OK) return st;
        return ep_dispatch(shape, x, topk_w, slot_of, payload, recv, recv_scales, recv_w, err_flags, stream);
    }
    // The same checks as ep_get_layout and ep_dispatch, before anything is launched.
    if (payload != EP_PAYLOAD_BF16 && payload != EP_PAYLOAD_FP8_E4M3 && payload != EP_PAYLOAD_FP8_E4M3_UE8M0)
        return fail(EP_ERR_INVALID_ARG, "payload = %d is not a payload format", payload);
    const bool fp8 = payload != EP_PAYLOAD_BF16;
    const bool ue8m0 = payload == EP_PAYLOAD_FP8_E4M3_UE8M0;
    if (fp8 && shape->H % 128 != 0) return fail(EP_ERR_INVALID_ARG, "fp8 payload needs H %% 128 == 0 (H = %d)", shape->H);
    if (topk_idx == nullptr || slot_of == nullptr || x == nullptr || recv == nullptr)
        return fail(EP_ERR_INVALID_ARG, "topk_idx / slot_of / x / recv is NULL");
    if (counts == nullptr || offsets == nullptr || part_counts == nullptr || part_offsets == nullptr ||
        src_token == nullptr || src_k == nullptr)
        return fail(EP_ERR_INVALID_ARG, "counts / offsets / part_counts / part_offsets / src_token / src_k is NULL");
    if (!aligned16(x) || !aligned16(recv)) return fail(EP_ERR_INVALID_ARG, "x and recv must be 16-byte aligned");
    if (fp8 && (recv_scales == nullptr || (!ue8m0 && !aligned16(recv_scales))))
        return fail(EP_ERR_INVALID_ARG, "fp8 payload needs recv_scales (16-byte aligned for f32 scales)");
    if (recv_w != nullptr && topk_w == nullptr) return fail(EP_ERR_INVALID_ARG, "recv_w needs topk_w");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::FusedLaunch f{};
    f.topk_idx = topk_idx;
    f.x = x;
    f.topk_w = topk_w;
    f.counts = counts;
    f.offsets = offsets;
    f.part_counts = part_counts;
    f.part_offsets = part_offsets;
    f.slot_of = slot_of;
    f.src_token = src_token;
    f.src_k = src_k;
    f.recv = recv;
    f.recv_scales = recv_scales;
    f.recv_w = recv_w;
    f.err_flags = err_flags;
    f.R = rows_of(shape);
    f.T = shape->T;
    f.H = shape->H;
    f.E = shape->E;
    f.k = shape->k;
    f.P = shape->num_partitions;
    f.mode = shape->mode;
    f.cap = shape->capacity;
    f.fp8 = fp8 ? 1 : 0;
    f.ue8m0 = ue8m0 ? 1 : 0;
    return launched(ep::launch_layout_dispatch(f, num_sms, reinterpret_cast<cudaStream_t>(stream)),
                    "layout+dispatch launch");
}

ep_status_t ep_combine(const ep_shape_t* shape, const void* y, const float* topk_w, const int32_t* slot_of,
                       void* out, uint32_t* err_flags, ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    if (shape->T == 0) return ok();
    if (y == nullptr || slot_of == nullptr || out == nullptr)
        return fail(EP_ERR_INVALID_ARG, "y / slot_of / out is NULL");
    if (!aligned16(y) || !aligned16(out)) return fail(EP_ERR_INVALID_ARG, "y and out must be 16-byte aligned");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::CombineParams p{};
    p.y = y;
    p.topk_w = topk_w;
    p.slot_of = slot_of;
    p.out = out;
    p.err_flags = err_flags;
    p.R = rows_of(shape);
    p.T = shape->T;
    p.H = shape->H;
    p.k = shape->k;
    return launched(ep::launch_combine(p, num_sms, reinterpret_cast<cudaStream_t>(stream)), "combine launch");
}

ep_status_t ep_combine_fp8(const ep_shape_t* shape, const void* y, const void* y_scales, int32_t payload,
                           const float* topk_w, const int32_t* slot_of, void* out, uint32_t* err_flags,
                           ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    if (payload != EP_PAYLOAD_FP8_E4M3 && payload != EP_PAYLOAD_FP8_E4M3_UE8M0)
        return fail(EP_ERR_INVALID_ARG, "payload = %d is not an fp8 payload format", payload);
    if (shape->H % 128 != 0) return fail(EP_ERR_INVALID_ARG, "fp8 expert outputs need H %% 128 == 0 (H = %d)", shape->H);
    if (shape->T == 0) return ok();
    const bool ue8m0 = payload == EP_PAYLOAD_FP8_E4M3_UE8M0;
    if (y == nullptr || y_scales == nullptr || slot_of == nullptr || out == nullptr)
        return fail(EP_ERR_INVALID_ARG, "y / y_scales / slot_of / out is NULL");
    if (!aligned16(y) || !aligned16(out)) return fail(EP_ERR_INVALID_ARG, "y and out must be 16-byte aligned");
    if (!ue8m0 && (reinterpret_cast<uintptr_t>(y_scales) & 3u))
        return fail(EP_ERR_INVALID_ARG, "f32 y_scales must be 4-byte aligned");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::CombineParams p{};
    p.y = y;
    p.y_scales = y_scales;
    p.fp8 = 1;
    p.ue8m0 = ue8m0 ? 1 : 0;
    p.topk_w = topk_w;
    p.slot_of = slot_of;
    p.out = out;
    p.err_flags = err_flags;
    p.R = rows_of(shape);
    p.T = shape->T;
    p.H = shape->H;
    p.k = shape->k;
    return launched(ep::launch_combine(p, num_sms, reinterpret_cast<cudaStream_t>(stream)), "combine launch");
}

size_t ep_combine_src_workspace_bytes(const ep_shape_t* shape) {
    if (check_shape(shape) != EP_OK) return 0;
    return ep::combine_src_workspace_bytes(shape->T, shape->k);
}

ep_status_t ep_combine_src(const ep_shape_t* shape, const void* y, const void* y_scales, int32_t payload,
                           const float* row_w, const int32_t* src_token, const int32_t* src_k, void* out,
                           void* workspace, size_t workspace_bytes, uint32_t* err_flags, ep_stream_t stream) {
    ep_status_t st = check_shape(shape);
    if (st != EP_OK) return st;
    if (payload != EP_PAYLOAD_BF16 && payload != EP_PAYLOAD_FP8_E4M3 && payload != EP_PAYLOAD_FP8_E4M3_UE8M0)
        return fail(EP_ERR_INVALID_ARG, "payload = %d is not a payload format", payload);
    const bool fp8 = payload != EP_PAYLOAD_BF16;
    const bool ue8m0 = payload == EP_PAYLOAD_FP8_E4M3_UE8M0;
    if (fp8 && shape->H % 128 != 0)
        return fail(EP_ERR_INVALID_ARG, "fp8 expert outputs need H %% 128 == 0 (H = %d)", shape->H);
    if (shape->T == 0) return ok();
    if (y == nullptr || out == nullptr || workspace == nullptr)
        return fail(EP_ERR_INVALID_ARG, "y / out / workspace is NULL");
    const int64_t R = rows_of(shape);
    if (R > 0 && (src_token == nullptr || src_k == nullptr))
        return fail(EP_ERR_INVALID_ARG, "src_token / src_k is NULL");
    if (fp8 && y_scales == nullptr) return fail(EP_ERR_INVALID_ARG, "fp8 expert outputs need y_scales");
    if (!aligned16(y) || !aligned16(out)) return fail(EP_ERR_INVALID_ARG, "y and out must be 16-byte aligned");
    if (fp8 && !ue8m0 && (reinterpret_cast<uintptr_t>(y_scales) & 3u))
        return fail(EP_ERR_INVALID_ARG, "f32 y_scales must be 4-byte aligned");
    const size_t need = ep::combine_src_workspace_bytes(shape->T, shape->k);
    if (workspace_bytes < need)
        return fail(EP_ERR_INVALID_ARG, "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 3u) return fail(EP_ERR_INVALID_ARG, "workspace is not 4-byte aligned");
    int num_sms = 0;
    st = device_info(&num_sms);
    if (st != EP_OK) return st;

    ep::CombineSrcParams p{};
    p.base.y = y;
    p.base.y_scales = fp8 ? y_scales : nullptr;
    p.base.fp8 = fp8 ? 1 : 0;
    p.base.ue8m0 = ue8m0 ? 1 : 0;
    p.base.out = out;
    p.base.err_flags = err_flags;
    p.base.R = R;
    p.base.T = shape->T;
    p.base.H = shape->H;
    p.base.k = shape->k;
    p.row_w = row_w;
    p.src_token = src_token;
    p.src_k = src_k;
    p.workspace = workspace;
    return launched(ep::launch_combine_src(p, num_sms, reinterpret_cast<cudaStream_t>(stream)), "combine_src launch");
}

}  // extern "C"
