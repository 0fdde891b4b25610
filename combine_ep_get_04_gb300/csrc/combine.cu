// combine.cu -- weighted top-k reduce of expert outputs back to token order
// (ep_combine): out[t] = bf16( sum_j w[t,j] * y[slot_of[t,j]] ), fp32
// accumulation in increasing j, one rounding to bf16.
//
// Combine is the reverse of dispatch and is measured beside it in "Pipeline
// direct NVLink dispatch with triple-buffered prefetch" (DeepEP PR #693),
// Validation table.  It reads k rows per token and writes one, so it is a
// gather bound by HBM reads: each thread owns 16 bytes (8 channels) of one
// token, issues the k independent 16-byte row loads before it does any
// arithmetic, and stores one 16-byte vector.  No tensor cores: there is no
// contraction, only k multiply-adds per output element.
#include "ep_device.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;   // rows loaded before they are summed

struct Args {
    const uint4* y;
    const float* topk_w;
    const int32_t* slot_of;
    uint4* out;
    uint32_t* err_flags;
    int64_t R;       // rows of y
    int64_t total;   // T * H8
    int H8;          // H / 8
    int k;
};

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void accumulate(float (&acc)[8], float w, const uint4& v) {
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(w, bf16_lo(words[q])));
        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(w, bf16_hi(words[q])));
    }
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const Args a) {
    const int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (g >= a.total) return;
    const int64_t t = g / a.H8;
    const int c = (int)(g - t * a.H8);
    const int32_t* so = a.slot_of + t * a.k;
    const float* wt = a.topk_w + t * a.k;

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;

    for (int j0 = 0; j0 < a.k; j0 += kBatch) {
        int32_t s[kBatch];
        float w[kBatch];
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            s[u] = (j0 + u < a.k) ? __ldg(so + j0 + u) : -1;
            if (s[u] < -1 || s[u] >= a.R) {
                if (c == 0 && a.err_flags != nullptr) atomicOr(a.err_flags, kErrBadSlot);
                s[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (s[u] >= 0) {
                w[u] = __ldg(wt + j0 + u);
                v[u] = load_stream(a.y + (int64_t)s[u] * a.H8 + c);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (s[u] >= 0) accumulate(acc, w[u], v[u]);
        }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    a.out[g] = o;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    if (p.T == 0) return cudaSuccess;
    Args a{};
    a.y = static_cast<const uint4*>(p.y);
    a.topk_w = p.topk_w;
    a.slot_of = p.slot_of;
    a.out = static_cast<uint4*>(p.out);
    a.err_flags = p.err_flags;
    a.R = p.R;
    a.H8 = p.H / 8;
    a.k = p.k;
    a.total = (int64_t)p.T * a.H8;
    const int64_t grid = (a.total + kThreads - 1) / kThreads;
    combine_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
