// Exhaustive check of the fp8 quantiser's arithmetic against CUDA's IEEE
// division: for every finite bf16 amax >= 0 (0x0000..0x7F7F) the block
// scale from block_scale() must equal RN32(max(amax, 1e-4) / 448) computed
// with __fdiv_rn (then bumped to a power of two for UE8M0), and for every
// finite bf16 x the e4m3 code of quotient_rn(x, s, RN(1/s)) must equal the
// code of __fdiv_rn(x, s); where |x| <= amax (the values a block with that
// amax can hold) and |x/s| >= 2^-10 the two fp32 quotients must also be
// bit-identical.  Codes for |x| > amax are counted apart: a quantiser never
// divides a value larger than its block's amax, and there x * RN(1/s) can
// overflow.  Prints one line of counts per scale format; exits 0 once it ran.
#include <cmath>
#include <cstdint>
#include <cstdio>

#include "ep_device.cuh"

using namespace ep;

struct Counts {
    unsigned long long pairs, scale_mismatch, code_mismatch_in, code_mismatch_out, quotient_mismatch_in;
};

__device__ float bf16_value(uint32_t bits) { return __uint_as_float(bits << 16); }

__global__ void check(Counts* c, int ue8m0) {
    const uint32_t mb = blockIdx.x * blockDim.x + threadIdx.x;
    if (mb > 0x7F7Fu) return;
    const float m = bf16_value(mb);
    float s_ref = __fdiv_rn(fmaxf(m, 1e-4f), 448.0f);
    if (ue8m0) {
        uint32_t b = __float_as_uint(s_ref);
        if (b & 0x007fffffu) b = (b & 0x7f800000u) + 0x00800000u;
        s_ref = __uint_as_float(b);
    }
    const float s = block_scale(m, ue8m0 != 0, recip_448());
    if (blockIdx.y == 0 && __float_as_uint(s) != __float_as_uint(s_ref)) atomicAdd(&c->scale_mismatch, 1ull);
    const float rs = __frcp_rn(s);
    unsigned long long n = 0, cin = 0, cout = 0, qin = 0;
    for (uint32_t xb = blockIdx.y * 256u; xb < blockIdx.y * 256u + 256u; ++xb) {
        const float x = bf16_value(xb);
        if (!isfinite(x)) continue;
        const float qr = __fdiv_rn(x, s_ref);
        const float qn = quotient_rn(x, s, rs);
        const bool in = fabsf(x) <= m;
        const uint32_t cr = pack_e4m3x2(qr, 0.0f) & 0xffu, cn = pack_e4m3x2(qn, 0.0f) & 0xffu;
        ++n;
        if (cr != cn) {
            if (in) ++cin; else ++cout;
        }
        if (in && fabsf(qr) >= 0x1p-10f && __float_as_uint(qr) != __float_as_uint(qn)) ++qin;
    }
    atomicAdd(&c->pairs, n);
    if (cin) atomicAdd(&c->code_mismatch_in, cin);
    if (cout) atomicAdd(&c->code_mismatch_out, cout);
    if (qin) atomicAdd(&c->quotient_mismatch_in, qin);
}

int main() {
    Counts* d = nullptr;
    if (cudaMalloc(&d, sizeof(Counts)) != cudaSuccess) return 2;
    for (int ue8m0 = 0; ue8m0 < 2; ++ue8m0) {
        cudaMemset(d, 0, sizeof(Counts));
        check<<<dim3((0x7F7F + 1 + 255) / 256, 256), 256>>>(d, ue8m0);
        Counts h{};
        if (cudaMemcpy(&h, d, sizeof(Counts), cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
        printf("ue8m0=%d pairs=%llu scale_mismatch=%llu code_mismatch_in=%llu code_mismatch_out=%llu "
               "quotient_mismatch_in=%llu\n", ue8m0, h.pairs, h.scale_mismatch, h.code_mismatch_in,
               h.code_mismatch_out, h.quotient_mismatch_in);
    }
    const cudaError_t e = cudaGetLastError();
    printf("cuda=%s\n", cudaGetErrorString(e));
    cudaFree(d);
    return e == cudaSuccess ? 0 : 4;
}
