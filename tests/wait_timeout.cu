// The bounded mbarrier wait every kernel of the library uses (mbar_wait in
// ep_device.cuh), made to run out on the GPU without a fault: one thread arms
// an mbarrier for 16 bytes that no copy ever delivers, waits, and on timeout
// ORs the library's timeout bit into a flag word and returns.  Then a real
// bulk copy is waited for (it must complete, no flag), and a plain kernel runs
// on the same context.  Prints one line; exit code 0 once all three ran.
#include <cstdint>
#include <cstdio>

#include "ep_device.cuh"

using namespace ep;

__global__ void never_delivered(uint32_t* flags, unsigned long long* waited_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, 16);      // no copy will bring these bytes
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait(&bar, 0);
        *waited_ns = global_timer_ns() - t0;
        if (!ok) atomicOr(flags, kErrTimeout);
    }
}

__global__ void delivered(const uint4* src, uint32_t* flags, uint4* out) {
    __shared__ __align__(128) uint4 buf[8];
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, sizeof(buf));
        bulk_load(buf, src, sizeof(buf), &bar);
        if (!mbar_wait(&bar, 0)) {
            atomicOr(flags, kErrTimeout);
        } else {
            out[0] = buf[7];
        }
    }
}

__global__ void plain(int* v) { v[threadIdx.x] = (int)threadIdx.x * 3; }

int main() {
    uint32_t* flags = nullptr;
    unsigned long long* waited = nullptr;
    uint4 *src = nullptr, *out = nullptr;
    int* v = nullptr;
    if (cudaMalloc(&flags, 8) || cudaMalloc(&waited, 8) || cudaMalloc(&src, 8 * sizeof(uint4)) ||
        cudaMalloc(&out, sizeof(uint4)) || cudaMalloc(&v, 32 * sizeof(int)))
        return 2;
    uint4 h_src[8];
    for (int i = 0; i < 8; ++i) h_src[i] = make_uint4(i, i + 1, i + 2, i + 3);
    cudaMemcpy(src, h_src, sizeof(h_src), cudaMemcpyHostToDevice);

    cudaMemset(flags, 0, 8);
    never_delivered<<<1, 32>>>(flags, waited);
    const cudaError_t e1 = cudaDeviceSynchronize();
    uint32_t f1 = 0;
    unsigned long long ns = 0;
    cudaMemcpy(&f1, flags, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(&ns, waited, 8, cudaMemcpyDeviceToHost);

    cudaMemset(flags, 0, 8);
    delivered<<<1, 32>>>(src, flags, out);
    const cudaError_t e2 = cudaDeviceSynchronize();
    uint32_t f2 = 0;
    uint4 got{};
    cudaMemcpy(&f2, flags, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(&got, out, sizeof(got), cudaMemcpyDeviceToHost);

    plain<<<1, 32>>>(v);
    const cudaError_t e3 = cudaDeviceSynchronize();
    int hv[32] = {};
    cudaMemcpy(hv, v, sizeof(hv), cudaMemcpyDeviceToHost);

    printf("timeout_flag=%u timeout_bit=%u waited_ms=%.1f err1=%s delivered_flag=%u delivered_ok=%d err2=%s "
           "plain_ok=%d err3=%s\n",
           f1, (unsigned)kErrTimeout, ns / 1e6, cudaGetErrorName(e1), f2, got.x == 7 && got.w == 10,
           cudaGetErrorName(e2), hv[31] == 93, cudaGetErrorName(e3));
    return 0;
}
