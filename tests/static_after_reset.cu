// ep_get_layout_static across a device reset.  The entry point caches the
// device address of its built-in scratch array per device context; after
// cudaDeviceReset() the next call runs in a new context, where the library's
// module is loaded again (its arrays possibly elsewhere), so the cached
// address must not be reused.  This program computes one layout that needs
// scratch (65536 routing entries, 256 experts) with ep_get_layout and a
// cudaMalloc'd workspace, then with ep_get_layout_static before and after a
// reset, and compares every output.  Prints one line; exit code 0 when all
// three agree.
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>

#include "ep.h"

namespace {

constexpr int T = 8192, H = 8, E = 256, K = 8, P = 32;
constexpr int N = T * K, R = T * K;

struct Outputs {
    std::vector<int32_t> counts, offsets, part_counts, part_offsets, slot_of, src_token, src_k;
    uint32_t err = 0;
    bool operator==(const Outputs& o) const {
        return counts == o.counts && offsets == o.offsets && part_counts == o.part_counts &&
               part_offsets == o.part_offsets && slot_of == o.slot_of && src_token == o.src_token &&
               src_k == o.src_k && err == o.err;
    }
};

#define CK(call)                                                                           \
    do {                                                                                   \
        cudaError_t e_ = (call);                                                           \
        if (e_ != cudaSuccess) {                                                           \
            std::printf("FAILED: %s: %s\n", #call, cudaGetErrorString(e_));                \
            return false;                                                                  \
        }                                                                                  \
    } while (0)

// One layout of `idx` on device 0; with_workspace selects ep_get_layout (a
// cudaMalloc'd workspace) or ep_get_layout_static.
bool run_layout(const std::vector<int32_t>& idx, bool with_workspace, Outputs& out) {
    const ep_shape_t shape = {T, H, E, K, P, EP_LAYOUT_PACKED, 0};
    int32_t *d_idx, *d_counts, *d_offsets, *d_pc, *d_po, *d_slot, *d_st, *d_sk;
    uint32_t* d_err;
    void* ws = nullptr;
    const size_t ws_bytes = ep_layout_workspace_bytes(&shape);
    if (ws_bytes == 0 || ws_bytes == (size_t)-1) {
        std::printf("FAILED: this shape should need layout scratch (%zu)\n", ws_bytes);
        return false;
    }
    CK(cudaMalloc(&d_idx, N * 4));
    CK(cudaMalloc(&d_counts, E * 4));
    CK(cudaMalloc(&d_offsets, (E + 1) * 4));
    CK(cudaMalloc(&d_pc, P * 4));
    CK(cudaMalloc(&d_po, (P + 1) * 4));
    CK(cudaMalloc(&d_slot, N * 4));
    CK(cudaMalloc(&d_st, R * 4));
    CK(cudaMalloc(&d_sk, R * 4));
    CK(cudaMalloc(&d_err, 4));
    if (with_workspace) CK(cudaMalloc(&ws, ws_bytes));
    CK(cudaMemcpy(d_idx, idx.data(), N * 4, cudaMemcpyHostToDevice));
    CK(cudaMemset(d_err, 0, 4));
    ep_status_t st = with_workspace
                         ? ep_get_layout(&shape, d_idx, d_counts, d_offsets, d_pc, d_po, d_slot, d_st, d_sk, ws,
                                         ws_bytes, d_err, nullptr)
                         : ep_get_layout_static(&shape, d_idx, d_counts, d_offsets, d_pc, d_po, d_slot, d_st, d_sk,
                                                d_err, nullptr);
    if (st != EP_OK) {
        std::printf("FAILED: layout call returned %d (%s)\n", (int)st, ep_last_error());
        return false;
    }
    CK(cudaDeviceSynchronize());
    out.counts.resize(E);
    out.offsets.resize(E + 1);
    out.part_counts.resize(P);
    out.part_offsets.resize(P + 1);
    out.slot_of.resize(N);
    out.src_token.resize(R);
    out.src_k.resize(R);
    CK(cudaMemcpy(out.counts.data(), d_counts, E * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.offsets.data(), d_offsets, (E + 1) * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.part_counts.data(), d_pc, P * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.part_offsets.data(), d_po, (P + 1) * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.slot_of.data(), d_slot, N * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.src_token.data(), d_st, R * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out.src_k.data(), d_sk, R * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&out.err, d_err, 4, cudaMemcpyDeviceToHost));
    for (void* p : {(void*)d_idx, (void*)d_counts, (void*)d_offsets, (void*)d_pc, (void*)d_po, (void*)d_slot,
                    (void*)d_st, (void*)d_sk, (void*)d_err, ws})
        if (p != nullptr) CK(cudaFree(p));
    return true;
}

}  // namespace

int main() {
    if (cudaSetDevice(0) != cudaSuccess) return 2;
    // skewed-looking routing: expert (t * 37 + j * j * 11) % E, duplicates allowed
    std::vector<int32_t> idx(N);
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < K; ++j) idx[t * K + j] = (int32_t)((t * 37u + j * j * 11u + (t >> 5)) % E);
    Outputs ref, before, after;
    if (!run_layout(idx, true, ref) || !run_layout(idx, false, before)) return 1;
    if (!(before == ref)) {
        std::printf("FAILED: static layout differs from the workspace layout\n");
        return 1;
    }
    if (cudaDeviceReset() != cudaSuccess || cudaSetDevice(0) != cudaSuccess) {
        std::printf("FAILED: device reset\n");
        return 1;
    }
    if (!run_layout(idx, false, after)) return 1;
    if (!(after == ref)) {
        std::printf("FAILED: static layout after the reset differs\n");
        return 1;
    }
    std::printf("static layout across a reset ok\n");
    return 0;
}
