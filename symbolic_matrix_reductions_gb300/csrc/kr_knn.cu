// K-min / ArgMin instances and launcher.
#include "kr_kernels_packed.cuh"

namespace kr {

namespace {
typedef void (*KernelFn)(const Args);

template <int DP, int KP>
KernelFn knn_instance() {
    if constexpr (knn_expand(DP))
        return knnx_kernel<DP, KP, rows_knn(DP, KP), knn_instance_tile(DP)>;
    else if constexpr (packed(DP))
        return knn2_kernel<DP, KP, rows_knn(DP, KP), knn_instance_tile(DP)>;
    else
        return knn_kernel<DP, KP, rows_knn(DP, KP), knn_instance_tile(DP)>;
}

template <int KP>
KernelFn knn_by_d(int dp) {
    switch (dp) {
        case 1: return knn_instance<1, KP>();
        case 2: return knn_instance<2, KP>();
        case 3: return knn_instance<3, KP>();
        case 4: return knn_instance<4, KP>();
        case 8: return knn_instance<8, KP>();
        case 16: return knn_instance<16, KP>();
        case 32: return knn_instance<32, KP>();
        case 50: return knn_instance<50, KP>();
        case 64: return knn_instance<64, KP>();
        case 128: return knn_instance<128, KP>();
        default: return nullptr;
    }
}

KernelFn knn_kernel_for(const Instance &inst) {
    switch (inst.ek_pad) {
        case 1: return knn_by_d<1>(inst.d_pad);
        case 4: return knn_by_d<4>(inst.d_pad);
        case 10: return knn_by_d<10>(inst.d_pad);
        case 16: return knn_by_d<16>(inst.d_pad);
        case 32: return knn_by_d<32>(inst.d_pad);
        default: return nullptr;
    }
}
}  // namespace

cudaError_t launch_knn(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s) {
    KernelFn k = knn_kernel_for(inst);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

int occupancy_knn(const Instance &inst) {
    KernelFn k = knn_kernel_for(inst);
    int n = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, 0) != cudaSuccess) return 0;
    return n;
}

}  // namespace kr
