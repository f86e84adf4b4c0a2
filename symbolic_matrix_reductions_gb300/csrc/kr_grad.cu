// x-gradient instances and launcher.
#include "kr_kernels_packed.cuh"

namespace kr {

namespace {
typedef void (*KernelFn)(const Args);

template <int DP, int EP>
KernelFn grad_instance() {
    if constexpr (packed_grad(DP))
        return grad2_kernel<DP, EP, rows_grad(DP, EP), tile_points_packed(pair_stride(DP, EP))>;
    else
        return grad_kernel<DP, EP, rows_grad(DP, EP), tile_points(pack_stride(DP, EP))>;
}

template <int EP>
KernelFn grad_by_d(int dp) {
    switch (dp) {
        case 1: return grad_instance<1, EP>();
        case 2: return grad_instance<2, EP>();
        case 3: return grad_instance<3, EP>();
        case 4: return grad_instance<4, EP>();
        case 8: return grad_instance<8, EP>();
        case 16: return grad_instance<16, EP>();
        case 32: return grad_instance<32, EP>();
        case 50: return grad_instance<50, EP>();
        case 64: return grad_instance<64, EP>();
        case 128: return grad_instance<128, EP>();
        default: return nullptr;
    }
}

KernelFn grad_kernel_for(const Instance &inst) {
    switch (inst.ek_pad) {
        case 1: return grad_by_d<1>(inst.d_pad);
        case 4: return grad_by_d<4>(inst.d_pad);
        case 16: return grad_by_d<16>(inst.d_pad);
        default: return nullptr;
    }
}
}  // namespace

cudaError_t launch_grad(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s) {
    KernelFn k = grad_kernel_for(inst);
    if (!k) return cudaErrorInvalidValue;
    k<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

int occupancy_grad(const Instance &inst) {
    KernelFn k = grad_kernel_for(inst);
    int n = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, 0) != cudaSuccess) return 0;
    return n;
}

}  // namespace kr
