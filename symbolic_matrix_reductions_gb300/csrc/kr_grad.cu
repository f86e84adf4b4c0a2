// x-gradient instances and launcher.
#include <mutex>
#include <utility>
#include <vector>

#include "kr_kernels_packed.cuh"

namespace kr {

namespace {
typedef void (*KernelFn)(const Args);

template <int DP, int EP>
KernelFn grad_instance() {
    if constexpr (packed_grad(DP))
        return grad2_kernel<DP, EP, rows_grad(DP, EP), tile_points_packed(pair_stride(DP, EP))>;
    else if constexpr (wide_grad(DP))
        return gradw_kernel<DP, EP, kWideGradTile>;
    else
        return grad_kernel<DP, EP, rows_grad(DP, EP), tile_points(pack_stride(DP, EP))>;
}

// Dynamic shared memory of an instance (the wide kernel's tile and running sums).
size_t grad_smem(const Instance &inst) {
    if (!wide_grad(inst.d_pad)) return 0;
    return ((size_t)kWideGradTile * pack_stride(inst.d_pad, inst.ek_pad) + 2 * (size_t)inst.d_pad * kThreads) *
           sizeof(float);
}

// Opts a wide instance in to its dynamic shared memory (above the 48 KB default), once.
cudaError_t grad_prepare(KernelFn k, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    static std::mutex mu;
    static std::vector<std::pair<int, KernelFn>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &dk : done)
        if (dk.first == dev && dk.second == k) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) done.emplace_back(dev, k);
    return e;
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
    const size_t smem = grad_smem(inst);
    const cudaError_t e = grad_prepare(k, smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

int occupancy_grad(const Instance &inst) {
    KernelFn k = grad_kernel_for(inst);
    int n = 0;
    const size_t smem = grad_smem(inst);
    if (!k || grad_prepare(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace kr
