// x-gradient instances and launcher.
#include "kr_kernels_packed.cuh"

namespace kr {

namespace {
typedef void (*KernelFn)(const Args);

// rec: the streamed variant of the packed kernel (records from the prepass).
template <int DP, int EP>
KernelFn grad_instance(bool rec) {
    if constexpr (packed_grad(DP)) {
        static_assert(!packed_grad(DP) || streamed(DP), "every packed gradient instance has a streamed variant");
        return rec ? grad2_kernel<DP, EP, rows_grad(DP, EP), tile_points_packed(pair_stride(DP, EP)), true>
                   : grad2_kernel<DP, EP, rows_grad(DP, EP), tile_points_packed(pair_stride(DP, EP)), false>;
    } else if constexpr (wide_grad(DP)) {
        return rec ? nullptr : gradw_kernel<DP, EP, kWideGradTile>;
    } else {
        return rec ? nullptr : grad_kernel<DP, EP, rows_grad(DP, EP), tile_points(pack_stride(DP, EP))>;
    }
}

// Dynamic shared memory of an instance (the wide kernel's tile and running sums; the
// streamed kernel's two record tiles).
size_t grad_smem(const Instance &inst) {
    if (inst.rec) return 2 * (size_t)record_tile_floats(inst.d_pad, inst.ek_pad, inst.tile) * sizeof(float);
    if (!wide_grad(inst.d_pad)) return 0;
    return ((size_t)kWideGradTile * pack_stride(inst.d_pad, inst.ek_pad) + 2 * (size_t)inst.d_pad * kThreads) *
           sizeof(float);
}

// Opts an instance in to its dynamic shared memory (above the 48 KB default), once.
cudaError_t grad_prepare(KernelFn k, size_t smem) { return set_dyn_smem((const void *)k, smem); }

template <int EP>
KernelFn grad_by_d(int dp, bool rec) {
    switch (dp) {
        case 1: return grad_instance<1, EP>(rec);
        case 2: return grad_instance<2, EP>(rec);
        case 3: return grad_instance<3, EP>(rec);
        case 4: return grad_instance<4, EP>(rec);
        case 8: return grad_instance<8, EP>(rec);
        case 16: return grad_instance<16, EP>(rec);
        case 32: return grad_instance<32, EP>(rec);
        case 50: return grad_instance<50, EP>(rec);
        case 64: return grad_instance<64, EP>(rec);
        case 128: return grad_instance<128, EP>(rec);
        default: return nullptr;
    }
}

KernelFn grad_kernel_for(const Instance &inst) {
    switch (inst.ek_pad) {
        case 1: return grad_by_d<1>(inst.d_pad, inst.rec);
        case 4: return grad_by_d<4>(inst.d_pad, inst.rec);
        case 16: return grad_by_d<16>(inst.d_pad, inst.rec);
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
