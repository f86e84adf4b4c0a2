// kr_records.cu -- the prepass of the streamed Sum / LogSumExp / x-gradient instances
// (D <= 16): the call's y and its signal, packed once into the pair records the
// reduction kernels read from shared memory, tile by tile, so that the kernels can copy
// each tile with plain 16-byte cp.async and keep two tiles in flight.
//
// Records of tile t (BN points j = t BN .. t BN + BN - 1, BN the instance's tile):
// BN / 2 pair records of PS2 floats; record m holds points 2m and 2m+1 interleaved
// field by field: the coordinates -c y_jd (d < DP; zero past D and for points past N),
// then the values: b_je (Sum, gradient; zero past E and N) or, for the LogSumExp,
// W_te - w'_je with w' = log2(e) w and W_te the largest w' of the tile's points (+inf
// for an empty weight), W_te itself going to wtile[t EP + e].  The same arithmetic as
// the kernels' own staging, so both give the same bits for the same tiles.
#include <mutex>
#include <utility>
#include <vector>

#include "kr_kernels_packed.cuh"

namespace kr {

template <int DP, int EP, bool LSE>
__global__ void __launch_bounds__(kThreads) pack_records_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PS2 = pair_stride(DP, EP);
    constexpr int BN = tile_points_packed(PS2);
    constexpr int TF = record_tile_floats(DP, EP, BN);
    constexpr float kLog2e = 1.4426950408889634f;
    __shared__ float wred[kThreads / 32][EP];
    const int64_t tt = blockIdx.x;
    const int64_t j0 = tt * BN;

    float W[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) W[e] = -f_inf();
    if (LSE) {
        for (int p = threadIdx.x; p < BN; p += kThreads) {
            const int64_t j = j0 + p;
#pragma unroll
            for (int e = 0; e < EP; ++e)
                if (j < a.N && e < a.E) W[e] = fmaxf(W[e], kLog2e * ldg_chk(a, a.b, j * a.E + e, a.N * a.E, KRD_B));
        }
#pragma unroll
        for (int e = 0; e < EP; ++e) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) W[e] = fmaxf(W[e], __shfl_xor_sync(0xffffffffu, W[e], o));
            if ((threadIdx.x & 31) == 0) wred[threadIdx.x >> 5][e] = W[e];
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            W[e] = wred[0][e];
#pragma unroll
            for (int w = 1; w < kThreads / 32; ++w) W[e] = fmaxf(W[e], wred[w][e]);
        }
        if (threadIdx.x == 0) {
#pragma unroll
            for (int e = 0; e < EP; ++e) st_chk(a, a.wtile, tt * EP + e, a.wtile_n, KRD_WS, W[e]);
        }
    }

    float *dst = a.rec + tt * TF;
    for (int m = threadIdx.x; m < BN / 2; m += kThreads) {
        float r[PS2];
#pragma unroll
        for (int f = 0; f < PS2; ++f) r[f] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t j = j0 + 2 * m + h;
            const bool ok = j < a.N;
#pragma unroll
            for (int d = 0; d < DP; ++d)
                r[2 * d + h] = (ok && d < a.D) ? -a.c * ldg_chk(a, a.y, j * a.D + d, a.N * a.D, KRD_Y) : 0.f;
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                if (!LSE) {
                    r[2 * (DP + e) + h] = (ok && e < a.E) ? ldg_chk(a, a.b, j * a.E + e, a.N * a.E, KRD_B) : 0.f;
                } else {
                    const float v = (ok && e < a.E) ? kLog2e * ldg_chk(a, a.b, j * a.E + e, a.N * a.E, KRD_B) : -f_inf();
                    r[2 * (DP + e) + h] = (v == -f_inf()) ? f_inf() : W[e] - v;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < PS2 / 4; ++k) {
            const int64_t o = (tt * TF + (int64_t)m * PS2) + 4 * k;
#ifdef KR_DEBUG
            if (o + 3 >= a.rec_n) {
                if (a.dbg) atomicOr(a.dbg, (unsigned)KRD_WS);
                continue;
            }
#endif
            reinterpret_cast<float4 *>(dst + (int64_t)m * PS2)[k] =
                make_float4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
        }
    }
}

namespace {
typedef void (*KernelFn)(const Args);

template <int EP, bool LSE>
KernelFn pack_by_d(int dp) {
    switch (dp) {
        case 1: return pack_records_kernel<1, EP, LSE>;
        case 2: return pack_records_kernel<2, EP, LSE>;
        case 3: return pack_records_kernel<3, EP, LSE>;
        case 4: return pack_records_kernel<4, EP, LSE>;
        case 8: return pack_records_kernel<8, EP, LSE>;
        case 16: return pack_records_kernel<16, EP, LSE>;
        default: return nullptr;
    }
}

template <bool LSE>
KernelFn pack_kernel_for(const Instance &inst) {
    switch (inst.ek_pad) {
        case 1: return pack_by_d<1, LSE>(inst.d_pad);
        case 4: return pack_by_d<4, LSE>(inst.d_pad);
        case 16: return pack_by_d<16, LSE>(inst.d_pad);
        default: return nullptr;
    }
}
}  // namespace

int64_t record_elems(const Instance &inst, int64_t N) {
    const int64_t tiles = (N + inst.tile - 1) / inst.tile;
    return tiles * (inst.tile / 2) * pair_stride(inst.d_pad, inst.ek_pad);
}

int64_t wtile_elems(int op, const Instance &inst, int64_t N) {
    return op == OP_LSE ? (N + inst.tile - 1) / inst.tile * inst.ek_pad : 0;
}

cudaError_t launch_pack(int op, const Instance &inst, const Args &a, int64_t tiles, cudaStream_t s) {
    if (tiles <= 0) return cudaSuccess;
    if (inst.tile != tile_points_packed(pair_stride(inst.d_pad, inst.ek_pad))) return cudaErrorInvalidValue;
    KernelFn k = op == OP_LSE ? pack_kernel_for<true>(inst) : pack_kernel_for<false>(inst);
    if (!k) return cudaErrorInvalidValue;
    k<<<dim3((unsigned)tiles, 1, (unsigned)(a.batch > 1 ? a.batch : 1)), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t set_dyn_smem(const void *fn, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    static std::mutex mu;
    static std::vector<std::pair<int, const void *>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &dk : done)
        if (dk.first == dev && dk.second == fn) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) done.emplace_back(dev, fn);
    return e;
}

}  // namespace kr
