// kr_probe.cu -- pipe-throughput probes used to state the FP32 / MUFU roofline of
// the reduction kernels.  Each probe runs 8 independent dependency chains per
// thread on every SM and reports, per block, the SM cycles the loop took
// (clock64), so throughput comes out in lanes per clock per SM, independent of the
// SM clock.  Built into libkrprobe.so, separate from the library's C ABI.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;

__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rsqrt_approx(float v) {
    float r;
    asm volatile("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float sqrt_approx(float v) {
    float r;
    asm volatile("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// kind 0: scalar FFMA; 1: packed FFMA2 (f32x2); 2: ex2.approx; 3: rcp.approx;
// 4: rsqrt.approx; 5: sqrt.approx (the transcendental-unit operations of the kernels).
template <int KIND>
__global__ void __launch_bounds__(256) probe_kernel(int iters, float seed, float *sink, long long *cycles) {
    float v[kChains];
    float2 w[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        v[c] = seed + 0.001f * (float)(threadIdx.x + c);
        w[c] = make_float2(v[c], v[c] + 0.5f);
    }
    const float2 m2 = make_float2(0.999f, 0.998f), a2 = make_float2(0.001f, 0.002f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) {
            if (KIND == 0) v[c] = fmaf(v[c], 0.999f, 0.001f);
            if (KIND == 1) w[c] = __ffma2_rn(w[c], m2, a2);
            if (KIND == 2) v[c] = ex2_approx(-v[c]);
            if (KIND == 3) v[c] = rcp_approx(v[c] + 0.5f);  // the add keeps 1/(1/v) from folding
            if (KIND == 4) v[c] = rsqrt_approx(v[c]);   // tends to 1
            if (KIND == 5) v[c] = sqrt_approx(v[c]);    // tends to 1
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += (KIND == 1) ? (w[c].x + w[c].y) : v[c];
    if (s == 12345.678f) sink[0] = s;  // keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

}  // namespace

extern "C" {

// Runs probe `kind` with `blocks` blocks of 256 threads, `iters` loop trips of 8
// chains each.  cycles_dev[blocks] receives each block's SM cycles; sink_dev is a
// 1-float device buffer.  Returns the cudaError_t of the launch.
int kr_probe_pipe(int kind, int blocks, int iters, float *sink_dev, long long *cycles_dev, void *stream) {
    cudaStream_t s = (cudaStream_t)stream;
    switch (kind) {
        case 0: probe_kernel<0><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        case 1: probe_kernel<1><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        case 2: probe_kernel<2><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        case 3: probe_kernel<3><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        case 4: probe_kernel<4><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        case 5: probe_kernel<5><<<blocks, 256, 0, s>>>(iters, 0.5f, sink_dev, cycles_dev); break;
        default: return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

// Lanes of work per chain step (2 for the packed probe) and chains per thread.
int kr_probe_lanes_per_op(int kind) { return kind == 1 ? 2 : 1; }
int kr_probe_chains(void) { return kChains; }

}  // extern "C"
