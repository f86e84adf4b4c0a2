// kr_noalloc.cu -- kernel_reduce_noalloc: the Sum / LogSumExp reduction in split-j
// mode, with its split partials in a fixed static device array instead of memory
// taken from the allocator.
//
// Who needs it: callers that cannot allocate device memory at call time -- for
// example a process that has already handed (almost) all device memory to its
// own arena, so any further cudaMalloc / cudaMallocAsync fails, or a
// latency-critical loop that must not wait on the driver's allocator.  Such a
// caller allocates its inputs and outputs itself, once, and this entry point
// touches no allocator at all.
//
// Scratch: kScratchBytes (16 MiB) of static device memory, reserved on every GPU
// that loads the library until the process exits.  In host code the array's name
// only stands for the symbol; the device address is obtained once per device
// with cudaGetSymbolAddress (with that device current) on the first call there.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "kr_internal.h"

namespace {

constexpr int64_t kScratchBytes = (int64_t)16 << 20;
constexpr int64_t kScratchFloats = kScratchBytes / (int64_t)sizeof(float);

// Split-j partials of every kernel_reduce_noalloc call on this device (shared by
// all calls; each call overwrites every element it later reads).
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (the current device); looked up
// once per device.
cudaError_t scratch_for_device(int dev, float **ptr) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        float *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress((void **)&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool on_device(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" int kernel_reduce_noalloc(const float *x, const float *y, const float *b, float *out, int64_t M,
                                     int64_t N, int D, int E, float sigma, int reduction, kr_stream_t stream) {
    using namespace kr;
    if (reduction != KR_SUM && reduction != KR_LSE) return KR_ERR_INVALID;
    if (M < 0 || N < 0 || D < 1 || E < 1) return KR_ERR_INVALID;
    if (!(std::isfinite(sigma) && sigma > 0.f)) return KR_ERR_INVALID;
    if (D > kMaxD || E > kMaxE) return KR_ERR_UNSUPPORTED;
    if (M == 0) return KR_OK;
    if (!x || !out || (N > 0 && (!y || !b))) return KR_ERR_INVALID;
    // Two splits of (hi, lo) or (m, acc) per output element must fit the scratch.
    if (M * (int64_t)E > kScratchFloats / 4) return KR_ERR_UNSUPPORTED;
    // the limits of kernel_reduce: int32 indices, element counts up to 2^60
    const int64_t kMaxElems = (int64_t)1 << 60;
    if (N > INT32_MAX - 1 || M > kMaxElems / D || N > kMaxElems / D || N > kMaxElems / E) return KR_ERR_UNSUPPORTED;
    // Host arrays would need staging memory: device (or managed) pointers only.
    if (!on_device(x) || !on_device(out) || (N > 0 && (!on_device(y) || !on_device(b)))) return KR_ERR_INVALID;
    const uintptr_t o0 = (uintptr_t)out, o1 = o0 + (uintptr_t)(M * E * (int64_t)sizeof(float));
    auto hits = [&](const void *p, int64_t bytes) {
        const uintptr_t p0 = (uintptr_t)p;
        return p && bytes > 0 && p0 < o1 && o0 < p0 + (uintptr_t)bytes;
    };
    if (hits(x, M * D * 4) || hits(y, N * D * 4) || hits(b, N * E * 4)) return KR_ERR_INVALID;

    const int op = reduction == KR_SUM ? OP_SUM : OP_LSE;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return KR_ERR_CUDA;
    float *scratch = nullptr;
    ce = scratch_for_device(dev, &scratch);
    if (ce != cudaSuccess) return KR_ERR_CUDA;
    int num_sms = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KR_ERR_CUDA;
    Instance in = choose_instance(op, D, E);
    in.rec = false;  // the kernels stage their own tiles: no records, which would need memory
    const int occ = op == OP_SUM ? occupancy_sum(in) : occupancy_lse(in);

    // The planner's split for the CUDA-core kernel, at least 2, at most what the
    // scratch holds.
    kr_options opt = {};
    opt.path = KR_PATH_CUDA_CORES;
    kr_plan_t p;
    int st = kr_plan(op, M, N, D, E, num_sms, occ, &opt, &p);
    if (st != KR_OK) return st;
    const int64_t fit = kScratchFloats / (2 * M * (int64_t)E);
    int S = p.split < 2 ? 2 : p.split;
    if (S > fit) S = (int)fit;
    opt.split = S;
    st = kr_plan(op, M, N, D, E, num_sms, occ, &opt, &p);
    if (st != KR_OK) return st;

    Args a{};
    a.x = x;
    a.y = y;
    a.b = b;
    a.out = out;
    a.M = M;
    a.N = N;
    a.D = D;
    a.E = E;
    a.c = (float)(std::sqrt(1.4426950408889634) / (double)sigma);
    a.S = p.split;
    a.chunk = p.chunk;
    a.out_n = M * E;
    a.ws_n = (int64_t)p.split * M * E;
#ifdef KR_DEBUG
    a.dbg = debug_word(dev);  // the index checks report where kr_device_status reads
#endif
    if (p.split > 1) {
        a.ws0 = scratch;
        a.ws1 = scratch + (int64_t)p.split * M * E;
    }
    const dim3 grid((unsigned)p.row_blocks, (unsigned)p.split);
    ce = op == OP_SUM ? launch_sum(in, a, grid, (cudaStream_t)stream) : launch_lse(in, a, grid, (cudaStream_t)stream);
    if (ce == cudaSuccess && p.split > 1) ce = launch_combine(op, in, a, (cudaStream_t)stream);
    return ce == cudaSuccess ? KR_OK : KR_ERR_CUDA;
}
