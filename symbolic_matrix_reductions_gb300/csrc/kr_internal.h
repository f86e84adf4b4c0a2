// kr_internal.h -- declarations shared by the host planner and the kernel instance files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kreduce.h"

namespace kr {

// K-min on the tensor cores: the largest |x|^2 + |y|^2 its screen takes (fp16 operands stay in
// range and the screen's margin, 2^-14 of the norms, stays below the distances that matter);
// above it the CUDA-core kernel does the call.
constexpr float kTcKnnNormLimit = 4096.f;

enum Op { OP_SUM = 0, OP_LSE = 1, OP_GRAD = 2, OP_KNN = 3, OP_MAX = 4 };
constexpr int kNumOps = 5;
constexpr int kNumKernels = 4;  // radial kernel kinds (KR_KERNEL_*)

constexpr int kThreads = 128;   // threads per block for every main kernel
constexpr int kMaxD = 128;
constexpr int kMaxE = 16;
constexpr int kMaxK = 32;
constexpr int kMaxSplit = 64;   // most j-ranges a call is split into
constexpr int kMaxBatch = 65535;  // most problems in one batched call (grid z)

// Everything a main kernel needs; passed by value as the kernel parameter.
struct Args {
    const float *x;      // M x D
    const float *y;      // N x D
    const float *b;      // N x E: signal (Sum, grad) or log-weight (LSE)
    const float *g;      // M x E upstream gradient (grad only)
    float *out;          // S == 1: final output (M x E, M x D or M x K distances)
    int32_t *idx;        // K-min indices, S == 1
    float *ws0;          // S > 1: first partial array  (S x M x W)
    float *ws1;          // S > 1: second partial array (S x M x W)
    int32_t *wsi;        // S > 1: K-min partial indices (S x M x K_pad)
    int64_t M, N;
    int D, E, K;
    float c;             // coordinate prescale sqrt(log2 e) / sigma (1 for K-min)
    float gscale;        // grad: -2 / (sigma^2 c)
    int64_t chunk;       // columns per split
    int S;
    const unsigned *tc_guard;  // non-null when the tensor-core kernel ran first; the CUDA-core
                               // kernel then works only if the guard failed it ...
    const uint8_t *tc_flags;   // ... or (x-gradient) on the rows this flag array (S x M) marks
    float vsign;         // Max/Min: +1 (Max) or -1 (Min, computed as -Max of k (-b))
    // Batch dimension: blockIdx.z selects one of `batch` independent problems whose
    // arrays follow each other in memory; the strides are in elements (0 when batch == 1).
    int batch;
    int64_t bs_x, bs_y, bs_b, bs_g, bs_out, bs_idx, bs_ws;
    // Block-sparse mode (radial kernels): block b owns rows blk[b].x..blk[b].y-1 and
    // reduces over the column ranges rng[blk[b].z .. blk[b].w-1]; null otherwise.
    const int4 *blk;
    const int2 *rng;
    // Element counts of the outputs and split partials of one problem, for the index
    // checks of debug builds (-DKR_DEBUG), which record a violated bound in *dbg.
    int64_t out_n, idx_n, ws_n;
    unsigned *dbg;
    // Streamed records (instances with Instance::rec): tile-major pair records of y (and the
    // signal or tile-relative log-weight), written by the prepass, read by cp.async; the
    // LogSumExp's tile frames (EP floats a tile, base 2).  Element counts of one problem
    // (rec_n, wtile_n) and batch strides (bs_rec, bs_wtile).
    float *rec;
    float *wtile;
    int64_t rec_n, wtile_n, bs_rec, bs_wtile;
};

// Bits of the debug status word (debug builds; kr_device_status reports them << 8).
enum DebugBits : unsigned {
    KRD_X = 1u, KRD_Y = 2u, KRD_B = 4u, KRD_G = 8u, KRD_OUT = 16u, KRD_IDX = 32u, KRD_WS = 64u, KRD_SMEM = 128u
};

// Compile-time shape of one kernel instance, chosen by the planner.
struct Instance {
    int d_pad, ek_pad, rows, tile;
    bool rec;  // y tiles streamed from prepass records (see streamed() in kr_config.h)
};

// Debug builds (-DKR_DEBUG): the device word of `dev` that the kernels' index checks
// write to (allocated once per device, kept for the life of the process); null when it
// could not be allocated.  Release builds never call it.
unsigned *debug_word(int dev);

// Instance selection (pure host logic).  kind: the kernel kind (KR_KERNEL_*) of a Sum; the
// streamed variant (rec) serves the Gaussian Sum, LogSumExp and x-gradient up to D = 16.
Instance choose_instance(int op, int D, int EK, int kind = 0);

// Launchers, one per kernel family; they dispatch on the instance and return the
// launch's cudaError_t.  grid = (row_blocks, S).
cudaError_t launch_sum(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_lse(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_grad(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_knn(const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_combine(int op, const Instance &inst, const Args &a, cudaStream_t s);
// Prepass of the streamed instances: packs y and b of op (Sum / grad: the signal; LSE: the
// tile-relative log-weight and the tile frames) into a.rec (and a.wtile); grid = (tiles, 1,
// batch).
cudaError_t launch_pack(int op, const Instance &inst, const Args &a, int64_t tiles, cudaStream_t s);
// Elements of the records and tile frames of one problem with N points.
int64_t record_elems(const Instance &inst, int64_t N);
int64_t wtile_elems(int op, const Instance &inst, int64_t N);
// Opts kernel `fn` in to `smem` bytes of dynamic shared memory on the current device when
// that is above the 48 KB default (once per device and kernel).
cudaError_t set_dyn_smem(const void *fn, size_t smem);
// Radial-kernel family (kr_radial.cuh): red 0 = Sum (Laplace, Cauchy, inverse
// multiquadric), 1 = Max/Min (every kind); one launcher per kernel kind.
cudaError_t launch_radial_gauss(int red, const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_radial_laplace(int red, const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_radial_cauchy(int red, const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
cudaError_t launch_radial_imq(int red, const Instance &inst, const Args &a, dim3 grid, cudaStream_t s);
int occupancy_radial_gauss(int red, const Instance &inst);
int occupancy_radial_laplace(int red, const Instance &inst);
int occupancy_radial_cauchy(int red, const Instance &inst);
int occupancy_radial_imq(int red, const Instance &inst);

// Resident blocks per SM of an instance (cudaOccupancyMaxActiveBlocksPerMultiprocessor);
// 0 if unknown.
int occupancy_sum(const Instance &inst);
int occupancy_lse(const Instance &inst);
int occupancy_grad(const Instance &inst);
int occupancy_knn(const Instance &inst);

}  // namespace kr
