// kr_tc.h -- the tensor-core path of the Gaussian Sum and LogSumExp (see kr_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kr_internal.h"

namespace kr {

// Threads of the tensor-core x-gradient's block: a TMA warp, an MMA warp and 16 evaluation
// warps (four per TMEM lane quarter, each with 32 of a tile's 128 points).
constexpr int kTcGradThreads = 64 + 32 * 16;

// Host-side description of one tensor-core Sum launch.
struct TcArgs {
    const __half *a_hi, *a_lo;  // m_pad x 64 augmented x operands (split fp16), m_pad % kTcRows == 0
    const __half *b_hi, *b_lo;  // n_pad x 64 augmented y operands, n_pad % kTcCols == 0
    const float *bpad;          // Sum: n_pad signal values (zero past N); LSE: log2 e w - tile frame
                                // (-inf past N); 16-byte aligned
    const float *fpad;          // LSE: n_pad / kTcCols tile frames (base 2); Sum: unused
    float *out;                 // S == 1: M outputs
    float *ws0, *ws1;           // S > 1: S x M (hi, lo) partials, as the CUDA-core Sum writes them
    const unsigned *guard;      // [0] max |x'|^2, [1] max |y'|^2 (float bits), written by the prepass
    uint64_t wait_ns;           // bound of every mbarrier wait (global time)
    bool starve;                // test hook: issue no B tile, so the waits run out
    int64_t M, N, m_pad, n_pad;
    int64_t chunk;              // points per split, a multiple of kTcCols (gradient: kTcGradCols)
    int S;
    bool lse;                   // LogSumExp (CUDA-core LSE partials) instead of the Sum
    // x-gradient (tc_launch_grad): x (M x D fp32), upstream g (M), prescale c, the factor
    // -2 / (sigma^2 c); out / ws0 / ws1 are then M x D (S x M x D partials).
    const float *x, *g;
    int D;
    float c, gscale;
    uint8_t *flags;  // x-gradient: S x M, 1 where the CUDA-core kernel must redo (split, row)
    // K-min (tc_launch_knn): y (N x D fp32) for the direct distances, K, the index output
    // (M x K; out: the distances, or null) and, with S > 1, the index partials (ws0: distances),
    // S x M x KP each; carry: M x KP, per row the distances of the best list any block of
    // the row has published (the x prepass sets them to +inf)
    const float *y;
    int32_t *idx, *wsi;
    int K, KP;
    float *carry;
};

// Kernel parameters: TMA descriptors of the four operand arrays plus the rest.
struct TcParams {
    CUtensorMap tm_a_hi, tm_a_lo, tm_b_hi, tm_b_lo;
    const float *bpad, *fpad;
    float *out, *ws0, *ws1;
    const unsigned *guard;
    uint64_t wait_ns;
    int starve;
    int64_t M, N, chunk;
    int S;
    const float *x, *g;  // x-gradient only (x: and K-min)
    int D;
    float c, gscale;
    uint8_t *flags;
    const float *y;  // K-min only
    int32_t *idx, *wsi;
    int K;
    float *carry;
};

int tc_smem_bytes();
int tc_occupancy();
bool tc_available();  // the driver offers cuTensorMapEncodeTiled
// Operand prepass.  lse: the operands carry the weight slot of the LogSumExp (A: 1; B: the
// log-weight relative to its tile's frame, which fpad receives; b holds the log-weights).
// Otherwise bpad receives b padded with zeros.
// natural_b: bpad in point order (the x-gradient) rather than the Sum's evaluation order.
// lo null: only the high halves are written.  carry non-null: carry[r * carry_w + k] = +inf
// for r < rows, k < carry_w.
cudaError_t tc_launch_prep(const float *src, int64_t rows, int64_t rows_pad, int D, float c, bool is_x, bool lse,
                           __half *hi, __half *lo, unsigned *guard, const float *b, float *bpad, float *fpad,
                           cudaStream_t s, bool natural_b = false, float *carry = nullptr, int carry_w = 0);
// x-gradient: guard[2] receives the largest |b| (float bits), from which the prepass of the
// y side scales bpad by a power of two into [-1, 1] (run before that prepass).
cudaError_t tc_launch_bmax(const float *b, int64_t n, unsigned *guard, cudaStream_t s);
// Opts the tensor-core kernels in to their dynamic shared memory on the current device.
cudaError_t tc_set_attributes();
cudaError_t tc_launch_sum(const TcArgs &a, dim3 grid, cudaStream_t s);
// The x-gradient on the tensor cores (32 <= D <= 62, E = 1): grid (ceil(M / 128), S).
cudaError_t tc_launch_grad(const TcArgs &a, dim3 grid, cudaStream_t s);
int tc_grad_occupancy();
// K-min on the tensor cores (32 <= D <= 62, K <= 32): grid (ceil(M / 128), S); a screen by the
// tensor product, direct fp32 distances for the points that pass.
cudaError_t tc_launch_knn(const TcArgs &a, dim3 grid, cudaStream_t s);
// Reads (and optionally clears) the sticky device status of the tensor-core kernels on the
// current device: bit 0 = a bounded wait gave up.  Synchronous.
cudaError_t tc_read_status(bool clear, unsigned *status);

}  // namespace kr
