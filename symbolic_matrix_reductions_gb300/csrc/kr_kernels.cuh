// kr_kernels.cuh -- sm_103a kernels of the tiled, on-the-fly kernel reductions.
//
// Scheme (KeOps README, symbolic-matrix paragraph: a tiled reduction whose matrix
// coefficients are evaluated on the fly, kept in registers rather than memory):
//   * a block owns kThreads * R rows of x; each thread keeps R rows x'_i and their
//     accumulators in registers for the whole j-range;
//   * the block walks its j-range in tiles of BN points: the tile of y (prescaled)
//     and its values (signal or log-weight) are staged into shared memory as
//     16-byte-aligned records, then every thread reads each record with broadcast
//     16-byte loads and evaluates R pairs from it;
//   * the Gaussian is exp(-|x-y|^2/sigma^2) = 2^(-|x'-y'|^2) with x' = c x,
//     y' = c y, c = sqrt(log2 e)/sigma, evaluated with ex2.approx.ftz;
//   * sums over j keep a fresh fp32 partial per tile and fold it into a
//     compensated (TwoSum) running pair once per tile;
//   * grid = (row blocks, S): with S > 1 each blockIdx.y owns one of S disjoint
//     j-ranges and writes a partial result, combined later in a fixed order.
// No kernel here waits on a flag or on another block: the only synchronisation
// is __syncthreads() inside a block.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kr_config.h"
#include "kr_internal.h"

namespace kr {

__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float lg2_approx(float v) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float f_inf() { return __int_as_float(0x7f800000); }

// The tensor-core K-min ran this call (its operand norms, written by its prepass, are within
// its limit); a finite sum is required, so NaN inputs take the CUDA-core kernel.
__device__ __forceinline__ bool tc_knn_ran(const unsigned *guard) {
    return __uint_as_float(guard[0]) + __uint_as_float(guard[1]) <= kTcKnnNormLimit;
}

// max(a, b, c) and min(a, b, c) in one instruction each (the three-input max.f32 /
// min.f32 of sm_100 and later); a NaN input is passed over as fmaxf / fminf pass it over.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Checked global accesses.  Release builds compile them to the plain access; debug
// builds (-DKR_DEBUG) first check the element index against the array's extent and, on
// a violation, set the array's bit in the status word a.dbg and skip the access (a load
// then returns 0), so a wrong index shows up as a status instead of a fault.
template <typename T>
__device__ __forceinline__ T ldg_chk(const Args &a, const T *p, int64_t k, int64_t n, unsigned bit) {
#ifdef KR_DEBUG
    if (k < 0 || k >= n) {
        if (a.dbg) atomicOr(a.dbg, bit);
        return T(0);
    }
#endif
    return __ldg(p + k);
}
template <typename T>
__device__ __forceinline__ void st_chk(const Args &a, T *p, int64_t k, int64_t n, unsigned bit, T v) {
#ifdef KR_DEBUG
    if (k < 0 || k >= n) {
        if (a.dbg) atomicOr(a.dbg, bit);
        return;
    }
#endif
    p[k] = v;
}
// Shared-memory index check (debug builds): false, and KRD_SMEM recorded, when k is
// outside [0, n).
__device__ __forceinline__ bool smem_ok(const Args &a, int64_t k, int64_t n) {
#ifdef KR_DEBUG
    if (k < 0 || k >= n) {
        if (a.dbg) atomicOr(a.dbg, (unsigned)KRD_SMEM);
        return false;
    }
#endif
    return true;
}

// The arguments of this block's problem: with a batch dimension (grid z), every
// array pointer moves to problem blockIdx.z.  Uniform across the block.
__device__ __forceinline__ Args batch_view(const Args &a) {
    if (a.batch <= 1) return a;
    Args v = a;
    const int64_t z = blockIdx.z;
    v.x += z * a.bs_x;
    v.y += z * a.bs_y;
    if (v.b) v.b += z * a.bs_b;
    if (v.g) v.g += z * a.bs_g;
    if (v.out) v.out += z * a.bs_out;
    if (v.idx) v.idx += z * a.bs_idx;
    if (v.ws0) v.ws0 += z * a.bs_ws;
    if (v.ws1) v.ws1 += z * a.bs_ws;
    if (v.wsi) v.wsi += z * a.bs_ws;
    if (v.rec) v.rec += z * a.bs_rec;
    if (v.wtile) v.wtile += z * a.bs_wtile;
    return v;
}

// ---------------------------------------------------------------------------
// Asynchronous tile copies (streamed records): 16-byte cp.async from global to shared
// memory through L2 only (.cg), grouped per tile; cp.async.wait_all plus the block
// barrier that follows make a tile visible to every thread.  These are hardware waits on
// the thread's own copies, not spin loops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Starts the copy of record tile `t` (TF floats, TF % 4 == 0) into `dst`: every thread
// copies 16-byte pieces t0 + threadIdx.x + k kThreads, coalesced.  Debug builds check the
// pieces against the records' extent (a.rec_n) and skip those outside.
template <int TF>
__device__ __forceinline__ void issue_record_tile(const Args &a, float *dst, int64_t t) {
    static_assert(TF % 4 == 0, "tiles are whole 16-byte pieces");
    const float *src = a.rec + t * TF;
    for (int c = threadIdx.x; c < TF / 4; c += kThreads) {
#ifdef KR_DEBUG
        if (t < 0 || t * TF + 4 * (int64_t)c + 3 >= a.rec_n) {
            if (a.dbg) atomicOr(a.dbg, (unsigned)KRD_WS);
            continue;
        }
#endif
        cp_async16(dst + 4 * c, src + 4 * c);
    }
    cp_async_commit();
}

// Dynamic shared memory of the streamed kernels (two record tiles).
extern __shared__ float4 kr_dyn_smem[];

// Knuth's TwoSum: (hi, lo) += v with the rounding error of hi + v kept in lo.
__device__ __forceinline__ void two_sum_add(float &hi, float &lo, float v) {
    const float s = __fadd_rn(hi, v);
    const float bv = __fsub_rn(s, hi);
    const float av = __fsub_rn(s, bv);
    const float err = __fadd_rn(__fsub_rn(hi, av), __fsub_rn(v, bv));
    hi = s;
    lo = __fadd_rn(lo, err);
}

// Reads one tile record (PS floats, 16-byte aligned) into registers.
template <int PS>
__device__ __forceinline__ void load_record(const float *rec, float (&pv)[PS]) {
    const float4 *p4 = reinterpret_cast<const float4 *>(rec);
#pragma unroll
    for (int k = 0; k < PS / 4; ++k) {
        const float4 v = p4[k];
        pv[4 * k + 0] = v.x;
        pv[4 * k + 1] = v.y;
        pv[4 * k + 2] = v.z;
        pv[4 * k + 3] = v.w;
    }
}

// Loads the R rows of x owned by this thread, times `scale`; rows past M and
// coordinates past D are zero.
template <int DP, int R>
__device__ __forceinline__ void load_rows(const Args &a, int64_t row0, float (&xr)[R][DP], float scale) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + threadIdx.x;
#pragma unroll
        for (int d = 0; d < DP; ++d)
            xr[r][d] = (i < a.M && d < a.D) ? scale * ldg_chk(a, a.x, i * a.D + d, a.M * a.D, KRD_X) : 0.f;
    }
}

// Stages the coordinates of points [jt, jt + nv) into tile records, times
// `scale`; padding records [nv, nvp) get coordinate 0 = `pad0` and zeros.
// Coordinates D..DP-1 are zeroed once per kernel by zero_pad_coords().
template <int DP, int PS>
__device__ __forceinline__ void stage_coords(const Args &a, float *tile, int64_t jt, int nv, int nvp,
                                             float scale, float pad0) {
    for (int p = threadIdx.x; p < nvp; p += kThreads) {
        float *dst = tile + p * PS;
        if (p < nv) {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) dst[d] = scale * ldg_chk(a, a.y, (jt + p) * a.D + d, a.N * a.D, KRD_Y);
        } else {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) dst[d] = (d == 0) ? pad0 : 0.f;
        }
    }
}

template <int DP, int PS, int BN>
__device__ __forceinline__ void zero_pad_coords(const Args &a, float *tile) {
    if (a.D < DP) {
        for (int f = threadIdx.x; f < BN * DP; f += kThreads) {
            const int p = f / DP, d = f % DP;
            if (d >= a.D) tile[p * PS + d] = 0.f;
        }
    }
}

// ---------------------------------------------------------------------------
// Sum and LogSumExp.
//
// Sum:  value slot e of record j holds b_je; per pair k = 2^(-q), part += k b.
// LSE (base-2 units, t'_ij = -q_ij + w'_j, w' = w log2 e):  for each tile the
//   block computes W_e = max_j w'_je and stores v_je = W_e - w'_je >= 0, so every
//   term 2^(t' - W) = 2^(-(q + v)) lies in [0, 1] and the tile costs what a Sum
//   tile costs.  The tile's partial p in frame F = W is folded into the row's
//   running (m, hi + lo), whose value is 2^m (hi + lo).  Terms below 2^-126 in
//   frame W flush to zero; that is harmless when the row's running total is
//   not far below 2^W (est >= W - 64) or when the tile's own partial is not
//   tiny (p >= 2^-60).  Otherwise the thread recomputes the tile in two passes
//   with the row's own tile maximum as the frame (the "careful" path).
// ---------------------------------------------------------------------------
template <int DP, int EP, int R, int BN, bool LSE>
__global__ void __launch_bounds__(kThreads) fwd_kernel(const Args a_) {
    const Args a = batch_view(a_);
    if (a.tc_guard && __uint_as_float(a.tc_guard[0]) + __uint_as_float(a.tc_guard[1]) <= kTcNormLimit)
        return;  // the tensor-core kernel computed this call
    constexpr int PS = pack_stride(DP, EP);
    constexpr int U = unroll_points(DP);
    constexpr float kLog2e = 1.4426950408889634f;
    static_assert(BN % U == 0, "tile must be a multiple of the unroll");
    __shared__ __align__(16) float tile[BN * PS];
    __shared__ float wmax[kThreads / 32][EP];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    zero_pad_coords<DP, PS, BN>(a, tile);
    float xr[R][DP];
    load_rows<DP, R>(a, row0, xr, a.c);

    float part[R][EP], hi[R][EP], lo[R][EP], m[R][EP], est[R][EP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            part[r][e] = hi[r][e] = lo[r][e] = 0.f;
            m[r][e] = est[r][e] = -f_inf();
        }

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + U - 1) / U * U;
        __syncthreads();  // every thread is done with the previous tile
        stage_coords<DP, PS>(a, tile, jt, nv, nvp, a.c, 0.f);

        float W[EP];
        if (!LSE) {
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e)
                    tile[p * PS + DP + e] = (p < nv && e < a.E) ? ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : 0.f;
            }
        } else {
            float lmax[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) lmax[e] = -f_inf();
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const float v = (p < nv && e < a.E) ? kLog2e * ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : -f_inf();
                    tile[p * PS + DP + e] = v;
                    lmax[e] = fmaxf(lmax[e], v);
                }
            }
#pragma unroll
            for (int e = 0; e < EP; ++e) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lmax[e] = fmaxf(lmax[e], __shfl_xor_sync(0xffffffffu, lmax[e], o));
                if ((t & 31) == 0) wmax[t >> 5][e] = lmax[e];
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                W[e] = wmax[0][e];
#pragma unroll
                for (int w = 1; w < kThreads / 32; ++w) W[e] = fmaxf(W[e], wmax[w][e]);
            }
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const float v = tile[p * PS + DP + e];
                    tile[p * PS + DP + e] = (v == -f_inf()) ? f_inf() : W[e] - v;
                }
            }
        }
        __syncthreads();  // tile staged

        // ---- fast pass: every pair once --------------------------------------
        for (int jj = 0; jj < nvp; jj += U) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float pv[PS];
                load_record<PS>(tile + (jj + u) * PS, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    constexpr int NC = dist_chains(DP);
                    float qc[NC];
#pragma unroll
                    for (int c = 0; c < NC; ++c) qc[c] = (c == 0 && LSE && EP == 1) ? pv[DP] : 0.f;
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        const float df = xr[r][d] - pv[d];
                        qc[d % NC] = fmaf(df, df, qc[d % NC]);
                    }
                    float q = qc[0];
#pragma unroll
                    for (int c = 1; c < NC; ++c) q += qc[c];
                    if (!LSE) {
                        const float k = ex2_approx(-q);
#pragma unroll
                        for (int e = 0; e < EP; ++e) part[r][e] = fmaf(k, pv[DP + e], part[r][e]);
                    } else if (EP == 1) {
                        part[r][0] += ex2_approx(-q);
                    } else {
#pragma unroll
                        for (int e = 0; e < EP; ++e) part[r][e] += ex2_approx(-(q + pv[DP + e]));
                    }
                }
            }
        }

        if (!LSE) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    two_sum_add(hi[r][e], lo[r][e], part[r][e]);
                    part[r][e] = 0.f;
                }
            continue;
        }

        // ---- LSE: frames, careful recomputation when needed -----------------
        bool careful = false;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < EP; ++e)
                careful |= !(W[e] <= est[r][e] + 64.f || part[r][e] >= 0x1p-60f);
        float F[R][EP];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < EP; ++e) F[r][e] = W[e];
        if (careful) {
            float umin[R][EP];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) umin[r][e] = f_inf();
            for (int jj = 0; jj < nvp; ++jj) {
                float pv[PS];
                load_record<PS>(tile + jj * PS, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float q = 0.f;
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        const float df = xr[r][d] - pv[d];
                        q = fmaf(df, df, q);
                    }
#pragma unroll
                    for (int e = 0; e < EP; ++e) umin[r][e] = fminf(umin[r][e], q + pv[DP + e]);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    part[r][e] = 0.f;
                    if (umin[r][e] == f_inf()) umin[r][e] = 0.f;  // column empty in this tile
                    F[r][e] = W[e] - umin[r][e];
                }
            for (int jj = 0; jj < nvp; ++jj) {
                float pv[PS];
                load_record<PS>(tile + jj * PS, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float q = 0.f;
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        const float df = xr[r][d] - pv[d];
                        q = fmaf(df, df, q);
                    }
#pragma unroll
                    for (int e = 0; e < EP; ++e) part[r][e] += ex2_approx(umin[r][e] - (q + pv[DP + e]));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const float p = part[r][e];
                if (p > 0.f) {
                    const float mn = fmaxf(m[r][e], F[r][e]);
                    const float so = ex2_approx(m[r][e] - mn);
                    const float sn = ex2_approx(F[r][e] - mn);
                    hi[r][e] *= so;
                    lo[r][e] *= so;
                    two_sum_add(hi[r][e], lo[r][e], p * sn);
                    m[r][e] = mn;
                    est[r][e] = mn + lg2_approx(hi[r][e] + lo[r][e]);
                }
                part[r][e] = 0.f;
            }
    }

    // ---- results ------------------------------------------------------------
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
        if (i >= a.M) continue;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (e >= a.E) continue;
            const int64_t o = i * a.E + e;
            if (!LSE) {
                if (a.S == 1) {
                    st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(hi[r][e] + lo[r][e]));
                } else {
                    const int64_t w = (int64_t)blockIdx.y * a.M * a.E + o;
                    st_chk(a, a.ws0, w, a.ws_n, KRD_WS, (float)(hi[r][e]));
                    st_chk(a, a.ws1, w, a.ws_n, KRD_WS, (float)(lo[r][e]));
                }
            } else {
                const float tot = hi[r][e] + lo[r][e];
                if (a.S == 1) {
                    st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(tot > 0.f ? (float)(0.6931471805599453 * ((double)m[r][e] + log2((double)tot)))
                                         : -f_inf()));
                } else {
                    const int64_t w = (int64_t)blockIdx.y * a.M * a.E + o;
                    st_chk(a, a.ws0, w, a.ws_n, KRD_WS, (float)(tot > 0.f ? m[r][e] : -f_inf()));
                    st_chk(a, a.ws1, w, a.ws_n, KRD_WS, (float)(tot));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Gradient wrt x of sum_ie g_ie a_ie:
//   gx_id = -(2/sigma^2) sum_j k_ij beta_ij (x_id - y_jd),  beta_ij = sum_e g_ie b_je.
// In prescaled units x - y = (x' - y')/c, so gx = gscale * sum_j k beta (x' - y')
// with gscale = -2/(sigma^2 c).  The differences of the distance are reused.
// For E = 1, g_i is factored out of the sum and applied at the end.
// ---------------------------------------------------------------------------
template <int DP, int EP, int R, int BN>
__global__ void __launch_bounds__(kThreads) grad_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PS = pack_stride(DP, EP);
    constexpr int U = unroll_points(DP);
    __shared__ __align__(16) float tile[BN * PS];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    zero_pad_coords<DP, PS, BN>(a, tile);
    float xr[R][DP];
    load_rows<DP, R>(a, row0, xr, a.c);
    float gr[R][EP];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
#pragma unroll
        for (int e = 0; e < EP; ++e) gr[r][e] = (i < a.M && e < a.E) ? ldg_chk(a, a.g, i * a.E + e, a.M * a.E, KRD_G) : 0.f;
    }
    float part[R][DP], hi[R][DP], lo[R][DP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int d = 0; d < DP; ++d) part[r][d] = hi[r][d] = lo[r][d] = 0.f;

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + U - 1) / U * U;
        __syncthreads();
        stage_coords<DP, PS>(a, tile, jt, nv, nvp, a.c, 0.f);
        for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
            for (int e = 0; e < EP; ++e)
                tile[p * PS + DP + e] = (p < nv && e < a.E) ? ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : 0.f;
        }
        __syncthreads();

        for (int jj = 0; jj < nvp; jj += U) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float pv[PS];
                load_record<PS>(tile + (jj + u) * PS, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    constexpr int NC = dist_chains(DP);
                    float df[DP];
                    float qc[NC];
#pragma unroll
                    for (int c = 0; c < NC; ++c) qc[c] = 0.f;
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        df[d] = xr[r][d] - pv[d];
                        qc[d % NC] = fmaf(df[d], df[d], qc[d % NC]);
                    }
                    float q = qc[0];
#pragma unroll
                    for (int c = 1; c < NC; ++c) q += qc[c];
                    float beta;
                    if (EP == 1) {
                        beta = pv[DP];
                    } else {
                        beta = 0.f;
#pragma unroll
                        for (int e = 0; e < EP; ++e) beta = fmaf(gr[r][e], pv[DP + e], beta);
                    }
                    const float kb = ex2_approx(-q) * beta;
#pragma unroll
                    for (int d = 0; d < DP; ++d) part[r][d] = fmaf(kb, df[d], part[r][d]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                two_sum_add(hi[r][d], lo[r][d], part[r][d]);
                part[r][d] = 0.f;
            }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
        if (i >= a.M) continue;
        const float sc = (EP == 1) ? a.gscale * gr[r][0] : a.gscale;
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            if (d >= a.D) continue;
            const int64_t o = i * a.D + d;
            if (a.S == 1) {
                st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)((hi[r][d] + lo[r][d]) * sc));
            } else {
                const int64_t w = (int64_t)blockIdx.y * a.M * a.D + o;
                st_chk(a, a.ws0, w, a.ws_n, KRD_WS, (float)(hi[r][d] * sc));
                st_chk(a, a.ws1, w, a.ws_n, KRD_WS, (float)(lo[r][d] * sc));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// K-min / ArgMin over d_ij = sum_d (x_id - y_jd)^2 (no prescale).
// Each row keeps a register list of the KP smallest (d, j), sorted ascending.
// Points are visited in increasing j and a new pair enters only when strictly
// smaller, so equal distances keep the lower index.
// ---------------------------------------------------------------------------
template <int KP>
__device__ __forceinline__ void knn_insert(float (&dk)[KP], int (&ik)[KP], float q, int j) {
    // Slot k takes the old slot k-1 when the new pair ranks above it, the new
    // pair when it lands exactly at k, and keeps its value otherwise.
#pragma unroll
    for (int k = KP - 1; k > 0; --k) {
        const float da = dk[k - 1], db = dk[k];
        const int ia = ik[k - 1], ib = ik[k];
        const bool above = q < da;
        const bool here = q < db;
        dk[k] = above ? da : (here ? q : db);
        ik[k] = above ? ia : (here ? j : ib);
    }
    if (q < dk[0]) {
        dk[0] = q;
        ik[0] = j;
    }
}

template <int DP, int KP, int R, int BN>
__global__ void __launch_bounds__(kThreads) knn_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PS = pack_stride(DP, 0);
    constexpr int U = unroll_points(DP);
    __shared__ __align__(16) float tile[BN * PS];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    zero_pad_coords<DP, PS, BN>(a, tile);
    float xr[R][DP];
    load_rows<DP, R>(a, row0, xr, 1.f);
    float dk[R][KP];
    int ik[R][KP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            dk[r][k] = f_inf();
            ik[r][k] = -1;
        }

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + U - 1) / U * U;
        __syncthreads();
        stage_coords<DP, PS>(a, tile, jt, nv, nvp, 1.f, f_inf());
        __syncthreads();

        for (int jj = 0; jj < nvp; jj += U) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float pv[PS];
                load_record<PS>(tile + (jj + u) * PS, pv);
                const int j = (int)(jt + jj + u);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    constexpr int NC = dist_chains(DP);  // interleaved partial sums
                    float qc[NC];
#pragma unroll
                    for (int c = 0; c < NC; ++c) qc[c] = 0.f;
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        const float df = xr[r][d] - pv[d];
                        qc[d % NC] = fmaf(df, df, qc[d % NC]);
                    }
                    float q = qc[0];
#pragma unroll
                    for (int c = 1; c < NC; ++c) q += qc[c];
                    if (q < dk[r][KP - 1]) knn_insert<KP>(dk[r], ik[r], q, j);
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
        if (i >= a.M) continue;
        if (a.S == 1) {
#pragma unroll
            for (int k = 0; k < KP; ++k) {
                if (k >= a.K) continue;
                st_chk(a, a.idx, i * a.K + k, a.idx_n, KRD_IDX, (int32_t)(ik[r][k]));
                if (a.out) st_chk(a, a.out, i * a.K + k, a.out_n, KRD_OUT, (float)(dk[r][k]));
            }
        } else {
            const int64_t w = ((int64_t)blockIdx.y * a.M + i) * KP;
#pragma unroll
            for (int k = 0; k < KP; ++k) {
                st_chk(a, a.ws0, w + k, a.ws_n, KRD_WS, (float)(dk[r][k]));
                st_chk(a, a.wsi, w + k, a.ws_n, KRD_WS, (int32_t)(ik[r][k]));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// x-gradient for wide points (32 <= D <= 64).  The same sums as grad_kernel, one row
// per thread, but the compensated running sums (hi, lo) of the D coordinates live in
// dynamic shared memory, laid out [coordinate][hi|lo][thread] so every access of a
// warp is to consecutive words; each thread folds its tile partials into its own
// slots, so no barrier is needed for them.  Registers hold x (D), the differences of
// the current pair (D) and the tile partials (D).  Dynamic shared memory:
// BN * PS + 2 * DP * kThreads floats.
// ---------------------------------------------------------------------------
template <int DP, int EP, int BN>
__global__ void __launch_bounds__(kThreads) gradw_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PS = pack_stride(DP, EP);
    extern __shared__ __align__(16) float wsm[];
    float *tile = wsm;
    float *acc = wsm + BN * PS;  // acc[(2 d + 0|1) kThreads + t] = hi | lo of coordinate d

    const int t = threadIdx.x;
    const int64_t i = (int64_t)blockIdx.x * kThreads + t;
    // After the tensor-core gradient: nothing to do if its guard held (norms, a finite signal),
    // except the rows of this split it flagged as too weak for its fp16 P tile.
    bool mine = true;
    if (a.tc_guard && __uint_as_float(a.tc_guard[0]) + __uint_as_float(a.tc_guard[1]) <= kTcNormLimit &&
        __uint_as_float(a.tc_guard[2]) <= 3.0e38f) {
        mine = a.tc_flags && i < a.M && a.tc_flags[(int64_t)blockIdx.y * a.M + i] != 0;
        if (!__syncthreads_or(mine)) return;
    }
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    zero_pad_coords<DP, PS, BN>(a, tile);
    float xr[DP];
#pragma unroll
    for (int d = 0; d < DP; ++d) xr[d] = (i < a.M && d < a.D) ? a.c * ldg_chk(a, a.x, i * a.D + d, a.M * a.D, KRD_X) : 0.f;
    float gr[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) gr[e] = (i < a.M && e < a.E) ? ldg_chk(a, a.g, i * a.E + e, a.M * a.E, KRD_G) : 0.f;
    float part[DP];
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        part[d] = 0.f;
        acc[(2 * d) * kThreads + t] = 0.f;
        acc[(2 * d + 1) * kThreads + t] = 0.f;
    }

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        __syncthreads();
        stage_coords<DP, PS>(a, tile, jt, nv, nv, a.c, 0.f);
        for (int p = t; p < nv; p += kThreads) {
#pragma unroll
            for (int e = 0; e < EP; ++e) tile[p * PS + DP + e] = e < a.E ? ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : 0.f;
        }
        __syncthreads();

        for (int jj = 0; jj < nv; ++jj) {
            const float4 *rec = reinterpret_cast<const float4 *>(tile + jj * PS);
            constexpr int NC = dist_chains(DP);
            float df[DP];
            float qc[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) qc[c] = 0.f;
#pragma unroll
            for (int k = 0; k < DP / 4; ++k) {  // the record in 16-byte pieces, used at once
                const float4 v = rec[k];
                const float yv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int d = 4 * k + u;
                    df[d] = xr[d] - yv[u];
                    qc[d % NC] = fmaf(df[d], df[d], qc[d % NC]);
                }
            }
#pragma unroll
            for (int d = DP / 4 * 4; d < DP; ++d) {  // the coordinates past the last whole piece
                df[d] = xr[d] - tile[jj * PS + d];
                qc[d % NC] = fmaf(df[d], df[d], qc[d % NC]);
            }
            float q = qc[0];
#pragma unroll
            for (int c = 1; c < NC; ++c) q += qc[c];
            float beta;
            if (EP == 1) {
                beta = tile[jj * PS + DP];
            } else {
                beta = 0.f;
#pragma unroll
                for (int e = 0; e < EP; ++e) beta = fmaf(gr[e], tile[jj * PS + DP + e], beta);
            }
            const float kb = ex2_approx(-q) * beta;
#pragma unroll
            for (int d = 0; d < DP; ++d) part[d] = fmaf(kb, df[d], part[d]);
        }
#pragma unroll
        for (int d = 0; d < DP; ++d) {  // fold the tile into this thread's own slots
            float h = acc[(2 * d) * kThreads + t], l = acc[(2 * d + 1) * kThreads + t];
            two_sum_add(h, l, part[d]);
            acc[(2 * d) * kThreads + t] = h;
            acc[(2 * d + 1) * kThreads + t] = l;
            part[d] = 0.f;
        }
    }

    if (i >= a.M || !mine) return;
    const float sc = (EP == 1) ? a.gscale * gr[0] : a.gscale;
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        if (d >= a.D) continue;
        const float h = acc[(2 * d) * kThreads + t], l = acc[(2 * d + 1) * kThreads + t];
        const int64_t o = i * a.D + d;
        if (a.S == 1) {
            st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)((h + l) * sc));
        } else {
            const int64_t w = (int64_t)blockIdx.y * a.M * a.D + o;
            st_chk(a, a.ws0, w, a.ws_n, KRD_WS, (float)(h * sc));
            st_chk(a, a.ws1, w, a.ws_n, KRD_WS, (float)(l * sc));
        }
    }
}

// ---------------------------------------------------------------------------
// Split-j combines: one thread per output element, partials visited in
// increasing split order, so the result does not depend on scheduling.
// ---------------------------------------------------------------------------
// Sum / grad: total = sum_s (hi_s + lo_s) in fp64.  `W` = E (Sum) or D (grad).
__global__ void combine_sum_kernel(const Args a, int W);
// LSE: (m_s, acc_s) merged as 2^M sum_s acc_s 2^(m_s - M), M = max_s m_s, in fp64.
__global__ void combine_lse_kernel(const Args a);
// K-min: S sorted lists of KP pairs merged by (d, j); empty slots rank last.
__global__ void combine_knn_kernel(const Args a, int KP);
// Max/Min: the largest (value, lowest index) over the splits, times the value sign.
__global__ void combine_max_kernel(const Args a);

}  // namespace kr
