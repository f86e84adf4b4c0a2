// kr_kernels_packed.cuh -- the reduction kernels with packed fp32x2 arithmetic.
//
// Same scheme and same per-pair arithmetic as kr_kernels.cuh, but every FP32
// instruction works on two points at once (FADD2 / FMUL2 / FFMA2 on register
// pairs): the SM's FP32 lanes are the same, but a pair of points now costs half
// the issue slots, so the FP32 pipe rather than instruction issue bounds the loop.
//   * the tile holds pair records: points 2m and 2m+1 interleaved field by field
//     (the coordinates are stored negated, -y', so x' - y' is one FADD2);
//   * each thread keeps its rows as (x'_d, x'_d) register pairs;
//   * the per-point partial sums of even and odd points are kept in the two
//     halves of a float2 and added once per tile.
// Used for D <= 64 (register pairs of x' cost 2 R D registers).
#pragma once

#include "kr_kernels.cuh"

namespace kr {

// Reads one pair record (PS2 floats, 16-byte aligned) as PS2/2 float2 fields.
template <int PS2>
__device__ __forceinline__ void load_pair_record(const float *rec, float2 (&pv)[PS2 / 2]) {
    const float4 *p4 = reinterpret_cast<const float4 *>(rec);
#pragma unroll
    for (int k = 0; k < PS2 / 4; ++k) {
        const float4 v = p4[k];
        pv[2 * k + 0] = make_float2(v.x, v.y);
        pv[2 * k + 1] = make_float2(v.z, v.w);
    }
}

// Rows of x owned by this thread, times `scale`, as duplicated register pairs.
template <int DP, int R>
__device__ __forceinline__ void load_rows_pairs(const Args &a, int64_t row0, float2 (&x2)[R][DP], float scale) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + threadIdx.x;
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            const float v = (i < a.M && d < a.D) ? scale * ldg_chk(a, a.x, i * a.D + d, a.M * a.D, KRD_X) : 0.f;
            x2[r][d] = make_float2(v, v);
        }
    }
}

// Field slot of point p: record p/2, half p%2.
template <int PS2>
__device__ __forceinline__ float *pair_slot(float *tile, int p, int field) {
    return tile + (p >> 1) * PS2 + 2 * field + (p & 1);
}

// Coordinates of points [jt, jt + nv) into pair records, times `scale`; padding
// points [nv, nvp) get coordinate 0 = `pad0` and zeros.
template <int DP, int PS2>
__device__ __forceinline__ void stage_coords_pairs(const Args &a, float *tile, int64_t jt, int nv, int nvp,
                                                   float scale, float pad0) {
    for (int p = threadIdx.x; p < nvp; p += kThreads) {
        if (p < nv) {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) *pair_slot<PS2>(tile, p, d) = scale * ldg_chk(a, a.y, (jt + p) * a.D + d, a.N * a.D, KRD_Y);
        } else {
#pragma unroll
            for (int d = 0; d < DP; ++d)
                if (d < a.D) *pair_slot<PS2>(tile, p, d) = (d == 0) ? pad0 : 0.f;
        }
    }
}

template <int DP, int PS2, int BN>
__device__ __forceinline__ void zero_pad_coords_pairs(const Args &a, float *tile) {
    if (a.D < DP) {
        for (int f = threadIdx.x; f < BN * DP; f += kThreads) {
            const int p = f / DP, d = f % DP;
            if (d >= a.D) *pair_slot<PS2>(tile, p, d) = 0.f;
        }
    }
}

// q = |x' - y'|^2 for the two points of a record (coordinates stored negated).
template <int DP, int PS2>
__device__ __forceinline__ float2 sq_dist_pair(const float2 (&x2)[DP], const float2 (&pv)[PS2 / 2], float2 q0,
                                               bool start_from_q0) {
    constexpr int NC = dist_chains(DP);  // interleaved partial sums (see kr_config.h)
    float2 qc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) qc[c] = q0;
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        const float2 df = __fadd2_rn(x2[d], pv[d]);
        const int c = d % NC;
        const bool first = d < NC && !(c == 0 && start_from_q0);
        qc[c] = first ? __fmul2_rn(df, df) : __ffma2_rn(df, df, qc[c]);
    }
    float2 q = qc[0];
#pragma unroll
    for (int c = 1; c < NC; ++c) q = __fadd2_rn(q, qc[c]);
    return q;
}

// ---------------------------------------------------------------------------
// Sum / LogSumExp (packed).  Value fields: b_je (Sum) or W_e - w'_je (LSE), as in
// fwd_kernel; the LSE tile frame and careful path are the same.
// ---------------------------------------------------------------------------
//
// REC (streamed records, D <= 16): the tiles come ready-made from the prepass (pack
// kernel below): pair records of -y' and b (Sum) or of -y' and W - w' (LSE), with the
// tile frame W in a.wtile.  They are copied into two shared-memory buffers with cp.async:
// while the block scans tile k, the copy of tile k + 1 is in flight, and one barrier per
// tile separates them.  a.chunk is then a multiple of BN, so every block's tiles are the
// prepass's tiles.
template <int DP, int EP, int R, int BN, bool LSE, bool REC>
__global__ void __launch_bounds__(kThreads) fwd2_kernel(const Args a_) {
    const Args a = batch_view(a_);
    if (a.tc_guard && __uint_as_float(a.tc_guard[0]) + __uint_as_float(a.tc_guard[1]) <= kTcNormLimit)
        return;  // the tensor-core kernel computed this call
    constexpr int PS2 = pair_stride(DP, EP);
    constexpr int UP = unroll_pairs(DP);
    constexpr int UPT = 2 * UP;
    constexpr int TF = record_tile_floats(DP, EP, BN);
    constexpr float kLog2e = 1.4426950408889634f;
    static_assert(BN % UPT == 0, "tile must be a multiple of the unroll");
    __shared__ __align__(16) float stile[REC ? 4 : TF];
    __shared__ float wmax[kThreads / 32][EP];
    float *const tbuf = REC ? reinterpret_cast<float *>(kr_dyn_smem) : stile;

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    if constexpr (REC) {
        if (j_begin < j_end) issue_record_tile<TF>(a, tbuf, j_begin / BN);
    } else {
        zero_pad_coords_pairs<DP, PS2, BN>(a, tbuf);
    }
    float2 x2[R][DP];
    load_rows_pairs<DP, R>(a, row0, x2, a.c);

    float2 part2[R][EP];
    float hi[R][EP], lo[R][EP], m[R][EP], est[R][EP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            part2[r][e] = make_float2(0.f, 0.f);
            hi[r][e] = lo[r][e] = 0.f;
            m[r][e] = est[r][e] = -f_inf();
        }

    int kt = 0;
    for (int64_t jt = j_begin; jt < j_end; jt += BN, ++kt) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + UPT - 1) / UPT * UPT;
        float W[EP];
        const float *tile;
        if constexpr (REC) {
            tile = tbuf + (kt & 1) * TF;
            if (LSE) {
#pragma unroll
                for (int e = 0; e < EP; ++e) W[e] = ldg_chk(a, (const float *)a.wtile, (jt / BN) * EP + e, a.wtile_n, KRD_WS);
            }
            cp_async_wait_all();
            __syncthreads();  // tile kt landed; every thread is done with the other buffer
            if (jt + BN < j_end) issue_record_tile<TF>(a, tbuf + ((kt + 1) & 1) * TF, jt / BN + 1);
        } else {
            tile = tbuf;
            __syncthreads();
            stage_coords_pairs<DP, PS2>(a, tbuf, jt, nv, nvp, -a.c, 0.f);
        }

        if (REC) {
        } else if (!LSE) {
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e)
                    *pair_slot<PS2>(tbuf, p, DP + e) = (p < nv && e < a.E) ? ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : 0.f;
            }
        } else {
            float lmax[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) lmax[e] = -f_inf();
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const float v = (p < nv && e < a.E) ? kLog2e * ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : -f_inf();
                    *pair_slot<PS2>(tbuf, p, DP + e) = v;
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
                    float *slot = pair_slot<PS2>(tbuf, p, DP + e);
                    const float v = *slot;
                    *slot = (v == -f_inf()) ? f_inf() : W[e] - v;
                }
            }
        }
        if (!REC) __syncthreads();

        // ---- fast pass ------------------------------------------------------------
        // the Sum's loop is unrolled four steps deep (4 % faster at D = 3); the LogSumExp's is
        // not (slower so)
#pragma unroll(LSE ? 1 : 4)
        for (int jj = 0; jj < nvp; jj += UPT) {
#pragma unroll
            for (int u = 0; u < UP; ++u) {
                float2 pv[PS2 / 2];
                load_pair_record<PS2>(tile + ((jj >> 1) + u) * PS2, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const bool fold = LSE && EP == 1;
                    const float2 q = sq_dist_pair<DP, PS2>(x2[r], pv, fold ? pv[DP] : make_float2(0.f, 0.f), fold);
                    if (!LSE) {
                        const float2 k2 = make_float2(ex2_approx(-q.x), ex2_approx(-q.y));
#pragma unroll
                        for (int e = 0; e < EP; ++e) part2[r][e] = __ffma2_rn(k2, pv[DP + e], part2[r][e]);
                    } else if (EP == 1) {
                        part2[r][0] = __fadd2_rn(part2[r][0], make_float2(ex2_approx(-q.x), ex2_approx(-q.y)));
                    } else {
#pragma unroll
                        for (int e = 0; e < EP; ++e) {
                            const float2 tq = __fadd2_rn(q, pv[DP + e]);
                            part2[r][e] = __fadd2_rn(part2[r][e], make_float2(ex2_approx(-tq.x), ex2_approx(-tq.y)));
                        }
                    }
                }
            }
        }

        float part[R][EP];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                part[r][e] = part2[r][e].x + part2[r][e].y;
                part2[r][e] = make_float2(0.f, 0.f);
            }
        if (!LSE) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) two_sum_add(hi[r][e], lo[r][e], part[r][e]);
            continue;
        }

        // ---- LSE: frames, careful recomputation when needed ---------------------
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
            for (int jj = 0; jj < nvp; jj += 2) {
                float2 pv[PS2 / 2];
                load_pair_record<PS2>(tile + (jj >> 1) * PS2, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 q = sq_dist_pair<DP, PS2>(x2[r], pv, make_float2(0.f, 0.f), false);
#pragma unroll
                    for (int e = 0; e < EP; ++e) {
                        const float2 tq = __fadd2_rn(q, pv[DP + e]);
                        umin[r][e] = fminf(umin[r][e], fminf(tq.x, tq.y));
                    }
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
            for (int jj = 0; jj < nvp; jj += 2) {
                float2 pv[PS2 / 2];
                load_pair_record<PS2>(tile + (jj >> 1) * PS2, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 q = sq_dist_pair<DP, PS2>(x2[r], pv, make_float2(0.f, 0.f), false);
#pragma unroll
                    for (int e = 0; e < EP; ++e) {
                        const float2 tq = __fadd2_rn(q, pv[DP + e]);
                        part[r][e] += ex2_approx(umin[r][e] - tq.x) + ex2_approx(umin[r][e] - tq.y);
                    }
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
            }
    }

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
// x-gradient (packed): the same sum as grad_kernel, two points per instruction.
// ---------------------------------------------------------------------------
// REC: the tiles are streamed from the prepass records (-y', b), double-buffered, as in
// fwd2_kernel.
template <int DP, int EP, int R, int BN, bool REC>
__global__ void __launch_bounds__(kThreads) grad2_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PS2 = pair_stride(DP, EP);
    constexpr int UP = unroll_pairs(DP);
    constexpr int UPT = 2 * UP;
    constexpr int TF = record_tile_floats(DP, EP, BN);
    static_assert(BN % UPT == 0, "tile must be a multiple of the unroll");
    __shared__ __align__(16) float stile[REC ? 4 : TF];
    float *const tbuf = REC ? reinterpret_cast<float *>(kr_dyn_smem) : stile;

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    if constexpr (REC) {
        if (j_begin < j_end) issue_record_tile<TF>(a, tbuf, j_begin / BN);
    } else {
        zero_pad_coords_pairs<DP, PS2, BN>(a, tbuf);
    }
    float2 x2[R][DP];
    load_rows_pairs<DP, R>(a, row0, x2, a.c);
    float gr[R][EP];
    float2 g2[R][EP];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            gr[r][e] = (i < a.M && e < a.E) ? ldg_chk(a, a.g, i * a.E + e, a.M * a.E, KRD_G) : 0.f;
            g2[r][e] = make_float2(gr[r][e], gr[r][e]);
        }
    }
    float2 part2[R][DP];
    float hi[R][DP], lo[R][DP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            part2[r][d] = make_float2(0.f, 0.f);
            hi[r][d] = lo[r][d] = 0.f;
        }

    int kt = 0;
    for (int64_t jt = j_begin; jt < j_end; jt += BN, ++kt) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + UPT - 1) / UPT * UPT;
        const float *tile;
        if constexpr (REC) {
            tile = tbuf + (kt & 1) * TF;
            cp_async_wait_all();
            __syncthreads();  // tile kt landed; every thread is done with the other buffer
            if (jt + BN < j_end) issue_record_tile<TF>(a, tbuf + ((kt + 1) & 1) * TF, jt / BN + 1);
        } else {
            tile = tbuf;
            __syncthreads();
            stage_coords_pairs<DP, PS2>(a, tbuf, jt, nv, nvp, -a.c, 0.f);
            for (int p = t; p < nvp; p += kThreads) {
#pragma unroll
                for (int e = 0; e < EP; ++e)
                    *pair_slot<PS2>(tbuf, p, DP + e) = (p < nv && e < a.E) ? ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B) : 0.f;
            }
            __syncthreads();
        }

        for (int jj = 0; jj < nvp; jj += UPT) {
#pragma unroll
            for (int u = 0; u < UP; ++u) {
                float2 pv[PS2 / 2];
                load_pair_record<PS2>(tile + ((jj >> 1) + u) * PS2, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float2 df[DP];
                    float2 q = make_float2(0.f, 0.f);
#pragma unroll
                    for (int d = 0; d < DP; ++d) {
                        df[d] = __fadd2_rn(x2[r][d], pv[d]);
                        q = d == 0 ? __fmul2_rn(df[d], df[d]) : __ffma2_rn(df[d], df[d], q);
                    }
                    float2 beta;
                    if (EP == 1) {
                        beta = pv[DP];
                    } else {
                        beta = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < EP; ++e) beta = __ffma2_rn(g2[r][e], pv[DP + e], beta);
                    }
                    const float2 kb = __fmul2_rn(make_float2(ex2_approx(-q.x), ex2_approx(-q.y)), beta);
#pragma unroll
                    for (int d = 0; d < DP; ++d) part2[r][d] = __ffma2_rn(kb, df[d], part2[r][d]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                two_sum_add(hi[r][d], lo[r][d], part2[r][d].x + part2[r][d].y);
                part2[r][d] = make_float2(0.f, 0.f);
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
// K-min (packed direct distances, 32 <= D <= 64; smaller D take the filtered kernel
// below).  The threshold test is taken once per row for a group of UPT points (the
// minimum of their distances against the list's last entry); a passing group's
// points are walked in increasing j from a bit mask and inserted into the sorted
// register list.  Insertion is strictly-smaller and in increasing j, so equal
// distances keep the lower index.
// ---------------------------------------------------------------------------
template <int DP, int KP, int R, int BN>
__global__ void __launch_bounds__(kThreads) knn2_kernel(const Args a_) {
    const Args a = batch_view(a_);
    if (a.tc_guard && tc_knn_ran(a.tc_guard)) return;  // the tensor-core K-min did this call
    constexpr int PS2 = pair_stride(DP, 0);
    constexpr int UP = unroll_pairs(DP);
    constexpr int UPT = 2 * UP;
    static_assert(BN % UPT == 0, "tile must be a multiple of the unroll");
    __shared__ __align__(16) float tile[(BN / 2) * PS2];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    zero_pad_coords_pairs<DP, PS2, BN>(a, tile);
    float2 x2[R][DP];
    load_rows_pairs<DP, R>(a, row0, x2, 1.f);
    float dk[R][KP];
    int ik[R][KP];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            dk[r][k] = f_inf();
            ik[r][k] = -1;
        }
    }

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + UPT - 1) / UPT * UPT;
        __syncthreads();
        stage_coords_pairs<DP, PS2>(a, tile, jt, nv, nvp, -1.f, -f_inf());
        __syncthreads();

        for (int jj = 0; jj < nvp; jj += UPT) {
            float2 q[UP][R];
#pragma unroll
            for (int u = 0; u < UP; ++u) {
                float2 pv[PS2 / 2];
                load_pair_record<PS2>(tile + ((jj >> 1) + u) * PS2, pv);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    q[u][r] = sq_dist_pair<DP, PS2>(x2[r], pv, make_float2(0.f, 0.f), false);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float mn = fminf(q[0][r].x, q[0][r].y);
#pragma unroll
                for (int u = 1; u < UP; ++u) mn = fminf(mn, fminf(q[u][r].x, q[u][r].y));
                if (mn < dk[r][KP - 1]) {
                    const float thr = dk[r][KP - 1];
                    unsigned mask = 0;
#pragma unroll
                    for (int u = 0; u < UP; ++u) {
                        mask |= (q[u][r].x < thr ? 1u : 0u) << (2 * u);
                        mask |= (q[u][r].y < thr ? 1u : 0u) << (2 * u + 1);
                    }
                    const int j0 = (int)(jt + jj);
                    while (mask) {
                        const int c = __ffs(mask) - 1;
                        mask &= mask - 1;
                        float2 qq = q[0][r];
#pragma unroll
                        for (int u = 1; u < UP; ++u) qq = ((c >> 1) == u) ? q[u][r] : qq;
                        knn_insert<KP>(dk[r], ik[r], (c & 1) ? qq.y : qq.x, j0 + c);
                    }
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
// K-min with an expansion filter (D <= 16).
//
// Which y_j rank first for a row x only depends on |y_j|^2 - 2 x.y_j (|x|^2 is the
// same for every j): D FMAs a pair, against D subtractions and D FMAs for |x - y|^2.
// In fp32 that value cancels when |x| and |y| are large against the distance, so here
// it only screens: a group of points whose filter values all lie above a bound T is
// skipped, T being placed so that a skipped point's direct fp32 distance cannot lie
// below the current K-th distance thr, i.e. it could not have been inserted.  Every
// other group gets the direct fp32 distance (the arithmetic of the unfiltered
// kernels, from the exact coordinates) and is inserted by that value, so the list is
// the one the unfiltered scan produces.
//
// The block subtracts c, the mean of its rows of x, from x and y before the filter
// (x~ = fl(x - c), y~ = fl(y - c)), so an offset common to the data does not loosen
// the bound.  For point j and row i:
//   f_ij = h_j + sum_d x~_id (-y~_jd),   h_j = fl(|y~_j|^2) (1 - kappa) / 2,
//   T_i  = ((thr_i + 2^-100 + kappa (|x~_i|^2 + thr_i)) - |x~_i|^2) / 2.
// f_ij > T_i means |x~ - y~|^2 > thr + 2^-100 + kappa Q (Q = |x~|^2 + |y~|^2 + thr) up
// to the rounding of f, h, T, of the centring and of the direct distance, which in
// all stays below (3D + 7) u Q (u = 2^-24) plus a few 2^-126 (flushed subnormals);
// kappa = (8D + 12) u is more than twice that and 2^-100 covers the absolute part,
// so the direct distance is >= thr.  A point with |y~|^2 not below 2^100 (or NaN)
// gets h = -inf and a row with |x~|^2 not below 2^100 gets T = +inf: they always
// pass, and the direct distance decides.  (Non-finite coordinates give a non-finite
// or NaN direct distance, which is never inserted, so their filter values need no
// bound.)
// ---------------------------------------------------------------------------
template <int DP>
__device__ __forceinline__ float knn_filter_bound(float thr, float xx) {
    constexpr float kappa = knn_kappa(DP);
    if (!(xx < 0x1p100f)) return f_inf();
    return 0.5f * (fmaf(kappa, xx + thr, thr + 0x1p-100f) - xx);
}

// |x~|^2 of a row held as duplicated register pairs (fp32 fma chain).
template <int DP>
__device__ __forceinline__ float sq_norm_pairs(const float2 (&x2)[DP]) {
    float s = x2[0].x * x2[0].x;
#pragma unroll
    for (int d = 1; d < DP; ++d) s = fmaf(x2[d].x, x2[d].x, s);
    return s;
}

// Filter values of the two points of a filter record (fields -y~_d, then h).
template <int DP, int PSF>
__device__ __forceinline__ float2 filter_pair(const float2 (&x2)[DP], const float2 (&pv)[PSF / 2]) {
    constexpr int NC = dist_chains(DP);
    float2 acc[NC];
    acc[0] = __ffma2_rn(x2[0], pv[0], pv[DP]);
#pragma unroll
    for (int c = 1; c < NC; ++c) acc[c] = __fmul2_rn(x2[c], pv[c]);
#pragma unroll
    for (int d = NC; d < DP; ++d) acc[d % NC] = __ffma2_rn(x2[d], pv[d], acc[d % NC]);
    float2 f = acc[0];
#pragma unroll
    for (int c = 1; c < NC; ++c) f = __fadd2_rn(f, acc[c]);
    return f;
}

// Exact coordinates of row i as duplicated register pairs (zero beyond M and D).
template <int DP>
__device__ __forceinline__ void load_row_exact(const Args &a, int64_t i, float2 (&xe)[DP]) {
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        const float v = (i < a.M && d < a.D) ? ldg_chk(a, a.x, i * a.D + d, a.M * a.D, KRD_X) : 0.f;
        xe[d] = make_float2(v, v);
    }
}

// Direct fp32 distances of the UP exact records from rec0 on.
template <int DP, int PSE, int UP>
__device__ __forceinline__ void knnx_exact_group(const float2 (&xe)[DP], const float *tileE, int rec0,
                                                 float2 (&q)[UP]) {
#pragma unroll
    for (int u = 0; u < UP; ++u) {
        float2 pv[PSE / 2];
        load_pair_record<PSE>(tileE + (rec0 + u) * PSE, pv);
        q[u] = sq_dist_pair<DP, PSE>(xe, pv, make_float2(0.f, 0.f), false);
    }
}

// Inserts the points of a group (distances q, first index j0) that beat the row's
// current K-th distance, in increasing j.
template <int KP, int UP>
__device__ __forceinline__ void knnx_insert_group(const float2 (&q)[UP], float (&dk)[KP], int (&ik)[KP], int64_t j0) {
    const float thr = dk[KP - 1];
    unsigned mask = 0;
#pragma unroll
    for (int u = 0; u < UP; ++u) {
        mask |= (q[u].x < thr ? 1u : 0u) << (2 * u);
        mask |= (q[u].y < thr ? 1u : 0u) << (2 * u + 1);
    }
    while (mask) {  // usually one point
        const int c = __ffs(mask) - 1;
        mask &= mask - 1;
        float2 qq = q[0];
#pragma unroll
        for (int u = 1; u < UP; ++u) qq = ((c >> 1) == u) ? q[u] : qq;
        knn_insert<KP>(dk, ik, (c & 1) ? qq.y : qq.x, (int)(j0 + c));
    }
}

// Tile of the filtered K-min: exact records -y (padding: -inf in coordinate 0, so the
// direct distance is +inf) and filter records -y~ and h (padding: zeros and h = +inf,
// so f = +inf).  Coordinates d >= D are zero in both.
template <int DP, int PSF, int PSE>
__device__ __forceinline__ void stage_knn_filter(const Args &a, float *tileF, float *tileE, const float *cen,
                                                 int64_t jt, int nv, int nvp) {
    constexpr float kH = 0.5f * (1.0f - knn_kappa(DP));
    for (int p = threadIdx.x; p < nvp; p += kThreads) {
        if (p < nv) {
            float yy = 0.f;
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                const float v = d < a.D ? ldg_chk(a, a.y, (jt + p) * a.D + d, a.N * a.D, KRD_Y) : 0.f;
                const float w = v - cen[d];
                *pair_slot<PSE>(tileE, p, d) = -v;
                *pair_slot<PSF>(tileF, p, d) = -w;
                yy = (d == 0) ? w * w : fmaf(w, w, yy);
            }
            *pair_slot<PSF>(tileF, p, DP) = (yy < 0x1p100f) ? kH * yy : -f_inf();
        } else {
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                *pair_slot<PSE>(tileE, p, d) = (d == 0) ? -f_inf() : 0.f;
                *pair_slot<PSF>(tileF, p, d) = 0.f;
            }
            *pair_slot<PSF>(tileF, p, DP) = f_inf();
        }
    }
}

// Drains the queues of one thread's rows, all 32 lanes together, in the order the
// entries were made.  An entry is (block << 8) | mask: bit g of mask marks group
// block * IB + g of the tile.  The groups of an entry are taken two at a time, both
// groups' distances computed before the first insertion (the second's test then sees
// the threshold the first left).
template <int DP, int KP, int R, int PSE, int UP, int IB>
__device__ __forceinline__ void knnx_drain(const Args &a, int64_t row0, const float2 (&x2)[R][DP], float (&T)[R],
                                           float (&dk)[R][KP], int (&ik)[R][KP], int (&nc)[R],
                                           const uint16_t *qbuf, const float *tileE, int64_t jt, int CB) {
    constexpr int UPT = 2 * UP;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int steps = __reduce_max_sync(0xffffffffu, nc[r]);
        if (steps == 0) continue;
        float2 xe[DP];
        load_row_exact<DP>(a, row0 + (int64_t)r * kThreads + threadIdx.x, xe);
        const uint16_t *slot = qbuf + r * CB * kThreads + threadIdx.x;
        for (int s = 0; s < steps; ++s) {
            const unsigned e = s < nc[r] ? (unsigned)slot[s * kThreads] : 0u;
            unsigned mask = e & 0xffu;
            const int g_base = (int)(e >> 8) * IB;
            while (mask) {
                const int g0 = g_base + __ffs(mask) - 1;
                mask &= mask - 1;
                const bool two = mask != 0;
                const int g1 = two ? g_base + __ffs(mask) - 1 : g0;
                mask &= mask - 1;
                float2 q0[UP], q1[UP];
                knnx_exact_group<DP, PSE, UP>(xe, tileE, g0 * UP, q0);
                knnx_exact_group<DP, PSE, UP>(xe, tileE, g1 * UP, q1);
                knnx_insert_group<KP, UP>(q0, dk[r], ik[r], jt + g0 * UPT);
                if (two) knnx_insert_group<KP, UP>(q1, dk[r], ik[r], jt + g1 * UPT);
            }
        }
        nc[r] = 0;
        T[r] = knn_filter_bound<DP>(dk[r][KP - 1], sq_norm_pairs<DP>(x2[r]));
    }
}

template <int DP, int KP, int R, int BN>
__global__ void __launch_bounds__(kThreads, knn_min_blocks(DP, KP)) knnx_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int PSF = pair_stride(DP, 1);
    constexpr int PSE = pair_stride(DP, 0);
    constexpr int UP = unroll_pairs(DP);
    constexpr int UPT = 2 * UP;
    constexpr int CB = knnx_queue(DP, KP);
    constexpr int IB = CB > 0 ? knnx_mask_groups(DP, KP) : 1;  // groups per block
    constexpr int BP = IB * UPT;                                 // points per block
    static_assert(IB <= 8, "a block's mask is one byte of the entry");
    static_assert(BN % BP == 0, "tile must be a multiple of the block");
    static_assert(BN / BP <= 256, "block index is one byte of the entry");
    static_assert(knn_tile_bytes(DP, BN) + (CB > 0 ? R * CB * kThreads * 2 : 0) <= 45056, "shared memory");
    __shared__ __align__(16) float tileF[(BN / 2) * PSF];
    __shared__ __align__(16) float tileE[(BN / 2) * PSE];
    // per row r, slot s, thread t: qbuf[(r CB + s) kThreads + t] = (block << 8) | pass mask
    __shared__ uint16_t qbuf[CB > 0 ? R * CB * kThreads : 1];
    __shared__ float cpart[kThreads / 32][2 * DP];
    __shared__ float cen[DP];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * (kThreads * R);
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);

    // Centre: mean of the block's rows of x, per coordinate over its finite values,
    // summed in a fixed order (lane 0 of each warp, then the warps in turn).
    float2 x2[R][DP];
    load_rows_pairs<DP, R>(a, row0, x2, 1.f);
    {
        float s[DP], n[DP];
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            s[d] = 0.f;
            n[d] = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float v = x2[r][d].x;
                if (row0 + (int64_t)r * kThreads + t < a.M && isfinite(v)) {
                    s[d] += v;
                    n[d] += 1.f;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s[d] += __shfl_xor_sync(0xffffffffu, s[d], o);
                n[d] += __shfl_xor_sync(0xffffffffu, n[d], o);
            }
        }
        if ((t & 31) == 0) {
#pragma unroll
            for (int d = 0; d < DP; ++d) {
                cpart[t >> 5][d] = s[d];
                cpart[t >> 5][DP + d] = n[d];
            }
        }
        __syncthreads();
        if (t < DP) {
            float S = 0.f, Nn = 0.f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                S += cpart[w][t];
                Nn += cpart[w][DP + t];
            }
            cen[t] = Nn > 0.f ? S / Nn : 0.f;
        }
        __syncthreads();
    }
    float T[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            const float w = x2[r][d].x - cen[d];
            x2[r][d] = make_float2(w, w);
        }
        T[r] = f_inf();
    }

    float dk[R][KP];
    int ik[R][KP];
    int nc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            dk[r][k] = f_inf();
            ik[r][k] = -1;
        }
        nc[r] = 0;
    }

    for (int64_t jt = j_begin; jt < j_end; jt += BN) {
        const int nv = (int)min((int64_t)BN, j_end - jt);
        const int nvp = (nv + BP - 1) / BP * BP;
        __syncthreads();
        stage_knn_filter<DP, PSF, PSE>(a, tileF, tileE, cen, jt, nv, nvp);
        __syncthreads();

        for (int jb = 0; jb < nvp; jb += BP) {
            unsigned m[R];
#pragma unroll
            for (int r = 0; r < R; ++r) m[r] = 0u;
#pragma unroll
            for (int gg = 0; gg < IB; ++gg) {
                const int jj = jb + gg * UPT;
                float2 f[UP][R];
#pragma unroll
                for (int u = 0; u < UP; ++u) {
                    float2 pv[PSF / 2];
                    load_pair_record<PSF>(tileF + ((jj >> 1) + u) * PSF, pv);
#pragma unroll
                    for (int r = 0; r < R; ++r) f[u][r] = filter_pair<DP, PSF>(x2[r], pv);
                }
                bool any = false;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float mn = fminf(f[0][r].x, f[0][r].y);
#pragma unroll
                    for (int u = 1; u < UP; ++u) mn = fmin3(mn, f[u][r].x, f[u][r].y);
                    const bool pass = !(mn > T[r]);
                    m[r] |= pass ? (1u << gg) : 0u;
                    any |= pass;
                }
                if (CB == 0 && any) {
                    // insert at once: one branch for all rows, rarely taken late in a scan
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (m[r] == 0u) continue;
                        float2 xe[DP], q[UP];
                        load_row_exact<DP>(a, row0 + (int64_t)r * kThreads + t, xe);
                        knnx_exact_group<DP, PSE, UP>(xe, tileE, jj >> 1, q);
                        knnx_insert_group<KP, UP>(q, dk[r], ik[r], jt + jj);
                        T[r] = knn_filter_bound<DP>(dk[r][KP - 1], sq_norm_pairs<DP>(x2[r]));
                    }
                }
            }
            if (CB > 0) {
                // one entry per row and block, kept (the count advanced) only if a bit is set
                int nm = 0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (smem_ok(a, nc[r], CB))
                        qbuf[(r * CB + nc[r]) * kThreads + t] = (uint16_t)(((jb / BP) << 8) | m[r]);
                    nc[r] += m[r] != 0u ? 1 : 0;
                    nm = max(nm, nc[r]);
                }
                if (__any_sync(0xffffffffu, nm >= CB))  // a full queue is drained before the next block
                    knnx_drain<DP, KP, R, PSE, UP, IB>(a, row0, x2, T, dk, ik, nc, qbuf, tileE, jt, CB > 0 ? CB : 1);
            }
        }
        if (CB > 0)  // the entries name points of this tile: drain before it is replaced
            knnx_drain<DP, KP, R, PSE, UP, IB>(a, row0, x2, T, dk, ik, nc, qbuf, tileE, jt, CB > 0 ? CB : 1);
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

}  // namespace kr
