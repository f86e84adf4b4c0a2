// kr_radial.cuh -- Sum and Max/Min reductions of k(x_i, y_j) b_je for the radial
// kernels other than the tuned Gaussian Sum:
//   Gaussian   exp(-|x-y|^2/sigma^2) = 2^(-|x'-y'|^2),  x' = x sqrt(log2 e)/sigma
//   Laplace    exp(-|x-y|/sigma)     = 2^(-|x'-y'|),    x' = x log2 e/sigma
//   Cauchy     1/(1 + |x-y|^2/sigma^2) = 1/(1 + |x'-y'|^2),       x' = x/sigma
//   inverse multiquadric 1/sqrt(1 + |x-y|^2/sigma^2) = rsqrt(1 + |x'-y'|^2)
// ("Kernel Operations on the GPU...", §2: reductions of generic formulas, sum /
// max / min / argmin; KeOps README: a wide range of formulas; Sum, Min, Max,
// ArgMin, ArgMax reductions).
//
// Same tiling as the Gaussian kernels: a thread keeps R rows of x' in registers,
// the block stages tiles of y' (negated, so x' - y' is one add) and b in shared
// memory, and every thread reads each record with broadcast 16-byte loads.  One
// body serves two lane widths: L = 2 evaluates two points per instruction on
// f32x2 register pairs (coordinate counts up to 64), L = 1 is the scalar form
// (128 coordinates, whose register pairs would not fit).
//
// Sum: per-tile fp32 partials folded into a compensated (TwoSum) running pair.
// Max: per (row, column) the best value and its index.  The values of a group of
// points are compared with the best once (their maximum); only when that test
// passes are the points walked in increasing j, replacing the best on a strictly
// larger value, so equal values keep the lowest index.  Min is Max of k (-b):
// the block stages -b and the result is negated on output.  Padding points carry
// b = NaN: k NaN is NaN, which neither wins a comparison nor survives fmaxf.  With
// one signal column (and packed lanes) the scan compares a key that falls as |k b|
// rises instead of the values (log_key), in a mode each block picks from the signs of
// its chunk's signal, and forms the value once a row; the value scan remains for the
// other cases.
#pragma once

#include <type_traits>

#include "kr_kernels_packed.cuh"

namespace kr {

enum RadialKind { KT_GAUSS = 0, KT_LAPLACE = 1, KT_CAUCHY = 2, KT_IMQ = 3 };

// +inf as a constant expression
KR_HD constexpr float f_inf_c() { return __builtin_huge_valf(); }
enum RadialRed { RR_SUM = 0, RR_MAX = 1 };

__device__ __forceinline__ float sqrt_approx(float v) {
    float r;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rsqrt_approx(float v) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// k as a function of the prescaled squared distance (plus 1 for Cauchy and the
// inverse multiquadric, folded into the start of the distance sum).
template <int KT>
__device__ __forceinline__ float radial_value(float q) {
    if (KT == KT_GAUSS) return ex2_approx(-q);
    if (KT == KT_LAPLACE) return ex2_approx(-sqrt_approx(q));
    if (KT == KT_CAUCHY) return rcp_approx(q);
    return rsqrt_approx(q);
}
template <int KT>
KR_HD constexpr float radial_q0() { return (KT == KT_CAUCHY || KT == KT_IMQ) ? 1.f : 0.f; }

// ---- lane-width abstraction: float (L = 1) or float2 (L = 2) ------------------------
template <int L> struct Lanes;
template <> struct Lanes<1> {
    typedef float T;
    static __device__ __forceinline__ T splat(float v) { return v; }
    // explicitly rounded, so no context contracts them differently (Max recomputes values)
    static __device__ __forceinline__ T add(T a, T b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ T mul(T a, T b) { return __fmul_rn(a, b); }
    static __device__ __forceinline__ T fma(T a, T b, T c) { return __fmaf_rn(a, b, c); }
    static __device__ __forceinline__ float lane(T v, int) { return v; }
    static __device__ __forceinline__ float hmax(T v) { return v; }
    static __device__ __forceinline__ float max_into(float m, T v) { return fmaxf(m, v); }
    static __device__ __forceinline__ float hsum(T v) { return v; }
    template <int KT>
    static __device__ __forceinline__ T kval(T q) { return radial_value<KT>(q); }
};
template <> struct Lanes<2> {
    typedef float2 T;
    static __device__ __forceinline__ T splat(float v) { return make_float2(v, v); }
    static __device__ __forceinline__ T add(T a, T b) { return __fadd2_rn(a, b); }
    static __device__ __forceinline__ T mul(T a, T b) { return __fmul2_rn(a, b); }
    static __device__ __forceinline__ T fma(T a, T b, T c) { return __ffma2_rn(a, b, c); }
    static __device__ __forceinline__ float lane(T v, int l) { return l ? v.y : v.x; }
    static __device__ __forceinline__ float hmax(T v) { return fmaxf(v.x, v.y); }
    static __device__ __forceinline__ float max_into(float m, T v) { return fmax3(m, v.x, v.y); }
    static __device__ __forceinline__ float hsum(T v) { return v.x + v.y; }
    template <int KT>
    static __device__ __forceinline__ T kval(T q) { return make_float2(radial_value<KT>(q.x), radial_value<KT>(q.y)); }
};

// Lane width, record floats and tile geometry of an instance.
KR_HD constexpr int radial_lanes(int DP) { return packed(DP) ? 2 : 1; }
KR_HD constexpr int radial_stride(int DP, int EP) { return packed(DP) ? pair_stride(DP, EP) : pack_stride(DP, EP); }
// Points per unrolled step (a multiple of the lane width).
KR_HD constexpr int radial_step(int DP) { return packed(DP) ? 2 * unroll_pairs(DP) : unroll_points(DP); }

// Field f (coordinate d, or DP + e for a value) of tile point p.
template <int L, int PS>
__device__ __forceinline__ float *radial_slot(float *tile, int p, int f) {
    if (L == 2) return pair_slot<PS>(tile, p, f);
    return tile + p * PS + f;
}

template <int L, int PS>
__device__ __forceinline__ void radial_load(const float *rec, typename Lanes<L>::T (&pv)[PS / L]) {
    if constexpr (L == 2)
        load_pair_record<PS>(rec, pv);
    else
        load_record<PS>(rec, pv);
}

// Max, dense mode, E = 1: steps per block of the running-maximum test.  A larger block
// tests less often but recomputes more points when a lane's maximum rose (and some lane
// of a warp usually does in each tile).
KR_HD constexpr int radial_max_block(int KT) { return 2; }
// The same for the Gaussian's log-domain scan (one compare a pair, no ex2 to hide it behind).
KR_HD constexpr int log_max_block() { return 2; }

// k of a row (coordinates xr, prescaled) against the L points of a record: the distance
// summed in dist_chains(DP) interleaved chains, then the kernel.  Max recomputes values
// with it, so the scan and the recomputation give the same bits.
template <int DP, int L, int PS, int KT>
__device__ __forceinline__ typename Lanes<L>::T radial_k(const typename Lanes<L>::T (&xr)[DP],
                                                         const typename Lanes<L>::T (&pv)[PS / L]) {
    typedef Lanes<L> V;
    typedef typename V::T T;
    constexpr int NC = dist_chains(DP);  // interleaved partial sums
    T qc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) qc[c] = V::splat(c == 0 ? radial_q0<KT>() : 0.f);
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        const T df = V::add(xr[d], pv[d]);
        const int c = d % NC;
        const bool first = d < NC && !(c == 0 && radial_q0<KT>() != 0.f);
        qc[c] = first ? V::mul(df, df) : V::fma(df, df, qc[c]);
    }
    T q = qc[0];
#pragma unroll
    for (int c = 1; c < NC; ++c) q = V::add(q, qc[c]);
    return V::template kval<KT>(q);
}

template <int L>
__device__ __forceinline__ typename Lanes<L>::T make_lanes_sqrt(typename Lanes<L>::T q) {
    if constexpr (L == 2) return make_float2(sqrt_approx(q.x), sqrt_approx(q.y));
    else return sqrt_approx(q);
}

// Max / Min with one signal column without forming k b: a key t of the pair that falls as
// |k b| rises, from the point's staged value slot s (two points a record, f32x2):
//   Gaussian  t = q - log2|b|         (s = -log2|b| starts the distance's chain),  |k b| = 2^-t
//   Laplace   t = sqrt(q) - log2|b|   (s = -log2|b|),                              |k b| = 2^-t
//   Cauchy    t = (1 + q) / |b|       (s = 1 / |b|; the chain starts at 1),        |k b| = 1 / t
//   inverse multiquadric  t = (1 + q) / b^2  (s = 1 / b^2),                         |k b| = 1 / sqrt(t)
// with q = |x'-y'|^2.  A point that cannot hold the extreme carries s = +-inf (t = +-inf).
// Used by the scan and by the index recomputation alike.
template <int KT>
__device__ __forceinline__ float log_slot(float v) {  // s of a signal value v != 0 (its magnitude)
    const float m = fabsf(v);
    if (KT == KT_GAUSS || KT == KT_LAPLACE) return -log2f(m);
    if (KT == KT_CAUCHY) return 1.0f / m;
    return 1.0f / (m * m);
}
template <int KT>
__device__ __forceinline__ float log_value(float t) {  // |k b| at the key t
    if (KT == KT_GAUSS || KT == KT_LAPLACE) return exp2f(-t);
    if (KT == KT_CAUCHY) return 1.0f / t;
    return 1.0f / sqrtf(t);
}
template <int DP, int L, int PS, int KT>
__device__ __forceinline__ typename Lanes<L>::T log_key(const typename Lanes<L>::T (&xr)[DP],
                                                        const typename Lanes<L>::T (&pv)[PS / L]) {
    typedef Lanes<L> V;
    typedef typename V::T T;
    constexpr int NC = dist_chains(DP);
    // the first chain starts at s (Gaussian), at 1 (Cauchy, inverse multiquadric) or at 0
    const T q0 = KT == KT_GAUSS ? pv[DP] : V::splat(radial_q0<KT>());
    const bool start = KT != KT_LAPLACE;
    T qc[NC];
#pragma unroll
    for (int d = 0; d < DP; ++d) {
        const T df = V::add(xr[d], pv[d]);
        const int c = d % NC;
        qc[c] = d < NC ? ((c == 0 && start) ? V::fma(df, df, q0) : V::mul(df, df)) : V::fma(df, df, qc[c]);
    }
    T q = qc[0];
#pragma unroll
    for (int c = 1; c < NC; ++c) q = V::add(q, qc[c]);
    if (KT == KT_LAPLACE) return V::add(make_lanes_sqrt<L>(q), pv[DP]);
    if (KT == KT_CAUCHY || KT == KT_IMQ) return V::mul(q, pv[DP]);
    return q;
}

template <int DP, int EP, int R, int BN, int KT, int RED>
__global__ void __launch_bounds__(kThreads) radial_kernel(const Args a_) {
    const Args a = batch_view(a_);
    constexpr int L = radial_lanes(DP);
    typedef Lanes<L> V;
    typedef typename V::T T;
    constexpr int PS = radial_stride(DP, EP);
    constexpr int UPT = radial_step(DP);      // points per step
    constexpr int UR = UPT / L;                // records per step
    // Max, dense mode, E = 1: the running maximum is tested once per block of IB steps
    // (wider signals keep the per-step walk: the block state would not fit in registers)
    constexpr bool kBlockMax = RED == RR_MAX && EP == 1;
    constexpr int IB = radial_max_block(KT);
    static_assert(BN % (IB * UPT) == 0, "tile must be a multiple of the step and of the block");
    __shared__ __align__(16) float tile[(BN / L) * PS];

    const int t = threadIdx.x;
    // Dense mode: row block blockIdx.x, split blockIdx.y's column chunk.  Block-sparse
    // mode: the work table gives the block's rows and its list of column ranges, which
    // need not be in increasing j, so Max/Min then breaks ties on the index itself;
    // with S splits, split blockIdx.y takes every S-th tile of the ranges.
    const bool ranged = a.blk != nullptr;
    // tiles are padded to whole steps, and for the dense Max to whole blocks of IB steps
    // (padding points carry b = NaN there, which never wins)
    const int BPT = (kBlockMax && !ranged) ? IB * UPT : UPT;
    int64_t row0 = (int64_t)blockIdx.x * (kThreads * R), row_end = a.M;
    int r_lo = 0, r_hi = 1;
    if (ranged) {
        const int4 w = a.blk[blockIdx.x];
        row0 = w.x;
        row_end = w.y;
        r_lo = w.z;
        r_hi = w.w;
    }
    const int64_t j_begin = (int64_t)blockIdx.y * a.chunk;
    const int64_t j_end = min(a.N, j_begin + a.chunk);
    const float nan = __int_as_float(0x7fc00000);

    // zero the padded coordinates D..DP-1 of every tile point once
    if (a.D < DP) {
        for (int f = t; f < BN * DP; f += kThreads) {
            const int p = f / DP, d = f % DP;
            if (d >= a.D) *radial_slot<L, PS>(tile, p, d) = 0.f;
        }
    }
    T xr[R][DP];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
#pragma unroll
        for (int d = 0; d < DP; ++d) xr[r][d] = V::splat((i < row_end && d < a.D) ? a.c * ldg_chk(a, a.x, i * a.D + d, a.M * a.D, KRD_X) : 0.f);
    }

    T part[R][EP];
    float hi[R][EP], lo[R][EP];  // Sum: compensated running pair; Max: best value, unused
    int bj[R][EP];               // Max: index of the best value
    int last[R][EP];             // Max, dense mode: the tile step that last raised it (-1: none)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            part[r][e] = V::splat(0.f);
            hi[r][e] = RED == RR_MAX ? -f_inf() : 0.f;
            lo[r][e] = 0.f;
            bj[r][e] = -1;
            last[r][e] = -1;
        }

    // Max / Min, dense mode, E = 1: the key scan (log_key).  With v_j = vsign b_j, the signs of
    // v over the block's column chunk fix where the extreme can come from, the same for all its
    // rows: some v_j > 0: the largest k v is |k v| at the smallest key over those points (mode
    // 1); all v_j < 0 (none zero): it is -|k v| at the largest key over them (mode 2);
    // otherwise (zeros without positives, only NaN, none) the value scan below (mode 0).  The
    // scan then needs no ex2 / rcp / rsqrt and no product per pair (the Laplace keeps its
    // sqrt), and the order of the keys is that of the values up to the rounding of t.  A row
    // that finds no finite key (infinite or NaN coordinates) sends its block back to the value
    // scan.
    constexpr bool kLogMax = RED == RR_MAX && EP == 1 && L == 2;
    constexpr int LB = log_max_block();
    static_assert(!kLogMax || BN % (LB * UPT) == 0, "tile must be a multiple of the log-domain block");
    int mode = 0;
    if constexpr (kLogMax) {
        if (!ranged) {
            // the range where the staged 1 / |v| (Cauchy) or 1 / v^2 (inverse multiquadric) is
            // exact and finite; outside it the chunk keeps the value scan
            constexpr float kLo = KT == KT_CAUCHY ? 0x1p-126f : KT == KT_IMQ ? 0x1p-62f : 0.f;
            constexpr float kHi = KT == KT_CAUCHY ? 0x1p126f : KT == KT_IMQ ? 0x1p62f : f_inf_c();
            int f = 0;
            for (int64_t j = j_begin + t; j < j_end; j += kThreads) {
                const float v = a.vsign * ldg_chk(a, a.b, j, a.N, KRD_B);
                f |= v > 0.f ? 1 : v < 0.f ? 2 : v == 0.f ? 4 : 0;
                if (v != 0.f && !(fabsf(v) >= kLo && fabsf(v) <= kHi)) f |= 8;
            }
            const bool any_pos = __syncthreads_or(f & 1), any_neg = __syncthreads_or(f & 2);
            const bool any_zero = __syncthreads_or(f & 4), out_of_range = __syncthreads_or(f & 8);
            mode = out_of_range ? 0 : any_pos ? 1 : (any_neg && !any_zero) ? 2 : 0;
        }
    }
    if constexpr (kLogMax) {
        if (mode != 0) {
            const bool neg = mode == 2;
            const float none = neg ? -f_inf() : f_inf();  // the key of a point that cannot win
            float tb[R];
#pragma unroll
            for (int r = 0; r < R; ++r) tb[r] = none;
            // one tile: blocks of IB steps tested once against the best key; the last block that
            // improved it is recomputed at the end of the tile for the first point attaining it
            auto log_tile = [&](auto negc, int64_t jt, int nvp) {
                constexpr bool NEG = decltype(negc)::value;
                int lastb[R];
#pragma unroll
                for (int r = 0; r < R; ++r) lastb[r] = -1;
                for (int jb = 0; jb < nvp; jb += LB * UPT) {
                    float bm[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) bm[r] = NEG ? -f_inf() : f_inf();
#pragma unroll
                    for (int g = 0; g < LB; ++g)
#pragma unroll
                        for (int u = 0; u < UR; ++u) {
                            T pv[PS / L];
                            radial_load<L, PS>(tile + ((jb + g * UPT) / L + u) * PS, pv);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const T k = log_key<DP, L, PS, KT>(xr[r], pv);
                                bm[r] = NEG ? fmax3(bm[r], k.x, k.y) : fmin3(bm[r], k.x, k.y);
                            }
                        }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        lastb[r] = (NEG ? bm[r] > tb[r] : bm[r] < tb[r]) ? jb : lastb[r];
                        tb[r] = NEG ? fmaxf(tb[r], bm[r]) : fminf(tb[r], bm[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int jb = lastb[r];
                    if (jb < 0) continue;
                    bool found = false;
                    for (int u = 0; u < LB * UR; ++u) {
                        T pv[PS / L];
                        radial_load<L, PS>(tile + (jb / L + u) * PS, pv);
                        const T k = log_key<DP, L, PS, KT>(xr[r], pv);
#pragma unroll
                        for (int l = 0; l < L; ++l) {
                            if (!found && V::lane(k, l) == tb[r]) {
                                bj[r][0] = (int)(jt + jb + u * L + l);
                                found = true;
                            }
                        }
                    }
                }
            };
            for (int64_t jt = j_begin; jt < j_end; jt += BN) {
                const int nv = (int)min((int64_t)BN, j_end - jt);
                const int nvp = (nv + LB * UPT - 1) / (LB * UPT) * (LB * UPT);
                __syncthreads();  // every thread is done with the previous tile
                for (int p = t; p < nvp; p += kThreads) {
                    float key = none;
                    if (p < nv) {
#pragma unroll
                        for (int d = 0; d < DP; ++d)
                            if (d < a.D) *radial_slot<L, PS>(tile, p, d) = -a.c * ldg_chk(a, a.y, (jt + p) * a.D + d, a.N * a.D, KRD_Y);
                        const float v = a.vsign * ldg_chk(a, a.b, jt + p, a.N, KRD_B);
                        if (neg ? v < 0.f : v > 0.f) key = log_slot<KT>(v);
                    } else {
#pragma unroll
                        for (int d = 0; d < DP; ++d)
                            if (d < a.D) *radial_slot<L, PS>(tile, p, d) = 0.f;
                    }
                    *radial_slot<L, PS>(tile, p, DP) = key;
                }
                __syncthreads();  // tile staged
                if (neg)
                    log_tile(std::true_type(), jt, nvp);
                else
                    log_tile(std::false_type(), jt, nvp);
            }
            bool open = false;
#pragma unroll
            for (int r = 0; r < R; ++r) open |= row0 + (int64_t)r * kThreads + t < row_end && bj[r][0] < 0;
            if (__syncthreads_or(open)) {
                mode = 0;  // the value scan redoes this block's chunk
#pragma unroll
                for (int r = 0; r < R; ++r) bj[r][0] = -1;
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) hi[r][0] = neg ? -log_value<KT>(tb[r]) : log_value<KT>(tb[r]);
            }
        }
    }

    int tk = 0;  // block-sparse: tiles seen over the block's ranges; split y takes tk = y mod S
    for (int rr = r_lo; rr < r_hi && mode == 0; ++rr) {
    const int64_t js = ranged ? (int64_t)a.rng[rr].x : j_begin;
    const int64_t je = ranged ? (int64_t)a.rng[rr].y : j_end;
    for (int64_t jt = js; jt < je; jt += BN) {
        if (ranged && (tk++ % a.S) != (int)blockIdx.y) continue;  // uniform across the block
        const int nv = (int)min((int64_t)BN, je - jt);
        const int nvp = (nv + BPT - 1) / BPT * BPT;
        __syncthreads();  // every thread is done with the previous tile
        for (int p = t; p < nvp; p += kThreads) {
            if (p < nv) {
#pragma unroll
                for (int d = 0; d < DP; ++d)
                    if (d < a.D) *radial_slot<L, PS>(tile, p, d) = -a.c * ldg_chk(a, a.y, (jt + p) * a.D + d, a.N * a.D, KRD_Y);
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    float v = RED == RR_MAX ? nan : 0.f;
                    if (e < a.E) {
                        v = ldg_chk(a, a.b, (jt + p) * a.E + e, a.N * a.E, KRD_B);
                        if (RED == RR_MAX) v *= a.vsign;
                    }
                    *radial_slot<L, PS>(tile, p, DP + e) = v;
                }
            } else {
#pragma unroll
                for (int d = 0; d < DP; ++d)
                    if (d < a.D) *radial_slot<L, PS>(tile, p, d) = 0.f;
#pragma unroll
                for (int e = 0; e < EP; ++e) *radial_slot<L, PS>(tile, p, DP + e) = RED == RR_MAX ? nan : 0.f;
            }
        }
        __syncthreads();  // tile staged

        // One pass over the tile.  Max, dense mode, E = 1: no branch in the pass; the
        // running maximum and the last block of IB steps that raised it are kept (one test
        // per block), and that block is recomputed after the pass to find the index
        // (strictly greater raises it, so ties keep the lowest j).  Otherwise (block-sparse
        // mode, whose ranges come in any order, or E > 1) a raising or tying step walks its
        // points at once and ties break on the index.
        auto eval_step = [&](int jj, T (&kv)[UR][R][EP]) {
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                T pv[PS / L];
                radial_load<L, PS>(tile + (jj / L + u) * PS, pv);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const T k = radial_k<DP, L, PS, KT>(xr[r], pv);
#pragma unroll
                    for (int e = 0; e < EP; ++e) {
                        if (RED == RR_SUM)
                            part[r][e] = V::fma(k, pv[DP + e], part[r][e]);
                        else
                            kv[u][r][e] = V::mul(k, pv[DP + e]);
                    }
                }
            }
        };
        if constexpr (RED == RR_SUM) {
            T kv[UR][R][EP];
            // E = 1: two steps deep (6 % faster at D = 3: the loop's own overhead); wider
            // signals would spill
#pragma unroll(EP == 1 ? 2 : 1)
            for (int jj = 0; jj < nvp; jj += UPT) eval_step(jj, kv);
        } else if (!kBlockMax || ranged) {
            for (int jj = 0; jj < nvp; jj += UPT) {
                T kv[UR][R][EP];
                eval_step(jj, kv);
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < EP; ++e) {
                        float m = V::hmax(kv[0][r][e]);
#pragma unroll
                        for (int u = 1; u < UR; ++u) m = fmaxf(m, V::hmax(kv[u][r][e]));
                        if (m >= hi[r][e]) {  // rare: walk the step's points
#pragma unroll
                            for (int u = 0; u < UR; ++u)
#pragma unroll
                                for (int l = 0; l < L; ++l) {
                                    const float f = V::lane(kv[u][r][e], l);
                                    const int j = (int)(jt + jj + u * L + l);
                                    if (f > hi[r][e] || (f == hi[r][e] && j < bj[r][e])) {
                                        hi[r][e] = f;
                                        bj[r][e] = j;
                                    }
                                }
                        }
                    }
            }
        } else if constexpr (kBlockMax) {
            for (int jb = 0; jb < nvp; jb += IB * UPT) {
                float bm[R][EP];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < EP; ++e) bm[r][e] = -f_inf();
#pragma unroll
                for (int g = 0; g < IB; ++g) {
                    T kv[UR][R][EP];
                    eval_step(jb + g * UPT, kv);
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int e = 0; e < EP; ++e)
#pragma unroll
                            for (int u = 0; u < UR; ++u) bm[r][e] = V::max_into(bm[r][e], kv[u][r][e]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int e = 0; e < EP; ++e) {
                        last[r][e] = bm[r][e] > hi[r][e] ? jb : last[r][e];
                        hi[r][e] = fmaxf(hi[r][e], bm[r][e]);
                    }
            }
            // the index of each raised maximum: the first point of its last raising block
            // whose recomputed value equals it
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const int jb = last[r][e];
                    if (jb < 0) continue;
                    last[r][e] = -1;
                    bool found = false;
                    for (int u = 0; u < IB * UR; ++u) {
                        T pv[PS / L];
                        radial_load<L, PS>(tile + (jb / L + u) * PS, pv);
                        const T f = V::mul(radial_k<DP, L, PS, KT>(xr[r], pv), pv[DP + e]);
#pragma unroll
                        for (int l = 0; l < L; ++l) {
                            if (!found && V::lane(f, l) == hi[r][e]) {
                                bj[r][e] = (int)(jt + jb + u * L + l);
                                found = true;
                            }
                        }
                    }
                }
        }
        if (RED == RR_SUM) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    two_sum_add(hi[r][e], lo[r][e], V::hsum(part[r][e]));
                    part[r][e] = V::splat(0.f);
                }
        }
    }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t i = row0 + (int64_t)r * kThreads + t;
        if (i >= row_end) continue;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (e >= a.E) continue;
            const int64_t o = i * a.E + e;
            if (a.S == 1) {
                if (RED == RR_SUM) {
                    st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(hi[r][e] + lo[r][e]));
                } else {
                    if (a.out) st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(a.vsign * hi[r][e]));
                    if (a.idx) st_chk(a, a.idx, o, a.idx_n, KRD_IDX, (int32_t)(bj[r][e]));
                }
            } else {
                const int64_t w = (int64_t)blockIdx.y * a.M * a.E + o;
                st_chk(a, a.ws0, w, a.ws_n, KRD_WS, (float)(hi[r][e]));
                if (RED == RR_SUM)
                    st_chk(a, a.ws1, w, a.ws_n, KRD_WS, (float)(lo[r][e]));
                else
                    st_chk(a, a.wsi, w, a.ws_n, KRD_WS, (int32_t)(bj[r][e]));
            }
        }
    }
}

}  // namespace kr
