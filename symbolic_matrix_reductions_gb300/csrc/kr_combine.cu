// Split-j combine kernels: deterministic, fixed split order.
#include "kr_kernels.cuh"

namespace kr {

__global__ void combine_sum_kernel(const Args a_, int W) {
    const Args a = batch_view(a_);
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = a.M * W;
    if (o >= total) return;
    double acc = 0.0;
    for (int s = 0; s < a.S; ++s) acc += (double)ldg_chk(a, a.ws0, s * total + o, a.ws_n, KRD_WS) + (double)ldg_chk(a, a.ws1, s * total + o, a.ws_n, KRD_WS);
    st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)acc);
}

__global__ void combine_lse_kernel(const Args a_) {
    const Args a = batch_view(a_);
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = a.M * a.E;
    if (o >= total) return;
    // A split that could not finish (a tensor-core wait that ran out) leaves NaN in its
    // frame; fmaxf would drop it, so NaN is looked for first and passed on to the output.
    float mmax = -f_inf();
    bool nan = false;
    for (int s = 0; s < a.S; ++s) {
        const float m = ldg_chk(a, a.ws0, s * total + o, a.ws_n, KRD_WS);
        nan |= m != m;
        mmax = fmaxf(mmax, m);
    }
    if (nan) {
        st_chk(a, a.out, o, a.out_n, KRD_OUT, __int_as_float(0x7fc00000));
        return;
    }
    if (mmax == -f_inf()) {
        st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(-f_inf()));
        return;
    }
    double acc = 0.0;
    for (int s = 0; s < a.S; ++s) {
        const float acc_s = ldg_chk(a, a.ws1, s * total + o, a.ws_n, KRD_WS);
        if (acc_s > 0.f) acc += (double)acc_s * exp2((double)ldg_chk(a, a.ws0, s * total + o, a.ws_n, KRD_WS) - (double)mmax);
    }
    st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(0.6931471805599453 * ((double)mmax + log2(acc))));
}

__global__ void combine_knn_kernel(const Args a_, int KP) {
    const Args a = batch_view(a_);
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.M) return;
    int head[kMaxSplit];
    for (int s = 0; s < a.S; ++s) head[s] = 0;
    for (int k = 0; k < a.K; ++k) {
        int best = -1;
        float bd = 0.f;
        int bj = 0;
        for (int s = 0; s < a.S; ++s) {
            if (head[s] >= KP) continue;
            const int64_t w = ((int64_t)s * a.M + i) * KP + head[s];
            const int j = ldg_chk(a, (const int32_t *)a.wsi, w, a.ws_n, KRD_WS);
            if (j < 0) continue;  // empty slot: ranks after every real pair
            const float d = ldg_chk(a, a.ws0, w, a.ws_n, KRD_WS);
            if (best < 0 || d < bd || (d == bd && j < bj)) {
                best = s;
                bd = d;
                bj = j;
            }
        }
        if (best < 0) {
            st_chk(a, a.idx, i * a.K + k, a.idx_n, KRD_IDX, (int32_t)(-1));
            if (a.out) st_chk(a, a.out, i * a.K + k, a.out_n, KRD_OUT, (float)(f_inf()));
        } else {
            st_chk(a, a.idx, i * a.K + k, a.idx_n, KRD_IDX, (int32_t)(bj));
            if (a.out) st_chk(a, a.out, i * a.K + k, a.out_n, KRD_OUT, (float)(bd));
            ++head[best];
        }
    }
}

__global__ void combine_max_kernel(const Args a_) {
    const Args a = batch_view(a_);
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = a.M * a.E;
    if (o >= total) return;
    float best = -f_inf();
    int bj = -1;
    for (int s = 0; s < a.S; ++s) {
        const float v = ldg_chk(a, a.ws0, s * total + o, a.ws_n, KRD_WS);
        const int j = ldg_chk(a, (const int32_t *)a.wsi, s * total + o, a.ws_n, KRD_WS);
        // larger value, or the same value at a lower index (block-sparse splits need
        // not hold increasing j; dense splits do, so there this keeps the earlier split)
        if (v > best || (v == best && j >= 0 && (bj < 0 || j < bj))) {
            best = v;
            bj = j;
        }
    }
    if (a.out) st_chk(a, a.out, o, a.out_n, KRD_OUT, (float)(a.vsign * best));
    if (a.idx) st_chk(a, a.idx, o, a.idx_n, KRD_IDX, (int32_t)(bj));
}

cudaError_t launch_combine(int op, const Instance &inst, const Args &a, cudaStream_t s) {
    const int threads = 256;
    int64_t n = 0;
    switch (op) {
        case OP_SUM:
            n = a.M * a.E;
            combine_sum_kernel<<<dim3((unsigned)((n + threads - 1) / threads), 1, (unsigned)(a.batch > 1 ? a.batch : 1)), threads, 0, s>>>(a, a.E);
            break;
        case OP_GRAD:
            n = a.M * a.D;
            combine_sum_kernel<<<dim3((unsigned)((n + threads - 1) / threads), 1, (unsigned)(a.batch > 1 ? a.batch : 1)), threads, 0, s>>>(a, a.D);
            break;
        case OP_LSE:
            n = a.M * a.E;
            combine_lse_kernel<<<dim3((unsigned)((n + threads - 1) / threads), 1, (unsigned)(a.batch > 1 ? a.batch : 1)), threads, 0, s>>>(a);
            break;
        case OP_MAX:
            n = a.M * a.E;
            combine_max_kernel<<<dim3((unsigned)((n + threads - 1) / threads), 1, (unsigned)(a.batch > 1 ? a.batch : 1)), threads, 0, s>>>(a);
            break;
        case OP_KNN:
            n = a.M;
            combine_knn_kernel<<<dim3((unsigned)((n + threads - 1) / threads), 1, (unsigned)(a.batch > 1 ? a.batch : 1)), threads, 0, s>>>(a, inst.ek_pad);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kr
