// Dtype-generic newest-query / causal-chunk attention on CUDA cores.
//
// [Ch37] "Keep the prefix, project only the new row", listing "Evaluate one
// newest query across the retained rows plus the candidate key/value row
// before committing the append": s_j = q.k_j / sqrt(d_h), numerically stable
// softmax, output sum_j a_j v_j.  [LCP5] section "先看一次历史编辑": a chunk
// row at slot n + i attends slots 0 .. n + i (with a sliding window of W, section
// "为什么滑窗部分命中必须回退", only slots n + i - W + 1 .. n + i).
//
// One warp per query row (b, h, i) streams its t = slot0[b] + i + 1 key/value
// rows with an online (running max, running sum) softmax.  The accumulator is
// float for bf16 / f32 storage and double for f64 storage.  This path serves
// every dtype and head width (2 .. 256); the bf16 head-width-128 kernels are
// the fast paths.
#include "device_common.cuh"
#include "kvc_internal.h"

namespace kvc {

template <typename A> __device__ __forceinline__ A exp_acc(A x);
template <> __device__ __forceinline__ float exp_acc<float>(float x) { return expf(x); }
template <> __device__ __forceinline__ double exp_acc<double>(double x) { return exp(x); }

template <typename T, typename A>
__global__ void __launch_bounds__(128) attend_generic_kernel(GenericAttendLaunch a) {
    using S = Storage<T>;
    constexpr int MAXE = 8;  // dims per lane: d_h <= 256
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int64_t nrows = (int64_t)a.B * a.Hq * a.S;
    if (row >= nrows) return;
    const int i = (int)(row % a.S);
    const int h = (int)((row / a.S) % a.Hq);
    const int b = (int)(row / ((int64_t)a.S * a.Hq));
    const int rows = a.seqlen ? a.seqlen[b] : a.S;
    if (i >= rows) return;
    const int t = a.slot0[b] + i + 1;
    if (!debug_check(t >= 1 && t <= a.C, lane == 0 ? a.err : nullptr)) return;
    const int g = h / (a.Hq / a.Hkv);
    const A* q = (const A*)a.qrot + row * a.d;
    const A scale = (A)1 / sqrt((A)a.d);

    A qv[MAXE], acc[MAXE];
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        qv[e] = c < a.d ? q[c] : (A)0;
        acc[e] = (A)0;
    }
    A m = -INFINITY, l = 0;
    const int lo = a.window > 0 && t > a.window ? t - a.window : 0;   // sliding window: the last `window` slots
    for (int j = lo; j < t; ++j) {
        const int64_t rj = kv_row(a.kv, b, g, j) * a.d;
        const T* kr = (const T*)a.K + rj;
        A dot = 0;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            if (c < a.d) dot += qv[e] * (A)S::to_f64(kr[c]);
        }
        const A s = warp_sum(dot) * scale;
        const A m_new = s > m ? s : m;
        const A corr = exp_acc<A>(m - m_new);
        const A p = exp_acc<A>(s - m_new);
        l = l * corr + p;
        const T* vr = (const T*)a.V + rj;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            if (c < a.d) acc[e] = acc[e] * corr + p * (A)S::to_f64(vr[c]);
        }
        m = m_new;
    }
    A* o = (A*)a.out + row * a.d;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (c < a.d) o[c] = acc[e] / l;
    }
}

cudaError_t launch_attend_generic(int dtype, const GenericAttendLaunch& a, cudaStream_t s) {
    const int64_t nrows = (int64_t)a.B * a.Hq * a.S;
    if (nrows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((nrows + 3) / 4);
    switch (dtype) {
        case KVC_BF16: attend_generic_kernel<__nv_bfloat16, float><<<blocks, 128, 0, s>>>(a); break;
        case KVC_F32: attend_generic_kernel<float, float><<<blocks, 128, 0, s>>>(a); break;
        case KVC_F64: attend_generic_kernel<double, double><<<blocks, 128, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvc
