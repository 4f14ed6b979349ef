// Fused RoPE-at-offset + key/value append.
//
// [Ch37] "Keep the prefix, project only the new row", section "Append along
// the position axis": the new key is rotated for its absolute position (the
// zero-based old length) and appended with the unrotated value; the query is
// rotated the same way for the current calculation only.  [LCP5] listing under
// "哪些东西必须一起裁剪": every slot also records its position.
//
// One thread handles P interleaved pairs (16 bytes of bf16, 8 of f64) of one
// row of one head of q, k or v.  Consecutive threads walk consecutive pairs of
// a row, then rows, then heads, so loads and stores are coalesced.  The
// rotation runs in float64 with separately rounded products and sums from a
// float64 cos/sin table, and the result is rounded once to its destination
// type, which makes the stored key bit-identical to the plain float64
// definition rounded to the storage dtype.
#include "device_common.cuh"
#include "kvc_internal.h"

namespace kvc {

template <typename T, int P>
struct alignas((2 * P * sizeof(T)) >= 16 ? 16 : (2 * P * sizeof(T))) Pack { T v[2 * P]; };

template <typename T, typename QO, int P>
__global__ void __launch_bounds__(256) rope_append_kernel(AppendLaunch a) {
    using S = Storage<T>;
    const int pairs_per_row = a.d / 2;
    const int chunks = pairs_per_row / P;
    const int heads_all = a.Hq + 2 * a.Hkv;
    const int64_t total = (int64_t)a.B * heads_all * a.S * chunks;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(u % chunks);
        int64_t r = u / chunks;
        const int i = (int)(r % a.S);
        r /= a.S;
        const int hh = (int)(r % heads_all);
        const int b = (int)(r / heads_all);
        const int rows = a.seqlen ? a.seqlen[b] : a.S;
        if (i >= rows) continue;
        const int slot = a.slot0[b] + i;
        const int pos = a.pos0[b] + i;
        if (slot < 0 || slot >= a.C || pos < 0 || (a.rope && pos >= a.max_positions)) {
            atomicOr(a.err, (uint32_t)DEV_ERR_SLOT);
            continue;
        }
        int kind, h;   // 0 = query, 1 = key, 2 = value
        if (hh < a.Hq) { kind = 0; h = hh; }
        else if (hh < a.Hq + a.Hkv) { kind = 1; h = hh - a.Hq; }
        else { kind = 2; h = hh - a.Hq - a.Hkv; }
        const int H = kind == 0 ? a.Hq : a.Hkv;
        const T* src = (const T*)(kind == 0 ? a.q : kind == 1 ? a.k : a.v) +
                       (((int64_t)b * H + h) * a.S + i) * a.d + 2 * P * c;
        Pack<T, P> in = *reinterpret_cast<const Pack<T, P>*>(src);
        if (kind == 2) {
            T* dst = (T*)a.V + (((int64_t)b * a.Hkv + h) * a.C + slot) * a.d + 2 * P * c;
            *reinterpret_cast<Pack<T, P>*>(dst) = in;
            continue;
        }
        double xr[2 * P];
#pragma unroll
        for (int e = 0; e < P; ++e) {
            const double x = S::to_f64(in.v[2 * e]);
            const double y = S::to_f64(in.v[2 * e + 1]);
            if (a.rope) {
                const double2 cs = a.rope[(int64_t)pos * pairs_per_row + P * c + e];
                rope_pair_f64(x, y, cs.x, cs.y, xr[2 * e], xr[2 * e + 1]);
            } else {
                xr[2 * e] = x;
                xr[2 * e + 1] = y;
            }
        }
        if (kind == 1) {
            Pack<T, P> o;
#pragma unroll
            for (int e = 0; e < 2 * P; ++e) o.v[e] = from_f64_rn<T>(xr[e]);
            T* dst = (T*)a.K + (((int64_t)b * a.Hkv + h) * a.C + slot) * a.d + 2 * P * c;
            *reinterpret_cast<Pack<T, P>*>(dst) = o;
            if (h == 0 && c == 0) a.positions[(int64_t)b * a.C + slot] = pos;
        } else {
            Pack<QO, P> o;
#pragma unroll
            for (int e = 0; e < 2 * P; ++e) o.v[e] = from_f64_rn<QO>(xr[e]);
            QO* dst = (QO*)a.qrot + (((int64_t)b * a.Hq + h) * a.S + i) * a.d + 2 * P * c;
            *reinterpret_cast<Pack<QO, P>*>(dst) = o;
        }
    }
}

template <typename T, typename QO>
static cudaError_t launch_typed(const AppendLaunch& a, cudaStream_t s) {
    constexpr int P_max = 16 / (2 * sizeof(T)) > 0 ? 16 / (2 * sizeof(T)) : 1;  // pairs per 16 bytes
    const int pairs = a.d / 2;
    int P = 1;
    if (P_max >= 4 && pairs % 4 == 0) P = 4;
    else if (P_max >= 2 && pairs % 2 == 0) P = 2;
    const int64_t total = (int64_t)a.B * (a.Hq + 2 * a.Hkv) * a.S * (pairs / P);
    if (total == 0) return cudaSuccess;
    int sms = 152;
    int dev;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    switch (P) {
        case 4: rope_append_kernel<T, QO, 4><<<(unsigned)blocks, 256, 0, s>>>(a); break;
        case 2: rope_append_kernel<T, QO, 2><<<(unsigned)blocks, 256, 0, s>>>(a); break;
        default: rope_append_kernel<T, QO, 1><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_rope_append(int dtype, const AppendLaunch& a, cudaStream_t s) {
    switch (dtype) {
        case KVC_BF16:
            if (a.qrot_kind == 2) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, s);
            return launch_typed<__nv_bfloat16, float>(a, s);
        case KVC_F32:
            return launch_typed<float, float>(a, s);
        case KVC_F64:
            return launch_typed<double, double>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kvc
