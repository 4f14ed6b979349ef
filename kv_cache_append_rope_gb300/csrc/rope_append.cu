// Fused RoPE-at-offset + key/value append.
//
// [Ch37] "Keep the prefix, project only the new row", section "Append along
// the position axis": the new key is rotated for its absolute position (the
// zero-based old length) and appended with the unrotated value; the query is
// rotated the same way for the current calculation only.  [LCP5] listing under
// "哪些东西必须一起裁剪": every slot also records its position.
//
// Two kernels.  bf16 storage with d_h a multiple of 8 (the long chunks) takes
// rope_append_bf16_kernel: a thread rotates one 16-byte chunk of one row for
// four heads at once, sharing the row's cos/sin load and keeping four
// independent loads in flight at 62 registers.  Other dtypes and head sizes
// take rope_append_kernel: one thread handles P interleaved pairs (16 bytes of
// bf16, 8 of f64) of up to four rows of one head.  In both, consecutive threads
// walk consecutive chunks of a row, then rows, so loads and stores are coalesced.
//
// The stored key is defined as the float64 evaluation of (x c - y s, x s + y c)
// -- every product and sum rounded separately, cos/sin from a float64 table --
// rounded once to the storage dtype.  f32 and f64 caches evaluate exactly that.
// bf16 caches (where float64 throughput would dominate a long chunk) evaluate
// it in float32 and prove, element by element, that rounding to bf16 gives the
// same bits: with r the float32 result and E a bound on |r - X| (X the float64
// value), rounding to nearest is monotone, so RN(r - E) == RN(r + E) implies
// RN(X) == RN(r).  Elements that fail the test (a bf16 rounding boundary
// within E, about one in a thousand) are evaluated in float64.  Queries are
// never stored and use the float32 rotation directly.
#include <type_traits>

#include "device_common.cuh"
#include "kvc_internal.h"

namespace kvc {

template <typename T, int P>
struct alignas((2 * P * sizeof(T)) >= 16 ? 16 : (2 * P * sizeof(T))) Pack { T v[2 * P]; };

constexpr int kRows = 4;   // rows of one (head, chunk) handled by a thread: 4 loads in flight

template <typename T, typename QO, int P, bool FAST>
__device__ __forceinline__ void rope_one(const AppendLaunch& a, int kind, int b, int h, int i, int slot, int pos,
                                         int c, const Pack<T, P>& in) {
    using S = Storage<T>;
    const int pairs_per_row = a.d / 2;
    if (kind == 2) {
        T* dst = (T*)a.V + kv_row(a.kv, b, h, slot) * a.d + 2 * P * c;
        *reinterpret_cast<Pack<T, P>*>(dst) = in;
        return;
    }
    const int64_t t0 = (int64_t)pos * pairs_per_row + P * c;
    if constexpr (FAST) {
        // bf16 storage: float32 rotation, bit-exact key rounding (see above)
        Pack<T, P> ok;
        Pack<QO, P> oq;
        if (!a.rope) {          // no rotation: keys are copied, queries converted
            ok = in;
#pragma unroll
            for (int e = 0; e < 2 * P; ++e) oq.v[e] = (QO)S::to_f32(in.v[e]);
        } else {
#pragma unroll
            for (int e = 0; e < P; ++e) {
                const float2 cs = a.rope_f[t0 + e];
                const float xf = S::to_f32(in.v[2 * e]);
                const float yf = S::to_f32(in.v[2 * e + 1]);
                if (kind == 1) {
                    ok.v[2 * e] = rope_bf16_exact(xf, yf, cs.x, cs.y, a.rope, pos, pairs_per_row, P * c + e, false);
                    ok.v[2 * e + 1] = rope_bf16_exact(xf, yf, cs.x, cs.y, a.rope, pos, pairs_per_row, P * c + e, true);
                } else {
                    oq.v[2 * e] = (QO)fmaf(xf, cs.x, -(yf * cs.y));
                    oq.v[2 * e + 1] = (QO)fmaf(yf, cs.x, xf * cs.y);
                }
            }
        }
        if (kind == 1) {
            T* dst = (T*)a.K + kv_row(a.kv, b, h, slot) * a.d + 2 * P * c;
            *reinterpret_cast<Pack<T, P>*>(dst) = ok;
            if (h == 0 && c == 0) a.positions[(int64_t)b * a.C + slot] = pos;
        } else {
            QO* dst = (QO*)a.qrot + (((int64_t)b * a.Hq + h) * a.S + i) * a.d + 2 * P * c;
            *reinterpret_cast<Pack<QO, P>*>(dst) = oq;
        }
    } else {
        double xr[2 * P];
#pragma unroll
        for (int e = 0; e < P; ++e) {
            const double x = S::to_f64(in.v[2 * e]);
            const double y = S::to_f64(in.v[2 * e + 1]);
            if (a.rope) {
                const double2 cs = a.rope[t0 + e];
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
            T* dst = (T*)a.K + kv_row(a.kv, b, h, slot) * a.d + 2 * P * c;
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

template <typename T, typename QO, int P, bool FAST>
__global__ void __launch_bounds__(256) rope_append_kernel(AppendLaunch a) {
    const int chunks = a.d / 2 / P;
    const int heads_all = a.Hq + 2 * a.Hkv;
    const int groups = (a.S + kRows - 1) / kRows;
    const int64_t total = (int64_t)a.B * heads_all * groups * chunks;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        // consecutive threads: the chunks of one row, then the heads of the same rows
        // (a warp shares their cos/sin entries in L1), then row groups, then sequences
        const int c = (int)(u % chunks);
        int64_t r = u / chunks;
        const int hh = (int)(r % heads_all);
        r /= heads_all;
        const int ig = (int)(r % groups);
        const int b = (int)(r / groups);
        const int rows = a.seqlen ? a.seqlen[b] : a.S;
        const int i0 = ig * kRows;
        if (i0 >= rows) continue;
        int kind, h;   // 0 = query, 1 = key, 2 = value
        if (hh < a.Hq) { kind = 0; h = hh; }
        else if (hh < a.Hq + a.Hkv) { kind = 1; h = hh - a.Hq; }
        else { kind = 2; h = hh - a.Hq - a.Hkv; }
        const int H = kind == 0 ? a.Hq : a.Hkv;
        const T* src = (const T*)(kind == 0 ? a.q : kind == 1 ? a.k : a.v) +
                       (((int64_t)b * H + h) * a.S + i0) * a.d + 2 * P * c;
        const int n = min(kRows, rows - i0);
        Pack<T, P> in[kRows];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr)
            if (rr < n) in[rr] = *reinterpret_cast<const Pack<T, P>*>(src + (int64_t)rr * a.d);
        const int slot0 = a.slot0[b] + i0;
        const int pos0 = a.pos0[b] + i0;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            if (rr >= n) break;
            const int slot = slot0 + rr, pos = pos0 + rr;
            if (slot < 0 || slot >= a.C || pos < 0 || (a.rope && pos >= a.max_positions)) {
                atomicOr(a.err, (uint32_t)DEV_ERR_SLOT);
                continue;
            }
            if (kind != 0 && !debug_check(kv_slot_ok(a.kv, b, slot), a.err)) continue;
            rope_one<T, QO, P, FAST>(a, kind, b, h, i0 + rr, slot, pos, c, in[rr]);
        }
    }
}

// ---- bf16 storage, d_h a multiple of 8: heads-grouped kernel ------------------
//
// A thread takes one 16-byte chunk (4 pairs) of one row for up to kHeads heads of
// the same kind, so the row's cos/sin entries are loaded once for all of them and
// the thread keeps kHeads independent 16-byte loads in flight.  Consecutive threads
// walk the chunks of a row, then the rows (contiguous in [B,H,S,d]), then head
// groups, then sequences.  Keys whose float32 rotation cannot be proved to round
// like the float64 one are stored first and then rewritten, element by element,
// by an out-of-line float64 pass (rare), so the common path carries no call.
constexpr int kHeads = 4;

__device__ __forceinline__ uint32_t pack2_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// One rotated key component rounded to bf16, or `fail` set when a bf16 rounding
// boundary lies within the float32 error bound (same test as rope_bf16_exact).
__device__ __forceinline__ __nv_bfloat16 rope_bf16_checked(float t1, float c, float t2, bool add, bool& fail) {
    const float r = add ? fmaf(t1, c, t2) : fmaf(t1, c, -t2);
    const float bound = 0x1p-20f * (fabsf(t1 * c) + fabsf(t2) + fabsf(r)) + 0x1p-140f;
    const __nv_bfloat16 lo = __float2bfloat16_rn(r - bound);
    const __nv_bfloat16 hi = __float2bfloat16_rn(r + bound);
    fail = __bfloat16_as_ushort(lo) != __bfloat16_as_ushort(hi);
    return lo;
}

template <typename QO>
__global__ void __launch_bounds__(256) rope_append_bf16_kernel(AppendLaunch a) {
    using bf = __nv_bfloat16;
    // blockIdx.y: (sequence, head group); x threads stride over (row, chunk) of that plane
    const int gq = (a.Hq + kHeads - 1) / kHeads, gk = (a.Hkv + kHeads - 1) / kHeads;
    const int groups = gq + 2 * gk;
    const int b = blockIdx.y / groups, gg = blockIdx.y % groups;
    int kind, h0, H;   // 0 = query, 1 = key, 2 = value
    if (gg < gq) { kind = 0; h0 = gg * kHeads; H = a.Hq; }
    else if (gg < gq + gk) { kind = 1; h0 = (gg - gq) * kHeads; H = a.Hkv; }
    else { kind = 2; h0 = (gg - gq - gk) * kHeads; H = a.Hkv; }
    const int nh = min(kHeads, H - h0);
    const int chunks = a.d >> 3;
    const int pairs = a.d >> 1;
    const int rows = a.seqlen ? a.seqlen[b] : a.S;
    const int slot0 = a.slot0[b], pos0 = a.pos0[b];
    const uint32_t total = (uint32_t)rows * chunks;
    const bf* base = (const bf*)(kind == 0 ? a.q : kind == 1 ? a.k : a.v) + ((int64_t)b * H + h0) * a.S * a.d;
    const int64_t hstride = (int64_t)a.S * a.d;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += gridDim.x * blockDim.x) {
        const int i = (int)(u / chunks), c = (int)(u % chunks);
        const int slot = slot0 + i, pos = pos0 + i;
        if (slot < 0 || slot >= a.C || pos < 0 || (a.rope && pos >= a.max_positions)) {
            atomicOr(a.err, (uint32_t)DEV_ERR_SLOT);
            continue;
        }
        if (kind != 0 && !debug_check(kv_slot_ok(a.kv, b, slot), a.err)) continue;
        const bf* src = base + (int64_t)i * a.d + 8 * c;
        uint4 in[kHeads];
#pragma unroll
        for (int e = 0; e < kHeads; ++e)
            if (e < nh) in[e] = __ldcs(reinterpret_cast<const uint4*>(src + e * hstride));
        if (kind == 2) {
#pragma unroll
            for (int e = 0; e < kHeads; ++e)
                if (e < nh) *reinterpret_cast<uint4*>((bf*)a.V + kv_row(a.kv, b, h0 + e, slot) * a.d + 8 * c) = in[e];
            continue;
        }
        const int64_t t0 = (int64_t)pos * pairs + 4 * c;
        float cf[4], sf[4];
        if (a.rope) {
            const float4 c01 = *reinterpret_cast<const float4*>(a.rope_f + t0);
            const float4 c23 = *reinterpret_cast<const float4*>(a.rope_f + t0 + 2);
            cf[0] = c01.x; sf[0] = c01.y; cf[1] = c01.z; sf[1] = c01.w;
            cf[2] = c23.x; sf[2] = c23.y; cf[3] = c23.z; sf[3] = c23.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) { cf[e] = 1.f; sf[e] = 0.f; }
        }
        uint32_t mask = 0;   // keys: bit 8 e + k flags element k of head h0 + e
#pragma unroll
        for (int e = 0; e < kHeads; ++e) {
            if (e >= nh) break;
            const uint32_t w[4] = {in[e].x, in[e].y, in[e].z, in[e].w};
            if (kind == 1) {
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float x = __uint_as_float(w[p] << 16), y = __uint_as_float(w[p] & 0xffff0000u);
                    bool f0, f1;
                    const bf r0 = rope_bf16_checked(x, cf[p], y * sf[p], false, f0);
                    const bf r1 = rope_bf16_checked(y, cf[p], x * sf[p], true, f1);
                    o[p] = a.rope ? pack2_bf16(r0, r1) : w[p];
                    if (a.rope) mask |= ((uint32_t)f0 | ((uint32_t)f1 << 1)) << (8 * e + 2 * p);
                }
                *reinterpret_cast<uint4*>((bf*)a.K + kv_row(a.kv, b, h0 + e, slot) * a.d + 8 * c) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                QO o[8];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float x = __uint_as_float(w[p] << 16), y = __uint_as_float(w[p] & 0xffff0000u);
                    o[2 * p] = (QO)fmaf(x, cf[p], -(y * sf[p]));
                    o[2 * p + 1] = (QO)fmaf(y, cf[p], x * sf[p]);
                }
                QO* dst = (QO*)a.qrot + (((int64_t)b * a.Hq + h0 + e) * a.S + i) * a.d + 8 * c;
                *reinterpret_cast<Pack<QO, 4>*>(dst) = *reinterpret_cast<const Pack<QO, 4>*>(o);
            }
        }
        if (kind == 1 && h0 == 0 && c == 0) a.positions[(int64_t)b * a.C + slot] = pos;
        // rare: rewrite the flagged key elements with the float64 evaluation (the same
        // thread stored the chunk just before, so program order makes this the final value)
        while (__builtin_expect(mask != 0, 0)) {
            const int k = __ffs(mask) - 1;
            mask &= mask - 1;
            const int e = k >> 3, el = k & 7, pr = el >> 1;
            const bf* s2 = src + e * hstride + 2 * pr;
            const double2 cs = a.rope[t0 + pr];
            double xr, yr;
            rope_pair_f64((double)__bfloat162float(s2[0]), (double)__bfloat162float(s2[1]), cs.x, cs.y, xr, yr);
            ((bf*)a.K)[kv_row(a.kv, b, h0 + e, slot) * a.d + 8 * c + el] = f64_to_bf16_rn((el & 1) ? yr : xr);
        }
    }
}

template <typename QO>
static cudaError_t launch_bf16(const AppendLaunch& a, cudaStream_t s) {
    const int groups = (a.Hq + kHeads - 1) / kHeads + 2 * ((a.Hkv + kHeads - 1) / kHeads);
    const int64_t planes = (int64_t)a.B * groups;
    const int64_t per_plane = (int64_t)a.S * (a.d / 8);
    if (planes == 0 || per_plane == 0) return cudaSuccess;
    if (planes > 65535 || per_plane > 0x7fffffff) return cudaErrorInvalidValue;
    int sms = 152;
    int dev;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about 32 resident 256-thread blocks' worth of threads per SM over the whole grid;
    // short chunks (decode: one row) get one small block per plane
    const int threads = per_plane >= 256 ? 256 : (int)((per_plane + 31) / 32 * 32);
    int64_t bx = (per_plane + threads - 1) / threads;
    const int64_t cap = ((int64_t)sms * 32 + planes - 1) / planes;
    if (bx > cap) bx = cap;
    rope_append_bf16_kernel<QO><<<dim3((unsigned)bx, (unsigned)planes), threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, typename QO>
static cudaError_t launch_typed(const AppendLaunch& a, cudaStream_t s) {
    constexpr int P_max = 16 / (2 * sizeof(T)) > 0 ? 16 / (2 * sizeof(T)) : 1;  // pairs per 16 bytes
    const int pairs = a.d / 2;
    int P = 1;
    if (P_max >= 4 && pairs % 4 == 0) P = 4;
    else if (P_max >= 2 && pairs % 2 == 0) P = 2;
    const int64_t total = (int64_t)a.B * (a.Hq + 2 * a.Hkv) * ((a.S + kRows - 1) / kRows) * (pairs / P);
    if (total == 0) return cudaSuccess;
    int sms = 152;
    int dev;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    constexpr bool FAST = std::is_same<T, __nv_bfloat16>::value;
    switch (P) {
        case 4: rope_append_kernel<T, QO, 4, FAST><<<(unsigned)blocks, 256, 0, s>>>(a); break;
        case 2: rope_append_kernel<T, QO, 2, FAST><<<(unsigned)blocks, 256, 0, s>>>(a); break;
        default: rope_append_kernel<T, QO, 1, FAST><<<(unsigned)blocks, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_rope_append(int dtype, const AppendLaunch& a, cudaStream_t s) {
    switch (dtype) {
        case KVC_BF16:
            if (a.d % 8 == 0)
                return a.qrot_kind == 2 ? launch_bf16<__nv_bfloat16>(a, s) : launch_bf16<float>(a, s);
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
