// Device helpers shared by the kvc kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvc {

// Error bits written to the handle's device error word.
enum DeviceError : uint32_t {
    DEV_ERR_SLOT = 1u,        // an append slot or position fell outside its buffer
    DEV_ERR_WAIT_TIMEOUT = 2u,// a bounded mbarrier wait gave up
    DEV_ERR_TMEM = 4u,        // tensor-memory allocation returned an unusable address
    DEV_ERR_FULL = 8u,        // a device-length decode step met a full sequence or a position
                              // beyond the RoPE table and was rejected as a whole
    DEV_ERR_CUT = 16u,        // a device-checked truncate met a cut beyond a length
    DEV_ERR_BOUNDS = 32u      // debug builds: a length or slot index outside the cache; the
                              // access was skipped
};

// Debug builds (compiled with -DKVC_DEBUG, libkvc_debug.so) check every length
// and slot index a kernel derives against the capacity before it touches
// storage; a failed check records DEV_ERR_BOUNDS in the error word and skips the
// access -- never a trap or an assert, so the context stays usable and
// kvc_check reports it.  Release builds compile the checks away.
#ifdef KVC_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif

// True when `ok` holds or the build has no debug checks; else records the bit.
__device__ __forceinline__ bool debug_check(bool ok, uint32_t* err) {
    if (!kDebug || ok) return true;
    if (err) atomicOr(err, (uint32_t)DEV_ERR_BOUNDS);
    return false;
}

// ---- storage dtype traits ------------------------------------------------

template <typename T> struct Storage;
template <> struct Storage<__nv_bfloat16> {
    __device__ static double to_f64(__nv_bfloat16 x) { return (double)__bfloat162float(x); }
    __device__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
};
template <> struct Storage<float> {
    __device__ static double to_f64(float x) { return (double)x; }
    __device__ static float to_f32(float x) { return x; }
};
template <> struct Storage<double> {
    __device__ static double to_f64(double x) { return x; }
    __device__ static float to_f32(double x) { return (float)x; }
};

// Round a double to the nearest bfloat16, ties to even, in one rounding.
// Truncate to binary32 (toward zero), then make the result "sticky" by setting
// the lowest significand bit when the truncation was inexact (round-to-odd at
// 24 bits), then round to nearest-even at 8 bits.  Rounding to odd at a
// precision at least two bits wider than the target and then rounding to
// nearest gives the correctly rounded result (Boldo & Melquiond, "Emulation of
// FMA and correctly rounded sums: proved algorithms using rounding to odd").
__device__ __forceinline__ __nv_bfloat16 f64_to_bf16_rn(double x) {
    float t = __double2float_rz(x);
    uint32_t bits = __float_as_uint(t);
    if ((double)t != x && (bits & 0x7f800000u) != 0x7f800000u) bits |= 1u;
    return __float2bfloat16_rn(__uint_as_float(bits));
}

template <typename T> __device__ __forceinline__ T from_f64_rn(double x);
template <> __device__ __forceinline__ __nv_bfloat16 from_f64_rn<__nv_bfloat16>(double x) { return f64_to_bf16_rn(x); }
template <> __device__ __forceinline__ float from_f64_rn<float>(double x) { return __double2float_rn(x); }
template <> __device__ __forceinline__ double from_f64_rn<double>(double x) { return x; }

// RoPE rotation of one interleaved pair in float64 with every product and sum
// rounded separately (no fused multiply-add), so that the result equals the
// plain IEEE evaluation of (x c - y s, x s + y c).
__device__ __forceinline__ void rope_pair_f64(double x, double y, double c, double s,
                                              double& xr, double& yr) {
    xr = __dsub_rn(__dmul_rn(x, c), __dmul_rn(y, s));
    yr = __dadd_rn(__dmul_rn(x, s), __dmul_rn(y, c));
}

// ---- bf16 keys: float32 rotation with a per-element exactness proof ----------
//
// The stored key is defined as the float64 evaluation of (x c - y s, x s + y c),
// every product and sum rounded separately, rounded once to bf16.  With r the
// float32 result and E a bound on |r - X| (X the float64 value), rounding to
// nearest is monotone, so RN(r - E) == RN(r + E) implies RN(X) == RN(r).
// Elements where a bf16 rounding boundary lies within E (about one in a
// thousand) are evaluated in float64.

// The rare exact evaluation, kept out of line so that the common path carries no
// (predicated) float64 instructions.
static __device__ __noinline__ __nv_bfloat16 rope_bf16_fallback(float xf, float yf, const double2* table, int64_t ti,
                                                         bool second) {
    double2 cs = make_double2(1.0, 0.0);
    if (table) cs = table[ti];
    double xr, yr;
    rope_pair_f64((double)xf, (double)yf, cs.x, cs.y, xr, yr);
    return f64_to_bf16_rn(second ? yr : xr);
}

// One component of the rotated pair (second: x s + y c, else x c - y s) in
// float32 with one fused multiply-add; the bound covers the float32 rounding of
// cos/sin, of the other product and of the fused operation with a factor of 4
// to spare (each is at most 2^-24 relative to the terms' magnitudes).
static __device__ __forceinline__ __nv_bfloat16 rope_bf16_exact(float xf, float yf, float cf, float sf,
                                                        const double2* table, int pos, int pairs, int j,
                                                        bool second) {
    const float t2 = second ? xf * sf : yf * sf;
    const float t1a = second ? yf : xf;
    const float r = second ? fmaf(t1a, cf, t2) : fmaf(t1a, cf, -t2);
    const float bound = 0x1p-20f * (fabsf(t1a * cf) + fabsf(t2) + fabsf(r)) + 0x1p-140f;
    const __nv_bfloat16 lo = __float2bfloat16_rn(r - bound);
    const __nv_bfloat16 hi = __float2bfloat16_rn(r + bound);
    if (__builtin_expect(__bfloat16_as_ushort(lo) == __bfloat16_as_ushort(hi), 1)) return lo;
    return rope_bf16_fallback(xf, yf, table, (int64_t)pos * pairs + j, second);
}

// ---- warp reductions -------------------------------------------------------

template <typename A> __device__ __forceinline__ A warp_sum(A v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace kvc
