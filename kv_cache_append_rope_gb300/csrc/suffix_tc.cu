// Suffix-chunk causal attention on the 5th-generation tensor cores (bf16, d_h = 128).
//
// [LCP5] "LLM 机制实验（五）：改了历史，能否只重算变化的后缀？", section "先看一次历史编辑"
// and the listing under "哪些东西必须一起裁剪": after truncation to `cut`, the
// suffix rows continue at slot/position cut and each attends the retained
// prefix plus the suffix rows up to itself.  [Ch37] listing "Evaluate one newest
// query across the retained rows plus the candidate key/value row before
// committing the append" fixes the score scale 1/sqrt(d_h) and the
// max-subtracted softmax.  A long suffix is a dense Q K^T / P V contraction,
// which is why this kernel uses tcgen05 tiles.
//
// One CTA per work item (sequence b, query head h, 128-row query tile qt),
// items ordered longest first.  Query row i (slot cut + i) attends key slots
// 0 .. cut + i; key tiles are 128 slots, the last ones masked element-wise.
//
// Warp roles (192 threads):
//   warp 0    TMA producer: the rotated Q tile once, then K and V tiles into a
//             two-stage ring (128-byte swizzle, no multicast).
//   warp 1    TMEM allocator (512 columns) and, on one elected thread, the MMA
//             issuer: S = Q K^T into one of two TMEM S buffers (so the next
//             tile's QK^T overlaps the current softmax), then O += P V into
//             the TMEM O accumulator, each completion signalled with
//             tcgen05.commit on an mbarrier.
//   warps 2-5 softmax (thread = query row = TMEM lane): tcgen05.ld of the S
//             row, causal mask, running max in log2 units, O rescaled through
//             TMEM only when the max grows by more than 2^8 (the final
//             division by the running sum makes the stale max exact), P
//             written as bf16 into a swizzled shared-memory tile for the PV
//             MMA, and the normalised O row written to global memory.
// Every mbarrier wait is bounded (DEV_ERR_WAIT_TIMEOUT), the MMA thread waits
// for its own last commit and the TMA thread for its own copies before the
// allocator warp frees the tensor memory.
#include <cuda.h>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int HALF = BM * 128;             // 128 rows x 64 bf16 (one TMA box)
constexpr int TILE = 2 * HALF;             // 128 rows x 128 bf16
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;        // two stages
constexpr int OFF_V = OFF_K + 2 * TILE;    // two stages
constexpr int OFF_P = OFF_V + 2 * TILE;
constexpr int OFF_BAR = OFF_P + TILE;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
constexpr float RESCALE_LOG2 = 8.0f;

struct Bars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, o_ready, mma_done;
    uint32_t tmem_base;
    int err;
};

__device__ __forceinline__ void fail_wait(Bars* bars, uint32_t* err) {
    *(volatile int*)&bars->err = 1;
    atomicOr(err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
}

// A bounded wait taken by every lane of a warp, with one verdict for the whole warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const uint32_t* abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
}

__global__ void __launch_bounds__(THREADS, 1) suffix_tc_kernel(const __grid_constant__ SuffixLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int4 w = a.work[blockIdx.x];
    const int b = w.x, h = w.y, qt = w.z, n = w.w;
    const int g = h / (a.Hq / a.Hkv);
    const int cut = a.slot0[b];
    const int rows_b = a.seqlen[b];

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
            mbar_init(smem_u32(&bars->s_full[s]), 1);
            mbar_init(smem_u32(&bars->s_free[s]), 4);
        }
        mbar_init(smem_u32(&bars->p_full), 4);
        mbar_init(smem_u32(&bars->o_ready), 1);
        mbar_init(smem_u32(&bars->mma_done), 1);
        bars->err = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&a.tmQ);
            prefetch_tmap(&a.tmK);
            prefetch_tmap(&a.tmV);
            const int qrow = (b * a.Hq + h) * a.S + qt * BM;
            const int kvrow = (b * a.Hkv + g) * a.C;
            const uint32_t qb = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(qb, TILE);
            tma_load_2d(smem_u32(smem + OFF_Q), &a.tmQ, 0, qrow, qb);
            tma_load_2d(smem_u32(smem + OFF_Q + HALF), &a.tmQ, 64, qrow, qb);
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < n && !*(volatile int*)&bars->err; ++j) {
                const int s = j & 1, use = j >> 1;
                if (j >= 2 && !mbar_wait_bounded(smem_u32(&bars->k_empty[s]), (use - 1) & 1, a.err)) {
                    fail_wait(bars, a.err);
                    break;
                }
                const uint32_t kb = smem_u32(&bars->k_full[s]);
                mbar_arrive_expect_tx(kb, TILE);
                tma_load_2d(smem_u32(smem + OFF_K + s * TILE), &a.tmK, 0, kvrow + j * BN, kb);
                tma_load_2d(smem_u32(smem + OFF_K + s * TILE + HALF), &a.tmK, 64, kvrow + j * BN, kb);
                issued_k = j + 1;
                if (j >= 2 && !mbar_wait_bounded(smem_u32(&bars->v_empty[s]), (use - 1) & 1, a.err)) {
                    fail_wait(bars, a.err);
                    break;
                }
                const uint32_t vb = smem_u32(&bars->v_full[s]);
                mbar_arrive_expect_tx(vb, TILE);
                tma_load_2d(smem_u32(smem + OFF_V + s * TILE), &a.tmV, 0, kvrow + j * BN, vb);
                tma_load_2d(smem_u32(smem + OFF_V + s * TILE + HALF), &a.tmV, 64, kvrow + j * BN, vb);
                issued_v = j + 1;
            }
            // Our own copies must have landed before the CTA's shared memory is released.
            mbar_wait_bounded(qb, 0, a.err);
            for (int t = issued_k - 2 < 0 ? 0 : issued_k - 2; t < issued_k; ++t)
                mbar_wait_bounded(smem_u32(&bars->k_full[t & 1]), (t >> 1) & 1, a.err);
            for (int t = issued_v - 2 < 0 ? 0 : issued_v - 2; t < issued_v; ++t)
                mbar_wait_bounded(smem_u32(&bars->v_full[t & 1]), (t >> 1) & 1, a.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
            const uint32_t q_s = smem_u32(smem + OFF_Q);
            const uint32_t p_s = smem_u32(smem + OFF_P);
            bool ok = mbar_wait_bounded(smem_u32(&bars->q_full), 0, a.err);
            if (!ok) fail_wait(bars, a.err);
            tc_fence_after();
            auto issue_qk = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait_bounded(smem_u32(&bars->k_full[s]), (j >> 1) & 1, a.err)) return false;
                if (j >= 2 && !mbar_wait_bounded(smem_u32(&bars->s_free[s]), ((j >> 1) - 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint32_t k_s = smem_u32(smem + OFF_K + s * TILE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
                    tc_mma_ss(tmem + (s ? COL_S1 : COL_S0), smem_desc_sw128(q_s + off, 16, 1024),
                              smem_desc_sw128(k_s + off, 16, 1024), idesc_qk, kk > 0);
                }
                tc_commit(smem_u32(&bars->s_full[s]));
                tc_commit(smem_u32(&bars->k_empty[s]));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n && !(ok = issue_qk(j + 1))) break;
                const int s = j & 1;
                if (!mbar_wait_bounded(smem_u32(&bars->p_full), j & 1, a.err) ||
                    !mbar_wait_bounded(smem_u32(&bars->v_full[s]), (j >> 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t v_s = smem_u32(smem + OFF_V + s * TILE);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // A = P (K-major over keys), B = V (rows = keys, contiguous head dims: MN-major)
                    const uint32_t poff = (kk >> 2) * HALF + (kk & 3) * 32;
                    tc_mma_ss(tmem + COL_O, smem_desc_sw128(p_s + poff, 16, 1024),
                              smem_desc_sw128(v_s + kk * 16 * 128, HALF, 1024), idesc_pv, (j > 0 || kk > 0));
                }
                tc_commit(smem_u32(&bars->o_ready));
                tc_commit(smem_u32(&bars->v_empty[s]));
            }
            if (!ok) fail_wait(bars, a.err);
            // every MMA issued by this thread completes before the tensor memory is freed
            tc_commit(smem_u32(&bars->mma_done));
            mbar_wait_bounded(smem_u32(&bars->mma_done), 0);  // no abort: the MMAs always finish
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroup
        const int sub = warp & 3;                    // TMEM sub-partition of this warp
        const int row = sub * 32 + lane;             // query row inside the tile = TMEM lane
        const int i = qt * BM + row;
        const int qslot = cut + i;
        const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
        uint8_t* prow = smem + OFF_P + row * 128;
        const float sl2 = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int s = j & 1;
            if (!warp_wait(smem_u32(&bars->s_full[s]), (j >> 1) & 1, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_addr + (s ? COL_S1 : COL_S0) + c * 32, x + c * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[s]));

            const int kbase = j * BN;
            if (kbase + BN - 1 > cut + qt * BM) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (kbase + c > qslot) x[c] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) mx = fmaxf(mx, x[c]);
            const float m_tile = mx * sl2;
            const bool grow = m_tile > m_run + RESCALE_LOG2 || (j == 0);
            const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
            if (j > 0) {
                // PV of the previous tile must be done: O is rescaled below and P is rewritten.
                if (!warp_wait(smem_u32(&bars->o_ready), (j - 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (grow && m_run > -INFINITY) {
                    const float corr = fast_exp2(m_run - m_new);
                    l_run *= corr;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(lane_addr + COL_O + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= corr;
                        tmem_st32(lane_addr + COL_O + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            m_run = m_new;
            const float mu = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
            for (int ch = 0; ch < BN / 8; ++ch) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = fast_exp2(fmaf(x[ch * 8 + 2 * e], sl2, -mu));
                    const float p1 = fast_exp2(fmaf(x[ch * 8 + 2 * e + 1], sl2, -mu));
                    l_run += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                const uint32_t addr = smem_u32(prow + (ch >> 3) * HALF + ((((ch & 7) ^ (row & 7))) << 4));
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[0]), "r"(pk[1]),
                             "r"(pk[2]), "r"(pk[3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
        }
        if (ok && n > 0) {
            if (!warp_wait(smem_u32(&bars->o_ready), (n - 1) & 1, a.err)) {
                ok = false;
            } else {
                tc_fence_after();
                const float inv = 1.0f / l_run;
                float* orow = a.out + (((int64_t)b * a.Hq + h) * a.S + i) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(lane_addr + COL_O + c * 32, o);
                    tmem_wait_ld();
                    if (i < rows_b) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *(float4*)(orow + c * 32 + e) =
                                make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
                    }
                }
            }
        }
        if (!ok) fail_wait(bars, a.err);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int suffix_tc_grid(int sms) { return sms; }

cudaError_t launch_suffix_tc(const SuffixLaunch& a, int grid, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(suffix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (grid <= 0) return cudaSuccess;
    suffix_tc_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
