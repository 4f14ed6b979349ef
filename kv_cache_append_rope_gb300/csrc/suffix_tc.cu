// Suffix-chunk causal attention on the 5th-generation tensor cores (bf16, d_h = 128).
//
// [LCP5] "LLM 机制实验（五）：改了历史，能否只重算变化的后缀？", section "先看一次历史编辑"
// and the listing under "哪些东西必须一起裁剪": after truncation to `cut`, the
// suffix rows continue at slot/position cut and each attends the retained
// prefix plus the suffix rows up to itself.  [Ch37] listing "Evaluate one newest
// query across the retained rows plus the candidate key/value row before
// committing the append" fixes the score scale 1/sqrt(d_h) and the
// max-subtracted softmax.  With a sliding window of W slots ([LCP5]
// "为什么滑窗部分命中必须回退") row cut + i sees slots cut + i - W + 1 .. cut + i:
// its key tiles start later and the first ones are masked from below too.  A long suffix is a dense Q K^T / P V contraction,
// which is why this kernel uses tcgen05 tiles.
//
// One CTA per work item (sequence b, query head h, 128-row query tile qt).
// Items are grouped by (b, h) -- the query tiles of one head launch together
// and walk its K/V tiles in step, so each tile comes from DRAM once and from
// L2 for the rest -- and the groups are ordered by total work, longest first.  Query row i (slot cut + i) attends key slots
// 0 .. cut + i; key tiles are 128 slots, the last ones masked element-wise.
//
// Warp roles (320 threads):
//   warp 0    TMA producers (128-byte swizzle, no multicast): lane 0 the
//             rotated Q tile once and K tiles into a 3-stage ring, lane 1 V
//             tiles into a 2-stage ring.
//   warp 1    TMEM allocator (512 columns) and, on one elected thread, the MMA
//             issuer: S = Q K^T into one of two TMEM S buffers (so the next
//             tile's QK^T overlaps the current softmax), then O += P V into
//             the TMEM O accumulator with P read from tensor memory, each
//             completion signalled with tcgen05.commit on an mbarrier.
// Tensor memory: S0, S1, O (128 columns each), P0, P1 (64 columns each).
//   warps 2-9 softmax, two warps per TMEM sub-partition, each thread one
//             query row (= TMEM lane) and one half of its 128 columns, the
//             pair exchanging row maxima through shared memory (an mbarrier
//             of 64 arrivals): tcgen05.ld of the S half-row, causal mask,
//             running max in log2 units, O rescaled through
//             TMEM only when the max grows by more than 2^8 (the final
//             division by the running sum makes the stale max exact), P
//             computed in registers while the previous tile's PV runs, then
//             written as packed bf16 into one of two 64-column tensor-memory
//             P buffers (tcgen05.st), from which the PV MMA reads its A
//             operand, and the normalised O row written to global memory.
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
constexpr int KST = 3, VST = 2;            // K and V ring stages (K is needed first)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;
constexpr int OFF_V = OFF_K + KST * TILE;
constexpr int OFF_BAR = OFF_V + VST * TILE;
constexpr int SMEM_BYTES = OFF_BAR + 8192 + 1024;
constexpr int WPS = 2;                     // softmax warps per TMEM sub-partition
constexpr int NSW = 4 * WPS;               // softmax warps
constexpr int THREADS = (2 + NSW) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256, COL_P0 = 384, COL_P1 = 448;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int kTileCache = 256;            // paged: key tiles whose row coordinates are staged in shared memory

struct Bars {
    float red_max[2][WPS][BM]; // [tile parity][column part][row]: partial row maxima
    float red_sum[WPS][BM];    // [column part][row]: partial row sums
    uint64_t q_full;
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2], pv_done[2], mma_done;
    uint64_t xchg[4][2];       // [sub-partition][tile parity]: the two softmax warps of a row block
    uint64_t fin[4];           // [sub-partition]: final partial sums
    uint32_t tmem_base;
    int err;
    int2 ty[kTileCache];       // paged: TMA row coordinates of the two halves of this item's key tiles
};

__device__ __forceinline__ void fail_wait(Bars* bars, uint32_t* err) {
    *(volatile int*)&bars->err = 1;
    atomicOr(err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
}

// Pool row of a slot in paged storage; a slot past the sequence's blocks (the
// second half of its last key tile) maps to rows -64..-1, where the TMA
// load fills zeros (those keys are masked).
__device__ __forceinline__ int paged_row(const KvLayout& L, int b, int h, int slot) {
    const int j = slot >> L.shift;
    const int blk = j < L.nblk ? L.table[(int64_t)b * L.nblk + j] : -1;
    return blk < 0 ? -64 : ((blk * L.Hkv + h) << L.shift) + (slot & (L.P - 1));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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
    // first key tile: 0, or with a sliding window the tile holding the earliest slot
    // any row of this query tile sees (its first row's slot - window + 1)
    const int j0 = a.window > 0 ? max(0, cut + qt * BM - a.window + 1) / BN : 0;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int s = 0; s < KST; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->s_full[s]), 1);
            mbar_init(smem_u32(&bars->s_free[s]), NSW);
            mbar_init(smem_u32(&bars->p_full[s]), NSW);
            mbar_init(smem_u32(&bars->pv_done[s]), 1);
        }
        mbar_init(smem_u32(&bars->mma_done), 1);
        for (int q = 0; q < 4; ++q) {
            mbar_init(smem_u32(&bars->xchg[q][0]), 32 * WPS);
            mbar_init(smem_u32(&bars->xchg[q][1]), 32 * WPS);
            mbar_init(smem_u32(&bars->fin[q]), 32 * WPS);
        }
        bars->err = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    // Paged storage: warp 0 looks up the pool rows of both 64-row halves of this item's
    // key tiles once, in parallel, and stages them in shared memory, so the producers'
    // path per tile is one shared load (tiles past the staged ones are looked up
    // directly).
    if (a.kv.table && warp == 0)
        for (int e = lane; e < min(n, kTileCache); e += 32)
            bars->ty[e] = make_int2(paged_row(a.kv, b, g, (j0 + e) * BN), paged_row(a.kv, b, g, (j0 + e) * BN + 64));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // lane 0 streams Q and the K ring, lane 1 the V ring, so that the K
        // look-ahead never waits behind a V stage that is still being read.
        if (lane < 2) {
            const int kvrow = (b * a.Hkv + g) * a.C;   // contiguous storage
            const bool is_k = lane == 0;
            const int NS = is_k ? KST : VST;
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
            const CUtensorMap* map = is_k ? &a.tmK : &a.tmV;
            uint8_t* ring = smem + (is_k ? OFF_K : OFF_V);
            prefetch_tmap(map);
            uint32_t qb = 0;
            if (is_k) {
                prefetch_tmap(&a.tmQ);
                const int qrow = (b * a.Hq + h) * a.S + qt * BM;
                qb = smem_u32(&bars->q_full);
                mbar_arrive_expect_tx(qb, TILE);
                tma_load_2d(smem_u32(smem + OFF_Q), &a.tmQ, 0, qrow, qb);
                tma_load_2d(smem_u32(smem + OFF_Q + HALF), &a.tmQ, 64, qrow, qb);
            }
            int issued = 0;
            for (int j = 0; j < n && !*(volatile int*)&bars->err; ++j) {
                const int s = j % NS, use = j / NS;
                if (j >= NS && !mbar_wait_bounded(smem_u32(&empty[s]), (use - 1) & 1, a.err)) {
                    fail_wait(bars, a.err);
                    break;
                }
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, TILE);
                if (!a.kv.table) {
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, kvrow + (j0 + j) * BN, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, kvrow + (j0 + j) * BN, fb);
                } else {
                    // paged: the two 64-row halves of the tile, each inside one block
                    // (64-row box map; same 128-byte-swizzled layout as one 128-row box)
                    const int2 yy = j < kTileCache ? bars->ty[j]
                                                   : make_int2(paged_row(a.kv, b, g, (j0 + j) * BN),
                                                               paged_row(a.kv, b, g, (j0 + j) * BN + 64));
                    const int ya = yy.x, yb = yy.y;
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, ya, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + 64 * 128), map, 0, yb, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, ya, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF + 64 * 128), map, 64, yb, fb);
                }
                issued = j + 1;
            }
            // Our own copies must have landed before the CTA's shared memory is released.
            if (is_k) mbar_wait_bounded(qb, 0, a.err);
            for (int t = issued - NS < 0 ? 0 : issued - NS; t < issued; ++t)
                mbar_wait_bounded(smem_u32(&full[t % NS]), (t / NS) & 1, a.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
            const uint32_t q_s = smem_u32(smem + OFF_Q);
            bool ok = mbar_wait_bounded(smem_u32(&bars->q_full), 0, a.err);
            if (!ok) fail_wait(bars, a.err);
            tc_fence_after();
            auto issue_qk = [&](int j) -> bool {
                const int s = j & 1, ks = j % KST;
                if (!mbar_wait_bounded(smem_u32(&bars->k_full[ks]), (j / KST) & 1, a.err)) return false;
                if (j >= 2 && !mbar_wait_bounded(smem_u32(&bars->s_free[s]), ((j >> 1) - 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint32_t k_s = smem_u32(smem + OFF_K + ks * TILE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
                    tc_mma_ss(tmem + (s ? COL_S1 : COL_S0), smem_desc_sw128(q_s + off, 16, 1024),
                              smem_desc_sw128(k_s + off, 16, 1024), idesc_qk, kk > 0);
                }
                tc_commit(smem_u32(&bars->s_full[s]));
                tc_commit(smem_u32(&bars->k_empty[ks]));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n && !(ok = issue_qk(j + 1))) break;
                const int s = j & 1, vs = j % VST;
                if (!mbar_wait_bounded(smem_u32(&bars->p_full[s]), (j >> 1) & 1, a.err) ||
                    !mbar_wait_bounded(smem_u32(&bars->v_full[vs]), (j / VST) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t v_s = smem_u32(smem + OFF_V + vs * TILE);
                const uint32_t p_t = tmem + (s ? COL_P1 : COL_P0);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // A = P from tensor memory (16 keys = 8 columns per step),
                    // B = V (rows = keys, contiguous head dims: MN-major)
                    tc_mma_ts(tmem + COL_O, p_t + kk * 8, smem_desc_sw128(v_s + kk * 16 * 128, HALF, 1024),
                              idesc_pv, (j > 0 || kk > 0));
                }
                tc_commit(smem_u32(&bars->pv_done[s]));
                tc_commit(smem_u32(&bars->v_empty[vs]));
            }
            if (!ok) fail_wait(bars, a.err);
            // every MMA issued by this thread completes before the tensor memory is freed
            tc_commit(smem_u32(&bars->mma_done));
            mbar_wait_bounded(smem_u32(&bars->mma_done), 0);  // no abort: the MMAs always finish
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        // Warp w reads TMEM lanes 32 * (w % 4) .. + 31 (its sub-partition); the
        // WPS warps of a sub-partition take consecutive column parts of those rows.
        constexpr int HC = BN / WPS;                 // columns per warp
        const int sub = warp & 3;
        const int half = (warp - 2) >> 2;            // column part
        const int row = sub * 32 + lane;             // query row inside the tile = TMEM lane
        const int i = qt * BM + row;
        const int qslot = cut + i;
        const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
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
            float x[HC];
            const uint32_t s_col = (s ? COL_S1 : COL_S0) + half * HC;
#pragma unroll
            for (int c = 0; c < HC / 32; ++c) tmem_ld32(lane_addr + s_col + c * 32, x + c * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->s_free[s]));

            const int kbase = (j0 + j) * BN + half * HC;
            // causal mask (keys after the row's slot) on diagonal tiles; with a window also
            // the keys before slot - window + 1 on the first tiles
            const bool past_window = a.window > 0 && kbase < cut + qt * BM + BM - a.window;
            if (kbase + HC - 1 > cut + qt * BM || past_window) {
                const int klo = a.window > 0 ? qslot - a.window + 1 : 0;
#pragma unroll
                for (int c = 0; c < HC; ++c) x[c] = (kbase + c > qslot || kbase + c < klo) ? -INFINITY : x[c];
            }
            // row maximum over this part (8 independent chains of 3-input maxima),
            // then over the other parts of the same rows
            float m8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) m8[q] = x[q];
#pragma unroll
            for (int c = 8; c + 16 <= HC; c += 16)
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = fmax3(m8[q], x[c + q], x[c + 8 + q]);
            if constexpr ((HC - 8) % 16 != 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = fmaxf(m8[q], x[HC - 8 + q]);
            }
            float mpart = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            bars->red_max[s][half][row] = mpart;
            mbar_arrive(smem_u32(&bars->xchg[sub][s]));
            if (!warp_wait(smem_u32(&bars->xchg[sub][s]), (j >> 1) & 1, a.err)) {
                ok = false;
                break;
            }
            float mx = mpart;
#pragma unroll
            for (int q = 0; q < WPS; ++q)
                if (q != half) mx = fmaxf(mx, bars->red_max[s][q][row]);
            const float m_tile = mx * sl2;
            const bool grow = m_tile > m_run + RESCALE_LOG2 || (j == 0);
            const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
            if (grow && j > 0 && m_run > -INFINITY) {
                // O holds the sum over earlier tiles: wait for PV of tile j-1, then rescale this half.
                if (!warp_wait(smem_u32(&bars->pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float corr = fast_exp2(m_run - m_new);
                l_run *= corr;
#pragma unroll
                for (int c = 0; c < HC / 32; ++c) {
                    float o[32];
                    const uint32_t oa = lane_addr + COL_O + half * HC + c * 32;
                    tmem_ld32(oa, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= corr;
                    tmem_st32(oa, o);
                }
                tmem_wait_st();
            }
            m_run = m_new;
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            // P in registers first: the exponentials overlap the previous tile's PV.
            // (packed float32x2 FMA for the arguments and packed adds for the sums:
            // the softmax warps are issue-bound, so fewer instructions matter)
            uint32_t pk[HC / 2];
            float2 l4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) l4[q] = make_float2(0.f, 0.f);
            const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
#pragma unroll
            for (int e = 0; e < HC / 2; ++e) {
                const float2 arg = __ffma2_rn(make_float2(x[2 * e], x[2 * e + 1]), sl2v, negmu);
                const float p0 = fast_exp2(arg.x);
                const float p1 = fast_exp2(arg.y);
                l4[e & 3] = __fadd2_rn(l4[e & 3], make_float2(p0, p1));
                pk[e] = pack_bf16(p0, p1);
            }
            l4[0] = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
            l_run += l4[0].x + l4[0].y;
            // P buffer s was last read by the PV of tile j-2.
            if (j >= 2 && !warp_wait(smem_u32(&bars->pv_done[s]), ((j >> 1) - 1) & 1, a.err)) {
                ok = false;
                break;
            }
            if constexpr (HC / 2 == 32) {
                tmem_st32u(lane_addr + (s ? COL_P1 : COL_P0) + half * (HC / 2), pk);
            } else {
                tmem_st16u(lane_addr + (s ? COL_P1 : COL_P0) + half * (HC / 2), pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[s]));
        }
        bars->red_sum[half][row] = l_run;
        mbar_arrive(smem_u32(&bars->fin[sub]));
        if (!warp_wait(smem_u32(&bars->fin[sub]), 0, a.err)) ok = false;
        if (ok && n > 0) {
            if (!warp_wait(smem_u32(&bars->pv_done[(n - 1) & 1]), ((n - 1) >> 1) & 1, a.err)) {
                ok = false;
            } else {
                tc_fence_after();
                float lsum = 0.f;
#pragma unroll
                for (int q = 0; q < WPS; ++q) lsum += bars->red_sum[q][row];
                const float inv = 1.0f / lsum;
                float* orow = a.out + (((int64_t)b * a.Hq + h) * a.S + i) * D + half * HC;
#pragma unroll
                for (int c = 0; c < HC / 32; ++c) {
                    float o[32];
                    tmem_ld32(lane_addr + COL_O + half * HC + c * 32, o);
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
