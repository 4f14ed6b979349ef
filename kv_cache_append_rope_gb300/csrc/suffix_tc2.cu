// Suffix-chunk causal attention on pairs of SMs (cta_group::2), selected with
// KVC_OPT_SUFFIX_KERNEL = 3 for contiguous bf16 storage with d_h = 128.
//
// Same computation as the one-SM tile kernel ([LCP5] "先看一次历史编辑": suffix row
// cut + i attends slots 0 .. cut + i; [Ch37] fixes the 1/sqrt(d_h) scale and the
// max-subtracted softmax), with the same softmax warp code per query row.
//
// A cluster of two CTAs computes four 128-row query tiles of one (sequence, head):
// CTA r holds tiles A_r = 4q + r and B_r = 4q + 2 + r.  The leader (rank 0) issues
// every MMA for the pair with cta_group::2 and M = 256: QK^T takes A = Q (each CTA's
// own 128 rows from its own shared memory) and B = K with the 128 keys of a tile
// split between the CTAs (64 each); PV takes A = P from each CTA's tensor memory and
// B = V with the 128 head dims split between the CTAs (64 each).  Per SM and key tile
// the shared-memory port then carries 160 KB instead of 256 KB, and each CTA loads
// half of every K and V tile.  MMA completions are multicast to both CTAs; P-ready
// arrivals go to the leader's barriers.  Both CTAs' TMA loads complete directly on
// the leader's barriers (the .cta_group::2 form of the bulk tensor copy signals the
// pair's leader); the leader's producer arms each stage for the bytes of both CTAs.
//
// Tensor memory: both CTAs execute tcgen05.alloc.cta_group::2 and receive the same
// base (the pair allocates together; 512 columns in each SM), and both free it after
// a cluster barrier, so that neither CTA leaves while the pair still uses its memory.
// Every mbarrier wait is bounded (DEV_ERR_WAIT_TIMEOUT), as in the one-SM kernel.
//
// Status: its results match the oracle, but on the B = 8 suffix workload the step
// takes longer than with the one-SM kernel, so the automatic choice is the one-SM kernel.
#include <cuda.h>

#include <type_traits>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int QT = 2;
constexpr int HALF = BM * 128;         // 128 rows x 64 bf16
constexpr int TILE = 2 * HALF;         // 128 rows x 128 bf16
constexpr int KHALF = 64 * 128;        // 64 rows x 64 bf16
constexpr int KSTAGE = 2 * KHALF;      // this CTA's 64 keys x 128 dims
constexpr int VSTAGE = HALF;           // 128 keys x this CTA's 64 dims
constexpr int KST = 4, VST = 4;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QT * TILE;
constexpr int OFF_V = OFF_K + KST * KSTAGE;
constexpr int OFF_BAR = OFF_V + VST * VSTAGE;
constexpr int SMEM_BYTES = OFF_BAR + 1024 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
constexpr int NSW = 4 * QT;
constexpr int THREADS = (4 + NSW) * 32;
constexpr int kLaunchRegs = 168, kRegsLow = 120, kRegsHigh = 192;
static_assert(128 * kRegsLow + 2 * 128 * kRegsHigh == THREADS * kLaunchRegs, "register split");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256;
constexpr float RESCALE_LOG2 = 8.0f;

struct Bars {
    uint64_t q_full;                       // leader: both CTAs' query tiles landed
    uint64_t k_full[KST], v_full[VST];     // leader: both halves of a stage landed
    uint64_t k_empty[KST], v_empty[VST];   // each CTA: the pair's MMAs released the stage
    uint64_t s_full[QT];                   // each CTA: S_X written
    uint64_t p_full[QT];                   // leader: P_X written in both CTAs
    uint64_t o_done;                       // each CTA: every MMA of the item completed
    uint32_t tmem_base;
    int err;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait (cluster-scope acquire): false after kWaitLimitNs or when `abort` is set.
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, const uint32_t* abort = nullptr) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (global_timer_ns() - t0 > kWaitLimitNs) return false;
            if (abort && *(const volatile uint32_t*)abort) return false;
        }
    }
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, const uint32_t* abort) {
    return __all_sync(0xffffffffu, wait_cluster(bar, parity, abort));
}
// Bulk tensor copy into this CTA's shared memory whose completion is counted on
// `bar`, a barrier of the pair's leader (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on `bar` in both CTAs of the pair once every MMA issued so far has completed.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void fail_wait(Bars* bars, uint32_t* err) {
    *(volatile int*)&bars->err = 1;
    atomicOr(err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
}

// Key tiles [lo, hi) of query tile qt (empty past the sequence's rows).
__device__ __forceinline__ void tile_range(int qt, int cut, int rows, int window, int& lo, int& hi) {
    const int r0 = qt * BM;
    if (r0 >= rows) {
        lo = hi = 0;
        return;
    }
    const int q_end = min(r0 + BM, rows);
    lo = window > 0 ? max(0, cut + r0 - window + 1) / BN : 0;
    hi = (cut + q_end - 1) / BN + 1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    suffix_tc2_kernel(const __grid_constant__ SuffixLaunch2 a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    const int4 w = a.work[blockIdx.x >> 1];
    const int b = w.x, h = w.y, quad = w.z;
    const int g = h / (a.Hq / a.Hkv);
    const int cut = a.slot0[b];
    const int rows_b = a.seqlen[b];
    // debug builds: both CTAs of the pair read the same item and leave together, before
    // any cluster barrier
    if (!debug_check(cut >= 0 && rows_b >= 0 && cut + rows_b <= a.C, threadIdx.x == 0 ? a.err : nullptr)) return;
    // pair tile X covers query tiles 4 quad + 2 X (in CTA 0) and + 1 (in CTA 1); its key
    // range is the union of theirs
    int jlo[QT], jhi[QT];
#pragma unroll
    for (int X = 0; X < QT; ++X) {
        int l0, h0, l1, h1;
        tile_range(4 * quad + 2 * X, cut, rows_b, a.window, l0, h0);
        tile_range(4 * quad + 2 * X + 1, cut, rows_b, a.window, l1, h1);
        jlo[X] = l0;
        jhi[X] = max(h0, h1);
        if (h0 == 0) jlo[X] = jhi[X] = 0;
    }
    const int j_first = jlo[0];
    const int n = max(jhi[0], jhi[1]) - j_first;
    const int my_tile[QT] = {4 * quad + (int)rank, 4 * quad + 2 + (int)rank};

    if (threadIdx.x == 0) {
        // full barriers: one arrival (the leader's producer, arming both CTAs' bytes)
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int s = 0; s < KST; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
        }
        for (int X = 0; X < QT; ++X) {
            mbar_init(smem_u32(&bars->s_full[X]), 1);
            mbar_init(smem_u32(&bars->p_full[X]), 8);
        }
        mbar_init(smem_u32(&bars->o_done), 1);
        bars->err = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers initialised and tensor memory allocated before any remote use
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 4) {
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane < 2) {
            // ------------------------------------------------------------ TMA producers
            // (both CTAs; every copy completes on the leader's barrier of its stage, which
            // the leader arms for both CTAs' bytes)
            const int kvrow = (b * a.Hkv + g) * a.C;
            const bool is_k = lane == 0;
            const int NS = is_k ? KST : VST;
            const uint32_t stage_bytes = is_k ? KSTAGE : VSTAGE;
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
            uint8_t* ring = smem + (is_k ? OFF_K : OFF_V);
            const CUtensorMap* map = is_k ? &a.tmK64 : &a.tmV128;
            prefetch_tmap(map);
            if (is_k) {
                prefetch_tmap(&a.tmQ);
                if (leader) mbar_arrive_expect_tx(smem_u32(&bars->q_full), 2 * QT * TILE);
                const uint32_t qb = mapa(smem_u32(&bars->q_full), 0);
#pragma unroll
                for (int X = 0; X < QT; ++X) {
                    const int qrow = (b * a.Hq + h) * a.S + my_tile[X] * BM;
                    tma_load_2d_pair(smem_u32(smem + OFF_Q + X * TILE), &a.tmQ, 0, qrow, qb);
                    tma_load_2d_pair(smem_u32(smem + OFF_Q + X * TILE + HALF), &a.tmQ, 64, qrow, qb);
                }
            }
            bool failed = false;
            for (int j = 0; j < n && !*(volatile int*)&bars->err && !*(volatile uint32_t*)a.err; ++j) {
                const int s = j % NS, use = j / NS;
                if (j >= NS && !wait_cluster(smem_u32(&empty[s]), (use - 1) & 1, a.err)) {
                    fail_wait(bars, a.err);
                    failed = true;
                    break;
                }
                if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * stage_bytes);
                const uint32_t fb = mapa(smem_u32(&full[s]), 0);
                const int key0 = kvrow + (j_first + j) * BN;
                if (is_k) {
                    // this CTA's 64 keys of the tile, both 64-dim halves
                    tma_load_2d_pair(smem_u32(ring + s * KSTAGE), map, 0, key0 + 64 * (int)rank, fb);
                    tma_load_2d_pair(smem_u32(ring + s * KSTAGE + KHALF), map, 64, key0 + 64 * (int)rank, fb);
                } else {
                    // all 128 keys of the tile, this CTA's 64 dims
                    tma_load_2d_pair(smem_u32(ring + s * VSTAGE), map, 64 * (int)rank, key0, fb);
                }
            }
            // Every copy issued here is consumed by the leader's MMAs, which wait for its
            // stage to complete, before the final cluster barrier: on the normal path the
            // shared memory is never released under a copy.  On an error path (a wait gave
            // up) some copies may be unconsumed: give them a bounded 200 us to land.
            if (failed || *(volatile int*)&bars->err || *(volatile uint32_t*)a.err) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) {
                }
            }
        } else if (warp == 1 && lane == 0 && leader) {
            // ------------------------------------------------------------ MMA issuer (leader)
            constexpr uint32_t idesc_qk = idesc_bf16_f32(2 * BM, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(2 * BM, D, false, true);
            bool ok = wait_cluster(smem_u32(&bars->q_full), 0, a.err);
            if (!ok) fail_wait(bars, a.err);
            tc_fence_after();
            auto active = [&](int X, int jj) { return jj >= jlo[X] && jj < jhi[X]; };
            const uint64_t dq = smem_desc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
            const uint64_t dk = smem_desc_sw128(smem_u32(smem + OFF_K), 16, 1024);
            const uint64_t dv = smem_desc_sw128(smem_u32(smem + OFF_V), HALF, 1024);
            auto issue_qk = [&](int X, int ks) {
                const uint64_t qd = dq + (uint64_t)((X * TILE) >> 4);
                const uint64_t kd = dk + (uint64_t)((ks * KSTAGE) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qoff = ((kk >> 2) * HALF + (kk & 3) * 32) >> 4;
                    const uint32_t koff = ((kk >> 2) * KHALF + (kk & 3) * 32) >> 4;
                    mma_ss_pair(tmem + COL_S + X * 128, qd + qoff, kd + koff, idesc_qk, kk > 0);
                }
                commit_pair(smem_u32(&bars->s_full[X]));
            };
            int pv_count[QT] = {0, 0};
            if (ok) {
                if (!wait_cluster(smem_u32(&bars->k_full[0]), 0, a.err)) ok = false;
                tc_fence_after();
                for (int X = 0; ok && X < QT; ++X)
                    if (active(X, j_first)) issue_qk(X, 0);
                if (ok) commit_pair(smem_u32(&bars->k_empty[0]));
            }
            for (int j = 0; ok && j < n; ++j) {
                const int jj = j_first + j, vs = j % VST;
                const bool next = j + 1 < n;
                const int ks1 = (j + 1) % KST;
                if (!wait_cluster(smem_u32(&bars->v_full[vs]), (j / VST) & 1, a.err) ||
                    (next && !wait_cluster(smem_u32(&bars->k_full[ks1]), ((j + 1) / KST) & 1, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t vd = dv + (uint64_t)((vs * VSTAGE) >> 4);
                for (int X = 0; ok && X < QT; ++X) {
                    if (active(X, jj)) {
                        if (!wait_cluster(smem_u32(&bars->p_full[X]), pv_count[X] & 1, a.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts_pair(tmem + COL_O + X * 128, tmem + COL_S + X * 128 + kk * 8,
                                        vd + (uint64_t)(kk * 16 * 128 >> 4), idesc_pv, (pv_count[X] > 0 || kk > 0));
                        pv_count[X] += 1;
                    }
                    if (next && active(X, jj + 1)) issue_qk(X, ks1);
                }
                if (!ok) break;
                commit_pair(smem_u32(&bars->v_empty[vs]));
                if (next) commit_pair(smem_u32(&bars->k_empty[ks1]));
            }
            if (!ok) fail_wait(bars, a.err);
            commit_pair(smem_u32(&bars->o_done));
            wait_cluster(smem_u32(&bars->o_done), 0);
        }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ------------------------------------------------------------ softmax (both CTAs)
        const int X = (warp - 4) >> 2;
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        const int qt = my_tile[X];
        const int i = qt * BM + row;
        const int qslot = cut + i;
        const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
        const uint32_t s_addr = lane_addr + COL_S + X * 128;
        const uint32_t o_addr = lane_addr + COL_O + X * 128;
        const uint32_t p_leader = mapa(smem_u32(&bars->p_full[X]), 0);
        const float sl2 = a.scale_log2;
        const int tile_slot0 = cut + qt * BM;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int c = 0;
        for (int jj = jlo[X]; jj < jhi[X]; ++jj, ++c) {
            if (!warp_wait_cluster(smem_u32(&bars->s_full[X]), c & 1, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // masked: diagonal or later tiles (the pair's range reaches the other CTA's rows),
            // and with a window the tiles that start before some row's window
            const bool masked =
                jj * BN + BN - 1 > tile_slot0 || (a.window > 0 && jj * BN < tile_slot0 + BM - a.window);
            auto tile = [&](auto mask_c) {
                float x[BN];
#pragma unroll
                for (int q = 0; q < BN / 32; ++q) tmem_ld32(s_addr + q * 32, x + q * 32);
                tmem_wait_ld();
                if constexpr (decltype(mask_c)::value) {
                    const int kb = jj * BN;
                    const int klo = a.window > 0 ? qslot - a.window + 1 : 0;
#pragma unroll
                    for (int e = 0; e < BN; ++e) x[e] = (kb + e > qslot || kb + e < klo) ? -INFINITY : x[e];
                }
                float m8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = fmax3(x[q], x[8 + q], x[16 + q]);
#pragma unroll
                for (int e = 24; e + 16 <= BN; e += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q) m8[q] = fmax3(m8[q], x[e + q], x[e + 8 + q]);
                m8[0] = fmax3(m8[0], x[120], x[121]);
                m8[1] = fmax3(m8[1], x[122], x[123]);
                m8[2] = fmax3(m8[2], x[124], x[125]);
                m8[3] = fmax3(m8[3], x[126], x[127]);
                const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                const float m_tile = mx * sl2;
                const bool grow = m_tile > m_run + RESCALE_LOG2 || c == 0;
                const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
                const bool rescale = grow && c > 0 && m_run > -INFINITY;
                if (__any_sync(0xffffffffu, rescale)) {
                    const float corr = rescale ? fast_exp2(m_run - m_new) : 1.0f;
                    l_run *= corr;
#pragma unroll 1
                    for (int q = 0; q < D / 32; ++q) {
                        float o[32];
                        tmem_ld32(o_addr + q * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= corr;
                        tmem_st32(o_addr + q * 32, o);
                    }
                    tmem_wait_st();
                }
                m_run = m_new;
                const float mu = m_run == -INFINITY ? 0.f : m_run;
                float2 l4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) l4[q] = make_float2(0.f, 0.f);
                const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
#pragma unroll
                for (int q = 0; q < BN / 32; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c2 = q * 32 + 2 * e;
                        const float2 arg = __ffma2_rn(make_float2(x[c2], x[c2 + 1]), sl2v, negmu);
                        const float p0 = fast_exp2(arg.x);
                        const float p1 = fast_exp2(arg.y);
                        l4[e & 3] = __fadd2_rn(l4[e & 3], make_float2(p0, p1));
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st16u(s_addr + q * 16, pk);
                }
                l4[0] = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
                l_run += l4[0].x + l4[0].y;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(p_leader);
            };
            if (masked)
                tile(std::true_type{});
            else
                tile(std::false_type{});
        }
        if (ok && c > 0) {
            if (!warp_wait_cluster(smem_u32(&bars->o_done), 0, a.err)) {
                ok = false;
            } else {
                tc_fence_after();
                const float inv = 1.0f / l_run;
                float4* stage = reinterpret_cast<float4*>(smem + OFF_Q) + (warp - 4) * 256;
                const int row0 = qt * BM + sub * 32;
                float* obase = a.out + (((int64_t)b * a.Hq + h) * a.S) * D;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    float o[32];
                    tmem_ld32(o_addr + q * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        stage[lane * 8 + (e ^ (lane & 7))] =
                            make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int rr = 4 * k + (lane >> 3), cc = lane & 7;
                        const float4 val = stage[rr * 8 + (cc ^ (rr & 7))];
                        if (row0 + rr < rows_b)
                            *reinterpret_cast<float4*>(obase + (int64_t)(row0 + rr) * D + q * 32 + cc * 4) = val;
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok) fail_wait(bars, a.err);
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves (or frees tensor memory) while the pair may still use it
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_suffix_tc2(const SuffixLaunch2& a, int items, cudaStream_t s) {
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, suffix_tc2_kernel);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(suffix_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (e != cudaSuccess) return e;
    if (items <= 0) return cudaSuccess;
    suffix_tc2_kernel<<<2 * items, THREADS, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
