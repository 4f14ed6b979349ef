// Suffix-chunk causal attention on the 5th-generation tensor cores, persistent form
// (bf16, d_h = 128, contiguous storage).
//
// Same computation, work items and per-item pipeline as the one-CTA-per-item tile
// kernel (suffix_tc.cu): [LCP5] "LLM 机制实验（五）：改了历史，能否只重算变化的后缀？",
// section "先看一次历史编辑" -- after truncation to `cut`, suffix row i (slot cut + i)
// attends slots 0 .. cut + i (or its `window` most recent ones, [LCP5]
// "为什么滑窗部分命中必须回退"); [Ch37] listing "Evaluate one newest query across the
// retained rows plus the candidate key/value row before committing the append" fixes
// the 1/sqrt(d_h) scale and the max-subtracted softmax.
//
// One CTA per SM takes work items from the list in order through a global counter (the
// list is grouped by (sequence, head) and longest first, so the CTAs working at one time
// share each head's K/V tiles through L2, and the longest items go first).  The K
// producer lane fetches each next item index and passes it to the other roles through a
// 4-entry ring in shared memory (item_full / item_empty).  Tensor memory is allocated
// once, the barriers keep counting across items, and the item boundary overlaps:
//   * the producer loads the next item's query tiles as soon as the MMAs that read the
//     current ones are done (q_empty, committed once the item's last QK^T is issued) and
//     streams its K/V tiles into the same rings, whose stage counters run on;
//   * the MMA thread issues the next item's first S_A, S_B = Q K_0^T while the softmax
//     warps still write the current item's O out; only its first P V into O_X waits
//     for that (o_free[X], which the softmax warps of tile X arrive on after reading O_X);
//   * the epilogue stages O through a shared-memory buffer of its own (the query tiles
//     hold the next item by then).
// Every role walks the same item sequence and skips the same (invalid) items, so phase
// parities derived from per-role counters agree; no barrier can run two phases ahead of
// its waiters (each phase of q_full, o_done, o_free, s_full, p_full is consumed before
// the producer of the next one can proceed).  Every wait is bounded (DEV_ERR_WAIT_TIMEOUT)
// and gives up when any CTA flags an error; the TMA lanes wait for their own copies and
// the MMA thread for its last commit before the tensor memory is freed.
#include <cuda.h>

#include <type_traits>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int QT = 2;                      // query tiles per item sharing each key/value tile
constexpr int HALF = BM * 128;             // 128 rows x 64 bf16 (one TMA box)
constexpr int TILE = 2 * HALF;             // 128 rows x 128 bf16
constexpr int KST = 2, VST = 2;            // K and V ring stages
constexpr int NSW = 4 * QT;                // softmax warps
constexpr int STG_WARP = 256 * 16;         // epilogue staging per softmax warp: 32 rows x 32 floats
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QT * TILE;
constexpr int OFF_V = OFF_K + KST * TILE;
constexpr int OFF_STG = OFF_V + VST * TILE;
constexpr int OFF_BAR = OFF_STG + NSW * STG_WARP;
constexpr int SMEM_BYTES = OFF_BAR + 1024 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
constexpr int THREADS = (4 + NSW) * 32;
constexpr int kLaunchRegs = 168, kRegsLow = 120, kRegsHigh = 192;
static_assert(128 * kRegsLow + 2 * 128 * kRegsHigh == THREADS * kLaunchRegs, "register split");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256; // S_X at 128 X, O_X at 256 + 128 X
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int IRING = 4;                   // item-index ring entries
constexpr int ITEM_READERS = 2 + NSW;      // V lane, MMA thread, softmax warps

struct Bars {
    uint64_t item_full[IRING], item_empty[IRING];
    int item_idx[IRING];                   // work index, or -1 when the list is done
    uint64_t q_full, q_empty;
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[QT], p_full[QT];
    uint64_t o_done, o_free[QT];
    uint32_t tmem_base;
    int err;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

__device__ __forceinline__ void fail_wait(Bars* bars, uint32_t* err) {
    *(volatile int*)&bars->err = 1;
    atomicOr(err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const uint32_t* abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
}

// One work item: (sequence b, query head h, pair of query tiles 2 qp and 2 qp + 1).
struct Item {
    int b, h, g, qp, cut, rows;
    int jlo[QT], jhi[QT];
    int j_first, n;                        // key tiles j_first .. j_first + n - 1
    bool ok;
};

__device__ __forceinline__ Item item_of(const SuffixLaunch& a, int idx) {
    Item I;
    const int4 w = a.work[idx];
    I.b = w.x;
    I.h = w.y;
    I.qp = w.z;
    I.g = I.h / (a.Hq / a.Hkv);
    I.cut = a.slot0[I.b];
    I.rows = a.seqlen[I.b];
    // debug builds: the item's query and key slots lie inside the sequence (every role
    // evaluates the same check, so an invalid item is skipped by all of them)
    I.ok = debug_check(I.cut >= 0 && I.rows >= 0 && I.cut + I.rows <= a.C, nullptr);
#pragma unroll
    for (int X = 0; X < QT; ++X) {
        const int qt = QT * I.qp + X, r0 = qt * BM;
        if (r0 >= I.rows) {
            I.jlo[X] = I.jhi[X] = 0;
        } else {
            const int q_end = min(r0 + BM, I.rows);
            I.jlo[X] = a.window > 0 ? max(0, I.cut + r0 - a.window + 1) / BN : 0;
            I.jhi[X] = (I.cut + q_end - 1) / BN + 1;
        }
    }
    I.j_first = I.jlo[0];
    I.n = max(I.jhi[0], I.jhi[1]) - I.j_first;
    if (I.n <= 0) I.ok = false;
    return I;
}

__global__ void __launch_bounds__(THREADS, 1) suffix_tcp_kernel(const __grid_constant__ SuffixLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int r = 0; r < IRING; ++r) {
            mbar_init(smem_u32(&bars->item_full[r]), 1);
            mbar_init(smem_u32(&bars->item_empty[r]), ITEM_READERS);
        }
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_empty), 1);
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
            mbar_init(smem_u32(&bars->p_full[X]), 4);
            mbar_init(smem_u32(&bars->o_free[X]), 4);
        }
        mbar_init(smem_u32(&bars->o_done), 1);
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
    auto failed = [&]() { return *(volatile int*)&bars->err != 0 || *(volatile uint32_t*)a.err != 0; };
    // The k-th item index of this CTA for the roles other than the fetcher: waits for its
    // ring entry, reads it and releases the entry (one arrival per reading thread or
    // warp).  -2 when the wait gave up.
    auto read_item = [&](int k, bool whole_warp) {
        const int r = k % IRING;
        const uint32_t full = smem_u32(&bars->item_full[r]);
        const bool got = whole_warp ? warp_wait(full, (k / IRING) & 1, a.err)
                                    : mbar_wait_bounded(full, (k / IRING) & 1, a.err);
        if (!got) return -2;
        const int idx = *(volatile int*)&bars->item_idx[r];
        if (whole_warp) __syncwarp();
        if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars->item_empty[r]));
        return idx;
    };

    if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producers
        // lane 0: each item's two query tiles, then its K tiles; lane 1: its V tiles.
        if (lane < 2) {
            const bool is_k = lane == 0;
            const int NS = is_k ? KST : VST;
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
            const CUtensorMap* map = is_k ? &a.tmK : &a.tmV;
            uint8_t* ring = smem + (is_k ? OFF_K : OFF_V);
            prefetch_tmap(map);
            if (is_k) prefetch_tmap(&a.tmQ);
            const uint32_t qb = smem_u32(&bars->q_full);
            int qloads = 0, gt = 0;                      // query-tile loads and K/V tiles issued
            bool bad = false;
            for (int k = 0; !bad && !failed(); ++k) {
                int it;
                if (is_k) {
                    // fetch the next item and publish it in the ring
                    const int r = k % IRING;
                    if (k >= IRING && !mbar_wait_bounded(smem_u32(&bars->item_empty[r]), ((k / IRING) - 1) & 1, a.err)) {
                        bad = true;
                        break;
                    }
                    it = atomicAdd(a.counter, 1);
                    if (it >= a.n_work) it = -1;
                    bars->item_idx[r] = it;
                    mbar_arrive(smem_u32(&bars->item_full[r]));
                } else {
                    it = read_item(k, false);
                    if (it == -2) {
                        bad = true;
                        break;
                    }
                }
                if (it < 0) break;
                const Item I = item_of(a, it);
                if (!I.ok) {
                    // debug builds: an item outside its sequence is recorded and skipped by all
                    if (is_k) atomicOr(a.err, (uint32_t)DEV_ERR_BOUNDS);
                    continue;
                }
                if (is_k) {
                    // the query tiles of the previous item are free once its QK^T completed
                    if (qloads > 0 && !mbar_wait_bounded(smem_u32(&bars->q_empty), (qloads - 1) & 1, a.err)) {
                        bad = true;
                        break;
                    }
                    mbar_arrive_expect_tx(qb, QT * TILE);
#pragma unroll
                    for (int X = 0; X < QT; ++X) {
                        // rows past the chunk belong to the next head or lie outside the map
                        // (zero filled); their results are never stored
                        const int qrow = (I.b * a.Hq + I.h) * a.S + (QT * I.qp + X) * BM;
                        tma_load_2d(smem_u32(smem + OFF_Q + X * TILE), &a.tmQ, 0, qrow, qb);
                        tma_load_2d(smem_u32(smem + OFF_Q + X * TILE + HALF), &a.tmQ, 64, qrow, qb);
                    }
                    ++qloads;
                }
                const int kvrow = (I.b * a.Hkv + I.g) * a.C;
                for (int j = 0; j < I.n; ++j, ++gt) {
                    const int s = gt % NS;
                    if (gt >= NS && !mbar_wait_bounded(smem_u32(&empty[s]), ((gt / NS) - 1) & 1, a.err)) {
                        bad = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, TILE);
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, kvrow + (I.j_first + j) * BN, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, kvrow + (I.j_first + j) * BN, fb);
                }
            }
            if (bad) fail_wait(bars, a.err);
            // Our own copies must have landed before the CTA's shared memory is released
            // (bounded in time only: an error raised elsewhere must not cut this short).
            if (qloads > 0) mbar_wait_bounded(qb, (qloads - 1) & 1);
            for (int t = gt - NS < 0 ? 0 : gt - NS; t < gt; ++t)
                mbar_wait_bounded(smem_u32(&full[t % NS]), (t / NS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
            // Descriptors are built once: the start address sits in the low 14 bits (in
            // 16-byte units, every shared address here is below 256 KB), so the descriptor
            // of base + off is the base's descriptor + off / 16.
            const uint64_t dq = smem_desc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
            const uint64_t dk = smem_desc_sw128(smem_u32(smem + OFF_K), 16, 1024);
            const uint64_t dv = smem_desc_sw128(smem_u32(smem + OFF_V), HALF, 1024);
            auto issue_qk = [&](int X, int ks) {
                const uint64_t qd = dq + (uint64_t)((X * TILE) >> 4);
                const uint64_t kd = dk + (uint64_t)((ks * TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * HALF + (kk & 3) * 32) >> 4;
                    tc_mma_ss(tmem + COL_S + X * 128, qd + off, kd + off, idesc_qk, kk > 0);
                }
                tc_commit(smem_u32(&bars->s_full[X]));
            };
            int items = 0, gt = 0;                    // items and key tiles consumed so far
            int pv_all[QT] = {0, 0};                  // P V products issued, all items
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int it = read_item(k, false);
                if (it == -2) {
                    ok = false;
                    break;
                }
                if (it < 0) break;
                const Item I = item_of(a, it);
                if (!I.ok) continue;
                auto active = [&](int X, int jj) {
                    return X == 0 ? (jj >= I.jlo[0] && jj < I.jhi[0]) : (jj >= I.jlo[1] && jj < I.jhi[1]);
                };
                if (!mbar_wait_bounded(smem_u32(&bars->q_full), items & 1, a.err) ||
                    !mbar_wait_bounded(smem_u32(&bars->k_full[gt % KST]), (gt / KST) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int X = 0; X < QT; ++X)
                    if (active(X, I.j_first)) issue_qk(X, gt % KST);
                tc_commit(smem_u32(&bars->k_empty[gt % KST]));
                int pv_item[QT] = {0, 0};
                for (int j = 0; ok && j < I.n; ++j) {
                    const int jj = I.j_first + j, gj = gt + j, vs = gj % VST;
                    const bool next = j + 1 < I.n;
                    const int ks1 = (gj + 1) % KST;
                    // every QK^T of this item is issued: the query tiles may be reloaded once
                    // they complete
                    if (!next) tc_commit(smem_u32(&bars->q_empty));
                    if (!mbar_wait_bounded(smem_u32(&bars->v_full[vs]), (gj / VST) & 1, a.err) ||
                        (next && !mbar_wait_bounded(smem_u32(&bars->k_full[ks1]), ((gj + 1) / KST) & 1, a.err))) {
                        ok = false;
                        break;
                    }
                    // the first P V of an item overwrites O_X: the previous item's epilogue
                    // must have read both O tiles
                    if (j == 0 && items > 0) {
#pragma unroll
                        for (int X = 0; X < QT; ++X)
                            if (!mbar_wait_bounded(smem_u32(&bars->o_free[X]), (items - 1) & 1, a.err)) ok = false;
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint64_t vd = dv + (uint64_t)((vs * TILE) >> 4);
#pragma unroll
                    for (int X = 0; X < QT; ++X) {
                        if (!ok) break;
                        if (active(X, jj)) {
                            if (!mbar_wait_bounded(smem_u32(&bars->p_full[X]), pv_all[X] & 1, a.err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                tc_mma_ts(tmem + COL_O + X * 128, tmem + COL_S + X * 128 + kk * 8,
                                          vd + (uint64_t)(kk * 16 * 128 >> 4), idesc_pv,
                                          (pv_item[X] > 0 || kk > 0));
                            pv_item[X] += 1;
                            pv_all[X] += 1;
                        }
                        // the next S_X overwrites P_X: issued after the PV that reads it
                        if (next && active(X, jj + 1)) issue_qk(X, ks1);
                    }
                    if (!ok) break;
                    tc_commit(smem_u32(&bars->v_empty[vs]));
                    if (next) tc_commit(smem_u32(&bars->k_empty[ks1]));
                }
                if (!ok) break;
                // every MMA of the item completes before its O is read
                tc_commit(smem_u32(&bars->o_done));
                gt += I.n;
                ++items;
            }
            // every MMA issued by this thread completes before the tensor memory is freed (no
            // abort: the MMAs always finish).  On the normal path that is the last item's
            // o_done phase -- another commit would complete a phase the softmax warps may
            // not have observed yet; after an error, a commit for the unfinished item.
            if (!ok) {
                fail_wait(bars, a.err);
                tc_commit(smem_u32(&bars->o_done));
                mbar_wait_bounded(smem_u32(&bars->o_done), items & 1);
            } else if (items > 0) {
                mbar_wait_bounded(smem_u32(&bars->o_done), (items - 1) & 1);
            }
        }
    }
    } else {
        setmaxnreg_inc<kRegsHigh>();
        // ------------------------------------------------------------ softmax warps
        // Warps 4-7 take query tile A, 8-11 tile B; warp w reads TMEM lanes
        // 32 * (w % 4) .. + 31, one query row per thread.
        const int X = (warp - 4) >> 2;
        const int sub = warp & 3;
        const int row = sub * 32 + lane;             // query row inside the tile = TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
        const uint32_t s_addr = lane_addr + COL_S + X * 128;
        const uint32_t o_addr = lane_addr + COL_O + X * 128;
        const float sl2 = a.scale_log2;
        float4* stage = reinterpret_cast<float4*>(smem + OFF_STG) + (warp - 4) * 256;
        int items = 0, cs = 0;                       // items done, S_X tiles consumed (all items)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int it = read_item(k, true);
            if (it == -2) {
                ok = false;
                break;
            }
            if (it < 0) break;
            const Item I = item_of(a, it);
            if (!I.ok) continue;
            const int qt = QT * I.qp + X;
            const int jlo = X == 0 ? I.jlo[0] : I.jlo[1], jhi = X == 0 ? I.jhi[0] : I.jhi[1];
            const int qslot = I.cut + qt * BM + row;
            const int tile_slot0 = I.cut + qt * BM;  // slot of the tile's first row
            float m_run = -INFINITY, l_run = 0.f;
            int c = 0;
            for (int jj = jlo; jj < jhi; ++jj, ++c, ++cs) {
                if (!warp_wait(smem_u32(&bars->s_full[X]), cs & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // causal mask (keys after the row's slot) on diagonal tiles; with a window
                // also the keys before slot - window + 1 on the first tiles.  The tile is
                // processed by one of two copies of the code, with and without the mask.
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
                    // row maximum (8 independent chains of 3-input maxima)
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
                    const float mx =
                        fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                    const float m_tile = mx * sl2;
                    const bool grow = m_tile > m_run + RESCALE_LOG2 || c == 0;
                    const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
                    // O holds the sum over this item's earlier tiles; the PV that last wrote
                    // it completed before this S (its QK^T was issued after that PV).
                    // tcgen05.ld/st are warp-collective, so the whole warp rescales when any
                    // of its rows must, the other rows by 1.
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
                    // P = exp2(x * scale - max), packed to bf16 pairs into columns 0 .. 63 of
                    // S_X (all of S is in registers already); packed float32x2 arithmetic
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
                    if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[X]));
                };
                if (masked)
                    tile(std::true_type{});
                else
                    tile(std::false_type{});
            }
            if (!ok) break;
            // every MMA of the item has completed: O_X is final
            if (!warp_wait(smem_u32(&bars->o_done), items & 1, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (c > 0) {
                const float inv = 1.0f / l_run;
                // O rows leave through this warp's staging buffer: each thread writes 32
                // columns of its row, the warp then stores 4 rows x 128 bytes per
                // instruction; 16-byte slots XOR-swizzled by row (mod 8)
                const int row0 = qt * BM + sub * 32;     // query row of lane 0
                float* obase = a.out + (((int64_t)I.b * a.Hq + I.h) * a.S) * D;
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
                        if (row0 + rr < I.rows)
                            *reinterpret_cast<float4*>(obase + (int64_t)(row0 + rr) * D + q * 32 + cc * 4) = val;
                    }
                    __syncwarp();
                }
            }
            // O_X has been read: the next item's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[X]));
            ++items;
        }
        if (!ok) fail_wait(bars, a.err);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_suffix_tcp(const SuffixLaunch& a, int sms, cudaStream_t s) {
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        // the register split assumes the launch allocation it was computed for
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, suffix_tcp_kernel);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(suffix_tcp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (e != cudaSuccess) return e;
    if (a.n_work <= 0 || sms <= 0) return cudaSuccess;
    if (a.kv.table || !a.counter) return cudaErrorInvalidValue;   // contiguous storage only
    e = cudaMemsetAsync(a.counter, 0, sizeof(int), s);                 // the items start at 0
    if (e != cudaSuccess) return e;
    suffix_tcp_kernel<<<a.n_work < sms ? a.n_work : sms, THREADS, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
