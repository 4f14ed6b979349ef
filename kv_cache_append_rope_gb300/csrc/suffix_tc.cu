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
// its key tiles start later and the first ones are masked from below too.
// A long suffix is a dense Q K^T / P V contraction, which is why this kernel
// uses tcgen05 tiles.
//
// One CTA per work item (sequence b, query head h, pair of 128-row query tiles
// A = 2p and B = 2p + 1).  Both query tiles use every key/value tile the CTA
// loads, which halves the key/value bytes each SM takes in per flop (with one
// query tile per CTA the kernel was bound by that feed).  Items are grouped by
// (b, h) -- the tile pairs of one head launch together and walk its K/V tiles
// in step, so each tile comes from DRAM once and from L2 for the rest -- and
// the groups are ordered by total work, longest first.  Query row i (slot
// cut + i) attends key slots 0 .. cut + i; key tiles are 128 slots, the
// diagonal ones masked element-wise.
//
// Warp roles (SPLIT = 1: 384 threads, three warpgroups):
//   warp 0    TMA producers (128-byte swizzle, no multicast): lane 0 both Q
//             tiles once and K tiles into a 2-stage ring, lane 1 V tiles into
//             a 2-stage ring.
//   warp 1    TMEM allocator (512 columns) and, on one elected thread, the MMA
//             issuer.  Per key tile j: O_A += P_A V_j, then S_A = Q_A K_{j+1}^T,
//             then O_B += P_B V_j, then S_B = Q_B K_{j+1}^T -- so that while one
//             query tile's softmax runs, the tensor pipe works for the other
//             (S = QK^T in the SS form, PV in the TS form with P read from tensor
//             memory); completions are signalled with tcgen05.commit on mbarriers.
// Tensor memory: S_A, S_B (128 columns each), O_A, O_B (128 each); P_X, packed
//             bf16, overwrites the first 64 columns of S_X once the softmax has
//             read S_X, and the next S_X = Q_X K^T is issued after the PV that
//             reads P_X (the MMAs of one thread execute in order).
//   warps 2-3 idle (they complete warpgroup 0, whose registers go to the softmax).
//   warps 4-7 softmax of tile A, warps 8-11 of tile B: one thread per query row
//             (= TMEM lane of its sub-partition) owning the whole 128-column row
//             -- no exchange between warps: tcgen05.ld of S, causal (and
//             window) mask, running max in log2 units, O rescaled through TMEM
//             only when the max grows by more than 2^8 (the final division by
//             the running sum makes the stale max exact), P written with
//             tcgen05.st, then the normalised O row stored to global memory.
// The SPLIT = 2 form (640 threads) gives each query tile two softmax warpgroups:
// warps 4-7 and 8-11 take the two 64-key halves of tile A's rows, warps 12-15 and
// 16-19 those of tile B.  The two warps of one TMEM lane quarter exchange their
// halves' row maxima (and their wait verdicts) through shared memory at a 64-thread
// named barrier per key tile and add their partial row sums at the end; part 1 writes
// its P columns (part 0's S columns) only after that barrier.
// Every mbarrier wait is bounded (DEV_ERR_WAIT_TIMEOUT); the MMA thread waits
// for its own last commit and the TMA thread for its own copies before the
// allocator warp frees the tensor memory.
#include <cuda.h>

#include <type_traits>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int QT = 2;                      // query tiles per CTA sharing each key/value tile
constexpr int HALF = BM * 128;             // 128 rows x 64 bf16 (one TMA box)
constexpr int TILE = 2 * HALF;             // 128 rows x 128 bf16
constexpr int KST = 2, VST = 2;            // K and V ring stages
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QT * TILE;
constexpr int OFF_V = OFF_K + KST * TILE;
constexpr int OFF_BAR = OFF_V + VST * TILE;
// split rows: the partners' row maxima (two buffers), wait verdicts (two buffers), row sums
constexpr int OFF_XCH = OFF_BAR + 4096;
constexpr int XCH_MAX = 0, XCH_FLAG = QT * 2 * 2 * 128 * 4, XCH_SUM = XCH_FLAG + QT * 2 * 4 * 2 * 4;
constexpr int XCH_BYTES = XCH_SUM + QT * 2 * 128 * 4;
// SPLIT softmax threads share one query row, each owning BN / SPLIT of its key columns
// (and D / SPLIT of its output columns).  SPLIT = 1: one thread per row, the whole
// 128-column row of S in its registers.  SPLIT = 2: two warpgroups per query tile halve
// the work on the softmax's critical path per key tile; the partners exchange their
// halves' row maxima through shared memory once per tile.
// Registers: the warps per SM sub-partition cap a thread at kLaunchRegs at launch;
// warpgroup 0 then gives registers back to the softmax warpgroups.  The split must add up
// to the launch allocation exactly (checked on the host against the built kernel's
// register count before the first launch).
template <int SPLIT> struct TileCfg;
template <> struct TileCfg<1> {
    static constexpr int kLaunchRegs = 168, kRegsLow = 120, kRegsHigh = 192;
};
template <> struct TileCfg<2> {
    static constexpr int kLaunchRegs = 96, kRegsLow = 64, kRegsHigh = 104;
};
template <int SPLIT> constexpr int kSoftmaxWarps = 4 * QT * SPLIT;   // one per TMEM sub-partition, tile, part
template <int SPLIT> constexpr int kThreads = (4 + kSoftmaxWarps<SPLIT>) * 32;  // + producer, MMA, 2 idle
template <int SPLIT> constexpr int kSmemBytes = OFF_XCH + (SPLIT > 1 ? XCH_BYTES : 0) + 1024;
static_assert(128 * TileCfg<1>::kRegsLow + 2 * 128 * TileCfg<1>::kRegsHigh == kThreads<1> * TileCfg<1>::kLaunchRegs,
              "register split");
static_assert(128 * TileCfg<2>::kRegsLow + 4 * 128 * TileCfg<2>::kRegsHigh == kThreads<2> * TileCfg<2>::kLaunchRegs,
              "register split");
// the epilogue stages 4 KB per softmax warp in the query tiles' shared memory
static_assert(kSoftmaxWarps<2> * 4096 <= QT * TILE, "epilogue staging");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256; // S_X at 128 X, O_X at 256 + 128 X
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int kTileCache = 256;            // paged: key tiles whose row coordinates are staged in shared memory

struct Bars {
    uint64_t q_full;
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[QT], p_full[QT];
    uint64_t o_done;
    uint32_t tmem_base;
    int err;
    int2 ty[kTileCache];       // paged: TMA row coordinates of the two halves of this item's key tiles
};
static_assert(sizeof(Bars) <= 4096, "barrier block");

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

// Key tiles [lo, hi) that query tile qt of a sequence reads (empty past its rows).
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

template <int SPLIT>
__global__ void __launch_bounds__(kThreads<SPLIT>, 1) suffix_tc_kernel(const __grid_constant__ SuffixLaunch a) {
    using Cfg = TileCfg<SPLIT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int4 w = a.work[blockIdx.x];
    const int b = w.x, h = w.y, qp = w.z;
    const int g = h / (a.Hq / a.Hkv);
    const int cut = a.slot0[b];
    const int rows_b = a.seqlen[b];
    // debug builds: the item's query and key slots lie inside the sequence (checked by
    // every thread alike, before any barrier or tensor-memory allocation)
    if (!debug_check(cut >= 0 && rows_b >= 0 && cut + rows_b <= a.C, threadIdx.x == 0 ? a.err : nullptr)) return;
    int jlo[QT], jhi[QT];
#pragma unroll
    for (int X = 0; X < QT; ++X) tile_range(QT * qp + X, cut, rows_b, a.window, jlo[X], jhi[X]);
    // the item walks key tiles j_first .. j_first + n - 1 (tile A is never empty; B may be)
    const int j_first = jlo[0];
    const int n = max(jhi[0], jhi[1]) - j_first;

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
        for (int X = 0; X < QT; ++X) {
            mbar_init(smem_u32(&bars->s_full[X]), 1);
            mbar_init(smem_u32(&bars->p_full[X]), 4 * SPLIT);
        }
        mbar_init(smem_u32(&bars->o_done), 1);
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
            bars->ty[e] = make_int2(paged_row(a.kv, b, g, (j_first + e) * BN),
                                    paged_row(a.kv, b, g, (j_first + e) * BN + 64));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (warp < 4) {
    setmaxnreg_dec<Cfg::kRegsLow>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // lane 0 streams both Q tiles and the K ring, lane 1 the V ring, so that the
        // K look-ahead never waits behind a V stage that is still being read.
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
                qb = smem_u32(&bars->q_full);
                mbar_arrive_expect_tx(qb, QT * TILE);
#pragma unroll
                for (int X = 0; X < QT; ++X) {
                    // rows past the chunk belong to the next head or lie outside the map
                    // (filled with zeros); their results are never stored
                    const int qrow = (b * a.Hq + h) * a.S + (QT * qp + X) * BM;
                    tma_load_2d(smem_u32(smem + OFF_Q + X * TILE), &a.tmQ, 0, qrow, qb);
                    tma_load_2d(smem_u32(smem + OFF_Q + X * TILE + HALF), &a.tmQ, 64, qrow, qb);
                }
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
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, kvrow + (j_first + j) * BN, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, kvrow + (j_first + j) * BN, fb);
                } else {
                    // paged: the two 64-row halves of the tile, each inside one block
                    // (64-row box map; same 128-byte-swizzled layout as one 128-row box)
                    const int2 yy = j < kTileCache ? bars->ty[j]
                                                   : make_int2(paged_row(a.kv, b, g, (j_first + j) * BN),
                                                               paged_row(a.kv, b, g, (j_first + j) * BN + 64));
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, yy.x, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + 64 * 128), map, 0, yy.y, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, yy.x, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF + 64 * 128), map, 64, yy.y, fb);
                }
                issued = j + 1;
            }
            // Our own copies must have landed before the CTA's shared memory is released
            // (bounded in time only: an error raised elsewhere must not cut this short).
            if (is_k) mbar_wait_bounded(qb, 0);
            for (int t = issued - NS < 0 ? 0 : issued - NS; t < issued; ++t)
                mbar_wait_bounded(smem_u32(&full[t % NS]), (t / NS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
            bool ok = mbar_wait_bounded(smem_u32(&bars->q_full), 0, a.err);
            if (!ok) fail_wait(bars, a.err);
            tc_fence_after();
            auto active = [&](int X, int jj) { return jj >= jlo[X] && jj < jhi[X]; };
            // S_X = Q_X K^T from K stage ks
            // Descriptors are built once: the start address sits in the low 14 bits (in
            // 16-byte units, and every shared address here is below 256 KB), so the
            // descriptor of base + off is the base's descriptor + off / 16.
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
            int pv_count[QT] = {0, 0};
            if (ok) {
                if (!mbar_wait_bounded(smem_u32(&bars->k_full[0]), 0, a.err)) ok = false;
                tc_fence_after();
                for (int X = 0; ok && X < QT; ++X)
                    if (active(X, j_first)) issue_qk(X, 0);
                if (ok) tc_commit(smem_u32(&bars->k_empty[0]));
            }
            for (int j = 0; ok && j < n; ++j) {
                const int jj = j_first + j, vs = j % VST;
                const bool next = j + 1 < n;
                const int ks1 = (j + 1) % KST;
                if (!mbar_wait_bounded(smem_u32(&bars->v_full[vs]), (j / VST) & 1, a.err) ||
                    (next && !mbar_wait_bounded(smem_u32(&bars->k_full[ks1]), ((j + 1) / KST) & 1, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t vd = dv + (uint64_t)((vs * TILE) >> 4);
                for (int X = 0; ok && X < QT; ++X) {
                    if (active(X, jj)) {
                        if (!mbar_wait_bounded(smem_u32(&bars->p_full[X]), pv_count[X] & 1, a.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            // A = P_X from tensor memory (16 keys = 8 columns per step),
                            // B = V (rows = keys, contiguous head dims: MN-major)
                            tc_mma_ts(tmem + COL_O + X * 128, tmem + COL_S + X * 128 + kk * 8,
                                      vd + (uint64_t)(kk * 16 * 128 >> 4), idesc_pv,
                                      (pv_count[X] > 0 || kk > 0));
                        }
                        pv_count[X] += 1;
                    }
                    // the next S_X overwrites P_X: issued after the PV that reads it
                    if (next && active(X, jj + 1)) issue_qk(X, ks1);
                }
                if (!ok) break;
                tc_commit(smem_u32(&bars->v_empty[vs]));
                if (next) tc_commit(smem_u32(&bars->k_empty[ks1]));
            }
            if (!ok) fail_wait(bars, a.err);
            // every MMA issued by this thread completes before O is read and the tensor memory freed
            tc_commit(smem_u32(&bars->o_done));
            mbar_wait_bounded(smem_u32(&bars->o_done), 0);  // no abort: the MMAs always finish
        }
    }
    } else {
        setmaxnreg_inc<Cfg::kRegsHigh>();
        // ------------------------------------------------------------ softmax warps
        // Query tile X has 4 * SPLIT warps; warp w reads TMEM lanes 32 * (w % 4) .. + 31, one
        // query row per thread, and part `half` of the row's key (and output) columns.
        constexpr int CW = BN / SPLIT;               // key columns per thread
        constexpr int OW = D / SPLIT;                // output columns per thread
        const int wi = warp - 4;
        const int X = wi / (4 * SPLIT);
        const int half = (wi >> 2) % SPLIT;
        const int sub = warp & 3;
        const int row = sub * 32 + lane;             // query row inside the tile = TMEM lane
        const int qt = QT * qp + X;
        const int i = qt * BM + row;
        const int qslot = cut + i;
        const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
        const uint32_t s_addr = lane_addr + COL_S + X * 128;
        const uint32_t sx_addr = s_addr + half * CW;         // this thread's columns of S
        const uint32_t p_addr = s_addr + half * (CW / 2);    // its packed bf16 columns of P
        const uint32_t o_addr = lane_addr + COL_O + X * 128 + half * OW;
        const float sl2 = a.scale_log2;
        const int tile_slot0 = cut + qt * BM;        // slot of the tile's first row
        auto kbase_of = [](int jj) { return jj * BN; };
        // SPLIT = 2: per (query tile, part) double-buffered row maxima, per warp wait verdicts
        float* xm = reinterpret_cast<float*>(smem + OFF_XCH + XCH_MAX);
        int* xf = reinterpret_cast<int*>(smem + OFF_XCH + XCH_FLAG);
        float* xs = reinterpret_cast<float*>(smem + OFF_XCH + XCH_SUM);
        const int pair_bar = 1 + X * 4 + sub;        // named barrier of the two partner warps
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int c = 0;
        for (int jj = jlo[X]; jj < jhi[X]; ++jj, ++c) {
            const bool okw = warp_wait(smem_u32(&bars->s_full[X]), c & 1, a.err);
            // SPLIT = 1 leaves at once; partners first agree on the verdict (below), so that
            // both leave at the same tile and neither waits at the named barrier alone
            if (SPLIT == 1 && !okw) {
                ok = false;
                break;
            }
            tc_fence_after();
            // causal mask (keys after the row's slot) on diagonal tiles; with a window also
            // the keys before slot - window + 1 on the first tiles.  The tile is processed
            // by one of two copies of the code, with and without the mask, so that the
            // unmasked tiles (nearly all) carry no masking instructions.
            const bool masked =
                kbase_of(jj) + BN - 1 > tile_slot0 || (a.window > 0 && kbase_of(jj) < tile_slot0 + BM - a.window);
            auto tile = [&](auto mask_c) -> bool {
                // The thread's columns of the row are read with one wait, then reduced to
                // their maximum, then turned into exponentials in place.
                float x[CW];
                if (SPLIT == 1 || okw) {
                    if constexpr (CW == 128)
                        tmem_ld128(sx_addr, x);
                    else
                        tmem_ld64(sx_addr, x);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < CW; ++e) x[e] = 0.f;   // not used: the partners leave below
                }
                if constexpr (decltype(mask_c)::value) {
                    const int kb = jj * BN + half * CW;
                    const int klo = a.window > 0 ? qslot - a.window + 1 : 0;
#pragma unroll
                    for (int e = 0; e < CW; ++e) x[e] = (kb + e > qslot || kb + e < klo) ? -INFINITY : x[e];
                }
                // maximum (8 independent chains of 3-input maxima)
                float m8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = fmax3(x[q], x[8 + q], x[16 + q]);
#pragma unroll
                for (int e = 24; e + 16 <= CW; e += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q) m8[q] = fmax3(m8[q], x[e + q], x[e + 8 + q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) m8[q] = fmax3(m8[q], x[CW - 8 + 2 * q], x[CW - 7 + 2 * q]);
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                if constexpr (SPLIT == 2) {
                    // the partner's maximum of the other half of the row (both partners have
                    // read their columns of S before either overwrites any with P)
                    const int buf = c & 1;
                    xm[((X * 2 + half) * 2 + buf) * 128 + row] = mx;
                    if (lane == 0) xf[((X * 2 + half) * 4 + sub) * 2 + buf] = okw;
                    tc_fence_before();
                    named_bar_sync(pair_bar, 64);
                    tc_fence_after();
                    const float mp = xm[((X * 2 + (half ^ 1)) * 2 + buf) * 128 + row];
                    const int okp = xf[((X * 2 + (half ^ 1)) * 4 + sub) * 2 + buf];
                    if (!okw || !okp) return false;
                    mx = fmaxf(mx, mp);
                }
                const float m_tile = mx * sl2;
                const bool grow = m_tile > m_run + RESCALE_LOG2 || c == 0;
                const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
                // O holds the sum over earlier tiles; the PV that last wrote it completed before
                // this S (its QK^T was issued after that PV).  tcgen05.ld/st are warp-collective
                // (.sync.aligned), so the whole warp rescales when any of its rows must, the
                // other rows by 1.
                const bool rescale = grow && c > 0 && m_run > -INFINITY;
                const float m_old = m_run;
                auto rescale_o = [&] {
                    if (__any_sync(0xffffffffu, rescale)) {
                        const float corr = rescale ? fast_exp2(m_old - m_new) : 1.0f;
                        l_run *= corr;
#pragma unroll 1
                        for (int q = 0; q < OW / 32; ++q) {
                            float o[32];
                            tmem_ld32(o_addr + q * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= corr;
                            tmem_st32(o_addr + q * 32, o);
                        }
                        tmem_wait_st();
                    }
                };
                // SPLIT = 2 rescales after the exponentials, when the row's S values no longer
                // occupy registers (only the arrive on p_full must follow it)
                if constexpr (SPLIT == 1) rescale_o();
                m_run = m_new;
                const float mu = m_run == -INFINITY ? 0.f : m_run;
                // P = exp2(x * scale - max), packed to bf16 pairs into the thread's P columns
                // (its S columns are in registers already; SPLIT = 2: part 1's P columns are
                // part 0's S columns, read before the named barrier); packed float32x2
                // arithmetic, since the softmax warps issue most of the kernel's instructions.
                float2 l4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) l4[q] = make_float2(0.f, 0.f);
                const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
                uint32_t pk[CW / 2];
#pragma unroll
                for (int e = 0; e < CW / 2; ++e) {
                    const int c2 = 2 * e;
                    const float2 arg = __ffma2_rn(make_float2(x[c2], x[c2 + 1]), sl2v, negmu);
                    const float p0 = fast_exp2(arg.x);
                    const float p1 = fast_exp2(arg.y);
                    l4[e & 3] = __fadd2_rn(l4[e & 3], make_float2(p0, p1));
                    pk[e] = pack_bf16(p0, p1);
                }
                if constexpr (CW == 128)
                    tmem_st64u(p_addr, pk);
                else
                    tmem_st32u(p_addr, pk);
                l4[0] = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
                if constexpr (SPLIT == 2) rescale_o();
                l_run += l4[0].x + l4[0].y;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[X]));
                return true;
            };
            const bool good = masked ? tile(std::true_type{}) : tile(std::false_type{});
            if (!good) {
                ok = false;
                break;
            }
        }
        if constexpr (SPLIT == 2) {
            // the row sum is the partners' two partial sums (taken before any further wait, so
            // that both partners reach this barrier: they left the loop at the same tile)
            if (ok && c > 0) {
                xs[(X * 2 + half) * 128 + row] = l_run;
                named_bar_sync(pair_bar, 64);
                l_run += xs[(X * 2 + (half ^ 1)) * 128 + row];
            }
        }
        if (ok && c > 0) {
            if (!warp_wait(smem_u32(&bars->o_done), 0, a.err)) {
                ok = false;
            } else {
                tc_fence_after();
                const float inv = 1.0f / l_run;
                // O rows leave through shared memory (the Q tiles, unused once every MMA has
                // completed): each thread writes 32 columns of its row, the warp then stores
                // 4 rows x 128 bytes per instruction -- whole lines instead of 32 scattered
                // 16-byte pieces.  16-byte slots are XOR-swizzled by row (mod 8), so both
                // sides take the minimum of 4 shared-memory wavefronts per instruction.
                float4* stage = reinterpret_cast<float4*>(smem + OFF_Q) + wi * 256;
                const int row0 = qt * BM + sub * 32;             // query row of lane 0
                float* obase = a.out + (((int64_t)b * a.Hq + h) * a.S) * D + half * OW;
#pragma unroll
                for (int q = 0; q < OW / 32; ++q) {
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
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int suffix_tc_grid(int sms) { return sms; }

namespace {

template <int SPLIT> cudaError_t launch_tile(const SuffixLaunch& a, int grid, cudaStream_t s) {
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        // the register split assumes the launch allocation it was computed for
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, suffix_tc_kernel<SPLIT>);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != TileCfg<SPLIT>::kLaunchRegs) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(suffix_tc_kernel<SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes<SPLIT>);
    });
    if (e != cudaSuccess) return e;
    if (grid <= 0) return cudaSuccess;
    suffix_tc_kernel<SPLIT><<<grid, kThreads<SPLIT>, kSmemBytes<SPLIT>, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_suffix_tc(const SuffixLaunch& a, int grid, cudaStream_t s, int split) {
    return split == 2 ? launch_tile<2>(a, grid, s) : launch_tile<1>(a, grid, s);
}

}  // namespace kvc
