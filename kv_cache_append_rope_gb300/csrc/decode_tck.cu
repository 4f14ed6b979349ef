// Tensor-core decode, stream-K form: one wave of CTAs, each over an equal run of key tiles
// of the concatenated lanes (bf16, d_h = 128, 16 < G = H_q / H_kv <= 32, contiguous
// storage, fused step with host lengths).
//
// Same computation as the tensor-core decode kernel (decode_tc.cu; [Ch37] "Keep the
// prefix, project only the new row" and the listing "Evaluate one newest query across
// the retained rows plus the candidate key/value row before committing the append":
// every new query scores all retained rows and the candidate row, q.k_j / sqrt(d_h),
// takes a max-subtracted softmax and mixes the values), with the work cut differently.
// The lanes (b, kv head) are laid end to end as runs of 128-key tiles (each lane's tiles
// start at its window start rounded down to 64 rows); CTA c of P takes tiles
// [c T / P, (c + 1) T / P) of the T in all, so every CTA gets the same number of tiles
// and one wave of P = #SMs CTAs finishes together.  A CTA's range cuts into segments,
// one per lane it touches; each segment's (O, max, sum) is a partial of its lane (slot
// c - first CTA of the lane), merged by decode_combine_kernel (a lane inside one CTA is
// normalised and stored directly).  The segment holding a lane's last tile appends the
// new key/value row first; the one holding its first tile commits the length (kv head 0).
//
// Per CTA the roles walk the same segment list (computed from c alone):
//   warp 0   per segment: the new row when the segment ends the lane, then its K and V
//            tiles into 2-stage rings whose counters run on across segments;
//   warp 1   tensor memory (512 columns), and on one thread the MMAs: S into one of two
//            buffers (alternating over all the CTA's tiles), O += P V; the first P V of a
//            segment waits until the previous segment's O was read (o_free);
//   warp 2   zeroes query rows 32 .. 127 once, then per segment, once the previous
//            segment's QK^T completed (q_empty), writes the lane's G rotated query rows;
//   warp 4   softmax (one thread per head row), per segment from a fresh running max and
//            sum; at the segment's end, once its MMAs completed (o_done), the partial or
//            the normalised output, then o_free.
// Every wait is bounded (DEV_ERR_WAIT_TIMEOUT); no barrier runs two phases ahead of its
// waiters (each phase is consumed before the role that completes the next one can go on).
#include <cuda.h>

#include <type_traits>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int D = 128, BN = 128, QROWS = 128;
constexpr int HALF = QROWS * 128;          // 128 rows x 64 bf16 (one TMA box)
constexpr int TILE = 2 * HALF;             // 128 rows x 128 bf16
constexpr int KST = 2, VST = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;
constexpr int OFF_V = OFF_K + KST * TILE;
constexpr int OFF_BAR = OFF_V + VST * TILE;
constexpr int SMEM_BYTES = OFF_BAR + 1024 + 1024;
constexpr int THREADS = 5 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256;   // S buffer u at 128 u, O at 256
constexpr float RESCALE_LOG2 = 8.0f;

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[2], p_full[2];
    uint64_t pv_done, o_done, o_free;
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

__device__ __forceinline__ void store_out(const DecodeLaunch& a, int64_t i, float x) {
    if (a.out_bf16)
        ((__nv_bfloat16*)a.out)[i] = __float2bfloat16_rn(x);
    else
        ((float*)a.out)[i] = x;
}

// One segment: the part of lane l = b H_kv + hkv that CTA c covers.
struct Seg {
    int b, hkv;
    int t, lo;                 // keys lo .. t - 1 attend
    int r0, r1;                // key rows of the segment
    int n;                     // 128-key tiles
    int slot;                  // partial slot of the lane (c - its first CTA)
    bool single, last, first;  // lane in one CTA; segment holds the lane's last / first tile
};

// First tile of CTA c.
__device__ __forceinline__ int tile_begin(const DecodeLaunch& a, int c) {
    return (int)(((int64_t)c * a.streamk_tiles) / a.streamk);
}

// Lane holding tile x: the last lane whose first tile is <= x.
__device__ __forceinline__ int lane_of_tile(const DecodeLaunch& a, int x) {
    const int lanes = a.B * a.Hkv;
    int lo_i = 0, hi_i = lanes;
    while (hi_i - lo_i > 1) {
        const int mid = (lo_i + hi_i) >> 1;
        if (a.item_start[mid] <= x) lo_i = mid;
        else hi_i = mid;
    }
    return lo_i;
}

__device__ __forceinline__ Seg seg_of(const DecodeLaunch& a, int l, int T0, int T1) {
    Seg s;
    s.b = l / a.Hkv;
    s.hkv = l - s.b * a.Hkv;
    s.t = a.old_len[s.b] + 1;
    s.lo = a.window > 0 ? max(0, s.t - a.window) : 0;
    const int base = s.lo & ~63;
    const int l0 = a.item_start[l], l1 = a.item_start[l + 1];
    const int j0 = max(T0, l0) - l0, j1 = min(T1, l1) - l0;
    s.r0 = base + j0 * BN;
    s.r1 = min(s.t, base + j1 * BN);
    s.n = j1 - j0;
    s.slot = (int)blockIdx.x - a.seq_of[l];
    s.single = a.seq_rows[l] == 1;
    s.last = T1 >= l1;
    s.first = T0 <= l0;
    return s;
}

__global__ void __launch_bounds__(THREADS, 1)
decode_tck_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ DecodeLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;
    const int T0 = tile_begin(a, blockIdx.x), T1 = tile_begin(a, blockIdx.x + 1);
    const int l_first = lane_of_tile(a, T0);
    // everything below may read what the previous kernel of the stream wrote
    grid_dependency_wait();
    launch_dependents();
    if (T1 <= T0) return;
    // debug builds: every lane's new-row slot lies inside the cache (checked by every thread
    // alike, before any barrier or tensor-memory allocation)
    if (kDebug) {
        bool ok = true;
        for (int l = l_first; l < a.B * a.Hkv && a.item_start[l] < T1; ++l) {
            const int ol = a.old_len[l / a.Hkv];
            ok = ok && ol >= 0 && ol < a.C;
        }
        if (!debug_check(ok, threadIdx.x == 0 ? a.err : nullptr)) return;
    }
    // the first segment of a lane, for kv head 0, commits its sequence's length
    if (threadIdx.x == 0 && !a.no_commit)
        for (int l = l_first; l < a.B * a.Hkv && a.item_start[l] < T1; ++l) {
            const Seg s = seg_of(a, l, T0, T1);
            if (s.first && s.hkv == 0) {
                a.len_out[s.b] = s.t;
                a.next_out[s.b] = a.pos[s.b] + 1;
            }
        }

    if (threadIdx.x == 0) {
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
        for (int u = 0; u < 2; ++u) {
            mbar_init(smem_u32(&bars->s_full[u]), 1);
            mbar_init(smem_u32(&bars->p_full[u]), 1);
        }
        mbar_init(smem_u32(&bars->pv_done), 1);
        mbar_init(smem_u32(&bars->o_done), 1);
        mbar_init(smem_u32(&bars->o_free), 1);
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
    const int lanes = a.B * a.Hkv;

    if (warp == 0) {
        // ------------------------------------------------------------ new rows, then TMA
        int gt = 0;                                  // tiles issued, all segments
        bool bad = false;
        for (int l = l_first; l < lanes && a.item_start[l] < T1 && !bad; ++l) {
            const Seg sg = seg_of(a, l, T0, T1);
            if (sg.last) {
                // The new row (slot t - 1) is in this segment: rotate and store the key
                // (bit-exact bf16 rounding), store the value and the position, then order
                // these generic-proxy writes before this warp's TMA reads of them.
                const int old_len = sg.t - 1, pos = a.pos[sg.b];
                const int64_t src = ((int64_t)sg.b * a.Hkv + sg.hkv) * D + lane * 4;
                const int64_t dst = (((int64_t)sg.b * a.Hkv + sg.hkv) * a.C + old_len) * D + lane * 4;
                const uint2 kraw = *(const uint2*)(a.k_in + src);
                const uint2 vraw = *(const uint2*)(a.v_in + src);
                const __nv_bfloat16* kin = (const __nv_bfloat16*)&kraw;
                __nv_bfloat16 kout[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float xf = __bfloat162float(kin[2 * e]), yf = __bfloat162float(kin[2 * e + 1]);
                    if (a.rope_f) {
                        const int j = lane * 2 + e;
                        const float2 cs = a.rope_f[(int64_t)pos * (D / 2) + j];
                        kout[2 * e] = rope_bf16_exact(xf, yf, cs.x, cs.y, a.rope, pos, D / 2, j, false);
                        kout[2 * e + 1] = rope_bf16_exact(xf, yf, cs.x, cs.y, a.rope, pos, D / 2, j, true);
                    } else {
                        kout[2 * e] = kin[2 * e];
                        kout[2 * e + 1] = kin[2 * e + 1];
                    }
                }
                *(uint2*)(a.K + dst) = *(const uint2*)kout;
                *(uint2*)(a.V + dst) = vraw;
                if (sg.hkv == 0 && lane == 0) a.positions[(int64_t)sg.b * a.C + old_len] = pos;
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            }
            if (lane < 2 && !a.test_stall) {
                const bool is_k = lane == 0;
                uint64_t* full = is_k ? bars->k_full : bars->v_full;
                uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
                const CUtensorMap* map = is_k ? &tmK : &tmV;
                uint8_t* ring = smem + (is_k ? OFF_K : OFF_V);
                const int NS = is_k ? KST : VST;
                if (l == l_first) prefetch_tmap(map);
                const int row0 = ((sg.b * a.Hkv + sg.hkv) * a.C) + sg.r0;    // contiguous storage
                for (int j = 0; j < sg.n && !*(volatile int*)&bars->err; ++j, ++gt) {
                    const int s = gt % NS;
                    if (gt >= NS && !mbar_wait_bounded(smem_u32(&empty[s]), ((gt / NS) - 1) & 1, a.err)) {
                        bad = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, TILE);
                    // rows past the segment belong to the next lane or lie outside the map
                    // (zero filled); their scores are masked and their values weighted by 0
                    tma_load_2d(smem_u32(ring + s * TILE), map, 0, row0 + j * BN, fb);
                    tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, row0 + j * BN, fb);
                }
            }
            bad = __shfl_sync(0xffffffffu, bad, 0) || __shfl_sync(0xffffffffu, bad, 1);
        }
        if (lane < 2) {
            if (bad) fail_wait(bars, a.err);
            // our own copies land before the CTA's shared memory is released (bounded in
            // time only: an error raised elsewhere must not cut this short)
            const int NS = lane == 0 ? KST : VST;
            uint64_t* full = lane == 0 ? bars->k_full : bars->v_full;
            for (int u = gt - NS < 0 ? 0 : gt - NS; u < gt; ++u)
                mbar_wait_bounded(smem_u32(&full[u % NS]), (u / NS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(QROWS, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(QROWS, D, false, true);
            const uint64_t dq = smem_desc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
            const uint64_t dk = smem_desc_sw128(smem_u32(smem + OFF_K), 16, 1024);
            const uint64_t dv = smem_desc_sw128(smem_u32(smem + OFF_V), HALF, 1024);
            auto issue_qk = [&](int u, int ks) {
                const uint64_t kd = dk + (uint64_t)((ks * TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * HALF + (kk & 3) * 32) >> 4;
                    tc_mma_ss(tmem + COL_S + u * 128, dq + off, kd + off, idesc_qk, kk > 0);
                }
                tc_commit(smem_u32(&bars->s_full[u]));
            };
            bool ok = true;
            int segs = 0, gt = 0;                    // segments and tiles consumed so far
            for (int l = l_first; ok && l < lanes && a.item_start[l] < T1; ++l) {
                const Seg sg = seg_of(a, l, T0, T1);
                if (!mbar_wait_bounded(smem_u32(&bars->q_full), segs & 1, a.err) ||
                    !mbar_wait_bounded(smem_u32(&bars->k_full[gt % KST]), (gt / KST) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_qk(gt & 1, gt % KST);
                tc_commit(smem_u32(&bars->k_empty[gt % KST]));
                for (int j = 0; j < sg.n; ++j) {
                    const int gj = gt + j, u = gj & 1;
                    if (j + 1 < sg.n) {
                        // S_{j+1} into the other buffer, whose P the P V issued for the previous
                        // tile has read (this thread's MMAs run in order)
                        const int ks = (gj + 1) % KST;
                        if (!mbar_wait_bounded(smem_u32(&bars->k_full[ks]), ((gj + 1) / KST) & 1, a.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_qk(u ^ 1, ks);
                        tc_commit(smem_u32(&bars->k_empty[ks]));
                    } else {
                        // every QK^T of the segment is issued: the query tile may be rewritten
                        // once they complete
                        tc_commit(smem_u32(&bars->q_empty));
                    }
                    const int vs = gj % VST;
                    if (!mbar_wait_bounded(smem_u32(&bars->v_full[vs]), (gj / VST) & 1, a.err) ||
                        !mbar_wait_bounded(smem_u32(&bars->p_full[u]), (gj >> 1) & 1, a.err) ||
                        (j == 0 && segs > 0 && !mbar_wait_bounded(smem_u32(&bars->o_free), (segs - 1) & 1, a.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t vd = dv + (uint64_t)((vs * TILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts(tmem + COL_O, tmem + COL_S + u * 128 + kk * 8, vd + (uint64_t)(kk * 16 * 128 >> 4),
                                  idesc_pv, (j > 0 || kk > 0));
                    tc_commit(smem_u32(&bars->v_empty[vs]));
                    tc_commit(smem_u32(&bars->pv_done));
                }
                if (!ok) break;
                tc_commit(smem_u32(&bars->o_done));     // every MMA of the segment: O is final
                gt += sg.n;
                ++segs;
            }
            // every MMA issued by this thread completes before the tensor memory is freed (no
            // abort: the MMAs always finish): the last segment's o_done phase, or after an
            // error a commit for the unfinished segment
            if (!ok) {
                fail_wait(bars, a.err);
                tc_commit(smem_u32(&bars->o_done));
                mbar_wait_bounded(smem_u32(&bars->o_done), segs & 1);
            } else if (segs > 0) {
                mbar_wait_bounded(smem_u32(&bars->o_done), (segs - 1) & 1);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ query rows
        uint8_t* qt = smem + OFF_Q;
        // rows 32 .. 127 stay zero for every segment
        for (int u = lane; u < (QROWS - 32) * 16; u += 32) {
            const int row = 32 + (u >> 4), c = u & 15;
            *reinterpret_cast<uint4*>(qt + (c >> 3) * HALF + swz128(row, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
        int segs = 0;
        bool ok = true;
        for (int l = l_first; ok && l < lanes && a.item_start[l] < T1; ++l, ++segs) {
            const Seg sg = seg_of(a, l, T0, T1);
            // the previous segment's QK^T read the tile
            if (segs > 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->q_empty), (segs - 1) & 1, a.err))) {
                ok = false;
                break;
            }
            // row g < G: query head hkv G + g rotated at the sequence's position; rows G .. 31
            // zero.  Lane l takes columns 4 l .. 4 l + 3 (rotation pairs 2 l, 2 l + 1) of
            // every row, so that all 32 row loads are in flight at once.
            const int pos = a.pos[sg.b];
            float2 cs[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
            if (a.rope_f) {
                cs[0] = a.rope_f[(int64_t)pos * (D / 2) + 2 * lane];
                cs[1] = a.rope_f[(int64_t)pos * (D / 2) + 2 * lane + 1];
            }
            const __nv_bfloat16* q0 = a.q_in + ((int64_t)sg.b * a.Hq + sg.hkv * G) * D + 4 * lane;
            uint2 raw[32];
#pragma unroll
            for (int g = 0; g < 32; ++g)
                raw[g] = g < G ? *reinterpret_cast<const uint2*>(q0 + (int64_t)g * D) : make_uint2(0u, 0u);
            const int chunk = lane >> 1;
#pragma unroll
            for (int g = 0; g < 32; ++g) {
                uint32_t w[2] = {raw[g].x, raw[g].y};
                if (a.rope_f && g < G) {
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float x = __uint_as_float(w[p] << 16), y = __uint_as_float(w[p] & 0xffff0000u);
                        w[p] = pack_bf16(fmaf(x, cs[p].x, -(y * cs[p].y)), fmaf(y, cs[p].x, x * cs[p].y));
                    }
                }
                *reinterpret_cast<uint2*>(qt + (chunk >> 3) * HALF + swz128(g, chunk & 7) + (lane & 1) * 8) =
                    make_uint2(w[0], w[1]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->q_full));
        }
        if (!ok) fail_wait(bars, a.err);
    } else if (warp == 4) {
        // ------------------------------------------------------------ softmax
        const int g = lane;                         // query row = TMEM lane
        const uint32_t lane_addr = tmem;            // warp 4 reads lanes 0 .. 31
        const uint32_t o_addr = lane_addr + COL_O;
        const float sl2 = 1.4426950408889634f * rsqrtf((float)D);
        bool ok = true;
        int segs = 0, gt = 0;
        for (int l = l_first; ok && l < lanes && a.item_start[l] < T1; ++l) {
            const Seg sg = seg_of(a, l, T0, T1);
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < sg.n; ++j) {
                const int gj = gt + j, u = gj & 1;
                const uint32_t s_addr = lane_addr + COL_S + u * 128;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->s_full[u]), (gj >> 1) & 1, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kb = sg.r0 + j * BN;          // key of column 0
                const bool masked = kb < sg.lo || kb + BN > sg.r1;
                auto tile = [&](auto mask_c) -> bool {
                    float x[BN];
                    tmem_ld128(s_addr, x);
                    tmem_wait_ld();
                    if constexpr (decltype(mask_c)::value) {
#pragma unroll
                        for (int e = 0; e < BN; ++e) x[e] = (kb + e >= sg.r1 || kb + e < sg.lo) ? -INFINITY : x[e];
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
                    const float mx =
                        fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                    const float m_tile = mx * sl2;
                    // the P V of the previous tile of this segment (issued once its P was
                    // stored) completes before this tile's P is stored: waiting here, before
                    // this P exists, the barrier is at most one phase ahead; the O rescale
                    // below may then rewrite O
                    if (j > 0 &&
                        !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->pv_done), (gj - 1) & 1, a.err)))
                        return false;
                    const bool grow = m_tile > m_run + RESCALE_LOG2 || j == 0;
                    if (__any_sync(0xffffffffu, grow)) {
                        const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
                        const bool rescale = grow && j > 0 && m_run > -INFINITY;
                        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                            tc_fence_after();
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
                    }
                    const float mu = m_run == -INFINITY ? 0.f : m_run;
                    float2 l4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) l4[q] = make_float2(0.f, 0.f);
                    const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
                    uint32_t pk[BN / 2];
#pragma unroll
                    for (int e = 0; e < BN / 2; ++e) {
                        const int c2 = 2 * e;
                        const float2 arg = __ffma2_rn(make_float2(x[c2], x[c2 + 1]), sl2v, negmu);
                        const float p0 = fast_exp2(arg.x);
                        const float p1 = fast_exp2(arg.y);
                        l4[e & 3] = __fadd2_rn(l4[e & 3], make_float2(p0, p1));
                        pk[e] = pack_bf16(p0, p1);
                    }
                    tmem_st64u(s_addr, pk);
                    l4[0] = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
                    l_run += l4[0].x + l4[0].y;
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[u]));
                    return true;
                };
                if (!(masked ? tile(std::true_type{}) : tile(std::false_type{}))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            // every MMA of the segment has completed: O is final
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->o_done), segs & 1, a.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int64_t qh = (int64_t)sg.b * a.Hq + sg.hkv * G + g;
            const float inv = 1.0f / l_run;
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
                float o[32];
                tmem_ld32(o_addr + q * 32, o);
                tmem_wait_ld();
                if (g < G) {
                    if (sg.single) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) store_out(a, qh * D + q * 32 + e, o[e] * inv);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(a.part_o + (qh * a.max_splits + sg.slot) * D + q * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
                    }
                }
            }
            if (g < G && !sg.single) a.part_ml[qh * a.max_splits + sg.slot] = make_float2(m_run, l_run);
            // O has been read: the next segment's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
            gt += sg.n;
            ++segs;
        }
        if (!ok) fail_wait(bars, a.err);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_decode_tck(const DecodeLaunch& a, cudaStream_t s) {
    static PerDeviceOnce attr;
    cudaError_t e = attr.run(
        [] { return cudaFuncSetAttribute(decode_tck_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES); });
    if (e != cudaSuccess) return e;
    const int G = a.Hq / a.Hkv;
    if (!a.fused || a.dev_len || a.kv.table || G <= 16 || G > 32 || a.streamk <= 0 || a.B * a.Hkv > kFusedMaxB)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attrs[1];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.streamk, 1);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_tck_kernel, *a.tmK128, *a.tmV128, a);
}

}  // namespace kvc
