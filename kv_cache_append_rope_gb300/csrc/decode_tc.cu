// Split-K decode on the 5th-generation tensor cores, for many query heads per
// key/value head (bf16, d_h = 128, 16 < G = H_q / H_kv <= 32: multi-query attention).
//
// [Ch37] "Keep the prefix, project only the new row", listing "Evaluate one newest
// query across the retained rows plus the candidate key/value row before committing
// the append": every new query scores all t retained rows (q.k_j / sqrt(d_h)), takes a
// max-subtracted softmax and mixes the values; [Ch37] "From causal attention to managed
// LLM inference state" cites multi-query attention because reloading the K/V prefix is
// the bandwidth bottleneck, so one CTA serves all G query heads of one key/value head.
// With G = 32 that is 32 flop per byte of K/V -- more than the m16n8k16 path of the
// decode kernel sustains at the HBM rate -- so this kernel runs the two contractions
// on tcgen05 instead: the G heads are rows 0 .. G-1 of a 128-row query tile (the rest
// zero), S = Q K^T for 128 keys at a time lands in tensor memory, one softmax warp
// (one thread per head) turns it into P in place, and O += P V accumulates in tensor
// memory.  The MMAs waste the padding rows but need only about a third of the tensor
// rate, where the HBM rate is the bound.
//
// Work decomposition and results are those of the fused decode step
// (decode_bf16_kernel, MODE 1): grid (split, b * H_kv + kv_head); a CTA owns key rows
// [r0, r1) of its lane; the last split of a lane rotates and stores the new key row
// (bit-exact bf16 rounding) and the value row before its loads; the split's (O, max,
// sum) go to the same scratch and decode_combine_kernel merges the splits (or a lane
// with one split writes its normalised output); one CTA per sequence commits the
// length.  Contiguous storage only.
//
// Warp roles (160 threads):
//   warp 0   the new row (last split), then TMA (128-byte swizzle, no multicast):
//            lane 0 K tiles, lane 1 V tiles, 128 keys per tile, 2-stage rings
//   warp 1   tensor-memory allocation; one thread issues the MMAs:
//            S_{j+1} = Q K_{j+1}^T (into the other S buffer) before O += P_j V_j, so
//            the next tile's scores are ready when the softmax finishes this one
//   warps 2-3 the query tile: warp 2 rotates the G new query rows (float32 cos/sin of
//            the row's position, one fused multiply-add per component), rounds them
//            to bf16 and stores them swizzled as rows 0 .. 31; warp 3 zeroes rows 32 .. 127
//   warp 4   softmax of rows 0 .. 31 (tensor-memory lanes 0 .. 31): the whole 128-key
//            row per thread, mask outside [lo, r1), running max in log2 units with the
//            O rescale deferred until the max grows by more than 2^8 (waiting for the
//            previous P V first), P as bf16 pairs over the first 64 columns of its S
//            buffer; at the end O / l (or the unnormalised partial) to global memory.
// Every mbarrier wait is bounded (DEV_ERR_WAIT_TIMEOUT); the MMA thread waits for its
// last commit and the TMA lanes for their own copies before the tensor memory is freed.
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
    uint64_t q_full;
    uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
    uint64_t s_full[2], p_full[2];
    uint64_t pv_done, o_done;
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

// Key rows a query at t - 1 reads, counted from its window start rounded down to a
// 64-row tile (the decode kernel's split convention).
__device__ __forceinline__ int key_span(int t, int window) {
    return window > 0 ? t - (max(0, t - window) & ~63) : t;
}

__device__ __forceinline__ void store_out(const DecodeLaunch& a, int64_t i, float x) {
    if (a.out_bf16)
        ((__nv_bfloat16*)a.out)[i] = __float2bfloat16_rn(x);
    else
        ((float*)a.out)[i] = x;
}

__global__ void __launch_bounds__(THREADS, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ DecodeLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars* bars = (Bars*)(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int split = blockIdx.x, b, hkv, split_rows = a.split_rows;
    if (a.pieces) {
        // the sequence whose CTA range holds this CTA, then its kv head and split
        int lo_i = 0, hi_i = a.B;
        while (hi_i - lo_i > 1) {
            const int mid = (lo_i + hi_i) >> 1;
            if (a.item_start[mid] <= (int)blockIdx.x) lo_i = mid;
            else hi_i = mid;
        }
        b = a.seq_of[lo_i];
        const int r = blockIdx.x - a.item_start[lo_i];
        const int ns = (a.item_start[lo_i + 1] - a.item_start[lo_i]) / a.Hkv;
        hkv = r / ns;
        split = r - hkv * ns;
        split_rows = a.seq_rows[b];
    } else {
        b = (int)blockIdx.y / a.Hkv;
        hkv = (int)blockIdx.y - b * a.Hkv;
    }
    const int G = a.Hq / a.Hkv;
    // everything below may read what the previous kernel of the stream wrote
    grid_dependency_wait();
    launch_dependents();

    const int old_len = a.old_len[b], pos = a.pos[b];
    if (!debug_check(old_len >= 0 && old_len < a.C, threadIdx.x == 0 ? a.err : nullptr)) return;
    if (split == 0 && hkv == 0 && threadIdx.x == 0 && !a.no_commit) {
        a.len_out[b] = old_len + 1;
        a.next_out[b] = pos + 1;
    }
    const int t = old_len + 1;
    const int lo = a.window > 0 ? max(0, t - a.window) : 0;
    const int r0 = (lo & ~63) + split * split_rows;
    if (r0 >= t) return;
    const int r1 = min(t, r0 + split_rows);
    const int n = (r1 - r0 + BN - 1) / BN;                       // 128-key tiles
    const int nsplit_lane = (key_span(t, a.window) + split_rows - 1) / split_rows;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 2);
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
        // ------------------------------------------------------------ new row, then TMA
        if (split == nsplit_lane - 1) {
            // The new row (slot old_len) belongs to this split: rotate and store the key
            // (bit-exact bf16 rounding), store the value and the position, then order
            // these generic-proxy writes before this warp's TMA reads of them.
            const int64_t src = ((int64_t)b * a.Hkv + hkv) * D + lane * 4;
            const int64_t dst = (((int64_t)b * a.Hkv + hkv) * a.C + old_len) * D + lane * 4;
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
            if (hkv == 0 && lane == 0) a.positions[(int64_t)b * a.C + old_len] = pos;
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
            prefetch_tmap(map);
            const int row0 = ((b * a.Hkv + hkv) * a.C) + r0;    // contiguous storage
            int issued = 0;
            for (int j = 0; j < n && !*(volatile int*)&bars->err; ++j) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait_bounded(smem_u32(&empty[s]), ((j / NS) - 1) & 1, a.err)) {
                    fail_wait(bars, a.err);
                    break;
                }
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, TILE);
                // rows past the split belong to the next lane or lie outside the map (zero
                // filled); their scores are masked and their values weighted by 0
                tma_load_2d(smem_u32(ring + s * TILE), map, 0, row0 + j * BN, fb);
                tma_load_2d(smem_u32(ring + s * TILE + HALF), map, 64, row0 + j * BN, fb);
                issued = j + 1;
            }
            // our own copies land before the CTA's shared memory is released (bounded in
            // time only: an error raised elsewhere must not cut this short)
            for (int u = issued - NS < 0 ? 0 : issued - NS; u < issued; ++u)
                mbar_wait_bounded(smem_u32(&full[u % NS]), (u / NS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(QROWS, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(QROWS, D, false, true);
            bool ok = mbar_wait_bounded(smem_u32(&bars->q_full), 0, a.err);
            tc_fence_after();
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
            if (ok) {
                ok = mbar_wait_bounded(smem_u32(&bars->k_full[0]), 0, a.err);
                tc_fence_after();
                if (ok) {
                    issue_qk(0, 0);
                    tc_commit(smem_u32(&bars->k_empty[0]));
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                const int u = j & 1;
                if (j + 1 < n) {
                    // S_{j+1} into the other buffer, whose P_{j-1} the P V issued in the
                    // previous iteration has read (this thread's MMAs run in order)
                    const int ks = (j + 1) % KST;
                    if (!mbar_wait_bounded(smem_u32(&bars->k_full[ks]), ((j + 1) / KST) & 1, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(u ^ 1, ks);
                    tc_commit(smem_u32(&bars->k_empty[ks]));
                }
                const int vs = j % VST;
                if (!mbar_wait_bounded(smem_u32(&bars->v_full[vs]), (j / VST) & 1, a.err) ||
                    !mbar_wait_bounded(smem_u32(&bars->p_full[u]), (j >> 1) & 1, a.err)) {
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
            if (!ok) fail_wait(bars, a.err);
            // every MMA issued by this thread completes before O is read and the memory freed
            tc_commit(smem_u32(&bars->o_done));
            mbar_wait_bounded(smem_u32(&bars->o_done), 0);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ query rows 0 .. 31
        // row g < G: query head hkv * G + g rotated at `pos`; rows G .. 31 zero.  Lane l
        // takes columns 4 l .. 4 l + 3 (rotation pairs 2 l, 2 l + 1) of every row, so that
        // all 32 row loads are in flight at once and the cos/sin pairs are loaded once.
        uint8_t* qt = smem + OFF_Q;
        float2 cs[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
        if (a.rope_f) {
            cs[0] = a.rope_f[(int64_t)pos * (D / 2) + 2 * lane];
            cs[1] = a.rope_f[(int64_t)pos * (D / 2) + 2 * lane + 1];
        }
        const __nv_bfloat16* q0 = a.q_in + ((int64_t)b * a.Hq + hkv * G) * D + 4 * lane;
        uint2 raw[32];
#pragma unroll
        for (int g = 0; g < 32; ++g) raw[g] = g < G ? *reinterpret_cast<const uint2*>(q0 + (int64_t)g * D) : make_uint2(0u, 0u);
        const int chunk = lane >> 1;                   // 16-byte chunk of the 256-byte row
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
    } else if (warp == 3) {
        // ------------------------------------------------------------ query rows 32 .. 127: zero
        uint8_t* qt = smem + OFF_Q;
        for (int u = lane; u < (QROWS - 32) * 16; u += 32) {
            const int row = 32 + (u >> 4), c = u & 15;
            *reinterpret_cast<uint4*>(qt + (c >> 3) * HALF + swz128(row, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->q_full));
    } else {
        // ------------------------------------------------------------ softmax (warp 4)
        const int g = lane;                         // query row = TMEM lane
        const uint32_t lane_addr = tmem;            // warp 4 reads lanes 0 .. 31
        const uint32_t o_addr = lane_addr + COL_O;
        const float sl2 = 1.4426950408889634f * rsqrtf((float)D);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int u = j & 1;
            const uint32_t s_addr = lane_addr + COL_S + u * 128;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->s_full[u]), (j >> 1) & 1, a.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kb = r0 + j * BN;             // key of column 0
            const bool masked = kb < lo || kb + BN > r1;
            auto tile = [&](auto mask_c) -> bool {
                float x[BN];
#pragma unroll
                for (int q = 0; q < BN / 32; ++q) tmem_ld32(s_addr + q * 32, x + q * 32);
                tmem_wait_ld();
                if constexpr (decltype(mask_c)::value) {
#pragma unroll
                    for (int e = 0; e < BN; ++e) x[e] = (kb + e >= r1 || kb + e < lo) ? -INFINITY : x[e];
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
                // P V of tile j - 1 (issued once P_{j-1} was stored) completes before this
                // tile's P is stored: waiting here, before P_j exists, the barrier can be at
                // most one phase ahead, so the parity wait is unambiguous; and the O rescale
                // below may then rewrite O
                if (j > 0 &&
                    !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->pv_done), (j - 1) & 1, a.err)))
                    return false;
                const bool grow = m_tile > m_run + RESCALE_LOG2 || j == 0;
                if (__any_sync(0xffffffffu, grow)) {
                    const float m_new = grow ? fmaxf(m_run, m_tile) : m_run;
                    const bool rescale = grow && j > 0 && m_run > -INFINITY;
                    if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                        // rewrite O (warp-collective ld/st)
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
                if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[u]));
                return true;
            };
            if (!(masked ? tile(std::true_type{}) : tile(std::false_type{}))) {
                ok = false;
                break;
            }
        }
        if (ok && n > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&bars->o_done), 0, a.err))) {
                ok = false;
            } else {
                tc_fence_after();
                const int64_t qh = (int64_t)b * a.Hq + hkv * G + g;
                const bool single = nsplit_lane == 1;
                const float inv = 1.0f / l_run;
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    float o[32];
                    tmem_ld32(o_addr + q * 32, o);
                    tmem_wait_ld();
                    if (g < G) {
                        if (single) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) store_out(a, qh * D + q * 32 + e, o[e] * inv);
                        } else {
                            float4* dst = reinterpret_cast<float4*>(a.part_o + (qh * a.max_splits + split) * D + q * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
                        }
                    }
                }
                if (g < G && !single) a.part_ml[qh * a.max_splits + split] = make_float2(m_run, l_run);
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

cudaError_t launch_decode_tc(const DecodeLaunch& a, cudaStream_t s) {
    static PerDeviceOnce attr;
    cudaError_t e = attr.run(
        [] { return cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES); });
    if (e != cudaSuccess) return e;
    const int G = a.Hq / a.Hkv;
    if (!a.fused || a.dev_len || a.kv.table || G <= 16 || G > 32) return cudaErrorInvalidValue;
    cudaLaunchAttribute attrs[1];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = a.pieces ? dim3(a.item_start[a.B], 1) : dim3(a.max_splits, a.B * a.Hkv);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel, *a.tmK128, *a.tmV128, a);
}

}  // namespace kvc
