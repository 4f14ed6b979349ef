// Split-K flash-decoding for bf16 caches with d_h = 128 (MHA, GQA and MQA).
//
// [Ch37] "Keep the prefix, project only the new row", listing "Evaluate one
// newest query across the retained rows plus the candidate key/value row
// before committing the append": each new query scores all t retained rows
// (s_j = q.k_j / sqrt(d_h)), takes a max-subtracted softmax and mixes the t
// values.  [Ch37] "From causal attention to managed LLM inference state"
// cites multi-query attention because reloading the K/V prefix is the
// memory-bandwidth bottleneck; here one CTA serves all G = H_q / H_kv query
// heads of one key/value head, so every K/V byte is read from HBM once.
//
// Work decomposition: grid (split, b * H_kv + kv_head).  A CTA owns key rows
// [split * R, min((split + 1) * R, t)) of its lane (t = old length + 1: the
// new row was already appended by the RoPE/append kernel).  One producer warp
// streams 64-row K and V tiles with TMA (128-byte swizzle, no multicast) into
// a ring of shared-memory stages guarded by mbarriers; four consumer warps
// each own one 16-row MMA tile of the G query heads (padded to 16 or 32 rows)
// and 16 (one tile) or 32 (two tiles) keys of every stage, and compute
// S = Q K^T and O += P V with m16n8k16 bf16 tensor-core MMAs (fp32
// accumulation).  The softmax is online per warp (running
// max and sum in log2 units, quad shuffles for row maxima); the four warps
// are merged through shared memory and the split's (O, max, sum) is written
// to scratch, or the normalised output when the lane has a single split.  A
// second kernel merges the splits of every query head by log-sum-exp.
//
// Fused step (one launch per decode step): the old lengths and RoPE positions
// arrive as kernel parameters (host mirrors); the producer warp of each lane's
// last split rotates and stores the new key row (bit-exact bf16 rounding) and
// the value row before its TMA loads read them; the consumers rotate the new
// queries in registers; the last CTA of a lane to finish (an atomic ticket, no
// waiting) merges the splits -- or, with more than 16 query heads per lane,
// the separate merge kernel does, spread over every query head -- and one CTA
// per sequence commits the new length.
#include <cuda.h>

#include "device_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int D = 128;
constexpr int KT = 64;                 // key rows per stage
constexpr int NCW = 4;                 // consumer warps
constexpr int THREADS = (NCW + 1) * 32;
constexpr int HALF_BYTES = KT * 128;   // 64 rows x 64 dims x 2 B
constexpr int TILE_BYTES = 2 * HALF_BYTES;
constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K and V

template <int STAGES>
constexpr int smem_bytes() { return STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/; }

template <int MT> struct Cfg;
template <> struct Cfg<1> { static constexpr int STAGES = 3; static constexpr int MINB = 2; };
template <> struct Cfg<2> { static constexpr int STAGES = 3; static constexpr int MINB = 2; };

// Key rows a query at t - 1 reads, counted from its window start rounded down to a
// 64-row tile (the splits cover exactly this span).
__device__ __forceinline__ int key_span(int t, int window) {
    return window > 0 ? t - (max(0, t - window) & ~(KT - 1)) : t;
}

// A query pair (x, y) rotated by (cos, sin) = cs in float32.
__device__ __forceinline__ float2 q_rotate(float x, float y, float2 cs) {
    return make_float2(fmaf(x, cs.x, -(y * cs.y)), fmaf(y, cs.x, x * cs.y));
}

// Rotated query pair (c, c+1) of row `row` (< G) of this lane, as float32 (fused step).
__device__ __forceinline__ float2 fused_q_pair(const DecodeLaunch& a, int b, int qh, int c, int pos) {
    const __nv_bfloat162 v = *(const __nv_bfloat162*)(a.q_in + ((int64_t)b * a.Hq + qh) * D + c);
    const float x = __low2float(v), y = __high2float(v);
    if (!a.rope_f) return make_float2(x, y);
    return q_rotate(x, y, a.rope_f[(int64_t)pos * (D / 2) + c / 2]);
}

// Final output element: float32, or rounded to bf16 when the caller asked for bf16 output.
__device__ __forceinline__ void store_out(const DecodeLaunch& a, int64_t i, float x) {
    if (a.out_bf16)
        ((__nv_bfloat16*)a.out)[i] = __float2bfloat16_rn(x);
    else
        ((float*)a.out)[i] = x;
}

// Log-sum-exp merge of one query head's ns split partials ((max, sum) in ml, O rows in po,
// already offset to one head dim): the loads of the first kMergeBatch splits are all issued
// before any is used (one memory round trip instead of two per split), and the sums run
// over the splits in order.
constexpr int kMergeBatch = 8;
__device__ __forceinline__ float merge_splits(const float2* ml, const float* po, int ns) {
    float2 mv[kMergeBatch];
    float ov[kMergeBatch];
#pragma unroll
    for (int s = 0; s < kMergeBatch; ++s) {
        if (s < ns) {
            mv[s] = __ldcg(&ml[s]);
            ov[s] = __ldcg(po + (int64_t)s * D);
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMergeBatch; ++s)
        if (s < ns) M = fmaxf(M, mv[s].x);
    for (int s = kMergeBatch; s < ns; ++s) M = fmaxf(M, __ldcg(&ml[s].x));
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int s = 0; s < kMergeBatch; ++s) {
        if (s < ns) {
            const float f = fast_exp2(mv[s].x - M);
            L += mv[s].y * f;
            O += ov[s] * f;
        }
    }
    for (int s = kMergeBatch; s < ns; ++s) {
        const float2 v = __ldcg(&ml[s]);
        const float f = fast_exp2(v.x - M);
        L += v.y * f;
        O += __ldcg(po + (int64_t)s * D) * f;
    }
    return O / L;
}

// One 64-key stage of a consumer warp: S = Q K^T for the warp's KW = 16 MT keys (key
// key_base + j), masked outside [lo, r1); the online softmax of rows qa and qa + 8 of
// its m tile; O += P V.  kt, vt: the stage's K and V tiles in shared memory.
template <int MT>
__device__ __forceinline__ void consume_stage(uint32_t kt, uint32_t vt, int key_base, int r1, int lo,
                                              const uint32_t (&qf)[8][4], float (&o)[16][4], float (&m)[2],
                                              float (&l)[2], int lane, int kofs) {
    constexpr int KW = 16 * MT;              // keys per warp per stage
    constexpr int NT = KW / 8;               // n8 tiles of S
    constexpr int KS = KW / 16;              // k16 steps of P V
    const int qc = (lane & 3) * 2;           // fragment column pair
    // ---- S = Q K^T for this warp's KW keys
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
    // (k-outer: the NT accumulators are independent chains, so consecutive MMAs
    // do not wait on one another)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int dim0 = kk * 32 + (lane >> 3) * 8;
        uint32_t bk[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = kofs + nt * 8 + (lane & 7);
            const uint32_t addr = kt + (dim0 >> 6) * HALF_BYTES + swz128(row, (dim0 & 63) >> 3);
            ldsm_x4(addr, bk[nt][0], bk[nt][1], bk[nt][2], bk[nt][3]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], qf[2 * kk], bk[nt][0], bk[nt][1]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], qf[2 * kk + 1], bk[nt][2], bk[nt][3]);
    }
    // ---- mask keys beyond this split
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int key = key_base + nt * 8 + qc + e;
            if (key >= r1 || key < lo) {
                sc[nt][e] = -INFINITY;
                sc[nt][2 + e] = -INFINITY;
            }
        }
    // ---- online softmax (rows qa and qa + 8 of this m tile)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mx = fmaxf(mx, fmaxf(sc[nt][2 * rr], sc[nt][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // The reference maximum moves only when a score passes it by more than 2^8
        // (log2 units): exponentials up to 2^8 are exact enough in float32 and bf16,
        // and the final division by the running sum cancels the reference, so a
        // stale one changes nothing but rounding.  O is rescaled only then (a
        // warp-wide decision: rows that did not move are multiplied by 1).
        const bool grow = mx > m[rr] + 8.f;
        if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? fmaxf(m[rr], mx) : m[rr];
            const float corr = grow && m[rr] > -INFINITY ? fast_exp2(m[rr] - m_new) : 1.f;
            m[rr] = m_new;
            l[rr] *= corr;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o[n][2 * rr] *= corr;
                o[n][2 * rr + 1] *= corr;
            }
        }
        const float m_use = m[rr] == -INFINITY ? 0.f : m[rr];
        float ps = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float p = fast_exp2(sc[nt][2 * rr + e] - m_use);
                sc[nt][2 * rr + e] = p;
                ps += p;
            }
        l[rr] += ps;
    }
    // ---- O += P V (V^T fragments through transposing ldmatrix)
#pragma unroll
    for (int k2 = 0; k2 < KS; ++k2) {
        uint32_t pf[4];
        pf[0] = pack_bf16(sc[2 * k2][0], sc[2 * k2][1]);
        pf[1] = pack_bf16(sc[2 * k2][2], sc[2 * k2][3]);
        pf[2] = pack_bf16(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
        pf[3] = pack_bf16(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
        const int vrow = kofs + k2 * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            const int dim = np * 16 + (lane >> 4) * 8;
            const uint32_t addr = vt + (dim >> 6) * HALF_BYTES + swz128(vrow, (dim & 63) >> 3);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            mma_bf16_16816(o[2 * np], pf, b0, b1);
            mma_bf16_16816(o[2 * np + 1], pf, b2, b3);
        }
    }
}

// MODE 0: separate-kernel step; 1: fused step, lengths from the host mirrors;
// 2: fused step, lengths from device memory.
template <int MT, int MODE>
__global__ void __launch_bounds__(THREADS, Cfg<MT>::MINB)
decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ DecodeLaunch a) {
    constexpr int STAGES = Cfg<MT>::STAGES;
    constexpr bool FUSED = MODE >= 1;
    const int split = blockIdx.x;
    const int lane_kv = blockIdx.y;
    const int b = lane_kv / a.Hkv;
    const int hkv = lane_kv - b * a.Hkv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    volatile int* s_err = (volatile int*)(empty + STAGES);   // s_err[1]: last-CTA flag
    // Everything below may read what the previous kernel of the stream wrote (the
    // previous step's row, lengths, split scratch): wait for it; and let the next
    // step's CTAs take the slots this grid leaves as it drains.
    grid_dependency_wait();
    launch_dependents();

    // Fused step: the old length and position come from the host mirrors, so no
    // kernel of the step reads the length this kernel commits.
    int old_len, pos, split_rows = a.split_rows;
    if constexpr (MODE == 2) {
        // Device-length step (the launch parameters do not depend on the lengths,
        // so it can be captured in a CUDA graph and replayed): every CTA reads its
        // sequence's length and position, and checks every sequence, from device
        // memory, then takes a ticket; the last CTA of the grid to do so -- all the
        // others have read by then -- commits every sequence.  A step in which
        // some sequence is full or would rotate beyond the table is rejected
        // whole, as the host checks reject it in the other modes.
        old_len = __ldcg(a.len_out + b);
        pos = __ldcg(a.next_out + b);
        int bad = 0;
        for (int i = threadIdx.x; i < a.B; i += THREADS) {
            const int L = __ldcg(a.len_out + i), P = __ldcg(a.next_out + i);
            bad |= (L < 0) | (L >= a.C) | (P < 0) | (a.rope_f != nullptr && P >= a.max_positions);
        }
        const bool reject = __syncthreads_or(bad) != 0;
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(a.step_ticket, 1u);
            s_err[1] = prev == gridDim.x * gridDim.y - 1;
        }
        __syncthreads();
        if (s_err[1]) {
            for (int i = threadIdx.x; i < a.B && !reject; i += THREADS) {
                a.len_out[i] = __ldcg(a.len_out + i) + 1;
                a.next_out[i] = __ldcg(a.next_out + i) + 1;
            }
            if (threadIdx.x == 0) {
                *a.step_ticket = 0;
                if (reject) atomicOr(a.err, (uint32_t)DEV_ERR_FULL);
            }
        }
        if (reject) return;
        // every sequence takes max_splits splits, sized from its own (windowed) key count
        const int nk = key_span(old_len + 1, a.window);
        split_rows = ((nk + a.max_splits - 1) / a.max_splits + KT - 1) / KT * KT;
    } else {
        old_len = FUSED ? a.old_len[b] : a.len[b];
        pos = FUSED ? a.pos[b] : 0;
        // debug builds: the new row's slot (and so every key row read) lies inside the lane
        if (!debug_check(old_len >= 0 && old_len < a.C, threadIdx.x == 0 ? a.err : nullptr)) return;
        if (FUSED && split == 0 && hkv == 0 && threadIdx.x == 0 && !a.no_commit) {
            a.len_out[b] = old_len + 1;
            a.next_out[b] = pos + 1;
        }
    }
    const int t = old_len + 1;
    // keys lo .. t-1: every retained row, or the `window` most recent ones; the
    // splits start at lo rounded down to a tile (keys before lo are masked), so
    // that a 64-row tile never crosses a block of paged storage
    const int lo = a.window > 0 ? max(0, t - a.window) : 0;
    const int r0 = (lo & ~(KT - 1)) + split * split_rows;
    if (r0 >= t) return;
    const int r1 = min(t, r0 + split_rows);
    const int ntiles = (r1 - r0 + KT - 1) / KT;
    const int G = a.Hq / a.Hkv;
    const int nsplit_lane = (key_span(t, a.window) + split_rows - 1) / split_rows;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), NCW);
        }
        *s_err = 0;
        fence_mbar_init();
    }
    __syncthreads();

    int issued = 0;
    float o[16][4];
    float m[2], l[2];

    if (warp == NCW) {
        // ---------------- producer ----------------
        if (FUSED && split == nsplit_lane - 1) {
            // The new row (slot old_len) belongs to this split: rotate and store the
            // key (bit-exact bf16 rounding), store the value and the position, then
            // order these generic-proxy writes before this warp's TMA reads of them.
            const int64_t src = ((int64_t)b * a.Hkv + hkv) * D + lane * 4;
            const bool slot_ok = debug_check(kv_slot_ok(a.kv, b, old_len), lane == 0 ? a.err : nullptr);
            const int64_t dst = slot_ok ? kv_row(a.kv, b, hkv, old_len) * D + lane * 4 : 0;
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
            if (slot_ok) {
                *(uint2*)(a.K + dst) = *(const uint2*)kout;
                *(uint2*)(a.V + dst) = vraw;
                if (hkv == 0 && lane == 0) a.positions[(int64_t)b * a.C + old_len] = pos;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
        }
        if (lane == 0 && !a.test_stall) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            // (paged storage: the next tile's block-table entry is loaded one tile ahead,
            // so its latency overlaps the wait for a free stage)
            int y_next = (int)kv_row(a.kv, b, hkv, r0);
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % STAGES;
                const int y = y_next;
                if (i + 1 < ntiles) y_next = (int)kv_row(a.kv, b, hkv, r0 + (i + 1) * KT);
                if (i >= STAGES && !mbar_wait_bounded(smem_u32(&empty[s]), ((i / STAGES) - 1) & 1)) {
                    *s_err = 1;
                    atomicOr(a.err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
                    break;
                }
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, STAGE_BYTES);
                uint8_t* st = smem + s * STAGE_BYTES;
                tma_load_2d(smem_u32(st), &tmK, 0, y, fb);
                tma_load_2d(smem_u32(st + HALF_BYTES), &tmK, 64, y, fb);
                tma_load_2d(smem_u32(st + TILE_BYTES), &tmV, 0, y, fb);
                tma_load_2d(smem_u32(st + TILE_BYTES + HALF_BYTES), &tmV, 64, y, fb);
                issued = i + 1;
            }
        }
    } else {
        // ---------------- consumers ----------------
        // Each consumer warp owns one 16-row MMA tile of the G query heads and
        // KW = 16 * MT keys of every 64-key stage: with MT = 2 (G up to 32),
        // warps 0-1 hold heads 0-15 and warps 2-3 heads 16-31, each pair
        // splitting the stage's keys, so that every warp keeps one tile of
        // accumulators in registers and two CTAs fit on an SM.
        constexpr int KW = 16 * MT;              // keys per warp per stage
        constexpr int NT = KW / 8;               // n8 tiles of S
        constexpr int KS = KW / 16;              // k16 steps of P V
        constexpr int WPM = NCW / MT;            // warps per m tile
        const int mtw = warp / WPM;
        const int kofs = (warp % WPM) * KW;
        const int qa = lane >> 2;                // fragment row (and row + 8)
        const int qc = (lane & 3) * 2;           // fragment column pair
        // Q fragments, pre-scaled so that scores come out in log2 units.
        const float qscale = 1.4426950408889634f * rsqrtf((float)D);
        uint32_t qf[8][4];
        {
            const int ra = mtw * 16 + qa, rb = ra + 8;
            const float* qra = a.qrot + ((int64_t)b * a.Hq + hkv * G + ra) * D;
            const float* qrb = a.qrot + ((int64_t)b * a.Hq + hkv * G + rb) * D;
            const int qpos = pos;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int c = ks * 16 + qc;
                float2 x0, x1, x2, x3;
                if (FUSED) {
                    const float2 z = make_float2(0.f, 0.f);
                    x0 = ra < G ? fused_q_pair(a, b, hkv * G + ra, c, qpos) : z;
                    x1 = rb < G ? fused_q_pair(a, b, hkv * G + rb, c, qpos) : z;
                    x2 = ra < G ? fused_q_pair(a, b, hkv * G + ra, c + 8, qpos) : z;
                    x3 = rb < G ? fused_q_pair(a, b, hkv * G + rb, c + 8, qpos) : z;
                } else {
                    x0 = ra < G ? *(const float2*)(qra + c) : make_float2(0.f, 0.f);
                    x1 = rb < G ? *(const float2*)(qrb + c) : make_float2(0.f, 0.f);
                    x2 = ra < G ? *(const float2*)(qra + c + 8) : make_float2(0.f, 0.f);
                    x3 = rb < G ? *(const float2*)(qrb + c + 8) : make_float2(0.f, 0.f);
                }
                qf[ks][0] = pack_bf16(x0.x * qscale, x0.y * qscale);
                qf[ks][1] = pack_bf16(x1.x * qscale, x1.y * qscale);
                qf[ks][2] = pack_bf16(x2.x * qscale, x2.y * qscale);
                qf[ks][3] = pack_bf16(x3.x * qscale, x3.y * qscale);
            }
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[n][e] = 0.f;

        for (int i = 0; i < ntiles; ++i) {
            const int s = i % STAGES;
            // one verdict for the warp: the MMAs below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (i / STAGES) & 1))) {
                *s_err = 1;
                atomicOr(a.err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
                break;
            }
            const uint32_t kt = smem_u32(smem + s * STAGE_BYTES);
            const uint32_t vt = kt + TILE_BYTES;
            const int key_base = r0 + i * KT + kofs;

            consume_stage<MT>(kt, vt, key_base, r1, lo, qf, o, m, l, lane, kofs);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
    }

    __syncthreads();
    if (*s_err) {
        // Let copies already issued land before the CTA's shared memory is released.
        if (warp == NCW && lane == 0) {
            for (int i = issued - STAGES < 0 ? 0 : issued - STAGES; i < issued; ++i)
                mbar_wait_bounded(smem_u32(&full[i % STAGES]), (i / STAGES) & 1);
        }
        __syncthreads();
        return;
    }

    // ---------------- merge the consumer warps of each m tile ----------------
    constexpr int WPMr = NCW / MT;                               // warps per m tile
    float* Om = (float*)smem;                                    // [NCW][16][D]
    float2* ML = (float2*)(smem + NCW * 16 * D * 4);             // [NCW][16]
    if (warp < NCW) {
        const int qa = lane >> 2, qc = (lane & 3) * 2;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float lr = l[rr];
            lr += __shfl_xor_sync(0xffffffffu, lr, 1);
            lr += __shfl_xor_sync(0xffffffffu, lr, 2);
            const int row = qa + rr * 8;
            float* dst = Om + ((size_t)warp * 16 + row) * D;
#pragma unroll
            for (int n = 0; n < 16; ++n) *(float2*)(dst + n * 8 + qc) = make_float2(o[n][2 * rr], o[n][2 * rr + 1]);
            if ((lane & 3) == 0) ML[warp * 16 + row] = make_float2(m[rr], lr);
        }
    }
    __syncthreads();
    for (int u = threadIdx.x; u < G * D; u += THREADS) {
        const int g = u / D, dim = u - g * D;
        const int w0 = (g >> 4) * WPMr, gl = g & 15;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WPMr; ++w) M = fmaxf(M, ML[(w0 + w) * 16 + gl].x);
        float O = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < WPMr; ++w) {
            const float2 ml = ML[(w0 + w) * 16 + gl];
            const float f = fast_exp2(ml.x - M);
            O += Om[((size_t)(w0 + w) * 16 + gl) * D + dim] * f;
            L += ml.y * f;
        }
        const int64_t qh = (int64_t)b * a.Hq + hkv * G + g;
        if (nsplit_lane == 1) {
            store_out(a, qh * D + dim, O / L);
        } else {
            const int64_t idx = qh * a.max_splits + split;
            a.part_o[idx * D + dim] = O;
            if (dim == 0) a.part_ml[idx] = make_float2(M, L);
        }
    }
    if (!FUSED || nsplit_lane == 1 || !a.merge_in_kernel) return;

    // Fused step: the last CTA of this lane to finish merges every split (a ticket,
    // no waiting), then resets the ticket for the next step.
    __threadfence();
    __syncthreads();
    volatile int* s_last = s_err + 1;
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&a.lane_ticket[lane_kv], 1u);
        *s_last = prev == (unsigned)(nsplit_lane - 1);
    }
    __syncthreads();
    if (!*s_last) return;
    __threadfence();
    for (int u = threadIdx.x; u < G * D; u += THREADS) {
        const int g = u / D, dim = u - g * D;
        const int64_t qh = (int64_t)b * a.Hq + hkv * G + g;
        store_out(a, qh * D + dim,
                  merge_splits(a.part_ml + qh * a.max_splits, a.part_o + qh * a.max_splits * D + dim, nsplit_lane));
    }
    if (threadIdx.x == 0) a.lane_ticket[lane_kv] = 0;
}

__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeLaunch a) {
    grid_dependency_wait();
    launch_dependents();
    const int qh = blockIdx.x;
    const int b = qh / a.Hq;
    int t, rows = a.split_rows;
    if (a.dev_len) {
        // after the step's commit (after a rejected step the output is undefined)
        t = __ldcg(a.len_out + b);
        if (t <= 0) return;
        rows = ((key_span(t, a.window) + a.max_splits - 1) / a.max_splits + KT - 1) / KT * KT;
    } else {
        t = (a.fused ? a.old_len[b] : a.len[b]) + 1;
        if (a.pieces) rows = a.seq_rows[b];
    }
    if (!debug_check(t >= 1 && t <= a.C, threadIdx.x == 0 ? a.err : nullptr)) return;
    // stream-K: the lane's partials, one per CTA its tiles touched
    const int ns = a.streamk ? a.seq_rows[b * a.Hkv + (qh - b * a.Hq) / (a.Hq / a.Hkv)]
                             : (key_span(t, a.window) + rows - 1) / rows;
    if (ns <= 1) return;
    store_out(a, (int64_t)qh * D + threadIdx.x,
              merge_splits(a.part_ml + (int64_t)qh * a.max_splits,
                           a.part_o + (int64_t)qh * a.max_splits * D + threadIdx.x, ns));
}

// ---- many short lanes per CTA ---------------------------------------------------
//
// Fused decode step for short contexts (every lane one split) with G <= 4 query heads
// per key/value head: a CTA walks lanes_per_cta lanes in turn -- sequences in the order
// seq_of[] (longest first), their key/value heads in order -- through one continuous
// ring of stages, so that the producer loads the next lane's tiles while the consumers
// finish the current one and the per-CTA set-up (barriers, pipeline fill) is paid once
// for all of them.  Per lane it does exactly what the fused step does for a lane with
// one split: the new key (bit-exact rotation) and value rows and the position are stored
// before the lane's loads (a lane's last, partial tile loads only its 16-row boxes that
// hold keys), the consumer warps process its 64-key stages (consume_stage), merge through a small shared-memory buffer behind a barrier of the
// four consumer warps only, and write the normalised output; the CTA of a sequence's
// key/value head 0 commits its length.
constexpr int kLanesMaxG = 4;
constexpr int kLanesQBytes = kLanesMaxG * D * 2;  // a lane's rotated, scaled bf16 queries
constexpr int kLanesMergeBytes = NCW * kLanesMaxG * D * 4 + NCW * kLanesMaxG * 8;

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, Cfg<1>::MINB)
decode_lanes_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
                    const __grid_constant__ DecodeLaunch a) {
    constexpr int STAGES = Cfg<1>::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    volatile int* s_err = (volatile int*)(empty + STAGES);
    float* Om = (float*)(smem + STAGES * STAGE_BYTES + 256);                 // [NCW][4][D]
    float2* ML = (float2*)(smem + STAGES * STAGE_BYTES + 256 + NCW * kLanesMaxG * D * 4);  // [NCW][4]
    // [STAGES][kLanesMaxG][D] bf16: the queries of the lane whose first tile is in stage s
    uint8_t* Qs = smem + STAGES * STAGE_BYTES + 256 + kLanesMergeBytes;
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);
    grid_dependency_wait();
    launch_dependents();
    const int G = a.Hq / a.Hkv;
    const int nlanes = a.B * a.Hkv;
    const int l_begin = blockIdx.x * a.lanes_per_cta;
    const int l_end = min(nlanes, l_begin + a.lanes_per_cta);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), NCW);
        }
        *s_err = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // lane li: the (li / H_kv)-th sequence of seq_of, key/value head li % H_kv
    auto lane_of = [&](int li, int& b, int& hkv) {
        b = a.seq_of[li / a.Hkv];
        hkv = li % a.Hkv;
    };
    int issued = 0;
    if (warp == NCW) {
        // ---------------- producer ----------------
        int gi = 0;
        for (int li = l_begin; li < l_end && !*s_err; ++li) {
            int b, hkv;
            lane_of(li, b, hkv);
            const int old_len = a.old_len[b], pos = a.pos[b];
            if (!debug_check(old_len >= 0 && old_len < a.C, lane == 0 ? a.err : nullptr)) continue;
            const int t = old_len + 1;
            const int lo = a.window > 0 ? max(0, t - a.window) : 0;
            const int r0 = lo & ~(KT - 1);
            const int ntiles = (t - r0 + KT - 1) / KT;
            // The new row (slot old_len), then its TMA reads: generic-proxy writes first.  The
            // lane's queries are loaded with it (one memory latency for both), rotated,
            // scaled and stored as bf16 in the query slot of the stage that takes the lane's
            // first tile: the consumers read them from shared memory once that stage is full,
            // instead of waiting for the loads at the start of every lane.
            uint2 qpk[kLanesMaxG];
            {
                const int64_t src = ((int64_t)b * a.Hkv + hkv) * D + lane * 4;
                const bool slot_ok = debug_check(kv_slot_ok(a.kv, b, old_len), lane == 0 ? a.err : nullptr);
                const int64_t dst = slot_ok ? kv_row(a.kv, b, hkv, old_len) * D + lane * 4 : 0;
                const uint2 kraw = *(const uint2*)(a.k_in + src);
                const uint2 vraw = *(const uint2*)(a.v_in + src);
                uint2 qraw[kLanesMaxG];
#pragma unroll
                for (int g = 0; g < kLanesMaxG; ++g)
                    if (g < G) qraw[g] = *(const uint2*)(a.q_in + ((int64_t)b * a.Hq + hkv * G + g) * D + lane * 4);
                float2 cs[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
                if (a.rope_f) {
                    cs[0] = a.rope_f[(int64_t)pos * (D / 2) + lane * 2];
                    cs[1] = a.rope_f[(int64_t)pos * (D / 2) + lane * 2 + 1];
                }
                const __nv_bfloat16* kin = (const __nv_bfloat16*)&kraw;
                __nv_bfloat16 kout[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float xf = __bfloat162float(kin[2 * e]), yf = __bfloat162float(kin[2 * e + 1]);
                    if (a.rope_f) {
                        const int j = lane * 2 + e;
                        kout[2 * e] = rope_bf16_exact(xf, yf, cs[e].x, cs[e].y, a.rope, pos, D / 2, j, false);
                        kout[2 * e + 1] = rope_bf16_exact(xf, yf, cs[e].x, cs[e].y, a.rope, pos, D / 2, j, true);
                    } else {
                        kout[2 * e] = kin[2 * e];
                        kout[2 * e + 1] = kin[2 * e + 1];
                    }
                }
#pragma unroll
                for (int g = 0; g < kLanesMaxG; ++g) {
                    if (g < G) {
                        const __nv_bfloat16* qin = (const __nv_bfloat16*)&qraw[g];
                        uint32_t w[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float2 x = make_float2(__bfloat162float(qin[2 * e]), __bfloat162float(qin[2 * e + 1]));
                            if (a.rope_f) x = q_rotate(x.x, x.y, cs[e]);
                            w[e] = pack_bf16(x.x * qscale, x.y * qscale);
                        }
                        qpk[g] = make_uint2(w[0], w[1]);
                    }
                }
                if (slot_ok) {
                    *(uint2*)(a.K + dst) = *(const uint2*)kout;
                    *(uint2*)(a.V + dst) = vraw;
                    if (hkv == 0 && lane == 0) a.positions[(int64_t)b * a.C + old_len] = pos;
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            }
            if (a.test_stall) continue;
            // the query slot belongs to the first tile's stage: free once that stage is
            {
                const int s0 = gi % STAGES;
                const bool free_ok =
                    gi < STAGES || __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty[s0]), ((gi / STAGES) - 1) & 1));
                if (!free_ok) {
                    if (lane == 0) {
                        *s_err = 1;
                        atomicOr(a.err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
                    }
                    break;
                }
#pragma unroll
                for (int g = 0; g < kLanesMaxG; ++g)
                    if (g < G) *(uint2*)(Qs + s0 * kLanesQBytes + (g * D + lane * 4) * 2) = qpk[g];
                __syncwarp();
            }
            if (lane == 0) {
                prefetch_tmap(&tmK16);
                prefetch_tmap(&tmV16);
                for (int i = 0; i < ntiles; ++i, ++gi) {
                    const int s = gi % STAGES;
                    if (gi >= STAGES && !mbar_wait_bounded(smem_u32(&empty[s]), ((gi / STAGES) - 1) & 1)) {
                        *s_err = 1;
                        atomicOr(a.err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
                        break;
                    }
                    const int y = (int)kv_row(a.kv, b, hkv, r0 + i * KT);
                    const uint32_t fb = smem_u32(&full[s]);
                    uint8_t* st = smem + s * STAGE_BYTES;
                    const int rows = min(KT, t - (r0 + i * KT));
                    if (rows == KT) {
                        mbar_arrive_expect_tx(fb, STAGE_BYTES);
                        tma_load_2d(smem_u32(st), &tmK, 0, y, fb);
                        tma_load_2d(smem_u32(st + HALF_BYTES), &tmK, 64, y, fb);
                        tma_load_2d(smem_u32(st + TILE_BYTES), &tmV, 0, y, fb);
                        tma_load_2d(smem_u32(st + TILE_BYTES + HALF_BYTES), &tmV, 64, y, fb);
                    } else {
                        // the lane's last, partial tile: only its 16-row boxes that hold keys
                        // (a 16-row box at a 2 KB offset keeps the tile's 128-byte swizzle
                        // phase).  The value rows beyond them are zero-filled by boxes that lie
                        // wholly outside the tensor (row -16): masked keys get probability 0,
                        // and 0 times whatever the shared memory held before could be NaN.
                        // (Key rows there are masked after the product, so they stay as they are.)
                        const int nb = (rows + 15) / 16;
                        mbar_arrive_expect_tx(fb, (uint32_t)(nb * 4 + (4 - nb) * 2) * 16 * 128);
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t o = q * 16 * 128;
                            if (q < nb) {
                                tma_load_2d(smem_u32(st) + o, &tmK16, 0, y + 16 * q, fb);
                                tma_load_2d(smem_u32(st + HALF_BYTES) + o, &tmK16, 64, y + 16 * q, fb);
                                tma_load_2d(smem_u32(st + TILE_BYTES) + o, &tmV16, 0, y + 16 * q, fb);
                                tma_load_2d(smem_u32(st + TILE_BYTES + HALF_BYTES) + o, &tmV16, 64, y + 16 * q, fb);
                            } else {
                                tma_load_2d(smem_u32(st + TILE_BYTES) + o, &tmV16, 0, -16, fb);
                                tma_load_2d(smem_u32(st + TILE_BYTES + HALF_BYTES) + o, &tmV16, 64, -16, fb);
                            }
                        }
                    }
                    issued = gi + 1;
                }
            }
            gi = __shfl_sync(0xffffffffu, gi, 0);
        }
    } else {
        // ---------------- consumers (one 16-row m tile, 16 keys of each stage per warp) ----------------
        const int kofs = warp * 16;
        const int qa = lane >> 2, qc = (lane & 3) * 2;
        int gi = 0;
        for (int li = l_begin; li < l_end; ++li) {
            int b, hkv;
            lane_of(li, b, hkv);
            const int old_len = a.old_len[b];
            if (!(old_len >= 0 && old_len < a.C) && kDebug) continue;
            const int t = old_len + 1;
            const int lo = a.window > 0 ? max(0, t - a.window) : 0;
            const int r0 = lo & ~(KT - 1);
            const int ntiles = (t - r0 + KT - 1) / KT;
            uint32_t qf[8][4];
            float o[16][4];
            float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
            bool ok = true;
            for (int i = 0; i < ntiles; ++i, ++gi) {
                const int s = gi % STAGES;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (gi / STAGES) & 1))) {
                    ok = false;
                    break;
                }
                if (i == 0) {
                    // the lane's queries, written by the producer before it armed this stage
                    const uint32_t* qs = (const uint32_t*)(Qs + s * kLanesQBytes) + qa * (D / 2);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        qf[ks][0] = qa < G ? qs[(ks * 16 + qc) / 2] : 0u;
                        qf[ks][1] = 0u;                      // rows 8 .. 15: beyond G <= 4
                        qf[ks][2] = qa < G ? qs[(ks * 16 + qc + 8) / 2] : 0u;
                        qf[ks][3] = 0u;
                    }
                }
                const uint32_t kt = smem_u32(smem + s * STAGE_BYTES);
                consume_stage<1>(kt, kt + TILE_BYTES, r0 + i * KT + kofs, t, lo, qf, o, m, l, lane, kofs);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            }
            if (!ok) {
                *s_err = 1;
                atomicOr(a.err, (uint32_t)DEV_ERR_WAIT_TIMEOUT);
            }
            // merge the four consumer warps (rows < G), behind the consumers' own barrier
            consumer_bar();
            if (*s_err) break;
            float lr = l[0];
            lr += __shfl_xor_sync(0xffffffffu, lr, 1);
            lr += __shfl_xor_sync(0xffffffffu, lr, 2);
            if (qa < G) {
                float* dst = Om + ((size_t)warp * kLanesMaxG + qa) * D;
#pragma unroll
                for (int n = 0; n < 16; ++n) *(float2*)(dst + n * 8 + qc) = make_float2(o[n][0], o[n][1]);
                if ((lane & 3) == 0) ML[warp * kLanesMaxG + qa] = make_float2(m[0], lr);
            }
            consumer_bar();
            for (int u = threadIdx.x; u < G * D; u += NCW * 32) {
                const int g = u / D, dim = u - g * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < NCW; ++w) M = fmaxf(M, ML[w * kLanesMaxG + g].x);
                float O = 0.f, L = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) {
                    const float2 ml = ML[w * kLanesMaxG + g];
                    const float f = fast_exp2(ml.x - M);
                    O += Om[((size_t)w * kLanesMaxG + g) * D + dim] * f;
                    L += ml.y * f;
                }
                store_out(a, ((int64_t)b * a.Hq + hkv * G + g) * D + dim, O / L);
            }
            if (threadIdx.x == 0 && hkv == 0 && !a.no_commit) {
                a.len_out[b] = old_len + 1;
                a.next_out[b] = a.pos[b] + 1;
            }
            consumer_bar();                          // the buffer is free for the next lane
        }
    }
    __syncthreads();
    if (*s_err && warp == NCW && lane == 0) {
        // let copies already issued land before the CTA's shared memory is released
        for (int i = issued - STAGES < 0 ? 0 : issued - STAGES; i < issued; ++i)
            mbar_wait_bounded(smem_u32(&full[i % STAGES]), (i / STAGES) & 1);
    }
}

// Launch attributes: programmatic stream serialization when a.pdl is set.
struct PdlConfig {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg{};
    PdlConfig(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
    }
};

template <int MT, int MODE>
cudaError_t launch_mt(const DecodeLaunch& a, cudaStream_t s) {
    constexpr int SMEM = smem_bytes<Cfg<MT>::STAGES>();
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        return cudaFuncSetAttribute(decode_bf16_kernel<MT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    });
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_splits, a.B * a.Hkv);
    PdlConfig pc(grid, dim3(THREADS), SMEM, s, a.pdl != 0 && MODE != 2);
    return cudaLaunchKernelEx(&pc.cfg, decode_bf16_kernel<MT, MODE>, *a.tmK, *a.tmV, a);
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeLaunch& a, cudaStream_t s) {
    PdlConfig pc(dim3(a.B * a.Hq), dim3(128), 0, s, a.pdl != 0);
    return cudaLaunchKernelEx(&pc.cfg, decode_combine_kernel, a);
}

int decode_bf16_ctas_per_sm(int group) { return group <= 16 ? Cfg<1>::MINB : Cfg<2>::MINB; }

cudaError_t launch_decode_lanes(const DecodeLaunch& a, cudaStream_t s) {
    constexpr int SMEM = smem_bytes<Cfg<1>::STAGES>() + kLanesMergeBytes + Cfg<1>::STAGES * kLanesQBytes;
    static PerDeviceOnce attr;
    cudaError_t e = attr.run(
        [] { return cudaFuncSetAttribute(decode_lanes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM); });
    if (e != cudaSuccess) return e;
    if (!a.fused || a.dev_len || a.Hq / a.Hkv > kLanesMaxG || a.lanes_per_cta < 1 || a.B > kFusedMaxB)
        return cudaErrorInvalidValue;
    const int ctas = (a.B * a.Hkv + a.lanes_per_cta - 1) / a.lanes_per_cta;
    PdlConfig pc(dim3(ctas), dim3(THREADS), SMEM, s, a.pdl != 0);
    return cudaLaunchKernelEx(&pc.cfg, decode_lanes_kernel, *a.tmK, *a.tmV, *a.tmK16, *a.tmV16, a);
}

cudaError_t launch_decode_bf16(const DecodeLaunch& a, cudaStream_t s) {
    const int G = a.Hq / a.Hkv;
    if (a.fused && a.B > kFusedMaxB) return cudaErrorInvalidValue;
    const int mode = a.fused ? (a.dev_len ? 2 : 1) : 0;
    if (G <= 16) return mode == 2 ? launch_mt<1, 2>(a, s) : mode == 1 ? launch_mt<1, 1>(a, s) : launch_mt<1, 0>(a, s);
    if (G <= 32) return mode == 2 ? launch_mt<2, 2>(a, s) : mode == 1 ? launch_mt<2, 1>(a, s) : launch_mt<2, 0>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace kvc
