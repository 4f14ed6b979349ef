// Internal state of a kvc handle and the launchers of its kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <vector>

#include "../../include/kvc.h"

namespace kvc {

// Where the stored row of (sequence b, key/value head h, slot) lives in a layer's
// key (or value) array, in rows of d_h elements.  Contiguous storage is
// [B][H_kv][C] rows; paged storage is a pool of blocks of P rows, [blocks][H_kv][P],
// with table[b][slot / P] naming the physical block of each logical block.
struct KvLayout {
    const int32_t* table;   // null: contiguous; else [B][nblk] physical block ids (device)
    int nblk;               // logical blocks per sequence: ceil(C / P)
    int P;                  // rows per block: a power of two >= 64
    int shift;              // log2(P)
    int C, Hkv;
    int nblocks;            // paged: physical blocks in the pool (debug-build checks)
};

// Debug builds: the stored row of (b, slot) exists -- slot inside the capacity and,
// for paged storage, a valid block behind it.
__host__ __device__ inline bool kv_slot_ok(const KvLayout& L, int b, int slot) {
    if (slot < 0 || slot >= L.C) return false;
    if (!L.table) return true;
    const int blk = L.table[(int64_t)b * L.nblk + (slot >> L.shift)];
    return blk >= 0 && blk < L.nblocks;
}

__host__ __device__ inline int64_t kv_row(const KvLayout& L, int b, int h, int slot) {
    if (!L.table) return ((int64_t)b * L.Hkv + h) * L.C + slot;
    const int blk = L.table[(int64_t)b * L.nblk + (slot >> L.shift)];
    return (((int64_t)blk * L.Hkv + h) << L.shift) + (slot & (L.P - 1));
}

// Host-pinned -> device staging of small per-call argument arrays (start
// positions, chunk lengths, cuts, work lists).  Each slot is reused only after
// the event recorded behind its consumers has completed.
struct ArgRing {
    // enough slots that a caller enqueuing a few steps ahead rarely waits for one
    static constexpr int kSlots = 32;
    void* host[kSlots] = {};
    void* mapped[kSlots] = {};   // device view of host[] (page-locked memory is mapped)
    void* dev[kSlots] = {};
    size_t cap[kSlots] = {};
    cudaEvent_t done[kSlots] = {};
    bool pending[kSlots] = {};
    int next = 0;
    int cur = -1;
    // buffers replaced by larger ones; freed by destroy(), since freeing device memory
    // would wait for the whole device in the middle of a pipeline
    std::vector<void*> retired_host, retired_dev;

    cudaError_t init();
    void destroy();
    // Returns a host staging buffer of at least `bytes` for the next slot.
    cudaError_t acquire(size_t bytes, void** host_ptr);
    // Enqueues the copy of the acquired slot; *dev_ptr is its device copy.
    cudaError_t upload(size_t bytes, cudaStream_t stream, void** dev_ptr);
    // Enqueues the copy of the acquired slot's first `bytes` to device memory `dst`.
    cudaError_t copy(void* dst, size_t bytes, cudaStream_t stream);
    // true: copies run as a small kernel reading the mapped slot (set while bulk copies
    // occupy the host-to-device copy engine), else as copy-engine transfers
    bool by_kernel = false;
    // Records the slot's release behind the work enqueued so far on `stream`.
    cudaError_t release(cudaStream_t stream);
};

struct Handle {
    kvc_config cfg{};
    int max_positions = 0;
    size_t elem_size = 0;       // bytes per storage element
    size_t layer_elems = 0;     // B * H_kv * C * d_h
    void* K = nullptr;          // [L][B][H_kv][C][d_h]
    void* V = nullptr;
    int32_t* positions = nullptr;  // [L][B][C]
    int32_t* len_d = nullptr;      // [L][B]
    int32_t* next_d = nullptr;     // [L][B]
    double2* rope = nullptr;       // [max_positions][d_h/2] (cos, sin), or null when rope_base == 0
    float2* rope_f = nullptr;      // the same table rounded to float32
    uint32_t* err_d = nullptr;     // device error word
    unsigned long long* nonfinite_d = nullptr;  // first non-finite flat index of key [0] and value [1]
    unsigned long long* nonfinite_h = nullptr;  // pinned mirror

    std::vector<int32_t> len_h, next_h;  // host mirrors [L][B]

    // decode scratch
    void* qrot = nullptr;          // [B][H_q][d_h] float (bf16/f32 storage) or double (f64)
    float* part_o = nullptr;       // [B*H_q][splits][d_h]
    float2* part_ml = nullptr;     // [B*H_q][splits] (max in log2 units, sum)
    size_t part_splits = 0;        // splits the partial buffers hold per query head
    // prefill scratch
    void* qrot_chunk = nullptr;    // [B][H_q][S][d_h] rotated queries of a chunk
    size_t qrot_chunk_bytes = 0;
    int* work_counter = nullptr;   // dynamic tile scheduler counter
    // host-buffer prefill (kvc_prefill_suffix_host): device staging of the inputs and
    // the output, the two copy streams and their events
    void* io_buf = nullptr;
    size_t io_bytes = 0;
    cudaStream_t io_h2d = nullptr, io_d2h = nullptr;
    std::vector<cudaEvent_t> io_ev;   // per chunk: inputs landed, results ready
    cudaEvent_t io_entry = nullptr;   // the caller's stream at entry
    cudaEvent_t io_last = nullptr;    // the last output copy of the previous call
    unsigned* lane_ticket = nullptr;  // [B*H_kv] split counters of the fused decode step
    unsigned* step_ticket = nullptr;  // [L] CTA counters of device-length decode steps

    // paged storage (cfg.block_rows > 0): one block table for every layer
    int nblk = 0;                       // logical blocks per sequence
    int nblocks = 0;                    // physical blocks in each layer's pool
    std::vector<int32_t> table_h;       // [B][nblk] physical block or -1
    int32_t* table_d = nullptr;         // device copy
    bool table_dirty = false;           // table_h changed since the last upload
    std::vector<int32_t> refcnt;        // [nblocks] sequences holding each block
    std::vector<int32_t> free_blocks;   // stack of unused blocks

    // TMA descriptors over each layer's keys and values (bf16, d_h = 128):
    // 64-row boxes for decode, 128-row boxes for the suffix-chunk kernel
    std::vector<CUtensorMap> tmap_k, tmap_v, tmap_k128, tmap_v128;
    std::vector<CUtensorMap> tmap_k16, tmap_v16;   // 16-row boxes: the partial last tile of a short lane
    bool have_tmaps = false;

    ArgRing ring;
    std::string last_error;

    // per-family launch counters and optional CUDA-event timing
    struct Timer {
        std::vector<cudaEvent_t> start, stop;
        size_t used = 0;
        double ms = 0;
        int64_t launches = 0;
    } timers[KVC_KERNEL_COUNT];
    bool timing = false;

    // options
    int64_t opt_split_rows = 0;
    int64_t opt_force_generic = 0;
    int64_t opt_suffix_kernel = 0;
    int64_t opt_decode_fused = 1;
    int64_t opt_test_stall = 0;
    int64_t opt_device_lengths = 0;
    int64_t opt_decode_pdl = 1;
    int64_t opt_decode_tc = 1;
    int64_t opt_decode_lanes = 1;
    int64_t opt_decode_streamk = 1;
    std::vector<uint64_t> layer_version;  // [L] bumped by every change of a layer's state or staged slot
    bool mirrors_stale = false;    // device-length steps ran since the mirrors were last read back

    int B() const { return cfg.batch; }
    int Hq() const { return cfg.heads_q; }
    int Hkv() const { return cfg.heads_kv; }
    int C() const { return cfg.capacity; }
    int D() const { return cfg.head_dim; }
    char* K_layer(int l) const { return (char*)K + (size_t)l * layer_elems * elem_size; }
    char* V_layer(int l) const { return (char*)V + (size_t)l * layer_elems * elem_size; }
    int32_t* pos_layer(int l) const { return positions + (size_t)l * cfg.batch * cfg.capacity; }
    int32_t* len_layer(int l) const { return len_d + (size_t)l * cfg.batch; }
    bool paged() const { return cfg.block_rows > 0; }
    KvLayout layout() const {
        KvLayout L{};
        L.table = paged() ? table_d : nullptr;
        L.nblk = nblk;
        L.P = cfg.block_rows;
        L.shift = 0;
        while ((1 << L.shift) < L.P) ++L.shift;
        L.C = cfg.capacity;
        L.Hkv = cfg.heads_kv;
        L.nblocks = nblocks;
        return L;
    }
    int32_t* next_layer(int l) const { return next_d + (size_t)l * cfg.batch; }
};

// One-time set-up of a kernel's attributes, done once per device: a function
// attribute (such as the dynamic shared-memory opt-in) belongs to the context of
// the device that was current when it was set, so a flag shared by the whole
// process would skip the set-up on a second GPU.  Safe to call from several host
// threads: the set-up is idempotent, so two threads may both run it.
class PerDeviceOnce {
public:
    template <typename F>
    cudaError_t run(F setup) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
        if (bit && (done_.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        e = setup();
        if (e == cudaSuccess && bit) done_.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }

private:
    std::atomic<uint64_t> done_{0};
};

// ---- kernel launchers (each returns the launch status) ----------------------

struct AppendLaunch {
    const void* q; const void* k; const void* v;   // [B,H_q,S,d], [B,H_kv,S,d]
    void* K; void* V; int32_t* positions;          // one layer's storage
    const int32_t* slot0;    // [B] device: slot of row 0 (the old length)
    const int32_t* pos0;     // [B] device: position of row 0
    const int32_t* seqlen;   // [B] device, or null: S rows each
    void* qrot;              // [B,H_q,S,d] rotated queries
    int qrot_kind;           // 0 = float, 1 = double, 2 = bf16
    const double2* rope;     // null: no rotation
    const float2* rope_f;    // the same table rounded to float32 (bf16 caches)
    uint32_t* err;
    int B, Hq, Hkv, S, C, d, max_positions;
    KvLayout kv;             // where stored rows live
};
cudaError_t launch_rope_append(int dtype, const AppendLaunch& a, cudaStream_t s);
cudaError_t launch_copy_args(const void* src_mapped, void* dst, size_t bytes, cudaStream_t s);

struct GenericAttendLaunch {
    const void* qrot;        // [B,H_q,S,d] float or double
    const void* K; const void* V;
    const int32_t* slot0;    // [B] device: slot of row 0
    const int32_t* seqlen;   // [B] device or null
    void* out;               // [B,H_q,S,d] float or double
    int B, Hq, Hkv, S, C, d;
    int window;              // 0, or each row attends its `window` most recent slots
    KvLayout kv;
    uint32_t* err;           // device error word (debug-build bounds checks)
};
cudaError_t launch_attend_generic(int dtype, const GenericAttendLaunch& a, cudaStream_t s);

constexpr int kFusedMaxB = 256;   // sequences whose lengths travel as kernel parameters

struct DecodeLaunch {
    const CUtensorMap* tmK; const CUtensorMap* tmV;       // 64-row boxes
    const CUtensorMap* tmK128; const CUtensorMap* tmV128; // 128-row boxes (tensor-core decode)
    const CUtensorMap* tmK16; const CUtensorMap* tmV16;   // 16-row boxes (short lanes' last tiles)
    const float* qrot;       // [B,H_q,128] rotated queries (separate-kernel step)
    const int32_t* len;      // [B] old length: t = len + 1 (separate-kernel step)
    float* part_o; float2* part_ml;
    void* out;               // [B,H_q,128] float, or bf16 when out_bf16
    uint32_t* err;
    int B, Hq, Hkv, C, split_rows, max_splits;
    int out_bf16;
    int window;              // 0, or the query attends only its `window` most recent slots
    KvLayout kv;             // where stored rows live (tiles of 64 rows never cross a block)
    // Fused step (append + attend + split merge + length commit in one launch).
    int fused;
    const __nv_bfloat16* q_in;           // [B,H_q,128] new queries, unrotated
    const __nv_bfloat16* k_in;           // [B,H_kv,128] new keys, unrotated
    const __nv_bfloat16* v_in;           // [B,H_kv,128] new values
    __nv_bfloat16* K; __nv_bfloat16* V;  // the layer's storage
    int32_t* positions;                  // [B][C]
    int32_t* len_out; int32_t* next_out; // device lengths / next positions to commit
    const float2* rope_f; const double2* rope;
    unsigned* lane_ticket;               // [B*H_kv] split counters, zero between launches
    int merge_in_kernel;                 // 1: the last CTA of a lane merges its splits
    int no_commit;                       // 1: a prepared step: leave the lengths to kvc_commit
    int test_stall;                      // test only: the producer issues no loads (waits run out)
    // Device-length step: old lengths and positions are read from len_out /
    // next_out instead of old_len / pos, every sequence uses max_splits splits
    // (rows per split from its own length), and the grid's last CTA to read
    // the lengths commits them.
    int dev_len;
    int pdl;                             // 1: launched as a programmatic dependent of the previous kernel
    unsigned* step_ticket;               // zero between launches
    int max_positions;
    int32_t old_len[kFusedMaxB];         // host mirrors: old length and RoPE position
    int32_t pos[kFusedMaxB];
    // Piece list (tensor-core decode): blockIdx.x enumerates only CTAs with work, sequence
    // by sequence in the order seq_of[0], seq_of[1], ... (largest pieces first, so that
    // the in-order dispatch of CTAs to free SMs balances the load); sequence seq_of[i] owns
    // CTAs item_start[i] .. item_start[i+1]-1: H_kv lanes x its own split count, each
    // split seq_rows[b] key rows.
    int pieces;
    int lanes_per_cta;                   // many-lane short-context step: lanes each CTA walks
    // Stream-K tensor-core decode (streamk = P CTAs, 0 = off): lane l = b H_kv + hkv owns
    // tiles item_start[l] .. item_start[l+1]-1 of streamk_tiles; CTA c takes tiles
    // [c T / P, (c+1) T / P); seq_of[l] is the lane's first CTA, seq_rows[l] its partials.
    int streamk;
    int streamk_tiles;
    int32_t item_start[kFusedMaxB + 1];
    int32_t seq_of[kFusedMaxB];
    int32_t seq_rows[kFusedMaxB];
};
cudaError_t launch_decode_bf16(const DecodeLaunch& a, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeLaunch& a, cudaStream_t s);
// Fused step with many short lanes per CTA (every lane one split, H_q / H_kv <= 4); lanes
// in the order of seq_of (sequences) x key/value heads.
cudaError_t launch_decode_lanes(const DecodeLaunch& a, cudaStream_t s);
// Tensor-core decode (fused step, contiguous storage, 16 < H_q / H_kv <= 32); one CTA per SM.
cudaError_t launch_decode_tc(const DecodeLaunch& a, cudaStream_t s);
// Stream-K form of the tensor-core decode: one wave of a.streamk CTAs.
cudaError_t launch_decode_tck(const DecodeLaunch& a, cudaStream_t s);
int decode_bf16_ctas_per_sm(int group);

cudaError_t launch_commit(int32_t* len, int32_t* next, const int32_t* pos0, const int32_t* seqlen,
                          int uniform_rows, int B, int C, uint32_t* err, cudaStream_t s);
cudaError_t launch_truncate(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B,
                            cudaStream_t s);
constexpr int kCommitMaxLayers = 64;      // layers one commit launch advances
struct CommitLayers { int32_t layer[kCommitMaxLayers]; int n; };
cudaError_t launch_commit_layers(int32_t* len, int32_t* next, const CommitLayers& layers, int B, int C,
                                 uint32_t* err, cudaStream_t s);
cudaError_t launch_truncate_checked(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B,
                                    uint32_t* err, cudaStream_t s);
// Copies whole blocks (src, dst) = pairs[i] of every layer's key and value pool.
cudaError_t launch_copy_blocks(char* K, char* V, size_t layer_bytes, int layers, size_t block_bytes,
                               const int2* pairs, int npairs, cudaStream_t s);
cudaError_t launch_set_lengths(int32_t* len, int32_t* next, int layers, int B, int b, int value, cudaStream_t s);
// Logical rows of one layer into [B, H_kv, R, d] arrays (rows >= len zero, positions -1).
cudaError_t launch_read_rows(const void* K, const void* V, const int32_t* pos, const int32_t* len, const KvLayout& kv,
                             void* Ko, void* Vo, int32_t* Po, int B, int Hkv, int R, int row_bytes, cudaStream_t s);
// Test-only: poison every storage row no sequence holds (keys 0, values vbits).
cudaError_t launch_poison(void* K, void* V, size_t layer_bytes, const int32_t* live, int layers, int groups, int Hkv,
                          int R, int d, int esz, unsigned long long vbits, cudaStream_t s);
// Test-only: the next kvc_decode_attend_noalloc call's producer issues no loads.
void noalloc_arm_test_stall();
cudaError_t launch_nonfinite(int dtype, const void* x, int64_t n, unsigned long long* first,
                             cudaStream_t s);

// Tensor-core suffix-chunk kernel (bf16, d_h = 128).
struct SuffixLaunch {
    CUtensorMap tmQ, tmK, tmV;   // Q: [B*H_q*S, 128] bf16 rotated queries; K/V: one layer
    const int32_t* slot0;        // [B] device, slot of suffix row 0 (= cut)
    const int32_t* seqlen;       // [B] device
    const int4* work;            // tiles: (b, h, q_tile, n_kv_tiles), longest first
    int n_work;
    int* counter;                // zeroed before launch
    float* out;                  // [B,H_q,S,128]
    uint32_t* err;
    int B, Hq, Hkv, S, C;
    int window;                  // 0, or each row attends its `window` most recent slots; the work
                                 // item's key tiles then start at tile (cut + 128 q_tile - window + 1) / 128
    KvLayout kv;                 // paged: K/V tiles load as two 64-row boxes (tmK/tmV 64-row maps)
    float scale_log2;            // log2(e) / sqrt(d_h)
};
// split: softmax threads per query row (1 or 2)
cudaError_t launch_suffix_tc(const SuffixLaunch& a, int grid, cudaStream_t s, int split);
// Persistent form: one CTA per SM (at most n_work) takes work items in list order through
// a global counter (zeroed before the launch); contiguous storage only.
cudaError_t launch_suffix_tcp(const SuffixLaunch& a, int sms, cudaStream_t s);

// Pair-of-SMs tile kernel (cta_group::2): a cluster of two CTAs per work item.
struct SuffixLaunch2 {
    CUtensorMap tmQ;      // rotated queries [B*Hq*S, 128] bf16, 128-row x 64-col boxes
    CUtensorMap tmK64;    // one layer's keys [B*Hkv*C, 128], 64-row x 64-col boxes
    CUtensorMap tmV128;   // one layer's values, 128-row x 64-col boxes
    const int32_t* slot0;
    const int32_t* seqlen;
    const int4* work;     // (b, h, quad of query tiles, weight)
    int n_work;
    float* out;
    uint32_t* err;
    int B, Hq, Hkv, S, C, window;
    float scale_log2;
};

cudaError_t launch_suffix_tc2(const SuffixLaunch2& a, int items, cudaStream_t s);
int suffix_tc_grid(int sms);

}  // namespace kvc
