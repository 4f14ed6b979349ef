/*
 * kvc.h -- C ABI of libkvc: cached incremental causal attention with RoPE on
 * one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section (or listing title):
 *   [Ch37] "Keep the prefix, project only the new row", learn_llm course,
 *          chapter 37 (intale.github.io/learn_llm/en/course/37-incremental-attention/)
 *   [LCP5] "LLM 机制实验（五）：改了历史，能否只重算变化的后缀？"
 *          (huhohoo.com/docs/llm/longest-prefix-reuse)
 *
 * Model.  A handle owns, for every layer, fixed-capacity key and value
 * buffers laid out [B, H_kv, C, d_h] in the storage dtype, a per-slot position
 * array [B, C] (int32), and per-sequence logical length and next position
 * (int32 [B]).  Rows are appended along the slot axis ([Ch37] "Append along
 * the position axis"); the key is stored rotated (RoPE at its absolute
 * position), the value unrotated, the query is never stored.
 *
 * Conventions shared by every entry point:
 *   - Device memory.  Tensor data pointers passed in kvc_tensor are DEVICE
 *     pointers (cudaMalloc / torch CUDA tensors), contiguous row-major, owned
 *     by the caller and only read (inputs) or written (outputs) during the
 *     call's stream work.  The handle owns its cache storage and scratch.
 *   - Host memory.  Plain int32_t* arguments (cut, start_pos, seqlen, ids,
 *     lengths) are HOST pointers, read before the call returns.
 *   - Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).  Work is enqueued asynchronously; calls on one handle
 *     must be issued from one host thread and in stream order.
 *   - Errors.  Every argument, shape, dtype, capacity and position check runs
 *     on the host, against host mirrors of the lengths, BEFORE any work is
 *     enqueued; a call that returns an error has changed neither storage nor
 *     lengths ([Ch37] "Reset or reject without corrupting retained state").
 *     kvc_last_error() gives the message of the handle's last failure.
 *   - Dtypes.  Inputs q, k, v carry the storage dtype.  Outputs are f32 for
 *     bf16 and f32 storage and f64 for f64 storage.
 */
#ifndef KVC_H
#define KVC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 5

typedef enum kvc_status {
    KVC_OK = 0,
    KVC_ERR_NULL = 1,                       /* a required pointer is NULL */
    KVC_ERR_ZERO_BATCH = 2,                 /* batch size 0 */
    KVC_ERR_ZERO_CAPACITY = 3,              /* capacity 0 */
    KVC_ERR_CAPACITY_EXCEEDS_POSITIONS = 4, /* capacity > RoPE position capacity */
    KVC_ERR_ELEMENT_OVERFLOW = 5,           /* B*H*C*d_h (or a byte count) overflows */
    KVC_ERR_ALLOC = 6,                      /* device allocation failed */
    KVC_ERR_FULL = 7,                       /* an append would pass capacity C */
    KVC_ERR_KEY_SHAPE = 8,                  /* key tensor shape / rank mismatch */
    KVC_ERR_VALUE_SHAPE = 9,                /* value tensor shape / rank mismatch */
    KVC_ERR_QUERY_SHAPE = 10,               /* query shape mismatch, or not a single token */
    KVC_ERR_OUTPUT_SHAPE = 11,              /* output shape mismatch */
    KVC_ERR_DTYPE = 12,                     /* tensor dtype differs from the handle's */
    KVC_ERR_LAYER = 13,                     /* layer index out of range */
    KVC_ERR_NONFINITE_KEY = 14,             /* checked mode: NaN/Inf in the appended key */
    KVC_ERR_NONFINITE_VALUE = 15,           /* checked mode: NaN/Inf in the appended value */
    KVC_ERR_CUT = 16,                       /* cut < 0 or cut > current length */
    KVC_ERR_EMPTY_QUERY = 17,               /* empty token-id query */
    KVC_ERR_POSITION = 18,                  /* a RoPE position outside [0, max_positions) */
    KVC_ERR_CONFIG = 19,                    /* invalid geometry or option */
    KVC_ERR_CUDA = 20,                      /* a CUDA runtime call failed (no device, ...) */
    KVC_ERR_DEVICE = 21,                    /* a kernel reported a fault or a timed-out wait */
    KVC_ERR_TICKET = 22                     /* a prepared-step ticket no longer matches its cache */
} kvc_status;

typedef enum kvc_dtype {
    KVC_BF16 = 0,
    KVC_F32 = 1,
    KVC_F64 = 2
} kvc_dtype;

/* Geometry and numerics of a cache ([Ch37] "Keep layer, logical length, and
 * capacity separate"; the RoPE configuration is captured at construction as in
 * the listing "Own a fixed layer-bound cache, append one checked row, and
 * reset logical length"). */
typedef struct kvc_config {
    int32_t batch;              /* B >= 1 sequences */
    int32_t heads_q;            /* H_q >= 1 query heads */
    int32_t heads_kv;           /* H_kv >= 1 key/value heads, divides H_q (query head h reads h / (H_q/H_kv)) */
    int32_t capacity;           /* C >= 1 slots per sequence and layer */
    int32_t head_dim;           /* d_h, even, 2 .. 256 */
    int32_t layers;             /* >= 1 independent layer caches */
    int32_t dtype;              /* kvc_dtype of storage and of q/k/v inputs */
    int32_t rope_max_positions; /* RoPE table size; 0 means C; must be >= C */
    double rope_base;           /* > 0: theta_j = base^(-2j/d_h); 0: no rotation */
    int32_t checked;            /* nonzero: reject NaN/Inf keys and values (adds a device sync per call) */
    int32_t device;             /* CUDA device ordinal */
    int32_t window;             /* 0: full causal attention; W >= 1: sliding window -- the row at
                                   slot s attends slots s - W + 1 .. s only ([LCP5] "为什么滑窗部分
                                   命中必须回退"); storage keeps every row up to C */
    int32_t block_rows;         /* 0: contiguous [B, H_kv, C, d_h] storage per layer.  P > 0 (a
                                   power of two >= 64): paged storage -- each layer holds a pool of
                                   blocks [blocks, H_kv, P, d_h] and one block table [B][ceil(C/P)]
                                   (shared by all layers) maps each sequence's logical blocks to
                                   physical ones; blocks are taken from the pool as rows are
                                   appended, returned by truncate/reset, and can be shared between
                                   sequences (kvc_share_prefix, copy-on-write) */
    int32_t blocks;             /* paged: physical blocks per layer pool; 0 means B * ceil(C/P) */
} kvc_config;

/* A contiguous row-major tensor on the device.  ndim <= 4. */
typedef struct kvc_tensor {
    void* data;
    int32_t dtype;              /* kvc_dtype */
    int32_t ndim;
    int64_t shape[4];
} kvc_tensor;

/* A prepared decode step of one layer (kvc_prepare_attend), committed by
 * kvc_commit.  Plain data owned by the caller; only the library writes it. */
typedef struct kvc_ticket {
    const void* handle;   /* the handle that prepared it */
    int32_t layer;
    int32_t reserved;
    uint64_t version;     /* the layer's state version when it was prepared */
} kvc_ticket;

typedef struct kvc_handle kvc_handle;

/* ABI version of the loaded library (KVC_ABI_VERSION). */
int32_t kvc_abi_version(void);

/* Static text for a status code. */
const char* kvc_status_string(kvc_status status);

/* Message of the last failed call on `h` (empty string if none).  With h ==
 * NULL: the last failure of kvc_create / kvc_create_ex on this thread. */
const char* kvc_last_error(const kvc_handle* h);

/*
 * kvc_create: a cache with H_q = H_kv = heads, bf16 storage, RoPE base 10000,
 * rope_max_positions = capacity, unchecked, device 0.
 * kvc_create_ex: any configuration.
 * [Ch37] listing "Own a fixed layer-bound cache, append one checked row, and
 * reset logical length" (construction): batch 0 -> KVC_ERR_ZERO_BATCH,
 * capacity 0 -> KVC_ERR_ZERO_CAPACITY, capacity > rope_max_positions ->
 * KVC_ERR_CAPACITY_EXCEEDS_POSITIONS, element-count overflow ->
 * KVC_ERR_ELEMENT_OVERFLOW, device allocation failure -> KVC_ERR_ALLOC.
 * Storage is zero-filled; every length and next position starts at 0.  On
 * success *out owns all device memory until kvc_destroy.  On failure *out is
 * set to NULL and nothing is allocated.
 */
kvc_status kvc_create(int32_t batch, int32_t heads, int32_t capacity, int32_t head_dim,
                      int32_t layers, kvc_handle** out);
kvc_status kvc_create_ex(const kvc_config* config, kvc_handle** out);

/* Frees every device and host resource of `h` (NULL is a no-op).  The caller
 * must ensure no enqueued work on the handle is still running. */
void kvc_destroy(kvc_handle* h);

/*
 * One decode step of one layer for all B sequences ([Ch37] "Predict the third
 * result before running the example", "Append along the position axis" and the
 * listing "Evaluate one newest query across the retained rows plus the
 * candidate key/value row before committing the append").
 *   q   [B, H_q, 1, d_h]   the new query rows (unrotated), storage dtype
 *   k   [B, H_kv, 1, d_h]  the new key rows (unrotated)
 *   v   [B, H_kv, 1, d_h]  the new value rows
 *   out [B, H_q, 1, d_h]   f32 (bf16/f32 storage) or f64 (f64 storage); with bf16
 *                          storage and d_h = 128 (the tensor-core decode path) also
 *                          bf16, each element rounded once from the float32 result
 * For each sequence b with old length n_b and next position p_b (p_b == n_b
 * except after a deliberately stale prefill): q and k are rotated at p_b; the
 * rotated key (rounded once to the storage dtype) and the value are written to
 * slot n_b, positions[b][n_b] = p_b; the new query of every head attends slots
 * 0 .. n_b with scores q.k/sqrt(d_h) and a max-subtracted softmax; then
 * n_b += 1 and p_b += 1.
 * Errors (no state change): KVC_ERR_LAYER, KVC_ERR_NULL, KVC_ERR_DTYPE,
 * KVC_ERR_QUERY_SHAPE (including more than one token), KVC_ERR_KEY_SHAPE,
 * KVC_ERR_VALUE_SHAPE, KVC_ERR_OUTPUT_SHAPE, KVC_ERR_FULL (some n_b == C, or a
 * paged pool without the free blocks the step needs),
 * KVC_ERR_POSITION (some p_b >= rope_max_positions), and in checked mode
 * KVC_ERR_NONFINITE_KEY / KVC_ERR_NONFINITE_VALUE.
 * With KVC_OPT_DEVICE_LENGTHS on, the length and position checks run on the
 * device instead (see that option) and KVC_ERR_CONFIG is returned when the
 * cache is not bf16 with d_h = 128 or holds more than 256 sequences.
 */
kvc_status kvc_append_attend(kvc_handle* h, int32_t layer, const kvc_tensor* q,
                             const kvc_tensor* k, const kvc_tensor* v,
                             const kvc_tensor* out, void* stream);

/*
 * The same step without its commit ([Ch37] listing "Evaluate one newest query
 * across the retained rows plus the candidate key/value row before committing
 * the append": the prepared result carries its candidate rows and the length it
 * expects; chapter 38, as that listing's comment announces, prepares one such
 * ticket per decoder block, finishes the model, checks that every ticket still
 * targets its cache and only then commits the whole stack).  Arguments,
 * checks and errors as kvc_append_attend; `out` receives the attention output
 * over the retained rows plus the candidate row.  The rotated key and the value
 * are staged in slot n_b -- beyond the logical length, so no call sees them --
 * and the length and next position stay unchanged until kvc_commit.
 * *ticket (caller-owned) records the layer and its state version.  Any later
 * change of the layer (an append, prepare, prefill, truncate, reset or commit
 * of it) makes the ticket stale.  Not available with KVC_OPT_DEVICE_LENGTHS
 * (KVC_ERR_CONFIG).
 */
kvc_status kvc_prepare_attend(kvc_handle* h, int32_t layer, const kvc_tensor* q,
                              const kvc_tensor* k, const kvc_tensor* v,
                              const kvc_tensor* out, kvc_ticket* ticket, void* stream);

/*
 * Commits n prepared steps at once: every ticket must come from `h`, name a
 * distinct layer and still match that layer's state version; then every
 * named layer's lengths and next positions advance by one, all in one
 * enqueued launch.  KVC_ERR_TICKET (nothing committed) when a ticket is
 * stale, foreign or repeats a layer; KVC_ERR_NULL for a NULL array with n > 0.
 * n == 0 commits nothing.  Dropping a ticket discards its step (the staged
 * rows stay beyond the length).
 */
kvc_status kvc_commit(kvc_handle* h, const kvc_ticket* tickets, int32_t n, void* stream);

/*
 * Append a chunk of rows per sequence and attend it causally against the
 * retained prefix plus the chunk ([LCP5] section "先看一次历史编辑": with the
 * same configuration and positions the prefix rows do not depend on later
 * tokens; listing under "哪些东西必须一起裁剪": continue from position cut).
 *   q   [B, H_q, S, d_h], k and v [B, H_kv, S, d_h]: row i < seqlen[b] of
 *       sequence b is new row i; rows >= seqlen[b] are ignored (padding).
 *       q may be NULL when out is NULL (append only).
 *   start_pos [B] host: position of row 0 (NULL -> each sequence's next
 *       position, the normal path; a different value is accepted and recorded,
 *       which is how a stale-position negative control is run).
 *   seqlen [B] host: rows per sequence, 0 .. S (NULL -> S for all).
 *   out [B, H_q, S, d_h] f32/f64, or NULL to append without attending
 *       (prefill of a prefix).  Rows >= seqlen[b] of out are left untouched.
 * Row i of sequence b goes to slot n_b + i with position start_pos[b] + i;
 * its query attends slots 0 .. n_b + i (the mask is by slot).  Afterwards
 * n_b += seqlen[b] and p_b = start_pos[b] + seqlen[b].
 * Errors as kvc_append_attend, plus KVC_ERR_FULL when n_b + seqlen[b] > C and
 * KVC_ERR_POSITION when a position leaves [0, rope_max_positions).
 */
kvc_status kvc_prefill_suffix(kvc_handle* h, int32_t layer, const kvc_tensor* q,
                              const kvc_tensor* k, const kvc_tensor* v,
                              const int32_t* start_pos, const int32_t* seqlen,
                              const kvc_tensor* out, void* stream);

/*
 * kvc_prefill_suffix with q, k, v and out in HOST memory (page-locked memory
 * lets the copies overlap the work; pageable memory works, without overlap).
 * Same arguments, layouts, results and errors as kvc_prefill_suffix, plus:
 *   chunk_sequences: sequences per pipeline stage (0 -> ceil(B / 8)); the stages take
 *                    the sequences smallest first, the second smallest last and the
 *                    others largest first (by seqlen), so that the first upload and the
 *                    last download are short.
 * Every check of the whole call (shapes, dtypes, capacity, positions, storage
 * blocks; in checked mode the finiteness of k and v, scanned on the host) runs
 * before any copy or launch; an error leaves the state unchanged.  The call
 * then copies rows 0 .. seqlen[b]-1 of each head of each sequence into device
 * staging owned by the handle, stage by stage, on an internal upload stream;
 * runs each stage's append and attention on `stream` as soon as its rows have
 * landed (the other sequences take 0 rows); and copies each stage's output rows
 * back on an internal download stream, so that the copies of one stage overlap
 * the work of another.  The call returns once everything is enqueued; `stream`
 * completes after the last output row is in host memory, and the host buffers
 * must stay valid and unchanged until then.  The results equal those of
 * kvc_prefill_suffix on the same inputs bit for bit.  Rows >= seqlen[b] of out
 * are left untouched.  KVC_ERR_CONFIG if a pointer is device memory;
 * KVC_ERR_ALLOC if the staging (the size of q, k, v and out) cannot be allocated.
 */
kvc_status kvc_prefill_suffix_host(kvc_handle* h, int32_t layer, const kvc_tensor* q,
                                   const kvc_tensor* k, const kvc_tensor* v,
                                   const int32_t* start_pos, const int32_t* seqlen,
                                   const kvc_tensor* out, int32_t chunk_sequences,
                                   void* stream);

/*
 * [Ch37] "Keep layer, logical length, and capacity separate" / "Reset or reject
 * without corrupting retained state": every layer's length and next position
 * become 0.  Storage, positions, capacity and allocation are unchanged.  A
 * device error recorded by an earlier call is cleared.
 */
kvc_status kvc_reset(kvc_handle* h, void* stream);

/*
 * [LCP5] listing under "哪些东西必须一起裁剪": for every layer and sequence b,
 * keep rows < cut[b] and set length = next position = cut[b].
 * cut [B] host.  KVC_ERR_CUT (no state change) if some cut[b] < 0 or
 * cut[b] > the current length of sequence b in any layer.  With
 * KVC_OPT_DEVICE_LENGTHS on, the second check runs on the device without a
 * synchronisation: a cut beyond a length then changes nothing and sets bit 16
 * of the device error word (kvc_check reports KVC_ERR_DEVICE).
 */
kvc_status kvc_truncate(kvc_handle* h, const int32_t* cut, void* stream);

/*
 * [LCP5] "先看一次历史编辑" and "查询流程与缓存所有权": cut = min(L, m - 1),
 * L the length of the run of equal ids from index 0 of cached[0..n) and
 * query[0..m).  Host only, no device.  n == 0 gives cut 0; m <= 0 ->
 * KVC_ERR_EMPTY_QUERY; NULL arrays (with a non-zero length) -> KVC_ERR_NULL.
 */
kvc_status kvc_lcp(const int32_t* cached, int64_t n, const int32_t* query, int64_t m,
                   int32_t* cut);

/*
 * [LCP5] "为什么滑窗部分命中必须回退": the cut for a sliding-window cache.  A
 * window cache has lost the early rows of its history, so only a full match of
 * the cached ids with a query that continues past them reuses it (cut = n);
 * every other case recomputes (cut = 0).  window == 0 gives kvc_lcp.  Host
 * only; errors as kvc_lcp, plus KVC_ERR_CONFIG for window < 0.
 */
kvc_status kvc_lcp_window(const int32_t* cached, int64_t n, const int32_t* query, int64_t m,
                          int32_t window, int32_t* cut);

/* Host mirrors of one layer's lengths and next positions, each [B] host
 * (either may be NULL).  After device-length decode steps (KVC_OPT_DEVICE_LENGTHS)
 * the mirrors lag behind until kvc_sync_lengths, kvc_check, kvc_truncate or
 * kvc_prefill_suffix reads the device lengths back. */
kvc_status kvc_get_lengths(const kvc_handle* h, int32_t layer, int32_t* lengths,
                           int32_t* next_positions);

/* The host mirror of one layer's logical lengths, [B] host ([Ch37] listing "Own a
 * fixed layer-bound cache, append one checked row, and reset logical length":
 * len()).  The same as kvc_get_lengths without the next positions; after
 * device-length decode steps call kvc_sync_lengths first.  KVC_ERR_NULL for a
 * NULL handle or array, KVC_ERR_LAYER for a layer out of range. */
kvc_status kvc_get_len(const kvc_handle* h, int32_t layer, int32_t* len_B);

/*
 * Logical snapshot of one layer ([Ch37] listing "Own a fixed layer-bound cache,
 * append one checked row, and reset logical length": keys() and values() copy
 * out the retained rows [B, H, len, d_h], never the unused capacity).
 *   keys, values  [B, H_kv, R, d_h] DEVICE tensors of the storage dtype,
 *                 1 <= R <= C, caller-owned; either may be NULL (not both)
 *   positions     [B, R] int32 DEVICE pointer, or NULL
 * Row r of sequence b receives stored row r (the rotated key, the value, the
 * recorded position) when r < length[b], gathered through the block table for
 * paged storage; rows r >= length[b] receive zeros and position -1.  The
 * lengths are the device lengths at the point of `stream` where the copy runs,
 * so the snapshot follows every earlier call on that stream (device-length
 * steps included).  Enqueued on `stream`; the storage is only read.  Errors (no
 * work enqueued): KVC_ERR_NULL, KVC_ERR_LAYER, KVC_ERR_DTYPE, KVC_ERR_KEY_SHAPE /
 * KVC_ERR_VALUE_SHAPE (shape, or R outside [1, C]), KVC_ERR_CONFIG (a pointer
 * that is not device memory of the handle's GPU, or misaligned).
 */
kvc_status kvc_read_rows(kvc_handle* h, int32_t layer, const kvc_tensor* keys, const kvc_tensor* values,
                         int32_t* positions, void* stream);

/* Waits for all work on the handle's device, then copies every layer's device
 * lengths and next positions into the host mirrors.  No other effect. */
kvc_status kvc_sync_lengths(kvc_handle* h);

/*
 * Paged storage ([LCP5] "这一轮留下的工程判断": blocked storage as the next step of
 * prefix reuse; section "查询流程与缓存所有权", step 4 keeps the reusable rows of a
 * cached entry and computes only the rest).  Sequence `dst` (empty in every
 * layer) takes the first `rows` rows of sequence `src` (rows <= src's length
 * in every layer) in every layer by sharing src's blocks -- no copy; a shared
 * block is copied only when either sequence later writes into it.  dst's
 * positions are copied from src; its length and next position become `rows`.
 * KVC_ERR_CONFIG for contiguous storage or dst == src; KVC_ERR_CUT when dst
 * is not empty or rows exceeds src's length; no state change on error.
 */
kvc_status kvc_share_prefix(kvc_handle* h, int32_t dst, int32_t src, int32_t rows, void* stream);

/*
 * Paged storage: the host copy of the block table, [B][ceil(C/P)] physical
 * block ids (-1: no block), and the number of unused blocks in the pool.
 * Either pointer may be NULL.  KVC_ERR_CONFIG for contiguous storage.
 */
kvc_status kvc_block_table(const kvc_handle* h, int32_t* table, int32_t* free_blocks);

/* The handle's configuration (rope_max_positions resolved). */
kvc_status kvc_get_config(const kvc_handle* h, kvc_config* out);

/* Device pointers of one layer's storage, for audits: keys and values
 * [B, H_kv, C, d_h] storage dtype (paged: the pool [blocks, H_kv, P, d_h]),
 * positions [B, C] int32.  Owned by the handle; valid until kvc_destroy.  Any
 * output pointer may be NULL. */
kvc_status kvc_storage(const kvc_handle* h, int32_t layer, void** keys, void** values,
                       int32_t** positions);

/*
 * Synchronises `stream`, then checks the device side: the kernels' error word
 * (bits: 1 an append slot or position out of range, 2 a bounded wait that gave
 * up, 4 tensor memory, 8 a rejected device-length step, 16 a device-checked cut
 * beyond a length, 32 a debug-build bounds check that skipped an access) and that the device
 * lengths and next positions equal the host mirrors.  KVC_ERR_DEVICE on any
 * difference (message names it), KVC_ERR_CUDA if the synchronisation fails.
 * A reported error word is cleared (while it is set, kernels stop early).
 */
kvc_status kvc_check(kvc_handle* h, void* stream);

/*
 * Decode attention that allocates nothing.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot let a library call
 * cudaMalloc -- a serving engine that owns all device memory through its own
 * arena (so a request never fails halfway on an out-of-memory error and no
 * allocation synchronises the device under running streams), or a host
 * framework that hands out only buffers it created.  It runs the split-K
 * decode kernel of kvc_append_attend over a cache the caller owns, with the
 * kernel's scratch in one static 8 MiB device array of the library (held on
 * every GPU that loads the library until the process exits).
 *   keys, values [B, H_kv, C, 128] bf16 device: rotated keys and values
 *   q_rot        [B, H_q, 128] f32 device: the new queries, already rotated
 *   lengths      [B] HOST int32: rows 0 .. lengths[b]-1 of sequence b are
 *                attended (1 <= lengths[b] <= C)
 *   out          [B, H_q, 128] f32 device
 * bf16 storage and d_h = 128 only; H_q / H_kv <= 32; B <= 4096 and
 * B * H_q <= 16099 (what the array holds) -- larger sizes return
 * KVC_ERR_CONFIG, lengths outside [1, C] KVC_ERR_FULL, NULL pointers
 * KVC_ERR_NULL, a failed CUDA call KVC_ERR_CUDA.  Runs on the current device.
 * The first call on a device resolves the array's device address there (make
 * it before any stream capture).  Every call shares the array and it keeps the
 * last call's contents; calls that overlap on the GPU race on it, so order
 * them on one stream.
 */
kvc_status kvc_decode_attend_noalloc(const void* keys, const void* values, const float* q_rot,
                                     const int32_t* lengths, float* out, int32_t batch, int32_t heads_q,
                                     int32_t heads_kv, int32_t capacity, void* stream);

/*
 * Device-side status of kvc_decode_attend_noalloc on the current device (no
 * page counterpart, like that call).  Synchronises `stream`, reads the error
 * word in the static array and clears it: KVC_ERR_DEVICE when some call since
 * the last check had a bounded wait give up (its `out` is then undefined),
 * KVC_OK otherwise (also before any call on this device), KVC_ERR_CUDA if the
 * synchronisation or the read fails.  Allocates nothing.  A wait that gives up
 * cannot be seen from the call that launched it (the call returns before the
 * kernel runs), so callers check after the steps whose outputs they consume.
 */
kvc_status kvc_noalloc_check(void* stream);

/* Tuning / test options (kvc_set_option). */
typedef enum kvc_option {
    KVC_OPT_DECODE_SPLIT_ROWS = 1, /* key rows per decode split (multiple of 64); 0 = automatic */
    KVC_OPT_FORCE_GENERIC = 2,     /* 1 = use the dtype-generic CUDA-core kernels even for bf16, d_h = 128 */
    KVC_OPT_SUFFIX_KERNEL = 3,     /* 0 = automatic, 1 = generic, 2 = tensor-core tile kernel, 3 = the tile
                                      kernel on pairs of SMs, 4 = the persistent tile kernel (one CTA per
                                      SM walking the work items; 3 and 4 need contiguous storage, else 2),
                                      5 = the tile kernel with two softmax threads per query row */
    KVC_OPT_TIMING = 4,            /* 1 = record a CUDA event pair around every kernel launch */
    KVC_OPT_DECODE_FUSED = 5,      /* 1 (default) = bf16 decode steps with B <= 256 append, attend and
                                      commit in one launch (plus a merge launch when H_q / H_kv > 16);
                                      0 = separate append, attend, merge and commit kernels */
    KVC_OPT_TEST_STALL = 6,        /* test only, applies to the next bf16 d_h = 128 decode step: its producer
                                      issues no loads, so the consumers' bounded waits give up (about 1 s)
                                      and the step reports a device error through kvc_check; the step's
                                      outputs are undefined and the cache should then be reset.  With a
                                      NULL handle it applies to the next kvc_decode_attend_noalloc call
                                      instead (reported by kvc_noalloc_check) */
    KVC_OPT_DEVICE_LENGTHS = 7,    /* 1 = decode steps read the lengths and next positions from device memory
                                      instead of the host mirrors, so that the launches of a step do not
                                      depend on them and can be captured in a CUDA graph and replayed:
                                      kvc_append_attend then enqueues one launch (two with more than 16
                                      query heads per key/value head), makes no synchronising call and
                                      no host length check.  The kernel checks every sequence of the layer
                                      first; if one is full or would rotate beyond the table it changes
                                      nothing and sets bit 8 of the device error word (kvc_check reports
                                      KVC_ERR_DEVICE).  The split count is fixed at the call (from the
                                      lengths last read back) and serves every later length.  Make one
                                      uncaptured call per layer before capturing, so that the split
                                      scratch is allocated outside the capture.  kvc_truncate then checks
                                      its cuts on the device too.  Changing the option, and
                                      kvc_prefill_suffix and kvc_check while it is on, synchronise the
                                      device and read the lengths back.  Paged storage cannot use it
                                      (blocks are taken on the host as rows are appended):
                                      KVC_ERR_CONFIG. */
    KVC_OPT_DECODE_PDL = 8,        /* 1 (default) = bf16 d_h = 128 decode and merge kernels are launched as
                                      programmatic dependents of the previous kernel in the stream (each
                                      CTA waits for it before touching global memory), so that a step's
                                      CTAs take the slots the previous step frees as it drains; 0 = plain
                                      launches.  Never used while the stream captures a graph or with
                                      KVC_OPT_DEVICE_LENGTHS. */
    KVC_OPT_TEST_POISON = 9,       /* test only: value 1 synchronises the device and fills every stored row
                                      that no sequence holds -- slots at or past a sequence's length
                                      (paged: past the held rows of a block, and every free block) -- in
                                      every layer with a large finite poison: keys 0, values 1e4 (9984 in
                                      bf16), so that a kernel reading a row it must not moves its output
                                      by about 1e4 / t.  Lengths and held rows are unchanged; a prepared,
                                      uncommitted step's staged row is overwritten.  0 does nothing. */
    KVC_OPT_TEST_PLANT_LENGTH = 10, /* test only, debug builds (libkvc_debug.so, compiled with KVC_DEBUG)
                                      only, else KVC_ERR_CONFIG: synchronises the device and writes `value`
                                      into the DEVICE length and next position of layer 0, sequence 0,
                                      leaving the host mirror alone -- a state the host checks never
                                      produce -- so that the debug build's device bounds checks can be
                                      seen to record KVC_ERR_DEVICE bit 32 and skip the access.  Reset
                                      the cache afterwards. */
    KVC_OPT_DECODE_TC = 11,        /* 1 (default) = decode steps with more than 16 (up to 32) query heads per
                                      key/value head run on the tensor-core decode kernel (tcgen05, the
                                      heads as rows of a 128-row query tile, S and O in tensor memory)
                                      when the step is fused, its lengths are host-held and the storage is
                                      contiguous; 0 = the m16n8k16 decode kernel for every group size */
    KVC_OPT_DECODE_LANES = 12,     /* 1 (default) = fused decode steps over many short lanes (every key span
                                      at most 512 rows, at least four waves of lanes, at most 4 query heads
                                      per key/value head) run with CTAs that walk several lanes each,
                                      longest sequences first; 0 = one CTA per lane and split */
    KVC_OPT_DECODE_STREAMK = 13    /* 1 (default) = tensor-core decode steps (see KVC_OPT_DECODE_TC) with at
                                      most 256 lanes (B x H_kv) run as one wave of CTAs, one per SM, each
                                      over an equal run of 128-key tiles of the lanes laid end to end (a
                                      CTA's run may span lanes; a lane's partials are merged after);
                                      0 = per-sequence pieces, about two waves, largest first */
} kvc_option;

kvc_status kvc_set_option(kvc_handle* h, int32_t option, int64_t value);

/* Kernel families counted by kvc_kernel_stats. */
typedef enum kvc_kernel {
    KVC_KERNEL_ROPE_APPEND = 0,     /* fused RoPE + key/value append */
    KVC_KERNEL_DECODE = 1,          /* split-K decode attention (bf16, d_h = 128) */
    KVC_KERNEL_DECODE_COMBINE = 2,  /* log-sum-exp merge of decode splits */
    KVC_KERNEL_SUFFIX = 3,          /* tensor-core suffix-chunk attention */
    KVC_KERNEL_GENERIC_ATTEND = 4,  /* dtype-generic attention */
    KVC_KERNEL_BOOKKEEPING = 5,     /* commit, truncate, finiteness check */
    KVC_KERNEL_COUNT = 6
} kvc_kernel;

/*
 * Launch count and (with KVC_OPT_TIMING on) summed device time in ms of one
 * kernel family since the handle was created or kvc_reset_stats was called;
 * kernel = -1 sums every family.  Reading the time synchronises on the
 * recorded events.  Either output pointer may be NULL.
 */
kvc_status kvc_kernel_stats(kvc_handle* h, int32_t kernel, double* total_ms, int64_t* launches);
kvc_status kvc_reset_stats(kvc_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
