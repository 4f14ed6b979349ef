// Host side of the kvc C ABI: handle lifetime, argument checks against host
// mirrors of the lengths (every rejection happens before any work is
// enqueued), launch planning and the per-call kernel sequence.
//
// [Ch37] "Keep the prefix, project only the new row": the listing "Own a fixed
// layer-bound cache, append one checked row, and reset logical length" defines
// construction checks (zero batch, zero capacity, capacity beyond the RoPE
// positions, element-count overflow, allocation), the append checks (key and
// value shape, full cache, non-finite rows) and reset; section "Reset or
// reject without corrupting retained state" requires that a rejected call
// changes neither stored rows nor lengths.  [LCP5] adds truncation to a cut
// with next_position = cut and the longest-common-prefix rule.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <limits>
#include <string>
#include <vector>

#include "kvc_internal.h"

using namespace kvc;

struct kvc_handle : public kvc::Handle {};

namespace {

thread_local std::string g_create_error;

std::string vformat(const char* fmt, va_list ap) {
    char buf[1024];
    vsnprintf(buf, sizeof(buf), fmt, ap);
    return std::string(buf);
}

kvc_status fail(kvc_handle* h, kvc_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::string msg = vformat(fmt, ap);
    va_end(ap);
    if (h) h->last_error = msg;
    else g_create_error = msg;
    return st;
}

kvc_status cuda_fail(kvc_handle* h, cudaError_t e, const char* what) {
    return fail(h, KVC_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(e));
}

#define KVC_CUDA(h, call)                                    \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
    } while (0)

size_t dtype_size(int dtype) {
    switch (dtype) {
        case KVC_BF16: return 2;
        case KVC_F32: return 4;
        case KVC_F64: return 8;
    }
    return 0;
}

const char* dtype_name(int dtype) {
    switch (dtype) {
        case KVC_BF16: return "bf16";
        case KVC_F32: return "f32";
        case KVC_F64: return "f64";
    }
    return "?";
}

int out_dtype(int storage) { return storage == KVC_F64 ? KVC_F64 : KVC_F32; }

bool mul_ok(size_t a, size_t b, size_t* out) {
    if (a != 0 && b > std::numeric_limits<size_t>::max() / a) return false;
    *out = a * b;
    return true;
}

std::string shape_str(const int64_t* s, int n) {
    std::string r = "[";
    for (int i = 0; i < n; ++i) {
        if (i) r += ", ";
        r += std::to_string(s[i]);
    }
    return r + "]";
}

// Checks a [B, H, S?, d] tensor.  S < 0 accepts any positive third extent.
kvc_status check_tensor(kvc_handle* h, const kvc_tensor* t, const char* name, kvc_status shape_err,
                        int dtype, int64_t d0, int64_t d1, int64_t d2, int64_t d3) {
    if (!t || !t->data) return fail(h, KVC_ERR_NULL, "%s tensor or its data pointer is NULL", name);
    if (t->dtype != dtype)
        return fail(h, KVC_ERR_DTYPE, "%s has dtype %s, the cache expects %s", name, dtype_name(t->dtype),
                    dtype_name(dtype));
    const int64_t want[4] = {d0, d1, d2, d3};
    bool ok = t->ndim == 4;
    for (int i = 0; ok && i < 4; ++i) ok = want[i] < 0 ? t->shape[i] > 0 : t->shape[i] == want[i];
    if (!ok) {
        int64_t shown[4];
        for (int i = 0; i < 4; ++i) shown[i] = want[i] < 0 ? -1 : want[i];
        return fail(h, shape_err, "%s must have shape %s, got %s", name, shape_str(shown, 4).c_str(),
                    shape_str(t->shape, t->ndim < 0 ? 0 : (t->ndim > 4 ? 4 : t->ndim)).c_str());
    }
    if (((uintptr_t)t->data & 15u) != 0)
        return fail(h, KVC_ERR_CONFIG, "%s data pointer is not 16-byte aligned", name);
    // A host pointer handed to a kernel would fault the device: insist on device memory
    // of the handle's GPU.
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, t->data) != cudaSuccess) {
        cudaGetLastError();
        return fail(h, KVC_ERR_CONFIG, "%s data pointer is not a CUDA allocation", name);
    }
    if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) || attr.device != h->cfg.device)
        return fail(h, KVC_ERR_CONFIG, "%s data must be device memory of GPU %d", name, h->cfg.device);
    return KVC_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2-D bf16 map over `rows` rows of 128 elements, box [box_rows x 64], 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, void* base, uint64_t rows, uint32_t box_rows) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches `fn` (returning cudaError_t) as one kernel of family `id`: counts it
// and, when timing is on, brackets it with a CUDA event pair on its stream.
template <typename F>
cudaError_t timed(kvc_handle* h, int id, cudaStream_t s, F fn) {
    auto& t = h->timers[id];
    t.launches += 1;
    if (!h->timing) return fn();
    if (t.used == t.start.size()) {
        cudaEvent_t a, b;
        cudaError_t e = cudaEventCreate(&a);
        if (e != cudaSuccess) return e;
        e = cudaEventCreate(&b);
        if (e != cudaSuccess) return e;
        t.start.push_back(a);
        t.stop.push_back(b);
    }
    cudaError_t e = cudaEventRecord(t.start[t.used], s);
    if (e != cudaSuccess) return e;
    e = fn();
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(t.stop[t.used], s);
    t.used += 1;
    return e;
}

cudaError_t collect_timer(kvc_handle* h, int id) {
    auto& t = h->timers[id];
    for (size_t i = 0; i < t.used; ++i) {
        cudaError_t e = cudaEventSynchronize(t.stop[i]);
        if (e != cudaSuccess) return e;
        float ms = 0;
        e = cudaEventElapsedTime(&ms, t.start[i], t.stop[i]);
        if (e != cudaSuccess) return e;
        t.ms += ms;
    }
    t.used = 0;
    return cudaSuccess;
}

bool fast_decode_ok(const kvc_handle* h) {
    return h->cfg.dtype == KVC_BF16 && h->cfg.head_dim == 128 && h->have_tmaps && !h->opt_force_generic &&
           h->Hq() / h->Hkv() <= 32;
}

int sm_count(int device) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 152;
    return n;
}

void free_all(kvc_handle* h) {
    cudaFree(h->K);
    cudaFree(h->V);
    cudaFree(h->positions);
    cudaFree(h->len_d);
    cudaFree(h->next_d);
    cudaFree(h->rope);
    cudaFree(h->rope_f);
    cudaFree(h->err_d);
    cudaFree(h->nonfinite_d);
    if (h->nonfinite_h) cudaFreeHost(h->nonfinite_h);
    cudaFree(h->qrot);
    cudaFree(h->part_o);
    cudaFree(h->part_ml);
    cudaFree(h->qrot_chunk);
    cudaFree(h->work_counter);
    cudaFree(h->lane_ticket);
    cudaFree(h->step_ticket);
    cudaFree(h->table_d);
    cudaFree(h->io_buf);
    for (auto e : h->io_ev) cudaEventDestroy(e);
    h->io_ev.clear();
    if (h->io_entry) cudaEventDestroy(h->io_entry);
    if (h->io_last) cudaEventDestroy(h->io_last);
    if (h->io_h2d) cudaStreamDestroy(h->io_h2d);
    if (h->io_d2h) cudaStreamDestroy(h->io_d2h);
    h->ring.destroy();
    for (auto& t : h->timers) {
        for (auto e : t.start) cudaEventDestroy(e);
        for (auto e : t.stop) cudaEventDestroy(e);
        t.start.clear();
        t.stop.clear();
    }
}

}  // namespace

// ---------------------------------------------------------------- ArgRing

namespace kvc {

cudaError_t ArgRing::init() {
    for (int i = 0; i < kSlots; ++i) {
        cudaError_t e = cudaEventCreateWithFlags(&done[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

void ArgRing::destroy() {
    for (int i = 0; i < kSlots; ++i) {
        if (pending[i]) cudaEventSynchronize(done[i]);
        if (host[i]) cudaFreeHost(host[i]);
        if (dev[i]) cudaFree(dev[i]);
        if (done[i]) cudaEventDestroy(done[i]);
        host[i] = dev[i] = mapped[i] = nullptr;
        done[i] = nullptr;
    }
    for (void* p : retired_host) cudaFreeHost(p);
    for (void* p : retired_dev) cudaFree(p);
    retired_host.clear();
    retired_dev.clear();
}

cudaError_t ArgRing::acquire(size_t bytes, void** host_ptr) {
    const int s = next;
    if (pending[s]) {
        cudaError_t e = cudaEventSynchronize(done[s]);
        if (e != cudaSuccess) return e;
        pending[s] = false;
    }
    if (cap[s] < bytes) {
        // grow geometrically; the replaced buffers are retired, not freed (their last
        // copy has completed, but freeing would synchronise the device)
        size_t c = std::max<size_t>(std::max<size_t>(bytes, 2 * cap[s]), 65536);
        if (host[s]) retired_host.push_back(host[s]);
        if (dev[s]) retired_dev.push_back(dev[s]);
        host[s] = dev[s] = mapped[s] = nullptr;
        cap[s] = 0;
        cudaError_t e = cudaHostAlloc(&host[s], c, cudaHostAllocMapped);
        if (e != cudaSuccess) return e;
        e = cudaHostGetDevicePointer(&mapped[s], host[s], 0);
        if (e != cudaSuccess) return e;
        e = cudaMalloc(&dev[s], c);
        if (e != cudaSuccess) return e;
        cap[s] = c;
    }
    cur = s;
    *host_ptr = host[s];
    return cudaSuccess;
}

cudaError_t ArgRing::upload(size_t bytes, cudaStream_t stream, void** dev_ptr) {
    *dev_ptr = dev[cur];
    return copy(dev[cur], bytes, stream);
}

cudaError_t ArgRing::copy(void* dst, size_t bytes, cudaStream_t stream) {
    if (by_kernel) return launch_copy_args(mapped[cur], dst, bytes, stream);
    return cudaMemcpyAsync(dst, host[cur], bytes, cudaMemcpyHostToDevice, stream);
}

cudaError_t ArgRing::release(cudaStream_t stream) {
    cudaError_t e = cudaEventRecord(done[cur], stream);
    pending[cur] = true;
    next = (cur + 1) % kSlots;
    cur = -1;
    return e;
}

}  // namespace kvc

// ---------------------------------------------------------------- C ABI

extern "C" {

int32_t kvc_abi_version(void) { return KVC_ABI_VERSION; }

const char* kvc_status_string(kvc_status s) {
    switch (s) {
        case KVC_OK: return "ok";
        case KVC_ERR_NULL: return "null pointer";
        case KVC_ERR_ZERO_BATCH: return "zero batch size";
        case KVC_ERR_ZERO_CAPACITY: return "zero capacity";
        case KVC_ERR_CAPACITY_EXCEEDS_POSITIONS: return "capacity exceeds RoPE positions";
        case KVC_ERR_ELEMENT_OVERFLOW: return "element count overflow";
        case KVC_ERR_ALLOC: return "device allocation failed";
        case KVC_ERR_FULL: return "cache full";
        case KVC_ERR_KEY_SHAPE: return "key shape mismatch";
        case KVC_ERR_VALUE_SHAPE: return "value shape mismatch";
        case KVC_ERR_QUERY_SHAPE: return "query shape mismatch";
        case KVC_ERR_OUTPUT_SHAPE: return "output shape mismatch";
        case KVC_ERR_DTYPE: return "dtype mismatch";
        case KVC_ERR_LAYER: return "layer out of range";
        case KVC_ERR_NONFINITE_KEY: return "non-finite key";
        case KVC_ERR_NONFINITE_VALUE: return "non-finite value";
        case KVC_ERR_CUT: return "invalid cut";
        case KVC_ERR_EMPTY_QUERY: return "empty query";
        case KVC_ERR_POSITION: return "position out of range";
        case KVC_ERR_CONFIG: return "invalid configuration";
        case KVC_ERR_CUDA: return "CUDA error";
        case KVC_ERR_DEVICE: return "device-side error";
        case KVC_ERR_TICKET: return "stale or foreign ticket";
    }
    return "unknown status";
}

const char* kvc_last_error(const kvc_handle* h) {
    return h ? h->last_error.c_str() : g_create_error.c_str();
}

kvc_status kvc_create(int32_t batch, int32_t heads, int32_t capacity, int32_t head_dim, int32_t layers,
                      kvc_handle** out) {
    kvc_config c{};
    c.batch = batch;
    c.heads_q = heads;
    c.heads_kv = heads;
    c.capacity = capacity;
    c.head_dim = head_dim;
    c.layers = layers;
    c.dtype = KVC_BF16;
    c.rope_max_positions = 0;
    c.rope_base = 10000.0;
    c.checked = 0;
    c.device = 0;
    return kvc_create_ex(&c, out);
}

kvc_status kvc_create_ex(const kvc_config* config, kvc_handle** out) {
    if (!out) return fail(nullptr, KVC_ERR_NULL, "output handle pointer is NULL");
    *out = nullptr;
    if (!config) return fail(nullptr, KVC_ERR_NULL, "configuration pointer is NULL");
    kvc_config c = *config;
    if (c.batch <= 0) return fail(nullptr, KVC_ERR_ZERO_BATCH, "batch size must be at least 1, got %d", c.batch);
    if (c.capacity <= 0)
        return fail(nullptr, KVC_ERR_ZERO_CAPACITY, "capacity must be at least 1, got %d", c.capacity);
    if (c.heads_q <= 0 || c.heads_kv <= 0 || c.heads_q % c.heads_kv)
        return fail(nullptr, KVC_ERR_CONFIG, "heads_q (%d) must be a positive multiple of heads_kv (%d)", c.heads_q,
                    c.heads_kv);
    if (c.head_dim < 2 || c.head_dim > 256 || c.head_dim % 2)
        return fail(nullptr, KVC_ERR_CONFIG, "head width must be even and in [2, 256], got %d", c.head_dim);
    if (c.layers <= 0) return fail(nullptr, KVC_ERR_CONFIG, "layer count must be at least 1, got %d", c.layers);
    if (!dtype_size(c.dtype)) return fail(nullptr, KVC_ERR_CONFIG, "unknown storage dtype %d", c.dtype);
    if (!(c.rope_base >= 0.0) || !std::isfinite(c.rope_base))
        return fail(nullptr, KVC_ERR_CONFIG, "RoPE base must be finite and >= 0");
    if (c.rope_max_positions < 0) return fail(nullptr, KVC_ERR_CONFIG, "rope_max_positions must be >= 0");
    if (c.window < 0) return fail(nullptr, KVC_ERR_CONFIG, "sliding window must be 0 (none) or >= 1, got %d", c.window);
    if (c.block_rows < 0 || (c.block_rows && (c.block_rows < 64 || (c.block_rows & (c.block_rows - 1)))))
        return fail(nullptr, KVC_ERR_CONFIG, "block rows must be 0 (contiguous) or a power of two >= 64, got %d",
                    c.block_rows);
    if (c.blocks < 0) return fail(nullptr, KVC_ERR_CONFIG, "block count must be >= 0, got %d", c.blocks);
    const bool paged = c.block_rows > 0;
    const int nblk = paged ? (int)(((int64_t)c.capacity + c.block_rows - 1) / c.block_rows) : 0;
    if (paged && c.blocks == 0) {
        if ((int64_t)c.batch * nblk > INT32_MAX) return fail(nullptr, KVC_ERR_ELEMENT_OVERFLOW, "too many blocks");
        c.blocks = c.batch * nblk;
    }
    if (!paged) c.blocks = 0;
    const int maxpos = c.rope_max_positions ? c.rope_max_positions : c.capacity;
    if (c.capacity > maxpos)
        return fail(nullptr, KVC_ERR_CAPACITY_EXCEEDS_POSITIONS,
                    "capacity %d is larger than the %d positions the RoPE table covers", c.capacity, maxpos);
    c.rope_max_positions = maxpos;

    size_t layer_elems, all_elems, bytes, t, store_rows;
    // rows of one layer's key (or value) array: [B][H_kv][C], or the pool [blocks][H_kv][P]
    const bool rows_ok = paged ? mul_ok(c.blocks, c.heads_kv, &t) && mul_ok(t, c.block_rows, &store_rows)
                               : mul_ok(c.batch, c.heads_kv, &t) && mul_ok(t, c.capacity, &store_rows);
    if (!rows_ok || !mul_ok(store_rows, c.head_dim, &layer_elems) ||
        !mul_ok(layer_elems, c.layers, &all_elems) || !mul_ok(all_elems, dtype_size(c.dtype), &bytes))
        return fail(nullptr, KVC_ERR_ELEMENT_OVERFLOW,
                    "element count overflows for batch %d, %d heads, capacity %d, head width %d, %d layers", c.batch,
                    c.heads_kv, c.capacity, c.head_dim, c.layers);
    if ((uint64_t)c.batch * c.heads_kv * c.capacity > (uint64_t)INT32_MAX || store_rows > (uint64_t)INT32_MAX)
        return fail(nullptr, KVC_ERR_ELEMENT_OVERFLOW,
                    "batch * heads_kv * capacity (and the pool's rows) must fit in 31 bits");

    cudaError_t e = cudaSetDevice(c.device);
    if (e != cudaSuccess) return fail(nullptr, KVC_ERR_CUDA, "cudaSetDevice(%d) failed: %s", c.device, cudaGetErrorString(e));

    kvc_handle* h = new kvc_handle();
    h->cfg = c;
    h->max_positions = maxpos;
    h->elem_size = dtype_size(c.dtype);
    h->layer_elems = layer_elems;
    const size_t LB = (size_t)c.layers * c.batch;
    auto alloc = [&](void** p, size_t n) -> bool {
        cudaError_t ae = cudaMalloc(p, n);
        if (ae != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        return true;
    };
    const size_t acc = c.dtype == KVC_F64 ? 8 : 4;
    bool ok = alloc(&h->K, bytes) && alloc(&h->V, bytes) &&
              alloc((void**)&h->positions, LB * c.capacity * sizeof(int32_t)) &&
              alloc((void**)&h->len_d, LB * sizeof(int32_t)) && alloc((void**)&h->next_d, LB * sizeof(int32_t)) &&
              alloc((void**)&h->err_d, sizeof(uint32_t)) &&
              alloc((void**)&h->nonfinite_d, 2 * sizeof(unsigned long long)) &&
              alloc(&h->qrot, (size_t)c.batch * c.heads_q * c.head_dim * acc) &&
              alloc((void**)&h->work_counter, 64) &&
              alloc((void**)&h->lane_ticket, (size_t)c.batch * c.heads_kv * sizeof(unsigned)) &&
              alloc((void**)&h->step_ticket, (size_t)c.layers * sizeof(unsigned));
    if (ok && paged) ok = alloc((void**)&h->table_d, (size_t)c.batch * nblk * sizeof(int32_t));
    if (ok && c.rope_base > 0.0)
        ok = alloc((void**)&h->rope, (size_t)maxpos * (c.head_dim / 2) * sizeof(double2)) &&
             alloc((void**)&h->rope_f, (size_t)maxpos * (c.head_dim / 2) * sizeof(float2));
    if (!ok) {
        free_all(h);
        delete h;
        return fail(nullptr, KVC_ERR_ALLOC, "cannot allocate %zu bytes of KV cache storage", 2 * bytes);
    }
    auto abort_cuda = [&](cudaError_t ce, const char* what) {
        free_all(h);
        delete h;
        return fail(nullptr, KVC_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(ce));
    };
    if ((e = cudaMemset(h->K, 0, bytes)) != cudaSuccess) return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->V, 0, bytes)) != cudaSuccess) return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->positions, 0, LB * c.capacity * sizeof(int32_t))) != cudaSuccess)
        return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->len_d, 0, LB * sizeof(int32_t))) != cudaSuccess) return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->next_d, 0, LB * sizeof(int32_t))) != cudaSuccess) return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->err_d, 0, sizeof(uint32_t))) != cudaSuccess) return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->lane_ticket, 0, (size_t)c.batch * c.heads_kv * sizeof(unsigned))) != cudaSuccess)
        return abort_cuda(e, "cudaMemset");
    if ((e = cudaMemset(h->step_ticket, 0, (size_t)c.layers * sizeof(unsigned))) != cudaSuccess)
        return abort_cuda(e, "cudaMemset");
    if (paged) {
        h->nblk = nblk;
        h->nblocks = c.blocks;
        h->table_h.assign((size_t)c.batch * nblk, -1);
        h->refcnt.assign(c.blocks, 0);
        h->free_blocks.resize(c.blocks);
        for (int i = 0; i < c.blocks; ++i) h->free_blocks[i] = c.blocks - 1 - i;   // handed out 0, 1, 2, ...
        if ((e = cudaMemset(h->table_d, 0xff, (size_t)c.batch * nblk * sizeof(int32_t))) != cudaSuccess)
            return abort_cuda(e, "cudaMemset");
    }
    if ((e = cudaHostAlloc((void**)&h->nonfinite_h, 2 * sizeof(unsigned long long), cudaHostAllocDefault)) !=
        cudaSuccess)
        return abort_cuda(e, "cudaHostAlloc");
    if ((e = h->ring.init()) != cudaSuccess) return abort_cuda(e, "cudaEventCreate");

    if (h->rope) {
        // cos/sin of phi = p * theta_j, theta_j = base^(-2j/d_h): one IEEE product and one
        // libm call per entry, computed once per handle.
        const int half = c.head_dim / 2;
        std::vector<double> inv(half);
        for (int j = 0; j < half; ++j) inv[j] = std::pow(c.rope_base, -(2.0 * j) / c.head_dim);
        std::vector<double2> tab((size_t)maxpos * half);
        for (int p = 0; p < maxpos; ++p)
            for (int j = 0; j < half; ++j) {
                const double ang = (double)p * inv[j];
                tab[(size_t)p * half + j] = make_double2(std::cos(ang), std::sin(ang));
            }
        if ((e = cudaMemcpy(h->rope, tab.data(), tab.size() * sizeof(double2), cudaMemcpyHostToDevice)) !=
            cudaSuccess)
            return abort_cuda(e, "cudaMemcpy");
        std::vector<float2> tabf(tab.size());
        for (size_t i = 0; i < tab.size(); ++i) tabf[i] = make_float2((float)tab[i].x, (float)tab[i].y);
        if ((e = cudaMemcpy(h->rope_f, tabf.data(), tabf.size() * sizeof(float2), cudaMemcpyHostToDevice)) !=
            cudaSuccess)
            return abort_cuda(e, "cudaMemcpy");
    }

    if (c.dtype == KVC_BF16 && c.head_dim == 128) {
        h->tmap_k.resize(c.layers);
        h->tmap_v.resize(c.layers);
        h->tmap_k128.resize(c.layers);
        h->tmap_v128.resize(c.layers);
        h->tmap_k16.resize(c.layers);
        h->tmap_v16.resize(c.layers);
        bool all = true;
        const uint64_t rows = store_rows;
        for (int l = 0; l < c.layers && all; ++l)
            all = encode_rows_map(&h->tmap_k[l], h->K_layer(l), rows, 64) &&
                  encode_rows_map(&h->tmap_v[l], h->V_layer(l), rows, 64) &&
                  encode_rows_map(&h->tmap_k128[l], h->K_layer(l), rows, 128) &&
                  encode_rows_map(&h->tmap_v128[l], h->V_layer(l), rows, 128) &&
                  encode_rows_map(&h->tmap_k16[l], h->K_layer(l), rows, 16) &&
                  encode_rows_map(&h->tmap_v16[l], h->V_layer(l), rows, 16);
        h->have_tmaps = all;
    }
    h->len_h.assign(LB, 0);
    h->next_h.assign(LB, 0);
    h->layer_version.assign(c.layers, 0);
    *out = h;
    return KVC_OK;
}

void kvc_destroy(kvc_handle* h) {
    if (!h) return;
    cudaSetDevice(h->cfg.device);
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
}

static kvc_status check_layer(kvc_handle* h, int32_t layer) {
    if (layer < 0 || layer >= h->cfg.layers)
        return fail(h, KVC_ERR_LAYER, "layer %d is outside [0, %d)", layer, h->cfg.layers);
    return KVC_OK;
}

// After device-length decode steps (and in that mode at any time, since a
// captured graph may have replayed steps without a host call) the device
// lengths are authoritative: wait for every enqueued step and read them back
// into the host mirrors.
static kvc_status refresh_mirrors(kvc_handle* h) {
    if (!h->mirrors_stale && !h->opt_device_lengths) return KVC_OK;
    const size_t n = (size_t)h->cfg.layers * h->B();
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    KVC_CUDA(h, cudaDeviceSynchronize());
    KVC_CUDA(h, cudaMemcpy(h->len_h.data(), h->len_d, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    KVC_CUDA(h, cudaMemcpy(h->next_h.data(), h->next_d, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    h->mirrors_stale = false;
    return KVC_OK;
}

// ---- paged storage: block allocation on the host, copies on the device -------------

static kvc_status upload_table(kvc_handle* h, cudaStream_t s) {
    if (!h->table_dirty) return KVC_OK;
    const size_t bytes = h->table_h.size() * sizeof(int32_t);
    void* hp;
    KVC_CUDA(h, h->ring.acquire(bytes, &hp));
    memcpy(hp, h->table_h.data(), bytes);
    KVC_CUDA(h, h->ring.copy(h->table_d, bytes, s));
    KVC_CUDA(h, h->ring.release(s));
    h->table_dirty = false;
    return KVC_OK;
}

// Gives every sequence b blocks for rows [from[b], to[b]) -- a block that is shared
// with another sequence is first copied (copy-on-write) -- then uploads the table.
// All or nothing: KVC_ERR_FULL, with no change, when the pool is short.
// Blocks that growing each sequence b from from[b] to to[b] rows takes from the pool: one
// per missing block and one per shared block written into (copied first).
static int64_t blocks_needed(kvc_handle* h, const int32_t* from, const int32_t* to) {
    const int B = h->B(), P = h->cfg.block_rows, nb = h->nblk;
    int64_t need = 0;
    for (int b = 0; b < B; ++b)
        for (int j = from[b] / P; from[b] < to[b] && j <= (to[b] - 1) / P; ++j) {
            const int blk = h->table_h[(size_t)b * nb + j];
            need += blk < 0 || h->refcnt[blk] > 1;
        }
    return need;
}

static kvc_status ensure_blocks(kvc_handle* h, const int32_t* from, const int32_t* to, cudaStream_t s) {
    if (!h->paged()) return KVC_OK;
    const int B = h->B(), P = h->cfg.block_rows, nb = h->nblk;
    const int64_t need = blocks_needed(h, from, to);
    if (need > (int64_t)h->free_blocks.size())
        return fail(h, KVC_ERR_FULL, "the block pool has %zu free blocks; the call needs %lld", h->free_blocks.size(),
                    (long long)need);
    std::vector<int2> cow;
    for (int b = 0; b < B; ++b)
        for (int j = from[b] / P; from[b] < to[b] && j <= (to[b] - 1) / P; ++j) {
            int32_t& slot = h->table_h[(size_t)b * nb + j];
            if (slot >= 0 && h->refcnt[slot] == 1) continue;
            const int fresh = h->free_blocks.back();
            h->free_blocks.pop_back();
            h->refcnt[fresh] = 1;
            if (slot >= 0) {
                h->refcnt[slot] -= 1;
                cow.push_back(make_int2(slot, fresh));
            }
            slot = fresh;
            h->table_dirty = true;
        }
    if (!cow.empty()) {
        void* hp;
        void* dp;
        const size_t bytes = cow.size() * sizeof(int2);
        KVC_CUDA(h, h->ring.acquire(bytes, &hp));
        memcpy(hp, cow.data(), bytes);
        KVC_CUDA(h, h->ring.upload(bytes, s, &dp));
        const size_t block_bytes = (size_t)h->Hkv() * P * h->D() * h->elem_size;
        KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] {
            return launch_copy_blocks((char*)h->K, (char*)h->V, h->layer_elems * h->elem_size, h->cfg.layers,
                                      block_bytes, (const int2*)dp, (int)cow.size(), s);
        }));
        KVC_CUDA(h, h->ring.release(s));
    }
    return upload_table(h, s);
}

// Returns the blocks of sequence b past its first `keep` rows to the pool.
static void release_blocks(kvc_handle* h, int b, int keep) {
    if (!h->paged()) return;
    const int P = h->cfg.block_rows;
    for (int j = (keep + P - 1) / P; j < h->nblk; ++j) {
        int32_t& slot = h->table_h[(size_t)b * h->nblk + j];
        if (slot < 0) continue;
        if (--h->refcnt[slot] == 0) h->free_blocks.push_back(slot);
        slot = -1;
        h->table_dirty = true;
    }
}

// True while `s` records a CUDA graph (or when that cannot be told): decode launches are
// then made without the programmatic-dependent-launch attribute.
static bool stream_capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return st != cudaStreamCaptureStatusNone;
}

static kvc_status ensure_partials(kvc_handle* h, size_t splits) {
    if (h->part_splits >= splits) return KVC_OK;
    cudaDeviceSynchronize();
    cudaFree(h->part_o);
    cudaFree(h->part_ml);
    h->part_o = nullptr;
    h->part_ml = nullptr;
    h->part_splits = 0;
    const size_t lanes = (size_t)h->B() * h->Hq();
    if (cudaMalloc((void**)&h->part_o, lanes * splits * 128 * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&h->part_ml, lanes * splits * sizeof(float2)) != cudaSuccess) {
        cudaGetLastError();
        return fail(h, KVC_ERR_ALLOC, "cannot allocate decode split scratch for %zu splits", splits);
    }
    h->part_splits = splits;
    return KVC_OK;
}

static kvc_status check_nonfinite(kvc_handle* h, const kvc_tensor* k, const kvc_tensor* v, int64_t nk,
                                  int64_t nv, cudaStream_t s) {
    KVC_CUDA(h, cudaMemsetAsync(h->nonfinite_d, 0xff, 2 * sizeof(unsigned long long), s));
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] { return launch_nonfinite(h->cfg.dtype, k->data, nk, h->nonfinite_d, s); }));
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] { return launch_nonfinite(h->cfg.dtype, v->data, nv, h->nonfinite_d + 1, s); }));
    KVC_CUDA(h, cudaMemcpyAsync(h->nonfinite_h, h->nonfinite_d, 2 * sizeof(unsigned long long),
                                cudaMemcpyDeviceToHost, s));
    KVC_CUDA(h, cudaStreamSynchronize(s));
    for (int which = 0; which < 2; ++which) {
        const unsigned long long idx = h->nonfinite_h[which];
        if (idx == ~0ull) continue;
        const kvc_tensor* t = which ? v : k;
        double val = 0;
        char raw[8] = {};
        if (cudaMemcpy(raw, (const char*)t->data + idx * h->elem_size, h->elem_size, cudaMemcpyDeviceToHost) ==
            cudaSuccess) {
            if (h->cfg.dtype == KVC_F64) memcpy(&val, raw, 8);
            else if (h->cfg.dtype == KVC_F32) { float f; memcpy(&f, raw, 4); val = f; }
            else { uint32_t u = (uint32_t)(*(uint16_t*)raw) << 16; float f; memcpy(&f, &u, 4); val = f; }
        }
        return fail(h, which ? KVC_ERR_NONFINITE_VALUE : KVC_ERR_NONFINITE_KEY,
                    "%s element at flat index %llu is not finite (%g); nothing was appended", which ? "value" : "key",
                    idx, val);
    }
    return KVC_OK;
}

}  // extern "C"

namespace kvc {
namespace {

// One decode step of one layer; `commit` false prepares it (kvc_prepare_attend):
// the candidate rows are staged in slot n_b and the lengths are left unchanged.
kvc_status append_attend_impl(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k,
                              const kvc_tensor* v, const kvc_tensor* out, bool commit, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    kvc_status st;
    if ((st = check_layer(h, layer)) != KVC_OK) return st;
    if (!commit && h->opt_device_lengths)
        return fail(h, KVC_ERR_CONFIG, "prepared steps need the host length mirrors (device-length mode is on)");
    const int B = h->B(), Hq = h->Hq(), Hkv = h->Hkv(), D = h->D(), C = h->C();
    const int dt = h->cfg.dtype;
    if (q && q->ndim == 4 && q->shape[2] != 1)
        return fail(h, KVC_ERR_QUERY_SHAPE, "one decode step takes a single token per sequence, got %lld",
                    (long long)q->shape[2]);
    if ((st = check_tensor(h, q, "query", KVC_ERR_QUERY_SHAPE, dt, B, Hq, 1, D)) != KVC_OK) return st;
    if ((st = check_tensor(h, k, "key", KVC_ERR_KEY_SHAPE, dt, B, Hkv, 1, D)) != KVC_OK) return st;
    if ((st = check_tensor(h, v, "value", KVC_ERR_VALUE_SHAPE, dt, B, Hkv, 1, D)) != KVC_OK) return st;
    const bool fast = fast_decode_ok(h);
    // bf16 storage on the tensor-core decode path may also return bf16 outputs
    const bool out_bf16 = out && out->dtype == KVC_BF16 && dt == KVC_BF16 && fast;
    if ((st = check_tensor(h, out, "output", KVC_ERR_OUTPUT_SHAPE, out_bf16 ? KVC_BF16 : out_dtype(dt), B, Hq, 1,
                           D)) != KVC_OK)
        return st;
    const bool dev_len = h->opt_device_lengths != 0;
    if (dev_len && !(fast && h->opt_decode_fused && B <= kFusedMaxB))
        return fail(h, KVC_ERR_CONFIG,
                    "device-length decode steps need bf16 storage, d_h = 128, the fused step and at most %d sequences",
                    kFusedMaxB);
    if (!dev_len && (st = refresh_mirrors(h)) != KVC_OK) return st;
    int32_t* lenh = &h->len_h[(size_t)layer * B];
    int32_t* nexth = &h->next_h[(size_t)layer * B];
    int max_t = 0;
    int64_t total_keys = 0;
    const int W = h->cfg.window;
    // key rows one query's splits cover: from its window start rounded down to a 64-row tile
    auto keys_of = [&](int t) { return W > 0 ? t - (std::max(0, t - W) & ~63) : t; };
    for (int b = 0; b < B && dev_len; ++b) {
        // the kernel checks the device lengths; the mirrors only size the splits
        max_t = std::max(max_t, keys_of(std::min(lenh[b], C - 1) + 1));
        total_keys += keys_of(std::min(lenh[b], C - 1) + 1);
    }
    for (int b = 0; b < B && !dev_len; ++b) {
        if (lenh[b] >= C)
            return fail(h, KVC_ERR_FULL, "sequence %d of layer %d already holds %d rows, the capacity", b, layer, C);
        if (h->rope && nexth[b] >= h->max_positions)
            return fail(h, KVC_ERR_POSITION, "sequence %d would be rotated at position %d, beyond the %d-position table",
                        b, nexth[b], h->max_positions);
        max_t = std::max(max_t, keys_of(lenh[b] + 1));
        total_keys += keys_of(lenh[b] + 1);
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    if (h->cfg.checked) {
        if ((st = check_nonfinite(h, k, v, (int64_t)B * Hkv * D, (int64_t)B * Hkv * D, s)) != KVC_OK) return st;
    }
    if (h->paged()) {
        std::vector<int32_t> to(B);
        for (int b = 0; b < B; ++b) to[b] = lenh[b] + 1;
        if ((st = ensure_blocks(h, lenh, to.data(), s)) != KVC_OK) return st;
    }
    AppendLaunch ap{};
    ap.q = q->data; ap.k = k->data; ap.v = v->data;
    ap.K = h->K_layer(layer); ap.V = h->V_layer(layer); ap.positions = h->pos_layer(layer);
    ap.slot0 = h->len_layer(layer); ap.pos0 = h->next_layer(layer); ap.seqlen = nullptr;
    ap.qrot = h->qrot; ap.qrot_kind = dt == KVC_F64 ? 1 : 0;
    ap.rope = h->rope; ap.rope_f = h->rope_f; ap.err = h->err_d;
    ap.B = B; ap.Hq = Hq; ap.Hkv = Hkv; ap.S = 1; ap.C = C; ap.d = D; ap.max_positions = h->max_positions;
    ap.kv = h->layout();

    int split_rows = 0, max_splits = 1;
    // Many query heads per key/value head on the fused step: the tensor-core decode kernel
    // (one CTA per SM) instead of the m16n8k16 one (two per SM)
    const bool tc_decode = fast && h->opt_decode_tc && h->opt_decode_fused && B <= kFusedMaxB && !dev_len &&
                           !h->paged() && Hq / Hkv > 16 && Hq / Hkv <= 32;
    struct {
        bool on = false;
        int32_t start[kFusedMaxB + 1];
        int32_t seq[kFusedMaxB];
        int32_t rows[kFusedMaxB];
    } pieces;
    int lanes_per_cta = 0;
    struct {
        bool on = false;
        int P = 0, T = 0;
        int32_t start[kFusedMaxB + 1];
        int32_t first[kFusedMaxB];
        int32_t ns[kFusedMaxB];
    } sk;
    if (fast) {
        if (h->opt_split_rows > 0) {
            split_rows = (int)h->opt_split_rows;
        } else if (tc_decode && h->opt_decode_streamk && (int64_t)B * Hkv <= kFusedMaxB) {
            // Stream-K: the lanes' 128-key tiles laid end to end, one wave of CTAs (one per
            // SM) over equal runs of them; a lane's partials: one per CTA its tiles touch.
            // CTA c starts at tile floor(c T / P); the CTA holding tile x is
            // floor(((x + 1) P - 1) / T).
            const int lanes = B * Hkv;
            int64_t T = 0;
            for (int l = 0; l < lanes; ++l) {
                sk.start[l] = (int32_t)T;
                T += (keys_of(lenh[l / Hkv] + 1) + 127) / 128;
            }
            sk.start[lanes] = (int32_t)T;
            const int64_t P = std::max<int64_t>(1, std::min<int64_t>(sm_count(h->cfg.device), T));
            max_splits = 1;
            for (int l = 0; l < lanes; ++l) {
                const int64_t x0 = sk.start[l], x1 = sk.start[l + 1] - 1;
                const int64_t c0 = ((x0 + 1) * P - 1) / T, c1 = ((x1 + 1) * P - 1) / T;
                sk.first[l] = (int32_t)c0;
                sk.ns[l] = (int32_t)(c1 - c0 + 1);
                max_splits = std::max(max_splits, sk.ns[l]);
            }
            sk.on = true;
            sk.P = (int)P;
            sk.T = (int)T;
            split_rows = 128;
        } else if (tc_decode) {
            // One CTA per SM: every sequence is cut into its own number of equal pieces,
            // about two waves of them in all, and the pieces are launched largest first,
            // so that the in-order dispatch of CTAs to free SMs ends with the small ones.
            const int64_t slots = 2 * (int64_t)sm_count(h->cfg.device);
            std::vector<int> keys(B);
            for (int b = 0; b < B; ++b) keys[b] = keys_of(lenh[b] + 1);
            auto count = [&](int64_t r) {
                int64_t c = 0;
                for (int b = 0; b < B; ++b) c += (int64_t)Hkv * ((keys[b] + r - 1) / r);
                return c;
            };
            int64_t R = std::max<int64_t>(1024, ((total_keys * Hkv + slots - 1) / slots + 63) / 64 * 64);
            while (count(R) > slots && R < ((int64_t)max_t + 63) / 64 * 64) R += 64;
            pieces.on = true;
            std::vector<int> order(B);
            for (int b = 0; b < B; ++b) {
                int ns = (keys[b] + (int)R - 1) / (int)R;
                // whole 128-key tiles (the kernel's tile), so only a lane's last piece ends
                // inside a tile
                pieces.rows[b] = ((keys[b] + ns - 1) / ns + 127) / 128 * 128;
                order[b] = b;
            }
            std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return pieces.rows[x] > pieces.rows[y]; });
            pieces.start[0] = 0;
            max_splits = 1;
            for (int i = 0; i < B; ++i) {
                const int b = order[i];
                const int ns = (keys[b] + pieces.rows[b] - 1) / pieces.rows[b];
                pieces.seq[i] = b;
                pieces.start[i + 1] = pieces.start[i] + Hkv * ns;
                max_splits = std::max(max_splits, ns);
            }
            split_rows = (int)R;
        } else {
            const int G = Hq / Hkv;
            const int64_t target = (int64_t)sm_count(h->cfg.device) * decode_bf16_ctas_per_sm(G) * 4;
            // about four waves of CTAs, but at least 256 rows per query head served
            // (a CTA's fixed work -- queries, pipeline fill, merge -- grows with G)
            // as long as that still leaves one CTA per SM
            const int64_t keys = total_keys * Hkv;
            int64_t r = (keys + target - 1) / target;
            r = std::max<int64_t>(r, std::min<int64_t>(256 * G, keys / sm_count(h->cfg.device)));
            r = (r + 63) / 64 * 64;
            // at most 4096 rows, in multiples of 512 from 1024 up: B = 64, H_kv = 8, 16-32K
            // contexts ran 1.5% faster with 4096-row splits than with the 10816 the wave
            // count alone gives (more, shorter CTAs drain more evenly), B = 32, H = 32, up to
            // 8K 0.4% faster with 3072 rows than with 3200
            r = std::min<int64_t>(r, 4096);
            if (r >= 1024) r = r / 512 * 512;
            r = std::min<int64_t>(r, ((int64_t)max_t + 63) / 64 * 64);
            split_rows = (int)r;
        }
        if (!pieces.on && !sk.on) max_splits = (max_t + split_rows - 1) / split_rows;
        // Short contexts with many lanes (at least four waves of one-split lanes, G <= 4):
        // CTAs that walk several lanes each, longest sequences first (decode_lanes_kernel).
        // Lanes per CTA: 2 .. 8, the count that minimises waves x (lanes + 0.5), the 0.5
        // being a CTA's own fixed cost in lanes -- a partial last wave costs as much as a
        // full one (B = 128, H = 32, lengths up to 256 on 152 SMs: 7 lanes, 586 CTAs in
        // two waves, 11% faster than 6 lanes and 683 CTAs in three).
        if (h->opt_decode_lanes && !tc_decode && h->opt_decode_fused && !dev_len && B <= kFusedMaxB &&
            Hq / Hkv <= 4 && !h->opt_split_rows && max_t <= 512) {
            const int64_t slots = (int64_t)sm_count(h->cfg.device) * decode_bf16_ctas_per_sm(Hq / Hkv);
            const int64_t lanes = (int64_t)B * Hkv;
            if (lanes >= 4 * slots) {
                double best = 0.0;
                for (int lpc = 2; lpc <= 8; ++lpc) {
                    const int64_t waves = ((lanes + lpc - 1) / lpc + slots - 1) / slots;
                    const double cost = (double)waves * (lpc + 0.5);
                    if (lanes_per_cta == 0 || cost < best) {
                        best = cost;
                        lanes_per_cta = lpc;
                    }
                }
                split_rows = (max_t + 63) / 64 * 64;
                max_splits = 1;
            }
        }
        if (dev_len) {
            // A device-length step keeps its grid for every later length (a captured
            // graph replays it) and each sequence takes max_splits splits of its own
            // size: as many as the mean length needs at the rows per split chosen
            // above, but as many as fit in one wave of CTAs and at most one per 64 rows.
            const int64_t lanes = (int64_t)B * Hkv;
            const int64_t mean_t = (total_keys + B - 1) / B;
            int64_t ns = (mean_t + split_rows - 1) / split_rows;
            // (whole CTAs per lane: rounding the fill up would leave a short second wave)
            const int64_t fill = (int64_t)sm_count(h->cfg.device) * decode_bf16_ctas_per_sm(Hq / Hkv) / lanes;
            ns = std::min<int64_t>(std::max<int64_t>(ns, fill), (C + 63) / 64);
            max_splits = (int)std::max<int64_t>(ns, 1);
        }
        if (max_splits > 1 && (st = ensure_partials(h, max_splits)) != KVC_OK) return st;
    }

    // One launch per step (append, attend, merge splits, commit lengths); beyond 16
    // query heads per key/value head the merge done by one CTA per lane costs more
    // than a separate merge kernel spread over every query head, so it follows.
    if (fast && h->opt_decode_fused && B <= kFusedMaxB) {
        DecodeLaunch dl{};
        dl.tmK = &h->tmap_k[layer]; dl.tmV = &h->tmap_v[layer];
        dl.tmK128 = &h->tmap_k128[layer]; dl.tmV128 = &h->tmap_v128[layer];
        dl.tmK16 = &h->tmap_k16[layer]; dl.tmV16 = &h->tmap_v16[layer];
        dl.part_o = h->part_o; dl.part_ml = h->part_ml; dl.out = out->data; dl.err = h->err_d;
        dl.B = B; dl.Hq = Hq; dl.Hkv = Hkv; dl.C = C; dl.split_rows = split_rows; dl.max_splits = max_splits;
        dl.out_bf16 = out_bf16;
        dl.window = W;
        dl.kv = h->layout();
        dl.fused = 1;
        dl.dev_len = dev_len;
        dl.step_ticket = h->step_ticket + layer;
        dl.max_positions = h->max_positions;
        dl.q_in = (const __nv_bfloat16*)q->data; dl.k_in = (const __nv_bfloat16*)k->data;
        dl.v_in = (const __nv_bfloat16*)v->data;
        dl.K = (__nv_bfloat16*)h->K_layer(layer); dl.V = (__nv_bfloat16*)h->V_layer(layer);
        dl.positions = h->pos_layer(layer);
        dl.len_out = h->len_layer(layer); dl.next_out = h->next_layer(layer);
        dl.rope_f = h->rope_f; dl.rope = h->rope; dl.lane_ticket = h->lane_ticket;
        dl.merge_in_kernel = Hq / Hkv <= 16;
        dl.no_commit = !commit;
        dl.pdl = h->opt_decode_pdl && !dev_len && !stream_capturing(s);
        dl.test_stall = (int)h->opt_test_stall;
        h->opt_test_stall = 0;
        for (int b = 0; b < B && !dev_len; ++b) {
            dl.old_len[b] = lenh[b];
            dl.pos[b] = nexth[b];
        }
        dl.pieces = pieces.on;
        dl.lanes_per_cta = lanes_per_cta;
        if (lanes_per_cta) {
            // sequences longest first: the last CTAs to start are the shortest
            std::vector<int> order(B);
            for (int b = 0; b < B; ++b) order[b] = b;
            std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return lenh[x] > lenh[y]; });
            for (int i = 0; i < B; ++i) dl.seq_of[i] = order[i];
        }
        if (sk.on) {
            dl.streamk = sk.P;
            dl.streamk_tiles = sk.T;
            memcpy(dl.item_start, sk.start, (B * Hkv + 1) * sizeof(int32_t));
            memcpy(dl.seq_of, sk.first, B * Hkv * sizeof(int32_t));
            memcpy(dl.seq_rows, sk.ns, B * Hkv * sizeof(int32_t));
        }
        if (pieces.on) {
            memcpy(dl.item_start, pieces.start, (B + 1) * sizeof(int32_t));
            memcpy(dl.seq_of, pieces.seq, B * sizeof(int32_t));
            memcpy(dl.seq_rows, pieces.rows, B * sizeof(int32_t));
        }
        KVC_CUDA(h, timed(h, KVC_KERNEL_DECODE, s, [&] {
            return tc_decode ? (sk.on ? launch_decode_tck(dl, s) : launch_decode_tc(dl, s))
                             : lanes_per_cta ? launch_decode_lanes(dl, s)
                                             : launch_decode_bf16(dl, s);
        }));
        if (!dl.merge_in_kernel && max_splits > 1)
            KVC_CUDA(h, timed(h, KVC_KERNEL_DECODE_COMBINE, s, [&] { return launch_decode_combine(dl, s); }));
        h->layer_version[layer] += 1;
        if (dev_len) {
            h->mirrors_stale = true;
            return KVC_OK;
        }
        for (int b = 0; b < B && commit; ++b) {
            lenh[b] += 1;
            nexth[b] += 1;
        }
        return KVC_OK;
    }
    KVC_CUDA(h, timed(h, KVC_KERNEL_ROPE_APPEND, s, [&] { return launch_rope_append(dt, ap, s); }));
    if (fast) {
        DecodeLaunch dl{};
        dl.tmK = &h->tmap_k[layer]; dl.tmV = &h->tmap_v[layer];
        dl.qrot = (const float*)h->qrot; dl.len = h->len_layer(layer);
        dl.part_o = h->part_o; dl.part_ml = h->part_ml; dl.out = out->data; dl.err = h->err_d;
        dl.B = B; dl.Hq = Hq; dl.Hkv = Hkv; dl.C = C; dl.split_rows = split_rows; dl.max_splits = max_splits;
        dl.out_bf16 = out_bf16;
        dl.window = W;
        dl.kv = h->layout();
        dl.pdl = h->opt_decode_pdl && !stream_capturing(s);
        dl.test_stall = (int)h->opt_test_stall;
        h->opt_test_stall = 0;
        KVC_CUDA(h, timed(h, KVC_KERNEL_DECODE, s, [&] { return launch_decode_bf16(dl, s); }));
        if (max_splits > 1)
            KVC_CUDA(h, timed(h, KVC_KERNEL_DECODE_COMBINE, s, [&] { return launch_decode_combine(dl, s); }));
    } else {
        GenericAttendLaunch g{};
        g.qrot = h->qrot; g.K = h->K_layer(layer); g.V = h->V_layer(layer);
        g.slot0 = h->len_layer(layer); g.seqlen = nullptr; g.out = out->data;
        g.B = B; g.Hq = Hq; g.Hkv = Hkv; g.S = 1; g.C = C; g.d = D; g.window = W; g.kv = h->layout(); g.err = h->err_d;
        KVC_CUDA(h, timed(h, KVC_KERNEL_GENERIC_ATTEND, s, [&] { return launch_attend_generic(dt, g, s); }));
    }
    h->layer_version[layer] += 1;
    if (!commit) return KVC_OK;
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] {
        return launch_commit(h->len_layer(layer), h->next_layer(layer), h->next_layer(layer), nullptr, 1, B, C,
                             h->err_d, s);
    }));
    for (int b = 0; b < B; ++b) {
        lenh[b] += 1;
        nexth[b] += 1;
    }
    return KVC_OK;
}


// kvc_prefill_suffix with device tensors; `check_finite` false skips the checked-mode
// scan (the host-buffer entry point scans its host inputs once for the whole call).
kvc_status prefill_impl(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k, const kvc_tensor* v,
                        const int32_t* start_pos, const int32_t* seqlen, const kvc_tensor* out, void* stream,
                        bool check_finite) {

    kvc_status st;
    if ((st = check_layer(h, layer)) != KVC_OK) return st;
    const int B = h->B(), Hq = h->Hq(), Hkv = h->Hkv(), D = h->D(), C = h->C();
    const int dt = h->cfg.dtype;
    // Appending without attending needs no query: q may then be NULL.
    const bool need_q = out != nullptr || q != nullptr;
    if (need_q && (st = check_tensor(h, q, "query", KVC_ERR_QUERY_SHAPE, dt, B, Hq, -1, D)) != KVC_OK) return st;
    if (!need_q && (st = check_tensor(h, k, "key", KVC_ERR_KEY_SHAPE, dt, B, Hkv, -1, D)) != KVC_OK) return st;
    const int64_t S64 = need_q ? q->shape[2] : k->shape[2];
    if (S64 > INT32_MAX) return fail(h, KVC_ERR_QUERY_SHAPE, "a chunk of %lld rows is too long", (long long)S64);
    const int S = (int)S64;
    if ((st = check_tensor(h, k, "key", KVC_ERR_KEY_SHAPE, dt, B, Hkv, S, D)) != KVC_OK) return st;
    if ((st = check_tensor(h, v, "value", KVC_ERR_VALUE_SHAPE, dt, B, Hkv, S, D)) != KVC_OK) return st;
    if (out && (st = check_tensor(h, out, "output", KVC_ERR_OUTPUT_SHAPE, out_dtype(dt), B, Hq, S, D)) != KVC_OK)
        return st;
    if ((st = refresh_mirrors(h)) != KVC_OK) return st;
    int32_t* lenh = &h->len_h[(size_t)layer * B];
    int32_t* nexth = &h->next_h[(size_t)layer * B];
    std::vector<int32_t> st_h(B), sl_h(B);
    for (int b = 0; b < B; ++b) {
        const int n = seqlen ? seqlen[b] : S;
        if (n < 0 || n > S)
            return fail(h, KVC_ERR_QUERY_SHAPE, "sequence %d declares %d rows, the chunk holds %d", b, n, S);
        const int p = start_pos ? start_pos[b] : nexth[b];
        if (lenh[b] + (int64_t)n > C)
            return fail(h, KVC_ERR_FULL, "sequence %d of layer %d holds %d rows; %d more exceed the capacity %d", b,
                        layer, lenh[b], n, C);
        if (p < 0 || (int64_t)p + n > (h->rope ? (int64_t)h->max_positions : (int64_t)INT32_MAX))
            return fail(h, KVC_ERR_POSITION, "sequence %d: positions %d .. %lld leave the %d-position table", b, p,
                        (long long)p + n - 1, h->max_positions);
        st_h[b] = p;
        sl_h[b] = n;
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    if (h->cfg.checked && check_finite) {
        const int64_t nk = (int64_t)B * Hkv * S * D;
        if ((st = check_nonfinite(h, k, v, nk, nk, s)) != KVC_OK) return st;
    }
    if (h->paged()) {
        std::vector<int32_t> to(B);
        for (int b = 0; b < B; ++b) to[b] = lenh[b] + sl_h[b];
        if ((st = ensure_blocks(h, lenh, to.data(), s)) != KVC_OK) return st;
    }
    // Attention kernel: the tensor-core tile kernel for bf16 with d_h = 128, else the generic one.
    const bool tc_ok = dt == KVC_BF16 && D == 128 && h->have_tmaps;
    if (out && h->opt_suffix_kernel >= 2 && !tc_ok)
        return fail(h, KVC_ERR_CONFIG, "the tensor-core suffix kernel needs bf16 storage and d_h = 128");
    const bool use_tc = out && tc_ok && !h->opt_force_generic && h->opt_suffix_kernel != 1;
    const bool use_tc2 = use_tc && h->opt_suffix_kernel == 3 && !h->paged();
    const bool use_tcp = use_tc && h->opt_suffix_kernel == 4 && !h->paged();
    std::vector<int4> work;
    if (use_tc2) {
        // one item per (sequence, query head, four 128-row query tiles): a pair of CTAs
        const int W = h->cfg.window;
        auto range = [&](int b, int qt, int& lo, int& hi) {
            if (qt * 128 >= sl_h[b]) { lo = hi = 0; return; }
            const int q_end = std::min(qt * 128 + 128, sl_h[b]);
            lo = W > 0 ? std::max(0, lenh[b] + qt * 128 - W + 1) / 128 : 0;
            hi = (lenh[b] + q_end + 127) / 128;
        };
        for (int b = 0; b < B; ++b)
            for (int hq = 0; hq < Hq; ++hq)
                for (int qd = 0; qd * 512 < sl_h[b]; ++qd) {
                    int wgt = 0;
                    for (int X = 0; X < 2; ++X) {
                        int l0, h0, l1, h1;
                        range(b, 4 * qd + 2 * X, l0, h0);
                        range(b, 4 * qd + 2 * X + 1, l1, h1);
                        if (h0 > 0) wgt += 2 * (std::max(h0, h1) - l0);
                    }
                    work.push_back(make_int4(b, hq, qd, wgt));
                }
        std::vector<int64_t> gw((size_t)B * Hq, 0);
        for (const int4& t : work) gw[(size_t)t.x * Hq + t.y] += t.w;
        std::stable_sort(work.begin(), work.end(), [&](const int4& x, const int4& y) {
            const int64_t wx = gw[(size_t)x.x * Hq + x.y], wy = gw[(size_t)y.x * Hq + y.y];
            if (wx != wy) return wx > wy;
            if (x.x != y.x) return x.x < y.x;
            if (x.y != y.y) return x.y < y.y;
            return x.w > y.w;
        });
        if ((uint64_t)B * Hq * S > (uint64_t)INT32_MAX)
            return fail(h, KVC_ERR_ELEMENT_OVERFLOW, "B * H_q * S must fit in 31 bits for the tile kernel");
    } else if (use_tc) {
        // one item per (sequence, query head, pair of 128-row query tiles); its weight is
        // the number of (query tile, key tile) products, key tiles from the window start
        // (tile 0 without a window) to the tile of the query tile's last row
        const int W = h->cfg.window;
        auto tiles_of = [&](int b, int qt) {
            if (qt * 128 >= sl_h[b]) return 0;
            const int q_end = std::min(qt * 128 + 128, sl_h[b]);
            const int j0 = W > 0 ? std::max(0, lenh[b] + qt * 128 - W + 1) / 128 : 0;
            return (lenh[b] + q_end + 127) / 128 - j0;
        };
        for (int b = 0; b < B; ++b)
            for (int hq = 0; hq < Hq; ++hq)
                for (int qp = 0; qp * 256 < sl_h[b]; ++qp)
                    work.push_back(make_int4(b, hq, qp, tiles_of(b, 2 * qp) + tiles_of(b, 2 * qp + 1)));
        // Group the query tiles of each (sequence, head) so they stream its K/V together
        // (L2 reuse); groups by total work, longest first; inside a group longest first.
        std::vector<int64_t> gw((size_t)B * Hq, 0);
        for (const int4& t : work) gw[(size_t)t.x * Hq + t.y] += t.w;
        std::stable_sort(work.begin(), work.end(), [&](const int4& x, const int4& y) {
            const int64_t wx = gw[(size_t)x.x * Hq + x.y], wy = gw[(size_t)y.x * Hq + y.y];
            if (wx != wy) return wx > wy;
            if (x.x != y.x) return x.x < y.x;
            if (x.y != y.y) return x.y < y.y;
            return x.w > y.w;
        });
        if ((uint64_t)B * Hq * S > (uint64_t)INT32_MAX)
            return fail(h, KVC_ERR_ELEMENT_OVERFLOW, "B * H_q * S must fit in 31 bits for the tile kernel");
    }
    // qrot scratch for the chunk: bf16 for the tile kernel, the accumulator dtype for the generic one
    const size_t acc = use_tc ? 2 : (dt == KVC_F64 ? 8 : 4);
    const size_t qbytes = (size_t)B * Hq * S * D * acc;
    if (out && qbytes > h->qrot_chunk_bytes) {
        cudaStreamSynchronize(s);
        cudaFree(h->qrot_chunk);
        h->qrot_chunk = nullptr;
        h->qrot_chunk_bytes = 0;
        if (cudaMalloc(&h->qrot_chunk, qbytes) != cudaSuccess) {
            cudaGetLastError();
            return fail(h, KVC_ERR_ALLOC, "cannot allocate %zu bytes of chunk scratch", qbytes);
        }
        h->qrot_chunk_bytes = qbytes;
    }
    const size_t arg_bytes = (2 * B * sizeof(int32_t) + 15) / 16 * 16;
    const size_t ring_bytes = arg_bytes + work.size() * sizeof(int4);
    void* hp;
    KVC_CUDA(h, h->ring.acquire(ring_bytes, &hp));
    memcpy(hp, st_h.data(), B * sizeof(int32_t));
    memcpy((int32_t*)hp + B, sl_h.data(), B * sizeof(int32_t));
    if (!work.empty()) memcpy((char*)hp + arg_bytes, work.data(), work.size() * sizeof(int4));
    void* dp;
    KVC_CUDA(h, h->ring.upload(ring_bytes, s, &dp));
    const int32_t* start_d = (const int32_t*)dp;
    const int32_t* seqlen_d = start_d + B;
    const int4* work_d = (const int4*)((const char*)dp + arg_bytes);

    AppendLaunch ap{};
    ap.q = out ? q->data : nullptr; ap.k = k->data; ap.v = v->data;
    ap.K = h->K_layer(layer); ap.V = h->V_layer(layer); ap.positions = h->pos_layer(layer);
    ap.slot0 = h->len_layer(layer); ap.pos0 = start_d; ap.seqlen = seqlen_d;
    ap.qrot = out ? h->qrot_chunk : nullptr; ap.qrot_kind = use_tc ? 2 : (dt == KVC_F64 ? 1 : 0);
    ap.rope = h->rope; ap.rope_f = h->rope_f; ap.err = h->err_d;
    ap.B = B; ap.Hq = out ? Hq : 0; ap.Hkv = Hkv; ap.S = S; ap.C = C; ap.d = D; ap.max_positions = h->max_positions;
    ap.kv = h->layout();
    // Without an output the query heads are skipped (Hq = 0 in the launch).
    KVC_CUDA(h, timed(h, KVC_KERNEL_ROPE_APPEND, s, [&] { return launch_rope_append(dt, ap, s); }));
    if (out && use_tc2 && !work.empty()) {
        SuffixLaunch2 sl{};
        if (!encode_rows_map(&sl.tmQ, h->qrot_chunk, (uint64_t)B * Hq * S, 128))
            return fail(h, KVC_ERR_CUDA, "cannot encode the query tensor map");
        sl.tmK64 = h->tmap_k[layer];
        sl.tmV128 = h->tmap_v128[layer];
        sl.slot0 = h->len_layer(layer); sl.seqlen = seqlen_d;
        sl.work = work_d; sl.n_work = (int)work.size();
        sl.out = (float*)out->data; sl.err = h->err_d;
        sl.B = B; sl.Hq = Hq; sl.Hkv = Hkv; sl.S = S; sl.C = C; sl.window = h->cfg.window;
        sl.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
        KVC_CUDA(h, timed(h, KVC_KERNEL_SUFFIX, s, [&] { return launch_suffix_tc2(sl, (int)work.size(), s); }));
    } else if (out && use_tc && !work.empty()) {
        SuffixLaunch sl{};
        if (!encode_rows_map(&sl.tmQ, h->qrot_chunk, (uint64_t)B * Hq * S, 128))
            return fail(h, KVC_ERR_CUDA, "cannot encode the query tensor map");
        // contiguous: 128-row boxes; paged: 64-row boxes, two per key tile
        sl.tmK = h->paged() ? h->tmap_k[layer] : h->tmap_k128[layer];
        sl.tmV = h->paged() ? h->tmap_v[layer] : h->tmap_v128[layer];
        sl.kv = h->layout();
        sl.slot0 = h->len_layer(layer); sl.seqlen = seqlen_d;
        sl.work = work_d; sl.n_work = (int)work.size(); sl.counter = h->work_counter;
        sl.out = (float*)out->data; sl.err = h->err_d;
        sl.B = B; sl.Hq = Hq; sl.Hkv = Hkv; sl.S = S; sl.C = C; sl.window = h->cfg.window;
        sl.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
        if (use_tcp) {
            const int sms = sm_count(h->cfg.device);
            KVC_CUDA(h, timed(h, KVC_KERNEL_SUFFIX, s, [&] { return launch_suffix_tcp(sl, sms, s); }));
        } else {
            const int split = h->opt_suffix_kernel == 5 ? 2 : 1;
            KVC_CUDA(h, timed(h, KVC_KERNEL_SUFFIX, s,
                              [&] { return launch_suffix_tc(sl, (int)work.size(), s, split); }));
        }
    } else if (out && !use_tc) {
        GenericAttendLaunch g{};
        g.qrot = h->qrot_chunk; g.K = h->K_layer(layer); g.V = h->V_layer(layer);
        g.slot0 = h->len_layer(layer); g.seqlen = seqlen_d; g.out = out->data;
        g.B = B; g.Hq = Hq; g.Hkv = Hkv; g.S = S; g.C = C; g.d = D; g.window = h->cfg.window; g.kv = h->layout(); g.err = h->err_d;
        KVC_CUDA(h, timed(h, KVC_KERNEL_GENERIC_ATTEND, s, [&] { return launch_attend_generic(dt, g, s); }));
    }
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] {
        return launch_commit(h->len_layer(layer), h->next_layer(layer), start_d, seqlen_d, S, B, C, h->err_d, s);
    }));
    KVC_CUDA(h, h->ring.release(s));
    for (int b = 0; b < B; ++b) {
        lenh[b] += sl_h[b];
        nexth[b] = st_h[b] + sl_h[b];
    }
    h->layer_version[layer] += 1;
    return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_append_attend(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k,
                             const kvc_tensor* v, const kvc_tensor* out, void* stream) {
    return append_attend_impl(h, layer, q, k, v, out, true, stream);
}

kvc_status kvc_prepare_attend(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k,
                              const kvc_tensor* v, const kvc_tensor* out, kvc_ticket* ticket, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    if (!ticket) return fail(h, KVC_ERR_NULL, "ticket pointer is NULL");
    kvc_status st = append_attend_impl(h, layer, q, k, v, out, false, stream);
    if (st != KVC_OK) return st;
    ticket->handle = h;
    ticket->layer = layer;
    ticket->reserved = 0;
    ticket->version = h->layer_version[layer];
    return KVC_OK;
}

kvc_status kvc_commit(kvc_handle* h, const kvc_ticket* tickets, int32_t n, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    if (n < 0) return fail(h, KVC_ERR_TICKET, "ticket count %d is negative", n);
    if (n > 0 && !tickets) return fail(h, KVC_ERR_NULL, "ticket array is NULL");
    const int L = h->cfg.layers, B = h->B();
    std::vector<char> seen(L, 0);
    for (int i = 0; i < n; ++i) {
        const kvc_ticket& t = tickets[i];
        if (t.handle != h) return fail(h, KVC_ERR_TICKET, "ticket %d was prepared by another cache", i);
        if (t.layer < 0 || t.layer >= L) return fail(h, KVC_ERR_TICKET, "ticket %d names layer %d", i, t.layer);
        if (seen[t.layer]) return fail(h, KVC_ERR_TICKET, "tickets repeat layer %d", t.layer);
        seen[t.layer] = 1;
        if (t.version != h->layer_version[t.layer])
            return fail(h, KVC_ERR_TICKET, "ticket %d of layer %d is stale: the layer changed after it was prepared",
                        i, t.layer);
    }
    if (n == 0) return KVC_OK;
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    for (int i0 = 0; i0 < n; i0 += kCommitMaxLayers) {
        CommitLayers cl{};
        cl.n = std::min(n - i0, kCommitMaxLayers);
        for (int i = 0; i < cl.n; ++i) cl.layer[i] = tickets[i0 + i].layer;
        KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] { return launch_commit_layers(h->len_d, h->next_d, cl, B, h->C(), h->err_d, s); }));
    }
    for (int i = 0; i < n; ++i) {
        const int l = tickets[i].layer;
        h->layer_version[l] += 1;
        for (int b = 0; b < B; ++b) {
            h->len_h[(size_t)l * B + b] += 1;
            h->next_h[(size_t)l * B + b] += 1;
        }
    }
    return KVC_OK;
}

kvc_status kvc_prefill_suffix(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k,
                              const kvc_tensor* v, const int32_t* start_pos, const int32_t* seqlen,
                              const kvc_tensor* out, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    return kvc::prefill_impl(h, layer, q, k, v, start_pos, seqlen, out, stream, true);
}

// ---------------------------------------------------------------- host-buffer prefill

namespace {

// Shape, dtype and alignment of a [B, H, S?, d] tensor in HOST memory (pinned or pageable).
kvc_status check_host_tensor(kvc_handle* h, const kvc_tensor* t, const char* name, kvc_status shape_err, int dtype,
                             int64_t d0, int64_t d1, int64_t d2, int64_t d3) {
    if (!t || !t->data) return fail(h, KVC_ERR_NULL, "%s tensor or its data pointer is NULL", name);
    if (t->dtype != dtype)
        return fail(h, KVC_ERR_DTYPE, "%s has dtype %s, the cache expects %s", name, dtype_name(t->dtype),
                    dtype_name(dtype));
    const int64_t want[4] = {d0, d1, d2, d3};
    bool ok = t->ndim == 4;
    for (int i = 0; ok && i < 4; ++i) ok = want[i] < 0 ? t->shape[i] > 0 : t->shape[i] == want[i];
    if (!ok) {
        int64_t shown[4];
        for (int i = 0; i < 4; ++i) shown[i] = want[i] < 0 ? -1 : want[i];
        return fail(h, shape_err, "%s must have shape %s, got %s", name, shape_str(shown, 4).c_str(),
                    shape_str(t->shape, t->ndim < 0 ? 0 : (t->ndim > 4 ? 4 : t->ndim)).c_str());
    }
    if (((uintptr_t)t->data & 15u) != 0)
        return fail(h, KVC_ERR_CONFIG, "%s data pointer is not 16-byte aligned", name);
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, t->data) != cudaSuccess) {
        cudaGetLastError();   // older drivers: an unregistered host pointer
        return KVC_OK;
    }
    if (attr.type == cudaMemoryTypeDevice)
        return fail(h, KVC_ERR_CONFIG, "%s data is device memory; the host-buffer call takes host memory", name);
    return KVC_OK;
}

// First non-finite element of `n` host elements of the storage dtype, or -1.
int64_t first_nonfinite_host(const void* p, int64_t n, int dtype) {
    if (dtype == KVC_BF16) {
        const uint16_t* u = (const uint16_t*)p;
        for (int64_t i = 0; i < n; ++i)
            if ((u[i] & 0x7f80u) == 0x7f80u) return i;
    } else if (dtype == KVC_F32) {
        const uint32_t* u = (const uint32_t*)p;
        for (int64_t i = 0; i < n; ++i)
            if ((u[i] & 0x7f800000u) == 0x7f800000u) return i;
    } else {
        const uint64_t* u = (const uint64_t*)p;
        for (int64_t i = 0; i < n; ++i)
            if ((u[i] & 0x7ff0000000000000ull) == 0x7ff0000000000000ull) return i;
    }
    return -1;
}

// Rows 0 .. n-1 of every head of the sequences seqs[0 .. count) of a [B, H, S, d] tensor:
// one strided copy per sequence (H runs of n rows, S rows apart).
cudaError_t copy_rows(char* dst, const char* src, const int* seqs, int count, const int32_t* n, int H, int S,
                      size_t row_bytes, cudaMemcpyKind kind, cudaStream_t st) {
    const size_t pitch = (size_t)S * row_bytes;
    for (int i = 0; i < count; ++i) {
        const int b = seqs[i];
        if (n[b] == 0) continue;
        const size_t off = (size_t)b * H * pitch;
        cudaError_t e = cudaMemcpy2DAsync(dst + off, pitch, src + off, pitch, (size_t)n[b] * row_bytes, (size_t)H,
                                          kind, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

kvc_status kvc_prefill_suffix_host(kvc_handle* h, int32_t layer, const kvc_tensor* q, const kvc_tensor* k,
                                   const kvc_tensor* v, const int32_t* start_pos, const int32_t* seqlen,
                                   const kvc_tensor* out, int32_t chunk_sequences, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    kvc_status st;
    if ((st = check_layer(h, layer)) != KVC_OK) return st;
    if (chunk_sequences < 0) return fail(h, KVC_ERR_CONFIG, "chunk_sequences is %d, must be >= 0", chunk_sequences);
    const int B = h->B(), Hq = h->Hq(), Hkv = h->Hkv(), D = h->D(), C = h->C();
    const int dt = h->cfg.dtype;
    const bool need_q = out != nullptr || q != nullptr;
    if (need_q && (st = check_host_tensor(h, q, "query", KVC_ERR_QUERY_SHAPE, dt, B, Hq, -1, D)) != KVC_OK) return st;
    if (!need_q && (st = check_host_tensor(h, k, "key", KVC_ERR_KEY_SHAPE, dt, B, Hkv, -1, D)) != KVC_OK) return st;
    const int64_t S64 = need_q ? q->shape[2] : k->shape[2];
    if (S64 > INT32_MAX) return fail(h, KVC_ERR_QUERY_SHAPE, "a chunk of %lld rows is too long", (long long)S64);
    const int S = (int)S64;
    if ((st = check_host_tensor(h, k, "key", KVC_ERR_KEY_SHAPE, dt, B, Hkv, S, D)) != KVC_OK) return st;
    if ((st = check_host_tensor(h, v, "value", KVC_ERR_VALUE_SHAPE, dt, B, Hkv, S, D)) != KVC_OK) return st;
    if (out && (st = check_host_tensor(h, out, "output", KVC_ERR_OUTPUT_SHAPE, out_dtype(dt), B, Hq, S, D)) != KVC_OK)
        return st;
    if ((st = refresh_mirrors(h)) != KVC_OK) return st;
    // The whole call is checked before any copy or launch, as kvc_prefill_suffix checks it.
    const int32_t* lenh = &h->len_h[(size_t)layer * B];
    const int32_t* nexth = &h->next_h[(size_t)layer * B];
    std::vector<int32_t> sl(B), sp(B);
    for (int b = 0; b < B; ++b) {
        const int n = seqlen ? seqlen[b] : S;
        if (n < 0 || n > S)
            return fail(h, KVC_ERR_QUERY_SHAPE, "sequence %d declares %d rows, the chunk holds %d", b, n, S);
        const int p = start_pos ? start_pos[b] : nexth[b];
        if (lenh[b] + (int64_t)n > C)
            return fail(h, KVC_ERR_FULL, "sequence %d of layer %d holds %d rows; %d more exceed the capacity %d", b,
                        layer, lenh[b], n, C);
        if (p < 0 || (int64_t)p + n > (h->rope ? (int64_t)h->max_positions : (int64_t)INT32_MAX))
            return fail(h, KVC_ERR_POSITION, "sequence %d: positions %d .. %lld leave the %d-position table", b, p,
                        (long long)p + n - 1, h->max_positions);
        sl[b] = n;
        sp[b] = p;
    }
    if (h->paged()) {
        // counted for the whole call as one kvc_prefill_suffix counts it (an upper bound on
        // what the chunks take one after another), so no chunk can run out of blocks
        std::vector<int32_t> to(B);
        for (int b = 0; b < B; ++b) to[b] = lenh[b] + sl[b];
        const int64_t need = blocks_needed(h, lenh, to.data());
        if (need > (int64_t)h->free_blocks.size())
            return fail(h, KVC_ERR_FULL, "the block pool has %zu free blocks; the call needs %lld",
                        h->free_blocks.size(), (long long)need);
    }
    const size_t esz = h->elem_size, osz = out_dtype(dt) == KVC_F64 ? 8 : 4;
    const size_t row_bytes = (size_t)D * esz;
    if (h->cfg.checked) {
        const int64_t nkv = (int64_t)B * Hkv * S * D;
        for (int which = 0; which < 2; ++which) {
            const int64_t idx = first_nonfinite_host(which ? v->data : k->data, nkv, dt);
            if (idx >= 0)
                return fail(h, which ? KVC_ERR_NONFINITE_VALUE : KVC_ERR_NONFINITE_KEY,
                            "%s element at flat index %lld is not finite; nothing was appended",
                            which ? "value" : "key", (long long)idx);
        }
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    // Device staging: q, k, v and the output, each laid out like the caller's buffer.
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t qb = need_q ? al((size_t)B * Hq * S * row_bytes) : 0;
    const size_t kb = al((size_t)B * Hkv * S * row_bytes);
    const size_t ob = out ? al((size_t)B * Hq * S * D * osz) : 0;
    const size_t total = qb + 2 * kb + ob;
    if (total > h->io_bytes) {
        if (h->io_h2d) KVC_CUDA(h, cudaStreamSynchronize(h->io_h2d));
        if (h->io_d2h) KVC_CUDA(h, cudaStreamSynchronize(h->io_d2h));
        KVC_CUDA(h, cudaStreamSynchronize(s));
        cudaFree(h->io_buf);
        h->io_buf = nullptr;
        h->io_bytes = 0;
        if (cudaMalloc(&h->io_buf, total) != cudaSuccess) {
            cudaGetLastError();
            return fail(h, KVC_ERR_ALLOC, "cannot allocate %zu bytes of staging for host buffers", total);
        }
        h->io_bytes = total;
    }
    if (!h->io_h2d) {
        KVC_CUDA(h, cudaStreamCreateWithFlags(&h->io_h2d, cudaStreamNonBlocking));
        KVC_CUDA(h, cudaStreamCreateWithFlags(&h->io_d2h, cudaStreamNonBlocking));
        KVC_CUDA(h, cudaEventCreateWithFlags(&h->io_entry, cudaEventDisableTiming));
        KVC_CUDA(h, cudaEventCreateWithFlags(&h->io_last, cudaEventDisableTiming));
        KVC_CUDA(h, cudaEventRecord(h->io_last, h->io_d2h));
    }
    const int cs = chunk_sequences > 0 ? std::min(chunk_sequences, B) : std::max(1, (B + 7) / 8);
    const int nchunks = (B + cs - 1) / cs;
    // Stage order: the pipeline waits for the first stage's upload before any work and for
    // the last stage's download after all of it, so the smallest sequence goes first, the
    // second smallest last, and the others largest first in between (the results do not
    // depend on the order: sequences are independent).
    std::vector<int> order(B);
    for (int b = 0; b < B; ++b) order[b] = b;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return sl[x] < sl[y]; });
    if (B > 2) {
        std::vector<int> o2;
        o2.push_back(order[0]);
        for (int i = B - 1; i >= 2; --i) o2.push_back(order[i]);
        o2.push_back(order[1]);
        order.swap(o2);
    }
    while ((int)h->io_ev.size() < 2 * nchunks) {
        cudaEvent_t e;
        KVC_CUDA(h, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        h->io_ev.push_back(e);
    }
    char* dq = (char*)h->io_buf;
    char* dk = dq + qb;
    char* dv = dk + kb;
    char* dout = dv + kb;
    // The staging is rewritten only after the caller's earlier work and the previous
    // call's output copies are done.
    KVC_CUDA(h, cudaEventRecord(h->io_entry, s));
    KVC_CUDA(h, cudaStreamWaitEvent(h->io_h2d, h->io_entry, 0));
    KVC_CUDA(h, cudaStreamWaitEvent(h->io_h2d, h->io_last, 0));
    // 1. every chunk's inputs, in chunk order, on the upload stream
    for (int c = 0; c < nchunks; ++c) {
        const int i0 = c * cs, i1 = std::min(B, i0 + cs);
        if (need_q)
            KVC_CUDA(h, copy_rows(dq, (const char*)q->data, order.data() + i0, i1 - i0, sl.data(), Hq, S, row_bytes,
                                  cudaMemcpyHostToDevice, h->io_h2d));
        KVC_CUDA(h, copy_rows(dk, (const char*)k->data, order.data() + i0, i1 - i0, sl.data(), Hkv, S, row_bytes,
                              cudaMemcpyHostToDevice, h->io_h2d));
        KVC_CUDA(h, copy_rows(dv, (const char*)v->data, order.data() + i0, i1 - i0, sl.data(), Hkv, S, row_bytes,
                              cudaMemcpyHostToDevice, h->io_h2d));
        KVC_CUDA(h, cudaEventRecord(h->io_ev[2 * c], h->io_h2d));
    }
    // 2. each chunk's append and attention on the caller's stream once its inputs have
    //    landed (the other sequences take 0 rows), then its output rows on the download stream
    kvc_tensor tq{}, tk{}, tv{}, to{};
    if (need_q) { tq = *q; tq.data = dq; }
    tk = *k; tk.data = dk;
    tv = *v; tv.data = dv;
    if (out) { to = *out; to.data = dout; }
    std::vector<int32_t> sl_c(B), sp_c(B);
    std::vector<char> in_stage(B);
    for (int c = 0; c < nchunks; ++c) {
        const int i0 = c * cs, i1 = std::min(B, i0 + cs);
        std::fill(in_stage.begin(), in_stage.end(), 0);
        for (int i = i0; i < i1; ++i) in_stage[order[i]] = 1;
        int rows = 0;
        for (int b = 0; b < B; ++b) {
            const bool in = in_stage[b] != 0;
            sl_c[b] = in ? sl[b] : 0;
            sp_c[b] = in ? sp[b] : h->next_h[(size_t)layer * B + b];
            rows += sl_c[b];
        }
        if (rows == 0) continue;
        KVC_CUDA(h, cudaStreamWaitEvent(s, h->io_ev[2 * c], 0));
        // the stage's small argument arrays must not wait behind the bulk uploads on the
        // copy engine: the SMs read them from the mapped ring slot instead
        h->ring.by_kernel = true;
        st = kvc::prefill_impl(h, layer, need_q ? &tq : nullptr, &tk, &tv, sp_c.data(), sl_c.data(),
                               out ? &to : nullptr, s, false);
        h->ring.by_kernel = false;
        if (st != KVC_OK) return st;
        if (out) {
            KVC_CUDA(h, cudaEventRecord(h->io_ev[2 * c + 1], s));
            KVC_CUDA(h, cudaStreamWaitEvent(h->io_d2h, h->io_ev[2 * c + 1], 0));
            KVC_CUDA(h, copy_rows((char*)out->data, dout, order.data() + i0, i1 - i0, sl.data(), Hq, S,
                                  (size_t)D * osz, cudaMemcpyDeviceToHost, h->io_d2h));
        }
    }
    // io_last follows every launch and output copy of this call (the next call's uploads
    // wait for it before they overwrite the staging); the caller's stream waits for it too,
    // so that its completion means the output rows are in host memory
    KVC_CUDA(h, cudaEventRecord(h->io_entry, s));
    KVC_CUDA(h, cudaStreamWaitEvent(h->io_d2h, h->io_entry, 0));
    KVC_CUDA(h, cudaEventRecord(h->io_last, h->io_d2h));
    KVC_CUDA(h, cudaStreamWaitEvent(s, h->io_last, 0));
    return KVC_OK;
}

kvc_status kvc_reset(kvc_handle* h, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    const size_t n = (size_t)h->cfg.layers * h->B();
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    KVC_CUDA(h, cudaMemsetAsync(h->len_d, 0, n * sizeof(int32_t), s));
    KVC_CUDA(h, cudaMemsetAsync(h->next_d, 0, n * sizeof(int32_t), s));
    KVC_CUDA(h, cudaMemsetAsync(h->lane_ticket, 0, (size_t)h->B() * h->Hkv() * sizeof(unsigned), s));
    KVC_CUDA(h, cudaMemsetAsync(h->err_d, 0, sizeof(uint32_t), s));
    for (int b = 0; b < h->B(); ++b) release_blocks(h, b, 0);
    kvc_status st = upload_table(h, s);
    if (st != KVC_OK) return st;
    std::fill(h->len_h.begin(), h->len_h.end(), 0);
    std::fill(h->next_h.begin(), h->next_h.end(), 0);
    for (auto& v : h->layer_version) v += 1;
    h->mirrors_stale = false;
    return KVC_OK;
}

kvc_status kvc_truncate(kvc_handle* h, const int32_t* cut, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    if (!cut) return fail(h, KVC_ERR_NULL, "cut array is NULL");
    const int B = h->B(), L = h->cfg.layers;
    // With device lengths the kernel checks cut <= length itself (no synchronisation).
    const bool dev_len = h->opt_device_lengths != 0;
    for (int b = 0; b < B; ++b) {
        if (cut[b] < 0) return fail(h, KVC_ERR_CUT, "cut %d of sequence %d is negative", cut[b], b);
        for (int l = 0; l < L && !dev_len; ++l)
            if (cut[b] > h->len_h[(size_t)l * B + b])
                return fail(h, KVC_ERR_CUT, "cut %d of sequence %d exceeds its length %d in layer %d", cut[b], b,
                            h->len_h[(size_t)l * B + b], l);
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    void* hp;
    KVC_CUDA(h, h->ring.acquire(B * sizeof(int32_t), &hp));
    memcpy(hp, cut, B * sizeof(int32_t));
    void* dp;
    KVC_CUDA(h, h->ring.upload(B * sizeof(int32_t), s, &dp));
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] {
        return dev_len ? launch_truncate_checked(h->len_d, h->next_d, (const int32_t*)dp, L, B, h->err_d, s)
                       : launch_truncate(h->len_d, h->next_d, (const int32_t*)dp, L, B, s);
    }));
    KVC_CUDA(h, h->ring.release(s));
    for (int b = 0; b < B; ++b) release_blocks(h, b, cut[b]);
    kvc_status ust = upload_table(h, s);
    if (ust != KVC_OK) return ust;
    for (int l = 0; l < L; ++l) {
        h->layer_version[l] += 1;
        for (int b = 0; b < B; ++b) {
            h->len_h[(size_t)l * B + b] = cut[b];
            h->next_h[(size_t)l * B + b] = cut[b];
        }
    }
    return KVC_OK;
}

kvc_status kvc_lcp(const int32_t* cached, int64_t n, const int32_t* query, int64_t m, int32_t* cut) {
    if (!cut) return KVC_ERR_NULL;
    if (m <= 0) return KVC_ERR_EMPTY_QUERY;
    if (!query || (n > 0 && !cached) || n < 0) return KVC_ERR_NULL;
    int64_t L = 0;
    const int64_t lim = std::min(n, m);
    while (L < lim && cached[L] == query[L]) ++L;
    const int64_t c = std::min(L, m - 1);
    if (c > INT32_MAX) return KVC_ERR_CUT;
    *cut = (int32_t)c;
    return KVC_OK;
}

kvc_status kvc_lcp_window(const int32_t* cached, int64_t n, const int32_t* query, int64_t m, int32_t window,
                          int32_t* cut) {
    if (window < 0) return KVC_ERR_CONFIG;
    if (window == 0) return kvc_lcp(cached, n, query, m, cut);
    if (!cut) return KVC_ERR_NULL;
    if (m <= 0) return KVC_ERR_EMPTY_QUERY;
    if (!query || (n > 0 && !cached) || n < 0) return KVC_ERR_NULL;
    int64_t L = 0;
    const int64_t lim = std::min(n, m);
    while (L < lim && cached[L] == query[L]) ++L;
    // the window is reused whole or not at all
    const int64_t c = (L == n && m > n) ? n : 0;
    if (c > INT32_MAX) return KVC_ERR_CUT;
    *cut = (int32_t)c;
    return KVC_OK;
}

kvc_status kvc_get_lengths(const kvc_handle* h, int32_t layer, int32_t* lengths, int32_t* next_positions) {
    if (!h) return KVC_ERR_NULL;
    if (layer < 0 || layer >= h->cfg.layers) return KVC_ERR_LAYER;
    const int B = h->B();
    if (lengths) memcpy(lengths, &h->len_h[(size_t)layer * B], B * sizeof(int32_t));
    if (next_positions) memcpy(next_positions, &h->next_h[(size_t)layer * B], B * sizeof(int32_t));
    return KVC_OK;
}

kvc_status kvc_get_len(const kvc_handle* h, int32_t layer, int32_t* len_B) {
    if (!len_B) return KVC_ERR_NULL;
    return kvc_get_lengths(h, layer, len_B, nullptr);
}

kvc_status kvc_read_rows(kvc_handle* h, int32_t layer, const kvc_tensor* keys, const kvc_tensor* values,
                         int32_t* positions, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    kvc_status st;
    if ((st = check_layer(h, layer)) != KVC_OK) return st;
    if (!keys && !values) return fail(h, KVC_ERR_NULL, "keys and values are both NULL");
    const int B = h->B(), Hkv = h->Hkv(), D = h->D(), dt = h->cfg.dtype;
    const kvc_tensor* first = keys ? keys : values;
    if (first->ndim != 4 || first->shape[2] < 1 || first->shape[2] > h->C())
        return fail(h, KVC_ERR_KEY_SHAPE, "the snapshot must have shape [%d, %d, R, %d] with 1 <= R <= %d", B, Hkv, D,
                    h->C());
    const int R = (int)first->shape[2];
    if (keys && (st = check_tensor(h, keys, "keys", KVC_ERR_KEY_SHAPE, dt, B, Hkv, R, D)) != KVC_OK) return st;
    if (values && (st = check_tensor(h, values, "values", KVC_ERR_VALUE_SHAPE, dt, B, Hkv, R, D)) != KVC_OK)
        return st;
    if (positions) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, positions) != cudaSuccess) {
            cudaGetLastError();
            return fail(h, KVC_ERR_CONFIG, "positions pointer is not a CUDA allocation");
        }
        if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
            attr.device != h->cfg.device)
            return fail(h, KVC_ERR_CONFIG, "positions must be device memory of GPU %d", h->cfg.device);
        if ((uintptr_t)positions & 3u) return fail(h, KVC_ERR_CONFIG, "positions pointer is not 4-byte aligned");
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s, [&] {
        return launch_read_rows(h->K_layer(layer), h->V_layer(layer), h->pos_layer(layer), h->len_layer(layer),
                                h->layout(), keys ? keys->data : nullptr, values ? values->data : nullptr,
                                positions, B, Hkv, R, (int)(D * h->elem_size), s);
    }));
    return KVC_OK;
}

kvc_status kvc_share_prefix(kvc_handle* h, int32_t dst, int32_t src, int32_t rows, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    if (!h->paged()) return fail(h, KVC_ERR_CONFIG, "sharing a prefix needs paged storage (block_rows > 0)");
    const int B = h->B(), L = h->cfg.layers, P = h->cfg.block_rows;
    if (dst < 0 || dst >= B || src < 0 || src >= B || dst == src)
        return fail(h, KVC_ERR_CONFIG, "sequences %d <- %d: need two distinct indices in [0, %d)", dst, src, B);
    for (int l = 0; l < L; ++l) {
        if (h->len_h[(size_t)l * B + dst] != 0)
            return fail(h, KVC_ERR_CUT, "sequence %d holds %d rows in layer %d; it must be empty", dst,
                        h->len_h[(size_t)l * B + dst], l);
        if (rows < 0 || rows > h->len_h[(size_t)l * B + src])
            return fail(h, KVC_ERR_CUT, "%d rows exceed the %d rows of sequence %d in layer %d", rows,
                        h->len_h[(size_t)l * B + src], src, l);
    }
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    release_blocks(h, dst, 0);        // blocks a prepared, uncommitted step may have taken
    for (int j = 0; j < (rows + P - 1) / P; ++j) {
        const int blk = h->table_h[(size_t)src * h->nblk + j];
        h->table_h[(size_t)dst * h->nblk + j] = blk;
        h->refcnt[blk] += 1;
        h->table_dirty = true;
    }
    kvc_status st = upload_table(h, s);
    if (st != KVC_OK) return st;
    const int C = h->C();
    for (int l = 0; l < L && rows > 0; ++l)
        KVC_CUDA(h, cudaMemcpyAsync(h->pos_layer(l) + (size_t)dst * C, h->pos_layer(l) + (size_t)src * C,
                                    (size_t)rows * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    KVC_CUDA(h, timed(h, KVC_KERNEL_BOOKKEEPING, s,
                      [&] { return launch_set_lengths(h->len_d, h->next_d, L, B, dst, rows, s); }));
    for (int l = 0; l < L; ++l) {
        h->len_h[(size_t)l * B + dst] = rows;
        h->next_h[(size_t)l * B + dst] = rows;
        h->layer_version[l] += 1;
    }
    return KVC_OK;
}

kvc_status kvc_block_table(const kvc_handle* h, int32_t* table, int32_t* free_blocks) {
    if (!h) return KVC_ERR_NULL;
    if (!h->paged()) return KVC_ERR_CONFIG;
    if (table) memcpy(table, h->table_h.data(), h->table_h.size() * sizeof(int32_t));
    if (free_blocks) *free_blocks = (int32_t)h->free_blocks.size();
    return KVC_OK;
}

kvc_status kvc_sync_lengths(kvc_handle* h) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    return refresh_mirrors(h);
}

kvc_status kvc_get_config(const kvc_handle* h, kvc_config* out) {
    if (!h || !out) return KVC_ERR_NULL;
    *out = h->cfg;
    return KVC_OK;
}

kvc_status kvc_storage(const kvc_handle* h, int32_t layer, void** keys, void** values, int32_t** positions) {
    if (!h) return KVC_ERR_NULL;
    if (layer < 0 || layer >= h->cfg.layers) return KVC_ERR_LAYER;
    if (keys) *keys = h->K_layer(layer);
    if (values) *values = h->V_layer(layer);
    if (positions) *positions = h->pos_layer(layer);
    return KVC_OK;
}

kvc_status kvc_check(kvc_handle* h, void* stream) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    KVC_CUDA(h, cudaStreamSynchronize(s));
    const size_t n = (size_t)h->cfg.layers * h->B();
    std::vector<int32_t> len(n), next(n);
    uint32_t err = 0;
    KVC_CUDA(h, cudaMemcpy(len.data(), h->len_d, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    KVC_CUDA(h, cudaMemcpy(next.data(), h->next_d, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    KVC_CUDA(h, cudaMemcpy(&err, h->err_d, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    // reported once: kernels stop early while the word is set, so it is cleared here
    if (err) KVC_CUDA(h, cudaMemset(h->err_d, 0, sizeof(uint32_t)));
    if (err)
        return fail(h, KVC_ERR_DEVICE,
                    "device error word 0x%x (1: slot out of range, 2: bounded wait timed out, 4: tensor memory, "
                    "8: cache full or position beyond the table in a device-length step, "
                    "16: cut beyond a length in a device-checked truncate, "
                    "32: debug-build bounds check skipped an access)",
                    err);
    if (h->mirrors_stale || h->opt_device_lengths) {
        h->len_h = len;
        h->next_h = next;
        h->mirrors_stale = false;
    }
    for (size_t i = 0; i < n; ++i)
        if (len[i] != h->len_h[i] || next[i] != h->next_h[i])
            return fail(h, KVC_ERR_DEVICE, "device length/next position (%d, %d) of entry %zu differ from the host (%d, %d)",
                        len[i], next[i], i, h->len_h[i], h->next_h[i]);
    return KVC_OK;
}

// KVC_OPT_TEST_POISON: every storage row that no sequence holds -- slot >= length in
// contiguous storage; past the held rows of a block, or the whole of a free block, in
// paged storage -- gets keys 0 and values 1e4 (in the storage dtype), in every layer.
static kvc_status poison_unheld_rows(kvc_handle* h) {
    kvc_status st = refresh_mirrors(h);
    if (st != KVC_OK) return st;
    const int L = h->cfg.layers, B = h->B(), Hkv = h->Hkv();
    const int groups = h->paged() ? h->nblocks : B;
    const int R = h->paged() ? h->cfg.block_rows : h->C();
    std::vector<int32_t> live((size_t)L * groups, 0);
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b) {
            const int n = h->len_h[(size_t)l * B + b];
            if (!h->paged()) {
                live[(size_t)l * groups + b] = n;
                continue;
            }
            for (int j = 0; j < h->nblk; ++j) {
                const int blk = h->table_h[(size_t)b * h->nblk + j];
                if (blk < 0) continue;
                const int held = std::max(0, std::min(R, n - j * R));
                int32_t& x = live[(size_t)l * groups + blk];
                x = std::max(x, held);
            }
        }
    unsigned long long vbits = 0;
    if (h->cfg.dtype == KVC_F64) { const double v = 1e4; memcpy(&vbits, &v, 8); }
    else if (h->cfg.dtype == KVC_F32) { const float v = 1e4f; uint32_t u; memcpy(&u, &v, 4); vbits = u; }
    else vbits = 0x461c;   // 1e4 rounded to bf16 (9984)
    int32_t* live_d = nullptr;
    KVC_CUDA(h, cudaSetDevice(h->cfg.device));
    KVC_CUDA(h, cudaDeviceSynchronize());
    KVC_CUDA(h, cudaMalloc((void**)&live_d, live.size() * sizeof(int32_t)));
    cudaError_t e = cudaMemcpy(live_d, live.data(), live.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = launch_poison(h->K, h->V, h->layer_elems * h->elem_size, live_d, L, groups, Hkv, R, h->D(),
                          (int)h->elem_size, vbits, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    cudaFree(live_d);
    if (e != cudaSuccess) return cuda_fail(h, e, "poisoning unheld rows");
    return KVC_OK;
}

kvc_status kvc_set_option(kvc_handle* h, int32_t option, int64_t value) {
    if (!h && option == KVC_OPT_TEST_STALL) {
        // no handle: the next kvc_decode_attend_noalloc call stalls (test only)
        if (value) noalloc_arm_test_stall();
        return KVC_OK;
    }
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    switch (option) {
        case KVC_OPT_TEST_POISON:
            return value ? poison_unheld_rows(h) : KVC_OK;
        case KVC_OPT_TEST_PLANT_LENGTH: {
#ifdef KVC_DEBUG
            if (value < INT32_MIN || value > INT32_MAX) return fail(h, KVC_ERR_CONFIG, "planted length out of range");
            const int32_t v = (int32_t)value;
            KVC_CUDA(h, cudaSetDevice(h->cfg.device));
            KVC_CUDA(h, cudaDeviceSynchronize());
            KVC_CUDA(h, cudaMemcpy(h->len_d, &v, sizeof(v), cudaMemcpyHostToDevice));
            KVC_CUDA(h, cudaMemcpy(h->next_d, &v, sizeof(v), cudaMemcpyHostToDevice));
            return KVC_OK;
#else
            return fail(h, KVC_ERR_CONFIG, "planting a device length needs the debug build (libkvc_debug.so)");
#endif
        }
        case KVC_OPT_DECODE_SPLIT_ROWS:
            if (value < 0 || value % 64 || value > (int64_t)1 << 30)
                return fail(h, KVC_ERR_CONFIG, "decode split rows must be 0 or a positive multiple of 64, got %lld",
                            (long long)value);
            h->opt_split_rows = value;
            return KVC_OK;
        case KVC_OPT_FORCE_GENERIC:
            h->opt_force_generic = value != 0;
            return KVC_OK;
        case KVC_OPT_SUFFIX_KERNEL:
            if (value < 0 || value > 5) return fail(h, KVC_ERR_CONFIG, "suffix kernel must be 0 .. 5");
            h->opt_suffix_kernel = value;
            return KVC_OK;
        case KVC_OPT_TIMING:
            h->timing = value != 0;
            return KVC_OK;
        case KVC_OPT_DECODE_FUSED:
            h->opt_decode_fused = value != 0;
            return KVC_OK;
        case KVC_OPT_TEST_STALL:
            h->opt_test_stall = value != 0;
            return KVC_OK;
        case KVC_OPT_DECODE_PDL:
            h->opt_decode_pdl = value != 0;
            return KVC_OK;
        case KVC_OPT_DECODE_TC:
            h->opt_decode_tc = value != 0;
            return KVC_OK;
        case KVC_OPT_DECODE_LANES:
            h->opt_decode_lanes = value != 0;
            return KVC_OK;
        case KVC_OPT_DECODE_STREAMK:
            h->opt_decode_streamk = value != 0;
            return KVC_OK;
        case KVC_OPT_DEVICE_LENGTHS: {
            if (value && h->paged())
                return fail(h, KVC_ERR_CONFIG, "device-held lengths need contiguous storage (blocks are taken on the host)");
            kvc_status st = refresh_mirrors(h);
            if (st != KVC_OK) return st;
            h->opt_device_lengths = value != 0;
            return KVC_OK;
        }
    }
    return fail(h, KVC_ERR_CONFIG, "unknown option %d", option);
}

kvc_status kvc_kernel_stats(kvc_handle* h, int32_t kernel, double* total_ms, int64_t* launches) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    if (kernel < -1 || kernel >= KVC_KERNEL_COUNT) return fail(h, KVC_ERR_CONFIG, "unknown kernel family %d", kernel);
    double ms = 0;
    int64_t n = 0;
    for (int id = 0; id < KVC_KERNEL_COUNT; ++id) {
        if (kernel != -1 && id != kernel) continue;
        KVC_CUDA(h, collect_timer(h, id));
        ms += h->timers[id].ms;
        n += h->timers[id].launches;
    }
    if (total_ms) *total_ms = ms;
    if (launches) *launches = n;
    return KVC_OK;
}

kvc_status kvc_reset_stats(kvc_handle* h) {
    if (!h) return fail(nullptr, KVC_ERR_NULL, "handle is NULL");
    for (int id = 0; id < KVC_KERNEL_COUNT; ++id) {
        KVC_CUDA(h, collect_timer(h, id));
        h->timers[id].ms = 0;
        h->timers[id].launches = 0;
    }
    return KVC_OK;
}

}  // extern "C"
