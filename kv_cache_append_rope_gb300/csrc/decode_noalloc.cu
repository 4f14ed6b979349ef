// kvc_decode_attend_noalloc: split-K decode attention that allocates nothing.
//
// Some callers cannot let a library call cudaMalloc: a serving engine that
// owns every byte of device memory through its own arena (so that a request
// can never fail halfway on an out-of-memory error, and so that no
// allocation implicitly synchronises the device while other streams run), or
// a host framework that hands out only the buffers it created.  For them this
// entry point runs the same split-K decode kernel as kvc_append_attend over a
// key/value cache the caller owns, and keeps the kernel's scratch (per-split
// partial outputs, maxima and sums, plus the per-sequence lengths and an error
// word) in one file-scope device array instead of cudaMalloc'd memory.
//
// The array is kNoallocScratchBytes (8 MiB) and lives on every GPU that loads
// the library until the process exits.  Host code cannot use the array's
// name as a device address, so the first call on each device (with that
// device current) resolves it with cudaGetSymbolAddress and caches the
// pointer; make that first call before any stream capture.  All calls share
// the array and it keeps the last call's contents: calls that overlap on the
// GPU (different streams, or different host threads without ordering) race
// on it.  Within one call every partial is written before it is read, and the
// lengths are rewritten by the call itself.  The error word is not: a bounded
// wait that gave up in any call sets a bit there, and the bit stays until
// kvc_noalloc_check reads it back and clears it, so a failed step is reported
// even when later calls ran in between.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;
constexpr int kMaxBatch = 4096;
constexpr size_t kHeaderBytes = 256 + kMaxBatch * sizeof(int32_t);      // error word, lengths
constexpr size_t kPartialBytes = 128 * sizeof(float) + sizeof(float2);   // one (query head, split)
constexpr size_t kMaxPartials = (kNoallocScratchBytes - kHeaderBytes) / kPartialBytes;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
std::atomic<int> g_test_stall{0};   // test only: the next call's producer issues no loads

// The array's device address on the current device (resolved on the first use
// there), or null if the lookup fails.  *fresh is set when this call resolved it.
void* scratch_on(int dev, bool* fresh = nullptr) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (fresh) *fresh = false;
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
        if (fresh) *fresh = true;
    }
    return g_scratch_ptr[dev];
}

struct LengthsParam {
    int32_t len_minus_one[256];
};

// Writes the old lengths (t - 1, the decode kernel's convention) of up to 256
// sequences into the scratch.
__global__ void noalloc_prologue(int32_t* lens_dst, LengthsParam p, int offset, int n) {
    const int i = threadIdx.x;
    if (i < n) lens_dst[offset + i] = p.len_minus_one[i];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool encode(CUtensorMap* map, const void* base, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

void noalloc_arm_test_stall() { g_test_stall.store(1); }

}  // namespace kvc

using namespace kvc;

extern "C" kvc_status kvc_decode_attend_noalloc(const void* keys, const void* values, const float* q_rot,
                                                const int32_t* lengths, float* out, int32_t batch,
                                                int32_t heads_q, int32_t heads_kv, int32_t capacity,
                                                void* stream) {
    if (!keys || !values || !q_rot || !lengths || !out) return KVC_ERR_NULL;
    if (batch <= 0) return KVC_ERR_ZERO_BATCH;
    if (capacity <= 0) return KVC_ERR_ZERO_CAPACITY;
    if (heads_q <= 0 || heads_kv <= 0 || heads_q % heads_kv || heads_q / heads_kv > 32) return KVC_ERR_CONFIG;
    if (batch > kMaxBatch || (size_t)batch * heads_q > kMaxPartials) return KVC_ERR_CONFIG;
    if ((uint64_t)batch * heads_kv * capacity > (uint64_t)INT32_MAX) return KVC_ERR_ELEMENT_OVERFLOW;
    if (((uintptr_t)keys | (uintptr_t)values | (uintptr_t)q_rot | (uintptr_t)out) & 15u) return KVC_ERR_CONFIG;
    int max_t = 0;
    int64_t total = 0;
    for (int b = 0; b < batch; ++b) {
        if (lengths[b] < 1 || lengths[b] > capacity) return KVC_ERR_FULL;
        max_t = lengths[b] > max_t ? lengths[b] : max_t;
        total += lengths[b];
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;

    bool fresh = false;
    void* base = scratch_on(dev, &fresh);
    if (!base) return KVC_ERR_CUDA;
    uint32_t* err = (uint32_t*)base;
    // the error word starts at zero on every device (it is cleared again only by
    // kvc_noalloc_check); everything else in the array is written before it is read
    if (fresh && cudaMemsetAsync(err, 0, sizeof(uint32_t), (cudaStream_t)stream) != cudaSuccess) return KVC_ERR_CUDA;
    int32_t* lens = (int32_t*)((uint8_t*)base + 256);
    uint8_t* parts = (uint8_t*)base + kHeaderBytes;

    // Split plan: as kvc_append_attend, then widened until the partials fit the array.
    const int G = heads_q / heads_kv;
    int sms = 152;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t target = (int64_t)sms * decode_bf16_ctas_per_sm(G) * 4;
    int64_t r = (total * heads_kv + target - 1) / target;
    r = (r + 63) / 64 * 64;
    if (r < 256) r = 256;
    const int64_t rmax = ((int64_t)max_t + 63) / 64 * 64;
    if (r > rmax) r = rmax;
    const size_t lanes_q = (size_t)batch * heads_q;
    while ((size_t)((max_t + r - 1) / r) * lanes_q > kMaxPartials) r += 64;
    const int max_splits = (int)((max_t + r - 1) / r);

    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)batch * heads_kv * capacity;
    if (!encode(&tmK, keys, rows) || !encode(&tmV, values, rows)) return KVC_ERR_CUDA;

    cudaStream_t s = (cudaStream_t)stream;
    for (int off = 0; off < batch; off += 256) {
        LengthsParam p;
        const int n = batch - off < 256 ? batch - off : 256;
        for (int i = 0; i < n; ++i) p.len_minus_one[i] = lengths[off + i] - 1;
        noalloc_prologue<<<1, 256, 0, s>>>(lens, p, off, n);
        if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
    }
    DecodeLaunch dl{};
    dl.tmK = &tmK;
    dl.tmV = &tmV;
    dl.qrot = q_rot;
    dl.len = lens;
    dl.part_ml = (float2*)parts;
    dl.part_o = (float*)(parts + lanes_q * max_splits * sizeof(float2));
    dl.out = out;
    dl.kv.C = capacity;          // contiguous [B][H_kv][C] rows
    dl.kv.Hkv = heads_kv;
    dl.err = err;
    dl.B = batch;
    dl.Hq = heads_q;
    dl.Hkv = heads_kv;
    dl.C = capacity;
    dl.split_rows = (int)r;
    dl.max_splits = max_splits;
    dl.test_stall = g_test_stall.exchange(0);
    if (launch_decode_bf16(dl, s) != cudaSuccess) return KVC_ERR_CUDA;
    if (max_splits > 1 && launch_decode_combine(dl, s) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

extern "C" kvc_status kvc_noalloc_check(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) return KVC_OK;   // no call has run on this device
    }
    uint32_t* err = (uint32_t*)scratch_on(dev);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KVC_ERR_CUDA;
    if (!word) return KVC_OK;
    if (cudaMemsetAsync(err, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return KVC_ERR_CUDA;
    return KVC_ERR_DEVICE;
}
