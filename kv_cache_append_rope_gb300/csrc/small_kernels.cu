// Length bookkeeping and input checks.
//
// commit:   [Ch37] "Bind the state, calculate completely, then commit" -- the
//           logical length grows only after the attention of the call has been
//           enqueued; every length and next position of one layer is updated
//           by one thread, so no kernel of the same call reads a half-updated
//           length.
// truncate: [LCP5] listing under "哪些东西必须一起裁剪" -- length and next
//           position of every layer become cut; stored rows are not touched.
// nonfinite: [Ch37] listing "Own a fixed layer-bound cache, append one checked
//           row, and reset logical length" rejects non-finite keys and values
//           before they are stored; this finds the first such flat index.
#include <algorithm>

#include "device_common.cuh"
#include "kvc_internal.h"

namespace kvc {

__global__ void commit_kernel(int32_t* len, int32_t* next, const int32_t* pos0, const int32_t* seqlen,
                              int uniform_rows, int B, int C, uint32_t* err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int n = seqlen ? seqlen[b] : uniform_rows;
    const int p = pos0[b];
    if (!debug_check(len[b] >= 0 && n >= 0 && len[b] + n <= C, err)) return;
    len[b] += n;
    next[b] = p + n;
}

cudaError_t launch_commit(int32_t* len, int32_t* next, const int32_t* pos0, const int32_t* seqlen,
                          int uniform_rows, int B, int C, uint32_t* err, cudaStream_t s) {
    commit_kernel<<<(B + 127) / 128, 128, 0, s>>>(len, next, pos0, seqlen, uniform_rows, B, C, err);
    return cudaGetLastError();
}

// kvc_commit: every listed layer advances by one row, in one launch.
__global__ void commit_layers_kernel(int32_t* len, int32_t* next, const CommitLayers layers, int B, int C,
                                     uint32_t* err) {
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < layers.n * B; u += gridDim.x * blockDim.x) {
        const int64_t i = (int64_t)layers.layer[u / B] * B + u % B;
        if (!debug_check(len[i] >= 0 && len[i] < C, err)) continue;
        len[i] += 1;
        next[i] += 1;
    }
}

cudaError_t launch_commit_layers(int32_t* len, int32_t* next, const CommitLayers& layers, int B, int C,
                                 uint32_t* err, cudaStream_t s) {
    const int n = layers.n * B;
    if (n <= 0) return cudaSuccess;
    commit_layers_kernel<<<(n + 255) / 256 < 64 ? (n + 255) / 256 : 64, 256, 0, s>>>(len, next, layers, B, C, err);
    return cudaGetLastError();
}

__global__ void truncate_kernel(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B) {
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= layers * B) return;
    const int c = cut[u % B];
    len[u] = c;
    next[u] = c;
}

cudaError_t launch_truncate(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B,
                            cudaStream_t s) {
    const int n = layers * B;
    truncate_kernel<<<(n + 127) / 128, 128, 0, s>>>(len, next, cut, layers, B);
    return cudaGetLastError();
}

// The same, with the host-side check moved to the device (lengths kept on the
// device): one block first checks every layer's length against the cut and
// changes nothing -- setting an error bit instead -- if some cut exceeds one.
__global__ void truncate_checked_kernel(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B,
                                        uint32_t* err) {
    const int n = layers * B;
    int bad = 0;
    for (int u = threadIdx.x; u < n; u += blockDim.x) bad |= cut[u % B] > len[u];
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) atomicOr(err, (uint32_t)DEV_ERR_CUT);
        return;
    }
    for (int u = threadIdx.x; u < n; u += blockDim.x) {
        const int c = cut[u % B];
        len[u] = c;
        next[u] = c;
    }
}

cudaError_t launch_truncate_checked(int32_t* len, int32_t* next, const int32_t* cut, int layers, int B,
                                    uint32_t* err, cudaStream_t s) {
    truncate_checked_kernel<<<1, 1024, 0, s>>>(len, next, cut, layers, B, err);
    return cudaGetLastError();
}

// Copy-on-write of paged blocks: one CTA per (pair, layer, key/value), 16-byte chunks.
__global__ void copy_blocks_kernel(char* K, char* V, size_t layer_bytes, size_t block_bytes, const int2* pairs,
                                   int layers) {
    const int pair = blockIdx.x / (2 * layers);
    const int rem = blockIdx.x % (2 * layers);
    char* pool = (rem & 1 ? V : K) + (size_t)(rem >> 1) * layer_bytes;
    const int2 p = pairs[pair];
    const uint4* src = (const uint4*)(pool + (size_t)p.x * block_bytes);
    uint4* dst = (uint4*)(pool + (size_t)p.y * block_bytes);
    for (size_t i = threadIdx.x; i < block_bytes / 16; i += blockDim.x) dst[i] = src[i];
}

cudaError_t launch_copy_blocks(char* K, char* V, size_t layer_bytes, int layers, size_t block_bytes,
                               const int2* pairs, int npairs, cudaStream_t s) {
    if (npairs <= 0) return cudaSuccess;
    copy_blocks_kernel<<<(unsigned)npairs * 2 * layers, 256, 0, s>>>(K, V, layer_bytes, block_bytes, pairs, layers);
    return cudaGetLastError();
}

// Small argument arrays read by the SMs straight from mapped page-locked host memory:
// unlike a copy-engine transfer, this does not queue behind bulk host-to-device copies
// that other streams have in flight.
__global__ void copy_args_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t bytes) {
    const size_t words = bytes / 16;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride)
        reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    for (size_t i = words * 16 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < bytes; i += stride)
        dst[i] = src[i];
}

cudaError_t launch_copy_args(const void* src_mapped, void* dst, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return cudaSuccess;
    if (((uintptr_t)src_mapped | (uintptr_t)dst) & 15u) return cudaErrorMisalignedAddress;
    const size_t words = (bytes + 15) / 16;
    const unsigned blocks = (unsigned)std::min<size_t>(64, (words + 255) / 256);
    copy_args_kernel<<<blocks, 256, 0, s>>>((const uint8_t*)src_mapped, (uint8_t*)dst, bytes);
    return cudaGetLastError();
}

// Length and next position of sequence b in every layer (shared-prefix setup).
__global__ void set_lengths_kernel(int32_t* len, int32_t* next, int layers, int B, int b, int value) {
    const int l = blockIdx.x * blockDim.x + threadIdx.x;
    if (l >= layers) return;
    len[(int64_t)l * B + b] = value;
    next[(int64_t)l * B + b] = value;
}

cudaError_t launch_set_lengths(int32_t* len, int32_t* next, int layers, int B, int b, int value, cudaStream_t s) {
    set_lengths_kernel<<<(layers + 127) / 128, 128, 0, s>>>(len, next, layers, B, b, value);
    return cudaGetLastError();
}

// Logical rows of one layer (kvc_read_rows): destination row (b, h, r) of a
// [B, H_kv, R, d] array receives stored row (b, h, r) when r < len[b] (gathered
// through the block table for paged storage) and zeros otherwise; positions[b][r]
// the recorded position, or -1.  W is the copy unit (16 bytes when a row is a
// multiple of 16 bytes, else 4).
template <typename W>
__global__ void read_rows_kernel(const char* __restrict__ K, const char* __restrict__ V,
                                 const int32_t* __restrict__ pos, const int32_t* __restrict__ len, KvLayout kv,
                                 char* __restrict__ Ko, char* __restrict__ Vo, int32_t* __restrict__ Po, int B,
                                 int Hkv, int R, int row_bytes) {
    const int units = row_bytes / (int)sizeof(W);
    const int64_t total = (int64_t)B * Hkv * R * units;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(u % units);
        int64_t r = u / units;
        const int slot = (int)(r % R);
        r /= R;
        const int h = (int)(r % Hkv);
        const int b = (int)(r / Hkv);
        const int n = min(len[b], kv.C);
        const int64_t dst = (((int64_t)b * Hkv + h) * R + slot) * row_bytes + (int64_t)c * sizeof(W);
        W kw{}, vw{};
        if (slot < n) {
            const int64_t src = kv_row(kv, b, h, slot) * row_bytes + (int64_t)c * sizeof(W);
            kw = *reinterpret_cast<const W*>(K + src);
            vw = *reinterpret_cast<const W*>(V + src);
        }
        if (Ko) *reinterpret_cast<W*>(Ko + dst) = kw;
        if (Vo) *reinterpret_cast<W*>(Vo + dst) = vw;
        if (Po && h == 0 && c == 0) Po[(int64_t)b * R + slot] = slot < n ? pos[(int64_t)b * kv.C + slot] : -1;
    }
}

cudaError_t launch_read_rows(const void* K, const void* V, const int32_t* pos, const int32_t* len, const KvLayout& kv,
                             void* Ko, void* Vo, int32_t* Po, int B, int Hkv, int R, int row_bytes, cudaStream_t s) {
    const bool wide = row_bytes % 16 == 0;
    const int64_t total = (int64_t)B * Hkv * R * (row_bytes / (wide ? 16 : 4));
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256, 152 * 16);
    if (wide)
        read_rows_kernel<uint4><<<blocks, 256, 0, s>>>((const char*)K, (const char*)V, pos, len, kv, (char*)Ko,
                                                       (char*)Vo, Po, B, Hkv, R, row_bytes);
    else
        read_rows_kernel<uint32_t><<<blocks, 256, 0, s>>>((const char*)K, (const char*)V, pos, len, kv, (char*)Ko,
                                                          (char*)Vo, Po, B, Hkv, R, row_bytes);
    return cudaGetLastError();
}

// Test-only poison (KVC_OPT_TEST_POISON): in every layer, row (g, h, r) of the
// storage viewed as [groups][H_kv][R] rows -- contiguous: groups = sequences,
// R = C; paged: groups = pool blocks, R = P -- is filled when r >= live[l][g]
// (the rows no sequence holds): keys with zeros, values with `vbits` (one
// element's bit pattern, `esz` bytes).
__global__ void poison_kernel(char* K, char* V, size_t layer_bytes, const int32_t* live, int layers, int groups,
                              int Hkv, int R, int d, int esz, unsigned long long vbits) {
    const int64_t total = (int64_t)layers * groups * Hkv * R * d;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = u / d;
        const int slot = (int)(r % R);
        r /= R;
        const int64_t gh = r;                          // (l * groups + g) * Hkv + h
        const int64_t lg = gh / Hkv;                   // l * groups + g
        if (slot < live[lg]) continue;
        const int l = (int)(lg / groups);
        const int64_t row_in_layer = (gh - (int64_t)l * groups * Hkv) * R + slot;
        const int64_t off = (int64_t)l * layer_bytes + (row_in_layer * d + u % d) * esz;
        for (int e = 0; e < esz; ++e) {
            K[off + e] = 0;
            V[off + e] = (char)((vbits >> (8 * e)) & 0xff);
        }
    }
}

cudaError_t launch_poison(void* K, void* V, size_t layer_bytes, const int32_t* live, int layers, int groups, int Hkv,
                          int R, int d, int esz, unsigned long long vbits, cudaStream_t s) {
    const int64_t total = (int64_t)layers * groups * Hkv * R * d;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256, 152 * 32);
    poison_kernel<<<blocks, 256, 0, s>>>((char*)K, (char*)V, layer_bytes, live, layers, groups, Hkv, R, d, esz, vbits);
    return cudaGetLastError();
}

template <typename T>
__global__ void nonfinite_kernel(const T* x, int64_t n, unsigned long long* first) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const double v = Storage<T>::to_f64(x[i]);
        if (!isfinite(v)) atomicMin(first, (unsigned long long)i);
    }
}

cudaError_t launch_nonfinite(int dtype, const void* x, int64_t n, unsigned long long* first,
                             cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    switch (dtype) {
        case KVC_BF16: nonfinite_kernel<<<(unsigned)blocks, 256, 0, s>>>((const __nv_bfloat16*)x, n, first); break;
        case KVC_F32: nonfinite_kernel<<<(unsigned)blocks, 256, 0, s>>>((const float*)x, n, first); break;
        case KVC_F64: nonfinite_kernel<<<(unsigned)blocks, 256, 0, s>>>((const double*)x, n, first); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvc
