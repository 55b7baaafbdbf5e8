// decode_noalloc.cu -- attn_decode_kvcache_noalloc: the paged decode with its split-KV
// partials kept in a scratch array that belongs to the library, for callers that cannot
// allocate device memory themselves.
//
// Who needs it: a caller that owns no allocator can still pass its inputs and outputs but has
// no way to obtain the workspace attn_decode_kvcache asks for -- for example a plugin behind a
// host ABI that hands over tensors only, a serving process that has reserved all free HBM
// for its KV cache before this library is loaded, or a latency-critical loop where a
// cudaMalloc (which may synchronise the device) is not acceptable.
//
// How: the partials live in kScratchBytes of file-scope __device__ memory, which every GPU
// that loads this library holds until the process exits.  The first call on a device looks up
// that device's address of the array with cudaGetSymbolAddress (the device must be current);
// later calls reuse it.  The call then runs exactly the attn_decode_kvcache path with that
// address as its workspace, so no device memory is ever allocated or freed here.
//
// Sharing: all calls on a device use the same array and it keeps the previous call's
// contents.  Nothing in it needs clearing, because the split kernel writes every partial slot
// (empty splits included) before the combine kernel of the same call reads it.  Two calls
// whose kernels overlap on the GPU (different streams, no ordering between them) race on the
// array and may return wrong results.
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "attn.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
attn_status_t scratch_address(void** out, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_decode_kvcache_noalloc(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* cache_seqlens,
                                          const int32_t* block_table, int page_size,
                                          int num_splits, void* out, float* lse, int batch,
                                          int nheads_q, int nheads_kv, int head_dim,
                                          int max_pages_per_seq, int num_pages,
                                          float softmax_scale, void* stream) {
    if (batch < 0 || nheads_q <= 0 || nheads_kv <= 0 || num_splits < 0 || num_splits > 64)
        return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (batch == 0) return ATTN_OK;
    void* scratch = nullptr;
    int num_sms = 0;
    const attn_status_t st = scratch_address(&scratch, &num_sms);
    if (st != ATTN_OK) return st;
    // Resolve the automatic split count the same way attn_decode_kvcache does, so the size
    // check below is exact rather than a worst case.
    const int splits = num_splits != 0 ? num_splits
                                       : attn_decode_num_splits(batch, nheads_q, nheads_kv,
                                                                max_pages_per_seq, page_size,
                                                                num_sms);
    const size_t need = attn_decode_workspace_bytes(batch, nheads_q, head_dim, splits);
    if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the built-in scratch
    return attn_decode_kvcache(q, k_cache, v_cache, cache_seqlens, block_table, page_size,
                               splits, out, lse, batch, nheads_q, nheads_kv, head_dim,
                               max_pages_per_seq, num_pages, softmax_scale, scratch,
                               kScratchBytes, stream);
}

}  // extern "C"
