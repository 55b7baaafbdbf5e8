// attn_api.cu -- the C ABI declared in include/attn.h: argument checks, TMA descriptors,
// the split-count heuristic and the kernel launches.  No call allocates device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <string.h>

#include "attn.h"
#include "kernels.h"
#include "tile_math.h"

namespace attn {
namespace {

__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    unsigned* status = nullptr;  // device address of g_status_word
    int num_sms = 0;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

attn_status_t device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        if (g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return ATTN_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (configure_fwd_kernels() != cudaSuccess) return ATTN_ERR_CUDA;
        if (configure_decode_kernels() != cudaSuccess) return ATTN_ERR_CUDA;
        s.status = static_cast<unsigned*>(addr);
        s.ready = true;
    }
    *out = &s;
    return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// An NVTX range around each computing entry point, so that profiler timelines show the C-ABI
// calls by name (NVTX is header-only and costs next to nothing without a tool attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// 3-D bf16 tensor [n2][n1][n0] (n0 contiguous), 128-byte swizzled boxes {64, b1, b2}.
attn_status_t encode_3d(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1,
                        uint64_t n2, uint32_t b1, uint32_t b2) {
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
    const cuuint32_t box[3] = {64, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D byte tensor [n2][n1][n0] (n0 innermost), box {b0, b1, b2}, 128-byte swizzle.
attn_status_t encode_3d_u8(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1,
                           uint64_t n2, uint32_t b0, uint32_t b1, uint32_t b2) {
    const cuuint64_t dims[3] = {n0, n1, n2};
    const cuuint64_t strides[2] = {n0, n0 * n1};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work items (pairs of 128-row Q tiles) the prefill list can hold.
long long fwd_capacity_pairs(int batch, int max_seqlen_q, int g) {
    const long long per = 2LL * tokens_per_tile(g);
    return static_cast<long long>(batch) * ((max_seqlen_q + per - 1) / per);
}

// a positive, finite, normal fp32 (its reciprocal is finite too)
bool scale_ok(float s) { return isfinite(s) && s >= 1.17549435e-38f; }

constexpr float kLog2eF = 1.44269504088896340736f;

// KV heads per group of the forward work list: as many as keep the group's K and V (all
// sequences) within 32 MiB, about a quarter of the L2, so the CTAs working on one group find
// the blocks other CTAs of the group already fetched.
int fwd_heads_per_group(int total_k, int nheads_kv, int head_dim) {
    const long long per_head = 4ll * total_k * head_dim;  // K and V, bf16
    if (per_head <= 0) return nheads_kv;
    const long long n = (32ll << 20) / per_head;
    return static_cast<int>(n < 1 ? 1 : (n > nheads_kv ? nheads_kv : n));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA call failed";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel wait exceeded its time limit";
        case ATTN_ERR_DEVICE_BOUNDS: return "a device-side index was out of range";
    }
    return "unknown status";
}

size_t attn_fwd_workspace_bytes(int batch, int max_seqlen_q, int nheads_q, int nheads_kv) {
    if (batch < 0 || max_seqlen_q < 0 || nheads_q <= 0 || nheads_kv <= 0 ||
        nheads_q % nheads_kv != 0 || nheads_q / nheads_kv > 128)
        return 0;
    const long long pairs = fwd_capacity_pairs(batch, max_seqlen_q, nheads_q / nheads_kv);
    return sizeof(FwdWorkspaceHeader) + align_up(sizeof(int) * (batch + 1), 16) +
           static_cast<size_t>(pairs) * nheads_kv * sizeof(int4);
}

int attn_kv_block_range(int i_min, int i_max, int seqlen_q, int seqlen_k, int block_n,
                        int causal, int window_left, int window_right, int* lo, int* hi) {
    if (!lo || !hi || block_n <= 0 || seqlen_k < 0 || seqlen_q < 0) return -1;
    const KvRange r = kv_block_range(i_min, i_max, seqlen_q, seqlen_k, block_n, causal,
                                     window_left, window_right);
    *lo = r.lo;
    *hi = r.hi;
    return 0;
}

int attn_kv_block_masked(int j, int i_min, int i_max, int seqlen_q, int seqlen_k, int block_n,
                         int causal, int window_left, int window_right) {
    return kv_block_masked(j, i_min, i_max, seqlen_q, seqlen_k, block_n, causal, window_left,
                           window_right)
               ? 1
               : 0;
}

}  // extern "C"

namespace {

attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                       int causal, int window_left, int window_right, void* workspace,
                       size_t workspace_bytes, void* stream, float softcap,
                       const float* alibi_slopes) {
    if (!(softcap == 0.f || (softcap >= 0x1p-20f && softcap <= 1e30f)) ||
        (alibi_slopes && !aligned(alibi_slopes, 4)))
        return ATTN_ERR_INVALID_ARG;
    if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        nheads_q <= 0 || nheads_kv <= 0 || window_left < -1 || window_right < -1 ||
        !scale_ok(softmax_scale))
        return ATTN_ERR_INVALID_ARG;
    if (nheads_q % nheads_kv != 0) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const int g = nheads_q / nheads_kv;
    if (g > 128) return ATTN_ERR_UNSUPPORTED;
    if (batch == 0 || total_q == 0) return ATTN_OK;  // nothing to compute
    if (total_k == 0) {  // no keys anywhere: k and v may be empty tensors without storage
        k = q;
        v = q;
    }
    if (!q || !k || !v || !out || !lse || !cu_seqlens_q || !cu_seqlens_k)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
        return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(total_q) * nheads_q > (1LL << 31) - 1 ||
        static_cast<long long>(total_k) * nheads_kv > (1LL << 31) - 1)
        return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_fwd_workspace_bytes(batch, max_seqlen_q, nheads_q, nheads_kv);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return ATTN_ERR_WORKSPACE;

    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int tpt = tokens_per_tile(g);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    FwdWorkspaceHeader* header = reinterpret_cast<FwdWorkspaceHeader*>(ws);
    int* prefix = reinterpret_cast<int*>(ws + sizeof(FwdWorkspaceHeader));
    int4* items = reinterpret_cast<int4*>(ws + sizeof(FwdWorkspaceHeader) +
                                          align_up(sizeof(int) * (batch + 1), 16));

    FwdPrepParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.cu_q = cu_seqlens_q;
    pp.cu_k = cu_seqlens_k;
    pp.prefix = prefix;
    pp.items = items;
    pp.header = header;
    pp.status = dev->status;
    pp.batch = batch;
    pp.total_q = total_q;
    pp.total_k = total_k;
    pp.max_seqlen_q = max_seqlen_q;
    pp.max_seqlen_k = max_seqlen_k;
    pp.Hkv = nheads_kv;
    pp.tpt = tpt;
    pp.capacity_pairs = static_cast<int>(fwd_capacity_pairs(batch, max_seqlen_q, g));
    pp.causal = causal ? 1 : 0;
    pp.wl = window_left;
    pp.wr = window_right;
    pp.heads_per_group = fwd_heads_per_group(total_k, nheads_kv, head_dim);

    FwdParams fp;
    memset(&fp, 0, sizeof(fp));
    if (encode_3d(&fp.tm_q, q, head_dim, nheads_q, total_q, g, tpt) != ATTN_OK ||
        encode_3d(&fp.tm_o, out, head_dim, nheads_q, total_q, g, tpt) != ATTN_OK ||
        encode_3d(&fp.tm_k, k, head_dim, nheads_kv, total_k > 0 ? total_k : 1, 1,
                  kFwdBlockN) != ATTN_OK ||
        encode_3d(&fp.tm_v, v, head_dim, nheads_kv, total_k > 0 ? total_k : 1, 1,
                  kFwdBlockN) != ATTN_OK)
        return ATTN_ERR_CUDA;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.cu_q = cu_seqlens_q;
    fp.cu_k = cu_seqlens_k;
    fp.items = items;
    fp.header = header;
    fp.status = dev->status;
    fp.Hq = nheads_q;
    fp.Hkv = nheads_kv;
    fp.g = g;
    fp.tpt = tpt;
    fp.total_q = total_q;
    fp.causal = pp.causal;
    fp.wl = window_left;
    fp.wr = window_right;
    fp.scale_log2 = softmax_scale * kLog2eF;
    fp.scale = softmax_scale;
    fp.softcap = softcap;
    fp.alibi = alibi_slopes;

    if (launch_fwd_prepare(pp, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_fwd(fp, head_dim, dev->num_sms, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                       int causal, int window_left, int window_right, void* workspace,
                       size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_range("attn_fwd");
    return fwd_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                    max_seqlen_q, max_seqlen_k, nheads_q, nheads_kv, head_dim, softmax_scale,
                    causal, window_left, window_right, workspace, workspace_bytes, stream, 0.f,
                    nullptr);
}

attn_status_t attn_fwd_mods(const void* q, const void* k, const void* v, void* out, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                            int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                            int causal, int window_left, int window_right, float softcap,
                            const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                            void* stream) {
    NvtxRange nvtx_range("attn_fwd_mods");
    return fwd_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                    max_seqlen_q, max_seqlen_k, nheads_q, nheads_kv, head_dim, softmax_scale,
                    causal, window_left, window_right, workspace, workspace_bytes, stream,
                    softcap, alibi_slopes);
}

attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8t,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* out, float* lse, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, int batch, int total_q, int total_k,
                           int max_seqlen_q, int max_seqlen_k, int nheads_q, int nheads_kv,
                           int head_dim, int key_blocks, float softmax_scale, int causal,
                           int window_left, int window_right, void* stream) {
    NvtxRange nvtx_range("attn_fwd_fp8");
    if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        nheads_q <= 0 || nheads_kv <= 0 || key_blocks < 0 || window_left < -1 ||
        window_right < -1 || !scale_ok(softmax_scale))
        return ATTN_ERR_INVALID_ARG;
    if (nheads_q % nheads_kv != 0) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const int g = nheads_q / nheads_kv;
    if (g > 128) return ATTN_ERR_UNSUPPORTED;
    if (batch == 0 || total_q == 0) return ATTN_OK;
    // no keys anywhere: k8 may be an empty tensor without storage (its map is never read)
    if (total_k == 0) k8 = v8t;
    if (!q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale || !out || !lse ||
        !cu_seqlens_q || !cu_seqlens_k || key_blocks == 0)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(out, 16) ||
        !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(lse, 4) ||
        !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
        return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(total_q) * nheads_q > (1LL << 31) - 1 ||
        static_cast<long long>(total_k) * nheads_kv > (1LL << 31) - 1 ||
        static_cast<long long>(key_blocks) * 128 * head_dim * nheads_kv > (1LL << 40) ||
        static_cast<long long>(batch) * nheads_kv > 65535)
        return ATTN_ERR_UNSUPPORTED;

    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;

    const int tpt = tokens_per_tile(g);
    Fp8Params fp;
    memset(&fp, 0, sizeof(fp));
    if (encode_3d_u8(&fp.tm_q, q8, head_dim, nheads_q, total_q, 128, g, tpt) != ATTN_OK ||
        encode_3d_u8(&fp.tm_k, k8, head_dim, nheads_kv, total_k > 0 ? total_k : 1, 128, 1, 128) != ATTN_OK ||
        encode_3d_u8(&fp.tm_v, v8t, 128ull * key_blocks, head_dim, nheads_kv, 128, 128, 1) != ATTN_OK ||
        encode_3d(&fp.tm_o, out, head_dim, nheads_q, total_q, g, tpt) != ATTN_OK)
        return ATTN_ERR_CUDA;
    fp.q_scale = q_scale;
    fp.k_scale = k_scale;
    fp.v_scale = v_scale;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.cu_q = cu_seqlens_q;
    fp.cu_k = cu_seqlens_k;
    fp.status = dev->status;
    fp.batch = batch;
    fp.Hq = nheads_q;
    fp.Hkv = nheads_kv;
    fp.g = g;
    fp.tpt = tpt;
    fp.total_q = total_q;
    fp.total_k = total_k;
    fp.max_seqlen_q = max_seqlen_q;
    fp.max_seqlen_k = max_seqlen_k;
    fp.nqb = (total_q + 127) / 128;
    fp.nkb = key_blocks;
    fp.causal = causal ? 1 : 0;
    fp.wl = window_left;
    fp.wr = window_right;
    fp.scale_log2 = softmax_scale * kLog2eF;
    if (launch_fwd_fp8(fp, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_quantize_fp8(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens_k, int batch, int total_q, int total_k,
                                int max_seqlen_k, int nheads_q, int nheads_kv, int head_dim,
                                int key_blocks, const float* signs, void* q8, float* q_scale,
                                void* k8, float* k_scale, void* v8t, float* v_scale,
                                void* stream) {
    NvtxRange nvtx_range("attn_quantize_fp8");
    if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_k < 0 || nheads_q <= 0 ||
        nheads_kv <= 0 || key_blocks < 0)
        return ATTN_ERR_INVALID_ARG;
    if (head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(total_q) * nheads_q > (1LL << 31) - 1 ||
        static_cast<long long>(total_k) * nheads_kv > (1LL << 31) - 1 ||
        static_cast<long long>(key_blocks) > 65535 || nheads_q > 65535 ||
        static_cast<long long>(batch) * nheads_kv > 65535 || (total_q + 127) / 128 > (1 << 30))
        return ATTN_ERR_UNSUPPORTED;
    if (batch == 0 && total_q == 0) return ATTN_OK;
    if (!q || !k || !v || !cu_seqlens_k || !q8 || !q_scale || !k8 || !k_scale || !v8t ||
        !v_scale)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q8, 16) ||
        !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(q_scale, 4) || !aligned(k_scale, 4) ||
        !aligned(v_scale, 4) || !aligned(cu_seqlens_k, 4) || (signs && !aligned(signs, 4)))
        return ATTN_ERR_INVALID_ARG;
    QuantParams qp;
    memset(&qp, 0, sizeof(qp));
    qp.q = static_cast<const __nv_bfloat16*>(q);
    qp.k = static_cast<const __nv_bfloat16*>(k);
    qp.v = static_cast<const __nv_bfloat16*>(v);
    qp.cu_k = cu_seqlens_k;
    qp.signs = signs;
    qp.q8 = static_cast<uint8_t*>(q8);
    qp.k8 = static_cast<uint8_t*>(k8);
    qp.v8t = static_cast<uint8_t*>(v8t);
    qp.q_scale = q_scale;
    qp.k_scale = k_scale;
    qp.v_scale = v_scale;
    qp.batch = batch;
    qp.total_q = total_q;
    qp.total_k = total_k;
    qp.max_seqlen_k = max_seqlen_k;
    qp.Hq = nheads_q;
    qp.Hkv = nheads_kv;
    qp.key_blocks = key_blocks;
    if (launch_quantize_fp8(qp, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t attn_fwd_kvcache_workspace_bytes(int batch, int total_q, int max_seqlen_q, int nheads_q,
                                        int nheads_kv, int head_dim, int rotary_dim) {
    const size_t list = attn_fwd_workspace_bytes(batch, max_seqlen_q, nheads_q, nheads_kv);
    if (list == 0 && batch > 0) return 0;
    if (total_q < 0 || (head_dim != 64 && head_dim != 128)) return 0;
    const size_t qrot =
        rotary_dim > 0 ? static_cast<size_t>(total_q) * nheads_q * head_dim * 2 : 0;
    return align_up(list, 256) + qrot;
}

attn_status_t attn_fwd_kvcache(const void* q, const void* k_new, const void* v_new, void* k_cache,
                               void* v_cache, const int32_t* cache_seqlens,
                               const int32_t* block_table, const int32_t* cu_seqlens_q,
                               const float* rotary_cos, const float* rotary_sin, int rotary_dim,
                               int rotary_rows, int rotary_interleaved, void* out, float* lse,
                               int batch, int total_q, int max_seqlen_q, int nheads_q,
                               int nheads_kv, int head_dim, int page_size,
                               int max_pages_per_seq, int num_pages, float softmax_scale,
                               int causal, int window_left, int window_right, void* workspace,
                               size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_range("attn_fwd_kvcache");
    if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || nheads_q <= 0 || nheads_kv <= 0 ||
        window_left < -1 || window_right < -1 || !scale_ok(softmax_scale) ||
        max_pages_per_seq <= 0 || num_pages <= 0 || page_size <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (nheads_q % nheads_kv != 0) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const int g = nheads_q / nheads_kv;
    if (g > 128) return ATTN_ERR_UNSUPPORTED;
    // pages hold whole 16-row boxes and a 128-key block is whole pages or part of one
    if (page_size % 16 != 0 || (kFwdBlockN % page_size != 0 && page_size % kFwdBlockN != 0))
        return ATTN_ERR_UNSUPPORTED;
    if (rotary_dim < 0 || rotary_dim > head_dim || rotary_dim % 16 != 0) return ATTN_ERR_UNSUPPORTED;
    if (rotary_dim > 0 && (!rotary_cos || !rotary_sin || rotary_rows <= 0 ||
                           !aligned(rotary_cos, 4) || !aligned(rotary_sin, 4)))
        return ATTN_ERR_INVALID_ARG;
    if (batch == 0 || total_q == 0) return ATTN_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !cache_seqlens || !block_table ||
        !cu_seqlens_q || !out || !lse)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(cache_seqlens, 4) || !aligned(block_table, 4) || !aligned(cu_seqlens_q, 4))
        return ATTN_ERR_INVALID_ARG;
    const long long cache_rows = static_cast<long long>(num_pages) * page_size;
    if (static_cast<long long>(total_q) * nheads_q > (1LL << 31) - 1 ||
        cache_rows * nheads_kv > (1LL << 31) - 1 ||
        static_cast<long long>(max_pages_per_seq) * page_size > (1LL << 30))
        return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_fwd_kvcache_workspace_bytes(batch, total_q, max_seqlen_q, nheads_q,
                                                         nheads_kv, head_dim, rotary_dim);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return ATTN_ERR_WORKSPACE;

    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int tpt = tokens_per_tile(g);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    FwdWorkspaceHeader* header = reinterpret_cast<FwdWorkspaceHeader*>(ws);
    int* prefix = reinterpret_cast<int*>(ws + sizeof(FwdWorkspaceHeader));
    int4* items = reinterpret_cast<int4*>(ws + sizeof(FwdWorkspaceHeader) +
                                          align_up(sizeof(int) * (batch + 1), 16));
    __nv_bfloat16* q_rot =
        rotary_dim > 0
            ? reinterpret_cast<__nv_bfloat16*>(
                  ws + align_up(attn_fwd_workspace_bytes(batch, max_seqlen_q, nheads_q, nheads_kv), 256))
            : nullptr;

    // 1. append the new keys (rotated) and values; rotate the queries
    AppendParams ap;
    ap.q = static_cast<const __nv_bfloat16*>(q);
    ap.k_new = static_cast<const __nv_bfloat16*>(k_new);
    ap.v_new = static_cast<const __nv_bfloat16*>(v_new);
    ap.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    ap.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    ap.q_rot = q_rot;
    ap.cu_q = cu_seqlens_q;
    ap.cache_seqlens = cache_seqlens;
    ap.block_table = block_table;
    ap.rot_cos = rotary_cos;
    ap.rot_sin = rotary_sin;
    ap.status = dev->status;
    ap.batch = batch;
    ap.total_q = total_q;
    ap.Hq = nheads_q;
    ap.Hkv = nheads_kv;
    ap.d = head_dim;
    ap.page_size = page_size;
    ap.max_pages = max_pages_per_seq;
    ap.num_pages = num_pages;
    ap.rot_dim = rotary_dim;
    ap.rot_rows = rotary_rows;
    ap.interleaved = rotary_interleaved ? 1 : 0;

    // 2. work list: sequence b has q_len_b query rows and cache_seqlens[b] + q_len_b keys
    FwdPrepParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.cu_q = cu_seqlens_q;
    pp.cu_k = nullptr;
    pp.cache_seqlens = cache_seqlens;
    pp.max_keys = max_pages_per_seq * page_size;
    pp.prefix = prefix;
    pp.items = items;
    pp.header = header;
    pp.status = dev->status;
    pp.batch = batch;
    pp.total_q = total_q;
    pp.max_seqlen_q = max_seqlen_q;
    pp.Hkv = nheads_kv;
    pp.tpt = tpt;
    pp.capacity_pairs = static_cast<int>(fwd_capacity_pairs(batch, max_seqlen_q, g));
    pp.causal = causal ? 1 : 0;
    pp.wl = window_left;
    pp.wr = window_right;
    pp.heads_per_group = nheads_kv;  // one group: the cache's layout is the caller's

    // 3. attention over the cache, K/V gathered through block_table
    const int box_rows = page_size < kFwdBlockN ? page_size : kFwdBlockN;
    FwdParams fp;
    memset(&fp, 0, sizeof(fp));
    if (encode_3d(&fp.tm_q, q_rot ? static_cast<const void*>(q_rot) : q, head_dim, nheads_q,
                  total_q, g, tpt) != ATTN_OK ||
        encode_3d(&fp.tm_o, out, head_dim, nheads_q, total_q, g, tpt) != ATTN_OK ||
        encode_3d(&fp.tm_k, k_cache, head_dim, nheads_kv, cache_rows, 1, box_rows) != ATTN_OK ||
        encode_3d(&fp.tm_v, v_cache, head_dim, nheads_kv, cache_rows, 1, box_rows) != ATTN_OK)
        return ATTN_ERR_CUDA;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.cu_q = cu_seqlens_q;
    fp.cu_k = nullptr;
    fp.items = items;
    fp.header = header;
    fp.status = dev->status;
    fp.Hq = nheads_q;
    fp.Hkv = nheads_kv;
    fp.g = g;
    fp.tpt = tpt;
    fp.total_q = total_q;
    fp.causal = pp.causal;
    fp.wl = window_left;
    fp.wr = window_right;
    fp.scale_log2 = softmax_scale * kLog2eF;
    fp.block_table = block_table;
    fp.cache_seqlens = cache_seqlens;
    fp.page_size = page_size;
    fp.max_pages = max_pages_per_seq;
    fp.num_pages = num_pages;
    fp.box_rows = box_rows;

    if (launch_kvcache_append(ap, dev->num_sms, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_fwd_prepare(pp, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_fwd(fp, head_dim, dev->num_sms, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int total_q, int nheads_q) {
    if (total_q < 0 || nheads_q <= 0) return 0;
    return align_up(static_cast<size_t>(total_q) * nheads_q * sizeof(float), 256);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                       int causal, int window_left, int window_right, void* workspace,
                       size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_range("attn_bwd");
    if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        nheads_q <= 0 || nheads_kv <= 0 || window_left < -1 || window_right < -1 ||
        !scale_ok(softmax_scale))
        return ATTN_ERR_INVALID_ARG;
    if (nheads_q % nheads_kv != 0) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const int g = nheads_q / nheads_kv;
    if (g > 128) return ATTN_ERR_UNSUPPORTED;
    if (batch == 0 || (total_q == 0 && total_k == 0)) return ATTN_OK;
    if (total_q == 0 || total_k == 0) {
        // One side without rows: with no queries every key's gradient is zero, with no keys
        // every query's.  The empty side's tensors may have no storage (NULL).
        void* g0 = total_q == 0 ? dk : dq;
        void* g1 = total_q == 0 ? dv : nullptr;
        const size_t bytes = static_cast<size_t>(total_q == 0 ? total_k : total_q) *
                             static_cast<size_t>(total_q == 0 ? nheads_kv : nheads_q) *
                             static_cast<size_t>(head_dim) * 2;
        if (!g0 || !aligned(g0, 16) || (total_q == 0 && (!g1 || !aligned(g1, 16))))
            return ATTN_ERR_INVALID_ARG;
        const cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(g0, 0, bytes, s) != cudaSuccess ||
            (g1 && cudaMemsetAsync(g1, 0, bytes, s) != cudaSuccess))
            return ATTN_ERR_CUDA;
        return ATTN_OK;
    }
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !cu_seqlens_q ||
        !cu_seqlens_k)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
        return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(total_q) * nheads_q > (1LL << 31) - 1 ||
        static_cast<long long>(total_k) * nheads_kv > (1LL << 31) - 1 ||
        static_cast<long long>(batch) * nheads_kv > 65535)
        return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_bwd_workspace_bytes(total_q, nheads_q);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return ATTN_ERR_WORKSPACE;

    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;

    const int tpt = tokens_per_tile(g);
    BwdParams bp;
    memset(&bp, 0, sizeof(bp));
    if (encode_3d(&bp.tm_q, q, head_dim, nheads_q, total_q > 0 ? total_q : 1, g, tpt) != ATTN_OK ||
        encode_3d(&bp.tm_do, dout, head_dim, nheads_q, total_q > 0 ? total_q : 1, g, tpt) != ATTN_OK ||
        encode_3d(&bp.tm_k, k, head_dim, nheads_kv, total_k > 0 ? total_k : 1, 1, 128) != ATTN_OK ||
        encode_3d(&bp.tm_v, v, head_dim, nheads_kv, total_k > 0 ? total_k : 1, 1, 128) != ATTN_OK)
        return ATTN_ERR_CUDA;
    bp.o = static_cast<const __nv_bfloat16*>(out);
    bp.dout = static_cast<const __nv_bfloat16*>(dout);
    bp.lse = lse;
    bp.dsum = static_cast<float*>(workspace);
    bp.dq = static_cast<__nv_bfloat16*>(dq);
    bp.dk = static_cast<__nv_bfloat16*>(dk);
    bp.dv = static_cast<__nv_bfloat16*>(dv);
    bp.cu_q = cu_seqlens_q;
    bp.cu_k = cu_seqlens_k;
    bp.status = dev->status;
    bp.batch = batch;
    bp.Hq = nheads_q;
    bp.Hkv = nheads_kv;
    bp.g = g;
    bp.tpt = tpt;
    bp.total_q = total_q;
    bp.total_k = total_k;
    bp.d = head_dim;
    bp.max_seqlen_q = max_seqlen_q;
    bp.max_seqlen_k = max_seqlen_k;
    bp.causal = causal ? 1 : 0;
    bp.wl = window_left;
    bp.wr = window_right;
    bp.scale = softmax_scale;
    bp.scale_log2 = softmax_scale * kLog2eF;
    if (launch_bwd(bp, dev->num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

int attn_decode_num_splits(int batch, int nheads_q, int nheads_kv, int max_pages_per_seq,
                           int page_size, int num_sms) {
    if (batch <= 0 || nheads_q <= 0 || nheads_kv <= 0 || nheads_q % nheads_kv != 0 ||
        max_pages_per_seq <= 0 || page_size <= 0)
        return 1;
    if (num_sms <= 0) num_sms = 1;
    const int g = nheads_q / nheads_kv;
    const long long groups =
        static_cast<long long>(batch) * nheads_kv * ((g + kDecRowsPerCta - 1) / kDecRowsPerCta);
    // About one split per 2048 keys of the longest sequence (so long and short sequences
    // produce CTAs of similar length), and at least about four waves of CTAs.
    const long long max_keys = static_cast<long long>(max_pages_per_seq) * page_size;
    long long by_len = (max_keys + 2047) / 2048;
    long long by_sms = (4LL * 2 * num_sms + groups - 1) / groups;
    long long s = by_len > by_sms ? by_len : by_sms;
    if (s < 1) s = 1;
    if (s > 16) s = 16;
    return static_cast<int>(s);
}

size_t attn_decode_workspace_bytes(int batch, int nheads_q, int head_dim, int num_splits) {
    if (batch < 0 || nheads_q <= 0 || (head_dim != 64 && head_dim != 128) || num_splits < 0 ||
        num_splits > 64)
        return 0;
    const int S = num_splits == 0 ? 16 : num_splits;
    if (S == 1 && num_splits == 1) return 0;
    const size_t rows = static_cast<size_t>(batch) * nheads_q * S;
    return align_up(rows * head_dim * sizeof(float), 256) + align_up(rows * sizeof(float), 256);
}

attn_status_t attn_decode_kvcache(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* cache_seqlens, const int32_t* block_table,
                                  int page_size, int num_splits, void* out, float* lse,
                                  int batch, int nheads_q, int nheads_kv, int head_dim,
                                  int max_pages_per_seq, int num_pages, float softmax_scale,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_range("attn_decode_kvcache");
    if (batch < 0 || nheads_q <= 0 || nheads_kv <= 0 || nheads_q % nheads_kv != 0 ||
        max_pages_per_seq < 0 || num_pages < 0 || num_splits < 0 || num_splits > 64 ||
        page_size <= 0 || !scale_ok(softmax_scale))
        return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (page_size % 16 != 0 || !(page_size % 64 == 0 || 64 % page_size == 0))
        return ATTN_ERR_UNSUPPORTED;
    if (batch > 65535) return ATTN_ERR_UNSUPPORTED;
    if (batch == 0) return ATTN_OK;
    if (!q || !k_cache || !v_cache || !cache_seqlens || !block_table || !out || !lse)
        return ATTN_ERR_INVALID_ARG;
    if (max_pages_per_seq == 0 || num_pages == 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(lse, 4) || !aligned(cache_seqlens, 4) ||
        !aligned(block_table, 4))
        return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(num_pages + 1) * page_size > (1LL << 31) - 1 ||
        static_cast<long long>(max_pages_per_seq) * page_size > (1LL << 31) - 1)
        return ATTN_ERR_UNSUPPORTED;

    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int S = num_splits == 0 ? attn_decode_num_splits(batch, nheads_q, nheads_kv,
                                                           max_pages_per_seq, page_size,
                                                           dev->num_sms)
                                  : num_splits;
    const int g = nheads_q / nheads_kv;
    DecParams dp;
    memset(&dp, 0, sizeof(dp));
    const int box_rows = page_size < kDecChunk ? page_size : kDecChunk;
    const uint64_t cache_rows = static_cast<uint64_t>(num_pages) * page_size;
    if (encode_3d(&dp.tm_k, k_cache, head_dim, nheads_kv, cache_rows, 1, box_rows) != ATTN_OK ||
        encode_3d(&dp.tm_v, v_cache, head_dim, nheads_kv, cache_rows, 1, box_rows) != ATTN_OK)
        return ATTN_ERR_CUDA;
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.out = static_cast<__nv_bfloat16*>(out);
    dp.lse = lse;
    dp.seqlens = cache_seqlens;
    dp.block_table = block_table;
    dp.status = dev->status;
    dp.batch = batch;
    dp.Hq = nheads_q;
    dp.Hkv = nheads_kv;
    dp.g = g;
    dp.hgroups = (g + kDecRowsPerCta - 1) / kDecRowsPerCta;
    dp.page_size = page_size;
    dp.box_rows = box_rows;
    dp.max_pages = max_pages_per_seq;
    dp.num_pages = num_pages;
    dp.num_splits = S;
    dp.scale_log2 = softmax_scale * kLog2eF;
    if (S > 1) {
        const size_t rows = static_cast<size_t>(batch) * nheads_q * S;
        const size_t need = align_up(rows * head_dim * sizeof(float), 256) +
                            align_up(rows * sizeof(float), 256);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
            return ATTN_ERR_WORKSPACE;
        dp.part_o = static_cast<float*>(workspace);
        dp.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                               align_up(rows * head_dim * sizeof(float), 256));
    }
    if (launch_decode(dp, head_dim, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (S > 1) {
        CombineParams cp;
        cp.part_o = dp.part_o;
        cp.part_lse = dp.part_lse;
        cp.out = dp.out;
        cp.lse = lse;
        cp.rows = batch * nheads_q;
        cp.num_splits = S;
        if (launch_combine(cp, head_dim, s) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(void* stream) {
    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    if (launch_watchdog_selftest(dev->status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_selftest_softcap(const float* scores, float* out, int n, float softmax_scale,
                                    float softcap, void* stream) {
    if (n < 0 || (n & 1) || !scale_ok(softmax_scale) || !(softcap >= 0x1p-20f && softcap <= 1e30f))
        return ATTN_ERR_INVALID_ARG;
    if (n == 0) return ATTN_OK;
    if (!scores || !out || !aligned(scores, 8) || !aligned(out, 8)) return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    if (launch_softcap_selftest(scores, out, n, softmax_scale, softcap,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_get_device_status(void* stream) {
    DeviceState* dev = nullptr;
    attn_status_t st = device_state(&dev);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word & kStatusTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
    if (word & kStatusBounds) return ATTN_ERR_DEVICE_BOUNDS;
    return ATTN_OK;
}

}  // extern "C"
