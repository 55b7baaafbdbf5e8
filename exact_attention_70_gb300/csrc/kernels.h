// kernels.h -- parameter blocks and launchers shared by the host API (attn_api.cu) and the
// kernel translation units.  Nothing here is part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Bits of the per-device status word the kernels raise instead of trapping.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBounds = 2u;

// Opt-in device bounds checks, for debugging (build with -DATTN_CHECK_BOUNDS, which
// exact_attention_70_gb300.build does for build(check_bounds=True)): a global store or a TMA
// coordinate that would leave its tensor raises the bounds bit of the status word and is
// skipped.  In the default build the check is the constant true and generates no code.
#ifdef ATTN_CHECK_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, unsigned* status) {
    if (!ok) atomicOr(status, kStatusBounds);
    return ok;
}
#define ATTN_IN_BOUNDS(cond, status) ::attn::in_bounds((cond), (status))
#else
#define ATTN_IN_BOUNDS(cond, status) true
#endif

// ---- prefill ----------------------------------------------------------------------------

constexpr int kFwdBlockN = 128;     // keys per KV tile
constexpr int kFwdTilesPerItem = 2; // Q tiles (of 128 packed rows) per work item
constexpr int kFwdThreads = 640;    // 4 softmax warpgroups + (TMA warp, 2 MMA warps, 1 idle)
constexpr int kPrepThreads = 1024;
constexpr int kPrepBins = 1024;     // cost histogram bins of the work-list sort

// Workspace layout of attn_fwd: [header 256 B][prefix int32 (batch+1), 16-B aligned][items]
struct FwdWorkspaceHeader {
    int n_items;
    int n_pairs;
    int next_item;  // the forward kernel's claim counter (reset by the work-list kernel)
    int pad[61];
};

struct FwdPrepParams {
    const int* cu_q;
    const int* cu_k;            // contiguous K/V: key offsets [batch + 1]; null when paged
    const int* cache_seqlens;   // paged K/V: cached tokens per sequence before the new ones
    int max_keys;               // paged K/V: max_pages_per_seq * page_size
    int* prefix;     // [batch + 1] work items per sequence, exclusive scan
    int4* items;     // [capacity_pairs * Hkv]
    FwdWorkspaceHeader* header;
    unsigned* status;
    int batch, total_q, total_k, max_seqlen_q, max_seqlen_k;
    int Hkv, tpt, capacity_pairs;
    int causal, wl, wr;
    int heads_per_group;  // KV heads whose items are listed together (1..Hkv)
};

struct FwdParams {
    CUtensorMap tm_q;  // 3-D over q   [total_q, Hq, d],  box {64, g, tpt}
    CUtensorMap tm_k;  // 3-D over k   [total_k, Hkv, d], box {64, 1, 128}
    CUtensorMap tm_v;  // 3-D over v   [total_k, Hkv, d], box {64, 1, 128}
    CUtensorMap tm_o;  // 3-D over out [total_q, Hq, d],  box {64, g, tpt}: stores of whole tiles
    __nv_bfloat16* out;
    float* lse;
    const int* cu_q;
    const int* cu_k;            // contiguous K/V; null when paged
    const int4* items;
    FwdWorkspaceHeader* header;  // n_items, and the claim counter the kernel advances
    unsigned* status;
    int Hq, Hkv, g, tpt, total_q;
    int causal, wl, wr;
    float scale_log2;  // softmax_scale * log2(e)
    // Score modifiers (the kernel instance built for them): softcap c > 0 maps the scaled
    // score s to c tanh(s / c); alibi (per q head, or null) adds -slope |pos - key|.
    float scale, softcap;
    const float* alibi;
    // Paged K/V (block_table != null): tm_k / tm_v are 3-D over [num_pages * page_size, Hkv, d]
    // with boxes {64, 1, box_rows}; sequence b holds cache_seqlens[b] + q_len_b keys.
    const int* block_table;     // [batch, max_pages]
    const int* cache_seqlens;
    int page_size, max_pages, num_pages, box_rows;
};

// ---- paged-cache append (chunked prefill) ---------------------------------------------------

struct AppendParams {
    const __nv_bfloat16* q;      // [total_q, Hq, d]
    const __nv_bfloat16* k_new;  // [total_q, Hkv, d]
    const __nv_bfloat16* v_new;
    __nv_bfloat16* k_cache;      // [num_pages, page_size, Hkv, d]
    __nv_bfloat16* v_cache;
    __nv_bfloat16* q_rot;        // [total_q, Hq, d] rotated queries (rotary only)
    const int* cu_q;
    const int* cache_seqlens;
    const int* block_table;
    const float* rot_cos;        // [rot_rows, rot_dim / 2]
    const float* rot_sin;
    unsigned* status;
    int batch, total_q, Hq, Hkv, d, page_size, max_pages, num_pages;
    int rot_dim, rot_rows, interleaved;
};

cudaError_t launch_kvcache_append(const AppendParams& p, int num_sms, cudaStream_t stream);

cudaError_t launch_fwd_prepare(const FwdPrepParams& p, cudaStream_t stream);
cudaError_t launch_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t stream);
int fwd_smem_bytes(int head_dim);

// ---- backward ------------------------------------------------------------------------------

struct BwdParams {
    CUtensorMap tm_q;   // 3-D over q    [total_q, Hq, d], box {64, g, tpt}
    CUtensorMap tm_do;  // 3-D over dout [total_q, Hq, d], box {64, g, tpt}
    CUtensorMap tm_k;   // 3-D over k    [total_k, Hkv, d], box {64, 1, 128}
    CUtensorMap tm_v;
    const __nv_bfloat16* o;     // [total_q, Hq, d]
    const __nv_bfloat16* dout;
    const float* lse;           // [Hq, total_q]
    float* dsum;                // [Hq, total_q]: D = rowsum(dout * o)
    __nv_bfloat16* dq;          // [total_q, Hq, d]
    __nv_bfloat16* dk;          // [total_k, Hkv, d]
    __nv_bfloat16* dv;
    const int* cu_q;
    const int* cu_k;
    unsigned* status;
    int batch, Hq, Hkv, g, tpt, total_q, total_k, d, max_seqlen_q, max_seqlen_k;
    int causal, wl, wr;
    float scale, scale_log2;
};

cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t stream);

// ---- FP8 (e4m3) prefill ----------------------------------------------------------------

// Scales: q_scale [Hq, nqb] per 128 consecutive packed query tokens; k_scale [Hkv, nkb] per
// 128-key block of a sequence (block kb0[b] + (t - k0) / 128, kb0 the prefix sum of
// ceil(Lk_b / 128)); v_scale [batch, Hkv].  V is stored transposed: v8t [Hkv, d, 128 nkb],
// key t of sequence b in column 128 (kb0[b]) + (t - k0).
struct Fp8Params {
    CUtensorMap tm_q;   // 3-D over q8  [total_q, Hq, d] u8, box {d, g, tpt}
    CUtensorMap tm_k;   // 3-D over k8  [total_k, Hkv, d] u8, box {d, 1, 128}
    CUtensorMap tm_v;   // 3-D over v8t [Hkv, d, 128 nkb] u8, box {128, d, 1}
    CUtensorMap tm_o;   // 3-D over out [total_q, Hq, d] bf16, box {64, g, tpt}: stores of whole tiles
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    __nv_bfloat16* out;
    float* lse;
    const int* cu_q;
    const int* cu_k;
    unsigned* status;
    int batch, Hq, Hkv, g, tpt, total_q, total_k, max_seqlen_q, max_seqlen_k, nqb, nkb;
    int causal, wl, wr;
    float scale_log2;
};

cudaError_t launch_fwd_fp8(const Fp8Params& p, cudaStream_t stream);

// bf16 Q, K, V -> the FP8 forward's inputs (layouts as above); signs: fp32 [128] of +-1 for
// the rotation of Q and K, or null.
struct QuantParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const int* cu_k;
    const float* signs;
    uint8_t* q8;
    uint8_t* k8;
    uint8_t* v8t;
    float* q_scale;
    float* k_scale;
    float* v_scale;
    int batch, total_q, total_k, max_seqlen_k, Hq, Hkv, key_blocks;
};

cudaError_t launch_quantize_fp8(const QuantParams& p, cudaStream_t stream);

// ---- failure-path self-test ------------------------------------------------------------

cudaError_t launch_watchdog_selftest(unsigned* status, cudaStream_t stream);
cudaError_t launch_softcap_selftest(const float* s, float* out, int n, float scale, float softcap,
                                    cudaStream_t stream);

// ---- decode -------------------------------------------------------------------------------

constexpr int kDecChunk = 64;       // keys per pipeline stage
constexpr int kDecThreads = 160;    // 4 MMA warps + 1 TMA warp
constexpr int kDecRowsPerCta = 16;  // query heads of one kv group handled by one CTA

struct DecParams {
    CUtensorMap tm_k;  // 3-D over k_cache [num_pages*page_size, Hkv, d], box {64, 1, box_rows}
    CUtensorMap tm_v;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;    // [batch, Hq, num_splits, d]  (num_splits > 1)
    float* part_lse;  // [batch, Hq, num_splits]
    const int* seqlens;
    const int* block_table;
    unsigned* status;
    int batch, Hq, Hkv, g, hgroups;
    int page_size, box_rows, max_pages, num_pages, num_splits;
    float scale_log2;
};

struct CombineParams {
    const float* part_o;
    const float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int rows;  // batch * Hq
    int num_splits;
};

cudaError_t launch_decode(const DecParams& p, int head_dim, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int head_dim, cudaStream_t stream);
int decode_smem_bytes(int head_dim);

// Configure the kernels' shared-memory limits on the current device (idempotent).
cudaError_t configure_fwd_kernels();
cudaError_t configure_decode_kernels();

}  // namespace attn
