/*
 * attn.h -- C ABI of libattn.so: exact tiled scaled-dot-product attention on GB300 (sm_103a).
 *
 * What is computed ("Attention kernels: FlashAttention and PagedAttention", section 二.1 and
 * section 三.2; "04 · FA4 (CuTeDSL) and engineering interfaces", sections 3-7):
 *   for every query row i of sequence b and query head h,
 *     S_ij  = softmax_scale * <q_i,h , k_j,kvh>        kvh = h / (nheads_q / nheads_kv)
 *     O_i,h = sum_j softmax_j(S_i.) v_j,kvh          over the keys j visible to row i
 *     LSE   = log sum_j exp(S_ij)                    (natural log)
 *   The kernels tile the key axis, keep a running row max and denominator, rescale the output
 *   accumulator when the max moves, and write only O and LSE: S and P never reach memory.
 *
 * Visibility (bottom-right aligned, "04 · FA4 ...", section 6.2 and the section 7 table):
 *   query row i of a sequence with Lq queries and Lk keys sits at key position p = i + Lk - Lq;
 *   key j < Lk is visible iff  j <= p + w_right  (causal forces w_right = 0; w_right == -1 with
 *   causal == 0 means no right bound)  and  j >= p - w_left  (w_left == -1: no left bound).
 *   A row that sees no key gets O = 0 and LSE = -inf.
 *
 * Conventions shared by every call:
 *   - All pointers marked "device" are device addresses on the current CUDA device; the caller
 *     owns every buffer.  The library never allocates, frees or retains memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *     Nothing synchronises the host except attn_get_device_status().
 *   - Tensors are dense row-major with the last dimension contiguous.  q, k, v, out, k_cache
 *     and v_cache must be 16-byte aligned; lse 4-byte aligned; workspace 256-byte aligned.
 *   - The library is stateless apart from a per-device status word and a per-device cache of
 *     kernel attributes; calls from several host threads on different streams are safe.
 *   - Errors: argument checks run before any launch and return ATTN_ERR_INVALID_ARG,
 *     ATTN_ERR_UNSUPPORTED or ATTN_ERR_WORKSPACE without touching the device.  A failed
 *     launch returns ATTN_ERR_CUDA.  Faults detected on the device (a wait that exceeded its
 *     time limit, an index outside its buffer in cu_seqlens, cache_seqlens or block_table)
 *     never trap: the kernel records a flag, skips the offending work and exits, and
 *     attn_get_device_status() reports it.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,    /* null pointer, bad size, misaligned buffer */
    ATTN_ERR_UNSUPPORTED = -2,    /* valid but not built: head_dim, group size, page size */
    ATTN_ERR_WORKSPACE = -3,      /* workspace missing or smaller than required */
    ATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
    ATTN_ERR_DEVICE_TIMEOUT = -5, /* a kernel wait exceeded its limit and the kernel gave up */
    ATTN_ERR_DEVICE_BOUNDS = -6   /* a device-side index (seqlens, page ids) was out of range */
} attn_status_t;

/*
 * attn_fwd -- varlen prefill ("flash_attn_varlen_func" in "04 · FA4 ...", sections 3-5;
 * tiling per "Attention kernels ...", sections 三.2 and 七).
 *
 *   q             device bf16 [total_q, nheads_q, head_dim]; sequence b owns rows
 *                 [cu_seqlens_q[b], cu_seqlens_q[b+1])
 *   k, v          device bf16 [total_k, nheads_kv, head_dim]; sequence b owns rows
 *                 [cu_seqlens_k[b], cu_seqlens_k[b+1])
 *   out           device bf16 [total_q, nheads_q, head_dim] (written for rows inside a sequence)
 *   lse           device fp32 [nheads_q, total_q], natural log
 *   cu_seqlens_q, cu_seqlens_k   device int32 [batch + 1], non-decreasing, last entry
 *                 <= total_q (resp. total_k); checked on the device (ATTN_ERR_DEVICE_BOUNDS)
 *   batch, total_q, total_k      host sizes (the C ABI needs them to describe the tensors)
 *   max_seqlen_q, max_seqlen_k   upper bounds on the per-sequence lengths (sizing only)
 *   nheads_q, nheads_kv          nheads_q % nheads_kv == 0, group nheads_q/nheads_kv <= 128
 *   head_dim      64 or 128
 *   softmax_scale finite and >= FLT_MIN (callers wanting the default pass head_dim^-0.5)
 *   causal, window_left, window_right   see "Visibility"; window values >= -1
 *   workspace     device scratch of at least attn_fwd_workspace_bytes(...) bytes, holding the
 *                 tile work list; contents need not be initialised; not retained after the
 *                 stream reaches the end of the call
 *   stream        cudaStream_t
 * Two calls that share a workspace must not overlap on the device.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                       int causal, int window_left, int window_right, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_fwd needs for these sizes (0 on invalid sizes). */
size_t attn_fwd_workspace_bytes(int batch, int max_seqlen_q, int nheads_q, int nheads_kv);

/*
 * attn_decode_kvcache -- seqlen_q = 1 decode over a paged KV cache with split-KV and an
 * LSE-weighted combine ("flash_attn_with_kvcache" in "04 · FA4 ...", sections 6.1-6.2;
 * "Attention kernels ...", sections 五.2, 五.3, 六.1 and 六.3).
 *
 *   q             device bf16 [batch, nheads_q, head_dim] (one new token per sequence)
 *   k_cache, v_cache   device bf16 [num_pages, page_size, nheads_kv, head_dim]
 *   cache_seqlens device int32 [batch]; sequence b attends to its keys 0 .. cache_seqlens[b]-1
 *                 (all of them: bottom-right causal with one query); must be in
 *                 [0, max_pages_per_seq * page_size] (checked on the device)
 *   block_table   device int32 [batch, max_pages_per_seq]; key j of sequence b is at
 *                 page block_table[b][j / page_size], slot j % page_size; entries past
 *                 ceil(cache_seqlens[b] / page_size) are never read; ids must be in
 *                 [0, num_pages) (checked on the device)
 *   page_size     a multiple of 16 that divides 64 or is a multiple of 64
 *   num_splits    0 = choose automatically (1..16), else 1..64; split s of sequence b covers a
 *                 contiguous range of whole 64-key chunks; an empty split has weight 0
 *   out           device bf16 [batch, nheads_q, head_dim]
 *   lse           device fp32 [batch, nheads_q], natural log
 *   batch, nheads_q, nheads_kv, head_dim, max_pages_per_seq, num_pages   host sizes;
 *                 head_dim 64 or 128; nheads_q % nheads_kv == 0
 *   softmax_scale finite and >= FLT_MIN
 *   workspace     device scratch of attn_decode_workspace_bytes(batch, nheads_q, head_dim,
 *                 num_splits) bytes for the split partials (may be NULL when that is 0)
 *   stream        cudaStream_t
 */
attn_status_t attn_decode_kvcache(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* cache_seqlens, const int32_t* block_table,
                                  int page_size, int num_splits, void* out, float* lse,
                                  int batch, int nheads_q, int nheads_kv, int head_dim,
                                  int max_pages_per_seq, int num_pages, float softmax_scale,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_kvcache_noalloc -- attn_decode_kvcache for callers that cannot allocate device
 * memory.  The pages describe no counterpart of this call; it exists because some callers own
 * no allocator: a plugin behind a host interface that passes tensors but no allocation hook,
 * a server that has reserved all free HBM for its KV cache, or a latency-bound loop where
 * cudaMalloc's possible device synchronisation is unacceptable.
 *
 * Arguments, layouts and results are those of attn_decode_kvcache without the workspace
 * pair; the caller still passes every input and output.  The split partials go to a 32 MiB
 * array of __device__ memory owned by the library (every GPU that loads the library holds it
 * until the process exits).  A request whose partials would exceed 32 MiB, i.e.
 * attn_decode_workspace_bytes(batch, nheads_q, head_dim, splits) > 33554432 with `splits` the
 * resolved split count, returns ATTN_ERR_WORKSPACE and launches nothing.
 *
 * The first call on a device looks up the array's address on that device (that device must be
 * current); make that first call before any stream capture.  The address is kept for the life
 * of the process and belongs to the device's primary context, the one the CUDA runtime uses:
 * do not call this entry point after cudaDeviceReset or with another context of that device
 * current.  No call allocates or frees device memory.  All calls on a device share the array and it keeps the last call's contents
 * (nothing needs clearing: each call rewrites every slot it reads); calls whose kernels
 * overlap on the GPU race on it, so order them on one stream or by events.
 */
attn_status_t attn_decode_kvcache_noalloc(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* cache_seqlens,
                                          const int32_t* block_table, int page_size,
                                          int num_splits, void* out, float* lse, int batch,
                                          int nheads_q, int nheads_kv, int head_dim,
                                          int max_pages_per_seq, int num_pages,
                                          float softmax_scale, void* stream);

/*
 * Chunked prefill against a paged KV cache, with the new keys and values appended in place
 * ("Attention kernels: FlashAttention and PagedAttention", section 五.1 and its chunked-prefill
 * figure; "04 · FA4 (CuTeDSL) and engineering interfaces", sections 6.1-6.2).
 *
 * Sequence b has q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens after
 * cache_seqlens[b] cached ones.  The call
 *   1. writes each new token's key (rotated, when rotary_dim > 0) and value into k_cache /
 *      v_cache at position cache_seqlens[b] + i through block_table;
 *   2. rotates the queries the same way (into the workspace; q itself is not modified);
 *   3. computes, for every query row, exact attention over the cache's keys
 *      0 .. cache_seqlens[b] + q_len_b - 1 with the bottom-right causal / window rule
 *      (query i sits at key position cache_seqlens[b] + i).
 * cache_seqlens is not advanced: the caller adds q_len_b after the call.
 *
 *   q            bf16 [total_q, nheads_q, head_dim]
 *   k_new, v_new bf16 [total_q, nheads_kv, head_dim]
 *   k_cache, v_cache  bf16 [num_pages, page_size, nheads_kv, head_dim], updated in place
 *   cache_seqlens int32 [batch], block_table int32 [batch, max_pages_per_seq] (device);
 *                entries past ceil((cache_seqlens[b] + q_len_b) / page_size) are not read
 *   cu_seqlens_q int32 [batch + 1] (device)
 *   rotary_cos, rotary_sin  fp32 [rotary_rows, rotary_dim / 2] (device), row = position;
 *                NULL with rotary_dim = 0 for no rotary embedding.  Planes pair
 *                (x_i, x_{i + rotary_dim/2}) or, with rotary_interleaved, (x_2i, x_2i+1):
 *                (a, b) -> (a cos - b sin, a sin + b cos), computed in fp32, stored as bf16.
 *   out bf16 [total_q, nheads_q, head_dim]; lse fp32 [nheads_q, total_q] (natural log)
 *   head_dim 64 or 128; page_size a multiple of 16 that divides 128 or is a multiple of 128;
 *   rotary_dim a multiple of 16 (0 = none); softmax_scale finite and >= FLT_MIN; windows -1 = unbounded.
 *   workspace: attn_fwd_kvcache_workspace_bytes(...) bytes, 256-byte aligned.
 * Ownership: caller's buffers; nothing is allocated.  Errors: argument checks before any
 * launch; an out-of-range page id, position or rotary row raises ATTN_ERR_DEVICE_BOUNDS
 * (read with attn_get_device_status) and that row is skipped.
 */
attn_status_t attn_fwd_kvcache(const void* q, const void* k_new, const void* v_new, void* k_cache,
                               void* v_cache, const int32_t* cache_seqlens,
                               const int32_t* block_table, const int32_t* cu_seqlens_q,
                               const float* rotary_cos, const float* rotary_sin, int rotary_dim,
                               int rotary_rows, int rotary_interleaved, void* out, float* lse,
                               int batch, int total_q, int max_seqlen_q, int nheads_q,
                               int nheads_kv, int head_dim, int page_size,
                               int max_pages_per_seq, int num_pages, float softmax_scale,
                               int causal, int window_left, int window_right, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Workspace bytes for attn_fwd_kvcache (the work list plus, with rotary, the rotated q). */
size_t attn_fwd_kvcache_workspace_bytes(int batch, int total_q, int max_seqlen_q, int nheads_q,
                                        int nheads_kv, int head_dim, int rotary_dim);

/*
 * Backward pass of attn_fwd: gradients of sum(out * dout) with respect to q, k and v
 * ("Attention kernels: FlashAttention and PagedAttention", section 四.3: S = Q K^T and
 * P = exp(S - LSE) are recomputed blockwise from the saved LSE; D = rowsum(dout * out);
 * dV = P^T dout, dS = P * (dout V^T - D), dQ = scale dS K, dK = scale dS^T Q; a kv head's
 * dK, dV sum over its query heads).  dQ of a row is accumulated inside one CTA, so results do
 * not depend on scheduling (no atomics).
 *
 *   q, out, dout, dq  bf16 [total_q, nheads_q, head_dim]
 *   k, v, dk, dv      bf16 [total_k, nheads_kv, head_dim]
 *   lse               fp32 [nheads_q, total_q] from attn_fwd (natural log)
 *   the remaining arguments as in attn_fwd (same sequences, mask, window and scale).
 *   workspace: attn_bwd_workspace_bytes(total_q, nheads_q) bytes, 256-byte aligned (D).
 * Rows without a visible key get zero gradient; keys no row sees get dk = dv = 0.  With
 * total_q == 0 only dk and dv are written (zeros) and q, out, dout, lse, dq may be NULL; with
 * total_k == 0 only dq is (zeros) and k, v, dk, dv may be NULL.
 * Ownership: caller's buffers.  Errors: argument checks before any launch; inconsistent
 * cu_seqlens raise ATTN_ERR_DEVICE_BOUNDS.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                       int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                       int causal, int window_left, int window_right, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Workspace bytes for attn_bwd (D, fp32 per (head, token)). */
size_t attn_bwd_workspace_bytes(int total_q, int nheads_q);

/*
 * attn_fwd with the score modifiers of "04 · FA4 (CuTeDSL) and engineering interfaces",
 * section 7, applied to each scaled score s = softmax_scale * q.k before the mask:
 *   softcap > 0     s -> softcap * tanh(s / softcap)      (0 = off)
 *   alibi_slopes    device fp32 [nheads_q] or NULL: s -> s - slope_h * |i + Lk - Lq - j|
 *                   (query i at its bottom-right position, key j)
 * LSE is that of the modified scores.  Other arguments, layouts and errors as attn_fwd;
 * softcap must be 0 or in [2^-20, 1e30].
 */
attn_status_t attn_fwd_mods(const void* q, const void* k, const void* v, void* out, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                            int nheads_q, int nheads_kv, int head_dim, float softmax_scale,
                            int causal, int window_left, int window_right, float softcap,
                            const float* alibi_slopes, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * FP8 (e4m3) forward ("Attention kernels: FlashAttention and PagedAttention", section 四.2,
 * FlashAttention-3): Q, K and V as e4m3 bytes with block-wise fp32 scales, V re-laid out
 * key-major; the result is the attention of the dequantized values.
 *   q8      device u8 e4m3 [total_q, nheads_q, head_dim]
 *   k8      device u8 e4m3 [total_k, nheads_kv, head_dim] (may be NULL when total_k == 0)
 *   v8t     device u8 e4m3 [nheads_kv, head_dim, 128 * key_blocks]: V transposed; key t of
 *           sequence b sits in column 128 * kb0[b] + (t - cu_seqlens_k[b]), kb0 the prefix sum
 *           of ceil(Lk_b / 128); columns past a sequence's keys must hold finite values (zero)
 *   q_scale device fp32 [nheads_q, ceil(total_q / 128)]: one scale per 128 consecutive packed
 *           query tokens (row value = code * scale)
 *   k_scale device fp32 [nheads_kv, key_blocks]: one scale per 128-key block of a sequence
 *           (block kb0[b] + (t - cu_seqlens_k[b]) / 128)
 *   v_scale device fp32 [batch, nheads_kv]: one scale per (sequence, kv head)
 *   key_blocks >= kb0[batch]; a sequence whose blocks run past it sets the device bounds flag.
 * out, lse, cu_seqlens, sizes, causal and window as attn_fwd; head_dim must be 128.  Within
 * the kernel P is rounded to e4m3 (as 16 P~ with P~ <= 16), S and O accumulate in fp32, and
 * LSE is computed from the unrounded P~.  The rounding of P is the only approximation added to
 * the exact attention of the dequantized inputs: each element of O differs from it by at most
 * 2^-4 sum_j P_j |v_j| (keys in e4m3's normal range, 16 P~ >= 2^-6) plus a term below
 * 2^-14 |v_j| / l per remaining key, plus the bf16 rounding of O.
 */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8t,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* out, float* lse, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, int batch, int total_q, int total_k,
                           int max_seqlen_q, int max_seqlen_k, int nheads_q, int nheads_kv,
                           int head_dim, int key_blocks, float softmax_scale, int causal,
                           int window_left, int window_right, void* stream);

/*
 * bf16 Q, K, V to the inputs of attn_fwd_fp8 (same page and section): for each block,
 * amax = max |x|, scale = amax / 448 (1 for an all-zero block), code = e4m3(x * (448 / amax)),
 * round to nearest even and saturating, each step one IEEE fp32 operation.
 *   q, k, v      device bf16 [total_q, nheads_q, 128], [total_k, nheads_kv, 128] x 2
 *   signs        device fp32 [128] of +1 / -1, or NULL: Q and K rows are first rotated by
 *                H diag(signs) / sqrt(128) (H the Walsh-Hadamard matrix, "incoherent
 *                processing"; Q K^T is unchanged); V is never rotated
 *   key_blocks   >= sum_b ceil(Lk_b / 128), e.g. ceil(total_k / 128) + batch
 *   outputs      q8, q_scale, k8, k_scale, v8t, v_scale in the layouts attn_fwd_fp8 reads;
 *                unused key blocks get scale 1 and zero V^T columns
 * cu_seqlens_k as attn_fwd (rows outside [0, total_k) are never read); head_dim must be 128.
 */
attn_status_t attn_quantize_fp8(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens_k, int batch, int total_q, int total_k,
                                int max_seqlen_k, int nheads_q, int nheads_kv, int head_dim,
                                int key_blocks, const float* signs, void* q8, float* q_scale,
                                void* k8, float* k_scale, void* v8t, float* v_scale,
                                void* stream);

/* Bytes of split-partial workspace for attn_decode_kvcache; num_splits 0 sizes for the
 * automatic choice (at most 16 splits).  0 when one split needs no workspace. */
size_t attn_decode_workspace_bytes(int batch, int nheads_q, int head_dim, int num_splits);

/* The split count num_splits = 0 resolves to, for these sizes on a GPU with num_sms SMs. */
int attn_decode_num_splits(int batch, int nheads_q, int nheads_kv, int max_pages_per_seq,
                           int page_size, int num_sms);

/*
 * Synchronises `stream`, then returns and clears the current device's status word:
 * ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_DEVICE_BOUNDS, ATTN_ERR_CUDA for a sticky CUDA error,
 * else ATTN_OK.
 */
attn_status_t attn_get_device_status(void* stream);

/*
 * Failure-path self-test.  Launches, on `stream`, one small kernel whose threads wait with the
 * attention kernels' bounded wait (limit shortened to 20 ms) on a barrier that nothing ever
 * completes.  The wait runs out, raises the timeout bit of the device status word and the
 * kernel returns normally: a following attn_get_device_status() returns
 * ATTN_ERR_DEVICE_TIMEOUT (and clears it) and the context stays usable.  Returns ATTN_OK once
 * the kernel is launched, ATTN_ERR_CUDA if the launch fails.
 */
attn_status_t attn_selftest_wait_timeout(void* stream);

/*
 * Softcap check.  Writes out[i] = softcap * tanh(softmax_scale * scores[i] / softcap) for
 * i < n, computed on `stream` by the device code attn_fwd_mods applies to each score
 * (tanh u = 1 - 2 / (e^(2u) + 1) with the hardware exp2 and reciprocal, u = scale s / c).
 * scores, out: device fp32 [n], 8-byte aligned, caller-owned; n even.
 * Returns ATTN_ERR_INVALID_ARG for a bad n, pointer, scale or softcap (which must lie in
 * [2^-20, 1e30]), ATTN_ERR_CUDA if the launch fails, else ATTN_OK.
 */
attn_status_t attn_selftest_softcap(const float* scores, float* out, int n, float softmax_scale,
                                    float softcap, void* stream);

/* Static description of a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * Host copy of the key-block range rule the prefill kernels use ("Attention kernels ...",
 * section 七.2-七.3; "04 · FA4 ...", section 7: n_block_min / n_block_max).  For query rows
 * i_min..i_max (0-based within the sequence) it stores in *lo, *hi the half-open range of
 * block_n-key blocks holding any visible key, and returns 0.  attn_kv_block_masked() returns 1
 * when block j holds a key invisible to some row of i_min..i_max (so the kernel masks it
 * element-wise), else 0.  Exposed so the integer work can be checked without a GPU.
 */
int attn_kv_block_range(int i_min, int i_max, int seqlen_q, int seqlen_k, int block_n,
                        int causal, int window_left, int window_right, int* lo, int* hi);
int attn_kv_block_masked(int j, int i_min, int i_max, int seqlen_q, int seqlen_k, int block_n,
                         int causal, int window_left, int window_right);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
