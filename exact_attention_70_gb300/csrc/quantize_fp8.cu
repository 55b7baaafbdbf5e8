// quantize_fp8.cu -- bf16 Q, K, V to the FP8 (e4m3) inputs of the FP8 forward pass.
//
// The method ("Attention kernels: FlashAttention and PagedAttention", section 四.2,
// FlashAttention-3): Q, K and V are rounded to e4m3 with one scale per block, after the
// optional "incoherent processing" that multiplies Q and K by the same random orthogonal matrix
// (here H diag(signs) / sqrt(d), H the Walsh-Hadamard matrix), and V is re-laid out key-major.
// For a block: amax = max |x|, scale = amax / 448 (1 when the block is zero), code = e4m3(x r)
// with r = 448 / amax formed once per block, round to nearest even, saturating.  Every fp32
// step is one IEEE operation.
//
// Layouts (as the FP8 forward reads them):
//   q8 [total_q, Hq, d], q_scale [Hq, ceil(total_q / 128)]: blocks of 128 packed tokens;
//   k8 [total_k, Hkv, d], k_scale [Hkv, key_blocks]: blocks of 128 keys of one sequence,
//       block kb0[b] + i (kb0 the prefix sum of ceil(Lk_b / 128)); unused blocks get scale 1;
//   v8t [Hkv, d, 128 key_blocks]: V transposed, key t of sequence b in column
//       128 kb0[b] + (t - k0), zero elsewhere; v_scale [batch, Hkv]: one per sequence and head.
// Kernels: quant_rows_kernel (Q or K, one CTA per block and head, a warp per 16 rows, a row
// per 8 lanes with 16 values a lane: four of the transform's seven butterfly stages inside the
// lane, three across lanes by shuffles), quant_v_amax_kernel
// (atomic max of |V| per sequence and head), quant_v_kernel (one CTA per key block and head,
// transposed through shared memory), quant_v_finalize_kernel (amax -> scale).  All of it is
// bandwidth-bound: each input byte is read once (V twice) and each output byte written once.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kQThreads = 256;  // 8 warps x 16 rows = one 128-row block
constexpr float kInvSqrt128 = 0.0883883476483184405f;  // 1 / sqrt(128), rounded to fp32 once

// Sequence b holding key block blk of the per-sequence numbering, and the block's index i
// within it; b = batch when blk is past the last sequence's blocks.
__device__ __forceinline__ void key_block_owner(const int* cu_k, int batch, int blk, int& b,
                                                int& i) {
    int kb0 = 0;
    for (b = 0; b < batch; ++b) {
        const int nb = (cu_k[b + 1] - cu_k[b] + 127) / 128;
        if (blk < kb0 + nb) {
            i = blk - kb0;
            return;
        }
        kb0 += nb;
    }
    i = 0;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    return pack_e4m3x4(a, b, c, d);
}

// One block of up to 128 rows (token rows t0.., of head h) of a [total, H, 128] bf16 tensor.
// kKeys: blocks are 128 keys of a sequence (K); otherwise 128 consecutive tokens (Q).
template <bool kKeys>
__global__ void __launch_bounds__(kQThreads) quant_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                                uint8_t* __restrict__ dst,
                                                                float* __restrict__ scale,
                                                                const int* __restrict__ cu_k,
                                                                const float* __restrict__ signs,
                                                                int batch, int total, int H,
                                                                int nblocks) {
    const int blk = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t0 = 128 * blk, t1 = min(total, t0 + 128);
    if (kKeys) {
        int b, i;
        key_block_owner(cu_k, batch, blk, b, i);
        if (b >= batch) {  // a block past the sequences: scale 1, no codes
            if (threadIdx.x == 0) scale[static_cast<size_t>(h) * nblocks + blk] = 1.f;
            return;
        }
        t0 = cu_k[b] + 128 * i;
        t1 = min(min(cu_k[b + 1], t0 + 128), total);  // (rows are clamped to the tensor)
        if (t0 < 0) t0 = t1;
    }
    // Each row is spread over a group of 8 lanes, 16 consecutive values a lane (element
    // i = 16 j + k, j = lane % 8): the transform's stages h = 1 .. 8 stay inside the lane and
    // h = 16, 32, 64 cross lanes j ^ 1, 2, 4.  A warp takes 4 rows at a time, 16 rows in all.
    const int j = lane & 7, sub = lane >> 3;
    float sg[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) sg[k] = signs != nullptr ? signs[16 * j + k] : 1.f;
    // all four rows' loads first, so that 128 bytes a lane are in flight at once
    uint4 raw[4][2];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int t = t0 + 16 * warp + 4 * it + sub;
        if (t < t1) {
            const uint4* src4 = reinterpret_cast<const uint4*>(src + (static_cast<size_t>(t) * H + h) * 128 + 16 * j);
            raw[it][0] = src4[0];
            raw[it][1] = src4[1];
        } else {
            raw[it][0] = raw[it][1] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    float x[4][16];
    float amax = 0.f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int t = t0 + 16 * warp + 4 * it + sub;
        float* v = x[it];
        {
            const uint32_t w[8] = {raw[it][0].x, raw[it][0].y, raw[it][0].z, raw[it][0].w,
                                   raw[it][1].x, raw[it][1].y, raw[it][1].z, raw[it][1].w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                v[2 * q] = __uint_as_float(w[q] << 16);
                v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            }
        }
        if (signs != nullptr) {
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], sg[k]);
            // pair (lower, upper) -> (lower + upper, lower - upper), stage by stage
#pragma unroll
            for (int hh = 1; hh < 16; hh <<= 1)
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if ((k & hh) == 0) {
                        const float a = v[k], c = v[k + hh];
                        v[k] = __fadd_rn(a, c);
                        v[k + hh] = __fsub_rn(a, c);
                    }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
                const bool upper = (j & m) != 0;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float other = __shfl_xor_sync(0xffffffffu, v[k], m);
                    v[k] = upper ? __fsub_rn(other, v[k]) : __fadd_rn(v[k], other);
                }
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], kInvSqrt128);
        }
        if (t < t1) {
#pragma unroll
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __shared__ float red[kQThreads / 32];
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const float rcp = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    if (threadIdx.x == 0) scale[static_cast<size_t>(h) * nblocks + blk] = s;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int t = t0 + 16 * warp + 4 * it + sub;
        const float* v = x[it];
        if (t < t1) {
            uint32_t c[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                c[q] = e4m3x4(__fmul_rn(v[4 * q], rcp), __fmul_rn(v[4 * q + 1], rcp),
                              __fmul_rn(v[4 * q + 2], rcp), __fmul_rn(v[4 * q + 3], rcp));
            *reinterpret_cast<uint4*>(dst + (static_cast<size_t>(t) * H + h) * 128 + 16 * j) =
                make_uint4(c[0], c[1], c[2], c[3]);
        }
    }
}

// max |V| per (sequence, kv head), as fp32 bits, into amax[b * Hkv + h] (zeroed first).
__global__ void __launch_bounds__(256) quant_v_amax_kernel(const __nv_bfloat16* __restrict__ v,
                                                           const int* __restrict__ cu_k,
                                                           unsigned* __restrict__ amax_bits,
                                                           int Hkv, int total_k) {
    const int b = blockIdx.y / Hkv, h = blockIdx.y % Hkv;
    const int k0 = max(cu_k[b], 0), k1 = min(cu_k[b + 1], total_k);
    const int t0 = k0 + 128 * blockIdx.x;
    // 128 rows x 16 pieces of 8 values, eight pieces a thread, all loads issued before any use
    uint4 u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int t = t0 + idx / 16;
        u[i] = t < k1 ? *reinterpret_cast<const uint4*>(v + (static_cast<size_t>(t) * Hkv + h) * 128 + 8 * (idx % 16))
                      : make_uint4(0u, 0u, 0u, 0u);
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax_bits + blockIdx.y, __float_as_uint(m));
}

// One 128-key block of V for kv head h: codes with the sequence's scale, written transposed
// (v8t row = one of the d dimensions, 128 key columns); padding keys and unused blocks are 0.
__global__ void __launch_bounds__(256) quant_v_kernel(const __nv_bfloat16* __restrict__ v,
                                                      const int* __restrict__ cu_k,
                                                      const unsigned* __restrict__ amax_bits,
                                                      uint8_t* __restrict__ v8t, int batch,
                                                      int Hkv, int key_blocks, int total_k) {
    __shared__ uint32_t tile[128][33];  // [d][key / 4] codes, padded against bank conflicts
    const int blk = blockIdx.x, h = blockIdx.y;
    int b, i;
    key_block_owner(cu_k, batch, blk, b, i);
    int t0 = 0, n = 0;
    float rcp = 1.f;
    if (b < batch) {
        t0 = max(cu_k[b], 0) + 128 * i;
        n = max(0, min(min(cu_k[b + 1], total_k) - t0, 128));  // (rows are clamped to the tensor)
        const float amax = __uint_as_float(amax_bits[static_cast<size_t>(b) * Hkv + h]);
        rcp = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    }
    // thread: key group kg (4 consecutive keys) and d-quad dq; codes of 4 keys x 4 dims
    for (int w = threadIdx.x; w < 32 * 32; w += blockDim.x) {
        const int kg = w / 32, dq = w % 32;
        float x[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int key = 4 * kg + kk;
            if (key < n) {
                const uint2 u = *reinterpret_cast<const uint2*>(v + (static_cast<size_t>(t0 + key) * Hkv + h) * 128 + 4 * dq);
                x[kk][0] = __uint_as_float(u.x << 16);
                x[kk][1] = __uint_as_float(u.x & 0xFFFF0000u);
                x[kk][2] = __uint_as_float(u.y << 16);
                x[kk][3] = __uint_as_float(u.y & 0xFFFF0000u);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) x[kk][e] = 0.f;
            }
        }
        // for dimension 4 dq + e: bytes of keys 4 kg .. 4 kg + 3
#pragma unroll
        for (int e = 0; e < 4; ++e)
            tile[4 * dq + e][kg] = e4m3x4(__fmul_rn(x[0][e], rcp), __fmul_rn(x[1][e], rcp),
                                          __fmul_rn(x[2][e], rcp), __fmul_rn(x[3][e], rcp));
    }
    __syncthreads();
    const size_t cols = static_cast<size_t>(128) * key_blocks;
    for (int w = threadIdx.x; w < 128 * 32; w += blockDim.x) {
        const int dd = w / 32, kg = w % 32;
        *reinterpret_cast<uint32_t*>(v8t + (static_cast<size_t>(h) * 128 + dd) * cols + 128 * static_cast<size_t>(blk) + 4 * kg) =
            tile[dd][kg];
    }
}

__global__ void quant_v_finalize_kernel(float* v_scale, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const float amax = v_scale[i];  // holds the amax bits
        v_scale[i] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    }
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantParams& p, cudaStream_t stream) {
    const int nqb = (p.total_q + 127) / 128;
    if (nqb > 0)
        quant_rows_kernel<false><<<dim3(nqb, p.Hq), kQThreads, 0, stream>>>(
            p.q, p.q8, p.q_scale, p.cu_k, p.signs, p.batch, p.total_q, p.Hq, nqb);
    if (p.key_blocks > 0)
        quant_rows_kernel<true><<<dim3(p.key_blocks, p.Hkv), kQThreads, 0, stream>>>(
            p.k, p.k8, p.k_scale, p.cu_k, p.signs, p.batch, p.total_k, p.Hkv, p.key_blocks);
    cudaError_t e = cudaMemsetAsync(p.v_scale, 0, sizeof(float) * p.batch * p.Hkv, stream);
    if (e != cudaSuccess) return e;
    const int vb = (p.max_seqlen_k + 127) / 128;
    if (vb > 0 && p.batch > 0)
        quant_v_amax_kernel<<<dim3(vb, p.batch * p.Hkv), 256, 0, stream>>>(
            p.v, p.cu_k, reinterpret_cast<unsigned*>(p.v_scale), p.Hkv, p.total_k);
    if (p.key_blocks > 0)
        quant_v_kernel<<<dim3(p.key_blocks, p.Hkv), 256, 0, stream>>>(
            p.v, p.cu_k, reinterpret_cast<const unsigned*>(p.v_scale), p.v8t, p.batch, p.Hkv,
            p.key_blocks, p.total_k);
    const int n = p.batch * p.Hkv;
    if (n > 0) quant_v_finalize_kernel<<<(n + 255) / 256, 256, 0, stream>>>(p.v_scale, n);
    return cudaGetLastError();
}

}  // namespace attn
