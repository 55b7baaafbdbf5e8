// kvcache.cu -- the in-place cache append of a chunked-prefill step, with rotary embedding.
//
// "Attention kernels: FlashAttention and PagedAttention", section 五.1 (chunked prefill: the
// new tokens' K/V are written into the cache and then read by the same step) and "04 · FA4
// (CuTeDSL) and engineering interfaces", sections 6.1-6.2 (block_table addressing,
// cache_seqlens, the in-place append of the new k, v that also applies the rotary
// embedding).  New token i of sequence b sits at position cache_seqlens[b] + i: its key
// (rotated) and value go to that position of the paged cache, and its queries are rotated
// into a separate buffer the attention kernel reads.
//
// Rotary embedding (the standard form; the pages name it without a formula): the first
// rot_dim components are rotated in rot_dim / 2 planes, (a, b) -> (a cos - b sin,
// a sin + b cos), with cos, sin from row `position` of the caller's tables; the planes pair
// (x_i, x_{i + rot_dim/2}) or, interleaved, (x_{2i}, x_{2i+1}).  Each rotated component is a
// difference of two products, evaluated in fp32 with Kahan's algorithm for a b - c d (error
// bounded by about 1.5 ulp of the result even under cancellation: C.-P. Jeannerod,
// N. Louvet, J.-M. Muller, "Further analysis of Kahan's algorithm for the accurate
// computation of 2x2 determinants", 2013), then rounded to bf16 (nearest, ties to even).
//
// One thread per 16 bytes (8 elements) of a row: memory-bound, every byte read and written
// once, apart from the partner half of a rotate-half plane, which is read twice.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

__device__ __forceinline__ int find_seq(const int* cu, int batch, int t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

// a b - c d: w = c d rounded, e = the exact rounding error of w (one FMA), then
// fma(a, b, -w) + e.
__device__ __forceinline__ float det2(float a, float b, float c, float d) {
    const float w = c * d;
    const float e = fmaf(-c, d, w);
    return fmaf(a, b, -w) + e;
}

// Rotated copy of the 8 elements [e0, e0 + 8) of a d-row; the whole row is at `row`.
__device__ __forceinline__ uint4 rotate8(const AppendParams& p, const __nv_bfloat16* row, int e0,
                                         int pos) {
    const uint4 own = *reinterpret_cast<const uint4*>(row + e0);
    if (e0 >= p.rot_dim) return own;
    const int half = p.rot_dim / 2;
    const float* cr = p.rot_cos + static_cast<size_t>(pos) * half;
    const float* sr = p.rot_sin + static_cast<size_t>(pos) * half;
    float x[8], y[8];
    unpack8(own, x);
    if (p.interleaved) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float c = cr[e0 / 2 + i], s = sr[e0 / 2 + i];
            y[2 * i] = det2(x[2 * i], c, x[2 * i + 1], s);
            y[2 * i + 1] = det2(x[2 * i], s, -x[2 * i + 1], c);
        }
    } else {
        float z[8];
        const bool first = e0 < half;  // plane partner lies rot_dim/2 further on, or before
        unpack8(*reinterpret_cast<const uint4*>(row + (first ? e0 + half : e0 - half)), z);
        const int tix = first ? e0 : e0 - half;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float c = cr[tix + i], s = sr[tix + i];
            y[i] = first ? det2(x[i], c, z[i], s) : det2(z[i], s, -x[i], c);
        }
    }
    return pack8(y);
}

__global__ void __launch_bounds__(256) kvcache_append_kernel(const AppendParams p) {
    const int chunks = p.d / 8;
    const int rows_per_tok = 2 * p.Hkv + (p.rot_dim > 0 ? p.Hq : 0);
    const long long total = static_cast<long long>(p.total_q) * rows_per_tok * chunks;
    for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < total;
         u += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int e0 = static_cast<int>(u % chunks) * 8;
        const long long rt = u / chunks;
        const int r = static_cast<int>(rt % rows_per_tok);
        const int t = static_cast<int>(rt / rows_per_tok);
        const int b = find_seq(p.cu_q, p.batch, t);
        const int pos = p.cache_seqlens[b] + (t - p.cu_q[b]);
        if (p.rot_dim > 0 && pos >= p.rot_rows) {
            atomicOr(p.status, kStatusBounds);
            continue;
        }
        if (r < 2 * p.Hkv) {  // key (r < Hkv) or value row of kv head r % Hkv
            const int kvh = r % p.Hkv;
            if (pos >= p.max_pages * p.page_size) {
                atomicOr(p.status, kStatusBounds);
                continue;
            }
            const int page = p.block_table[static_cast<size_t>(b) * p.max_pages + pos / p.page_size];
            if (page < 0 || page >= p.num_pages) {
                atomicOr(p.status, kStatusBounds);
                continue;
            }
            const size_t dst =
                ((static_cast<size_t>(page) * p.page_size + pos % p.page_size) * p.Hkv + kvh) * p.d + e0;
            const size_t src = (static_cast<size_t>(t) * p.Hkv + kvh) * p.d;
            if (!ATTN_IN_BOUNDS(t < p.total_q && kvh < p.Hkv && e0 + 8 <= p.d, p.status)) continue;
            if (r < p.Hkv) {
                const uint4 w = p.rot_dim > 0 ? rotate8(p, p.k_new + src, e0, pos)
                                              : *reinterpret_cast<const uint4*>(p.k_new + src + e0);
                *reinterpret_cast<uint4*>(p.k_cache + dst) = w;
            } else {
                *reinterpret_cast<uint4*>(p.v_cache + dst) =
                    *reinterpret_cast<const uint4*>(p.v_new + src + e0);
            }
        } else {  // rotated query row of head r - 2 Hkv
            const int h = r - 2 * p.Hkv;
            const size_t row = (static_cast<size_t>(t) * p.Hq + h) * p.d;
            if (!ATTN_IN_BOUNDS(t < p.total_q && h < p.Hq && e0 + 8 <= p.d, p.status)) continue;
            *reinterpret_cast<uint4*>(p.q_rot + row + e0) = rotate8(p, p.q + row, e0, pos);
        }
    }
}

}  // namespace

cudaError_t launch_kvcache_append(const AppendParams& p, int num_sms, cudaStream_t stream) {
    const long long total =
        static_cast<long long>(p.total_q) * (2 * p.Hkv + (p.rot_dim > 0 ? p.Hq : 0)) * (p.d / 8);
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    kvcache_append_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
