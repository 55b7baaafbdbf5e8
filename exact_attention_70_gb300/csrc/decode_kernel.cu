// decode_kernel.cu -- seqlen_q = 1 decode over a paged KV cache: split-KV partials and the
// LSE-weighted combine.
//
// The method ("Attention kernels: FlashAttention and PagedAttention", sections 五.2-五.3,
// 六.1 and 六.3; "04 · FA4 (CuTeDSL) and engineering interfaces", sections 5, 6.1 and 6.2):
// the keys of sequence b are split into num_splits contiguous ranges; for each (b, kv head,
// split) one CTA gathers its K/V through block_table and runs the online softmax over the
// range with the g query heads of that kv head packed as rows, so every K/V byte is read from
// HBM once; each split emits (O_s normalised, LSE_s) and a second kernel merges them with
// weights exp(LSE_s - LSE).
//
// GB300 mapping.  The work is HBM-bound (about g FLOP per byte), so the design goal is bytes
// in flight: warp 4 issues one TMA box per (page piece, 64 columns of d) into a 3-stage ring
// of 64-key chunks (32 KiB per stage at d = 128), two CTAs per SM.  Warps 0-3 each take 16
// keys of every chunk; the tiny GEMMs (16 packed rows x 16 keys x d) run on the warp-level
// mma.sync tensor path straight from the 128-byte-swizzled TMA tiles via ldmatrix, leaving
// the FP32 pipes idle.  Row max and sum are reduced with quad shuffles; the four warps'
// (m, l, O) are merged through shared memory at the end.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr float kLn2f = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct DecCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = kDecChunk * 128;       // 64 keys x 128 B
    static constexpr int kKvBytes = kHalves * kHalfBytes;     // K (or V) of one chunk
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kStages = D == 128 ? 3 : 6;
    static constexpr int kOffBar = kStages * kStageBytes;
    static constexpr int kMergeStride = D + 4;                // floats per merged row
    static constexpr int kMergeBytes = 4 * kDecRowsPerCta * kMergeStride * 4 + 2 * 4 * 16 * 4;
    static_assert(kMergeBytes <= kOffBar, "merge buffer must fit in the stage ring");
    static constexpr int kSmem = kOffBar + 256 + 1024;
};

struct DecBars {
    uint64_t full[8], empty[8];
    int abort_flag;
};

__device__ __forceinline__ uint32_t swz(int row, int oct) {
    return static_cast<uint32_t>(row * 128 + ((oct ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_split_kernel(const __grid_constant__ DecParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    DecBars* bars = reinterpret_cast<DecBars*>(smem + C::kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.hgroups, hg = blockIdx.y % p.hgroups;
    const int b = blockIdx.z;
    const int S = p.num_splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 4);
        }
        bars->abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const Watchdog wd{&bars->abort_flag, p.status};

    // Key range of this split, in whole 64-key chunks.
    int L = p.seqlens[b];
    const int Lmax = p.max_pages * p.page_size;
    if (L < 0 || L > Lmax) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBounds);
        L = L < 0 ? 0 : Lmax;
    }
    const int nch = (L + kDecChunk - 1) / kDecChunk;
    const int per = (nch + S - 1) / S;
    const int c0 = min(split * per, nch), c1 = min(c0 + per, nch);

    const int rows = min(kDecRowsPerCta, p.g - hg * kDecRowsPerCta);  // valid packed rows
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    if (warp == 4) {
        // ---- producer: gather pages through block_table ----
        if (lane == 0 && c1 > c0) {
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            const int* bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
            const int pieces = kDecChunk / p.box_rows;
            uint32_t issued = 0;
            for (int c = c0; c < c1; ++c, ++issued) {
                const uint32_t st = issued % C::kStages;
                if (issued >= C::kStages &&
                    !wd.wait(&bars->empty[st], ((issued / C::kStages) - 1) & 1))
                    break;
                mbar_arrive_expect_tx(&bars->full[st], C::kStageBytes);
                uint8_t* kdst = smem + st * C::kStageBytes;
                uint8_t* vdst = kdst + C::kKvBytes;
                for (int pc = 0; pc < pieces; ++pc) {
                    const int tok = c * kDecChunk + pc * p.box_rows;
                    // A piece wholly past the sequence end (possible in the last chunk when
                    // pages are shorter than a chunk) is aimed past the end of the cache, so
                    // TMA fills it with zeros and its block_table entry is never read.
                    int page = p.num_pages;
                    if (tok < L) {
                        page = bt[tok / p.page_size];
                        if (page < 0 || page >= p.num_pages) {
                            // an out-of-range id loads zeros (TMA fills outside the tensor)
                            atomicOr(p.status, kStatusBounds);
                            page = p.num_pages;
                        }
                    }
                    const int row = page * p.page_size + tok % p.page_size;
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h) {
                        tma_load_3d(kdst + h * C::kHalfBytes + pc * p.box_rows * 128, &p.tm_k,
                                    &bars->full[st], h * 64, kvh, row);
                        tma_load_3d(vdst + h * C::kHalfBytes + pc * p.box_rows * 128, &p.tm_v,
                                    &bars->full[st], h * 64, kvh, row);
                    }
                }
            }
            // wait for every load still in flight before the ring is reused for the merge; a
            // load that never lands raises the timeout status and the abort flag, so that
            // nothing is merged or stored from this CTA
            const uint32_t n_st = issued < C::kStages ? issued : C::kStages;
            for (uint32_t st = 0; st < n_st; ++st) {
                const uint32_t last = st + C::kStages * ((issued - 1 - st) / C::kStages);
                const unsigned long long t0 = global_ns();
                bool landed = true;
                while (!mbar_try(&bars->full[st], (last / C::kStages) & 1)) {
                    if (global_ns() - t0 > kWaitLimitNs) {
                        landed = false;
                        break;
                    }
                }
                if (!landed) {
                    wd.fail();
                    break;
                }
            }
        }
    } else {
        // ---- consumers: warp w owns keys [16 w, 16 w + 16) of every chunk ----
        const int gq = lane >> 2, tq = lane & 3;
        // Q as the A operand (16 packed rows x d), rows >= `rows` are zero.
        uint32_t qa[D / 16][4];
        {
            const int r0 = gq, r1 = gq + 8;
            const __nv_bfloat16* qb =
                p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.g + hg * kDecRowsPerCta) * D;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = kk * 16 + 2 * tq;
                qa[kk][0] = r0 < rows ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + c) : 0u;
                qa[kk][1] = r1 < rows ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + c) : 0u;
                qa[kk][2] =
                    r0 < rows ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + c + 8) : 0u;
                qa[kk][3] =
                    r1 < rows ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + c + 8) : 0u;
            }
        }
        const float sl2 = p.scale_log2;
        const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix id, row within matrix
        for (int c = c0; c < c1; ++c) {
            const uint32_t n = c - c0, st = n % C::kStages;
            if (!__all_sync(0xffffffffu, wd.wait(&bars->full[st], (n / C::kStages) & 1))) break;
            uint8_t* kst = smem + st * C::kStageBytes;
            uint8_t* vst = kst + C::kKvBytes;
            const int key0 = c * kDecChunk + warp * 16;
            const int nvalid = min(16, L - key0);
            if (nvalid < 16) {
                // keys past the sequence end: zero their V rows so 0 * garbage cannot be NaN
                for (int i = lane; i < (16 - max(nvalid, 0)) * C::kHalves * 8; i += 32) {
                    const int r = warp * 16 + max(nvalid, 0) + i / (C::kHalves * 8);
                    const int rest = i % (C::kHalves * 8);
                    *reinterpret_cast<uint4*>(vst + (rest / 8) * C::kHalfBytes + r * 128 +
                                              (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (nvalid > 0) {
                // S (16 rows x 16 keys) = Q K^T
                float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const uint32_t kbase = smem_u32(kst);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int key = warp * 16 + (mi >> 1) * 8 + ri;
                    const int oct = 2 * kk + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(kbase + (oct >> 3) * C::kHalfBytes + swz(key, oct & 7), b0, b1,
                                b2, b3);
                    mma_bf16_16816(s[0], qa[kk], b0, b1);
                    mma_bf16_16816(s[1], qa[kk], b2, b3);
                }
                // mask keys past the end, then the online softmax in the exp2 domain
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = nt * 8 + 2 * tq + (e & 1);
                        s[nt][e] = col < nvalid ? s[nt][e] * sl2 : -INFINITY;
                    }
                float mx[2];
                mx[0] = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                mx[1] = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                }
                float alpha[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float m_new = fmaxf(m_run[r], mx[r]);
                    alpha[r] = ex2_approx(m_run[r] - m_new);
                    m_run[r] = m_new;
                }
                uint32_t pa[4];
                float rs[2] = {0.f, 0.f};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float p0 = ex2_approx(s[nt][0] - m_run[0]);
                    const float p1 = ex2_approx(s[nt][1] - m_run[0]);
                    const float p2 = ex2_approx(s[nt][2] - m_run[1]);
                    const float p3 = ex2_approx(s[nt][3] - m_run[1]);
                    rs[0] += p0 + p1;
                    rs[1] += p2 + p3;
                    pa[2 * nt + 0] = pack_bf16x2(p0, p1);
                    pa[2 * nt + 1] = pack_bf16x2(p2, p3);
                }
                l_run[0] = l_run[0] * alpha[0] + rs[0];
                l_run[1] = l_run[1] * alpha[1] + rs[1];
                // A fragment of P: (row g, keys 2t..) (row g+8, ..) (row g, keys 8+2t..) ...
                const uint32_t pfrag[4] = {pa[0], pa[1], pa[2], pa[3]};
                const uint32_t vbase = smem_u32(vst);
#pragma unroll
                for (int nn = 0; nn < D / 8; nn += 2) {
                    const int key = warp * 16 + (mi & 1) * 8 + ri;
                    const int oct = nn + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(vbase + (oct >> 3) * C::kHalfBytes + swz(key, oct & 7), b0,
                                      b1, b2, b3);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o[nn][e] *= alpha[e >> 1];
                        o[nn + 1][e] *= alpha[e >> 1];
                    }
                    mma_bf16_16816(o[nn], pfrag, b0, b1);
                    mma_bf16_16816(o[nn + 1], pfrag, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->empty[st]);
        }
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
    }
    __syncthreads();  // the ring is idle from here on: reuse it for the cross-warp merge
    if (wd.aborted()) return;  // a wait ran out: the status word says so, nothing is stored

    float* mo = reinterpret_cast<float*>(smem);  // [4 warps][16 rows][kMergeStride]
    float* mm = mo + 4 * kDecRowsPerCta * C::kMergeStride;  // [4][16] running max
    float* ml = mm + 4 * 16;                                 // [4][16] denominators
    if (warp < 4) {
        const int gq = lane >> 2, tq = lane & 3;
        float* w = mo + warp * kDecRowsPerCta * C::kMergeStride;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            *reinterpret_cast<float2*>(w + gq * C::kMergeStride + n * 8 + 2 * tq) =
                make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2*>(w + (gq + 8) * C::kMergeStride + n * 8 + 2 * tq) =
                make_float2(o[n][2], o[n][3]);
        }
        if (tq == 0) {
            mm[warp * 16 + gq] = m_run[0];
            mm[warp * 16 + gq + 8] = m_run[1];
            ml[warp * 16 + gq] = l_run[0];
            ml[warp * 16 + gq + 8] = l_run[1];
        }
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        for (int e = threadIdx.x; e < rows * D; e += 128) {
            const int r = e / D, d = e % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) M = fmaxf(M, mm[w * 16 + r]);
            float lsum = 0.f, acc = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float sc = ex2_approx(mm[w * 16 + r] - M);
                    lsum += ml[w * 16 + r] * sc;
                    acc += mo[(w * kDecRowsPerCta + r) * C::kMergeStride + d] * sc;
                }
            }
            const float out = lsum > 0.f ? acc / lsum : 0.f;
            const float lse = lsum > 0.f ? (M + __log2f(lsum)) * kLn2f : -INFINITY;
            const int head = kvh * p.g + hg * kDecRowsPerCta + r;
            const size_t bh = static_cast<size_t>(b) * p.Hq + head;
            if (!ATTN_IN_BOUNDS(head < p.Hq && b < p.batch, p.status)) continue;
            if (S == 1) {
                p.out[bh * D + d] = __float2bfloat16_rn(out);
                if (d == 0) p.lse[bh] = lse;
            } else {
                p.part_o[(bh * S + split) * D + d] = out;
                if (d == 0) p.part_lse[bh * S + split] = lse;
            }
        }
    }
}

// One warp per (b, h): LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s
// ("Attention kernels ...", section 六.3; an empty split has LSE_s = -inf and weight 0).
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(CombineParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= p.rows) return;
    const int S = p.num_splits;
    const float* pl = p.part_lse + static_cast<size_t>(row) * S;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, pl[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    constexpr int E = D / 32;  // elements per lane
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float sum = 0.f;
        for (int s = lane; s < S; s += 32) sum += ex2_approx((pl[s] - M) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        lse = M + __logf(sum);
        const float* po = p.part_o + static_cast<size_t>(row) * S * D + lane * E;
        for (int s = 0; s < S; ++s) {
            const float w = ex2_approx((pl[s] - lse) * kLog2e);
            const float* src = po + static_cast<size_t>(s) * D;
            if constexpr (E == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
    __nv_bfloat16* dst = p.out + static_cast<size_t>(row) * D + lane * E;
    if constexpr (E == 4) {
        uint2 v;
        v.x = pack_bf16x2(acc[0], acc[1]);
        v.y = pack_bf16x2(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(dst) = v;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
    }
    if (lane == 0) p.lse[row] = lse;
}

}  // namespace

int decode_smem_bytes(int head_dim) {
    return head_dim == 128 ? DecCfg<128>::kSmem : DecCfg<64>::kSmem;
}

cudaError_t configure_decode_kernels() {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecCfg<128>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_split_kernel<64>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<64>::kSmem);
}

cudaError_t launch_decode(const DecParams& p, int head_dim, cudaStream_t stream) {
    const dim3 grid(p.num_splits, p.Hkv * p.hgroups, p.batch);
    if (head_dim == 128)
        decode_split_kernel<128><<<grid, kDecThreads, DecCfg<128>::kSmem, stream>>>(p);
    else
        decode_split_kernel<64><<<grid, kDecThreads, DecCfg<64>::kSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, int head_dim, cudaStream_t stream) {
    const int grid = (p.rows + 3) / 4;
    if (head_dim == 128)
        decode_combine_kernel<128><<<grid, 128, 0, stream>>>(p);
    else
        decode_combine_kernel<64><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
