// bwd_kernel.cu -- backward pass of exact attention on tcgen05 tensor cores.
//
// The method ("Attention kernels: FlashAttention and PagedAttention", section 四.3; "04 · FA4
// (CuTeDSL) and engineering interfaces", section 2 for the preprocess / postprocess split):
// only O and the row log-sum-exp L were kept by the forward pass, so the backward recomputes
// S = Q K^T blockwise and P = exp(S - L) in one step, forms D_i = rowsum(dO_i * O_i),
// dP = dO V^T and dS = P * (dP - D), and accumulates dV = P^T dO, dK = scale dS^T Q and
// dQ = scale dS K.
//
// GB300 mapping: three kernels, no atomics (dQ is accumulated in one CTA, so the result does
// not depend on scheduling):
//   * bwd_preprocess_kernel: D per (token, head), one warp per row;
//   * bwd_dkdv_kernel: one CTA per 128-key block of one (sequence, kv head); it walks the
//     128-row Q tiles (tokens x the g query heads, packed as in the forward pass) that see
//     the block, with S^T = K Q^T and dP^T = V dO^T in TMEM, P^T and dS^T written back over
//     them as bf16, and dV += P^T dO, dK += dS^T Q accumulated in TMEM;
//   * bwd_dq_kernel: one CTA per Q tile, walking the key blocks it sees, with S, dP in TMEM,
//     dS written back over S as bf16 and dQ += dS K accumulated in TMEM.
//   Roles per CTA: warps 0-7 the elementwise work (two warps per TMEM lane quarter, each
//   taking half of the columns), warp 8 TMA, warp 9 the MMA issuer and TMEM owner.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_math.h"

namespace attn {

namespace {

constexpr float kLog2e = 1.44269504088896341f;
constexpr int kBwdThreads = 384;

template <int D>
struct BwdCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kAtomBytes = 128 * 128;
    static constexpr int kTile = kHalves * kAtomBytes;  // 128 rows x D bf16, 128-B swizzle
};

struct BwdBars {
    uint64_t kv_full[2], kv_empty[2], q_full[2], q_empty[2];
    uint64_t s_full, p_full, mm_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Per packed row of a Q tile: -L * log2(e) (or -inf when the row has no gradient), D, and
// the row's visible key interval.
struct RowInfo {
    float nl[128];
    float dd[128];
    int kmin[128];
    int kmax[128];
};

__device__ void bwd_drain(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > 200000000ull) return;
}

// The sequence of (b, kvh) a CTA serves, checked against the tensors.
struct BwdSeq {
    int b, kvh, q0, Lq, k0, Lk;
    bool ok;
};

__device__ __forceinline__ BwdSeq bwd_seq(const BwdParams& p) {
    BwdSeq s;
    s.b = blockIdx.y / p.Hkv;
    s.kvh = blockIdx.y % p.Hkv;
    s.q0 = p.cu_q[s.b];
    s.Lq = p.cu_q[s.b + 1] - s.q0;
    s.k0 = p.cu_k[s.b];
    s.Lk = p.cu_k[s.b + 1] - s.k0;
    s.ok = s.q0 >= 0 && s.Lq >= 0 && s.q0 + s.Lq <= p.total_q && s.Lq <= p.max_seqlen_q &&
           s.k0 >= 0 && s.Lk >= 0 && s.k0 + s.Lk <= p.total_k && s.Lk <= p.max_seqlen_k;
    return s;
}

// Fill row information of Q tile i for packed rows r = 0..127 (threads 0..127 of the warps
// 0-7).  Rows past the tile's tokens or the sequence get no gradient (nl = -inf, D = 0).
__device__ void fill_rows(const BwdParams& p, const BwdSeq& sq, int i, bool masked, RowInfo& ri,
                          int r) {
    const int tok = i * p.tpt + r / p.g;
    const int head = sq.kvh * p.g + r % p.g;
    const bool valid = r < p.g * p.tpt && tok < sq.Lq;
    float nl = -INFINITY, dd = 0.f;
    int kmin = 1, kmax = 0;
    if (valid) {
        const size_t at = static_cast<size_t>(head) * p.total_q + sq.q0 + tok;
        const float l = p.lse[at];
        if (l != -INFINITY) nl = -l * kLog2e;
        dd = p.dsum[at];
        if (masked) row_key_interval(tok, sq.Lq, sq.Lk, p.causal, p.wl, p.wr, kmin, kmax);
    }
    ri.nl[r] = nl;
    ri.dd[r] = dd;
    ri.kmin[r] = kmin;
    ri.kmax[r] = kmax;
}

// ---- D = rowsum(dO * O) ---------------------------------------------------------------------

__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(p.total_q) * p.Hq;
    const long long step = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += step) {
        const uint32_t* o = reinterpret_cast<const uint32_t*>(p.o + r * p.d);
        const uint32_t* g = reinterpret_cast<const uint32_t*>(p.dout + r * p.d);
        float acc = 0.f;
        for (int e = lane; e < p.d / 2; e += 32) {
            const uint32_t a = o[e], b = g[e];
            acc += __uint_as_float(a << 16) * __uint_as_float(b << 16) +
                   __uint_as_float(a & 0xFFFF0000u) * __uint_as_float(b & 0xFFFF0000u);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            const long long t = r / p.Hq;
            const int h = static_cast<int>(r % p.Hq);
            p.dsum[static_cast<size_t>(h) * p.total_q + t] = acc;
        }
    }
}

// ---- dK, dV: one CTA per key block --------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + C::kTile;
    uint8_t* sQ = smem + 2 * C::kTile;   // two stages
    uint8_t* sDO = smem + 4 * C::kTile;  // two stages
    RowInfo* info = reinterpret_cast<RowInfo*>(smem + 6 * C::kTile);  // two stages
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + 6 * C::kTile + 2 * sizeof(RowInfo));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const BwdSeq sq = bwd_seq(p);
    if (!sq.ok) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int j = blockIdx.x;  // key block
    if (j * 128 >= sq.Lk) return;
    const int n_qt = (sq.Lq + p.tpt - 1) / p.tpt;
    // Does Q tile i see key block j?  (the forward pass's block range, per tile)
    auto sees = [&](int i) {
        const KvRange r = kv_block_range(i * p.tpt, min(i * p.tpt + p.tpt, sq.Lq) - 1, sq.Lq,
                                         sq.Lk, 128, p.causal, p.wl, p.wr);
        return r.lo <= j && j < r.hi;
    };

    // Rows of Q and dO past the packed tokens are never written by TMA but are part of the
    // contractions over query rows: clear both stages once.
    for (int u = threadIdx.x; u < 4 * C::kTile / 16; u += blockDim.x)
        st_shared_v4(smem_u32(sQ) + u * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->p_full, 8);
        mbar_init(&bars->mm_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    // TMEM: S^T / P^T [0, 128), dP^T / dS^T [128, 256), dV [256, 256 + D), dK [256 + D, ...)
    constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

    // Registers: launched at 168 per thread; warpgroup 2 (TMA, MMA, two idle warps) drops to
    // 80 and the elementwise warps rise to 208: 128 * 80 + 256 * 208 = 63488 <= 384 * 168.
    // (Each role sets its own count inside its branch.)
    if (warp == 8) {
        regs_decrease<80>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_do);
            mbar_arrive_expect_tx(&bars->kv_full[0], 2 * C::kTile);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(sK + h * C::kAtomBytes, &p.tm_k, &bars->kv_full[0], h * 64, sq.kvh,
                            sq.k0 + j * 128);
                tma_load_3d(sV + h * C::kAtomBytes, &p.tm_v, &bars->kv_full[0], h * 64, sq.kvh,
                            sq.k0 + j * 128);
            }
            const uint32_t box = 64u * p.g * p.tpt * 2u * C::kHalves;
            uint32_t n = 0;
            for (int i = 0; i < n_qt; ++i) {
                if (!sees(i)) continue;
                const int s = n & 1;
                if (n >= 2 && !wd.wait(&bars->q_empty[s], ((n >> 1) - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->q_full[s], 2 * box);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    tma_load_3d(sQ + s * C::kTile + h * C::kAtomBytes, &p.tm_q, &bars->q_full[s],
                                h * 64, sq.kvh * p.g, sq.q0 + i * p.tpt);
                    tma_load_3d(sDO + s * C::kTile + h * C::kAtomBytes, &p.tm_do,
                                &bars->q_full[s], h * 64, sq.kvh * p.g, sq.q0 + i * p.tpt);
                }
                ++n;
            }
            bwd_drain(&bars->kv_full[0], 0);
            for (uint32_t s = 0; s < 2 && s < n; ++s)
                bwd_drain(&bars->q_full[s], ((n - 1 - s) >> 1) & 1);
        }
    } else if (warp == 9) {
        regs_decrease<80>();
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);
            const uint64_t dk_ = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv_ = sdesc_sw128(smem_u32(sV), 16, 1024);
            uint32_t n = 0;
            if (wd.wait(&bars->kv_full[0], 0)) {
                for (int i = 0; i < n_qt; ++i) {
                    if (!sees(i)) continue;
                    const int s = n & 1;
                    if (!wd.wait(&bars->q_full[s], (n >> 1) & 1)) break;
                    // S^T and dP^T overwrite P^T and dS^T of the previous tile
                    if (n > 0 && !wd.wait(&bars->mm_done, (n - 1) & 1)) break;
                    tc_fence_after();
                    const uint32_t q_base = smem_u32(sQ + s * C::kTile);
                    const uint32_t do_base = smem_u32(sDO + s * C::kTile);
                    const uint64_t dq_ = sdesc_sw128(q_base, 16, 1024);
                    const uint64_t ddo = sdesc_sw128(do_base, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (((kk >> 2) * C::kAtomBytes + (kk & 3) * 32) >> 4);
                        umma_ss(tmem + kColS, dk_ + off, dq_ + off, kIdS, kk > 0);
                        umma_ss(tmem + kColDP, dv_ + off, ddo + off, kIdS, kk > 0);
                    }
                    umma_commit(&bars->s_full);
                    if (!wd.wait(&bars->p_full, n & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk) {
                        const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
                        umma_ts(tmem + kColDV, tmem + kColS + kk * 8,
                                sdesc_sw128(do_base + kk * 2048, C::kAtomBytes, 1024), kIdG, acc);
                        umma_ts(tmem + kColDK, tmem + kColDP + kk * 8,
                                sdesc_sw128(q_base + kk * 2048, C::kAtomBytes, 1024), kIdG, acc);
                    }
                    umma_commit(&bars->mm_done);
                    umma_commit(&bars->q_empty[s]);
                    ++n;
                }
            }
            umma_commit(&bars->drain);
            bwd_drain(&bars->drain, 0);
        }
    } else if (warp >= 10) {
        regs_decrease<80>();
    } else {
        regs_increase<208>();
        const int quarter = warp & 3, ch = warp >> 2;
        const int kr = 32 * quarter + lane;  // key row of the block
        const int key = j * 128 + kr;
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
        // Every compute warp passes both named barriers on every tile, even after a wait has
        // run out (ok == false skips the work), so no warp is left waiting at one.
        bool ok = true;
        uint32_t n = 0;
        for (int i = 0; i < n_qt; ++i) {
            if (!sees(i)) continue;
            const int s = n & 1;
            const int imin = i * p.tpt, imax = min(imin + p.tpt, sq.Lq) - 1;
            const bool masked = kv_block_masked(j, imin, imax, sq.Lq, sq.Lk, 128, p.causal, p.wl,
                                                p.wr);
            if (threadIdx.x < 128) fill_rows(p, sq, i, masked, info[s], threadIdx.x);
            named_bar_sync(1, 256);
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->s_full, n & 1));
            tc_fence_after();
            const RowInfo& ri = info[s];
            uint32_t pp[32], pd[32];
#pragma unroll
            for (int c2 = 0; c2 < 2 && ok; ++c2) {
                const int col0 = 64 * ch + 32 * c2;
                uint32_t sv[32], dv[32];
                tmem_ld32(tmem + lane_off + kColS + col0, sv);
                tmem_ld32(tmem + lane_off + kColDP + col0, dv);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float pe[2], de[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = col0 + e + u;
                        float x = fmaf(__uint_as_float(sv[e + u]), p.scale_log2, ri.nl[c]);
                        if (masked && (key < ri.kmin[c] || key > ri.kmax[c])) x = -INFINITY;
                        pe[u] = ex2_approx(x);
                        de[u] = pe[u] * (__uint_as_float(dv[e + u]) - ri.dd[c]);
                    }
                    pp[16 * c2 + e / 2] = pack_bf16x2(pe[0], pe[1]);
                    pd[16 * c2 + e / 2] = pack_bf16x2(de[0], de[1]);
                }
            }
            // every warp has read S^T and dP^T before any overwrites them with P^T and dS^T
            named_bar_sync(2, 256);
            if (ok) {
                tmem_st32(tmem + lane_off + kColS + 32 * ch, pp);
                tmem_st32(tmem + lane_off + kColDP + 32 * ch, pd);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full);
            }
            ++n;
        }
        // Epilogue: dV and scale * dK rows of this key block, bf16.
        if (n > 0) {
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->mm_done, (n - 1) & 1));
            tc_fence_after();
        }
        const bool valid = ok && key < sq.Lk;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t col = (which == 0 ? kColDV : kColDK) + (D / 2) * ch;
            const float mul = which == 0 ? 1.f : p.scale;
            __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) +
                                 (static_cast<size_t>(sq.k0 + key) * p.Hkv + sq.kvh) * D + (D / 2) * ch;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t o[32];
                if (n > 0 && ok) {
                    tmem_ld32(tmem + lane_off + col + 32 * c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        d4[v] = make_uint4(
                            pack_bf16x2(__uint_as_float(o[8 * v + 0]) * mul, __uint_as_float(o[8 * v + 1]) * mul),
                            pack_bf16x2(__uint_as_float(o[8 * v + 2]) * mul, __uint_as_float(o[8 * v + 3]) * mul),
                            pack_bf16x2(__uint_as_float(o[8 * v + 4]) * mul, __uint_as_float(o[8 * v + 5]) * mul),
                            pack_bf16x2(__uint_as_float(o[8 * v + 6]) * mul, __uint_as_float(o[8 * v + 7]) * mul));
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- dQ: one CTA per Q tile ---------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sDO = smem + C::kTile;
    uint8_t* sK = smem + 2 * C::kTile;  // two stages
    uint8_t* sV = smem + 4 * C::kTile;  // two stages
    RowInfo* info = reinterpret_cast<RowInfo*>(smem + 6 * C::kTile);
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + 6 * C::kTile + 2 * sizeof(RowInfo));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const BwdSeq sq = bwd_seq(p);
    if (!sq.ok) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int i = blockIdx.x;  // Q tile
    if (i * p.tpt >= sq.Lq) return;
    const int imin = i * p.tpt, imax = min(imin + p.tpt, sq.Lq) - 1;
    const KvRange kr_ = kv_block_range(imin, imax, sq.Lq, sq.Lk, 128, p.causal, p.wl, p.wr);
    const int lo = kr_.lo, hi = kr_.hi;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->q_full[0], 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->p_full, 8);
        mbar_init(&bars->mm_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    // TMEM: S / dS [0, 128), dP [128, 256), dQ [256, 256 + D)
    constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

    if (warp == 8) {
        if (lane == 0 && hi > lo) {
            const uint32_t box = 64u * p.g * p.tpt * 2u * C::kHalves;
            mbar_arrive_expect_tx(&bars->q_full[0], 2 * box);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(sQ + h * C::kAtomBytes, &p.tm_q, &bars->q_full[0], h * 64,
                            sq.kvh * p.g, sq.q0 + imin);
                tma_load_3d(sDO + h * C::kAtomBytes, &p.tm_do, &bars->q_full[0], h * 64,
                            sq.kvh * p.g, sq.q0 + imin);
            }
            uint32_t n = 0;
            for (int j = lo; j < hi; ++j, ++n) {
                const int s = n & 1;
                if (n >= 2 && !wd.wait(&bars->kv_empty[s], ((n >> 1) - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->kv_full[s], 2 * C::kTile);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    tma_load_3d(sK + s * C::kTile + h * C::kAtomBytes, &p.tm_k, &bars->kv_full[s],
                                h * 64, sq.kvh, sq.k0 + j * 128);
                    tma_load_3d(sV + s * C::kTile + h * C::kAtomBytes, &p.tm_v, &bars->kv_full[s],
                                h * 64, sq.kvh, sq.k0 + j * 128);
                }
            }
            bwd_drain(&bars->q_full[0], 0);
            for (uint32_t s = 0; s < 2 && s < n; ++s)
                bwd_drain(&bars->kv_full[s], ((n - 1 - s) >> 1) & 1);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);
            const uint64_t dq_ = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t ddo = sdesc_sw128(smem_u32(sDO), 16, 1024);
            uint32_t n = 0;
            if (hi > lo && wd.wait(&bars->q_full[0], 0)) {
                for (int j = lo; j < hi; ++j, ++n) {
                    const int s = n & 1;
                    if (!wd.wait(&bars->kv_full[s], (n >> 1) & 1)) break;
                    // S and dP overwrite dS of the previous block, which dQ read
                    if (n > 0 && !wd.wait(&bars->mm_done, (n - 1) & 1)) break;
                    tc_fence_after();
                    const uint32_t k_base = smem_u32(sK + s * C::kTile);
                    const uint64_t dk_ = sdesc_sw128(k_base, 16, 1024);
                    const uint64_t dv_ = sdesc_sw128(smem_u32(sV + s * C::kTile), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (((kk >> 2) * C::kAtomBytes + (kk & 3) * 32) >> 4);
                        umma_ss(tmem + kColS, dq_ + off, dk_ + off, kIdS, kk > 0);
                        umma_ss(tmem + kColDP, ddo + off, dv_ + off, kIdS, kk > 0);
                    }
                    umma_commit(&bars->s_full);
                    if (!wd.wait(&bars->p_full, n & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk)
                        umma_ts(tmem + kColDQ, tmem + kColS + kk * 8,
                                sdesc_sw128(k_base + kk * 2048, C::kAtomBytes, 1024), kIdG,
                                (n > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&bars->mm_done);
                    umma_commit(&bars->kv_empty[s]);
                }
            }
            umma_commit(&bars->drain);
            bwd_drain(&bars->drain, 0);
        }
    } else if (warp < 8) {
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = 32 * quarter + lane;  // packed row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
        if (threadIdx.x < 128) fill_rows(p, sq, i, true, info[0], threadIdx.x);
        named_bar_sync(1, 256);
        const float nl = info[0].nl[r], dd = info[0].dd[r];
        const int kmin = info[0].kmin[r], kmax = info[0].kmax[r];
        const bool row_valid = nl != -INFINITY;
        bool ok = true;  // as in the dK/dV kernel: the named barrier is passed on every block
        uint32_t n = 0;
        for (int j = lo; j < hi; ++j, ++n) {
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->s_full, n & 1));
            tc_fence_after();
            const bool masked = kv_block_masked(j, imin, imax, sq.Lq, sq.Lk, 128, p.causal, p.wl,
                                                p.wr);
            uint32_t pd[32];
#pragma unroll
            for (int c2 = 0; c2 < 2 && ok; ++c2) {
                const int col0 = 64 * ch + 32 * c2;
                uint32_t sv[32], dv[32];
                tmem_ld32(tmem + lane_off + kColS + col0, sv);
                tmem_ld32(tmem + lane_off + kColDP + col0, dv);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float de[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int key = j * 128 + col0 + e + u;
                        float x = fmaf(__uint_as_float(sv[e + u]), p.scale_log2, nl);
                        if (masked && (key < kmin || key > kmax)) x = -INFINITY;
                        const float pe = ex2_approx(x);
                        de[u] = row_valid ? pe * (__uint_as_float(dv[e + u]) - dd) : 0.f;
                    }
                    pd[16 * c2 + e / 2] = pack_bf16x2(de[0], de[1]);
                }
            }
            named_bar_sync(2, 256);
            if (ok) {
                tmem_st32(tmem + lane_off + kColS + 32 * ch, pd);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full);
            }
        }
        // Epilogue: scale * dQ rows of this tile, bf16.
        if (n > 0) {
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->mm_done, (n - 1) & 1));
            tc_fence_after();
        }
        const int tok = imin + r / p.g;
        const bool valid = ok && r < p.g * p.tpt && tok < sq.Lq;
        __nv_bfloat16* dst = p.dq + (static_cast<size_t>(sq.q0 + tok) * p.Hq + sq.kvh * p.g + r % p.g) * D +
                             (D / 2) * ch;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            if (n > 0 && ok) {
                tmem_ld32(tmem + lane_off + kColDQ + (D / 2) * ch + 32 * c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (valid) {
                uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    d4[v] = make_uint4(
                        pack_bf16x2(__uint_as_float(o[8 * v + 0]) * p.scale, __uint_as_float(o[8 * v + 1]) * p.scale),
                        pack_bf16x2(__uint_as_float(o[8 * v + 2]) * p.scale, __uint_as_float(o[8 * v + 3]) * p.scale),
                        pack_bf16x2(__uint_as_float(o[8 * v + 4]) * p.scale, __uint_as_float(o[8 * v + 5]) * p.scale),
                        pack_bf16x2(__uint_as_float(o[8 * v + 6]) * p.scale, __uint_as_float(o[8 * v + 7]) * p.scale));
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
constexpr int bwd_smem() {
    return 6 * BwdCfg<D>::kTile + 2 * static_cast<int>(sizeof(RowInfo)) + 256 + 1024;
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t stream) {
    {
        const long long rows = static_cast<long long>(p.total_q) * p.Hq;
        long long blocks = (rows + 7) / 8;
        if (blocks > static_cast<long long>(num_sms) * 16) blocks = static_cast<long long>(num_sms) * 16;
        if (blocks > 0) bwd_preprocess_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    }
    const dim3 grid_kv((p.max_seqlen_k + 127) / 128, p.batch * p.Hkv);
    const dim3 grid_q((p.max_seqlen_q + p.tpt - 1) / p.tpt, p.batch * p.Hkv);
    if (p.d == 128) {
        constexpr int sm = bwd_smem<128>();
        cudaFuncSetAttribute(bwd_dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        cudaFuncSetAttribute(bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        if (grid_kv.x > 0) bwd_dkdv_kernel<128><<<grid_kv, kBwdThreads, sm, stream>>>(p);
        if (grid_q.x > 0) bwd_dq_kernel<128><<<grid_q, kBwdThreads, sm, stream>>>(p);
    } else {
        constexpr int sm = bwd_smem<64>();
        cudaFuncSetAttribute(bwd_dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        cudaFuncSetAttribute(bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        if (grid_kv.x > 0) bwd_dkdv_kernel<64><<<grid_kv, kBwdThreads, sm, stream>>>(p);
        if (grid_q.x > 0) bwd_dq_kernel<64><<<grid_q, kBwdThreads, sm, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace attn
