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
//   * bwd_dkdv_kernel: one CTA per 128-key block of one (sequence, kv head), walking the
//     128-row Q tiles (tokens x query heads, packed as in the forward pass) that see it;
//   * bwd_dq_kernel: one CTA per 128-row Q tile, walking the 128-key blocks it sees.
//   Every MMA is 128 x 128 (x D) so the tensor pipe runs at its full rate.  The elementwise
//   warps (0-7, two per TMEM lane quarter) pull S and dP of a block into registers, which
//   frees that TMEM for the next MMA while they work; the gradient operand goes back to TMEM
//   as packed bf16 (over S^T and dP^T in the dK/dV kernel, into two spare slots in the dQ
//   kernel) for MMAs that take their A operand from TMEM.  Two warps issue MMAs, one per
//   stream (9: S and dP; 11: the gradients), so neither stream waits behind the other; warp 8
//   streams operands by TMA, and in the dK/dV kernel warp 10 stages the query rows' L, D and
//   key intervals a tile ahead.
#include <cuda_bf16.h>

#include <cstddef>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_math.h"

namespace attn {

namespace {

constexpr float kLog2e = 1.44269504088896341f;
constexpr int kBwdThreads = 384;
constexpr int kStages = 2;  // streamed operand ring (and row information ring)
constexpr int kKStages = 3; // K ring of the dQ kernel

template <int D>
struct BwdCfg {
    static constexpr int kHalves = D / 64;      // 128-byte swizzle atoms across d
    static constexpr int kAtom = 128 * 128;     // one atom of 128 rows x 128 bytes
    static constexpr int kTile = kHalves * kAtom;
};

struct BwdBars {
    uint64_t fixed_full;                               // loaded once (dK/dV: K, V; dQ: Q, dO)
    uint64_t in_full[kKStages], in_empty[kKStages];    // streamed operands (dK/dV: Q, dO; dQ: K)
    uint64_t v_full[kStages], v_empty[kStages];        // dQ: V
    uint64_t info_full[kStages], info_empty[kStages];  // row information (dK/dV)
    uint64_t s_full, s_free;                           // dQ: S / dP in TMEM, loaded to registers
    uint64_t p_full[2], p_empty[2];                    // dQ: dS slots in TMEM
    uint64_t sa_full, sb_full, pa_full, pb_full;       // dK/dV: S^T, dP^T in; P^T, dS^T out
    uint64_t dv_done, dk_done;                         // dK/dV: gradient MMAs have read P^T / dS^T
    uint64_t mm_done, drain[2];
    uint32_t tmem_base;
    int abort_flag;
};

__device__ void init_bars(BwdBars* b) {
    mbar_init(&b->fixed_full, 1);
    for (int s = 0; s < kKStages; ++s) {
        mbar_init(&b->in_full[s], 1);
        mbar_init(&b->in_empty[s], 1);
    }
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&b->v_full[s], 1);
        mbar_init(&b->v_empty[s], 1);
        mbar_init(&b->info_full[s], 32);
        mbar_init(&b->info_empty[s], 8);
    }
    mbar_init(&b->s_full, 1);
    mbar_init(&b->s_free, 8);
    mbar_init(&b->p_full[0], 8);
    mbar_init(&b->p_full[1], 8);
    mbar_init(&b->p_empty[0], 1);
    mbar_init(&b->p_empty[1], 1);
    mbar_init(&b->sa_full, 1);
    mbar_init(&b->sb_full, 1);
    mbar_init(&b->pa_full, 8);
    mbar_init(&b->pb_full, 8);
    mbar_init(&b->dv_done, 1);
    mbar_init(&b->dk_done, 1);
    mbar_init(&b->mm_done, 1);
    mbar_init(&b->drain[0], 1);
    mbar_init(&b->drain[1], 1);
    b->abort_flag = 0;
}

// Per packed row of a 128-row Q tile: -L * log2(e) (or -inf when the row has no gradient),
// D, and the row's visible key interval.
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

// 32 fp32 accumulator columns times mul, as bf16, to 64 contiguous bytes of global memory.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&o)[32], float mul) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < 4; ++v)
        d4[v] = make_uint4(
            pack_bf16x2(__uint_as_float(o[8 * v + 0]) * mul, __uint_as_float(o[8 * v + 1]) * mul),
            pack_bf16x2(__uint_as_float(o[8 * v + 2]) * mul, __uint_as_float(o[8 * v + 3]) * mul),
            pack_bf16x2(__uint_as_float(o[8 * v + 4]) * mul, __uint_as_float(o[8 * v + 5]) * mul),
            pack_bf16x2(__uint_as_float(o[8 * v + 6]) * mul, __uint_as_float(o[8 * v + 7]) * mul));
}

// P = exp2(s * scale_log2 + nl) and dS = P (dp - dd) for two elements, with the paired fp32
// instructions (two lanes of work per issue); a masked element gets P = 0.
__device__ __forceinline__ void p_ds_pair(uint32_t s0, uint32_t s1, uint32_t dp0, uint32_t dp1,
                                          uint64_t scale2, uint64_t nl2, uint64_t ndd2, bool m0,
                                          bool m1, uint32_t& p_out, uint32_t& ds_out) {
    float x0, x1;
    f2_split(f2_fma(f2_make(__uint_as_float(s0), __uint_as_float(s1)), scale2, nl2), x0, x1);
    const float p0 = ex2_approx(m0 ? -INFINITY : x0);
    const float p1 = ex2_approx(m1 ? -INFINITY : x1);
    const uint64_t pv = f2_make(p0, p1);
    float d0, d1;
    f2_split(f2_mul(pv, f2_add(f2_make(__uint_as_float(dp0), __uint_as_float(dp1)), ndd2)), d0, d1);
    p_out = pack_bf16x2(p0, p1);
    ds_out = pack_bf16x2(d0, d1);
}

// dS = exp2(s * scale_log2 + nl) (dp - dd) for two unmasked elements, packed as bf16.
__device__ __forceinline__ uint32_t ds_pair(uint32_t s0, uint32_t s1, uint32_t dp0, uint32_t dp1,
                                            uint64_t scale2, uint64_t nl2, uint64_t ndd2) {
    float x0, x1;
    f2_split(f2_fma(f2_make(__uint_as_float(s0), __uint_as_float(s1)), scale2, nl2), x0, x1);
    const uint64_t pv = f2_make(ex2_approx(x0), ex2_approx(x1));
    float d0, d1;
    f2_split(f2_mul(pv, f2_add(f2_make(__uint_as_float(dp0), __uint_as_float(dp1)), ndd2)), d0, d1);
    return pack_bf16x2(d0, d1);
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
//
// The CTA walks the 128-row Q tiles that see key block j.  TMEM: region F = [0, 128) holds
// S^T and then packed P^T, region G = [128, 256) holds dP^T and then packed dS^T, dV is at
// [256, 256 + D) and dK at [256 + D, 256 + 2 D).  Tile n:
//   warps 0-7:   phase A: their 64 columns of S^T to registers, P^T = exp2(S^T scale log2(e) -
//                L log2(e)) kept in fp32, packed bf16 P^T over their own S^T columns;
//                phase B: per 32-column chunk of dP^T, dS^T = P^T (dP^T - D), packed bf16 over
//                the chunk's own dP^T columns;
//   warp 9:      S^T(n) = K Q(n)^T into F once dV(n-1) has read P^T(n-1), then dP^T(n) =
//                V dO(n)^T into G once dK(n-1) has read dS^T(n-1);
//   warp 11:     dV += P^T(n) dO(n) after phase A and dK += dS^T(n) Q(n) after phase B, with
//                A from TMEM;
//   warp 10:     the rows' -L log2(e), D and key intervals, a tile ahead;
//   warp 8:      TMA of K, V (once) and of Q, dO tiles (two stages).
// So the tensor pipe runs S^T, dP^T, dV, dK of one tile back to back while the elementwise
// warps work phase by phase.

template <int D>
struct DkdvSmem {
    using C = BwdCfg<D>;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = C::kTile;
    static constexpr int kOffQ = 2 * C::kTile;                 // kStages stages
    static constexpr int kOffDO = kOffQ + kStages * C::kTile;   // kStages stages
    static constexpr int kOffInfo = kOffDO + kStages * C::kTile;
    static constexpr int kOffBars = kOffInfo + kStages * static_cast<int>(sizeof(RowInfo));
    static constexpr int kBytes = kOffBars + static_cast<int>(sizeof(BwdBars)) + 1024;
};
static_assert(DkdvSmem<128>::kBytes <= 227 * 1024, "dK/dV shared memory");

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    using L = DkdvSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem + L::kOffK;
    uint8_t* sV = smem + L::kOffV;
    uint8_t* sQ = smem + L::kOffQ;
    uint8_t* sDO = smem + L::kOffDO;
    RowInfo* info = reinterpret_cast<RowInfo*>(smem + L::kOffInfo);
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kOffBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const BwdSeq sq = bwd_seq(p);
    if (!sq.ok) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int j = blockIdx.x;  // key block
    if (j * 128 >= sq.Lk) return;
    const int n_qt = (sq.Lq + p.tpt - 1) / p.tpt;
    // (the lambdas take copies: a reference to the parameter block would turn each use into a
    // load through a generic pointer)
    const int tpt = p.tpt, causal = p.causal, wl = p.wl, wr = p.wr, Lq = sq.Lq, Lk = sq.Lk;
    auto tok_hi = [=](int i) { return min(i * tpt + tpt, Lq) - 1; };
    // Does Q tile i see key block j?  (the forward pass's block range, per tile)
    auto sees = [=](int i) {
        const KvRange r = kv_block_range(i * tpt, min(i * tpt + tpt, Lq) - 1, Lq, Lk, 128, causal,
                                         wl, wr);
        return r.lo <= j && j < r.hi;
    };

    // Rows of Q and dO past the packed tokens are never written by TMA but are part of the
    // contractions over query rows: clear both stages once.
    for (int u = threadIdx.x; u < 2 * kStages * C::kTile / 16; u += blockDim.x)
        st_shared_v4(smem_u32(sQ) + u * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        init_bars(bars);
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    constexpr uint32_t kColF = 0, kColG = 128, kColDV = 256, kColDK = 256 + D;
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);

    // Registers: launched at 168 per thread; warps 8-11 drop to 80 and the elementwise warps
    // rise to 208: 128 * 80 + 256 * 208 = 63488 <= 384 * 168.  (Each role sets its own count.)
    if (warp == 8) {
        regs_decrease<80>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_do);
            mbar_arrive_expect_tx(&bars->fixed_full, 2 * C::kTile);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(sK + h * C::kAtom, &p.tm_k, &bars->fixed_full, h * 64, sq.kvh,
                            sq.k0 + j * 128);
                tma_load_3d(sV + h * C::kAtom, &p.tm_v, &bars->fixed_full, h * 64, sq.kvh,
                            sq.k0 + j * 128);
            }
            const uint32_t box = 128u * p.g * p.tpt * C::kHalves;  // bytes of one operand
            int n = 0;
            for (int i = 0; i < n_qt; ++i) {
                if (!sees(i)) continue;
                const int st = n & 1;
                if (n >= 2 && !wd.wait(&bars->in_empty[st], ((n >> 1) - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->in_full[st], 2 * box);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    tma_load_3d(sQ + st * C::kTile + h * C::kAtom, &p.tm_q, &bars->in_full[st],
                                h * 64, sq.kvh * p.g, sq.q0 + i * p.tpt);
                    tma_load_3d(sDO + st * C::kTile + h * C::kAtom, &p.tm_do, &bars->in_full[st],
                                h * 64, sq.kvh * p.g, sq.q0 + i * p.tpt);
                }
                ++n;
            }
            bwd_drain(&bars->fixed_full, 0);
            for (int m = n > 2 ? n - 2 : 0; m < n; ++m) bwd_drain(&bars->in_full[m & 1], (m >> 1) & 1);
        }
    } else if (warp == 9) {
        regs_decrease<80>();
        if (lane == 0) {
            // X^T = A B^T over d into TMEM column col, B a Q / dO stage
            auto s_mma = [&](uint32_t col, const uint8_t* a, const uint8_t* b) {
                const uint64_t ad = sdesc_sw128(smem_u32(a), 16, 1024);
                const uint64_t bd = sdesc_sw128(smem_u32(b), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (((kk >> 2) * C::kAtom + (kk & 3) * 32) >> 4);
                    umma_ss(tmem + col, ad + off, bd + off, kIdS, kk > 0);
                }
            };
            int n = 0;
            bool ok = wd.wait(&bars->fixed_full, 0);
            for (int i = 0; ok && i < n_qt; ++i) {
                if (!sees(i)) continue;
                const int st = n & 1;
                // S^T(n) into F once dV(n-1) has read P^T(n-1)
                ok = wd.wait(&bars->in_full[st], (n >> 1) & 1) &&
                     (n == 0 || wd.wait(&bars->dv_done, (n - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                s_mma(kColF, sK, sQ + st * C::kTile);
                umma_commit(&bars->sa_full);
                // dP^T(n) into G once dK(n-1) has read dS^T(n-1)
                ok = n == 0 || wd.wait(&bars->dk_done, (n - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                s_mma(kColG, sV, sDO + st * C::kTile);
                umma_commit(&bars->sb_full);
                ++n;
            }
            umma_commit(&bars->drain[0]);
            bwd_drain(&bars->drain[0], 0);
        }
    } else if (warp == 11) {
        regs_decrease<80>();
        if (lane == 0) {
            int n = 0;
            bool ok = true;
            for (int i = 0; ok && i < n_qt; ++i) {
                if (!sees(i)) continue;
                const int st = n & 1;
                const uint32_t q_base = smem_u32(sQ + st * C::kTile);
                const uint32_t do_base = smem_u32(sDO + st * C::kTile);
                // dV += P^T dO: K-step kk (query rows 16 kk ..) packed at F + 64 (kk / 4) +
                // 8 (kk % 4)
                ok = wd.wait(&bars->pa_full, n & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColDV, tmem + kColF + 64 * (kk >> 2) + 8 * (kk & 3),
                            sdesc_sw128(do_base + kk * 2048, C::kAtom, 1024), kIdG,
                            (n > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bars->dv_done);
                // dK += dS^T Q: K-step kk packed at G + 32 (kk / 2) + 8 (kk % 2)
                ok = wd.wait(&bars->pb_full, n & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColDK, tmem + kColG + 32 * (kk >> 1) + 8 * (kk & 1),
                            sdesc_sw128(q_base + kk * 2048, C::kAtom, 1024), kIdG,
                            (n > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bars->dk_done);
                umma_commit(&bars->in_empty[st]);
                ++n;
            }
            umma_commit(&bars->mm_done);
            umma_commit(&bars->drain[1]);
            bwd_drain(&bars->drain[1], 0);
        }
    } else if (warp == 10) {
        regs_decrease<80>();
        // Row information of each tile: lane l fills packed rows l, l + 32, l + 64, l + 96.
        int n = 0;
        for (int i = 0; i < n_qt; ++i) {
            if (!sees(i)) continue;
            const int st = n & 1;
            if (n >= 2 && !wd.wait(&bars->info_empty[st], ((n >> 1) - 1) & 1)) break;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int r = lane + 32 * h;
                const int tok = i * p.tpt + r / p.g;
                float nl = -INFINITY, dd = 0.f;
                int kmin = 1, kmax = 0;
                if (r < p.g * p.tpt && tok < sq.Lq) {
                    const size_t at =
                        static_cast<size_t>(sq.kvh * p.g + r % p.g) * p.total_q + sq.q0 + tok;
                    const float l = p.lse[at];
                    if (l != -INFINITY) nl = -l * kLog2e;
                    dd = p.dsum[at];
                    row_key_interval(tok, sq.Lq, sq.Lk, p.causal, p.wl, p.wr, kmin, kmax);
                }
                info[st].nl[r] = nl;
                info[st].dd[r] = -dd;
                info[st].kmin[r] = kmin;
                info[st].kmax[r] = kmax;
            }
            mbar_arrive(&bars->info_full[st]);
            ++n;
        }
    } else {
        regs_increase<208>();
        const int quarter = warp & 3, ch = warp >> 2;
        const int kr = 32 * quarter + lane;  // key row of the block
        const int key = j * 128 + kr;
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
        const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
        bool ok = true;
        int n = 0;
        for (int i = 0; i < n_qt; ++i) {
            if (!sees(i)) continue;
            const int st = n & 1;
            const bool masked = kv_block_masked(j, i * p.tpt, tok_hi(i), sq.Lq, sq.Lk, 128,
                                                p.causal, p.wl, p.wr);
            // this warp's 64 query rows (columns) of the row information
            const uint32_t ib = smem_u32(&info[st]) + 4 * 64 * ch;
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->info_full[st], (n >> 1) & 1));
            // phase A: P^T from S^T
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->sa_full, n & 1));
            tc_fence_after();
            uint32_t pv[64];  // S^T, then P^T in fp32
            if (ok) {
                tmem_ld32(tmem + lane_off + kColF + 64 * ch, *reinterpret_cast<uint32_t(*)[32]>(pv));
                tmem_ld32(tmem + lane_off + kColF + 64 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(pv + 32));
                tmem_wait_ld();
                if (!masked) {
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) {
                        const uint4 nl4 = ld_shared_v4(ib + offsetof(RowInfo, nl) + 16 * e4);
                        const int e = 4 * e4;
                        float x0, x1, x2, x3;
                        f2_split(f2_fma(f2_make(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), scale2,
                                        f2_make(__uint_as_float(nl4.x), __uint_as_float(nl4.y))), x0, x1);
                        f2_split(f2_fma(f2_make(__uint_as_float(pv[e + 2]), __uint_as_float(pv[e + 3])), scale2,
                                        f2_make(__uint_as_float(nl4.z), __uint_as_float(nl4.w))), x2, x3);
                        pv[e] = __float_as_uint(ex2_approx(x0));
                        pv[e + 1] = __float_as_uint(ex2_approx(x1));
                        pv[e + 2] = __float_as_uint(ex2_approx(x2));
                        pv[e + 3] = __float_as_uint(ex2_approx(x3));
                    }
                } else {
#pragma unroll
                    for (int e4 = 0; e4 < 16; ++e4) {
                        const uint4 nl4 = ld_shared_v4(ib + offsetof(RowInfo, nl) + 16 * e4);
                        const uint4 lo4 = ld_shared_v4(ib + offsetof(RowInfo, kmin) + 16 * e4);
                        const uint4 hi4 = ld_shared_v4(ib + offsetof(RowInfo, kmax) + 16 * e4);
                        const uint32_t nlv[4] = {nl4.x, nl4.y, nl4.z, nl4.w};
                        const uint32_t lov[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
                        const uint32_t hiv[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int e = 4 * e4 + u;
                            const bool vis = key >= static_cast<int>(lov[u]) && key <= static_cast<int>(hiv[u]);
                            const float x = fmaf(__uint_as_float(pv[e]), p.scale_log2, __uint_as_float(nlv[u]));
                            pv[e] = __float_as_uint(ex2_approx(vis ? x : -INFINITY));
                        }
                    }
                }
                // packed query columns 64 ch + 2 c, 2 c + 1 at F + 64 ch + c: own columns
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pp[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        pp[c] = pack_bf16x2(__uint_as_float(pv[32 * h + 2 * c]),
                                            __uint_as_float(pv[32 * h + 2 * c + 1]));
                    tmem_st16(tmem + lane_off + kColF + 64 * ch + 16 * h, pp);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->pa_full);
            // phase B: dS^T from dP^T
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->sb_full, n & 1));
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const uint32_t col = kColG + 64 * ch + 32 * c2;
                    uint32_t dv[32], pd[16];
                    tmem_ld32(tmem + lane_off + col, dv);
                    tmem_wait_ld();
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const uint4 dd4 = ld_shared_v4(ib + offsetof(RowInfo, dd) + 4 * 32 * c2 + 16 * e4);
                        const int e = 32 * c2 + 4 * e4;
                        float d[4];
                        f2_split(f2_mul(f2_make(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])),
                                        f2_add(f2_make(__uint_as_float(dv[4 * e4]), __uint_as_float(dv[4 * e4 + 1])),
                                               f2_make(__uint_as_float(dd4.x), __uint_as_float(dd4.y)))),
                                 d[0], d[1]);
                        f2_split(f2_mul(f2_make(__uint_as_float(pv[e + 2]), __uint_as_float(pv[e + 3])),
                                        f2_add(f2_make(__uint_as_float(dv[4 * e4 + 2]), __uint_as_float(dv[4 * e4 + 3])),
                                               f2_make(__uint_as_float(dd4.z), __uint_as_float(dd4.w)))),
                                 d[2], d[3]);
                        pd[2 * e4] = pack_bf16x2(d[0], d[1]);
                        pd[2 * e4 + 1] = pack_bf16x2(d[2], d[3]);
                    }
                    // packed into the first 16 of the chunk's own 32 dP^T columns
                    tmem_st16(tmem + lane_off + col, pd);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars->pb_full);
                mbar_arrive(&bars->info_empty[st]);
            }
            ++n;
        }
        // Epilogue: dV and scale * dK rows of this key block, bf16.
        if (n > 0) {
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->mm_done, 0));
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
                if (valid) store_row32(dst + 32 * c, o, mul);
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
//
// The CTA walks the 128-key blocks its 128 packed query rows see.  TMEM: S at [0, 128), dP at
// [128, 256), dQ at [256, 256 + D), two slots of packed bf16 dS at [384, 448) and [448, 512).
// Block n:
//   warps 0-7:  load their 64 columns of S(n) and dP(n) to registers (both regions are free
//               again), form dS = P (dP - D) and write it packed to slot n % 2;
//   warp 9:     S(n+1) = Q K(n+1)^T and dP(n+1) = dO V(n+1)^T as soon as S(n), dP(n) are in
//               registers;
//   warp 11:    dQ += dS(n) K(n) with dS from TMEM;
//   warp 8:     TMA of Q, dO (once), of K blocks into a three-stage ring (a K block is read
//               until its dQ step) and of V blocks into a two-stage ring (read by dP only).

template <int D>
struct DqSmem {
    using C = BwdCfg<D>;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = C::kTile;
    static constexpr int kOffK = 2 * C::kTile;                // kKStages stages
    static constexpr int kOffV = kOffK + kKStages * C::kTile;  // kStages stages
    static constexpr int kOffBars = kOffV + kStages * C::kTile;
    static constexpr int kBytes = kOffBars + static_cast<int>(sizeof(BwdBars)) + 1024;
};
static_assert(DqSmem<128>::kBytes <= 227 * 1024, "dQ shared memory");

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    using L = DqSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + L::kOffQ;
    uint8_t* sDO = smem + L::kOffDO;
    uint8_t* sK = smem + L::kOffK;
    uint8_t* sV = smem + L::kOffV;
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kOffBars);
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

    // Rows of Q and dO past the packed tokens are never written by TMA: clear them once so
    // that their S, dP and dS rows are zero.
    for (int u = threadIdx.x; u < 2 * C::kTile / 16; u += blockDim.x)
        st_shared_v4(smem_u32(sQ) + u * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        init_bars(bars);
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;

    if (warp == 8) {
        regs_decrease<80>();
        if (lane == 0 && hi > lo) {
            const uint32_t box = 128u * p.g * p.tpt * C::kHalves;  // bytes of one operand
            mbar_arrive_expect_tx(&bars->fixed_full, 2 * box);
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(sQ + h * C::kAtom, &p.tm_q, &bars->fixed_full, h * 64, sq.kvh * p.g,
                            sq.q0 + imin);
                tma_load_3d(sDO + h * C::kAtom, &p.tm_do, &bars->fixed_full, h * 64,
                            sq.kvh * p.g, sq.q0 + imin);
            }
            int nk = 0, nv = 0;  // K, V blocks loaded
            for (int j = lo; j < hi; ++j) {
                const int sk = nk % kKStages, sv = nv & 1;
                if (nk >= kKStages && !wd.wait(&bars->in_empty[sk], ((nk / kKStages) - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->in_full[sk], C::kTile);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(sK + sk * C::kTile + h * C::kAtom, &p.tm_k, &bars->in_full[sk],
                                h * 64, sq.kvh, sq.k0 + j * 128);
                ++nk;
                if (nv >= 2 && !wd.wait(&bars->v_empty[sv], ((nv >> 1) - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->v_full[sv], C::kTile);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(sV + sv * C::kTile + h * C::kAtom, &p.tm_v, &bars->v_full[sv],
                                h * 64, sq.kvh, sq.k0 + j * 128);
                ++nv;
            }
            bwd_drain(&bars->fixed_full, 0);
            for (int m = nk > kKStages ? nk - kKStages : 0; m < nk; ++m)
                bwd_drain(&bars->in_full[m % kKStages], (m / kKStages) & 1);
            for (int m = nv > 2 ? nv - 2 : 0; m < nv; ++m) bwd_drain(&bars->v_full[m & 1], (m >> 1) & 1);
        }
    } else if (warp == 9) {
        regs_decrease<80>();
        if (lane == 0) {
            // S(n) = Q K(n)^T, dP(n) = dO V(n)^T once S(n-1), dP(n-1) are in registers
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
            const uint64_t dq_ = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t ddo = sdesc_sw128(smem_u32(sDO), 16, 1024);
            int n = 0;
            bool ok = hi > lo && wd.wait(&bars->fixed_full, 0);
            for (int j = lo; ok && j < hi; ++j, ++n) {
                const int sk = n % kKStages, sv = n & 1;
                ok = wd.wait(&bars->in_full[sk], (n / kKStages) & 1) &&
                     wd.wait(&bars->v_full[sv], (n >> 1) & 1) &&
                     (n == 0 || wd.wait(&bars->s_free, (n - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint64_t dk_ = sdesc_sw128(smem_u32(sK + sk * C::kTile), 16, 1024);
                const uint64_t dv_ = sdesc_sw128(smem_u32(sV + sv * C::kTile), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (((kk >> 2) * C::kAtom + (kk & 3) * 32) >> 4);
                    umma_ss(tmem + kColS, dq_ + off, dk_ + off, kIdS, kk > 0);
                    umma_ss(tmem + kColDP, ddo + off, dv_ + off, kIdS, kk > 0);
                }
                umma_commit(&bars->s_full);
                umma_commit(&bars->v_empty[sv]);
            }
            umma_commit(&bars->drain[0]);
            bwd_drain(&bars->drain[0], 0);
        }
    } else if (warp == 11) {
        regs_decrease<80>();
        if (lane == 0) {
            // dQ += dS(n) K(n) (K in stage n % 3), dS from TMEM slot n % 2: K-steps of 16
            // keys, keys 64 c .. 64 c + 63 packed at slot + 32 c
            constexpr uint32_t kIdG = idesc_bf16_f32(128, D, false, true);
            int n = 0;
            bool ok = true;
            for (int j = lo; ok && j < hi; ++j, ++n) {
                const int sk = n % kKStages;
                ok = wd.wait(&bars->p_full[n & 1], (n >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sK + sk * C::kTile);
                const uint32_t slot = kColDS + 64 * (n & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tmem + kColDQ, tmem + slot + 32 * (kk >> 2) + 8 * (kk & 3),
                            sdesc_sw128(k_base + kk * 2048, C::kAtom, 1024), kIdG,
                            (n > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bars->p_empty[n & 1]);
                umma_commit(&bars->in_empty[sk]);
            }
            umma_commit(&bars->mm_done);
            umma_commit(&bars->drain[1]);
            bwd_drain(&bars->drain[1], 0);
        }
    } else if (warp == 10) {
        regs_decrease<80>();
    } else {
        regs_increase<208>();
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = 32 * quarter + lane;  // packed row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
        const int tok = imin + r / p.g;
        const bool in_tile = r < p.g * p.tpt && tok < sq.Lq;
        float nl = -INFINITY, dd = 0.f;
        int kmin = 1, kmax = 0;
        if (in_tile) {
            const size_t at = static_cast<size_t>(sq.kvh * p.g + r % p.g) * p.total_q + sq.q0 + tok;
            const float l = p.lse[at];
            if (l != -INFINITY) nl = -l * kLog2e;
            dd = p.dsum[at];
            row_key_interval(tok, sq.Lq, sq.Lk, p.causal, p.wl, p.wr, kmin, kmax);
        }
        const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
        const uint64_t nl2 = f2_make(nl, nl), ndd2 = f2_make(-dd, -dd);
        bool ok = true;
        int n = 0;
        for (int j = lo; j < hi; ++j, ++n) {
            const bool masked = kv_block_masked(j, imin, imax, sq.Lq, sq.Lk, 128, p.causal, p.wl,
                                                p.wr);
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->s_full, n & 1));
            tc_fence_after();
            uint32_t sv[64], dv[64];
            if (ok) {
                tmem_ld32(tmem + lane_off + kColS + 64 * ch, *reinterpret_cast<uint32_t(*)[32]>(sv));
                tmem_ld32(tmem + lane_off + kColS + 64 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
                tmem_ld32(tmem + lane_off + kColDP + 64 * ch, *reinterpret_cast<uint32_t(*)[32]>(dv));
                tmem_ld32(tmem + lane_off + kColDP + 64 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free);
            uint32_t pd[32];  // computed and stored only when the scores above were loaded
            if (ok && !masked) {
#pragma unroll
                for (int e = 0; e < 64; e += 2)
                    pd[e / 2] = ds_pair(sv[e], sv[e + 1], dv[e], dv[e + 1], scale2, nl2, ndd2);
            } else if (ok) {
                const int k0 = j * 128 + 64 * ch;
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    uint32_t pk;
                    p_ds_pair(sv[e], sv[e + 1], dv[e], dv[e + 1], scale2, nl2, ndd2,
                              k0 + e < kmin || k0 + e > kmax, k0 + e + 1 < kmin || k0 + e + 1 > kmax,
                              pk, pd[e / 2]);
                    (void)pk;
                }
            }
            // slot n % 2 is free once dQ of block n - 2 has read it
            if (n >= 2)
                ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->p_empty[n & 1], ((n - 2) >> 1) & 1));
            if (ok) {
                tmem_st32(tmem + lane_off + kColDS + 64 * (n & 1) + 32 * ch, pd);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[n & 1]);
        }
        // Epilogue: scale * dQ rows of this tile, bf16.
        if (n > 0) {
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->mm_done, 0));
            tc_fence_after();
        }
        const bool valid = ok && in_tile;
        __nv_bfloat16* dst =
            p.dq + (static_cast<size_t>(sq.q0 + tok) * p.Hq + sq.kvh * p.g + r % p.g) * D + (D / 2) * ch;
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
            if (valid) store_row32(dst + 32 * c, o, p.scale);
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
        constexpr int a = DkdvSmem<128>::kBytes, b = DqSmem<128>::kBytes;
        cudaFuncSetAttribute(bwd_dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, a);
        cudaFuncSetAttribute(bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, b);
        if (grid_kv.x > 0) bwd_dkdv_kernel<128><<<grid_kv, kBwdThreads, a, stream>>>(p);
        if (grid_q.x > 0) bwd_dq_kernel<128><<<grid_q, kBwdThreads, b, stream>>>(p);
    } else {
        constexpr int a = DkdvSmem<64>::kBytes, b = DqSmem<64>::kBytes;
        cudaFuncSetAttribute(bwd_dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, a);
        cudaFuncSetAttribute(bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, b);
        if (grid_kv.x > 0) bwd_dkdv_kernel<64><<<grid_kv, kBwdThreads, a, stream>>>(p);
        if (grid_q.x > 0) bwd_dq_kernel<64><<<grid_q, kBwdThreads, b, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace attn
