// fwd_fp8_kernel.cu -- FP8 (e4m3) forward pass of exact attention on tcgen05 tensor cores.
//
// The method ("Attention kernels: FlashAttention and PagedAttention", section 四.2,
// FlashAttention-3): Q, K and V go to the 8-bit MMA as e4m3 values with block-wise scales, and
// V is re-laid out so that the P V product reads it key-major.  Around the two products the
// tiled online softmax is the one of the bf16 path (same page, section 三; "04 · FA4
// (CuTeDSL) and engineering interfaces", sections 4-5 for varlen and GQA packing): a running
// row maximum m and sum l, P~ = exp2(x - m), O rescaled when m moves.
//
// GB300 mapping: persistent CTAs, one per SM, each walking work items (pairs of 128-row packed
// Q tiles: tokens x the g query heads of a kv head) in a static snake order, the pairs that see
// the most keys first; barrier phases run on across items.  320 threads:
//   warps 0-7: the softmax, warps 4t..4t+3 for tile t, one thread per row (TMEM lane quarter =
//              warp % 4).  S of a key block is pulled into registers whole, so its TMEM region
//              is free again at once; P goes to shared memory as e4m3 bytes of 16 P~ (P~ <= 2^4
//              with the lazy rescale below, so 16 P~ <= 256 stays inside e4m3's range and its
//              normal grid covers P~ >= 2^-10);
//   warp 8:    TMA of each item's two Q tiles and of its K and V^T blocks into three-stage
//              rings, each block serving both tiles;
//   (an item's O leaves by TMA tensor store from the tile's P buffers when the tile's rows all
//   belong to its sequence, so the stores drain while the next item starts; ragged tiles store
//   row by row)
//   warp 9:    the MMA issuer: S_t(n) = Q_t K(n)^T (kind::f8f6f4, K = 32 per instruction) as
//              soon as tile t's softmax holds S_t(n-1) in registers, then O_t += P_t(n-1) V(n-1)
//              (A = P from shared memory, B = the V^T block, both K-major).
//   TMEM: tile t has S at [256 t, 256 t + 128) and O at [256 t + 128, 256 t + 256).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_math.h"

namespace attn {

namespace {

constexpr int kF8Threads = 320;
constexpr int kF8Stages = 3;
constexpr int kAtom = 128 * 128;      // 128 rows x 128 bytes, 128-byte swizzle
constexpr float kPLog2 = 4.f;         // P is stored as 2^4 P~
constexpr float kLazyLog2 = 4.f;      // O and l are rescaled only when m grows by more than this

struct F8Bars {
    uint64_t q_full, q_empty;               // the two Q tiles of the current item
    uint64_t k_full[kF8Stages], k_empty[kF8Stages];
    uint64_t v_full[kF8Stages], v_empty[kF8Stages];
    uint64_t s_full[2], s_free[2];          // per tile
    uint64_t p_full[2][2], p_empty[2][2];   // per tile and P buffer
    uint64_t pv_done[2];                    // per tile
    uint64_t o_done;                        // an item's last P V has finished
    uint64_t o_free[2];                     // tile t's softmax has read O_t of its item
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Shared memory: two Q tiles, K ring, V^T ring, two P buffers per tile (one atom each), barriers.
constexpr int kOffQ = 0;
constexpr int kOffK = 2 * kAtom;
constexpr int kOffV = kOffK + kF8Stages * kAtom;
constexpr int kOffP = kOffV + kF8Stages * kAtom;
constexpr int kOffBars = kOffP + 4 * kAtom;
constexpr int kF8Smem = kOffBars + static_cast<int>(sizeof(F8Bars)) + 1024;
static_assert(kF8Smem <= 227 * 1024, "FP8 forward shared memory");

__device__ void f8_drain(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > 200000000ull) return;
}

// One work item: a pair of 128-row packed Q tiles (tiles tile0, tile0 + 1) of one (sequence,
// kv head).  Items are numbered so that the pairs that see the most keys come first: item v
// is pair T - 1 - v / (batch Hkv) of (sequence, kv head) v % (batch Hkv), T pairs per sequence
// of max_seqlen_q tokens.  Every role derives the same item from v.
struct F8Item {
    int b, kvh, q0, Lq, k0, Lk, tile0, lo, hi, kb0;
    bool any;  // the item has rows (and its sequence's offsets are valid)
    bool bad;  // the sequence's offsets or the tables are out of bounds
};

__device__ F8Item f8_item(const Fp8Params& p, int v, int pairs) {
    F8Item it;
    const int bh = p.batch * p.Hkv;
    const int pair = pairs - 1 - v / bh, rem = v % bh;
    it.b = rem / p.Hkv;
    it.kvh = rem % p.Hkv;
    it.q0 = p.cu_q[it.b];
    it.Lq = p.cu_q[it.b + 1] - it.q0;
    it.k0 = p.cu_k[it.b];
    it.Lk = p.cu_k[it.b + 1] - it.k0;
    it.tile0 = 2 * pair;
    it.lo = it.hi = it.kb0 = 0;
    it.bad = it.q0 < 0 || it.Lq < 0 || it.q0 + it.Lq > p.total_q || it.Lq > p.max_seqlen_q ||
             it.k0 < 0 || it.Lk < 0 || it.k0 + it.Lk > p.total_k || it.Lk > p.max_seqlen_k;
    it.any = !it.bad && it.tile0 * p.tpt < it.Lq;
    if (!it.any) return it;
    // first 128-key block of this sequence in the V^T columns and the k_scale rows
    int kb0 = 0;
    for (int s = 0; s < it.b; ++s) kb0 += (p.cu_k[s + 1] - p.cu_k[s] + 127) / 128;
    it.kb0 = kb0;
    if (kb0 + (it.Lk + 127) / 128 > p.nkb) {  // the scale and V^T tables are too short
        it.bad = true;
        it.any = false;
        return it;
    }
    // key blocks seen by either tile (consecutive tiles see overlapping or adjacent ranges)
    const KvRange r0 = kv_block_range(it.tile0 * p.tpt, min(it.tile0 * p.tpt + p.tpt, it.Lq) - 1,
                                      it.Lq, it.Lk, 128, p.causal, p.wl, p.wr);
    it.lo = r0.lo;
    it.hi = r0.hi;
    if ((it.tile0 + 1) * p.tpt < it.Lq) {
        const KvRange r1 = kv_block_range((it.tile0 + 1) * p.tpt,
                                          min((it.tile0 + 2) * p.tpt, it.Lq) - 1, it.Lq, it.Lk,
                                          128, p.causal, p.wl, p.wr);
        if (it.hi <= it.lo) {
            it.lo = r1.lo;
            it.hi = r1.hi;
        } else if (r1.hi > r1.lo) {
            it.lo = min(it.lo, r1.lo);
            it.hi = max(it.hi, r1.hi);
        }
    }
    if (it.hi < it.lo) it.hi = it.lo;
    return it;
}

// Persistent schedule: round k hands CTA c the item k G + c (even rounds) or k G + G - 1 - c
// (odd rounds); with the longest pairs first this snake order evens out the per-CTA totals.
__device__ __forceinline__ int f8_item_index(int k, int c, int G) {
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

__global__ void __launch_bounds__(kF8Threads, 1) fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    F8Bars* bars = reinterpret_cast<F8Bars*>(smem + kOffBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pairs = (p.max_seqlen_q + 2 * p.tpt - 1) / (2 * p.tpt);
    const int n_items = pairs * p.batch * p.Hkv;
    const int G = gridDim.x, cta = blockIdx.x;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < kF8Stages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->s_free[t], 4);
            mbar_init(&bars->pv_done[t], 1);
            mbar_init(&bars->o_free[t], 4);
            for (int s = 0; s < 2; ++s) {
                mbar_init(&bars->p_full[t][s], 4);
                mbar_init(&bars->p_empty[t][s], 1);
            }
        }
        mbar_init(&bars->o_done, 1);
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

    if (warp == 8) {
        // TMA: each item's two Q tiles, then its K and V^T blocks through the rings
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            int nk = 0, nv = 0;
            uint32_t items = 0;
            bool ok = true;
            for (int k = 0; ok && k * G < n_items; ++k) {
                const int v = f8_item_index(k, cta, G);
                if (v >= n_items) continue;
                const F8Item it = f8_item(p, v, pairs);
                if (it.bad) atomicOr(p.status, kStatusBounds);
                if (!it.any) continue;
                // the previous item's last S has read the Q tiles
                if (items > 0 && !wd.wait(&bars->q_empty, (items - 1) & 1)) break;
                mbar_arrive_expect_tx(&bars->q_full, 2 * 128u * p.g * p.tpt);
                tma_load_3d(smem + kOffQ, &p.tm_q, &bars->q_full, 0, it.kvh * p.g,
                            it.q0 + it.tile0 * p.tpt);
                tma_load_3d(smem + kOffQ + kAtom, &p.tm_q, &bars->q_full, 0, it.kvh * p.g,
                            it.q0 + (it.tile0 + 1) * p.tpt);
                ++items;
                for (int j = it.lo; j < it.hi; ++j) {
                    const int sk = nk % kF8Stages;
                    if (nk >= kF8Stages && !wd.wait(&bars->k_empty[sk], ((nk / kF8Stages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->k_full[sk], kAtom);
                    tma_load_3d(smem + kOffK + sk * kAtom, &p.tm_k, &bars->k_full[sk], 0, it.kvh,
                                it.k0 + j * 128);
                    ++nk;
                    const int sv = nv % kF8Stages;
                    if (nv >= kF8Stages && !wd.wait(&bars->v_empty[sv], ((nv / kF8Stages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->v_full[sv], kAtom);
                    tma_load_3d(smem + kOffV + sv * kAtom, &p.tm_v, &bars->v_full[sv],
                                128 * (it.kb0 + j), 0, it.kvh);
                    ++nv;
                }
            }
            // every load this thread issued has landed before the CTA's shared memory goes
            if (items > 0) f8_drain(&bars->q_full, (items - 1) & 1);
            for (int m = nk > kF8Stages ? nk - kF8Stages : 0; m < nk; ++m)
                f8_drain(&bars->k_full[m % kF8Stages], (m / kF8Stages) & 1);
            for (int m = nv > kF8Stages ? nv - kF8Stages : 0; m < nv; ++m)
                f8_drain(&bars->v_full[m % kF8Stages], (m / kF8Stages) & 1);
        }
    } else if (warp == 9) {
        // the MMA issuer: S_t(n) as soon as tile t's softmax holds S_t(n-1), then the previous
        // block's P V; block counters run on across items
        if (lane == 0) {
            constexpr uint32_t kId = idesc_e4m3_f32(128, 128);
            uint32_t items = 0;
            // O_t += P_t(m) V(m) for both tiles: K-steps of 32 keys (32 bytes) along both
            // K-major operands.  An item's first P V overwrites O_t, so it waits for the previous
            // item's epilogue to have read O_t.
            auto pv = [&](int m, bool first) {
                const int sv = m % kF8Stages, bm = m & 1;
                if (!wd.wait(&bars->v_full[sv], (m / kF8Stages) & 1)) return false;
                const uint64_t vd = sdesc_sw128(smem_u32(smem + kOffV + sv * kAtom), 16, 1024);
                for (int t = 0; t < 2; ++t) {
                    if (!wd.wait(&bars->p_full[t][bm], (m >> 1) & 1)) return false;
                    if (first && items > 0 && !wd.wait(&bars->o_free[t], (items - 1) & 1))
                        return false;
                    tc_fence_after();
                    const uint64_t pd =
                        sdesc_sw128(smem_u32(smem + kOffP + (2 * t + bm) * kAtom), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_ss_f8(tmem + 256 * t + 128, pd + 2 * kk, vd + 2 * kk, kId,
                                   (!first || kk > 0) ? 1u : 0u);
                    umma_commit(&bars->p_empty[t][bm]);
                    umma_commit(&bars->pv_done[t]);
                }
                umma_commit(&bars->v_empty[sv]);
                return true;
            };
            int n = 0;
            bool ok = true;
            for (int k = 0; ok && k * G < n_items; ++k) {
                const int v = f8_item_index(k, cta, G);
                if (v >= n_items) continue;
                const F8Item it = f8_item(p, v, pairs);
                if (!it.any) continue;
                ok = wd.wait(&bars->q_full, items & 1);
                if (!ok) break;
                const int n0 = n;
                for (int j = it.lo; ok && j < it.hi; ++j) {
                    const int sk = n % kF8Stages;
                    ok = wd.wait(&bars->k_full[sk], (n / kF8Stages) & 1);
                    if (!ok) break;
                    const uint64_t kd = sdesc_sw128(smem_u32(smem + kOffK + sk * kAtom), 16, 1024);
                    for (int t = 0; t < 2 && ok; ++t) {
                        // S_t(n) over S_t(n-1), which tile t's softmax holds in registers
                        ok = n == 0 || wd.wait(&bars->s_free[t], (n - 1) & 1);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t qd = sdesc_sw128(smem_u32(smem + kOffQ + t * kAtom), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ss_f8(tmem + 256 * t, qd + 2 * kk, kd + 2 * kk, kId, kk > 0 ? 1u : 0u);
                        umma_commit(&bars->s_full[t]);
                    }
                    if (!ok) break;
                    umma_commit(&bars->k_empty[sk]);
                    if (j == it.hi - 1) umma_commit(&bars->q_empty);  // the item's last S
                    if (n > n0 && !pv(n - 1, n - 1 == n0)) {
                        ok = false;
                        break;
                    }
                    ++n;
                }
                if (!ok) break;
                if (n > n0) {
                    if (!pv(n - 1, n - 1 == n0)) break;
                } else {
                    // no key block: Q is released at once and O's previous reader is awaited
                    // here, so every item consumes one phase of q_empty and of o_free
                    umma_commit(&bars->q_empty);
                    if (items > 0 && !(wd.wait(&bars->o_free[0], (items - 1) & 1) &&
                                       wd.wait(&bars->o_free[1], (items - 1) & 1)))
                        break;
                }
                umma_commit(&bars->o_done);
                ++items;
            }
            umma_commit(&bars->drain);
            f8_drain(&bars->drain, 0);
        }
    } else {
        // softmax: tile t, thread = packed row r of the tile
        const int t = warp >> 2, quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
        const uint32_t col_s = 256 * t, col_o = 256 * t + 128;
        bool ok = true;
        int n = 0;  // key blocks of this CTA so far (barrier phases run on across items)
        uint32_t items = 0;
        // A whole tile's O leaves through its two P buffers by TMA store; before P or O is
        // written there again, the store must have read them (the same for all four warps of
        // the tile, so the named barrier is met alike).
        bool epi_pending = false;
        auto release_staging = [&]() {
            if (epi_pending) {
                if (quarter == 0 && lane == 0) bulk_wait_group_read_all();
                named_bar_sync(1 + t, 128);
                epi_pending = false;
            }
        };
        for (int k = 0; k * G < n_items; ++k) {
            const int v = f8_item_index(k, cta, G);
            if (v >= n_items) continue;
            const F8Item it = f8_item(p, v, pairs);
            if (!it.any) continue;
            const int Lq = it.Lq, Lk = it.Lk;
            const int imin = (it.tile0 + t) * p.tpt;
            const bool tile_ok = imin < Lq;
            const int imax = tile_ok ? min(imin + p.tpt, Lq) - 1 : imin;
            const int tok = imin + r / p.g, head = it.kvh * p.g + r % p.g;
            const bool valid = tile_ok && r < p.g * p.tpt && tok < Lq;
            int kmin = 1, kmax = 0;
            float qs = 0.f;
            if (valid) {
                row_key_interval(tok, Lq, Lk, p.causal, p.wl, p.wr, kmin, kmax);
                qs = p.q_scale[static_cast<size_t>(head) * p.nqb + (it.q0 + tok) / 128];
            }
            const float* ks_row = p.k_scale + static_cast<size_t>(it.kvh) * p.nkb + it.kb0;
            // this thread's row of the tile's P buffers: 128 keys as bytes, 16-byte chunk c at
            // c ^ (r % 8)
            const uint32_t row_p = smem_u32(smem + kOffP + 2 * t * kAtom) + r * 128;
            float m_used = -INFINITY, l = 0.f;
            const int n0 = n;
            // blocks needing the element mask are a prefix and a suffix of [lo, hi): the rest,
            // [full_lo, full_hi), is found once per item
            int full_lo = it.lo, full_hi = it.hi;
            while (full_lo < full_hi &&
                   kv_block_masked(full_lo, imin, imax, Lq, Lk, 128, p.causal, p.wl, p.wr))
                ++full_lo;
            while (full_hi > full_lo &&
                   kv_block_masked(full_hi - 1, imin, imax, Lq, Lk, 128, p.causal, p.wl, p.wr))
                --full_hi;
            // each block's K scale, loaded a block ahead
            float ks_next = it.hi > it.lo ? ks_row[it.lo] : 0.f;
            for (int j = it.lo; j < it.hi; ++j, ++n) {
                const int bn = n & 1;
                const float ks = ks_next;
                if (j + 1 < it.hi) ks_next = ks_row[j + 1];
                const bool masked = !valid || j < full_lo || j >= full_hi;
                // (kept positive so that a masked -inf never meets a zero multiplier)
                const float c = fmaxf(qs * ks * p.scale_log2, 1.17549435e-38f);
                ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->s_full[t], n & 1));
                tc_fence_after();
                uint32_t s[128];
                if (ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld32(tmem + lane_off + col_s + 32 * q,
                                  *reinterpret_cast<uint32_t(*)[32]>(s + 32 * q));
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 128; ++e) s[e] = 0u;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_free[t]);
                if (masked) {
#pragma unroll
                    for (int e = 0; e < 128; ++e) {
                        const int key = j * 128 + e;
                        if (!valid || key < kmin || key > kmax) s[e] = __float_as_uint(-INFINITY);
                    }
                }
                // row maximum of the raw scores (c > 0 keeps the order)
                // (four independent chains)
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 128; e += 8)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        mq[u] = fmax3(mq[u], __uint_as_float(s[e + 2 * u]), __uint_as_float(s[e + 2 * u + 1]));
                const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                const float xm = mx == -INFINITY ? -INFINITY : mx * c;
                // lazy rescale: move m only when the block's maximum exceeds it by > 2^4
                const bool grow = xm > m_used + kLazyLog2;
                float alpha = 1.f;
                if (grow) {
                    if (m_used != -INFINITY) alpha = exp2f(m_used - xm);
                    l *= alpha;
                    m_used = xm;
                }
                // Buffer bn is free once P V of block n - 2 has read it.  Waited for before the
                // rescale below: pv_done's phases are told apart by parity only, so the wait for
                // P V n - 1 there is exact only once P V n - 2 is known to have finished.
                if (n >= 2)
                    ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->p_empty[t][bn], ((n - 2) >> 1) & 1));
                if (__any_sync(0xffffffffu, grow && alpha != 1.f) && n > n0) {
                    // O_t holds earlier blocks of this item: wait for its last P V, then scale
                    // its rows
                    ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->pv_done[t], (n - 1) & 1));
                    tc_fence_after();
                    if (ok) {
                        // in 8-column pieces: the block's 128 scores stay live meanwhile
#pragma unroll 1
                        for (int q = 0; q < 16; ++q) {
                            uint32_t o[8];
                            tmem_ld8(tmem + lane_off + col_o + 8 * q, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st8(tmem + lane_off + col_o + 8 * q, o);
                        }
                        tmem_wait_st();
                    }
                    // the rescaled O_t before the P V that p_full releases (issued by another
                    // thread): the stores are ordered before that arrive
                    tc_fence_before();
                }
                release_staging();
                // P = 2^4 exp2(x - m), x = s c; an empty row so far uses m = 0 (no -inf - -inf);
                // each 16 keys go to shared memory as they are done
                const float off = kPLog2 - (m_used == -INFINITY ? 0.f : m_used);
                const uint64_t c2 = f2_make(c, c), off2 = f2_make(off, off);
                const uint32_t row = row_p + bn * kAtom;
                float su[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial sums
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t pk[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 16 * cc + 4 * u;
                        float x0, x1, x2, x3;
                        f2_split(f2_fma(f2_make(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), c2, off2), x0, x1);
                        f2_split(f2_fma(f2_make(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])), c2, off2), x2, x3);
                        x0 = ex2_approx(x0);
                        x1 = ex2_approx(x1);
                        x2 = ex2_approx(x2);
                        x3 = ex2_approx(x3);
                        su[u] += (x0 + x1) + (x2 + x3);
                        pk[u] = pack_e4m3x4(x0, x1, x2, x3);
                    }
                    if (ok)
                        st_shared_v4(row + static_cast<uint32_t>(((cc ^ (r & 7)) * 16)), pk[0], pk[1],
                                     pk[2], pk[3]);
                }
                l += (su[0] + su[1]) + (su[2] + su[3]);
                if (ok) fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[t][bn]);
            }
            // Epilogue: O = v_scale O~ / l as bf16, LSE = ln 2 (m + log2 l - 4).  Every item
            // ends with one o_done phase; O_t is released (o_free) once read.
            ok = ok && __all_sync(0xffffffffu, wd.wait(&bars->o_done, items & 1));
            tc_fence_after();
            const bool had_blocks = n > n0;
            // the item's place in the output, derived again here from v (volatile loads) so
            // that none of it stays live through the block loop
            const int bh = p.batch * p.Hkv, grp = v % bh;
            const int eb = grp / p.Hkv, ekvh = grp % p.Hkv;
            const int eq0 = *reinterpret_cast<const volatile int*>(p.cu_q + eb);
            const int eLq = *reinterpret_cast<const volatile int*>(p.cu_q + eb + 1) - eq0;
            const int etile = 2 * (pairs - 1 - v / bh) + t;
            const int etok = etile * p.tpt + r / p.g, ehead = ekvh * p.g + r % p.g;
            const float vs = p.v_scale[static_cast<size_t>(eb) * p.Hkv + ekvh];
            const float mul = l > 0.f ? vs / l : 0.f;
            // A tile whose rows all belong to the sequence is staged in its two P buffers (free:
            // every P V of the item has finished) in the layout of a 128-byte-swizzled TMA box
            // {64 columns, g heads, tpt tokens} and stored by TMA, asynchronously; a ragged tile
            // is stored row by row.
            const bool whole = (etile + 1) * p.tpt <= eLq;
            if (whole) release_staging();
            __nv_bfloat16* dst = p.out + (static_cast<size_t>(eq0 + etok) * p.Hq + ehead) * 128;
            const bool stored =
                ATTN_IN_BOUNDS(!valid || (eq0 + etok < p.total_q && ehead < p.Hq), p.status);
            const uint32_t stage = smem_u32(smem + kOffP + 2 * t * kAtom) + r * 128;
            // the row's 128 columns in one go (one wait for the four loads)
            uint32_t ob[128];
            if (had_blocks && ok) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld32(tmem + lane_off + col_o + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(ob + 32 * q));
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 128; ++e) ob[e] = 0u;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t* o = ob + 32 * q;
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
                if (whole) {
                    // 16-byte chunk c (of 16) of the row: buffer c / 8, position (c % 8) ^ (r % 8)
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const int c = 4 * q + v4;
                        st_shared_v4(stage + static_cast<uint32_t>((c >> 3) * kAtom + (((c & 7) ^ (r & 7)) * 16)),
                                     w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                    }
                } else if (valid && ok && stored) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * q);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        d4[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                }
            }
            // O_t has been read: the next item's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free[t]);
            if (whole) {
                fence_proxy_async_smem();
                named_bar_sync(1 + t, 128);
                if (quarter == 0 && lane == 0) {
                    const int row0 = eq0 + etile * p.tpt;
                    if (ok && ATTN_IN_BOUNDS(row0 >= 0 && row0 + p.tpt <= p.total_q && (ekvh + 1) * p.g <= p.Hq,
                                             p.status)) {
                        tma_store_3d(&p.tm_o, smem + kOffP + 2 * t * kAtom, 0, ekvh * p.g, row0);
                        tma_store_3d(&p.tm_o, smem + kOffP + (2 * t + 1) * kAtom, 64, ekvh * p.g, row0);
                    }
                    bulk_commit_group();
                }
                epi_pending = true;
            }
            if (valid && ok && stored)
                p.lse[static_cast<size_t>(ehead) * p.total_q + eq0 + etok] =
                    l > 0.f ? (m_used + log2f(l) - kPLog2) * 0.69314718055994531f : -INFINITY;
            ++items;
        }
        // the O stores this thread issued have completed before the CTA's memory goes
        if (quarter == 0 && lane == 0) bulk_wait_group_all();
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

cudaError_t launch_fwd_fp8(const Fp8Params& p, cudaStream_t stream) {
    int dev = 0, num_sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 1;
    const long long tiles = (p.max_seqlen_q + p.tpt - 1) / p.tpt;
    const long long items = (tiles + 1) / 2 * p.batch * p.Hkv;
    const int grid = static_cast<int>(items < num_sms ? items : num_sms);
    cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (grid > 0) fwd_fp8_kernel<<<grid, kF8Threads, kF8Smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
