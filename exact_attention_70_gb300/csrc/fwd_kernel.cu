// fwd_kernel.cu -- varlen / GQA / causal / sliding-window prefill on tcgen05 tensor cores.
//
// The method ("Attention kernels: FlashAttention and PagedAttention", sections 三.2 and 四.1;
// "04 · FA4 (CuTeDSL) and engineering interfaces", sections 2, 4 and 5): for each tile of
// query rows, walk the key blocks it can see; per block compute S = Q K^T, mask it where
// needed, update the running row max m and denominator l in the exp2 domain, rescale the
// output accumulator when m moves, and accumulate P V; finally write O / l and
// LSE = (m + log2 l) ln 2.  S and P never leave the SM.
//
// GB300 mapping (one CTA per SM, persistent):
//   * a work item is two 128-row Q tiles of one (sequence, kv head); its rows pack
//     tokens x the g query heads of that kv head (pack_gqa), so each K/V block is loaded once
//     for 256 query rows;
//   * warp 8 issues TMA loads (Q once per item; K and V blocks into 2-stage rings);
//   * warp 9 owns the tensor memory and issues every tcgen05.mma from one thread;
//     S_t = Q_t K^T lands in TMEM columns [128 t, 128 t + 128), O_t in [256 + d t, ...);
//   * warps 10-11 only complete warpgroup 2, whose registers (80 per thread) go to the
//     softmax warpgroups (208 per thread) through setmaxnreg;
//   * warps 0-3 (tile 0) and 4-7 (tile 1) run the online softmax, one thread per TMEM lane,
//     i.e. one thread per query row; they write P as bf16 back over the first 64 columns of
//     S_t, and the MMA warp reads it from there as the A operand of O_t += P V;
//   * the MMA warp issues, per tile, PV_t(j) and then S_t(j+1) once PV_t(j) has completed
//     (S_t(j+1) overwrites the columns PV_t(j) reads), alternating between the two tiles so
//     one tile's softmax overlaps the other tile's MMAs;
//   * the running max only moves the accumulator's reference when it grows by more than
//     2^8 (the result is exact for any reference; this only bounds P <= 256), so the O
//     rescale through TMEM is rare after the first blocks.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_math.h"

namespace attn {

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdCfg {
    static constexpr int kHalves = D / 64;                 // 128-byte swizzle atoms along d
    static constexpr int kAtomBytes = 128 * 128;           // 128 rows x 128 B
    static constexpr int kQTile = kHalves * kAtomBytes;    // one 128-row Q tile
    static constexpr int kKvTile = kHalves * kAtomBytes;   // one 128-key K or V block
    static constexpr int kNK = D == 128 ? 2 : 4;           // K ring stages
    static constexpr int kNV = D == 128 ? 2 : 4;           // V ring stages
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kFwdTilesPerItem * kQTile;
    static constexpr int kOffV = kOffK + kNK * kKvTile;
    static constexpr int kOffBar = kOffV + kNV * kKvTile;
    static constexpr int kSmem = kOffBar + 1024 + 1024;    // barriers + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S_t (fp32, later P_t as bf16 pairs) and O_t
    __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + D * t; }
};

struct FwdBars {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4];
    uint64_t v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Geometry of one work item, derived identically by every role.
struct Item {
    int b, kvh, q0, Lq, k0, Lk;
    int tok0[2], imin[2], imax[2], lo[2], hi[2];
    bool rows[2], mma[2];
    int jlo, jhi;
    bool any;
};

__device__ __forceinline__ Item load_item(const FwdParams& p, int idx) {
    Item it;
    const int4 w = p.items[idx];
    it.b = w.x;
    it.kvh = w.y;
    const int m = w.z;
    it.q0 = p.cu_q[it.b];
    it.Lq = p.cu_q[it.b + 1] - it.q0;
    it.k0 = p.cu_k[it.b];
    it.Lk = p.cu_k[it.b + 1] - it.k0;
    it.jlo = 1 << 30;
    it.jhi = 0;
    it.any = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        it.tok0[t] = (2 * m + t) * p.tpt;
        it.rows[t] = it.tok0[t] < it.Lq;
        it.imin[t] = it.tok0[t];
        it.imax[t] = min(it.tok0[t] + p.tpt, it.Lq) - 1;
        it.lo[t] = it.hi[t] = 0;
        it.mma[t] = false;
        if (it.rows[t]) {
            const KvRange r = kv_block_range(it.imin[t], it.imax[t], it.Lq, it.Lk, kFwdBlockN,
                                             p.causal, p.wl, p.wr);
            it.lo[t] = r.lo;
            it.hi[t] = r.hi;
            it.mma[t] = r.hi > r.lo;
            if (it.mma[t]) {
                it.jlo = min(it.jlo, r.lo);
                it.jhi = max(it.jhi, r.hi);
                it.any = true;
            }
        }
    }
    return it;
}

// Persistent schedule: round k hands CTA c the item k*G + c (even rounds) or
// k*G + G-1-c (odd rounds); the list is sorted longest-first, so the snake order evens out
// the per-CTA totals.
__device__ __forceinline__ int item_index(int k, int c, int G) {
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Wait, ignoring the abort flag, for a barrier phase that TMA or the tensor core still owes
// us, so shared memory and TMEM are quiet before the CTA exits.
__device__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity)) {
        if (global_ns() - t0 > 200000000ull) return;
    }
}

// ---- TMA producer (one thread) -----------------------------------------------------------

template <int D>
__device__ void fwd_producer_loop(const FwdParams& p, uint8_t* smem, FwdBars* bars,
                                  const Watchdog& wd, int n_items, uint32_t& q_cnt,
                                  uint32_t& k_cnt, uint32_t& v_cnt) {
    using C = FwdCfg<D>;
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    const int G = gridDim.x, c = blockIdx.x;
    const uint32_t q_box_bytes = 64u * p.g * p.tpt * 2u;
    for (int k = 0; k * G < n_items; ++k) {
        const int idx = item_index(k, c, G);
        if (idx >= n_items) continue;
        const Item it = load_item(p, idx);
        if (!it.any) continue;
        if (q_cnt > 0 && !wd.wait(&bars->q_empty, (q_cnt - 1) & 1)) return;
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (it.mma[t]) qbytes += q_box_bytes * C::kHalves;
        mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!it.mma[t]) continue;
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h)
                tma_load_3d(smem + C::kOffQ + t * C::kQTile + h * C::kAtomBytes, &p.tm_q,
                            &bars->q_full, h * 64, it.kvh * p.g, it.q0 + it.tok0[t]);
        }
        ++q_cnt;
        for (int j = it.jlo; j < it.jhi; ++j) {
            {
                const uint32_t st = k_cnt % C::kNK;
                if (k_cnt >= C::kNK && !wd.wait(&bars->k_empty[st], ((k_cnt / C::kNK) - 1) & 1))
                    return;
                mbar_arrive_expect_tx(&bars->k_full[st], C::kKvTile);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(smem + C::kOffK + st * C::kKvTile + h * C::kAtomBytes, &p.tm_k,
                                &bars->k_full[st], h * 64, it.kvh, it.k0 + j * kFwdBlockN);
                ++k_cnt;
            }
            {
                const uint32_t st = v_cnt % C::kNV;
                if (v_cnt >= C::kNV && !wd.wait(&bars->v_empty[st], ((v_cnt / C::kNV) - 1) & 1))
                    return;
                mbar_arrive_expect_tx(&bars->v_full[st], C::kKvTile);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(smem + C::kOffV + st * C::kKvTile + h * C::kAtomBytes, &p.tm_v,
                                &bars->v_full[st], h * 64, it.kvh, it.k0 + j * kFwdBlockN);
                ++v_cnt;
            }
        }
    }
}

template <int D>
__device__ void fwd_producer(const FwdParams& p, uint8_t* smem, FwdBars* bars,
                             const Watchdog& wd, int n_items) {
    using C = FwdCfg<D>;
    uint32_t q_cnt = 0, k_cnt = 0, v_cnt = 0;
    fwd_producer_loop<D>(p, smem, bars, wd, n_items, q_cnt, k_cnt, v_cnt);
    // Every stage holds at most one load in flight: wait for the latest load of each one.
    if (q_cnt > 0) drain_wait(&bars->q_full, (q_cnt - 1) & 1);
    for (uint32_t st = 0; st < C::kNK && st < k_cnt; ++st)
        drain_wait(&bars->k_full[st], ((k_cnt - 1 - st) / C::kNK) & 1);
    for (uint32_t st = 0; st < C::kNV && st < v_cnt; ++st)
        drain_wait(&bars->v_full[st], ((v_cnt - 1 - st) / C::kNV) & 1);
}

// ---- MMA issuer (one thread) ---------------------------------------------------------------

template <int D>
__device__ void fwd_mma(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem,
                        const Watchdog& wd, int n_items) {
    using C = FwdCfg<D>;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, kFwdBlockN, false, false);
    constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
    const uint32_t q_base = smem_u32(smem + C::kOffQ);
    const uint32_t k_base = smem_u32(smem + C::kOffK);
    const uint32_t v_base = smem_u32(smem + C::kOffV);
    const int G = gridDim.x, cta = blockIdx.x;
    uint32_t q_cnt = 0, k_cnt = 0, v_cnt = 0;
    uint32_t pv_cnt[2] = {0, 0};   // PV_t issued so far (== P_t consumed)
    uint32_t o_items[2] = {0, 0};  // items in which tile t accumulated into O_t
    for (int k = 0; k * G < n_items; ++k) {
        const int idx = item_index(k, cta, G);
        if (idx >= n_items) continue;
        const Item it = load_item(p, idx);
        if (!it.any) continue;
        if (!wd.wait(&bars->q_full, q_cnt & 1)) return;
        ++q_cnt;
        tc_fence_after();
        int nS[2], nPV[2];
        bool first_pv[2] = {true, true};
#pragma unroll
        for (int t = 0; t < 2; ++t) nS[t] = nPV[t] = it.lo[t];
        bool q_released = false;
        unsigned long long t_idle = 0;
        uint32_t idle_spins = 0;
        while (true) {
            bool done = true, progress = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!it.mma[t]) continue;
                const int t2 = 1 - t;
                if (nPV[t] < it.hi[t]) done = false;
                // S_t(j) = Q_t K_j^T: needs K_j and the completion of PV_t(j-1), which reads P
                // from the columns S_t(j) overwrites.
                if (nS[t] < it.hi[t] && nS[t] == nPV[t]) {
                    const int j = nS[t];
                    const uint32_t n = k_cnt + (j - it.jlo);
                    const uint32_t st = n % C::kNK;
                    if (mbar_test(&bars->k_full[st], (n / C::kNK) & 1) &&
                        (pv_cnt[t] == 0 || mbar_test(&bars->pv_done[t], (pv_cnt[t] - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t qa = q_base + t * C::kQTile;
                        const uint32_t kb = k_base + st * C::kKvTile;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * C::kAtomBytes + (kk & 3) * 32;
                            umma_ss(tmem + C::col_s(t), sdesc_sw128(qa + off, 16, 1024),
                                    sdesc_sw128(kb + off, 16, 1024), kIdescS, kk > 0);
                        }
                        umma_commit(&bars->s_full[t]);
                        ++nS[t];
                        const bool other_needs =
                            it.mma[t2] && it.lo[t2] <= j && j < it.hi[t2] && nS[t2] <= j;
                        if (!other_needs) umma_commit(&bars->k_empty[st]);
                        if (!q_released && (!it.mma[0] || nS[0] == it.hi[0]) &&
                            (!it.mma[1] || nS[1] == it.hi[1])) {
                            umma_commit(&bars->q_empty);
                            q_released = true;
                        }
                        progress = true;
                    }
                }
                // O_t (+)= P_t(j) V_j: needs P_t(j), V_j and, for the item's first block, the
                // previous item's epilogue to have read O_t.
                if (nPV[t] < nS[t]) {
                    const int j = nPV[t];
                    const uint32_t n = v_cnt + (j - it.jlo);
                    const uint32_t st = n % C::kNV;
                    const bool o_ok = !first_pv[t] || o_items[t] == 0 ||
                                      mbar_test(&bars->o_free[t], (o_items[t] - 1) & 1);
                    if (o_ok && mbar_test(&bars->p_full[t], pv_cnt[t] & 1) &&
                        mbar_test(&bars->v_full[st], (n / C::kNV) & 1)) {
                        tc_fence_after();
                        const uint32_t vb = v_base + st * C::kKvTile;
#pragma unroll
                        for (int kk = 0; kk < kFwdBlockN / 16; ++kk) {
                            umma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8,
                                    sdesc_sw128(vb + kk * 16 * 128, C::kAtomBytes, 1024),
                                    kIdescO, (first_pv[t] && kk == 0) ? 0u : 1u);
                        }
                        umma_commit(&bars->pv_done[t]);
                        ++pv_cnt[t];
                        first_pv[t] = false;
                        ++nPV[t];
                        const bool other_needs =
                            it.mma[t2] && it.lo[t2] <= j && j < it.hi[t2] && nPV[t2] <= j;
                        if (!other_needs) umma_commit(&bars->v_empty[st]);
                        progress = true;
                    }
                }
            }
            if (done) break;
            if (progress) {
                idle_spins = 0;
            } else if ((++idle_spins & 63u) == 0) {
                if (wd.aborted()) return;
                const unsigned long long now = global_ns();
                if (t_idle == 0) {
                    t_idle = now;
                } else if (now - t_idle > kWaitLimitNs) {
                    wd.fail();
                    return;
                }
            }
            if (progress) t_idle = 0;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (it.mma[t]) ++o_items[t];
        k_cnt += it.jhi - it.jlo;
        v_cnt += it.jhi - it.jlo;
    }
}

// ---- softmax / correction / epilogue (one warpgroup per Q tile, one thread per row) -------

template <int D, int t>
__device__ void fwd_softmax(const FwdParams& p, FwdBars* bars, uint32_t tmem,
                            const Watchdog& wd, int n_items, int quarter, int lane) {
    using C = FwdCfg<D>;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const float sl2 = p.scale_log2;
    const int G = gridDim.x, cta = blockIdx.x;
    const int g = p.g;
    const int row_tok = row / g, row_head = row % g;
    const bool row_in_tile = row < g * p.tpt;
    uint32_t blk = 0;  // blocks of tile t processed so far (== S_t consumed == P_t produced)
    for (int k = 0; k * G < n_items; ++k) {
        const int idx = item_index(k, cta, G);
        if (idx >= n_items) continue;
        const Item it = load_item(p, idx);
        if (!it.rows[t]) continue;
        const int tok = it.tok0[t] + row_tok;
        const bool valid = row_in_tile && tok < it.Lq;
        const int head = it.kvh * g + row_head;
        int kmin, kmax;
        row_key_interval(tok, it.Lq, it.Lk, p.causal, p.wl, p.wr, kmin, kmax);
        float m_run = -INFINITY, l_run = 0.f;
        __nv_bfloat16* orow =
            p.out + (static_cast<size_t>(it.q0 + tok) * p.Hq + head) * D;
        if (it.mma[t]) {
            for (int j = it.lo[t]; j < it.hi[t]; ++j) {
                if (!__all_sync(0xffffffffu, wd.wait(&bars->s_full[t], blk & 1))) return;
                tc_fence_after();
                uint32_t s[128];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    tmem_ld32(tS + c4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c4 * 32]));
                tmem_wait_ld();
                if (kv_block_masked(j, it.imin[t], it.imax[t], it.Lq, it.Lk, kFwdBlockN,
                                    p.causal, p.wl, p.wr)) {
                    const int key0 = j * kFwdBlockN;
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const int key = key0 + c;
                        if (key < kmin || key > kmax) s[c] = __float_as_uint(-INFINITY);
                    }
                }
                // row max: eight independent chains of 3-input max, then a short tree
                float acc[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    float m = __uint_as_float(s[a]);
#pragma unroll
                    for (int i = 1; i < 15; i += 2)
                        m = fmax3(m, __uint_as_float(s[a + 8 * i]),
                                  __uint_as_float(s[a + 8 * (i + 1)]));
                    acc[a] = fmaxf(m, __uint_as_float(s[a + 120]));
                }
                const float mx = fmaxf(fmax3(acc[0], acc[1], acc[2]),
                                       fmax3(fmax3(acc[3], acc[4], acc[5]), acc[6], acc[7]));
                const float m_blk = mx * sl2;
                const bool need = m_blk > m_run + kRescaleThreshold;
                const float m_new = need ? m_blk : m_run;
                const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
                l_run *= alpha;
                m_run = m_new;
                const float mref = (m_run == -INFINITY) ? 0.f : m_run;
                // P = exp2(s * scale*log2e - m): paired FFMA, MUFU ex2, paired sums
                const uint64_t sl2x2 = f2_make(sl2, sl2);
                const uint64_t negm2 = f2_make(-mref, -mref);
                uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c = h * 64 + 2 * e;
                        const uint64_t x2 = f2_fma(
                            f2_make(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2,
                            negm2);
                        float x0, x1;
                        f2_split(x2, x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        sum2[e & 3] = f2_add(sum2[e & 3], f2_make(p0, p1));
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + h * 32, pk);
                }
                float sum;
                {
                    const uint64_t t2 = f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3]));
                    float lo, hi;
                    f2_split(t2, lo, hi);
                    sum = lo + hi;
                }
                l_run += sum;
                if (__any_sync(0xffffffffu, need) && j > it.lo[t]) {
                    // O_t holds PV_t(j-1); it completed before S_t(j) was issued.
                    if (!__all_sync(0xffffffffu, wd.wait(&bars->pv_done[t], (blk - 1) & 1)))
                        return;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[t]);
                ++blk;
            }
            // Epilogue: O / l from TMEM, bf16, straight to global memory.
            if (!__all_sync(0xffffffffu, wd.wait(&bars->pv_done[t], (blk - 1) & 1))) return;
            tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l,
                                          __uint_as_float(o[8 * v + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l,
                                          __uint_as_float(o[8 * v + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l,
                                          __uint_as_float(o[8 * v + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l,
                                          __uint_as_float(o[8 * v + 7]) * inv_l);
                        dst[v] = w;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free[t]);
        } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
        }
        if (valid) {
            p.lse[static_cast<size_t>(head) * p.total_q + it.q0 + tok] =
                l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars->k_full[i], 1);
            mbar_init(&bars->k_empty[i], 1);
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->v_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], 4);
            mbar_init(&bars->pv_done[t], 1);
            mbar_init(&bars->o_free[t], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    const int n_items = p.header->n_items;

    // Registers: launched at 168 per thread (384 threads); warpgroup 2 (TMA, MMA, 2 idle
    // warps) drops to 80 and the two softmax warpgroups rise to 208:
    // 128 * 80 + 256 * 208 = 63488 <= 384 * 168 = 64512.
    if (warp >= 8) {
        regs_decrease<80>();
        if (warp == 8) {
            if (lane == 0) fwd_producer<D>(p, smem, bars, wd, n_items);
        } else if (warp == 9) {
            if (lane == 0) {
                fwd_mma<D>(p, smem, bars, tmem, wd, n_items);
                // every tcgen05 op this thread issued has finished before TMEM is released
                umma_commit(&bars->drain);
                drain_wait(&bars->drain, 0);
            }
        }
    } else {
        regs_increase<208>();
        if (warp < 4)
            fwd_softmax<D, 0>(p, bars, tmem, wd, n_items, warp & 3, lane);
        else
            fwd_softmax<D, 1>(p, bars, tmem, wd, n_items, warp & 3, lane);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---- work-list construction (one CTA) ------------------------------------------------------

// Block-wide exclusive scan of one int per thread (blockDim.x == kPrepThreads).
__device__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    total = warp_tot[31];
    __syncthreads();
    return before;
}

__device__ int item_cost(const FwdPrepParams& p, int Lq, int Lk, int m) {
    int cost = 0;
    for (int t = 0; t < 2; ++t) {
        const int tok0 = (2 * m + t) * p.tpt;
        if (tok0 >= Lq) continue;
        const KvRange r = kv_block_range(tok0, min(tok0 + p.tpt, Lq) - 1, Lq, Lk, kFwdBlockN,
                                         p.causal, p.wl, p.wr);
        cost += r.hi - r.lo;
    }
    return cost;
}

__global__ void __launch_bounds__(kPrepThreads) fwd_prepare_kernel(FwdPrepParams p) {
    __shared__ int hist[kPrepBins];
    __shared__ int warp_tot[32];
    __shared__ int err;
    const int tid = threadIdx.x;
    if (tid == 0) err = 0;
    __syncthreads();
    // 1. the sequence boundaries must describe rows inside the tensors
    for (int b = tid; b < p.batch; b += blockDim.x) {
        const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
        if (q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.max_seqlen_q || k0 < 0 ||
            k1 < k0 || k1 > p.total_k || k1 - k0 > p.max_seqlen_k)
            err = 1;
    }
    __syncthreads();
    if (err) {
        if (tid == 0) {
            atomicOr(p.status, kStatusBounds);
            p.header->n_items = 0;
            p.header->n_pairs = 0;
        }
        return;
    }
    // 2. work items (pairs of Q tiles) per sequence, prefix-summed
    const int per_item = 2 * p.tpt;
    int carry = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
        const int b = base + tid;
        int n = 0;
        if (b < p.batch) n = (p.cu_q[b + 1] - p.cu_q[b] + per_item - 1) / per_item;
        int total;
        const int ex = block_exclusive_scan(n, warp_tot, total);
        if (b < p.batch) p.prefix[b] = carry + ex;
        carry += total;
    }
    if (tid == 0) p.prefix[p.batch] = carry;
    const int n_pairs = carry;
    if (n_pairs > p.capacity_pairs) {
        if (tid == 0) {
            atomicOr(p.status, kStatusBounds);
            p.header->n_items = 0;
            p.header->n_pairs = 0;
        }
        return;
    }
    __threadfence_block();
    __syncthreads();
    // 3. counting sort of the items by cost, longest first
    for (int i = tid; i < kPrepBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int q = tid; q < n_pairs; q += blockDim.x) {
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.prefix[mid] <= q) lo = mid; else hi = mid - 1;
        }
        const int b = lo, m = q - p.prefix[b];
        const int cost = item_cost(p, p.cu_q[b + 1] - p.cu_q[b], p.cu_k[b + 1] - p.cu_k[b], m);
        atomicAdd(&hist[kPrepBins - 1 - min(cost, kPrepBins - 1)], 1);
    }
    __syncthreads();
    int total;
    const int off = block_exclusive_scan(tid < kPrepBins ? hist[tid] : 0, warp_tot, total);
    if (tid < kPrepBins) hist[tid] = off;
    __syncthreads();
    for (int q = tid; q < n_pairs; q += blockDim.x) {
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.prefix[mid] <= q) lo = mid; else hi = mid - 1;
        }
        const int b = lo, m = q - p.prefix[b];
        const int cost = item_cost(p, p.cu_q[b + 1] - p.cu_q[b], p.cu_k[b + 1] - p.cu_k[b], m);
        const int slot = atomicAdd(&hist[kPrepBins - 1 - min(cost, kPrepBins - 1)], 1);
        for (int h = 0; h < p.Hkv; ++h)
            p.items[static_cast<size_t>(slot) * p.Hkv + h] = make_int4(b, h, m, cost);
    }
    if (tid == 0) {
        p.header->n_pairs = n_pairs;
        p.header->n_items = n_pairs * p.Hkv;
    }
}

}  // namespace

int fwd_smem_bytes(int head_dim) {
    return head_dim == 128 ? FwdCfg<128>::kSmem : FwdCfg<64>::kSmem;
}

cudaError_t configure_fwd_kernels() {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdCfg<128>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdCfg<64>::kSmem);
}

cudaError_t launch_fwd_prepare(const FwdPrepParams& p, cudaStream_t stream) {
    fwd_prepare_kernel<<<1, kPrepThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t stream) {
    if (head_dim == 128)
        fwd_kernel<128><<<grid, kFwdThreads, FwdCfg<128>::kSmem, stream>>>(p);
    else
        fwd_kernel<64><<<grid, kFwdThreads, FwdCfg<64>::kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
