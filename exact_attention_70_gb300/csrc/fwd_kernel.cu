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
//   * warp 16 issues TMA loads: Q once per item, then the item's K and V blocks through one
//     ring of shared-memory slots, in the order the tensor core consumes them
//     (K_0, K_1, V_0, K_2, V_1, ..., V_{m-1});
//   * warp 17 issues every S_t = Q_t K^T (fp32 into TMEM columns [128 t, 128 t + 128)) and
//     warp 18 every O_t += P_t V (O_t in TMEM columns [256 + d t, ...)), both with operands in
//     shared memory.  An issuing thread blocks until the tensor pipe accepts each instruction
//     and the pipe holds little beyond the one executing, so a wait between two groups on a
//     single issuer idles the tensor cores; with two issuers one thread's waits overlap the
//     other thread's MMAs;
//   * warps 0-7 (tile 0) and 8-15 (tile 1) run the online softmax, 16 query rows per warp in
//     the MMA accumulator-fragment layout.  They release S_t as soon as it is in registers,
//     so S_t(j+1) is computed while they exponentiate block j, and write P_t as bf16 to
//     shared memory, with stmatrix, in the 128-byte-swizzled K-major layout the tensor core
//     reads as the A operand;
//   * warps 16-19 (warpgroup 4) give registers to the softmax warpgroups through setmaxnreg;
//   * the running max only moves the accumulator's reference when it grows by more than
//     2^8 (the result is exact for any reference; this only bounds P <= 256), so the O
//     rescale through TMEM is rare after the first blocks.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "softcap.cuh"
#include "tile_math.h"

namespace attn {

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct FwdCfg {
    static constexpr int kHalves = D / 64;                 // 128-byte swizzle atoms along d
    static constexpr int kAtomBytes = 128 * 128;           // 128 rows x 128 B
    static constexpr int kQTile = kHalves * kAtomBytes;    // one 128-row Q tile
    static constexpr int kKvTile = kHalves * kAtomBytes;   // one 128-key K or V block
    static constexpr int kPTile = 2 * kAtomBytes;          // 128 rows x 128 keys of P, bf16
    static constexpr int kSlots = D == 128 ? 3 : 8;        // K/V ring slots
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kFwdTilesPerItem * kQTile;
    static constexpr int kOffKV = kOffP + kFwdTilesPerItem * kPTile;
    static constexpr int kOffBar = kOffKV + kSlots * kKvTile;
    static constexpr int kSmem = kOffBar + 512 + 1024;     // barriers + alignment slack
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns of S_t (fp32) and O_t (fp32)
    __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + D * t; }
};

struct FwdBars {
    uint64_t q_full, q_empty;
    // One ring of K/V slots.  A slot alternates between K and V blocks, and K is consumed by the
    // S issuer while V is consumed by the PV issuer, so each slot has one "full" barrier per
    // kind: every waiter then sees every phase of its barrier in order, which is what a parity
    // wait needs (on a shared barrier the S issuer could wait for a K while the slot's previous
    // V was still landing, and its parity wait would read the phase before as complete).
    uint64_t k_full[8], v_full[8], kv_empty[8];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_free[2];
    uint64_t epi_full[2], epi_free[2];  // O staged in P_t for a TMA store / the store read it
    uint64_t drain[2];
    uint64_t idx_full[4], idx_empty[4];  // the claimed item indices (fwd_claim_item)
    int idx_ring[4];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(FwdBars) <= 512, "barrier block");

// Per-slot parity of the K (or V) loads a role has seen go into each ring slot: bit s flips at
// every load of that kind into slot s, and before a wait it is the parity of the awaited phase.
__device__ __forceinline__ uint32_t slot_parity(uint32_t bits, uint32_t st) {
    return (bits >> st) & 1u;
}

// Geometry of one work item, derived identically by every role.
struct Item {
    int b, kvh, q0, Lq, k0, Lk;
    int tok0[2], imin[2], imax[2], lo[2], hi[2];
    bool rows[2], mma[2];
    int jlo, jhi;
    bool any;
};

template <bool kPaged>
__device__ __forceinline__ Item load_item(const FwdParams& p, int idx) {
    Item it;
    const int4 w = p.items[idx];
    it.b = w.x;
    it.kvh = w.y;
    const int m = w.z;
    it.q0 = p.cu_q[it.b];
    it.Lq = p.cu_q[it.b + 1] - it.q0;
    if constexpr (kPaged) {  // the cached prefix, then this call's new tokens
        it.k0 = 0;
        it.Lk = p.cache_seqlens[it.b] + it.Lq;
    } else {
        it.k0 = p.cu_k[it.b];
        it.Lk = p.cu_k[it.b + 1] - it.k0;
    }
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

__device__ __forceinline__ bool tile_uses(const Item& it, int t, int j) {
    return it.mma[t] && it.lo[t] <= j && j < it.hi[t];
}

// Positions in the K/V ring, relative to the item's first slot, of K_i and V_i for an item of
// m key blocks.  The two tiles' key ranges overlap or touch, so their union [jlo, jhi) has no
// gap; the producer fills 2m slots in the order K_0, K_1, V_0, K_2, V_1, ..., K_{m-1},
// V_{m-2}, V_{m-1}.
__device__ __forceinline__ uint32_t ring_pos_k(int i) { return i == 0 ? 0u : 2u * i - 1u; }
__device__ __forceinline__ uint32_t ring_pos_v(int i, int m) {
    return i == m - 1 ? 2u * m - 1u : 2u * i + 2u;
}

// Persistent schedule with dynamic claims.  The work list comes in groups of KV heads, each
// sorted longest-first; a CTA's TMA producer claims the next index from a global counter while
// the CTA still works on its current item (after that item's first loads), so CTAs take items
// in list order as they free up: the longest-first order evens out the finishing times, and
// the CTAs running at any moment share the few KV heads of one or two groups, whose K/V
// blocks then stay in L2 between the items that read them.  The producer hands each index to
// the CTA's other roles through a four-slot ring in shared memory; every role derives the item
// from the index (load_item), and -1 ends the loop.
constexpr uint32_t kIdxRing = 4;
constexpr uint32_t kIdxReaders = 18;  // the two MMA issuers and the 16 softmax warps

// The producer's claim of ring position r (false: a wait gave up).  Slot r % 4 last held
// position r - 4, which every reader took before its own item r - 3.
__device__ __forceinline__ bool fwd_claim_item(const FwdParams& p, FwdBars* bars,
                                               const Watchdog& wd, int n_items, uint32_t r,
                                               int& idx) {
    const uint32_t slot = r % kIdxRing;
    if (r >= kIdxRing && !wd.wait(&bars->idx_empty[slot], ((r / kIdxRing) - 1) & 1))
        return false;
    idx = atomicAdd(&p.header->next_item, 1);
    if (idx >= n_items) idx = -1;
    bars->idx_ring[slot] = idx;
    mbar_arrive(&bars->idx_full[slot]);  // release: the index is visible to the readers
    return true;
}

// The item index of ring position r for one reading thread, and r advanced (-2: a wait gave
// up, -1: no more items).
__device__ __forceinline__ int fwd_take_item(FwdBars* bars, const Watchdog& wd, uint32_t& r) {
    const uint32_t slot = r % kIdxRing;
    if (!wd.wait(&bars->idx_full[slot], (r / kIdxRing) & 1)) return -2;
    const int idx = *reinterpret_cast<volatile int*>(&bars->idx_ring[slot]);
    mbar_arrive(&bars->idx_empty[slot]);
    ++r;
    return idx;
}

// The same for a whole warp: lane 0 releases the slot once every lane has the index.
__device__ __forceinline__ int fwd_take_item_warp(FwdBars* bars, const Watchdog& wd,
                                                  uint32_t& r, int lane) {
    const uint32_t slot = r % kIdxRing;
    if (!__all_sync(0xffffffffu, wd.wait(&bars->idx_full[slot], (r / kIdxRing) & 1))) return -2;
    const int idx = *reinterpret_cast<volatile int*>(&bars->idx_ring[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->idx_empty[slot]);
    ++r;
    return idx;
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

// What the producer has put into the ring: the slot loads so far and, per slot, the parity of
// its K and of its V loads and whether its latest load was a V.
struct RingState {
    uint32_t n = 0, kpar = 0, vpar = 0, lastv = 0;
};

template <int D, bool kPaged>
__device__ void fwd_producer_loop(const FwdParams& p, uint8_t* smem, FwdBars* bars,
                                  const Watchdog& wd, int n_items, uint32_t& q_cnt,
                                  RingState& ring) {
    using C = FwdCfg<D>;
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    const uint32_t q_box_bytes = 64u * p.g * p.tpt * 2u;
    uint32_t claims = 0;
    int idx;
    if (!fwd_claim_item(p, bars, wd, n_items, claims++, idx)) return;
    while (idx >= 0) {
        const Item it = load_item<kPaged>(p, idx);
        int next = -1;
        bool claimed = false;
        if (!it.any) {
            if (!fwd_claim_item(p, bars, wd, n_items, claims++, next)) return;
            idx = next;
            continue;
        }
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
        const int m = it.jhi - it.jlo;
        for (int r = 0; r < 2 * m; ++r) {
            // inverse of ring_pos_k / ring_pos_v
            const bool last = r == 2 * m - 1;
            const bool is_v = last || (r > 0 && (r & 1) == 0);
            const int i = is_v ? (last ? m - 1 : (r - 2) / 2) : (r + 1) / 2;
            const uint32_t n = ring.n;
            const uint32_t st = n % C::kSlots;
            if (n >= C::kSlots && !wd.wait(&bars->kv_empty[st], ((n / C::kSlots) - 1) & 1))
                return;
            uint64_t* const full = is_v ? &bars->v_full[st] : &bars->k_full[st];
            mbar_arrive_expect_tx(full, C::kKvTile);
            ++ring.n;
            if (is_v) {
                ring.vpar ^= 1u << st;
                ring.lastv |= 1u << st;
            } else {
                ring.kpar ^= 1u << st;
                ring.lastv &= ~(1u << st);
            }
            const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
            uint8_t* const slot = smem + C::kOffKV + st * C::kKvTile;
            if constexpr (!kPaged) {
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(slot + h * C::kAtomBytes, map, full, h * 64, it.kvh,
                                it.k0 + (it.jlo + i) * kFwdBlockN);
            } else {
                // Gather the block's keys page by page through block_table.  Boxes wholly past
                // the sequence end (whose table entries need not be valid) and boxes of a bad
                // page id are aimed past the end of the cache, so TMA fills them with zeros.
                const int* bt = p.block_table + static_cast<size_t>(it.b) * p.max_pages;
                const int oob_row = p.num_pages * p.page_size;
                for (int r0 = 0; r0 < kFwdBlockN; r0 += p.box_rows) {
                    const int key = (it.jlo + i) * kFwdBlockN + r0;
                    int row = oob_row;
                    if (key < it.Lk) {
                        const int page = bt[key / p.page_size];
                        if (page >= 0 && page < p.num_pages)
                            row = page * p.page_size + key % p.page_size;
                        else
                            atomicOr(p.status, kStatusBounds);
                    }
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(slot + h * C::kAtomBytes + r0 * 128, map, full, h * 64,
                                    it.kvh, row);
                }
            }
            // claim the next item two key blocks before this one's last load: late enough
            // that claims follow the order in which CTAs free up, early enough that the
            // claim's round trip is hidden behind the blocks still to come
            if (!claimed && r == max(min(1, 2 * m - 1), 2 * m - 5)) {
                if (!fwd_claim_item(p, bars, wd, n_items, claims++, next)) return;
                claimed = true;
            }
        }
        idx = next;
    }
}

template <int D, bool kPaged>
__device__ void fwd_producer(const FwdParams& p, uint8_t* smem, FwdBars* bars,
                             const Watchdog& wd, int n_items) {
    using C = FwdCfg<D>;
    uint32_t q_cnt = 0;
    RingState ring;
    fwd_producer_loop<D, kPaged>(p, smem, bars, wd, n_items, q_cnt, ring);
    // Every slot holds at most one load in flight: wait for the latest load of each one (its
    // phase has the parity before that load's flip).
    if (q_cnt > 0) drain_wait(&bars->q_full, (q_cnt - 1) & 1);
    for (uint32_t st = 0; st < C::kSlots && st < ring.n; ++st) {
        const bool v = slot_parity(ring.lastv, st) != 0;
        drain_wait(v ? &bars->v_full[st] : &bars->k_full[st],
                   slot_parity(v ? ring.vpar : ring.kpar, st) ^ 1u);
    }
}

// ---- MMA issuers: warp 17 issues S = Q K^T, warp 18 issues O += P V (one thread each) -----

// S_t(j) for every (j, t) of every item.  S_t(j) overwrites the TMEM columns of S_t(j-1), so
// it waits for tile t's softmax to have read them (s_free).
template <int D, bool kPaged>
__device__ void fwd_mma_s(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem,
                          const Watchdog& wd, int n_items) {
    using C = FwdCfg<D>;
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, kFwdBlockN, false, false);
    // K-major operand descriptors (128-byte swizzle, 8-row groups 1024 B apart), as halves
    const uint64_t dq = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dkv = sdesc_sw128(smem_u32(smem + C::kOffKV), 16, 1024);
    const uint32_t q_lo = static_cast<uint32_t>(dq), d_hi = static_cast<uint32_t>(dq >> 32);
    const uint32_t kv_lo = static_cast<uint32_t>(dkv);
    uint32_t q_cnt = 0, kv_cnt = 0;
    uint32_t kpar = 0;                // per-slot parity of the K blocks consumed so far
    uint32_t s_cnt0 = 0, s_cnt1 = 0;  // S_t issued so far
    for (uint32_t rd = 0;;) {
        const int idx = fwd_take_item(bars, wd, rd);
        if (idx < 0) return;
        const Item it = load_item<kPaged>(p, idx);
        if (!it.any) continue;
        if (!wd.wait(&bars->q_full, q_cnt & 1)) return;
        ++q_cnt;
        const int m = it.jhi - it.jlo;
        for (int i = 0; i < m; ++i) {
            const int j = it.jlo + i;
            const uint32_t n = kv_cnt + ring_pos_k(i);
            const uint32_t st = n % C::kSlots;
            if (!wd.wait(&bars->k_full[st], slot_parity(kpar, st))) return;
            kpar ^= 1u << st;
            const uint32_t k_lo = kv_lo + st * (C::kKvTile >> 4);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!tile_uses(it, t, j)) continue;
                uint32_t& sc = t ? s_cnt1 : s_cnt0;
                if (sc > 0 && !wd.wait(&bars->s_free[t], (sc - 1) & 1)) return;
                tc_fence_after();
                const uint32_t a_lo = q_lo + t * (C::kQTile >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kAtomBytes + (kk & 3) * 32) >> 4;
                    umma_ss_lh(tmem + C::col_s(t), a_lo + off, d_hi, k_lo + off, d_hi, kIdesc,
                               kk > 0);
                }
                umma_commit(&bars->s_full[t]);
                ++sc;
            }
            umma_commit(&bars->kv_empty[st]);  // both tiles' S_t(j) have read K_j
        }
        umma_commit(&bars->q_empty);
        kv_cnt += 2 * m;
    }
}

// O_t (+)= P_t(j) V_j for every (j, t) of every item, P_t from shared memory.  The item's
// first PV_t overwrites O_t, so it first waits for the previous item's epilogue to have read
// O_t (o_free).
template <int D, bool kPaged>
__device__ void fwd_mma_pv(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem,
                           const Watchdog& wd, int n_items) {
    using C = FwdCfg<D>;
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, false, true);
    // A = P_t (K-major), B = V (MN-major: 64-wide d atoms kAtomBytes apart), as halves
    const uint64_t dp = sdesc_sw128(smem_u32(smem + C::kOffP), 16, 1024);
    const uint64_t dv = sdesc_sw128(smem_u32(smem + C::kOffKV), C::kAtomBytes, 1024);
    const uint32_t p_lo = static_cast<uint32_t>(dp), p_hi = static_cast<uint32_t>(dp >> 32);
    const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
    uint32_t kv_cnt = 0;
    uint32_t vpar = 0;                    // per-slot parity of the V blocks consumed so far
    uint32_t pv_cnt0 = 0, pv_cnt1 = 0;    // PV_t issued so far (== P_t consumed)
    uint32_t o_items0 = 0, o_items1 = 0;  // items in which tile t accumulated into O_t
    for (uint32_t rd = 0;;) {
        const int idx = fwd_take_item(bars, wd, rd);
        if (idx < 0) return;
        const Item it = load_item<kPaged>(p, idx);
        if (!it.any) continue;
        bool first0 = true, first1 = true;
        const int m = it.jhi - it.jlo;
        for (int i = 0; i < m; ++i) {
            const int j = it.jlo + i;
            const uint32_t n = kv_cnt + ring_pos_v(i, m);
            const uint32_t st = n % C::kSlots;
            if (!wd.wait(&bars->v_full[st], slot_parity(vpar, st))) return;
            vpar ^= 1u << st;
            const uint32_t b_lo = v_lo + st * (C::kKvTile >> 4);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!tile_uses(it, t, j)) continue;
                bool& first = t ? first1 : first0;
                const uint32_t oi = t ? o_items1 : o_items0;
                if (first && oi > 0 && !wd.wait(&bars->o_free[t], (oi - 1) & 1)) return;
                uint32_t& pc = t ? pv_cnt1 : pv_cnt0;
                if (!wd.wait(&bars->p_full[t], pc & 1)) return;
                tc_fence_after();
                const uint32_t a_lo = p_lo + t * (C::kPTile >> 4);
#pragma unroll
                for (int kk = 0; kk < kFwdBlockN / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kAtomBytes + (kk & 3) * 32) >> 4;
                    umma_ss_lh(tmem + C::col_o(t), a_lo + off, p_hi, b_lo + kk * (16 * 128 >> 4),
                               v_hi, kIdesc, (first && kk == 0) ? 0u : 1u);
                }
                umma_commit(&bars->pv_done[t]);
                ++pc;
                first = false;
            }
            umma_commit(&bars->kv_empty[st]);  // both tiles' PV_t(j) have read V_j
        }
        if (it.mma[0]) ++o_items0;
        if (it.mma[1]) ++o_items1;
        kv_cnt += 2 * m;
    }
}

// ---- softmax / correction / epilogue (eight warps per Q tile, 16 rows per warp) ----------
//
// Warp k of tile t (k = 0..7) owns rows 32 (k % 4) + 16 (k / 4) + [0, 16) of the tile (a warp
// may only address the TMEM lanes of its own quarter, 32 (warp % 4) + [0, 32)).  S is read
// with the 16-lane shape, so thread i holds rows i/4 and i/4 + 8 of those 16, two columns of
// every 8-column chunk: 64 values, the row max and sum are completed across the 4 threads of a
// quad, and P goes to shared memory with stmatrix.  Four such warps share each SM
// sub-partition, enough to overlap one warp's TMEM and shared-memory latency with another's
// exponentials.

// One Q tile's view of an item (the tile index is a run-time value: every softmax warp runs
// the same instruction stream, which keeps the instruction cache shared between them).
struct TileView {
    bool rows, mma;
    int tok0, imin, imax, lo, hi;
};

__device__ __forceinline__ TileView tile_view(const Item& it, int t) {
    TileView v;
    v.rows = t ? it.rows[1] : it.rows[0];
    v.mma = t ? it.mma[1] : it.mma[0];
    v.tok0 = t ? it.tok0[1] : it.tok0[0];
    v.imin = t ? it.imin[1] : it.imin[0];
    v.imax = t ? it.imax[1] : it.imax[0];
    v.lo = t ? it.lo[1] : it.lo[0];
    v.hi = t ? it.hi[1] : it.hi[0];
    return v;
}

// Address of the 16-byte unit u (8 bf16 columns) of row r in a 128-row tile stored as
// 128-byte-swizzled atoms of 64 columns.
__device__ __forceinline__ uint32_t sw128_unit(uint32_t base, int r, int u) {
    return base + (u >> 3) * (128 * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4);
}

template <int D, bool kPaged, bool kMods>
__device__ void fwd_softmax(const FwdParams& p, uint8_t* smem, FwdBars* bars, uint32_t tmem,
                            const Watchdog& wd, int n_items, int t, int k, int lane) {
    using C = FwdCfg<D>;
    uint64_t* const s_full = &bars->s_full[t];
    uint64_t* const s_free = &bars->s_free[t];
    uint64_t* const p_full = &bars->p_full[t];
    uint64_t* const pv_done = &bars->pv_done[t];
    uint64_t* const o_free = &bars->o_free[t];
    uint64_t* const epi_full = &bars->epi_full[t];
    uint64_t* const epi_free = &bars->epi_free[t];
    // Whole tiles leave through a TMA store of the O rows staged in P_t, issued by lane 0 of
    // the tile's warp 0 and left running; before P_t is written again the tile waits until that
    // store has read it (epi_free).  epi_cnt counts such stores, epi_pending marks one whose
    // read has not been waited for yet.
    uint32_t epi_cnt = 0;
    bool epi_pending = false;
    const int rbase = 32 * (k & 3) + 16 * (k >> 2);   // this warp's first row
    const int ra = rbase + (lane >> 2);                // this thread's rows ra and ra + 8
    const int cpair = 2 * (lane & 3);                  // its columns in each 8-column chunk
    const uint32_t tS = tmem + (static_cast<uint32_t>(rbase) << 16) + C::col_s(t);
    const uint32_t tO = tmem + (static_cast<uint32_t>(rbase) << 16) + C::col_o(t);
    const uint32_t p_tile = smem_u32(smem + C::kOffP + t * C::kPTile);
    // stmatrix: this thread addresses row (lane % 8) of matrix lane / 8, where matrix m holds
    // rows rbase + 8 (m % 2) + [0, 8) of 8-column chunk (base chunk + m / 2)
    const int st_row = rbase + 8 * ((lane >> 3) & 1) + (lane & 7);
    const int st_dc = lane >> 4;
    // Its row address for 8-column chunk u = 2 c + st_dc (c = 0..7) is
    // st_addr[c % 4] + (c / 4) * atom: unit (u % 8) ^ (row % 8) of atom u / 8.
    uint32_t st_addr[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_addr[c] = p_tile + st_row * 128 + ((((2 * c + st_dc) ^ lane) & 7) << 4);
    // log2(e) times what turns an S value into a logit: the scale, or c where a softcap has
    // made S tanh(scale S / c)
    const bool capped = kMods && p.softcap > 0.f;
    const float sl2 = capped ? p.softcap * kLog2e : p.scale_log2;
    // ALiBi biases are added to S in S's own units (the logit over the scale, or over c), and
    // for causal attention every visible key lies at or before the query's position, so the
    // bias is linear in the key: slope (key - pos)
    const float alibi_unit = capped ? 1.f / p.softcap : 1.f / p.scale;
    const bool alibi_linear = p.causal || p.wr == 0;
    const uint64_t sl2x2 = f2_make(sl2, sl2);
    const int g = p.g;
    const int tile_rows = g * p.tpt;
    uint32_t blk = 0;  // blocks of tile t processed so far (== S_t consumed == P_t produced)
    uint32_t kv_cnt = 0;  // K/V ring slots filled for earlier items (locates paged V blocks)
    uint32_t vpar = 0;    // per-slot parity of the V blocks loaded for earlier items (paged)
    for (uint32_t rd = 0;;) {
        const int idx = fwd_take_item_warp(bars, wd, rd, lane);
        if (idx < 0) break;
        const Item it = load_item<kPaged>(p, idx);
        const uint32_t kv_base = kv_cnt;
        const uint32_t vpar_item = vpar;
        if (it.any) {
            const int m = it.jhi - it.jlo;
            kv_cnt += 2 * m;
            if constexpr (kPaged)
                for (int i = 0; i < m; ++i) vpar ^= 1u << ((kv_base + ring_pos_v(i, m)) % C::kSlots);
        }
        const TileView tv = tile_view(it, t);
        if (!tv.rows) continue;
        // this thread's rows ra and ra + 8; packed row r is token tok0 + r / g, head kvh g + r % g
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;  // l: this thread's part
        // ALiBi: the rows' slopes and bottom-right key positions
        float slope_a = 0.f, slope_b = 0.f, pos_a = 0.f, pos_b = 0.f;
        if constexpr (kMods) {
            if (p.alibi != nullptr) {
                slope_a = p.alibi[it.kvh * g + ra % g] * alibi_unit;
                slope_b = p.alibi[it.kvh * g + (ra + 8) % g] * alibi_unit;
                pos_a = static_cast<float>(tv.tok0 + ra / g + it.Lk - it.Lq);
                pos_b = static_cast<float>(tv.tok0 + (ra + 8) / g + it.Lk - it.Lq);
            }
        }
        // Blocks needing the element mask are a prefix and a suffix of [lo, hi) (left window
        // edge; diagonal, right window edge, ragged end): the rest, [full_lo, full_hi), is
        // found once per item.
        int full_lo = tv.lo, full_hi = tv.hi;
        while (full_lo < full_hi && kv_block_masked(full_lo, tv.imin, tv.imax, it.Lq, it.Lk,
                                                    kFwdBlockN, p.causal, p.wl, p.wr))
            ++full_lo;
        while (full_hi > full_lo && kv_block_masked(full_hi - 1, tv.imin, tv.imax, it.Lq, it.Lk,
                                                    kFwdBlockN, p.causal, p.wl, p.wr))
            --full_hi;
        if (tv.mma) {
            for (int j = tv.lo; j < tv.hi; ++j) {
                if (!__all_sync(0xffffffffu, wd.wait(s_full, blk & 1))) return;
                tc_fence_after();
                uint32_t s[64];
                tmem_ld16x256_x8(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld16x256_x8(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_wait_ld();
                // S_t is in registers: the tensor core may overwrite it with S_t(j+1)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                // per-row constants of this block added to the logits in log2 units (ALiBi)
                float ca = 0.f, cb = 0.f;    // this thread's columns
                float qa = 0.f, qb = 0.f;    // S-unit shift of its columns to the block start
                float ra0 = 0.f, rb0 = 0.f;  // the rows' constants at the block start
                if constexpr (kMods) {
                    // softcap: S -> tanh(scale S / c), c applied through sl2; then the ALiBi
                    // bias; the element mask below comes after them
                    if (capped) {
                        const float ku = softcap_ku(p.scale, p.softcap);
                        const uint64_t ku2 = f2_make(ku, ku);
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            float s0 = __uint_as_float(s[c]), s1 = __uint_as_float(s[c + 1]);
                            softcap_tanh2(s0, s1, ku2);
                            s[c] = __float_as_uint(s0);
                            s[c + 1] = __float_as_uint(s1);
                        }
                    }
                    if (p.alibi != nullptr && alibi_linear) {
                        // slope (key - pos) = slope (8 c + e) + slope (key0 - pos): one FFMA per
                        // score with a constant, and a per-row constant of the block
                        const float key0 = static_cast<float>(j * kFwdBlockN + cpair);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float o = static_cast<float>(8 * c + e);
                                s[4 * c + e] = __float_as_uint(fmaf(slope_a, o, __uint_as_float(s[4 * c + e])));
                                s[4 * c + 2 + e] =
                                    __float_as_uint(fmaf(slope_b, o, __uint_as_float(s[4 * c + 2 + e])));
                            }
                        }
                        ca = slope_a * (key0 - pos_a) * sl2;
                        cb = slope_b * (key0 - pos_b) * sl2;
                        // the four threads of a row hold columns key0 = block start + cpair:
                        // their maxima below are moved to the block start so the quad agrees
                        qa = slope_a * static_cast<float>(cpair);
                        qb = slope_b * static_cast<float>(cpair);
                        ra0 = slope_a * (static_cast<float>(j * kFwdBlockN) - pos_a) * sl2;
                        rb0 = slope_b * (static_cast<float>(j * kFwdBlockN) - pos_b) * sl2;
                    } else if (p.alibi != nullptr) {
                        // -slope |pos - key| with key = key0 + 8 c + e: (pos - key0) once per
                        // block, then one subtraction of a constant per score (all values are
                        // integers below 2^24, exact in fp32)
                        const float key0 = static_cast<float>(j * kFwdBlockN + cpair);
                        const float da = pos_a - key0, db = pos_b - key0;
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float o = static_cast<float>(8 * c + e);
                                s[4 * c + e] = __float_as_uint(
                                    fmaf(-slope_a, fabsf(da - o), __uint_as_float(s[4 * c + e])));
                                s[4 * c + 2 + e] = __float_as_uint(
                                    fmaf(-slope_b, fabsf(db - o), __uint_as_float(s[4 * c + 2 + e])));
                            }
                        }
                    }
                }
                if (j < full_lo || j >= full_hi) {
                    const int key0 = j * kFwdBlockN + cpair;
                    int kmin_a, kmax_a, kmin_b, kmax_b;
                    row_key_interval(tv.tok0 + ra / g, it.Lq, it.Lk, p.causal, p.wl, p.wr,
                                     kmin_a, kmax_a);
                    row_key_interval(tv.tok0 + (ra + 8) / g, it.Lq, it.Lk, p.causal, p.wl, p.wr,
                                     kmin_b, kmax_b);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = key0 + 8 * c + e;
                            if (key < kmin_a || key > kmax_a) s[4 * c + e] = __float_as_uint(-INFINITY);
                            if (key < kmin_b || key > kmax_b)
                                s[4 * c + 2 + e] = __float_as_uint(-INFINITY);
                        }
                    }
                }
                // row maxima: this thread's 32 values of each row (16 chunks of 4: chunks 0 and 1
                // start four chains, then chunks c and c + 1 for even c >= 2 join them), then across the quad
                float xa0 = fmaxf(__uint_as_float(s[0]), __uint_as_float(s[4]));
                float xa1 = fmaxf(__uint_as_float(s[1]), __uint_as_float(s[5]));
                float xb0 = fmaxf(__uint_as_float(s[2]), __uint_as_float(s[6]));
                float xb1 = fmaxf(__uint_as_float(s[3]), __uint_as_float(s[7]));
#pragma unroll
                for (int c = 2; c < 16; c += 2) {
                    xa0 = fmax3(xa0, __uint_as_float(s[4 * c]), __uint_as_float(s[4 * c + 4]));
                    xa1 = fmax3(xa1, __uint_as_float(s[4 * c + 1]), __uint_as_float(s[4 * c + 5]));
                    xb0 = fmax3(xb0, __uint_as_float(s[4 * c + 2]), __uint_as_float(s[4 * c + 6]));
                    xb1 = fmax3(xb1, __uint_as_float(s[4 * c + 3]), __uint_as_float(s[4 * c + 7]));
                }
                float mxa = fmaxf(xa0, xa1), mxb = fmaxf(xb0, xb1);
                if constexpr (kMods) {
                    mxa += qa;
                    mxb += qb;
                }
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
                float mba, mbb;
                if constexpr (kMods) {
                    mba = fmaf(mxa, sl2, ra0);
                    mbb = fmaf(mxb, sl2, rb0);
                } else {
                    mba = mxa * sl2;
                    mbb = mxb * sl2;
                }
                const bool need_a = mba > m_a + kRescaleThreshold;
                const bool need_b = mbb > m_b + kRescaleThreshold;
                const float mna = need_a ? mba : m_a, mnb = need_b ? mbb : m_b;
                const float alpha_a = need_a ? ex2_approx(m_a - mna) : 1.f;
                const float alpha_b = need_b ? ex2_approx(m_b - mnb) : 1.f;
                l_a *= alpha_a;
                l_b *= alpha_b;
                m_a = mna;
                m_b = mnb;
                const float ra_ref = (m_a == -INFINITY) ? 0.f : m_a;
                const float rb_ref = (m_b == -INFINITY) ? 0.f : m_b;
                uint64_t nma, nmb;
                if constexpr (kMods) {
                    nma = f2_make(ca - ra_ref, ca - ra_ref);
                    nmb = f2_make(cb - rb_ref, cb - rb_ref);
                } else {
                    nma = f2_make(-ra_ref, -ra_ref);
                    nmb = f2_make(-rb_ref, -rb_ref);
                }
                // P = exp2(s * scale*log2e - m): paired FFMA, MUFU ex2, paired sums
                uint64_t suma = 0, sumb = 0;
                uint32_t pka[16], pkb[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint64_t xa = f2_fma(f2_make(__uint_as_float(s[4 * c]), __uint_as_float(s[4 * c + 1])),
                                               sl2x2, nma);
                    const uint64_t xb = f2_fma(f2_make(__uint_as_float(s[4 * c + 2]), __uint_as_float(s[4 * c + 3])),
                                               sl2x2, nmb);
                    float a0, a1, b0, b1;
                    f2_split(xa, a0, a1);
                    f2_split(xb, b0, b1);
                    const float pa0 = ex2_approx(a0), pa1 = ex2_approx(a1);
                    const float pb0 = ex2_approx(b0), pb1 = ex2_approx(b1);
                    suma = f2_add(suma, f2_make(pa0, pa1));
                    sumb = f2_add(sumb, f2_make(pb0, pb1));
                    pka[c] = pack_bf16x2(pa0, pa1);
                    pkb[c] = pack_bf16x2(pb0, pb1);
                }
                {
                    float lo, hi;
                    f2_split(suma, lo, hi);
                    l_a += lo + hi;
                    f2_split(sumb, lo, hi);
                    l_b += lo + hi;
                }
                // Paged K/V: the last block's rows past the sequence end come from cache slots
                // nobody wrote; their P is 0 but 0 * NaN would still poison O, so this tile's
                // warps clear those V rows (whole rows: the swizzle only permutes within a row).
                if (kPaged && (j + 1) * kFwdBlockN > it.Lk) {
                    const int m = it.jhi - it.jlo;
                    uint32_t bits = vpar_item;  // V parities before V_j's load
                    for (int i = 0; i < j - it.jlo; ++i)
                        bits ^= 1u << ((kv_base + ring_pos_v(i, m)) % C::kSlots);
                    const uint32_t st = (kv_base + ring_pos_v(j - it.jlo, m)) % C::kSlots;
                    if (!__all_sync(0xffffffffu, wd.wait(&bars->v_full[st], slot_parity(bits, st))))
                        return;
                    const int valid = it.Lk - j * kFwdBlockN;
                    const uint32_t vslot = smem_u32(smem + C::kOffKV + st * C::kKvTile);
                    const int units = (kFwdBlockN - valid) * C::kHalves * 8;
                    for (int u = k * 32 + lane; u < units; u += 8 * 32) {
                        const int r = valid + u / (C::kHalves * 8);
                        const int hc = u % (C::kHalves * 8);
                        st_shared_v4(vslot + (hc >> 3) * C::kAtomBytes + r * 128 + (hc & 7) * 16,
                                     0u, 0u, 0u, 0u);
                    }
                }
                // PV_t of the previous block has finished reading P_t from shared memory and
                // accumulating into O_t.
                if (blk > 0) {
                    if (!__all_sync(0xffffffffu, wd.wait(pv_done, (blk - 1) & 1))) return;
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, need_a || need_b) && j > tv.lo) {
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[16];
                        tmem_ld16x256_x4(tO + 32 * cc, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            o[4 * c] = __float_as_uint(__uint_as_float(o[4 * c]) * alpha_a);
                            o[4 * c + 1] = __float_as_uint(__uint_as_float(o[4 * c + 1]) * alpha_a);
                            o[4 * c + 2] = __float_as_uint(__uint_as_float(o[4 * c + 2]) * alpha_b);
                            o[4 * c + 3] = __float_as_uint(__uint_as_float(o[4 * c + 3]) * alpha_b);
                        }
                        tmem_st16x256_x4(tO + 32 * cc, o);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                if (epi_pending) {
                    // the previous item's O store out of P_t must have read it
                    if (k == 0 && lane == 0) {
                        bulk_wait_group_read_all();
                        mbar_arrive(epi_free);
                    }
                    if (!__all_sync(0xffffffffu, wd.wait(epi_free, (epi_cnt - 1) & 1))) return;
                    epi_pending = false;
                }
                // P_t rows of this warp: chunks (2 cp, 2 cp + 1) x (rows ra, ra + 8) per stmatrix
#pragma unroll
                for (int cp = 0; cp < 8; ++cp)
                    stmatrix_x4(st_addr[cp & 3] + (cp >> 2) * C::kAtomBytes, pka[2 * cp],
                                pkb[2 * cp], pka[2 * cp + 1], pkb[2 * cp + 1]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                ++blk;
            }
            // Epilogue: full row sums, O / l from TMEM as bf16 staged through this warp's rows
            // of P_t (free once the last PV_t completed), then row-contiguous global stores.
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
            if (!__all_sync(0xffffffffu, wd.wait(pv_done, (blk - 1) & 1))) return;
            tc_fence_after();
            const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
            const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t o[32];
                tmem_ld16x256_x8(tO + 64 * cc, o);
                tmem_wait_ld();
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    const int c = 2 * cp;
                    stmatrix_x4(st_addr[cp] + cc * C::kAtomBytes,
                                pack_bf16x2(__uint_as_float(o[4 * c]) * inv_a,
                                            __uint_as_float(o[4 * c + 1]) * inv_a),
                                pack_bf16x2(__uint_as_float(o[4 * c + 2]) * inv_b,
                                            __uint_as_float(o[4 * c + 3]) * inv_b),
                                pack_bf16x2(__uint_as_float(o[4 * c + 4]) * inv_a,
                                            __uint_as_float(o[4 * c + 5]) * inv_a),
                                pack_bf16x2(__uint_as_float(o[4 * c + 6]) * inv_b,
                                            __uint_as_float(o[4 * c + 7]) * inv_b));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            if (tv.tok0 + p.tpt <= it.Lq) {
                // Every packed row of the tile is a row of this sequence: one TMA store per
                // 64 columns writes the tile's g * tpt rows, asynchronously.
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(epi_full);
                if (k == 0) {
                    if (!__all_sync(0xffffffffu, wd.wait(epi_full, epi_cnt & 1))) return;
                    if (lane == 0) {
                        if (ATTN_IN_BOUNDS(it.q0 + tv.tok0 >= 0 && it.q0 + tv.tok0 + p.tpt <= p.total_q &&
                                               (it.kvh + 1) * g <= p.Hq,
                                           p.status)) {
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_store_3d(&p.tm_o, smem + C::kOffP + t * C::kPTile + h * C::kAtomBytes,
                                             h * 64, it.kvh * g, it.q0 + tv.tok0);
                        }
                        bulk_commit_group();
                    }
                }
                ++epi_cnt;
                epi_pending = true;
            } else if constexpr (!kPaged && !kMods) {
                // each store instruction writes whole rows: 32 / (D / 8) rows of D / 8 16-byte
                // units; packed row r is token r / g, head r % g (the quotient taken in fp32:
                // (r + 1/2) / g is at least 1/(2 g) away from an integer, far beyond the error)
                constexpr int kRowUnits = D / 8;
                constexpr int kRowsPerPass = 32 / kRowUnits;
                const int u = lane % kRowUnits;
                const float inv_g = 1.f / static_cast<float>(g);
#pragma unroll
                for (int v = 0; v < 16 / kRowsPerPass; ++v) {
                    const int r = rbase + v * kRowsPerPass + lane / kRowUnits;
                    const int rt = static_cast<int>((static_cast<float>(r) + 0.5f) * inv_g);
                    const int tok = tv.tok0 + rt;
                    if (r < tile_rows && tok < it.Lq) {
                        const int head = it.kvh * g + (r - rt * g);
                        uint4* dst = reinterpret_cast<uint4*>(
                            p.out + (static_cast<size_t>(it.q0 + tok) * p.Hq + head) * D);
                        if (ATTN_IN_BOUNDS(it.q0 + tok < p.total_q && head < p.Hq, p.status))
                            dst[u] = ld_shared_v4(sw128_unit(p_tile, r, u));
                    }
                }
            } else {
                // two threads per row: row rbase + lane / 2, units of half (lane % 2).  The
                // paged and modifier instances keep this layout: with their larger live state
                // the per-row index arithmetic above cost them more than the wider stores
                // saved (3-4% measured).
                constexpr int kUnits = D / 16;
                const int r = rbase + (lane >> 1);
                const int tok = tv.tok0 + r / g;
                if (r < tile_rows && tok < it.Lq) {
                    const int head = it.kvh * g + r % g;
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.out + (static_cast<size_t>(it.q0 + tok) * p.Hq + head) * D);
                    if (ATTN_IN_BOUNDS(it.q0 + tok < p.total_q && head < p.Hq, p.status)) {
#pragma unroll
                        for (int v = 0; v < kUnits; ++v) {
                            const int u = (lane & 1) * kUnits + v;
                            dst[u] = ld_shared_v4(sw128_unit(p_tile, r, u));
                        }
                    }
                }
            }
            __syncwarp();  // staging reads done before this warp's next P_t stores
        } else {
            // no visible key at all: O = 0 (each thread of the quad writes D/4 columns)
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = ra + 8 * h;
                const int tok = tv.tok0 + r / g;
                if (r < tile_rows && tok < it.Lq) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.out + (static_cast<size_t>(it.q0 + tok) * p.Hq + it.kvh * g + r % g) * D);
                    if (ATTN_IN_BOUNDS(it.q0 + tok < p.total_q && it.kvh * g + r % g < p.Hq, p.status)) {
#pragma unroll
                        for (int v = 0; v < D / 32; ++v) dst[(lane & 3) * (D / 32) + v] = z;
                    }
                }
            }
        }
        const int tok_a = tv.tok0 + ra / g, tok_b = tv.tok0 + (ra + 8) / g;
        const bool valid_a = ra < tile_rows && tok_a < it.Lq;
        const bool valid_b = ra + 8 < tile_rows && tok_b < it.Lq;
        if ((lane & 3) == 0) {
            if (valid_a && ATTN_IN_BOUNDS(it.q0 + tok_a < p.total_q, p.status))
                p.lse[static_cast<size_t>(it.kvh * g + ra % g) * p.total_q + it.q0 + tok_a] =
                    l_a > 0.f ? (m_a + __log2f(l_a)) * kLn2 : -INFINITY;
            if (valid_b && ATTN_IN_BOUNDS(it.q0 + tok_b < p.total_q, p.status))
                p.lse[static_cast<size_t>(it.kvh * g + (ra + 8) % g) * p.total_q + it.q0 + tok_b] =
                    l_b > 0.f ? (m_b + __log2f(l_b)) * kLn2 : -INFINITY;
        }
    }
}

template <int D, bool kPaged, bool kMods>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kSoftmaxWarps = 16;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&bars->k_full[i], 1);
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->s_free[t], kSoftmaxWarps / 2);
            mbar_init(&bars->p_full[t], kSoftmaxWarps / 2);
            mbar_init(&bars->pv_done[t], 1);
            mbar_init(&bars->o_free[t], kSoftmaxWarps / 2);
            mbar_init(&bars->epi_full[t], kSoftmaxWarps / 2);
            mbar_init(&bars->epi_free[t], 1);
            mbar_init(&bars->drain[t], 1);
        }
        for (uint32_t i = 0; i < kIdxRing; ++i) {
            mbar_init(&bars->idx_full[i], 1);
            mbar_init(&bars->idx_empty[i], kIdxReaders);
        }
        bars->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kSoftmaxWarps + 1) tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Watchdog wd{&bars->abort_flag, p.status};
    // (launched as a programmatic dependent of the work-list kernel: the set-up above overlaps
    // that kernel; the list is read only once it has finished)
    griddep_wait();
    const int n_items = p.header->n_items;

    // Registers: launched at 96 per thread (640 threads); warpgroup 4 (TMA, two MMA issuers,
    // one idle warp) drops to 64 and the four softmax warpgroups rise to 104:
    // 128 * 64 + 512 * 104 = 61440 = 640 * 96.
    if (warp >= kSoftmaxWarps) {
        regs_decrease<64>();
        if (warp == kSoftmaxWarps) {
            if (lane == 0) fwd_producer<D, kPaged>(p, smem, bars, wd, n_items);
        } else if (warp == kSoftmaxWarps + 1 || warp == kSoftmaxWarps + 2) {
            if (lane == 0) {
                const int w = warp - kSoftmaxWarps - 1;
                if (w == 0)
                    fwd_mma_s<D, kPaged>(p, smem, bars, tmem, wd, n_items);
                else
                    fwd_mma_pv<D, kPaged>(p, smem, bars, tmem, wd, n_items);
                // every tcgen05 op this thread issued has finished before TMEM is released
                umma_commit(&bars->drain[w]);
                drain_wait(&bars->drain[w], 0);
            }
        }
    } else {
        regs_increase<104>();
        fwd_softmax<D, kPaged, kMods>(p, smem, bars, tmem, wd, n_items, warp >> 3, warp & 7, lane);
        // the output stores this thread issued have completed before the CTA's memory goes
        if ((warp & 7) == 0 && lane == 0) bulk_wait_group_all();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kSoftmaxWarps + 1) {
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

// Keys of sequence b: the contiguous K/V's range, or the cached prefix plus the new tokens.
__device__ __forceinline__ int seq_keys(const FwdPrepParams& p, int b) {
    return p.cache_seqlens != nullptr ? p.cache_seqlens[b] + (p.cu_q[b + 1] - p.cu_q[b])
                                      : p.cu_k[b + 1] - p.cu_k[b];
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
    griddep_launch_dependents();  // the forward kernel may set up while the list is built
    if (tid == 0) err = 0;
    __syncthreads();
    // 1. the sequence boundaries must describe rows inside the tensors
    for (int b = tid; b < p.batch; b += blockDim.x) {
        const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
        if (q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.max_seqlen_q) err = 1;
        if (p.cache_seqlens != nullptr) {
            const int ctx = p.cache_seqlens[b];
            if (ctx < 0 || static_cast<long long>(ctx) + (q1 - q0) > p.max_keys) err = 1;
        } else {
            const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
            if (k0 < 0 || k1 < k0 || k1 > p.total_k || k1 - k0 > p.max_seqlen_k) err = 1;
        }
    }
    __syncthreads();
    if (err) {
        if (tid == 0) {
            atomicOr(p.status, kStatusBounds);
            p.header->n_items = 0;
            p.header->n_pairs = 0;
            p.header->next_item = 0;
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
            p.header->next_item = 0;
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
        const int cost = item_cost(p, p.cu_q[b + 1] - p.cu_q[b], seq_keys(p, b), m);
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
        const int cost = item_cost(p, p.cu_q[b + 1] - p.cu_q[b], seq_keys(p, b), m);
        const int slot = atomicAdd(&hist[kPrepBins - 1 - min(cost, kPrepBins - 1)], 1);
        // groups of heads_per_group KV heads, one after the other; inside a group the pairs
        // longest-first, each pair's heads side by side
        for (int h = 0; h < p.Hkv; ++h) {
            const int h0 = h - h % p.heads_per_group;
            const int width = min(p.heads_per_group, p.Hkv - h0);
            p.items[static_cast<size_t>(n_pairs) * h0 + static_cast<size_t>(slot) * width +
                    (h - h0)] = make_int4(b, h, m, cost);
        }
    }
    if (tid == 0) {
        p.header->n_pairs = n_pairs;
        p.header->n_items = n_pairs * p.Hkv;
        p.header->next_item = 0;
    }
}

}  // namespace

int fwd_smem_bytes(int head_dim) {
    return head_dim == 128 ? FwdCfg<128>::kSmem : FwdCfg<64>::kSmem;
}

cudaError_t configure_fwd_kernels() {
    const cudaFuncAttribute smem = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<128, false, false>, smem, FwdCfg<128>::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<64, false, false>, smem, FwdCfg<64>::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<128, true, false>, smem, FwdCfg<128>::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<64, true, false>, smem, FwdCfg<64>::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<128, false, true>, smem, FwdCfg<128>::kSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<64, false, true>, smem, FwdCfg<64>::kSmem);
    return e;
}

cudaError_t launch_fwd_prepare(const FwdPrepParams& p, cudaStream_t stream) {
    fwd_prepare_kernel<<<1, kPrepThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// The forward kernel goes out as a programmatic dependent of the work-list kernel just before
// it: its CTAs initialise barriers and TMEM while the list is built (griddep_wait in the kernel).
template <int D, bool kPaged, bool kMods>
cudaError_t launch_fwd_instance(const FwdParams& p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFwdThreads);
    cfg.dynamicSmemBytes = FwdCfg<D>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_kernel<D, kPaged, kMods>, p);
}

// K/V through block_table when p.block_table is set, else contiguous; the score-modifier
// instance when softcap or ALiBi is requested (contiguous K/V only).
cudaError_t launch_fwd(const FwdParams& p, int head_dim, int grid, cudaStream_t stream) {
    const bool paged = p.block_table != nullptr;
    const bool mods = p.softcap > 0.f || p.alibi != nullptr;
    if (paged && mods) return cudaErrorInvalidValue;
    if (head_dim == 128) {
        if (paged) return launch_fwd_instance<128, true, false>(p, grid, stream);
        if (mods) return launch_fwd_instance<128, false, true>(p, grid, stream);
        return launch_fwd_instance<128, false, false>(p, grid, stream);
    }
    if (paged) return launch_fwd_instance<64, true, false>(p, grid, stream);
    if (mods) return launch_fwd_instance<64, false, true>(p, grid, stream);
    return launch_fwd_instance<64, false, false>(p, grid, stream);
}

}  // namespace attn
