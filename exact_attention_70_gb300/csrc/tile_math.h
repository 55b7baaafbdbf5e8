// tile_math.h -- integer work shared by the host and the kernels: which key blocks a block of
// query rows needs, which of them need an element-wise mask, and how query rows are packed.
//
// Visibility ("04 · FA4 (CuTeDSL) and engineering interfaces", section 6.2 and the section 7
// table; "Attention kernels: FlashAttention and PagedAttention", sections 七.2-七.3): query i
// of a sequence with Lq queries and Lk keys sits at key position p = i + Lk - Lq; key j < Lk is
// visible iff j <= p + wr (causal: wr = 0; wr < 0 and not causal: unbounded) and
// j >= p - wl (wl < 0: unbounded).
#pragma once

#ifndef __CUDACC__
#define TM_HD inline
#else
#define TM_HD __host__ __device__ __forceinline__
#endif

namespace attn {

struct KvRange {
    int lo, hi;  // half-open range of key blocks
};

// Key blocks of width bn holding a key visible to some query row in [i_min, i_max].
TM_HD KvRange kv_block_range(int i_min, int i_max, int Lq, int Lk, int bn, int causal, int wl,
                             int wr) {
    const int nblk = Lk > 0 ? (Lk + bn - 1) / bn : 0;
    const long long shift = static_cast<long long>(Lk) - Lq;
    const int right = causal ? 0 : wr;
    int hi = nblk;
    if (right >= 0) {
        const long long last_key = i_max + shift + right;  // right edge of the last row
        if (last_key < 0) {
            hi = 0;
        } else {
            const long long h = last_key / bn + 1;
            hi = h < nblk ? static_cast<int>(h) : nblk;
        }
    }
    int lo = 0;
    if (wl >= 0) {
        const long long first_key = i_min + shift - wl;  // left edge of the first row
        if (first_key > 0) {
            const long long l = first_key / bn;
            lo = l < nblk ? static_cast<int>(l) : nblk;
        }
    }
    if (lo > hi) lo = hi;
    return KvRange{lo, hi};
}

// Does key block j hold a key that some row in [i_min, i_max] must not see?
TM_HD bool kv_block_masked(int j, int i_min, int i_max, int Lq, int Lk, int bn, int causal,
                           int wl, int wr) {
    const long long k_first = static_cast<long long>(j) * bn;
    const long long k_last = k_first + bn - 1;
    if (k_last >= Lk) return true;  // ragged tail
    const long long shift = static_cast<long long>(Lk) - Lq;
    const int right = causal ? 0 : wr;
    if (right >= 0 && k_last > i_min + shift + right) return true;
    if (wl >= 0 && k_first < i_max + shift - wl) return true;
    return false;
}

// Visible key interval [kmin, kmax] of query row i (may be empty: kmin > kmax).
TM_HD void row_key_interval(int i, int Lq, int Lk, int causal, int wl, int wr, int& kmin,
                            int& kmax) {
    const long long p = static_cast<long long>(i) + Lk - Lq;
    const int right = causal ? 0 : wr;
    long long hi = Lk - 1;
    if (right >= 0 && p + right < hi) hi = p + right;
    long long lo = 0;
    if (wl >= 0 && p - wl > lo) lo = p - wl;
    if (hi < -1) hi = -1;
    if (lo > static_cast<long long>(Lk)) lo = Lk;
    kmin = static_cast<int>(lo);
    kmax = static_cast<int>(hi);
}

// Query rows of a prefill tile: 128 TMEM lanes hold tokens_per_tile(g) consecutive tokens of
// one sequence times the g query heads sharing a kv head (pack_gqa, "04 · FA4 ...",
// section 5): row r is token r / g, head kvh * g + r % g.
TM_HD int tokens_per_tile(int g) { return 128 / g; }

}  // namespace attn
