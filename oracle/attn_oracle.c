/*
 * attn_oracle.c -- the oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header, table or
 * helper with the CUDA path and includes nothing from it.
 *
 * It is the plain definition, written out in fp64, and deliberately slow:
 *
 *   "Attention kernels: FlashAttention and PagedAttention" (arganzheng.life), section 二.1-二.2:
 *     for one head, S = scale * Q K^T, P = softmax(S) row-wise, O = P V, with S and P
 *     materialised.  Here every query row materialises its full row of S and of P
 *     (Lk doubles each) before O is formed; nothing is tiled, fused or reordered.
 *   same page, section 四.3: the per-row log-sum-exp L = m + log(sum exp(s - m)), natural log.
 *   "04 · FA4 (CuTeDSL) and engineering interfaces" (llm-infra-atlas), sections 4-6:
 *     varlen batches through cu_seqlens prefix sums (section 4), query head h reads kv head
 *     h / (Hq/Hkv) (section 5), paged K/V through block_table (section 6.1), split-KV partials
 *     merged by LSE (section 6.2), causal aligned bottom-right for the kv-cache call
 *     (section 6.2) and the sliding window [i - w_left, i + w_right] (section 7 table).
 *
 * Readings where the pages are silent or disagree:
 *   - causal is aligned bottom-right everywhere: key j is visible to query i iff
 *     j <= i + (Lk - Lq) (+ w_right when not causal); this equals top-left when Lq == Lk;
 *   - window follows the API's (w_left, w_right) pair; -1 means unbounded on that side;
 *     causal forces w_right = 0;
 *   - a row with no visible key has O = 0 and LSE = -inf (no epsilon anywhere);
 *   - an empty split has LSE = -inf and weight 0 in the merge.
 *
 * Inputs are either fp64 (dtype 0) or bf16 bit patterns (dtype 1); bf16 is widened to fp64
 * exactly.  All arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F64 0
#define ORACLE_BF16 1

typedef struct {
    long long flops;       /* 2d per visible (query, key) pair for QK^T + 2d for PV */
    long long s_elems;     /* elements of S materialised (written once, read once by softmax) */
    long long p_elems;     /* elements of P materialised (written once, read once by PV) */
    long long qkvo_bytes;  /* bf16 bytes of Q, K, V read once and O written once */
} oracle_counts_t;

/* ---- element access ------------------------------------------------------------------ */

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Copy n consecutive elements starting at element index idx into dst as fp64. */
static void load_row(const void* base, int dtype, int64_t idx, int n, double* dst) {
    if (dtype == ORACLE_F64) {
        const double* p = (const double*)base + idx;
        for (int e = 0; e < n; ++e) dst[e] = p[e];
    } else {
        const uint16_t* p = (const uint16_t*)base + idx;
        for (int e = 0; e < n; ++e) dst[e] = bf16_to_f64(p[e]);
    }
}

/* ---- the visibility rule -------------------------------------------------------------- */

/* Is key j visible to query row i of a sequence with Lq queries and Lk keys?
 * Bottom-right alignment: query i sits at absolute key position i + (Lk - Lq). */
int oracle_allowed(long long i, long long j, long long Lq, long long Lk, int causal,
                   int window_left, int window_right) {
    if (j < 0 || j >= Lk || i < 0 || i >= Lq) return 0;
    long long pos = i + (Lk - Lq);
    int wr = causal ? 0 : window_right;
    if (wr >= 0 && j > pos + wr) return 0;
    if (window_left >= 0 && j < pos - window_left) return 0;
    return 1;
}

/* ---- one query row of standard attention ---------------------------------------------- */

/*
 * Materialise one row of S and P for query vector qrow over the keys whose element offsets
 * are koff[0..Lk) (the same offsets index V), then form O and the row's LSE.
 * vis[j] != 0 marks visible keys.  s_row and p_row are caller scratch of Lk doubles.
 */
/* Optional score modifiers ("04 · FA4 ...", section 7): softcap s -> c tanh(s / c) of the
 * scaled score, then the ALiBi bias -slope |pos - j| with pos the query's key position. */
typedef struct {
    double softcap;  /* 0: off */
    double slope;    /* 0: no ALiBi */
    int64_t pos;
} score_mod_t;

static void attention_row(const double* qrow, const void* k, const void* v, int dtype,
                          const int64_t* koff, const unsigned char* vis, int64_t Lk, int d,
                          double scale, double* s_row, double* p_row, double* kbuf,
                          double* out, double* lse, long long* pairs, const score_mod_t* mod) {
    /* S row: s_j = scale * <q, k_j> (then the modifiers) for visible keys, -inf otherwise. */
    long long visible = 0;
    for (int64_t j = 0; j < Lk; ++j) {
        if (!vis[j]) { s_row[j] = -INFINITY; continue; }
        load_row(k, dtype, koff[j], d, kbuf);
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += qrow[e] * kbuf[e];
        s_row[j] = scale * acc;
        if (mod) {
            if (mod->softcap > 0.0) s_row[j] = mod->softcap * tanh(s_row[j] / mod->softcap);
            if (mod->slope != 0.0) s_row[j] -= mod->slope * fabs((double)(mod->pos - j));
        }
        ++visible;
    }
    if (pairs) *pairs += visible;
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (visible == 0) {          /* no visible key: O = 0, LSE = -inf */
        for (int64_t j = 0; j < Lk; ++j) p_row[j] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* P row: exp(s - m) / sum exp(s - m). */
    double m = -INFINITY;
    for (int64_t j = 0; j < Lk; ++j) if (s_row[j] > m) m = s_row[j];
    double denom = 0.0;
    for (int64_t j = 0; j < Lk; ++j) {
        p_row[j] = vis[j] ? exp(s_row[j] - m) : 0.0;
        denom += p_row[j];
    }
    for (int64_t j = 0; j < Lk; ++j) p_row[j] /= denom;
    /* O row: sum_j P_j v_j. */
    for (int64_t j = 0; j < Lk; ++j) {
        if (p_row[j] == 0.0) continue;
        load_row(v, dtype, koff[j], d, kbuf);
        for (int e = 0; e < d; ++e) out[e] += p_row[j] * kbuf[e];
    }
    *lse = m + log(denom);
}

/* Sequence index containing packed token t (cu has batch + 1 entries). */
static int find_seq(const int32_t* cu, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static int check_common(int batch, int Hq, int Hkv, int d) {
    if (batch < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

/* ---- prefill: every row, with the standard implementation's accounting ---------------- */

/*
 * q [total_q, Hq, d], k and v [total_k, Hkv, d]; out [total_q, Hq, d]; lse [Hq, total_q].
 * Sequence b owns query rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]).
 */
int oracle_attn_fwd(const void* q, const void* k, const void* v, int dtype,
                    const int32_t* cu_q, const int32_t* cu_k, int batch, int Hq, int Hkv,
                    int d, double scale, int causal, int window_left, int window_right,
                    double* out, double* lse, long long total_q, oracle_counts_t* counts) {
    if (check_common(batch, Hq, Hkv, d)) return -1;
    for (int b = 0; b < batch; ++b)
        if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -1;
    if (batch > 0 && cu_q[batch] > total_q) return -1;
    const int g = Hq / Hkv;
    long long flops = 0, s_el = 0, p_el = 0, qkvo = 0;
    const long long n_bh = (long long)batch * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : flops, s_el, p_el, qkvo)
    for (long long bh = 0; bh < n_bh; ++bh) {
        const int b = (int)(bh / Hq), h = (int)(bh % Hq), kvh = h / g;
        const int64_t Lq = cu_q[b + 1] - cu_q[b], Lk = cu_k[b + 1] - cu_k[b];
        int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (Lk > 0 ? Lk : 1));
        unsigned char* vis = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* qrow = (double*)malloc(sizeof(double) * d);
        double* kbuf = (double*)malloc(sizeof(double) * d);
        for (int64_t j = 0; j < Lk; ++j) koff[j] = ((int64_t)(cu_k[b] + j) * Hkv + kvh) * d;
        for (int64_t i = 0; i < Lq; ++i) {
            const int64_t t = cu_q[b] + i;
            for (int64_t j = 0; j < Lk; ++j)
                vis[j] = (unsigned char)oracle_allowed(i, j, Lq, Lk, causal, window_left,
                                                       window_right);
            load_row(q, dtype, (t * Hq + h) * d, d, qrow);
            long long pairs = 0;
            attention_row(qrow, k, v, dtype, koff, vis, Lk, d, scale, s_row, p_row, kbuf,
                          out + (t * Hq + h) * d, lse + (int64_t)h * total_q + t, &pairs, NULL);
            flops += 4LL * d * pairs;
            s_el += Lk;
            p_el += Lk;
        }
        qkvo += 2LL * d * (2 * Lq + 2 * Lk); /* Q and O rows, K and V rows, bf16 */
        free(koff); free(vis); free(s_row); free(p_row); free(qrow); free(kbuf);
    }
    if (counts) {
        counts->flops = flops;
        counts->s_elems = s_el;
        counts->p_elems = p_el;
        counts->qkvo_bytes = qkvo;
    }
    return 0;
}

/* ---- prefill: a chosen set of (packed token, query head) rows ------------------------- */

int oracle_attn_fwd_rows(const void* q, const void* k, const void* v, int dtype,
                         const int32_t* cu_q, const int32_t* cu_k, int batch, int Hq, int Hkv,
                         int d, double scale, int causal, int window_left, int window_right,
                         const int64_t* row_tok, const int32_t* row_head, long long nrows,
                         double* out, double* lse) {
    if (check_common(batch, Hq, Hkv, d) || batch == 0) return -1;
    const int g = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (long long r = 0; r < nrows; ++r) {
        const int64_t t = row_tok[r];
        const int h = row_head[r];
        if (t < cu_q[0] || t >= cu_q[batch] || h < 0 || h >= Hq) { bad |= 1; continue; }
        const int b = find_seq(cu_q, batch, t), kvh = h / g;
        const int64_t Lq = cu_q[b + 1] - cu_q[b], Lk = cu_k[b + 1] - cu_k[b];
        const int64_t i = t - cu_q[b];
        int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (Lk > 0 ? Lk : 1));
        unsigned char* vis = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* qrow = (double*)malloc(sizeof(double) * d);
        double* kbuf = (double*)malloc(sizeof(double) * d);
        for (int64_t j = 0; j < Lk; ++j) {
            koff[j] = ((int64_t)(cu_k[b] + j) * Hkv + kvh) * d;
            vis[j] = (unsigned char)oracle_allowed(i, j, Lq, Lk, causal, window_left,
                                                   window_right);
        }
        load_row(q, dtype, (t * Hq + h) * d, d, qrow);
        attention_row(qrow, k, v, dtype, koff, vis, Lk, d, scale, s_row, p_row, kbuf,
                      out + r * d, lse + r, NULL, NULL);
        free(koff); free(vis); free(s_row); free(p_row); free(qrow); free(kbuf);
    }
    return bad ? -1 : 0;
}

/* ---- merge of split partials ------------------------------------------------------------ */

/*
 * "Attention kernels: FlashAttention and PagedAttention", section 六.3: partials
 * (m_i, l_i, O_i) with O_i already normalised by l_i merge as
 *   m = max_i m_i,  l = sum_i l_i e^(m_i - m),  O = sum_i O_i l_i e^(m_i - m) / l.
 * A split with l_i == 0 (no visible key) contributes nothing.  Result LSE = m + log l.
 */
int oracle_merge(int nsplits, int d, const double* m_i, const double* l_i, const double* o_i,
                 double* out, double* lse) {
    double m = -INFINITY;
    for (int s = 0; s < nsplits; ++s)
        if (l_i[s] > 0.0 && m_i[s] > m) m = m_i[s];
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return 0; }
    double l = 0.0;
    for (int s = 0; s < nsplits; ++s)
        if (l_i[s] > 0.0) l += l_i[s] * exp(m_i[s] - m);
    for (int s = 0; s < nsplits; ++s) {
        if (!(l_i[s] > 0.0)) continue;
        const double w = l_i[s] * exp(m_i[s] - m) / l;
        for (int e = 0; e < d; ++e) out[e] += w * o_i[(int64_t)s * d + e];
    }
    *lse = m + log(l);
    return 0;
}

/* ---- decode over a paged KV cache ------------------------------------------------------- */

/*
 * q [batch, Hq, d] (one query per sequence); k_cache and v_cache
 * [num_pages, page_size, Hkv, d]; key j of sequence b lives in physical page
 * block_table[b * max_pages + j / page_size] at offset j % page_size
 * ("Attention kernels ...", section 六.1; "04 · FA4 ...", section 6.1).
 * All cache_seqlens[b] keys are visible (bottom-right causal with Lq = 1).
 *
 * num_splits == 0: one pass over all keys.  num_splits >= 1: split s takes keys
 * [s*C, min((s+1)*C, L)) with C = ceil(L / num_splits); each split materialises its own S and P
 * rows and yields (m_s, l_s, O_s); the splits are merged by oracle_merge.
 *
 * Rows are (b, h) pairs; rows_b == NULL means all batch*Hq rows in (b, h) order.
 * out [nrows, d], lse [nrows].  Returns -1 on an invalid page index or length.
 */
int oracle_decode(const void* q, const void* k_cache, const void* v_cache, int dtype,
                  const int32_t* cache_seqlens, const int32_t* block_table, int max_pages,
                  int page_size, int num_pages, int batch, int Hq, int Hkv, int d,
                  double scale, int num_splits, const int32_t* rows_b, const int32_t* rows_h,
                  long long nrows, double* out, double* lse) {
    if (check_common(batch, Hq, Hkv, d) || page_size <= 0 || num_splits < 0) return -1;
    const int g = Hq / Hkv;
    const long long n = rows_b ? nrows : (long long)batch * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (long long r = 0; r < n; ++r) {
        const int b = rows_b ? rows_b[r] : (int)(r / Hq);
        const int h = rows_b ? rows_h[r] : (int)(r % Hq);
        if (b < 0 || b >= batch || h < 0 || h >= Hq) { bad |= 1; continue; }
        const int kvh = h / g;
        const int64_t L = cache_seqlens[b];
        if (L < 0 || L > (int64_t)max_pages * page_size) { bad |= 1; continue; }
        int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (L > 0 ? L : 1));
        int page_bad = 0;
        for (int64_t j = 0; j < L; ++j) {
            const int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
            if (page < 0 || page >= num_pages) { page_bad = 1; koff[j] = 0; continue; }
            koff[j] = (((int64_t)page * page_size + j % page_size) * Hkv + kvh) * d;
        }
        if (page_bad) { bad |= 1; free(koff); continue; }
        double* qrow = (double*)malloc(sizeof(double) * d);
        double* kbuf = (double*)malloc(sizeof(double) * d);
        double* s_row = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
        double* p_row = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
        unsigned char* vis = (unsigned char*)malloc(L > 0 ? L : 1);
        load_row(q, dtype, ((int64_t)b * Hq + h) * d, d, qrow);
        if (num_splits == 0) {
            for (int64_t j = 0; j < L; ++j)
                vis[j] = (unsigned char)oracle_allowed(0, j, 1, L, 1, -1, -1);
            attention_row(qrow, k_cache, v_cache, dtype, koff, vis, L, d, scale, s_row, p_row,
                          kbuf, out + r * d, lse + r, NULL, NULL);
        } else {
            const int S = num_splits;
            const int64_t C = (L + S - 1) / S;
            double* m_i = (double*)malloc(sizeof(double) * S);
            double* l_i = (double*)malloc(sizeof(double) * S);
            double* o_i = (double*)malloc(sizeof(double) * S * d);
            for (int s = 0; s < S; ++s) {
                const int64_t j0 = (int64_t)s * C < L ? (int64_t)s * C : L;
                const int64_t j1 = j0 + C < L ? j0 + C : L;
                const int64_t n_s = j1 - j0;
                for (int64_t j = 0; j < n_s; ++j)
                    vis[j] = (unsigned char)oracle_allowed(0, j0 + j, 1, L, 1, -1, -1);
                double lse_s;
                attention_row(qrow, k_cache, v_cache, dtype, koff + j0, vis, n_s, d, scale,
                              s_row, p_row, kbuf, o_i + (int64_t)s * d, &lse_s, NULL, NULL);
                /* express the partial as (m_s, l_s) with O_s normalised */
                if (lse_s == -INFINITY) { m_i[s] = -INFINITY; l_i[s] = 0.0; }
                else {
                    double m = -INFINITY;
                    for (int64_t j = 0; j < n_s; ++j) if (s_row[j] > m) m = s_row[j];
                    double l = 0.0;
                    for (int64_t j = 0; j < n_s; ++j)
                        if (vis[j]) l += exp(s_row[j] - m);
                    m_i[s] = m;
                    l_i[s] = l;
                }
            }
            oracle_merge(S, d, m_i, l_i, o_i, out + r * d, lse + r);
            free(m_i); free(l_i); free(o_i);
        }
        free(koff); free(qrow); free(kbuf); free(s_row); free(p_row); free(vis);
    }
    return bad ? -1 : 0;
}

/*
 * Standard attention with the score modifiers of "04 · FA4 ...", section 7: softcap
 * (s -> c tanh(s / c) on the scaled score; c = 0 off) and ALiBi (a linear position bias,
 * here -slope_h |i + Lk - Lq - j|; slopes == NULL off), then the visibility mask and softmax.
 * Rows are (packed token, q head) pairs; rows_t == NULL means all total_q * Hq rows in
 * (token, head) order.  out [nrows, d], lse [nrows].
 */
int oracle_attn_fwd_mods(const void* q, const void* k, const void* v, int dtype,
                         const int32_t* cu_q, const int32_t* cu_k, int batch, int Hq, int Hkv,
                         int d, double scale, int causal, int wl, int wr, double softcap,
                         const double* slopes, const int64_t* rows_t, const int32_t* rows_h,
                         long long nrows, double* out, double* lse) {
    if (check_common(batch, Hq, Hkv, d) || softcap < 0.0) return -1;
    const int g = Hq / Hkv;
    const int64_t total_q = cu_q[batch];
    const long long n = rows_t ? nrows : total_q * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 8) reduction(| : bad)
    for (long long r = 0; r < n; ++r) {
        const int64_t t = rows_t ? rows_t[r] : r / Hq;
        const int h = rows_t ? rows_h[r] : (int)(r % Hq);
        if (t < 0 || t >= total_q || h < 0 || h >= Hq) { bad |= 1; continue; }
        const int b = find_seq(cu_q, batch, t);
        const int64_t i = t - cu_q[b];
        const int64_t Lq = (int64_t)cu_q[b + 1] - cu_q[b];
        const int64_t k0 = cu_k[b], Lk = (int64_t)cu_k[b + 1] - k0;
        const int kvh = h / g;
        double* qrow = (double*)malloc(sizeof(double) * d);
        double* kbuf = (double*)malloc(sizeof(double) * d);
        int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (Lk > 0 ? Lk : 1));
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* vis = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        load_row(q, dtype, (t * Hq + h) * d, d, qrow);
        for (int64_t j = 0; j < Lk; ++j) {
            koff[j] = ((k0 + j) * Hkv + kvh) * d;
            vis[j] = (unsigned char)oracle_allowed(i, j, Lq, Lk, causal, wl, wr);
        }
        score_mod_t mod;
        mod.softcap = softcap;
        mod.slope = slopes ? slopes[h] : 0.0;
        mod.pos = i + Lk - Lq;
        attention_row(qrow, k, v, dtype, koff, vis, Lk, d, scale, s_row, p_row, kbuf,
                      out + r * d, lse + r, NULL, &mod);
        free(qrow); free(kbuf); free(koff); free(s_row); free(p_row); free(vis);
    }
    return bad ? -1 : 0;
}

/* ---- backward pass ---------------------------------------------------------------------- */

/*
 * Gradients of L = sum(O * dO) for the standard attention of oracle_attn_fwd ("Attention
 * kernels ...", section 四.3: the backward recomputes S = Q K^T and P = exp(S - LSE), and with
 * D_i = rowsum(dO_i * O_i) forms dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = scale dS K,
 * dK = scale dS^T Q).  Written out per query row from the definition: the row's S, P and dP
 * are materialised, D_i = sum_j P_ij dP_ij (which equals dO_i . O_i), and the row's
 * contributions go to dQ_i, dK_j, dV_j.  A kv head's dK, dV sum the contributions of its g
 * query heads.  Parallel over (sequence, kv head), so no two threads touch one dK or dV row.
 * dq [total_q, Hq, d], dk / dv [total_k, Hkv, d], dsum (D) [Hq, total_q]; all fp64.
 */
int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
                    const int32_t* cu_q, const int32_t* cu_k, int batch, int Hq, int Hkv, int d,
                    double scale, int causal, int wl, int wr, double* dq, double* dk, double* dv,
                    double* dsum) {
    if (check_common(batch, Hq, Hkv, d)) return -1;
    const int g = Hq / Hkv;
    const int64_t total_q = cu_q[batch], total_k = cu_k[batch];
    for (int64_t i = 0; i < total_q * Hq * d; ++i) dq[i] = 0.0;
    for (int64_t i = 0; i < total_k * Hkv * d; ++i) { dk[i] = 0.0; dv[i] = 0.0; }
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < batch; ++b) {
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            const int64_t q0 = cu_q[b], k0 = cu_k[b];
            const int64_t Lq = cu_q[b + 1] - q0, Lk = cu_k[b + 1] - k0;
            if (Lq < 0 || Lk < 0) { bad |= 1; continue; }
            const int64_t n = Lk > 0 ? Lk : 1;
            double* qrow = (double*)malloc(sizeof(double) * d);
            double* dorow = (double*)malloc(sizeof(double) * d);
            double* kbuf = (double*)malloc(sizeof(double) * d);
            double* s_row = (double*)malloc(sizeof(double) * n);
            double* p_row = (double*)malloc(sizeof(double) * n);
            double* dp_row = (double*)malloc(sizeof(double) * n);
            for (int64_t i = 0; i < Lq; ++i) {
                for (int hh = 0; hh < g; ++hh) {
                    const int h = kvh * g + hh;
                    const int64_t t = q0 + i;
                    load_row(q, dtype, (t * Hq + h) * d, d, qrow);
                    load_row(dout, dtype, (t * Hq + h) * d, d, dorow);
                    /* S and P rows */
                    double m = -INFINITY;
                    for (int64_t j = 0; j < Lk; ++j) {
                        if (!oracle_allowed(i, j, Lq, Lk, causal, wl, wr)) { s_row[j] = -INFINITY; continue; }
                        load_row(k, dtype, ((k0 + j) * Hkv + kvh) * d, d, kbuf);
                        double acc = 0.0;
                        for (int e = 0; e < d; ++e) acc += qrow[e] * kbuf[e];
                        s_row[j] = scale * acc;
                        if (s_row[j] > m) m = s_row[j];
                    }
                    if (m == -INFINITY) {          /* no visible key: O = 0, no gradient */
                        dsum[(int64_t)h * total_q + t] = 0.0;
                        continue;
                    }
                    double denom = 0.0;
                    for (int64_t j = 0; j < Lk; ++j) {
                        p_row[j] = s_row[j] == -INFINITY ? 0.0 : exp(s_row[j] - m);
                        denom += p_row[j];
                    }
                    for (int64_t j = 0; j < Lk; ++j) p_row[j] /= denom;
                    /* dP row, D_i */
                    double D = 0.0;
                    for (int64_t j = 0; j < Lk; ++j) {
                        if (p_row[j] == 0.0) { dp_row[j] = 0.0; continue; }
                        load_row(v, dtype, ((k0 + j) * Hkv + kvh) * d, d, kbuf);
                        double acc = 0.0;
                        for (int e = 0; e < d; ++e) acc += dorow[e] * kbuf[e];
                        dp_row[j] = acc;
                        D += p_row[j] * acc;
                    }
                    dsum[(int64_t)h * total_q + t] = D;
                    /* dS = P (dP - D); dQ_i, dK_j, dV_j */
                    double* dqrow = dq + (t * Hq + h) * d;
                    for (int64_t j = 0; j < Lk; ++j) {
                        if (p_row[j] == 0.0) continue;
                        const double ds = p_row[j] * (dp_row[j] - D);
                        const int64_t kv = ((k0 + j) * Hkv + kvh) * d;
                        load_row(k, dtype, kv, d, kbuf);
                        for (int e = 0; e < d; ++e) dqrow[e] += scale * ds * kbuf[e];
                        for (int e = 0; e < d; ++e) {
                            dk[kv + e] += scale * ds * qrow[e];
                            dv[kv + e] += p_row[j] * dorow[e];
                        }
                    }
                }
            }
            free(qrow); free(dorow); free(kbuf); free(s_row); free(p_row); free(dp_row);
        }
    }
    return bad ? -1 : 0;
}

/* ---- chunked prefill over a paged cache, with KV append and rotary embedding ---------- */

/*
 * Round x to the nearest bf16 value, ties to even, straight from the fp64 value (no detour
 * through fp32, which could round twice).  bf16 keeps 8 significant bits and fp32's exponent
 * range; below 2^-126 its grid spacing is 2^-133.
 */
uint16_t oracle_f64_to_bf16(double x) {
    uint32_t u;
    float f;
    if (isnan(x)) return 0x7FC0u;
    if (x == 0.0) {
        f = (float)x;  /* keeps the sign of zero */
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    int e;
    (void)frexp(x, &e);                  /* |x| = m 2^e, 0.5 <= m < 1 */
    int q = e - 8;                       /* 8 significant bits: spacing 2^(e-8) */
    if (q < -133) q = -133;              /* bf16 subnormal spacing */
    double r = rint(ldexp(x, -q));       /* nearest integer, ties to even */
    r = ldexp(r, q);
    if (fabs(r) >= 0x1.0p128) r = copysign(INFINITY, x);   /* beyond the largest finite bf16 */
    f = (float)r;                        /* exact: r has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/*
 * Rotary position embedding of one d-vector x at table row pos: the first rot components are
 * rotated in rot/2 planes by the angles whose cosines and sines are the table row
 * (cosr[i], sinr[i]); components rot.. are left as they are.  Plane i pairs (x_i, x_{i+rot/2})
 * (rotate-half form) or (x_{2i}, x_{2i+1}) (interleaved form):
 *   (a, b) -> (a cos - b sin, a sin + b cos).
 */
static void rope_row(double* x, int rot, int interleaved, const double* cosr, const double* sinr) {
    const int half = rot / 2;
    for (int i = 0; i < half; ++i) {
        const int ia = interleaved ? 2 * i : i;
        const int ib = interleaved ? 2 * i + 1 : i + half;
        const double a = x[ia], b = x[ib];
        x[ia] = a * cosr[i] - b * sinr[i];
        x[ib] = a * sinr[i] + b * cosr[i];
    }
}

/* Store fp64 row src (d elements) at element index idx of a bf16 or fp64 array. */
static void store_row(void* base, int dtype, int64_t idx, int n, const double* src) {
    if (dtype == ORACLE_F64) {
        double* p = (double*)base + idx;
        for (int e = 0; e < n; ++e) p[e] = src[e];
    } else {
        uint16_t* p = (uint16_t*)base + idx;
        for (int e = 0; e < n; ++e) p[e] = oracle_f64_to_bf16(src[e]);
    }
}

/*
 * Chunked prefill against a paged cache ("Attention kernels ...", section 五.1 and its
 * chunked-prefill figure; "04 · FA4 ...", sections 6.1-6.2 for block_table, cache_seqlens and
 * the in-place append of new k, v with rotary embedding).  Sequence b has q_len_b new tokens
 * (cu_q) after ctx_b = cache_seqlens[b] cached ones.
 *   1. Every new token i of b sits at position ctx_b + i.  Its keys (rotated when rot_dim > 0)
 *      and values are written into k_cache / v_cache at that position through block_table
 *      (bf16 arrays store the value rounded to bf16).
 *   2. Every query row is rotated the same way (and rounded to bf16 for bf16 data).
 *   3. Query i of b attends, by the visibility rule with Lq = q_len_b and
 *      Lk = ctx_b + q_len_b (bottom-right aligned), over the cache's keys 0 .. Lk - 1.
 * k_cache, v_cache are updated in place.  Rows are (packed token, q head) pairs; rows_t ==
 * NULL means every total_q * Hq row in (token, head) order.  rot_cos, rot_sin are
 * [rot_rows, rot_dim / 2].  Returns -1 on an invalid argument, length or page index.
 */
int oracle_kvcache_prefill(const void* q, const void* k_new, const void* v_new, int dtype,
                           void* k_cache, void* v_cache, const int32_t* cache_seqlens,
                           const int32_t* block_table, int max_pages, int page_size,
                           int num_pages, const int32_t* cu_q, int batch, int Hq, int Hkv, int d,
                           const double* rot_cos, const double* rot_sin, int rot_dim,
                           int rot_rows, int interleaved, double scale, int causal, int wl,
                           int wr, const int64_t* rows_t, const int32_t* rows_h,
                           long long nrows, double* out, double* lse) {
    if (check_common(batch, Hq, Hkv, d) || page_size <= 0 || max_pages < 0) return -1;
    if (rot_dim < 0 || rot_dim > d || (rot_dim & 1) || (rot_dim > 0 && (!rot_cos || !rot_sin)))
        return -1;
    const int g = Hq / Hkv;
    const int64_t total_q = cu_q[batch];
    /* lengths, positions and pages */
    for (int b = 0; b < batch; ++b) {
        const int64_t ql = (int64_t)cu_q[b + 1] - cu_q[b];
        const int64_t ctx = cache_seqlens[b];
        if (ql < 0 || ctx < 0 || ctx + ql > (int64_t)max_pages * page_size) return -1;
        if (rot_dim > 0 && ctx + ql > rot_rows) return -1;
        for (int64_t j = 0; j < ctx + ql; ++j) {
            const int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
            if (page < 0 || page >= num_pages) return -1;
        }
    }
    /* 1. append the new keys (rotated) and values */
    double* buf = (double*)malloc(sizeof(double) * d);
    for (int b = 0; b < batch; ++b) {
        for (int64_t t = cu_q[b]; t < cu_q[b + 1]; ++t) {
            const int64_t pos = cache_seqlens[b] + (t - cu_q[b]);
            const int32_t page = block_table[(int64_t)b * max_pages + pos / page_size];
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                const int64_t dst = (((int64_t)page * page_size + pos % page_size) * Hkv + kvh) * d;
                const int64_t src = (t * Hkv + kvh) * d;
                load_row(k_new, dtype, src, d, buf);
                if (rot_dim > 0)
                    rope_row(buf, rot_dim, interleaved, rot_cos + pos * (rot_dim / 2),
                             rot_sin + pos * (rot_dim / 2));
                store_row(k_cache, dtype, dst, d, buf);
                load_row(v_new, dtype, src, d, buf);
                store_row(v_cache, dtype, dst, d, buf);
            }
        }
    }
    free(buf);
    /* 2-3. rotated queries against the updated cache */
    const long long n = rows_t ? nrows : total_q * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (long long r = 0; r < n; ++r) {
        const int64_t t = rows_t ? rows_t[r] : r / Hq;
        const int h = rows_t ? rows_h[r] : (int)(r % Hq);
        if (t < 0 || t >= total_q || h < 0 || h >= Hq) { bad |= 1; continue; }
        const int b = find_seq(cu_q, batch, t);
        const int64_t i = t - cu_q[b];
        const int64_t Lq = (int64_t)cu_q[b + 1] - cu_q[b];
        const int64_t Lk = cache_seqlens[b] + Lq;
        const int kvh = h / g;
        double* qrow = (double*)malloc(sizeof(double) * d);
        double* kbuf = (double*)malloc(sizeof(double) * d);
        int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (Lk > 0 ? Lk : 1));
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* vis = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        load_row(q, dtype, (t * Hq + h) * d, d, qrow);
        if (rot_dim > 0) {
            const int64_t pos = cache_seqlens[b] + i;
            rope_row(qrow, rot_dim, interleaved, rot_cos + pos * (rot_dim / 2),
                     rot_sin + pos * (rot_dim / 2));
            if (dtype == ORACLE_BF16)
                for (int e = 0; e < d; ++e) qrow[e] = bf16_to_f64(oracle_f64_to_bf16(qrow[e]));
        }
        for (int64_t j = 0; j < Lk; ++j) {
            const int32_t page = block_table[(int64_t)b * max_pages + j / page_size];
            koff[j] = (((int64_t)page * page_size + j % page_size) * Hkv + kvh) * d;
            vis[j] = (unsigned char)oracle_allowed(i, j, Lq, Lk, causal, wl, wr);
        }
        attention_row(qrow, k_cache, v_cache, dtype, koff, vis, Lk, d, scale, s_row, p_row, kbuf,
                      out + r * d, lse + r, NULL, NULL);
        free(qrow); free(kbuf); free(koff); free(s_row); free(p_row); free(vis);
    }
    return bad ? -1 : 0;
}

/* ---- the tiled method's traffic model (for the roofline discussion) -------------------- */

/*
 * "Attention kernels ...", section 三.3: with Q read once and O written once, and K and V
 * each read once per query block of Br rows, the HBM bytes of one head are
 * 2*N*d*2 (Q, O) + 2 * (N / Br) * N*d*2 (K, V re-reads), bf16.
 */
long long oracle_tiled_traffic_bytes(long long N, long long d, long long Br) {
    const long long blocks = (N + Br - 1) / Br;
    return 2 * N * d * 2 + 2 * blocks * N * d * 2;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- FP8 (e4m3) inputs ------------------------------------------------------------------- */

/*
 * "Attention kernels: FlashAttention and PagedAttention", section 四.2 (FlashAttention-3): the
 * FP8 forward feeds Q, K and V to the 8-bit MMA as e4m3 values with block-wise scales.  The
 * e4m3 format itself is the standard 8-bit float (OCP 8-bit floating point, E4M3): a sign bit,
 * 4 exponent bits with bias 7 and 3 mantissa bits; exponent field 0 holds the subnormals
 * (m / 8) 2^-6; exponent field 15 with mantissa 7 is NaN; there is no infinity, so the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_to_f64(int code) {
    const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * The e4m3 code nearest to x, ties to the code with the even mantissa, with magnitudes beyond
 * 448 saturated to 448 (a saturating conversion); NaN gives 0x7F.  A plain search over the
 * 127 non-negative finite codes, whose values increase with the code.
 */
int oracle_f64_to_e4m3(double x) {
    if (isnan(x)) return 0x7F;
    const int sign = signbit(x) ? 0x80 : 0;
    const double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_d = a;  /* distance to code 0 (value 0) */
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs(a - oracle_e4m3_to_f64(c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;
}

/* ---- FP8 quantization with block scales and the optional rotation ------------------------ */

/*
 * "Attention kernels: FlashAttention and PagedAttention", section 四.2 (FlashAttention-3): the
 * FP8 inputs carry one scale per block, and "incoherent processing" multiplies Q and K by the
 * same random orthogonal matrix (Q K^T is unchanged) to spread outliers before they are
 * rounded.  The orthogonal matrix taken here is the normalised Walsh-Hadamard matrix times a
 * diagonal of random signs, the usual construction of that kind; the signs are an input.
 *
 * Walsh-Hadamard transform of n = 2^k values in place (Sylvester order), fp32: stages
 * h = 1, 2, ..., n/2; in each, every pair (i, i + h) with i & h == 0 becomes
 * (x_i + x_{i+h}, x_i - x_{i+h}).
 */
static void fwht_f32(float* x, int n) {
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; ++i)
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/*
 * One block of n rows of d bf16 values (row-major bits) to e4m3 codes and one fp32 scale:
 *   1. optionally each row x -> H (signs * x) / sqrt(d) (fp32, 1/sqrt(d) rounded to fp32 once);
 *   2. amax = max |x| over the block; scale = amax / 448 in fp32 (1 for an all-zero block);
 *   3. code = the e4m3 code nearest to x * r with r = 448 / amax (fp32, formed once per block;
 *      1 for an all-zero block), ties to even, saturating.
 * Every fp32 operation is a single IEEE operation, so a device implementation doing the same
 * operations gets the same bits.
 */
int oracle_fp8_quantize_rows(const uint16_t* src, long long n, int d, const float* signs,
                             uint8_t* codes, float* scale) {
    if (n < 0 || d <= 0 || (d & (d - 1)) != 0) return -1;
    float* buf = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1) * (size_t)d);
    if (!buf) return -1;
    const float inv = (float)(1.0 / sqrt((double)d));
    float amax = 0.f;
    for (long long r = 0; r < n; ++r) {
        float* x = buf + r * d;
        for (int e = 0; e < d; ++e) x[e] = (float)bf16_to_f64(src[r * d + e]);
        if (signs) {
            for (int e = 0; e < d; ++e) x[e] = x[e] * signs[e];
            fwht_f32(x, d);
            for (int e = 0; e < d; ++e) x[e] = x[e] * inv;
        }
        for (int e = 0; e < d; ++e) amax = fabsf(x[e]) > amax ? fabsf(x[e]) : amax;
    }
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    const float rcp = amax > 0.f ? 448.f / amax : 1.f;
    for (long long i = 0; i < n * d; ++i) codes[i] = (uint8_t)oracle_f64_to_e4m3((double)(buf[i] * rcp));
    *scale = s;
    free(buf);
    return 0;
}
