/*
 * hp_oracle.c -- fp64 CPU reference for shared-prefix (cascade) decode attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call this file.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * What it computes.  The cascade method is exact: splitting the keys at the
 * prefix boundary (or at every vertex of a prefix tree) and merging the parts
 * by their log-sum-exp reaches the attention of the unsplit key set (Hydragen,
 * "Attention Decomposition Across Subsequences", Eq. 5 and its proof in
 * Appendix A).  So the reference is the plain definition, evaluated in double
 * precision over the exact bf16 input values:
 *
 *     s_j   = scale * sum_i q_i k_{j,i}                     (scaled scores)
 *     LSE   = log sum_j exp(s_j)      (natural log, Hydragen's LSE(Q,K))
 *     O     = sum_j exp(s_j - LSE) v_j                        (SDP(Q,K,V))
 *
 * LSE is evaluated as m + log sum_j exp(s_j - m) with m = max_j s_j, the same
 * value written so that exp() cannot overflow.  An empty key set gives
 * O = 0 and LSE = -inf (its merge weight is exactly zero).
 *
 * The two-part merge follows Hydragen Eq. 5 in the max-subtracted form of its
 * combine_lse step; the chunk partial state (O, m, n) and its reduction follow
 * ChunkAttention Eq. 1 (partial_attn) and Eq. 2 (attn_reduce).
 *
 * Query head h reads KV head h / (Hq / Hkv) (consecutive query heads share a
 * KV head: the grouped-query reading of "each KV head serves its group of
 * query heads", shared-prefix KV caching blog, "Splitting attention at the
 * prefix boundary").
 *
 * Reduced-precision KV (Hydragen, "Implications and Future Directions": the
 * suffix pass stays memory-bound, and quantising the KV cache is the
 * complementary remedy).  A level may store its keys and values as 8-bit
 * E4M3 codes with one f32 scale per (page, KV head) for K and one for V: the
 * stored value is decode(code) * scale.  The oracle decodes every code by the
 * format's definition (hpo_e4m3_to_f64) and then evaluates the same plain
 * definition above in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32, so widening is exact. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * SDP over an explicit key list (the definition).
 * q: [d]; keys are given as row pointers into bf16 storage.
 * ------------------------------------------------------------------------- */
static void sdp_rows_bf16(int d, const double *q, int nk, const uint16_t *const *krow,
                          const uint16_t *const *vrow, double scale, double *o, double *lse,
                          double *s /* scratch [nk] */)
{
    int j, i;
    for (i = 0; i < d; ++i)
        o[i] = 0.0;
    if (nk == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (i = 0; i < d; ++i)
            acc += q[i] * bf16_to_f64(krow[j][i]);
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    double sum = 0.0;
    for (j = 0; j < nk; ++j)
        sum += exp(s[j] - m);
    double L = m + log(sum);
    for (j = 0; j < nk; ++j) {
        double w = exp(s[j] - L);
        for (i = 0; i < d; ++i)
            o[i] += w * bf16_to_f64(vrow[j][i]);
    }
    *lse = L;
}

/* SDP and LSE of dense fp64 matrices: Q [nq][d], K,V [nk][d] -> O [nq][d], lse [nq]. */
void hpo_sdp_f64(int nq, int nk, int d, const double *Q, const double *K, const double *V,
                 double scale, double *O, double *lse)
{
    int r;
#pragma omp parallel for schedule(dynamic, 1) if (nq > 8)
    for (r = 0; r < nq; ++r) {
        const double *q = Q + (size_t)r * d;
        double *o = O + (size_t)r * d;
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        int j, i;
        for (i = 0; i < d; ++i)
            o[i] = 0.0;
        if (nk == 0) {
            lse[r] = -INFINITY;
            free(s);
            continue;
        }
        double m = -INFINITY;
        for (j = 0; j < nk; ++j) {
            double acc = 0.0;
            for (i = 0; i < d; ++i)
                acc += q[i] * K[(size_t)j * d + i];
            s[j] = scale * acc;
            if (s[j] > m)
                m = s[j];
        }
        double sum = 0.0;
        for (j = 0; j < nk; ++j)
            sum += exp(s[j] - m);
        double L = m + log(sum);
        for (j = 0; j < nk; ++j) {
            double w = exp(s[j] - L);
            for (i = 0; i < d; ++i)
                o[i] += w * V[(size_t)j * d + i];
        }
        lse[r] = L;
        free(s);
    }
}

/* ---------------------------------------------------------------------------
 * Two-part merge (Hydragen Eq. 5, max-subtracted):
 *   M = max(L1, L2); w1 = exp(L1 - M); w2 = exp(L2 - M)
 *   O = (w1 O1 + w2 O2) / (w1 + w2);  L = M + log(w1 + w2)
 * Both parts empty (L1 = L2 = -inf) gives O = 0, L = -inf.
 * ------------------------------------------------------------------------- */
void hpo_merge(long n, int d, const double *O1, const double *L1, const double *O2,
               const double *L2, double *O, double *L)
{
    long r;
    for (r = 0; r < n; ++r) {
        int i;
        double a = L1[r], b = L2[r];
        if (a == -INFINITY && b == -INFINITY) {
            for (i = 0; i < d; ++i)
                O[r * d + i] = 0.0;
            L[r] = -INFINITY;
            continue;
        }
        double M = a > b ? a : b;
        double w1 = exp(a - M), w2 = exp(b - M);
        double den = w1 + w2;
        for (i = 0; i < d; ++i)
            O[r * d + i] = (w1 * O1[r * d + i] + w2 * O2[r * d + i]) / den;
        L[r] = M + log(den);
    }
}

/* ---------------------------------------------------------------------------
 * ChunkAttention partial state.
 * partial_attn (Eq. 1) for one query row against one chunk of c keys:
 *   W = scale * q K^T;  m = max W;  E = exp(W - m);  n = sum E;  o = E V
 * attn_reduce (Eq. 2) folds a chunk state into a running state (O, m, n):
 *   x = exp(m_c - max(m_c, m)); y = exp(m - max(m_c, m))
 *   O <- x o_c + y O;  n <- x n_c + y n;  m <- max(m_c, m)
 * The final output is O / n.  The running state starts at m = -inf (an empty
 * state), n = 0, O = 0.
 * ------------------------------------------------------------------------- */
void hpo_partial_attn(int d, int c, const double *q, const double *Kc, const double *Vc,
                      double scale, double *o, double *m_out, double *n_out)
{
    int j, i;
    double m = -INFINITY;
    double *w = (double *)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
    for (j = 0; j < c; ++j) {
        double acc = 0.0;
        for (i = 0; i < d; ++i)
            acc += q[i] * Kc[(size_t)j * d + i];
        w[j] = scale * acc;
        if (w[j] > m)
            m = w[j];
    }
    double n = 0.0;
    for (i = 0; i < d; ++i)
        o[i] = 0.0;
    for (j = 0; j < c; ++j) {
        double e = exp(w[j] - m);
        n += e;
        for (i = 0; i < d; ++i)
            o[i] += e * Vc[(size_t)j * d + i];
    }
    *m_out = m;
    *n_out = n;
    free(w);
}

void hpo_attn_reduce(int d, const double *o_c, double m_c, double n_c, double *O, double *m,
                     double *n)
{
    int i;
    if (m_c == -INFINITY)
        return; /* empty chunk: nothing to add */
    double mx = m_c > *m ? m_c : *m;
    double x = exp(m_c - mx);
    double y = (*m == -INFINITY) ? 0.0 : exp(*m - mx);
    for (i = 0; i < d; ++i)
        O[i] = x * o_c[i] + y * O[i];
    *n = x * n_c + y * *n;
    *m = mx;
}

/* ---------------------------------------------------------------------------
 * 8-bit E4M3 codes (the OCP 8-bit floating-point format E4M3, which has no
 * infinities): bit 7 is the sign s, bits 6..3 the exponent field e (bias 7),
 * bits 2..0 the mantissa field m.
 *   e = 0:               (-1)^s * 2^-6 * (m / 8)       (zero and subnormals)
 *   e = 1..15:           (-1)^s * 2^(e - 7) * (1 + m / 8)
 *   e = 15 and m = 7:    not a number (the largest finite value is 448)
 * ------------------------------------------------------------------------- */
double hpo_e4m3_to_f64(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

void hpo_e4m3_decode(long n, const uint8_t *codes, double *out)
{
    long i;
    for (i = 0; i < n; ++i)
        out[i] = hpo_e4m3_to_f64(codes[i]);
}

/* One key of a row's key list: its K and V rows (bf16, or E4M3 codes with the
 * scales of their page and KV head). */
typedef struct {
    const void *k, *v;
    double k_scale, v_scale;
    int e4m3;
} hpo_key;

static double key_elem(const void *row, int e4m3, double sc, int i)
{
    if (e4m3)
        return hpo_e4m3_to_f64(((const uint8_t *)row)[i]) * sc;
    return bf16_to_f64(((const uint16_t *)row)[i]);
}

/* SDP over an explicit key list of mixed storage (the definition, as in
 * sdp_rows_bf16, with each element decoded from its storage first). */
static void sdp_keys(int d, const double *q, int nk, const hpo_key *keys, double scale, double *o,
                     double *lse, double *s)
{
    int j, i;
    for (i = 0; i < d; ++i)
        o[i] = 0.0;
    if (nk == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (i = 0; i < d; ++i)
            acc += q[i] * key_elem(keys[j].k, keys[j].e4m3, keys[j].k_scale, i);
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    double sum = 0.0;
    for (j = 0; j < nk; ++j)
        sum += exp(s[j] - m);
    double L = m + log(sum);
    for (j = 0; j < nk; ++j) {
        double w = exp(s[j] - L);
        for (i = 0; i < d; ++i)
            o[i] += w * key_elem(keys[j].v, keys[j].e4m3, keys[j].v_scale, i);
    }
    *lse = L;
}

/* ---------------------------------------------------------------------------
 * Cascade attention over a level-by-level prefix tree stored in pages.
 *
 * Pool layout [page][Hkv][ps][d] bf16.  Level l has num_nodes[l] nodes, each
 * (seq_begin, seq_end, kv_len, page_off); node tokens t = 0..kv_len-1 sit at
 * page page_ids[l][page_off + t/ps], slot t%ps.  Sequence b's key list is the
 * concatenation over levels of the tokens of the node covering b.
 *
 * rows: n_rows pairs (b, h); outputs O [n_rows][d], lse [n_rows].
 * q: [B][Hq][d] bf16, dense.
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *k_pool;
    const uint16_t *v_pool;
    int page_size;
    int num_nodes;
    const int32_t *nodes; /* [num_nodes][4] */
    const int32_t *page_ids;
} hpo_level;

static int seq_keys(const hpo_level *lv, int num_levels, int Hkv, int d, int b, int kvh,
                    const uint16_t **krow, const uint16_t **vrow)
{
    int n = 0, l, k, t;
    for (l = 0; l < num_levels; ++l) {
        const hpo_level *L = &lv[l];
        for (k = 0; k < L->num_nodes; ++k) {
            const int32_t *nd = L->nodes + 4 * k;
            if (b < nd[0] || b >= nd[1])
                continue;
            for (t = 0; t < nd[2]; ++t) {
                long page = L->page_ids[nd[3] + t / L->page_size];
                long slot = t % L->page_size;
                size_t off = (((size_t)page * Hkv + kvh) * L->page_size + slot) * d;
                if (krow) {
                    krow[n] = L->k_pool + off;
                    vrow[n] = L->v_pool + off;
                }
                ++n;
            }
            break; /* nodes of one level cover disjoint ranges */
        }
    }
    return n;
}

static void load_q(int d, const uint16_t *q, double *qd)
{
    int i;
    for (i = 0; i < d; ++i)
        qd[i] = bf16_to_f64(q[i]);
}

int hpo_cascade(int B, int Hq, int Hkv, int d, double scale, const uint16_t *q,
                int num_levels, const uint16_t *const *k_pools, const uint16_t *const *v_pools,
                const int32_t *page_sizes, const int32_t *num_nodes,
                const int32_t *const *nodes, const int32_t *const *page_ids, long n_rows,
                const int32_t *rows, double *O, double *lse)
{
    long r;
    int l, G;
    hpo_level *lv;
    if (Hkv <= 0 || Hq % Hkv != 0 || num_levels < 0)
        return -1;
    for (r = 0; r < n_rows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= Hq)
            return -2;
    G = Hq / Hkv;
    lv = (hpo_level *)malloc(sizeof(hpo_level) * (size_t)(num_levels > 0 ? num_levels : 1));
    for (l = 0; l < num_levels; ++l) {
        lv[l].k_pool = k_pools[l];
        lv[l].v_pool = v_pools[l];
        lv[l].page_size = page_sizes[l];
        lv[l].num_nodes = num_nodes[l];
        lv[l].nodes = nodes[l];
        lv[l].page_ids = page_ids[l];
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n_rows; ++r) {
        int b = rows[2 * r], h = rows[2 * r + 1];
        int kvh = h / G;
        int nk = seq_keys(lv, num_levels, Hkv, d, b, kvh, NULL, NULL);
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nk + 1));
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nk + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        seq_keys(lv, num_levels, Hkv, d, b, kvh, krow, vrow);
        load_q(d, q + ((size_t)b * Hq + h) * d, qd);
        sdp_rows_bf16(d, qd, nk, krow, vrow, scale, O + (size_t)r * d, lse + r, s);
        free(krow);
        free(vrow);
        free(s);
        free(qd);
    }
    free(lv);
    return 0;
}

/* Cascade attention over a tree whose levels may store E4M3 codes:
 * kv_dtypes[l] = 0 for bf16 pools, 1 for E4M3 pools ([page][Hkv][ps][d]
 * bytes) with f32 scales k_scales[l][page * Hkv + kvh] (and v_scales[l]
 * likewise).  Otherwise as hpo_cascade. */
int hpo_cascade_q(int B, int Hq, int Hkv, int d, double scale, const uint16_t *q, int num_levels,
                  const void *const *k_pools, const void *const *v_pools, const int32_t *kv_dtypes,
                  const float *const *k_scales, const float *const *v_scales, const int32_t *page_sizes,
                  const int32_t *num_nodes, const int32_t *const *nodes, const int32_t *const *page_ids,
                  long n_rows, const int32_t *rows, double *O, double *lse)
{
    long r;
    int G;
    if (Hkv <= 0 || Hq % Hkv != 0 || num_levels < 0)
        return -1;
    for (r = 0; r < n_rows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= Hq)
            return -2;
    G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n_rows; ++r) {
        int b = rows[2 * r], h = rows[2 * r + 1];
        int kvh = h / G;
        int nk = 0, l, k, t;
        for (l = 0; l < num_levels; ++l)
            for (k = 0; k < num_nodes[l]; ++k) {
                const int32_t *nd = nodes[l] + 4 * k;
                if (b >= nd[0] && b < nd[1]) {
                    nk += nd[2];
                    break;
                }
            }
        hpo_key *keys = (hpo_key *)malloc(sizeof(hpo_key) * (size_t)(nk + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        int n = 0;
        for (l = 0; l < num_levels; ++l) {
            const int ps = page_sizes[l];
            for (k = 0; k < num_nodes[l]; ++k) {
                const int32_t *nd = nodes[l] + 4 * k;
                if (b < nd[0] || b >= nd[1])
                    continue;
                for (t = 0; t < nd[2]; ++t, ++n) {
                    long page = page_ids[l][nd[3] + t / ps];
                    long slot = t % ps;
                    size_t off = (((size_t)page * Hkv + kvh) * ps + slot) * d;
                    keys[n].e4m3 = kv_dtypes[l] == 1;
                    if (keys[n].e4m3) {
                        keys[n].k = (const uint8_t *)k_pools[l] + off;
                        keys[n].v = (const uint8_t *)v_pools[l] + off;
                        keys[n].k_scale = k_scales[l][page * Hkv + kvh];
                        keys[n].v_scale = v_scales[l][page * Hkv + kvh];
                    } else {
                        keys[n].k = (const uint16_t *)k_pools[l] + off;
                        keys[n].v = (const uint16_t *)v_pools[l] + off;
                        keys[n].k_scale = keys[n].v_scale = 1.0;
                    }
                }
                break; /* nodes of one level cover disjoint ranges */
            }
        }
        load_q(d, q + ((size_t)b * Hq + h) * d, qd);
        sdp_keys(d, qd, nk, keys, scale, O + (size_t)r * d, lse + r, s);
        free(keys);
        free(s);
        free(qd);
    }
    return 0;
}

/* Per-sequence paged decode over E4M3 pools (codes [page][Hkv][ps][d] bytes,
 * f32 scales [page][Hkv] for K and for V); otherwise as hpo_paged_decode. */
int hpo_paged_decode_e4m3(int B, int Hq, int Hkv, int d, double scale, const uint16_t *q, long q_sb,
                          long q_sh, const uint8_t *k_pool, const uint8_t *v_pool, const float *k_scale,
                          const float *v_scale, int page_size, const int32_t *page_table, int pt_stride,
                          const int32_t *seq_lens, double *O, double *lse)
{
    long r;
    int G;
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < (long)B * Hq; ++r) {
        int b = (int)(r / Hq), h = (int)(r % Hq), kvh = h / G, t;
        int nk = seq_lens[b];
        hpo_key *keys = (hpo_key *)malloc(sizeof(hpo_key) * (size_t)(nk + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        for (t = 0; t < nk; ++t) {
            long page = page_table[(size_t)b * pt_stride + t / page_size];
            size_t off = (((size_t)page * Hkv + kvh) * page_size + t % page_size) * d;
            keys[t].k = k_pool + off;
            keys[t].v = v_pool + off;
            keys[t].k_scale = k_scale[page * Hkv + kvh];
            keys[t].v_scale = v_scale[page * Hkv + kvh];
            keys[t].e4m3 = 1;
        }
        load_q(d, q + (size_t)b * q_sb + (size_t)h * q_sh, qd);
        sdp_keys(d, qd, nk, keys, scale, O + (size_t)r * d, lse + r, s);
        free(keys);
        free(s);
        free(qd);
    }
    return 0;
}

/* Per-sequence paged decode: sequence b attends over its first seq_lens[b]
 * tokens, token t at page page_table[b*pt_stride + t/ps], slot t%ps.
 * q row (b,h) at q + b*q_sb + h*q_sh.  Outputs O [B][Hq][d], lse [B][Hq]. */
int hpo_paged_decode(int B, int Hq, int Hkv, int d, double scale, const uint16_t *q, long q_sb,
                     long q_sh, const uint16_t *k_pool, const uint16_t *v_pool, int page_size,
                     const int32_t *page_table, int pt_stride, const int32_t *seq_lens, double *O,
                     double *lse)
{
    long r;
    int G;
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < (long)B * Hq; ++r) {
        int b = (int)(r / Hq), h = (int)(r % Hq), kvh = h / G, t;
        int nk = seq_lens[b];
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nk + 1));
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nk + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        for (t = 0; t < nk; ++t) {
            long page = page_table[(size_t)b * pt_stride + t / page_size];
            size_t off = (((size_t)page * Hkv + kvh) * page_size + t % page_size) * d;
            krow[t] = k_pool + off;
            vrow[t] = v_pool + off;
        }
        load_q(d, q + (size_t)b * q_sb + (size_t)h * q_sh, qd);
        sdp_rows_bf16(d, qd, nk, krow, vrow, scale, O + (size_t)r * d, lse + r, s);
        free(krow);
        free(vrow);
        free(s);
        free(qd);
    }
    return 0;
}

/* Attention of nb query sequences against one contiguous prefix.
 * Prefix layout: token t, KV head g at k + t*kv_st + g*kv_sh (elements).
 * q row (b,h) at q + b*q_sb + h*q_sh.  Outputs O [nb][Hq][d], lse [nb][Hq]. */
int hpo_prefix(int nb, int Hq, int Hkv, int d, double scale, const uint16_t *q, long q_sb,
               long q_sh, const uint16_t *k, const uint16_t *v, long kv_st, long kv_sh, int len,
               double *O, double *lse)
{
    long r;
    int G;
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < (long)nb * Hq; ++r) {
        int b = (int)(r / Hq), h = (int)(r % Hq), kvh = h / G, t;
        const uint16_t **krow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(len + 1));
        const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(len + 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(len + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        for (t = 0; t < len; ++t) {
            krow[t] = k + (size_t)t * kv_st + (size_t)kvh * kv_sh;
            vrow[t] = v + (size_t)t * kv_st + (size_t)kvh * kv_sh;
        }
        load_q(d, q + (size_t)b * q_sb + (size_t)h * q_sh, qd);
        sdp_rows_bf16(d, qd, len, krow, vrow, scale, O + (size_t)r * d, lse + r, s);
        free(krow);
        free(vrow);
        free(s);
        free(qd);
    }
    return 0;
}

int hpo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void hpo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
