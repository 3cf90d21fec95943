/*
 * oracle.c -- plain, slow, single-threaded CPU oracle of the multi-column
 * embedding front end.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or constant generator with the CUDA library under
 * sparse_lookup_gb300/; neither side includes or links the other.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (see oracle/build.py).
 * -ffp-contract=off keeps every fp32 operation a separately rounded IEEE
 * operation on both x86-64 and aarch64, so stored expected values do not
 * depend on the machine that wrote them.
 *
 * Pages this follows (cited by title and section):
 *  [RecIS]   "RecIS: Unifying Sparse and Dense Computation for Efficient
 *            Recommendation Training" -- §3.1 (FeatureEngine transforms:
 *            hashing, modulo, bucketization), §3.2 "Index-aware segment
 *            reduction" with Algorithm 1 (forward CSR sum; backward
 *            per-contributor gradient w_r * G[s(r),:]), Figure 3 (local
 *            reduce-ID with inverse map), §4.3 (sparse learning rate).
 *  [RECom]   "RECom: A Compiler Approach to Accelerating Recommendation Model
 *            Inference with Massive Embedding Columns" -- "Why this problem is
 *            worth solving" (column = preprocess, translate to index by hashing
 *            or bucketing, safety: drop out-of-range indices and fill a default
 *            for a missing feature, lookup, reduce).
 *  [Monolith] "Di Dalam Monolit ByteDance: Mesin yang Memberdayakan Umpan
 *            Konten yang Lebih Cerdas dan Cepat" -- §2.1 "Tabel Hash"
 *            (collision-free table, admission after an occurrence threshold,
 *            expiry of IDs idle longer than a per-table period).
 *
 * Readings where the pages are silent (each is restated in the design notes):
 *  - hash transform = one output step of SplitMix64 (Steele, Lea & Flood,
 *    OOPSLA 2014, as in Vigna's splitmix64.c) with the state set to the ID
 *    reinterpreted as u64, then unsigned 64-bit modulo the table rows;
 *  - bucketize: row = #{j : bnd[j] <= x}; NaN -> 0; rows = nb + 1;
 *  - a dropped ID does not count in the mean denominator; a bag with no valid
 *    ID yields the column's default vector (zeros when none is given) and
 *    passes no gradient;
 *  - Adagrad: torch.optim.Adagrad's update with lr_decay = weight_decay = 0,
 *    eps outside the square root, evaluated in fp32 in the order
 *    g = (float)ghat; a = acc + g*g; w = w - (lr*g) / (sqrt(a) + eps);
 *  - hash admission: every occurrence counts; admission is decided after the
 *    whole batch is counted and takes effect in the same call; newly admitted
 *    keys are ordered by (table id, key) ascending and take the lowest free
 *    rows: the free list in ascending order first, then a bump pointer;
 *  - expiry: an entry (admitted or still counting) is removed when
 *    now - last_seen > ttl; its row returns to the free list;
 *  - sequence truncation: a SUM / MEAN column with max_len > 0 uses only the
 *    first max_len values of each bag (dropped IDs among them stay dropped).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_OOM = 3, ORC_ERR_FULL = 5 };

enum { ORC_IDENTITY = 0, ORC_HASH_MOD = 1, ORC_BUCKETIZE = 2, ORC_ROWS_GIVEN = 3 };
enum { ORC_SUM = 0, ORC_MEAN = 1, ORC_PADDED = 2 };

/* One embedding column as the oracle sees it [RECom, "Why this problem is
 * worth solving": each column owns one embedding table]. */
typedef struct {
    int32_t transform;        /* ORC_IDENTITY .. ORC_ROWS_GIVEN               */
    int32_t pooling;          /* ORC_SUM, ORC_MEAN, ORC_PADDED                */
    int64_t num_rows;         /* rows of the table                            */
    int32_t dim;              /* floats per row                               */
    int32_t table;            /* which physical table (columns may share one) */
    const float* boundaries;  /* BUCKETIZE: sorted boundaries                 */
    int32_t num_boundaries;
    int32_t pad_len;          /* PADDED: padded sequence length               */
    const float* default_vec; /* [dim] or NULL => zeros                       */
    int64_t out_col;          /* pooled: float offset of the column in a row of
                                 the concatenated output                      */
    int32_t max_len;          /* SUM / MEAN: a bag is its first max_len values
                                 (sequence truncation; 0 = all)               */
    int32_t reserved;
    const float* weights;     /* SUM: per-value weights w_r (NULL = all 1)     */
    int32_t table_dtype;      /* ORC_DT_*: how the table's elements are stored */
    int32_t reserved2;
    const float* row_scale;   /* ORC_DT_I8: [num_rows] scale of each row        */
} orc_col;

/* Element storage of a table [the RecIS evaluation lists an int8 table beside
 * fp32 ones, Table 3; the reading here: bf16, IEEE binary16, or int8 with
 * one fp32 scale per row]. */
enum { ORC_DT_F32 = 0, ORC_DT_BF16 = 1, ORC_DT_F16 = 2, ORC_DT_I8 = 3 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds zero and the subnormals (fraction x 2^-24),
 * exponent 31 infinity (fraction 0) and NaN. */
static double half_value(uint16_t h)
{
    const int sign = h >> 15, ex = (h >> 10) & 31, fr = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)fr, -24);
    else if (ex == 31) v = fr ? NAN : INFINITY;
    else v = ldexp((double)(fr | 1024), ex - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (same sign and exponent,
 * 7 fraction bits). */
static double bf16_value(uint16_t h)
{
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element d of row r of the column's table, exactly (int8: scale * q). */
static double table_value(const orc_col* c, const void* E, int64_t r, int32_t d)
{
    const int64_t e = r * c->dim + d;
    switch (c->table_dtype) {
    case ORC_DT_BF16: return bf16_value(((const uint16_t*)E)[e]);
    case ORC_DT_F16: return half_value(((const uint16_t*)E)[e]);
    case ORC_DT_I8: return (double)c->row_scale[r] * (double)((const int8_t*)E)[e];
    default: return (double)((const float*)E)[e];
    }
}

/* Weight of value t of a column: w_t for a weighted SUM column [RecIS §3.2,
 * Algorithm 1: y_s = sum_r w_r E[idx_r], and the backward passes w_r G[s]
 * to row idx_r], else 1. */
static double value_weight(const orc_col* c, int64_t t)
{
    return (c->pooling == ORC_SUM && c->weights) ? (double)c->weights[t] : 1.0;
}

/* End of the values of bag [lo, hi) that the column uses: PADDED keeps the
 * first pad_len, a truncated pooled column the first max_len [RecIS §2.1,
 * SeqTrunc: a long sequence feature keeps its first elements]. */
static int64_t bag_end(const orc_col* c, int64_t lo, int64_t hi)
{
    if (c->pooling == ORC_PADDED && hi - lo > c->pad_len) return lo + c->pad_len;
    if (c->pooling != ORC_PADDED && c->max_len > 0 && hi - lo > c->max_len) return lo + c->max_len;
    return hi;
}

/* ------------------------------------------------------------------------ */
/* a1: feature transform                                                     */
/* ------------------------------------------------------------------------ */

/* One output of SplitMix64 with the generator state equal to x. */
uint64_t orc_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Row of one value, before the safety check.  [RecIS §3.1: the hash, modulo
 * and bucket transforms turn a feature value into a table index.] */
static int64_t transform_one(const orc_col* c, int64_t id, float x)
{
    switch (c->transform) {
    case ORC_IDENTITY:
    case ORC_ROWS_GIVEN:
        return id;
    case ORC_HASH_MOD:
        return (int64_t)(orc_splitmix64((uint64_t)id) % (uint64_t)c->num_rows);
    case ORC_BUCKETIZE: {
        /* number of boundaries that are <= x, counted one by one */
        int64_t n = 0;
        for (int32_t j = 0; j < c->num_boundaries; ++j)
            if (c->boundaries[j] <= x) ++n;
        return n;
    }
    }
    return -1;
}

/* a1 + a2: transformed row of every value of one column, -1 when the value is
 * dropped by the safety check (row outside [0, num_rows)).  [RECom, "Why this
 * problem is worth solving": a column's safety step discards indices that fall
 * outside its table.] */
int orc_column_rows(const orc_col* c, int64_t n, const int64_t* ids,
                    const float* fvals, int64_t* rows_out)
{
    if (!c || (n > 0 && !rows_out)) return ORC_ERR_ARG;
    for (int64_t t = 0; t < n; ++t) {
        int64_t id = 0;
        float x = 0.0f;
        if (c->transform == ORC_BUCKETIZE) x = fvals[t]; else id = ids[t];
        int64_t r = transform_one(c, id, x);
        rows_out[t] = (r >= 0 && r < c->num_rows) ? r : -1;
    }
    return ORC_OK;
}

static int check_offsets(const int32_t* off, int32_t B)
{
    if (off[0] != 0) return ORC_ERR_ARG;
    for (int32_t b = 0; b < B; ++b)
        if (off[b + 1] < off[b]) return ORC_ERR_ARG;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a2 + a3 + a4: forward                                                     */
/* ------------------------------------------------------------------------ */

/* Forward of all columns.
 * offsets[c]: int32 [B+1] CSR of column c (relative to its own values);
 * ids[c] (int64) or fvals[c] (fp32, BUCKETIZE) hold its values;
 * tables[t]: row-major [num_rows, dim] of physical table t, elements stored
 *   as the columns' table_dtype says (fp32 unless stated);
 * out: [B, ldo] fp32, column c pooled into out[b*ldo + out_col + d];
 * seq_out[c]: PADDED columns, [B, pad_len, dim]; rows_out[c]: optional rows.
 *
 * Pooling follows Algorithm 1's forward [RecIS §3.2]: each output element is
 * the sum over the bag's CSR range [o_s, o_{s+1}) of the gathered rows (all
 * weights 1; MEAN divides by the number of valid IDs).  The sum is taken in
 * fp64 and rounded to fp32 once.  A bag with no valid ID gets the default
 * vector [RECom, "Why this problem is worth solving": a missing feature is
 * given a default; RecIS §3.2: an empty segment pools to zero]. */
int orc_forward(const orc_col* cols, int32_t C, int32_t B,
                const int32_t* const* offsets, const int64_t* const* ids,
                const float* const* fvals, const void* const* tables,
                float* out, int64_t ldo, float* const* seq_out,
                int64_t* const* rows_out)
{
    if (!cols || C < 0 || B < 0) return ORC_ERR_ARG;
    for (int32_t ci = 0; ci < C; ++ci) {
        const orc_col* c = &cols[ci];
        const int32_t* off = offsets[ci];
        if (check_offsets(off, B)) return ORC_ERR_ARG;
        int64_t n = off[B];
        int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
        double* S = (double*)malloc(sizeof(double) * (size_t)c->dim);
        if (!rows || !S) { free(rows); free(S); return ORC_ERR_OOM; }
        orc_column_rows(c, n, ids ? ids[ci] : NULL, fvals ? fvals[ci] : NULL, rows);
        if (rows_out && rows_out[ci]) memcpy(rows_out[ci], rows, sizeof(int64_t) * (size_t)n);
        const void* E = tables[c->table];
        for (int32_t b = 0; b < B; ++b) {
            int64_t lo = off[b], hi = off[b + 1];
            if (c->pooling == ORC_PADDED) {
                float* y = seq_out[ci] + (int64_t)b * c->pad_len * c->dim;
                for (int32_t t = 0; t < c->pad_len; ++t) {
                    int64_t r = (lo + t < hi) ? rows[lo + t] : -1;
                    for (int32_t d = 0; d < c->dim; ++d)
                        y[(int64_t)t * c->dim + d] = (r >= 0) ? (float)table_value(c, E, r, d) : 0.0f;
                }
                continue;
            }
            hi = bag_end(c, lo, hi);
            int64_t nv = 0;
            for (int32_t d = 0; d < c->dim; ++d) S[d] = 0.0;
            for (int64_t t = lo; t < hi; ++t) {
                int64_t r = rows[t];
                if (r < 0) continue;
                ++nv;
                const double wt = value_weight(c, t);
                for (int32_t d = 0; d < c->dim; ++d) S[d] += wt * table_value(c, E, r, d);
            }
            float* y = out + (int64_t)b * ldo + c->out_col;
            for (int32_t d = 0; d < c->dim; ++d) {
                if (nv == 0)
                    y[d] = c->default_vec ? c->default_vec[d] : 0.0f;
                else if (c->pooling == ORC_MEAN)
                    y[d] = (float)(S[d] / (double)nv);
                else
                    y[d] = (float)S[d];
            }
        }
        free(rows);
        free(S);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a5 + a6 + a7: backward, unique rows, aggregated gradient, sparse Adagrad  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t table;
    int32_t col;
    int64_t row;
    int64_t seq;    /* position in the order the contributions were listed  */
    int32_t b, t;   /* bag and position inside it                           */
    double scale;   /* w_r (1 unweighted) for SUM, 1 for PADDED, 1/n_valid for MEAN */
} contrib;

static int cmp_contrib(const void* pa, const void* pb)
{
    const contrib* a = (const contrib*)pa;
    const contrib* b = (const contrib*)pb;
    if (a->table != b->table) return a->table < b->table ? -1 : 1;
    if (a->row != b->row) return a->row < b->row ? -1 : 1;
    if (a->seq != b->seq) return a->seq < b->seq ? -1 : 1;
    return 0;
}

/* One Adagrad step on one element, fp32, in the order stated in the header. */
static void adagrad_elem(float* w, float* a, double ghat, float lr, float eps)
{
    float g = (float)ghat;
    float acc = *a + g * g;
    float den = sqrtf(acc) + eps;
    *a = acc;
    *w = *w - (lr * g) / den;
}

/* Backward of the forward above followed by sparse Adagrad.
 *
 * For every valid contribution r of bag (c, b) the gradient reaching its row
 * is scale_r * G[b, out_col + d] (PADDED columns: Gseq[c][b, t, d]); this is
 * the per-contributor term w_r G[s(r),:] of Algorithm 1's backward
 * [RecIS §3.2], with w_r = 1 (SUM, PADDED) or 1/n_valid (MEAN).  All
 * contributions to one physical row (table, row) are summed in fp64; the
 * rows are listed once each, ascending by (table, row), which is the local
 * reduce-ID of [RecIS §3.2, Figure 3 step 1] with counts.  Each listed row
 * then takes one Adagrad step (header).
 *
 * W[t], acc[t]: host tables [num_rows, dim] of table t, updated in place.
 * Optional outputs (NULL to skip): u_table/u_row/u_count [cap] per unique row;
 * u_grad: the fp32-rounded aggregated gradients, row after row, dim floats
 * each (grad_cap floats at most).  *n_unique receives the unique count. */
int orc_backward_adagrad(const orc_col* cols, int32_t C, int32_t B,
                         const int32_t* const* offsets, const int64_t* const* ids,
                         const float* const* fvals, const float* G, int64_t ldG,
                         const float* const* Gseq, float* const* W, float* const* acc,
                         float lr, float eps, int64_t cap, int64_t* n_unique,
                         int32_t* u_table, int64_t* u_row, int64_t* u_count,
                         float* u_grad, int64_t grad_cap)
{
    if (!cols || C < 0 || B < 0) return ORC_ERR_ARG;
    int64_t total = 0;
    for (int32_t ci = 0; ci < C; ++ci) {
        if (check_offsets(offsets[ci], B)) return ORC_ERR_ARG;
        total += offsets[ci][B];
    }
    contrib* list = (contrib*)malloc(sizeof(contrib) * (size_t)(total > 0 ? total : 1));
    if (!list) return ORC_ERR_OOM;
    int64_t n = 0;
    for (int32_t ci = 0; ci < C; ++ci) {
        const orc_col* c = &cols[ci];
        const int32_t* off = offsets[ci];
        int64_t nvals = off[B];
        int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nvals > 0 ? nvals : 1));
        if (!rows) { free(list); return ORC_ERR_OOM; }
        orc_column_rows(c, nvals, ids ? ids[ci] : NULL, fvals ? fvals[ci] : NULL, rows);
        for (int32_t b = 0; b < B; ++b) {
            int64_t lo = off[b], hi = off[b + 1];
            hi = bag_end(c, lo, hi);
            int64_t nv = 0;
            for (int64_t t = lo; t < hi; ++t) nv += rows[t] >= 0;
            for (int64_t t = lo; t < hi; ++t) {
                if (rows[t] < 0) continue;
                contrib* e = &list[n];
                e->table = c->table;
                e->col = ci;
                e->row = rows[t];
                e->seq = n;
                e->b = b;
                e->t = (int32_t)(t - lo);
                e->scale = (c->pooling == ORC_MEAN) ? 1.0 / (double)nv : value_weight(c, t);
                ++n;
            }
        }
        free(rows);
    }
    qsort(list, (size_t)n, sizeof(contrib), cmp_contrib);

    int64_t nu = 0, gpos = 0;
    int64_t i = 0;
    int32_t maxdim = 1;
    for (int32_t ci = 0; ci < C; ++ci) if (cols[ci].dim > maxdim) maxdim = cols[ci].dim;
    double* S = (double*)malloc(sizeof(double) * (size_t)maxdim);
    if (!S) { free(list); return ORC_ERR_OOM; }
    while (i < n) {
        int64_t j = i;
        while (j < n && list[j].table == list[i].table && list[j].row == list[i].row) ++j;
        const orc_col* c0 = &cols[list[i].col];
        int32_t dim = c0->dim;
        for (int32_t d = 0; d < dim; ++d) S[d] = 0.0;
        for (int64_t k = i; k < j; ++k) {
            const orc_col* c = &cols[list[k].col];
            const float* src;
            if (c->pooling == ORC_PADDED)
                src = Gseq[list[k].col] + ((int64_t)list[k].b * c->pad_len + list[k].t) * c->dim;
            else
                src = G + (int64_t)list[k].b * ldG + c->out_col;
            for (int32_t d = 0; d < dim; ++d) S[d] += list[k].scale * (double)src[d];
        }
        float* w = W[list[i].table] + list[i].row * dim;
        float* a = acc[list[i].table] + list[i].row * dim;
        for (int32_t d = 0; d < dim; ++d) adagrad_elem(&w[d], &a[d], S[d], lr, eps);
        if (nu < cap) {
            if (u_table) u_table[nu] = list[i].table;
            if (u_row) u_row[nu] = list[i].row;
            if (u_count) u_count[nu] = j - i;
        }
        if (u_grad && gpos + dim <= grad_cap)
            for (int32_t d = 0; d < dim; ++d) u_grad[gpos + d] = (float)S[d];
        gpos += dim;
        ++nu;
        i = j;
    }
    if (n_unique) *n_unique = nu;
    free(S);
    free(list);
    return ORC_OK;
}

/* The same backward for a chosen set of rows only, for workloads whose
 * tables are too large to copy to the host: targets (t_table[i], t_row[i]),
 * strictly ascending by (table, row).  Every valid contribution is visited in
 * the order orc_backward_adagrad lists them; one whose row is a target adds
 * scale_r * G to that target's fp64 sum (and |scale_r * G| to t_abs), so each
 * target's sum is formed in the same order as in orc_backward_adagrad.  Then
 * each target row takes its Adagrad step on the compact host rows
 * W_rows / acc_rows ([n_targets, ld], the target's dim floats used).
 * Outputs: t_count [n_targets]; t_grad [n_targets, ld] fp32-rounded sums;
 * t_abs [n_targets, ld] fp64 sums of magnitudes (NULL to skip). */
static int64_t find_target(int64_t n, const int32_t* tt, const int64_t* tr, int32_t table, int64_t row)
{
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (tt[mid] < table || (tt[mid] == table && tr[mid] < row)) lo = mid + 1; else hi = mid;
    }
    return (lo < n && tt[lo] == table && tr[lo] == row) ? lo : -1;
}

int orc_backward_rows(const orc_col* cols, int32_t C, int32_t B,
                      const int32_t* const* offsets, const int64_t* const* ids,
                      const float* const* fvals, const float* G, int64_t ldG,
                      const float* const* Gseq, int64_t n_targets, const int32_t* t_table,
                      const int64_t* t_row, float* W_rows, float* acc_rows, int32_t ld,
                      float lr, float eps, int64_t* t_count, float* t_grad, double* t_abs)
{
    if (!cols || C < 0 || B < 0 || n_targets < 0 || ld < 1) return ORC_ERR_ARG;
    for (int64_t i = 1; i < n_targets; ++i)
        if (t_table[i] < t_table[i - 1] || (t_table[i] == t_table[i - 1] && t_row[i] <= t_row[i - 1]))
            return ORC_ERR_ARG;
    for (int32_t ci = 0; ci < C; ++ci)
        if (check_offsets(offsets[ci], B)) return ORC_ERR_ARG;
    size_t cells = (size_t)(n_targets > 0 ? n_targets : 1) * (size_t)ld;
    double* S = (double*)calloc(cells, sizeof(double));
    double* A = (double*)calloc(cells, sizeof(double));
    int32_t* tdim = (int32_t*)calloc((size_t)(n_targets > 0 ? n_targets : 1), sizeof(int32_t));
    if (!S || !A || !tdim) { free(S); free(A); free(tdim); return ORC_ERR_OOM; }
    for (int64_t i = 0; i < n_targets; ++i) t_count[i] = 0;
    for (int32_t ci = 0; ci < C; ++ci) {
        const orc_col* c = &cols[ci];
        if (c->dim > ld) { free(S); free(A); free(tdim); return ORC_ERR_ARG; }
        const int32_t* off = offsets[ci];
        int64_t nvals = off[B];
        int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nvals > 0 ? nvals : 1));
        if (!rows) { free(S); free(A); free(tdim); return ORC_ERR_OOM; }
        orc_column_rows(c, nvals, ids ? ids[ci] : NULL, fvals ? fvals[ci] : NULL, rows);
        for (int32_t b = 0; b < B; ++b) {
            int64_t lo = off[b], hi = off[b + 1];
            hi = bag_end(c, lo, hi);
            int64_t nv = 0;
            for (int64_t t = lo; t < hi; ++t) nv += rows[t] >= 0;
            for (int64_t t = lo; t < hi; ++t) {
                if (rows[t] < 0) continue;
                int64_t k = find_target(n_targets, t_table, t_row, c->table, rows[t]);
                if (k < 0) continue;
                double scale = (c->pooling == ORC_MEAN) ? 1.0 / (double)nv : value_weight(c, t);
                const float* src;
                if (c->pooling == ORC_PADDED)
                    src = Gseq[ci] + ((int64_t)b * c->pad_len + (t - lo)) * c->dim;
                else
                    src = G + (int64_t)b * ldG + c->out_col;
                for (int32_t d = 0; d < c->dim; ++d) {
                    S[k * ld + d] += scale * (double)src[d];
                    A[k * ld + d] += fabs(scale * (double)src[d]);
                }
                tdim[k] = c->dim;
                t_count[k] += 1;
            }
        }
        free(rows);
    }
    for (int64_t k = 0; k < n_targets; ++k) {
        for (int32_t d = 0; d < tdim[k]; ++d) {
            adagrad_elem(&W_rows[k * ld + d], &acc_rows[k * ld + d], S[k * ld + d], lr, eps);
            if (t_grad) t_grad[k * ld + d] = (float)S[k * ld + d];
            if (t_abs) t_abs[k * ld + d] = A[k * ld + d];
        }
    }
    free(S);
    free(A);
    free(tdim);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a8 + a9: collision-free hash table with frequency filter and expiry       */
/* [Monolith §2.1 "Tabel Hash"]                                              */
/* ------------------------------------------------------------------------ */

/* The oracle keeps the key -> entry map as separate chaining: distinct keys
 * never share an entry, which is the collision-free property the page asks
 * for; where an entry lives inside the map is not part of the result. */
typedef struct {
    int64_t key;
    int32_t tid;
    int32_t admitted;
    int64_t row;        /* admitted: its row; else -1 */
    int64_t count;      /* occurrences since the entry was created */
    uint32_t last_seen; /* step of the last lookup */
    int64_t next;       /* chain link, -1 ends the chain */
} orc_entry;

typedef struct orc_hash {
    int64_t row_capacity;
    int32_t dim;
    int32_t threshold;
    uint64_t seed;
    float init_scale;
    float* W;           /* caller-owned host row pool [row_capacity, dim] */
    float* acc;         /* caller-owned host accumulators, same shape     */
    int64_t nbuckets;   /* power of two */
    int64_t* heads;
    orc_entry* ent;
    int64_t n_ent, cap_ent;
    int64_t free_ent;   /* chain of reusable entry records, -1 if none */
    int64_t live;
    int64_t* free_rows; /* rows released by expiry */
    int64_t n_free, cap_free;
    int64_t bump;       /* rows >= bump were never handed out */
    int64_t* admitted;  /* rows handed out by the last lookup, in admission order */
    int64_t n_admitted, cap_admitted;
} orc_hash;

static uint64_t bucket_of(const orc_hash* h, int32_t tid, int64_t key)
{
    return orc_splitmix64((uint64_t)key ^ ((uint64_t)(uint32_t)tid * 0xD6E8FEB86659FD93ULL)) &
           (uint64_t)(h->nbuckets - 1);
}

orc_hash* orc_hash_create(int64_t row_capacity, int32_t dim, int32_t threshold,
                          uint64_t seed, float init_scale, float* W, float* acc)
{
    if (row_capacity <= 0 || dim <= 0 || threshold < 1 || !W || !acc) return NULL;
    orc_hash* h = (orc_hash*)calloc(1, sizeof(orc_hash));
    if (!h) return NULL;
    h->row_capacity = row_capacity;
    h->dim = dim;
    h->threshold = threshold;
    h->seed = seed;
    h->init_scale = init_scale;
    h->W = W;
    h->acc = acc;
    h->nbuckets = 1 << 16;
    h->heads = (int64_t*)malloc(sizeof(int64_t) * (size_t)h->nbuckets);
    h->cap_ent = 1 << 16;
    h->ent = (orc_entry*)malloc(sizeof(orc_entry) * (size_t)h->cap_ent);
    h->cap_free = 1 << 10;
    h->free_rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)h->cap_free);
    h->cap_admitted = 1 << 10;
    h->admitted = (int64_t*)malloc(sizeof(int64_t) * (size_t)h->cap_admitted);
    if (!h->heads || !h->ent || !h->free_rows || !h->admitted) {
        free(h->heads); free(h->ent); free(h->free_rows); free(h->admitted); free(h);
        return NULL;
    }
    for (int64_t i = 0; i < h->nbuckets; ++i) h->heads[i] = -1;
    h->free_ent = -1;
    return h;
}

void orc_hash_destroy(orc_hash* h)
{
    if (!h) return;
    free(h->heads);
    free(h->ent);
    free(h->free_rows);
    free(h->admitted);
    free(h);
}

static int grow_buckets(orc_hash* h)
{
    int64_t nb = h->nbuckets * 2;
    int64_t* heads = (int64_t*)malloc(sizeof(int64_t) * (size_t)nb);
    if (!heads) return ORC_ERR_OOM;
    for (int64_t i = 0; i < nb; ++i) heads[i] = -1;
    int64_t old = h->nbuckets;
    int64_t* oldh = h->heads;
    h->nbuckets = nb;
    h->heads = heads;
    for (int64_t bkt = 0; bkt < old; ++bkt) {
        int64_t e = oldh[bkt];
        while (e >= 0) {
            int64_t nx = h->ent[e].next;
            uint64_t nbk = bucket_of(h, h->ent[e].tid, h->ent[e].key);
            h->ent[e].next = heads[nbk];
            heads[nbk] = e;
            e = nx;
        }
    }
    free(oldh);
    return ORC_OK;
}

static int64_t find_entry(const orc_hash* h, int32_t tid, int64_t key)
{
    int64_t e = h->heads[bucket_of(h, tid, key)];
    while (e >= 0 && !(h->ent[e].tid == tid && h->ent[e].key == key)) e = h->ent[e].next;
    return e;
}

static int64_t new_entry(orc_hash* h, int32_t tid, int64_t key)
{
    if (h->live + 1 > h->nbuckets && grow_buckets(h)) return -1;
    int64_t e;
    if (h->free_ent >= 0) {
        e = h->free_ent;
        h->free_ent = h->ent[e].next;
    } else {
        if (h->n_ent == h->cap_ent) {
            int64_t nc = h->cap_ent * 2;
            orc_entry* ne = (orc_entry*)realloc(h->ent, sizeof(orc_entry) * (size_t)nc);
            if (!ne) return -1;
            h->ent = ne;
            h->cap_ent = nc;
        }
        e = h->n_ent++;
    }
    orc_entry* x = &h->ent[e];
    x->key = key;
    x->tid = tid;
    x->admitted = 0;
    x->row = -1;
    x->count = 0;
    x->last_seen = 0;
    uint64_t bkt = bucket_of(h, tid, key);
    x->next = h->heads[bkt];
    h->heads[bkt] = e;
    h->live++;
    return e;
}

/* Initial value of element d of a newly admitted key's row: a uniform draw in
 * [-1, 1) with 24 random bits, times init_scale.  Every step is exact in fp32
 * except the final multiply, which rounds once. */
float orc_hash_init_value(uint64_t seed, int32_t tid, int64_t key, int32_t d, float init_scale)
{
    uint64_t h = orc_splitmix64((uint64_t)key ^ ((uint64_t)(uint32_t)tid << 48) ^ seed ^ (uint64_t)(uint32_t)d);
    int32_t v = (int32_t)(h >> 40) - 8388608;
    float f = (float)v * (1.0f / 8388608.0f);
    return f * init_scale;
}

typedef struct { int32_t tid; int64_t key; int64_t e; } newkey;

static int cmp_newkey(const void* pa, const void* pb)
{
    const newkey* a = (const newkey*)pa;
    const newkey* b = (const newkey*)pb;
    if (a->tid != b->tid) return a->tid < b->tid ? -1 : 1;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    return 0;
}

static int cmp_i64(const void* pa, const void* pb)
{
    int64_t a = *(const int64_t*)pa, b = *(const int64_t*)pb;
    return a < b ? -1 : (a > b);
}

/* Lookup-or-insert of one batch of n (table id, key) occurrences at `step`.
 * rows_out[i] receives the row of occurrence i, or -1 while its key is below
 * the admission threshold.  Returns ORC_ERR_FULL when the row pool ran out
 * (the keys that found no row stay counting and return -1). */
int orc_hash_lookup_or_insert(orc_hash* h, const int32_t* tids, const int64_t* keys,
                              int64_t n, uint32_t step, int64_t* rows_out)
{
    if (!h || n < 0) return ORC_ERR_ARG;
    int status = ORC_OK;
    h->n_admitted = 0;
    /* 1. count every occurrence and touch its entry */
    int64_t n_new = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t e = find_entry(h, tids[i], keys[i]);
        if (e < 0) e = new_entry(h, tids[i], keys[i]);
        if (e < 0) return ORC_ERR_OOM;
        orc_entry* x = &h->ent[e];
        x->last_seen = step;
        if (!x->admitted) {
            x->count += 1;
            if (x->count >= h->threshold) ++n_new; /* upper bound on new keys */
        }
    }
    /* 2. admit the keys that reached the threshold, in (tid, key) order; a
     *    key that found no free row earlier is listed again */
    if (n_new > 0) {
        newkey* nk = (newkey*)malloc(sizeof(newkey) * (size_t)n_new);
        if (!nk) return ORC_ERR_OOM;
        int64_t m = 0;
        for (int64_t i = 0; i < n; ++i) {
            int64_t e = find_entry(h, tids[i], keys[i]);
            orc_entry* x = &h->ent[e];
            if (!x->admitted && x->count >= h->threshold && x->row != -2) {
                x->row = -2; /* listed once */
                nk[m].tid = x->tid;
                nk[m].key = x->key;
                nk[m].e = e;
                ++m;
            }
        }
        qsort(nk, (size_t)m, sizeof(newkey), cmp_newkey);
        if (m > h->cap_admitted) {
            int64_t* na = (int64_t*)realloc(h->admitted, sizeof(int64_t) * (size_t)m);
            if (!na) { free(nk); return ORC_ERR_OOM; }
            h->admitted = na;
            h->cap_admitted = m;
        }
        qsort(h->free_rows, (size_t)h->n_free, sizeof(int64_t), cmp_i64);
        int64_t used_free = 0;
        for (int64_t k = 0; k < m; ++k) {
            orc_entry* x = &h->ent[nk[k].e];
            int64_t row;
            if (used_free < h->n_free) row = h->free_rows[used_free++];
            else if (h->bump < h->row_capacity) row = h->bump++;
            else { x->row = -1; status = ORC_ERR_FULL; continue; }
            x->admitted = 1;
            x->row = row;
            h->admitted[h->n_admitted++] = row;
            for (int32_t d = 0; d < h->dim; ++d) {
                h->W[row * h->dim + d] = orc_hash_init_value(h->seed, x->tid, x->key, d, h->init_scale);
                h->acc[row * h->dim + d] = 0.0f;
            }
        }
        memmove(h->free_rows, h->free_rows + used_free, sizeof(int64_t) * (size_t)(h->n_free - used_free));
        h->n_free -= used_free;
        free(nk);
    }
    /* 3. answer every occurrence */
    if (rows_out)
        for (int64_t i = 0; i < n; ++i) {
            const orc_entry* x = &h->ent[find_entry(h, tids[i], keys[i])];
            rows_out[i] = x->admitted ? x->row : -1;
        }
    return status;
}

/* Expiry sweep: remove every entry with now - last_seen > ttl.  Returns the
 * number of entries removed (admitted and counting). */
int64_t orc_hash_evict(orc_hash* h, uint32_t now, uint32_t ttl)
{
    int64_t removed = 0;
    for (int64_t bkt = 0; bkt < h->nbuckets; ++bkt) {
        int64_t* link = &h->heads[bkt];
        while (*link >= 0) {
            int64_t e = *link;
            orc_entry* x = &h->ent[e];
            if ((int64_t)now - (int64_t)x->last_seen > (int64_t)ttl) {
                if (x->admitted) {
                    if (h->n_free == h->cap_free) {
                        int64_t nc = h->cap_free * 2;
                        int64_t* nf = (int64_t*)realloc(h->free_rows, sizeof(int64_t) * (size_t)nc);
                        if (!nf) return -1;
                        h->free_rows = nf;
                        h->cap_free = nc;
                    }
                    h->free_rows[h->n_free++] = x->row;
                }
                *link = x->next;
                x->next = h->free_ent;
                h->free_ent = e;
                h->live--;
                ++removed;
            } else {
                link = &x->next;
            }
        }
    }
    return removed;
}

/* Every live entry, in no particular order.  Returns the number of entries
 * (all of them are written when cap allows). */
int64_t orc_hash_export(const orc_hash* h, int32_t* tids, int64_t* keys, int64_t* rows,
                        int64_t* counts, uint32_t* last_seen, int64_t cap)
{
    int64_t k = 0;
    for (int64_t bkt = 0; bkt < h->nbuckets; ++bkt)
        for (int64_t e = h->heads[bkt]; e >= 0; e = h->ent[e].next) {
            if (k < cap) {
                const orc_entry* x = &h->ent[e];
                if (tids) tids[k] = x->tid;
                if (keys) keys[k] = x->key;
                if (rows) rows[k] = x->admitted ? x->row : -1;
                if (counts) counts[k] = x->count;
                if (last_seen) last_seen[k] = x->last_seen;
            }
            ++k;
        }
    return k;
}

/* Rows the last lookup handed out (and initialised), in admission order.
 * Returns their number (all are written when cap allows). */
int64_t orc_hash_last_admitted(const orc_hash* h, int64_t* rows, int64_t cap)
{
    if (!h) return 0;
    for (int64_t i = 0; i < h->n_admitted && i < cap; ++i) rows[i] = h->admitted[i];
    return h->n_admitted;
}

int64_t orc_hash_size(const orc_hash* h) { return h ? h->live : 0; }
int64_t orc_hash_bump(const orc_hash* h) { return h ? h->bump : 0; }
int64_t orc_hash_free_count(const orc_hash* h) { return h ? h->n_free : 0; }
