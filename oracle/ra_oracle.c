/*
 * ra_oracle.c -- plain, slow fp64 CPU definition of masked attention with the
 * ring (out, lse) merge.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * library links, includes or calls this file; only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark use it.
 *
 * Sources (page title, then the section on it):
 *   [RS]   "ejkernel ... ring_attention._ring_splash" module source:
 *          _update_out_and_lse, _ring_attention_forward, _ring_attention_backward.
 *   [RSAPI] the API page of the same module (defaults such as mask_value).
 *   [KVAX] "Kvax: Flash Attention for JAX": flash_attention arguments,
 *          create_attention_mask, context-parallel token permutation.
 *
 * Everything is fp64; inputs arrive already widened from their stored bf16 /
 * fp32 values.  Layouts: q, out, dq [B][Lq][Hq][D]; k, v, dk, dv
 * [B][Lkv][Hkv][D]; lse [B][Hq][Lq]; positions / segment ids [B][L] int32;
 * sinks [Hq].
 *
 * Readings of points the pages leave open (each repeated at its use):
 *   R-excl   masked logits are excluded from the softmax (not given a large
 *            finite value); a row with nothing visible has O = 0, lse = -inf.
 *   R-pad    the padding segment id is never visible on either side.
 *   R-sink   a sink is one raw logit per query head, shared over the batch,
 *            counted once per row (the ring counts it on step 0 only).
 *   R-order  s = scale * <q,k>, then the soft cap, then the mask.
 *   R-pos    the causal predicate is q_pos >= kv_pos on positions; absent
 *            positions mean the token's index in the sequence as given.
 *   R-gqa    kv head of query head h is h / (Hq / Hkv).
 *   R-zig    zigzag: 2N chunks, virtual device d holds chunks d and 2N-1-d.
 *   R-local  without causal masking the ring of [RS] (_ring_attention_forward,
 *            non-causal branch) applies the one 2-D mask given to
 *            make_ring_attention -- local query length x local kv length --
 *            at every ring step; the pair (i, j) is then visible only where
 *            local_mask[i mod Lq_s][j mod Lkv_s] is set (Lq_s, Lkv_s = the
 *            per-device lengths), in addition to the segment rule.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORA_TILE 128

typedef struct {
    int B, Lq, Lkv, Hq, Hkv, D;
    double scale;     /* multiplies <q,k>            ([KVAX] flash_attention `scale`) */
    double soft_cap;  /* <= 0 : no cap               ([RS] logits_soft_cap) */
    int causal;       /* q_pos >= kv_pos             ([RS] causal_mask_fn) */
    int pad_segment_id;
    const int32_t *q_pos, *kv_pos; /* NULL -> index in the sequence */
    const int32_t *q_seg, *kv_seg; /* NULL -> one segment, no padding */
    const double *sinks;           /* NULL -> no sink */
    const uint8_t *local_mask;     /* [lq_s][lk_s], nonzero = visible; NULL -> none (R-local) */
    int lq_s, lk_s;                /* per-device query / kv lengths of local_mask */
} ora_params;

/* ------------------------------------------------------------------ */
/* visibility of one (query, key) pair: same non-padding segment, if causal
 * query position >= key position, and the local mask if one is given.
 * [KVAX] flash_attention (segment ids, positions, PADDING_SEGMENT_ID);
 * [RS] causal_mask_fn and the non-causal ring's per-step mask. */
static int ora_visible(const ora_params *p, int b, int i, int j)
{
    if (p->q_seg || p->kv_seg) {
        int sq = p->q_seg ? p->q_seg[(size_t)b * p->Lq + i] : 0;
        int sk = p->kv_seg ? p->kv_seg[(size_t)b * p->Lkv + j] : 0;
        if (sq != sk) return 0;
        if (sq == p->pad_segment_id) return 0; /* R-pad */
    }
    if (p->causal) {
        int pq = p->q_pos ? p->q_pos[(size_t)b * p->Lq + i] : i;
        int pk = p->kv_pos ? p->kv_pos[(size_t)b * p->Lkv + j] : j;
        if (pq < pk) return 0;
    }
    if (p->local_mask && !p->local_mask[(size_t)(i % p->lq_s) * p->lk_s + (j % p->lk_s)])
        return 0; /* R-local */
    return 1;
}

/* The scale and soft cap applied to a finished dot product (R-order). */
static double ora_cap(const ora_params *p, double acc)
{
    double s = p->scale * acc;
    if (p->soft_cap > 0.0) s = p->soft_cap * tanh(s / p->soft_cap);
    return s;
}

/* logit of one pair after scale and soft cap (R-order) */
static double ora_logit(const ora_params *p, const double *qrow, const double *krow)
{
    double acc = 0.0;
    for (int d = 0; d < p->D; ++d) acc += qrow[d] * krow[d];
    return ora_cap(p, acc);
}

static inline const double *qrow_of(const ora_params *p, const double *q, int b, int i, int h)
{
    return q + (((size_t)b * p->Lq + i) * p->Hq + h) * p->D;
}
static inline const double *krow_of(const ora_params *p, const double *k, int b, int j, int g)
{
    return k + (((size_t)b * p->Lkv + j) * p->Hkv + g) * p->D;
}

/* Attention of query rows [i0, i1) of (b, h) over key rows [j0, j1), with the
 * row mask given as materialised bytes vis[(i - i0) * Lkv + j].  The sink, if
 * use_sink, adds exp(sink_h) to the denominator only (R-sink).  Writes the
 * normalised output and the natural-log lse of each row (R-excl). */
static void ora_rows(const ora_params *p, const double *q, const double *k, const double *v,
                     int b, int h, int i0, int i1, int j0, int j1, const uint8_t *vis,
                     int use_sink, double *out_rows /* [(i1-i0)][D] */, double *lse_rows,
                     double *sbuf /* [Lkv] */)
{
    const int g = h / (p->Hq / p->Hkv); /* R-gqa */
    const int D = p->D;
    for (int i = i0; i < i1; ++i) {
        const uint8_t *vrow = vis + (size_t)(i - i0) * p->Lkv;
        const double *qr = qrow_of(p, q, b, i, h);
        double m = -INFINITY;
        int any = 0;
        for (int j = j0; j < j1; ++j) {
            if (!vrow[j]) continue;
            double s = ora_logit(p, qr, krow_of(p, k, b, j, g));
            sbuf[j] = s;
            if (s > m) m = s;
            any = 1;
        }
        double sink = (use_sink && p->sinks) ? p->sinks[h] : -INFINITY;
        if (sink > m) m = sink;
        double *o = out_rows + (size_t)(i - i0) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (!any && !(use_sink && p->sinks)) {
            lse_rows[i - i0] = -INFINITY;
            continue;
        }
        double z = (use_sink && p->sinks) ? exp(sink - m) : 0.0;
        for (int j = j0; j < j1; ++j)
            if (vrow[j]) z += exp(sbuf[j] - m);
        double lse = m + log(z);
        lse_rows[i - i0] = lse;
        for (int j = j0; j < j1; ++j) {
            if (!vrow[j]) continue;
            double w = exp(sbuf[j] - lse);
            const double *vr = krow_of(p, v, b, j, g);
            for (int d = 0; d < D; ++d) o[d] += w * vr[d];
        }
    }
}

/* Threads that ran at least one task of the last parallel call (the CPU
 * baseline reports it as the core count it used). */
static int ora_threads_used = 1;

static int ora_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int ora_thread_id(void)
{
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

static void ora_count_threads(const unsigned char *ran, int n)
{
    int c = 0;
    for (int t = 0; t < n; ++t) c += ran[t] != 0;
    ora_threads_used = c > 0 ? c : 1;
}

/* Rows per task of a parallel loop over `rows` rows of `B` batch rows (and
 * `units` independent heads or groups): small enough that there are about
 * four tasks per thread, at most one 128-row tile.  Only the schedule depends
 * on it, never the arithmetic of a row. */
static int ora_rows_per_task(int rows, int B, int units)
{
    const long want = 4L * ora_max_threads();
    long per = ((long)rows * B * (units > 0 ? units : 1) + want - 1) / want;
    if (per > ORA_TILE) per = ORA_TILE;
    if (per < 1) per = 1;
    return (int)per;
}

static void ora_fill_mask(const ora_params *p, int b, int i0, int i1, uint8_t *vis)
{
    for (int i = i0; i < i1; ++i)
        for (int j = 0; j < p->Lkv; ++j)
            vis[(size_t)(i - i0) * p->Lkv + j] = (uint8_t)ora_visible(p, b, i, j);
}

static int ora_check(const ora_params *p)
{
    if (p->B <= 0 || p->Lq <= 0 || p->Lkv <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0) return -1;
    if (p->Hq % p->Hkv) return -1;
    return 0;
}

/* Plain definition: every (b, h, i) over all keys, sink counted once.
 * Only query heads [heads_lo, heads_hi) and query rows [rows_lo, rows_hi)
 * are computed (an empty range means all); the rest of out / lse is left
 * untouched.  Restricting rows or heads changes which rows are computed,
 * never how a row is computed.  Tasks are blocks of rows of one batch row;
 * each materialises its block's mask once and runs every head over it. */
int ora_attn_fwd(const ora_params *p, const double *q, const double *k, const double *v,
                 double *out, double *lse, int heads_lo, int heads_hi, int rows_lo, int rows_hi)
{
    if (ora_check(p)) return -1;
    if (heads_hi <= heads_lo) { heads_lo = 0; heads_hi = p->Hq; }
    if (rows_hi <= rows_lo) { rows_lo = 0; rows_hi = p->Lq; }
    if (heads_lo < 0 || heads_hi > p->Hq || rows_lo < 0 || rows_hi > p->Lq) return -1;
    const int R = ora_rows_per_task(rows_hi - rows_lo, p->B, 1);
    const int nblk = (rows_hi - rows_lo + R - 1) / R;
    const int D = p->D;
    const int nthr = ora_max_threads();
    unsigned char *ran = (unsigned char *)calloc((size_t)nthr, 1);
    if (!ran) return -2;
    int err = 0;
#pragma omp parallel
    {
        uint8_t *vis = (uint8_t *)malloc((size_t)R * p->Lkv);
        double *sbuf = (double *)malloc(sizeof(double) * p->Lkv);
        double *orow = (double *)malloc(sizeof(double) * (size_t)R * D);
        double *lrow = (double *)malloc(sizeof(double) * R);
        if (!vis || !sbuf || !orow || !lrow) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (int b = 0; b < p->B; ++b)
                for (int blk = 0; blk < nblk; ++blk) {
                    const int i0 = rows_lo + blk * R;
                    const int i1 = i0 + R < rows_hi ? i0 + R : rows_hi;
                    ran[ora_thread_id()] = 1;
                    ora_fill_mask(p, b, i0, i1, vis);
                    for (int h = heads_lo; h < heads_hi; ++h) {
                        ora_rows(p, q, k, v, b, h, i0, i1, 0, p->Lkv, vis, 1, orow, lrow, sbuf);
                        for (int i = i0; i < i1; ++i) {
                            memcpy(out + (((size_t)b * p->Lq + i) * p->Hq + h) * D,
                                   orow + (size_t)(i - i0) * D, sizeof(double) * D);
                            lse[((size_t)b * p->Hq + h) * p->Lq + i] = lrow[i - i0];
                        }
                    }
                }
        }
        free(vis); free(sbuf); free(orow); free(lrow);
    }
    ora_count_threads(ran, nthr);
    free(ran);
    return err;
}

/* Numerically stable logistic sigmoid and softplus; both give 0 at -inf.
 * [RS] _update_out_and_lse uses jax.nn.sigmoid / jax.nn.softplus. */
static double ora_sigmoid(double x)
{
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}
static double ora_softplus(double x)
{
    double a = x > 0.0 ? x : 0.0;
    return a + log1p(exp(-fabs(x)));
}

/* [RS] _update_out_and_lse: merge one chunk's (block_out, block_lse) into the
 * running (out, lse) of a row.  First chunk (lse == -inf) takes the block. */
static void ora_merge_row(double *o, double *l, const double *bo, double bl, int D)
{
    if (*l == -INFINITY) {
        for (int d = 0; d < D; ++d) o[d] = bo[d];
        *l = bl;
        return;
    }
    double w = ora_sigmoid(bl - *l);
    for (int d = 0; d < D; ++d) o[d] = o[d] - w * (o[d] - bo[d]);
    *l = *l + ora_softplus(bl - *l);
}

/* Elementwise merge over out [B][L][H][D], lse [B][H][L] (in place). */
void ora_merge(double *out, double *lse, const double *bout, const double *blse,
               int B, int L, int H, int D)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < L; ++i)
            for (int h = 0; h < H; ++h) {
                size_t r = (((size_t)b * L + i) * H + h) * D;
                size_t li = ((size_t)b * H + h) * L + i;
                ora_merge_row(out + r, lse + li, bout + r, blse[li], D);
            }
}

/* Key/value source held by virtual device d at ring step t: the initial
 * source is the device's own index and each step takes the previous source
 * minus one, modulo N ([RS] _ring_attention_forward: initial_kv_source,
 * kv_source_next).  Closed form (d - t) mod N. */
int ora_ring_source(int d, int t, int n)
{
    int src = d;
    for (int i = 0; i < t; ++i) src = (src - 1 + n) % n;
    return src;
}

/* Ring mode, taken literally from [RS] _ring_attention_forward with N virtual
 * devices on one machine: device d owns query rows [d*Lq/N, (d+1)*Lq/N);
 * at step t it holds the key/value chunk of source s = (d - t) mod N
 * (initial source = own index, next = source - 1 mod N), computes the
 * chunk's partial (out, lse) with the sink only at t == 0, and merges it into
 * the running state, which starts at (0, -inf).  The mask is the global one
 * (positions and segments of the whole sequence), which for absent positions
 * is the pages' per-step causal offset d*Lq_local - s*Lkv_local. */
int ora_attn_fwd_ring(const ora_params *p, int n_shards, const double *q, const double *k,
                      const double *v, double *out, double *lse, int heads_lo, int heads_hi)
{
    if (ora_check(p) || n_shards <= 0 || p->Lq % n_shards || p->Lkv % n_shards) return -1;
    if (heads_hi <= heads_lo) { heads_lo = 0; heads_hi = p->Hq; }
    const int N = n_shards, D = p->D;
    const int lq = p->Lq / N, lk = p->Lkv / N;
    const int R = lq < ORA_TILE ? lq : ORA_TILE;
    const int nblk = (lq + R - 1) / R;
    int err = 0;
#pragma omp parallel
    {
        uint8_t *vis = (uint8_t *)malloc((size_t)R * p->Lkv);
        double *sbuf = (double *)malloc(sizeof(double) * p->Lkv);
        double *orun = (double *)malloc(sizeof(double) * (size_t)R * D);
        double *lrun = (double *)malloc(sizeof(double) * R);
        double *oblk = (double *)malloc(sizeof(double) * (size_t)R * D);
        double *lblk = (double *)malloc(sizeof(double) * R);
        if (!vis || !sbuf || !orun || !lrun || !oblk || !lblk) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(3)
            for (int b = 0; b < p->B; ++b)
                for (int dev = 0; dev < N; ++dev)
                    for (int blk = 0; blk < nblk; ++blk) {
                        int i0 = dev * lq + blk * R;
                        int i1 = i0 + R < (dev + 1) * lq ? i0 + R : (dev + 1) * lq;
                        ora_fill_mask(p, b, i0, i1, vis);
                        for (int h = heads_lo; h < heads_hi; ++h) {
                            for (int r = 0; r < i1 - i0; ++r) {
                                lrun[r] = -INFINITY;
                                for (int d = 0; d < D; ++d) orun[(size_t)r * D + d] = 0.0;
                            }
                            for (int t = 0; t < N; ++t) {
                                const int src = ora_ring_source(dev, t, N);
                                ora_rows(p, q, k, v, b, h, i0, i1, src * lk, (src + 1) * lk, vis,
                                         t == 0, oblk, lblk, sbuf);
                                for (int r = 0; r < i1 - i0; ++r)
                                    ora_merge_row(orun + (size_t)r * D, lrun + r,
                                                  oblk + (size_t)r * D, lblk[r], D);
                            }
                            for (int i = i0; i < i1; ++i) {
                                memcpy(out + (((size_t)b * p->Lq + i) * p->Hq + h) * D,
                                       orun + (size_t)(i - i0) * D, sizeof(double) * D);
                                lse[((size_t)b * p->Hq + h) * p->Lq + i] = lrun[i - i0];
                            }
                        }
                    }
        }
        free(vis); free(sbuf); free(orun); free(lrun); free(oblk); free(lblk);
    }
    return err;
}

/* dS of one visible pair (the soft-cap factor included) and its P:
 *   P = exp(s - lse),  dP = <dO_i, v_j>,  dS = P (dP - Delta_i) (1 - (s/cap)^2) */
static void ora_pair_grad(const ora_params *p, const double *qr, const double *kr,
                          const double *vr, const double *go, double l, double delta,
                          double *pij_out, double *ds_out)
{
    double s = ora_logit(p, qr, kr);
    double pij = exp(s - l);
    double dp = 0.0;
    for (int d = 0; d < p->D; ++d) dp += go[d] * vr[d];
    double dsij = pij * (dp - delta);
    if (p->soft_cap > 0.0) {
        double t = s / p->soft_cap;
        dsij *= 1.0 - t * t;
    }
    *pij_out = pij;
    *ds_out = dsij;
}

/* Exact gradient of the plain forward (its own forward is recomputed here,
 * so no input comes from elsewhere).  Only pairs (i, j) with query row i in
 * [rows_lo, rows_hi), key row j in [keys_lo, keys_hi) and query head in
 * [heads_lo, heads_hi) contribute (an empty range means all); dq of rows and
 * dk / dv of keys outside the ranges stay 0, and dsinks sums the rows of the
 * row range.  The result is the full gradient when every range is all.
 * Summing per-chunk contributions as [RS] _ring_attention_backward does gives
 * the same sums.
 *   Delta_i = <dO_i, O_i>,  P_ij = exp(s_ij - lse_i) on visible pairs
 *   dV_j  += P_ij dO_i ;  dP_ij = <dO_i, v_j> ;  dS_ij = P_ij (dP_ij - Delta_i)
 *   dR_ij  = dS_ij * (1 - (s_ij / cap)^2)   (cap > 0; 1 otherwise)
 *   dQ_i  += scale dR_ij k_j ;  dK_j += scale dR_ij q_i
 *   dsink_h = - sum_{b,i} exp(sink_h - lse_i) Delta_i
 * dk, dv sum over the query heads sharing a kv head (R-gqa).  Two parallel
 * passes that own their outputs: dq by (b, h, block of query rows), summing
 * keys in ascending order; dk / dv by (b, kv head, block of keys), summing
 * the heads of the group, then query rows, in ascending order. */
int ora_attn_bwd(const ora_params *p, const double *q, const double *k, const double *v,
                 const double *dout, double *dq, double *dk, double *dv, double *dsinks,
                 double *out_ws, double *lse_ws, int heads_lo, int heads_hi, int rows_lo,
                 int rows_hi, int keys_lo, int keys_hi)
{
    if (ora_check(p)) return -1;
    if (heads_hi <= heads_lo) { heads_lo = 0; heads_hi = p->Hq; }
    if (rows_hi <= rows_lo) { rows_lo = 0; rows_hi = p->Lq; }
    if (keys_hi <= keys_lo) { keys_lo = 0; keys_hi = p->Lkv; }
    if (keys_lo < 0 || keys_hi > p->Lkv) return -1;
    int rc = ora_attn_fwd(p, q, k, v, out_ws, lse_ws, heads_lo, heads_hi, rows_lo, rows_hi);
    if (rc) return rc;
    int used = ora_threads_used;
    const int D = p->D, G = p->Hq / p->Hkv, H = heads_hi - heads_lo;
    memset(dq, 0, sizeof(double) * (size_t)p->B * p->Lq * p->Hq * D);
    memset(dk, 0, sizeof(double) * (size_t)p->B * p->Lkv * p->Hkv * D);
    memset(dv, 0, sizeof(double) * (size_t)p->B * p->Lkv * p->Hkv * D);
    const size_t nrow = (size_t)p->B * p->Hq * p->Lq;
    double *delta = (double *)calloc(nrow, sizeof(double));
    if (!delta) return -2;
    const int nthr = ora_max_threads();
    unsigned char *ran = (unsigned char *)calloc((size_t)nthr, 1);
    if (!ran) { free(delta); return -2; }

    /* Delta of every row in range; dsinks per head, rows in ascending order */
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < p->B; ++b)
        for (int h = heads_lo; h < heads_hi; ++h)
            for (int i = rows_lo; i < rows_hi; ++i) {
                const double *o = out_ws + (((size_t)b * p->Lq + i) * p->Hq + h) * D;
                const double *go = dout + (((size_t)b * p->Lq + i) * p->Hq + h) * D;
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += go[d] * o[d];
                delta[((size_t)b * p->Hq + h) * p->Lq + i] = s;
            }
    if (dsinks) {
        for (int h = 0; h < p->Hq; ++h) dsinks[h] = 0.0;
        if (p->sinks)
            for (int h = heads_lo; h < heads_hi; ++h) {
                double tot = 0.0;
                for (int b = 0; b < p->B; ++b) {
                    double acc = 0.0;
                    for (int i = rows_lo; i < rows_hi; ++i) {
                        const size_t r = ((size_t)b * p->Hq + h) * p->Lq + i;
                        if (lse_ws[r] != -INFINITY) acc -= exp(p->sinks[h] - lse_ws[r]) * delta[r];
                    }
                    tot += acc;
                }
                dsinks[h] = tot;
            }
    }

    /* pass 1: dq */
    const int Rq = ora_rows_per_task(rows_hi - rows_lo, p->B, H);
    const int nbq = (rows_hi - rows_lo + Rq - 1) / Rq;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < p->B; ++b)
        for (int h = heads_lo; h < heads_hi; ++h)
            for (int blk = 0; blk < nbq; ++blk) {
                ran[ora_thread_id()] = 1;
                const int g = h / G;
                const int i0 = rows_lo + blk * Rq;
                const int i1 = i0 + Rq < rows_hi ? i0 + Rq : rows_hi;
                for (int i = i0; i < i1; ++i) {
                    const size_t r = ((size_t)b * p->Hq + h) * p->Lq + i;
                    const double l = lse_ws[r];
                    if (l == -INFINITY) continue;
                    const double *qr = qrow_of(p, q, b, i, h);
                    const double *go = dout + (((size_t)b * p->Lq + i) * p->Hq + h) * D;
                    double *gq = dq + (((size_t)b * p->Lq + i) * p->Hq + h) * D;
                    for (int j = keys_lo; j < keys_hi; ++j) {
                        if (!ora_visible(p, b, i, j)) continue;
                        const double *kr = krow_of(p, k, b, j, g);
                        double pij, dsij;
                        ora_pair_grad(p, qr, kr, krow_of(p, v, b, j, g), go, l, delta[r], &pij,
                                      &dsij);
                        for (int d = 0; d < D; ++d) gq[d] += p->scale * dsij * kr[d];
                    }
                }
            }

    /* pass 2: dk, dv */
    const int Rk = ora_rows_per_task(keys_hi - keys_lo, p->B, p->Hkv);
    const int nbk = (keys_hi - keys_lo + Rk - 1) / Rk;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int b = 0; b < p->B; ++b)
        for (int g = 0; g < p->Hkv; ++g)
            for (int blk = 0; blk < nbk; ++blk) {
                const int h0 = g * G > heads_lo ? g * G : heads_lo;
                const int h1 = (g + 1) * G < heads_hi ? (g + 1) * G : heads_hi;
                if (h0 >= h1) continue;
                ran[ora_thread_id()] = 1;
                const int j0 = keys_lo + blk * Rk;
                const int j1 = j0 + Rk < keys_hi ? j0 + Rk : keys_hi;
                for (int j = j0; j < j1; ++j) {
                    const double *kr = krow_of(p, k, b, j, g);
                    const double *vr = krow_of(p, v, b, j, g);
                    double *gk = dk + (((size_t)b * p->Lkv + j) * p->Hkv + g) * D;
                    double *gv = dv + (((size_t)b * p->Lkv + j) * p->Hkv + g) * D;
                    for (int h = h0; h < h1; ++h)
                        for (int i = rows_lo; i < rows_hi; ++i) {
                            const size_t r = ((size_t)b * p->Hq + h) * p->Lq + i;
                            const double l = lse_ws[r];
                            if (l == -INFINITY || !ora_visible(p, b, i, j)) continue;
                            const double *qr = qrow_of(p, q, b, i, h);
                            const double *go = dout + (((size_t)b * p->Lq + i) * p->Hq + h) * D;
                            double pij, dsij;
                            ora_pair_grad(p, qr, kr, vr, go, l, delta[r], &pij, &dsij);
                            for (int d = 0; d < D; ++d) {
                                gv[d] += pij * go[d];
                                gk[d] += p->scale * dsij * qr[d];
                            }
                        }
                }
            }
    ora_count_threads(ran, nthr);
    if (ora_threads_used < used) ora_threads_used = used;
    free(ran);
    free(delta);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Block map on the canonical 128 x 128 tile grid.  Class of tile (qt, kt):
 * 0 = EMPTY (no visible pair), 2 = FULL (all 128*128 pairs visible),
 * 1 = PARTIAL.  [RS] MaskInfo / make_ring_attention (forward and dkv infos),
 * [KVAX] create_attention_mask (skip_pad_tokens).
 *   cls       [B][nq][nk]
 *   fwd_cnt   [B*nq]       number of non-empty tiles of each query-tile row
 *   fwd_idx   [B*nq][nk]   their kt, ascending, then -1
 *   bwd_cnt   [B*nk]       number of non-empty tiles of each key-tile column
 *   bwd_idx   [B*nk][nq]   their qt, ascending, then -1
 *   fwd_order [B*nq]       row ids b*nq+qt by descending count, ties by id
 *   bwd_order [B*nk]       column ids b*nk+kt, same rule
 * Counts are taken pair by pair from the visibility definition. */
typedef struct { int key; int id; } ora_kv;
static int ora_cmp_desc(const void *a, const void *b)
{
    const ora_kv *x = (const ora_kv *)a, *y = (const ora_kv *)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    return x->id < y->id ? -1 : (x->id > y->id ? 1 : 0);
}

/* The same classification on a grid of bq query rows x bk key rows (the
 * backward's own block sizes, [RS] make_ring_attention with
 * block_sizes.has_backward_blocks: the dkv MaskInfo built on the
 * (block_q_dkv, block_kv_dkv) grid; [KVAX] create_attention_mask computing
 * the backward mask).  nq = Lq / bq, nk = Lkv / bk; arrays as above with
 * those nq, nk. */
int ora_block_mask_sized(const ora_params *p, int bq, int bk, uint8_t *cls, int32_t *fwd_cnt,
                         int32_t *fwd_idx, int32_t *bwd_cnt, int32_t *bwd_idx, int32_t *fwd_order,
                         int32_t *bwd_order)
{
    if (bq <= 0 || bk <= 0 || p->Lq % bq || p->Lkv % bk || p->B <= 0) return -1;
    const int nq = p->Lq / bq, nk = p->Lkv / bk;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < p->B; ++b)
        for (int qt = 0; qt < nq; ++qt)
            for (int kt = 0; kt < nk; ++kt) {
                long cnt = 0;
                for (int i = qt * bq; i < (qt + 1) * bq; ++i)
                    for (int j = kt * bk; j < (kt + 1) * bk; ++j)
                        cnt += ora_visible(p, b, i, j);
                cls[((size_t)b * nq + qt) * nk + kt] =
                    cnt == 0 ? 0 : (cnt == (long)bq * bk ? 2 : 1);
            }
    for (int b = 0; b < p->B; ++b) {
        for (int qt = 0; qt < nq; ++qt) {
            int c = 0;
            int32_t *row = fwd_idx + ((size_t)b * nq + qt) * nk;
            for (int kt = 0; kt < nk; ++kt)
                if (cls[((size_t)b * nq + qt) * nk + kt]) row[c++] = kt;
            fwd_cnt[b * nq + qt] = c;
            for (int r = c; r < nk; ++r) row[r] = -1;
        }
        for (int kt = 0; kt < nk; ++kt) {
            int c = 0;
            int32_t *col = bwd_idx + ((size_t)b * nk + kt) * nq;
            for (int qt = 0; qt < nq; ++qt)
                if (cls[((size_t)b * nq + qt) * nk + kt]) col[c++] = qt;
            bwd_cnt[b * nk + kt] = c;
            for (int r = c; r < nq; ++r) col[r] = -1;
        }
    }
    ora_kv *tmp = (ora_kv *)malloc(sizeof(ora_kv) * (size_t)p->B * (nq > nk ? nq : nk));
    if (!tmp) return -2;
    for (int r = 0; r < p->B * nq; ++r) { tmp[r].key = fwd_cnt[r]; tmp[r].id = r; }
    qsort(tmp, (size_t)p->B * nq, sizeof(ora_kv), ora_cmp_desc);
    for (int r = 0; r < p->B * nq; ++r) fwd_order[r] = tmp[r].id;
    for (int r = 0; r < p->B * nk; ++r) { tmp[r].key = bwd_cnt[r]; tmp[r].id = r; }
    qsort(tmp, (size_t)p->B * nk, sizeof(ora_kv), ora_cmp_desc);
    for (int r = 0; r < p->B * nk; ++r) bwd_order[r] = tmp[r].id;
    free(tmp);
    return 0;
}

int ora_block_mask(const ora_params *p, uint8_t *cls, int32_t *fwd_cnt, int32_t *fwd_idx,
                   int32_t *bwd_cnt, int32_t *bwd_idx, int32_t *fwd_order, int32_t *bwd_order)
{
    return ora_block_mask_sized(p, ORA_TILE, ORA_TILE, cls, fwd_cnt, fwd_idx, bwd_cnt, bwd_idx,
                                fwd_order, bwd_order);
}

/* ------------------------------------------------------------------ */
/* Zigzag load-balancing permutation along the sequence ([KVAX] context
 * parallelism: permute tokens, positions and segment ids; unpermute outputs).
 * Reading R-zig: split L into 2N chunks of c = L/(2N) tokens; virtual device
 * d holds chunk d followed by chunk 2N-1-d.  Permuted row p = d*(L/N) + r
 * takes source row d*c + r when r < c, else (2N-1-d)*c + (r - c).
 * inverse == 0: out[p] = in[src(p)];  inverse != 0: out[src(p)] = in[p]. */
int ora_zigzag_source(int L, int n, int pidx)
{
    const int c = L / (2 * n), per = L / n;
    const int d = pidx / per, r = pidx % per;
    return r < c ? d * c + r : (2 * n - 1 - d) * c + (r - c);
}

int ora_permute(const uint8_t *in, uint8_t *out, int B, int L, size_t row_bytes, int n,
                int inverse)
{
    if (n <= 0 || L % (2 * n)) return -1;
    for (int b = 0; b < B; ++b)
        for (int pidx = 0; pidx < L; ++pidx) {
            int s = ora_zigzag_source(L, n, pidx);
            size_t dst = inverse ? (size_t)s : (size_t)pidx;
            size_t src = inverse ? (size_t)pidx : (size_t)s;
            memcpy(out + ((size_t)b * L + dst) * row_bytes, in + ((size_t)b * L + src) * row_bytes,
                   row_bytes);
        }
    return 0;
}

int ora_num_threads(void) { return ora_max_threads(); }

/* Threads that ran work in the last ora_attn_fwd / ora_attn_bwd call (for
 * the backward: the larger of its forward and gradient phases). */
int ora_last_threads(void) { return ora_threads_used; }
