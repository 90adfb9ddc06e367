/*
 * attn_oracle.c -- fp64 CPU oracle for exact attention (forward pass).
 *
 * TEST INFRASTRUCTURE ONLY.  The product library neither links nor calls
 * this file.  Only tests/, the package smoke check and the CPU-baseline /
 * reference leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * What it computes (the plain definition that FlashAttention-2 reproduces):
 *
 *   For every batch b, head h and query row i, over the allowed keys j
 *     s_ij  = scale * sum_d q_id * k_jd
 *     m_i   = max_j s_ij
 *     p_ij  = exp(s_ij - m_i) / sum_j exp(s_ij - m_i)
 *     o_id  = sum_j p_ij * v_jd
 *     lse_i = m_i + ln sum_j exp(s_ij - m_i)
 *
 *   Source walk-through "FlashAttention-2 相比 FlashAttention-1，到底改了什么",
 *   section "第二处源码差异：kernel 主循环怎么组织": the online-softmax loop
 *   computes O = acc / l, and the text under it states that v1 and v2 follow
 *   the same softmax mathematics; its interview summary ("面试速答") says FA2
 *   changes parallelism and work partitioning, not the formula.  The same
 *   section's epilogue comment names the two outputs, O and LSE.  So the
 *   oracle is the definition itself, with S and P written out in full.
 *
 * Mask (allowed keys).  j < Sk always; causal keeps j <= i (the causal mask
 * of "FlashAttention-2 — L3 Cross-Paper Synthesis", §3 item 4 and §5 item 4);
 * an optional window keeps i - wl <= j <= i + wr (the sliding-window
 * generalisation named in the same page's §5 item 4); wl or wr < 0 means
 * unbounded on that side.  Masked scores are -inf, i.e. probability zero.
 *
 * Readings where the pages are silent (each restated in the design notes):
 *   - scale multiplies the dot product before the max and the exponential;
 *   - LSE is the natural log of the sum of exponentials of the scaled scores;
 *   - causal alignment is top-left (j <= i); for Sq == Sk it is the only one;
 *   - a query row with no allowed key is an error (ORC_ERR_EMPTY_ROW),
 *     because softmax over an empty set has no value.
 *
 * bf16 front ends take raw bf16 bit patterns (uint16) and widen them exactly
 * to fp64 (a bf16 value is the top half of an IEEE binary32).
 *
 * Threads: work items are (batch*head, slab of up to ORC_SLAB query rows),
 * taken from a shared counter by nthreads pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_NOMEM (-2)
#define ORC_ERR_EMPTY_ROW (-3)

#define ORC_SLAB 256L

/* exact widening of a bf16 bit pattern to fp64 */
static double bf16_bits_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int key_allowed(long i, long j, long Sk, int causal, long wl, long wr) {
    if (j < 0 || j >= Sk) return 0;
    if (causal && j > i) return 0;
    if (wl >= 0 && j < i - wl) return 0;
    if (wr >= 0 && j > i + wr) return 0;
    return 1;
}

/*
 * One block of query rows of one (b,h): S and P are materialised as
 * nr x Sk arrays.  qbh/kbh/vbh are the fp64 [S, D] slices of this head.
 * rows[r] is the query index of row r; orow[r] / lrow[r] where it goes.
 */
static int attn_rows(const double *qbh, const double *kbh, const double *vbh,
                     const long *rows, long nr, double *const *orow, double *lrow_base,
                     const long *lidx, long Sk, long D, double scale, int causal,
                     long wl, long wr, double *S, double *P) {
    /* step 1: scores s_ij = scale * q_i . k_j, -inf where not allowed */
    for (long r = 0; r < nr; ++r) {
        const long i = rows[r];
        const double *qi = qbh + i * D;
        for (long j = 0; j < Sk; ++j) {
            if (!key_allowed(i, j, Sk, causal, wl, wr)) {
                S[r * Sk + j] = -INFINITY;
                continue;
            }
            const double *kj = kbh + j * D;
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
            S[r * Sk + j] = scale * dot;
        }
    }
    /* steps 2-3: row max, probabilities, log-sum-exp */
    for (long r = 0; r < nr; ++r) {
        double m = -INFINITY;
        for (long j = 0; j < Sk; ++j)
            if (S[r * Sk + j] > m) m = S[r * Sk + j];
        if (m == -INFINITY) return ORC_ERR_EMPTY_ROW;
        double sum = 0.0;
        for (long j = 0; j < Sk; ++j) {
            const double e = exp(S[r * Sk + j] - m); /* exp(-inf) == 0 */
            P[r * Sk + j] = e;
            sum += e;
        }
        for (long j = 0; j < Sk; ++j) P[r * Sk + j] /= sum;
        lrow_base[lidx[r]] = m + log(sum);
    }
    /* step 4: o_i = sum_j p_ij v_j */
    for (long r = 0; r < nr; ++r) {
        double *o = orow[r];
        for (long d = 0; d < D; ++d) o[d] = 0.0;
        for (long j = 0; j < Sk; ++j) {
            const double p = P[r * Sk + j];
            if (p == 0.0) continue;
            const double *vj = vbh + j * D;
            for (long d = 0; d < D; ++d) o[d] += p * vj[d];
        }
    }
    return ORC_OK;
}

typedef struct {
    const void *q, *k, *v;
    int bf16;
    double *o, *lse;
    long B, H, Sq, Sk, D;
    double scale;
    int causal;
    long wl, wr;
    /* selected rows (NULL: every row); sorted by bh */
    const long *sel_bh, *sel_row;
    long nsel;
    /* work list */
    long nitems;
    long *item_bh, *item_begin, *item_end; /* rows [begin,end) of a run */
    long next;
    int status;
    pthread_mutex_t mu;
} job_t;

static const double *slice_f64(const job_t *jb, const void *base, long bh, long S,
                               double *buf) {
    const long n = S * jb->D;
    if (!jb->bf16) return (const double *)base + bh * n;
    const uint16_t *src = (const uint16_t *)base + bh * n;
    for (long t = 0; t < n; ++t) buf[t] = bf16_bits_to_f64(src[t]);
    return buf;
}

static void *worker(void *arg) {
    job_t *jb = (job_t *)arg;
    const long D = jb->D, Sq = jb->Sq, Sk = jb->Sk;
    double *qb = NULL, *kb = NULL, *vb = NULL;
    if (jb->bf16) {
        qb = (double *)malloc(sizeof(double) * (size_t)(Sq * D));
        kb = (double *)malloc(sizeof(double) * (size_t)(Sk * D));
        vb = (double *)malloc(sizeof(double) * (size_t)(Sk * D));
    }
    double *S = (double *)malloc(sizeof(double) * (size_t)(ORC_SLAB * Sk));
    double *P = (double *)malloc(sizeof(double) * (size_t)(ORC_SLAB * Sk));
    long rows[ORC_SLAB], lidx[ORC_SLAB];
    double *orow[ORC_SLAB];
    int st = ORC_OK;
    if (!S || !P || (jb->bf16 && (!qb || !kb || !vb))) st = ORC_ERR_NOMEM;
    long last_bh = -1;
    const double *qbh = NULL, *kbh = NULL, *vbh = NULL;
    while (st == ORC_OK) {
        pthread_mutex_lock(&jb->mu);
        const long it = jb->next++;
        const int failed = jb->status != ORC_OK;
        pthread_mutex_unlock(&jb->mu);
        if (it >= jb->nitems || failed) break;
        const long bh = jb->item_bh[it];
        if (bh != last_bh) {
            qbh = slice_f64(jb, jb->q, bh, Sq, qb);
            kbh = slice_f64(jb, jb->k, bh, Sk, kb);
            vbh = slice_f64(jb, jb->v, bh, Sk, vb);
            last_bh = bh;
        }
        const long b0 = jb->item_begin[it], b1 = jb->item_end[it];
        const long nr = b1 - b0;
        for (long r = 0; r < nr; ++r) {
            if (jb->sel_row) {
                rows[r] = jb->sel_row[b0 + r];
                lidx[r] = b0 + r;
                orow[r] = jb->o + (b0 + r) * D;
            } else {
                rows[r] = b0 + r;
                lidx[r] = bh * Sq + b0 + r;
                orow[r] = jb->o + (bh * Sq + b0 + r) * D;
            }
        }
        st = attn_rows(qbh, kbh, vbh, rows, nr, orow, jb->lse, lidx, Sk, D, jb->scale,
                       jb->causal, jb->wl, jb->wr, S, P);
    }
    if (st != ORC_OK) {
        pthread_mutex_lock(&jb->mu);
        if (jb->status == ORC_OK) jb->status = st;
        pthread_mutex_unlock(&jb->mu);
    }
    free(S);
    free(P);
    free(qb);
    free(kb);
    free(vb);
    return NULL;
}

static int check_shape(long B, long H, long Sq, long Sk, long D) {
    return (B >= 1 && H >= 1 && Sq >= 1 && Sk >= 1 && D >= 1) ? ORC_OK : ORC_ERR_ARG;
}

static int run(job_t *jb, int nthreads) {
    /* build the work list: runs of rows of one bh, at most ORC_SLAB long */
    long cap;
    if (jb->sel_row)
        cap = jb->nsel + 1;
    else
        cap = jb->B * jb->H * ((jb->Sq + ORC_SLAB - 1) / ORC_SLAB);
    jb->item_bh = (long *)malloc(sizeof(long) * (size_t)cap);
    jb->item_begin = (long *)malloc(sizeof(long) * (size_t)cap);
    jb->item_end = (long *)malloc(sizeof(long) * (size_t)cap);
    if (!jb->item_bh || !jb->item_begin || !jb->item_end) {
        free(jb->item_bh);
        free(jb->item_begin);
        free(jb->item_end);
        return ORC_ERR_NOMEM;
    }
    long n = 0;
    if (jb->sel_row) {
        long s = 0;
        while (s < jb->nsel) {
            long e = s + 1;
            while (e < jb->nsel && jb->sel_bh[e] == jb->sel_bh[s] && e - s < ORC_SLAB) ++e;
            jb->item_bh[n] = jb->sel_bh[s];
            jb->item_begin[n] = s;
            jb->item_end[n] = e;
            ++n;
            s = e;
        }
    } else {
        for (long bh = 0; bh < jb->B * jb->H; ++bh)
            for (long r0 = 0; r0 < jb->Sq; r0 += ORC_SLAB) {
                jb->item_bh[n] = bh;
                jb->item_begin[n] = r0;
                jb->item_end[n] = (r0 + ORC_SLAB < jb->Sq) ? r0 + ORC_SLAB : jb->Sq;
                ++n;
            }
    }
    jb->nitems = n;
    jb->next = 0;
    jb->status = ORC_OK;
    pthread_mutex_init(&jb->mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    if (th)
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, worker, jb) != 0) break;
    if (started == 0) worker(jb); /* no thread could start: run inline */
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
    free(jb->item_bh);
    free(jb->item_begin);
    free(jb->item_end);
    return jb->status;
}

/* ------------------------------------------------------------------------ */
/* Entry points.  Tensors are [B, H, S, D] contiguous (row-major), the       */
/* layout the attention call uses; lse is [B, H, Sq].                       */

int oracle_attn_fwd_f64(const double *q, const double *k, const double *v, double *o,
                        double *lse, long B, long H, long Sq, long Sk, long D,
                        double scale, int causal, long wl, long wr, int nthreads) {
    if (!q || !k || !v || !o || !lse || check_shape(B, H, Sq, Sk, D)) return ORC_ERR_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.bf16 = 0; jb.o = o; jb.lse = lse;
    jb.B = B; jb.H = H; jb.Sq = Sq; jb.Sk = Sk; jb.D = D;
    jb.scale = scale; jb.causal = causal; jb.wl = wl; jb.wr = wr;
    return run(&jb, nthreads);
}

int oracle_attn_fwd_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *o,
                         double *lse, long B, long H, long Sq, long Sk, long D,
                         double scale, int causal, long wl, long wr, int nthreads) {
    if (!q || !k || !v || !o || !lse || check_shape(B, H, Sq, Sk, D)) return ORC_ERR_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.bf16 = 1; jb.o = o; jb.lse = lse;
    jb.B = B; jb.H = H; jb.Sq = Sq; jb.Sk = Sk; jb.D = D;
    jb.scale = scale; jb.causal = causal; jb.wl = wl; jb.wr = wr;
    return run(&jb, nthreads);
}

/*
 * Selected rows only: row t of the output is query row sel_row[t] of head
 * sel_bh[t] (= b*H + h).  sel_bh must be non-decreasing.  o is [n, D],
 * lse is [n].  Same arithmetic, in the same order, as the full call.
 */
int oracle_attn_fwd_rows_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const long *sel_bh, const long *sel_row, long n, double *o,
                              double *lse, long B, long H, long Sq, long Sk, long D,
                              double scale, int causal, long wl, long wr, int nthreads) {
    if (!q || !k || !v || !o || !lse || !sel_bh || !sel_row || n < 1 ||
        check_shape(B, H, Sq, Sk, D))
        return ORC_ERR_ARG;
    for (long t = 0; t < n; ++t) {
        if (sel_bh[t] < 0 || sel_bh[t] >= B * H || sel_row[t] < 0 || sel_row[t] >= Sq)
            return ORC_ERR_ARG;
        if (t > 0 && sel_bh[t] < sel_bh[t - 1]) return ORC_ERR_ARG;
    }
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.bf16 = 1; jb.o = o; jb.lse = lse;
    jb.B = B; jb.H = H; jb.Sq = Sq; jb.Sk = Sk; jb.D = D;
    jb.scale = scale; jb.causal = causal; jb.wl = wl; jb.wr = wr;
    jb.sel_bh = sel_bh; jb.sel_row = sel_row; jb.nsel = n;
    return run(&jb, nthreads);
}

/*
 * The tiled online-softmax loop, in the order and notation of the
 * walk-through's pseudocode ("第二处源码差异：kernel 主循环怎么组织"): for each
 * query block, m = -inf, l = 0, acc = 0; for each key/value block,
 * S = Q K^T (scaled), masked; m_new = max(m, rowmax S); P = exp(S - m_new);
 * acc = acc * exp(m - m_new) + P V; l = l * exp(m - m_new) + rowsum P;
 * m = m_new; finally O = acc / l, LSE = m + ln l.  Key blocks go in
 * ascending order.  A block in which a row has no allowed key leaves that
 * row's m, l and acc unchanged (it contributes nothing).  fp64, one thread.
 * Used only to show that the tiled loop and the definition agree.
 */
int oracle_attn_fwd_tiled_f64(const double *q, const double *k, const double *v, double *o,
                              double *lse, long B, long H, long Sq, long Sk, long D,
                              double scale, int causal, long wl, long wr, long bm, long bn) {
    if (!q || !k || !v || !o || !lse || check_shape(B, H, Sq, Sk, D) || bm < 1 || bn < 1)
        return ORC_ERR_ARG;
    double *Sblk = (double *)malloc(sizeof(double) * (size_t)(bm * bn));
    double *acc = (double *)malloc(sizeof(double) * (size_t)(bm * D));
    double *m = (double *)malloc(sizeof(double) * (size_t)bm);
    double *l = (double *)malloc(sizeof(double) * (size_t)bm);
    int st = ORC_OK;
    if (!Sblk || !acc || !m || !l) st = ORC_ERR_NOMEM;
    for (long bh = 0; st == ORC_OK && bh < B * H; ++bh) {
        const double *Q = q + bh * Sq * D, *K = k + bh * Sk * D, *V = v + bh * Sk * D;
        for (long i0 = 0; st == ORC_OK && i0 < Sq; i0 += bm) {
            const long ni = (i0 + bm <= Sq) ? bm : Sq - i0;
            for (long r = 0; r < ni; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (long d = 0; d < D; ++d) acc[r * D + d] = 0.0;
            }
            for (long j0 = 0; j0 < Sk; j0 += bn) {
                const long nj = (j0 + bn <= Sk) ? bn : Sk - j0;
                /* S = Q K^T, then apply_mask */
                for (long r = 0; r < ni; ++r)
                    for (long c = 0; c < nj; ++c) {
                        const long i = i0 + r, j = j0 + c;
                        double dot = 0.0;
                        for (long d = 0; d < D; ++d) dot += Q[i * D + d] * K[j * D + d];
                        Sblk[r * bn + c] = key_allowed(i, j, Sk, causal, wl, wr)
                                               ? scale * dot : -INFINITY;
                    }
                for (long r = 0; r < ni; ++r) {
                    double rowmax = -INFINITY;
                    for (long c = 0; c < nj; ++c)
                        if (Sblk[r * bn + c] > rowmax) rowmax = Sblk[r * bn + c];
                    if (rowmax == -INFINITY) continue; /* no allowed key here */
                    const double m_new = (m[r] > rowmax) ? m[r] : rowmax;
                    const double corr = exp(m[r] - m_new); /* exp(-inf) = 0 at start */
                    double rowsum = 0.0;
                    for (long d = 0; d < D; ++d) acc[r * D + d] *= corr;
                    for (long c = 0; c < nj; ++c) {
                        const double p = exp(Sblk[r * bn + c] - m_new);
                        rowsum += p;
                        if (p == 0.0) continue;
                        const double *vj = V + (j0 + c) * D;
                        for (long d = 0; d < D; ++d) acc[r * D + d] += p * vj[d];
                    }
                    l[r] = l[r] * corr + rowsum;
                    m[r] = m_new;
                }
            }
            for (long r = 0; r < ni; ++r) {
                if (m[r] == -INFINITY) {
                    st = ORC_ERR_EMPTY_ROW;
                    break;
                }
                for (long d = 0; d < D; ++d) o[(bh * Sq + i0 + r) * D + d] = acc[r * D + d] / l[r];
                lse[bh * Sq + i0 + r] = m[r] + log(l[r]);
            }
        }
    }
    free(Sblk);
    free(acc);
    free(m);
    free(l);
    return st;
}

/* ------------------------------------------------------------------------ */
/*
 * Backward pass of the same attention, from the definition (no tiling):
 * given dO (the gradient of a loss with respect to O), for each (b, h)
 *   S_ij  = scale q_i.k_j (allowed keys; -inf elsewhere),  P = softmax_j(S)
 *   O_i   = sum_j P_ij v_j
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   Delta_i = dO_i . O_i
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
 * ("FlashAttention-2 — L3 Cross-Paper Synthesis", §3 item 1 and §5 item 2:
 * the backward pass and its five matrix products.)  All of S, P, dP and dS
 * of a head are materialised; one thread per (batch, head).
 */
typedef struct {
    const void *q, *k, *v, *dout;
    int bf16;
    double *dq, *dk, *dv;
    long B, H, Sq, Sk, D;
    double scale;
    int causal;
    long wl, wr;
    long next;
    int status;
    pthread_mutex_t mu;
} bwd_job_t;

static void *bwd_worker(void *arg) {
    bwd_job_t *jb = (bwd_job_t *)arg;
    const long Sq = jb->Sq, Sk = jb->Sk, D = jb->D;
    double *qb = (double *)malloc(sizeof(double) * (size_t)(Sq * D));
    double *kb = (double *)malloc(sizeof(double) * (size_t)(Sk * D));
    double *vb = (double *)malloc(sizeof(double) * (size_t)(Sk * D));
    double *gb = (double *)malloc(sizeof(double) * (size_t)(Sq * D));
    double *P = (double *)malloc(sizeof(double) * (size_t)(Sq * Sk));
    double *dS = (double *)malloc(sizeof(double) * (size_t)(Sq * Sk));
    double *O = (double *)malloc(sizeof(double) * (size_t)(Sq * D));
    double *delta = (double *)malloc(sizeof(double) * (size_t)Sq);
    int st = ORC_OK;
    if (!qb || !kb || !vb || !gb || !P || !dS || !O || !delta) st = ORC_ERR_NOMEM;
    while (st == ORC_OK) {
        pthread_mutex_lock(&jb->mu);
        const long bh = jb->next++;
        const int failed = jb->status != ORC_OK;
        pthread_mutex_unlock(&jb->mu);
        if (bh >= jb->B * jb->H || failed) break;
        job_t view;  /* reuse the widening helper */
        memset(&view, 0, sizeof view);
        view.bf16 = jb->bf16;
        view.D = D;
        const double *Q = slice_f64(&view, jb->q, bh, Sq, qb);
        const double *K = slice_f64(&view, jb->k, bh, Sk, kb);
        const double *V = slice_f64(&view, jb->v, bh, Sk, vb);
        const double *G = slice_f64(&view, jb->dout, bh, Sq, gb);
        /* S -> P (row softmax over allowed keys), O */
        for (long i = 0; i < Sq && st == ORC_OK; ++i) {
            double m = -INFINITY;
            for (long j = 0; j < Sk; ++j) {
                double s = -INFINITY;
                if (key_allowed(i, j, Sk, jb->causal, jb->wl, jb->wr)) {
                    double dot = 0.0;
                    for (long d = 0; d < D; ++d) dot += Q[i * D + d] * K[j * D + d];
                    s = jb->scale * dot;
                }
                P[i * Sk + j] = s;
                if (s > m) m = s;
            }
            if (m == -INFINITY) {
                st = ORC_ERR_EMPTY_ROW;
                break;
            }
            double sum = 0.0;
            for (long j = 0; j < Sk; ++j) {
                P[i * Sk + j] = exp(P[i * Sk + j] - m);
                sum += P[i * Sk + j];
            }
            for (long j = 0; j < Sk; ++j) P[i * Sk + j] /= sum;
            for (long d = 0; d < D; ++d) {
                double o = 0.0;
                for (long j = 0; j < Sk; ++j) o += P[i * Sk + j] * V[j * D + d];
                O[i * D + d] = o;
            }
        }
        if (st != ORC_OK) break;
        /* Delta, dP -> dS */
        for (long i = 0; i < Sq; ++i) {
            double dl = 0.0;
            for (long d = 0; d < D; ++d) dl += G[i * D + d] * O[i * D + d];
            delta[i] = dl;
            for (long j = 0; j < Sk; ++j) {
                double dp = 0.0;
                for (long d = 0; d < D; ++d) dp += G[i * D + d] * V[j * D + d];
                dS[i * Sk + j] = P[i * Sk + j] * (dp - dl);
            }
        }
        double *dq = jb->dq + bh * Sq * D, *dk = jb->dk + bh * Sk * D, *dv = jb->dv + bh * Sk * D;
        for (long i = 0; i < Sq; ++i)
            for (long d = 0; d < D; ++d) {
                double a = 0.0;
                for (long j = 0; j < Sk; ++j) a += dS[i * Sk + j] * K[j * D + d];
                dq[i * D + d] = jb->scale * a;
            }
        for (long j = 0; j < Sk; ++j)
            for (long d = 0; d < D; ++d) {
                double a = 0.0, b = 0.0;
                for (long i = 0; i < Sq; ++i) {
                    a += dS[i * Sk + j] * Q[i * D + d];
                    b += P[i * Sk + j] * G[i * D + d];
                }
                dk[j * D + d] = jb->scale * a;
                dv[j * D + d] = b;
            }
    }
    if (st != ORC_OK) {
        pthread_mutex_lock(&jb->mu);
        if (jb->status == ORC_OK) jb->status = st;
        pthread_mutex_unlock(&jb->mu);
    }
    free(qb); free(kb); free(vb); free(gb); free(P); free(dS); free(O); free(delta);
    return NULL;
}

static int run_bwd(bwd_job_t *jb, int nthreads) {
    jb->next = 0;
    jb->status = ORC_OK;
    pthread_mutex_init(&jb->mu, NULL);
    const long n = jb->B * jb->H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)n;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    if (th)
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, bwd_worker, jb) != 0) break;
    if (started == 0) bwd_worker(jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&jb->mu);
    return jb->status;
}

static int bwd_entry(const void *q, const void *k, const void *v, const void *dout, int bf16, double *dq,
                     double *dk, double *dv, long B, long H, long Sq, long Sk, long D, double scale,
                     int causal, long wl, long wr, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || check_shape(B, H, Sq, Sk, D)) return ORC_ERR_ARG;
    bwd_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.dout = dout; jb.bf16 = bf16;
    jb.dq = dq; jb.dk = dk; jb.dv = dv;
    jb.B = B; jb.H = H; jb.Sq = Sq; jb.Sk = Sk; jb.D = D;
    jb.scale = scale; jb.causal = causal; jb.wl = wl; jb.wr = wr;
    return run_bwd(&jb, nthreads);
}

int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *dout, double *dq,
                        double *dk, double *dv, long B, long H, long Sq, long Sk, long D, double scale,
                        int causal, long wl, long wr, int nthreads) {
    return bwd_entry(q, k, v, dout, 0, dq, dk, dv, B, H, Sq, Sk, D, scale, causal, wl, wr, nthreads);
}

int oracle_attn_bwd_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                         double *dq, double *dk, double *dv, long B, long H, long Sq, long Sk, long D,
                         double scale, int causal, long wl, long wr, int nthreads) {
    return bwd_entry(q, k, v, dout, 1, dq, dk, dv, B, H, Sq, Sk, D, scale, causal, wl, wr, nthreads);
}
