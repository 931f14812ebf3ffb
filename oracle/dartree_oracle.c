/*
 * DARTree supertree oracle: a plain, slow, single-threaded CPU definition of
 * what the GPU build computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls this file.
 * Only the tests, the package smoke check and the bench's CPU-baseline /
 * reference leg load it.  It shares no code, header, table or constant with
 * the CUDA path; both sides are fed the same seeded host arrays.
 *
 * Sources (page title -- section):
 *   [P1] "DARTree: Teaching a Chain-Trained Corrector to Think in Trees"
 *        -- Core Mechanism (level-by-level construction; best-first pruning
 *        on scores already computed), Key Concepts (marginal vs conditional),
 *        Framework Shift (one head call per depth, not per node).
 *   [P2] "Technische Samenvatting: DARTree" -- Methodologie, 1. Depth-Wise
 *        Parallel AR Expansie (batched correction, cumulative corrected
 *        score, keep top-W and carry correction states) and 2. Deferred
 *        Best-First Pruning (one global Top-B over all materialised prefixes;
 *        Lemma 1: with a non-positive depth bonus it equals a sequential
 *        best-first max-heap).
 *   [P3] "Accelerating Language Models with Diffusion Draft Trees" -- Summary
 *        & Methodology Analysis (a global top-W over each depth's children,
 *        state update, global top-B, prefix tree verified with a tree-attention
 *        mask).
 *
 * The correction head's architecture is not given by the pages.  The fixed
 * synthetic stand-in used throughout is
 *      s'      = q(tanh(A s + E[tok]))          (state after committing tok)
 *      logits  = z_d + s' Wout^T                 (corrected logits at depth d)
 * with q() = round to bf16 (nearest, ties to even) when the weights are bf16
 * and the identity when they are fp32.  The root state is q(state0).
 *
 * Precision (readings where the pages are silent): every dot product, the
 * tanh and the log-sum-exp are evaluated in double; logits and log-probs are
 * rounded to fp32 once; cumulative scores and Top-B keys are single fp32
 * operations in the stated order.  Build with -ffp-contract=off so that no
 * multiply-add is fused.
 *
 * Orders (readings; the pages give no tie-breaks):
 *   top-K of a row      : (logit desc, token asc)
 *   top-W of candidates : (score desc, candidate index i*K+j asc)
 *   Top-B of the pool   : (key desc, pool index asc), key = score + beta*depth
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_CLOSURE 2
#define ORC_ERR_ORDER 3
#define ORC_ERR_MEM 4

int orc_version(void) { return 1; }

/* ---------------------------------------------------------------- helpers */

/* bf16 bit pattern -> value: the 16 bits are the top half of an fp32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double weight(const void *w, int bf16, size_t i) {
    if (bf16) return bf16_to_double(((const uint16_t *)w)[i]);
    return (double)((const float *)w)[i];
}

/* Round an fp32 value to bf16 precision, nearest with ties to even, by its
 * definition: keep the top 16 bits, adding half an ulp of the kept part
 * (minus one when the kept part is even, so that exact halves go to even). */
float orc_round_bf16(float x) {
    uint32_t u;
    if (x != x) {                                    /* NaN stays a NaN */
        u = 0x7FC00000u;
    } else {                                         /* finite or inf */
        memcpy(&u, &x, sizeof u);
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
        u &= 0xFFFF0000u;
    }
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

static float qstate(int bf16, float x) { return bf16 ? orc_round_bf16(x) : x; }

/* "a is better than b" under (value desc, index asc). */
static int better(float va, int64_t ia, float vb, int64_t ib) {
    return va > vb || (va == vb && ia < ib);
}

/* ------------------------------------------------------- head (stand-in) */

/* State after committing token tok on top of the parent's state:
 * s_out[h] = q( tanh( sum_j A[h,j] s_par[j] + E[tok,h] ) ).
 * [P2] Methodologie 1 ("carries their correction states forward"),
 * [P3] Summary ("updates their states").
 * A == NULL is the Markov head: the state is a function of the last token
 * alone, s_out[h] = q(tanh(E[tok,h])) -- the A = 0 case of the same form.
 * [P2] Experimentele Resultaten, Ablatie (Generaliseerbaarheid: the DSpark
 * drafter with a Markov correction head). */
void orc_state_step(int H, int bf16, const void *A, const void *E,
                    const float *s_par, int32_t tok, float *s_out) {
    for (int h = 0; h < H; ++h) {
        double u = 0.0;
        if (A)
            for (int j = 0; j < H; ++j)
                u += weight(A, bf16, (size_t)h * H + j) * (double)s_par[j];
        u += weight(E, bf16, (size_t)tok * H + h);
        s_out[h] = qstate(bf16, (float)tanh(u));
    }
}

/* Corrected logits of one path and their log-sum-exp over the vocabulary.
 * ell[v] = fp32( z_d[v] + sum_h s[h] Wout[v,h] );
 * lse    = m + log sum_v exp(ell[v] - m), m = max ell, in double.
 * [P1] Core Mechanism (one corrected distribution per branch, conditioned
 * on that branch's own tokens). */
void orc_logits_row(int V, int H, int bf16, const float *z_d, const void *Wout,
                    const float *s, float *ell, double *lse) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double acc = (double)z_d[v];
        for (int h = 0; h < H; ++h)
            acc += (double)s[h] * weight(Wout, bf16, (size_t)v * H + h);
        ell[v] = (float)acc;
        if ((double)ell[v] > m) m = (double)ell[v];
    }
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    double sum = 0.0;
    for (int v = 0; v < V; ++v) sum += exp((double)ell[v] - m);
    *lse = m + log(sum);
}

/* Top-K of one row by (logit desc, token asc), by insertion into a sorted
 * list.  gap = ell_(K) - ell_(K+1) (+inf when V == K).
 * [P1] Core Mechanism (every frontier node is expanded by its K best
 * children). */
void orc_topk_row(int V, const float *ell, int K, int32_t *tok, float *val,
                  float *gap) {
    int n = 0;
    for (int v = 0; v < V; ++v) {
        if (n == K && !better(ell[v], v, val[K - 1], tok[K - 1])) continue;
        int p = (n < K) ? n : K - 1;
        while (p > 0 && better(ell[v], v, val[p - 1], tok[p - 1])) {
            val[p] = val[p - 1];
            tok[p] = tok[p - 1];
            --p;
        }
        val[p] = ell[v];
        tok[p] = v;
        if (n < K) ++n;
    }
    /* the (K+1)-th value: best entry not in the list */
    float next = -INFINITY;
    int32_t next_tok = -1;
    for (int v = 0; v < V; ++v) {
        int in = 0;
        for (int j = 0; j < K; ++j)
            if (tok[j] == v) { in = 1; break; }
        if (in) continue;
        if (next_tok < 0 || better(ell[v], v, next, next_tok)) {
            next = ell[v];
            next_tok = v;
        }
    }
    *gap = (next_tok < 0) ? INFINITY : val[K - 1] - next;
}

/* Base-logit candidate variant of one head row.  The K candidates ctok are
 * the top-K of the base logits z_d (shared by every branch); the row's
 * corrected logits are evaluated at those tokens only,
 *   e_j = fp32( z_d[c_j] + sum_h s[h] Wout[c_j,h] ),
 * and normalised over the K candidates: lse = m + log sum_j exp(e_j - m).
 * Output: the K candidates ordered by (e desc, token asc) in tok/val.
 * [P2] Methodologie 1 (Kandidaat Selectie: top-K candidate tokens from the
 * base logits at every depth; Gebatchte Correctie: the correction head
 * evaluates those candidates for all branches in one batch). */
void orc_cand_row(int H, int bf16, const float *z_d, const void *Wout,
                  const float *s, int K, const int32_t *ctok, int32_t *tok,
                  float *val, double *lse) {
    for (int j = 0; j < K; ++j) {                 /* insertion by (e, token) */
        int32_t c = ctok[j];
        double acc = (double)z_d[c];
        for (int h = 0; h < H; ++h)
            acc += (double)s[h] * weight(Wout, bf16, (size_t)c * H + h);
        float e = (float)acc;
        int p = j;
        while (p > 0 && better(e, c, val[p - 1], tok[p - 1])) {
            val[p] = val[p - 1];
            tok[p] = tok[p - 1];
            --p;
        }
        val[p] = e;
        tok[p] = c;
    }
    double m = (double)val[0];
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    double sum = 0.0;
    for (int j = 0; j < K; ++j) sum += exp((double)val[j] - m);
    *lse = m + log(sum);
}

/* --------------------------------------------------------- construction */

typedef struct { float c; int32_t idx; } cand_t;

static int cand_cmp(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (better(x->c, x->idx, y->c, y->idx)) return -1;
    if (better(y->c, y->idx, x->c, x->idx)) return 1;
    return 0;
}

/* Frontier sizes: |F_0| = 1, |F_d| = min(W, K |F_{d-1}|). */
static int frontier(int d, int W, int K) {
    int f = 1;
    for (int i = 0; i < d; ++i) f = (K * f < W) ? K * f : W;
    return f;
}

int orc_pool_size(int D, int W, int K) {
    int p = 0;
    for (int d = 1; d <= D; ++d) p += frontier(d, W, K);
    return p;
}

/*
 * One depth of the construction, callable on its own so that any depth of a
 * build can be replayed from given frontier states and scores.
 * [P1] Core Mechanism: the frontier's paths go through the head in ONE call;
 * each is expanded by its top-k children, ranked by cumulative path
 * log-probability; the W best survive.  [P2] Methodologie 1 and [P3] Summary:
 * one global top-W over the depth's children.
 *
 * Inputs: fp frontier rows with head states st [fp][H] and cumulative scores
 * score [fp]; the depth's base logits zd [V]; Wout [V,H] (bf16 bits or fp32).
 * cand_base != 0 takes the candidates from the base logits (orc_cand_row);
 * the row gap reported is then the base logits' K/K+1 gap, which alone
 * decides the candidate set.
 *   head call (one per depth): ell_i = corrected logits, lse_i, top-K of ell_i;
 *   candidates: c_ij = score[i] + logp_ij (one fp32 add), index i*K + j;
 *   own top-W : the first fd = min(W, fp*K) candidates by (c desc, index asc).
 * The kept frontier is force_slot/force_tok [fd] when given (teacher
 * forcing: slot in [0, fp), token in [0, V)), else the own top-W; the oracle
 * scores forced nodes in its own arithmetic.
 *
 * Outputs: own_slot/own_tok/own_score [fd]; kept frontier sel_slot/sel_tok,
 * sel_score (cumulative) and sel_logp (its log-prob given its parent) [fd];
 * force_margin [fd] = ell(slot, tok) - ell_(K)(slot) for forced nodes, else 0;
 * per row row_lse [fp], row_tok/row_logp [fp*K], row_kgap [fp]; w_cut [2] =
 * own W-th and (W+1)-th candidate score (-inf if none).
 */
int orc_depth(int V, int H, int fp, int W, int K, int bf16, int cand_base,
              const float *zd, const void *Wout, const float *st, const float *score,
              const int32_t *force_slot, const int32_t *force_tok,
              int32_t *own_slot, int32_t *own_tok, float *own_score,
              int32_t *sel_slot, int32_t *sel_tok, float *sel_score, float *sel_logp,
              float *force_margin, double *row_lse, int32_t *row_tok, float *row_logp,
              float *row_kgap, float *w_cut) {
    if (V < 1 || H < 1 || fp < 1 || W < 1 || K < 1 || K > V) return ORC_ERR_ARG;
    int rc = ORC_OK;
    const int fd = (K * fp < W) ? K * fp : W;
    float *ell = malloc(sizeof(float) * (size_t)fp * V);     /* full rows */
    cand_t *cand = malloc(sizeof(cand_t) * (size_t)fp * K);
    float *kth = malloc(sizeof(float) * (size_t)fp);         /* K-th logit */
    int32_t *tk = malloc(sizeof(int32_t) * (size_t)K);
    float *tv = malloc(sizeof(float) * (size_t)K);
    int32_t *ctok = malloc(sizeof(int32_t) * (size_t)K);    /* base candidates */
    float *cval = malloc(sizeof(float) * (size_t)K);
    if (!ell || !cand || !kth || !tk || !tv || !ctok || !cval) {
        rc = ORC_ERR_MEM;
        goto done;
    }

    float zgap = 0.0f;
    if (cand_base) orc_topk_row(V, zd, K, ctok, cval, &zgap);
    /* the batched head call over every frontier row */
    for (int i = 0; i < fp; ++i) {
        double lse;
        float kgap;
        if (cand_base) {
            orc_cand_row(H, bf16, zd, Wout, st + (size_t)i * H, K, ctok, tk, tv, &lse);
            for (int j = 0; j < K; ++j) ell[(size_t)i * V + tk[j]] = tv[j];
            kgap = zgap;     /* the candidate set is decided by z alone */
        } else {
            orc_logits_row(V, H, bf16, zd, Wout, st + (size_t)i * H,
                           ell + (size_t)i * V, &lse);
            orc_topk_row(V, ell + (size_t)i * V, K, tk, tv, &kgap);
        }
        row_lse[i] = lse;
        row_kgap[i] = kgap;
        kth[i] = tv[K - 1];
        for (int j = 0; j < K; ++j) {
            float logp = (float)((double)tv[j] - lse);
            row_tok[(size_t)i * K + j] = tk[j];
            row_logp[(size_t)i * K + j] = logp;
            cand[i * K + j].c = score[i] + logp;       /* one fp32 add */
            cand[i * K + j].idx = i * K + j;
        }
    }
    /* own global top-W over the fp*K candidates */
    qsort(cand, (size_t)fp * K, sizeof(cand_t), cand_cmp);
    for (int q = 0; q < fd; ++q) {
        own_slot[q] = cand[q].idx / K;
        own_tok[q] = row_tok[(size_t)own_slot[q] * K + cand[q].idx % K];
        own_score[q] = cand[q].c;
    }
    w_cut[0] = cand[fd - 1].c;
    w_cut[1] = (fp * K > fd) ? cand[fd].c : -INFINITY;

    /* the frontier that is kept: forced or own */
    for (int q = 0; q < fd; ++q) {
        int32_t slot, tok;
        if (force_slot) {
            slot = force_slot[q];
            tok = force_tok[q];
            if (slot < 0 || slot >= fp || tok < 0 || tok >= V) {
                rc = ORC_ERR_ARG;
                goto done;
            }
            if (cand_base) {              /* only a candidate can be kept */
                int in = 0;
                for (int j = 0; j < K; ++j) in |= (ctok[j] == tok);
                if (!in) { rc = ORC_ERR_ARG; goto done; }
            }
            float e = ell[(size_t)slot * V + tok];
            sel_logp[q] = (float)((double)e - row_lse[slot]);
            sel_score[q] = score[slot] + sel_logp[q];
            force_margin[q] = cand_base ? 0.0f : e - kth[slot];
        } else {
            slot = own_slot[q];
            tok = own_tok[q];
            sel_score[q] = own_score[q];
            sel_logp[q] = row_logp[(size_t)slot * K + cand[q].idx % K];
            force_margin[q] = 0.0f;
        }
        sel_slot[q] = slot;
        sel_tok[q] = tok;
    }

done:
    free(ell); free(cand); free(kth); free(tk); free(tv); free(ctok); free(cval);
    return rc;
}

/*
 * Depth-wise batched construction of the supertree for one request.
 * [P1] Core Mechanism: at depth d the W surviving paths go through the head
 * in ONE call; each is expanded by its top-k children (W*k candidates),
 * ranked by cumulative path log-probability; the W best survive; after D levels
 * exactly D head calls have been made and a pool of scored nodes is held.
 * [P2] Methodologie 1 and [P3] Summary: one global top-W over each depth's
 * children, whose correction states go on to the next depth.
 *
 * Inputs: z [D,V] fp32, state0 [H] fp32, A [H,H], E [V,H], Wout [V,H]
 * (bf16 bits or fp32).  Depth 1 has |F_1| = min(W, K) nodes.
 * A == NULL selects the Markov head (see orc_state_step).  cand_base != 0
 * takes each depth's candidates from the base logits (see orc_depth).
 *
 * Teacher forcing: when force_slot/force_tok are given ([P] each, laid out
 * like the pool), the frontier kept at each depth is the forced one (parent
 * slot in F_{d-1}, token) instead of the oracle's own top-W; the oracle still
 * records its own choice and scores the forced nodes in its own arithmetic.
 * When force_state is given ([D][W][H] fp32), the head rows of depth d use
 * those states instead of the oracle's own (state-level forcing, to compare
 * each head call on identical inputs: the bf16-rounded tanh recurrence
 * amplifies accumulation-order differences from depth to depth).
 *
 * Outputs ([P] = pool size, rows = W per depth):
 *   pool_parent/token/depth/score [P]: the pool that was kept, pool index =
 *       depth-major, rank order within a depth; parent -1 at depth 1;
 *       pool_logp [P] (may be NULL): each kept node's log-prob given its parent.
 *   own_slot/own_tok/own_score [P]: the oracle's own top-W at each depth
 *       given the kept previous frontier.
 *   force_margin [P]: for kept nodes, ell(parent,tok) - ell_(K)(parent).
 *   row_lse [D*W], row_tok/row_logp [D*W*K], row_kgap [D*W]: per head row.
 *   w_cut [2*D]: own W-th and (W+1)-th candidate score (-inf if none).
 *   calls: number of batched head calls made (== D).
 */
int orc_build_ex(int V, int H, int D, int W, int K, int bf16, int cand_base,
                 const float *z, const float *state0,
                 const void *A, const void *E, const void *Wout,
                 const int32_t *force_slot, const int32_t *force_tok,
                 const float *force_state,
                 int32_t *pool_parent, int32_t *pool_token, int32_t *pool_depth,
                 float *pool_score, float *pool_logp,
                 int32_t *own_slot, int32_t *own_tok, float *own_score,
                 float *force_margin,
                 double *row_lse, int32_t *row_tok, float *row_logp,
                 float *row_kgap, float *w_cut, int64_t *calls) {
    if (V < 1 || H < 1 || D < 1 || W < 1 || K < 1 || K > V) return ORC_ERR_ARG;
    int rc = ORC_OK;
    float *st = malloc(sizeof(float) * (size_t)W * H);      /* row states */
    float *st_next = malloc(sizeof(float) * (size_t)W * H);
    float *score = malloc(sizeof(float) * (size_t)W);        /* row scores */
    int32_t *sel_slot = malloc(sizeof(int32_t) * (size_t)W);
    int32_t *sel_tok = malloc(sizeof(int32_t) * (size_t)W);
    float *sel_score = malloc(sizeof(float) * (size_t)W);
    float *sel_logp = malloc(sizeof(float) * (size_t)W);
    if (!st || !st_next || !score || !sel_slot || !sel_tok || !sel_score || !sel_logp) {
        rc = ORC_ERR_MEM;
        goto done;
    }

    *calls = 0;
    int fp = 1, off_prev = 0, off = 0;
    for (int h = 0; h < H; ++h) st[h] = qstate(bf16, state0[h]);  /* root */
    score[0] = 0.0f;

    for (int d = 1; d <= D; ++d) {
        int fd = (K * fp < W) ? K * fp : W;
        if (force_state)
            memcpy(st, force_state + (size_t)(d - 1) * W * H, sizeof(float) * (size_t)fp * H);
        *calls += 1;                   /* one batched head call per depth */
        size_t r0 = (size_t)(d - 1) * W;
        rc = orc_depth(V, H, fp, W, K, bf16, cand_base, z + (size_t)(d - 1) * V, Wout, st,
                       score, force_slot ? force_slot + off : NULL,
                       force_tok ? force_tok + off : NULL, own_slot + off, own_tok + off,
                       own_score + off, sel_slot, sel_tok, sel_score, sel_logp,
                       force_margin + off, row_lse + r0, row_tok + r0 * K, row_logp + r0 * K,
                       row_kgap + r0, w_cut + 2 * (d - 1));
        if (rc != ORC_OK) goto done;
        for (int q = 0; q < fd; ++q) {
            pool_parent[off + q] = (d == 1) ? -1 : off_prev + sel_slot[q];
            pool_token[off + q] = sel_tok[q];
            pool_depth[off + q] = d;
            pool_score[off + q] = sel_score[q];
            if (pool_logp) pool_logp[off + q] = sel_logp[q];
        }
        /* carry the correction states forward to the kept nodes */
        if (d < D) {
            for (int q = 0; q < fd; ++q)
                orc_state_step(H, bf16, A, E, st + (size_t)sel_slot[q] * H,
                               sel_tok[q], st_next + (size_t)q * H);
            float *t = st; st = st_next; st_next = t;
        }
        for (int q = 0; q < fd; ++q) score[q] = sel_score[q];
        off_prev = off;
        off += fd;
        fp = fd;
    }

done:
    free(st); free(st_next); free(score); free(sel_slot); free(sel_tok);
    free(sel_score); free(sel_logp);
    return rc;
}

/* Cumulative path scores of a pool from each node's log-prob given its parent:
 * score[n] = score[parent[n]] + logp[n] (one fp32 add), 0 + logp[n] at depth 1
 * (parent -1).  Parents precede their children in pool order.  Returns
 * ORC_ERR_ORDER if a parent index is not below its child's.
 * [P1] Core Mechanism (children ranked by accumulated path log-probability). */
int orc_path_scores(int P, const int32_t *parent, const float *logp, float *score) {
    for (int n = 0; n < P; ++n) {
        int32_t p = parent[n];
        if (p >= n) return ORC_ERR_ORDER;
        score[n] = (p < 0 ? 0.0f : score[p]) + logp[n];
    }
    return ORC_OK;
}

/* The construction with the candidates of [P1] (top-K of each branch's
 * corrected distribution over the whole vocabulary). */
int orc_build(int V, int H, int D, int W, int K, int bf16,
              const float *z, const float *state0,
              const void *A, const void *E, const void *Wout,
              const int32_t *force_slot, const int32_t *force_tok,
              const float *force_state,
              int32_t *pool_parent, int32_t *pool_token, int32_t *pool_depth,
              float *pool_score,
              int32_t *own_slot, int32_t *own_tok, float *own_score,
              float *force_margin,
              double *row_lse, int32_t *row_tok, float *row_logp,
              float *row_kgap, float *w_cut, int64_t *calls) {
    return orc_build_ex(V, H, D, W, K, bf16, 0, z, state0, A, E, Wout,
                        force_slot, force_tok, force_state, pool_parent,
                        pool_token, pool_depth, pool_score, NULL, own_slot, own_tok,
                        own_score, force_margin, row_lse, row_tok, row_logp,
                        row_kgap, w_cut, calls);
}

/* ------------------------------------------------------ deferred pruning */

typedef struct { float key; int32_t idx; } key_t_;

static int key_cmp(const void *a, const void *b) {
    const key_t_ *x = (const key_t_ *)a, *y = (const key_t_ *)b;
    if (better(x->key, x->idx, y->key, y->idx)) return -1;
    if (better(y->key, y->idx, x->key, x->idx)) return 1;
    return 0;
}

/* key = score + beta * depth, two fp32 operations in that order. */
static float prune_key(float score, int32_t depth, float beta) {
    float bd = beta * (float)depth;
    return score + bd;
}

/*
 * Deferred global Top-B, compaction and the tree-attention mask.
 * [P2] Methodologie 2: one global Top-B over every materialised prefix of
 * the supertree, with a non-positive depth bonus; [P1] Core Mechanism: the
 * selected nodes form the verification tree, and its ancestor mask lets a
 * single target forward verify all branches at once; [P3] Summary.
 *
 * Canonical output order = the selection order (key desc, pool index asc).
 * out_parent = rank of the parent in that order (-1 at depth 1).
 * out_mask: B rows of ceil(B/32) words; bit j%32 of word j/32 of row i is
 * set iff node j is node i or one of its ancestors.  Rows at or beyond
 * n_out are parent/token -1, depth 0, score 0, mask 0.
 * order[r] = pool index of rank r.  Returns ORC_ERR_CLOSURE when a selected
 * node's parent is not selected, ORC_ERR_ORDER when a parent ranks after its
 * child (neither can happen for beta <= 0; see Lemma 1).
 */
int orc_topb(int P, const int32_t *pool_parent, const int32_t *pool_token,
             const int32_t *pool_depth, const float *pool_score, int B,
             float beta, int32_t *out_parent, int32_t *out_token,
             int32_t *out_depth, float *out_score, uint32_t *out_mask,
             int32_t *n_out, int32_t *order) {
    if (P < 0 || B < 1) return ORC_ERR_ARG;
    int rc = ORC_OK;
    int words = (B + 31) / 32;
    key_t_ *k = malloc(sizeof(key_t_) * (size_t)(P > 0 ? P : 1));
    int32_t *map = malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    if (!k || !map) { rc = ORC_ERR_MEM; goto done; }
    for (int n = 0; n < P; ++n) {
        k[n].key = prune_key(pool_score[n], pool_depth[n], beta);
        k[n].idx = n;
        map[n] = -1;
    }
    qsort(k, (size_t)P, sizeof(key_t_), key_cmp);
    int n_sel = P < B ? P : B;
    *n_out = n_sel;
    for (int r = 0; r < n_sel; ++r) {
        order[r] = k[r].idx;
        map[k[r].idx] = r;
    }
    memset(out_mask, 0, sizeof(uint32_t) * (size_t)B * words);
    for (int r = 0; r < B; ++r) {
        if (r >= n_sel) {
            out_parent[r] = -1; out_token[r] = -1; out_depth[r] = 0;
            out_score[r] = 0.0f;
            continue;
        }
        int n = order[r];
        int32_t pp = pool_parent[n];
        int32_t par = (pp < 0) ? -1 : map[pp];
        if (pp >= 0 && par < 0) { rc = ORC_ERR_CLOSURE; par = -1; }
        if (par >= r) { rc = ORC_ERR_ORDER; par = -1; }
        out_parent[r] = par;
        out_token[r] = pool_token[n];
        out_depth[r] = pool_depth[n];
        out_score[r] = pool_score[n];
        uint32_t *row = out_mask + (size_t)r * words;
        if (par >= 0) memcpy(row, out_mask + (size_t)par * words,
                             sizeof(uint32_t) * (size_t)words);
        row[r / 32] |= 1u << (r % 32);
    }
done:
    free(k); free(map);
    return rc;
}

/*
 * Sequential best-first pruning on the pool's stored scores with a max-heap:
 * seed with the depth-1 nodes, then B times pop the best node and push its
 * children from the pool.  [P1] Core Mechanism (the best-first pruning works
 * on scores already computed, so its sequential heap steps run no model);
 * Expert Assessment (EAGLE-2's heap moved
 * after the forwards).  Used to check Lemma 1 against orc_topb.
 * pop_order[r] = pool index popped at step r; returns the number of pops.
 */
int orc_heap_prune(int P, const int32_t *pool_parent, const int32_t *pool_depth,
                   const float *pool_score, int B, float beta,
                   int32_t *pop_order) {
    key_t_ *heap = malloc(sizeof(key_t_) * (size_t)(P > 0 ? P : 1));
    if (!heap) return -ORC_ERR_MEM;
    int hn = 0, pops = 0;
    /* push = sift up; "max" under (key desc, idx asc) */
#define ORC_PUSH(node)                                                        \
    do {                                                                      \
        key_t_ e_ = { prune_key(pool_score[node], pool_depth[node], beta),   \
                      (int32_t)(node) };                                      \
        int i_ = hn++;                                                        \
        while (i_ > 0) {                                                      \
            int p_ = (i_ - 1) / 2;                                            \
            if (!better(e_.key, e_.idx, heap[p_].key, heap[p_].idx)) break;   \
            heap[i_] = heap[p_];                                              \
            i_ = p_;                                                          \
        }                                                                     \
        heap[i_] = e_;                                                        \
    } while (0)
    for (int n = 0; n < P; ++n)
        if (pool_parent[n] < 0) ORC_PUSH(n);
    while (pops < B && hn > 0) {
        key_t_ top = heap[0];
        key_t_ last = heap[--hn];
        int i = 0;
        for (;;) {                                    /* sift down */
            int l = 2 * i + 1, r = l + 1, b = i;
            key_t_ bv = last;
            if (l < hn && better(heap[l].key, heap[l].idx, bv.key, bv.idx)) {
                b = l; bv = heap[l];
            }
            if (r < hn && better(heap[r].key, heap[r].idx, bv.key, bv.idx)) {
                b = r; bv = heap[r];
            }
            if (b == i) break;
            heap[i] = heap[b];
            i = b;
        }
        if (hn > 0) heap[i] = last;
        pop_order[pops++] = top.idx;
        for (int n = 0; n < P; ++n)
            if (pool_parent[n] == top.idx) ORC_PUSH(n);
    }
#undef ORC_PUSH
    free(heap);
    return pops;
}

/* ------------------------------------------- sequential best-first build */

/*
 * Node-by-node best-first construction with one head call per expanded
 * node: the sequential baseline that DARTree's depth-wise batching replaces.
 * [P2] Probleemstelling (Causale Correctie: a standard best-first build with
 * a max-heap makes the correction head run node by node -- pop one node,
 * correct it, push its children, and only then expand the next) and
 * Experimentele Resultaten, Ablatie (latency of the sequential heap build);
 * [P1] Core Mechanism (the expansion by top-k children and the scores).
 *
 * Nodes get ids in order of creation.  Head call 0 expands the root (state
 * q(state0), score 0, children at depth 1 from z_1).  Then for rank
 * q = 0 .. B-1: pop the best node under (key desc, id asc), key = score +
 * beta*depth (the orc_topb key); it becomes output rank q.  If q + 1 < B and
 * its depth d < D, head call q + 1 expands it: its state is the state step
 * of its parent's state (the root's for depth 1) with its token, the call
 * scores its children at depth d + 1 (z_{d+1}), and its top-K children are
 * created in rank order with score = node score + logp (one fp32 add);
 * otherwise call q + 1 is not made.  Stops early when no node is left.
 *
 * Children come from the corrected top-K as in orc_build.  Teacher forcing:
 * force_tok/force_logp ([B][K], by call) replace the children of each call
 * (the call's own row is still computed and reported); force_state ([B][H],
 * by call) replaces the state the call is made with.
 *
 * Outputs: the tree in pop order (parent rank, -1 at depth 1; token; depth;
 * score; ancestor mask as in orc_topb), n_out, call_rank[B] (rank expanded
 * by each call, -1 for the root, -2 if the call was not made), the call
 * states call_state[B][H], per-call rows (row_lse [B], row_tok/row_logp
 * [B][K], row_kgap [B]) and calls = head calls made.
 */
int orc_bestfirst(int V, int H, int D, int K, int B, int bf16, float beta,
                  const float *z, const float *state0,
                  const void *A, const void *E, const void *Wout,
                  const int32_t *force_tok, const float *force_logp,
                  const float *force_state,
                  int32_t *out_parent, int32_t *out_token, int32_t *out_depth,
                  float *out_score, uint32_t *out_mask, int32_t *n_out,
                  int32_t *call_rank, float *call_state,
                  double *row_lse, int32_t *row_tok, float *row_logp,
                  float *row_kgap, int64_t *calls) {
    if (V < 1 || H < 1 || D < 1 || K < 1 || K > V || B < 1) return ORC_ERR_ARG;
    int rc = ORC_OK;
    const int words = (B + 31) / 32;
    const int max_nodes = B * K;
    int32_t *n_par = malloc(sizeof(int32_t) * (size_t)max_nodes);   /* parent id */
    int32_t *n_tok = malloc(sizeof(int32_t) * (size_t)max_nodes);
    int32_t *n_dep = malloc(sizeof(int32_t) * (size_t)max_nodes);
    float *n_score = malloc(sizeof(float) * (size_t)max_nodes);
    int32_t *n_rank = malloc(sizeof(int32_t) * (size_t)max_nodes);  /* -1: not popped */
    key_t_ *heap = malloc(sizeof(key_t_) * (size_t)max_nodes);
    float *s_root = malloc(sizeof(float) * (size_t)H);
    float *s_rank = malloc(sizeof(float) * (size_t)B * H);           /* state per rank */
    float *ell = malloc(sizeof(float) * (size_t)V);
    int32_t *tk = malloc(sizeof(int32_t) * (size_t)K);
    float *tv = malloc(sizeof(float) * (size_t)K);
    if (!n_par || !n_tok || !n_dep || !n_score || !n_rank || !heap || !s_root ||
        !s_rank || !ell || !tk || !tv) {
        rc = ORC_ERR_MEM;
        goto done;
    }
    for (int h = 0; h < H; ++h) s_root[h] = qstate(bf16, state0[h]);
    for (int c = 0; c < B; ++c) call_rank[c] = -2;
    memset(out_mask, 0, sizeof(uint32_t) * (size_t)B * words);
    for (int q = 0; q < B; ++q) {
        out_parent[q] = -1; out_token[q] = -1; out_depth[q] = 0; out_score[q] = 0.0f;
    }
    *calls = 0;
    int n_nodes = 0, hn = 0, pops = 0;
    int expand = -1;                 /* node expanded by the next call: -1 = root */
    for (int c = 0; c < B; ++c) {
        if (expand >= -1) {
            /* ---- head call c expands the root (c = 0) or rank c-1 */
            int dep = (expand < 0) ? 0 : n_dep[expand];
            float sc = (expand < 0) ? 0.0f : n_score[expand];
            float *s = call_state + (size_t)c * H;
            if (expand < 0) {
                memcpy(s, s_root, sizeof(float) * (size_t)H);
            } else {
                int p = n_par[expand];
                const float *sp = (p < 0) ? s_root : s_rank + (size_t)n_rank[p] * H;
                orc_state_step(H, bf16, A, E, sp, n_tok[expand], s);
            }
            if (force_state) memcpy(s, force_state + (size_t)c * H, sizeof(float) * (size_t)H);
            if (expand >= 0) memcpy(s_rank + (size_t)n_rank[expand] * H, s, sizeof(float) * (size_t)H);
            call_rank[c] = (expand < 0) ? -1 : n_rank[expand];
            *calls += 1;
            double lse;
            float kgap;
            orc_logits_row(V, H, bf16, z + (size_t)dep * V, Wout, s, ell, &lse);
            orc_topk_row(V, ell, K, tk, tv, &kgap);
            row_lse[c] = lse;
            row_kgap[c] = kgap;
            for (int j = 0; j < K; ++j) {
                row_tok[(size_t)c * K + j] = tk[j];
                row_logp[(size_t)c * K + j] = (float)((double)tv[j] - lse);
            }
            /* ---- its children enter the heap, ids in rank order */
            for (int j = 0; j < K; ++j) {
                int id = n_nodes++;
                n_par[id] = expand;
                n_tok[id] = force_tok ? force_tok[(size_t)c * K + j] : row_tok[(size_t)c * K + j];
                float lp = force_logp ? force_logp[(size_t)c * K + j] : row_logp[(size_t)c * K + j];
                n_dep[id] = dep + 1;
                n_score[id] = sc + lp;                   /* one fp32 add */
                n_rank[id] = -1;
                key_t_ e = { prune_key(n_score[id], n_dep[id], beta), id };
                int i = hn++;                            /* sift up */
                while (i > 0) {
                    int pi = (i - 1) / 2;
                    if (!better(e.key, e.idx, heap[pi].key, heap[pi].idx)) break;
                    heap[i] = heap[pi];
                    i = pi;
                }
                heap[i] = e;
            }
        }
        /* ---- pop rank c */
        expand = -2;
        if (hn == 0) break;
        key_t_ top = heap[0];
        key_t_ last = heap[--hn];
        int i = 0;
        for (;;) {                                       /* sift down */
            int l = 2 * i + 1, r = l + 1, b = i;
            key_t_ bv = last;
            if (l < hn && better(heap[l].key, heap[l].idx, bv.key, bv.idx)) { b = l; bv = heap[l]; }
            if (r < hn && better(heap[r].key, heap[r].idx, bv.key, bv.idx)) { b = r; bv = heap[r]; }
            if (b == i) break;
            heap[i] = heap[b];
            i = b;
        }
        if (hn > 0) heap[i] = last;
        int m = top.idx, q = pops++;
        n_rank[m] = q;
        int pr = (n_par[m] < 0) ? -1 : n_rank[n_par[m]];
        out_parent[q] = pr;
        out_token[q] = n_tok[m];
        out_depth[q] = n_dep[m];
        out_score[q] = n_score[m];
        uint32_t *row = out_mask + (size_t)q * words;
        if (pr >= 0) memcpy(row, out_mask + (size_t)pr * words, sizeof(uint32_t) * (size_t)words);
        row[q / 32] |= 1u << (q % 32);
        if (n_dep[m] < D) expand = m;                    /* call c+1 expands it */
    }
    *n_out = pops;
done:
    free(n_par); free(n_tok); free(n_dep); free(n_score); free(n_rank);
    free(heap); free(s_root); free(s_rank); free(ell); free(tk); free(tv);
    return rc;
}

/* ------------------------------------------- verification: tree attention */

/*
 * One attention layer of the target's verification forward over the prefix
 * and the draft tree.  [P1] Core Mechanism (with the tree and its mask a
 * single target forward verifies all branches, and the longest prefix the
 * target agrees with is kept); [P2] Methodologie 2
 * (Verificatie: one forward pass with tree attention); [P3] Summary.
 *
 * Query rows: row 0 is the root (the last verified token, whose key and
 * value are the last prefix position), rows 1..B are the tree nodes in the
 * build's canonical order.  Row 0 attends to the Lp prefix positions; row
 * i >= 1 attends to the prefix and to the tree nodes j with bit j of mask
 * row i-1 (its ancestors and itself).  Grouped heads: query head h reads
 * key/value head h / (Hq / Hkv).
 *   O[i,h] = sum_j softmax_j(scale * q[i,h] . k[j,h']) v[j,h']   (fp64)
 * Layouts (one request): Q [B+1][Hq][dh], Kp/Vp [Lp][Hkv][dh],
 * Kt/Vt [B][Hkv][dh] (bf16 bits or fp32 as `bf16` says), mask [B][words],
 * O [B+1][Hq][dh] fp32.
 */
int orc_tree_attention(int Lp, int B, int Hq, int Hkv, int dh, int bf16, float scale,
                       const void *Q, const void *Kp, const void *Vp,
                       const void *Kt, const void *Vt, const uint32_t *mask,
                       float *O) {
    if (Lp < 0 || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || dh < 1 || Lp + B < 1)
        return ORC_ERR_ARG;
    const int words = (B + 31) / 32;
    const int g = Hq / Hkv;
    double *s = malloc(sizeof(double) * (size_t)(Lp + B > 0 ? Lp + B : 1));
    if (!s) return ORC_ERR_MEM;
    for (int i = 0; i <= B; ++i) {
        for (int h = 0; h < Hq; ++h) {
            const int hk = h / g;
            const size_t qo = ((size_t)i * Hq + h) * dh;
            double m = -INFINITY;
            /* scores of every key the row may see; -inf for the others */
            for (int j = 0; j < Lp + B; ++j) {
                int visible;
                const void *K;
                size_t ko;
                if (j < Lp) {
                    visible = 1;
                    K = Kp;
                    ko = ((size_t)j * Hkv + hk) * dh;
                } else {
                    const int t = j - Lp;
                    visible = i >= 1 && ((mask[(size_t)(i - 1) * words + t / 32] >> (t % 32)) & 1u);
                    K = Kt;
                    ko = ((size_t)t * Hkv + hk) * dh;
                }
                if (!visible) { s[j] = -INFINITY; continue; }
                double acc = 0.0;
                for (int c = 0; c < dh; ++c)
                    acc += weight(Q, bf16, qo + c) * weight(K, bf16, ko + c);
                s[j] = (double)scale * acc;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < Lp + B; ++j) l += (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
            for (int c = 0; c < dh; ++c) {
                double acc = 0.0;
                for (int j = 0; j < Lp + B; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const size_t vo = (j < Lp) ? ((size_t)j * Hkv + hk) * dh
                                               : ((size_t)(j - Lp) * Hkv + hk) * dh;
                    acc += exp(s[j] - m) * weight(j < Lp ? Vp : Vt, bf16, vo + c);
                }
                O[qo + c] = (l > 0.0) ? (float)(acc / l) : 0.0f;
            }
        }
    }
    free(s);
    return ORC_OK;
}

/*
 * Longest accepted prefix.  pred[0] is the target's token after the root,
 * pred[i] (i = 1..B) its token after tree node i-1.  Starting at the root,
 * the child (among the first n_out nodes, parent rank = current node, -1 for
 * the root) whose token equals the current node's prediction is accepted
 * and becomes the current node; siblings carry distinct tokens, so at most
 * one child matches.  [P1] Core Mechanism (the longest prefix the target
 * agrees with is accepted).  Outputs: accept_len, accept_nodes[0..accept_len) (ranks),
 * bonus = the prediction at the last accepted node (the root's if none).
 */
int orc_accept(int B, int n_out, const int32_t *parent, const int32_t *token,
               const int32_t *pred, int32_t *accept_len, int32_t *accept_nodes,
               int32_t *bonus) {
    if (B < 0 || n_out < 0 || n_out > B) return ORC_ERR_ARG;
    int cur = -1, len = 0;
    for (;;) {
        const int32_t want = pred[cur + 1];
        int next = -1;
        for (int n = 0; n < n_out; ++n)
            if (parent[n] == cur && token[n] == want) { next = n; break; }
        if (next < 0) break;
        accept_nodes[len++] = next;
        cur = next;
    }
    *accept_len = len;
    *bonus = pred[cur + 1];
    return ORC_OK;
}
