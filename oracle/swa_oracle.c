/*
 * swa_oracle.c -- fp64 CPU oracle for causal / sliding-window attention with
 * grouped-query heads: forward (output and per-row logsumexp) and the
 * closed-form softmax backward (dq, dk, dv).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion or reordering.  There are Lq query rows and Lk >= Lq key rows; the
 * queries are the last Lq positions of the key sequence, so query i sits at
 * position a = i + off with off = Lk - Lq (off = 0 for self-attention):
 *
 *   s_ij  = scale * q_i . k_j                         for every key j < Lk
 *   s_ij  = -inf  when j is outside band(i)
 *   causal:      band(i) = { j : j <= a  and  (W == 0  or  a - j < W) }
 *   non-causal:  band(i) = { j : W == 0  or  |a - j| < W }
 *   lse_i = m_i + ln sum_j exp(s_ij - m_i),  m_i = max_j s_ij
 *   P_ij  = exp(s_ij - lse_i)                  (exactly 0 outside the band)
 *   o_i   = sum_j P_ij v_j
 *   dP_ij = dO_i . v_j
 *   Delta_i = sum_j P_ij dP_ij                 (checked against dO_i . o_i)
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dq_i  = scale * sum_j dS_ij k_j
 *   dk_j  = scale * sum_{h in group} sum_i dS_ij q_i
 *   dv_j  = sum_{h in group} sum_i P_ij dO_i
 *
 * Shared prompt prefix ("Training -- design (ORPO, flash-CCE head, prefix
 * sharing, segmented backward)", section 5.4 "Shared prompt-prefix
 * forward"): one self-attention pass over [prompt (P rows); chosen response
 * (Rc rows); rejected response (Rr rows)], L = P + Rc + Rr, with the
 * block-sparse mask "causal AND NOT rejected->chosen" and the window measured
 * on logical positions, where each response starts at logical position P
 * (block-wise positions).  Written out, with lp(x) = x - Rc for x >= P + Rc
 * (a rejected row) and lp(x) = x otherwise:
 *
 *   key j visible to query i  iff  j <= i
 *                              and not (i >= P + Rc and P <= j < P + Rc)
 *                              and (W == 0 or lp(i) - lp(j) < W)
 *
 * The *_px entry points take (P, Rc); they are causal self-attention.
 *
 * Attention sinks (the *_sk entry points): one logit c_h per query head, a
 * term of every row's softmax normaliser that carries no value.  The pages
 * name sinks only as a parameter of the attention backward primitive,
 * beside scale and causal ("Lab 028 lab detail: Off NVIDIA, you fix the
 * platform yourself", "What I changed, in plain terms" item 2); the reading
 * taken is the per-head logit that the softmax normalises against:
 *
 *   lse_i = ln( sum_j exp(s_ij) + exp(c_h) )
 *   P_ij  = exp(s_ij - lse_i),   o_i = sum_j P_ij v_j
 *   dq, dk, dv and Delta_i as above (with this lse)
 *   dc_h  = - sum_{b, i} exp(c_h - lse_i) Delta_i
 *
 * The last line is d(loss)/dc_h: c_h enters o_i only through lse_i, and
 * d o_i / d c_h = -exp(c_h - lse_i) o_i, so the chain rule with dO_i gives
 * -exp(c_h - lse_i) dO_i . o_i = -exp(c_h - lse_i) Delta_i.  A sink of -inf
 * is no sink.
 *
 * Passages followed:
 *  - Mask rule: "Lab 028 lab detail: Off NVIDIA, you fix the platform
 *    yourself", "Plan for the build" step 4 (P is zeroed where
 *    j < i + diag_off - window_size + 1) and "What I changed, in plain
 *    terms" item 4 (a key that is window_size or more positions from the
 *    query's diagonal is zeroed); causal tiles above the diagonal are skipped
 *    ("What the code says", with the diagonal shifted by diag_off).  A window
 *    of 0 is read as no window.  The same page's item 3 (a non-causal window
 *    also skips tiles more than window_size ahead) and item 6 (windows tested
 *    "causal and not", including qL < kL) give the non-causal band and the
 *    suffix case; item 5(b) says keys behind every query's window get zero
 *    dK and dV, which the definition below gives (every term is zero).
 *  - Forward writes the logsumexp, the per-row softmax normaliser the
 *    backward reuses: same page, "What I changed, in plain terms" item 1.
 *  - Backward stores the per-row LSE and recomputes P: "Training -- design
 *    (ORPO, flash-CCE head, prefix sharing, segmented backward)" section 6
 *    "Kernel-fusion notes"; ground truth is the dense matmul / softmax
 *    decomposition of section 5.2 "Attention backward".
 *  - Grouped-query heads: query head h reads kv head h / (Hq / Hkv):
 *    "MiniCPM5 Decode Megakernel -- end-to-end build plan", section 4.1
 *    stage 5 and section 6 "Pitfalls".
 *
 * Layout: every tensor is row-major [B, H, L, D] (lse / delta [B, Hq, L]).
 * Inputs are either raw bf16 bit patterns (uint16) or fp64; bf16 values are
 * widened exactly to fp64.  All arithmetic is fp64.
 *
 * The backward is organised in two passes over the definition: a row pass
 * (per query row: s, lse, P, o, Delta, dq) and a column pass (per key row:
 * dk, dv, summing over every query row and every head of the group in
 * ascending order).  Both passes evaluate the same formulas above; the
 * column pass takes lse_i and Delta_i from the row pass.
 *
 * "band_only" skips the key (or query) positions outside the band.  Those
 * terms are exact zeros (exp(-inf) = 0), and the in-band terms are summed in
 * the same ascending order, so both modes give bitwise-equal results; this
 * is checked by a test.  It exists only to make the timed CPU baseline finish
 * on long sequences.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const void *q, *k, *v, *dO;
    int is_f64;               /* 1: fp64 arrays, 0: bf16 bit patterns */
    long B, Hq, Hkv, Lq, Lk, D, W;
    int causal;
    double scale;
    int band_only;
    long off;                 /* Lk - Lq: position of query 0 among the keys */
    int plan;                 /* 1: shared-prefix mask over [prompt; chosen; rejected] */
    long P, Rc;               /* prompt and chosen-response lengths (plan only) */
    const double* sinks;      /* [Hq] sink logits, or NULL for none */
} ctx_t;

/* Logical position of sequence position x under the shared-prefix plan: the
 * rejected response restarts at logical position P, right after the prompt. */
static long logical_pos(const ctx_t* c, long x) {
    return (c->plan && x >= c->P + c->Rc) ? x - c->Rc : x;
}

static double bf16_bits_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double ld(const ctx_t* c, const void* base, long idx) {
    if (c->is_f64) return ((const double*)base)[idx];
    return bf16_bits_to_f64(((const uint16_t*)base)[idx]);
}

/* Offset of query-side row i (q, dO, o, dq) of head h of batch b. */
static long qrow_off(const ctx_t* c, long b, long h, long i) {
    return ((b * c->Hq + h) * c->Lq + i) * c->D;
}

/* Offset of key-side row j (k, v, dk, dv) of kv head kvh of batch b. */
static long krow_off(const ctx_t* c, long b, long kvh, long j) {
    return ((b * c->Hkv + kvh) * c->Lk + j) * c->D;
}

/* Key j is visible to query i (at position a = i + off). */
static int in_band(const ctx_t* c, long i, long j) {
    const long a = i + c->off;
    if (c->plan) {
        if (j > i) return 0;                                          /* causal */
        if (i >= c->P + c->Rc && j >= c->P && j < c->P + c->Rc) return 0;  /* rejected -> chosen */
        if (c->W > 0 && logical_pos(c, i) - logical_pos(c, j) >= c->W) return 0;
        return 1;
    }
    if (c->causal) {
        if (j > a) return 0;
        if (c->W > 0 && a - j >= c->W) return 0;
        return 1;
    }
    if (c->W > 0 && (a - j >= c->W || j - a >= c->W)) return 0;
    return 1;
}

/* Range of key positions the row pass visits for query i. */
static void key_range(const ctx_t* c, long i, long* j0, long* j1) {
    *j0 = 0;
    *j1 = c->Lk - 1;
    if (!c->band_only) return;
    const long a = i + c->off;
    if (c->plan) {
        /* the smallest visible key has logical position lp(i) - W + 1 (a
           prompt key, or a key of i's own segment); keys in between that
           the mask drops are exact zeros */
        const long lo = logical_pos(c, i) - c->W + 1;
        if (c->W > 0 && lo > 0) *j0 = lo;
        *j1 = i;
        return;
    }
    if (c->W > 0 && a - c->W + 1 > 0) *j0 = a - c->W + 1;
    if (c->causal) *j1 = a;
    else if (c->W > 0 && a + c->W - 1 < c->Lk - 1) *j1 = a + c->W - 1;
}

/* Range of query rows the column pass visits for key j (empty if i1 < i0). */
static void query_range(const ctx_t* c, long j, long* i0, long* i1) {
    *i0 = 0;
    *i1 = c->Lq - 1;
    if (!c->band_only) return;
    if (c->plan) {
        /* rows i >= j with lp(i) <= lp(j) + W - 1; a rejected row sits Rc
           positions after its logical position */
        *i0 = j;
        if (c->W > 0 && logical_pos(c, j) + c->W - 1 + c->Rc < *i1) *i1 = logical_pos(c, j) + c->W - 1 + c->Rc;
        return;
    }
    /* positions a that see key j: a >= j (causal) or a >= j - W + 1
       (non-causal window), and a <= j + W - 1 (any window) */
    long alo = c->causal ? j : (c->W > 0 ? j - c->W + 1 : c->off);
    if (alo - c->off > *i0) *i0 = alo - c->off;
    if (c->W > 0 && j + c->W - 1 - c->off < *i1) *i1 = j + c->W - 1 - c->off;
}

/*
 * Row pass for query row i of head h (batch b).  s and dp are scratch of Lk
 * doubles.  Writes o_row[D], *lse; when dO is given also *delta (sum_j P dP),
 * *delta_alt (dO_i . o_i) and, if dq_row is not NULL, dq_row[D].
 */
static void row_pass(const ctx_t* c, long b, long h, long i, double* s, double* dp,
                     double* o_row, double* lse, double* delta, double* delta_alt,
                     double* dq_row) {
    const long D = c->D;
    const long kvh = h / (c->Hq / c->Hkv);
    const long qo = qrow_off(c, b, h, i);
    long j0, j1;
    key_range(c, i, &j0, &j1);

    /* scores */
    double m = -INFINITY;
    for (long j = j0; j <= j1; ++j) {
        if (!in_band(c, i, j)) { s[j] = -INFINITY; continue; }
        const long ko = krow_off(c, b, kvh, j);
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += ld(c, c->q, qo + d) * ld(c, c->k, ko + d);
        s[j] = c->scale * acc;
        if (s[j] > m) m = s[j];
    }
    /* logsumexp (with the head's sink logit as one more term) */
    const double sink = c->sinks ? c->sinks[h] : -INFINITY;
    if (sink > m) m = sink;
    double sum = 0.0;
    for (long j = j0; j <= j1; ++j) sum += exp(s[j] - m);
    if (c->sinks) sum += exp(sink - m);
    const double lse_i = m + log(sum);
    *lse = lse_i;
    /* output */
    for (long d = 0; d < D; ++d) o_row[d] = 0.0;
    for (long j = j0; j <= j1; ++j) {
        const double p = exp(s[j] - lse_i);
        const long vo = krow_off(c, b, kvh, j);
        for (long d = 0; d < D; ++d) o_row[d] += p * ld(c, c->v, vo + d);
    }
    if (!c->dO) return;

    /* dP, Delta (both forms) */
    const long go = qrow_off(c, b, h, i);
    double dl = 0.0;
    for (long j = j0; j <= j1; ++j) {
        const long vo = krow_off(c, b, kvh, j);
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += ld(c, c->dO, go + d) * ld(c, c->v, vo + d);
        dp[j] = acc;
        dl += exp(s[j] - lse_i) * acc;
    }
    double da = 0.0;
    for (long d = 0; d < D; ++d) da += ld(c, c->dO, go + d) * o_row[d];
    *delta = dl;
    *delta_alt = da;
    if (!dq_row) return;

    /* dq */
    for (long d = 0; d < D; ++d) dq_row[d] = 0.0;
    for (long j = j0; j <= j1; ++j) {
        const double p = exp(s[j] - lse_i);
        const double ds = p * (dp[j] - dl);
        const long ko = krow_off(c, b, kvh, j);
        for (long d = 0; d < D; ++d) dq_row[d] += c->scale * ds * ld(c, c->k, ko + d);
    }
}

/*
 * Column pass for key row j of kv head kvh (batch b): dk_row[D], dv_row[D].
 * lse and delta are [B, Hq, Lq] arrays from the row pass; only the rows of
 * the group's heads that can see key j are read.
 */
static void col_pass(const ctx_t* c, long b, long kvh, long j, const double* lse,
                     const double* delta, double* dk_row, double* dv_row) {
    const long D = c->D;
    const long G = c->Hq / c->Hkv;
    const long ko = krow_off(c, b, kvh, j);
    long i0, i1;
    query_range(c, j, &i0, &i1);
    for (long d = 0; d < D; ++d) { dk_row[d] = 0.0; dv_row[d] = 0.0; }
    for (long g = 0; g < G; ++g) {
        const long h = kvh * G + g;
        for (long i = i0; i <= i1; ++i) {
            const long qo = qrow_off(c, b, h, i);
            const long ri = (b * c->Hq + h) * c->Lq + i;
            double s;
            if (in_band(c, i, j)) {
                double acc = 0.0;
                for (long d = 0; d < D; ++d) acc += ld(c, c->q, qo + d) * ld(c, c->k, ko + d);
                s = c->scale * acc;
            } else {
                s = -INFINITY;
            }
            const double p = exp(s - lse[ri]);
            double dpv = 0.0;
            for (long d = 0; d < D; ++d) dpv += ld(c, c->dO, qo + d) * ld(c, c->v, ko + d);
            const double ds = p * (dpv - delta[ri]);
            for (long d = 0; d < D; ++d) {
                dk_row[d] += c->scale * ds * ld(c, c->q, qo + d);
                dv_row[d] += p * ld(c, c->dO, qo + d);
            }
        }
    }
}

static int check_shape(long B, long Hq, long Hkv, long Lq, long Lk, long D, long W) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < Lq || D < 1 || W < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

static ctx_t make_ctx(const void* q, const void* k, const void* v, const void* dO, int is_f64, long B,
                      long Hq, long Hkv, long Lq, long Lk, long D, long W, int causal, double scale,
                      int band_only) {
    ctx_t c = {q, k, v, dO, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal ? 1 : 0, scale, band_only, Lk - Lq, 0, 0, 0,
               NULL};
    return c;
}

/* The shared-prefix plan, for self-attention over L = Lq = Lk rows.  A plan
 * needs 0 <= P and 0 <= Rc with P + Rc <= L. */
static int set_plan(ctx_t* c, long P, long Rc) {
    if (P < 0 || Rc < 0 || P + Rc > c->Lk || c->Lq != c->Lk) return -1;
    c->plan = 1;
    c->P = P;
    c->Rc = Rc;
    c->causal = 1;
    return 0;
}

int swa_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over every row.  o: [B,Hq,Lq,D], lse: [B,Hq,Lq]. */
static int fwd_impl(const ctx_t* cp, double* o, double* lse) {
    const ctx_t c = *cp;
    const long B = c.B, Hq = c.Hq, Lq = c.Lq, Lk = c.Lk, D = c.D;
    const long rows = B * Hq * Lq;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        if (!s) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s) continue;
            const long i = r % Lq, bh = r / Lq, h = bh % Hq, b = bh / Hq;
            row_pass(&c, b, h, i, s, NULL, o + r * D, lse + r, NULL, NULL, NULL);
        }
        free(s);
    }
    return err;
}

/*
 * Forward and backward over every row and key.  Outputs o, dq: [B,Hq,Lq,D];
 * dk, dv: [B,Hkv,Lk,D]; lse, delta: [B,Hq,Lq].  *delta_gap receives
 * max_i |sum_j P dP - dO_i . o_i|.
 */
static int bwd_impl(const ctx_t* cp, double* o, double* lse, double* delta, double* dq, double* dk,
                    double* dv, double* delta_gap) {
    const ctx_t c = *cp;
    const long B = c.B, Hq = c.Hq, Hkv = c.Hkv, Lq = c.Lq, Lk = c.Lk, D = c.D;
    const long rows = B * Hq * Lq;
    const long keys = B * Hkv * Lk;
    double gap = 0.0;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
        double my_gap = 0.0;
        if (!s || !dp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s || !dp) continue;
            const long i = r % Lq, bh = r / Lq, h = bh % Hq, b = bh / Hq;
            double da;
            row_pass(&c, b, h, i, s, dp, o + r * D, lse + r, delta + r, &da, dq + r * D);
            const double g = fabs(delta[r] - da);
            if (g > my_gap) my_gap = g;
        }
#pragma omp critical
        if (my_gap > gap) gap = my_gap;
        free(s);
        free(dp);
    }
    if (err) return err;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < keys; ++r) {
        const long j = r % Lk, bh = r / Lk, kvh = bh % Hkv, b = bh / Hkv;
        col_pass(&c, b, kvh, j, lse, delta, dk + r * D, dv + r * D);
    }
    if (delta_gap) *delta_gap = gap;
    return 0;
}

/*
 * Selected query rows of one head: o, dq [n, D]; lse, delta [n].
 * dO may be NULL (forward only; delta and dq are then left untouched).
 */
static int rows_impl(const ctx_t* cp, long b, long h, const long* rows, long n, double* o, double* lse,
                     double* delta, double* dq) {
    const ctx_t c = *cp;
    const void* dO = c.dO;
    const long D = c.D, Lk = c.Lk;
    if (b < 0 || b >= c.B || h < 0 || h >= c.Hq) return -1;
    for (long t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= c.Lq) return -1;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
        if (!s || !dp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < n; ++t) {
            if (!s || !dp) continue;
            double da;
            row_pass(&c, b, h, rows[t], s, dp, o + t * D, lse + t, dO ? delta + t : NULL, &da,
                     dO ? dq + t * D : NULL);
        }
        free(s);
        free(dp);
    }
    return err;
}

/*
 * Selected key rows of one kv head: dk, dv [n, D].  First runs the row pass
 * for every query row, of every head in the group, that can see one of the
 * selected keys (lse_i and Delta_i), then the column pass for each key.
 */
static int key_rows_impl(const ctx_t* cp, long b, long kvh, const long* keys, long n, double* dk,
                         double* dv) {
    const ctx_t c = *cp;
    const long B = c.B, Hq = c.Hq, Hkv = c.Hkv, Lq = c.Lq, Lk = c.Lk, D = c.D;
    if (b < 0 || b >= B || kvh < 0 || kvh >= Hkv || n < 1 || !c.dO) return -1;
    for (long t = 0; t < n; ++t)
        if (keys[t] < 0 || keys[t] >= Lk) return -1;
    const long G = Hq / Hkv;
    /* query rows that can see any selected key (the others add exact zeros) */
    long ilo = Lq, ihi = -1;
    ctx_t cb = c;
    cb.band_only = 1;
    for (long t = 0; t < n; ++t) {
        long a, z;
        query_range(&cb, keys[t], &a, &z);
        if (a <= z) {
            if (a < ilo) ilo = a;
            if (z > ihi) ihi = z;
        }
    }
    if (ihi < ilo) { ilo = 0; ihi = -1; }
    const long nr = ihi - ilo + 1;
    /* lse / delta laid out as full [B, Hq, Lq] arrays so col_pass can index them */
    double* lse = (double*)calloc((size_t)(B * Hq * Lq), sizeof(double));
    double* delta = (double*)calloc((size_t)(B * Hq * Lq), sizeof(double));
    double* obuf = (double*)malloc(sizeof(double) * (size_t)((G * nr > 0 ? G * nr : 1) * D));
    if (!lse || !delta || !obuf) {
        free(lse); free(delta); free(obuf);
        return -2;
    }
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
        if (!s || !dp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < G * nr; ++r) {
            if (!s || !dp) continue;
            const long g = r / nr, i = ilo + r % nr, h = kvh * G + g;
            const long ri = (b * Hq + h) * Lq + i;
            double da;
            row_pass(&c, b, h, i, s, dp, obuf + r * D, lse + ri, delta + ri, &da, NULL);
        }
        free(s);
        free(dp);
    }
    if (!err) {
#pragma omp parallel for schedule(dynamic, 1)
        for (long t = 0; t < n; ++t) col_pass(&c, b, kvh, keys[t], lse, delta, dk + t * D, dv + t * D);
    }
    free(lse);
    free(delta);
    free(obuf);
    return err;
}

/* Forward over every row.  o: [B,Hq,Lq,D], lse: [B,Hq,Lq]. */
int swa_oracle_fwd_ex(const void* q, const void* k, const void* v, int is_f64, long B, long Hq,
                      long Hkv, long Lq, long Lk, long D, long W, int causal, double scale,
                      int band_only, double* o, double* lse) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W)) return -1;
    const ctx_t c = make_ctx(q, k, v, NULL, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, band_only);
    return fwd_impl(&c, o, lse);
}

/*
 * Forward and backward over every row and key.  Outputs o, dq: [B,Hq,Lq,D];
 * dk, dv: [B,Hkv,Lk,D]; lse, delta: [B,Hq,Lq].  *delta_gap receives
 * max_i |sum_j P dP - dO_i . o_i|.
 */
int swa_oracle_bwd_ex(const void* q, const void* k, const void* v, const void* dO, int is_f64,
                      long B, long Hq, long Hkv, long Lq, long Lk, long D, long W, int causal,
                      double scale, int band_only, double* o, double* lse, double* delta,
                      double* dq, double* dk, double* dv, double* delta_gap) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W)) return -1;
    const ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, band_only);
    return bwd_impl(&c, o, lse, delta, dq, dk, dv, delta_gap);
}

/*
 * Selected query rows of one head: o, dq [n, D]; lse, delta [n].
 * dO may be NULL (forward only; delta and dq are then left untouched).
 */
int swa_oracle_rows_ex(const void* q, const void* k, const void* v, const void* dO, int is_f64,
                       long B, long Hq, long Hkv, long Lq, long Lk, long D, long W, int causal,
                       double scale, int band_only, long b, long h, const long* rows, long n,
                       double* o, double* lse, double* delta, double* dq) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W)) return -1;
    const ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, band_only);
    return rows_impl(&c, b, h, rows, n, o, lse, delta, dq);
}

/*
 * Selected key rows of one kv head: dk, dv [n, D].  First runs the row pass
 * for every query row, of every head in the group, that can see one of the
 * selected keys (lse_i and Delta_i), then the column pass for each key.
 */
int swa_oracle_key_rows_ex(const void* q, const void* k, const void* v, const void* dO,
                           int is_f64, long B, long Hq, long Hkv, long Lq, long Lk, long D, long W,
                           int causal, double scale, int band_only, long b, long kvh,
                           const long* keys, long n, double* dk, double* dv) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W)) return -1;
    const ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, band_only);
    return key_rows_impl(&c, b, kvh, keys, n, dk, dv);
}

/* The same four over [prompt (P); chosen (Rc); rejected (L - P - Rc)] with
 * the shared-prefix mask (causal self-attention, Lq = Lk = L). */
int swa_oracle_fwd_px(const void* q, const void* k, const void* v, int is_f64, long B, long Hq, long Hkv,
                      long L, long D, long W, long P, long Rc, double scale, int band_only, double* o,
                      double* lse) {
    if (check_shape(B, Hq, Hkv, L, L, D, W)) return -1;
    ctx_t c = make_ctx(q, k, v, NULL, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only);
    if (set_plan(&c, P, Rc)) return -1;
    return fwd_impl(&c, o, lse);
}

int swa_oracle_bwd_px(const void* q, const void* k, const void* v, const void* dO, int is_f64, long B,
                      long Hq, long Hkv, long L, long D, long W, long P, long Rc, double scale,
                      int band_only, double* o, double* lse, double* delta, double* dq, double* dk,
                      double* dv, double* delta_gap) {
    if (check_shape(B, Hq, Hkv, L, L, D, W)) return -1;
    ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only);
    if (set_plan(&c, P, Rc)) return -1;
    return bwd_impl(&c, o, lse, delta, dq, dk, dv, delta_gap);
}

int swa_oracle_rows_px(const void* q, const void* k, const void* v, const void* dO, int is_f64, long B,
                       long Hq, long Hkv, long L, long D, long W, long P, long Rc, double scale,
                       int band_only, long b, long h, const long* rows, long n, double* o, double* lse,
                       double* delta, double* dq) {
    if (check_shape(B, Hq, Hkv, L, L, D, W)) return -1;
    ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only);
    if (set_plan(&c, P, Rc)) return -1;
    return rows_impl(&c, b, h, rows, n, o, lse, delta, dq);
}

int swa_oracle_key_rows_px(const void* q, const void* k, const void* v, const void* dO, int is_f64, long B,
                           long Hq, long Hkv, long L, long D, long W, long P, long Rc, double scale,
                           int band_only, long b, long kvh, const long* keys, long n, double* dk,
                           double* dv) {
    if (check_shape(B, Hq, Hkv, L, L, D, W)) return -1;
    ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only);
    if (set_plan(&c, P, Rc)) return -1;
    return key_rows_impl(&c, b, kvh, keys, n, dk, dv);
}

/* Self-attention (Lq = Lk = L), causal: the entry points the tests started with. */
int swa_oracle_fwd(const void* q, const void* k, const void* v, int is_f64, long B, long Hq,
                   long Hkv, long L, long D, long W, double scale, int band_only, double* o,
                   double* lse) {
    return swa_oracle_fwd_ex(q, k, v, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only, o, lse);
}

int swa_oracle_bwd(const void* q, const void* k, const void* v, const void* dO, int is_f64,
                   long B, long Hq, long Hkv, long L, long D, long W, double scale,
                   int band_only, double* o, double* lse, double* delta, double* dq,
                   double* dk, double* dv, double* delta_gap) {
    return swa_oracle_bwd_ex(q, k, v, dO, is_f64, B, Hq, Hkv, L, L, D, W, 1, scale, band_only, o, lse,
                             delta, dq, dk, dv, delta_gap);
}

/*
 * With attention sinks (see the header): sinks [Hq] fp64.  The forward and
 * backward are those of the _ex entry points with the sink term in every
 * row's normaliser; the backward also writes dsinks [Hq], summed over the
 * batch and the rows in ascending order.
 */
int swa_oracle_fwd_sk(const void* q, const void* k, const void* v, const double* sinks, int is_f64, long B,
                      long Hq, long Hkv, long Lq, long Lk, long D, long W, int causal, double scale, double* o,
                      double* lse) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W) || !sinks) return -1;
    ctx_t c = make_ctx(q, k, v, NULL, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, 0);
    c.sinks = sinks;
    return fwd_impl(&c, o, lse);
}

int swa_oracle_bwd_sk(const void* q, const void* k, const void* v, const void* dO, const double* sinks,
                      int is_f64, long B, long Hq, long Hkv, long Lq, long Lk, long D, long W, int causal,
                      double scale, double* o, double* lse, double* delta, double* dq, double* dk, double* dv,
                      double* dsinks, double* delta_gap) {
    if (check_shape(B, Hq, Hkv, Lq, Lk, D, W) || !sinks || !dsinks) return -1;
    ctx_t c = make_ctx(q, k, v, dO, is_f64, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, 0);
    c.sinks = sinks;
    const int err = bwd_impl(&c, o, lse, delta, dq, dk, dv, delta_gap);
    if (err) return err;
    for (long h = 0; h < Hq; ++h) {
        double acc = 0.0;
        for (long b = 0; b < B; ++b)
            for (long i = 0; i < Lq; ++i) {
                const long r = (b * Hq + h) * Lq + i;
                acc += exp(sinks[h] - lse[r]) * delta[r];
            }
        dsinks[h] = -acc;
    }
    return 0;
}
