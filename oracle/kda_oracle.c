/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * recurrent-state path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code,
 * header, table or helper with the CUDA library; neither includes the other.
 *
 * What it computes (per head, token by token, in double precision):
 *
 *   g_t    = -softplus(raw_gate_t)          per key channel   (alpha_t = exp(g_t))
 *   beta_t = sigmoid(raw_beta_t)            one scalar per (token, head)
 *   X      = Diag(alpha_t) S_{t-1}
 *   u_t    = beta_t (v_t - X^T k_t)
 *   S_t    = X + k_t u_t^T
 *   o_t    = S_t^T (scale q_t)
 *
 * This is the per-head KDA recurrence as the serving pages state it (the
 * "Kimi Delta Attention" state S of d_k x d_v per head, "state semantics"
 * page section 1 and the RecoverSSM page, implementation breakdown step 3).
 * The gate and beta activations follow the reading that every entry point
 * receives raw values and activates them itself (state-semantics page,
 * section 4, the kimi_linear.py comment on where gates are activated).
 *
 * Storage: the state of one head is held transposed, ST[v][k] = S[k][v]
 * (d_v rows of d_k contiguous values), the layout of the SGLang snapshot
 * store "track_state[seq, head, v_index, :]" (SGLang PR 34820 page, Helion
 * kernel listing).  Activations are [token][head][channel].
 *
 * Each entry below writes out the recurrence literally; there is no chunking,
 * blocking or reordering.  Units (sequence-or-request, head) are independent
 * and are spread over POSIX threads; each unit's arithmetic is sequential.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_GATE_LOG 1u    /* gate input already holds g (log of the decay)        */
#define ORC_BETA_ACT 2u    /* beta input already holds beta                        */
#define ORC_QK_L2NORM 32u  /* q and k of every row divided by sqrt(sum x^2 + eps)  */
#define ORC_L2NORM_EPS 1e-6

/* status bits returned by the oracle (host-side mirror of the semantics) */
#define ORC_BAD_SLOT 1
#define ORC_BAD_TRACK 2
#define ORC_BAD_ACCEPT 4
#define ORC_BAD_SEQLEN 8

/* g = -softplus(raw), written in the overflow-safe split form. */
static double orc_gate(double raw, unsigned flags)
{
    if (flags & ORC_GATE_LOG) return raw;
    if (raw > 0.0) return -(raw + log1p(exp(-raw)));
    return -log1p(exp(raw));
}

static double orc_beta(double raw, unsigned flags)
{
    if (flags & ORC_BETA_ACT) return raw;
    return 1.0 / (1.0 + exp(-raw));
}

/* The factor a row of q or k is multiplied by: 1 / sqrt(sum_i x_i^2 + eps) under
 * ORC_QK_L2NORM (the per-head L2 normalisation of the serving configurations,
 * "q, k ~ N(0,1) then L2-normalised per head", done inside the path), else 1. */
static double orc_norm(const double *x, int n, unsigned flags)
{
    if (!(flags & ORC_QK_L2NORM)) return 1.0;
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    return 1.0 / sqrt(ss + ORC_L2NORM_EPS);
}

/*
 * One recurrence step on the transposed state ST (dv rows of dk).
 * k, q, gate_raw: dk values; v: dv values.  Writes u (dv) and o (dv) if given.
 */
static void orc_step(double *ST, int dk, int dv, const double *q, const double *k,
                     const double *v, double beta_raw, const double *gate_raw,
                     double scale, unsigned flags, double *alpha_tmp, double *u_out,
                     double *o_out)
{
    double beta = orc_beta(beta_raw, flags);
    const double nk = orc_norm(k, dk, flags), nq = orc_norm(q, dk, flags);
    for (int i = 0; i < dk; ++i) alpha_tmp[i] = exp(orc_gate(gate_raw[i], flags));
    for (int c = 0; c < dv; ++c) {
        double *row = ST + (size_t)c * dk;
        /* X = Diag(alpha) S  ;  (X^T k)[c] = sum_i X[i][c] k[i] */
        double xk = 0.0;
        for (int i = 0; i < dk; ++i) {
            row[i] *= alpha_tmp[i];
            xk += row[i] * (k[i] * nk);
        }
        double u = beta * (v[c] - xk);
        /* S = X + k u^T ; o[c] = sum_i S[i][c] (scale q[i]) */
        double o = 0.0;
        for (int i = 0; i < dk; ++i) {
            row[i] += (k[i] * nk) * u;
            o += row[i] * (scale * (q[i] * nq));
        }
        if (u_out) u_out[c] = u;
        if (o_out) o_out[c] = o;
    }
}

/* ------------------------------------------------------------------------ */
/* minimal thread fan-out over independent units                             */

typedef void (*orc_unit_fn)(void *ctx, long unit, double *scratch);

typedef struct {
    orc_unit_fn fn;
    void *ctx;
    long n_units;
    int n_threads;
    int tid;
    size_t scratch_doubles;
} orc_job;

static void *orc_worker(void *p)
{
    orc_job *j = (orc_job *)p;
    double *scratch = (double *)malloc(j->scratch_doubles * sizeof(double));
    if (!scratch) return NULL;
    for (long u = j->tid; u < j->n_units; u += j->n_threads) j->fn(j->ctx, u, scratch);
    free(scratch);
    return NULL;
}

static void orc_parallel(orc_unit_fn fn, void *ctx, long n_units, int n_threads,
                         size_t scratch_doubles)
{
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long)n_threads > n_units) n_threads = (int)(n_units > 0 ? n_units : 1);
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].n_units = n_units;
        jobs[t].n_threads = n_threads;
        jobs[t].tid = t;
        jobs[t].scratch_doubles = scratch_doubles;
    }
    if (n_threads == 1) {
        orc_worker(&jobs[0]);
        return;
    }
    for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* prefill: the recurrence over each packed sequence, with snapshots         */

typedef struct {
    const double *q, *k, *v, *beta, *gate;
    const int32_t *cu_seqlens;
    int N, H, dk, dv, chunk, M;
    double scale;
    unsigned flags;
    const double *S0;           /* [N,H,dv,dk] or NULL: zero initial state */
    const int32_t *track;       /* [N,M], -1 unused */
    double *snap;               /* [N,M,H,dv,dk] */
    double *S_final;            /* [N,H,dv,dk] */
    double *out;                /* [T,H,dv] */
} orc_prefill_ctx;

static void orc_prefill_unit(void *vctx, long unit, double *scratch)
{
    orc_prefill_ctx *c = (orc_prefill_ctx *)vctx;
    const int n = (int)(unit / c->H), h = (int)(unit % c->H);
    const int dk = c->dk, dv = c->dv, H = c->H;
    const size_t ssz = (size_t)dk * dv;
    double *ST = scratch, *alpha = scratch + ssz, *o = alpha + dk;
    if (c->S0)
        memcpy(ST, c->S0 + ((size_t)n * H + h) * ssz, ssz * sizeof(double));
    else
        memset(ST, 0, ssz * sizeof(double));
    const int t0 = c->cu_seqlens[n], t1 = c->cu_seqlens[n + 1];
    for (int t = t0; t < t1; ++t) {
        const int local = t - t0;
        if (local % c->chunk == 0) {
            /* snapshot index j names the state after exactly j*chunk tokens */
            const int j = local / c->chunk;
            for (int m = 0; m < c->M; ++m)
                if (c->track[(size_t)n * c->M + m] == j)
                    memcpy(c->snap + (((size_t)n * c->M + m) * H + h) * ssz, ST,
                           ssz * sizeof(double));
        }
        const size_t th = (size_t)t * H + h;
        orc_step(ST, dk, dv, c->q + th * dk, c->k + th * dk, c->v + th * dv, c->beta[th],
                 c->gate + th * dk, c->scale, c->flags, alpha, NULL, o);
        memcpy(c->out + th * dv, o, dv * sizeof(double));
    }
    memcpy(c->S_final + ((size_t)n * H + h) * ssz, ST, ssz * sizeof(double));
}

/*
 * Returns a status bitmask (ORC_BAD_SEQLEN if cu_seqlens is not monotone,
 * ORC_BAD_TRACK if a track index lies outside [-1, n_chunks-1]).  Invalid
 * track entries simply never match, so their snapshot is left untouched.
 */
int kda_oracle_prefill(const double *q, const double *k, const double *v, const double *beta,
                       const double *gate, const int32_t *cu_seqlens, int N, int H, int dk,
                       int dv, double scale, unsigned flags, const double *S0, int chunk,
                       const int32_t *track, int M, double *snap, double *S_final,
                       double *out, int n_threads)
{
    int status = 0;
    if (cu_seqlens[0] != 0) return ORC_BAD_SEQLEN;
    for (int n = 0; n < N; ++n) {
        const int L = cu_seqlens[n + 1] - cu_seqlens[n];
        if (L < 0) return ORC_BAD_SEQLEN;
        const int n_chunks = (L + chunk - 1) / chunk;
        for (int m = 0; m < M; ++m) {
            const int j = track[(size_t)n * M + m];
            if (j < -1 || j >= n_chunks) status |= ORC_BAD_TRACK;
        }
    }
    orc_prefill_ctx c = {q, k, v, beta, gate, cu_seqlens, N, H, dk, dv, chunk, M,
                         scale, flags, S0, track, snap, S_final, out};
    orc_parallel(orc_prefill_unit, &c, (long)N * H, n_threads,
                 (size_t)dk * dv + dk + dv + 16);
    return status;
}

/* ------------------------------------------------------------------------ */
/* decode: one recurrence step per request, in place in a slot pool           */

typedef struct {
    const double *q, *k, *v, *beta, *gate;
    int R, H, dk, dv;
    double scale;
    unsigned flags;
    double *pool;
    long P;
    const int32_t *slot;
    double *out;
} orc_decode_ctx;

static void orc_decode_unit(void *vctx, long unit, double *scratch)
{
    orc_decode_ctx *c = (orc_decode_ctx *)vctx;
    const int r = (int)(unit / c->H), h = (int)(unit % c->H);
    const int dk = c->dk, dv = c->dv, H = c->H;
    const size_t th = (size_t)r * H + h;
    const int s = c->slot[r];
    if (s < 0 || s >= c->P) {
        memset(c->out + th * dv, 0, dv * sizeof(double));
        return;
    }
    double *ST = c->pool + ((size_t)s * H + h) * dk * dv;
    orc_step(ST, dk, dv, c->q + th * dk, c->k + th * dk, c->v + th * dv, c->beta[th],
             c->gate + th * dk, c->scale, c->flags, scratch, NULL, c->out + th * dv);
}

/* Slot < 0 skips the request (output row zero); slot >= P also sets ORC_BAD_SLOT. */
int kda_oracle_decode(const double *q, const double *k, const double *v, const double *beta,
                      const double *gate, int R, int H, int dk, int dv, double scale,
                      unsigned flags, double *pool, long P, const int32_t *slot, double *out,
                      int n_threads)
{
    int status = 0;
    for (int r = 0; r < R; ++r)
        if (slot[r] >= P) status |= ORC_BAD_SLOT;
    orc_decode_ctx c = {q, k, v, beta, gate, R, H, dk, dv, scale, flags, pool, P, slot, out};
    orc_parallel(orc_decode_unit, &c, (long)R * H, n_threads, (size_t)dk + 16);
    return status;
}

/* ------------------------------------------------------------------------ */
/* speculative verify: K steps from one checkpoint, never written back        */

typedef struct {
    const double *q, *k, *v, *beta, *gate;
    int R, K, H, dk, dv;
    const int32_t *q_len;
    double scale;
    unsigned flags;
    const double *pool;
    long P;
    const int32_t *ckpt;
    double *rec_u;  /* [R,H,K,dv] */
    double *rec_kg; /* [R,H,K,2dk] */
    double *out;    /* [R*K,H,dv] */
} orc_verify_ctx;

static void orc_verify_unit(void *vctx, long unit, double *scratch)
{
    orc_verify_ctx *c = (orc_verify_ctx *)vctx;
    const int r = (int)(unit / c->H), h = (int)(unit % c->H);
    const int dk = c->dk, dv = c->dv, H = c->H, K = c->K;
    const size_t ssz = (size_t)dk * dv;
    const int s = c->ckpt[r];
    int ql = c->q_len ? c->q_len[r] : K;
    const int ok = (s >= 0 && s < c->P && ql >= 0 && ql <= K);
    if (!ok) ql = 0;
    double *ST = scratch, *alpha = scratch + ssz;
    if (ok) memcpy(ST, c->pool + ((size_t)s * H + h) * ssz, ssz * sizeof(double));
    for (int t = 0; t < K; ++t) {
        const size_t row = (size_t)r * K + t, th = row * H + h;
        double *ru = c->rec_u + (((size_t)r * H + h) * K + t) * dv;
        double *rkg = c->rec_kg + (((size_t)r * H + h) * K + t) * 2 * dk;
        double *o = c->out + th * dv;
        if (t < ql) {
            orc_step(ST, dk, dv, c->q + th * dk, c->k + th * dk, c->v + th * dv, c->beta[th],
                     c->gate + th * dk, c->scale, c->flags, alpha, ru, o);
            memcpy(rkg, c->k + th * dk, dk * sizeof(double));
            memcpy(rkg + dk, c->gate + th * dk, dk * sizeof(double));
        } else {
            memset(o, 0, dv * sizeof(double));
            memset(ru, 0, dv * sizeof(double));
            memset(rkg, 0, 2 * dk * sizeof(double));
        }
    }
}

int kda_oracle_verify(const double *q, const double *k, const double *v, const double *beta,
                      const double *gate, int R, int K, const int32_t *q_len, int H, int dk,
                      int dv, double scale, unsigned flags, const double *pool, long P,
                      const int32_t *ckpt, double *rec_u, double *rec_kg, double *out,
                      int n_threads)
{
    int status = 0;
    for (int r = 0; r < R; ++r) {
        if (ckpt[r] >= P) status |= ORC_BAD_SLOT;
        if (q_len && (q_len[r] < 0 || q_len[r] > K)) status |= ORC_BAD_ACCEPT;
    }
    orc_verify_ctx c = {q,     k,     v,    beta, gate,  R,     K,      H,   dk, dv, q_len,
                        scale, flags, pool, P,    ckpt, rec_u, rec_kg, out};
    orc_parallel(orc_verify_unit, &c, (long)R * H, n_threads,
                 (size_t)dk * dv + dk + 16);
    return status;
}

/* ------------------------------------------------------------------------ */
/* commit: re-run the first a recorded steps from the checkpoint              */

typedef struct {
    double *pool;
    long P;
    const int32_t *ckpt, *dst, *acc, *q_len;
    int R, K, H, dk, dv;
    unsigned flags;
    const double *rec_u, *rec_kg;
} orc_commit_ctx;

static int orc_commit_valid(const orc_commit_ctx *c, int r)
{
    const int src = c->ckpt[r], dst = c->dst ? c->dst[r] : src;
    const int ql = c->q_len ? c->q_len[r] : c->K;
    const int a = c->acc[r];
    if (src < 0 || src >= c->P || dst < 0 || dst >= c->P) return 0;
    if (ql < 0 || ql > c->K || a < 0 || a > ql) return 0;
    return 1;
}

/*
 * Brute force: S <- Diag(alpha_t) S + k_t u_t^T for t = 1..a, where k_t and the
 * raw gate come from the key/gate record and u_t from the correction record
 * (RecoverSSM page, implementation breakdown steps 3 and 4).  a = 0 leaves the
 * checkpoint as it is and copies it when the destination differs.
 */
static void orc_commit_unit(void *vctx, long unit, double *scratch)
{
    orc_commit_ctx *c = (orc_commit_ctx *)vctx;
    const int r = (int)(unit / c->H), h = (int)(unit % c->H);
    if (!orc_commit_valid(c, r)) return;
    const int dk = c->dk, dv = c->dv, H = c->H, K = c->K;
    const size_t ssz = (size_t)dk * dv;
    const int src = c->ckpt[r], dst = c->dst ? c->dst[r] : src, a = c->acc[r];
    double *ST = scratch, *alpha = scratch + ssz;
    memcpy(ST, c->pool + ((size_t)src * H + h) * ssz, ssz * sizeof(double));
    for (int t = 0; t < a; ++t) {
        const double *u = c->rec_u + (((size_t)r * H + h) * K + t) * dv;
        const double *kg = c->rec_kg + (((size_t)r * H + h) * K + t) * 2 * dk;
        const double nk = orc_norm(kg, dk, c->flags);  /* the record holds k as given */
        for (int i = 0; i < dk; ++i) alpha[i] = exp(orc_gate(kg[dk + i], c->flags));
        for (int cc = 0; cc < dv; ++cc)
            for (int i = 0; i < dk; ++i)
                ST[(size_t)cc * dk + i] = alpha[i] * ST[(size_t)cc * dk + i] + (kg[i] * nk) * u[cc];
    }
    if (a > 0 || dst != src)
        memcpy(c->pool + ((size_t)dst * H + h) * ssz, ST, ssz * sizeof(double));
}

/*
 * plan_out[r] = (a, src, dst) for valid requests, (-1, src, dst) otherwise.
 * Returns ORC_BAD_ACCEPT / ORC_BAD_SLOT bits for skipped requests.
 */
int kda_oracle_commit(double *pool, long P, const int32_t *ckpt, const int32_t *dst,
                      const int32_t *acc, const int32_t *q_len, int R, int K, int H, int dk,
                      int dv, unsigned flags, const double *rec_u, const double *rec_kg,
                      int32_t *plan_out, int n_threads)
{
    orc_commit_ctx c = {pool, P, ckpt, dst, acc, q_len, R, K, H, dk, dv, flags, rec_u, rec_kg};
    int status = 0;
    for (int r = 0; r < R; ++r) {
        const int src = ckpt[r], d = dst ? dst[r] : src;
        const int ql = q_len ? q_len[r] : K;
        int ok = orc_commit_valid(&c, r);
        if (!ok) {
            if (src < 0 || src >= P || d < 0 || d >= P) status |= ORC_BAD_SLOT;
            else status |= ORC_BAD_ACCEPT;
        }
        (void)ql;
        if (plan_out) {
            plan_out[3 * r + 0] = ok ? acc[r] : -1;
            plan_out[3 * r + 1] = src;
            plan_out[3 * r + 2] = d;
        }
    }
    orc_parallel(orc_commit_unit, &c, (long)R * H, n_threads, (size_t)dk * dv + dk + 16);
    return status;
}
