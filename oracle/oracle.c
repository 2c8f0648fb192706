/*
 * oracle.c -- plain, slow fp64 CPU oracle for the selected-token logprob and
 * the train/rollout mismatch statistics.
 *
 * TEST INFRASTRUCTURE.  Only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this code.  It
 * shares nothing with the CUDA library (no header, no helper, no table) and
 * neither side includes or links the other.
 *
 * Everything is computed in double from the exact values of the inputs
 * (bf16 and fp32 convert to double exactly).  No blocking, fusion or
 * reordering: every sum runs in index order exactly as the definition reads.
 *
 * Sources (page title + section):
 *  - token logprob: icarus "RL: Training Inference Mismatch", section "log p"
 *    (hidden state -> LM head -> log-softmax -> gather at the token id, and
 *    its PyTorch statement log_softmax(logits, -1).gather(-1, ids)); LoongSage
 *    "Train-Inference Consistency" section 3 "FP32 LM head" (the head is
 *    computed at higher precision than bf16).  The pages' head has a bias;
 *    the library's call has none, so neither has this oracle.
 *  - mismatch: VeXact summary page, "Formal Definition" eq. (1)
 *    (delta = log pi_train - log pi_rollout) and "KL Estimators" (K1 = -log r,
 *    K3 = (r - 1) - log r); llm-infra-atlas section 2 (Delta = l_theta - l_mu,
 *    r = e^Delta); icarus "KL estimators" table (k2 = 0.5 (log r)^2) and
 *    "monitoring" steps 2-3 (mean over a completion's tokens, then mean over
 *    completions); icarus compute_consistency_and_kl_metrics
 *    (rel_diff = |delta| / (|logp_train| + 1e-8), masked mean); LoongSage
 *    section 4 (IS weight pi_old/pi_rollout, clipped when out of bounds) and
 *    section 5 (is_approx_k3_kl, is_clip_ratio, is_nan_ratio); VeXact
 *    "Algorithmic TIM Compensation" (sequence rejection on K3 / K1 of
 *    r_corr = pi_train / pi_rollout, thresholds tau_seq).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - w = min(r, C) (one-sided truncation), clip = r > C (strict);
 *  - a token "used" = mask != 0 and delta finite; a masked token with a
 *    non-finite delta counts as nan, gets w = 0 and is left out of the means;
 *  - integer decisions (finite, clip) use delta rounded to fp32, the
 *    precision the device computes it in; values use the exact fp64 delta;
 *  - log r is taken as delta itself (r = e^delta by definition), and
 *    r - 1 as expm1(delta), so that k3 does not lose digits to cancellation;
 *  - a sequence with no used token has all means 0, flag 0, and is left out
 *    of the mean over sequences;
 *  - rejection: mean k3 > tau (estimator 3) or |mean k1| > tau (estimator 1),
 *    strict; tau NaN means the default k3(C) = (C - 1) - ln C.
 *  - target outside [0, V) (the -100 ignore label): logp = NaN, lse valid.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ token logprob */

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One row of the definition: z_v = (sum_d h_d W[v, d]) / temperature
 * (d ascending; the sampling distribution softmax(z / tau) of the icarus
 * "logits processor" section, tau = 1 for raw logits), m = max_v z_v,
 * S = sum_v exp(z_v - m) (v ascending), lse = m + log S, logp = z_a - lse.
 * W is bf16 (W) or, for the FP32 LM head of LoongSage "Train-Inference
 * Consistency" section 3, fp32 (Wf, used when not NULL). */
static void oracle_row(const uint16_t *h_row, const uint16_t *W, const float *Wf, int32_t a,
                       int64_t D, int64_t V, double temperature, double *hd, double *z,
                       double *out_logp, double *out_lse)
{
    for (int64_t d = 0; d < D; ++d)
        hd[d] = bf16_value(h_row[d]);
    for (int64_t v = 0; v < V; ++v) {
        double acc = 0.0;
        if (Wf) {
            const float *w = Wf + v * D;
            for (int64_t d = 0; d < D; ++d)
                acc += hd[d] * (double)w[d];
        } else {
            const uint16_t *w = W + v * D;
            for (int64_t d = 0; d < D; ++d)
                acc += hd[d] * bf16_value(w[d]);
        }
        z[v] = acc / temperature;
    }
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (z[v] > m)
            m = z[v];
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v)
        S += exp(z[v] - m);
    double lse = m + log(S);
    *out_lse = lse;
    *out_logp = (a >= 0 && (int64_t)a < V) ? z[a] - lse : NAN;
}

typedef struct {
    const uint16_t *h, *W;
    const float *Wf;
    const int32_t *targets;
    const int64_t *rows;
    int64_t R, D, V;
    double temperature;
    double *out_logp, *out_lse;
    int tid, nthreads, failed;
} row_job;

static void *row_worker(void *p)
{
    row_job *j = (row_job *)p;
    double *hd = (double *)malloc(sizeof(double) * (size_t)j->D);
    double *z = (double *)malloc(sizeof(double) * (size_t)j->V);
    if (!hd || !z) {
        j->failed = 1;
        free(hd);
        free(z);
        return NULL;
    }
    for (int64_t i = j->tid; i < j->R; i += j->nthreads) {
        int64_t t = j->rows ? j->rows[i] : i;
        oracle_row(j->h + t * j->D, j->W, j->Wf, j->targets[t], j->D, j->V, j->temperature, hd, z,
                   j->out_logp + i, j->out_lse + i);
    }
    free(hd);
    free(z);
    return NULL;
}

/* Rows `rows[0..R)` of h (all N rows when rows == NULL, then R = N).
 * h bf16 [N, D], W bf16 [V, D], targets int32 [N], temperature > 0 (1 for raw
 * logits); outputs double [R].
 * Rows are spread over `nthreads` threads; each row is computed alone.
 * Returns 0, or -1 on bad arguments / allocation failure. */
static int token_logprob_rows(const uint16_t *h, const uint16_t *W, const float *Wf, const int32_t *targets,
                              const int64_t *rows, int64_t R, int64_t D, int64_t V, double temperature,
                              double *out_logp, double *out_lse, int nthreads)
{
    if (R < 0 || D <= 0 || V <= 0 || !h || (!W && !Wf) || !targets || !out_logp || !out_lse)
        return -1;
    if (!(temperature > 0.0) || !isfinite(temperature))
        return -1;
    if (R == 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > R)
        nthreads = (int)R;
    row_job *jobs = (row_job *)calloc((size_t)nthreads, sizeof(row_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    int rc = 0;
    for (int k = 0; k < nthreads; ++k) {
        jobs[k] = (row_job){h, W, Wf, targets, rows, R, D, V, temperature, out_logp, out_lse, k, nthreads, 0};
        if (pthread_create(&th[k], NULL, row_worker, &jobs[k]) != 0) {
            row_worker(&jobs[k]); /* run inline if no thread could be made */
            th[k] = 0;
        }
    }
    for (int k = 0; k < nthreads; ++k) {
        if (th[k])
            pthread_join(th[k], NULL);
        if (jobs[k].failed)
            rc = -1;
    }
    free(jobs);
    free(th);
    return rc;
}

int oracle_token_logprob(const uint16_t *h, const uint16_t *W, const int32_t *targets,
                         const int64_t *rows, int64_t R, int64_t D, int64_t V, double temperature,
                         double *out_logp, double *out_lse, int nthreads)
{
    if (!W)
        return -1;
    return token_logprob_rows(h, W, NULL, targets, rows, R, D, V, temperature, out_logp, out_lse, nthreads);
}

/* The same with fp32 weights W [V, D] (FP32 LM head): every product of a bf16
 * hidden value and an fp32 weight is taken exactly in fp64. */
int oracle_token_logprob_f32w(const uint16_t *h, const float *W, const int32_t *targets,
                              const int64_t *rows, int64_t R, int64_t D, int64_t V, double temperature,
                              double *out_logp, double *out_lse, int nthreads)
{
    if (!W)
        return -1;
    return token_logprob_rows(h, NULL, W, targets, rows, R, D, V, temperature, out_logp, out_lse, nthreads);
}

/* ------------------------------------------------------------------ mismatch stats */

enum { /* per-sequence record, in this order */
    SQ_N_MASK, SQ_N_USED, SQ_N_NAN, SQ_N_CLIP, SQ_MEAN_DELTA, SQ_MEAN_ABS_DELTA,
    SQ_MAX_ABS_DELTA, SQ_MEAN_K1, SQ_MEAN_K2, SQ_MEAN_K3, SQ_MEAN_W, SQ_MEAN_REL,
    SQ_FIELDS
};
enum { /* batch record, in this order */
    BT_N_MASK, BT_N_USED, BT_N_NAN, BT_N_CLIP, BT_MEAN_DELTA, BT_MEAN_ABS_DELTA,
    BT_MAX_ABS_DELTA, BT_MEAN_K1, BT_MEAN_K2, BT_MEAN_K3, BT_MEAN_W, BT_MEAN_REL,
    BT_SEQMEAN_K1, BT_SEQMEAN_K2, BT_SEQMEAN_K3, BT_CLIP_RATIO, BT_NAN_RATIO,
    BT_REJECT_RATIO, BT_N_SEQS_NONEMPTY, BT_N_REJECTED, BT_FIELDS
};

int oracle_seq_fields(void) { return SQ_FIELDS; }
int oracle_batch_fields(void) { return BT_FIELDS; }

/* sum / count, or 0 for an empty set. */
static double mean_or_zero(double sum, double count) { return count > 0 ? sum / count : 0.0; }

/* Per-token quantities of the definition. */
typedef struct {
    int used, nan, clip;
    double delta, k1, k2, k3, w, rel;
} token_terms;

static token_terms oracle_token(float l_tr, float l_ro, uint8_t mask, double C, double logC)
{
    token_terms q;
    memset(&q, 0, sizeof q);
    float d32 = l_tr - l_ro;                     /* device precision, decisions only */
    int in = mask != 0;
    int fin = isfinite(d32);
    q.used = in && fin;
    q.nan = in && !fin;
    if (!q.used)
        return q;
    double d = (double)l_tr - (double)l_ro;      /* delta = log pi_train - log pi_rollout */
    double log_r = d;                            /* r = e^delta, so log r = delta */
    double r = exp(d);
    double r_minus_1 = expm1(d);                 /* r - 1 without cancellation */
    q.delta = d;
    q.k1 = -log_r;
    q.k2 = 0.5 * log_r * log_r;
    q.k3 = r_minus_1 - log_r;
    q.w = r < C ? r : C;                         /* truncated IS weight min(r, C) */
    q.clip = (double)d32 > logC;                 /* r > C, decided on the fp32 delta */
    q.rel = fabs(d) / (fabs((double)l_tr) + 1e-8);
    return q;
}

/* Sums of one sequence over its tokens, in token order. */
typedef struct {
    double n_mask, n_used, n_nan, n_clip;
    double sd, sad, sk1, sk2, sk3, sw, srel, mx;
} seq_sums;

static seq_sums oracle_sequence(const float *logp_train, const float *logp_rollout, const uint8_t *mask,
                                int64_t t0, int64_t t1, double C, double logC, double *token_weight)
{
    seq_sums z;
    memset(&z, 0, sizeof z);
    for (int64_t t = t0; t < t1; ++t) {
        token_terms q = oracle_token(logp_train[t], logp_rollout[t], mask[t], C, logC);
        z.n_mask += mask[t] != 0;
        z.n_nan += q.nan;
        if (!q.used)
            continue;
        z.n_used += 1;
        z.n_clip += q.clip;
        z.sd += q.delta;
        z.sad += fabs(q.delta);
        z.sk1 += q.k1;
        z.sk2 += q.k2;
        z.sk3 += q.k3;
        z.sw += q.w;
        z.srel += q.rel;
        if (fabs(q.delta) > z.mx)
            z.mx = fabs(q.delta);
        if (token_weight)
            token_weight[t] = q.w;
    }
    return z;
}

/* Sequences [s0, s1) of a batch, on one thread: their sums into `sums`. */
typedef struct {
    const float *lt, *lr;
    const uint8_t *m;
    const int32_t *off;
    int32_t s0, s1;
    double C, logC;
    double *w;
    seq_sums *sums;
} seq_job;

static void *seq_worker(void *p)
{
    seq_job *j = (seq_job *)p;
    for (int32_t s = j->s0; s < j->s1; ++s)
        j->sums[s] = oracle_sequence(j->lt, j->lr, j->m, j->off[s], j->off[s + 1], j->C, j->logC, j->w);
    return NULL;
}

/* logp_train, logp_rollout fp32 [N]; mask uint8 [N]; seq_offsets int32 [S+1].
 * Outputs: token_weight double [N] (may be NULL), seq_stats double [S][SQ_FIELDS],
 * seq_flags int32 [S], batch double [BT_FIELDS].
 * Each sequence is summed alone in token order (the sequences are spread over
 * `nthreads` threads, which changes no arithmetic); then one thread adds the
 * sequences' sums into the batch totals in sequence order.
 * Returns 0, or -1 on bad arguments / bad offsets, -2 when out of memory. */
int oracle_mismatch_stats_threads(const float *logp_train, const float *logp_rollout, const uint8_t *mask,
                                  const int32_t *seq_offsets, int32_t S, int64_t N, double C,
                                  double tau_seq, int32_t seq_estimator, double *token_weight,
                                  double *seq_stats, int32_t *seq_flags, double *batch, int nthreads)
{
    if (S < 0 || N < 0 || !(C > 0.0) || !seq_offsets || !batch)
        return -1;
    if (N > 0 && (!logp_train || !logp_rollout || !mask))
        return -1;
    if (S > 0 && (!seq_stats || !seq_flags))
        return -1;
    if (seq_estimator != 1 && seq_estimator != 3)
        return -1;
    if (seq_offsets[0] != 0 || (int64_t)seq_offsets[S] != N)
        return -1;
    for (int32_t s = 0; s < S; ++s)
        if (seq_offsets[s + 1] < seq_offsets[s])
            return -1;

    const double logC = log(C);
    const double tau = isnan(tau_seq) ? (C - 1.0) - logC : tau_seq;

    if (token_weight)
        for (int64_t t = 0; t < N; ++t)
            token_weight[t] = 0.0;

    seq_sums *sums = (seq_sums *)malloc(sizeof(seq_sums) * (size_t)(S > 0 ? S : 1));
    if (!sums)
        return -2;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > S)
        nthreads = S > 0 ? S : 1;
    seq_job *jobs = (seq_job *)calloc((size_t)nthreads, sizeof(seq_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !tids || !started) {
        free(sums);
        free(jobs);
        free(tids);
        free(started);
        return -2;
    }
    for (int i = 0; i < nthreads; ++i)
        jobs[i] = (seq_job){logp_train, logp_rollout, mask, seq_offsets, (int32_t)((int64_t)S * i / nthreads),
                            (int32_t)((int64_t)S * (i + 1) / nthreads), C, logC, token_weight, sums};
    for (int i = 1; i < nthreads; ++i)
        started[i] = pthread_create(&tids[i], NULL, seq_worker, &jobs[i]) == 0;
    seq_worker(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) {
        if (started[i])
            pthread_join(tids[i], NULL);
        else
            seq_worker(&jobs[i]);   /* no thread could be made: run it here */
    }
    free(jobs);
    free(tids);
    free(started);

    /* batch totals, accumulated sequence by sequence in index order */
    double b_mask = 0, b_used = 0, b_nan = 0, b_clip = 0;
    double b_sd = 0, b_sad = 0, b_sk1 = 0, b_sk2 = 0, b_sk3 = 0, b_sw = 0, b_srel = 0, b_max = 0;
    double b_mk1 = 0, b_mk2 = 0, b_mk3 = 0, b_nonempty = 0, b_rej = 0;

    for (int32_t s = 0; s < S; ++s) {
        const seq_sums *z = &sums[s];
        const double n_used = z->n_used;
        double *o = seq_stats + (size_t)s * SQ_FIELDS;
        o[SQ_N_MASK] = z->n_mask;
        o[SQ_N_USED] = n_used;
        o[SQ_N_NAN] = z->n_nan;
        o[SQ_N_CLIP] = z->n_clip;
        o[SQ_MAX_ABS_DELTA] = z->mx;
        o[SQ_MEAN_DELTA] = mean_or_zero(z->sd, n_used);
        o[SQ_MEAN_ABS_DELTA] = mean_or_zero(z->sad, n_used);
        o[SQ_MEAN_K1] = mean_or_zero(z->sk1, n_used);
        o[SQ_MEAN_K2] = mean_or_zero(z->sk2, n_used);
        o[SQ_MEAN_K3] = mean_or_zero(z->sk3, n_used);
        o[SQ_MEAN_W] = mean_or_zero(z->sw, n_used);
        o[SQ_MEAN_REL] = mean_or_zero(z->srel, n_used);
        int flag = 0;
        if (n_used > 0) {
            double stat = seq_estimator == 3 ? o[SQ_MEAN_K3] : fabs(o[SQ_MEAN_K1]);
            flag = stat > tau;
            b_nonempty += 1;
            b_mk1 += o[SQ_MEAN_K1];
            b_mk2 += o[SQ_MEAN_K2];
            b_mk3 += o[SQ_MEAN_K3];
            b_rej += flag;
        }
        seq_flags[s] = flag;

        b_mask += z->n_mask;
        b_used += n_used;
        b_nan += z->n_nan;
        b_clip += z->n_clip;
        b_sd += z->sd;
        b_sad += z->sad;
        b_sk1 += z->sk1;
        b_sk2 += z->sk2;
        b_sk3 += z->sk3;
        b_sw += z->sw;
        b_srel += z->srel;
        if (z->mx > b_max)
            b_max = z->mx;
    }
    free(sums);

    batch[BT_N_MASK] = b_mask;
    batch[BT_N_USED] = b_used;
    batch[BT_N_NAN] = b_nan;
    batch[BT_N_CLIP] = b_clip;
    batch[BT_MEAN_DELTA] = mean_or_zero(b_sd, b_used);
    batch[BT_MEAN_ABS_DELTA] = mean_or_zero(b_sad, b_used);
    batch[BT_MAX_ABS_DELTA] = b_max;
    batch[BT_MEAN_K1] = mean_or_zero(b_sk1, b_used);
    batch[BT_MEAN_K2] = mean_or_zero(b_sk2, b_used);
    batch[BT_MEAN_K3] = mean_or_zero(b_sk3, b_used);
    batch[BT_MEAN_W] = mean_or_zero(b_sw, b_used);
    batch[BT_MEAN_REL] = mean_or_zero(b_srel, b_used);
    batch[BT_SEQMEAN_K1] = mean_or_zero(b_mk1, b_nonempty);
    batch[BT_SEQMEAN_K2] = mean_or_zero(b_mk2, b_nonempty);
    batch[BT_SEQMEAN_K3] = mean_or_zero(b_mk3, b_nonempty);
    batch[BT_CLIP_RATIO] = mean_or_zero(b_clip, b_mask);
    batch[BT_NAN_RATIO] = mean_or_zero(b_nan, b_mask);
    batch[BT_REJECT_RATIO] = mean_or_zero(b_rej, b_nonempty);
    batch[BT_N_SEQS_NONEMPTY] = b_nonempty;
    batch[BT_N_REJECTED] = b_rej;
    return 0;
}

int oracle_mismatch_stats(const float *logp_train, const float *logp_rollout, const uint8_t *mask,
                          const int32_t *seq_offsets, int32_t S, int64_t N, double C,
                          double tau_seq, int32_t seq_estimator, double *token_weight,
                          double *seq_stats, int32_t *seq_flags, double *batch)
{
    return oracle_mismatch_stats_threads(logp_train, logp_rollout, mask, seq_offsets, S, N, C, tau_seq,
                                         seq_estimator, token_weight, seq_stats, seq_flags, batch, 1);
}

/* ------------------------------------------------------------------ TIS-weighted PPO surrogate
 *
 * VeXact summary, eq. (2): the clipped PPO surrogate of ratio r and advantage
 * A; eq. (3), recompute mode: r = pi_theta / pi_old^train, and the TIS
 * correction multiplies the surrogate by the correction ratio pi_old^train /
 * pi_old^rollout truncated at C (LoongSage section 4 clips the same IS weight
 * when it leaves its bounds); HN page, section on clipped importance ratios:
 * separate eps_low / eps_high, and no gradient flows from a token whose
 * clipped term is the one taken.
 *
 * Per token with mask != 0 and finite inputs ("used"):
 *   r = exp(l_theta - l_old), w = min(exp(l_old - l_rollout), C),
 *   loss = -w min(r A, clip(r, 1 - eps_low, 1 + eps_high) A),
 *   grad = d loss / d l_theta = -w r A where r A is the minimum, else 0.
 * Readings: the clipped branch is taken only where it is strictly smaller
 * (ties keep the gradient); the decisions (clipped PPO branch, w capped) are
 * taken on the log-ratios rounded to fp32, the precision the device computes
 * them in, against the exact thresholds log(1 + eps_high), log(1 - eps_low),
 * log C; values use the exact fp64 log-ratios.  Unused tokens: loss 0, grad 0.
 * Outputs: token_loss, token_grad [N] (may be NULL), seq_loss [S] = mean loss
 * over the sequence's used tokens (0 if none), batch [PPO_FIELDS]. */
enum {
    PB_N_MASK, PB_N_USED, PB_N_PPO_CLIPPED, PB_N_TIS_CLIPPED, PB_MEAN_LOSS, PB_SEQMEAN_LOSS,
    PB_PPO_CLIP_RATIO, PB_TIS_CLIP_RATIO, PB_N_SEQS_NONEMPTY, PB_FIELDS
};

int oracle_ppo_fields(void) { return PB_FIELDS; }

int oracle_tis_ppo(const float *l_theta, const float *l_old, const float *l_rollout, const float *adv,
                   const uint8_t *mask, const int32_t *seq_offsets, int32_t S, int64_t N, double eps_low,
                   double eps_high, double C, double *token_loss, double *token_grad, double *seq_loss,
                   double *batch)
{
    if (S < 0 || N < 0 || !(C > 0.0) || !(eps_low >= 0.0 && eps_low < 1.0) || !(eps_high >= 0.0) ||
        !seq_offsets || !batch)
        return -1;
    if (N > 0 && (!l_theta || !l_old || !l_rollout || !adv || !mask))
        return -1;
    if (S > 0 && !seq_loss)
        return -1;
    if (seq_offsets[0] != 0 || (int64_t)seq_offsets[S] != N)
        return -1;
    for (int32_t s = 0; s < S; ++s)
        if (seq_offsets[s + 1] < seq_offsets[s])
            return -1;
    const double log_hi = log1p(eps_high), log_lo = log1p(-eps_low), log_c = log(C);
    double b_mask = 0, b_used = 0, b_ppo = 0, b_tis = 0, b_loss = 0, b_seqmean = 0, b_nonempty = 0;
    for (int32_t s = 0; s < S; ++s) {
        double n_used = 0, sum_loss = 0;
        for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t) {
            double loss = 0.0, grad = 0.0;
            const int in = mask[t] != 0;
            b_mask += in;
            const float dt32 = l_theta[t] - l_old[t];     /* decisions in fp32 */
            const float dc32 = l_old[t] - l_rollout[t];
            const int used = in && isfinite(dt32) && isfinite(dc32) && isfinite(adv[t]);
            if (used) {
                const double A = adv[t];
                const double r = exp((double)l_theta[t] - (double)l_old[t]);
                const double rc = exp((double)l_old[t] - (double)l_rollout[t]);
                const double w = rc < C ? rc : C;
                const int tis_clipped = (double)dc32 > log_c;
                const int ppo_clipped = (A > 0.0 && (double)dt32 > log_hi) || (A < 0.0 && (double)dt32 < log_lo);
                const double rclip = A > 0.0 ? 1.0 + eps_high : 1.0 - eps_low;
                loss = ppo_clipped ? -w * rclip * A : -w * r * A;
                grad = ppo_clipped ? 0.0 : -w * r * A;
                n_used += 1;
                sum_loss += loss;
                b_ppo += ppo_clipped;
                b_tis += tis_clipped;
            }
            if (token_loss)
                token_loss[t] = loss;
            if (token_grad)
                token_grad[t] = grad;
        }
        seq_loss[s] = mean_or_zero(sum_loss, n_used);
        b_used += n_used;
        b_loss += sum_loss;
        if (n_used > 0) {
            b_nonempty += 1;
            b_seqmean += seq_loss[s];
        }
    }
    batch[PB_N_MASK] = b_mask;
    batch[PB_N_USED] = b_used;
    batch[PB_N_PPO_CLIPPED] = b_ppo;
    batch[PB_N_TIS_CLIPPED] = b_tis;
    batch[PB_MEAN_LOSS] = mean_or_zero(b_loss, b_used);
    batch[PB_SEQMEAN_LOSS] = mean_or_zero(b_seqmean, b_nonempty);
    batch[PB_PPO_CLIP_RATIO] = mean_or_zero(b_ppo, b_used);
    batch[PB_TIS_CLIP_RATIO] = mean_or_zero(b_tis, b_used);
    batch[PB_N_SEQS_NONEMPTY] = b_nonempty;
    return 0;
}

/* ------------------------------------------------------------------ mismatch monitor
 *
 * llm-infra-atlas section 7, the list of mismatch metrics compared per
 * response token over a rollout dump: the p95 of |logp_train - logp_rollout|,
 * the 0.01 / 0.5 / 0.99 quantiles of the ratio r = pi_train / pi_rollout =
 * e^delta, and the fraction of tokens with |delta| > tau; VeXact summary,
 * calibration of the token-level threshold tau_tok (a token is rejected when
 * |delta| > tau_tok).
 * Readings: the statistics run over the used tokens of the batch (mask != 0,
 * finite fp32 delta); the quantile of a sample x_(0) <= ... <= x_(n-1) at
 * level q is the linear interpolation at h = (n - 1) q between x_(floor h)
 * and the next order statistic (the default of numpy and torch); an empty
 * sample gives NaN quantiles.  Order statistics of r are those of delta (e^x
 * is increasing), so r quantiles interpolate e^delta at delta's order
 * statistics.  Outputs: out[MON_FIELDS]; reject[N] (may be NULL): 1 for a used
 * token with |delta| > tau_tok, else 0. */
enum { MO_N_USED, MO_P95_ABS_DELTA, MO_RATIO_Q01, MO_RATIO_Q50, MO_RATIO_Q99, MO_N_EXTREME, MO_FRAC_EXTREME,
       MO_FIELDS };

int oracle_monitor_fields(void) { return MO_FIELDS; }

static int cmp_double(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return x < y ? -1 : x > y ? 1 : 0;
}

/* quantile at level q of the sorted sample x[0..n-1], n > 0 */
static double quantile_sorted(const double *x, int64_t n, double q, int exp_values)
{
    const double h = (double)(n - 1) * q;
    const double fl = floor(h);
    const int64_t k = (int64_t)fl;
    const int64_t k1 = k + 1 < n ? k + 1 : k;
    const double lo = exp_values ? exp(x[k]) : x[k];
    const double hi = exp_values ? exp(x[k1]) : x[k1];
    return lo + (h - fl) * (hi - lo);
}

int oracle_mismatch_monitor(const float *logp_train, const float *logp_rollout, const uint8_t *mask, int64_t N,
                            double tau_tok, double *out, uint8_t *reject)
{
    if (N < 0 || !out || !(tau_tok >= 0.0))
        return -1;
    if (N > 0 && (!logp_train || !logp_rollout || !mask))
        return -1;
    double *ad = N > 0 ? (double *)malloc(sizeof(double) * (size_t)N) : NULL;
    double *d = N > 0 ? (double *)malloc(sizeof(double) * (size_t)N) : NULL;
    if (N > 0 && (!ad || !d)) {
        free(ad);
        free(d);
        return -2;
    }
    int64_t n = 0, n_ext = 0;
    for (int64_t t = 0; t < N; ++t) {
        const float d32 = logp_train[t] - logp_rollout[t];
        const int used = mask[t] != 0 && isfinite(d32);
        const int ext = used && fabs((double)d32) > tau_tok;
        if (reject)
            reject[t] = (uint8_t)ext;
        if (used) {
            d[n] = (double)d32;
            ad[n] = fabs((double)d32);
            ++n;
            n_ext += ext;
        }
    }
    out[MO_N_USED] = (double)n;
    out[MO_N_EXTREME] = (double)n_ext;
    out[MO_FRAC_EXTREME] = mean_or_zero((double)n_ext, (double)n);
    if (n == 0) {
        out[MO_P95_ABS_DELTA] = out[MO_RATIO_Q01] = out[MO_RATIO_Q50] = out[MO_RATIO_Q99] = NAN;
    } else {
        qsort(ad, (size_t)n, sizeof(double), cmp_double);
        qsort(d, (size_t)n, sizeof(double), cmp_double);
        out[MO_P95_ABS_DELTA] = quantile_sorted(ad, n, 0.95, 0);
        out[MO_RATIO_Q01] = quantile_sorted(d, n, 0.01, 1);
        out[MO_RATIO_Q50] = quantile_sorted(d, n, 0.5, 1);
        out[MO_RATIO_Q99] = quantile_sorted(d, n, 0.99, 1);
    }
    free(ad);
    free(d);
    return 0;
}

/* ------------------------------------------------------------------ token logprob backward
 *
 * The trainer differentiates the selected-token logprob (Thinking Machines
 * page, "Unclipped importance sampling": the token gradient is a weight times
 * the gradient of log q_t).  With an upstream weight g_t per token and
 * l_t = z_t[a_t] / tau - log sum_v exp(z_t[v] / tau), z_t = h_t W^T:
 *   dz_t[v] = d (sum_t g_t l_t) / d z_t[v] = g_t (1[v = a_t] - p_t[v]) / tau,
 *   p_t = softmax(z_t / tau),  dh = dz W  [N, D],  dW = dz^T h  [V, D].
 * Written from the definition: z_t and p_t recomputed in fp64 per row (as the
 * forward oracle), then both products summed in index order.  Rows whose
 * target lies outside [0, V) take no one-hot term.  dz [N, V] may be NULL. */
int oracle_token_logprob_backward(const uint16_t *h, const uint16_t *W, const int32_t *targets, const float *grad,
                                  int64_t N, int64_t D, int64_t V, double temperature, double *dh, double *dW,
                                  double *dz_out)
{
    if (N < 0 || D <= 0 || V <= 0 || !(temperature > 0.0) || !isfinite(temperature))
        return -1;
    if (N > 0 && (!h || !W || !targets || !grad || !dh || !dW))
        return -1;
    double *hd = (double *)malloc(sizeof(double) * (size_t)D);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    if (!hd || !z) {
        free(hd);
        free(z);
        return -2;
    }
    for (int64_t i = 0; i < V * D; ++i)
        dW[i] = 0.0;
    for (int64_t t = 0; t < N; ++t) {
        double lp, lse;
        oracle_row(h + t * D, W, NULL, targets[t], D, V, temperature, hd, z, &lp, &lse);
        double *dht = dh + t * D;
        for (int64_t d = 0; d < D; ++d)
            dht[d] = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            const double p = exp(z[v] - lse);
            const double dzv = (double)grad[t] * ((v == targets[t] ? 1.0 : 0.0) - p) / temperature;
            if (dz_out)
                dz_out[t * V + v] = dzv;
            const uint16_t *w = W + v * D;
            double *dwv = dW + v * D;
            for (int64_t d = 0; d < D; ++d) {
                dht[d] += dzv * bf16_value(w[d]);
                dwv[d] += dzv * hd[d];
            }
        }
    }
    free(hd);
    free(z);
    return 0;
}
