/*
 * tim.h -- C ABI of the GB300 (sm_103a) train/rollout logprob-mismatch library
 * (libtim.so).
 *
 * Two calls make up the hot path of a trainer's mismatch check:
 *
 *   tim_token_logprob   the trainer-side selected-token log-probability
 *                       l_t = log softmax(h_t W^T)[a_t], computed as one fused
 *                       pass (bf16 x bf16 -> fp32 LM head, online
 *                       log-sum-exp over the vocabulary, gather at the target
 *                       id) that never writes the [N, V] logits to memory;
 *   tim_mismatch_stats  the segmented pass that scores l_train against the
 *                       rollout engine's logprobs: delta, r, k1/k2/k3, the
 *                       truncated importance weight and masked per-sequence /
 *                       per-batch means with a sequence rejection flag.
 *
 * Determinism and batch invariance.  Every reduction runs in an order fixed by
 * D and V (token logprob) or by a token's index inside its own sequence
 * (mismatch statistics); no split depends on N, S or on where a row or a
 * sequence sits in the batch.  A row's outputs, and a sequence's record, are
 * bit-identical whatever else is in the batch, and from run to run.
 *
 * Conventions for every call:
 *  - all array arguments are caller-owned DEVICE pointers of the current CUDA
 *    device; nothing is retained after the call returns;
 *  - calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream); a non-zero return means nothing was launched and the outputs are
 *    untouched;
 *  - host-side argument errors return TIM_ERR_INVALID_ARG; a device that is
 *    not sm_103 returns TIM_ERR_UNSUPPORTED_DEVICE; a failing CUDA runtime call
 *    returns TIM_ERR_CUDA; tim_last_error() gives a message for the calling
 *    thread;
 *  - bad DATA found on the device (bad sequence offsets; a pipeline wait that
 *    ran out of time) never traps: the kernel records a status word that
 *    tim_check() returns, and writes NaN into the affected outputs.
 */
#ifndef TIM_H
#define TIM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TIM_API __attribute__((visibility("default")))
#else
#define TIM_API
#endif

/* Same object as cudaStream_t; declared here so that this header needs no CUDA header. */
typedef struct CUstream_st *tim_stream_t;

typedef enum {
    TIM_OK = 0,
    TIM_ERR_INVALID_ARG = -1,        /* host-side argument check failed */
    TIM_ERR_UNSUPPORTED_DEVICE = -2, /* current device is not sm_103 (GB300) */
    TIM_ERR_CUDA = -3,               /* a CUDA runtime call failed */
    TIM_ERR_TIMEOUT = -4,            /* a pipeline wait inside a kernel ran out of time */
    TIM_ERR_BAD_INPUT = -5           /* the device found bad data (sequence offsets) */
} tim_status;

/* ------------------------------------------------------------------ token logprob
 *
 * l_t = log softmax(h_t W^T)[a_t] and lse_t = log sum_v exp(h_t . W_v).
 *
 * Defined by the icarus page "RL: Training Inference Mismatch", section "log p"
 * (final hidden states -> LM head -> log-softmax -> gather at the token id, and
 * its PyTorch statement log_softmax(logits, -1).gather(-1, ids)); the head is
 * kept above bf16 precision as in LoongSage "Train-Inference Consistency"
 * section 3 "FP32 LM head" -- here as bf16 operands with fp32 accumulation.
 * The pages' head has a bias; this call has none.  Temperature is 1 (raw
 * logits, icarus section "logits processor").  Batch invariance and fixed
 * reduction order: llm-infra-atlas "训推一致性与 determinism" sections 1.2 and 6.
 *
 *   h        bf16 [N, D] row-major (final hidden states), 16-byte aligned
 *   W        bf16 [V, D] row-major (LM-head weight, one row per vocabulary id),
 *            16-byte aligned
 *   targets  int32 [N]: a_t, already shifted by the caller so that row t of h
 *            predicts targets[t] (icarus section "shift and mask"); an id
 *            outside [0, V) (e.g. the -100 ignore label) gives out_logp = NaN
 *   N        rows, N >= 0 (N = 0 is a no-op returning TIM_OK), N < 2^31
 *   D        hidden size, D > 0 and D % 8 == 0 (16-byte row stride), D <= 65536
 *   V        vocabulary size, 0 < V < 2^31, with ceil(N / 128) * ceil(V / 1024)
 *            < 2^31 (N * V below about 2^48)
 *   out_logp fp32 [N]: l_t in nats
 *   out_lse  fp32 [N]: log-sum-exp of the raw logits, in nats
 *
 * Scratch: the call takes a split-V workspace of about 8 * N * ceil(V / 1024)
 * bytes from a stream-ordered memory pool of its own (cudaMallocFromPoolAsync
 * on `stream`) and gives it back on the same stream; the pool keeps the memory
 * for the next call.  Tolerance against an fp64 evaluation of the definition:
 * a few 1e-6 absolute on l_t and lse for the pages' head shapes.
 */
TIM_API int tim_token_logprob(const void *h, const void *W, const int32_t *targets,
                      int64_t N, int64_t D, int64_t V,
                      float *out_logp, float *out_lse, tim_stream_t stream);

/* Same, at a sampling temperature: l_t = log softmax(h_t W^T / temperature)[a_t]
 * and lse_t = log sum_v exp(h_t . W_v / temperature).  The rollout engine samples
 * from softmax(z / tau) (icarus page, section "logits processor"), and both sides
 * must use the same tau.  temperature > 0 and finite (else TIM_ERR_INVALID_ARG);
 * temperature = 1 gives the bits of tim_token_logprob.  Everything else as above. */
TIM_API int tim_token_logprob_temperature(const void *h, const void *W, const int32_t *targets,
                                          int64_t N, int64_t D, int64_t V, float temperature,
                                          float *out_logp, float *out_lse, tim_stream_t stream);

/* ------------------------------------------------------------------ token logprob backward
 *
 * The trainer's gradient through the selected-token logprob (Thinking Machines
 * page, "Unclipped importance sampling": each token weights the gradient of
 * log q_t).  With an upstream gradient g_t = dL / dl_t per token (for example
 * the TIS-weighted PPO surrogate's token_grad) and the forward's lse:
 *   dz_t[v] = g_t (1[v = a_t] - p_t[v]) / tau,  p_t = softmax(h_t W^T / tau),
 *   dh = dz W  (fp32 [N, D]),  dW = dz^T h  (fp32 [V, D]).
 * The logits are recomputed by the fused kernel and turned into dz (bf16) in
 * its epilogue, chunk by chunk of at most 4096 rows (the fp32 logits never
 * reach HBM); per chunk two cuBLAS GEMMs (bf16 operands, fp32 accumulation)
 * give that chunk's rows of dh and add its share of dW, chunks in row order,
 * so dW's reduction order is fixed and the results repeat bit for bit.
 *   h, W, targets, N, D, V, temperature   as tim_token_logprob_temperature
 *   grad_logp     fp32 [N], 4-byte aligned
 *   lse           fp32 [N]: out_lse of the forward at the same temperature
 *   dh            out: fp32 [N, D], 16-byte aligned
 *   dW            out: fp32 [V, D], 16-byte aligned; accumulate_dW != 0 adds into it
 * A target outside [0, V) takes no one-hot term.  Scratch: min(N, 4096) rows
 * x V bf16 from the library's stream-ordered pool (1.2 GB at V = 151936). */
TIM_API int tim_token_logprob_backward(const void *h, const void *W, const int32_t *targets,
                                       const float *grad_logp, const float *lse, int64_t N, int64_t D,
                                       int64_t V, float temperature, float *dh, float *dW, int accumulate_dW,
                                       tim_stream_t stream);

/* ------------------------------------------------------------------ FP32 LM head
 *
 * LoongSage "Train-Inference Consistency" section 3: the LM head's weights and
 * arithmetic stay in fp32, so that rounding to bf16 does not reach the
 * log-probabilities.  The hidden states stay bf16 (the model's activations;
 * exact in fp32).  The weights are first cut, once per weight update, into
 * three bf16 parts whose sum is each fp32 weight exactly; the fused kernel then
 * runs over the parts (three times the tensor work of the bf16 head) with fp32
 * accumulation: bf16 x bf16 products are exact in fp32.
 *
 * tim_split_weight_bytes(V, D): bytes of the split, V * 3 * Dp * 2 with Dp = D
 * rounded up to a multiple of 64; -1 for sizes out of range.
 * tim_split_weight_fp32(W, V, D, W_split, stream):
 *   W        fp32 [V, D] row-major, 16-byte aligned, D % 8 == 0
 *   W_split  out: caller-owned device buffer of tim_split_weight_bytes(V, D)
 *            bytes, 16-byte aligned; row v is [part 1 | part 2 | part 3], each
 *            Dp bf16 columns, zero past D.  Exact for |w| >= 2^-110 (smaller
 *            weights lose their last bits, below 2^-133); a non-finite weight
 *            goes whole into part 1.
 * tim_token_logprob_fp32_head(h, W_split, targets, N, D, V, temperature,
 *                             out_logp, out_lse, stream):
 *   as tim_token_logprob_temperature, with the split weights in place of W. */
TIM_API int64_t tim_split_weight_bytes(int64_t V, int64_t D);
TIM_API int tim_split_weight_fp32(const float *W, int64_t V, int64_t D, void *W_split, tim_stream_t stream);
TIM_API int tim_token_logprob_fp32_head(const void *h, const void *W_split, const int32_t *targets, int64_t N,
                                        int64_t D, int64_t V, float temperature, float *out_logp,
                                        float *out_lse, tim_stream_t stream);

/* ------------------------------------------------------------------ token logprob, no allocation
 *
 * No counterpart on the pages: a library-side variant of tim_token_logprob for
 * callers that cannot have the library allocate device memory -- an engine that
 * has reserved its whole device-memory budget for its own allocator (where a
 * hidden allocation fails or escapes its accounting), or code where the
 * stream-ordered allocator is unavailable.  Same arguments, results and
 * tolerance as tim_token_logprob; it calls no cudaMalloc / cudaFree / pool
 * routine.  Its split-V scratch is one fixed device array inside libtim.so of
 * TIM_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the library
 * until the process exits.  A call needs
 *   ceil(8 * N * ceil(V / 1024) / 256) * 256 + ceil(4 * N / 256) * 256
 *   + (N % 16 != 0 ? ceil(256 * D / 256) * 256 : 0) + 256
 * bytes of it (split-V partials, target logits, a zero-padded copy of the last
 * 128-row tile of h when N is not a multiple of 16 -- the same fast loads as
 * tim_token_logprob -- and a unit counter); calls needing more return
 * TIM_ERR_INVALID_ARG without launching anything.  At V = 151936 and D = 4096
 * that admits every N <= 13150 and multiples of 16 up to 14016.
 * The first call on a device sets that device up (it looks up the array's
 * device address, sets the kernel's shared-memory size and fetches the
 * tensor-map encoder); make that first call before any stream capture.
 * Every call shares the array; two calls whose kernels overlap on the GPU
 * (different streams or threads) race on it, so callers must order them.
 */
#define TIM_NOALLOC_SCRATCH_BYTES (16u << 20)
TIM_API int tim_token_logprob_noalloc(const void *h, const void *W, const int32_t *targets,
                                      int64_t N, int64_t D, int64_t V,
                                      float *out_logp, float *out_lse, tim_stream_t stream);

/* ------------------------------------------------------------------ mismatch stats
 *
 * Per token t with mask_t != 0 (VeXact summary eq. (1); llm-infra-atlas
 * section 2; icarus KL-estimator table; LoongSage sections 4-5):
 *   delta = l_train - l_rollout,  r = e^delta,
 *   k1 = -log r,  k2 = (log r)^2 / 2,  k3 = (r - 1) - log r,
 *   w = min(r, C)  (truncated importance weight; 0 for tokens not used),
 *   clip = r > C,  rel = |delta| / (|l_train| + 1e-8).
 * A token is "used" when mask != 0 and delta is finite; a masked-in token with a
 * non-finite delta is counted as nan and left out of every mean.
 * Per sequence s (tokens seq_offsets[s] .. seq_offsets[s+1]-1): means over its
 * used tokens, then the rejection flag (VeXact "Algorithmic TIM Compensation"):
 *   estimator 3: mean k3 > tau_seq;  estimator 1: |mean k1| > tau_seq.
 * Per batch: token means over all used tokens, the mean over non-empty sequences
 * of the per-sequence means (icarus monitoring steps 2-3), clip / nan ratios
 * over masked-in tokens and the rejected fraction of non-empty sequences.
 * A sequence with no used token has all means 0 and flag 0.
 */
#define TIM_SEQ_FIELDS 12
enum tim_seq_field {
    TIM_SEQ_N_MASK = 0,        /* masked-in tokens */
    TIM_SEQ_N_USED,            /* masked-in tokens with finite delta */
    TIM_SEQ_N_NAN,             /* masked-in tokens with non-finite delta */
    TIM_SEQ_N_CLIP,            /* used tokens with r > C */
    TIM_SEQ_MEAN_DELTA,
    TIM_SEQ_MEAN_ABS_DELTA,
    TIM_SEQ_MAX_ABS_DELTA,
    TIM_SEQ_MEAN_K1,
    TIM_SEQ_MEAN_K2,
    TIM_SEQ_MEAN_K3,
    TIM_SEQ_MEAN_W,
    TIM_SEQ_MEAN_REL
};

#define TIM_BATCH_FIELDS 20
enum tim_batch_field {
    TIM_BATCH_N_MASK = 0,
    TIM_BATCH_N_USED,
    TIM_BATCH_N_NAN,
    TIM_BATCH_N_CLIP,
    TIM_BATCH_MEAN_DELTA,      /* token means over all used tokens ... */
    TIM_BATCH_MEAN_ABS_DELTA,
    TIM_BATCH_MAX_ABS_DELTA,
    TIM_BATCH_MEAN_K1,
    TIM_BATCH_MEAN_K2,
    TIM_BATCH_MEAN_K3,         /* is_approx_k3_kl */
    TIM_BATCH_MEAN_W,
    TIM_BATCH_MEAN_REL,        /* consistency_rel_diff */
    TIM_BATCH_SEQMEAN_K1,      /* mean over non-empty sequences of the sequence means */
    TIM_BATCH_SEQMEAN_K2,
    TIM_BATCH_SEQMEAN_K3,
    TIM_BATCH_CLIP_RATIO,      /* n_clip / n_mask (is_clip_ratio) */
    TIM_BATCH_NAN_RATIO,       /* n_nan / n_mask (is_nan_ratio) */
    TIM_BATCH_REJECT_RATIO,    /* rejected / non-empty sequences */
    TIM_BATCH_N_SEQS_NONEMPTY,
    TIM_BATCH_N_REJECTED
};

/* Words of one sequence record: the per-sequence sums and counts the batch
 * record is folded from (see tim_mismatch_fold). */
#define TIM_SEQ_RECORD_WORDS 16

/* Sizes and outputs of tim_mismatch_stats.  The struct lives in host memory;
 * the pointers in it are device pointers.  It carries N and S so that the host
 * never has to read seq_offsets back from the device. */
typedef struct {
    int32_t num_seqs;        /* in: S >= 0 (S = 0: only batch_stats is written, all 0) */
    int64_t num_tokens;      /* in: N >= 0; must equal seq_offsets[S] (checked on device) */
    float tau_seq;           /* in: rejection threshold; NaN selects (C - 1) - ln C,
                                k3 at r = C (a reading: the pages give no value) */
    int32_t seq_estimator;   /* in: 3 = K3 (default when 0), 1 = |K1| */
    float *token_weight;     /* out, optional (NULL = not written): fp32 [N], w_t */
    float *seq_stats;        /* out: fp32 [S][TIM_SEQ_FIELDS] */
    int32_t *seq_flags;      /* out: int32 [S], 1 = rejected */
    double *batch_stats;     /* out: fp64 [TIM_BATCH_FIELDS] */
    uint32_t *seq_records;   /* out, optional (NULL = kept internal): [S][TIM_SEQ_RECORD_WORDS],
                                16-byte aligned; a record depends on its own sequence only */
} tim_mismatch_out;

/*   logp_train, logp_rollout  fp32 [N], 16-byte aligned
 *   mask                      uint8 [N], 16-byte aligned: 0 = not counted (prompt / padding), else counted
 *   seq_offsets               int32 [S + 1]: seq_offsets[0] = 0, non-decreasing,
 *                             seq_offsets[S] = N (sequences packed back to back)
 *   C                         truncation cap of the importance weight, C > 0, finite
 *   out                       host struct described above
 * Bad offsets found on the device set TIM_ERR_BAD_INPUT (see tim_check) and
 * make every output NaN for the affected sequences and for the batch record.
 * Scratch: about 64 * S bytes from the library's stream-ordered pool. */
TIM_API int tim_mismatch_stats(const float *logp_train, const float *logp_rollout,
                       const uint8_t *mask, const int32_t *seq_offsets, float C,
                       const tim_mismatch_out *out, tim_stream_t stream);

/* The batch record of a batch whose sequences were scored in parts (a batch
 * sharded across data-parallel ranks, or across calls): the sequence records
 * of the parts (tim_mismatch_out.seq_records), concatenated in the batch's
 * sequence order, folded exactly as tim_mismatch_stats folds its own.  A
 * sequence's record does not depend on where it was packed, so the result has
 * the bits tim_mismatch_stats gives over the whole batch (the per-batch
 * aggregation of the icarus page's monitoring steps 2-3, across parts).
 *   seq_records  [S][TIM_SEQ_RECORD_WORDS] device memory, 16-byte aligned
 *   num_seqs     S >= 0 (S = 0: an all-zero record)
 *   batch_stats  out: fp64 [TIM_BATCH_FIELDS], 8-byte aligned device memory
 * A record marked invalid (bad offsets in its part) makes the record NaN and
 * sets TIM_ERR_BAD_INPUT, as in tim_mismatch_stats.  Scratch: about S / 6
 * bytes from the library's stream-ordered pool. */
TIM_API int tim_mismatch_fold(const uint32_t *seq_records, int32_t num_seqs, double *batch_stats,
                              tim_stream_t stream);

/* ------------------------------------------------------------------ mismatch monitor
 *
 * Distribution of the mismatch over the used tokens of a batch (mask != 0 and
 * finite fp32 delta = logp_train - logp_rollout), as listed among the
 * per-token mismatch metrics of llm-infra-atlas section 7: the p95 of |delta|,
 * the 0.01 / 0.5 / 0.99 quantiles of the ratio r = e^delta and the fraction of
 * tokens with |delta| > tau_tok; plus the token-level rejection of the VeXact
 * summary (a used token is rejected when |delta| > tau_tok).
 * Quantile at level q of n values: the linear interpolation at h = (n - 1) q
 * between the order statistics floor(h) and floor(h) + 1 (numpy's and torch's
 * default).  The order statistics are selected exactly (the same tokens as a
 * sort would pick); NaN quantiles when no token is used.
 */
#define TIM_MON_FIELDS 7
enum tim_monitor_field {
    TIM_MON_N_USED = 0,
    TIM_MON_P95_ABS_DELTA,
    TIM_MON_RATIO_Q01,
    TIM_MON_RATIO_Q50,
    TIM_MON_RATIO_Q99,
    TIM_MON_N_EXTREME,          /* used tokens with |delta| > tau_tok */
    TIM_MON_FRAC_EXTREME        /* n_extreme / n_used (0 when n_used = 0) */
};

/*   logp_train, logp_rollout  fp32 [N], 16-byte aligned
 *   mask                      uint8 [N], 16-byte aligned
 *   N                         tokens, 0 <= N < 2^31
 *   tau_tok                   rejection threshold on |delta|, >= 0 and finite
 *   token_reject              out, optional (NULL = not written): uint8 [N], 16-byte aligned
 *   out                       out: fp64 [TIM_MON_FIELDS]
 * One pass over the tokens (9 bytes read per token) after a sample of at most
 * 2^20 of them; exact selection among the few percent of tokens near each
 * quantile (over all tokens when a sample-based bound misses).  Scratch:
 * 3254 KB + N bytes + 1 MB from the library's stream-ordered pool (the state
 * and histograms, then four lists of N / 16 + 65536 keys). */
TIM_API int tim_mismatch_monitor(const float *logp_train, const float *logp_rollout, const uint8_t *mask,
                                 int64_t N, float tau_tok, uint8_t *token_reject, double *out,
                                 tim_stream_t stream);

/* ------------------------------------------------------------------ TIS-weighted PPO surrogate
 *
 * The clipped PPO surrogate of VeXact summary eq. (2) in recompute mode
 * (eq. (3): r = pi_theta / pi_old^train), multiplied by the truncated
 * importance weight that corrects for the rollout engine (TIS: the ratio
 * pi_old^train / pi_old^rollout truncated at C; LoongSage section 4), with
 * separate lower and upper clip ranges and no gradient through a token whose
 * clipped term is taken (HN page, section on clipped importance ratios).
 * Per token t with mask_t != 0 and finite logp_theta - logp_old,
 * logp_old - logp_rollout and A_t ("used"):
 *   r = e^(l_theta - l_old),  w = min(e^(l_old - l_rollout), C),
 *   loss = -w min(r A, clip(r, 1 - eps_low, 1 + eps_high) A),
 *   grad = d loss / d l_theta = -w r A where r A is the minimum, else 0.
 * The clipped branch is taken only where it is strictly smaller (A > 0 and
 * r > 1 + eps_high, or A < 0 and r < 1 - eps_low); both decisions, and
 * w = C, are taken on the fp32 log-ratios against the exact thresholds
 * log(1 + eps_high), log(1 - eps_low), log C.  Tokens not used: loss 0, grad 0.
 * Per sequence: the mean loss over its used tokens (0 if none).  Per batch: the
 * mean over used tokens, the mean of the sequence means over non-empty
 * sequences, and the fractions of used tokens whose PPO term or TIS weight
 * was clipped.
 */
#define TIM_PPO_FIELDS 9
enum tim_ppo_field {
    TIM_PPO_N_MASK = 0,        /* masked-in tokens */
    TIM_PPO_N_USED,            /* masked-in tokens with finite inputs */
    TIM_PPO_N_PPO_CLIPPED,     /* used tokens on the clipped (zero-gradient) branch */
    TIM_PPO_N_TIS_CLIPPED,     /* used tokens with w = C, i.e. l_old - l_rollout > log C */
    TIM_PPO_MEAN_LOSS,         /* token mean over used tokens */
    TIM_PPO_SEQMEAN_LOSS,      /* mean over non-empty sequences of the sequence means */
    TIM_PPO_PPO_CLIP_RATIO,    /* n_ppo_clipped / n_used */
    TIM_PPO_TIS_CLIP_RATIO,    /* n_tis_clipped / n_used */
    TIM_PPO_N_SEQS_NONEMPTY
};

/* Sizes and outputs of tim_tis_ppo.  Host struct; the pointers are device
 * pointers. */
typedef struct {
    int32_t num_seqs;        /* in: S >= 0 (S = 0: only batch_stats is written, all 0) */
    int64_t num_tokens;      /* in: N >= 0; must equal seq_offsets[S] (checked on device) */
    float *token_loss;       /* out, optional (NULL = not written): fp32 [N] */
    float *token_grad;       /* out, optional (NULL = not written): fp32 [N], d token_loss / d logp_theta */
    float *seq_loss;         /* out: fp32 [S] */
    double *batch_stats;     /* out: fp64 [TIM_PPO_FIELDS] */
} tim_ppo_out;

/*   logp_theta, logp_old, logp_rollout  fp32 [N]: current policy, trainer's
 *                             recompute of the rollout policy, rollout engine
 *   advantages                fp32 [N], A_t (a per-sequence advantage is broadcast by the caller)
 *   mask                      uint8 [N]: 0 = not counted (prompt / padding), else counted
 *   seq_offsets               int32 [S + 1]: seq_offsets[0] = 0, non-decreasing, seq_offsets[S] = N
 *   eps_low                   lower clip range, 0 <= eps_low < 1
 *   eps_high                  upper clip range, 0 <= eps_high, finite
 *   C                         truncation cap of the TIS weight, C > 0, finite
 * Token arrays need 4-byte alignment only.  Bad offsets found on the device set
 * TIM_ERR_BAD_INPUT (see tim_check) and make the affected sequences' seq_loss
 * and the whole batch record NaN.  Scratch: about 24 * S bytes from the
 * library's stream-ordered pool. */
TIM_API int tim_tis_ppo(const float *logp_theta, const float *logp_old, const float *logp_rollout,
                        const float *advantages, const uint8_t *mask, const int32_t *seq_offsets,
                        float eps_low, float eps_high, float C, const tim_ppo_out *out,
                        tim_stream_t stream);

/* ------------------------------------------------------------------ failure-detection self-test
 *
 * No counterpart on the pages.  Runs the library's bounded-wait path on purpose,
 * without any fault: one warp waits on an mbarrier that nothing arrives on and
 * gives up after budget_us microseconds (1 .. 1000000), recording
 * TIM_ERR_TIMEOUT in the status word exactly as an expired pipeline wait in
 * the compute kernels does.  Asynchronous on `stream`; tim_check() then
 * returns TIM_ERR_TIMEOUT, and the device stays usable.
 */
TIM_API int tim_selftest_wait_timeout(uint32_t budget_us, tim_stream_t stream);

/* ------------------------------------------------------------------ checked build
 *
 * No counterpart on the pages (the stand-in for a memory checker, which this
 * library's users may not have): libtim_debug.so is the same library built
 * with TIM_DEBUG.  Its kernels also check, without ever trapping,
 *   - their own invariants: every TMA coordinate's innermost part is a whole
 *     16 bytes, every row or column they store lies inside its buffer, every
 *     claimed work unit is below the unit count, every bulk copy is 16-byte
 *     aligned and sized;
 *   - the input contracts the release build passes over silently: a target id
 *     >= V (negative ids are the ignore label and stay legal), a mask byte
 *     other than 0 or 1, a non-finite logit (h or W holds inf or NaN), a
 *     non-finite lse or upstream gradient in the backward, a non-finite
 *     advantage in the PPO surrogate.
 * The first violation on a device sets TIM_ERR_BAD_INPUT in the status word
 * (tim_check returns it) and is recorded; later ones only set the status.
 * tim_debug_violation(out, stream) synchronises `stream`, writes the record
 *   out[0] = check (TIM_CHECK_*, 0 if none), out[1] = index (the token, row,
 *   unit or coordinate concerned), out[2] = value (its bits), out[3] = 0,
 * and clears it; returns TIM_OK or a CUDA error.  tim_debug_build() is 1 in
 * libtim_debug.so and 0 in libtim.so (where the record stays zero).
 */
enum {
    TIM_CHECK_NONE = 0,
    TIM_CHECK_TARGET = 1,          /* target id >= V */
    TIM_CHECK_MASK = 2,            /* mask byte not 0 or 1 */
    TIM_CHECK_LOGIT = 3,           /* non-finite logit */
    TIM_CHECK_BACKWARD_INPUT = 4,  /* non-finite lse or upstream gradient */
    TIM_CHECK_ADVANTAGE = 5,       /* non-finite PPO advantage */
    TIM_CHECK_TMA_COORD = 6,       /* a TMA load's innermost coordinate not a whole 16 bytes, or negative */
    TIM_CHECK_STORE = 7,           /* a store outside its buffer */
    TIM_CHECK_UNIT = 8,            /* a claimed work unit out of range */
    TIM_CHECK_BULK = 9             /* a bulk copy not 16-byte aligned or sized */
};
TIM_API int tim_debug_violation(int64_t out[4], tim_stream_t stream);
TIM_API int tim_debug_build(void);

/* ------------------------------------------------------------------ status */

/* Synchronises `stream`, then returns and clears the status word the kernels
 * of the current device recorded since the last tim_check (TIM_OK if none). */
TIM_API int tim_check(tim_stream_t stream);

/* Message for the last non-OK return on the calling thread ("" if none). */
TIM_API const char *tim_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
TIM_API int tim_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TIM_H */
