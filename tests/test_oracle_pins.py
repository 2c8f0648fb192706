"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test names the passage it follows.  None of them re-types the oracle's
own formula as the expected value: the expected values are the pages'
printed numbers, closed forms from probability (KL divergence, log-normal
moments, normal tail), library routines that compute the same quantity by a
different route (scipy's entropy / log_expit, torch's float64 log_softmax),
or exact special cases.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import workloads as wl
from workloads import bf16_round, bf16_to_f32

F = {n: i for i, n in enumerate(oracle.SEQ_FIELDS)}
B = {n: i for i, n in enumerate(oracle.BATCH_FIELDS)}


def _table1(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "table1_qwen3_8b.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tok, lro, ltr, d = line.split()
            rows.append((tok, float(lro), float(ltr), float(d)))
    return rows


# --------------------------------------------------------------- mismatch: pages' numbers
def test_table1_delta_row_reproduced(golden_dir):
    """VeXact summary, Table 1: delta recomputed from the printed logprobs
    matches the printed delta row (fixes delta = train - rollout)."""
    rows = _table1(golden_dir)
    lro = np.array([r[1] for r in rows], np.float32)
    ltr = np.array([r[2] for r in rows], np.float32)
    # one token per sequence: each sequence's mean delta is that token's delta
    off = np.arange(len(rows) + 1, dtype=np.int32)
    out = oracle.mismatch_stats(ltr, lro, np.ones(len(rows), np.uint8), off, C=2.0)
    d = out["seq_stats"][:, F["mean_delta"]]
    for (tok, _, _, printed), got in zip(rows, d):
        assert round(got, 3) == pytest.approx(printed, abs=1e-12), tok


def test_table1_sequence_statistics(golden_dir):
    """Table 1 as one 8-token sequence: mean delta / |delta| / max |delta|
    follow from the printed delta row; nothing is clipped at C = 2 and the
    sequence is not rejected (max |delta| 0.133 is far below the default
    threshold)."""
    rows = _table1(golden_dir)
    lro = np.array([r[1] for r in rows], np.float32)
    ltr = np.array([r[2] for r in rows], np.float32)
    printed = [r[3] for r in rows]
    out = oracle.mismatch_stats(ltr, lro, np.ones(8, np.uint8), np.array([0, 8], np.int32), C=2.0)
    s = out["seq_stats"][0]
    tol = 2e-6  # the inputs are the printed decimals rounded to fp32
    assert s[F["mean_delta"]] == pytest.approx(sum(printed) / 8, abs=tol)
    assert s[F["mean_abs_delta"]] == pytest.approx(sum(abs(x) for x in printed) / 8, abs=tol)
    assert s[F["max_abs_delta"]] == pytest.approx(0.133, abs=tol)
    assert s[F["mean_k1"]] == pytest.approx(-sum(printed) / 8, abs=tol)
    assert s[F["n_used"]] == 8 and s[F["n_clip"]] == 0 and s[F["n_nan"]] == 0
    assert out["seq_flags"][0] == 0
    # k2 = (log r)^2 / 2 with the printed deltas (icarus KL estimator table)
    assert s[F["mean_k2"]] == pytest.approx(sum(x * x for x in printed) / 16, rel=1e-4)


# --------------------------------------------------------------- mismatch: probability pins
def test_k1_and_k3_means_are_the_kl_divergence():
    """Under tokens drawn from the rollout policy mu, E[k1] = E[k3] =
    KL(mu || pi_train) and E[r] = 1 (icarus: k1 and k3 are unbiased KL
    estimators; LoongSage section 4: the IS weight pi_old / pi_rollout).
    Token frequencies equal to mu make the sequence mean the exact expectation."""
    mu = np.array([0.5, 0.25, 0.125, 0.125])
    q = np.array([0.1, 0.2, 0.3, 0.4])
    counts = [4, 2, 1, 1]
    idx = np.repeat(np.arange(4), counts)
    l_ro = np.log(mu)[idx].astype(np.float32)
    l_tr = np.log(q)[idx].astype(np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(8, np.uint8), np.array([0, 8], np.int32), C=1e30)
    kl = scipy.stats.entropy(mu, q)
    s = out["seq_stats"][0]
    assert s[F["mean_k1"]] == pytest.approx(kl, abs=1e-6)
    assert s[F["mean_k3"]] == pytest.approx(kl, abs=1e-6)
    assert s[F["mean_w"]] == pytest.approx(1.0, abs=1e-6)


def test_lognormal_moments_and_normal_tail():
    """delta ~ N(0, s^2): E[k2] = s^2/2, E[k3] = E[r] - 1 = e^{s^2/2} - 1,
    E[min(r, C)] and P(r > C) from the log-normal law.  Tolerances are 6
    standard errors of the sample mean."""
    rng = np.random.default_rng(123)
    n, s = 400_000, 0.5
    C = 1.5
    l_ro = (-rng.gamma(2.0, 1.0, size=n)).astype(np.float32)
    d = rng.normal(0.0, s, size=n)
    l_tr = (l_ro.astype(np.float64) + d).astype(np.float32)
    delta = l_tr.astype(np.float64) - l_ro.astype(np.float64)    # the delta actually fed
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(n, np.uint8), np.array([0, n], np.int32), C=C)
    st = out["seq_stats"][0]
    se = lambda x: 6 * np.std(x) / math.sqrt(n)
    assert st[F["mean_k2"]] == pytest.approx(s * s / 2, abs=se(delta ** 2 / 2))
    assert st[F["mean_k3"]] == pytest.approx(math.exp(s * s / 2) - 1, abs=se(np.exp(delta)))
    lc = math.log(C)
    Ew = math.exp(s * s / 2) * scipy.stats.norm.cdf((lc - s * s) / s) + C * scipy.stats.norm.sf(lc / s)
    assert st[F["mean_w"]] == pytest.approx(Ew, abs=se(np.minimum(np.exp(delta), C)))
    p = scipy.stats.norm.sf(lc / s)
    assert st[F["n_clip"]] / n == pytest.approx(p, abs=6 * math.sqrt(p * (1 - p) / n))
    assert out["batch"][B["clip_ratio"]] == st[F["n_clip"]] / n


def test_small_delta_expansion():
    """k3 - k2 = delta^3/6 + O(delta^4) (Taylor expansion of e^x - 1 - x
    against x^2/2): catches a dropped or extra term in either estimator."""
    for c in (1e-2, -1e-2, 3e-3, -3e-3):
        l_ro = np.full(16, -1.0, np.float32)
        l_tr = (l_ro + np.float32(c)).astype(np.float32)
        d = float(np.float64(l_tr[0]) - np.float64(l_ro[0]))
        out = oracle.mismatch_stats(l_tr, l_ro, np.ones(16, np.uint8), np.array([0, 16], np.int32))
        s = out["seq_stats"][0]
        assert abs((s[F["mean_k3"]] - s[F["mean_k2"]]) - d ** 3 / 6) < d ** 4 / 20


def test_equal_logprobs_give_zero_mismatch():
    """Synced weights and no optimizer step: delta = 0, r = 1 (icarus
    "RL collapse and log p mismatch" section and the debugging checklist)."""
    rng = np.random.default_rng(5)
    l = (-rng.gamma(0.6, 3.0, size=1000)).astype(np.float32)
    off = np.array([0, 300, 300, 1000], np.int32)
    out = oracle.mismatch_stats(l, l, np.ones(1000, np.uint8), off, C=2.0)
    s = out["seq_stats"]
    for f in ("mean_delta", "mean_abs_delta", "max_abs_delta", "mean_k1", "mean_k2", "mean_k3",
              "mean_rel", "n_clip", "n_nan"):
        assert np.all(s[:, F[f]] == 0.0), f
    assert np.all(s[[0, 2], F["mean_w"]] == 1.0)
    assert np.all(out["seq_flags"] == 0)
    b = out["batch"]
    assert b[B["mean_k3"]] == 0 and b[B["mean_w"]] == 1.0 and b[B["n_seqs_nonempty"]] == 2


def test_k3_and_k2_nonnegative_random():
    rng = np.random.default_rng(9)
    n = 20000
    l_ro = (-rng.gamma(0.6, 3.0, size=n)).astype(np.float32)
    l_tr = (l_ro + rng.normal(0, 0.3, size=n)).astype(np.float32)
    off = np.arange(0, n + 1, 10, dtype=np.int32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(n, np.uint8), off)
    assert np.all(out["seq_stats"][:, F["mean_k3"]] >= 0)
    assert np.all(out["seq_stats"][:, F["mean_k2"]] >= 0)
    assert np.all(out["token_weight"] > 0)


def test_rel_diff_uses_train_logprob():
    """icarus compute_consistency_and_kl_metrics: |train - infer| / (|train| + 1e-8)."""
    l_tr = np.array([-1.0, -2.0], np.float32)
    l_ro = np.array([-3.0, -2.02], np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(2, np.uint8), np.array([0, 1, 2], np.int32))
    rel = out["seq_stats"][:, F["mean_rel"]]
    assert rel[0] == pytest.approx(2.0, rel=1e-7)        # not 2/3
    assert rel[1] == pytest.approx(0.01, rel=1e-5)       # the pages' 1% threshold case


def test_per_sequence_then_batch_aggregation():
    """icarus monitoring steps 2-3: mean over a completion's tokens, then mean
    over completions; the token mean over the batch is reported beside it."""
    l_ro = np.zeros(4, np.float32)
    l_tr = np.array([-1.0, 0.0, 0.0, 0.0], np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(4, np.uint8), np.array([0, 1, 4], np.int32))
    b = out["batch"]
    assert b[B["mean_k1"]] == pytest.approx(0.25)          # token mean of k1 = -delta
    assert b[B["seqmean_k1"]] == pytest.approx(0.5)        # (1 + 0) / 2
    assert b[B["mean_delta"]] == pytest.approx(-0.25)
    assert b[B["n_used"]] == 4 and b[B["n_seqs_nonempty"]] == 2


def test_mask_and_nonfinite_tokens():
    """Masked tokens (prompt / padding) never enter the statistics; a masked-in
    token with a non-finite log-ratio is counted in nan_ratio and left out
    (LoongSage section 5, is_nan_ratio)."""
    l_ro = np.array([-1, -1, -1, -1, -1, -1], np.float32)
    l_tr = np.array([-1.5, -1, np.nan, -1, np.inf, 100.0], np.float32)
    mask = np.array([1, 1, 1, 1, 0, 0], np.uint8)
    out = oracle.mismatch_stats(l_tr, l_ro, mask, np.array([0, 6], np.int32), C=2.0)
    s = out["seq_stats"][0]
    assert s[F["n_mask"]] == 4 and s[F["n_used"]] == 3 and s[F["n_nan"]] == 1
    assert s[F["mean_delta"]] == pytest.approx(-0.5 / 3)
    assert out["token_weight"][2] == 0 and out["token_weight"][5] == 0
    assert out["batch"][B["nan_ratio"]] == pytest.approx(0.25)


def test_empty_and_all_masked_sequences():
    l = np.zeros(5, np.float32)
    off = np.array([0, 0, 2, 2, 5], np.int32)
    mask = np.array([0, 0, 1, 1, 1], np.uint8)
    out = oracle.mismatch_stats(l, l - np.float32(0.1), mask, off)
    s = out["seq_stats"]
    assert np.all(s[[0, 1, 2]] == 0)                  # empty, all-masked, empty
    assert s[3, F["n_used"]] == 3
    assert out["batch"][B["n_seqs_nonempty"]] == 1
    # the mean over sequences of per-sequence means (icarus monitoring steps 2-3)
    # leaves out sequences without a used token (the reading for them: no mean
    # to take): with one non-empty sequence it is that sequence's own mean
    for k in ("k1", "k2", "k3"):
        assert out["batch"][B["seqmean_" + k]] == s[3, F["mean_" + k]] != 0
    z = oracle.mismatch_stats(np.zeros(0, np.float32), np.zeros(0, np.float32),
                              np.zeros(0, np.uint8), np.array([0], np.int32))
    assert np.all(z["batch"] == 0)


@pytest.mark.parametrize("est,delta,flag", [
    (3, 0.8, 1), (3, 0.6, 0), (3, -1.0, 1), (3, -0.9, 0),
    (1, 0.35, 1), (1, -0.35, 1), (1, 0.30, 0),
])
def test_sequence_rejection_default_threshold(est, delta, flag):
    """VeXact "Algorithmic TIM Compensation": reject a sequence whose K3 (or K1)
    of r_corr = pi_train / pi_rollout is too large.  With constant delta the
    sequence mean is the single-token value; the default threshold is k3 at
    r = C, (C - 1) - ln C = 0.30685 for C = 2."""
    l_ro = np.full(10, -2.0, np.float32)
    l_tr = (l_ro + np.float32(delta)).astype(np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(10, np.uint8), np.array([0, 10], np.int32),
                                C=2.0, seq_estimator=est)
    assert out["seq_flags"][0] == flag


def test_clip_is_strict_and_decided_on_fp32_delta():
    """r > C is strict; the fp32 delta nearest above ln 2 clips, the one just
    below does not."""
    ln2 = np.float32(math.log(2.0))
    below = ln2 if float(ln2) < math.log(2.0) else np.nextafter(ln2, np.float32(-1))
    above = np.nextafter(below, np.float32(1))
    l_ro = np.zeros(2, np.float32)
    l_tr = np.array([below, above], np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(2, np.uint8), np.array([0, 1, 2], np.int32), C=2.0)
    assert list(out["seq_stats"][:, F["n_clip"]]) == [0, 1]


def test_clip_is_strict_at_C_equal_one():
    """C = 1 is the one cap whose log (0) an fp32 delta can equal: a token with
    delta = 0 has r = C exactly and is not clipped (r > C is strict); the next
    fp32 delta above it is.  Both weights are min(r, C) = 1."""
    l_ro = np.full(2, -3.0, np.float32)
    l_tr = np.array([-3.0, np.nextafter(np.float32(-3.0), np.float32(0))], np.float32)
    out = oracle.mismatch_stats(l_tr, l_ro, np.ones(2, np.uint8), np.array([0, 1, 2], np.int32), C=1.0)
    assert list(out["seq_stats"][:, F["n_clip"]]) == [0, 1]
    assert list(out["token_weight"]) == [1.0, 1.0]


def test_clip_and_nan_ratios_count_every_masked_in_token():
    """LoongSage sections 4-5, is_clip_ratio and is_nan_ratio over the same
    population, the masked-in tokens: four masked-in tokens, one clipped
    (delta = 1 > ln 2), one non-finite, two at delta = 0, and one masked-out
    clipped token -> both ratios 1/4."""
    l_ro = np.full(5, -1.0, np.float32)
    l_tr = np.array([-1.0, 0.0, np.nan, -1.0, 0.0], np.float32)
    mask = np.array([1, 1, 1, 1, 0], np.uint8)
    out = oracle.mismatch_stats(l_tr, l_ro, mask, np.array([0, 5], np.int32), C=2.0)
    b = out["batch"]
    assert (b[B["n_mask"]], b[B["n_used"]], b[B["n_nan"]], b[B["n_clip"]]) == (4, 3, 1, 1)
    assert b[B["clip_ratio"]] == 0.25 and b[B["nan_ratio"]] == 0.25


def test_bad_offsets_rejected():
    l = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.mismatch_stats(l, l, np.ones(4, np.uint8), np.array([0, 3, 2, 4], np.int32))
    with pytest.raises(ValueError):
        oracle.mismatch_stats(l, l, np.ones(4, np.uint8), np.array([0, 3], np.int32))


# --------------------------------------------------------------- token logprob pins
def _rand_head(N, D, V, seed, w_std=0.05):
    rng = np.random.default_rng(seed)
    h = bf16_round(rng.standard_normal((N, D)).astype(np.float32))
    W = bf16_round((rng.standard_normal((V, D)) * w_std).astype(np.float32))
    a = rng.integers(0, V, size=N).astype(np.int32)
    return h, W, a


def test_zero_weight_gives_uniform():
    """W = 0: every logit is 0, so l_t = -log V and lse = log V."""
    for V in (1, 2, 1000, 1024):
        h, _, a = _rand_head(5, 64, V, 1)
        W = np.zeros((V, 64), np.uint16)
        logp, lse = oracle.token_logprob(h, W, a)
        assert np.all(logp == -math.log(V)) and np.all(lse == math.log(V))


def test_probabilities_sum_to_one_and_lse_is_shared():
    """sum_v exp(log p(v | h)) = 1: replicate one row V times with targets
    0..V-1; every copy has the same lse."""
    V, D = 257, 72
    h, W, _ = _rand_head(1, D, V, 2, w_std=0.2)
    hh = np.repeat(h, V, axis=0)
    logp, lse = oracle.token_logprob(hh, W, np.arange(V, dtype=np.int32))
    assert abs(math.fsum(np.exp(logp)) - 1.0) < 1e-12
    assert np.all(lse == lse[0])


def test_against_torch_float64_log_softmax_gather():
    """The icarus page's PyTorch statement log_softmax(logits).gather(ids),
    run in float64 by torch, on tiny shapes; catches a transposed operand."""
    torch = pytest.importorskip("torch")
    for (N, D, V) in ((64, 256, 1024), (7, 72, 130), (3, 8, 1)):
        h, W, a = _rand_head(N, D, V, N + D + V)
        logp, lse = oracle.token_logprob(h, W, a)
        ht = torch.from_numpy(bf16_to_f32(h).astype(np.float64))
        Wt = torch.from_numpy(bf16_to_f32(W).astype(np.float64))
        z = ht @ Wt.T
        ref = torch.log_softmax(z, dim=-1).gather(-1, torch.from_numpy(a.astype(np.int64))[:, None])[:, 0]
        np.testing.assert_allclose(logp, ref.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse, torch.logsumexp(z, -1).numpy(), rtol=0, atol=1e-11)


def test_two_class_closed_form():
    """V = 2: log p(1) = log sigmoid(z1 - z0) (scipy.special.log_expit)."""
    D = 16
    h, W, _ = _rand_head(32, D, 2, 3, w_std=0.5)
    logp, _ = oracle.token_logprob(h, W, np.ones(32, np.int32))
    z = bf16_to_f32(h).astype(np.float64) @ bf16_to_f32(W).astype(np.float64).T
    np.testing.assert_allclose(logp, scipy.special.log_expit(z[:, 1] - z[:, 0]), rtol=0, atol=1e-12)


def test_logit_shift_moves_lse_only():
    """Adding c to every logit (h[:, D-1] = 1, W[:, D-1] = c) raises lse by c
    and leaves log p unchanged (softmax is shift invariant)."""
    N, D, V = 6, 40, 300
    h, W, a = _rand_head(N, D, V, 4)
    h[:, D - 1] = bf16_round(np.float32(1.0))
    W0 = W.copy()
    W0[:, D - 1] = 0
    Wc = W.copy()
    Wc[:, D - 1] = bf16_round(np.float32(3.0))
    l0, s0 = oracle.token_logprob(h, W0, a)
    l1, s1 = oracle.token_logprob(h, Wc, a)
    np.testing.assert_allclose(l1, l0, atol=1e-12)
    np.testing.assert_allclose(s1 - s0, 3.0, atol=1e-12)


def test_one_hot_margin_and_bad_targets():
    """A target whose logit dominates by a wide margin has log p -> 0; a target
    outside [0, V) (the -100 ignore label) gives NaN with a valid lse."""
    D, V = 8, 50
    h = np.zeros((3, D), np.uint16)
    h[:, 0] = bf16_round(np.float32(1.0))
    W = np.zeros((V, D), np.uint16)
    W[7, 0] = bf16_round(np.float32(200.0))
    logp, lse = oracle.token_logprob(h, W, np.array([7, -100, V], np.int32))
    assert abs(logp[0]) < 1e-80
    assert np.isnan(logp[1]) and np.isnan(logp[2])
    assert np.all(np.isfinite(lse)) and lse[1] == pytest.approx(200.0)


def test_row_subset_matches_full():
    h, W, a = _rand_head(20, 32, 100, 6)
    lf, sf = oracle.token_logprob(h, W, a)
    rows = np.array([19, 0, 7])
    lr, sr = oracle.token_logprob(h, W, a, rows=rows, nthreads=2)
    assert np.array_equal(lr, lf[rows]) and np.array_equal(sr, sf[rows])


# --------------------------------------------------------------- temperature
def test_temperature_matches_scaled_weights_exactly():
    """softmax(z / 2) with W equals softmax(z) with W / 2 (an exact bf16 scale):
    the temperature divides the logits, not the probabilities (icarus, section
    "logits processor": sampling uses softmax(z / tau))."""
    h, W, a = _rand_head(9, 48, 700, 21, w_std=0.3)
    W_half = wl.bf16_round(wl.bf16_to_f32(W) * np.float32(0.5))
    l2, s2 = oracle.token_logprob(h, W, a, temperature=2.0)
    l1, s1 = oracle.token_logprob(h, W_half, a)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-13)


def test_temperature_limits_and_two_class_form():
    """tau -> infinity flattens to -log V; V = 2 gives log sigmoid((z1 - z0) / tau)."""
    h, W, a = _rand_head(5, 32, 300, 22, w_std=0.5)
    l, _ = oracle.token_logprob(h, W, a, temperature=1e9)
    assert np.max(np.abs(l + math.log(300))) < 1e-6
    h2, W2, _ = _rand_head(16, 16, 2, 23, w_std=0.5)
    lp, _ = oracle.token_logprob(h2, W2, np.ones(16, np.int32), temperature=0.7)
    z = bf16_to_f32(h2).astype(np.float64) @ bf16_to_f32(W2).astype(np.float64).T
    np.testing.assert_allclose(lp, scipy.special.log_expit((z[:, 1] - z[:, 0]) / 0.7), rtol=0, atol=1e-12)
    with pytest.raises(RuntimeError):
        oracle.token_logprob(h2, W2, np.ones(16, np.int32), temperature=0.0)


# --------------------------------------------------------------- TIS-weighted PPO surrogate
P = {n: i for i, n in enumerate(oracle.PPO_FIELDS)}
NO_CLIP = dict(eps_low=0.999999, eps_high=1e9, C=1e30)


def _ppo(lt, lo, lr, A, mask=None, offsets=None, **kw):
    lt, lo, lr, A = (np.asarray(x, np.float32) for x in (lt, lo, lr, A))
    n = lt.size
    m = np.ones(n, np.uint8) if mask is None else np.asarray(mask, np.uint8)
    off = np.array([0, n], np.int32) if offsets is None else np.asarray(offsets, np.int32)
    return oracle.tis_ppo(lt, lo, lr, A, m, off, **kw)


def test_ppo_importance_sampling_identity():
    """Tokens drawn from the rollout policy, weighted by pi_old / pi_rollout
    (TIS with no truncation) and by r = pi_theta / pi_old: the mean surrogate
    is -E_{pi_theta}[A], the on-policy objective (VeXact summary eq. (3) and
    the TIS correction; LoongSage section 4).  The rollout distribution is
    realised exactly by token counts; swapping old and rollout, or theta and
    old, moves the mean far off."""
    counts = np.array([400, 250, 200, 100, 50])            # p_rollout = counts / 1000
    p_ro = counts / 1000.0
    p_old = np.array([0.30, 0.30, 0.15, 0.15, 0.10])
    p_th = np.array([0.20, 0.35, 0.25, 0.05, 0.15])
    A = np.array([1.5, -0.5, 2.0, -3.0, 0.75])
    tok = np.repeat(np.arange(5), counts)
    o = _ppo(np.log(p_th)[tok], np.log(p_old)[tok], np.log(p_ro)[tok], A[tok], **NO_CLIP)
    exact = -float(np.dot(p_th, A))
    assert abs(o["batch"][P["mean_loss"]] - exact) < 1e-6
    assert o["batch"][P["n_ppo_clipped"]] == 0 and o["batch"][P["n_tis_clipped"]] == 0
    swapped = _ppo(np.log(p_th)[tok], np.log(p_ro)[tok], np.log(p_old)[tok], A[tok], **NO_CLIP)
    assert abs(swapped["batch"][P["mean_loss"]] - exact) > 0.05


def test_ppo_on_policy_is_minus_advantage():
    """r = 1 and w = 1 (theta = old = rollout): the surrogate of every token is
    -A and its gradient -A (eq. (2) at r = 1, whatever eps)."""
    rng = np.random.default_rng(40)
    l = -rng.gamma(0.6, 3.0, 64).astype(np.float32)
    A = rng.standard_normal(64).astype(np.float32)
    o = _ppo(l, l, l, A, eps_low=0.1, eps_high=0.3, C=1.5)
    np.testing.assert_array_equal(o["token_loss"], -A.astype(np.float64))
    np.testing.assert_array_equal(o["token_grad"], -A.astype(np.float64))
    assert o["batch"][P["n_ppo_clipped"]] == 0 and o["batch"][P["n_tis_clipped"]] == 0


def test_ppo_case_form_of_the_clipped_objective():
    """The clipped surrogate as a function of r (eq. (2)): for A > 0 it is
    -A min(r, 1 + eps_high), for A < 0 it is -A max(r, 1 - eps_low); the
    gradient is zero exactly where the clipped value is the one taken (HN
    page, "Clipped importance ratios"); eps_low and eps_high act on their own
    sides.  w = 1 here (old = rollout)."""
    eps_low, eps_high = 0.2, 0.28
    r = np.array([0.3, 0.79, 0.81, 1.0, 1.27, 1.29, 3.0])
    lo = np.full(r.size, -1.0)
    lt = (np.log(r) + lo).astype(np.float32)
    r32 = np.exp(lt.astype(np.float64) - np.float32(-1.0))
    for sign in (1.0, -1.0):
        A = np.full(r.size, 1.7 * sign, np.float32).astype(np.float64)
        o = _ppo(lt, lo, lo, A, eps_low=eps_low, eps_high=eps_high, C=2.0)
        taken = np.minimum(r32, 1 + eps_high) if sign > 0 else np.maximum(r32, 1 - eps_low)
        np.testing.assert_allclose(o["token_loss"], -A * taken, rtol=1e-15, atol=0)
        flat = r32 > 1 + eps_high if sign > 0 else r32 < 1 - eps_low
        assert np.array_equal(o["token_grad"] == 0, flat)
        assert o["batch"][P["n_ppo_clipped"]] == flat.sum()
        np.testing.assert_allclose(o["batch"][P["ppo_clip_ratio"]], flat.mean(), rtol=1e-15)


def test_ppo_ties_keep_the_gradient():
    """With eps = 0 the ratio r = 1 sits on both clip bounds: both terms of the
    min are equal there and the token keeps its gradient (the reading: the
    clipped branch is taken only where it is strictly smaller); the next fp32
    log-ratio above 0 is clipped for A > 0 and not for A < 0."""
    lo = np.full(4, -2.0, np.float32)
    up = np.nextafter(np.float32(-2.0), np.float32(0))
    lt = np.array([-2.0, -2.0, up, up], np.float32)
    A = np.array([1.5, -1.5, 1.5, -1.5])
    o = _ppo(lt, lo, lo, A, eps_low=0.0, eps_high=0.0, C=2.0)
    assert o["token_grad"][0] == -1.5 and o["token_grad"][1] == 1.5
    assert o["token_grad"][2] == 0 and o["token_grad"][3] != 0
    assert o["batch"][P["n_ppo_clipped"]] == 1


def test_ppo_gradient_is_the_derivative_of_the_loss():
    """token_grad = d token_loss / d logp_theta, checked by central differences
    of the oracle's own loss (step 2^-9, tokens at least 4 steps away from a
    clip boundary)."""
    rng = np.random.default_rng(41)
    n = 400
    lo = -rng.gamma(0.6, 3.0, n).astype(np.float32)
    lt = (lo + rng.normal(0, 0.25, n)).astype(np.float32)
    lr = (lo + rng.normal(0, 0.4, n)).astype(np.float32)
    A = rng.standard_normal(n).astype(np.float32)
    kw = dict(eps_low=0.2, eps_high=0.28, C=1.8)
    hstep = np.float32(2.0 ** -9)
    d = lt.astype(np.float64) - lo
    far = (np.abs(d - math.log1p(0.28)) > 4 * hstep) & (np.abs(d - math.log1p(-0.2)) > 4 * hstep)
    o = _ppo(lt, lo, lr, A, **kw)
    up = _ppo(lt + hstep, lo, lr, A, **kw)["token_loss"]
    dn = _ppo(lt - hstep, lo, lr, A, **kw)["token_loss"]
    fd = (up - dn) / (2 * float(hstep))
    exact_steps = ((lt + hstep) - (lt - hstep)).astype(np.float64) == 2 * float(hstep)
    sel = far & exact_steps
    assert sel.sum() > 300
    np.testing.assert_allclose(o["token_grad"][sel], fd[sel], rtol=2e-5, atol=1e-9)


def test_ppo_tis_weight_truncation():
    """w = min(pi_old / pi_rollout, C) (LoongSage section 4): below the cap the
    loss scales with 1 / pi_rollout; above it, lowering pi_rollout further
    changes nothing, and the token counts as TIS-clipped."""
    lt = np.array([-1.0, -2.0], np.float32)
    lo = np.array([-1.1, -2.2], np.float32)
    A = np.array([0.5, -2.0], np.float32)
    C = 3.0
    base = _ppo(lt, lo, lo + np.float32(0.25), A, eps_low=0.2, eps_high=0.2, C=C)
    down = _ppo(lt, lo, lo - np.float32(0.25), A, eps_low=0.2, eps_high=0.2, C=C)
    np.testing.assert_allclose(down["token_loss"], base["token_loss"] * math.exp(0.5), rtol=1e-6)
    capped = _ppo(lt, lo, lo - np.float32(2.0), A, eps_low=0.2, eps_high=0.2, C=C)
    capped2 = _ppo(lt, lo, lo - np.float32(5.0), A, eps_low=0.2, eps_high=0.2, C=C)
    np.testing.assert_array_equal(capped["token_loss"], capped2["token_loss"])
    w1 = _ppo(lt, lo, lo, A, eps_low=0.2, eps_high=0.2, C=C)
    np.testing.assert_allclose(capped["token_loss"], C * w1["token_loss"], rtol=1e-15)
    assert capped["batch"][P["n_tis_clipped"]] == 2 and base["batch"][P["n_tis_clipped"]] == 0


def test_ppo_masks_nonfinite_and_means():
    """Masked and non-finite tokens contribute nothing; the token mean divides
    by used tokens, the sequence mean averages non-empty sequences."""
    lt = np.array([-1.0, -1.0, np.nan, -1.0, -1.0, -1.0, -1.0], np.float32)
    lo = lt.copy()
    lo[2] = -1.0
    A = np.array([1.0, 2.0, 5.0, 7.0, 3.0, 3.0, 100.0], np.float32)
    mask = np.array([1, 1, 1, 0, 1, 1, 0], np.uint8)
    off = np.array([0, 4, 4, 6, 7], np.int32)     # seq 1 empty, seq 3 fully masked
    o = _ppo(lt, lo, lo, A, mask=mask, offsets=off, eps_low=0.2, eps_high=0.2, C=2.0)
    assert o["token_loss"][2] == 0 and o["token_loss"][3] == 0 and o["token_grad"][6] == 0
    np.testing.assert_array_equal(o["seq_loss"], [-1.5, 0.0, -3.0, 0.0])
    b = o["batch"]
    assert (b[P["n_mask"]], b[P["n_used"]], b[P["n_seqs_nonempty"]]) == (5, 4, 2)
    assert b[P["mean_loss"]] == -9.0 / 4 and b[P["seqmean_loss"]] == -2.25


def test_ppo_bad_arguments_rejected():
    z = np.zeros(3, np.float32)
    for kw in (dict(eps_low=1.0), dict(eps_low=-0.1), dict(eps_high=-0.1), dict(C=0.0), dict(C=float("nan"))):
        with pytest.raises(ValueError):
            oracle.tis_ppo(z, z, z, z, np.ones(3, np.uint8), np.array([0, 3], np.int32), **kw)
    with pytest.raises(ValueError):
        oracle.tis_ppo(z, z, z, z, np.ones(3, np.uint8), np.array([0, 2], np.int32))


# --------------------------------------------------------------- mismatch monitor
MF = {n: i for i, n in enumerate(oracle.MONITOR_FIELDS)}


def _delta32(lt, lr):
    return (np.asarray(lt, np.float32) - np.asarray(lr, np.float32)).astype(np.float64)


def test_monitor_quantiles_match_numpy_linear_quantile():
    """The quantiles are numpy's default ("linear", h = (n - 1) q) over the used
    tokens: |delta| at 0.95, r = e^delta at 0.01 / 0.5 / 0.99 (llm-infra-atlas
    section 7's metric list).  Masked and non-finite tokens are left out."""
    rng = np.random.default_rng(50)
    for n in (1, 2, 3, 10, 101, 5000):
        lt = wl.draw_train_logprobs(n, 50 + n)
        lr = (lt + rng.normal(0, 0.05, n)).astype(np.float32)
        mask = (rng.random(n) < 0.8).astype(np.uint8)
        if n > 3:
            lt[1] = np.nan
            lr[2] = -np.inf
            mask[[1, 2]] = 1
        o = oracle.mismatch_monitor(lt, lr, mask, 0.1)["batch"]
        d = _delta32(lt, lr)
        used = (mask != 0) & np.isfinite(d)
        assert o[MF["n_used"]] == used.sum()
        if used.sum() == 0:
            assert np.isnan(o[MF["p95_abs_delta"]])
            continue
        du = d[used]
        np.testing.assert_allclose(o[MF["p95_abs_delta"]], np.quantile(np.abs(du), 0.95), rtol=1e-14)
        for f, q in (("ratio_q01", 0.01), ("ratio_q50", 0.5), ("ratio_q99", 0.99)):
            np.testing.assert_allclose(o[MF[f]], np.quantile(np.exp(du), q), rtol=1e-14)


def test_monitor_normal_law():
    """delta ~ N(0, s^2): p95 |delta| -> 1.95996 s, median ratio -> 1,
    q99 ratio -> e^{2.32635 s}, P(|delta| > tau) -> 2 (1 - Phi(tau / s)) among
    the used tokens (30 % of the batch masked out, with |delta| = 1 there);
    tolerances are five standard errors of the sample quantile / fraction."""
    N, s, tau = 1_400_000, 0.05, 0.08
    rng = np.random.default_rng(51)
    lr = wl.draw_train_logprobs(N, 51)
    lt = (lr.astype(np.float64) + rng.normal(0, s, N)).astype(np.float32)
    mask = (rng.random(N) >= 0.3).astype(np.uint8)
    lt[mask == 0] = lr[mask == 0] + np.float32(1.0)
    n = int(mask.sum())
    o = oracle.mismatch_monitor(lt, lr, mask, tau)["batch"]
    assert o[MF["n_used"]] == n
    z95 = scipy.stats.norm.ppf(0.975)
    se = math.sqrt(0.95 * 0.05 / n) / (2 * scipy.stats.norm.pdf(z95) / s)
    assert abs(o[MF["p95_abs_delta"]] - z95 * s) < 5 * se
    se50 = math.sqrt(0.25 / n) / (scipy.stats.norm.pdf(0) / s)
    assert abs(math.log(o[MF["ratio_q50"]])) < 5 * se50
    z99 = scipy.stats.norm.ppf(0.99)
    se99 = math.sqrt(0.99 * 0.01 / n) / (scipy.stats.norm.pdf(z99) / s)
    assert abs(math.log(o[MF["ratio_q99"]]) - z99 * s) < 5 * se99
    assert abs(math.log(o[MF["ratio_q01"]]) + z99 * s) < 5 * se99
    p = 2 * scipy.stats.norm.sf(tau / s)
    assert abs(o[MF["frac_extreme"]] - p) < 5 * math.sqrt(p * (1 - p) / n)


def test_monitor_exact_small_cases_and_rejection():
    """Single token: every quantile is that token; two tokens: the median is
    the midpoint of the two ratios; the reject flag is |delta| > tau_tok,
    strict, only for used tokens (VeXact summary, tau_tok)."""
    one = oracle.mismatch_monitor(np.float32([-1.0]), np.float32([-1.5]), np.uint8([1]), 0.5)
    b = one["batch"]
    assert b[MF["p95_abs_delta"]] == 0.5 and b[MF["ratio_q01"]] == b[MF["ratio_q99"]] == math.exp(0.5)
    assert one["reject"][0] == 0 and b[MF["n_extreme"]] == 0          # |delta| = tau exactly: kept
    two = oracle.mismatch_monitor(np.float32([-1.0, -2.0]), np.float32([-1.25, -1.5]), np.uint8([1, 1]), 0.3)
    assert two["batch"][MF["ratio_q50"]] == pytest.approx((math.exp(0.25) + math.exp(-0.5)) / 2, rel=1e-15)
    assert list(two["reject"]) == [0, 1] and two["batch"][MF["frac_extreme"]] == 0.5
    masked = oracle.mismatch_monitor(np.float32([0.0, -3.0]), np.float32([-5.0, -3.0]), np.uint8([0, 1]), 0.1)
    assert list(masked["reject"]) == [0, 0] and masked["batch"][MF["ratio_q50"]] == 1.0
    empty = oracle.mismatch_monitor(np.float32([np.nan]), np.float32([0.0]), np.uint8([1]), 0.1)["batch"]
    assert empty[MF["n_used"]] == 0 and np.isnan(empty[MF["ratio_q50"]]) and empty[MF["frac_extreme"]] == 0


def test_monitor_is_order_free():
    rng = np.random.default_rng(52)
    n = 3001
    lt = wl.draw_train_logprobs(n, 52)
    lr = (lt + rng.normal(0, 0.1, n)).astype(np.float32)
    m = (rng.random(n) < 0.7).astype(np.uint8)
    p = rng.permutation(n)
    a = oracle.mismatch_monitor(lt, lr, m, 0.15)
    b = oracle.mismatch_monitor(lt[p], lr[p], m[p], 0.15)
    assert np.array_equal(a["batch"], b["batch"]) and np.array_equal(a["reject"][p], b["reject"])


# --------------------------------------------------------------- FP32 LM head
def test_f32_weights_holding_bf16_values_match_the_bf16_oracle():
    """fp32 weights that are exactly bf16 values give the bf16 oracle's bits
    (both sides take the same exact products)."""
    h, W, a = _rand_head(11, 40, 300, 60, w_std=0.2)
    l1, s1 = oracle.token_logprob(h, W, a)
    l2, s2 = oracle.token_logprob_f32w(h, bf16_to_f32(W), a)
    assert np.array_equal(l1, l2) and np.array_equal(s1, s2)


def test_f32_weights_against_torch_float64():
    """fp32 weights that are not bf16 values: torch float64 log_softmax of
    h W^T / tau (another route to the same definition), tau 1 and 0.8."""
    import torch
    rng = np.random.default_rng(61)
    N, D, V = 7, 48, 500
    h = bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = (rng.standard_normal((V, D)) * 0.1).astype(np.float32)
    a = rng.integers(0, V, N).astype(np.int32)
    for tau in (1.0, 0.8):
        lp, lse = oracle.token_logprob_f32w(h, W, a, temperature=tau)
        z = torch.from_numpy(bf16_to_f32(h).astype(np.float64)) @ torch.from_numpy(W.astype(np.float64)).T / tau
        ref = torch.log_softmax(z, dim=-1).gather(1, torch.from_numpy(a.astype(np.int64))[:, None])[:, 0]
        np.testing.assert_allclose(lp, ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, torch.logsumexp(z, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_f32_weights_differ_from_their_bf16_rounding():
    """The fp32 head is not the bf16 head in disguise: rounding W to bf16
    moves the logprobs by ~1e-3 (the error the FP32 head removes)."""
    rng = np.random.default_rng(62)
    N, D, V = 6, 512, 800
    h = bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = (rng.standard_normal((V, D)) * 0.05).astype(np.float32)
    a = rng.integers(0, V, N).astype(np.int32)
    lf, _ = oracle.token_logprob_f32w(h, W, a)
    lb, _ = oracle.token_logprob(h, bf16_round(W), a)
    assert 1e-5 < np.max(np.abs(lf - lb)) < 1e-1


# --------------------------------------------------------------- token logprob backward
def _bw_case(N, D, V, seed, w_std=0.2):
    h, W, a = _rand_head(N, D, V, seed, w_std=w_std)
    g = np.random.default_rng(seed + 1).standard_normal(N).astype(np.float32)
    return h, W, a, g


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_backward_against_torch_autograd(tau):
    """dh and dW equal torch float64 autograd of sum_t g_t log_softmax(h W^T / tau)[a_t]
    (reverse-mode differentiation: another route than the closed form)."""
    import torch
    h, W, a, g = _bw_case(6, 24, 50, 80)
    o = oracle.token_logprob_backward(h, W, a, g, temperature=tau, want_dz=True)
    ht = torch.tensor(bf16_to_f32(h).astype(np.float64), requires_grad=True)
    Wt = torch.tensor(bf16_to_f32(W).astype(np.float64), requires_grad=True)
    lp = torch.log_softmax(ht @ Wt.T / tau, dim=-1).gather(1, torch.from_numpy(a.astype(np.int64))[:, None])[:, 0]
    (lp * torch.from_numpy(g.astype(np.float64))).sum().backward()
    np.testing.assert_allclose(o["dh"], ht.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["dW"], Wt.grad.numpy(), rtol=0, atol=1e-12)
    assert np.max(np.abs(o["dz"].sum(axis=1))) < 1e-12   # softmax gradient rows sum to zero


def test_backward_dW_by_central_differences():
    """dW[v, d] = d (sum_t g_t l_t) / d W[v, d] by central differences of the
    fp32-weight forward oracle (weights on a 2^-12 grid, step 2^-10, exact in
    fp32); the bf16 weights of the backward are the same values."""
    rng = np.random.default_rng(81)
    N, D, V = 5, 16, 40
    h = bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    Wq = (np.round(rng.standard_normal((V, D)) * 0.3 * 64) / 64).astype(np.float32)   # bf16-exact, 2^-6 grid
    W = bf16_round(Wq)
    assert np.array_equal(bf16_to_f32(W), Wq)
    a = rng.integers(0, V, N).astype(np.int32)
    g = rng.standard_normal(N).astype(np.float32)
    o = oracle.token_logprob_backward(h, W, a, g)
    step = 2.0 ** -10
    for (v, d) in [(0, 0), (int(a[0]), 3), (17, 15), (39, 7), (int(a[2]), 0)]:
        Wp, Wm = Wq.copy(), Wq.copy()
        Wp[v, d] += np.float32(step)
        Wm[v, d] -= np.float32(step)
        lp, _ = oracle.token_logprob_f32w(h, Wp, a)
        lm, _ = oracle.token_logprob_f32w(h, Wm, a)
        fd = float(np.dot(g.astype(np.float64), lp - lm)) / (2 * step)
        assert abs(fd - o["dW"][v, d]) < 1e-6 * max(1.0, abs(fd)), (v, d, fd, o["dW"][v, d])


def test_backward_invariants():
    """Every column sum of dW is zero (each row's softmax gradient sums to
    zero); <dW, W> = <dh, h> (both equal sum_t sum_v dz z); g = 0 gives zero;
    a target outside [0, V) drops the one-hot term only."""
    h, W, a, g = _bw_case(8, 32, 60, 82)
    o = oracle.token_logprob_backward(h, W, a, g)
    Wf = bf16_to_f32(W).astype(np.float64)
    hf = bf16_to_f32(h).astype(np.float64)
    assert np.max(np.abs(o["dW"].sum(axis=0))) < 1e-12
    assert abs(np.sum(o["dW"] * Wf) - np.sum(o["dh"] * hf)) < 1e-10
    z = oracle.token_logprob_backward(h, W, a, np.zeros(8, np.float32))
    assert not z["dh"].any() and not z["dW"].any()
    a2 = a.copy()
    a2[0] = -100
    o2 = oracle.token_logprob_backward(h, W, a2, g)
    np.testing.assert_allclose(o2["dh"][0], o["dh"][0] - float(g[0]) * Wf[a[0]], rtol=0, atol=1e-12)


def test_mismatch_stats_on_several_threads_gives_the_same_bits():
    """The oracle sums each sequence alone in token order and folds the
    sequences in index order, so spreading the sequences over threads changes
    no bit of any output (empty sequences, masks and non-finite tokens
    included)."""
    rng = np.random.default_rng(77)
    lens = rng.integers(0, 300, size=700)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 77)
    l_ro = (l_tr + rng.normal(0, 0.3, N)).astype(np.float32)
    l_ro[::101] = np.inf
    mask = (rng.random(N) < 0.7).astype(np.uint8)
    one = oracle.mismatch_stats(l_tr, l_ro, mask, off, C=1.5)
    for nt in (2, 3, 8, 1000):
        many = oracle.mismatch_stats(l_tr, l_ro, mask, off, C=1.5, nthreads=nt)
        for k in one:
            assert np.array_equal(one[k].view(np.uint8), many[k].view(np.uint8)), (nt, k)
