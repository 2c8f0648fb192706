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
