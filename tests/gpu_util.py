"""Helpers shared by the GPU parity tests: comparison rules against the oracle.

Tolerances (written here, used by every GPU test):
  * token logprob and lse: 2e-3 absolute (the stated contract), per element;
  * mismatch statistics: 1e-5 relative.  Counts must be exact; ratios of
    counts within 1e-6 relative (the device divides in fp32).  Signed means (mean delta, mean k1) compare against the natural
    scale of their cancellation, max(|oracle|, oracle mean |delta|).  The
    rejection flag may differ only where the oracle's statistic is within
    1e-5 relative of the threshold.
  * TIS-weighted PPO surrogate: token loss and gradient 1e-5 relative per
    element (fp32 exp2 and three roundings stay below 2e-6 for |log-ratio| < 10);
    the clip decisions exact (same zero-gradient tokens, same counts); sequence
    and batch means 1e-5 of the matching mean |loss| (advantages of both signs
    cancel in the sums).
"""
import math

import numpy as np

import oracle

LOGP_ATOL = 2e-3
STAT_RTOL = 1e-5

SF = {n: i for i, n in enumerate(oracle.SEQ_FIELDS)}
BF = {n: i for i, n in enumerate(oracle.BATCH_FIELDS)}

_COUNTS = ("n_mask", "n_used", "n_nan", "n_clip")
_SIGNED = ("mean_delta", "mean_k1")
_POS = ("mean_abs_delta", "max_abs_delta", "mean_k2", "mean_k3", "mean_w", "mean_rel")


def _close(g, o, scale, what):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    scale = np.asarray(scale, np.float64)
    bad = ~(np.abs(g - o) <= STAT_RTOL * scale + 1e-30)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError("%s: %d mismatches, first at %d: gpu %r oracle %r scale %r"
                             % (what, int(bad.sum()), i, g.flat[i], o.flat[i], scale.flat[i]))


def assert_seq_stats_match(g_seq, o_seq):
    g = np.asarray(g_seq, np.float64)
    o = np.asarray(o_seq, np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    for f in _COUNTS:
        assert np.array_equal(g[:, SF[f]], o[:, SF[f]]), f
    for f in _SIGNED:
        _close(g[:, SF[f]], o[:, SF[f]], np.maximum(np.abs(o[:, SF[f]]), o[:, SF["mean_abs_delta"]]), f)
    for f in _POS:
        _close(g[:, SF[f]], o[:, SF[f]], np.abs(o[:, SF[f]]), f)


def assert_flags_match(g_flags, o_flags, o_seq, tau, estimator=3):
    g = np.asarray(g_flags)
    o = np.asarray(o_flags)
    stat = o_seq[:, SF["mean_k3"]] if estimator == 3 else np.abs(o_seq[:, SF["mean_k1"]])
    near = np.abs(stat - tau) <= STAT_RTOL * abs(tau)
    assert np.all((g == o) | near), np.nonzero((g != o) & ~near)


def assert_batch_match(g_b, o_b):
    g = np.asarray(g_b, np.float64)
    o = np.asarray(o_b, np.float64)
    for f in ("n_mask", "n_used", "n_nan", "n_clip", "n_seqs_nonempty"):
        assert g[BF[f]] == o[BF[f]], (f, g[BF[f]], o[BF[f]])
    for f in ("clip_ratio", "nan_ratio", "reject_ratio"):   # quotients of exact counts
        _close(g[BF[f]], o[BF[f]], abs(o[BF[f]]) * 0.1, f)
    for f in ("mean_delta", "mean_k1"):
        _close(g[BF[f]], o[BF[f]], max(abs(o[BF[f]]), o[BF["mean_abs_delta"]]), f)
    for f in ("mean_abs_delta", "max_abs_delta", "mean_k2", "mean_k3", "mean_w", "mean_rel",
              "seqmean_k2", "seqmean_k3"):
        _close(g[BF[f]], o[BF[f]], abs(o[BF[f]]), f)
    # the mean over sequences of a signed mean: scale by the sequences' mean |delta|
    _close(g[BF["seqmean_k1"]], o[BF["seqmean_k1"]], max(abs(o[BF["seqmean_k1"]]), o[BF["mean_abs_delta"]]),
           "seqmean_k1")


def default_tau(C):
    return (C - 1.0) - math.log(C)


PF = {n: i for i, n in enumerate(oracle.PPO_FIELDS)}


def assert_ppo_match(g, o, off, what=""):
    """g: dict of numpy arrays from the device (token_loss / token_grad may be
    None); o: the oracle's dict on the same inputs."""
    o_loss = o["token_loss"]
    if g.get("token_loss") is not None:
        _close(g["token_loss"], o_loss, np.abs(o_loss), what + " token_loss")
    if g.get("token_grad") is not None:
        assert np.array_equal(g["token_grad"] == 0, o["token_grad"] == 0), what + " clipped set"
        _close(g["token_grad"], o["token_grad"], np.abs(o["token_grad"]), what + " token_grad")
    off = np.asarray(off, np.int64)
    S = off.size - 1
    abs_loss = np.abs(o_loss)
    csum = np.concatenate([[0.0], np.cumsum(abs_loss)])
    cnz = np.concatenate([[0], np.cumsum(o_loss != 0)])
    # a sequence's scale: the mean |loss| over its tokens with a nonzero loss
    seq_scale = (csum[off[1:]] - csum[off[:-1]]) / np.maximum(cnz[off[1:]] - cnz[off[:-1]], 1)
    o_seq = o["seq_loss"]
    _close(g["seq_loss"], o_seq, np.maximum(np.abs(o_seq), seq_scale), what + " seq_loss")
    gb, ob = np.asarray(g["batch"], np.float64), o["batch"]
    for f in ("n_mask", "n_used", "n_ppo_clipped", "n_tis_clipped", "n_seqs_nonempty"):
        assert gb[PF[f]] == ob[PF[f]], (what, f, gb[PF[f]], ob[PF[f]])
    for f in ("ppo_clip_ratio", "tis_clip_ratio"):
        _close(gb[PF[f]], ob[PF[f]], abs(ob[PF[f]]) * 0.1, what + " " + f)
    n_used = max(ob[PF["n_used"]], 1.0)
    _close(gb[PF["mean_loss"]], ob[PF["mean_loss"]], max(abs(ob[PF["mean_loss"]]), abs_loss.sum() / n_used),
           what + " mean_loss")
    ne = max(ob[PF["n_seqs_nonempty"]], 1.0)
    _close(gb[PF["seqmean_loss"]], ob[PF["seqmean_loss"]],
           max(abs(ob[PF["seqmean_loss"]]), np.abs(o_seq).sum() / ne), what + " seqmean_loss")
    assert S == len(o_seq)
