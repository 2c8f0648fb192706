"""GPU parity of tim_mismatch_stats against the fp64 oracle, plus its
determinism properties.  Every call goes through the C ABI (via the binding)."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import (BF, SF, assert_batch_match, assert_flags_match, assert_seq_stats_match,
                      default_tau)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_both(l_tr, l_ro, mask, off, C=2.0, tau=math.nan, est=3, weights=True):
    g = tim.mismatch_stats(_dev(l_tr), _dev(l_ro), _dev(mask), _dev(off), C=C, tau_seq=tau,
                           seq_estimator=est, token_weight=weights)
    tim.check()
    o = oracle.mismatch_stats(l_tr, l_ro, mask, off, C=C, tau_seq=tau, seq_estimator=est)
    gs = {k: (v.cpu().numpy() if v is not None else None) for k, v in g.items()}
    return gs, o


def check_all(gs, o, C=2.0, tau=math.nan, est=3, weights=True):
    assert_seq_stats_match(gs["seq_stats"], o["seq_stats"])
    t = default_tau(C) if math.isnan(tau) else float(np.float32(tau))
    assert_flags_match(gs["seq_flags"], o["seq_flags"], o["seq_stats"], t, est)
    assert_batch_match(gs["batch"], o["batch"])
    if weights:
        w_o = o["token_weight"]
        np.testing.assert_allclose(gs["token_weight"], w_o, rtol=1e-5, atol=0)


def _config_inputs(name, seed=0):
    cfg = wl.CONFIGS[name]
    off = wl.draw_segments(cfg, seed=seed)
    N = int(off[-1])
    mask = wl.draw_mask(cfg, off, seed=seed)
    l_tr = wl.draw_train_logprobs(N, seed)
    l_ro = wl.draw_rollout(cfg, l_tr, seed=seed)
    return cfg, l_tr, l_ro, mask, off


@pytest.mark.parametrize("name", ["qwen3_8b", "llama3_8b", "dsv3"])
def test_config_shapes(name):
    cfg, l_tr, l_ro, mask, off = _config_inputs(name)
    gs, o = run_both(l_tr, l_ro, mask, off, C=cfg.C)
    check_all(gs, o, C=cfg.C)
    # the outliers of the Llama-shaped config exceed C and must clip
    if name == "llama3_8b":
        assert o["batch"][BF["n_clip"]] > 0


def test_tiny_config_from_oracle_logprobs():
    cfg = wl.CONFIGS["tiny"]
    h, W = wl.draw_head(cfg)
    a = wl.draw_targets(cfg, cfg.N)
    l_tr = oracle.token_logprob(h, W, a)[0].astype(np.float32)
    l_ro = wl.draw_rollout(cfg, l_tr)
    off = wl.draw_segments(cfg)
    mask = wl.draw_mask(cfg, off)
    gs, o = run_both(l_tr, l_ro, mask, off)
    check_all(gs, o)


def test_edge_cases_empty_masked_nonfinite():
    rng = np.random.default_rng(7)
    lens = [0, 1, 5, 0, 300, 257, 0, 1024, 3, 8192, 8193, 9000, 2]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 3)
    l_ro = (l_tr + rng.normal(0, 0.3, N)).astype(np.float32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    mask[off[4]:off[5]] = 0                       # an all-masked sequence
    l_tr[10] = np.nan
    l_ro[20] = np.inf
    l_tr[30] = -np.inf
    l_ro[31] = np.nan
    mask[[10, 20, 30]] = 1
    gs, o = run_both(l_tr, l_ro, mask, off)
    check_all(gs, o)
    assert gs["batch"][BF["n_nan"]] >= 3


@pytest.mark.parametrize("C,tau,est", [(2.0, math.nan, 1), (1.2, 0.01, 3), (0.8, math.nan, 3),
                                       (50.0, 0.05, 1)])
def test_caps_thresholds_estimators(C, tau, est):
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 700, size=40)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 5)
    scale = np.repeat(rng.choice([0.01, 0.2, 0.6], size=40), lens)
    l_ro = (l_tr + rng.normal(0, 1, N) * scale).astype(np.float32)
    mask = np.ones(N, np.uint8)
    gs, o = run_both(l_tr, l_ro, mask, off, C=C, tau=tau, est=est)
    check_all(gs, o, C=C, tau=tau, est=est)


def test_cap_one_with_exact_ties():
    """C = 1: a token with delta = 0 exactly has r = C and is not clipped (r > C
    is strict), any delta above 0 is; the default threshold (C - 1) - ln C is 0,
    so only sequences of exact ties stay unflagged.  Non-finite tokens mixed in."""
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 300, size=30)
    lens[:3] = (1, 64, 257)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 8)
    l_ro = (l_tr + rng.normal(0, 0.05, N)).astype(np.float32)
    tie = rng.random(N) < 0.3
    tie[off[0]:off[3]] = True                       # three sequences of exact ties only
    l_ro[tie] = l_tr[tie]
    mask = (rng.random(N) < 0.9).astype(np.uint8)
    l_tr[off[5]] = np.nan
    mask[off[5]] = 1
    gs, o = run_both(l_tr, l_ro, mask, off, C=1.0)
    check_all(gs, o, C=1.0)
    assert np.all(gs["seq_flags"][:3] == 0) and gs["batch"][BF["n_clip"]] > 0


def test_long_sequence_and_without_weights():
    """One 300k-token sequence (many compensated folds) next to short ones."""
    N = 300_000 + 77
    off = np.array([0, 40, 300_040, N], np.int32)
    l_tr = wl.draw_train_logprobs(N, 9)
    l_ro = (l_tr + np.random.default_rng(9).normal(0, 0.02, N)).astype(np.float32)
    mask = np.ones(N, np.uint8)
    gs, o = run_both(l_tr, l_ro, mask, off, weights=False)
    check_all(gs, o, weights=False)
    assert gs["token_weight"] is None


def test_no_sequences_and_no_tokens():
    z = np.zeros(0, np.float32)
    gs, o = run_both(z, z, np.zeros(0, np.uint8), np.array([0], np.int32))
    assert np.all(gs["batch"] == 0) and gs["seq_stats"].shape == (0, 12)
    gs, o = run_both(z, z, np.zeros(0, np.uint8), np.array([0, 0, 0], np.int32))
    assert np.all(gs["seq_stats"] == 0) and np.all(gs["batch"] == 0)


def test_table1_worked_example(golden_dir):
    """Table 1 of the VeXact summary through the GPU path (one 8-token sequence)."""
    import os
    rows = [l.split() for l in open(os.path.join(golden_dir, "table1_qwen3_8b.txt"))
            if l.strip() and not l.startswith("#")]
    l_ro = np.array([float(r[1]) for r in rows], np.float32)
    l_tr = np.array([float(r[2]) for r in rows], np.float32)
    gs, o = run_both(l_tr, l_ro, np.ones(8, np.uint8), np.array([0, 8], np.int32))
    check_all(gs, o)
    assert gs["seq_stats"][0, SF["max_abs_delta"]] == pytest.approx(0.133, abs=1e-6)


def test_sequence_records_do_not_depend_on_packing():
    """A sequence's record is bit-identical wherever it sits in the pack and
    whatever else is in the batch (the reduction order follows the token's
    index inside its own sequence)."""
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 3000, size=25)
    lens[[3, 11]] = [8193, 20000]            # two sequences take the whole-CTA path
    seqs = []
    for i, L in enumerate(lens):
        lt = wl.draw_train_logprobs(int(L), 100 + i)
        lr = (lt + rng.normal(0, 0.05, L)).astype(np.float32)
        m = (rng.random(L) < 0.7).astype(np.uint8)
        seqs.append((lt, lr, m))

    def pack(order, extra):
        parts = [seqs[i] for i in order] + extra
        off = np.concatenate([[0], np.cumsum([len(p[0]) for p in parts])]).astype(np.int32)
        cat = [np.concatenate([p[k] for p in parts]) for k in range(3)]
        g = tim.mismatch_stats(_dev(cat[0]), _dev(cat[1]), _dev(cat[2]), _dev(off), token_weight=True)
        tim.check()
        return g["seq_stats"].cpu().numpy(), g["token_weight"].cpu().numpy(), off

    base, wb, offb = pack(list(range(25)), [])
    perm = list(rng.permutation(25))
    filler = (wl.draw_train_logprobs(333, 1), wl.draw_train_logprobs(333, 2), np.ones(333, np.uint8))
    other, wo, offo = pack(perm, [filler])
    for j, i in enumerate(perm):
        assert np.array_equal(base[i].view(np.uint32), other[j].view(np.uint32)), i
        assert np.array_equal(wb[offb[i]:offb[i + 1]], wo[offo[j]:offo[j + 1]])


def test_repeat_runs_are_bitwise_identical():
    cfg, l_tr, l_ro, mask, off = _config_inputs("llama3_8b", seed=3)
    args = [_dev(x) for x in (l_tr, l_ro, mask, off)]
    r1 = tim.mismatch_stats(*args, token_weight=True)
    r2 = tim.mismatch_stats(*args, token_weight=True)
    tim.check()
    for k in ("seq_stats", "seq_flags", "batch", "token_weight"):
        assert torch.equal(r1[k], r2[k]), k


def test_bad_offsets_are_reported_not_trapped():
    l = _dev(np.zeros(10, np.float32))
    m = _dev(np.ones(10, np.uint8))
    for off in ([0, 6, 4, 10], [0, 4, 9], [1, 4, 10], [0, 4, 12]):
        g = tim.mismatch_stats(l, l, m, _dev(np.array(off, np.int32)))
        with pytest.raises(tim.TimError) as e:
            tim.check()
        assert e.value.code == tim.TIM_ERR_BAD_INPUT
        assert torch.isnan(g["batch"]).all()
    # the status word is cleared by the check: a good call afterwards is clean
    tim.mismatch_stats(l, l, m, _dev(np.array([0, 10], np.int32)))
    tim.check()


def test_many_sequences_take_the_two_level_fold():
    """5000 short sequences: more than one fold CTA (1024 sequences each), so
    the partials go through the final fold kernel."""
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 40, size=5000)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 21)
    l_ro = (l_tr + rng.normal(0, 0.05, N)).astype(np.float32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    gs, o = run_both(l_tr, l_ro, mask, off)
    check_all(gs, o)


def test_full_size_bandwidth_batch():
    """The bandwidth measurement's size: 2^27 tokens in ~116k lognormal
    sequences (median 1024, clipped to [128, 4096]), 30% masked, weights
    written, in the same launch configuration; every record against the
    oracle."""
    off, mask, _, l_tr, l_ro, _ = wl.draw_ppo_inputs(1 << 27, 22)
    gs, o = run_both(l_tr, l_ro, mask, off)
    check_all(gs, o)


def _part(l_tr, l_ro, mask, off, s0, s1):
    """Sequences s0 .. s1 - 1 of a packed batch as a batch of their own."""
    b, e = int(off[s0]), int(off[s1])
    return l_tr[b:e], l_ro[b:e], mask[b:e], (off[s0:s1 + 1] - off[s0]).astype(np.int32)


@pytest.mark.parametrize("cuts", [(0, 1, 5000), (0, 1700, 1701, 3333, 5000), (0, 2500, 2500, 5000)])
def test_batch_scored_in_parts_folds_to_the_same_bits(cuts):
    """A batch split into parts (as across data-parallel ranks; a part may be
    empty): each part's sequence records, concatenated in sequence order and
    folded by mismatch_fold, give the whole batch's record bit for bit, and
    the records themselves are the whole call's; the oracle agrees."""
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 60, size=5000)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    l_tr = wl.draw_train_logprobs(N, 31)
    l_ro = (l_tr + rng.normal(0, 0.05, N)).astype(np.float32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    whole = tim.mismatch_stats(_dev(l_tr), _dev(l_ro), _dev(mask), _dev(off), seq_records=True)
    recs = []
    for s0, s1 in zip(cuts[:-1], cuts[1:]):
        p = _part(l_tr, l_ro, mask, off, s0, s1)
        recs.append(tim.mismatch_stats(*(_dev(x) for x in p), seq_records=True)["seq_records"])
    folded = tim.mismatch_fold(torch.cat(recs, 0).contiguous())
    tim.check()
    assert torch.equal(torch.cat(recs, 0), whole["seq_records"])
    assert torch.equal(folded.view(torch.int64), whole["batch"].view(torch.int64))
    o = oracle.mismatch_stats(l_tr, l_ro, mask, off)
    assert_batch_match(folded.cpu().numpy(), o["batch"])


def test_fold_of_no_sequences_is_all_zero():
    out = tim.mismatch_fold(torch.zeros((0, tim.SEQ_RECORD_WORDS), dtype=torch.int32, device="cuda"))
    tim.check()
    assert torch.count_nonzero(out).item() == 0
