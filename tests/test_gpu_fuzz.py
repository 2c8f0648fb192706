"""Seeded random shapes and layouts for every entry point, each against the
oracle with the tolerances of its own parity tests: sizes that do not divide
any tile, chunk, warp or group size, empty and one-token sequences, extreme
masks."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import LOGP_ATOL, assert_batch_match, assert_ppo_match, assert_seq_stats_match

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16_dev(u16):
    return _dev(u16.view(np.int16)).view(torch.bfloat16)


def _segments(rng, N):
    lens, tot = [], 0
    while tot < N:
        L = int(min(N - tot, rng.choice([0, 1, 2, 31, 33, 200, 1000, 5000, 9000])))
        lens.append(L)
        tot += L
    if rng.random() < 0.5:
        lens.insert(int(rng.integers(0, len(lens) + 1)), 0)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@pytest.mark.parametrize("case", range(12))
def test_token_logprob_random_shapes(case):
    rng = np.random.default_rng(1000 + case)
    N = int(rng.integers(1, 700))
    D = int(rng.integers(1, 160)) * 8
    V = int(rng.integers(1, 5000))
    tau = float(np.float32(rng.choice([1.0, 0.5, 1.7])))
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.3 / math.sqrt(D / 8)))
    a = rng.integers(-2, V + 2, size=N).astype(np.int32)
    lp, lse = tim.token_logprob(_bf16_dev(h), _bf16_dev(W), _dev(a), temperature=tau)
    tim.check()
    o_lp, o_lse = oracle.token_logprob(h, W, a, temperature=tau)
    lp, lse = lp.cpu().numpy(), lse.cpu().numpy()
    ok = np.isfinite(o_lp)
    assert np.array_equal(np.isnan(lp), ~ok), (N, D, V)
    assert np.max(np.abs(lse - o_lse)) <= LOGP_ATOL, (N, D, V)
    if ok.any():
        assert np.max(np.abs(lp[ok] - o_lp[ok])) <= LOGP_ATOL, (N, D, V)


@pytest.mark.parametrize("case", range(10))
def test_mismatch_ppo_monitor_random_layouts(case):
    rng = np.random.default_rng(2000 + case)
    N = int(rng.integers(1, 40000))
    off = _segments(rng, N)
    lt = wl.draw_train_logprobs(N, 2000 + case)
    lr = (lt + rng.normal(0, rng.choice([1e-4, 0.02, 0.5]), N)).astype(np.float32)
    mask = (rng.random(N) < rng.choice([0.0, 0.3, 1.0, 1.0])).astype(np.uint8)
    bad = rng.random(N) < 0.002
    lt[bad] = np.nan
    C = float(np.float32(rng.choice([1.0, 2.0, 5.0])))

    g = tim.mismatch_stats(_dev(lt), _dev(lr), _dev(mask), _dev(off), C=C, token_weight=True)
    tim.check()
    o = oracle.mismatch_stats(lt, lr, mask, off, C=C)
    assert_seq_stats_match(g["seq_stats"].cpu().numpy(), o["seq_stats"])
    assert_batch_match(g["batch"].cpu().numpy(), o["batch"])

    l_th = wl.draw_policy_update(lt, 0.15, 2000 + case)
    adv = wl.draw_advantages(off, 2000 + case)
    pp = tim.tis_ppo(_dev(l_th), _dev(lt), _dev(lr), _dev(adv), _dev(mask), _dev(off), C=C)
    tim.check()
    op = oracle.tis_ppo(l_th, lt, lr, adv, mask, off, C=C)
    assert_ppo_match({k: (None if v is None else v.cpu().numpy()) for k, v in pp.items()}, op, off)

    tau = float(np.float32(rng.choice([0.0, 0.01, 0.3])))
    mon = tim.mismatch_monitor(_dev(lt), _dev(lr), _dev(mask), tau)
    tim.check()
    om = oracle.mismatch_monitor(lt, lr, mask, tau)
    gm = mon["batch"].cpu().numpy()
    assert gm[0] == om["batch"][0] and gm[5] == om["batch"][5]
    assert np.array_equal(mon["token_reject"].cpu().numpy(), om["reject"])
    if om["batch"][0] > 0:
        np.testing.assert_allclose(gm[1:5], om["batch"][1:5], rtol=1e-6)
    else:
        assert np.isnan(gm[1:5]).all()
