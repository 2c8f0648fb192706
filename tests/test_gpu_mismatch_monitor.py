"""GPU parity of tim_mismatch_monitor against the fp64 oracle: exact order
statistics (the same tokens a sort picks), counts and rejection flags, on
ragged sizes, ties, empty batches and the full-size batch the benchmark
times; repeat determinism."""
import numpy as np
import pytest

import oracle
import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402

MF = {n: i for i, n in enumerate(oracle.MONITOR_FIELDS)}
RATIOS = ("ratio_q01", "ratio_q50", "ratio_q99")


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def gpu_monitor(lt, lr, mask, tau):
    out = tim.mismatch_monitor(_dev(lt), _dev(lr), _dev(mask), tau)
    tim.check()
    return out["batch"].cpu().numpy(), out["token_reject"].cpu().numpy()


def assert_monitor_match(g, g_rej, o, what=""):
    ob, orej = o["batch"], o["reject"]
    for f in ("n_used", "n_extreme"):
        assert g[MF[f]] == ob[MF[f]], (what, f, g[MF[f]], ob[MF[f]])
    assert np.array_equal(g_rej, orej), what
    if ob[MF["n_used"]] == 0:
        assert all(np.isnan(g[MF[f]]) for f in ("p95_abs_delta",) + RATIOS), what
        return
    # |delta| order statistics are fp32 values on both sides and the
    # interpolation is the same fp64 expression: equal to rounding
    np.testing.assert_allclose(g[MF["p95_abs_delta"]], ob[MF["p95_abs_delta"]], rtol=1e-15, err_msg=what)
    for f in RATIOS:   # e^delta: fp32 expf on the device
        np.testing.assert_allclose(g[MF[f]], ob[MF[f]], rtol=1e-6, err_msg=what + " " + f)
    np.testing.assert_allclose(g[MF["frac_extreme"]], ob[MF["frac_extreme"]], rtol=1e-15, err_msg=what)


def _batch(N, seed, spread=0.05, tau=0.1):
    rng = np.random.default_rng(seed)
    lt = wl.draw_train_logprobs(N, seed)
    lr = (lt + rng.normal(0, spread, N) * (rng.random(N) < 0.9)).astype(np.float32)   # 10% exact ties at 0
    mask = (rng.random(N) < 0.75).astype(np.uint8)
    if N > 8:
        lt[3] = np.nan
        lr[5] = np.inf
        mask[[3, 5]] = 1
    return lt, lr, mask


@pytest.mark.parametrize("N", [1, 2, 3, 5, 31, 1000, 4099, 100003, 1 << 20])
def test_ragged_sizes(N):
    """Sizes that are not multiples of the 4-token groups, below one warp,
    and across many CTAs; a tenth of the tokens tie at delta = 0."""
    lt, lr, mask = _batch(N, N)
    tau = float(np.float32(0.08))
    g, rej = gpu_monitor(lt, lr, mask, tau)
    assert_monitor_match(g, rej, oracle.mismatch_monitor(lt, lr, mask, tau), "N=%d" % N)


def test_ties_signed_zero_and_empty():
    N = 5000
    lt = wl.draw_train_logprobs(N, 3)
    g, _ = gpu_monitor(lt, lt.copy(), np.ones(N, np.uint8), 0.0)           # every delta = +0
    assert g[MF["ratio_q01"]] == g[MF["ratio_q99"]] == 1.0 and g[MF["p95_abs_delta"]] == 0.0
    assert g[MF["n_extreme"]] == 0                                          # |delta| = tau = 0: kept
    lz = np.zeros(8, np.float32)
    lz[::2] = -0.0                                                          # -0 - (+0) = -0
    g2, _ = gpu_monitor(lz, np.zeros(8, np.float32), np.ones(8, np.uint8), 0.1)
    assert g2[MF["ratio_q50"]] == 1.0
    g3, rej3 = gpu_monitor(lt, lt, np.zeros(N, np.uint8), 0.1)             # nothing used
    assert g3[MF["n_used"]] == 0 and np.isnan(g3[MF["ratio_q50"]]) and not rej3.any()
    e = tim.mismatch_monitor(torch.zeros(0, device="cuda"), torch.zeros(0, device="cuda"),
                             torch.zeros(0, dtype=torch.uint8, device="cuda"), 0.1)
    tim.check()
    assert e["batch"][MF["n_used"]].item() == 0


def test_heavy_tail_and_thresholds():
    """Outliers of +-1 nat on 0.5% of tokens (the Llama-shaped rollout): the
    p99 / p01 ratios sit in the tail; several thresholds."""
    cfg = wl.CONFIGS["llama3_8b"]
    lt = wl.draw_train_logprobs(cfg.N, 4)
    lr = wl.draw_rollout(cfg, lt, seed=4)
    off = wl.draw_segments(cfg, seed=4)
    mask = wl.draw_mask(cfg, off, seed=4)
    for tau in (0.0, 0.01, 0.05, 0.5, 2.0):
        t = float(np.float32(tau))
        g, rej = gpu_monitor(lt, lr, mask, t)
        assert_monitor_match(g, rej, oracle.mismatch_monitor(lt, lr, mask, t), "tau=%g" % tau)


def test_repeat_runs_are_bitwise_identical():
    lt, lr, mask = _batch(1 << 20, 7)
    a = tim.mismatch_monitor(_dev(lt), _dev(lr), _dev(mask), 0.1)
    b = tim.mismatch_monitor(_dev(lt), _dev(lr), _dev(mask), 0.1)
    tim.check()
    assert torch.equal(a["batch"], b["batch"]) and torch.equal(a["token_reject"], b["token_reject"])


def test_full_size_batch():
    """2^27 tokens with the benchmark's recipe (30% masked, delta ~ N(0, 0.02^2)
    on -Gamma(0.6, 3) logprobs), in the launch configuration it times."""
    N = 1 << 27
    off, mask, _, lo, lr, _ = wl.draw_ppo_inputs(N, 6)
    tau = float(np.float32(0.05))
    g, rej = gpu_monitor(lo, lr, mask, tau)
    assert_monitor_match(g, rej, oracle.mismatch_monitor(lo, lr, mask, tau), "2^27")


def sampled_tokens(N, runs=1024, run=1024, region=1 << 18):
    """The tokens the monitor's sample reads when N exceeds runs x run: run r
    starts at g (N - region) / 63 rounded down to a multiple of 4, plus
    j region / 16 (g = r / 16, j = r mod 16)."""
    s = np.zeros(N, bool)
    for r in range(runs):
        s0 = ((r >> 4) * (N - region) // 63 & ~3) + (r & 15) * (region // 16)
        s[s0:s0 + run] = True
    return s


def test_sample_that_misses_the_bulk_and_mass_ties():
    """Batches larger than the 2^20-token sample where the sample misleads:
    the sampled runs (half the tokens at N = 2^21) hold delta = 0 and the rest
    delta = 1, so the quantiles lie outside the sample's bounds; and a batch
    of identical deltas, so the collected list overflows.  Both take the
    selection over all tokens (three radix passes with grid barriers) and stay
    exact."""
    N = 1 << 21
    rng = np.random.default_rng(9)
    lr = wl.draw_train_logprobs(N, 9)
    lt = (lr + np.where(sampled_tokens(N), np.float32(0.0), np.float32(1.0))).astype(np.float32)
    mask = (rng.random(N) < 0.9).astype(np.uint8)
    tau = float(np.float32(0.5))
    g, rej = gpu_monitor(lt, lr, mask, tau)
    assert_monitor_match(g, rej, oracle.mismatch_monitor(lt, lr, mask, tau), "misleading sample")
    same = lr.copy()
    g2, rej2 = gpu_monitor(same, lr, np.ones(N, np.uint8), tau)
    assert_monitor_match(g2, rej2, oracle.mismatch_monitor(same, lr, np.ones(N, np.uint8), tau), "all ties")


def test_signed_zeros_and_subnormals_at_the_ranks():
    """Half the deltas are zeros of either sign (-0 - +0 = -0), most of the rest
    subnormals of either sign, 3% normal: the median sits where -0, +0 and the
    smallest subnormals meet and p95 |delta| among the subnormals, in a batch
    larger than the sample so that the collected lists are used."""
    N = 1 << 21
    rng = np.random.default_rng(11)
    u = rng.random(N)
    tiny = (rng.integers(1, 1000, N) * np.float32(2.0 ** -149)).astype(np.float32)
    sign = np.where(rng.random(N) < 0.5, np.float32(-1.0), np.float32(1.0))
    lt = np.where(u < 0.5, np.float32(0.0), np.where(u < 0.97, sign * tiny,
                  sign * rng.uniform(0.005, 0.05, N).astype(np.float32))).astype(np.float32)
    lt[(u < 0.5) & (sign < 0)] = -0.0
    lr = np.zeros(N, np.float32)
    mask = (rng.random(N) < 0.9).astype(np.uint8)
    assert np.signbit(lt[u < 0.5]).any() and (lt[(u >= 0.5) & (u < 0.97)] != 0).all()
    for tau in (0.0, float(np.float32(2.0 ** -140))):
        g, rej = gpu_monitor(lt, lr, mask, tau)
        assert_monitor_match(g, rej, oracle.mismatch_monitor(lt, lr, mask, tau), "zeros tau=%g" % tau)


def test_just_above_the_sample_with_a_ragged_tail():
    """N just above the 2^20 tokens the sample reads, not a multiple of 4 or of
    the full pass's chunk: the sample's 64 regions overlap (some tokens are
    sampled twice) and the last chunk is read from global memory; the
    collected lists are used and the result stays exact."""
    N = (1 << 20) + 12345
    off, mask, _, lo, lr, _ = wl.draw_ppo_inputs(N, 21)
    tau = float(np.float32(0.03))
    g, rej = gpu_monitor(lo, lr, mask, tau)
    assert_monitor_match(g, rej, oracle.mismatch_monitor(lo, lr, mask, tau), "2^20 + 12345")


def test_sequences_that_differ_in_their_mismatch():
    """Each sequence has its own mismatch scale and shift (lognormal scales
    spread by a factor e^1.5): the sample's runs (mostly one sequence each)
    are then the independent units and its quantile estimates far noisier
    than their token count says, so a bound misses and the selection runs
    over all tokens; the result stays exact."""
    rng = np.random.default_rng(41)
    lens = rng.integers(256, 2048, size=4096)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = int(off[-1])
    seq = np.repeat(np.arange(len(lens)), lens)
    scale = (0.02 * np.exp(1.5 * rng.standard_normal(len(lens)))).astype(np.float32)[seq]
    shift = (0.02 * rng.standard_normal(len(lens))).astype(np.float32)[seq]
    lr = wl.draw_train_logprobs(N, 41)
    lt = (lr + shift + scale * rng.standard_normal(N).astype(np.float32)).astype(np.float32)
    mask = (rng.random(N) < 0.7).astype(np.uint8)
    tau = float(np.float32(0.05))
    g, rej = gpu_monitor(lt, lr, mask, tau)
    assert_monitor_match(g, rej, oracle.mismatch_monitor(lt, lr, mask, tau), "per-sequence mismatch")
