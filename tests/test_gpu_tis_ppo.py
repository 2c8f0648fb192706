"""GPU parity of tim_tis_ppo (the TIS-weighted PPO clipped surrogate) against
the fp64 oracle: every output on ragged packed batches with edge cases, the
full-size batch the benchmark times, packing invariance and determinism."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import PF, assert_ppo_match

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def gpu_ppo(lt, lo, lr, A, mask, off, eps_low=0.2, eps_high=0.2, C=2.0, token_outputs=True):
    out = tim.tis_ppo(_dev(lt), _dev(lo), _dev(lr), _dev(A), _dev(mask), _dev(off.astype(np.int32)),
                      eps_low=eps_low, eps_high=eps_high, C=C, token_outputs=token_outputs)
    tim.check()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}


def oracle_ppo(lt, lo, lr, A, mask, off, eps_low=0.2, eps_high=0.2, C=2.0):
    # the device receives fp32 parameters: the oracle gets the same values
    f = lambda x: float(np.float32(x))   # noqa: E731
    return oracle.tis_ppo(lt, lo, lr, A, mask, off, eps_low=f(eps_low), eps_high=f(eps_high), C=f(C))


def ragged_batch(lens, seed, update_std=0.15):
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(off[-1])
    rng = np.random.default_rng(seed)
    lo = wl.draw_train_logprobs(N, seed)
    lr = (lo + rng.normal(0, 0.05, N)).astype(np.float32)
    lr[rng.random(N) < 0.01] -= np.float32(2.0)           # rollout outliers past the TIS cap
    lt = wl.draw_policy_update(lo, update_std, seed)
    A = wl.draw_advantages(off, seed)
    A[rng.random(N) < 0.05] = rng.standard_normal() * 3   # some per-token advantages
    mask = (rng.random(N) >= 0.2).astype(np.uint8)
    return off, mask, lt, lo, lr, A


LENS = [0, 1, 31, 33, 64, 255, 256, 257, 1000, 0, 8192, 8193, 20000, 5, 300]


@pytest.mark.parametrize("eps_low,eps_high,C", [(0.2, 0.2, 2.0), (0.2, 0.28, 1.5), (0.0, 0.0, 1.0),
                                                (0.9, 5.0, 10.0)])
def test_ragged_full(eps_low, eps_high, C):
    """Every output, on sequences of every length class: empty, shorter than a
    warp, across 256-token steps, exactly at and past the one-warp limit
    (8192), and long ones reduced by a whole CTA."""
    off, mask, lt, lo, lr, A = ragged_batch(LENS, 11)
    g = gpu_ppo(lt, lo, lr, A, mask, off, eps_low, eps_high, C)
    o = oracle_ppo(lt, lo, lr, A, mask, off, eps_low, eps_high, C)
    assert_ppo_match(g, o, off, "eps %g/%g C %g" % (eps_low, eps_high, C))
    assert o["batch"][PF["n_ppo_clipped"]] > 0 or eps_high > 1


def test_exact_ties_at_zero_eps_and_unit_cap():
    """eps = 0 and C = 1: tokens whose log-ratios are exactly 0 sit on the clip
    bounds and on the cap; they keep their gradient and are not counted as
    clipped (both decisions are strict), like the oracle."""
    off, mask, lt, lo, lr, A = ragged_batch(LENS, 23)
    rng = np.random.default_rng(23)
    tie = rng.random(lt.size) < 0.3
    lt[tie] = lo[tie]
    tie_c = rng.random(lt.size) < 0.3
    lr[tie_c] = lo[tie_c]
    g = gpu_ppo(lt, lo, lr, A, mask, off, 0.0, 0.0, 1.0)
    o = oracle_ppo(lt, lo, lr, A, mask, off, 0.0, 0.0, 1.0)
    assert_ppo_match(g, o, off, "ties at eps 0, C 1")
    used_tie = tie & (mask != 0) & (A != 0)
    assert np.all(g["token_grad"][used_tie] != 0)

def test_nonfinite_zero_advantage_and_extremes():
    """NaN / inf inputs are not used (loss and gradient 0); A = 0 gives 0 even
    where r overflows fp32; large log-ratios stay finite where the oracle's are."""
    off, mask, lt, lo, lr, A = ragged_batch([700, 900, 64], 12)
    lt[[3, 10]] = [np.nan, np.inf]
    lr[[20, 21]] = [-np.inf, np.nan]
    A[[30, 31]] = [np.nan, np.inf]
    lo[40] = np.nan
    mask[[3, 10, 20, 21, 30, 31, 40]] = 1
    A[[50, 51, 52]] = 0.0
    lt[[50, 51]] = lo[[50, 51]] + np.float32(100.0)          # r = e^100: fp32 overflow, times A = 0
    lt[[60, 61]] = lo[[60, 61]] + np.float32(8.0)            # far past the clip range
    A[60], A[61] = 1.0, -1.0
    mask[[50, 51, 60, 61]] = 1
    g = gpu_ppo(lt, lo, lr, A, mask, off)
    o = oracle_ppo(lt, lo, lr, A, mask, off)
    assert_ppo_match(g, o, off, "nonfinite")
    bad = [3, 10, 20, 21, 30, 31, 40]
    assert np.all(g["token_loss"][bad] == 0) and np.all(g["token_grad"][bad] == 0)
    assert np.all(g["token_loss"][[50, 51, 52]] == 0)
    assert g["token_grad"][60] == 0 and g["token_grad"][61] != 0


def test_token_outputs_are_optional():
    off, mask, lt, lo, lr, A = ragged_batch(LENS, 13)
    g1 = gpu_ppo(lt, lo, lr, A, mask, off)
    g0 = gpu_ppo(lt, lo, lr, A, mask, off, token_outputs=False)
    assert g0["token_loss"] is None and g0["token_grad"] is None
    assert np.array_equal(g0["seq_loss"].view(np.uint32), g1["seq_loss"].view(np.uint32))
    assert np.array_equal(g0["batch"].view(np.uint64), g1["batch"].view(np.uint64))


def test_packing_invariance_and_repeat_determinism():
    """A sequence's mean has the same bits wherever it is packed and whatever
    its neighbours are; repeated calls give identical bits everywhere."""
    off, mask, lt, lo, lr, A = ragged_batch([1000, 9000, 77], 14)
    g = gpu_ppo(lt, lo, lr, A, mask, off)
    g2 = gpu_ppo(lt, lo, lr, A, mask, off)
    for k in ("token_loss", "token_grad", "seq_loss", "batch"):
        assert np.array_equal(g[k].view(np.uint8), g2[k].view(np.uint8)), k
    # the same three sequences behind other material, in another order
    o2, m2, t2, l2, r2, a2 = ragged_batch([333, 5000], 15)
    def seg(x, s):
        return x[off[s]:off[s + 1]]
    parts = [(t2[:333], l2[:333], r2[:333], a2[:333], m2[:333])]
    order = [2, 1, 0]
    for s in order:
        parts.append((seg(lt, s), seg(lo, s), seg(lr, s), seg(A, s), seg(mask, s)))
    cat = [np.concatenate([p[i] for p in parts]) for i in range(5)]
    lens = [333] + [int(off[s + 1] - off[s]) for s in order]
    off_b = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    gb = gpu_ppo(cat[0], cat[1], cat[2], cat[3], cat[4], off_b)
    for j, s in enumerate(order):
        assert gb["seq_loss"][j + 1].view(np.uint32) == g["seq_loss"][s].view(np.uint32), s


def test_bad_offsets_and_empty_batch():
    off, mask, lt, lo, lr, A = ragged_batch([100, 200, 300], 16)
    bad = off.copy()
    bad[1], bad[2] = 250, 120      # decreasing
    with pytest.raises(tim.TimError) as e:
        gpu_ppo(lt, lo, lr, A, mask, bad)
    assert e.value.code == tim.TIM_ERR_BAD_INPUT
    z = np.zeros(0, np.float32)
    g = gpu_ppo(z, z, z, z, np.zeros(0, np.uint8), np.zeros(1, np.int32))
    assert np.all(g["batch"] == 0)


@pytest.mark.parametrize("tokens", [1 << 27])
def test_full_size_batch(tokens):
    """The benchmark's batch (2^27 tokens, lognormal sequences, 30% masked),
    in the launch configuration it times: every sequence mean and the batch
    record against the oracle over all tokens, token outputs on a sample."""
    off, mask, lt, lo, lr, A = wl.draw_ppo_inputs(tokens, 5)
    g = gpu_ppo(lt, lo, lr, A, mask, off)
    o = oracle_ppo(lt, lo, lr, A, mask, off)
    rng = np.random.default_rng(5)
    pick = np.unique(np.concatenate([rng.integers(0, tokens, 1 << 20), [0, tokens - 1]]))
    sub = {"token_loss": g["token_loss"][pick], "token_grad": g["token_grad"][pick]}
    o_sub = {"token_loss": o["token_loss"][pick], "token_grad": o["token_grad"][pick]}
    from gpu_util import _close
    _close(sub["token_loss"], o_sub["token_loss"], np.abs(o_sub["token_loss"]), "sampled token_loss")
    assert np.array_equal(sub["token_grad"] == 0, o_sub["token_grad"] == 0)
    _close(sub["token_grad"], o_sub["token_grad"], np.abs(o_sub["token_grad"]), "sampled token_grad")
    g_rest = {"token_loss": None, "token_grad": None, "seq_loss": g["seq_loss"], "batch": g["batch"]}
    assert_ppo_match(g_rest, o, off, "2^27")


def test_four_byte_aligned_views():
    """The surrogate needs 4-byte alignment only: inputs and outputs as views
    that start one element into their buffers give the same bits as aligned
    ones."""
    off, mask, lt, lo, lr, A = ragged_batch([300, 9000, 41], 17)
    N = int(off[-1])
    def shifted(x, dtype):
        buf = torch.zeros(N + 1, dtype=dtype, device="cuda")
        buf[1:] = _dev(x)
        return buf[1:]
    args = [shifted(lt, torch.float32), shifted(lo, torch.float32), shifted(lr, torch.float32),
            shifted(A, torch.float32), shifted(mask, torch.uint8), _dev(off)]
    out = {"token_loss": torch.empty(N + 1, device="cuda")[1:], "token_grad": torch.empty(N + 1, device="cuda")[1:],
           "seq_loss": torch.empty(len(off), device="cuda")[1:], "batch": torch.empty(9, dtype=torch.float64, device="cuda")}
    tim.tis_ppo(*args, out=out)
    tim.check()
    g = gpu_ppo(lt, lo, lr, A, mask, off)
    for k in ("token_loss", "token_grad", "seq_loss", "batch"):
        assert np.array_equal(out[k].cpu().numpy().view(np.uint8), g[k].view(np.uint8)), k
