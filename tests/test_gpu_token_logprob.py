"""GPU parity of tim_token_logprob against the fp64 oracle: full outputs on
small ragged shapes, sampled rows at the pages' head shapes in the launch
configuration the benchmark times, and exact special cases."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import LOGP_ATOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16_dev(u16):
    return _dev(u16.view(np.int16)).view(torch.bfloat16)


def gpu_logprob(h, W, a):
    lp, lse = tim.token_logprob(_bf16_dev(h), _bf16_dev(W), _dev(a.astype(np.int32)))
    tim.check()
    return lp.cpu().numpy(), lse.cpu().numpy()


def assert_parity(g_lp, g_lse, o_lp, o_lse, what=""):
    ok_t = np.isfinite(o_lp)
    assert np.array_equal(np.isnan(g_lp), ~ok_t), what
    e_lp = np.max(np.abs(g_lp[ok_t] - o_lp[ok_t])) if ok_t.any() else 0.0
    e_lse = np.max(np.abs(g_lse - o_lse))
    assert e_lp <= LOGP_ATOL and e_lse <= LOGP_ATOL, (what, e_lp, e_lse)
    return e_lp, e_lse


def _rand(N, D, V, seed, w_std=0.02):
    rng = np.random.default_rng(seed)
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(w_std))
    a = rng.integers(0, V, size=N).astype(np.int32)
    return h, W, a


def test_tiny_config_full():
    cfg = wl.CONFIGS["tiny"]
    h, W = wl.draw_head(cfg)
    a = wl.draw_targets(cfg, cfg.N)
    g = gpu_logprob(h, W, a)
    o = oracle.token_logprob(h, W, a)
    e = assert_parity(*g, *o, "tiny")
    print("tiny max |dlogp| %.3g max |dlse| %.3g" % e)


@pytest.mark.parametrize("N,D,V", [
    (1, 64, 1), (7, 72, 130), (130, 256, 1000), (129, 128, 257), (300, 520, 2049),
    (64, 8, 1027), (200, 1024, 4099), (5, 4096, 3000), (257, 200, 1024),
])
def test_ragged_shapes_full(N, D, V):
    """Tails in every dimension: N not a multiple of 128, D not a multiple of
    64 (and D < 64), V not a multiple of 256 or of the 1024-id chunk."""
    h, W, a = _rand(N, D, V, N * 7 + D * 3 + V, w_std=0.2 / math.sqrt(D / 64))
    g = gpu_logprob(h, W, a)
    o = oracle.token_logprob(h, W, a)
    assert_parity(*g, *o, (N, D, V))


def test_uniform_when_weight_is_zero():
    N, D, V = 300, 256, 5000
    h, _, a = _rand(N, D, V, 1)
    W = np.zeros((V, D), np.uint16)
    lp, lse = gpu_logprob(h, W, a)
    assert np.max(np.abs(lp + math.log(V))) <= 1e-6
    assert np.max(np.abs(lse - math.log(V))) <= 1e-6


def test_probabilities_sum_to_one_and_rows_do_not_interact():
    """One row replicated V times with targets 0..V-1: sum of exp(logp) is 1,
    and every copy's lse has the same bits (a row's result does not depend on
    where it sits in the batch)."""
    V, D = 1500, 512
    h, W, _ = _rand(1, D, V, 2, w_std=0.1)
    lp, lse = gpu_logprob(np.repeat(h, V, axis=0), W, np.arange(V, dtype=np.int32))
    assert abs(math.fsum(np.exp(lp.astype(np.float64))) - 1.0) < 1e-4
    assert np.all(lse.view(np.uint32) == lse.view(np.uint32)[0])


def test_out_of_range_targets_give_nan():
    N, D, V = 9, 128, 700
    h, W, a = _rand(N, D, V, 3)
    a[[0, 3, 8]] = [-100, V, np.iinfo(np.int32).min]
    lp, lse = gpu_logprob(h, W, a)
    o_lp, o_lse = oracle.token_logprob(h, W, a)
    assert_parity(lp, lse, o_lp, o_lse)
    assert np.isnan(lp[[0, 3, 8]]).all() and np.isfinite(lse).all()


def test_repeat_runs_are_bitwise_identical():
    h, W, a = _rand(1000, 512, 9000, 4)
    hd, Wd, ad = _bf16_dev(h), _bf16_dev(W), _dev(a)
    r1 = tim.token_logprob(hd, Wd, ad)
    r2 = tim.token_logprob(hd, Wd, ad)
    tim.check()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])


def _rows_per_m_tile(N):
    """One row in every 128-row m-tile (so both CTAs of every pair, every h
    band and every cluster's units are compared), at an offset that walks
    through the tile's four TMEM lane quarters, plus the first and last rows."""
    mt = np.arange((N + 127) // 128)
    rows = np.minimum(mt * 128 + (mt * 37 + 5) % 128, N - 1)
    return np.unique(np.concatenate([[0, N - 1], rows])).astype(np.int64)


@pytest.mark.parametrize("name", ["qwen3_8b", "llama3_8b", "dsv3"])
def test_head_shapes_sampled_rows(name):
    """Full-size heads as the benchmark runs them; the oracle recomputes one
    row of every 128-row m-tile (64, 256 and 128 rows) on all host cores."""
    cfg = wl.CONFIGS[name]
    h, W = wl.draw_head(cfg)
    hd, Wd = _bf16_dev(h), _bf16_dev(W)
    top5 = None
    if cfg.target_mode == "top5mix":
        top5 = top5_ids(hd, Wd)
    a = wl.draw_targets(cfg, cfg.N, top5=top5)
    lp, lse = tim.token_logprob(hd, Wd, _dev(a))
    tim.check()
    lp, lse = lp.cpu().numpy(), lse.cpu().numpy()
    rows = _rows_per_m_tile(cfg.N)
    o_lp, o_lse = oracle.token_logprob(h, W, a, rows=rows)
    e = assert_parity(lp[rows], lse[rows], o_lp, o_lse, name)
    print("%s %d sampled rows: max |dlogp| %.3g max |dlse| %.3g" % (name, len(rows), *e))
    assert np.isfinite(lp).all() and np.isfinite(lse).all()


def top5_ids(hd, Wd, chunk=2048):
    """Input shaping for the DeepSeek-V3-shaped targets: the five largest
    logits of each row from a plain bf16 torch matmul (not the library)."""
    out = []
    for s in range(0, hd.shape[0], chunk):
        z = hd[s:s + chunk] @ Wd.T
        out.append(torch.topk(z.float(), 5, dim=-1).indices.int().cpu())
        del z
    return torch.cat(out).numpy()


# --------------------------------------------------------------- temperature
@pytest.mark.parametrize("tau", [0.7, 2.5])
def test_temperature_parity(tau):
    """log softmax(h W^T / tau) against the oracle (icarus, "logits processor")."""
    h, W, a = _rand(300, 512, 5000, 31, w_std=0.05)
    lp, lse = tim.token_logprob(_bf16_dev(h), _bf16_dev(W), _dev(a), temperature=tau)
    tim.check()
    o_lp, o_lse = oracle.token_logprob(h, W, a, temperature=tau)
    assert_parity(lp.cpu().numpy(), lse.cpu().numpy(), o_lp, o_lse, tau)


def test_temperature_one_and_power_of_two_are_exact():
    """tau = 1 gives the bits of the plain call; tau = 2 on W gives the bits of
    tau = 1 on W / 2 (an exact rescale of every logit)."""
    h, W, a = _rand(1000, 1024, 9000, 32)
    hd, Wd, ad = _bf16_dev(h), _bf16_dev(W), _dev(a)
    p0 = tim.token_logprob(hd, Wd, ad)
    p1 = tim.token_logprob(hd, Wd, ad, temperature=1.0)
    lp_bits = torch.empty_like(p0[0])
    rc = tim.tim_token_logprob_temperature(hd.data_ptr(), Wd.data_ptr(), ad.data_ptr(), 1000, 1024, 9000, 1.0,
                                           lp_bits.data_ptr(), p1[1].data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
    assert rc == tim.TIM_OK
    Wh = (Wd.float() * 0.5).to(torch.bfloat16)
    q2 = tim.token_logprob(hd, Wd, ad, temperature=2.0)
    q1 = tim.token_logprob(hd, Wh, ad)
    tim.check()
    assert torch.equal(p0[0], lp_bits) and torch.equal(p0[1], p1[1])
    assert torch.equal(q2[0], q1[0]) and torch.equal(q2[1], q1[1])


def test_temperature_rejects_bad_values():
    for tau in (0.0, -1.0, float("inf"), float("nan")):
        assert tim.tim_token_logprob_temperature(16, 16, 16, 4, 64, 10, tau, 16, 16, None) == tim.TIM_ERR_INVALID_ARG
