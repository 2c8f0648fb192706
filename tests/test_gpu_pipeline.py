"""The hot path chained on the GPU, against the same chain in the oracle: the
trainer's token logprobs (fused head), the mismatch statistics against the
rollout engine's logprobs, the TIS-weighted PPO surrogate and its gradient,
and that gradient taken back through the head (dh, dW).

Each stage reads the previous stage's GPU output, the oracle chain its own.
The old-policy logprobs are built from the oracle's l_theta so that no token
lies within 1e-3 of a PPO clip boundary or of the TIS cap: the two chains then
take the same clip decisions, and the tolerances are those of the single
stages (2e-3 on logprobs, 1e-5 relative on statistics and per-token
surrogate terms, the bf16-dz scale rule on dh and dW)."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import LOGP_ATOL, assert_batch_match

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16_dev(u16):
    return _dev(u16.view(np.int16)).view(torch.bfloat16)


def _away(x, edges, gap, rng):
    """Moves each value of x that is within `gap` of an edge to `2 gap` past it."""
    x = x.copy()
    for e in edges:
        near = np.abs(x - e) < gap
        x[near] = e + np.where(rng.random(near.sum()) < 0.5, -2 * gap, 2 * gap)
    return x


def test_forward_stats_surrogate_backward_chain():
    rng = np.random.default_rng(100)
    N, D, V = 512, 512, 6000
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.05))
    a = rng.integers(0, V, N).astype(np.int32)
    lens = [100, 1, 250, 0, 161]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    adv = wl.draw_advantages(off, 100)
    eps_low, eps_high, C = float(np.float32(0.2)), float(np.float32(0.28)), 2.0

    # oracle chain
    o_lp, o_lse = oracle.token_logprob(h, W, a)
    l_theta_o = o_lp.astype(np.float32)
    dt = _away(rng.normal(0, 0.2, N), [math.log1p(eps_high), math.log1p(-eps_low)], 1e-3, rng)
    l_old = (l_theta_o.astype(np.float64) - dt).astype(np.float32)
    dc = _away(rng.normal(0, 0.3, N), [math.log(C)], 1e-3, rng)
    l_ro = (l_old.astype(np.float64) - dc).astype(np.float32)
    o_stats = oracle.mismatch_stats(l_theta_o, l_ro, mask, off, C=C)
    o_ppo = oracle.tis_ppo(l_theta_o, l_old, l_ro, adv, mask, off, eps_low=eps_low, eps_high=eps_high, C=C)
    n_used = o_ppo["batch"][oracle.PPO_FIELDS.index("n_used")]
    g_o = (o_ppo["token_grad"] / n_used).astype(np.float32)   # gradient of the token-mean loss
    o_bw = oracle.token_logprob_backward(h, W, a, g_o, want_dz=True)

    # GPU chain
    hd, Wd, ad = _bf16_dev(h), _bf16_dev(W), _dev(a)
    lp, lse = tim.token_logprob(hd, Wd, ad)
    st = tim.mismatch_stats(lp, _dev(l_ro), _dev(mask), _dev(off), C=C)
    pp = tim.tis_ppo(lp, _dev(l_old), _dev(l_ro), _dev(adv), _dev(mask), _dev(off), eps_low=eps_low,
                     eps_high=eps_high, C=C)
    n_used_g = pp["batch"][oracle.PPO_FIELDS.index("n_used")]
    grad = (pp["token_grad"] / n_used_g).float()
    dh, dW = tim.token_logprob_backward(hd, Wd, ad, grad, lse)
    tim.check()

    assert np.max(np.abs(lp.cpu().numpy() - o_lp)) <= LOGP_ATOL
    assert_batch_match(st["batch"].cpu().numpy(), o_stats["batch"])
    g_grad = pp["token_grad"].cpu().numpy()
    assert np.array_equal(g_grad == 0, o_ppo["token_grad"] == 0)   # the same clip decisions
    np.testing.assert_allclose(g_grad, o_ppo["token_grad"], rtol=2e-5, atol=1e-7)
    assert n_used_g.item() == n_used
    hf = wl.bf16_to_f32(h).astype(np.float64)
    Wf = wl.bf16_to_f32(W).astype(np.float64)
    dz2 = o_bw["dz"] ** 2
    for g_arr, o_arr, scale, what in ((dh.cpu().numpy(), o_bw["dh"], np.sqrt(dz2 @ Wf ** 2), "dh"),
                                      (dW.cpu().numpy(), o_bw["dW"], np.sqrt(dz2.T @ hf ** 2), "dW")):
        # bf16 dz scale rule, plus the upstream gradient's own relative error (2e-5)
        bound = 2.0 ** -7 * scale + 3e-5 * np.abs(o_arr) + 1e-6 * np.max(np.abs(o_arr))
        assert np.all(np.abs(g_arr - o_arr) <= bound), what


def test_wrappers_reject_wrong_output_buffers():
    """Every torch wrapper checks the caller's output buffers (dtype, shape,
    device) before anything is launched: a buffer shorter than the outputs
    raises instead of being written past its end."""
    f32 = dict(dtype=torch.float32, device="cuda")
    N, D, V, S = 64, 64, 300, 2
    h = torch.zeros((N, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((V, D), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(N, dtype=torch.int32, device="cuda")
    l = torch.zeros(N, **f32)
    m = torch.ones(N, dtype=torch.uint8, device="cuda")
    off = torch.tensor([0, 32, N], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        tim.token_logprob(h, W, a, out_logp=torch.empty(N - 1, **f32))
    with pytest.raises(ValueError):
        tim.token_logprob(h, W, a, out_lse=torch.empty(N + 1, **f32))
    with pytest.raises(TypeError):
        tim.token_logprob(h, W, a, out_logp=torch.empty(N, dtype=torch.float64, device="cuda"))
    with pytest.raises(ValueError):
        tim.token_logprob_backward(h, W, a, l, l, dh=torch.empty((N, D - 8), **f32))
    with pytest.raises(ValueError):
        tim.token_logprob_backward(h, W, a, l, l, dW=torch.empty((V - 1, D), **f32))
    good = {"seq_stats": torch.empty((S, 12), **f32), "seq_flags": torch.empty(S, dtype=torch.int32, device="cuda"),
            "batch": torch.empty(20, dtype=torch.float64, device="cuda"), "token_weight": None}
    for key, bad in (("seq_stats", torch.empty((S - 1, 12), **f32)),
                     ("seq_flags", torch.empty(S, **f32)),
                     ("batch", torch.empty(19, dtype=torch.float64, device="cuda")),
                     ("token_weight", torch.empty(N - 4, **f32))):
        with pytest.raises((ValueError, TypeError)):
            tim.mismatch_stats(l, l, m, off, out=dict(good, **{key: bad}))
    with pytest.raises(ValueError):
        tim.mismatch_monitor(l, l, m, 0.1, out={"batch": torch.empty(6, dtype=torch.float64, device="cuda"),
                                                "token_reject": None})
    with pytest.raises(ValueError):
        tim.mismatch_monitor(l, l, m, 0.1, out={"batch": torch.empty(7, dtype=torch.float64, device="cuda"),
                                                "token_reject": torch.empty(N - 1, dtype=torch.uint8, device="cuda")})
    ppo = {"token_loss": None, "token_grad": None, "seq_loss": torch.empty(S, **f32),
           "batch": torch.empty(9, dtype=torch.float64, device="cuda")}
    with pytest.raises(ValueError):
        tim.tis_ppo(l, l, l, l, m, off, out=dict(ppo, seq_loss=torch.empty(S + 1, **f32)))
    with pytest.raises(ValueError):
        tim.tis_ppo(l, l, l, l, m, off, out=dict(ppo, token_grad=torch.empty(N // 2, **f32)))
    # the same buffers at the right sizes are accepted and computed into
    r = tim.mismatch_stats(l, l, m, off, out=good)
    tim.tis_ppo(l, l, l, l, m, off, out=ppo)
    tim.check()
    assert r["batch"][1].item() == N
