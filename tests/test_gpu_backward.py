"""GPU parity of tim_token_logprob_backward against the fp64 oracle.

Tolerance: the logit gradient dz is rounded to bf16 (relative error at most
2^-9 per element, round to nearest) before two GEMMs with fp32 accumulation,
so an element of dh = dz W carries an error of about 2^-9 / sqrt(3) times its
natural scale s_dh[t, d] = sqrt(sum_v (dz[t, v] W[v, d])^2) (likewise
s_dW[v, d] = sqrt(sum_t (dz[t, v] h[t, d])^2)).  The test allows 2^-7 times
that scale (about seven standard deviations), plus 4e-6 times
sum_v (|dz| + |g| onehot)[t, v] |W[v, d]| (resp. the same over t with |h|)
for p = 2^(z log2e / tau - lse log2e) in fp32 (about 1e-6 relative to p,
which matters where p ~ 1 and dz ~ 0), plus 1e-6 of the largest element for
the fp32 accumulation.  At the full head shape, where the
oracle's cost allows a few rows of dh only, dW is checked through the
identity <dW, W> = <dh, h> (both equal sum_t sum_v dz z) and dh on sampled
rows."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16_dev(u16):
    return _dev(u16.view(np.int16)).view(torch.bfloat16)


def _case(N, D, V, seed, w_std):
    rng = np.random.default_rng(seed)
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(w_std))
    a = rng.integers(0, V, size=N).astype(np.int32)
    g = rng.standard_normal(N).astype(np.float32)
    return h, W, a, g


def gpu_backward(h, W, a, g, tau=1.0):
    hd, Wd, ad = _bf16_dev(h), _bf16_dev(W), _dev(a)
    _, lse = tim.token_logprob(hd, Wd, ad, temperature=tau)
    dh, dW = tim.token_logprob_backward(hd, Wd, ad, _dev(g), lse, temperature=tau)
    tim.check()
    return dh.cpu().numpy(), dW.cpu().numpy()


def assert_close(gv, ov, scale, p_term, what):
    gv = np.asarray(gv, np.float64)
    bound = 2.0 ** -7 * scale + 4e-6 * p_term + 1e-6 * np.max(np.abs(ov))
    bad = np.abs(gv - ov) > bound
    assert not bad.any(), (what, int(bad.sum()), float(np.max(np.abs(gv - ov) / np.maximum(bound, 1e-300))))


def _abs_p(dz, a, g):
    """|dz| + |g| at the target: bounds |g| p elementwise."""
    ap = np.abs(dz)
    ok = (a >= 0) & (a < dz.shape[1])
    ap[np.nonzero(ok)[0], a[ok]] += np.abs(g[ok].astype(np.float64))
    return ap


def check_against_oracle(h, W, a, g, tau=1.0, what=""):
    dh, dW = gpu_backward(h, W, a, g, tau)
    o = oracle.token_logprob_backward(h, W, a, g, temperature=tau, want_dz=True)
    dz2 = o["dz"] ** 2
    hf = wl.bf16_to_f32(h).astype(np.float64)
    Wf = wl.bf16_to_f32(W).astype(np.float64)
    ap = _abs_p(o["dz"], a, g)
    assert_close(dh, o["dh"], np.sqrt(dz2 @ Wf ** 2), ap @ np.abs(Wf), what + " dh")
    assert_close(dW, o["dW"], np.sqrt(dz2.T @ hf ** 2), ap.T @ np.abs(hf), what + " dW")
    return dh, dW, o


@pytest.mark.parametrize("N,D,V", [(7, 72, 130), (130, 256, 1000), (300, 520, 2049), (200, 1024, 4099),
                                   (5, 4096, 3000), (1, 64, 1)])
def test_ragged_shapes(N, D, V):
    h, W, a, g = _case(N, D, V, N + 3 * D + V, w_std=0.3 / math.sqrt(D / 64))
    check_against_oracle(h, W, a, g, what=str((N, D, V)))


def test_temperature_and_bad_targets():
    h, W, a, g = _case(129, 256, 1500, 90, w_std=0.05)
    a[[0, 7]] = [-100, 1500]
    check_against_oracle(h, W, a, g, tau=0.7, what="tau 0.7")


def test_several_row_chunks_accumulate_and_repeat():
    """N = 4396 spans two row chunks (4096 + 300): dW sums the chunks in row
    order; accumulate_dW adds a second call's gradient; repeats are
    bit-identical."""
    h, W, a, g = _case(4396, 128, 2000, 91, w_std=0.1)
    dh, dW, o = check_against_oracle(h, W, a, g, what="two chunks")
    hd, Wd, ad, gd = _bf16_dev(h), _bf16_dev(W), _dev(a), _dev(g)
    _, lse = tim.token_logprob(hd, Wd, ad)
    dh1, dW1 = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
    dh2, dW2 = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
    dWa = dW1.clone()
    tim.token_logprob_backward(hd, Wd, ad, gd, lse, dW=dWa, accumulate_dW=True)
    tim.check()
    assert torch.equal(dh1, dh2) and torch.equal(dW1, dW2)
    # (dW + C1) + C2 against 2 (C1 + C2): fp32 rounding of partial sums, ~1 ulp of the largest
    w1 = dW1.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(dWa.cpu().numpy(), 2 * w1, rtol=0, atol=1e-6 * np.max(np.abs(w1)))


def test_zero_gradient_gives_zero():
    h, W, a, _ = _case(64, 128, 700, 92, w_std=0.1)
    dh, dW = gpu_backward(h, W, a, np.zeros(64, np.float32))
    assert not dh.any() and not dW.any()


def test_qwen_shape_sampled_rows_and_identity():
    """The Qwen3-8B-shaped head (N = 8192 in two row chunks, D = 4096,
    V = 151936): dh on sampled rows against the oracle; dW through
    <dW, W> = <dh, h>."""
    cfg = wl.CONFIGS["qwen3_8b"]
    h, W = wl.draw_head(cfg)
    a = wl.draw_targets(cfg, cfg.N)
    g = np.random.default_rng(93).standard_normal(cfg.N).astype(np.float32)
    dh, dW = gpu_backward(h, W, a, g)
    rows = np.array([0, 4095, 4096, cfg.N - 1])
    o = oracle.token_logprob_backward(h[rows], W, a[rows], g[rows], want_dz=True)
    Wf = wl.bf16_to_f32(W).astype(np.float64)
    assert_close(dh[rows], o["dh"], np.sqrt(o["dz"] ** 2 @ Wf ** 2), _abs_p(o["dz"], a[rows], g[rows]) @ np.abs(Wf),
                 "qwen dh rows")
    hf = wl.bf16_to_f32(h).astype(np.float64)
    lhs = float(np.sum(dW.astype(np.float64) * Wf))
    rhs = float(np.sum(dh.astype(np.float64) * hf))
    scale = float(np.sum(np.abs(dh.astype(np.float64) * hf)))
    print("qwen <dW, W> %.6g  <dh, h> %.6g  scale %.3g" % (lhs, rhs, scale))
    assert abs(lhs - rhs) <= 1e-4 * scale
    assert np.isfinite(dW).all() and np.isfinite(dh).all()
