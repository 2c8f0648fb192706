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
rows; dW is checked element by element on a batch of three row chunks.
Every contraction is the library's own tcgen05 GEMM with a reduction order
fixed by V (dh) or by the row order (dW), so a row of dh has the same bits
whatever batch it is in."""
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
                                   (5, 4096, 3000), (1, 64, 1),
                                   # long k loops for dh (K = V) over several m-blocks
                                   (130, 128, 45000), (257, 64, 83000)])
def test_ragged_shapes(N, D, V):
    h, W, a, g = _case(N, D, V, N + 3 * D + V, w_std=0.3 / math.sqrt(D / 64))
    check_against_oracle(h, W, a, g, what=str((N, D, V)))


def test_temperature_and_bad_targets():
    h, W, a, g = _case(129, 256, 1500, 90, w_std=0.05)
    a[[0, 7]] = [-100, 1500]
    check_against_oracle(h, W, a, g, tau=0.7, what="tau 0.7")


ROWS_PER_CHUNK = 16384   # rows of one backward chunk in the library (dz of a chunk kept whole)


def test_three_row_chunks_elementwise_accumulate_and_repeat():
    """N = 2 x 16384 + 237 spans three row chunks: dh and dW element by element
    against the oracle (dW sums the chunks in row order); accumulate_dW adds a
    second call's gradient; repeats are bit-identical."""
    N = 2 * ROWS_PER_CHUNK + 237
    h, W, a, g = _case(N, 64, 1000, 91, w_std=0.1)
    dh, dW, o = check_against_oracle(h, W, a, g, what="three chunks")
    hd, Wd, ad, gd = _bf16_dev(h), _bf16_dev(W), _dev(a), _dev(g)
    _, lse = tim.token_logprob(hd, Wd, ad)
    dh1, dW1 = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
    dh2, dW2 = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
    dWa = dW1.clone()
    tim.token_logprob_backward(hd, Wd, ad, gd, lse, dW=dWa, accumulate_dW=True)
    tim.check()
    assert torch.equal(dh1, dh2) and torch.equal(dW1, dW2)
    # (dW + C1) + C2 + C3 against 2 (C1 + C2 + C3): fp32 rounding of partial sums
    w1 = dW1.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(dWa.cpu().numpy(), 2 * w1, rtol=0, atol=2e-6 * np.max(np.abs(w1)))


def test_dh_rows_bit_identical_across_batch_sizes():
    """Probe rows of the Qwen3-8B-shaped head (D = 4096, V = 151936) alone
    (N = 1) and inside batches of N = 300, 4096 and 8192 other rows: each
    probe's dh row has the same bits in every batch (its reduction order is a
    function of V alone), as do its lse and logprob."""
    cfg = wl.CONFIGS["qwen3_8b"]
    D, V = cfg.D, cfg.V
    _, W = wl.draw_head(cfg, N=1)
    Wd = _bf16_dev(W)
    P = 4
    rng = np.random.default_rng(94)
    probes_h = wl.draw_h_rows(cfg, seed=95, N=P)
    probes_a = rng.integers(0, V, size=P).astype(np.int32)
    probes_g = rng.standard_normal(P).astype(np.float32)
    ref = None
    for N in (1, 300, 4096, 8192):
        if N == 1:
            rows = []
            for i in range(P):
                hd, ad, gd = _bf16_dev(probes_h[i:i + 1]), _dev(probes_a[i:i + 1]), _dev(probes_g[i:i + 1])
                _, lse = tim.token_logprob(hd, Wd, ad)
                dh, _ = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
                rows.append(dh[0].cpu().numpy())
            got = np.stack(rows)
        else:
            h = wl.draw_h_rows(cfg, seed=100 + N, N=N)
            a = rng.integers(0, V, size=N).astype(np.int32)
            g = rng.standard_normal(N).astype(np.float32)
            pos = rng.choice(N, size=P, replace=False)
            h[pos], a[pos], g[pos] = probes_h, probes_a, probes_g
            hd, ad, gd = _bf16_dev(h), _dev(a), _dev(g)
            _, lse = tim.token_logprob(hd, Wd, ad)
            dh, _ = tim.token_logprob_backward(hd, Wd, ad, gd, lse)
            got = dh.cpu().numpy()[pos]
        tim.check()
        assert np.isfinite(got).all()
        if ref is None:
            ref = got
        else:
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), N


def test_zero_gradient_gives_zero():
    h, W, a, _ = _case(64, 128, 700, 92, w_std=0.1)
    dh, dW = gpu_backward(h, W, a, np.zeros(64, np.float32))
    assert not dh.any() and not dW.any()


def test_qwen_shape_sampled_rows_and_identity():
    """The Qwen3-8B-shaped head (N = 8192 in one row chunk, D = 4096,
    V = 151936): dh on sampled rows (both CTAs of a pair, first and last row
    blocks) against the oracle; dW through <dW, W> = <dh, h>."""
    cfg = wl.CONFIGS["qwen3_8b"]
    h, W = wl.draw_head(cfg)
    a = wl.draw_targets(cfg, cfg.N)
    g = np.random.default_rng(93).standard_normal(cfg.N).astype(np.float32)
    dh, dW = gpu_backward(h, W, a, g)
    rows = np.array([0, 200, 4095, 4096, cfg.N - 1])
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
