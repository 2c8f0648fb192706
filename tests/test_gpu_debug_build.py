"""The checked build (libtim_debug.so, compiled with TIM_DEBUG): its kernels
also check their own invariants (TMA coordinates, store ranges, claimed work
units, bulk-copy alignment) and the input contracts the release build passes
over silently, and record the first violation without trapping.  Clean calls
must record nothing and give the release build's bits; a planted contract
violation (made on the host, no fault anywhere) must come back from
tim_check as TIM_ERR_BAD_INPUT with its kind and index."""
import numpy as np
import pytest

import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16(u16):
    return _dev(u16.view(np.int16)).view(torch.bfloat16)


def _head(N, D, V, seed):
    rng = np.random.default_rng(seed)
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.05))
    a = rng.integers(0, V, size=N).astype(np.int32)
    return h, W, a


def _seq_inputs(N, seed):
    off = np.array([0, 100, 100, 700, N], dtype=np.int32)
    rng = np.random.default_rng(seed)
    l_tr = wl.draw_train_logprobs(N, seed)
    l_ro = (l_tr + rng.normal(0, 0.05, N)).astype(np.float32)
    mask = (rng.random(N) < 0.8).astype(np.uint8)
    adv = rng.standard_normal(N).astype(np.float32)
    return off, l_tr, l_ro, mask, adv


def _all_calls(h, W, a, off, l_tr, l_ro, mask, adv):
    """Every entry point once; returns their outputs as host arrays."""
    hd, Wd, ad = _bf16(h), _bf16(W), _dev(a)
    lp, lse = tim.token_logprob(hd, Wd, ad)
    g = torch.linspace(-1, 1, h.shape[0], device="cuda")
    dh, dW = tim.token_logprob_backward(hd, Wd, ad, g, lse)
    ms = tim.mismatch_stats(_dev(l_tr), _dev(l_ro), _dev(mask), _dev(off), token_weight=True)
    pp = tim.tis_ppo(_dev(l_tr + 0.01), _dev(l_tr), _dev(l_ro), _dev(adv), _dev(mask), _dev(off))
    mon = tim.mismatch_monitor(_dev(l_tr), _dev(l_ro), _dev(mask), 0.1)
    out = [lp, lse, dh, dW, ms["seq_stats"], ms["batch"], ms["token_weight"], pp["token_loss"], pp["batch"],
           mon["record"] if isinstance(mon, dict) and "record" in mon else mon]
    return [o.cpu().numpy() if isinstance(o, torch.Tensor) else
            {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in o.items()} for o in out]


def _same_bits(x, y):
    if isinstance(x, dict):
        return all(_same_bits(x[k], y[k]) for k in x)
    if x is None:
        return y is None
    return np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))


def test_clean_calls_record_nothing_and_match_the_release_bits():
    h, W, a = _head(300, 256, 3000, 1)
    ins = _seq_inputs(2000, 2)
    ref = _all_calls(h, W, a, *ins)
    tim.check()
    assert tim.tim_debug_build() == 0
    with tim.checked():
        assert tim.tim_debug_build() == 1
        got = _all_calls(h, W, a, *ins)
        tim.check()
        assert tim.tim_debug_violation() == ("none", 0, 0)
    for r, g in zip(ref, got):
        assert _same_bits(r, g)


def _expect(kind, index):
    with pytest.raises(tim.TimError) as e:
        tim.check()
    assert e.value.code == tim.TIM_ERR_BAD_INPUT
    rec = tim.tim_debug_violation()
    assert rec[0] == kind and rec[1] == index, rec
    return rec


def test_target_id_at_or_past_V():
    h, W, a = _head(200, 128, 1000, 3)
    a[5] = 1003          # >= V: a bug in the caller (negative ids are the ignore label)
    a[9] = -100
    with tim.checked():
        lp, _ = tim.token_logprob(_bf16(h), _bf16(W), _dev(a))
        rec = _expect("target", 5)
        assert rec[2] == 1003
        assert torch.isnan(lp[[5, 9]]).all()
    # the release build gives the same NaNs and records nothing
    tim.token_logprob(_bf16(h), _bf16(W), _dev(a))
    tim.check()
    assert tim.tim_debug_violation() == ("none", 0, 0)


def test_non_finite_hidden_state_gives_a_non_finite_logit():
    h, W, a = _head(300, 128, 1000, 4)
    h[177, 3] = 0x7FC0   # a bf16 NaN in row 177
    with tim.checked():
        tim.token_logprob(_bf16(h), _bf16(W), _dev(a))
        _expect("logit", 177)


def test_mask_byte_other_than_0_or_1():
    off, l_tr, l_ro, mask, adv = _seq_inputs(2000, 5)
    mask[1234] = 2
    with tim.checked():
        tim.mismatch_stats(_dev(l_tr), _dev(l_ro), _dev(mask), _dev(off))
        rec = _expect("mask", 1234)
        assert rec[2] == 2


def test_non_finite_advantage_of_a_used_token():
    off, l_tr, l_ro, mask, adv = _seq_inputs(2000, 6)
    mask[:] = 1
    adv[901] = np.inf
    with tim.checked():
        tim.tis_ppo(_dev(l_tr + 0.01), _dev(l_tr), _dev(l_ro), _dev(adv), _dev(mask), _dev(off))
        _expect("advantage", 901)


def test_non_finite_lse_in_the_backward():
    h, W, a = _head(200, 128, 1000, 7)
    hd, Wd, ad = _bf16(h), _bf16(W), _dev(a)
    _, lse = tim.token_logprob(hd, Wd, ad)
    tim.check()
    lse[33] = float("nan")
    with tim.checked():
        tim.token_logprob_backward(hd, Wd, ad, torch.ones(200, device="cuda"), lse)
        _expect("backward_input", 33)
