"""The seeded input generators: bf16 rounding and the workload layouts."""
import numpy as np
import pytest

import workloads as wl


def test_bf16_rounding_order_example():
    """HN "Train-infer mismatch" page, "Rounding depends on the order of
    additions": in bf16, 1 + 2^-8 rounds to 1, while (2^-8 + 2^-8) + 1 is
    exactly 1 + 2^-7, the next value above 1."""
    one = np.float32(1.0)
    e8 = np.float32(2.0 ** -8)
    assert wl.bf16_to_f32(wl.bf16_round(one + e8)) == one
    assert wl.bf16_to_f32(wl.bf16_round((e8 + e8) + one)) == np.float32(1 + 2.0 ** -7)
    # ties go to the even neighbour: 1 + 3*2^-8 sits between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert wl.bf16_to_f32(wl.bf16_round(np.float32(1 + 3 * 2.0 ** -8))) == np.float32(1 + 2.0 ** -6)


def test_bf16_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 50
    ours = wl.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_draws_are_seeded_and_chunk_independent():
    cfg = wl.HeadConfig("t", N=10, D=48, V=33)
    h1, W1 = wl.draw_head(cfg)
    h2, W2 = wl.draw_head(cfg)
    assert np.array_equal(h1, h2) and np.array_equal(W1, W2)
    a = wl._normal_bf16(np.random.default_rng(3), (7, 9), 0.1, chunk=5)
    b = wl._normal_bf16(np.random.default_rng(3), (7, 9), 0.1, chunk=1000)
    assert np.array_equal(a, b)
    # W does not depend on N
    _, W3 = wl.draw_head(cfg, N=3)
    assert np.array_equal(W1, W3)


def test_segment_layouts():
    q = wl.CONFIGS["qwen3_8b"]
    off = wl.draw_segments(q)
    assert off[0] == 0 and off[-1] == q.N and len(off) == 17 and np.all(np.diff(off) == 512)
    m = wl.draw_mask(q, off)
    assert m.sum() == 16 * 384
    ll = wl.CONFIGS["llama3_8b"]
    off = wl.draw_segments(ll)
    lens = np.diff(off)
    assert off[-1] == ll.N and np.all(lens[:-1] >= 128) and np.all(lens <= 4096) and lens[-1] >= 1
    assert 700 < np.median(lens) < 1400
    m = wl.draw_mask(ll, off)
    assert abs(1 - m.mean() - 0.3) < 0.01


def test_rollout_noise_and_outliers():
    ll = wl.CONFIGS["llama3_8b"]
    lt = wl.draw_train_logprobs(200_000, 0)
    lr = wl.draw_rollout(ll, lt)
    d = lr.astype(np.float64) - lt
    big = np.abs(d) > 0.5
    assert abs(big.mean() - 0.005) < 0.001
    assert abs(np.std(d[~big]) - 0.02) < 0.001
    assert np.all(lt <= 0)


def test_top5_targets_need_top5():
    ds = wl.CONFIGS["dsv3"]
    with pytest.raises(ValueError):
        wl.draw_targets(ds, 4)
    top5 = np.tile(np.arange(5, dtype=np.int32), (1000, 1)) + 100
    t = wl.draw_targets(ds, 1000, top5=top5)
    frac = np.mean((t >= 100) & (t < 105))
    assert 0.65 < frac < 0.75
