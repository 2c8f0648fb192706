"""tim_token_logprob_noalloc: the token logprob for callers that cannot let a
library allocate device memory (an engine that reserved its device-memory
budget for its own allocator, or code without the stream-ordered allocator).
Its scratch is a fixed device array inside libtim.so shared by every call, so
it must give the bits of tim_token_logprob (same kernels, same reduction
order, same operand values), call after call, with nothing left over from the
previous call -- also when that call was larger -- and match the oracle.
This file runs last: it checks an addition, and a failure here must not hide
the results of the other tests."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import LOGP_ATOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _inputs(N, D, V, seed):
    rng = np.random.default_rng(seed)
    h = wl.bf16_round(rng.standard_normal((N, D), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.02))
    a = rng.integers(0, V, size=N).astype(np.int32)
    a[::97] = -100                                    # some ignored positions
    dev = torch.device("cuda", 0)
    hd = torch.from_numpy(h.view(np.int16)).to(dev).view(torch.bfloat16)
    Wd = torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16)
    return (h, W, a), (hd, Wd, torch.from_numpy(a).to(dev))


def _call(fn, hd, Wd, ad):
    N, D = hd.shape
    V = Wd.shape[0]
    lp = torch.full((N,), 123.0, dtype=torch.float32, device=hd.device)
    lse = torch.full((N,), 123.0, dtype=torch.float32, device=hd.device)
    rc = fn(hd.data_ptr(), Wd.data_ptr(), ad.data_ptr(), N, D, V, lp.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream(hd.device).cuda_stream)
    assert rc == tim.TIM_OK, tim.tim_last_error()
    return lp, lse


def _bits(t):
    return t.view(torch.int32).cpu().numpy()


def test_noalloc_matches_the_pool_entry_point_bit_for_bit_two_calls_in_a_row():
    torch.cuda.set_device(0)
    # N % 16 != 0 (padded last m-tile), a multiple of 16, and the first case
    # again after the larger second one has filled more of the shared array
    cases = [(3000, 1024, 32000, 1), (1216, 4096, 151936, 2), (3000, 1024, 32000, 1), (1, 512, 5000, 3)]
    for N, D, V, seed in cases:
        (h, W, a), (hd, Wd, ad) = _inputs(N, D, V, seed)
        lp_n, lse_n = _call(tim.tim_token_logprob_noalloc, hd, Wd, ad)
        lp_p, lse_p = _call(tim.tim_token_logprob, hd, Wd, ad)
        tim.check()
        assert np.array_equal(_bits(lp_n), _bits(lp_p)), (N, D, V)
        assert np.array_equal(_bits(lse_n), _bits(lse_p)), (N, D, V)
        assert int(torch.isnan(lp_n).sum()) == len(range(0, N, 97))
        # sampled rows (the first, the last, one per 128-row m-tile) against the oracle
        rows = np.unique(np.concatenate([[0, N - 1], np.arange(5, N, 128)]))
        o_lp, o_lse = oracle.token_logprob(h.view(np.uint16), W.view(np.uint16), a, rows=rows)
        g_lp = lp_n.cpu().numpy()[rows].astype(np.float64)
        g_lse = lse_n.cpu().numpy()[rows].astype(np.float64)
        assert np.array_equal(np.isnan(g_lp), np.isnan(o_lp))
        ok = ~np.isnan(o_lp)
        assert np.max(np.abs(g_lp[ok] - o_lp[ok]), initial=0.0) <= LOGP_ATOL
        assert np.max(np.abs(g_lse - o_lse)) <= LOGP_ATOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch.cuda.set_device(0)
    N, D, V = 20000, 64, 151936            # 20000 x 149 x 8 bytes > 16 MiB
    rc = tim.tim_token_logprob_noalloc(16, 16, 16, N, D, V, 16, 16, None)
    assert rc == tim.TIM_ERR_INVALID_ARG
    assert "TIM_NOALLOC_SCRATCH_BYTES" in tim.tim_last_error()
