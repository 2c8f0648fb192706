"""tim_token_logprob_noalloc: the token logprob for callers that cannot let a
library allocate device memory (an engine that reserved its device-memory
budget for its own allocator, or code without the stream-ordered allocator).
Its scratch is a fixed device array inside libtim.so, so it must give the same
results as tim_token_logprob, call after call, with nothing left over from the
previous call.  This file runs last: it checks an addition, and a failure here
must not hide the results of the other tests."""
import numpy as np
import pytest

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
    return hd, Wd, torch.from_numpy(a).to(dev)


def _call(fn, hd, Wd, ad):
    N, D = hd.shape
    V = Wd.shape[0]
    lp = torch.full((N,), 123.0, dtype=torch.float32, device=hd.device)
    lse = torch.full((N,), 123.0, dtype=torch.float32, device=hd.device)
    rc = fn(hd.data_ptr(), Wd.data_ptr(), ad.data_ptr(), N, D, V, lp.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream(hd.device).cuda_stream)
    assert rc == tim.TIM_OK, tim.tim_last_error()
    return lp, lse


def test_noalloc_matches_the_pool_entry_point_two_calls_in_a_row():
    torch.cuda.set_device(0)
    cases = [(3000, 1024, 32000, 1), (1200, 4096, 151936, 2)]
    for N, D, V, seed in cases:
        hd, Wd, ad = _inputs(N, D, V, seed)
        lp_n, lse_n = _call(tim.tim_token_logprob_noalloc, hd, Wd, ad)
        lp_p, lse_p = _call(tim.tim_token_logprob, hd, Wd, ad)
        tim.check()
        nan_n, nan_p = torch.isnan(lp_n), torch.isnan(lp_p)
        assert torch.equal(nan_n, nan_p) and int(nan_n.sum()) == len(range(0, N, 97))
        ok = ~nan_p
        assert float((lp_n[ok] - lp_p[ok]).abs().max()) <= LOGP_ATOL
        assert float((lse_n - lse_p).abs().max()) <= LOGP_ATOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch.cuda.set_device(0)
    N, D, V = 20000, 64, 151936            # 20000 x 149 x 8 bytes > 16 MiB
    rc = tim.tim_token_logprob_noalloc(16, 16, 16, N, D, V, 16, 16, None)
    assert rc == tim.TIM_ERR_INVALID_ARG
    assert "TIM_NOALLOC_SCRATCH_BYTES" in tim.tim_last_error()
