"""Failure detection without a GPU fault: the bounded-wait path of the kernels'
pipelines reports TIM_ERR_TIMEOUT through tim_check, and the context stays
usable afterwards; bad data is reported, not trapped (see also the offsets
test of the mismatch pass)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_expired_wait_is_reported_and_the_device_stays_usable():
    torch.cuda.set_device(0)
    tim.check()                                   # start from a clean status
    assert tim.tim_selftest_wait_timeout(2000, _stream()) == tim.TIM_OK   # 2 ms
    with pytest.raises(tim.TimError) as e:
        tim.check()
    assert e.value.code == tim.TIM_ERR_TIMEOUT
    # the status word was cleared and the context still computes correctly
    tim.check()
    h = torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device="cuda")
    lp, lse = tim.token_logprob(h, W, torch.tensor([0, 5, 99], dtype=torch.int32, device="cuda"))
    tim.check()
    assert torch.allclose(lp, torch.full((3,), -float(np.log(100)), device="cuda"))


def test_selftest_rejects_bad_budget():
    assert tim.tim_selftest_wait_timeout(0, _stream()) == tim.TIM_ERR_INVALID_ARG
    assert tim.tim_selftest_wait_timeout(2_000_000, _stream()) == tim.TIM_ERR_INVALID_ARG
