"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol include/tim.h declares, and rejects bad arguments on the host before any
CUDA call (no compute call is made here)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

import rollout_logprob_mismatch_gb300 as tim
from rollout_logprob_mismatch_gb300 import build as tim_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tim.h")


@pytest.fixture(scope="module")
def lib():
    tim_build.build()
    return tim.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"TIM_API\s+[\w\s\*]*?\b(tim_\w+)\s*\(", text)


def test_header_declares_the_api():
    names = declared_functions()
    assert {"tim_token_logprob", "tim_mismatch_stats", "tim_check", "tim_last_error",
            "tim_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", tim.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c_and_struct_layout_matches(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "tim.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(tim_mismatch_out),"
        "offsetof(tim_mismatch_out,num_seqs),offsetof(tim_mismatch_out,num_tokens),"
        "offsetof(tim_mismatch_out,tau_seq),offsetof(tim_mismatch_out,seq_estimator),"
        "offsetof(tim_mismatch_out,token_weight),offsetof(tim_mismatch_out,seq_stats),"
        "offsetof(tim_mismatch_out,seq_flags),offsetof(tim_mismatch_out,batch_stats),"
        "offsetof(tim_mismatch_out,seq_records));"
        "return TIM_SEQ_FIELDS == 12 && TIM_BATCH_FIELDS == 20 && TIM_SEQ_RECORD_WORDS == 16 ? 0 : 1;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                    "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    S = tim.tim_mismatch_out
    want = [ctypes.sizeof(S)] + [getattr(S, f).offset for f in
                                 ("num_seqs", "num_tokens", "tau_seq", "seq_estimator", "token_weight",
                                  "seq_stats", "seq_flags", "batch_stats", "seq_records")]
    assert vals == want
    assert len(tim.SEQ_FIELDS) == 12 and len(tim.BATCH_FIELDS) == 20 and tim.SEQ_RECORD_WORDS == 16


def test_version(lib):
    assert tim.tim_version() >= 100


@pytest.mark.parametrize("N,D,V", [(-1, 64, 10), (4, 0, 10), (4, 12, 10), (4, 64, 0), (4, 64, 1 << 31),
                                   (1 << 31, 64, 10), (4, 65544, 10)])
def test_token_logprob_rejects_bad_sizes(lib, N, D, V):
    rc = tim.tim_token_logprob(16, 16, 16, N, D, V, 16, 16, None)
    assert rc == tim.TIM_ERR_INVALID_ARG
    assert tim.tim_last_error()


def test_token_logprob_rejects_null_and_misaligned(lib):
    assert tim.tim_token_logprob(None, 16, 16, 4, 64, 10, 16, 16, None) == tim.TIM_ERR_INVALID_ARG
    assert tim.tim_token_logprob(16, 16, 16, 4, 64, 10, None, 16, None) == tim.TIM_ERR_INVALID_ARG
    assert tim.tim_token_logprob(8, 16, 16, 4, 64, 10, 16, 16, None) == tim.TIM_ERR_INVALID_ARG
    assert "aligned" in tim.tim_last_error()


def test_token_logprob_empty_is_noop(lib):
    assert tim.tim_token_logprob(None, None, None, 0, 64, 10, None, None, None) == tim.TIM_OK


def test_noalloc_rejects_bad_arguments_on_the_host(lib):
    """The no-alloc entry point checks sizes, pointers, alignment and its fixed
    scratch (N x ceil(V / 1024) partials) before any CUDA call."""
    E = tim.TIM_ERR_INVALID_ARG
    call = tim.tim_token_logprob_noalloc
    for N, D, V in ((-1, 64, 10), (4, 12, 10), (4, 64, 0), (1 << 31, 64, 10), (4, 65544, 10)):
        assert call(16, 16, 16, N, D, V, 16, 16, None) == E, (N, D, V)
    assert call(None, 16, 16, 4, 64, 10, 16, 16, None) == E
    assert call(16, 8, 16, 4, 64, 10, 16, 16, None) == E
    assert call(16, 16, 18, 4, 64, 10, 16, 16, None) == E
    # 14080 rows of 149 chunks (V = 151936) need 16.8 MB of partials, more than the 16 MiB scratch
    assert call(16, 16, 16, 14080, 4096, 151936, 16, 16, None) == E
    assert "TIM_NOALLOC_SCRATCH_BYTES" in tim.tim_last_error()
    assert call(None, None, None, 0, 64, 10, None, None, None) == tim.TIM_OK


def test_selftest_rejects_bad_budget_on_the_host(lib):
    for budget in (0, 1000001):
        assert tim.tim_selftest_wait_timeout(budget, None) == tim.TIM_ERR_INVALID_ARG


def _out(S=1, N=4, est=3, batch=16, seq=16, flags=16):
    d = tim.tim_mismatch_out()
    d.num_seqs, d.num_tokens, d.tau_seq, d.seq_estimator = S, N, math.nan, est
    d.token_weight, d.seq_stats, d.seq_flags, d.batch_stats = None, seq, flags, batch
    return d


def test_mismatch_stats_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    ok_ptrs = (16, 16, 16, 16)
    assert lib.tim_mismatch_stats(*ok_ptrs, 2.0, None, None) == E
    for C in (0.0, -1.0, math.nan, math.inf):
        assert tim.tim_mismatch_stats(*ok_ptrs, C, _out(), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(S=-1), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(S=0, N=5), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(est=2), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(batch=None), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(seq=None), None) == E
    assert tim.tim_mismatch_stats(None, 16, 16, 16, 2.0, _out(), None) == E
    assert tim.tim_mismatch_stats(16, 16, 16, None, 2.0, _out(), None) == E
    assert tim.tim_mismatch_stats(18, 16, 16, 16, 2.0, _out(), None) == E
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, _out(batch=20), None) == E
    d = _out()
    d.seq_records = 24   # caller-owned records must be 16-byte aligned
    assert tim.tim_mismatch_stats(*ok_ptrs, 2.0, d, None) == E


def test_mismatch_fold_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    assert tim.tim_mismatch_fold(16, -1, 16, None) == E
    assert tim.tim_mismatch_fold(None, 3, 16, None) == E
    assert tim.tim_mismatch_fold(16, 3, None, None) == E
    assert tim.tim_mismatch_fold(24, 3, 16, None) == E      # records not 16-byte aligned
    assert tim.tim_mismatch_fold(16, 3, 20, None) == E      # batch record not 8-byte aligned
    assert "aligned" in tim.tim_last_error()


def test_ppo_struct_layout_matches(tmp_path):
    src = tmp_path / "ppo_layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "tim.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(tim_ppo_out),"
        "offsetof(tim_ppo_out,num_seqs),offsetof(tim_ppo_out,num_tokens),offsetof(tim_ppo_out,token_loss),"
        "offsetof(tim_ppo_out,token_grad),offsetof(tim_ppo_out,seq_loss),offsetof(tim_ppo_out,batch_stats));"
        "return TIM_PPO_FIELDS == 9 && TIM_PPO_N_SEQS_NONEMPTY == 8 ? 0 : 1;}\n")
    exe = tmp_path / "ppo_layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                    "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    S = tim.tim_ppo_out
    want = [ctypes.sizeof(S)] + [getattr(S, f).offset for f in
                                 ("num_seqs", "num_tokens", "token_loss", "token_grad", "seq_loss", "batch_stats")]
    assert vals == want
    assert len(tim.PPO_FIELDS) == 9


def _ppo_out(S=1, N=4, seq=16, batch=16, loss=None, grad=None):
    d = tim.tim_ppo_out()
    d.num_seqs, d.num_tokens = S, N
    d.token_loss, d.token_grad, d.seq_loss, d.batch_stats = loss, grad, seq, batch
    return d


def test_tis_ppo_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    p6 = (16, 16, 16, 16, 16, 16)
    assert lib.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, None, None) == E
    for lo, hi, C in ((1.0, 0.2, 2.0), (-0.1, 0.2, 2.0), (math.nan, 0.2, 2.0), (0.2, -0.1, 2.0),
                      (0.2, math.inf, 2.0), (0.2, math.nan, 2.0), (0.2, 0.2, 0.0), (0.2, 0.2, math.inf)):
        assert tim.tim_tis_ppo(*p6, lo, hi, C, _ppo_out(), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(S=-1), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(S=0, N=3), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(seq=None), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(batch=None), None) == E
    assert tim.tim_tis_ppo(None, 16, 16, 16, 16, 16, 0.2, 0.2, 2.0, _ppo_out(), None) == E
    assert tim.tim_tis_ppo(16, 16, 16, 16, 16, None, 0.2, 0.2, 2.0, _ppo_out(), None) == E
    assert tim.tim_tis_ppo(18, 16, 16, 16, 16, 16, 0.2, 0.2, 2.0, _ppo_out(), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(grad=18), None) == E
    assert tim.tim_tis_ppo(*p6, 0.2, 0.2, 2.0, _ppo_out(batch=20), None) == E
    assert "aligned" in tim.tim_last_error()


def test_mismatch_monitor_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    assert tim.tim_mismatch_monitor(16, 16, 16, -1, 0.1, None, 16, None) == E
    assert tim.tim_mismatch_monitor(16, 16, 16, 1 << 31, 0.1, None, 16, None) == E
    for tau in (-0.1, math.nan, math.inf):
        assert tim.tim_mismatch_monitor(16, 16, 16, 4, tau, None, 16, None) == E
    assert tim.tim_mismatch_monitor(16, 16, 16, 4, 0.1, None, None, None) == E
    assert tim.tim_mismatch_monitor(None, 16, 16, 4, 0.1, None, 16, None) == E
    assert tim.tim_mismatch_monitor(16, 16, 20, 4, 0.1, None, 16, None) == E
    assert tim.tim_mismatch_monitor(16, 16, 16, 4, 0.1, 8, 16, None) == E
    assert tim.tim_mismatch_monitor(16, 16, 16, 4, 0.1, None, 12, None) == E
    assert "aligned" in tim.tim_last_error()
    assert len(tim.MONITOR_FIELDS) == 7


def test_fp32_head_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    assert tim.tim_split_weight_bytes(10, 100) == 10 * 3 * 128 * 2
    assert tim.tim_split_weight_bytes(10, 64) == 10 * 3 * 64 * 2
    assert tim.tim_split_weight_bytes(0, 64) == -1 and tim.tim_split_weight_bytes(10, 65537) == -1
    assert tim.tim_split_weight_fp32(16, 0, 64, 16, None) == E
    assert tim.tim_split_weight_fp32(16, 10, 12, 16, None) == E
    assert tim.tim_split_weight_fp32(None, 10, 64, 16, None) == E
    assert tim.tim_split_weight_fp32(16, 10, 64, 8, None) == E
    assert tim.tim_split_weight_fp32(20, 10, 64, 16, None) == E
    for tau in (0.0, -1.0, math.inf, math.nan):
        assert tim.tim_token_logprob_fp32_head(16, 16, 16, 4, 64, 10, tau, 16, 16, None) == E
    assert tim.tim_token_logprob_fp32_head(16, 16, 16, 4, 12, 10, 1.0, 16, 16, None) == E
    assert tim.tim_token_logprob_fp32_head(16, 8, 16, 4, 64, 10, 1.0, 16, 16, None) == E


def test_backward_rejects_bad_arguments(lib):
    E = tim.TIM_ERR_INVALID_ARG
    ok = dict(h=16, W=16, t=16, g=16, l=16, N=4, D=64, V=10, tau=1.0, dh=16, dW=16)

    def call(**kw):
        a = dict(ok, **kw)
        return tim.tim_token_logprob_backward(a["h"], a["W"], a["t"], a["g"], a["l"], a["N"], a["D"], a["V"],
                                              a["tau"], a["dh"], a["dW"], 0, None)
    for bad in (dict(N=-1), dict(D=12), dict(D=0), dict(V=0), dict(tau=0.0), dict(tau=math.nan), dict(W=None),
                dict(dW=None), dict(h=None), dict(g=None), dict(l=None), dict(dh=None), dict(h=8), dict(dh=24),
                dict(dW=8), dict(g=18)):
        assert call(**bad) == E, bad


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(tim, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(tim, "_DEBUG_LIB_PATH", str(tmp_path / "absent_debug.so"))
    monkeypatch.setattr(tim, "_lib", None)
    monkeypatch.setattr(tim, "_release", None)
    monkeypatch.setattr(tim, "_debug", None)
    with pytest.raises(tim.TimError):
        tim.load()
    with pytest.raises(tim.TimError):
        tim.load_debug()


def test_checked_build_exports_the_same_api_and_says_so(lib):
    """libtim_debug.so (TIM_DEBUG) exports every declared symbol; the two
    builds tell themselves apart without touching a GPU."""
    out = subprocess.run(["nm", "-D", "--defined-only", tim._DEBUG_LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
    assert tim.tim_debug_build() == 0
    with tim.checked():
        assert tim.tim_debug_build() == 1
    assert tim.tim_debug_build() == 0


def test_torch_wrappers_reject_host_tensors_and_wrong_types():
    """The torch wrappers check their tensors before any library call: host
    tensors, wrong dtypes and non-tensors raise (there is no CPU path)."""
    torch = pytest.importorskip("torch")
    h = torch.zeros((4, 64), dtype=torch.bfloat16)
    W = torch.zeros((10, 64), dtype=torch.bfloat16)
    a = torch.zeros(4, dtype=torch.int32)
    l = torch.zeros(4, dtype=torch.float32)
    m = torch.ones(4, dtype=torch.uint8)
    off = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tim.token_logprob(h, W, a)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tim.mismatch_stats(l, l, m, off)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tim.mismatch_monitor(l, l, m, 0.1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tim.tis_ppo(l, l, l, l, m, off)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tim.split_weight_fp32(torch.zeros((10, 64)))
    with pytest.raises(TypeError):
        tim.token_logprob([[0.0]], W, a)
