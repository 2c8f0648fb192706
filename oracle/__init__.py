"""fp64 CPU oracle (plain C, ``oracle.c``) and its ctypes binding.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library; the two sides meet only in the seeded
input generators of ``workloads``.

``token_logprob``  -- the selected-token logprob by the definition (icarus
"RL: Training Inference Mismatch", section "log p"): z = h W^T in fp64,
lse = log sum exp z, logp = z[a] - lse.
``token_logprob_backward`` -- dh, dW (and dz) of sum_t g_t l_t (Thinking
Machines page, "Unclipped importance sampling": gradients of log q_t).
``token_logprob_f32w`` -- the same with fp32 weights (the FP32 LM head of
LoongSage "Train-Inference Consistency" section 3).
``tis_ppo``        -- the TIS-weighted PPO clipped surrogate, its gradient and
masked means (VeXact summary eq. (2)-(3); HN "Clipped importance ratios").
``mismatch_monitor`` -- p95 |delta|, ratio quantiles 0.01 / 0.5 / 0.99, extreme
token fraction and token rejection (llm-infra-atlas section 7; VeXact tau_tok).
``mismatch_stats`` -- delta, r, k1/k2/k3, truncated-IS weight, masked
per-sequence and batch means and the rejection flag (VeXact summary eq. (1)
and "KL Estimators"; llm-infra-atlas section 2; icarus "KL estimators",
monitoring steps and compute_consistency_and_kl_metrics; LoongSage sections
4-5).  Field orders are ``SEQ_FIELDS`` and ``BATCH_FIELDS``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

SEQ_FIELDS = ("n_mask", "n_used", "n_nan", "n_clip", "mean_delta", "mean_abs_delta",
              "max_abs_delta", "mean_k1", "mean_k2", "mean_k3", "mean_w", "mean_rel")
BATCH_FIELDS = ("n_mask", "n_used", "n_nan", "n_clip", "mean_delta", "mean_abs_delta",
                "max_abs_delta", "mean_k1", "mean_k2", "mean_k3", "mean_w", "mean_rel",
                "seqmean_k1", "seqmean_k2", "seqmean_k3", "clip_ratio", "nan_ratio",
                "reject_ratio", "n_seqs_nonempty", "n_rejected")


PPO_FIELDS = ("n_mask", "n_used", "n_ppo_clipped", "n_tis_clipped", "mean_loss", "seqmean_loss",
              "ppo_clip_ratio", "tis_clip_ratio", "n_seqs_nonempty")

MONITOR_FIELDS = ("n_used", "p95_abs_delta", "ratio_q01", "ratio_q50", "ratio_q99", "n_extreme",
                  "frac_extreme")


def build(force: bool = False) -> str:
    """Compile oracle.c with plain gcc -O2 (no fast-math) into _liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            lib.oracle_token_logprob.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_double, P, P, ctypes.c_int]
            lib.oracle_token_logprob.restype = ctypes.c_int
            lib.oracle_token_logprob_f32w.argtypes = lib.oracle_token_logprob.argtypes
            lib.oracle_token_logprob_f32w.restype = ctypes.c_int
            lib.oracle_token_logprob_backward.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64,
                                                          ctypes.c_int64, ctypes.c_double, P, P, P]
            lib.oracle_token_logprob_backward.restype = ctypes.c_int
            lib.oracle_mismatch_stats.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int64,
                                                  ctypes.c_double, ctypes.c_double, ctypes.c_int32,
                                                  P, P, P, P]
            lib.oracle_mismatch_stats.restype = ctypes.c_int
            lib.oracle_mismatch_stats_threads.argtypes = lib.oracle_mismatch_stats.argtypes + [ctypes.c_int]
            lib.oracle_mismatch_stats_threads.restype = ctypes.c_int
            lib.oracle_tis_ppo.argtypes = [P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_double,
                                           ctypes.c_double, ctypes.c_double, P, P, P, P]
            lib.oracle_tis_ppo.restype = ctypes.c_int
            lib.oracle_mismatch_monitor.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_double, P, P]
            lib.oracle_mismatch_monitor.restype = ctypes.c_int
            assert lib.oracle_monitor_fields() == len(MONITOR_FIELDS)
            assert lib.oracle_ppo_fields() == len(PPO_FIELDS)
            assert lib.oracle_seq_fields() == len(SEQ_FIELDS)
            assert lib.oracle_batch_fields() == len(BATCH_FIELDS)
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def token_logprob(h_bf16: np.ndarray, W_bf16: np.ndarray, targets: np.ndarray,
                  rows=None, nthreads: int | None = None, temperature: float = 1.0):
    """(logp, lse) as float64 arrays, for `rows` of h (all rows if None), of
    log softmax(h W^T / temperature) at the targets.

    h_bf16 uint16 [N, D], W_bf16 uint16 [V, D] (bf16 bit patterns),
    targets int32 [N]."""
    lib = _load()
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16)
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    a = np.ascontiguousarray(targets, dtype=np.int32)
    N, D = h.shape
    V, D2 = W.shape
    assert D == D2 and a.shape == (N,)
    if rows is None:
        r = None
        R = N
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < N))
        R = r.size
    logp = np.empty(R, dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    nt = nthreads or max(1, len(os.sched_getaffinity(0)))
    rc = lib.oracle_token_logprob(_ptr(h), _ptr(W), _ptr(a), None if r is None else _ptr(r), R,
                                  D, V, float(temperature), _ptr(logp), _ptr(lse), nt)
    if rc != 0:
        raise RuntimeError("oracle_token_logprob failed")
    return logp, lse


def token_logprob_f32w(h_bf16: np.ndarray, W_f32: np.ndarray, targets: np.ndarray,
                       rows=None, nthreads: int | None = None, temperature: float = 1.0):
    """token_logprob with fp32 weights W [V, D] (the FP32 LM head of LoongSage
    "Train-Inference Consistency" section 3): (logp, lse) float64."""
    lib = _load()
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16)
    W = np.ascontiguousarray(W_f32, dtype=np.float32)
    a = np.ascontiguousarray(targets, dtype=np.int32)
    N, D = h.shape
    V, D2 = W.shape
    assert D == D2 and a.shape == (N,)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    R = N if r is None else r.size
    if r is not None:
        assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < N))
    logp = np.empty(R, dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    nt = nthreads or max(1, len(os.sched_getaffinity(0)))
    rc = lib.oracle_token_logprob_f32w(_ptr(h), _ptr(W), _ptr(a), None if r is None else _ptr(r), R,
                                       D, V, float(temperature), _ptr(logp), _ptr(lse), nt)
    if rc != 0:
        raise RuntimeError("oracle_token_logprob_f32w failed")
    return logp, lse


def token_logprob_backward(h_bf16, W_bf16, targets, grad, temperature: float = 1.0, want_dz: bool = False):
    """Gradients of sum_t grad_t l_t with respect to h and W (l_t the token
    logprob at `temperature`): dict with dh [N, D], dW [V, D] (and dz [N, V]
    when want_dz), float64.  Cost N V D: small shapes only."""
    lib = _load()
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16)
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    a = np.ascontiguousarray(targets, dtype=np.int32)
    g = np.ascontiguousarray(grad, dtype=np.float32)
    N, D = h.shape
    V, D2 = W.shape
    assert D == D2 and a.shape == (N,) and g.shape == (N,)
    dh = np.empty((N, D), dtype=np.float64)
    dW = np.empty((V, D), dtype=np.float64)
    dz = np.empty((N, V), dtype=np.float64) if want_dz else None
    rc = lib.oracle_token_logprob_backward(_ptr(h), _ptr(W), _ptr(a), _ptr(g), N, D, V, float(temperature),
                                           _ptr(dh), _ptr(dW), None if dz is None else _ptr(dz))
    if rc != 0:
        raise ValueError("oracle_token_logprob_backward rejected its arguments")
    out = {"dh": dh, "dW": dW}
    if want_dz:
        out["dz"] = dz
    return out


def mismatch_stats(logp_train, logp_rollout, mask, seq_offsets, C: float = 2.0,
                   tau_seq: float = float("nan"), seq_estimator: int = 3, nthreads: int = 1):
    """dict with token_weight [N], seq_stats [S, 12], seq_flags [S], batch [20]
    (all float64 except seq_flags int32).  nthreads > 1 sums the sequences on
    that many threads; the arithmetic, and so every bit, is the same."""
    lib = _load()
    lt = np.ascontiguousarray(logp_train, dtype=np.float32)
    lr = np.ascontiguousarray(logp_rollout, dtype=np.float32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    off = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    N = lt.size
    S = off.size - 1
    assert lr.size == N and m.size == N and S >= 0
    w = np.empty(N, dtype=np.float64)
    seq = np.empty((S, len(SEQ_FIELDS)), dtype=np.float64)
    flags = np.empty(S, dtype=np.int32)
    batch = np.empty(len(BATCH_FIELDS), dtype=np.float64)
    rc = lib.oracle_mismatch_stats_threads(_ptr(lt), _ptr(lr), _ptr(m), _ptr(off), S, N, float(C),
                                           float(tau_seq), int(seq_estimator), _ptr(w), _ptr(seq),
                                           _ptr(flags), _ptr(batch), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_mismatch_stats rejected its arguments")
    return {"token_weight": w, "seq_stats": seq, "seq_flags": flags, "batch": batch}


def tis_ppo(logp_theta, logp_old, logp_rollout, advantages, mask, seq_offsets, eps_low: float = 0.2,
            eps_high: float = 0.2, C: float = 2.0):
    """TIS-weighted PPO clipped surrogate (VeXact summary eq. (2)-(3), TIS by
    r_corr truncated at C; HN page, clipped importance ratios).  dict with
    token_loss [N], token_grad [N] (d loss / d logp_theta), seq_loss [S],
    batch [9] (PPO_FIELDS), all float64."""
    lib = _load()
    arrs = [np.ascontiguousarray(x, dtype=np.float32) for x in (logp_theta, logp_old, logp_rollout, advantages)]
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    off = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    N = arrs[0].size
    S = off.size - 1
    assert all(x.size == N for x in arrs) and m.size == N and S >= 0
    loss = np.empty(N, dtype=np.float64)
    grad = np.empty(N, dtype=np.float64)
    seq = np.empty(S, dtype=np.float64)
    batch = np.empty(len(PPO_FIELDS), dtype=np.float64)
    rc = lib.oracle_tis_ppo(*[_ptr(x) for x in arrs], _ptr(m), _ptr(off), S, N, float(eps_low), float(eps_high),
                            float(C), _ptr(loss), _ptr(grad), _ptr(seq), _ptr(batch))
    if rc != 0:
        raise ValueError("oracle_tis_ppo rejected its arguments")
    return {"token_loss": loss, "token_grad": grad, "seq_loss": seq, "batch": batch}


def mismatch_monitor(logp_train, logp_rollout, mask, tau_tok: float):
    """Distribution monitor of delta = logp_train - logp_rollout over the used
    tokens (llm-infra-atlas section 7; VeXact tau_tok): dict with batch
    [7] (MONITOR_FIELDS, float64) and reject [N] uint8."""
    lib = _load()
    lt = np.ascontiguousarray(logp_train, dtype=np.float32)
    lr = np.ascontiguousarray(logp_rollout, dtype=np.float32)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    N = lt.size
    assert lr.size == N and m.size == N
    out = np.empty(len(MONITOR_FIELDS), dtype=np.float64)
    rej = np.empty(N, dtype=np.uint8)
    rc = lib.oracle_mismatch_monitor(_ptr(lt), _ptr(lr), _ptr(m), N, float(tau_tok), _ptr(out), _ptr(rej))
    if rc != 0:
        raise ValueError("oracle_mismatch_monitor rejected its arguments")
    return {"batch": out, "reject": rej}
