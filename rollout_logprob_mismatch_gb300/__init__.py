"""GB300 (sm_103a) fused selected-token logprob and train/rollout mismatch statistics.

A thin ctypes binding over ``libtim.so`` (C ABI in ``include/tim.h``).  The
functions named like the C entry points (``tim_token_logprob``,
``tim_mismatch_stats``, ``tim_check``) take raw device pointers and sizes;
``token_logprob`` and ``mismatch_stats`` take torch CUDA tensors and only
marshal them.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU fallback: if ``libtim.so`` is missing, importing the
binding succeeds but every call raises ``TimError``.

Method: the trainer recomputes l_t = log softmax(h_t W^T)[a_t] from its final
hidden states (icarus "RL: Training Inference Mismatch", section "log p") and
compares it with the rollout engine's logprob through delta = l_train -
l_rollout, r = e^delta, the k1/k2/k3 KL estimators, the truncated importance
weight min(r, C) and masked per-sequence / per-batch means with a sequence
rejection flag (VeXact summary, eq. (1) and "Algorithmic TIM Compensation";
LoongSage "Train-Inference Consistency", sections 4-5).  ``tis_ppo`` gives the
clipped PPO surrogate weighted by the truncated importance weight, its
gradient and masked means (VeXact summary eq. (2)-(3)).
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

__all__ = [
    "TimError", "SEQ_FIELDS", "BATCH_FIELDS", "PPO_FIELDS", "MONITOR_FIELDS", "tim_mismatch_out", "tim_ppo_out", "lib_path", "load",
    "tim_token_logprob", "tim_token_logprob_temperature", "tim_token_logprob_noalloc", "tim_mismatch_stats",
    "tim_mismatch_fold", "SEQ_RECORD_WORDS", "mismatch_fold",
    "tim_tis_ppo", "tim_mismatch_monitor", "tim_split_weight_bytes", "tim_split_weight_fp32",
    "tim_token_logprob_fp32_head", "tim_token_logprob_backward", "tim_selftest_wait_timeout", "tim_check", "tim_last_error", "tim_version",
    "tim_debug_violation", "tim_debug_build", "load_debug", "checked", "CHECKS",
    "token_logprob", "token_logprob_backward", "split_weight_fp32", "token_logprob_fp32_head", "mismatch_stats", "mismatch_monitor", "tis_ppo", "check",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtim.so")
_DEBUG_LIB_PATH = os.path.join(_PKG, "libtim_debug.so")

TIM_OK = 0
TIM_ERR_INVALID_ARG = -1
TIM_ERR_UNSUPPORTED_DEVICE = -2
TIM_ERR_CUDA = -3
TIM_ERR_TIMEOUT = -4
TIM_ERR_BAD_INPUT = -5
NOALLOC_SCRATCH_BYTES = 16 << 20   # TIM_NOALLOC_SCRATCH_BYTES in include/tim.h

# TIM_CHECK_* of include/tim.h: what the checked build (libtim_debug.so) records
CHECKS = {0: "none", 1: "target", 2: "mask", 3: "logit", 4: "backward_input", 5: "advantage",
          6: "tma_coord", 7: "store", 8: "unit", 9: "bulk"}

SEQ_RECORD_WORDS = 16   # TIM_SEQ_RECORD_WORDS
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


class TimError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("tim error %d: %s" % (code, msg))
        self.code = code


class tim_mismatch_out(ctypes.Structure):
    """Mirror of the C struct tim_mismatch_out (host struct of device pointers)."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_tokens", ctypes.c_int64),
        ("tau_seq", ctypes.c_float),
        ("seq_estimator", ctypes.c_int32),
        ("token_weight", ctypes.c_void_p),
        ("seq_stats", ctypes.c_void_p),
        ("seq_flags", ctypes.c_void_p),
        ("batch_stats", ctypes.c_void_p),
        ("seq_records", ctypes.c_void_p),
    ]


class tim_ppo_out(ctypes.Structure):
    """Mirror of the C struct tim_ppo_out (host struct of device pointers)."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_tokens", ctypes.c_int64),
        ("token_loss", ctypes.c_void_p),
        ("token_grad", ctypes.c_void_p),
        ("seq_loss", ctypes.c_void_p),
        ("batch_stats", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None          # the library calls go to (libtim.so, or libtim_debug.so inside `checked()`)
_release = None
_debug = None


def lib_path() -> str:
    return _LIB_PATH


def _open(path: str, what: str):
    if not os.path.exists(path):
        raise TimError(TIM_ERR_CUDA, "%s is not built (%s); run "
                       "`python -m rollout_logprob_mismatch_gb300.build`" % (what, path))
    lib = ctypes.CDLL(path)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.tim_token_logprob.argtypes = [P, P, P, I64, I64, I64, P, P, P]
    lib.tim_token_logprob.restype = ctypes.c_int
    lib.tim_token_logprob_temperature.argtypes = [P, P, P, I64, I64, I64, ctypes.c_float, P, P, P]
    lib.tim_token_logprob_temperature.restype = ctypes.c_int
    lib.tim_token_logprob_noalloc.argtypes = [P, P, P, I64, I64, I64, P, P, P]
    lib.tim_token_logprob_noalloc.restype = ctypes.c_int
    lib.tim_mismatch_stats.argtypes = [P, P, P, P, ctypes.c_float, ctypes.POINTER(tim_mismatch_out), P]
    lib.tim_mismatch_stats.restype = ctypes.c_int
    lib.tim_mismatch_fold.argtypes = [P, ctypes.c_int32, P, P]
    lib.tim_mismatch_fold.restype = ctypes.c_int
    F = ctypes.c_float
    lib.tim_tis_ppo.argtypes = [P, P, P, P, P, P, F, F, F, ctypes.POINTER(tim_ppo_out), P]
    lib.tim_tis_ppo.restype = ctypes.c_int
    lib.tim_split_weight_bytes.argtypes = [I64, I64]
    lib.tim_split_weight_bytes.restype = ctypes.c_int64
    lib.tim_split_weight_fp32.argtypes = [P, I64, I64, P, P]
    lib.tim_split_weight_fp32.restype = ctypes.c_int
    lib.tim_token_logprob_fp32_head.argtypes = [P, P, P, I64, I64, I64, ctypes.c_float, P, P, P]
    lib.tim_token_logprob_fp32_head.restype = ctypes.c_int
    lib.tim_token_logprob_backward.argtypes = [P, P, P, P, P, I64, I64, I64, ctypes.c_float, P, P,
                                               ctypes.c_int, P]
    lib.tim_token_logprob_backward.restype = ctypes.c_int
    lib.tim_mismatch_monitor.argtypes = [P, P, P, I64, F, P, P, P]
    lib.tim_mismatch_monitor.restype = ctypes.c_int
    lib.tim_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.tim_selftest_wait_timeout.restype = ctypes.c_int
    lib.tim_check.argtypes = [P]
    lib.tim_check.restype = ctypes.c_int
    lib.tim_debug_violation.argtypes = [ctypes.POINTER(ctypes.c_int64), P]
    lib.tim_debug_violation.restype = ctypes.c_int
    lib.tim_debug_build.argtypes = []
    lib.tim_debug_build.restype = ctypes.c_int
    lib.tim_last_error.argtypes = []
    lib.tim_last_error.restype = ctypes.c_char_p
    lib.tim_version.argtypes = []
    lib.tim_version.restype = ctypes.c_int
    return lib


def load():
    """The library calls go to: libtim.so (libtim_debug.so inside `checked()`);
    raises TimError when it has not been built."""
    global _lib, _release
    with _lock:
        if _lib is None:
            if _release is None:
                _release = _open(_LIB_PATH, "libtim.so")
            _lib = _release
    return _lib


def load_debug():
    """libtim_debug.so: the same library built with TIM_DEBUG (its kernels also
    check indices, TMA coordinates and input contracts; see include/tim.h)."""
    global _debug
    with _lock:
        if _debug is None:
            _debug = _open(_DEBUG_LIB_PATH, "libtim_debug.so")
    return _debug


@contextlib.contextmanager
def checked():
    """Within the block every call of this module goes to libtim_debug.so
    (one thread at a time); tim_debug_violation() then reports the first
    violation its kernels found."""
    global _lib
    dbg = load_debug()
    prev = load()
    _lib = dbg
    try:
        yield dbg
    finally:
        _lib = prev


# ----------------------------------------------------------------------------- raw C ABI
def tim_token_logprob(h, W, targets, N, D, V, out_logp, out_lse, stream) -> int:
    """C ABI call with integer device addresses; returns the tim_status code."""
    return load().tim_token_logprob(h, W, targets, N, D, V, out_logp, out_lse, stream)


def tim_token_logprob_temperature(h, W, targets, N, D, V, temperature, out_logp, out_lse, stream) -> int:
    """C ABI call of the token logprob at a sampling temperature; returns the tim_status code."""
    return load().tim_token_logprob_temperature(h, W, targets, N, D, V, float(temperature), out_logp,
                                                out_lse, stream)


def tim_token_logprob_noalloc(h, W, targets, N, D, V, out_logp, out_lse, stream) -> int:
    """C ABI call of the variant that allocates nothing (its scratch is a fixed
    NOALLOC_SCRATCH_BYTES device array of the library); returns the tim_status code."""
    return load().tim_token_logprob_noalloc(h, W, targets, N, D, V, out_logp, out_lse, stream)


def tim_mismatch_stats(logp_train, logp_rollout, mask, seq_offsets, C, out: tim_mismatch_out,
                       stream) -> int:
    return load().tim_mismatch_stats(logp_train, logp_rollout, mask, seq_offsets, float(C),
                                     ctypes.byref(out), stream)


def tim_mismatch_fold(seq_records, num_seqs, batch_stats, stream) -> int:
    return load().tim_mismatch_fold(seq_records, int(num_seqs), batch_stats, stream)


def tim_tis_ppo(logp_theta, logp_old, logp_rollout, advantages, mask, seq_offsets, eps_low, eps_high, C,
                out: tim_ppo_out, stream) -> int:
    return load().tim_tis_ppo(logp_theta, logp_old, logp_rollout, advantages, mask, seq_offsets,
                              float(eps_low), float(eps_high), float(C), ctypes.byref(out), stream)


def tim_token_logprob_backward(h, W, targets, grad_logp, lse, N, D, V, temperature, dh, dW, accumulate_dW,
                               stream) -> int:
    return load().tim_token_logprob_backward(h, W, targets, grad_logp, lse, N, D, V, float(temperature), dh, dW,
                                             int(accumulate_dW), stream)


def tim_split_weight_bytes(V, D) -> int:
    return load().tim_split_weight_bytes(V, D)


def tim_split_weight_fp32(W, V, D, W_split, stream) -> int:
    return load().tim_split_weight_fp32(W, V, D, W_split, stream)


def tim_token_logprob_fp32_head(h, W_split, targets, N, D, V, temperature, out_logp, out_lse, stream) -> int:
    return load().tim_token_logprob_fp32_head(h, W_split, targets, N, D, V, float(temperature), out_logp,
                                              out_lse, stream)


def tim_mismatch_monitor(logp_train, logp_rollout, mask, N, tau_tok, token_reject, out, stream) -> int:
    return load().tim_mismatch_monitor(logp_train, logp_rollout, mask, N, float(tau_tok), token_reject, out,
                                       stream)


def tim_selftest_wait_timeout(budget_us, stream) -> int:
    """C ABI: a kernel waits on a barrier nothing arrives on, for budget_us
    microseconds, and records TIM_ERR_TIMEOUT (no fault; see include/tim.h)."""
    return load().tim_selftest_wait_timeout(budget_us, stream)


def tim_check(stream) -> int:
    return load().tim_check(stream)


def tim_last_error() -> str:
    return load().tim_last_error().decode(errors="replace")


def tim_version() -> int:
    return load().tim_version()


def tim_debug_build() -> int:
    """1 when calls go to the checked build (libtim_debug.so), else 0."""
    return load().tim_debug_build()


def tim_debug_violation(stream=None):
    """The first violation the checked build's kernels recorded since the last
    call, as (check name, index, value bits), cleared on read; ("none", 0, 0)
    if none (always so in libtim.so).  Synchronises the stream."""
    import torch
    out = (ctypes.c_int64 * 4)()
    s = 0 if stream is None and not torch.cuda.is_available() else _stream_handle(stream, None)
    _raise_if(load().tim_debug_violation(out, s))
    return CHECKS.get(int(out[0]), str(int(out[0]))), int(out[1]), int(out[2])


def _raise_if(rc: int):
    if rc != TIM_OK:
        raise TimError(rc, tim_last_error())


# ----------------------------------------------------------------------------- torch wrappers
def _stream_handle(stream, device):
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _need(t, name, dtype, ndim, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must be %d-D" % (name, ndim))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _need_out(t, name, dtype, shape, device):
    """An output buffer the kernels write in full: exact dtype, shape, device,
    contiguous (a shorter buffer would be written past its end)."""
    _need(t, name, dtype, len(shape), device)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def token_logprob(h, W, targets, out_logp=None, out_lse=None, stream=None, temperature: float = 1.0):
    """(logp [N] fp32, lse [N] fp32) for bf16 h [N, D], bf16 W [V, D], int32 targets [N]:
    log softmax(h W^T / temperature) at the targets (temperature 1: raw logits)."""
    import torch
    _need(h, "h", torch.bfloat16, 2)
    dev = h.device
    _need(W, "W", torch.bfloat16, 2, dev)
    _need(targets, "targets", torch.int32, 1, dev)
    N, D = h.shape
    V = W.shape[0]
    if W.shape[1] != D or targets.shape[0] != N:
        raise ValueError("shape mismatch: h %s, W %s, targets %s" % (tuple(h.shape), tuple(W.shape),
                                                                       tuple(targets.shape)))
    if out_logp is None:
        out_logp = torch.empty(N, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(N, dtype=torch.float32, device=dev)
    _need_out(out_logp, "out_logp", torch.float32, (N,), dev)
    _need_out(out_lse, "out_lse", torch.float32, (N,), dev)
    with torch.cuda.device(dev):
        if temperature == 1.0:
            rc = tim_token_logprob(h.data_ptr(), W.data_ptr(), targets.data_ptr(), N, D, V,
                                   out_logp.data_ptr(), out_lse.data_ptr(), _stream_handle(stream, dev))
        else:
            rc = tim_token_logprob_temperature(h.data_ptr(), W.data_ptr(), targets.data_ptr(), N, D, V,
                                               temperature, out_logp.data_ptr(), out_lse.data_ptr(),
                                               _stream_handle(stream, dev))
    _raise_if(rc)
    return out_logp, out_lse


def token_logprob_backward(h, W, targets, grad_logp, lse, temperature: float = 1.0, dh=None, dW=None,
                           accumulate_dW: bool = False, stream=None):
    """(dh fp32 [N, D], dW fp32 [V, D]): gradients of sum_t grad_logp_t l_t
    for bf16 h [N, D], bf16 W [V, D], int32 targets, the forward's lse [N]
    at the same temperature.  With accumulate_dW the gradient is added to dW."""
    import torch
    _need(h, "h", torch.bfloat16, 2)
    dev = h.device
    _need(W, "W", torch.bfloat16, 2, dev)
    _need(targets, "targets", torch.int32, 1, dev)
    _need(grad_logp, "grad_logp", torch.float32, 1, dev)
    _need(lse, "lse", torch.float32, 1, dev)
    N, D = h.shape
    V = W.shape[0]
    if W.shape[1] != D or any(t.shape[0] != N for t in (targets, grad_logp, lse)):
        raise ValueError("shape mismatch")
    if dh is None:
        dh = torch.empty((N, D), dtype=torch.float32, device=dev)
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs dW")
        dW = torch.empty((V, D), dtype=torch.float32, device=dev)
    _need_out(dh, "dh", torch.float32, (N, D), dev)
    _need_out(dW, "dW", torch.float32, (V, D), dev)
    with torch.cuda.device(dev):
        rc = tim_token_logprob_backward(h.data_ptr(), W.data_ptr(), targets.data_ptr(), grad_logp.data_ptr(),
                                        lse.data_ptr(), N, D, V, temperature, dh.data_ptr(), dW.data_ptr(),
                                        accumulate_dW, _stream_handle(stream, dev))
    _raise_if(rc)
    return dh, dW


def split_weight_fp32(W, out=None, stream=None):
    """fp32 W [V, D] -> its three bf16 parts, a bf16 tensor [V, 3 * Dp]
    (Dp = D rounded up to 64): the operand of token_logprob_fp32_head."""
    import torch
    _need(W, "W", torch.float32, 2)
    dev = W.device
    V, D = W.shape
    nbytes = tim_split_weight_bytes(V, D)
    if nbytes < 0:
        raise ValueError("W shape %s out of range" % (tuple(W.shape),))
    cols = nbytes // (2 * V)
    if out is None:
        out = torch.empty((V, cols), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 2, dev)
    if tuple(out.shape) != (V, cols):
        raise ValueError("out must be [%d, %d]" % (V, cols))
    with torch.cuda.device(dev):
        rc = tim_split_weight_fp32(W.data_ptr(), V, D, out.data_ptr(), _stream_handle(stream, dev))
    _raise_if(rc)
    return out


def token_logprob_fp32_head(h, W_split, targets, out_logp=None, out_lse=None, stream=None,
                            temperature: float = 1.0):
    """(logp, lse) fp32 [N] of log softmax(h W^T / temperature) at the targets
    with fp32 weights W, given as split_weight_fp32(W); h bf16 [N, D]."""
    import torch
    _need(h, "h", torch.bfloat16, 2)
    dev = h.device
    _need(W_split, "W_split", torch.bfloat16, 2, dev)
    _need(targets, "targets", torch.int32, 1, dev)
    N, D = h.shape
    V = W_split.shape[0]
    if tim_split_weight_bytes(V, D) != W_split.numel() * 2 or targets.shape[0] != N:
        raise ValueError("shape mismatch: h %s, W_split %s, targets %s"
                         % (tuple(h.shape), tuple(W_split.shape), tuple(targets.shape)))
    if out_logp is None:
        out_logp = torch.empty(N, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(N, dtype=torch.float32, device=dev)
    _need_out(out_logp, "out_logp", torch.float32, (N,), dev)
    _need_out(out_lse, "out_lse", torch.float32, (N,), dev)
    with torch.cuda.device(dev):
        rc = tim_token_logprob_fp32_head(h.data_ptr(), W_split.data_ptr(), targets.data_ptr(), N, D, V,
                                         temperature, out_logp.data_ptr(), out_lse.data_ptr(),
                                         _stream_handle(stream, dev))
    _raise_if(rc)
    return out_logp, out_lse


def mismatch_stats(logp_train, logp_rollout, mask, seq_offsets, C: float = 2.0,
                   tau_seq: float = math.nan, seq_estimator: int = 3, token_weight: bool = False,
                   stream=None, out=None, seq_records: bool = False):
    """Mismatch statistics of packed sequences.

    logp_train, logp_rollout fp32 [N]; mask bool/uint8 [N]; seq_offsets int32 [S + 1].
    Returns a dict: seq_stats fp32 [S, 12] (SEQ_FIELDS), seq_flags int32 [S],
    batch fp64 [20] (BATCH_FIELDS), token_weight fp32 [N] or None, and with
    seq_records=True seq_records int32 [S, SEQ_RECORD_WORDS] (the records the
    batch record is folded from; see mismatch_fold).
    """
    import torch
    _need(logp_train, "logp_train", torch.float32, 1)
    dev = logp_train.device
    _need(logp_rollout, "logp_rollout", torch.float32, 1, dev)
    _need(mask, "mask", (torch.uint8, torch.bool), 1, dev)
    _need(seq_offsets, "seq_offsets", torch.int32, 1, dev)
    N = logp_train.shape[0]
    S = seq_offsets.shape[0] - 1
    if logp_rollout.shape[0] != N or mask.shape[0] != N or S < 0:
        raise ValueError("shape mismatch")
    if out is None:
        out = {
            "seq_stats": torch.empty((S, len(SEQ_FIELDS)), dtype=torch.float32, device=dev),
            "seq_flags": torch.empty(S, dtype=torch.int32, device=dev),
            "batch": torch.empty(len(BATCH_FIELDS), dtype=torch.float64, device=dev),
            "token_weight": torch.empty(N, dtype=torch.float32, device=dev) if token_weight else None,
            "seq_records": torch.empty((S, SEQ_RECORD_WORDS), dtype=torch.int32, device=dev)
            if seq_records else None,
        }
    _need_out(out["seq_stats"], "seq_stats", torch.float32, (S, len(SEQ_FIELDS)), dev)
    _need_out(out["seq_flags"], "seq_flags", torch.int32, (S,), dev)
    _need_out(out["batch"], "batch", torch.float64, (len(BATCH_FIELDS),), dev)
    if out.get("token_weight") is not None:
        _need_out(out["token_weight"], "token_weight", torch.float32, (N,), dev)
    if out.get("seq_records") is not None:
        _need_out(out["seq_records"], "seq_records", torch.int32, (S, SEQ_RECORD_WORDS), dev)
        if out["seq_records"].data_ptr() % 16:
            raise ValueError("seq_records must be 16-byte aligned")
    d = tim_mismatch_out()
    d.num_seqs = S
    d.num_tokens = N
    d.tau_seq = float(tau_seq)
    d.seq_estimator = int(seq_estimator)
    d.token_weight = out["token_weight"].data_ptr() if out.get("token_weight") is not None else None
    d.seq_stats = out["seq_stats"].data_ptr()
    d.seq_flags = out["seq_flags"].data_ptr()
    d.batch_stats = out["batch"].data_ptr()
    d.seq_records = out["seq_records"].data_ptr() if out.get("seq_records") is not None else None
    with torch.cuda.device(dev):
        rc = tim_mismatch_stats(logp_train.data_ptr(), logp_rollout.data_ptr(), mask.data_ptr(),
                                seq_offsets.data_ptr(), C, d, _stream_handle(stream, dev))
    _raise_if(rc)
    return out


def mismatch_fold(seq_records, out=None, stream=None):
    """The batch record (fp64 [20], BATCH_FIELDS) of a batch scored in parts:
    the parts' seq_records (int32 [S_part, SEQ_RECORD_WORDS] each, from
    mismatch_stats(..., seq_records=True)) concatenated in the batch's sequence
    order.  Bit-identical to mismatch_stats over the whole batch."""
    import torch
    _need(seq_records, "seq_records", torch.int32, 2)
    dev = seq_records.device
    if seq_records.shape[1] != SEQ_RECORD_WORDS:
        raise ValueError("seq_records must have %d columns" % SEQ_RECORD_WORDS)
    if seq_records.data_ptr() % 16:
        raise ValueError("seq_records must be 16-byte aligned")
    if out is None:
        out = torch.empty(len(BATCH_FIELDS), dtype=torch.float64, device=dev)
    _need_out(out, "out", torch.float64, (len(BATCH_FIELDS),), dev)
    with torch.cuda.device(dev):
        rc = tim_mismatch_fold(seq_records.data_ptr(), seq_records.shape[0], out.data_ptr(),
                               _stream_handle(stream, dev))
    _raise_if(rc)
    return out


def mismatch_monitor(logp_train, logp_rollout, mask, tau_tok: float, token_reject: bool = True, stream=None,
                     out=None):
    """Mismatch monitor over the used tokens: batch fp64 [7] (MONITOR_FIELDS:
    n_used, p95 |delta|, ratio quantiles 0.01 / 0.5 / 0.99, n_extreme,
    frac_extreme) and token_reject uint8 [N] (None unless requested)."""
    import torch
    _need(logp_train, "logp_train", torch.float32, 1)
    dev = logp_train.device
    _need(logp_rollout, "logp_rollout", torch.float32, 1, dev)
    _need(mask, "mask", (torch.uint8, torch.bool), 1, dev)
    N = logp_train.shape[0]
    if logp_rollout.shape[0] != N or mask.shape[0] != N:
        raise ValueError("shape mismatch")
    if out is None:
        out = {"batch": torch.empty(len(MONITOR_FIELDS), dtype=torch.float64, device=dev),
               "token_reject": torch.empty(N, dtype=torch.uint8, device=dev) if token_reject else None}
    _need_out(out["batch"], "batch", torch.float64, (len(MONITOR_FIELDS),), dev)
    rej = out.get("token_reject")
    if rej is not None:
        _need_out(rej, "token_reject", torch.uint8, (N,), dev)
    with torch.cuda.device(dev):
        rc = tim_mismatch_monitor(logp_train.data_ptr(), logp_rollout.data_ptr(), mask.data_ptr(), N, tau_tok,
                                  None if rej is None else rej.data_ptr(), out["batch"].data_ptr(),
                                  _stream_handle(stream, dev))
    _raise_if(rc)
    return out


def tis_ppo(logp_theta, logp_old, logp_rollout, advantages, mask, seq_offsets, eps_low: float = 0.2,
            eps_high: float = 0.2, C: float = 2.0, token_outputs: bool = True, stream=None, out=None):
    """TIS-weighted PPO clipped surrogate of packed sequences.

    logp_theta, logp_old, logp_rollout, advantages fp32 [N]; mask bool/uint8 [N];
    seq_offsets int32 [S + 1].  Returns a dict: token_loss, token_grad fp32 [N]
    (None unless token_outputs), seq_loss fp32 [S], batch fp64 [9] (PPO_FIELDS).
    """
    import torch
    _need(logp_theta, "logp_theta", torch.float32, 1)
    dev = logp_theta.device
    for name, t in (("logp_old", logp_old), ("logp_rollout", logp_rollout), ("advantages", advantages)):
        _need(t, name, torch.float32, 1, dev)
    _need(mask, "mask", (torch.uint8, torch.bool), 1, dev)
    _need(seq_offsets, "seq_offsets", torch.int32, 1, dev)
    N = logp_theta.shape[0]
    S = seq_offsets.shape[0] - 1
    if any(t.shape[0] != N for t in (logp_old, logp_rollout, advantages, mask)) or S < 0:
        raise ValueError("shape mismatch")
    if out is None:
        out = {
            "token_loss": torch.empty(N, dtype=torch.float32, device=dev) if token_outputs else None,
            "token_grad": torch.empty(N, dtype=torch.float32, device=dev) if token_outputs else None,
            "seq_loss": torch.empty(S, dtype=torch.float32, device=dev),
            "batch": torch.empty(len(PPO_FIELDS), dtype=torch.float64, device=dev),
        }
    for name in ("token_loss", "token_grad"):
        if out.get(name) is not None:
            _need_out(out[name], name, torch.float32, (N,), dev)
    _need_out(out["seq_loss"], "seq_loss", torch.float32, (S,), dev)
    _need_out(out["batch"], "batch", torch.float64, (len(PPO_FIELDS),), dev)
    d = tim_ppo_out()
    d.num_seqs = S
    d.num_tokens = N
    d.token_loss = out["token_loss"].data_ptr() if out.get("token_loss") is not None else None
    d.token_grad = out["token_grad"].data_ptr() if out.get("token_grad") is not None else None
    d.seq_loss = out["seq_loss"].data_ptr()
    d.batch_stats = out["batch"].data_ptr()
    with torch.cuda.device(dev):
        rc = tim_tis_ppo(logp_theta.data_ptr(), logp_old.data_ptr(), logp_rollout.data_ptr(),
                         advantages.data_ptr(), mask.data_ptr(), seq_offsets.data_ptr(), eps_low, eps_high, C,
                         d, _stream_handle(stream, dev))
    _raise_if(rc)
    return out


def check(stream=None, device=None):
    """Synchronises the stream and raises TimError if a kernel recorded a status."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _raise_if(tim_check(_stream_handle(stream, dev)))
