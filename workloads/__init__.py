"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the method itself (no logits, no
log-softmax, no mismatch statistics).  It only draws random numbers, rounds
fp32 draws to bf16, lays out packed sequences and masks, and adds noise to a
logprob vector handed in by the caller.  Every draw comes from
``numpy.random.default_rng(seed)`` (PCG64), so the same call gives the same
bytes on x86 and on Arm.

Workload shapes follow the pages' Qwen3-8B / Llama-3-8B / DeepSeek-V3 LM
heads (the final-hidden-state -> LM head -> log-softmax -> gather chain on
the icarus "RL: Training Inference Mismatch" page, "log p" section, and the
Qwen3-8B bf16 drift of Table 1 on the VeXact summary page).  No model
weights or datasets are used: shapes and value distributions only.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "CONFIGS", "HeadConfig", "bf16_round", "bf16_to_f32", "draw_head", "draw_targets",
    "draw_segments", "draw_mask", "draw_rollout", "draw_train_logprobs", "draw_h_rows",
]


# ----------------------------------------------------------------------------- bf16
def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    The VeXact/HN "Rounding depends on the order of additions" figure fixes the
    rounding rule this must follow: 1 + 2^-8 is a tie between 1 and 1 + 2^-7
    and goes to the even neighbour 1; tests pin that case.
    """
    f = np.array(x, dtype=np.float32, copy=True, order="C")
    shape = f.shape
    f = f.reshape(-1)
    u = f.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out.reshape(shape)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 (exact)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 24,
                 outlier_frac: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    """Draw N(0, std^2) fp32 values in row-major order, optionally scale an iid
    fraction of entries, round to bf16.  Drawn chunk by chunk from one stream,
    so the result does not depend on the chunk size."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if outlier_frac > 0.0:
            sel = rng.random(e - s, dtype=np.float32) < np.float32(outlier_frac)
            v[sel] *= np.float32(outlier_scale)
        out[s:e] = bf16_round(v)
    return out.reshape(shape)


# ----------------------------------------------------------------------------- configs
@dataclasses.dataclass(frozen=True)
class HeadConfig:
    name: str
    N: int
    D: int
    V: int
    h_std: float = 1.0
    w_std: float = 0.02
    h_outlier_frac: float = 0.0
    h_outlier_scale: float = 1.0
    seq_layout: str = "fixed"        # "fixed" (num_seqs x seq_len) or "lognormal"
    num_seqs: int = 1
    seq_len: int = 0
    len_median: float = 1024.0
    len_sigma: float = 0.5           # unstated on the pages; this is the reading used
    len_min: int = 128
    len_max: int = 4096
    prompt_len: int = 0              # first tokens of each sequence masked as prompt
    mask_drop: float = 0.0           # iid probability that a token is masked out
    rollout_std: float = 1e-3
    outlier_frac: float = 0.0        # iid fraction of rollout tokens shifted by +-outlier_shift
    outlier_shift: float = 0.0
    target_mode: str = "uniform"     # "uniform" or "top5mix"
    C: float = 2.0
    seed: int = 0


CONFIGS = {
    "tiny": HeadConfig("tiny", N=64, D=256, V=1024, num_seqs=1, seq_len=64, rollout_std=1e-3),
    "qwen3_8b": HeadConfig("qwen3_8b", N=8192, D=4096, V=151936, num_seqs=16, seq_len=512,
                           prompt_len=128, rollout_std=0.01),
    "llama3_8b": HeadConfig("llama3_8b", N=32768, D=4096, V=128256, seq_layout="lognormal",
                            mask_drop=0.3, rollout_std=0.02, outlier_frac=0.005, outlier_shift=1.0),
    "dsv3": HeadConfig("dsv3", N=16384, D=7168, V=129280, w_std=0.015, h_outlier_frac=0.01,
                       h_outlier_scale=20.0, num_seqs=32, seq_len=512, rollout_std=0.05,
                       target_mode="top5mix"),
}

# batch-invariance sweep: one W (seed 1), 512 probe rows (seed 1), batch sizes below
SWEEP = dict(D=4096, V=151936, probes=512, seed=1, batch_sizes=(1, 7, 512, 4096, 32768))


# ----------------------------------------------------------------------------- draws
def draw_head(cfg: HeadConfig, seed: int | None = None, N: int | None = None):
    """(h, W) as bf16 bit patterns: h [N, D], W [V, D], both row-major.

    W is drawn first from its own stream (seed), h from stream (seed + 1), so
    that W does not change when N changes.
    """
    seed = cfg.seed if seed is None else seed
    N = cfg.N if N is None else N
    W = _normal_bf16(np.random.default_rng([seed, 0]), (cfg.V, cfg.D), cfg.w_std)
    h = draw_h_rows(cfg, seed, N)
    return h, W


def draw_h_rows(cfg: HeadConfig, seed: int, N: int) -> np.ndarray:
    return _normal_bf16(np.random.default_rng([seed, 1]), (N, cfg.D), cfg.h_std,
                        outlier_frac=cfg.h_outlier_frac, outlier_scale=cfg.h_outlier_scale)


def draw_targets(cfg: HeadConfig, N: int, seed: int | None = None, top5: np.ndarray | None = None):
    """int32 [N] target ids.

    uniform: U[0, V).  top5mix: with probability 0.7 a uniform pick among the
    row's five highest logits (``top5`` [N, 5], supplied by the caller from a
    plain fp32 matmul; ties do not matter because this only shapes inputs),
    otherwise U[0, V).
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng([seed, 2])
    t = rng.integers(0, cfg.V, size=N, dtype=np.int64).astype(np.int32)
    if cfg.target_mode == "top5mix":
        if top5 is None:
            raise ValueError("top5mix targets need the rows' top-5 ids")
        pick = rng.random(N) < 0.7
        col = rng.integers(0, 5, size=N)
        t = np.where(pick, np.asarray(top5)[np.arange(N), col], t).astype(np.int32)
    return t


def draw_segments(cfg: HeadConfig, N: int | None = None, seed: int | None = None) -> np.ndarray:
    """int32 seq_offsets [S + 1] (CSR), off[0] = 0, off[S] = N."""
    N = cfg.N if N is None else N
    seed = cfg.seed if seed is None else seed
    if cfg.seq_layout == "fixed":
        S = cfg.num_seqs
        if S * cfg.seq_len != N:
            L = max(1, N // S)
            lens = [L] * (S - 1) + [N - L * (S - 1)]
        else:
            lens = [cfg.seq_len] * S
    else:
        rng = np.random.default_rng([seed, 3])
        lens, tot = [], 0
        while tot < N:
            L = int(round(math.exp(rng.normal(math.log(cfg.len_median), cfg.len_sigma))))
            L = min(max(L, cfg.len_min), cfg.len_max)
            L = min(L, N - tot)   # the last one is truncated so that the sum is N
            lens.append(L)
            tot += L
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    return off.astype(np.int32)


def draw_mask(cfg: HeadConfig, seq_offsets: np.ndarray, seed: int | None = None) -> np.ndarray:
    """uint8 [N] response mask (1 = token counts in the statistics)."""
    seed = cfg.seed if seed is None else seed
    off = np.asarray(seq_offsets, dtype=np.int64)
    N = int(off[-1])
    m = np.ones(N, dtype=np.uint8)
    if cfg.prompt_len > 0:
        for s in range(len(off) - 1):
            m[off[s]: min(off[s + 1], off[s] + cfg.prompt_len)] = 0
    if cfg.mask_drop > 0.0:
        rng = np.random.default_rng([seed, 4])
        m[rng.random(N) < cfg.mask_drop] = 0
    return m


def draw_rollout(cfg: HeadConfig, logp_train: np.ndarray, seed: int | None = None) -> np.ndarray:
    """fp32 rollout logprobs = train logprobs + N(0, rollout_std^2) (+ iid
    outlier tokens shifted by +-outlier_shift with a fair sign)."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng([seed, 5])
    lt = np.asarray(logp_train)
    noise = rng.normal(0.0, cfg.rollout_std, size=lt.shape)
    if cfg.outlier_frac > 0.0:
        hit = rng.random(lt.shape) < cfg.outlier_frac
        u = rng.random(lt.shape)
        noise[hit] += np.where(u[hit] < 0.5, -1.0, 1.0) * cfg.outlier_shift
        del u, hit
    noise += lt
    return noise.astype(np.float32)


def draw_train_logprobs(N: int, seed: int) -> np.ndarray:
    """Stand-in trainer logprobs for tests of the mismatch pass alone: fp32,
    <= 0, most mass near 0 with a long tail (a Gamma(0.6, 3) magnitude)."""
    rng = np.random.default_rng([seed, 6])
    return (-rng.gamma(0.6, 3.0, size=N)).astype(np.float32)


def draw_policy_update(logp_old: np.ndarray, std: float, seed: int) -> np.ndarray:
    """Stand-in current-policy logprobs for the PPO surrogate: fp32
    logp_old + N(0, std^2), the drift of a few optimiser steps since the
    rollout policy's snapshot."""
    rng = np.random.default_rng([seed, 7])
    lo = np.asarray(logp_old, dtype=np.float64)
    return (lo + rng.normal(0.0, std, size=lo.shape)).astype(np.float32)


def draw_advantages(seq_offsets: np.ndarray, seed: int) -> np.ndarray:
    """fp32 [N] advantages, one N(0, 1) value per sequence broadcast to its
    tokens (an outcome reward normalised over its group, as in GRPO)."""
    off = np.asarray(seq_offsets, dtype=np.int64)
    rng = np.random.default_rng([seed, 8])
    per_seq = rng.standard_normal(len(off) - 1)
    return np.repeat(per_seq, np.diff(off)).astype(np.float32)


def draw_ppo_inputs(N: int, seed: int, update_std: float = 0.1):
    """Packed inputs of the TIS-weighted PPO surrogate, N tokens: Llama-like
    segments (lognormal lengths, median 1024, clipped to [128, 4096]), 30% of
    tokens masked out, trainer logprobs l_old as in ``draw_train_logprobs``,
    rollout logprobs l_old + N(0, 0.02^2) with 0.5% outliers shifted by +-1
    (l_old has the law of ``draw_train_logprobs``, drawn in fp32 for speed),
    current-policy logprobs l_old + N(0, update_std^2), per-sequence N(0, 1)
    advantages.  Returns (seq_offsets, mask, l_theta, l_old, l_rollout, adv)."""
    cfg = HeadConfig("ppo", N=N, D=8, V=8, seq_layout="lognormal", mask_drop=0.3, rollout_std=0.02,
                     outlier_frac=0.005, outlier_shift=1.0, seed=seed)
    off = draw_segments(cfg)
    mask = draw_mask(cfg, off)
    rng = np.random.default_rng([seed, 9])
    l_old = rng.standard_gamma(0.6, size=N, dtype=np.float32)
    l_old *= np.float32(-3.0)
    l_ro = draw_rollout(cfg, l_old)
    l_th = draw_policy_update(l_old, update_std, seed)
    adv = draw_advantages(off, seed)
    return off, mask, l_th, l_old, l_ro, adv


def draw_weight_f32(cfg: HeadConfig, seed: int | None = None, chunk: int = 1 << 24) -> np.ndarray:
    """fp32 W [V, D] ~ N(0, w_std^2), not rounded to bf16: the weights of an
    FP32 LM head (own stream, so the bf16 W of the same config is unchanged)."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng([seed, 10])
    W = np.empty(cfg.V * cfg.D, dtype=np.float32)
    for s in range(0, W.size, chunk):
        n = min(chunk, W.size - s)
        W[s:s + n] = rng.standard_normal(n, dtype=np.float32) * np.float32(cfg.w_std)
    return W.reshape(cfg.V, cfg.D)
