"""Batch-invariance sweep of tim_token_logprob (llm-infra-atlas
"训推一致性与 determinism", section 1.2: a request's result must not depend on
which other requests share its batch).

One Qwen3-8B-shaped head (D = 4096, V = 151936, seed 1) and 512 fixed probe
rows (seed 1).  The probes run alone (N = 1), one per batch of 7 among 6
random rows, all together (N = 512), and scattered among random rows at
N = 4096 and N = 32768.  Every probe's logp and lse must have the same bits
everywhere and across three repeats; a sample of probes is also checked
against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import LOGP_ATOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import rollout_logprob_mismatch_gb300 as tim  # noqa: E402

SW = wl.SWEEP


@pytest.fixture(scope="module")
def head():
    cfg = wl.HeadConfig("sweep", N=SW["probes"], D=SW["D"], V=SW["V"])
    h, W = wl.draw_head(cfg, seed=SW["seed"])
    a = wl.draw_targets(cfg, SW["probes"], seed=SW["seed"])
    hd = torch.from_numpy(h.view(np.int16)).cuda().view(torch.bfloat16)
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    return cfg, h, W, a, hd, Wd, torch.from_numpy(a).cuda()


def _batch(hd, ad, Wd, N, probe_idx, pos, seed, cfg):
    """A batch of N rows with probe rows probe_idx at positions pos, the other
    rows random (seed)."""
    fill = wl.draw_h_rows(cfg, seed, N)
    hb = torch.from_numpy(fill.view(np.int16)).cuda().view(torch.bfloat16)
    ab = torch.from_numpy(np.random.default_rng(seed).integers(0, cfg.V, N).astype(np.int32)).cuda()
    p = torch.from_numpy(np.asarray(probe_idx)).cuda().long()
    q = torch.from_numpy(np.asarray(pos)).cuda().long()
    hb[q] = hd[p]
    ab[q] = ad[p]
    lp, lse = tim.token_logprob(hb, Wd, ab)
    return lp[q], lse[q]


def test_probe_bits_identical_across_batch_sizes(head):
    cfg, h, W, a, hd, Wd, ad = head
    P = SW["probes"]
    results = {}
    for rep in range(3):
        # N = 1
        lp1 = torch.empty(P, device="cuda")
        lse1 = torch.empty(P, device="cuda")
        for i in range(P):
            lp, lse = tim.token_logprob(hd[i:i + 1], Wd, ad[i:i + 1])
            lp1[i], lse1[i] = lp[0], lse[0]
        results[(1, rep)] = (lp1, lse1)
        # N = 7: one probe per batch at a random position among 6 random rows
        lp7 = torch.empty(P, device="cuda")
        lse7 = torch.empty(P, device="cuda")
        rng = np.random.default_rng(1000 + rep)
        for i in range(P):
            lp, lse = _batch(hd, ad, Wd, 7, [i], [int(rng.integers(0, 7))], 2000 + i, cfg)
            lp7[i], lse7[i] = lp[0], lse[0]
        results[(7, rep)] = (lp7, lse7)
        # N = 512: the probes alone, shuffled
        perm = np.random.default_rng(3000 + rep).permutation(P)
        lp, lse = tim.token_logprob(hd[torch.from_numpy(perm).cuda()], Wd, ad[torch.from_numpy(perm).cuda()])
        inv = np.argsort(perm)
        results[(512, rep)] = (lp[torch.from_numpy(inv).cuda()], lse[torch.from_numpy(inv).cuda()])
        # N = 4096 and 32768: probes scattered among random rows
        for N in (4096, 32768):
            pos = np.random.default_rng(100 + N + rep).choice(N, size=P, replace=False)
            results[(N, rep)] = _batch(hd, ad, Wd, N, np.arange(P), pos, 100 + N + rep, cfg)
    tim.check()
    ref_lp, ref_lse = results[(1, 0)]
    for key, (lp, lse) in results.items():
        assert torch.equal(lp.view(torch.int32), ref_lp.view(torch.int32)), key
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), key
    # and the probes are right
    rows = np.arange(0, P, 37)
    o_lp, o_lse = oracle.token_logprob(h, W, a, rows=rows)
    g_lp = ref_lp.cpu().numpy()[rows]
    g_lse = ref_lse.cpu().numpy()[rows]
    assert np.max(np.abs(g_lp - o_lp)) <= LOGP_ATOL and np.max(np.abs(g_lse - o_lse)) <= LOGP_ATOL
