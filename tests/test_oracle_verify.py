"""Pins of the oracle's verification step (CPU only).

Each test fixes the oracle against something other than itself: the closed
form E[tokens per verify] printed on the cheatsheet, the exact law of the
step by enumeration (losslessness theorem), chi-square against the target
distribution, the two-token example of the AV article's footnote, argmax
matching for greedy rows, and plain numpy for emitted-token bookkeeping.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from conftest import golden
from exact_law import depth_marginals, step_law
from speculative_decoding_verification_03_gb300 import synth


def _run(w, seed=0, draft_len=None, theta=None):
    return oracle.verify(synth.logits_np(w.target), synth.logits_np(w.draft), w.draft_tokens.numpy(),
                         w.temperature.numpy(), seed, draft_len=draft_len, theta=theta)


def _resample_drafts(w, q, seed):
    """Fresh drafts d_i ~ q_i for every sequence (the drafter's role)."""
    rng = np.random.default_rng(seed)
    K = w.K
    toks = np.empty((w.B, K), np.int32)
    for i in range(K):
        toks[:, i] = rng.choice(q.shape[1], size=w.B, p=q[i] / q[i].sum())
    w.draft_tokens = torch.from_numpy(toks)
    return w


def _pooled_chisq(obs, exp_p, min_expected=5.0):
    """Chi-square p-value with categories of small expected count pooled."""
    n = obs.sum()
    e = exp_p * n
    order = np.argsort(e)
    o_s, e_s = obs[order].astype(float), e[order]
    bins_o, bins_e, acc_o, acc_e = [], [], 0.0, 0.0
    for oo, ee in zip(o_s, e_s):
        acc_o += oo
        acc_e += ee
        if acc_e >= min_expected:
            bins_o.append(acc_o)
            bins_e.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        bins_o[-1] += acc_o
        bins_e[-1] += acc_e
    return stats.chisquare(bins_o, bins_e).pvalue


def test_tokens_per_verify_closed_form():
    rows = {r[0]: r[1:] for r in golden("tokens_per_verify.txt")}
    alpha, K = float(rows["alpha"][0]), int(rows["K"][0])
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert round(closed, int(rows["printed_decimals"][0])) == float(rows["printed"][0])
    B = 200_000
    w = synth.alpha_exact(alpha, B=B, K=K, V=16, seed=1)
    q = w.meta["q"].numpy()
    w = _resample_drafts(w, q, seed=2)
    r = _run(w, seed=3)
    a = r["accept_len"].astype(np.float64)
    m, se = (a + 1).mean(), (a + 1).std() / np.sqrt(B)
    assert abs(m - closed) < 5 * se, (m, closed, se)
    # the accept length is a geometric law truncated at K
    law = np.array([alpha ** j * (1 - alpha) for j in range(K)] + [alpha ** K])
    assert stats.chisquare(np.bincount(r["accept_len"], minlength=K + 1), law * B).pvalue > 1e-3


@pytest.mark.parametrize("K", [2, 3])
def test_exact_enumeration_v8(K):
    V = 8
    rng = np.random.default_rng(K)
    zt = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zd = (zt[:K] + rng.normal(0, 0.8, (K, V))).astype(np.float32)
    p = np.exp(zt.astype(np.float64))
    p /= p.sum(1, keepdims=True)
    q = np.exp(zd.astype(np.float64))
    q /= q.sum(1, keepdims=True)
    law = step_law(p, q)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    marg, reach = depth_marginals(law, K, V)
    for j in range(K + 1):
        # losslessness: given depth j is reached, the token there follows p_j
        assert np.abs(marg[j] - p[j]).max() < 1e-12
    # the oracle's Monte-Carlo outcome frequencies follow the exact law
    B = 200_000
    w = synth.Workload("v8", B, K, V, torch.float32,
                       torch.from_numpy(np.broadcast_to(zt, (B, K + 1, V)).copy()),
                       torch.from_numpy(np.broadcast_to(zd, (B, K, V)).copy()),
                       torch.zeros((B, K), dtype=torch.int32), torch.ones(B))
    w = _resample_drafts(w, q, seed=10 + K)
    r = _run(w, seed=K)
    keys = list(law.keys())
    index = {k: n for n, k in enumerate(keys)}
    obs = np.zeros(len(keys))
    for b in range(B):
        a = r["accept_len"][b]
        obs[index[tuple(int(t) for t in r["tokens"][b, :a + 1])]] += 1
    assert _pooled_chisq(obs, np.array([law[k] for k in keys])) > 1e-3


def test_first_token_follows_target_tiny():
    base = synth.tiny(seed=0)
    B = 200_000
    zt, zd = base.target[0].numpy(), base.draft[0].numpy()
    p0 = np.exp(zt[0].astype(np.float64))
    p0 /= p0.sum()
    q = np.exp(zd.astype(np.float64))
    q /= q.sum(1, keepdims=True)
    w = synth.Workload("tiny_rep", B, base.K, base.V, torch.float32,
                       torch.from_numpy(np.broadcast_to(zt, (B,) + zt.shape).copy()),
                       torch.from_numpy(np.broadcast_to(zd, (B,) + zd.shape).copy()),
                       torch.zeros((B, base.K), dtype=torch.int32), torch.ones(B))
    w = _resample_drafts(w, q, seed=5)
    r = _run(w, seed=0)
    obs = np.bincount(r["tokens"][:, 0], minlength=base.V)
    assert _pooled_chisq(obs, p0) > 1e-3


def test_footnote_two_token_example():
    g = {r[0]: [float(x) for x in r[1:]] for r in golden("footnote_two_token.txt")}
    p, q = np.array(g["p"]), np.array(g["q"])
    ratio_b = min(1.0, p[1] / q[1])
    assert ratio_b == g["ratio_b"][0]
    res = np.maximum(p - q, 0)
    assert list(res / res.sum()) == g["residual"]
    B = 400_000
    w = synth.two_token_example(B, seed=1)
    d = w.draft_tokens.numpy()[:, 0]
    # untrimmed: lossless
    r = _run(w, seed=7)
    t0 = r["tokens"][:, 0]
    rejected = r["accept_len"] == 0
    assert np.all(t0[rejected] == 0)                     # the residual is [1, 0]
    acc_b = (r["accept_len"][d == 1] == 1).mean()        # P(accept | b drafted) = 0.625
    assert abs(acc_b - ratio_b) < 5 * np.sqrt(ratio_b * (1 - ratio_b) / (d == 1).sum())
    assert np.all(r["accept_len"][d == 0] == 1)          # ratio(a) = 2.5 > 1: always accepted
    assert stats.chisquare(np.bincount(t0, minlength=2), np.array(g["untrimmed_output"]) * B).pvalue > 1e-3
    # trimming on q_sampled (verify only drafts with q(d) >= 0.5) biases the law to [0.4, 0.6]
    trim_len = np.where(q[d] < 0.5, 0, 1).astype(np.int32)
    r2 = _run(w, seed=7, draft_len=trim_len)
    assert stats.chisquare(np.bincount(r2["tokens"][:, 0], minlength=2),
                           np.array(g["trimmed_on_q_sampled_output"]) * B).pvalue > 1e-3
    # trimming on q_max (0.8 for every draft) does not look at the drafted token: lossless
    keep = np.full(B, 1 if q.max() >= 0.5 else 0, np.int32)
    r3 = _run(w, seed=7, draft_len=keep)
    assert stats.chisquare(np.bincount(r3["tokens"][:, 0], minlength=2), p * B).pvalue > 1e-3


def test_greedy_is_argmax_matching():
    for seed in range(4):
        w = synth.tiny(seed=seed, B=64, greedy=True)
        # make about half of the drafts disagree with the target argmax
        toks = w.draft_tokens.numpy().copy()
        rng = np.random.default_rng(seed)
        flip = rng.random(toks.shape) < 0.3
        toks[flip] = rng.integers(0, w.V, flip.sum())
        w.draft_tokens = torch.from_numpy(toks)
        r = _run(w, seed=seed)
        am = np.argmax(w.target.numpy(), axis=-1)  # first index on ties
        for b in range(w.B):
            match = toks[b] == am[b, :w.K]
            a = w.K if match.all() else int(np.argmin(match))
            assert r["accept_len"][b] == a
            assert list(r["tokens"][b, :a]) == list(toks[b, :a])
            assert r["tokens"][b, a] == am[b, a]
            assert np.all(r["tokens"][b, a + 1:] == -1)
            assert r["ndraws"][b] == 0


def test_draft_equal_target_always_accepts():
    base = synth.tiny(seed=1)
    B = 100_000
    z = base.target[0].numpy()
    w = synth.Workload("same", B, base.K, base.V, torch.float32,
                       torch.from_numpy(np.broadcast_to(z, (B,) + z.shape).copy()),
                       torch.from_numpy(np.broadcast_to(z[:base.K], (B, base.K, base.V)).copy()),
                       torch.zeros((B, base.K), dtype=torch.int32), torch.ones(B))
    p = np.exp(z.astype(np.float64))
    p /= p.sum(1, keepdims=True)
    w = _resample_drafts(w, p[:base.K], seed=3)
    r = _run(w, seed=2)
    assert np.all(r["accept_len"] == base.K)
    assert _pooled_chisq(np.bincount(r["tokens"][:, base.K], minlength=base.V), p[base.K]) > 1e-3


def test_output_layout_and_margins_tiny():
    w = synth.tiny(seed=0)
    r = _run(w, seed=0)
    for b in range(w.B):
        a = r["accept_len"][b]
        assert 0 <= a <= w.K
        assert list(r["tokens"][b, :a]) == list(w.draft_tokens[b, :a].numpy())
        assert 0 <= r["tokens"][b, a] < w.V
        assert np.all(r["tokens"][b, a + 1:] == -1)
        assert r["ndraws"][b] == (a + 2 if a < w.K else w.K + 1)
        assert r["margin"][b] > 0
    assert np.isnan(r["conf"]).all()  # AV off


def test_kept_len_zero_emits_plain_decode_token():
    w = synth.tiny(seed=2, B=8)
    r = _run(w, seed=4, draft_len=np.zeros(8, np.int32))
    assert np.all(r["accept_len"] == 0)
    assert np.all(r["tokens"][:, 1:] == -1)
    assert np.all(r["ndraws"] == 1)


def test_error_flags():
    w = synth.tiny(seed=0, B=4)
    toks = w.draft_tokens.numpy().copy()
    toks[1, 0] = w.V + 3
    w.draft_tokens = torch.from_numpy(toks)
    tgt = w.target.numpy().copy()
    tgt[2, 0, 5] = np.nan
    w.target = torch.from_numpy(tgt)
    r = _run(w, seed=0, draft_len=np.array([4, 4, 4, 9], np.int32))
    assert r["flags"][0] == 0
    assert r["flags"][1] & oracle.FLAG_TOKEN_RANGE
    assert r["accept_len"][1] == 0  # an out-of-range draft is rejected
    assert r["flags"][2] & oracle.FLAG_NONFINITE
    assert r["flags"][3] & oracle.FLAG_BAD_LEN


def test_temperature_is_applied_to_both_rows():
    # scaling both logit rows by s and the temperature by s leaves every result unchanged
    w = synth.tiny(seed=4, B=16)
    r1 = _run(w, seed=9)
    s = 2.0  # exact in fp32
    w2 = synth.Workload("scaled", w.B, w.K, w.V, torch.float32, w.target * s, w.draft * s, w.draft_tokens,
                        w.temperature * s)
    r2 = _run(w2, seed=9)
    assert np.array_equal(r1["tokens"], r2["tokens"])
    assert np.array_equal(r1["accept_len"], r2["accept_len"])


# Seeds whose uniform lands exactly on a tie (found by exhaustive search over
# seeds; each test re-checks the uniform before using it).
SEED_U0_IS_ZERO = 12121362      # U(seed, b=0, pos=0, draw 0) == 0
SEED_U1_POS1_IS_HALF = 3321324  # U(seed, b=0, pos=1, draw 1) == 0.5


def test_acceptance_tie_is_a_rejection():
    # u < min(1, ratio) is strict: u = 0 against ratio = 0 (p(d) = 0) rejects
    assert oracle.uniform(SEED_U0_IS_ZERO, 0, 0, 0) == 0.0
    tgt = np.array([[[-np.inf, 0.0], [0.0, 0.0]]], np.float32)
    drf = np.array([[[0.0, 0.0]]], np.float32)
    r = oracle.verify(tgt, drf, np.array([[0]], np.int32), np.ones(1, np.float32), SEED_U0_IS_ZERO)
    assert r["accept_len"][0] == 0
    assert r["tokens"][0, 0] == 1  # residual max(p - q, 0) = [0, 0.5]


def test_cdf_tie_picks_the_next_token():
    # smallest v with C(v) > u R is strict: C(0) = 0.5 = u R picks v = 1
    assert oracle.uniform(SEED_U1_POS1_IS_HALF, 0, 1, 1) == 0.5
    tgt = np.zeros((1, 2, 2), np.float32)           # p = [0.5, 0.5] in both rows (exact)
    drf = np.array([[[0.0, -1.0]]], np.float32)     # ratio(token 0) > 1: accepted, bonus follows
    r = oracle.verify(tgt, drf, np.array([[0]], np.int32), np.ones(1, np.float32), SEED_U1_POS1_IS_HALF)
    assert r["accept_len"][0] == 1
    assert r["tokens"][0, 1] == 1
    assert r["margin"][0] == 0.0  # flagged as a near-tie


def test_zero_draft_probability_accepts():
    # the cheatsheet's loop ("algorithm loop in code") sets the ratio to +inf
    # when the drafter gave the drafted token probability 0: always accepted,
    # whatever the uniform
    tgt = np.zeros((1, 2, 2), np.float32)                  # p = [0.5, 0.5] in both rows
    drf = np.array([[[0.0, -np.inf]]], np.float32)         # q = [1, 0]: token 1 has q = 0
    for seed in range(64):
        r = oracle.verify(tgt, drf, np.array([[1]], np.int32), np.ones(1, np.float32), seed)
        assert r["accept_len"][0] == 1 and r["tokens"][0, 0] == 1
        assert r["flags"][0] == 0


def test_threaded_oracle_equals_single_thread():
    """orc_verify_threads (the all-core timing of the oracle) splits the
    sequences over threads; every output equals one single-threaded call,
    with and without explicit sequence ids."""
    w = synth.c2(seed=3, B=24, V=2003)
    t, d = synth.logits_np(w.target), synth.logits_np(w.draft)
    toks, tau = w.draft_tokens.numpy(), w.temperature.numpy()
    th = np.concatenate([[0.7], 0.3 - 0.1 * np.arange(w.K)])
    dl = np.arange(w.B, dtype=np.int32) % (w.K + 1)
    for kw in (dict(), dict(seq_ids=np.arange(100, 124, dtype=np.int32), draft_len=dl)):
        one = oracle.verify(t, d, toks, tau, 9, theta=th, **kw)
        for n in (2, 5, 64):
            many = oracle.verify(t, d, toks, tau, 9, theta=th, threads=n, **kw)
            for k in one:
                assert np.array_equal(one[k], many[k], equal_nan=True), (n, k)
