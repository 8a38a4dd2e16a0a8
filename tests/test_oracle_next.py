"""Pins of the oracle's steps around verification (CPU only): the AV global
budget, the post-verification update, the TTS distillation signal and the
tree acceptance walk.  Each test fixes the oracle against something other
than its own formula: brute force over subsets, closed forms, a hand-worked
example, the cheatsheet's cache bookkeeping replayed step by step, a library
KL divergence, finite differences, the linear oracle, and chi-square tests
of losslessness."""
import itertools

import numpy as np
import pytest
from scipy import special, stats

import oracle
from conftest import golden


# ----------------------------------------------------------------------------- budget
def _costs(N, seed=0):
    rng = np.random.default_rng(seed)
    dc = np.cumsum(rng.uniform(0.05, 0.4, N + 1)).astype(np.float32)
    vc = (5.0 + 0.02 * np.ceil(np.arange(N + 1) / 4.0) * 4.0).astype(np.float32)
    return dc, vc


@pytest.mark.parametrize("seed", range(6))
def test_budget_brute_force_over_subsets(seed):
    rng = np.random.default_rng(seed)
    B, K = 2, 3
    conf = rng.uniform(0.05, 1.0, (B, K)).astype(np.float32)
    n_req = int(rng.integers(1, 5))
    dc, vc = _costs(B * K, seed)
    r = oracle.av_budget(conf, n_req, dc, vc)
    s = np.cumprod(conf.astype(np.float64), axis=1).ravel()
    N = s.size
    best = []
    for n in range(N + 1):
        # the largest achievable sum of n survivals over ALL subsets
        m = max((sum(s[list(c)]) for c in itertools.combinations(range(N), n)), default=0.0)
        best.append(m)
        assert abs(r["est"][n] - (n_req + m)) < 1e-6
    ratio = (n_req + np.array(best)) / (dc.astype(np.float64) + vc.astype(np.float64))[:N + 1]
    assert r["budget"] == int(np.argmax(ratio))
    # the kept drafts are each request's first kept_len positions, and they
    # are the budget largest survivals
    kept = [(b, i) for b in range(B) for i in range(r["kept_len"][b])]
    assert len(kept) == r["budget"]
    if 0 < r["budget"] < N:
        worst_in = min(s[b * K + i] for b, i in kept)
        best_out = max(s[b * K + i] for b in range(B) for i in range(K) if (b, i) not in kept)
        assert worst_in >= best_out - 1e-6


def test_budget_constant_cost_keeps_everything():
    conf = np.random.default_rng(3).uniform(0.2, 0.9, (5, 4)).astype(np.float32)
    N = conf.size
    r = oracle.av_budget(conf, 5, np.zeros(N + 1, np.float32), np.full(N + 1, 7.0, np.float32))
    assert r["budget"] == N and np.all(r["kept_len"] == 4)


@pytest.mark.parametrize("c,a,bcost,expect_all", [(0.6, 10.0, 0.5, True), (0.6, 10.0, 1.0, False)])
def test_budget_linear_cost_closed_form(c, a, bcost, expect_all):
    # K = 1, equal confidences: est[n]/cost[n] = (R + n c)/(a + b n) is monotone,
    # increasing iff c a > R b
    B = 8
    conf = np.full((B, 1), c, np.float32)
    n = np.arange(B + 1, dtype=np.float32)
    r = oracle.av_budget(conf, B, np.zeros(B + 1, np.float32), (a + bcost * n).astype(np.float32))
    assert (c * a > B * bcost) == expect_all
    assert r["budget"] == (B if expect_all else 0)


def test_budget_tie_takes_the_smallest_budget():
    # est / cost equal for every n (est = [2, 3, 4] over cost = [2, 3, 4], all
    # exact): the budget is the first n attaining the maximum, n = 0
    conf = np.ones((2, 1), np.float32)
    r = oracle.av_budget(conf, 2, np.zeros(3, np.float32), np.array([2.0, 3.0, 4.0], np.float32))
    assert list(r["ratio"]) == [1.0, 1.0, 1.0]
    assert r["budget"] == 0 and list(r["kept_len"]) == [0, 0]


def test_budget_ragged_rows_and_survival_rounding():
    rng = np.random.default_rng(9)
    conf = rng.uniform(0.3, 1.0, (6, 5)).astype(np.float32)
    dl = np.array([0, 5, 2, 3, 1, 4])
    dc, vc = _costs(30, 1)
    r = oracle.av_budget(conf, 6, dc, vc, draft_len=dl)
    assert np.all(r["kept_len"] <= dl) and r["est"].size == dl.sum() + 1
    s64 = np.cumprod(conf.astype(np.float64), axis=1)
    s32 = oracle.survival(conf)
    assert np.all(np.abs(s32 - s64) <= 5 * 2.0**-24 * s64 + 1e-30)


# ----------------------------------------------------------------------------- post-verify
def _golden_cases():
    cases = {}
    for row in golden("post_verify_worked.txt"):
        cases.setdefault(row[0], {})[row[1]] = row[2:]
    return cases


def test_post_verify_hand_worked_cases():
    cases = _golden_cases()
    names = sorted(cases)
    ins = np.array([[int(v) for v in cases[n]["in"]] for n in names], np.int32)
    outs = np.array([[int(v) for v in cases[n]["out"]] for n in names], np.int32)
    acc = np.array([int(cases[n]["accept"][0]) for n in names])
    kl = np.array([int(cases[n]["klen"][0]) for n in names])
    B = len(names)
    r = oracle.post_verify(ins, outs, acc, np.full(B, 10), np.full(B, 10), np.zeros((B, 16), np.int32), draft_len=kl)
    for i, n in enumerate(names):
        assert list(r["next_in"][i]) == [int(v) for v in cases[n]["next_in"]], n
        assert r["kv_len"][i] == int(cases[n]["kv_len"][0]), n
        assert r["seq_len"][i] == int(cases[n]["seq_len"][0]), n
        want = np.zeros(16, np.int32)
        for kv in cases[n]["hist"]:
            pos, tok = kv.split(":")
            want[int(pos)] = int(tok)
        assert np.array_equal(r["history"][i], want), n
    assert np.all(r["flags"] == 0)


class _Cache:
    """The cheatsheet's cache bookkeeping, replayed operation by operation."""

    def __init__(self, n):
        self.n = n

    def extend(self, k):
        self.n += k

    def truncate_to(self, n):
        self.n = n


@pytest.mark.parametrize("seed", range(4))
def test_post_verify_kv_matches_the_cheatsheet_loop(seed):
    rng = np.random.default_rng(seed)
    B, K = 40, 6
    kl = rng.integers(0, K + 1, B)
    acc = np.array([rng.integers(0, k + 1) for k in kl])
    prefix = rng.integers(5, 50, B)
    outs = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        outs[b, :acc[b] + 1] = rng.integers(0, 1000, acc[b] + 1)
    ins = rng.integers(0, 1000, (B, K + 1)).astype(np.int32)
    hist = rng.integers(0, 1000, (B, 64)).astype(np.int32)
    r = oracle.post_verify(ins, outs, acc, prefix, prefix, hist, draft_len=kl)
    for b in range(B):
        cache, emitted = _Cache(int(prefix[b])), []
        for i in range(int(kl[b])):
            if i < acc[b]:
                emitted.append(outs[b, i])
                cache.extend(1)
            else:
                emitted.append(outs[b, i])
                cache.truncate_to(int(prefix[b]) + len(emitted))
                break
        else:
            emitted.append(outs[b, kl[b]])  # bonus: no cache entry
        assert r["kv_len"][b] == cache.n
        assert r["seq_len"][b] == prefix[b] + len(emitted)
        assert list(r["history"][b, prefix[b]:prefix[b] + len(emitted)]) == emitted
        assert np.array_equal(r["history"][b, :prefix[b]], hist[b, :prefix[b]])
        assert list(r["next_in"][b, :len(emitted)]) == emitted


def test_post_verify_flags():
    ins = np.zeros((3, 3), np.int32)
    outs = np.array([[4, 5, -1], [4, -1, -1], [1, 2, 3]], np.int32)
    r = oracle.post_verify(ins, outs, [1, 1, 2], [0, 0, 3], [0, 0, 0], np.zeros((3, 4), np.int32))
    assert r["flags"][0] == 0
    assert r["flags"][1] == oracle.post_verify.__globals__["FLAG_BAD_INPUT"]  # emitted token missing
    assert r["flags"][2] == oracle.post_verify.__globals__["FLAG_OVERFLOW"]   # 3 + 3 > capacity 4
    assert list(r["history"][2]) == [0, 0, 0, 1]


# ----------------------------------------------------------------------------- TTS
def test_tts_kl_against_library_and_identity():
    rng = np.random.default_rng(0)
    B, K, V = 3, 4, 50
    t = rng.normal(0, 2, (B, K + 1, V))
    d = t[:, :K] + rng.normal(0, 0.7, (B, K, V))
    tau = np.array([1.0, 0.6, 0.0])
    w = np.array([1.0, 0.8, 0.64, 0.512])
    r = oracle.tts_signal(t, d, tau, w)
    for b in range(B):
        tb = tau[b] if tau[b] > 0 else 1.0
        for k in range(K):
            p = special.softmax(t[b, k] / tb)
            q = special.softmax(d[b, k] / tb)
            assert abs(r["kl"][b, k] - w[k] * stats.entropy(p, q)) < 1e-12
    same = oracle.tts_signal(d, d, tau, w)
    assert np.all(np.abs(same["kl"]) < 1e-12) and np.all(np.abs(same["grad"]) < 1e-15)
    assert np.all(np.abs(r["grad"].sum(axis=2)) < 1e-12)


def test_tts_gradient_by_finite_differences():
    rng = np.random.default_rng(1)
    V = 12
    t = rng.normal(0, 1.5, (1, 1, V))
    d = rng.normal(0, 1.5, (1, 1, V))
    for tau in (1.0, 0.7):
        g = oracle.tts_signal(t, d, [tau], [0.9])["grad"][0, 0]
        h = 1e-6
        for v in range(V):
            dp, dm = d.copy(), d.copy()
            dp[0, 0, v] += h
            dm[0, 0, v] -= h
            num = (oracle.tts_signal(t, dp, [tau], [0.9], want_grad=False)["kl"][0, 0] -
                   oracle.tts_signal(t, dm, [tau], [0.9], want_grad=False)["kl"][0, 0]) / (2 * h)
            assert abs(num - g[v]) < 1e-6


# ----------------------------------------------------------------------------- tree
def test_tree_chain_equals_linear_verification():
    rng = np.random.default_rng(5)
    B, K, V = 64, 4, 40
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 0.8, (B, K, V))).astype(np.float32)
    tau = np.where(np.arange(B) % 5 == 0, 0.0, 1.0).astype(np.float32)
    toks = np.array([[rng.choice(V, p=special.softmax(d[b, i].astype(np.float64) / (tau[b] or 1.0)))
                      for i in range(K)] for b in range(B)], np.int32)
    lin = oracle.verify(t, d, toks, tau, 123)
    # chain: node n + 1 carries draft n; the draft distribution after node n is draft row n
    N = K + 1
    dd = np.concatenate([d, np.zeros((B, 1, V), np.float32)], axis=1)
    tk = np.concatenate([np.zeros((B, 1), np.int32), toks], axis=1)
    par = np.tile(np.arange(-1, K), (B, 1))
    tr = oracle.verify_tree(t, dd, tk, par, tau, 123)
    clear = lin["margin"] > 1e-9
    assert clear.mean() > 0.9
    assert np.array_equal(tr["accept_len"][clear], lin["accept_len"][clear])
    assert np.array_equal(tr["tokens"][clear], lin["tokens"][clear])
    assert np.all(tr["path"][clear][:, :1] == np.where(lin["accept_len"][clear] > 0, 1, -1)[:, None])


def test_tree_greedy_walk_by_hand():
    # root -> {1: tok 2, 2: tok 3}; 1 -> {3: tok 0}; 2 -> {4: tok 1, 5: tok 3}
    V = 4
    par = np.array([[-1, 0, 0, 1, 2, 2]])
    tok = np.array([[0, 2, 3, 0, 1, 3]])
    t = np.zeros((1, 6, V))
    t[0, 0, 3] = 5.0   # root argmax 3 -> child 2
    t[0, 2, 3] = 5.0   # node 2 argmax 3 -> child 5
    t[0, 5, 1] = 5.0   # node 5 is a leaf: bonus 1
    r = oracle.verify_tree(t, np.zeros_like(t), tok, par, [0.0], 0)
    assert list(r["tokens"][0]) == [3, 3, 1, -1, -1, -1]
    assert r["accept_len"][0] == 2 and list(r["path"][0][:2]) == [2, 5]
    t[0, 2, 3] = 0.0
    t[0, 2, 0] = 5.0   # node 2 argmax 0: no child matches, emit 0
    r = oracle.verify_tree(t, np.zeros_like(t), tok, par, [0.0], 0)
    assert list(r["tokens"][0][:2]) == [3, 0] and r["accept_len"][0] == 1


def _chi2_ok(counts, probs, min_p=1e-3):
    exp = probs * counts.sum()
    return stats.chisquare(counts, exp).pvalue > min_p


@pytest.mark.parametrize("branch", [1, 2, 3])
def test_tree_walk_is_lossless(branch):
    """Children drawn i.i.d. from q at each node: the first emitted token is
    distributed as p at the root, and the token after an accepted child c as
    p at c."""
    rng = np.random.default_rng(branch)
    V, B = 5, 20000
    # a two-level tree: root with `branch` children, each with 2 children
    N = 1 + branch + 2 * branch
    par = [-1] + [0] * branch + [1 + c for c in range(branch) for _ in range(2)]
    t_rows = rng.normal(0, 1.2, (N, V))
    d_rows = t_rows + rng.normal(0, 1.0, (N, V))
    p0 = special.softmax(t_rows[0])
    q = [special.softmax(r) for r in d_rows]
    tok = np.zeros((B, N), np.int64)
    for n in range(1, N):
        tok[:, n] = rng.choice(V, size=B, p=q[par[n]])
    T = np.broadcast_to(t_rows, (B, N, V))
    D = np.broadcast_to(d_rows, (B, N, V))
    P = np.broadcast_to(np.array(par), (B, N))
    r = oracle.verify_tree(T, D, tok, P, np.ones(B), 77)
    first = np.bincount(r["tokens"][:, 0], minlength=V)
    assert _chi2_ok(first, p0)
    # second token given the walk accepted child 1 (node index 1)
    sel = r["path"][:, 0] == 1
    second = np.bincount(r["tokens"][sel, 1], minlength=V)
    assert sel.sum() > 1000 and _chi2_ok(second, special.softmax(t_rows[1]))
