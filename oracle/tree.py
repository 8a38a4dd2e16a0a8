"""Acceptance walk over a token tree (test infrastructure only; see
oracle/__init__.py).

Sources:
  - "Accelerating Sonar through Speculation", section "EAGLE": the drafter
    explores several draft sequences as a tree (top candidates at each node
    instead of one chain); the target scores the tree in one pass (with a
    tree attention mask, outside this step), the best-fitting branch is kept
    and one extra token from the target is appended.
  - "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet, "one speculative
    step": accept left to right with probability min(1, p/q), at the first
    rejection sample the normalised positive residual, and a bonus token when
    everything was accepted; its lesson table lists a tree verification mask.

Readings:
  - a request's tree has N nodes in topological order; node 0 is the last
    committed token, node n >= 1 carries draft token tok[n] and parent
    par[n] < n; children are tried in ascending node order;
  - target[n] is the target's next-token distribution after node n; draft[n]
    the draft distribution after node n, from which node n's children were
    drawn independently (with replacement);
  - at node c the walk tries each child x in turn: accept with probability
    min(1, p(x)/q(x)) where p is the target distribution at c, replaced after
    every rejected child by the normalised positive residual max(p - q, 0)
    (the cheatsheet's rule applied once per child); an accepted child becomes
    the current node; when no child is accepted, or c is a leaf, one token is
    drawn from the current p and the walk ends;
  - uniforms: the test of child j at depth t uses word 0 of Philox block
    (b, t, j, 0); the final draw at depth t uses word 1 of block (b, t, 0, 0)
    (a chain tree therefore reproduces linear verification exactly);
  - tau_b <= 0 is a greedy row: the first child whose token is the target's
    argmax (lowest index on ties) is accepted; otherwise, and at a leaf, the
    argmax itself is emitted;
  - a residual with no mass left (rounding only) keeps the previous p and
    raises FLAG_ZERO_RESIDUAL.
"""
from __future__ import annotations

import numpy as np

from . import philox4x32_10

FLAG_ZERO_RESIDUAL = 1
FLAG_BAD_TREE = 2


def tree_uniform(seed: int, b: int, depth: int, child: int, word: int) -> float:
    key = (int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF)
    r = philox4x32_10((b, depth, child, 0), key)
    return float(int(r[word]) >> 8) * (1.0 / 16777216.0)


def _softmax(z):
    y = z - np.max(z)
    e = np.exp(y)
    return e / np.sum(e)


def _draw(p, u):
    """Smallest v with C(v) > u * R, C the ascending cumulative sum of p;
    also the distance of u * R to the nearer edge of v's step, over R."""
    c = np.cumsum(p)
    R = c[-1]
    idx = np.nonzero(c > u * R)[0]
    if idx.size:
        v = int(idx[0])
        lo = c[v - 1] if v > 0 else 0.0
        return v, min(u * R - lo, c[v] - u * R) / R
    nz = np.nonzero(p > 0)[0]
    return (int(nz[-1]) if nz.size else int(np.argmax(p))), 0.0


def verify_tree(target, draft, tokens, parents, temperature, seed: int, n_nodes=None, seq_ids=None):
    """target, draft [B][N][V] floats; tokens, parents [B][N] int; temperature [B].
    Returns dict(tokens [B][N] (emitted, -1 after), accept_len [B], path [B][N-1]
    (accepted node indices, -1 after), flags [B], margin [B]: the smallest
    distance of a decision to its boundary -- |u - p(x)/q(x)| over the child
    tests and the final draw's distance to its step edge (over R);
    acc_margin [B] and smp_margin [B]: the same over the child tests only and
    over the final draw only; ndraws [B]: child tests that drew a uniform).
    seq_ids [B] or None: the request indices that key the uniforms."""
    t = np.asarray(target, dtype=np.float64)
    d = np.asarray(draft, dtype=np.float64)
    tok = np.asarray(tokens, dtype=np.int64)
    par = np.asarray(parents, dtype=np.int64)
    B, N, V = t.shape
    tau = np.asarray(temperature, dtype=np.float64).reshape(B)
    nn = np.full(B, N, np.int64) if n_nodes is None else np.asarray(n_nodes, dtype=np.int64)
    out = np.full((B, N), -1, np.int32)
    path = np.full((B, max(N - 1, 1)), -1, np.int32)
    acc = np.zeros(B, np.int32)
    flags = np.zeros(B, np.int32)
    margin = np.full(B, np.inf)
    acc_margin = np.full(B, np.inf)
    smp_margin = np.full(B, np.inf)
    ndraws = np.zeros(B, np.int32)
    sid = np.arange(B) if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    for b in range(B):
        key = int(sid[b])
        n_b = int(nn[b])
        if n_b < 1 or n_b > N or any(not (0 <= par[b, n] < n) for n in range(1, n_b)):
            flags[b] |= FLAG_BAD_TREE
            continue
        greedy = not (tau[b] > 0)
        tb = 1.0 if greedy else tau[b]
        cur, depth = 0, 0
        while True:
            kids = [n for n in range(1, n_b) if par[b, n] == cur]
            if greedy:
                best = int(np.argmax(t[b, cur]))
                nxt = next((c for c in kids if tok[b, c] == best), None)
                if nxt is None:
                    out[b, depth] = best
                    break
            else:
                p = _softmax(t[b, cur] / tb)
                q = _softmax(d[b, cur] / tb)
                nxt = None
                for j, c in enumerate(kids):
                    x = int(tok[b, c])
                    u = tree_uniform(seed, key, depth, j, 0)
                    ratio = 0.0
                    if 0 <= x < V:
                        ratio = np.inf if q[x] == 0 else p[x] / q[x]
                    margin[b] = min(margin[b], abs(u - ratio))
                    acc_margin[b] = min(acc_margin[b], abs(u - ratio))
                    ndraws[b] += 1
                    if u < ratio:
                        nxt = c
                        break
                    r = np.maximum(p - q, 0.0)
                    if np.sum(r) > 0:
                        p = r / np.sum(r)
                    else:
                        flags[b] |= FLAG_ZERO_RESIDUAL
                if nxt is None:
                    out[b, depth], m = _draw(p, tree_uniform(seed, key, depth, 0, 1))
                    margin[b] = min(margin[b], m)
                    smp_margin[b] = min(smp_margin[b], m)
                    break
            out[b, depth] = tok[b, nxt]
            path[b, depth] = nxt
            cur = nxt
            depth += 1
        acc[b] = depth
    return dict(tokens=out, accept_len=acc, path=path, flags=flags, margin=margin, acc_margin=acc_margin,
                smp_margin=smp_margin, ndraws=ndraws)
