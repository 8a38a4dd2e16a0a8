"""Exact law of one verification step on a small vocabulary, by enumeration.

Independent of the oracle: works on probability vectors in fp64 numpy and
walks every drafted tuple (V^K of them) with its probability prod_i q_i(d_i),
branching on accept (min(1, p/q)) or reject (normalised positive residual)
as the cheatsheet "Speculative Decoding: Draft, EAGLE, MTP" describes in its
section "one speculative step".  Used to pin the oracle, never the reverse.
"""
from __future__ import annotations

import itertools
from collections import defaultdict

import numpy as np


def residual(p, q):
    r = np.maximum(p - q, 0.0)
    s = r.sum()
    return r / s if s > 0 else p.copy()


def step_law(p, q):
    """p: [K+1][V] target probabilities, q: [K][V] draft probabilities.

    Returns dict mapping the emitted token tuple (accepted drafts then the
    residual/bonus token) to its exact probability."""
    K1, V = p.shape
    K = K1 - 1
    law = defaultdict(float)
    for d in itertools.product(range(V), repeat=K):
        w = 1.0
        for i in range(K):
            w *= q[i, d[i]]
        if w == 0.0:
            continue
        reach = w
        for i in range(K + 1):
            if i == K:
                for v in range(V):
                    law[tuple(d[:K]) + (v,)] += reach * p[K, v]
                break
            qi, pi = q[i, d[i]], p[i, d[i]]
            acc = 1.0 if qi == 0.0 else min(1.0, pi / qi)
            rej = 1.0 - acc
            if rej > 0.0:
                r = residual(p[i], q[i])
                for v in range(V):
                    if r[v] > 0.0:
                        law[tuple(d[:i]) + (v,)] += reach * rej * r[v]
            reach *= acc
            if reach == 0.0:
                break
    return dict(law)


def depth_marginals(law, K, V):
    """P(token at depth j = v | depth j reached), j = 0..K, from the exact law."""
    num = np.zeros((K + 1, V))
    for seq, pr in law.items():
        for j, v in enumerate(seq):
            num[j, v] += pr
    reach = num.sum(axis=1, keepdims=True)
    return num / np.where(reach > 0, reach, 1.0), reach.ravel()
