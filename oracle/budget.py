"""AV global draft budget (test infrastructure only; see oracle/__init__.py).

Source: "Adaptive Verification without a confidence head" (German version
"Adaptive Verification ohne Confidence Head"), section "Other features
considered": drafts are ranked by their survival probability (the running
product of the per-position confidences along each request), the estimated
number of accepted tokens for a budget of n drafts is the number of sampling
requests plus the sum of the n largest survivals, and the budget is the n
that maximises that estimate divided by the measured cost of drafting and
verifying n tokens; the n best-ranked drafts are kept.

Readings where the page leaves a step open:
  - the survivals are the running product of the fp32 confidences, taken in
    fp32 in position order (the same precision as the kernel, so that the
    ranking -- an integer decision -- is identical on both sides);
  - only positions i < draft_len[b] are candidates;
  - ranking: survival descending, ties by flat index b * K + i ascending (so
    every request keeps a prefix of its drafts);
  - est[n] = n_req + sum of the n largest survivals, n = 0 .. N (N = number
    of candidates), summed in fp64 in ranking order; cost[n] = draft_cost[n] +
    verify_cost[n] from a cost table of at least N + 1 entries (synthetic
    here: the page's table is measured on its serving system);
  - a survival that is NaN is not a candidate; one at or below 0 counts as 0;
  - budget = the first n attaining the maximum of est[n] / cost[n] over the n
    with cost[n] > 0 and a finite ratio (0 when there is none);
  - kept_len[b] = the number of request b's drafts among the n best.
"""
from __future__ import annotations

import numpy as np


def survival(conf, draft_len=None):
    """Running product of the confidences along each row, fp32, position order."""
    c = np.asarray(conf, dtype=np.float32)
    B, K = c.shape
    s = np.zeros((B, K), np.float32)
    for b in range(B):
        run = np.float32(1.0)
        for i in range(K):
            run = np.float32(run * c[b, i])
            s[b, i] = run
    return s


def av_budget(conf, n_req: int, draft_cost, verify_cost, draft_len=None):
    """Returns dict(budget, kept_len [B], est [N+1], ratio [N+1], order [N])."""
    c = np.asarray(conf, dtype=np.float32)
    B, K = c.shape
    s = survival(c)
    kl = np.full(B, K, np.int64) if draft_len is None else np.clip(np.asarray(draft_len), 0, K)
    cand = [(max(float(s[b, i]), 0.0), b * K + i) for b in range(B) for i in range(int(kl[b]))
            if not np.isnan(s[b, i])]
    # survival descending, flat index ascending
    cand.sort(key=lambda t: (-t[0], t[1]))
    N = len(cand)
    est = np.zeros(N + 1, np.float64)
    est[0] = float(n_req)
    run = float(n_req)
    for j, (sv, _) in enumerate(cand):
        run = run + sv
        est[j + 1] = run
    dc = np.asarray(draft_cost, dtype=np.float32).astype(np.float64)
    vc = np.asarray(verify_cost, dtype=np.float32).astype(np.float64)
    assert dc.size >= N + 1 and vc.size >= N + 1
    cost = dc[:N + 1] + vc[:N + 1]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = est / cost
    budget, best = 0, None
    for n in range(N + 1):
        if cost[n] > 0 and np.isfinite(ratio[n]) and (best is None or ratio[n] > best):
            budget, best = n, ratio[n]
    kept = np.zeros(B, np.int32)
    for _, idx in cand[:budget]:
        kept[idx // K] += 1
    return dict(budget=budget, kept_len=kept, est=est, ratio=ratio, order=np.array([i for _, i in cand], np.int64))
