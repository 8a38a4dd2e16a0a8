"""Test-time speculation (TTS) distillation signal (test infrastructure only;
see oracle/__init__.py).

Source: "Technical summary: Test-Time Speculation (TTS)", section
"Algorithm", step 3 "Distillation loss": after verification the drafter
takes a gradient step on L(q) = KL~(p || q) + lambda KL~(q_t || q) over the
canvas, with position weights w_k favouring early positions; p is the target
(teacher), q the draft being trained (student), q_t the draft as it was.

Readings:
  - KL~ over the canvas is the w_k-weighted per-position KL divergence over the
    whole vocabulary; the signal is computed at q = q_t, where the second
    term and its gradient vanish;
  - p = softmax(z_target[b][k] / tau_b), q = softmax(z_draft[b][k] / tau_b) for
    canvas positions k = 0 .. K-1; a row with tau_b <= 0 (greedy) uses tau = 1;
  - outputs per (b, k): kl = w_k * sum_v p_v (ln p_v - ln q_v) (terms with
    p_v = 0 contribute 0), and the gradient of that term with respect to the
    draft logits, g_v = w_k * (q_v - p_v) / tau_b.
"""
from __future__ import annotations

import numpy as np


def _log_softmax(z):
    m = np.max(z)
    y = z - m
    return y - np.log(np.sum(np.exp(y)))


def tts_signal(target, draft, temperature, weights, want_grad: bool = True):
    """target [B][K(+1)][V] and draft [B][K][V] as float arrays (fp64 math);
    returns dict(kl [B][K], grad [B][K][V] or None)."""
    t = np.asarray(target, dtype=np.float64)
    d = np.asarray(draft, dtype=np.float64)
    B, K, V = d.shape
    tau = np.asarray(temperature, dtype=np.float64).reshape(B)
    w = np.asarray(weights, dtype=np.float64).reshape(K)
    kl = np.zeros((B, K), np.float64)
    grad = np.zeros((B, K, V), np.float64) if want_grad else None
    for b in range(B):
        tb = tau[b] if tau[b] > 0 else 1.0
        for k in range(K):
            lp = _log_softmax(t[b, k] / tb)
            lq = _log_softmax(d[b, k] / tb)
            p = np.exp(lp)
            q = np.exp(lq)
            with np.errstate(invalid="ignore"):  # p = 0 where lp = -inf: the term is 0
                terms = np.where(p > 0, p * (lp - lq), 0.0)
            kl[b, k] = w[k] * np.sum(terms)
            if want_grad:
                grad[b, k] = w[k] * (q - p) / tb
    return dict(kl=kl, grad=grad)
