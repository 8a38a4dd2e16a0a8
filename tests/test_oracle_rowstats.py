"""Pins of the oracle's row statistics, AV feature, confidence and survival
(CPU only), against scipy / numpy routines and closed forms."""
import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp

import oracle
from speculative_decoding_verification_03_gb300 import synth


def _bf16_row(V, seed, scale=3.0, boost=0.0):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(V, generator=g) * scale
    if boost:
        z[int(torch.randint(0, V, (1,), generator=g))] += boost
    t = z.to(torch.bfloat16)
    return synth.logits_np(t), t.double().numpy()


@pytest.mark.parametrize("V,tau,boost", [(64, 1.0, 0.0), (32000, 1.0, 8.0), (1000, 0.37, 4.0), (7, 2.5, 0.0)])
def test_row_stats_match_logsumexp(V, tau, boost):
    bits, z = _bf16_row(V, seed=V, boost=boost)
    st = oracle.row_stats(bits, tau)
    y = z / tau
    assert st["m"] == y.max()
    assert st["argmax"] == int(np.argmax(y))
    assert abs((st["m"] + st["lnS"]) - logsumexp(y)) < 1e-12 * max(1.0, abs(logsumexp(y)))
    others = np.delete(y, int(np.argmax(y)))
    assert abs(st["E"] - np.exp(others - y.max()).sum()) <= 1e-12 * np.exp(others - y.max()).sum()


def test_row_stats_fp32_and_ties():
    z = np.array([1.0, 3.0, -2.0, 3.0, 0.5], dtype=np.float32)
    st = oracle.row_stats(z, 1.0)
    assert st["argmax"] == 1  # lowest index among equal maxima
    # exactly one copy of the max is excluded from E: the other 3.0 counts as exp(0) = 1
    want = 1.0 + np.exp(1.0 - 3.0) + np.exp(-5.0) + np.exp(0.5 - 3.0)
    assert abs(st["E"] - want) < 1e-15
    assert not st["nonfinite"]


def test_row_stats_nonfinite():
    assert oracle.row_stats(np.array([0.0, np.nan, 1.0], np.float32))["nonfinite"]
    assert oracle.row_stats(np.array([0.0, np.inf, 1.0], np.float32))["nonfinite"]
    assert oracle.row_stats(np.array([-np.inf, -np.inf], np.float32))["nonfinite"]
    st = oracle.row_stats(np.array([-np.inf, 2.0, -np.inf], np.float32))
    assert not st["nonfinite"] and st["E"] == 0.0 and st["argmax"] == 1


@pytest.mark.parametrize("V,seed", [(100, 1), (5000, 2), (64, 3)])
def test_feature_is_logit_of_qmax(V, seed):
    bits, z = _bf16_row(V, seed, scale=2.0, boost=3.0)
    q = np.exp(z - logsumexp(z))
    qmax = q.max()
    st = oracle.row_stats(bits, 1.0)
    x = oracle.feature(st["E"])
    assert abs(x - np.log(qmax / (1 - qmax))) < 1e-9


def test_feature_clamp():
    assert oracle.feature(0.0) == 30.0
    assert oracle.feature(1e-20) == 30.0
    assert oracle.feature(1e20) == -30.0
    assert oracle.feature(1.0) == 0.0


def test_conf_closed_forms():
    # omega = 1, beta = 0: sigmoid(logit(q_max)) = q_max
    for qmax in [0.05, 0.3, 0.5, 0.9, 0.999]:
        x = np.log(qmax / (1 - qmax))
        assert abs(oracle.conf(1.0, 0.0, x) - qmax) < 1e-14
    for w, b, x in [(0.5, 0.55, 2.0), (0.45, -1.0, -3.0), (0.59, 0.1, 7.0)]:
        assert abs(oracle.conf(w, b, x) - expit(w * x + b)) < 1e-15


def test_kept_len_survival():
    conf = np.array([0.9, 0.8, 0.6, 0.9, 0.5])
    surv = np.cumprod(conf)  # 0.9 0.72 0.432 0.3888 0.1944
    assert oracle.kept_len(conf, 0.3) == int((surv >= 0.3).sum()) == 4
    assert oracle.kept_len(conf, 0.0) == 5  # no threshold: keep all
    assert oracle.kept_len(conf, 0.95) == 0
    assert oracle.kept_len(np.array([0.5, 0.6]), 0.3) == 2  # survival 0.3 exactly is kept (>=)


def test_av_score_matches_row_by_row():
    w = synth.tiny(seed=3)
    th = np.array([0.52, 0.55, 0.3, 0.1, -0.2])
    r = oracle.av_score(w.draft.numpy(), w.temperature.numpy(), th, 0.3)
    for b in range(w.B):
        for i in range(w.K):
            st = oracle.row_stats(w.draft[b, i].numpy(), 1.0)
            x = oracle.feature(st["E"])
            assert r["feature"][b, i] == x
            assert abs(r["conf"][b, i] - expit(th[0] * x + th[1 + i])) < 1e-15
        assert r["kept_len"][b] == int((np.cumprod(r["conf"][b]) >= 0.3).sum())
