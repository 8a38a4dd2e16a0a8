"""sv_verify_fit: verification and the AV refit step in one launch, checked
against the two-launch path (sv_verify, then sv_av_fit_step on its features
and accept lengths) and against the oracle's refit ("Adaptive Verification
without a confidence head", "Fitting the coefficients").  Tokens, accept
lengths, features and confidences come from the same code as sv_verify and
must be identical; theta differs only by the order of the label sums."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, assert_rel
from speculative_decoding_verification_03_gb300 import binding, synth

pytestmark = pytest.mark.gpu

# theta is O(1): compared as |a - b| <= tol * max(1, |b|); the two paths sum
# the same fp32 per-label terms in a different order and precision
THETA_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    binding.build()
    oracle.build()
    torch.cuda.init()


def _theta(K):
    return np.concatenate([[0.52], 0.55 - 0.2 * np.arange(K)])


def _two_launch(w, seed, theta, st, draft_len=None, round_len=1):
    out = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, draft_len=draft_len, theta=theta,
                         want_feature=True)
    st.fit_step(theta, out["feature"], out["accept_len"], kept_len=draft_len, round_len=round_len)
    return out


def _fused(w, seed, theta, st, draft_len=None, round_len=1):
    return binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, draft_len=draft_len, theta=theta,
                          want_feature=True, av_state=st, round_len=round_len)


def _same_outputs(a, b):
    for k in ("tokens", "accept_len"):
        assert torch.equal(a[k], b[k]), k
    for k in ("feature", "conf"):
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        assert np.array_equal(np.isnan(x), np.isnan(y)), k
        m = ~np.isnan(x)
        assert np.array_equal(x[m], y[m]), k


@pytest.mark.parametrize("name", ["tiny", "c2", "c3"])
def test_fused_fit_matches_two_launches_and_oracle(name):
    dev = torch.device("cuda")
    w = synth.WORKLOADS[name](seed=3, device=dev)
    th = _theta(w.K)
    t1 = torch.tensor(th, dtype=torch.float32, device=dev)
    t2 = t1.clone()
    s1, s2 = binding.AVState(w.K, device=dev), binding.AVState(w.K, device=dev)
    a = _two_launch(w, 21, t1, s1)
    b = _fused(w, 21, t2, s2)
    _same_outputs(a, b)
    assert not torch.equal(t2, torch.tensor(th, dtype=torch.float32, device=dev)), "theta was not updated"
    assert_close(t2.cpu().numpy(), t1.cpu().numpy(), tol=THETA_TOL, what="theta fused vs two launches")
    # the oracle's refit on the GPU's own labels and features
    fit = oracle.AVFit(t1.new_tensor(th).double().cpu().numpy())
    fit.step(b["feature"].double().cpu().numpy(), b["accept_len"].cpu().numpy())
    assert_close(t2.cpu().numpy(), fit.theta, tol=THETA_TOL, what="theta fused vs oracle")
    for st, ws in ((s2, b["ws"]),):
        assert binding.status(st.buf) == (0, 0)
        assert binding.status(ws) == (0, 0)


def test_fused_fit_greedy_rows():
    dev = torch.device("cuda")
    w = synth.tiny(seed=8, B=96, K=6, V=300, greedy=True, device=dev)
    th = _theta(w.K)
    t1 = torch.tensor(th, dtype=torch.float32, device=dev)
    t2 = t1.clone()
    s1, s2 = binding.AVState(w.K, device=dev), binding.AVState(w.K, device=dev)
    _same_outputs(_two_launch(w, 2, t1, s1), _fused(w, 2, t2, s2))
    assert_close(t2.cpu().numpy(), t1.cpu().numpy(), tol=THETA_TOL, what="theta greedy")


def test_fused_fit_rounds_with_draft_len():
    """Round of 3 steps, 7 steps, ragged draft lengths: theta after every
    step, and the confidences each step computes from it, follow the
    two-launch path and the oracle."""
    dev = torch.device("cuda")
    K, rl = 5, 3
    th = _theta(K)
    t1 = torch.tensor(th, dtype=torch.float32, device=dev)
    t2 = t1.clone()
    s1, s2 = binding.AVState(K, device=dev), binding.AVState(K, device=dev)
    fit = oracle.AVFit(th, round_len=rl, damping_c=10.0)
    rng = np.random.default_rng(12)
    for step in range(7):
        w = synth.tiny(seed=40 + step, B=200, K=K, V=700, device=dev)
        dl = torch.tensor(rng.integers(0, K + 1, w.B), dtype=torch.int32, device=dev)
        a = _two_launch(w, 100 + step, t1, s1, draft_len=dl, round_len=rl)
        b = _fused(w, 100 + step, t2, s2, draft_len=dl, round_len=rl)
        for k in ("tokens", "accept_len"):
            assert torch.equal(a[k], b[k]), (step, k)
        fit.step(b["feature"].double().cpu().numpy(), b["accept_len"].cpu().numpy(), dl.cpu().numpy())
        torch.cuda.synchronize()
        assert_close(t2.cpu().numpy(), t1.cpu().numpy(), tol=THETA_TOL, what="theta step %d" % step)
        assert_close(t2.cpu().numpy(), fit.theta, tol=THETA_TOL, what="theta vs oracle step %d" % step)
        ca, cb = a["conf"].cpu().numpy(), b["conf"].cpu().numpy()
        m = ~np.isnan(ca)
        assert np.array_equal(m, ~np.isnan(cb))
        assert_rel(cb[m], ca[m], tol=THETA_TOL * 10, what="conf step %d" % step)
    assert binding.status(s2.buf) == (0, 0)


def test_fused_fit_empty_batch_advances_round():
    dev = torch.device("cuda")
    K = 4
    th = _theta(K)
    t1 = torch.tensor(th, dtype=torch.float32, device=dev)
    t2 = t1.clone()
    s1, s2 = binding.AVState(K, device=dev), binding.AVState(K, device=dev)
    e = synth.tiny(seed=1, B=0, K=K, V=64, device=dev)
    _two_launch(e, 5, t1, s1, round_len=2)
    _fused(e, 5, t2, s2, round_len=2)
    assert torch.equal(t1, t2) and torch.equal(t2, t1.new_tensor(th))  # one step of two: no update yet
    w = synth.tiny(seed=2, B=64, K=K, V=64, device=dev)
    _two_launch(w, 6, t1, s1, round_len=2)
    _fused(w, 6, t2, s2, round_len=2)
    assert not torch.equal(t2, t2.new_tensor(th)), "the round's second step did not update theta"
    assert_close(t2.cpu().numpy(), t1.cpu().numpy(), tol=THETA_TOL, what="theta after empty step")


def test_fused_fit_rejects_missing_state():
    dev = torch.device("cuda")
    w = synth.tiny(seed=1, device=dev)
    st = binding.AVState(w.K, device=dev)
    with pytest.raises(ValueError):
        binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, 1, av_state=st)
    small = binding.AVState(w.K, device=dev)
    small.buf = small.buf[:256]  # shorter than sv_av_state_bytes
    theta = torch.tensor(_theta(w.K), dtype=torch.float32, device=dev)
    with pytest.raises(RuntimeError):
        binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, 1, theta=theta, av_state=small)
