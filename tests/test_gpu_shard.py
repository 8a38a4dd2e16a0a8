"""The refit over a batch sharded across GPUs, checked on one GPU: the
accumulate-only rounds of two halves of a batch, their accumulator blocks
summed (what the all-reduce does between GPUs) and solved with sv_av_solve,
give the theta of the whole batch refitted at once, and the oracle's
("Adaptive Verification without a confidence head", "Fitting the
coefficients": gradient and Hessian sums over every label of the round, one
solve at its end)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close
from speculative_decoding_verification_03_gb300 import binding, shard, synth

pytestmark = pytest.mark.gpu

THETA_TOL = 1e-5  # |a - b| <= tol * max(1, |b|): the halves sum the same fp32 terms in another order


@pytest.fixture(scope="module", autouse=True)
def _built():
    binding.build()
    oracle.build()
    torch.cuda.init()


def _theta(K):
    return np.concatenate([[0.52], 0.55 - 0.2 * np.arange(K)])


def _labels(name, seed, dev):
    w = synth.WORKLOADS[name](seed=seed, device=dev)
    th = torch.tensor(_theta(w.K), dtype=torch.float32, device=dev)
    out = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, theta=th, want_feature=True)
    return w, out["feature"], out["accept_len"]


@pytest.mark.parametrize("name", ["tiny", "c2"])
def test_two_halves_summed_equal_the_whole_batch(name):
    dev = torch.device("cuda")
    w, feat, acc = _labels(name, 7, dev)
    B, K = w.B, w.K
    kept = torch.tensor(np.random.default_rng(3).integers(0, K + 1, B), dtype=torch.int32, device=dev)
    acc = torch.minimum(acc, kept)
    th0 = _theta(K)
    # the whole batch, one round of one step
    t_whole = torch.tensor(th0, dtype=torch.float32, device=dev)
    s_whole = binding.AVState(K, device=dev)
    s_whole.fit_step(t_whole, feat, acc, kept_len=kept, round_len=1)
    # two shards, accumulate only, blocks summed, solved on each shard
    parts = [shard.shard_range(B, 2, r) for r in range(2)]
    states = [binding.AVState(K, device=dev) for _ in parts]
    thetas = [torch.tensor(th0, dtype=torch.float32, device=dev) for _ in parts]
    for (b0, b1), s, t in zip(parts, states, thetas):
        s.fit_step(t, feat[b0:b1].contiguous(), acc[b0:b1].contiguous(), kept_len=kept[b0:b1].contiguous(),
                   round_len=0)
    torch.cuda.synchronize()
    assert torch.equal(thetas[0], t_whole.new_tensor(th0))  # accumulate only: theta unchanged
    # each shard's block equals the oracle's sums over its sequences (layout of sv_av_accum_bytes)
    for (b0, b1), s in zip(parts, states):
        d = oracle.av_accumulate(th0, feat[b0:b1].double().cpu().numpy(), acc[b0:b1].cpu().numpy(),
                                 kept[b0:b1].cpu().numpy())
        want = shard.block_from_dense(d["g"], d["H"], d["n"])
        got = s.accum().cpu().numpy()
        np.testing.assert_allclose(got, want, rtol=1e-4, atol=1e-4 * np.abs(want).max())
    total = states[0].accum() + states[1].accum()
    for s, t in zip(states, thetas):
        s.accum().copy_(total)
        s.solve(t, damping_c=10.0)
    torch.cuda.synchronize()
    assert torch.equal(thetas[0], thetas[1])
    assert_close(thetas[0].cpu().numpy(), t_whole.cpu().numpy(), tol=THETA_TOL, what="sharded vs whole")
    fit = oracle.AVFit(th0, round_len=1, damping_c=10.0)
    fit.step(feat.double().cpu().numpy(), acc.cpu().numpy(), kept.cpu().numpy())
    assert_close(thetas[0].cpu().numpy(), fit.theta, tol=THETA_TOL, what="sharded vs oracle")
    assert not np.allclose(fit.theta, th0)
    # the solve cleared the block and the round
    assert float(states[0].accum().abs().max()) == 0.0
    for s in states + [s_whole]:
        assert binding.status(s.buf) == (0, 0)


def test_fused_accumulate_only_rounds_then_solve():
    """sv_verify_fit with round_len = 0 on two shards of a C2 batch for three
    steps, then one sum and one solve: the oracle's three-step round over
    the same labels."""
    dev = torch.device("cuda")
    K = 4
    th0 = _theta(K)
    states = [binding.AVState(K, device=dev) for _ in range(2)]
    thetas = [torch.tensor(th0, dtype=torch.float32, device=dev) for _ in range(2)]
    fit = oracle.AVFit(th0, round_len=3, damping_c=10.0)
    for step in range(3):
        w = synth.c2(seed=20 + step, device=dev)
        feats, accs = [], []
        for r in range(2):
            b0, b1 = shard.shard_range(w.B, 2, r)
            out = binding.verify(w.target[b0:b1], w.draft[b0:b1], w.draft_tokens[b0:b1], w.temperature[b0:b1],
                                 1000 * r + step, theta=thetas[r], want_feature=True, av_state=states[r],
                                 round_len=0)
            feats.append(out["feature"])
            accs.append(out["accept_len"])
        fit.step(torch.cat(feats).double().cpu().numpy(), torch.cat(accs).cpu().numpy())
    total = states[0].accum() + states[1].accum()
    for s, t in zip(states, thetas):
        s.accum().copy_(total)
        s.solve(t, damping_c=10.0)
    torch.cuda.synchronize()
    assert torch.equal(thetas[0], thetas[1])
    assert_close(thetas[0].cpu().numpy(), fit.theta, tol=THETA_TOL, what="fused sharded rounds vs oracle")
    assert not np.allclose(fit.theta, th0)


def test_solve_without_labels_keeps_theta():
    dev = torch.device("cuda")
    K = 3
    s = binding.AVState(K, device=dev)
    t = torch.tensor(_theta(K), dtype=torch.float32, device=dev)
    s.solve(t)
    torch.cuda.synchronize()
    assert torch.equal(t, t.new_tensor(_theta(K)))
    assert binding.status(s.buf) == (0, 0)
