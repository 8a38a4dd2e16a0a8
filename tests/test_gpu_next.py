"""GPU parity of the steps around verification, through the C ABI, against
the oracle on the same inputs: the AV global budget (sv_av_budget), the
post-verification update (sv_post_verify), the TTS distillation signal
(sv_tts_signal) and the tree acceptance walk (sv_verify_tree)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_03_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    binding.build()
    oracle.build()
    torch.cuda.init()


# ----------------------------------------------------------------------------- budget
def _budget_check(conf, n_req, dc, vc, draft_len=None):
    dev = torch.device("cuda")
    g_b, g_k = binding.av_budget(conf.to(dev), n_req, dc.to(dev), vc.to(dev),
                                 draft_len=None if draft_len is None else draft_len.to(dev))
    gb, gk = int(g_b.item()), g_k.cpu().numpy()
    r = oracle.av_budget(conf.numpy(), n_req, dc.numpy(), vc.numpy(),
                         draft_len=None if draft_len is None else draft_len.numpy())
    if gb != r["budget"]:
        # only a near-tie may differ (the device sums the ranked survivals in
        # another order): both budgets attain the maximum to 1e-12
        best = np.nanmax(np.where(np.isfinite(r["ratio"]), r["ratio"], -np.inf))
        assert abs(r["ratio"][gb] - best) <= 1e-12 * abs(best), (gb, r["budget"])
    # the kept drafts are the gb best-ranked ones
    K = conf.shape[1]
    want = np.bincount(r["order"][:gb] // K, minlength=conf.shape[0])
    assert np.array_equal(gk, want)
    return gb, r


@pytest.mark.parametrize("B,K", [(4, 4), (64, 4), (256, 5), (512, 16), (1024, 7), (1000, 16)])
def test_budget_parity(B, K):
    conf, dc, vc = synth.budget_inputs(B, K, seed=B + K)
    gb, r = _budget_check(conf, B, dc, vc)
    assert 0 < gb <= B * K


def test_budget_ragged_ties_and_edges():
    conf, dc, vc = synth.budget_inputs(300, 8, seed=3)
    conf[::7] = 0.5                       # many equal survivals: ties by index
    conf[5, 2] = float("nan")             # no score: positions 2.. of row 5 drop out
    conf[9] = 0.0                         # survivals of 0
    dl = torch.from_numpy(np.random.default_rng(1).integers(0, 9, 300).astype(np.int32))
    _budget_check(conf, 300, dc, vc, draft_len=dl)
    # a flat cost keeps every candidate; a negative cost entry is skipped
    flat = torch.full((300 * 8 + 1,), 5.0)
    gb, r = _budget_check(conf, 300, torch.zeros_like(flat), flat, draft_len=dl)
    assert gb == np.count_nonzero(np.diff(r["est"]) > 0)  # every positive survival
    dc2 = dc.clone()
    dc2[:50] = -100.0
    _budget_check(conf, 300, dc2, vc, draft_len=dl)
    # nothing to rank
    _budget_check(torch.full((3, 4), float("nan")), 3, dc[:13], vc[:13])


# ----------------------------------------------------------------------------- post-verify
def _pv_inputs(B, K, seed, cap=48):
    rng = np.random.default_rng(seed)
    kl = rng.integers(0, K + 1, B).astype(np.int32)
    acc = np.array([rng.integers(0, k + 1) for k in kl], np.int32)
    outs = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        outs[b, :acc[b] + 1] = rng.integers(0, 150000, acc[b] + 1)
    ins = rng.integers(0, 150000, (B, K + 1)).astype(np.int32)
    sl = rng.integers(0, cap, B).astype(np.int32)      # some rows run past the capacity
    kv = sl.copy()
    hist = rng.integers(0, 150000, (B, cap)).astype(np.int32)
    bad = rng.random(B) < 0.03
    acc[bad] = kl[bad] + 1                                # invalid accept lengths
    return ins, outs, acc, kl, sl, kv, hist


@pytest.mark.parametrize("B,K", [(1, 0), (37, 3), (3000, 7), (4096, 16)])
def test_post_verify_parity(B, K):
    ins, outs, acc, kl, sl, kv, hist = _pv_inputs(B, K, seed=B)
    dev = torch.device("cuda")
    T = lambda a: torch.from_numpy(a).to(dev)
    g_sl, g_kv, g_hist = T(sl), T(kv), T(hist)
    nxt, fl = binding.post_verify(T(ins), T(outs), T(acc), g_sl, g_kv, history=g_hist, draft_len=T(kl))
    r = oracle.post_verify(ins, outs, acc, sl, kv, hist, draft_len=kl)
    assert np.array_equal(nxt.cpu().numpy(), r["next_in"])
    assert np.array_equal(g_sl.cpu().numpy(), r["seq_len"])
    assert np.array_equal(g_kv.cpu().numpy(), r["kv_len"])
    assert np.array_equal(g_hist.cpu().numpy(), r["history"])
    assert np.array_equal(fl.cpu().numpy(), r["flags"])
    assert (r["flags"] & 2).any() or B < 100


def test_post_verify_after_verify_c2():
    """The device chain verify -> post-verify without the host in between."""
    dev = torch.device("cuda")
    w = synth.c2(seed=4, device=dev)
    out = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, 9)
    last = torch.randint(0, w.V, (w.B, 1), dtype=torch.int32, device=dev)
    ins = torch.cat([last, w.draft_tokens], dim=1).contiguous()
    sl = torch.full((w.B,), 100, dtype=torch.int32, device=dev)
    kv = sl.clone()
    hist = torch.zeros((w.B, 128), dtype=torch.int32, device=dev)
    nxt, fl = binding.post_verify(ins, out["tokens"], out["accept_len"], sl, kv, history=hist)
    r = oracle.post_verify(ins.cpu().numpy(), out["tokens"].cpu().numpy(), out["accept_len"].cpu().numpy(),
                           np.full(w.B, 100), np.full(w.B, 100), np.zeros((w.B, 128), np.int32))
    assert np.array_equal(nxt.cpu().numpy(), r["next_in"]) and np.array_equal(hist.cpu().numpy(), r["history"])
    assert np.array_equal(sl.cpu().numpy(), r["seq_len"]) and np.array_equal(kv.cpu().numpy(), r["kv_len"])
    assert not fl.any()
