"""GPU parity of the steps around verification, through the C ABI, against
the oracle on the same inputs: the AV global budget (sv_av_budget), the
post-verification update (sv_post_verify), the TTS distillation signal
(sv_tts_signal) and the tree acceptance walk (sv_verify_tree)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import oracle_verify
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


@pytest.mark.parametrize("B,K", [(4, 4), (64, 4), (256, 5), (512, 16), (1024, 7), (1000, 16), (1024, 16)])
def test_budget_parity(B, K):
    conf, dc, vc = synth.budget_inputs(B, K, seed=B + K)
    gb, r = _budget_check(conf, B, dc, vc)
    assert 0 < gb <= B * K


@pytest.mark.parametrize("B,K", [(200, 8), (1000, 8), (1024, 4), (2000, 8), (8192, 2), (16384, 1)])
def test_budget_ends_inside_a_tie_group(B, K):
    # equal confidences: the survivals of one position tie across all
    # requests, and these cost tables end the budget part-way through a
    # group, so only the requests with the smallest index keep that position.
    # The runner-up ratios lie 2e-9 .. 4e-6 below the maximum: inside the
    # coarse fp32 window, so several candidates reach the fp64 comparison.
    # Sizes cover every keys-per-thread count of the sort (2, 4, 8, 16) and
    # the largest table (B*K = 16384, K = 2 without the padded row stride).
    conf = torch.full((B, K), 0.9)
    nk = B * K
    n = np.arange(nk + 1, dtype=np.float64)
    for q in (0.3, 2.0):
        vc = torch.from_numpy((B + 0.5 * n + q * n * n / nk).astype(np.float32))
        gb, r = _budget_check(conf, B, torch.zeros(nk + 1), vc)
        assert gb == r["budget"] and gb % B != 0, (gb, r["budget"])


def test_budget_exact_tie_takes_the_smallest_budget():
    # est / cost is exactly 1 for n = 0, 1, 2: the first maximum, n = 0
    dev = torch.device("cuda")
    conf = torch.ones((2, 1), dtype=torch.float32)
    dc, vc = torch.zeros(3), torch.tensor([2.0, 3.0, 4.0])
    g_b, g_k = binding.av_budget(conf.to(dev), 2, dc.to(dev), vc.to(dev))
    r = oracle.av_budget(conf.numpy(), 2, dc.numpy(), vc.numpy())
    assert int(g_b.item()) == r["budget"] == 0
    assert list(g_k.cpu().numpy()) == [0, 0]


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


def test_budget_ragged_edges_sixteen_keys_per_thread():
    # the same edge mix at B*K = 16000 (16 sort keys per thread): ragged
    # lengths, a NaN that cuts a request short, rows of zero survivals and
    # groups of tied survivals
    conf, dc, vc = synth.budget_inputs(2000, 8, seed=11)
    conf[::5] = 0.75
    conf[17, 3] = float("nan")
    conf[40:60] = 0.0
    dl = torch.from_numpy(np.random.default_rng(4).integers(0, 9, 2000).astype(np.int32))
    gb, r = _budget_check(conf, 2000, dc, vc, draft_len=dl)
    assert 0 < gb < np.count_nonzero(r["est"][1:] > r["est"][:-1])


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


# ----------------------------------------------------------------------------- TTS
def _tts_case(w, weights, pairs=None):
    dev = torch.device("cuda")
    g = w if w.target.is_cuda else w.to(dev)
    wt = torch.tensor(weights, dtype=torch.float32, device=dev)
    kl, grad = binding.tts_signal(g.target, g.draft, g.temperature, wt)
    kl = kl.cpu().numpy()
    t, d, tau = synth.logits_np(w.target), synth.logits_np(w.draft), w.temperature.cpu().numpy()
    if w.target.dtype == torch.bfloat16:  # bf16 bit patterns -> values
        t = (t.astype(np.uint32) << 16).view(np.float32)
        d = (d.astype(np.uint32) << 16).view(np.float32)
    if pairs is None:
        pairs = [(b, k) for b in range(w.B) for k in range(w.K)]
    for b, k in pairs:
        r = oracle.tts_signal(t[b:b + 1, k:k + 1], d[b:b + 1, k:k + 1], tau[b:b + 1], [weights[k]])
        ko = r["kl"][0, 0]
        if np.isinf(ko):  # a draft logit of -inf where p > 0
            assert kl[b, k] == ko, (b, k, kl[b, k], ko)
        else:
            assert abs(kl[b, k] - ko) <= 1e-4 * abs(ko) + 1e-9, (b, k, kl[b, k], ko)
        go = r["grad"][0, 0]
        gg = grad[b, k].float().cpu().numpy()
        tb = tau[b] if tau[b] > 0 else 1.0
        p = np.exp(t[b, k] / tb - np.max(t[b, k] / tb))
        p /= p.sum()
        q = np.exp(d[b, k] / tb - np.max(d[b, k] / tb))
        q /= q.sum()
        # bf16 rounding, plus the fp32 normalisation of p and q (their sums
        # over the row are kept to a few 1e-7): the error of q_v - p_v is
        # bounded relative to the larger of the two
        tol = 1.01 * 2.0**-8 * np.abs(go) + 2e-6 * abs(weights[k]) / tb * np.maximum(p, q) + 1e-38
        bad = np.abs(gg - go) > tol
        assert not bad.any(), (b, k, np.nonzero(bad)[0][:5], gg[bad][:5], go[bad][:5])
    return kl


def test_tts_tiny_and_unaligned():
    w = synth.tiny(seed=3, B=6, K=4, V=64)
    w.temperature = torch.tensor([1.0, 0.5, 0.0, 1.3, 1.0, 0.8])
    _tts_case(w, [1.0, 0.9, 0.81, 0.729])
    for V, dt in ((1001, torch.bfloat16), (37, torch.float32), (7, torch.bfloat16)):
        g = torch.Generator().manual_seed(V)
        z = torch.randn((5, 4, V), generator=g) * 2
        dd = z[:, :3] + torch.randn((5, 3, V), generator=g) * 0.5
        ww = synth.Workload("u", 5, 3, V, dt, z.to(dt).contiguous(), dd.to(dt).contiguous(),
                            torch.zeros((5, 3), dtype=torch.int32), torch.ones(5))
        _tts_case(ww, [1.0, 0.5, 0.25])


def _tts_rows(B, K, V, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((B, K + 1, V), generator=g) * 2
    dd = z[:, :K] + torch.randn((B, K, V), generator=g) * 0.5
    return synth.Workload("t", B, K, V, dtype, z.to(dtype).contiguous(), dd.to(dtype).contiguous(),
                          torch.zeros((B, K), dtype=torch.int32), torch.ones(B))


def test_tts_c4_vocabulary():
    # V = 151936 bf16: another group size and slice length than the C3 rows
    _tts_case(_tts_rows(3, 3, 151936, torch.bfloat16, 11), [1.0, 0.7, 0.5])


def test_tts_fp32_rows():
    # V = 128256 fp32: slices of 16-byte vectors of four elements
    _tts_case(_tts_rows(2, 2, 128256, torch.float32, 12), [1.0, 0.6])


def test_tts_wide_rows_two_resident_slices():
    # V = 700000 bf16: three pair slices per CTA fit no group of at most 32
    # CTAs, so two do (and fewer pairs than groups)
    _tts_case(_tts_rows(1, 2, 700000, torch.bfloat16, 14), [1.0, 0.8])


def test_tts_maximum_vocabulary():
    # V = 2^24 bf16 (SV_MAX_V): slices too long for shared memory, so the
    # kernel that reads each pair twice (the second time from L2) runs
    V = 1 << 24
    g = torch.Generator().manual_seed(15)
    z = torch.randn((1, 2, V), generator=g) * 2
    d = z[:, :1] + torch.randn((1, 1, V), generator=g) * 0.5
    w = synth.Workload("t", 1, 1, V, torch.bfloat16, z.to(torch.bfloat16).contiguous(),
                       d.to(torch.bfloat16).contiguous(), torch.zeros((1, 1), dtype=torch.int32), torch.ones(1))
    _tts_case(w, [0.9])


def test_tts_masked_logits_and_degenerate_weights():
    # target logits of -inf and far below the rest (p = 0 or an underflow, the
    # warps holding them take the general path), a draft logit of -inf where
    # p > 0 (KL = +inf), a zero and a negative weight
    w = _tts_rows(4, 3, 32000, torch.bfloat16, 13)
    w.target[0, 0, :300] = float("-inf")
    w.target[1, 1, 4000:4064] = -3.0e4
    w.target[2, 2, 31990:] = float("-inf")
    w.draft[3, 0, 7] = float("-inf")
    w.temperature = torch.tensor([1.0, 0.5, 1.7, 1.0])
    _tts_case(w, [1.0, 0.0, -0.5])


def test_tts_wait_timeout_is_reported_and_the_next_call_recovers():
    """A TTS wait that runs out: with sv_set_wait_test's withhold no row copy
    is issued, so the compute warps' copy waits can only end by their limit
    (200 us).  The call reports SV_ERR_TIMEOUT through the workspace status,
    every KL value is NaN and no gradient is written; the next call on the
    same workspace returns SV_OK and matches the oracle."""
    dev = torch.device("cuda")
    w = _tts_rows(4, 2, 32000, torch.bfloat16, 21).to(dev)
    wt = torch.tensor([1.0, 0.7], dtype=torch.float32, device=dev)
    ws = binding.tts_workspace(dev)
    grad = torch.full((w.B, w.K, w.V), 7.0, dtype=torch.bfloat16, device=dev)
    binding.set_wait_test(limit_ns=200_000, withhold=True)
    try:
        kl, _ = binding.tts_signal(w.target, w.draft, w.temperature, wt, out_grad=grad, workspace=ws)
    finally:
        binding.set_wait_test(0, False)
    rc, flags = binding.status(ws)
    assert rc == 6 and flags & binding.FLAG_TIMEOUT, (rc, flags)  # SV_ERR_TIMEOUT
    assert bool(torch.isnan(kl).all())
    assert bool((grad == 7.0).all())  # nothing was written
    kl2, _ = binding.tts_signal(w.target, w.draft, w.temperature, wt, out_grad=grad, workspace=ws)
    rc, flags = binding.status(ws)
    assert rc == 0 and flags == 0, (rc, flags)
    ref = _tts_case(w, [1.0, 0.7])  # another call, checked against the oracle
    assert np.array_equal(kl2.cpu().numpy(), ref)  # the launch is deterministic


def test_tts_identical_rows_give_zero():
    w = synth.c2(seed=2)
    w.draft = w.target[:, :w.K].contiguous()
    dev = torch.device("cuda")
    kl, grad = binding.tts_signal(w.target.to(dev), w.draft.to(dev), w.temperature.to(dev),
                                  torch.ones(w.K, device=dev))
    assert torch.all(kl.abs() < 1e-7) and torch.all(grad.float().abs() < 1e-7)


def test_tts_c2_all_pairs():
    w = synth.c2(seed=5)
    _tts_case(w, [1.0, 0.8, 0.6, 0.4])


def test_tts_c3_sampled_pairs():
    w = synth.c3(seed=6, device="cuda")
    rng = np.random.default_rng(0)
    pairs = [(int(b), int(k)) for b, k in zip(rng.integers(0, w.B, 12), rng.integers(0, w.K, 12))]
    kl = _tts_case(w, [1.0, 0.9, 0.8, 0.7, 0.6], pairs=pairs)
    assert np.all(np.isfinite(kl)) and np.all(kl >= 0)


def test_tts_c3_every_kl():
    # the full C3 launch (the bench's configuration): every one of the 1280
    # KL values against the oracle (the gradient is sampled above)
    w = synth.c3(seed=7, device="cuda")
    weights = [1.0, 0.9, 0.8, 0.7, 0.6]
    kl, _ = binding.tts_signal(w.target, w.draft, w.temperature,
                               torch.tensor(weights, dtype=torch.float32, device="cuda"), want_grad=False)
    kl = kl.cpu().numpy()
    t = (synth.logits_np(w.target).astype(np.uint32) << 16).view(np.float32)
    d = (synth.logits_np(w.draft).astype(np.uint32) << 16).view(np.float32)
    ko = oracle.tts_signal(t, d, w.temperature.cpu().numpy(), weights, want_grad=False)["kl"]
    assert np.all(np.abs(kl - ko) <= 1e-4 * np.abs(ko) + 1e-9), np.max(np.abs(kl - ko) / (np.abs(ko) + 1e-9))


# ----------------------------------------------------------------------------- tree
# The parity contract of the linear path, applied to the tree walk: paths,
# tokens and accept lengths identical to the oracle; decisions within 1e-5
# of their boundary (|u - ratio| for a child test, the draw's distance to its
# CDF step edge over R) are counted, must match as well, and child-test ties
# must stay under 1e-4 of the child tests over the statistics run.
TREE_TIE = 1e-5


def _tree_values(t):
    a = synth.logits_np(t)
    return (a.astype(np.uint32) << 16).view(np.float32) if t.dtype == torch.bfloat16 else a


def _tree_compare(w, seed, idx=None):
    dev = torch.device("cuda")
    g = w.to(dev)
    out = binding.verify_tree(g.target, g.draft, g.tokens, g.parents, g.temperature, seed)
    res = {k: v.cpu().numpy() for k, v in out.items()}
    assert not (res["flags"] & 2).any()
    sel = np.arange(w.B) if idx is None else np.asarray(idx)
    T, D = _tree_values(w.target), _tree_values(w.draft)
    r = oracle.verify_tree(T[sel], D[sel], w.tokens.numpy()[sel], w.parents.numpy()[sel],
                           w.temperature.numpy()[sel], seed, seq_ids=sel)
    ok = (res["accept_len"][sel] == r["accept_len"]) & np.all(res["tokens"][sel] == r["tokens"], axis=1) & \
        np.all(res["path"][sel] == r["path"], axis=1)
    acc_tie = r["acc_margin"] < TREE_TIE
    tie = acc_tie | (r["smp_margin"] < TREE_TIE)
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, ("mismatch (tie flags %s)" % tie[bad][:4], sel[bad][:4], res["tokens"][sel][bad][:2],
                           r["tokens"][bad][:2], r["acc_margin"][bad][:4], r["smp_margin"][bad][:4])
    return res, r, int(acc_tie.sum()), int(r["ndraws"].sum()), int(tie.sum())


@pytest.mark.parametrize("dtype,V", [(torch.float32, 300), (torch.bfloat16, 2000), (torch.bfloat16, 1001)])
def test_tree_parity_small(dtype, V):
    w = synth.tree(seed=V, B=48, V=V, dtype=dtype)
    res, r, acc_ties, draws, ties = _tree_compare(w, 17)
    print("tree", V, "draws", draws, "acceptance ties", acc_ties, "all ties", ties, "mean accept",
          res["accept_len"].mean())
    assert res["accept_len"].max() >= 2


def test_tree_parity_tie_statistics():
    """Many requests at a small vocabulary: every decision identical, and
    child-test near-ties under 1e-4 of the child tests."""
    w = synth.tree(seed=77, B=8192, V=64, dtype=torch.float32)
    res, r, acc_ties, draws, ties = _tree_compare(w, 23)
    print("tree statistics: draws", draws, "acceptance ties", acc_ties, "all ties", ties)
    assert draws > 20000
    assert acc_ties / draws < 1e-4, (acc_ties, draws)


def test_tree_parity_vocab_32000_sampled():
    w = synth.tree(seed=5, B=96, V=32000)
    _tree_compare(w, 3, idx=np.arange(0, 96, 6))


def test_tree_parity_vocab_128256_rows_from_l2():
    # two 256 KB rows per node do not fit in shared memory: every pass reads them from L2
    w = synth.tree(seed=11, B=8, V=128256)
    _tree_compare(w, 5)


def test_tree_parity_maximum_vocabulary():
    # V = 2^24 (SV_MAX_V): every pass streams its rows from L2/HBM and a
    # thread sums tens of thousands of terms per row
    w = synth.tree(seed=13, B=2, V=1 << 24, levels=(2, 2))
    _tree_compare(w, 9)


def test_tree_chain_equals_sv_verify():
    """A chain tree is linear verification: identical to sv_verify except
    sequences in which the oracle flags a near-tie (counted), and those must
    agree too."""
    dev = torch.device("cuda")
    w = synth.c2(seed=7, device=dev)
    B, K, V = w.B, w.K, w.V
    lin = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, 11)
    N = K + 1
    draft = torch.cat([w.draft, torch.zeros((B, 1, V), dtype=w.draft.dtype, device=dev)], dim=1).contiguous()
    toks = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device=dev), w.draft_tokens], dim=1).contiguous()
    par = torch.arange(-1, K, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    tr = binding.verify_tree(w.target, draft, toks, par, w.temperature, 11)
    same = ((tr["accept_len"] == lin["accept_len"]) & torch.all(tr["tokens"] == lin["tokens"], dim=1)).cpu().numpy()
    ref = oracle_verify(w, 11)
    tie = ref["margin"] < TREE_TIE
    print("chain tree: ties", int(tie.sum()), "of", B)
    assert same.all(), (np.nonzero(~same)[0][:8], tie[~same][:8])


def test_tree_greedy_by_hand_and_bad_trees():
    dev = torch.device("cuda")
    V, N = 4, 6
    par = torch.tensor([[-1, 0, 0, 1, 2, 2], [-1, 0, 0, 1, 2, 2], [-1, 0, 3, 1, 2, 2]], dtype=torch.int32)
    tok = torch.tensor([[0, 2, 3, 0, 1, 3]] * 3, dtype=torch.int32)
    t = torch.zeros((3, N, V))
    t[:, 0, 3] = 5.0
    t[:, 2, 3] = 5.0
    t[:, 5, 1] = 5.0
    t[1, 2, 3], t[1, 2, 0] = 0.0, 5.0
    out = binding.verify_tree(t.to(dev), torch.zeros_like(t).to(dev), tok.to(dev), par.to(dev),
                              torch.zeros(3, device=dev), 0)
    o = {k: v.cpu().numpy() for k, v in out.items()}
    assert list(o["tokens"][0]) == [3, 3, 1, -1, -1, -1] and o["accept_len"][0] == 2
    assert list(o["path"][0][:2]) == [2, 5]
    assert list(o["tokens"][1][:3]) == [3, 0, -1] and o["accept_len"][1] == 1
    assert o["flags"][2] == 2 and o["accept_len"][2] == 0 and (o["tokens"][2] == -1).all()
