"""GPU edge cases: empty and ragged canvases, unaligned and tiny vocabularies,
split rows, error flags, workspace reuse, determinism, invariances."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_rel, compare, gpu_verify, oracle_verify
from speculative_decoding_verification_03_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    binding.build()
    oracle.build()


def _rand_workload(B, K, V, dtype=torch.float32, seed=0, noise=0.7, scale=2.0, tau=1.0):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((B, K + 1, V), generator=g) * scale
    d = z[:, :K] + torch.randn((B, K, V), generator=g) * noise
    t, dd = z.to(dtype), d.to(dtype)
    probs = torch.softmax(dd.float() / tau, -1).reshape(-1, V) if K > 0 else None
    toks = (torch.multinomial(probs, 1, generator=g).view(B, K) if K > 0 else torch.zeros((B, 0), dtype=torch.int64))
    return synth.Workload("rand", B, K, V, dtype, t.contiguous(), dd.contiguous(), toks.to(torch.int32),
                          torch.full((B,), float(tau)))


def _check(w, seed, theta=None, draft_len=None):
    g = gpu_verify(w, seed, theta=theta, draft_len=draft_len)
    assert g["rc"] == 0, g["flags"]
    r = oracle_verify(w, seed, theta=theta, draft_len=draft_len)
    compare(g, r)
    if theta is not None:
        assert_rel(g["conf"], r["conf"], what="conf")
    return g, r


def test_k0_is_plain_sampling():
    w = _rand_workload(16, 0, 100, seed=1)
    g, r = _check(w, 3)
    assert np.all(g["accept_len"] == 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_draft_len(dtype):
    w = _rand_workload(64, 6, 500, dtype=dtype, seed=2)
    dl = np.random.default_rng(0).integers(0, 7, 64).astype(np.int32)
    dl[:3] = [0, 6, 1]
    th = np.concatenate([[0.5], np.linspace(0.5, -0.5, 6)])
    g, r = _check(w, 4, theta=th, draft_len=dl)
    assert np.all(g["accept_len"] <= dl)
    assert np.isnan(g["conf"][0]).all()  # nothing verified: no score


@pytest.mark.parametrize("V,dtype", [(1001, torch.bfloat16), (37, torch.float32), (1, torch.float32),
                                     (2, torch.bfloat16), (7, torch.bfloat16), (8195, torch.float32),
                                     (32001, torch.bfloat16)])
def test_unaligned_and_tiny_vocab(V, dtype):
    w = _rand_workload(24, 3, V, dtype=dtype, seed=V)
    th = np.array([0.6, 0.4, 0.1, -0.3])
    g, r = _check(w, V, theta=th)
    if V == 1:
        assert np.all(g["accept_len"] == 3) and np.all(g["tokens"] == 0)


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 128256), (torch.float32, 300007)])
def test_split_rows(dtype, V):
    # few rows with a long vocabulary: each row is split into chunks merged on the device
    w = _rand_workload(2, 1, V, dtype=dtype, seed=5, scale=3.0, noise=1.0)
    th = np.array([0.5, 0.3])
    _check(w, 11, theta=th)


def test_draft_equal_target_accepts_all():
    w = _rand_workload(128, 4, 256, seed=6, noise=0.0)
    w.draft = w.target[:, :4].contiguous()
    p = torch.softmax(w.draft, -1).reshape(-1, 256)
    w.draft_tokens = torch.multinomial(p, 1, generator=torch.Generator().manual_seed(1)).view(128, 4).to(torch.int32)
    g, r = _check(w, 1)
    assert np.all(g["accept_len"] == 4)


def test_mixed_temperatures_and_greedy_rows():
    w = _rand_workload(96, 5, 3000, dtype=torch.bfloat16, seed=7)
    tau = np.random.default_rng(1).uniform(0.3, 1.2, 96).astype(np.float32)
    tau[::7] = 0.0
    w.temperature = torch.from_numpy(tau)
    th = np.concatenate([[0.5], np.zeros(5)])
    _check(w, 8, theta=th)


def test_temperature_scaling_invariance():
    w = _rand_workload(64, 4, 777, dtype=torch.bfloat16, seed=8, tau=0.7)
    g1 = gpu_verify(w, 5)
    w2 = synth.Workload("s", w.B, w.K, w.V, w.dtype, w.target * 2, w.draft * 2, w.draft_tokens, w.temperature * 2)
    g2 = gpu_verify(w2, 5)
    assert np.array_equal(g1["tokens"], g2["tokens"]) and np.array_equal(g1["accept_len"], g2["accept_len"])


def test_determinism_and_workspace_reuse():
    w = synth.c2(seed=3, device="cuda")
    th = np.concatenate([[1.0], np.zeros(w.K)])
    ws = binding.workspace(256, 5, 128256)  # larger than needed, reused
    g1 = gpu_verify(w, 1, theta=th, ws=ws)
    g2 = gpu_verify(w, 1, theta=th, ws=ws)
    for k in ("tokens", "accept_len", "conf", "feature"):
        assert np.array_equal(g1[k], g2[k], equal_nan=True), k
    small = _rand_workload(8, 2, 64, seed=9)
    gs = gpu_verify(small, 2, ws=ws)
    rs = oracle_verify(small, 2)
    compare(gs, rs)
    g3 = gpu_verify(w, 1, theta=th, ws=ws)
    assert np.array_equal(g1["tokens"], g3["tokens"])


def test_error_flags_are_reported_not_trapped():
    w = _rand_workload(6, 3, 200, seed=10)
    toks = w.draft_tokens.clone()
    toks[1, 0] = 200 + 5
    toks[2, 1] = -3
    w.draft_tokens = toks
    g = gpu_verify(w, 1)
    assert g["rc"] == 5, g
    assert g["flags"] & binding.FLAG_TOKEN_RANGE
    r = oracle_verify(w, 1)
    compare(g, r)
    assert g["accept_len"][1] == 0
    # status is cleared by reading it
    rc, flags = binding.status(g["ws"])
    assert rc == 0 and flags == 0

    w2 = _rand_workload(4, 2, 64, seed=11)
    w2.target[2, 1, 7] = float("nan")
    g2 = gpu_verify(w2, 1)
    assert g2["rc"] == 4 and g2["flags"] & binding.FLAG_NONFINITE
    ok = np.array([0, 1, 3])
    r2 = oracle_verify(w2, 1)
    assert np.array_equal(g2["tokens"][ok], r2["tokens"][ok])
    assert np.all((g2["tokens"] >= -1) & (g2["tokens"] < 64))

    w3 = _rand_workload(4, 2, 64, seed=12)
    g3 = gpu_verify(w3, 1, draft_len=np.array([2, 5, -1, 1], np.int32))
    assert g3["rc"] == 8 and g3["flags"] & binding.FLAG_BAD_LEN
    r3 = oracle_verify(w3, 1, draft_len=np.array([2, 5, -1, 1], np.int32))
    assert np.array_equal(g3["tokens"], r3["tokens"])

    w4 = _rand_workload(4, 2, 64, seed=13)
    w4.temperature = torch.tensor([1.0, -0.5, 1.0, float("nan")])
    g4 = gpu_verify(w4, 1)
    assert g4["rc"] == 9 and g4["flags"] & binding.FLAG_BAD_TEMP
    r4 = oracle_verify(w4, 1)
    assert np.array_equal(g4["tokens"], r4["tokens"])


def test_host_checks_with_gpu_present():
    dev = torch.device("cuda")
    t = torch.zeros((2, 3, 64), device=dev)
    d = torch.zeros((2, 2, 64), device=dev)
    toks = torch.zeros((2, 2), dtype=torch.int32, device=dev)
    tau = torch.ones(2, device=dev)
    with pytest.raises(binding.SVError) as e:
        binding.verify(t, d, toks, tau, 0, ws=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.code == 7
    out = binding.verify(t, d, toks, tau, 0)
    L = binding.lib()
    import ctypes
    rc = L.sv_verify(2, 2, 64, 1, ctypes.c_void_p(t.data_ptr() + 2), ctypes.c_void_p(d.data_ptr()),
                     ctypes.c_void_p(toks.data_ptr()), None, ctypes.c_void_p(tau.data_ptr()), 0, None, None,
                     ctypes.c_void_p(out["tokens"].data_ptr()), ctypes.c_void_p(out["accept_len"].data_ptr()),
                     None, None, ctypes.c_void_p(out["ws"].data_ptr()), out["ws"].numel(), None)
    assert rc == 1  # logits not aligned to their element size


def test_early_exit_uses_no_target_row_past_the_first_rejection():
    """Target rows a_b + 1 .. K of every sequence (a_b from the oracle) are
    filled with NaN: the walk must not use them (no non-finite flag) and the
    outputs must not change.  (Row a_b + 1 may be read one step ahead on
    small launches, and is then discarded.)"""
    w = synth.c2(seed=9)
    th = np.concatenate([[0.6], np.linspace(0.4, -0.4, w.K)])
    r = oracle_verify(w, 13, theta=th)
    g0 = gpu_verify(w, 13, theta=th)
    poisoned = w.target.clone()
    for b in range(w.B):
        a = int(r["accept_len"][b])
        if a < w.K:
            poisoned[b, a + 1:] = float("nan")
    w2 = synth.Workload("p", w.B, w.K, w.V, w.dtype, poisoned, w.draft, w.draft_tokens, w.temperature)
    g = gpu_verify(w2, 13, theta=th)
    assert g["rc"] == 0 and g["flags"] == 0, g["flags"]
    assert np.array_equal(g["tokens"], g0["tokens"]) and np.array_equal(g["accept_len"], g0["accept_len"])
    assert np.array_equal(g["conf"], g0["conf"])
    assert (r["accept_len"] < w.K).sum() > w.B // 2  # most sequences had rows to skip


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_draft_probability_accepts(dtype):
    """A drafted token the drafter gave probability 0 (logit -inf) has ratio
    +inf and is always accepted, as in the cheatsheet's loop; the bonus token
    then follows the target row."""
    B, K, V = 64, 3, 256
    g = torch.Generator().manual_seed(11)
    t = (torch.randn((B, K + 1, V), generator=g) * 2.0).to(dtype)
    d = (torch.randn((B, K, V), generator=g) * 2.0)
    toks = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    d.scatter_(2, toks.long().unsqueeze(-1), float("-inf"))
    w = synth.Workload("qzero", B, K, V, dtype, t.contiguous(), d.to(dtype).contiguous(), toks, torch.ones(B))
    g_out, r = _check(w, 21)
    assert np.all(g_out["accept_len"] == K) and np.all(r["accept_len"] == K)


@pytest.mark.parametrize("name", ["tiny", "c2"])
def test_wait_timeout_is_reported_and_the_next_call_recovers(name):
    """A device wait that runs out: with sv_set_wait_test's withhold, the
    producer warps stage nothing, so every other warp's first wait can only
    end by its limit (200 us here).  The call reports SV_ERR_TIMEOUT through
    the workspace status, writes no output, and leaves the GPU usable: the
    next call on the same workspace returns SV_OK and matches the oracle."""
    dev = torch.device("cuda")
    w = synth.WORKLOADS[name](seed=5)
    g = w.to(dev)
    B, K = w.B, w.K
    ws = binding.workspace(B, K, w.V, dev)
    th = torch.tensor(np.concatenate([[1.0], np.zeros(K)]), dtype=torch.float32, device=dev)
    out = dict(tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
               accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
               feature=torch.full((B, K), -7.0, device=dev), conf=torch.full((B, K), -7.0, device=dev))
    binding.set_wait_test(limit_ns=200_000, withhold=True)
    try:
        binding.verify(g.target, g.draft, g.draft_tokens, g.temperature, 3, theta=th, want_feature=True, ws=ws,
                       out=out)
    finally:
        binding.set_wait_test(0, False)
    rc, flags = binding.status(ws)
    assert rc == 6 and flags & binding.FLAG_TIMEOUT, (rc, flags)  # SV_ERR_TIMEOUT
    for k in ("tokens", "accept_len", "feature", "conf"):
        assert bool((out[k] == -7).all()), k  # nothing was written
    res = gpu_verify(w, 3, theta=np.concatenate([[1.0], np.zeros(K)]), ws=ws)
    assert res["rc"] == 0 and res["flags"] == 0, (res["rc"], res["flags"])
    ref = oracle_verify(w, 3, theta=np.concatenate([[1.0], np.zeros(K)]))
    compare(res, ref)
    assert_rel(res["conf"], ref["conf"], what="conf after a time-out")


def test_wait_limit_without_withholding_changes_nothing():
    """The limit alone (a generous 5 s) leaves results and status unchanged."""
    w = synth.c2(seed=9)
    th = np.concatenate([[1.0], np.zeros(w.K)])
    base = gpu_verify(w, 4, theta=th)
    binding.set_wait_test(limit_ns=5_000_000_000, withhold=False)
    try:
        res = gpu_verify(w, 4, theta=th)
    finally:
        binding.set_wait_test(0, False)
    assert res["rc"] == 0 and base["rc"] == 0
    assert np.array_equal(res["tokens"], base["tokens"]) and np.array_equal(res["accept_len"], base["accept_len"])


@pytest.fixture(scope="module")
def max_vocab_workload():
    return synth.tiny(seed=31, B=2, K=2, V=1 << 24)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_maximum_vocabulary(dtype, max_vocab_workload):
    """V = 2^24 (SV_MAX_V), B = 2, K = 2: the largest rows the library
    accepts (16 split chunks per static row, a queued target row of 2^24
    elements on one SM, 16 draw parts of 4096 sub-chunks).  At this V a
    draw's CDF steps are about R / V wide, so nearly every draw lies within
    1e-5 R of a step edge (a sampling near-tie); those are counted and must
    still agree with the oracle."""
    import dataclasses
    w = max_vocab_workload
    if dtype == torch.bfloat16:
        w = dataclasses.replace(w, target=w.target.to(dtype).contiguous(), draft=w.draft.to(dtype).contiguous(),
                                dtype=dtype)
    for seed in (0, 1):
        th = np.array([1.0, 0.0, 0.0])
        g = gpu_verify(w, seed, theta=th)
        assert g["rc"] == 0 and g["flags"] == 0, (g["rc"], g["flags"])
        r = oracle_verify(w, seed, theta=th)
        t = compare(g, r)
        print("V = 2^24", dtype, "seed", seed, t)
        assert t.tie_mismatch == 0, t
        assert_rel(g["conf"], r["conf"], what="conf")
