"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same bytes, and compare under the parity contract:
tokens and accept lengths bit-exact except sequences in which the oracle saw
a draw within 1e-5 of its decision boundary (counted, and required to stay a
small fraction); floating-point outputs within 1e-4 relative."""
import numpy as np
import torch

import oracle
from speculative_decoding_verification_03_gb300 import binding, synth

NEAR_TIE = 1e-5
REL_TOL = 1e-4


def gpu_verify(w, seed, theta=None, draft_len=None, draft_stats=None, want_feature=True, ws=None):
    dev = torch.device("cuda")
    g = w if w.target.is_cuda else w.to(dev)
    th = None if theta is None else torch.as_tensor(np.asarray(theta), dtype=torch.float32, device=dev)
    dl = None if draft_len is None else torch.as_tensor(np.asarray(draft_len), dtype=torch.int32, device=dev)
    out = binding.verify(g.target, g.draft, g.draft_tokens, g.temperature, seed, draft_len=dl, theta=th,
                         draft_stats=draft_stats, want_feature=want_feature, ws=ws)
    rc, flags = binding.status(out["ws"])
    res = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) and k != "ws" else v) for k, v in out.items()}
    res["rc"], res["flags"] = rc, flags
    return res


def oracle_verify(w, seed, theta=None, draft_len=None, idx=None):
    """Oracle on all sequences, or on the subset idx (keyed by global index)."""
    t, d, toks, tau = w.target, w.draft, w.draft_tokens, w.temperature
    sid = None
    if idx is not None:
        it = torch.as_tensor(idx, device=t.device)
        t, d, toks, tau = t[it], d[it], toks[it], tau[it]
        sid = np.asarray(idx, dtype=np.int32)
        if draft_len is not None:
            draft_len = np.asarray(draft_len)[np.asarray(idx)]
    return oracle.verify(synth.logits_np(t), synth.logits_np(d), toks.cpu().numpy(), tau.cpu().numpy(), seed,
                         draft_len=draft_len, theta=theta, seq_ids=sid)


class Tally:
    """Counts of one comparison: draws, near-ties by kind, mismatches inside the band."""

    def __init__(self):
        self.seqs = self.draws = self.acc_ties = self.smp_ties = self.tie_mismatch = 0

    def __repr__(self):
        return "Tally(seqs=%d draws=%d acc_ties=%d smp_ties=%d tie_mismatch=%d)" % (
            self.seqs, self.draws, self.acc_ties, self.smp_ties, self.tie_mismatch)


def compare(gpu, ref, idx=None, max_acc_tie_frac=None):
    """Bit-exact tokens and accept lengths for every sequence without a
    near-tie draw (oracle margin < 1e-5, acceptance or sampling); sequences
    with one are counted, and so are the ones among them that differ."""
    gt, ga = gpu["tokens"], gpu["accept_len"]
    if idx is not None:
        gt, ga = gt[np.asarray(idx)], ga[np.asarray(idx)]
    acc_tie = ref["acc_margin"] < NEAR_TIE
    smp_tie = ref["smp_margin"] < NEAR_TIE
    flagged = acc_tie | smp_tie
    ok = (ga == ref["accept_len"]) & np.all(gt == ref["tokens"], axis=1)
    bad = np.nonzero(~ok & ~flagged)[0]
    assert bad.size == 0, "mismatch in unflagged sequences %s: gpu %s / %s, oracle %s / %s, margins %s %s" % (
        bad[:5], gt[bad[:3]], ga[bad[:3]], ref["tokens"][bad[:3]], ref["accept_len"][bad[:3]],
        ref["acc_margin"][bad[:3]], ref["smp_margin"][bad[:3]])
    t = Tally()
    t.seqs, t.draws = len(ga), int(ref["ndraws"].sum())
    t.acc_ties, t.smp_ties = int(acc_tie.sum()), int(smp_tie.sum())
    t.tie_mismatch = int((~ok & flagged).sum())
    if max_acc_tie_frac is not None and t.draws > 0:
        assert t.acc_ties / t.draws < max_acc_tie_frac, t
    return t


def assert_close(a, b, tol=REL_TOL, what=""):
    """|a - b| <= tol * max(1, |b|): for features, which cross zero."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert np.array_equal(np.isnan(a), np.isnan(b)), what + ": NaN pattern differs"
    m = ~np.isnan(b)
    err = np.abs(a[m] - b[m]) / np.maximum(np.abs(b[m]), 1.0)
    assert err.size == 0 or err.max() <= tol, "%s: max err %.3g" % (what, err.max())


def assert_rel(a, b, tol=REL_TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    assert np.array_equal(np.isnan(a), np.isnan(b)), what + ": NaN pattern differs"
    a, b = a[~both_nan], b[~both_nan]
    err = np.abs(a - b) / np.maximum(np.abs(b), 1e-30)
    assert err.size == 0 or err.max() <= tol, "%s: max rel err %.3g at %s (gpu %r, oracle %r)" % (
        what, err.max(), np.argmax(err), a.ravel()[np.argmax(err)], b.ravel()[np.argmax(err)])
