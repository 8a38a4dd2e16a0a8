"""Post-verification state update (test infrastructure only; see
oracle/__init__.py).

Sources:
  - "Accelerating Sonar through Speculation", section "MTP schedule for one
    token": after verification a device kernel shifts the target's input
    tokens and plugs the next target tokens into their positions, so that the
    draft re-runs on the same batch layout without a CPU-GPU synchronisation;
    the draft's input buffer is the target's, shifted one step left.
  - "Speculative Decoding: Draft, EAGLE, MTP" cheatsheet, "one speculative
    step" and the loop under "algorithm loop in code": the key-value cache
    grows by one entry per accepted draft and, at the first rejection, is cut
    back to the prefix length plus the number of emitted tokens.

Readings:
  - the verify input row of request b is in[b] = [t_last, d_0, ..., d_{K-1}]
    (the last committed token, then the drafts); the emitted tokens are
    out[b][0..a] (a accepted drafts, then the correction or bonus token);
  - next_in[b][j] = out[b][j] for j <= a (the shifted accepted drafts with the
    target's token plugged in at position a), in[b][j + 1] for a < j < k (the
    drafts that were not accepted, which the draft re-run recomputes and the
    next step discards), -1 elsewhere; k = draft_len[b] (K when absent);
  - the token history gets the a + 1 emitted tokens at positions
    seq_len[b] .. seq_len[b] + a, and seq_len[b] += a + 1; a write past the
    history's capacity is skipped and flagged;
  - kv_len follows the cheatsheet's loop: += a + 1 at a rejection (a < k),
    += k when every draft was accepted (the bonus token has no cache entry
    yet).
"""
from __future__ import annotations

import numpy as np

FLAG_OVERFLOW = 1   # history capacity exceeded (the write was skipped)
FLAG_BAD_INPUT = 2  # accept_len outside [0, k] or a missing emitted token


def post_verify(in_tokens, out_tokens, accept_len, seq_len, kv_len, history, draft_len=None):
    """Returns dict(next_in [B][K+1], seq_len [B], kv_len [B], history [B][H], flags [B]);
    the inputs are not modified."""
    inp = np.asarray(in_tokens, dtype=np.int32)
    out = np.asarray(out_tokens, dtype=np.int32)
    B, K1 = out.shape
    K = K1 - 1
    al = np.asarray(accept_len, dtype=np.int64)
    sl = np.array(seq_len, dtype=np.int64)
    kv = np.array(kv_len, dtype=np.int64)
    hist = np.array(history, dtype=np.int32)
    H = hist.shape[1]
    kl = np.full(B, K, np.int64) if draft_len is None else np.clip(np.asarray(draft_len, dtype=np.int64), 0, K)
    nxt = np.full((B, K1), -1, np.int32)
    flags = np.zeros(B, np.int32)
    for b in range(B):
        a, k = int(al[b]), int(kl[b])
        if a < 0 or a > k or out[b, a] < 0:
            flags[b] |= FLAG_BAD_INPUT
            continue
        for j in range(K1):
            if j <= a:
                nxt[b, j] = out[b, j]
            elif j < k:
                nxt[b, j] = inp[b, j + 1]
        for j in range(a + 1):
            pos = int(sl[b]) + j
            if 0 <= pos < H:
                hist[b, pos] = out[b, j]
            else:
                flags[b] |= FLAG_OVERFLOW
        sl[b] += a + 1
        kv[b] += (a + 1) if a < k else k
    return dict(next_in=nxt, seq_len=sl.astype(np.int32), kv_len=kv.astype(np.int32), history=hist, flags=flags)
