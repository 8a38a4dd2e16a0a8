"""sv_verify_noalloc: verification for callers that cannot allocate device
memory (a plain C host holding only pointers to tensors another framework
owns, or a serving runtime that reserved all device memory for its KV-cache
pool and forbids later cudaMalloc).  It uses a scratch array compiled into
the library instead of a caller workspace.  Checked here, through the C ABI,
against sv_verify on the same inputs, on two calls in a row (the scratch
keeps the previous call's contents, so the second call shows that each call
clears what it needs).  Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import assert_rel
from speculative_decoding_verification_03_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    binding.build()
    L = binding.lib()
    P, I, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    L.sv_verify_noalloc.argtypes = [I, I, I, I, P, P, P, P, P, U64, P, P, P, P, P, P, P]
    L.sv_verify_noalloc.restype = I
    L.sv_noalloc_status_holder.argtypes = []
    L.sv_noalloc_status_holder.restype = P
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(L, w, seed, theta):
    B, K, V = w.B, w.K, w.V
    dev = w.target.device
    tok = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    feat = torch.empty((B, K), dtype=torch.float32, device=dev)
    conf = torch.empty((B, K), dtype=torch.float32, device=dev)
    code = binding.SV_BF16 if w.dtype == torch.bfloat16 else binding.SV_FP32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.sv_verify_noalloc(B, K, V, code, _p(w.target), _p(w.draft), _p(w.draft_tokens), None,
                             _p(w.temperature), ctypes.c_uint64(seed), _p(theta), None, _p(tok), _p(acc),
                             _p(feat), _p(conf), stream)
    assert rc == 0, binding.strerror(rc)
    flags = ctypes.c_uint32(0)
    rc = L.sv_status(ctypes.c_void_p(L.sv_noalloc_status_holder()), stream, ctypes.byref(flags))
    assert rc == 0 and flags.value == 0, (rc, flags.value)
    return tok.cpu().numpy(), acc.cpu().numpy(), feat.cpu().numpy(), conf.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "c2", "c3"])
def test_noalloc_matches_sv_verify_twice(lib, name):
    dev = torch.device("cuda")
    w = synth.WORKLOADS[name](seed=5, device=dev)
    theta = torch.tensor([0.52] + [0.4 - 0.1 * i for i in range(w.K)], dtype=torch.float32, device=dev)
    for seed in (11, 12):  # two calls in a row on the shared scratch
        tok, acc, feat, conf = _noalloc(lib, w, seed, theta)
        ref = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, theta=theta,
                             want_feature=True)
        assert np.array_equal(tok, ref["tokens"].cpu().numpy())
        assert np.array_equal(acc, ref["accept_len"].cpu().numpy())
        assert_rel(conf, ref["conf"].cpu().numpy(), what="conf")
        assert_rel(feat, ref["feature"].cpu().numpy(), what="feature")


def test_noalloc_smaller_call_after_a_larger_one(lib):
    """The largest shape first, then the smallest, on the shared scratch: the
    small call's counters and queue entries sit where the large call left
    other values, so this shows that each call clears what its own layout
    needs."""
    dev = torch.device("cuda")
    for name, seed in (("c3", 21), ("tiny", 22), ("c2", 23), ("tiny", 24)):
        w = synth.WORKLOADS[name](seed=seed, device=dev)
        theta = torch.tensor([0.52] + [0.4 - 0.1 * i for i in range(w.K)], dtype=torch.float32, device=dev)
        tok, acc, feat, conf = _noalloc(lib, w, seed, theta)
        ref = binding.verify(w.target, w.draft, w.draft_tokens, w.temperature, seed, theta=theta,
                             want_feature=True)
        assert np.array_equal(tok, ref["tokens"].cpu().numpy()), name
        assert np.array_equal(acc, ref["accept_len"].cpu().numpy()), name
        assert_rel(conf, ref["conf"].cpu().numpy(), what="conf " + name)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    B, K, V = 1024, 16, 1 << 22
    assert lib.sv_workspace_bytes(B, K, V) > (8 << 20)
    rc = lib.sv_verify_noalloc(B, K, V, binding.SV_BF16, None, None, None, None, None, ctypes.c_uint64(0), None,
                               None, None, None, None, None, None)
    assert rc == 7  # SV_ERR_WORKSPACE: needs more scratch than the library holds
