"""The C ABI library loads, exports every function include/specverify.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_03_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    binding.build()
    return binding.lib()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(lib):
    assert lib.sv_workspace_bytes(0, 0, 1) > 0
    assert lib.sv_workspace_bytes(-1, 4, 64) == 0
    assert lib.sv_workspace_bytes(4, 17, 64) == 0
    assert lib.sv_workspace_bytes(4, 4, 0) == 0
    assert lib.sv_workspace_bytes(4, 4, (1 << 24) + 1) == 0
    a = lib.sv_workspace_bytes(256, 5, 128256)
    assert a % 256 == 0 and a < 4 << 20
    assert lib.sv_workspace_bytes(1024, 16, 151936) > a
    assert lib.sv_av_state_bytes(5) > 0 and lib.sv_av_state_bytes(17) == 0
    # the refit's accumulator block: 4K + 2 fp64 values inside the AV state
    for K in (0, 1, 5, 16):
        off, n = lib.sv_av_accum_offset(), lib.sv_av_accum_bytes(K)
        assert off % 256 == 0 and n == (4 * K + 2) * 8
        assert off + n <= lib.sv_av_state_bytes(K)
    assert lib.sv_av_accum_bytes(-1) == 0 and lib.sv_av_accum_bytes(17) == 0


def _verify(lib, B=2, K=2, V=64, dtype=1, tgt=0x10000, drf=0x20000, toks=0x30000, tau=0x40000, theta=None,
            out_tok=0x50000, out_len=0x60000, conf=None, ws=0x100000, wsb=1 << 20):
    P = ctypes.c_void_p
    return lib.sv_verify(B, K, V, dtype, P(tgt) if tgt else None, P(drf) if drf else None,
                         P(toks) if toks else None, None, P(tau) if tau else None, 0,
                         P(theta) if theta else None, None, P(out_tok) if out_tok else None,
                         P(out_len) if out_len else None, None, P(conf) if conf else None,
                         P(ws) if ws else None, wsb, None)


def test_host_argument_checks(lib):
    INVALID, WORKSPACE = 1, 7
    assert _verify(lib, K=17) == INVALID
    assert _verify(lib, V=0) == INVALID
    assert _verify(lib, dtype=5) == INVALID
    assert _verify(lib, tgt=0) == INVALID
    assert _verify(lib, drf=0) == INVALID
    assert _verify(lib, toks=0) == INVALID
    assert _verify(lib, tau=0) == INVALID
    assert _verify(lib, out_tok=0) == INVALID
    assert _verify(lib, conf=0x70000) == INVALID          # conf without theta
    assert _verify(lib, tgt=0x10001) == INVALID           # not aligned to 4 bytes (fp32)
    assert _verify(lib, ws=0) == WORKSPACE
    assert _verify(lib, ws=0x100010) == WORKSPACE         # not 256-byte aligned
    assert _verify(lib, wsb=16) == WORKSPACE
    assert _verify(lib, B=0) == 0                        # nothing to do
    P = ctypes.c_void_p
    assert lib.sv_av_fit_step(4, 4, P(0x1000), P(0x2000), 1 << 20, -1, 10.0, P(0x3000), P(0x4000), None, None) == INVALID
    assert lib.sv_av_fit_step(4, 4, P(0x1000), P(0x2000), 1 << 20, 1, -1.0, P(0x3000), P(0x4000), None, None) == INVALID
    assert lib.sv_av_fit_step(4, 4, P(0x1000), P(0x2000), 16, 1, 10.0, P(0x3000), P(0x4000), None, None) == WORKSPACE
    assert lib.sv_av_score(4, 4, 64, 1, P(0x1000), P(0x2000), None, 0.3, P(0x3000), P(0x4000), None, None,
                           P(0x100000), 1 << 20, None) == INVALID      # theta missing
    assert lib.sv_philox(0, -1, 4, P(0x1000), None) == INVALID
    assert lib.sv_av_solve(17, P(0x1000), P(0x2000), 1 << 20, 10.0, None) == INVALID
    assert lib.sv_av_solve(4, None, P(0x2000), 1 << 20, 10.0, None) == INVALID
    assert lib.sv_av_solve(4, P(0x1000), P(0x2000), 1 << 20, -1.0, None) == INVALID
    assert lib.sv_av_solve(4, P(0x1000), P(0x2000), 16, 10.0, None) == WORKSPACE
    assert lib.sv_av_solve(4, P(0x1000), P(0x2010), 1 << 20, 10.0, None) == WORKSPACE
    assert lib.sv_status(None, None, None) == INVALID


def test_strerror(lib):
    for code in range(0, 11):
        assert lib.sv_strerror(code)
    assert binding.strerror(7).startswith("workspace")


def test_no_gpu_means_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid host arguments reach the device query, which fails loudly without a GPU
    assert _verify(lib) in (2, 3)


def _tts(lib, B=2, K=2, V=64, dtype=1, tgt=0x10000, drf=0x20000, tau=0x40000, wts=0x50000, kl=0x60000,
         grad=None, ws=0x100000, wsb=None):
    P = ctypes.c_void_p
    if wsb is None:
        wsb = lib.sv_tts_workspace_bytes()
    return lib.sv_tts_signal(B, K, V, dtype, P(tgt) if tgt else None, P(drf) if drf else None,
                             P(tau) if tau else None, P(wts) if wts else None, P(kl) if kl else None,
                             P(grad) if grad else None, P(ws) if ws else None, wsb, None)


def test_tts_host_argument_checks(lib):
    INVALID, WORKSPACE = 1, 7
    n = lib.sv_tts_workspace_bytes()
    assert n > 0 and n % 256 == 0 and n < 1 << 20
    assert _tts(lib, K=17) == INVALID
    assert _tts(lib, V=0) == INVALID
    assert _tts(lib, dtype=5) == INVALID
    assert _tts(lib, ws=0) == WORKSPACE
    assert _tts(lib, ws=0x100010) == WORKSPACE           # not 256-byte aligned
    assert _tts(lib, wsb=n - 1) == WORKSPACE
    assert _tts(lib, B=0) == 0                           # nothing to do
    assert _tts(lib, tgt=0) == INVALID
    assert _tts(lib, kl=0) == INVALID
    assert _tts(lib, grad=0x70001) == INVALID            # gradient not aligned to 2 bytes
