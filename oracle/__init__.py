"""Plain fp64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does: the CUDA
library in ``speculative_decoding_verification_03_gb300`` shares no code with
``oracle.c`` and neither side imports the other.

The arithmetic lives in ``oracle.c`` (single thread, fp64, every step the
obvious one).  This module only compiles it with gcc and marshals numpy
arrays through ctypes.  Logit arrays are passed as raw bytes: bf16 as
``uint16`` bit patterns (dtype code 0), fp32 as ``float32`` (dtype code 1).

Functions whose result is not pinned by a test against the pages or the
mathematics: none (see the test files ``tests/test_oracle_*.py``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FLAG_ZERO_RESIDUAL = 1
FLAG_NONFINITE = 2
FLAG_TOKEN_RANGE = 4
FLAG_BAD_LEN = 8
FLAG_BAD_TEMP = 16


_CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math,
    no FMA contraction, so x86 and Arm give the same bits)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_source(src: str, out: str) -> str:
    """gcc with the oracle's flags: one C source into a shared library."""
    subprocess.run(["gcc"] + _CFLAGS + [src, "-o", out, "-lm"], check=True)
    return out


class _RowStats(ctypes.Structure):
    _fields_ = [("m", ctypes.c_double), ("lnS", ctypes.c_double), ("E", ctypes.c_double),
                ("argmax", ctypes.c_int), ("nonfinite", ctypes.c_int)]


def _bind(path: str):
    """Load a compiled oracle and declare its functions' signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_philox4x32_10.restype = None
    lib.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
    lib.orc_uniform.restype = ctypes.c_double
    lib.orc_row_stats.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.POINTER(_RowStats)]
    lib.orc_row_stats.restype = None
    lib.orc_feature.argtypes = [ctypes.c_double]
    lib.orc_feature.restype = ctypes.c_double
    lib.orc_conf.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
    lib.orc_conf.restype = ctypes.c_double
    lib.orc_kept_len.argtypes = [P, ctypes.c_int, ctypes.c_double]
    lib.orc_kept_len.restype = ctypes.c_int
    lib.orc_av_score.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P,
                                 ctypes.c_double, P, P, P]
    lib.orc_av_score.restype = None
    lib.orc_verify.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P,
                               ctypes.c_uint64, P, P, P, P, P, P, P, P]
    lib.orc_verify.restype = None
    lib.orc_verify_threads.argtypes = [ctypes.c_int] + lib.orc_verify.argtypes
    lib.orc_verify_threads.restype = None
    lib.orc_av_accumulate.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P]
    lib.orc_av_accumulate.restype = None
    lib.orc_av_solve_update.argtypes = [ctypes.c_int, P, P, P, ctypes.c_double, P, P]
    lib.orc_av_solve_update.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the oracle's Python functions on another compiled copy of oracle.c
    (the pin tests use this to check that planted mistakes are caught)."""
    global _lib
    prev = _load()
    with _lock:
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """Return (contiguous array, dtype code) for bf16-as-uint16 or float32 logits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 0
    if a.dtype == np.float32:
        return a, 1
    raise TypeError("logits must be uint16 (bf16 bits) or float32, got %s" % a.dtype)


# --------------------------------------------------------------------------
# Philox4x32-10 and the uniform stream
# --------------------------------------------------------------------------
def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, pos: int, draw: int) -> float:
    return _load().orc_uniform(seed, b, pos, draw)


# --------------------------------------------------------------------------
# Row statistics, feature, confidence
# --------------------------------------------------------------------------
def row_stats(row, tau: float = 1.0):
    """Softmax statistics of one row at temperature tau: dict(m, lnS, E, argmax, nonfinite)."""
    r, code = _logits(row)
    st = _RowStats()
    _load().orc_row_stats(_ptr(r), code, int(r.size), float(tau), ctypes.byref(st))
    return dict(m=st.m, lnS=st.lnS, E=st.E, argmax=st.argmax, nonfinite=bool(st.nonfinite))


def feature(E: float) -> float:
    return _load().orc_feature(float(E))


def conf(omega: float, beta: float, x: float) -> float:
    return _load().orc_conf(float(omega), float(beta), float(x))


def kept_len(conf_row, threshold: float) -> int:
    c = np.ascontiguousarray(np.asarray(conf_row, dtype=np.float64))
    return _load().orc_kept_len(_ptr(c), int(c.size), float(threshold))


def av_score(draft, temperature, theta, keep_threshold: float = 0.0):
    """draft [B][K][V] -> dict(feature [B][K], conf [B][K], kept_len [B])."""
    d, code = _logits(draft)
    B, K, V = d.shape
    t = np.ascontiguousarray(np.asarray(temperature, dtype=np.float32).reshape(B))
    th = np.ascontiguousarray(np.asarray(theta, dtype=np.float64).reshape(K + 1))
    feat = np.zeros((B, K), np.float64)
    cf = np.zeros((B, K), np.float64)
    kl = np.zeros(B, np.int32)
    _load().orc_av_score(B, K, V, code, _ptr(d), _ptr(t), _ptr(th), float(keep_threshold),
                         _ptr(feat), _ptr(cf), _ptr(kl))
    return dict(feature=feat, conf=cf, kept_len=kl)


# --------------------------------------------------------------------------
# Verification step
# --------------------------------------------------------------------------
def verify(target, draft, draft_tokens, temperature, seed: int, draft_len=None, theta=None, seq_ids=None,
           threads: int = 1):
    """One verification step.

    target [B][K+1][V], draft [B][K][V] (uint16 bf16 bits or float32),
    draft_tokens [B][K] int32, temperature [B] float32, draft_len [B] or None,
    seq_ids [B] or None: global sequence indices keying the uniforms.
    Returns dict(tokens [B][K+1], accept_len [B], feature [B][K], conf [B][K],
    acc_margin [B] (smallest |u - ratio| over the acceptance draws),
    smp_margin [B] (distance of u R to the chosen CDF step's nearer edge, / R),
    margin [B] (the smaller of the two), ndraws [B], flags [B]).
    threads > 1 splits the sequences over that many host threads
    (orc_verify_threads); the results are the same.
    """
    t, code = _logits(target)
    d, code2 = _logits(draft)
    assert code == code2
    B, K1, V = t.shape
    K = K1 - 1
    assert d.shape == (B, K, V)
    dt = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, K))
    tau = np.ascontiguousarray(np.asarray(temperature, dtype=np.float32).reshape(B))
    dl = None if draft_len is None else np.ascontiguousarray(np.asarray(draft_len, dtype=np.int32).reshape(B))
    th = None if theta is None else np.ascontiguousarray(np.asarray(theta, dtype=np.float64).reshape(K + 1))
    sid = None if seq_ids is None else np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int32).reshape(B))
    out = dict(tokens=np.zeros((B, K + 1), np.int32), accept_len=np.zeros(B, np.int32),
               feature=np.zeros((B, K), np.float64), conf=np.zeros((B, K), np.float64),
               margins=np.zeros((B, 2), np.float64), ndraws=np.zeros(B, np.int32), flags=np.zeros(B, np.int32))
    args = (B, K, V, code, _ptr(t), _ptr(d), _ptr(dt), _ptr(dl), _ptr(sid), _ptr(tau), int(seed) & (2**64 - 1),
            _ptr(th), _ptr(out["tokens"]), _ptr(out["accept_len"]), _ptr(out["feature"]), _ptr(out["conf"]),
            _ptr(out["margins"]), _ptr(out["ndraws"]), _ptr(out["flags"]))
    if threads > 1:
        _load().orc_verify_threads(int(threads), *args)
    else:
        _load().orc_verify(*args)
    out["acc_margin"] = out["margins"][:, 0].copy()
    out["smp_margin"] = out["margins"][:, 1].copy()
    out["margin"] = out["margins"].min(axis=1)
    del out["margins"]
    return out


# --------------------------------------------------------------------------
# AV refit
# --------------------------------------------------------------------------
def av_accumulate(theta, feature, accept_len, kept_len=None, acc=None):
    """Add one decode step's labelled drafts to acc = dict(g, H, n) at fixed theta."""
    feature = np.ascontiguousarray(np.asarray(feature, dtype=np.float64))
    B, K = feature.shape
    th = np.ascontiguousarray(np.asarray(theta, dtype=np.float64).reshape(K + 1))
    al = np.ascontiguousarray(np.asarray(accept_len, dtype=np.int32).reshape(B))
    kl = None if kept_len is None else np.ascontiguousarray(np.asarray(kept_len, dtype=np.int32).reshape(B))
    if acc is None:
        acc = dict(g=np.zeros(K + 1), H=np.zeros((K + 1, K + 1)), n=np.zeros(K))
    _load().orc_av_accumulate(B, K, _ptr(th), _ptr(feature), _ptr(al), _ptr(kl),
                              _ptr(acc["g"]), _ptr(acc["H"]), _ptr(acc["n"]))
    return acc


def av_solve_update(theta, acc, damping_c: float = 10.0):
    """Damped Newton step; returns (new theta, delta, status)."""
    K = acc["n"].size
    th = np.array(theta, dtype=np.float64).reshape(K + 1).copy()
    delta = np.zeros(K + 1)
    g = np.ascontiguousarray(acc["g"])
    H = np.ascontiguousarray(acc["H"])
    n = np.ascontiguousarray(acc["n"])
    st = _load().orc_av_solve_update(K, _ptr(g), _ptr(H), _ptr(n), float(damping_c), _ptr(th), _ptr(delta))
    return th, delta, st


class AVFit:
    """Round bookkeeping of the refit: accumulate for round_len steps at
    fixed theta, then solve and update ([AV] "Fitting the coefficients")."""

    def __init__(self, theta, round_len: int = 1, damping_c: float = 10.0):
        self.theta = np.array(theta, dtype=np.float64)
        self.round_len = int(round_len)
        self.damping_c = float(damping_c)
        self.acc = None
        self.steps = 0

    def step(self, feature, accept_len, kept_len=None):
        self.acc = av_accumulate(self.theta, feature, accept_len, kept_len, self.acc)
        self.steps += 1
        status = None
        if self.steps == self.round_len:
            self.theta, _, status = av_solve_update(self.theta, self.acc, self.damping_c)
            self.acc = None
            self.steps = 0
        return status


# --------------------------------------------------------------------------
# The steps around verification, in plain numpy (budget.py, post_verify.py,
# tts.py, tree.py)
# --------------------------------------------------------------------------
from .budget import av_budget, survival  # noqa: E402
from .post_verify import post_verify  # noqa: E402
from .tree import tree_uniform, verify_tree  # noqa: E402
from .tts import tts_signal  # noqa: E402
