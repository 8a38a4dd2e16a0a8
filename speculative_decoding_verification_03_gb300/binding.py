"""ctypes binding of ``libspecverify.so`` (the C ABI in ``include/specverify.h``).

Argument marshalling only: every step of the verification path runs in the
library's CUDA kernels.  Torch tensors provide device memory and the current
stream.  There is no fallback: if the library was not built, or the device
is not a GB300 (sm_103), the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
_SOURCES = ["api.cu", "rowpass.cu", "sample.cu", "avfit.cu", "postverify.cu", "budget.cu", "tts.cu", "tree.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC"]

SV_BF16, SV_FP32 = 0, 1
STATUS_NAMES = {0: "SV_OK", 1: "SV_ERR_INVALID", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_CUDA",
                4: "SV_ERR_NONFINITE", 5: "SV_ERR_TOKEN_RANGE", 6: "SV_ERR_TIMEOUT", 7: "SV_ERR_WORKSPACE",
                8: "SV_ERR_BAD_LEN", 9: "SV_ERR_BAD_TEMP"}
FLAG_NONFINITE, FLAG_TOKEN_RANGE, FLAG_TIMEOUT, FLAG_BAD_LEN, FLAG_BAD_TEMP = 1, 2, 4, 8, 16
FLAG_ZERO_RESIDUAL, FLAG_FIT_SINGULAR = 32, 64


class SVError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, STATUS_NAMES.get(code, "?"), code))


def build(force: bool = False, nvcc: str = "nvcc") -> str:
    """Compile the CUDA sources for sm_103a into libspecverify.so (in-tree)."""
    csrc = os.path.join(_HERE, "csrc")
    srcs = [os.path.join(csrc, s) for s in _SOURCES]
    deps = srcs + [os.path.join(csrc, h) for h in ("sv_device.cuh", "sv_internal.h", "sample_common.cuh", "rowstats.cuh",
                                                   "avfit_common.cuh")] + \
        [os.path.join(_ROOT, "include", "specverify.h")]
    if not force and os.path.exists(LIB_PATH) and \
            os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(d) for d in deps):
        return LIB_PATH
    bdir = os.path.join(_HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    inc = ["-I" + os.path.join(_ROOT, "include")]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        subprocess.run([nvcc] + NVCC_FLAGS + inc + ["-c", src, "-o", obj], check=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None
_lock = threading.Lock()


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libspecverify.so is not built (run __graft_entry__.build()); "
                                   "there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            P, I, U64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
            L.sv_workspace_bytes.argtypes = [I, I, I]
            L.sv_workspace_bytes.restype = SZ
            L.sv_verify.argtypes = [I, I, I, I, P, P, P, P, P, U64, P, P, P, P, P, P, P, SZ, P]
            L.sv_verify.restype = I
            L.sv_verify_fit.argtypes = [I, I, I, I, P, P, P, P, P, U64, P, P, P, P, P, P, P, SZ, I, F, P, SZ, P]
            L.sv_verify_fit.restype = I
            L.sv_av_score.argtypes = [I, I, I, I, P, P, P, F, P, P, P, P, P, SZ, P]
            L.sv_av_score.restype = I
            L.sv_av_state_bytes.argtypes = [I]
            L.sv_av_state_bytes.restype = SZ
            L.sv_av_reset.argtypes = [I, P, SZ, P]
            L.sv_av_reset.restype = I
            L.sv_av_fit_step.argtypes = [I, I, P, P, SZ, I, F, P, P, P, P]
            L.sv_av_fit_step.restype = I
            L.sv_av_accum_offset.argtypes = []
            L.sv_av_accum_offset.restype = SZ
            L.sv_av_accum_bytes.argtypes = [I]
            L.sv_av_accum_bytes.restype = SZ
            L.sv_av_solve.argtypes = [I, P, P, SZ, F, P]
            L.sv_av_solve.restype = I
            L.sv_philox.argtypes = [U64, I, I, P, P]
            L.sv_philox.restype = I
            L.sv_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
            L.sv_status.restype = I
            L.sv_set_wait_test.argtypes = [U64, I]
            L.sv_set_wait_test.restype = I
            L.sv_set_launch_events.argtypes = [P, P]
            L.sv_set_launch_events.restype = I
            L.sv_post_verify.argtypes = [I, I, P, P, P, P, P, P, P, I, P, P, P]
            L.sv_post_verify.restype = I
            L.sv_av_budget.argtypes = [I, I, P, P, I, P, P, P, P, P]
            L.sv_av_budget.restype = I
            L.sv_tts_workspace_bytes.argtypes = []
            L.sv_tts_workspace_bytes.restype = SZ
            L.sv_tts_signal.argtypes = [I, I, I, I, P, P, P, P, P, P, P, SZ, P]
            L.sv_tts_signal.restype = I
            L.sv_verify_tree.argtypes = [I, I, I, I, P, P, P, P, P, P, U64, P, P, P, P, P]
            L.sv_verify_tree.restype = I
            L.sv_strerror.argtypes = [I]
            L.sv_strerror.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != 0:
        raise SVError(rc, where)


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_FP32
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def workspace_bytes(B: int, K: int, V: int) -> int:
    return int(lib().sv_workspace_bytes(B, K, V))


def workspace(B: int, K: int, V: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(B, K, V)
    if n == 0:
        raise ValueError("invalid shape")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def verify(target, draft, draft_tokens, temperature, seed: int, draft_len=None, theta=None, draft_stats=None,
           want_feature: bool = False, want_conf: bool | None = None, ws=None, out=None, stream=None,
           av_state: "AVState | None" = None, round_len: int = 1, damping_c: float = 10.0):
    """One verification step on the GPU.  Returns dict(tokens [B][K+1] int32,
    accept_len [B] int32, feature [B][K] or None, conf [B][K] or None, ws).
    With av_state (and theta) the AV refit step runs in the same launch
    (sv_verify_fit) and theta is updated in place at the end of a round."""
    B, K1, V = target.shape
    K = K1 - 1
    code = _dtype_code(target)
    _dev(target, "target")
    _dev(draft, "draft", target.dtype)
    _dev(draft_tokens, "draft_tokens", torch.int32)
    _dev(temperature, "temperature", torch.float32)
    _dev(draft_len, "draft_len", torch.int32)
    _dev(theta, "theta", torch.float32)
    _dev(draft_stats, "draft_stats", torch.int32)
    if want_conf is None:
        want_conf = theta is not None
    dev = target.device
    if out is None:
        out = dict(tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                   accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   feature=torch.empty((B, K), dtype=torch.float32, device=dev) if want_feature else None,
                   conf=torch.empty((B, K), dtype=torch.float32, device=dev) if want_conf else None)
    if ws is None:
        ws = workspace(B, K, V, dev)
    out["ws"] = ws
    if av_state is not None:
        if theta is None:
            raise ValueError("the fused refit needs theta")
        rc = lib().sv_verify_fit(B, K, V, code, _ptr(target), _ptr(draft), _ptr(draft_tokens), _ptr(draft_len),
                                 _ptr(temperature), ctypes.c_uint64(int(seed) & (2**64 - 1)), _ptr(theta),
                                 _ptr(draft_stats), _ptr(out["tokens"]), _ptr(out["accept_len"]),
                                 _ptr(out["feature"]), _ptr(out["conf"]), _ptr(av_state.buf), av_state.buf.numel(),
                                 int(round_len), float(damping_c), _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "sv_verify_fit")
        return out
    rc = lib().sv_verify(B, K, V, code, _ptr(target), _ptr(draft), _ptr(draft_tokens), _ptr(draft_len),
                         _ptr(temperature), ctypes.c_uint64(int(seed) & (2**64 - 1)), _ptr(theta),
                         _ptr(draft_stats), _ptr(out["tokens"]), _ptr(out["accept_len"]), _ptr(out["feature"]),
                         _ptr(out["conf"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "sv_verify")
    return out


def av_score(draft, temperature, theta, keep_threshold: float = 0.0, want_stats: bool = False, ws=None,
             out=None, stream=None):
    """AV scoring of the drafts.  Returns dict(feature, conf, kept_len, stats or None, ws)."""
    B, K, V = draft.shape
    code = _dtype_code(draft)
    _dev(draft, "draft")
    _dev(temperature, "temperature", torch.float32)
    _dev(theta, "theta", torch.float32)
    dev = draft.device
    if out is None:
        out = dict(feature=torch.empty((B, K), dtype=torch.float32, device=dev),
                   conf=torch.empty((B, K), dtype=torch.float32, device=dev),
                   kept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   stats=torch.empty((B, K, 4), dtype=torch.int32, device=dev) if want_stats else None)
    if ws is None:
        ws = workspace(B, K, V, dev)
    out["ws"] = ws
    rc = lib().sv_av_score(B, K, V, code, _ptr(draft), _ptr(temperature), _ptr(theta), float(keep_threshold),
                           _ptr(out["feature"]), _ptr(out["conf"]), _ptr(out["kept_len"]), _ptr(out["stats"]),
                           _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "sv_av_score")
    return out


class AVState:
    """Device state of the AV refit (round accumulators, step counter, status)."""

    def __init__(self, K: int, device="cuda", stream=None):
        self.K = K
        n = int(lib().sv_av_state_bytes(K))
        self.buf = torch.empty(n, dtype=torch.uint8, device=device)
        self.reset(stream)

    def reset(self, stream=None):
        _check(lib().sv_av_reset(self.K, _ptr(self.buf), self.buf.numel(), _stream(stream)), "sv_av_reset")

    def fit_step(self, theta, feature, accept_len, kept_len=None, round_len: int = 1, damping_c: float = 10.0,
                 stream=None):
        B = accept_len.shape[0]
        _dev(theta, "theta", torch.float32)
        _dev(feature, "feature", torch.float32)
        _dev(accept_len, "accept_len", torch.int32)
        _dev(kept_len, "kept_len", torch.int32)
        rc = lib().sv_av_fit_step(B, self.K, _ptr(theta), _ptr(self.buf), self.buf.numel(), int(round_len),
                                  float(damping_c), _ptr(feature), _ptr(accept_len), _ptr(kept_len),
                                  _stream(stream))
        _check(rc, "sv_av_fit_step")

    def accum(self) -> torch.Tensor:
        """The round's accumulator block (sv_av_accum_offset / sv_av_accum_bytes):
        a float64 view into the state, 4K + 2 values g[0..K], H_ww, H_wb[K],
        H_bb[K], n[K].  Summing it over the shards of a batch (in place, e.g.
        torch.distributed.all_reduce) before solve() gives the refit of the
        whole batch."""
        off = int(lib().sv_av_accum_offset())
        n = int(lib().sv_av_accum_bytes(self.K))
        return self.buf[off:off + n].view(torch.float64)

    def solve(self, theta, damping_c: float = 10.0, stream=None):
        """sv_av_solve: end the round now (solve from the accumulator block,
        update theta in place, clear the block)."""
        _dev(theta, "theta", torch.float32)
        rc = lib().sv_av_solve(self.K, _ptr(theta), _ptr(self.buf), self.buf.numel(), float(damping_c),
                               _stream(stream))
        _check(rc, "sv_av_solve")


class HostSession:
    """Verification from host buffers: each step copies the inputs from
    (pinned) host tensors into device buffers allocated once, runs
    sv_verify_fit (verification and the refit step in one launch), and copies
    the emitted tokens and accept lengths back into host tensors.  All on one
    stream, no synchronisation: the host outputs are valid after the stream
    is synchronised."""

    def __init__(self, B, K, V, dtype, device, theta0, round_len=1, damping_c=10.0):
        self.B, self.K, self.V = B, K, V
        self.dev = torch.device(device)
        self.target = torch.empty((B, K + 1, V), dtype=dtype, device=self.dev)
        self.draft = torch.empty((B, K, V), dtype=dtype, device=self.dev)
        self.draft_tokens = torch.empty((B, K), dtype=torch.int32, device=self.dev)
        self.temperature = torch.empty((B,), dtype=torch.float32, device=self.dev)
        self.theta = torch.tensor(theta0, dtype=torch.float32, device=self.dev)
        self.ws = workspace(B, K, V, self.dev)
        self.state = AVState(K, device=self.dev)
        self.round_len, self.damping_c = round_len, damping_c
        self.out = dict(tokens=torch.empty((B, K + 1), dtype=torch.int32, device=self.dev),
                        accept_len=torch.empty((B,), dtype=torch.int32, device=self.dev),
                        feature=torch.empty((B, K), dtype=torch.float32, device=self.dev),
                        conf=torch.empty((B, K), dtype=torch.float32, device=self.dev))

    def step(self, host, seed, tokens_out, accept_out):
        for name in ("target", "draft", "draft_tokens", "temperature"):
            getattr(self, name).copy_(host[name], non_blocking=True)
        verify(self.target, self.draft, self.draft_tokens, self.temperature, seed, theta=self.theta,
               want_feature=True, ws=self.ws, out=self.out, av_state=self.state, round_len=self.round_len,
               damping_c=self.damping_c)
        tokens_out.copy_(self.out["tokens"], non_blocking=True)
        accept_out.copy_(self.out["accept_len"], non_blocking=True)


def post_verify(in_tokens, out_tokens, accept_len, seq_len, kv_len, history=None, draft_len=None,
                next_in=None, flags=None, stream=None):
    """sv_post_verify: updates seq_len, kv_len and history in place, fills
    next_in and flags (allocated when not given); returns (next_in, flags)."""
    B, K1 = out_tokens.shape
    dev = out_tokens.device
    for t, n in ((in_tokens, "in_tokens"), (out_tokens, "out_tokens"), (accept_len, "accept_len"),
                 (seq_len, "seq_len"), (kv_len, "kv_len"), (history, "history"), (draft_len, "draft_len")):
        _dev(t, n, torch.int32)
    if next_in is None:
        next_in = torch.empty((B, K1), dtype=torch.int32, device=dev)
    if flags is None:
        flags = torch.empty((B,), dtype=torch.int32, device=dev)
    cap = 0 if history is None else history.shape[1]
    rc = lib().sv_post_verify(B, K1 - 1, _ptr(in_tokens), _ptr(out_tokens), _ptr(accept_len), _ptr(draft_len),
                              _ptr(seq_len), _ptr(kv_len), _ptr(history), cap, _ptr(next_in), _ptr(flags),
                              _stream(stream))
    _check(rc, "sv_post_verify")
    return next_in, flags


def av_budget(conf, n_req: int, draft_cost, verify_cost, draft_len=None, out_budget=None, out_kept_len=None,
              stream=None):
    """sv_av_budget: returns (budget [1] int32, kept_len [B] int32) device tensors."""
    B, K = conf.shape
    _dev(conf, "conf", torch.float32)
    _dev(draft_cost, "draft_cost", torch.float32)
    _dev(verify_cost, "verify_cost", torch.float32)
    _dev(draft_len, "draft_len", torch.int32)
    if draft_cost.numel() < B * K + 1 or verify_cost.numel() < B * K + 1:
        raise ValueError("cost tables need B*K + 1 entries")
    if out_budget is None:
        out_budget = torch.empty((1,), dtype=torch.int32, device=conf.device)
    if out_kept_len is None:
        out_kept_len = torch.empty((B,), dtype=torch.int32, device=conf.device)
    rc = lib().sv_av_budget(B, K, _ptr(conf), _ptr(draft_len), int(n_req), _ptr(draft_cost), _ptr(verify_cost),
                            _ptr(out_budget), _ptr(out_kept_len), _stream(stream))
    _check(rc, "sv_av_budget")
    return out_budget, out_kept_len


def tts_workspace(device=None):
    """A workspace for sv_tts_signal (sv_tts_workspace_bytes() bytes)."""
    return torch.empty(int(lib().sv_tts_workspace_bytes()), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def tts_signal(target, draft, temperature, weights, want_grad: bool = True, out_kl=None, out_grad=None,
               workspace=None, stream=None):
    """sv_tts_signal: returns (kl [B][K] float32, grad [B][K][V] bfloat16 or None).
    `workspace` (tts_workspace()) is allocated per call when not given."""
    B, K, V = draft.shape
    code = _dtype_code(target)
    if _dtype_code(draft) != code or target.shape != (B, K + 1, V):
        raise ValueError("target must be [B][K+1][V] and draft [B][K][V] of one dtype")
    _dev(target, "target")
    _dev(draft, "draft")
    _dev(temperature, "temperature", torch.float32)
    _dev(weights, "weights", torch.float32)
    if out_kl is None:
        out_kl = torch.empty((B, K), dtype=torch.float32, device=draft.device)
    if want_grad and out_grad is None:
        out_grad = torch.empty((B, K, V), dtype=torch.bfloat16, device=draft.device)
    if workspace is None:
        workspace = tts_workspace(draft.device)
    _dev(workspace, "workspace", torch.uint8)
    rc = lib().sv_tts_signal(B, K, V, code, _ptr(target), _ptr(draft), _ptr(temperature), _ptr(weights),
                             _ptr(out_kl), _ptr(out_grad) if want_grad else None, _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(rc, "sv_tts_signal")
    return out_kl, (out_grad if want_grad else None)


def verify_tree(target, draft, tokens, parents, temperature, seed: int, n_nodes=None, stream=None):
    """sv_verify_tree: returns dict(tokens [B][N], accept_len [B], path [B][N-1], flags [B])."""
    B, N, V = target.shape
    code = _dtype_code(target)
    if _dtype_code(draft) != code or draft.shape != target.shape:
        raise ValueError("target and draft must both be [B][N][V] of one dtype")
    for t, n in ((target, "target"), (draft, "draft")):
        _dev(t, n)
    for t, n in ((tokens, "tokens"), (parents, "parents"), (n_nodes, "n_nodes")):
        _dev(t, n, torch.int32)
    _dev(temperature, "temperature", torch.float32)
    dev = target.device
    out = dict(tokens=torch.empty((B, N), dtype=torch.int32, device=dev),
               accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
               path=torch.empty((B, max(N - 1, 1)), dtype=torch.int32, device=dev),
               flags=torch.empty((B,), dtype=torch.int32, device=dev))
    rc = lib().sv_verify_tree(B, N, V, code, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(parents),
                              _ptr(n_nodes), _ptr(temperature), ctypes.c_uint64(int(seed) & (2**64 - 1)),
                              _ptr(out["tokens"]), _ptr(out["accept_len"]), _ptr(out["path"]), _ptr(out["flags"]),
                              _stream(stream))
    _check(rc, "sv_verify_tree")
    return out


def status(holder: torch.Tensor, stream=None):
    """Synchronise, read and clear the status word of a workspace or AV state: (code, flags)."""
    flags = ctypes.c_uint32(0)
    rc = lib().sv_status(_ptr(holder), _stream(stream), ctypes.byref(flags))
    return rc, flags.value


def philox(seed: int, nb: int, npos: int, device="cuda", stream=None) -> torch.Tensor:
    out = torch.empty((nb, npos, 4), dtype=torch.int32, device=device)
    _check(lib().sv_philox(ctypes.c_uint64(int(seed) & (2**64 - 1)), nb, npos, _ptr(out), _stream(stream)),
           "sv_philox")
    return out


def set_launch_events(begin=None, end=None):
    """Record torch.cuda.Event pair around the row-pass kernel of later calls
    from this thread (None, None turns it off)."""
    for ev in (begin, end):
        if ev is not None and not ev.cuda_event:
            ev.record()  # torch creates the underlying event lazily
    b = None if begin is None else ctypes.c_void_p(begin.cuda_event)
    e = None if end is None else ctypes.c_void_p(end.cuda_event)
    _check(lib().sv_set_launch_events(b, e), "sv_set_launch_events")


def set_wait_test(limit_ns: int = 0, withhold: bool = False):
    """sv_set_wait_test (failure-detection tests): the device waits' limit for
    later calls from this thread (0 = default) and whether the producers
    withhold all work so that the waits run out."""
    _check(lib().sv_set_wait_test(ctypes.c_uint64(int(limit_ns)), 1 if withhold else 0), "sv_set_wait_test")


def strerror(code: int) -> str:
    return lib().sv_strerror(code).decode()
