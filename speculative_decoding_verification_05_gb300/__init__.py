"""Python binding of libspecverify (GB300 speculative-decoding verification).

Argument marshalling only: every step of the verification runs in the CUDA
kernels of ``libspecverify.so`` (built in-tree by ``build.py``). PyTorch is
used for device memory and streams. There is no CPU fallback: if the library
is missing or no CUDA device is present the calls raise.

Entry points (same names as the C ABI in ``include/specverify.h``):

* ``verify``         modified rejection sampling with temperature / top-k / top-p
* ``verify_tree``    greedy exact-match verification of a REST draft tree
* ``verify_mentor``  the lossy, KL-bounded mentor variant
* ``sample``         one draw per row from the transformed distribution

Tensors may live on the GPU (the normal case) or in (pinned) host memory; host
inputs are copied to the current device, and outputs come back to the host.
"""

import contextlib
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
# the same library built with device-side index checks (build.py --debug)
DEBUG_LIB_PATH = os.path.join(_HERE, "libspecverify_debug.so")

SPEC_OK, SPEC_EINVAL, SPEC_ECUDA, SPEC_ETIMEOUT, SPEC_EDATA, SPEC_EBOUNDS = 0, 1, 2, 3, 4, 5
SPEC_F32, SPEC_BF16 = 0, 1
PURPOSE_ACCEPT, PURPOSE_RESAMPLE, PURPOSE_DRAFT = 0, 1, 2

EXPORTED = [
    "spec_verify_workspace_size", "spec_verify", "spec_verify_lenient",
    "spec_verify_tree_workspace_size", "spec_verify_tree", "spec_tree_build", "spec_acceptance_rate",
    "spec_expected_tokens", "spec_walltime_factor", "spec_ops_factor", "spec_best_gamma",
    "spec_verify_mentor_workspace_size", "spec_verify_mentor",
    "spec_sample_workspace_size", "spec_sample",
    "spec_philox_uniform", "spec_verify_noalloc", "spec_status_string", "spec_last_cuda_error",
    "spec_version", "spec_debug_build", "spec_debug_failures", "spec_debug_withhold_copy",
]


class SpecSampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float), ("top_k", ctypes.c_int32)]


class SpecError(RuntimeError):
    pass


_libs = {}
_current = [LIB_PATH]
_lock = threading.Lock()
_P = ctypes.c_void_p
_I = ctypes.c_int
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t


def load_library(path=None):
    """Load the library (default: the one ``use_library`` selected, normally
    libspecverify.so) and declare its C signatures (no CUDA call)."""
    with _lock:
        path = path or _current[0]
        lib = _libs.get(path)
        if lib is not None:
            return lib
        if not os.path.exists(path):
            raise SpecError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        lib.spec_verify_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.spec_verify_workspace_size.restype = _SZ
        lib.spec_verify.argtypes = [_P, _P, _I, _P, _I, _I, _I, SpecSampling, _U64, _U64,
                                    _P, _P, _P, _P, _P, _P, _SZ, _P]
        lib.spec_verify.restype = _I
        lib.spec_verify_lenient.argtypes = [_P, _P, _I, _P, _I, _I, _I, SpecSampling, ctypes.c_float, _U64, _U64,
                                            _P, _P, _P, _P, _P, _P, _SZ, _P]
        lib.spec_verify_lenient.restype = _I
        lib.spec_verify_tree_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.spec_verify_tree_workspace_size.restype = _SZ
        lib.spec_verify_tree.argtypes = [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                         _P, _SZ, _P]
        lib.spec_verify_tree.restype = _I
        lib.spec_tree_build.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
        lib.spec_tree_build.restype = _I
        lib.spec_acceptance_rate.argtypes = [_P, _P, _I, _I, _I, _I, SpecSampling, _P, _P, _P, _SZ, _P]
        lib.spec_acceptance_rate.restype = _I
        _D = ctypes.c_double
        lib.spec_expected_tokens.argtypes = [_D, _I]
        lib.spec_expected_tokens.restype = _D
        lib.spec_walltime_factor.argtypes = [_D, _I, _D]
        lib.spec_walltime_factor.restype = _D
        lib.spec_ops_factor.argtypes = [_D, _I, _D]
        lib.spec_ops_factor.restype = _D
        lib.spec_best_gamma.argtypes = [_D, _D, _I]
        lib.spec_best_gamma.restype = _I
        lib.spec_verify_mentor_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.spec_verify_mentor_workspace_size.restype = _SZ
        lib.spec_verify_mentor.argtypes = [_P, _P, _I, _P, _I, _I, _I, ctypes.c_float, ctypes.c_float,
                                           _I, _U64, _U64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        lib.spec_verify_mentor.restype = _I
        lib.spec_sample_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.spec_sample_workspace_size.restype = _SZ
        lib.spec_sample.argtypes = [_P, _I, _I, _I, _I, SpecSampling, _U64, _U64, ctypes.c_uint32,
                                    ctypes.c_uint32, _P, _P, _P, _SZ, _P]
        lib.spec_sample.restype = _I
        lib.spec_verify_noalloc.argtypes = [_P, _P, _I, _P, _I, _I, _I, SpecSampling, _U64, _U64,
                                            _P, _P, _P, _P, _P, _P]
        lib.spec_verify_noalloc.restype = _I
        lib.spec_philox_uniform.argtypes = [_U64, _U64, ctypes.c_uint32, ctypes.c_uint32, _I, _P, _P]
        lib.spec_philox_uniform.restype = _I
        lib.spec_status_string.argtypes = [_I]
        lib.spec_status_string.restype = ctypes.c_char_p
        lib.spec_last_cuda_error.argtypes = []
        lib.spec_last_cuda_error.restype = ctypes.c_char_p
        lib.spec_version.argtypes = []
        lib.spec_version.restype = _I
        lib.spec_debug_build.argtypes = []
        lib.spec_debug_build.restype = _I
        lib.spec_debug_failures.argtypes = [_P]
        lib.spec_debug_failures.restype = _I
        lib.spec_debug_withhold_copy.argtypes = [_I]
        lib.spec_debug_withhold_copy.restype = _I
        _libs[path] = lib
        return lib


@contextlib.contextmanager
def use_library(path):
    """Route the calls of this module to the library at `path` (for example
    the debug build, DEBUG_LIB_PATH) inside the block."""
    load_library(path)
    with _lock:
        saved = _current[0]
        _current[0] = path
    try:
        yield
    finally:
        with _lock:
            _current[0] = saved


def _check(rc):
    if rc != SPEC_OK:
        lib = load_library()
        msg = lib.spec_status_string(rc).decode()
        if rc == SPEC_ECUDA:
            msg += ": " + lib.spec_last_cuda_error().decode()
        raise SpecError(msg)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise SpecError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


_ws_cache = {}


def workspace(nbytes, device, stream):
    """A workspace of at least nbytes, cached per (device, stream).

    The library clears what it needs at the start of every call, so the
    buffer is reused as is; calls on one stream never overlap on the GPU.
    """
    key = (device.index if device.index is not None else torch.cuda.current_device(), stream.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        with torch.cuda.stream(stream):
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


class _Staging:
    """Moves host inputs to the device and device outputs back (end-to-end calls)."""

    def __init__(self, ref):
        self.host = ref.device.type == "cpu"
        if self.host and not torch.cuda.is_available():
            raise SpecError("libspecverify needs a CUDA device; none is available")
        self.device = torch.device("cuda", torch.cuda.current_device()) if self.host else ref.device

    def dev(self, t, dtype=None):
        if t is None:
            return None
        if dtype is not None and t.dtype != dtype:
            t = t.to(dtype)
        if t.device != self.device:
            t = t.to(self.device, non_blocking=True)
        return t.contiguous()

    def out(self, shape, dtype=torch.int32):
        return torch.empty(shape, dtype=dtype, device=self.device)

    def back(self, d):
        """Device outputs to host tensors: one asynchronous copy per output
        into a reused pinned buffer, one synchronisation, then copies into
        ordinary host tensors that the caller owns."""
        if not self.host:
            return d
        tens = {k: v for k, v in d.items() if isinstance(v, torch.Tensor)}
        total = sum(_al16(v.numel() * v.element_size()) for v in tens.values())
        with _pin_lock:
            buf = _pinned.get(self.device.index)
            if buf is None or buf.numel() < total:
                buf = torch.empty(max(total, 1 << 16), dtype=torch.uint8, pin_memory=True)
                _pinned[self.device.index] = buf
            views, o = {}, 0
            for k, v in tens.items():
                n = v.numel() * v.element_size()
                h = buf[o:o + n].view(v.dtype).view(v.shape)
                h.copy_(v, non_blocking=True)
                views[k] = h
                o += _al16(n)
            torch.cuda.current_stream(self.device).synchronize()
            res = {k: (views[k].clone() if k in views else v) for k, v in d.items()}
        return res


def _al16(n):
    return (n + 15) & ~15


_pinned = {}
_pin_lock = threading.Lock()


def verify(target, draft, draft_tokens, temperature=1.0, top_p=1.0, top_k=0, seed=0, offset=0,
           debug=False, out=None, lenience=1.0):
    """Modified rejection sampling over target [B, gamma+1, V] and draft [B, gamma, V].

    Returns a dict of tensors: accepted [B], tokens [B, gamma+1], next_token [B],
    status [B] and, with debug=True, probs [B, gamma, 2] = (q(x_k), p(x_k)).
    ``out`` may pass preallocated output tensors under the same keys.
    ``lenience`` l < 1 selects spec_verify_lenient (acceptance min(1, q/(l p)),
    residual max(0, q - l p)); l = 1 is spec_verify.
    """
    lib = load_library()
    sg = _Staging(target)
    target = sg.dev(target)
    draft = sg.dev(draft) if (draft is not None and temperature != 0) else None
    toks = sg.dev(draft_tokens, torch.int32)
    B, G1, V = target.shape
    gamma = G1 - 1
    if toks.shape != (B, gamma) or (draft is not None and draft.shape != (B, gamma, V)):
        raise SpecError("shape mismatch between target, draft and draft_tokens")
    if draft is not None and draft.dtype != target.dtype:
        raise SpecError("target and draft must share a dtype")
    o = dict(out or {})
    o.setdefault("accepted", sg.out((B,)))
    o.setdefault("tokens", sg.out((B, G1)))
    o.setdefault("next_token", sg.out((B,)))
    o.setdefault("status", sg.out((B,)))
    if debug:
        o.setdefault("probs", sg.out((B, gamma, 2), torch.float32))
    dt = _dtype_code(target)
    stream = torch.cuda.current_stream(sg.device)
    nbytes = lib.spec_verify_workspace_size(B, gamma, V, dt)
    ws = workspace(nbytes, sg.device, stream)
    smp = SpecSampling(float(temperature), float(top_p), int(top_k))
    outs = (_ptr(o["accepted"]), _ptr(o["tokens"]), _ptr(o["next_token"]), _ptr(o["status"]),
            _ptr(o.get("probs")), _ptr(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    if lenience == 1.0:
        rc = lib.spec_verify(_ptr(target), _ptr(draft), dt, _ptr(toks), B, gamma, V, smp, int(seed), int(offset),
                             *outs)
    else:
        rc = lib.spec_verify_lenient(_ptr(target), _ptr(draft), dt, _ptr(toks), B, gamma, V, smp,
                                     float(lenience), int(seed), int(offset), *outs)
    _check(rc)
    return sg.back(o)


def verify_tree(target, node_tokens, parent, depth, max_depth):
    """Greedy exact-match verification of BFS-ordered draft trees [B, N, V].

    Returns accept_len [B], path_nodes [B, max_depth+1], tokens [B, max_depth+1],
    bonus [B], status [B].
    """
    lib = load_library()
    sg = _Staging(target)
    target = sg.dev(target)
    tok, par, dep = (sg.dev(t, torch.int32) for t in (node_tokens, parent, depth))
    B, N, V = target.shape
    W = max_depth + 1
    o = {"accept_len": sg.out((B,)), "path_nodes": sg.out((B, W)), "tokens": sg.out((B, W)),
         "bonus": sg.out((B,)), "status": sg.out((B,))}
    dt = _dtype_code(target)
    stream = torch.cuda.current_stream(sg.device)
    ws = workspace(lib.spec_verify_tree_workspace_size(B, N, V, dt), sg.device, stream)
    rc = lib.spec_verify_tree(_ptr(target), dt, _ptr(tok), _ptr(par), _ptr(dep), B, N, V, int(max_depth),
                              _ptr(o["accept_len"]), _ptr(o["path_nodes"]), _ptr(o["tokens"]),
                              _ptr(o["bonus"]), _ptr(o["status"]), _ptr(ws), ws.numel(),
                              ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return sg.back(o)


def tree_build(candidates, root_token, V, N, counts=None, with_mask=True):
    """REST draft trees from retrieved continuations candidates [B, C, L] (-1 ends one).

    Returns node_tokens, parent, depth [B, N] (the layout ``verify_tree`` takes),
    mask [B, N, N] uint8 (when ``with_mask``), n_nodes [B] and status [B].
    """
    lib = load_library()
    sg = _Staging(candidates)
    cand = sg.dev(candidates, torch.int32)
    root = sg.dev(root_token, torch.int32)
    cnt = sg.dev(counts, torch.int32)
    B, C, L = cand.shape
    o = {"node_tokens": sg.out((B, N)), "parent": sg.out((B, N)), "depth": sg.out((B, N)),
         "n_nodes": sg.out((B,)), "status": sg.out((B,))}
    if with_mask:
        o["mask"] = sg.out((B, N, N), torch.uint8)
    stream = torch.cuda.current_stream(sg.device)
    rc = lib.spec_tree_build(_ptr(cand), _ptr(cnt), _ptr(root), B, C, L, int(V), int(N),
                             _ptr(o["node_tokens"]), _ptr(o["parent"]), _ptr(o["depth"]), _ptr(o.get("mask")),
                             _ptr(o["n_nodes"]), _ptr(o["status"]), ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return sg.back(o)


def acceptance_rate(target, draft, temperature=1.0, top_p=1.0, top_k=0):
    """beta [B, gamma] = sum_x min(q_k(x), p_k(x)) per position (temperature > 0),
    and status [B]; the mean of beta estimates the acceptance rate alpha."""
    lib = load_library()
    sg = _Staging(target)
    target, draft = sg.dev(target), sg.dev(draft)
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft.shape != (B, gamma, V) or draft.dtype != target.dtype:
        raise SpecError("shape or dtype mismatch between target and draft")
    o = {"beta": sg.out((B, gamma), torch.float32), "status": sg.out((B,))}
    dt = _dtype_code(target)
    stream = torch.cuda.current_stream(sg.device)
    ws = workspace(lib.spec_verify_workspace_size(B, gamma, V, dt), sg.device, stream)
    rc = lib.spec_acceptance_rate(_ptr(target), _ptr(draft), dt, B, gamma, V,
                                  SpecSampling(float(temperature), float(top_p), int(top_k)),
                                  _ptr(o["beta"]), _ptr(o["status"]), _ptr(ws), ws.numel(),
                                  ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return sg.back(o)


def expected_tokens(alpha, gamma):
    """E[#tokens per target call] for acceptance rate alpha and draft length gamma."""
    return load_library().spec_expected_tokens(float(alpha), int(gamma))


def walltime_factor(alpha, gamma, c):
    """Expected walltime improvement for draft cost ratio c."""
    return load_library().spec_walltime_factor(float(alpha), int(gamma), float(c))


def ops_factor(alpha, gamma, c_hat):
    """Expected factor on the total number of operations."""
    return load_library().spec_ops_factor(float(alpha), int(gamma), float(c_hat))


def best_gamma(alpha, c, gamma_max):
    """The draft length in 1..gamma_max with the largest walltime factor."""
    return load_library().spec_best_gamma(float(alpha), float(c), int(gamma_max))


def verify_mentor(target, draft, draft_tokens, temperature=1.0, kl_bound=0.0, bisect_iters=30,
                  seed=0, offset=0, debug=False):
    """Lossy mentor verification; returns the ``verify`` outputs plus alpha and beta [B, gamma]."""
    lib = load_library()
    sg = _Staging(target)
    target, draft = sg.dev(target), sg.dev(draft)
    toks = sg.dev(draft_tokens, torch.int32)
    B, G1, V = target.shape
    gamma = G1 - 1
    if draft.shape != (B, gamma, V) or toks.shape != (B, gamma) or draft.dtype != target.dtype:
        raise SpecError("shape or dtype mismatch between target, draft and draft_tokens")
    o = {"accepted": sg.out((B,)), "tokens": sg.out((B, G1)), "next_token": sg.out((B,)),
         "status": sg.out((B,)), "alpha": sg.out((B, gamma), torch.float32),
         "beta": sg.out((B, gamma), torch.float32)}
    if debug:
        o["probs"] = sg.out((B, gamma, 2), torch.float32)
    dt = _dtype_code(target)
    stream = torch.cuda.current_stream(sg.device)
    ws = workspace(lib.spec_verify_mentor_workspace_size(B, gamma, V, dt), sg.device, stream)
    rc = lib.spec_verify_mentor(_ptr(target), _ptr(draft), dt, _ptr(toks), B, gamma, V,
                                float(temperature), float(kl_bound), int(bisect_iters), int(seed),
                                int(offset), _ptr(o["accepted"]), _ptr(o["tokens"]),
                                _ptr(o["next_token"]), _ptr(o["status"]), _ptr(o["alpha"]),
                                _ptr(o["beta"]), _ptr(o.get("probs")), _ptr(ws), ws.numel(),
                                ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return sg.back(o)


def sample(logits, temperature=1.0, top_p=1.0, top_k=0, seed=0, offset=0, pos0=0,
           purpose=PURPOSE_DRAFT):
    """One draw per row of logits [B, P, V]; returns tokens [B, P] and status [B]."""
    lib = load_library()
    sg = _Staging(logits)
    logits = sg.dev(logits)
    B, P, V = logits.shape
    o = {"tokens": sg.out((B, P)), "status": sg.out((B,))}
    dt = _dtype_code(logits)
    stream = torch.cuda.current_stream(sg.device)
    ws = workspace(lib.spec_sample_workspace_size(B, P, V, dt), sg.device, stream)
    rc = lib.spec_sample(_ptr(logits), dt, B, P, V, SpecSampling(float(temperature), float(top_p), int(top_k)),
                         int(seed), int(offset), int(pos0), int(purpose), _ptr(o["tokens"]),
                         _ptr(o["status"]), _ptr(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return sg.back(o)


def philox_uniform(seed, row0, position, purpose, n, device=None):
    """The library's uniforms U(seed, row0 + i, position, purpose), i < n (device float32)."""
    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    out = torch.empty(n, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    _check(lib.spec_philox_uniform(int(seed), int(row0), int(position), int(purpose), int(n), _ptr(out),
                                   ctypes.c_void_p(stream.cuda_stream)))
    return out


__all__ = ["use_library", "DEBUG_LIB_PATH", "philox_uniform", "verify", "verify_tree", "tree_build", "acceptance_rate", "expected_tokens",
           "walltime_factor", "ops_factor", "best_gamma", "verify_mentor", "sample", "load_library", "workspace",
           "SpecError", "SpecSampling", "EXPORTED", "LIB_PATH"]
