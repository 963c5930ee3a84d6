"""CPU oracle for the mHC seam -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports it, and it never imports them.

The arithmetic lives in ``mhc_oracle.c`` (plain C: fp64, plus the exact fp32
collapse); this module only compiles it with gcc, loads it with ctypes and
converts numpy arrays.  Each function cites the passage of the vLLM pull
request pages it restates ("Use AITER mHC for the delayed pre block" #56503;
"Fix TileLang mHC pre on 64-wide wavefronts" #56342).

Pins: see ``tests/test_oracle_pins.py``.  Not pinned: whether the gate and
Sinkhorn readings equal the production model's code, which the pages do not
print (parity unpinned against that model).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# Reading of the pages' constants (RMS eps 1e-6 for both the projection scale
# and the fold; eps added once to the comb after the first row softmax).
RMS_EPS = 1e-6
NORM_EPS = 1e-6
SINKHORN_EPS = 1e-6
SINKHORN_ITERS = 20

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mhc_oracle.c`` into ``_build/liboracle.so`` with gcc.

    ``-ffp-contract=off`` keeps every fp32 product of the collapse rounded on
    its own (no fused multiply-add), as the bit-exact collapse requires.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.mhc_oracle_pre_delayed.argtypes = [
                P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                P, P, P, P, P, P, ctypes.c_int]
            lib.mhc_oracle_pre_delayed.restype = ctypes.c_int
            lib.mhc_oracle_gates_from_logits.argtypes = [
                P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P, P]
            lib.mhc_oracle_gates_from_logits.restype = ctypes.c_int
            lib.mhc_oracle_post.argtypes = [
                P, P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
            lib.mhc_oracle_post.restype = ctypes.c_int
            lib.mhc_oracle_bf16_round.argtypes = [P, ctypes.c_int64, P]
            lib.mhc_oracle_bf16_round.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def bf16_round(v) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even); returns uint16 bits."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().mhc_oracle_bf16_round(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16)."""
    b = _c(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def pre_delayed(x_bits, pre_in, fn, bias, alpha, norm_w_bits=None, *,
                iters=SINKHORN_ITERS, rms_eps=RMS_EPS, norm_eps=NORM_EPS,
                sinkhorn_eps=SINKHORN_EPS, nthreads=1) -> dict:
    """Delayed mHC pre block for every token (the #56503 page: the block
    collapses a sublayer's input with the previous seam's pre-mix and returns
    this seam's pre-mix, the post and comb gates and the collapsed
    layer_input; the
    #56342 page, "Measurements": the optional RMSNorm fold, rounded once).

    x_bits: uint16 [T, n, C] (bf16 bits); pre_in: float32 [T, n];
    fn: float32 [2n+n^2, n*C]; bias: float32 [2n+n^2]; alpha: float32 [3];
    norm_w_bits: uint16 [C] or None (no fold).

    Returns fp64 ``logits`` [T, M], ``pre`` [T, n], ``post`` [T, n],
    ``comb`` [T, n, n]; the exact fp32 collapse ``h32`` [T, C]; and
    ``layer_input`` as bf16 bits [T, C].
    """
    x_bits = _c(x_bits, np.uint16)
    T, n, C = x_bits.shape
    M = 2 * n + n * n
    pre_in = _c(pre_in, np.float32).reshape(T, n)
    fn = _c(fn, np.float32).reshape(M, n * C)
    bias = _c(bias, np.float32).reshape(M)
    alpha = _c(alpha, np.float32).reshape(3)
    nw = None if norm_w_bits is None else _c(norm_w_bits, np.uint16).reshape(C)
    out = {
        "logits": np.empty((T, M), np.float64),
        "pre": np.empty((T, n), np.float64),
        "post": np.empty((T, n), np.float64),
        "comb": np.empty((T, n, n), np.float64),
        "h32": np.empty((T, C), np.float32),
        "layer_input": np.empty((T, C), np.uint16),
    }
    rc = _load().mhc_oracle_pre_delayed(
        _ptr(x_bits), _ptr(pre_in), _ptr(fn), _ptr(bias), _ptr(alpha), _ptr(nw),
        T, n, C, int(iters), float(rms_eps), float(norm_eps), float(sinkhorn_eps),
        _ptr(out["logits"]), _ptr(out["pre"]), _ptr(out["post"]), _ptr(out["comb"]),
        _ptr(out["h32"]), _ptr(out["layer_input"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad arguments to pre_delayed")
    return out


def pre_nondelayed(x_bits, fn, bias, alpha, norm_w_bits=None, *, pre_mix=None, iters=SINKHORN_ITERS,
                   rms_eps=RMS_EPS, norm_eps=NORM_EPS, sinkhorn_eps=SINKHORN_EPS, nthreads=1) -> dict:
    """Non-delayed mHC pre block (the #56503 page, "Why V4.1 cannot just reuse
    MHCPreOp": the V4 block collapses a sublayer's input with the pre-mix it
    computes itself, where V4.1 uses the previous seam's): the gates of
    ``pre_delayed`` (which do not depend on the incoming pre-mix) and the
    collapse with this block's own pre-mix rounded to fp32 -- the kernel's
    stored values.  ``pre_mix`` (float32 [T, n]) replaces that rounding with
    given values (a kernel's own pre, for a layered bit-exact check of the
    collapse); otherwise the fp64 pre is rounded to nearest fp32 here.

    A composition of ``pre_delayed`` calls, so it rests on that function's
    pins; ``tests/test_oracle_pins.py`` adds the invariants specific to it."""
    x_bits = _c(x_bits, np.uint16)
    T, n, C = x_bits.shape
    gates = pre_delayed(x_bits, np.zeros((T, n), np.float32), fn, bias, alpha, norm_w_bits, iters=iters,
                        rms_eps=rms_eps, norm_eps=norm_eps, sinkhorn_eps=sinkhorn_eps, nthreads=nthreads)
    mix = gates["pre"].astype(np.float32) if pre_mix is None else _c(pre_mix, np.float32).reshape(T, n)
    coll = pre_delayed(x_bits, mix, fn, bias, alpha, norm_w_bits, iters=iters, rms_eps=rms_eps,
                       norm_eps=norm_eps, sinkhorn_eps=sinkhorn_eps, nthreads=nthreads)
    out = dict(gates)
    out["h32"], out["layer_input"], out["pre_mix"] = coll["h32"], coll["layer_input"], mix
    return out


def broadcast_streams(x_bits, n: int = 4) -> np.ndarray:
    """The model-entry residual: n copies of the hidden state x [T, C] as the
    streams of a [T, n, C] residual (the #56503 page, "Approach": at the
    model's entry the projection's operand is x itself, narrower than the
    streams)."""
    x_bits = _c(x_bits, np.uint16)
    T, C = x_bits.shape
    return np.ascontiguousarray(np.broadcast_to(x_bits[:, None, :], (T, n, C)))


def pre_delayed_broadcast(x_bits, pre_in, fn, bias, alpha, norm_w_bits=None, n: int = 4, **kw) -> dict:
    """Delayed pre block of the model-entry broadcast seam: by definition the
    delayed block on the broadcast residual (pre_in: the model-entry
    pre-mix, the #56503 page, "Test Plan")."""
    return pre_delayed(broadcast_streams(x_bits, n), pre_in, fn, bias, alpha, norm_w_bits, **kw)


def pre_nondelayed_broadcast(x_bits, fn, bias, alpha, norm_w_bits=None, n: int = 4, **kw) -> dict:
    """Non-delayed pre block of the model-entry broadcast seam (definition)."""
    return pre_nondelayed(broadcast_streams(x_bits, n), fn, bias, alpha, norm_w_bits, **kw)


def gates_from_logits(logits, n=4, *, iters=SINKHORN_ITERS,
                      sinkhorn_eps=SINKHORN_EPS) -> dict:
    """pre = sigmoid(l[:n]), post = 2 sigmoid(l[n:2n]), comb = Sinkhorn of
    l[2n:] as an n x n row-major matrix (the #56503 page, "Approach": one
    stage forms the post and comb gates and runs all the Sinkhorn iterations,
    20 of them); fp64 from the given logits."""
    lg = _c(logits, np.float64)
    M = 2 * n + n * n
    lg = lg.reshape(-1, M)
    T = lg.shape[0]
    pre = np.empty((T, n), np.float64)
    post = np.empty((T, n), np.float64)
    comb = np.empty((T, n, n), np.float64)
    rc = _load().mhc_oracle_gates_from_logits(
        _ptr(lg), T, n, int(iters), float(sinkhorn_eps), _ptr(pre), _ptr(post), _ptr(comb))
    if rc != 0:
        raise ValueError("oracle: bad arguments to gates_from_logits")
    return {"pre": pre, "post": post, "comb": comb}


def post(x_bits, y_bits, comb, post_gate, *, nthreads=1) -> tuple[np.ndarray, np.ndarray]:
    """mHC post (MHCPostOp on the #56503 page): x_new[j] = bf16(sum_i
    comb[i, j] x[i] + post[j] y), exact in fp64 then rounded once.
    Returns (x_new bf16 bits [T, n, C], exact fp64 values [T, n, C])."""
    x_bits = _c(x_bits, np.uint16)
    T, n, C = x_bits.shape
    y_bits = _c(y_bits, np.uint16).reshape(T, C)
    comb = _c(comb, np.float32).reshape(T, n, n)
    post_gate = _c(post_gate, np.float32).reshape(T, n)
    xn = np.empty((T, n, C), np.uint16)
    x64 = np.empty((T, n, C), np.float64)
    rc = _load().mhc_oracle_post(_ptr(x_bits), _ptr(y_bits), _ptr(comb), _ptr(post_gate),
                                 T, n, C, _ptr(xn), _ptr(x64), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad arguments to post")
    return xn, x64


def post_broadcast(x_bits, y_bits, comb, post_gate, n: int = 4, *, nthreads=1):
    """Post of the model-entry broadcast seam: by definition ``post`` on the
    broadcast residual; returns x_new [T, n, C] as ``post`` does."""
    return post(broadcast_streams(x_bits, n), y_bits, comb, post_gate, nthreads=nthreads)
