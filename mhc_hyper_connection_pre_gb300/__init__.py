"""GB300 (sm_103a) mHC seam: Python binding of libmhc.so.

Thin ctypes marshalling over the C ABI declared in ``include/mhc.h``: it
checks dtypes, devices and contiguity, allocates outputs with torch when the
caller passes none, and hands raw device pointers plus the current CUDA
stream to the library.  Every step of the seam runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If the library is missing or
cannot be loaded, every call raises.

    pre_delayed(x, pre_in, fn, bias, alpha, norm_weight=None, ...) -> dict
    post(x, y, comb, post_gate, out=None) -> Tensor
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["pre_delayed", "pre_delayed_noalloc", "post", "pre_plan", "device_status", "workspace_for",
           "library_path", "load_library", "MhcError", "SINKHORN_ITERS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libmhc.so")
SINKHORN_ITERS = 20
_STATUS = {0: "MHC_OK", 1: "MHC_ERR_INVALID_ARGUMENT", 2: "MHC_ERR_UNSUPPORTED",
           3: "MHC_ERR_CUDA", 4: "MHC_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class MhcError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libmhc.so (built by ``build.py``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libmhc.so not found at {_LIB_PATH}: build it with "
                "`python -m mhc_hyper_connection_pre_gb300.build` (no fallback exists)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.mhc_pre_delayed.argtypes = [P, P, P, P, P, P, I64, I, I, I, F, F, F, P, P, P, P, P,
                                         P, ctypes.c_size_t, P]
        lib.mhc_pre_delayed.restype = I
        lib.mhc_pre_delayed_noalloc.argtypes = [P, P, P, P, P, P, I64, I, I, I, F, F, F, P, P, P, P, P, P]
        lib.mhc_pre_delayed_noalloc.restype = I
        lib.mhc_pre_workspace_bytes.argtypes = [I64, I, I]
        lib.mhc_pre_workspace_bytes.restype = ctypes.c_size_t
        lib.mhc_post.argtypes = [P, P, P, P, I64, I, I, P, P]
        lib.mhc_post.restype = I
        lib.mhc_post_pre_delayed.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I, I, I, F, F, F, P, P, P, P, P,
                                             P, ctypes.c_size_t, P]
        lib.mhc_post_pre_delayed.restype = I
        lib.mhc_pre.argtypes = [P, P, P, P, P, I64, I, I, I, F, F, F, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.mhc_pre.restype = I
        lib.mhc_pre_delayed_broadcast.argtypes = lib.mhc_pre_delayed.argtypes
        lib.mhc_pre_delayed_broadcast.restype = I
        lib.mhc_pre_broadcast.argtypes = lib.mhc_pre.argtypes
        lib.mhc_pre_broadcast.restype = I
        lib.mhc_post_broadcast.argtypes = lib.mhc_post.argtypes
        lib.mhc_post_broadcast.restype = I
        lib.mhc_pre_packed_bytes.argtypes = [I, I]
        lib.mhc_pre_packed_bytes.restype = ctypes.c_size_t
        lib.mhc_pre_pack.argtypes = [P, I, I, P, ctypes.c_size_t, P]
        lib.mhc_pre_pack.restype = I
        lib.mhc_pre_delayed_packed.argtypes = [P, P, P, P, ctypes.c_size_t, P, P, P, I64, I, I, I, F, F, F,
                                               P, P, P, P, P, P]
        lib.mhc_pre_delayed_packed.restype = I
        lib.mhc_seam_host_workspace_bytes.argtypes = [I64, I, I]
        lib.mhc_seam_host_workspace_bytes.restype = ctypes.c_size_t
        lib.mhc_seam_host.argtypes = [P, P, P, P, P, P, P, I64, I, I, I, F, F, F, P, P, P, P, P, P,
                                      ctypes.c_size_t, P]
        lib.mhc_seam_host.restype = I
        lib.mhc_status_string.argtypes = [I]
        lib.mhc_status_string.restype = ctypes.c_char_p
        lib.mhc_pre_delayed_plan.argtypes = [I64, I, I, P, P, P, P]
        lib.mhc_pre_delayed_plan.restype = I
        lib.mhc_version.argtypes = []
        lib.mhc_version.restype = I
        lib.mhc_device_status.argtypes = []
        lib.mhc_device_status.restype = I
        lib.mhc_set_launch_overlap.argtypes = [I]
        lib.mhc_set_launch_overlap.restype = I
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        lib = load_library()
        raise MhcError(fn, status, lib.mhc_status_string(status).decode())


def _dev_ptr(t: torch.Tensor | None, name: str, dtype: torch.dtype, device) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on the same CUDA device as x (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _device_index(device) -> int:
    d = torch.device(device)
    return d.index if d.index is not None else torch.cuda.current_device()


def workspace_for(T: int, n: int, C: int, device, stream=None) -> torch.Tensor | None:
    """A cached device workspace big enough for ``mhc_pre_delayed`` at this
    shape (None when the shape needs none).  One buffer per (device, stream),
    grown on demand and allocated on that stream, so calls on different
    streams never share one; ``stream`` defaults to the device's current
    stream."""
    dev = _device_index(device)
    with torch.cuda.device(dev):
        need = int(load_library().mhc_pre_workspace_bytes(T, n, C))
        if need == 0:
            return None
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        key = (dev, s.cuda_stream)
        buf = _workspaces.get(key)
        if buf is None or buf.numel() < need:
            with torch.cuda.stream(s):
                buf = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", dev))
            _workspaces[key] = buf
    return buf


def _stream_ptr(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _pre_outputs(o: dict, T: int, n: int, C: int, dev, return_logits: bool) -> dict:
    M = 2 * n + n * n
    if "pre" not in o:
        o["pre"] = torch.empty(T, n, dtype=torch.float32, device=dev)
    if "post" not in o:
        o["post"] = torch.empty(T, n, dtype=torch.float32, device=dev)
    if "comb" not in o:
        o["comb"] = torch.empty(T, n, n, dtype=torch.float32, device=dev)
    if "layer_input" not in o:
        o["layer_input"] = torch.empty(T, C, dtype=torch.bfloat16, device=dev)
    if return_logits and "logits" not in o:
        o["logits"] = torch.empty(T, M, dtype=torch.float32, device=dev)
    return o


def _pre_call(fname: str, x: torch.Tensor, pre_in: torch.Tensor | None, fn: torch.Tensor, bias: torch.Tensor,
              alpha: torch.Tensor, norm_weight: torch.Tensor | None, T: int, n: int, C: int, sinkhorn_iters: int,
              rms_eps: float, norm_eps: float, sinkhorn_eps: float, out: dict | None, return_logits: bool,
              workspace: torch.Tensor | None, stream) -> dict:
    """Marshal one pre-block call (delayed or not, four-stream or broadcast
    x) into the C entry point ``fname``."""
    lib = load_library()
    dev = x.device
    M = 2 * n + n * n
    o = _pre_outputs(dict(out) if out else {}, T, n, C, dev, return_logits)
    if fn.numel() != M * n * C or bias.numel() != M or alpha.numel() != 3:
        raise ValueError("fn / bias / alpha have the wrong number of elements")
    if pre_in is not None and pre_in.numel() != T * n:
        raise ValueError("pre_in must have T * n elements")
    if norm_weight is not None and norm_weight.numel() != C:
        raise ValueError("norm_weight must have C elements")
    args = [_dev_ptr(x, "x", torch.bfloat16, dev)]
    if pre_in is not None:
        args.append(_dev_ptr(pre_in, "pre_in", torch.float32, dev))
    args += [_dev_ptr(fn, "fn", torch.float32, dev), _dev_ptr(bias, "bias", torch.float32, dev),
             _dev_ptr(alpha, "alpha", torch.float32, dev), _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, dev)]
    outs = [_dev_ptr(o["pre"], "pre", torch.float32, dev), _dev_ptr(o["post"], "post", torch.float32, dev),
            _dev_ptr(o["comb"], "comb", torch.float32, dev),
            _dev_ptr(o["layer_input"], "layer_input", torch.bfloat16, dev),
            _dev_ptr(o.get("logits"), "logits", torch.float32, dev)]
    if workspace is None:
        workspace = workspace_for(T, n, C, dev, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8, dev)
        ws_bytes = workspace.numel()
    with torch.cuda.device(dev):
        st = getattr(lib, fname)(*args, T, n, C, int(sinkhorn_iters), float(rms_eps), float(norm_eps),
                                 float(sinkhorn_eps), *outs, ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    _check(fname, st)
    return o


def _shape3(x: torch.Tensor):
    if x.dim() != 3:
        raise ValueError("x must be [T, n, C]")
    return x.shape


def _shape2(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("x must be [T, C] (the model-entry broadcast seam)")
    return x.shape


def pre_delayed(x: torch.Tensor, pre_in: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor,
                alpha: torch.Tensor, norm_weight: torch.Tensor | None = None, *,
                sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6,
                norm_eps: float = 1e-6, sinkhorn_eps: float = 1e-6, out: dict | None = None,
                return_logits: bool = False, workspace: torch.Tensor | None = None,
                stream=None) -> dict:
    """Delayed mHC pre block (``mhc_pre_delayed`` in include/mhc.h).

    x bf16 [T, 4, C]; pre_in fp32 [T, 4] (previous seam's pre-mix);
    fn fp32 [24, 4C]; bias fp32 [24]; alpha fp32 [3]; norm_weight bf16 [C]
    or None.  Returns {"pre", "post", "comb", "layer_input"[, "logits"]}
    (``out`` may supply preallocated tensors under the same keys).
    ``workspace``: uint8 device buffer of at least ``mhc_pre_workspace_bytes``;
    by default a cached per-device buffer is used.
    """
    T, n, C = _shape3(x)
    return _pre_call("mhc_pre_delayed", x, pre_in, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters,
                     rms_eps, norm_eps, sinkhorn_eps, out, return_logits, workspace, stream)


def pre(x: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor, alpha: torch.Tensor,
        norm_weight: torch.Tensor | None = None, *, sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6,
        norm_eps: float = 1e-6, sinkhorn_eps: float = 1e-6, out: dict | None = None, return_logits: bool = False,
        workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Non-delayed mHC pre block (``mhc_pre``): as ``pre_delayed`` but the
    collapse uses each token's own pre-mix (no pre_in)."""
    T, n, C = _shape3(x)
    return _pre_call("mhc_pre", x, None, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters, rms_eps,
                     norm_eps, sinkhorn_eps, out, return_logits, workspace, stream)


def pre_pack(fn: torch.Tensor, n: int = 4, C: int | None = None, *, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """Pack fn into the tensor-core kernel's bf16 planes (``mhc_pre_pack``);
    returns the uint8 device buffer for ``pre_delayed_packed``.  Re-pack
    after writing fn."""
    lib = load_library()
    if C is None:
        C = fn.numel() // ((2 * n + n * n) * n)
    need = int(lib.mhc_pre_packed_bytes(n, C))
    if need == 0:
        raise ValueError(f"no packed planes for n={n}, C={C} (the tensor-core kernel does not take it)")
    dev = fn.device
    if out is None:
        out = torch.empty(need, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = lib.mhc_pre_pack(_dev_ptr(fn, "fn", torch.float32, dev), n, C,
                              _dev_ptr(out, "packed", torch.uint8, dev), out.numel(), _stream_ptr(stream, dev))
    _check("mhc_pre_pack", st)
    return out


def pre_delayed_packed(x: torch.Tensor, pre_in: torch.Tensor, fn: torch.Tensor, packed: torch.Tensor,
                       bias: torch.Tensor, alpha: torch.Tensor, norm_weight: torch.Tensor | None = None, *,
                       sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6, norm_eps: float = 1e-6,
                       sinkhorn_eps: float = 1e-6, out: dict | None = None, return_logits: bool = False,
                       stream=None) -> dict:
    """``pre_delayed`` with fn's planes packed ahead by ``pre_pack``
    (``mhc_pre_delayed_packed``): the same bits, no per-call conversion, no
    workspace."""
    lib = load_library()
    T, n, C = _shape3(x)
    dev = x.device
    M = 2 * n + n * n
    o = _pre_outputs(dict(out) if out else {}, T, n, C, dev, return_logits)
    if fn.numel() != M * n * C or bias.numel() != M or alpha.numel() != 3 or pre_in.numel() != T * n:
        raise ValueError("pre_in / fn / bias / alpha have the wrong number of elements")
    if norm_weight is not None and norm_weight.numel() != C:
        raise ValueError("norm_weight must have C elements")
    with torch.cuda.device(dev):
        st = lib.mhc_pre_delayed_packed(
            _dev_ptr(x, "x", torch.bfloat16, dev), _dev_ptr(pre_in, "pre_in", torch.float32, dev),
            _dev_ptr(fn, "fn", torch.float32, dev), _dev_ptr(packed, "packed", torch.uint8, dev), packed.numel(),
            _dev_ptr(bias, "bias", torch.float32, dev), _dev_ptr(alpha, "alpha", torch.float32, dev),
            _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, dev), T, n, C, int(sinkhorn_iters),
            float(rms_eps), float(norm_eps), float(sinkhorn_eps), _dev_ptr(o["pre"], "pre", torch.float32, dev),
            _dev_ptr(o["post"], "post", torch.float32, dev), _dev_ptr(o["comb"], "comb", torch.float32, dev),
            _dev_ptr(o["layer_input"], "layer_input", torch.bfloat16, dev),
            _dev_ptr(o.get("logits"), "logits", torch.float32, dev), _stream_ptr(stream, dev))
    _check("mhc_pre_delayed_packed", st)
    return o


def pre_delayed_broadcast(x: torch.Tensor, pre_in: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor,
                          alpha: torch.Tensor, norm_weight: torch.Tensor | None = None, *, n: int = 4,
                          sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6, norm_eps: float = 1e-6,
                          sinkhorn_eps: float = 1e-6, out: dict | None = None, return_logits: bool = False,
                          workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Model-entry broadcast seam, delayed (``mhc_pre_delayed_broadcast``):
    ``pre_delayed`` on x bf16 [T, C] read as all n streams; pre_in is the
    model-entry pre-mix [T, n]."""
    T, C = _shape2(x)
    return _pre_call("mhc_pre_delayed_broadcast", x, pre_in, fn, bias, alpha, norm_weight, T, n, C,
                     sinkhorn_iters, rms_eps, norm_eps, sinkhorn_eps, out, return_logits, workspace, stream)


def pre_broadcast(x: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor, alpha: torch.Tensor,
                  norm_weight: torch.Tensor | None = None, *, n: int = 4, sinkhorn_iters: int = SINKHORN_ITERS,
                  rms_eps: float = 1e-6, norm_eps: float = 1e-6, sinkhorn_eps: float = 1e-6,
                  out: dict | None = None, return_logits: bool = False, workspace: torch.Tensor | None = None,
                  stream=None) -> dict:
    """Model-entry broadcast seam, non-delayed (``mhc_pre_broadcast``)."""
    T, C = _shape2(x)
    return _pre_call("mhc_pre_broadcast", x, None, fn, bias, alpha, norm_weight, T, n, C, sinkhorn_iters,
                     rms_eps, norm_eps, sinkhorn_eps, out, return_logits, workspace, stream)


def post_pre_delayed(x: torch.Tensor, y: torch.Tensor, comb: torch.Tensor, post: torch.Tensor,
                     pre_in: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor, alpha: torch.Tensor,
                     norm_weight: torch.Tensor | None = None, *, x_new: torch.Tensor | None = None,
                     sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6, norm_eps: float = 1e-6,
                     sinkhorn_eps: float = 1e-6, out: dict | None = None, return_logits: bool = False,
                     workspace: torch.Tensor | None = None, stream=None) -> dict:
    """One seam boundary (``mhc_post_pre_delayed``): the previous seam's post
    on (x, y, comb, post) into ``x_new`` (default: a new tensor; may be x),
    then this seam's delayed pre on x_new.  Returns the pre outputs as
    ``pre_delayed`` does, plus "x_new".  ``out["comb"]`` / ``out["post"]``
    may be the very tensors passed as comb / post."""
    lib = load_library()
    if x.dim() != 3:
        raise ValueError("x must be [T, n, C]")
    T, n, C = x.shape
    dev = x.device
    M = 2 * n + n * n
    if x_new is None:
        x_new = torch.empty_like(x)
    o = dict(out) if out else {}
    if "pre" not in o:
        o["pre"] = torch.empty(T, n, dtype=torch.float32, device=dev)
    if "post" not in o:
        o["post"] = torch.empty(T, n, dtype=torch.float32, device=dev)
    if "comb" not in o:
        o["comb"] = torch.empty(T, n, n, dtype=torch.float32, device=dev)
    if "layer_input" not in o:
        o["layer_input"] = torch.empty(T, C, dtype=torch.bfloat16, device=dev)
    if return_logits and "logits" not in o:
        o["logits"] = torch.empty(T, M, dtype=torch.float32, device=dev)
    if y.numel() != T * C or comb.numel() != T * n * n or post.numel() != T * n or x_new.shape != x.shape:
        raise ValueError("y / comb / post / x_new have the wrong shape")
    if pre_in.numel() != T * n or fn.numel() != M * n * C or bias.numel() != M or alpha.numel() != 3:
        raise ValueError("pre_in / fn / bias / alpha have the wrong number of elements")
    if norm_weight is not None and norm_weight.numel() != C:
        raise ValueError("norm_weight must have C elements")
    args = [_dev_ptr(x, "x", torch.bfloat16, dev), _dev_ptr(y, "y", torch.bfloat16, dev),
            _dev_ptr(comb, "comb", torch.float32, dev), _dev_ptr(post, "post", torch.float32, dev),
            _dev_ptr(x_new, "x_new", torch.bfloat16, dev), _dev_ptr(pre_in, "pre_in", torch.float32, dev),
            _dev_ptr(fn, "fn", torch.float32, dev), _dev_ptr(bias, "bias", torch.float32, dev),
            _dev_ptr(alpha, "alpha", torch.float32, dev), _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, dev)]
    outs = [_dev_ptr(o["pre"], "pre", torch.float32, dev), _dev_ptr(o["post"], "post", torch.float32, dev),
            _dev_ptr(o["comb"], "comb", torch.float32, dev),
            _dev_ptr(o["layer_input"], "layer_input", torch.bfloat16, dev),
            _dev_ptr(o.get("logits"), "logits", torch.float32, dev)]
    if workspace is None:
        workspace = workspace_for(T, n, C, dev, stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8, dev)
        ws_bytes = workspace.numel()
    with torch.cuda.device(dev):
        st = lib.mhc_post_pre_delayed(*args, T, n, C, int(sinkhorn_iters), float(rms_eps), float(norm_eps),
                                      float(sinkhorn_eps), *outs, ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    _check("mhc_post_pre_delayed", st)
    o["x_new"] = x_new
    return o


def pre_delayed_noalloc(x: torch.Tensor, pre_in: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor,
                        alpha: torch.Tensor, norm_weight: torch.Tensor | None = None, *,
                        sinkhorn_iters: int = SINKHORN_ITERS, rms_eps: float = 1e-6,
                        norm_eps: float = 1e-6, sinkhorn_eps: float = 1e-6, out: dict,
                        return_logits: bool = False, stream=None) -> dict:
    """``mhc_pre_delayed_noalloc``: the delayed pre block for callers that
    cannot allocate device memory (the library uses a fixed scratch array of
    ``MHC_NOALLOC_SCRATCH_BYTES`` per GPU instead of a workspace).  ``out``
    must hold preallocated "pre", "post", "comb", "layer_input" (and
    "logits" when ``return_logits``); nothing is allocated here."""
    lib = load_library()
    if x.dim() != 3:
        raise ValueError("x must be [T, n, C]")
    T, n, C = x.shape
    dev = x.device
    args = [
        _dev_ptr(x, "x", torch.bfloat16, dev), _dev_ptr(pre_in, "pre_in", torch.float32, dev),
        _dev_ptr(fn, "fn", torch.float32, dev), _dev_ptr(bias, "bias", torch.float32, dev),
        _dev_ptr(alpha, "alpha", torch.float32, dev),
        _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, dev),
    ]
    outs = [_dev_ptr(out["pre"], "pre", torch.float32, dev), _dev_ptr(out["post"], "post", torch.float32, dev),
            _dev_ptr(out["comb"], "comb", torch.float32, dev),
            _dev_ptr(out["layer_input"], "layer_input", torch.bfloat16, dev),
            _dev_ptr(out.get("logits") if return_logits else None, "logits", torch.float32, dev)]
    # the library's scratch address belongs to the current device: make x's current
    with torch.cuda.device(dev):
        st = lib.mhc_pre_delayed_noalloc(*args, T, n, C, int(sinkhorn_iters), float(rms_eps), float(norm_eps),
                                         float(sinkhorn_eps), *outs, _stream_ptr(stream, dev))
    _check("mhc_pre_delayed_noalloc", st)
    return out


def _post_call(fname: str, x: torch.Tensor, y: torch.Tensor, comb: torch.Tensor, post_gate: torch.Tensor,
               T: int, n: int, C: int, out: torch.Tensor, stream) -> torch.Tensor:
    dev = x.device
    if y.numel() != T * C or comb.numel() != T * n * n or post_gate.numel() != T * n or \
            tuple(out.shape) != (T, n, C):
        raise ValueError("y / comb / post / out have the wrong shape")
    with torch.cuda.device(dev):
        st = getattr(load_library(), fname)(
            _dev_ptr(x, "x", torch.bfloat16, dev), _dev_ptr(y, "y", torch.bfloat16, dev),
            _dev_ptr(comb, "comb", torch.float32, dev), _dev_ptr(post_gate, "post", torch.float32, dev), T, n, C,
            _dev_ptr(out, "out", torch.bfloat16, dev), _stream_ptr(stream, dev))
    _check(fname, st)
    return out


def post(x: torch.Tensor, y: torch.Tensor, comb: torch.Tensor, post_gate: torch.Tensor, *,
         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """mHC post block (``mhc_post``): x_new[j] = sum_i comb[i, j] x[i] + post[j] y.
    x bf16 [T, 4, C]; y bf16 [T, C]; comb fp32 [T, 4, 4]; post_gate fp32 [T, 4].
    ``out`` may be ``x`` itself (in place)."""
    T, n, C = _shape3(x)
    if out is None:
        out = torch.empty_like(x)
    return _post_call("mhc_post", x, y, comb, post_gate, T, n, C, out, stream)


def post_broadcast(x: torch.Tensor, y: torch.Tensor, comb: torch.Tensor, post_gate: torch.Tensor, *,
                   n: int = 4, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Model-entry broadcast seam's post (``mhc_post_broadcast``): ``post`` on
    x bf16 [T, C] read as all n streams; returns x_new bf16 [T, n, C]."""
    T, C = _shape2(x)
    if out is None:
        out = torch.empty(T, n, C, dtype=torch.bfloat16, device=x.device)
    return _post_call("mhc_post_broadcast", x, y, comb, post_gate, T, n, C, out, stream)


def _host_ptr(t: torch.Tensor | None, name: str, dtype: torch.dtype) -> int | None:
    if t is None:
        return None
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a page-locked (pinned) host tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    return t.data_ptr()


def seam_host(x: torch.Tensor, y: torch.Tensor, pre_in: torch.Tensor, fn: torch.Tensor, bias: torch.Tensor,
              alpha: torch.Tensor, norm_weight: torch.Tensor | None = None, *, sinkhorn_iters: int = SINKHORN_ITERS,
              rms_eps: float = 1e-6, norm_eps: float = 1e-6, sinkhorn_eps: float = 1e-6, out: dict | None = None,
              outputs: tuple = ("x_new", "pre"), workspace: torch.Tensor | None = None, device=None,
              stream=None) -> dict:
    """One seam on pinned HOST activations (``mhc_seam_host``): the delayed
    pre block, then the post block, with the chunked copies and kernels
    overlapped inside the library.  x bf16 [T, 4, C], y bf16 [T, C], pre_in
    fp32 [T, 4] (pinned host); fn, bias, alpha, norm_weight on the device.
    Returns pinned host tensors {"x_new", "pre"[, "post", "comb",
    "layer_input"]} (``outputs`` names the optional ones to copy back;
    ``out`` may supply them)."""
    lib = load_library()
    if x.dim() != 3:
        raise ValueError("x must be [T, n, C]")
    T, n, C = x.shape
    dev = fn.device if device is None else torch.device(device)
    o = dict(out) if out else {}
    shapes = {"x_new": ((T, n, C), torch.bfloat16), "pre": ((T, n), torch.float32),
              "post": ((T, n), torch.float32), "comb": ((T, n, n), torch.float32),
              "layer_input": ((T, C), torch.bfloat16)}
    for k in ("x_new", "pre") + tuple(k for k in outputs if k not in ("x_new", "pre")):
        if k not in o:
            shp, dt = shapes[k]
            o[k] = torch.empty(shp, dtype=dt, pin_memory=True)
    if workspace is None:
        di = _device_index(dev)
        with torch.cuda.device(di):
            need = int(lib.mhc_seam_host_workspace_bytes(T, n, C))
            s = stream if stream is not None else torch.cuda.current_stream(di)
            key = ("seam_host", di, s.cuda_stream)
            workspace = _workspaces.get(key)
            if workspace is None or workspace.numel() < need:
                with torch.cuda.stream(s):
                    workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=torch.device("cuda", di))
                _workspaces[key] = workspace
    with torch.cuda.device(dev):
        st = lib.mhc_seam_host(
            _host_ptr(x, "x", torch.bfloat16), _host_ptr(y, "y", torch.bfloat16),
            _host_ptr(pre_in, "pre_in", torch.float32), _dev_ptr(fn, "fn", torch.float32, dev),
            _dev_ptr(bias, "bias", torch.float32, dev), _dev_ptr(alpha, "alpha", torch.float32, dev),
            _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, dev), T, n, C, int(sinkhorn_iters),
            float(rms_eps), float(norm_eps), float(sinkhorn_eps), _host_ptr(o["x_new"], "x_new", torch.bfloat16),
            _host_ptr(o["pre"], "pre", torch.float32), _host_ptr(o.get("post"), "post", torch.float32),
            _host_ptr(o.get("comb"), "comb", torch.float32),
            _host_ptr(o.get("layer_input"), "layer_input", torch.bfloat16),
            _dev_ptr(workspace, "workspace", torch.uint8, dev), workspace.numel(), _stream_ptr(stream, dev))
    _check("mhc_seam_host", st)
    return o


def device_status() -> int:
    """Synchronise the current device and read-and-clear the library's device
    status word (``mhc_device_status``): 0 = OK, 4 = a bounded in-kernel wait
    timed out since the last check."""
    return load_library().mhc_device_status()


def set_launch_overlap(enable: bool) -> bool:
    """Turn programmatic dependent launch of the decode pre kernel and of
    ``post`` on or off (``mhc_set_launch_overlap``); returns the previous
    setting.  While on, fn, bias, alpha and norm_w must not be written by the
    kernel issued just before ``pre_delayed`` on the same stream."""
    return bool(load_library().mhc_set_launch_overlap(1 if enable else 0))


def pre_plan(T: int, n: int = 4, C: int = 5120) -> dict:
    """Launch plan of ``mhc_pre_delayed`` for a shape (``mhc_pre_delayed_plan``)."""
    lib = load_library()
    k, g, c, tt = (ctypes.c_int(0) for _ in range(4))
    st = lib.mhc_pre_delayed_plan(T, n, C, ctypes.byref(k), ctypes.byref(g), ctypes.byref(c),
                                  ctypes.byref(tt))
    _check("mhc_pre_delayed_plan", st)
    return {"kernel": k.value, "grid": g.value, "cluster": c.value, "tokens_per_tile": tt.value}
