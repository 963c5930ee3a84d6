"""CUDA-graph capture of seam calls through the CUDA runtime (ctypes).

The pages run decode under CUDA graphs (page "Use AITER mHC for the delayed
pre block", section "Test Plan": graph mode, median of 5 x 200 calls).
``SeamGraph`` records whatever a callable launches on one stream into a
graph, reports how many kernel nodes the graph holds (the launches per
seam), and replays it.  All buffers the callable touches must be allocated
before capture; nothing here allocates device memory during capture.
"""
from __future__ import annotations

import ctypes

import torch

_CUDART_NAMES = ("libcudart.so.13", "libcudart.so.12", "libcudart.so",
                 "/usr/local/cuda/lib64/libcudart.so")
_KERNEL_NODE = 0            # cudaGraphNodeTypeKernel
_CAPTURE_THREAD_LOCAL = 1   # cudaStreamCaptureModeThreadLocal

_rt = None


def cudart():
    global _rt
    if _rt is None:
        err = None
        for name in _CUDART_NAMES:
            try:
                _rt = ctypes.CDLL(name)
                break
            except OSError as e:
                err = e
        if _rt is None:
            raise RuntimeError(f"cannot load the CUDA runtime library: {err}")
        P = ctypes.c_void_p
        _rt.cudaStreamBeginCapture.argtypes = [P, ctypes.c_int]
        _rt.cudaStreamEndCapture.argtypes = [P, ctypes.POINTER(P)]
        _rt.cudaGraphGetNodes.argtypes = [P, P, ctypes.POINTER(ctypes.c_size_t)]
        _rt.cudaGraphNodeGetType.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        _rt.cudaGraphInstantiate.argtypes = [ctypes.POINTER(P), P, ctypes.c_ulonglong]
        _rt.cudaGraphLaunch.argtypes = [P, P]
        _rt.cudaGraphExecDestroy.argtypes = [P]
        _rt.cudaGraphDestroy.argtypes = [P]
        _rt.cudaGetErrorString.argtypes = [ctypes.c_int]
        _rt.cudaGetErrorString.restype = ctypes.c_char_p
    return _rt


def _ck(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed: {cudart().cudaGetErrorString(rc).decode()} ({rc})")


class SeamGraph:
    """Capture ``fn(stream)`` into a CUDA graph on ``stream`` and instantiate it."""

    def __init__(self, fn, stream: torch.cuda.Stream):
        rt = cudart()
        self.stream = stream
        s = ctypes.c_void_p(stream.cuda_stream)
        torch.cuda.synchronize()
        _ck(rt.cudaStreamBeginCapture(s, _CAPTURE_THREAD_LOCAL), "cudaStreamBeginCapture")
        try:
            fn(stream)
        finally:
            g = ctypes.c_void_p()
            rc = rt.cudaStreamEndCapture(s, ctypes.byref(g))
        _ck(rc, "cudaStreamEndCapture")
        self.graph = g
        n = ctypes.c_size_t(0)
        _ck(rt.cudaGraphGetNodes(g, None, ctypes.byref(n)), "cudaGraphGetNodes")
        nodes = (ctypes.c_void_p * max(1, n.value))()
        _ck(rt.cudaGraphGetNodes(g, nodes, ctypes.byref(n)), "cudaGraphGetNodes")
        self.num_nodes = n.value
        kinds = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            _ck(rt.cudaGraphNodeGetType(nodes[i], ctypes.byref(t)), "cudaGraphNodeGetType")
            kinds.append(t.value)
        self.kernel_nodes = sum(1 for k in kinds if k == _KERNEL_NODE)
        ex = ctypes.c_void_p()
        _ck(rt.cudaGraphInstantiate(ctypes.byref(ex), g, 0), "cudaGraphInstantiate")
        self.exec = ex

    def replay(self, count: int = 1):
        rt = cudart()
        s = ctypes.c_void_p(self.stream.cuda_stream)
        for _ in range(count):
            _ck(rt.cudaGraphLaunch(self.exec, s), "cudaGraphLaunch")

    def close(self):
        rt = cudart()
        if getattr(self, "exec", None):
            rt.cudaGraphExecDestroy(self.exec)
            self.exec = None
        if getattr(self, "graph", None):
            rt.cudaGraphDestroy(self.graph)
            self.graph = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
