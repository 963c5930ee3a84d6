"""CUDA-graph capture of seam calls through the CUDA runtime (ctypes).

The pages run decode under CUDA graphs (page "Use AITER mHC for the delayed
pre block", section "Test Plan": graph mode, median of 5 x 200 calls).
``SeamGraph`` records whatever a callable launches on one stream into a
graph, reports how many kernel nodes the graph holds (the launches per
seam), and replays it.  All buffers the callable touches must be allocated
before capture; nothing here allocates device memory during capture.

Early launch.  A kernel launched with programmatic dependent launch is
recorded with a programmatic edge from the kernel before it, taken from that
kernel's trigger port: the dependent starts when every block of the upstream
kernel has triggered or exited.  A PyTorch kernel never triggers, so after one
the dependent starts only when it ends.  ``early_launch=True`` moves those
edges to the upstream's launch-completion port (every block of it has
started).  The dependent then sets itself up while the upstream runs; its
``griddepcontrol.wait`` still blocks until the upstream has completed and its
writes are visible, which is the only ordering a kernel launched this way may
rely on (a trigger carries no memory ordering).  The seam kernels read only
weights before that wait.  Edges of the default type are left as captured.
"""
from __future__ import annotations

import ctypes

import torch

_CUDART_NAMES = ("libcudart.so.13", "libcudart.so.12", "libcudart.so",
                 "/usr/local/cuda/lib64/libcudart.so")
_KERNEL_NODE = 0            # cudaGraphNodeTypeKernel
_CAPTURE_THREAD_LOCAL = 1   # cudaStreamCaptureModeThreadLocal
_PORT_PROGRAMMATIC = 1      # cudaGraphKernelNodePortProgrammatic
_PORT_LAUNCH_COMPLETION = 2  # cudaGraphKernelNodePortLaunchCompletion
_DEP_PROGRAMMATIC = 1       # cudaGraphDependencyTypeProgrammatic


class _EdgeData(ctypes.Structure):
    """cudaGraphEdgeData: upstream port, downstream port, dependency type."""
    _fields_ = [("from_port", ctypes.c_ubyte), ("to_port", ctypes.c_ubyte), ("type", ctypes.c_ubyte),
                ("reserved", ctypes.c_ubyte * 5)]

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
        # edge-data forms of the dependency calls: the plain names from CUDA
        # 13 on, the _v2 names in CUDA 12
        for name in ("cudaGraphGetEdges", "cudaGraphRemoveDependencies", "cudaGraphAddDependencies"):
            f = getattr(_rt, name + "_v2") if hasattr(_rt, name + "_v2") else getattr(_rt, name)
            f.argtypes = [P, P, P, P, ctypes.POINTER(ctypes.c_size_t) if name == "cudaGraphGetEdges"
                          else ctypes.c_size_t]
            setattr(_rt, "_mhc_" + name, f)
    return _rt


def _ck(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed: {cudart().cudaGetErrorString(rc).decode()} ({rc})")


def _edges(graph):
    """All edges of ``graph``: (from nodes, to nodes, edge data, count)."""
    rt = cudart()
    n = ctypes.c_size_t(0)
    _ck(rt._mhc_cudaGraphGetEdges(graph, None, None, None, ctypes.byref(n)), "cudaGraphGetEdges")
    fr = (ctypes.c_void_p * max(1, n.value))()
    to = (ctypes.c_void_p * max(1, n.value))()
    ed = (_EdgeData * max(1, n.value))()
    _ck(rt._mhc_cudaGraphGetEdges(graph, fr, to, ed, ctypes.byref(n)), "cudaGraphGetEdges")
    return fr, to, ed, n.value


def launch_early(graph) -> int:
    """Move every programmatic edge of ``graph`` that leaves its upstream
    kernel's trigger port to that kernel's launch-completion port (the
    downstream kernel may start once every upstream block has started; its
    griddepcontrol.wait still waits for the upstream's completion).  Returns
    the number of edges moved."""
    rt = cudart()
    fr, to, ed, n = _edges(graph)
    moved = 0
    for i in range(n):
        if ed[i].type != _DEP_PROGRAMMATIC or ed[i].from_port != _PORT_PROGRAMMATIC:
            continue
        f, t = ctypes.c_void_p(fr[i]), ctypes.c_void_p(to[i])
        old = _EdgeData(from_port=_PORT_PROGRAMMATIC, type=_DEP_PROGRAMMATIC)
        new = _EdgeData(from_port=_PORT_LAUNCH_COMPLETION, type=_DEP_PROGRAMMATIC)
        _ck(rt._mhc_cudaGraphRemoveDependencies(graph, ctypes.byref(f), ctypes.byref(t), ctypes.byref(old), 1),
            "cudaGraphRemoveDependencies")
        _ck(rt._mhc_cudaGraphAddDependencies(graph, ctypes.byref(f), ctypes.byref(t), ctypes.byref(new), 1),
            "cudaGraphAddDependencies")
        moved += 1
    return moved


def edge_ports(graph) -> dict:
    """Histogram of the graph's edges by (upstream port, dependency type)."""
    fr, to, ed, n = _edges(graph)
    hist = {}
    for i in range(n):
        k = (ed[i].from_port, ed[i].type)
        hist[k] = hist.get(k, 0) + 1
    return hist


class SeamGraph:
    """Capture ``fn(stream)`` into a CUDA graph on ``stream`` and instantiate
    it; ``early_launch`` applies ``launch_early`` before instantiation
    (``moved_edges`` counts the edges it moved)."""

    def __init__(self, fn, stream: torch.cuda.Stream, early_launch: bool = False):
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
        self.moved_edges = launch_early(g) if early_launch else 0
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
