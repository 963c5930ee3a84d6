"""Host-only checks of the C ABI (no GPU needed): the library loads, exports
every function include/mhc.h declares, and rejects bad arguments on the host
before any CUDA call (fake pointer values are never dereferenced because
every call here is rejected by the host checks)."""
import ctypes
import os
import re

import pytest

import mhc_hyper_connection_pre_gb300 as mhc
from mhc_hyper_connection_pre_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, CUDA_ERR = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mhc.load_library()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mhc_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_function(lib):
    names = _declared_functions()
    assert {"mhc_pre_delayed", "mhc_post", "mhc_status_string"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"libmhc.so does not export {name}"


def test_status_strings(lib):
    for code in range(5):
        s = lib.mhc_status_string(code).decode()
        assert s.startswith("MHC_")
    assert lib.mhc_status_string(99).decode() == "unknown mhc_status"
    assert lib.mhc_version() >= 1


A = 0x10000  # a 16-byte aligned fake address; never dereferenced here


def _pre(lib, **kw):
    args = dict(x=A, pre_in=A + 0x100000, fn=A + 0x200000, bias=A + 0x3000000, alpha=A + 0x3001000,
                norm_weight=None, T=16, n=4, C=5120, iters=20, rms_eps=1e-6, norm_eps=1e-6,
                sk_eps=1e-6, pre_out=A + 0x4000000, post_out=A + 0x4100000, comb_out=A + 0x4200000,
                layer_input=A + 0x4300000, logits_out=None, workspace=None, workspace_bytes=0,
                stream=None)
    args.update(kw)
    return lib.mhc_pre_delayed(*args.values())


def test_pre_rejects_bad_shapes(lib):
    assert _pre(lib, n=3) == UNSUPPORTED
    assert _pre(lib, C=5121) == UNSUPPORTED
    assert _pre(lib, C=5124) == UNSUPPORTED
    assert _pre(lib, C=6152) == UNSUPPORTED
    assert _pre(lib, T=-1) == INVALID
    assert _pre(lib, iters=0) == INVALID
    assert _pre(lib, n=0) == INVALID
    assert _pre(lib, rms_eps=-1.0) == INVALID
    assert _pre(lib, norm_eps=float("nan")) == INVALID


def test_pre_zero_tokens_is_a_no_op(lib):
    # T == 0 returns before any pointer is looked at or any launch
    assert _pre(lib, T=0, x=None, pre_in=None, fn=None) == OK


def test_pre_rejects_null_misaligned_and_overlapping(lib):
    assert _pre(lib, x=None) == INVALID
    assert _pre(lib, fn=None) == INVALID
    assert _pre(lib, layer_input=None) == INVALID
    assert _pre(lib, x=A + 8) == INVALID
    assert _pre(lib, comb_out=A + 0x4200004) == INVALID
    assert _pre(lib, norm_weight=A + 0x5000002) == INVALID
    # pre_out aliasing pre_in (the carried pre-mix must be ping-ponged)
    assert _pre(lib, pre_out=A + 0x100000) == INVALID
    # layer_input inside x
    assert _pre(lib, layer_input=A + 0x1000) == INVALID
    # two outputs overlapping
    assert _pre(lib, post_out=A + 0x4000010) == INVALID
    # workspace overlapping an input or an output
    assert _pre(lib, workspace=A + 0x10, workspace_bytes=1 << 20) == INVALID
    assert _pre(lib, workspace=A + 0x4300000, workspace_bytes=64) == INVALID


def test_workspace_bytes_host_only(lib):
    # no GPU in this process: every shape reports 0 (the tensor-core plan, and
    # with it the workspace, is sized on the device); bad shapes report 0
    assert lib.mhc_pre_workspace_bytes(16, 4, 5120) == 0
    assert lib.mhc_pre_workspace_bytes(16, 3, 5120) == 0


def _post(lib, **kw):
    args = dict(x=A, y=A + 0x1000000, comb=A + 0x2000000, post=A + 0x2100000, T=16, n=4, C=5120,
                x_new=A + 0x3000000, stream=None)
    args.update(kw)
    return lib.mhc_post(*args.values())


def test_post_rejects_bad_arguments(lib):
    assert _post(lib, n=2) == UNSUPPORTED
    assert _post(lib, C=100) == UNSUPPORTED
    assert _post(lib, T=-5) == INVALID
    assert _post(lib, T=0, x=None) == OK
    assert _post(lib, y=None) == INVALID
    assert _post(lib, comb=A + 0x2000004) == INVALID
    assert _post(lib, x_new=A + 0x10) == INVALID           # overlaps x, not equal
    assert _post(lib, x_new=A + 0x1000000) == INVALID      # overlaps y


def test_plan_shape_checks(lib):
    kernel, grid, cluster, tt = (ctypes.c_int(-1) for _ in range(4))
    st = lib.mhc_pre_delayed_plan(16, 4, 5120, ctypes.byref(kernel), ctypes.byref(grid),
                                  ctypes.byref(cluster), ctypes.byref(tt))
    assert st == OK
    assert kernel.value == 1 and cluster.value == 16 and tt.value == 16
    st = lib.mhc_pre_delayed_plan(100, 4, 5120, None, None, None, ctypes.byref(tt))
    assert st == OK and tt.value == 32
    assert lib.mhc_pre_delayed_plan(16, 4, 5121, None, None, None, None) == UNSUPPORTED


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mhc.post(x, torch.zeros(2, 64, dtype=torch.bfloat16), torch.zeros(2, 4, 4),
                 torch.zeros(2, 4))


def _fused(lib, **kw):
    args = dict(x=A, y=A + 0x1000000, comb=A + 0x2000000, post=A + 0x2100000, x_new=A + 0x6000000,
                pre_in=A + 0x100000, fn=A + 0x200000, bias=A + 0x3000000, alpha=A + 0x3001000,
                norm_weight=None, T=16, n=4, C=5120, iters=20, rms_eps=1e-6, norm_eps=1e-6, sk_eps=1e-6,
                pre_out=A + 0x4000000, post_out=A + 0x4100000, comb_out=A + 0x4200000,
                layer_input=A + 0x4300000, logits_out=None, workspace=None, workspace_bytes=0, stream=None)
    args.update(kw)
    return lib.mhc_post_pre_delayed(*args.values())


def test_fused_rejects_on_the_host(lib):
    # x (0x10000) spans 655,360 bytes at T = 16; y sits at +0x1000000 and so on
    assert _fused(lib, y=None) == INVALID
    assert _fused(lib, comb=A + 0x2000008) == INVALID            # misaligned
    assert _fused(lib, x_new=A + 0x100) == INVALID                # partial overlap with x
    assert _fused(lib, x_new=A + 0x1000000) == INVALID            # overlaps y
    assert _fused(lib, comb_out=A + 0x2000040) == INVALID         # partial overlap with comb
    assert _fused(lib, pre_out=A + 0x100000) == INVALID           # pre_out aliases pre_in
    assert _fused(lib, n=3) == UNSUPPORTED
    assert _fused(lib, T=0, x=None, y=None) == OK


def test_fused_exact_aliases_pass_the_host_checks(lib):
    # x_new == x, comb_out == comb, post_out == post are allowed: with no GPU
    # in this process the call gets past every argument check and then fails
    # to find a device (MHC_ERR_CUDA), instead of MHC_ERR_INVALID_ARGUMENT
    assert _fused(lib, x_new=A) == CUDA_ERR
    assert _fused(lib, comb_out=A + 0x2000000, post_out=A + 0x2100000) == CUDA_ERR


def test_broadcast_entry_points_size_x_as_t_by_c(lib):
    """The broadcast calls take x as [T, C]: an output just past T*C*2 bytes
    of x passes the host checks (and then finds no device), where the
    four-stream call sees it inside x; x_new may never alias a broadcast x."""
    just_past = A + 16 * 5120 * 2            # T * C * 2 bytes after x
    assert _pre(lib, layer_input=just_past) == INVALID
    args = dict(x=A, pre_in=A + 0x100000, fn=A + 0x200000, bias=A + 0x3000000, alpha=A + 0x3001000,
                norm_weight=None, T=16, n=4, C=5120, iters=20, rms_eps=1e-6, norm_eps=1e-6,
                sk_eps=1e-6, pre_out=A + 0x4000000, post_out=A + 0x4100000, comb_out=A + 0x4200000,
                layer_input=just_past, logits_out=None, workspace=None, workspace_bytes=0, stream=None)
    assert lib.mhc_pre_delayed_broadcast(*args.values()) == CUDA_ERR
    args["layer_input"] = A + 0x100
    assert lib.mhc_pre_delayed_broadcast(*args.values()) == INVALID
    args["layer_input"] = just_past
    del args["pre_in"]
    assert lib.mhc_pre_broadcast(*args.values()) == CUDA_ERR
    args["n"] = 3
    assert lib.mhc_pre_broadcast(*args.values()) == UNSUPPORTED
    post = dict(x=A, y=A + 0x1000000, comb=A + 0x2000000, post=A + 0x2100000, T=16, n=4, C=5120,
                x_new=A, stream=None)
    assert _post(lib, x_new=A) == CUDA_ERR                          # in place is allowed for mhc_post
    assert lib.mhc_post_broadcast(*post.values()) == INVALID        # never for the broadcast x
    post["x_new"] = just_past
    assert _post(lib, x_new=just_past) == INVALID
    assert lib.mhc_post_broadcast(*post.values()) == CUDA_ERR


def _seam_host(lib, **kw):
    args = dict(x=A, y=A + 0x1000000, pre_in=A + 0x2000000, fn=A + 0x3000000, bias=A + 0x4000000,
                alpha=A + 0x4001000, norm_weight=None, T=16, n=4, C=5120, iters=20, rms_eps=1e-6, norm_eps=1e-6,
                sk_eps=1e-6, x_new=A + 0x5000000, pre_out=A + 0x6000000, post_out=None, comb_out=None,
                layer_input=None, workspace=A + 0x7000000, workspace_bytes=1 << 30,
                stream=None)
    args.update(kw)
    return lib.mhc_seam_host(*args.values())


def test_seam_host_rejects_on_the_host(lib):
    """mhc_seam_host checks shapes, pointers, host overlaps, the workspace
    and page-locked host memory before touching a device (here there is
    none: memory that is not page-locked is what every fake address is)."""
    assert _seam_host(lib, T=0, x=None) == OK
    assert _seam_host(lib, n=3) == UNSUPPORTED
    assert _seam_host(lib, C=100) == UNSUPPORTED
    assert _seam_host(lib, T=-1) == INVALID
    assert _seam_host(lib, x=None) == INVALID
    assert _seam_host(lib, pre_out=None) == INVALID
    assert _seam_host(lib, workspace=None) == INVALID
    assert _seam_host(lib, x_new=A + 0x100) == INVALID            # partial overlap with x
    assert _seam_host(lib, pre_out=A + 0x1000000) == INVALID      # inside y
    assert _seam_host(lib, workspace=A + 0x7000010) == INVALID    # not 256-byte aligned
    assert _seam_host(lib, workspace_bytes=16) == INVALID         # too small
    assert _seam_host(lib) == INVALID                             # not page-locked
    assert lib.mhc_seam_host_workspace_bytes(0, 4, 5120) == 0
    assert lib.mhc_seam_host_workspace_bytes(16, 3, 5120) == 0
    assert lib.mhc_seam_host_workspace_bytes(16, 4, 5120) > 16 * 4 * 5120 * 2


def test_packed_weights_host_checks(lib):
    """Sizes and host-side rejections of the packed-weight calls (no device
    here: a well-formed call finds none)."""
    assert lib.mhc_pre_packed_bytes(4, 5120) == 16 * 20 * 9216
    assert lib.mhc_pre_packed_bytes(4, 136) == 0          # not a tensor-core hidden size
    assert lib.mhc_pre_packed_bytes(3, 5120) == 0
    P = A + 0x8000000
    assert lib.mhc_pre_pack(A + 0x200000, 4, 5120, P, 16 * 20 * 9216, None) == CUDA_ERR
    assert lib.mhc_pre_pack(A + 0x200000, 4, 136, P, 1 << 20, None) == UNSUPPORTED
    assert lib.mhc_pre_pack(A + 0x200000, 4, 5120, P + 16, 1 << 22, None) == INVALID   # not 256-aligned
    assert lib.mhc_pre_pack(A + 0x200000, 4, 5120, P, 1024, None) == INVALID           # too small
    assert lib.mhc_pre_pack(A + 0x200000, 4, 5120, A + 0x200000, 1 << 22, None) == INVALID   # overlaps fn
    args = dict(x=A, pre_in=A + 0x100000, fn=A + 0x200000, packed=P, packed_bytes=16 * 20 * 9216,
                bias=A + 0x3000000, alpha=A + 0x3001000, norm_weight=None, T=16, n=4, C=5120, iters=20,
                rms_eps=1e-6, norm_eps=1e-6, sk_eps=1e-6, pre_out=A + 0x4000000, post_out=A + 0x4100000,
                comb_out=A + 0x4200000, layer_input=A + 0x4300000, logits_out=None, stream=None)
    assert lib.mhc_pre_delayed_packed(*args.values()) == CUDA_ERR
    assert lib.mhc_pre_delayed_packed(*dict(args, packed=None).values()) == INVALID
    assert lib.mhc_pre_delayed_packed(*dict(args, packed_bytes=1024).values()) == INVALID
    assert lib.mhc_pre_delayed_packed(*dict(args, pre_out=P + 64).values()) == INVALID    # output inside packed
