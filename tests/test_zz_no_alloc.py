"""The allocation-free entry point, mhc_pre_delayed_noalloc.

It serves callers that cannot allocate device memory (and so cannot hand
mhc_pre_delayed a workspace): the library keeps the tensor-core kernel's
scratch in a fixed device array instead.  The GPU test calls it through the
C ABI twice in a row, on different inputs and weights (so the second call
cannot lean on what the first left in the shared array), and checks each
result against mhc_pre_delayed on the same inputs, within the parity
tolerances of the other GPU tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import mhc_hyper_connection_pre_gb300 as mhc
from mhc_hyper_connection_pre_gb300 import build as mbuild
from parity import assert_gates, assert_bf16
from workloads import seam_inputs

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mhc.load_library()


def test_noalloc_rejects_on_the_host(lib):
    A = 0x10000  # fake, 16-byte aligned; every call below is rejected before any CUDA call
    args = dict(x=A, pre_in=A + 0x100000, fn=A + 0x200000, bias=A + 0x3000000, alpha=A + 0x3001000,
                norm_weight=None, T=300, n=4, C=5120, iters=20, rms_eps=1e-6, norm_eps=1e-6,
                sk_eps=1e-6, pre_out=A + 0x4000000, post_out=A + 0x4100000, comb_out=A + 0x4200000,
                layer_input=A + 0x4300000, logits_out=None, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return lib.mhc_pre_delayed_noalloc(*a.values())

    assert call(C=6144) == UNSUPPORTED      # beyond the tensor-core kernel's hidden-size limit (5120)
    assert call(C=1000) == UNSUPPORTED      # not a multiple of 256
    assert call(n=3) == UNSUPPORTED
    assert call(x=None) == INVALID
    assert call(pre_out=A + 0x100000) == INVALID
    assert call(T=0, x=None) == OK


def _noalloc(lib, d, o, stream=None):
    T, n, C = d["x"].shape
    nw = d["norm_w"].data_ptr() if d["norm_w"] is not None else None
    return lib.mhc_pre_delayed_noalloc(
        d["x"].data_ptr(), d["pre_in"].data_ptr(), d["fn"].data_ptr(), d["bias"].data_ptr(),
        d["alpha"].data_ptr(), nw, T, n, C, 20, 1e-6, 1e-6, 1e-6, o["pre"].data_ptr(),
        o["post"].data_ptr(), o["comb"].data_ptr(), o["layer_input"].data_ptr(),
        o["logits"].data_ptr() if "logits" in o else None,
        stream if stream is not None else torch.cuda.current_stream(d["x"].device).cuda_stream)


def _run_both(lib, d):
    T, n, C = d["x"].shape
    dev = d["x"].device

    def outs():
        return {"pre": torch.empty(T, n, device=dev), "post": torch.empty(T, n, device=dev),
                "comb": torch.empty(T, n, n, device=dev),
                "layer_input": torch.empty(T, C, dtype=torch.bfloat16, device=dev)}

    ref = mhc.pre_delayed(d["x"], d["pre_in"], d["fn"], d["bias"], d["alpha"], d["norm_w"], out=outs())
    o = outs()
    st = _noalloc(lib, d, o)
    assert st == OK, lib.mhc_status_string(st).decode()
    torch.cuda.synchronize(dev)
    assert mhc.device_status() == 0
    return ref, o


@pytest.mark.gpu
def test_noalloc_matches_mhc_pre_delayed_twice_in_a_row(lib):
    cases = [seam_inputs(300, seed=901, fold=True), seam_inputs(1000, seed=902, fold=True)]
    for d in cases:
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        ref, got = _run_both(lib, d)
        for k in ("pre", "post", "comb"):
            assert_gates(got[k].cpu().numpy(), ref[k].cpu().numpy().astype(np.float64), k)
        gl = got["layer_input"].cpu().view(torch.int16).numpy().view(np.uint16)
        rl = ref["layer_input"].cpu().view(torch.int16).numpy().view(np.uint16)
        assert_bf16(gl, rl, "layer_input")


@pytest.mark.gpu
@pytest.mark.parametrize("T,C,fold", [(1, 5120, True), (7, 5120, False), (128, 5120, True), (300, 256, True),
                                      (33, 768, False)])
def test_noalloc_against_the_oracle(lib, T, C, fold):
    """Decode-sized calls (one cluster, one tile: below 256 tokens only this
    entry point runs the tensor-core kernel) and small hidden sizes, against
    the CPU oracle at the parity tolerances."""
    import oracle
    from workloads import bf16_bits
    from parity import assert_bitexact
    oracle.build()
    d = seam_inputs(T, C=C, seed=910 + T + C, fold=fold)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    o = {"pre": torch.empty(T, 4, device="cuda"), "post": torch.empty(T, 4, device="cuda"),
         "comb": torch.empty(T, 4, 4, device="cuda"),
         "layer_input": torch.empty(T, C, dtype=torch.bfloat16, device="cuda")}
    st = _noalloc(lib, g, o)
    assert st == OK, lib.mhc_status_string(st).decode()
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    nw = None if d["norm_w"] is None else bf16_bits(d["norm_w"])
    ref = oracle.pre_delayed(bf16_bits(d["x"]), d["pre_in"].numpy(), d["fn"].numpy(), d["bias"].numpy(),
                             d["alpha"].numpy(), nw)
    for k in ("pre", "post", "comb"):
        assert_gates(o[k].cpu().numpy(), ref[k], k)
    li = o["layer_input"].cpu().view(torch.int16).numpy().view(np.uint16)
    if fold:
        assert_bf16(li, ref["layer_input"], "layer_input (fold)")
    else:
        assert_bitexact(li, ref["layer_input"], "layer_input (collapse)")


@pytest.mark.gpu
def test_noalloc_allocates_nothing_and_checks_the_device(lib):
    """After a first call on the device (its one-time set-up), further calls
    leave the device's free memory unchanged; x in host memory is rejected
    before anything is launched."""
    d = seam_inputs(300, seed=920, fold=True)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    o = {"pre": torch.empty(300, 4, device="cuda"), "post": torch.empty(300, 4, device="cuda"),
         "comb": torch.empty(300, 4, 4, device="cuda"),
         "layer_input": torch.empty(300, 5120, dtype=torch.bfloat16, device="cuda")}
    assert _noalloc(lib, g, o) == OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(lib, g, o) == OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert mhc.device_status() == 0
    hx = d["x"].pin_memory()
    bad = dict(g, x=hx)
    assert _noalloc(lib, bad, o, stream=torch.cuda.current_stream().cuda_stream) == INVALID
