"""GPU parity: the CUDA seam (through the C ABI) against the CPU oracle on
the same seeded inputs, element by element, plus launch-count, graph-replay
and determinism checks.  Needs a GB300 and a built libmhc.so."""
import os

import numpy as np
import pytest
import torch

import oracle
import mhc_hyper_connection_pre_gb300 as mhc
from mhc_hyper_connection_pre_gb300.graphs import SeamGraph, edge_ports
from workloads import seam_inputs, bf16_bits, chain_seam_params, chain_stub_delta
from parity import (assert_gates, assert_bf16, assert_bitexact, assert_logits, logit_bound,
                    post_abs_scale)

pytestmark = pytest.mark.gpu

NTHREADS = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mhc.load_library()
    oracle.build()


def _to_dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _gpu_pre(g, **kw):
    out = mhc.pre_delayed(g["x"], g["pre_in"], g["fn"], g["bias"], g["alpha"], g["norm_w"],
                          return_logits=True, **kw)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0, "a bounded in-kernel wait timed out"
    return {k: v.cpu() for k, v in out.items()}


def _oracle_pre(d, rows=None):
    x = bf16_bits(d["x"])
    pre_in = d["pre_in"].cpu().numpy()
    if rows is not None:
        x, pre_in = x[rows], pre_in[rows]
    nw = None if d["norm_w"] is None else bf16_bits(d["norm_w"])
    return oracle.pre_delayed(x, pre_in, d["fn"].cpu().numpy(), d["bias"].cpu().numpy(),
                              d["alpha"].cpu().numpy(), nw, nthreads=NTHREADS), x


def _check_pre(g, o, x_bits, d, fold, rows=None):
    sl = slice(None) if rows is None else rows
    li = g["layer_input"].view(torch.int16).numpy().view(np.uint16)[sl]
    if fold:
        assert_bf16(li, o["layer_input"], "layer_input (fold)")
    else:
        assert_bitexact(li, o["layer_input"], "layer_input (collapse)")
    assert_gates(g["pre"].numpy()[sl], o["pre"], "pre")
    assert_gates(g["post"].numpy()[sl], o["post"], "post")
    assert_gates(g["comb"].numpy()[sl], o["comb"], "comb")
    bound = logit_bound(x_bits, d["fn"].cpu().numpy(), d["alpha"].cpu().numpy(), o["logits"])
    assert_logits(g["logits"].numpy()[sl], o["logits"], bound)


def test_config0_pr1_reference():
    """T=16, seed 0, no fold: collapse bit-exact, gates within 2e-5."""
    d = seam_inputs(16, seed=0)
    g = _gpu_pre(_to_dev(d))
    o, xb = _oracle_pre(d)
    _check_pre(g, o, xb, d, fold=False)


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16, 32, 64, 128])
def test_config1_decode_sweep(T):
    """Decode sweep with the fused RMSNorm fold, seed = T."""
    d = seam_inputs(T, seed=T, fold=True)
    g = _gpu_pre(_to_dev(d))
    o, xb = _oracle_pre(d)
    _check_pre(g, o, xb, d, fold=True)


@pytest.mark.parametrize("T,C,fold", [
    (1, 8, False), (3, 8, True), (7, 136, True), (31, 1000, False), (9, 2056, True),
    (127, 5120, False), (129, 5120, True), (17, 6144, True), (64, 6144, False),
    (1000, 5120, True), (33, 4096, False), (5, 128, True), (2, 2048, True),
    (300, 1000, True), (500, 6144, False), (225, 136, False),
    # tile sizes at the projection's form boundaries: 4 tokens (the largest
    # fp32-FMA tile), 16 (the largest single m-tile), 17 and 32 (two m-tiles
    # sharing each fn fragment)
    (26, 5120, True), (112, 5120, False), (113, 5120, True), (224, 5120, True),
])
def test_token_and_hidden_sweep(T, C, fold):
    """Ragged token tails (tile sizes that do not divide T), hidden sizes
    whose 8-column groups do not split evenly over the 16 CTA slices, slices
    with no columns at all (C = 8), and cluster-kernel shapes with more tiles
    than co-resident clusters (several rounds per cluster: T = 225..500 at
    hidden sizes the tensor-core kernel does not take)."""
    d = seam_inputs(T, C=C, seed=100 + T + C, fold=fold)
    g = _gpu_pre(_to_dev(d))
    o, xb = _oracle_pre(d)
    _check_pre(g, o, xb, d, fold=fold)


@pytest.mark.parametrize("T,C,fold", [
    (256, 5120, True), (257, 5120, False), (300, 256, True), (512, 4096, True),
    (640, 2048, False), (1383, 5120, True), (4096, 5120, False), (700, 768, True),
])
def test_tensor_core_path(T, C, fold):
    """Shapes that take the tensor-core kernel (128-token tiles, fn split in
    three bf16 planes): ragged last tiles, one 16-column stage per CTA
    (C = 256), an odd number of stages per tile (C = 768), other slice
    widths, more tiles than co-resident clusters."""
    assert mhc.pre_plan(T, 4, C)["kernel"] == 2
    d = seam_inputs(T, C=C, seed=700 + T, fold=fold)
    g = _gpu_pre(_to_dev(d))
    assert mhc.device_status() == 0
    o, xb = _oracle_pre(d)
    _check_pre(g, o, xb, d, fold=fold)


def test_kernel_choice():
    assert mhc.pre_plan(1)["kernel"] == 1
    assert mhc.pre_plan(255)["kernel"] == 1
    assert mhc.pre_plan(256)["kernel"] == 2
    assert mhc.pre_plan(16384)["kernel"] == 2
    assert mhc.pre_plan(4096, 4, 6144)["kernel"] == 1      # slice too wide for the TMEM park
    assert mhc.pre_plan(4096, 4, 1000)["kernel"] == 1      # C not a multiple of 256
    assert mhc.pre_plan(4096, 4, 640)["kernel"] == 1
    p = mhc.pre_plan(16384)
    assert p["cluster"] == 16 and p["tokens_per_tile"] == 128 and p["grid"] % 16 == 0


def test_tensor_core_workspace_is_one_plane_copy():
    """From 256 tokens mhc_pre_delayed first packs fn's planes into the
    workspace (one copy that every cluster reads): the workspace it asks for
    is that copy plus mhc_pre's T x 16-byte scratch; a workspace of just the
    copy gives the same bits as the default one, and one 256-byte step less
    is rejected before anything launches."""
    lib = mhc.load_library()
    T, C = 300, 5120
    packed = int(lib.mhc_pre_packed_bytes(4, C))
    assert int(lib.mhc_pre_workspace_bytes(T, 4, C)) == packed + (T * 16 + 255) // 256 * 256
    gd = _to_dev(seam_inputs(T, seed=1700, fold=True))
    ref = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    ws = torch.empty(packed, dtype=torch.uint8, device="cuda")
    got = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], workspace=ws)
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    with pytest.raises(mhc.MhcError):
        mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                        workspace=ws[: packed - 256])
    assert mhc.device_status() == 0


def test_alpha_and_sinkhorn_parameters():
    """Non-unit alphas, another iteration count and eps reach the kernel."""
    d = seam_inputs(24, seed=5, fold=True)
    d["alpha"] = torch.tensor([0.5, 1.7, 2.5])
    gd = _to_dev(d)
    out = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                          sinkhorn_iters=3, sinkhorn_eps=1e-3, rms_eps=1e-5, norm_eps=1e-4,
                          return_logits=True)
    torch.cuda.synchronize()
    g = {k: v.cpu() for k, v in out.items()}
    o = oracle.pre_delayed(bf16_bits(d["x"]), d["pre_in"].numpy(), d["fn"].numpy(), d["bias"].numpy(),
                           d["alpha"].numpy(), bf16_bits(d["norm_w"]), iters=3, sinkhorn_eps=1e-3,
                           rms_eps=float(np.float32(1e-5)), norm_eps=float(np.float32(1e-4)),
                           nthreads=NTHREADS)
    li = g["layer_input"].view(torch.int16).numpy().view(np.uint16)
    assert_bf16(li, o["layer_input"], "layer_input")
    for k in ("pre", "post", "comb"):
        assert_gates(g[k].numpy(), o[k], k)


def test_staggering_invariance():
    """Changing the incoming pre-mix leaves logits, gates and comb
    bit-identical (the #56503 page: the staggering does not change the
    gates); feeding pre_in := this seam's pre gives the non-delayed collapse."""
    d = seam_inputs(40, seed=6, fold=False)
    gd = _to_dev(d)
    a = _gpu_pre(gd)
    gd2 = dict(gd)
    gd2["pre_in"] = torch.rand(40, 4, device="cuda")
    b = _gpu_pre(gd2)
    for k in ("pre", "post", "comb", "logits"):
        assert torch.equal(a[k], b[k]), k
    gd3 = dict(gd)
    gd3["pre_in"] = a["pre"].cuda()
    c = _gpu_pre(gd3)
    o = oracle.pre_delayed(bf16_bits(d["x"]), a["pre"].numpy(), d["fn"].numpy(), d["bias"].numpy(),
                           d["alpha"].numpy(), None, nthreads=NTHREADS)
    assert_bitexact(c["layer_input"].view(torch.int16).numpy().view(np.uint16), o["layer_input"],
                    "non-delayed collapse")


@pytest.mark.parametrize("T", [100, 3000])
def test_deterministic(T):
    d = _to_dev(seam_inputs(T, seed=8, fold=True))
    a, b = _gpu_pre(d), _gpu_pre(d)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert mhc.device_status() == 0


def test_zero_tokens():
    x = torch.empty(0, 4, 5120, dtype=torch.bfloat16, device="cuda")
    out = mhc.pre_delayed(x, torch.empty(0, 4, device="cuda"), torch.zeros(24, 20480, device="cuda"),
                          torch.zeros(24, device="cuda"), torch.ones(3, device="cuda"))
    assert out["layer_input"].shape == (0, 5120)
    xn = mhc.post(x, torch.empty(0, 5120, dtype=torch.bfloat16, device="cuda"),
                  torch.empty(0, 4, 4, device="cuda"), torch.empty(0, 4, device="cuda"))
    assert xn.shape == (0, 4, 5120)


def _post_case(T, C, seed):
    d = seam_inputs(T, C=C, seed=seed, fold=True, with_y=True)
    gd = _to_dev(d)
    pre = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    return d, gd, pre


@pytest.mark.parametrize("T,C", [(1, 5120), (5, 5120), (64, 5120), (1000, 5120), (3, 8), (17, 2056)])
def test_post_parity(T, C):
    d, gd, pre = _post_case(T, C, seed=200 + T)
    xn = mhc.post(gd["x"], gd["y"], pre["comb"], pre["post"])
    torch.cuda.synchronize()
    comb, pg = pre["comb"].cpu().numpy(), pre["post"].cpu().numpy()
    xb, yb = bf16_bits(d["x"]), bf16_bits(d["y"])
    o_bits, _ = oracle.post(xb, yb, comb, pg)
    g_bits = xn.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16(g_bits, o_bits, "x_new", abs_scale=post_abs_scale(xb, yb, comb, pg))


def test_post_in_place():
    d, gd, pre = _post_case(50, 5120, seed=301)
    ref = mhc.post(gd["x"], gd["y"], pre["comb"], pre["post"])
    x2 = gd["x"].clone()
    mhc.post(x2, gd["y"], pre["comb"], pre["post"], out=x2)
    torch.cuda.synchronize()
    assert torch.equal(ref, x2)


def _fused_case(T, C, fold, seed):
    """Previous seam's gates (from a pre call on other weights) plus this
    seam's inputs; x is the residual entering the previous seam's post."""
    d = seam_inputs(T, C=C, seed=seed, fold=fold, with_y=True)
    gd = _to_dev(d)
    prev = chain_seam_params(seed % 97, C=C, device="cuda")
    g = mhc.pre_delayed(gd["x"], gd["pre_in"], prev["fn"], prev["bias"], prev["alpha"], prev["norm_w"])
    torch.cuda.synchronize()
    return d, gd, g["comb"].clone(), g["post"].clone()


@pytest.mark.parametrize("T,C,fold", [(1, 5120, True), (5, 5120, False), (20, 5120, True), (32, 5120, True),
                                      (100, 5120, True), (120, 5120, False), (33, 1000, False), (300, 1000, True),
                                      (300, 5120, True), (7, 8, True),
                                      # from 256 tokens: a ragged last tile, other hidden sizes,
                                      # several tiles per cluster, a half last stage (C = 768)
                                      (1383, 5120, False), (4097, 4096, True), (300, 2048, False),
                                      (2000, 5120, True), (600, 768, True)])
def test_fused_seam_is_bit_identical_to_post_then_pre(T, C, fold):
    """mhc_post_pre_delayed gives exactly the bits of mhc_post followed by
    mhc_pre_delayed: one kernel below 256 tokens (and at C = 1000, multi-round
    tiles at T = 300), the post kernel then the tensor-core pre from 256
    tokens."""
    d, gd, comb, post = _fused_case(T, C, fold, seed=1100 + T + C)
    xn_ref = mhc.post(gd["x"], gd["y"], comb, post)
    ref = mhc.pre_delayed(xn_ref, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    got = mhc.post_pre_delayed(gd["x"], gd["y"], comb, post, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"],
                               gd["norm_w"], return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    assert torch.equal(got["x_new"], xn_ref)
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got[k], ref[k]), k


@pytest.mark.parametrize("T", [4, 300])
def test_fused_seam_in_place_and_shared_gate_buffers(T):
    """x_new == x and comb_out / post_out == the incoming comb / post."""
    d, gd, comb, post = _fused_case(T, 5120, True, seed=1300 + T)
    xn_ref = mhc.post(gd["x"], gd["y"], comb, post)
    ref = mhc.pre_delayed(xn_ref, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    x = gd["x"].clone()
    out = {"comb": comb, "post": post}
    got = mhc.post_pre_delayed(x, gd["y"], comb, post, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"],
                               gd["norm_w"], x_new=x, out=out)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    assert torch.equal(x, xn_ref)
    for k in ("pre", "post", "comb", "layer_input"):
        assert torch.equal(got[k], ref[k]), k


@pytest.mark.parametrize("T", [24, 300])
def test_fused_seam_against_the_oracle(T):
    """The fused call checked against the oracle directly: x_new against the
    oracle's post, the pre outputs against the oracle's pre on that x_new
    (T = 300: the post kernel, then the tensor-core pre)."""
    C = 5120
    d, gd, comb, post = _fused_case(T, C, True, seed=1500)
    got = mhc.post_pre_delayed(gd["x"], gd["y"], comb, post, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"],
                               gd["norm_w"], return_logits=True)
    torch.cuda.synchronize()
    xb, yb = bf16_bits(d["x"]), bf16_bits(d["y"])
    cb, pb = comb.cpu().numpy(), post.cpu().numpy()
    o_bits, _ = oracle.post(xb, yb, cb, pb)
    g_bits = got["x_new"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16(g_bits, o_bits, "x_new", abs_scale=post_abs_scale(xb, yb, cb, pb))
    d2 = dict(d, x=got["x_new"].cpu())
    o, xb2 = _oracle_pre(d2)
    _check_pre({k: v.cpu() for k, v in got.items() if k != "x_new"}, o, xb2, d2, fold=True)


@pytest.mark.parametrize("T,nodes", [(4, 1), (300, 3)])
def test_fused_seam_is_one_launch_in_a_graph(T, nodes):
    """One kernel node below 256 tokens (the cluster kernel); from 256
    tokens the post kernel, the fn-plane packing and the tensor-core pre."""
    d, gd, comb, post = _fused_case(T, 5120, True, seed=1600)
    out = {"pre": torch.empty(T, 4, device="cuda"), "post": torch.empty(T, 4, device="cuda"),
           "comb": torch.empty(T, 4, 4, device="cuda"),
           "layer_input": torch.empty(T, 5120, dtype=torch.bfloat16, device="cuda")}
    xn = torch.empty_like(gd["x"])
    s = torch.cuda.Stream()
    g = SeamGraph(lambda st: mhc.post_pre_delayed(gd["x"], gd["y"], comb, post, gd["pre_in"], gd["fn"],
                                                  gd["bias"], gd["alpha"], gd["norm_w"], x_new=xn, out=out,
                                                  stream=st), s)
    assert g.kernel_nodes == nodes, g.kernel_nodes
    g.replay(3)
    s.synchronize()
    assert mhc.device_status() == 0
    g.close()


@pytest.mark.parametrize("T,C,fold", [(1, 5120, True), (7, 5120, False), (26, 5120, True), (33, 5120, True),
                                      (128, 5120, False), (100, 1000, True), (300, 1000, False), (300, 5120, True),
                                      (1000, 5120, False),
                                      (5, 8, True), (2000, 768, True), (2000, 768, False), (4097, 4096, True),
                                      (600, 6144, True), (600, 6144, False), (256, 5120, True), (257, 2048, False)])
def test_nondelayed_pre_equals_delayed_with_its_own_pre(T, C, fold):
    """mhc_pre's gates are those of mhc_pre_delayed (they do not depend on the
    incoming pre-mix), and its layer input is bit for bit the delayed call's
    with pre_in set to the pre it returned: the cluster kernel below 256
    tokens, the two-pass path above (gates-only tensor-core pass, then the
    streaming collapse in the tensor-core kernel's order), multi-round tiles
    at C=1000; C=768 has an odd number of stages per slice and several
    rounds per cluster at T=2000, so stage groups alternate between rounds;
    C=6144 (the widest residual) streams with one CTA per SM under the fold
    and two without."""
    d = seam_inputs(T, C=C, seed=1700 + T + C, fold=fold)
    gd = _to_dev(d)
    got = mhc.pre(gd["x"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    ref = mhc.pre_delayed(gd["x"], got["pre"].clone(), gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                          return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got[k], ref[k]), k


@pytest.mark.parametrize("T,C,fold", [(1, 5120, True), (33, 5120, False), (300, 5120, True), (17, 2056, False)])
def test_nondelayed_pre_against_the_oracle(T, C, fold):
    """Gates within the gate tolerance of the oracle's; the collapse (no
    fold: bit-exact) and the fold (1 ulp) against the oracle's non-delayed
    block fed the kernel's own fp32 pre, so that a rounding of pre near a
    tie cannot move the comparison."""
    d = seam_inputs(T, C=C, seed=1800 + T + C, fold=fold)
    gd = _to_dev(d)
    got = mhc.pre(gd["x"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    g = {k: v.cpu() for k, v in got.items()}
    xb = bf16_bits(d["x"])
    nw = None if d["norm_w"] is None else bf16_bits(d["norm_w"])
    o = oracle.pre_nondelayed(xb, d["fn"].numpy(), d["bias"].numpy(), d["alpha"].numpy(), nw,
                              pre_mix=g["pre"].numpy(), nthreads=NTHREADS)
    _check_pre(g, o, xb, d, fold)
    # the pre-mix the kernel used is its own, not a stale or zero one
    o_own = oracle.pre_nondelayed(xb, d["fn"].numpy(), d["bias"].numpy(), d["alpha"].numpy(), nw,
                                  nthreads=NTHREADS)
    assert_gates(g["pre"].numpy(), o_own["pre"], "pre")


def test_nondelayed_pre_is_one_launch_in_a_graph_below_256_tokens():
    d = seam_inputs(16, C=5120, seed=1900, fold=True)
    gd = _to_dev(d)
    out = {"pre": torch.empty(16, 4, device="cuda"), "post": torch.empty(16, 4, device="cuda"),
           "comb": torch.empty(16, 4, 4, device="cuda"),
           "layer_input": torch.empty(16, 5120, dtype=torch.bfloat16, device="cuda")}
    ref = mhc.pre(gd["x"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    s = torch.cuda.Stream()
    g = SeamGraph(lambda st: mhc.pre(gd["x"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], out=out,
                                     stream=st), s)
    assert g.kernel_nodes == 1, g.kernel_nodes
    g.replay(5)
    s.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input"):
        assert torch.equal(out[k], ref[k]), k
    g.close()


def _bcast_case(T, C, fold, seed):
    d = seam_inputs(T, C=C, seed=seed, fold=fold, with_y=True)
    d["x"] = d["x"][:, 0, :].contiguous()          # the model-entry hidden state [T, C]
    return d, _to_dev(d)


@pytest.mark.parametrize("T,C,fold", [(1, 5120, True), (7, 5120, False), (33, 5120, True), (128, 5120, False),
                                      (300, 1000, True), (300, 5120, True), (1000, 5120, False), (5, 8, True),
                                      (700, 6144, True)])
def test_broadcast_pre_is_bit_identical_to_the_copied_residual(T, C, fold):
    """mhc_pre_delayed_broadcast / mhc_pre_broadcast on x [T, C] give every
    output bit for bit as the four-stream calls on x copied into four
    streams (decode kernel, multi-round tiles at C = 1000, tensor-core
    kernel from 256 tokens at C = 5120)."""
    d, gd = _bcast_case(T, C, fold, seed=2000 + T + C)
    xb = gd["x"][:, None, :].expand(T, 4, C).contiguous()
    got = mhc.pre_delayed_broadcast(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                                    return_logits=True)
    ref = mhc.pre_delayed(xb, gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    got_nd = mhc.pre_broadcast(gd["x"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    ref_nd = mhc.pre(xb, gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got[k], ref[k]), k
        assert torch.equal(got_nd[k], ref_nd[k]), "non-delayed " + k


@pytest.mark.parametrize("T,C", [(1, 5120), (64, 5120), (1000, 5120), (17, 2056)])
def test_broadcast_post_is_bit_identical_to_the_copied_residual(T, C):
    d, gd = _bcast_case(T, C, False, seed=2100 + T)
    comb = torch.rand(T, 4, 4, device="cuda")
    post = 2 * torch.rand(T, 4, device="cuda")
    xb = gd["x"][:, None, :].expand(T, 4, C).contiguous()
    got = mhc.post_broadcast(gd["x"], gd["y"], comb, post)
    ref = mhc.post(xb, gd["y"], comb, post)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("T,C,fold", [(24, 5120, True), (300, 5120, False)])
def test_broadcast_seam_against_the_oracle(T, C, fold):
    """The entry seam against the oracle's broadcast definitions: gates
    within 2e-5, collapse bit-exact or fold within 1 ulp, logits within the
    dot-product bound; the entry post's x_new within 1 ulp."""
    d, gd = _bcast_case(T, C, fold, seed=2200 + T)
    got = mhc.pre_delayed_broadcast(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                                    return_logits=True)
    xn = mhc.post_broadcast(gd["x"], gd["y"], got["comb"], got["post"])
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    g = {k: v.cpu() for k, v in got.items()}
    x1 = bf16_bits(d["x"])
    nw = None if d["norm_w"] is None else bf16_bits(d["norm_w"])
    o = oracle.pre_delayed_broadcast(x1, d["pre_in"].numpy(), d["fn"].numpy(), d["bias"].numpy(),
                                     d["alpha"].numpy(), nw, nthreads=NTHREADS)
    _check_pre(g, o, oracle.broadcast_streams(x1), d, fold)
    yb, cb, pb = bf16_bits(d["y"]), g["comb"].numpy(), g["post"].numpy()
    o_bits, _ = oracle.post_broadcast(x1, yb, cb, pb, nthreads=NTHREADS)
    g_bits = xn.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16(g_bits, o_bits, "x_new", abs_scale=post_abs_scale(oracle.broadcast_streams(x1), yb, cb, pb))


def test_graph_seam_is_two_launches_and_replays_exactly():
    """One seam (pre + post) captured in a CUDA graph holds exactly 2 kernel
    nodes; 200 replays give the eager result bit for bit."""
    d, gd, pre = _post_case(4, 5120, seed=400)
    eager_pre = {k: v.clone() for k, v in pre.items()}
    eager_xn = mhc.post(gd["x"], gd["y"], pre["comb"], pre["post"])
    out = {k: torch.empty_like(v) for k, v in pre.items()}
    xn = torch.empty_like(gd["x"])
    s = torch.cuda.Stream()

    def seam(stream):
        mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                        out=out, stream=stream)
        mhc.post(gd["x"], gd["y"], out["comb"], out["post"], out=xn, stream=stream)

    g = SeamGraph(seam, s)
    assert g.kernel_nodes == 2, g.kernel_nodes
    g.replay(200)
    s.synchronize()
    for k in eager_pre:
        assert torch.equal(out[k], eager_pre[k]), k
    assert torch.equal(xn, eager_xn)
    g.close()


def _chain_buffers(T, seams, C, dev):
    return {"x": torch.empty(T, 4, C, dtype=torch.bfloat16, device=dev),
            "pre": [torch.empty(T, 4, device=dev), torch.empty(T, 4, device=dev)],
            "outs": [{"post": torch.empty(T, 4, device=dev), "comb": torch.empty(T, 4, 4, device=dev),
                      "layer_input": torch.empty(T, C, dtype=torch.bfloat16, device=dev)}
                     for _ in range(seams)]}


def _seam_chain(b, params, ys, stream):
    """(pre, post) per seam back to back on one stream, launches only: each
    pre reads the x the previous post wrote and the pre-mix the previous pre
    wrote."""
    for si, o in enumerate(b["outs"]):
        p = params[si]
        out = dict(o, pre=b["pre"][(si + 1) & 1])
        mhc.pre_delayed(b["x"], b["pre"][si & 1], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=out,
                        stream=stream)
        mhc.post(b["x"], ys[si], o["comb"], o["post"], out=b["x"], stream=stream)


def _chain_result(b):
    return [b["x"].clone(), b["pre"][0].clone(), b["pre"][1].clone()] + \
        [v.clone() for o in b["outs"] for v in o.values()]


@pytest.mark.parametrize("T", [4, 100])
def test_launch_overlap_is_bit_identical(T):
    """With programmatic dependent launch on, a chain of seams whose kernels
    each consume the previous kernel's output (eager and graph-captured) gives
    the same bits as with it off."""
    seams, C, dev = 6, 5120, "cuda"
    params = [chain_seam_params(si, device=dev) for si in range(seams)]
    ys = [chain_stub_delta(si, T=T, device=dev) for si in range(seams)]
    d = seam_inputs(T, seed=900 + T, device=dev)
    b = _chain_buffers(T, seams, C, dev)
    s = torch.cuda.Stream()

    def reset():
        b["x"].copy_(d["x"])
        b["pre"][0].copy_(d["pre_in"])
        torch.cuda.synchronize()

    prev = mhc.set_launch_overlap(False)
    try:
        reset()
        _seam_chain(b, params, ys, s)
        s.synchronize()
        ref = _chain_result(b)
        mhc.set_launch_overlap(True)
        reset()
        _seam_chain(b, params, ys, s)
        s.synchronize()
        assert mhc.device_status() == 0
        for got, want in zip(_chain_result(b), ref):
            assert torch.equal(got, want)
        g = SeamGraph(lambda st: _seam_chain(b, params, ys, st), s)
        assert g.kernel_nodes == 2 * seams, g.kernel_nodes
        reset()
        g.replay(1)
        s.synchronize()
        assert mhc.device_status() == 0
        for got, want in zip(_chain_result(b), ref):
            assert torch.equal(got, want)
        g.close()
    finally:
        mhc.set_launch_overlap(prev)


def _fused_chain(b, params, ys, stream):
    """The same chain with each post(s - 1) fused into pre(s): pre(0), then
    (post(s - 1) + pre(s)) for s >= 1, then post of the last seam."""
    outs = b["outs"]
    for si, o in enumerate(outs):
        p = params[si]
        out = dict(o, pre=b["pre"][(si + 1) & 1])
        if si == 0:
            mhc.pre_delayed(b["x"], b["pre"][0], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=out,
                            stream=stream)
        else:
            q = outs[si - 1]
            mhc.post_pre_delayed(b["x"], ys[si - 1], q["comb"], q["post"], b["pre"][si & 1], p["fn"], p["bias"],
                                 p["alpha"], p["norm_w"], x_new=b["x"], out=out, stream=stream)
    mhc.post(b["x"], ys[len(outs) - 1], outs[-1]["comb"], outs[-1]["post"], out=b["x"], stream=stream)


@pytest.mark.parametrize("T", [4, 100])
def test_fused_chain_matches_and_overlaps_exactly(T):
    """A chain of fused seams equals the chain of separate calls bit for bit,
    with launch overlap off and on, eager and graph-captured."""
    seams, C, dev = 6, 5120, "cuda"
    params = [chain_seam_params(si, device=dev) for si in range(seams)]
    ys = [chain_stub_delta(si, T=T, device=dev) for si in range(seams)]
    d = seam_inputs(T, seed=950 + T, device=dev)
    b = _chain_buffers(T, seams, C, dev)
    s = torch.cuda.Stream()

    def reset():
        b["x"].copy_(d["x"])
        b["pre"][0].copy_(d["pre_in"])
        torch.cuda.synchronize()

    prev = mhc.set_launch_overlap(False)
    try:
        reset()
        _seam_chain(b, params, ys, s)
        s.synchronize()
        ref = _chain_result(b)
        for ov in (False, True):
            mhc.set_launch_overlap(ov)
            reset()
            _fused_chain(b, params, ys, s)
            s.synchronize()
            assert mhc.device_status() == 0
            for got, want in zip(_chain_result(b), ref):
                assert torch.equal(got, want)
        g = SeamGraph(lambda st: _fused_chain(b, params, ys, st), s)
        assert g.kernel_nodes == seams + 1, g.kernel_nodes
        reset()
        g.replay(1)
        s.synchronize()
        assert mhc.device_status() == 0
        for got, want in zip(_chain_result(b), ref):
            assert torch.equal(got, want)
        g.close()
    finally:
        mhc.set_launch_overlap(prev)


def _stub_chain(b, params, deltas, y, stream, fused):
    """The decode step as the benchmark runs it: each seam's sublayer is a
    PyTorch kernel (y = layer_input + D_s) between pre and post; with
    ``fused``, post(s - 1) runs inside pre(s) and the last post alone."""
    outs = b["outs"]
    for si, o in enumerate(outs):
        p = params[si]
        out = dict(o, pre=b["pre"][(si + 1) & 1])
        if fused and si > 0:
            q = outs[si - 1]
            mhc.post_pre_delayed(b["x"], y, q["comb"], q["post"], b["pre"][si & 1], p["fn"], p["bias"],
                                 p["alpha"], p["norm_w"], x_new=b["x"], out=out, stream=stream)
        else:
            mhc.pre_delayed(b["x"], b["pre"][si & 1], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=out,
                            stream=stream)
        with torch.cuda.stream(stream):
            torch.add(o["layer_input"], deltas[si], out=y)
        if not fused:
            mhc.post(b["x"], y, o["comb"], o["post"], out=b["x"], stream=stream)
    if fused:
        mhc.post(b["x"], y, outs[-1]["comb"], outs[-1]["post"], out=b["x"], stream=stream)


@pytest.mark.parametrize("T,fused", [(4, False), (4, True), (100, False), (100, True), (300, False), (300, True)])
def test_early_launch_after_a_torch_kernel_is_bit_identical(T, fused):
    """A graph whose programmatic edges leave the upstream kernel's
    launch-completion port (SeamGraph early_launch), with a PyTorch kernel
    between pre and post, gives the bits of the same chain run eagerly with
    launch overlap off.  Every programmatic edge is moved: below 256 tokens
    one into each seam kernel that follows another kernel; from 256 tokens
    (the pre is the plane pack and the tensor-core kernel, launched without
    programmatic serialization) one into each post, while the edges into the
    pack launches stay as captured."""
    seams, C, dev = 8, 5120, "cuda"
    params = [chain_seam_params(si, device=dev) for si in range(seams)]
    deltas = [chain_stub_delta(si, T=T, device=dev) for si in range(seams)]
    d = seam_inputs(T, seed=970 + T, device=dev)
    b = _chain_buffers(T, seams, C, dev)
    y = torch.empty(T, C, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()

    def reset():
        b["x"].copy_(d["x"])
        b["pre"][0].copy_(d["pre_in"])
        y.zero_()
        torch.cuda.synchronize()

    prev = mhc.set_launch_overlap(False)
    try:
        reset()
        _stub_chain(b, params, deltas, y, s, fused)
        s.synchronize()
        ref = _chain_result(b) + [y.clone()]
        mhc.set_launch_overlap(True)
        g = SeamGraph(lambda st: _stub_chain(b, params, deltas, y, st, fused), s, early_launch=True)
        if T >= 256:
            assert g.kernel_nodes == 4 * seams, g.kernel_nodes
            assert g.moved_edges == seams, g.moved_edges
        else:
            assert g.kernel_nodes == (2 * seams + 1 if fused else 3 * seams), g.kernel_nodes
            assert g.moved_edges == (seams if fused else 2 * seams - 1), g.moved_edges
        ports = edge_ports(g.graph)
        assert ports.get((1, 1), 0) == 0 and ports.get((2, 1), 0) == g.moved_edges, ports
        for _ in range(3):
            reset()
            g.replay(1)
            s.synchronize()
            assert mhc.device_status() == 0
            for got, want in zip(_chain_result(b) + [y], ref):
                assert torch.equal(got, want)
        g.close()
    finally:
        mhc.set_launch_overlap(prev)


def _stub_sublayer_oracle(li_bits: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """The chain's synthetic sublayer y = bf16(float(layer_input) + D_s): the
    two bf16 values added in fp32, the sum rounded once to bf16."""
    s32 = (oracle.bf16_to_f64(li_bits).astype(np.float32) + oracle.bf16_to_f64(d_bits).astype(np.float32))
    return oracle.bf16_round(s32.astype(np.float64))


def test_config3_decode_chain_against_the_oracle():
    """The full-model decode step: 80 seams at T = 4, each with its own
    weights, the pre-mix carried seam to seam (delayed), a synthetic
    sublayer between pre and post (the #56503 page: 80 seams per decode
    step).  Every seam's outputs are checked against the oracle fed that
    seam's GPU inputs (x and pre-mix): logits within the fp32 dot bound,
    gates within 2e-5, layer_input within 1 bf16 ulp, x_new within 1 ulp.
    The same chain captured in one CUDA graph (as the benchmark runs it) gives
    the eager chain's bits.  The drift of the final x against a chain run
    wholly in the oracle is reported."""
    seams, T, C = 80, 4, 5120
    params_cpu = [chain_seam_params(si) for si in range(seams)]
    deltas_cpu = [chain_stub_delta(si, T=T) for si in range(seams)]
    params = [_to_dev(p) for p in params_cpu]
    deltas = [dl.cuda() for dl in deltas_cpu]
    d0 = seam_inputs(T, seed=0)
    cx = d0["x"].cuda()
    cp = [d0["pre_in"].cuda(), torch.empty(T, 4, device="cuda")]
    co = {"post": torch.empty(T, 4, device="cuda"), "comb": torch.empty(T, 4, 4, device="cuda"),
          "layer_input": torch.empty(T, C, dtype=torch.bfloat16, device="cuda"),
          "logits": torch.empty(T, 24, device="cuda")}
    cy = torch.empty(T, C, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def seam(si, st):
        p = params[si]
        o = dict(co, pre=cp[(si + 1) & 1])
        mhc.pre_delayed(cx, cp[si & 1], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=o, stream=st)
        with torch.cuda.stream(st):
            torch.add(co["layer_input"], deltas[si], out=cy)
        mhc.post(cx, cy, co["comb"], co["post"], out=cx, stream=st)

    snaps = []
    for si in range(seams):
        x_in, p_in = bf16_bits(cx), cp[si & 1].cpu().numpy().copy()
        seam(si, s)
        s.synchronize()
        snaps.append({"x": x_in, "pre_in": p_in, "pre": cp[(si + 1) & 1].cpu().numpy().copy(),
                      "post": co["post"].cpu().numpy().copy(), "comb": co["comb"].cpu().numpy().copy(),
                      "logits": co["logits"].cpu().numpy().copy(), "layer_input": bf16_bits(co["layer_input"]),
                      "y": bf16_bits(cy), "x_new": bf16_bits(cx)})
    assert mhc.device_status() == 0
    eager_final = cx.clone()

    # the graph-captured chain from the same start
    cx.copy_(d0["x"].cuda())
    cp[0].copy_(d0["pre_in"].cuda())
    torch.cuda.synchronize()
    g = SeamGraph(lambda st: [seam(si, st) for si in range(seams)], s)
    g.replay(1)
    s.synchronize()
    assert mhc.device_status() == 0
    assert torch.equal(cx, eager_final), "graph-captured chain differs from the eager chain"
    g.close()

    for si, sn in enumerate(snaps):
        p = params_cpu[si]
        o = oracle.pre_delayed(sn["x"], sn["pre_in"], p["fn"].numpy(), p["bias"].numpy(), p["alpha"].numpy(),
                               bf16_bits(p["norm_w"]), nthreads=NTHREADS)
        what = f"seam {si}: "
        bound = logit_bound(sn["x"], p["fn"].numpy(), p["alpha"].numpy(), o["logits"])
        assert_logits(sn["logits"], o["logits"], bound, what + "logits")
        assert_gates(sn["pre"], o["pre"], what + "pre")
        assert_gates(sn["post"], o["post"], what + "post")
        assert_gates(sn["comb"], o["comb"], what + "comb")
        assert_bf16(sn["layer_input"], o["layer_input"], what + "layer_input")
        assert np.array_equal(sn["y"], _stub_sublayer_oracle(sn["layer_input"], bf16_bits(deltas_cpu[si])))
        xo, _ = oracle.post(sn["x"], sn["y"], sn["comb"], sn["post"])
        assert_bf16(sn["x_new"], xo, what + "x_new",
                    abs_scale=post_abs_scale(sn["x"], sn["y"], sn["comb"], sn["post"]))

    # the whole chain in the oracle, for the drift report
    x, pin = bf16_bits(d0["x"]), d0["pre_in"].numpy()
    for si in range(seams):
        p = params_cpu[si]
        o = oracle.pre_delayed(x, pin, p["fn"].numpy(), p["bias"].numpy(), p["alpha"].numpy(),
                               bf16_bits(p["norm_w"]), nthreads=NTHREADS)
        y = _stub_sublayer_oracle(o["layer_input"], bf16_bits(deltas_cpu[si]))
        x, _ = oracle.post(x, y, o["comb"], o["post"])
        pin = o["pre"]
    from parity import ulp_distance_bf16
    dist = ulp_distance_bf16(snaps[-1]["x_new"], x)
    hist = {int(k): int(v) for k, v in zip(*np.unique(np.minimum(dist, 8), return_counts=True))}
    print(f"\n80-seam chain, final x against the all-oracle chain: ulp histogram "
          f"(8 = 8 or more) {hist}; max {int(dist.max())}")
    assert np.median(dist) <= 1


# ------------------------------------------------- stress and full sizes ---

def _check_comb_properties(comb: np.ndarray, logits: np.ndarray):
    """The Sinkhorn invariants on every token: finite, non-negative, column
    sums 1 within 1e-6 (the last step normalises columns; sums in fp64 of the
    fp32 comb).  Row sums: twenty iterations do not bring every row within
    1e-3 even in exact arithmetic once the comb logits reach the tens (the
    C = 5120 workloads: about a third of the tokens at config 2, most of
    them under stress), so every token's comb is held to the oracle's
    Sinkhorn of the GPU's own logits -- within 2e-5 per entry, row sums
    within 1e-5 of the oracle's -- and the 1e-3 row bar to the tokens where
    the oracle itself meets it."""
    c = comb.astype(np.float64)
    assert np.all(np.isfinite(c))
    assert np.all(c >= 0)
    col = np.abs(c.sum(1) - 1.0)
    assert col.max() <= 1e-6, f"column sums off by up to {col.max():.3e}"
    og = oracle.gates_from_logits(np.asarray(logits, np.float64))["comb"]
    assert_gates(comb, og, "comb (every token, from gpu logits)")
    orow = og.sum(2)
    row_gap = np.abs(c.sum(2) - orow)
    assert row_gap.max() <= 1e-5, f"row sums differ from the oracle's by up to {row_gap.max():.3e}"
    conv = np.all(np.abs(orow - 1.0) <= 1e-3, axis=1)
    row = np.abs(c.sum(2) - 1.0)[conv]
    assert row.size == 0 or row.max() <= 1e-3 + 1e-5, f"row sums off by up to {row.max():.3e}"


def test_stress_small_layered():
    """Config-4 distribution at T=2048: comb logits of order +-300, 1% rows
    scaled by 1e3, 1% zero rows.  Layered check: logits within the fp32 dot
    bound; gates and comb recomputed by the oracle from the GPU's own logits
    within 2e-5; pre/post end to end; no NaN/Inf; Sinkhorn invariants."""
    T = 2048
    d = seam_inputs(T, seed=0, fold=True, stress=True)
    g = _gpu_pre(_to_dev(d))
    o, xb = _oracle_pre(d)
    bound = logit_bound(xb, d["fn"].numpy(), d["alpha"].numpy(), o["logits"])
    assert_logits(g["logits"].numpy(), o["logits"], bound)
    og = oracle.gates_from_logits(g["logits"].numpy().astype(np.float64))
    for k in ("pre", "post", "comb"):
        assert_gates(g[k].numpy(), og[k], k + " (from gpu logits)")
    assert_gates(g["pre"].numpy(), o["pre"], "pre")
    assert_gates(g["post"].numpy(), o["post"], "post")
    assert_bf16(g["layer_input"].view(torch.int16).numpy().view(np.uint16), o["layer_input"],
                "layer_input")
    _check_comb_properties(g["comb"].numpy(), g["logits"].numpy())
    zero = np.all(xb.reshape(T, -1) == 0, axis=1)
    assert zero.sum() == T // 100
    assert np.all(g["layer_input"].view(torch.int16).numpy()[zero] == 0)


def _sample_rows(T, extra=()):
    rng = np.random.default_rng(T)
    rows = set(rng.choice(T, size=min(T, 48), replace=False).tolist())
    rows |= {0, 1, 7, 8, T // 2, T - 9, T - 8, T - 1}
    rows |= set(int(r) for r in extra)
    return np.array(sorted(r for r in rows if 0 <= r < T))


def test_config2_prefill_full_size_sampled():
    """T=16384 with the fold, the launch configuration the benchmark times:
    pre and post on all tokens, compared with the oracle on sampled tokens,
    and properties checked on every token."""
    T = 16384
    gd = seam_inputs(T, seed=0, fold=True, with_y=True, device="cuda")
    out = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                          return_logits=True)
    xn = mhc.post(gd["x"], gd["y"], out["comb"], out["post"])
    torch.cuda.synchronize()
    rows = _sample_rows(T)
    g = {k: v.cpu() for k, v in out.items()}
    o, xb = _oracle_pre(gd, rows)
    _check_pre(g, o, xb, gd, fold=True, rows=rows)
    _check_comb_properties(g["comb"].numpy(), g["logits"].numpy())
    comb, pg = g["comb"].numpy()[rows], g["post"].numpy()[rows]
    yb = bf16_bits(gd["y"])[rows]
    o_bits, _ = oracle.post(xb, yb, comb, pg)
    g_bits = xn[rows.tolist()].cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16(g_bits, o_bits, "x_new", abs_scale=post_abs_scale(xb, yb, comb, pg))


def test_config4_stress_full_size_sampled():
    T = 65536
    gd = seam_inputs(T, seed=0, fold=True, stress=True, device="cuda")
    out = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                          return_logits=True)
    torch.cuda.synchronize()
    g = {k: v.cpu() for k, v in out.items()}
    for k in g:
        if g[k].dtype == torch.float32:
            assert torch.isfinite(g[k]).all(), k
    # Sinkhorn invariants on all 65,536 tokens (rows held to the oracle's
    # Sinkhorn of the GPU's logits: the +-300 stress logits do not converge
    # in 20 iterations even in exact arithmetic)
    _check_comb_properties(g["comb"].numpy(), g["logits"].numpy())
    xr = gd["x"].reshape(T, -1)
    zero = (xr == 0).all(1)
    big = xr.abs().amax(1) > 100
    extra = torch.nonzero(zero).flatten()[:8].tolist() + torch.nonzero(big).flatten()[:8].tolist()
    rows = _sample_rows(T, extra)
    o, xb = _oracle_pre(gd, rows)
    bound = logit_bound(xb, gd["fn"].cpu().numpy(), gd["alpha"].cpu().numpy(), o["logits"])
    assert_logits(g["logits"].numpy()[rows], o["logits"], bound)
    og = oracle.gates_from_logits(g["logits"].numpy()[rows].astype(np.float64))
    for k in ("pre", "post", "comb"):
        assert_gates(g[k].numpy()[rows], og[k], k + " (from gpu logits)")
    assert_bf16(g["layer_input"].view(torch.int16).numpy().view(np.uint16)[rows], o["layer_input"],
                "layer_input")
    assert torch.all(g["layer_input"].view(torch.int16)[zero.cpu()] == 0)


def test_entry_points_full_size_properties():
    """T = 16384 with the fold, the benchmark's launch configuration, for the
    other entry points: the broadcast pre and post equal the four-stream calls
    on the copied residual bit for bit; the non-delayed pre equals the
    delayed call fed its own pre bit for bit (two tensor-core passes against
    one); sampled rows of the broadcast seam against the oracle."""
    T = 16384
    gd = seam_inputs(T, seed=3, fold=True, with_y=True, device="cuda")
    xe = gd["x"][:, 0, :].contiguous()
    xb4 = xe[:, None, :].expand(T, 4, xe.shape[1]).contiguous()
    args = (gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    got_b = mhc.pre_delayed_broadcast(xe, gd["pre_in"], *args, return_logits=True)
    ref_b = mhc.pre_delayed(xb4, gd["pre_in"], *args, return_logits=True)
    xn_b = mhc.post_broadcast(xe, gd["y"], got_b["comb"], got_b["post"])
    xn_4 = mhc.post(xb4, gd["y"], got_b["comb"], got_b["post"])
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got_b[k], ref_b[k]), "broadcast " + k
    assert torch.equal(xn_b, xn_4)
    del xb4, ref_b, xn_4
    got_n = mhc.pre(gd["x"], *args, return_logits=True)
    ref_n = mhc.pre_delayed(gd["x"], got_n["pre"].clone(), *args, return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got_n[k], ref_n[k]), "non-delayed " + k
    rows = _sample_rows(T)
    g = {k: v.cpu() for k, v in got_b.items()}
    x1 = bf16_bits(xe)[rows]
    nw = bf16_bits(gd["norm_w"])
    o = oracle.pre_delayed_broadcast(x1, gd["pre_in"].cpu().numpy()[rows], gd["fn"].cpu().numpy(),
                                     gd["bias"].cpu().numpy(), gd["alpha"].cpu().numpy(), nw, nthreads=NTHREADS)
    _check_pre(g, o, oracle.broadcast_streams(x1), gd, fold=True, rows=rows)


def _pinned(t):
    return t.cpu().pin_memory()


@pytest.mark.parametrize("T", [1, 100, 300, 1000, 2048, 3000, 4097, 16384])
def test_seam_host_is_bit_identical_to_the_device_calls(T):
    """mhc_seam_host on pinned host activations (chunked, copies and kernels
    on three streams) gives the bits of mhc_pre_delayed + mhc_post on device
    copies: one chunk below 512 tokens, two chunks (384 + 616) at 1000; from
    2048 a 256-token head, 1024-token chunks, 512 tokens plus the remainder
    and a 256-token tail (2048: 256 + 1024 + 512 + 256; 3000: a 1464-token
    chunk, the largest, which sizes the buffers; 4097: a 513-token chunk)."""
    gd = seam_inputs(T, seed=2300 + T, fold=True, with_y=True, device="cuda")
    ref = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    xn_ref = mhc.post(gd["x"], gd["y"], ref["comb"], ref["post"])
    hx, hy, hp = _pinned(gd["x"]), _pinned(gd["y"]), _pinned(gd["pre_in"])
    got = mhc.seam_host(hx, hy, hp, gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                        outputs=("x_new", "pre", "post", "comb", "layer_input"))
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    assert torch.equal(got["x_new"], xn_ref.cpu())
    for k in ("pre", "post", "comb", "layer_input"):
        assert torch.equal(got[k], ref[k].cpu()), k


def test_seam_host_in_place_and_in_a_graph():
    """x_new may be the input buffer itself; the call captures into a CUDA
    graph (the library's copy streams fork from and join the capturing
    stream) and replays to the same bits."""
    T = 1000
    gd = seam_inputs(T, seed=2400, fold=True, with_y=True, device="cuda")
    ref = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"])
    xn_ref = mhc.post(gd["x"], gd["y"], ref["comb"], ref["post"]).cpu()
    hy, hp = _pinned(gd["y"]), _pinned(gd["pre_in"])
    hx = _pinned(gd["x"])
    got = mhc.seam_host(hx, hy, hp, gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], out={"x_new": hx})
    torch.cuda.synchronize()
    assert torch.equal(hx, xn_ref)
    assert torch.equal(got["pre"], ref["pre"].cpu())
    hx2 = _pinned(gd["x"])
    out = {"x_new": torch.empty_like(hx2).pin_memory(), "pre": torch.empty(T, 4).pin_memory()}
    s = torch.cuda.Stream()
    g = SeamGraph(lambda st: mhc.seam_host(hx2, hy, hp, gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"],
                                           out=out, stream=st), s)
    out["x_new"].zero_()
    g.replay(2)
    s.synchronize()
    assert mhc.device_status() == 0
    assert torch.equal(out["x_new"], xn_ref)
    assert torch.equal(out["pre"], ref["pre"].cpu())
    g.close()


@pytest.mark.parametrize("T,C,fold", [(4, 5120, True), (300, 5120, True), (1383, 5120, False), (700, 768, True),
                                      (16384, 5120, True)])
def test_packed_weights_are_bit_identical(T, C, fold):
    """mhc_pre_delayed_packed (planes packed once by mhc_pre_pack, one copy
    shared by the clusters, no per-call conversion) gives the bits of
    mhc_pre_delayed; below 256 tokens it runs the cluster kernel on fn."""
    gd = seam_inputs(T, C=C, seed=2500 + T, fold=fold, device="cuda")
    packed = mhc.pre_pack(gd["fn"], C=C)
    ref = mhc.pre_delayed(gd["x"], gd["pre_in"], gd["fn"], gd["bias"], gd["alpha"], gd["norm_w"], return_logits=True)
    got = mhc.pre_delayed_packed(gd["x"], gd["pre_in"], gd["fn"], packed, gd["bias"], gd["alpha"], gd["norm_w"],
                                 return_logits=True)
    torch.cuda.synchronize()
    assert mhc.device_status() == 0
    for k in ("pre", "post", "comb", "layer_input", "logits"):
        assert torch.equal(got[k], ref[k]), k
