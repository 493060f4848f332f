"""The debug build (libbeam_moe_debug.so, BEAM_DEBUG=1): device-side checks of
every index a kernel takes from the workspace.  A workspace corrupted on
purpose (route positions out of range, an inconsistent per-expert schedule)
is reported in the status word as BEAM_ERR_DEVICE_CHECK with the place of
the check, the bad accesses are skipped, and the context stays usable; on a
clean call the debug build gives the release build's bits.  The corruptions
are only ever fed to the debug build, whose checks cover every access they
could reach."""
import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
from group_limited_routing_03_b300 import inputs
from parity_helpers import seeded_routing

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEVICE_CHECK = 6


@pytest.fixture(scope="module")
def debug_lib():
    from group_limited_routing_03_b300 import _build

    _build.build()
    _build.build(debug=True)
    release = moe.load()
    dbg = moe.load_debug()
    assert dbg.beam_moe_debug_build() == 1 and release.beam_moe_debug_build() == 0
    return release, dbg


@pytest.fixture
def use_debug(debug_lib, monkeypatch):
    """The binding's calls go to the debug build for the test."""
    monkeypatch.setattr(moe, "_lib", debug_lib[1])
    return debug_lib[1]


def _setup(w_dtype, T=40, H=512, I=256, seed=3):
    """w_dtype "nvfp4_a4": the NVFP4 weights with W4A4 GEMMs."""
    fp4 = w_dtype in ("nvfp4", "nvfp4_a4")
    wl = inputs.workload("nvfp4" if fp4 else "tiny", T=T, H=H, I=I, x_dtype="bf16",
                         w_dtype="nvfp4" if fp4 else w_dtype, seed=seed)
    d = inputs.generate(wl, DEV)
    keys = ("gate", "up", "down") + (("gate_rs", "up_rs", "down_rs") if w_dtype == "fp8" else ()) + (
        ("gate_sf", "up_sf", "down_sf", "gate_gs", "up_gs", "down_gs") if fp4 else ())
    weights = {k: d[k] for k in keys}
    if w_dtype == "nvfp4_a4":
        weights["activations"] = "nvfp4"
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh, w_dtype)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((T, 8), dtype=torch.float32, device=DEV)
    call = moe.ForwardCall(sh, d["x"], d["router_w"], None, weights, y, ids, w, ws)
    return sh, ws, y, call, moe.workspace_layout(sh, w_dtype)


def _i32(ws, off, n):
    return ws[off:off + 4 * n].view(torch.int32)


@pytest.mark.parametrize("w_dtype,where", [("bf16", 22), ("fp8", 26), ("nvfp4", 27), ("nvfp4_a4", 27)])
def test_bad_route_positions_before_the_gather(use_debug, w_dtype, where):
    sh, ws, y, call, lay = _setup(w_dtype)
    R = sh.T * 8
    call.stage(0)
    call.stage(1)
    pos = _i32(ws, lay["pos"], R)
    pos[5] = 10 ** 8
    pos[17] = R
    pos[3] = -7
    for i in range(2, 6):
        call.stage(i)
    code, at = moe.beam_moe_read_device_status(ws)
    assert (code, at) == (DEVICE_CHECK, where)
    assert torch.isfinite(y.float()).all()
    call.run()  # the context is still usable (and a clean call reports nothing)
    assert moe.beam_moe_read_device_status(ws)[0] == 0


@pytest.mark.parametrize("residual,where", [(False, 23), (True, 28)])
def test_bad_route_positions_before_the_combine(use_debug, residual, where):
    sh, ws, y, call, lay = _setup("bf16")
    if residual:
        stream = torch.randn((sh.T, sh.H), device=DEV).to(torch.bfloat16)
        g = torch.ones(sh.H, device=DEV)
        a = call._keep
        call = moe.ForwardCall(sh, a[0], a[1], a[2], a[3], None, a[5], a[6], ws,
                               residual=(stream, stream, g, 1e-6, 3))
    for i in range(5):
        call.stage(i)
    pos = _i32(ws, lay["pos"], sh.T * 8)
    pos[9] = 1 << 30
    call.stage(5)
    code, at = moe.beam_moe_read_device_status(ws)
    assert (code, at) == (DEVICE_CHECK, where)


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8", "nvfp4"])
def test_inconsistent_schedule_before_the_gemms(use_debug, w_dtype):
    """counts no longer match offsets: the check before the gate/up GEMM
    reports it and leaves the GEMM no work (it would store past the routes)."""
    sh, ws, y, call, lay = _setup(w_dtype)
    for i in range(3):
        call.stage(i)
    counts = _i32(ws, lay["counts"], 256)
    counts[7] += 1000
    for i in range(3, 6):
        call.stage(i)
    code, at = moe.beam_moe_read_device_status(ws)
    assert (code, at) == (DEVICE_CHECK, 24)
    assert moe.beam_moe_stage_kernel_count(sh, 3, moe.BEAM_BF16, w_dtype) == 2  # the check, the GEMM


def test_expert_ids_out_of_range(use_debug):
    """Ids outside [0, 256) given to the experts call are dropped (both
    builds check them): the other tokens' outputs keep their bits."""
    T, H, I = 64, 256, 256
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype="bf16", seed=12)
    d = inputs.generate(wl, DEV)
    wts = {k: d[k].to(torch.bfloat16).contiguous() for k in ("gate", "up", "down")}
    ids, w = seeded_routing(T, seed=4)
    bad = ids.clone()
    bad[10, 3] = 300
    bad[20, 0] = -1
    sh = moe.shape(T, H, I)
    outs = []
    for i in (ids, bad):
        ws = moe.alloc_workspace(sh)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        moe.beam_moe_experts(sh, d["x"], wts, i.to(DEV), w.to(DEV), y, ws)
        outs.append((y, moe.beam_moe_read_device_status(ws)))
    assert outs[0][1][0] == 0
    assert outs[1][1] == (DEVICE_CHECK, 20)
    keep = torch.ones(T, dtype=torch.bool)
    keep[[10, 20]] = False
    assert torch.equal(outs[0][0][keep.to(DEV)], outs[1][0][keep.to(DEV)])


@pytest.mark.parametrize("w_dtype", ["bf16", "fp8", "nvfp4", "nvfp4_a4"])
def test_debug_build_gives_the_release_bits(debug_lib, monkeypatch, w_dtype):
    release, dbg = debug_lib
    res = []
    for lib in (release, dbg):
        monkeypatch.setattr(moe, "_lib", lib)
        sh, ws, y, call, _ = _setup(w_dtype, T=70, seed=8)
        call.run()
        assert moe.beam_moe_read_device_status(ws)[0] == 0
        res.append((y, call._keep[5], call._keep[6]))
    for a, b in zip(*res):
        assert torch.equal(a, b)
