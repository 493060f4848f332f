"""The allocation-free routing entry point against the workspace one.

beam_moe_route_noalloc serves callers that cannot allocate device memory (a
host framework that owns all device memory and gives a plugin only its
inputs and outputs, or a serving loop that must never allocate); its scratch
is a static device buffer inside the library.  This file is collected last
so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
from group_limited_routing_03_b300 import inputs
from parity_helpers import MARGIN, compare_routing, host_act

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from group_limited_routing_03_b300 import _build

    _build.build()
    moe.load()


def _route_both(wl, d):
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh)
    ids_ws = torch.empty((wl.T, 8), dtype=torch.int32, device="cuda")
    w_ws = torch.empty((wl.T, 8), dtype=torch.float32, device="cuda")
    moe.beam_moe_route(sh, d["x"], d["router_w"], d.get("bias"), ids_ws, w_ws, ws)
    ids_na = torch.full((wl.T, 8), -1, dtype=torch.int32, device="cuda")
    w_na = torch.zeros((wl.T, 8), dtype=torch.float32, device="cuda")
    moe.beam_moe_route_noalloc(sh, d["x"], d["router_w"], d.get("bias"), ids_na, w_na)
    torch.cuda.synchronize()
    return (ids_ws.cpu().numpy(), w_ws.cpu().numpy()), (ids_na.cpu().numpy(), w_na.cpu().numpy())


@pytest.mark.parametrize("name,T,H", [("decode", 64, 5120), ("skew", 300, 1024)])
def test_noalloc_route_matches_workspace_route_twice(name, T, H):
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        wl = inputs.workload(name, T=T, H=H, seed=100 * call + T)
        d = inputs.generate(wl, "cuda", experts=False)
        (ids_a, w_a), (ids_b, w_b) = _route_both(wl, d)
        b = None if d.get("bias") is None else d["bias"].cpu().numpy()
        ref = oracle.route(host_act(d["x"]), d["router_w"].cpu().numpy(), b)
        safe = ref["margin"] > MARGIN
        assert safe.mean() > 0.5
        np.testing.assert_array_equal(ids_b[safe], ids_a[safe])
        np.testing.assert_allclose(w_b[safe], w_a[safe], rtol=1e-5, atol=1e-6)
        assert ((ids_b >= 0) & (ids_b < 256)).all()


@pytest.mark.parametrize("name,T,H,x_dtype", [
    ("prefill", 600, 1024, "bf16"),    # BF16, T >= 512: the workspace route runs on the tensor cores
    ("prefill", 4097, 1024, "bf16"),   # T > 2048: one hidden-dimension split per tile
    ("skew", 5000, 1024, "f32"),       # past both split regimes, FP32 x, router bias
    ("prefill", 65536, 1024, "bf16"),  # the largest T: the 2 MiB histogram region exactly full
    ("prefill", 65536, 512, "f32"),
])
def test_noalloc_route_at_its_limits(name, T, H, x_dtype):
    """Both routing entry points against the oracle by the parity rules (ids
    exact where the margin is clear, in order where the adjacent score gaps
    are; near-ties validity-checked; weights to 1e-5)."""
    wl = inputs.workload(name, T=T, H=H, x_dtype=x_dtype, seed=7 * T + H)
    d = inputs.generate(wl, "cuda", experts=False)
    (ids_a, w_a), (ids_b, w_b) = _route_both(wl, d)
    b = None if d.get("bias") is None else d["bias"].cpu().numpy()
    ref = oracle.route(host_act(d["x"]), d["router_w"].cpu().numpy(), b, want_scores=True)
    compare_routing(ids_a, w_a, ref, bias=b)
    compare_routing(ids_b, w_b, ref, bias=b)


def test_noalloc_rejects_sizes_beyond_its_buffer():
    sh = moe.shape(65537, 256, 128)
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")  # never read: rejected on the host
    wr = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    ids = torch.zeros((16, 8), dtype=torch.int32, device="cuda")
    w = torch.zeros((16, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.BeamError) as ei:
        moe.beam_moe_route_noalloc(sh, x, wr, None, ids, w)
    assert ei.value.code == moe.BEAM_ERR_UNSUPPORTED
    # the shape rules of beam_moe_route apply too (one validation for both)
    for bad, code in ((moe.shape(16, 256, 100), moe.BEAM_ERR_UNSUPPORTED),
                      (moe.shape(16, 256, 128, routed_scale=float("inf")), moe.BEAM_ERR_INVALID_ARG)):
        with pytest.raises(moe.BeamError) as ei:
            moe.beam_moe_route_noalloc(bad, x, wr, None, ids, w)
        assert ei.value.code == code
