"""GPU parity of the post-norm residual update fused into the combine (Beam
launch post, section "Residual Stream"): the new stream against the oracle's
``residual_update`` of the oracle's own block output, on the same seeded
inputs.  Comparison rules as in parity_helpers; the stream adds one rounding
of the output to its dtype (2^-8 relative for BF16) to the block's tolerance."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import Y_TOL, compare_routing, host_act, oracle_route, oracle_y, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = float(np.float32(inputs.RESIDUAL_EPS))  # the kernel's eps is FP32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from group_limited_routing_03_b300 import _build

    _build.build()
    moe.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _tol(x_dtype, w_dtype):
    return Y_TOL[w_dtype] + (2.0 ** -8 if x_dtype == "bf16" else 0.0)


def _run(wl, d, weights, stream, g, k, *, out=None, want_y=True):
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh, "nvfp4" if wl.w_dtype == "nvfp4" else "bf16")
    out = torch.empty_like(stream) if out is None else out
    y = torch.empty_like(d["x"]) if want_y else None
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_forward_residual(sh, d["x"], d["router_w"], d.get("bias"), weights, stream, out, g, EPS, k, ids,
                                  w, ws, y=y)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, f"device status {code} where {where}"
    return out, y, ids, w


def _plain_y(wl, d, weights):
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh, "nvfp4" if wl.w_dtype == "nvfp4" else "bf16")
    y = torch.empty_like(d["x"])
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_forward(sh, d["x"], d["router_w"], d.get("bias"), weights, y, ids, w, ws)
    torch.cuda.synchronize()
    return y


# ---------------------------------------------------------------------------
# small shapes, every token compared; the row split of few tokens (clusters of
# 2..8 CTAs) and of many (one CTA per token, several passes per row)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,H,I,x_dtype,k", [(128, 256, 128, "f32", 2), (33, 256, 128, "bf16", 105),
                                             (300, 384, 256, "bf16", 3), (1, 256, 128, "bf16", 7),
                                             (77, 1024, 512, "f32", 50), (1100, 256, 128, "bf16", 4),
                                             (1030, 2048, 128, "f32", 9)])
def test_residual_small_all_tokens(T, H, I, x_dtype, k):
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype=x_dtype, seed=T + H + 7)
    dc = inputs.generate(wl, "cpu")
    dg = {kk: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for kk, v in dc.items()}
    weights = {kk: dg[kk].to(torch.bfloat16).contiguous() for kk in ("gate", "up", "down")}
    stream, g = inputs.residual_inputs(wl, "cpu")
    stream, g = stream.to(DEV), g.to(DEV)
    out, y, ids, w = _run(wl, dg, weights, stream, g, k)
    ref = oracle_route(dg)
    r = compare_routing(ids.cpu().numpy(), w.cpu().numpy(), ref)
    ow = {kk: dc[kk].numpy() for kk in ("gate", "up", "down")}
    y_ref = oracle_y(dg, np.arange(T), r.ids, r.weights, oracle_weights=ow)
    out_ref = oracle.residual_update(y_ref, host_act(stream), g.cpu().numpy(), EPS, k)
    err = rel_err(out.cpu().double().numpy(), out_ref)
    assert err <= _tol(x_dtype, "bf16"), err
    # the block output written beside the stream is the plain combine, bit for bit
    assert torch.equal(y, _plain_y(wl, dg, weights))
    if x_dtype == "f32":
        # with FP32 activations the kernel's y is the written y: the update
        # itself (norm, weights, scale) then agrees to FP32 rounding
        yy = y.double()
        inv = torch.rsqrt((yy * yy).mean(1, keepdim=True) + EPS)
        prop = np.sqrt((k - 1) / k) * stream.double() + yy * inv * g.double() / np.sqrt(k)
        e2 = float(((out.double() - prop).abs().max() / prop.abs().max()).item())
        assert e2 <= 1e-5, e2


def test_residual_in_place_and_without_y():
    """out == stream (in place) gives the same bits as a separate out; y may be
    omitted; the stage API with the residual at its combine step agrees."""
    wl = inputs.workload("tiny", T=200, H=512, I=256, x_dtype="bf16", seed=11)
    dg = inputs.generate(wl, DEV)
    weights = {kk: dg[kk].to(torch.bfloat16).contiguous() for kk in ("gate", "up", "down")}
    stream, g = inputs.residual_inputs(wl, DEV)
    ref_out, _, _, _ = _run(wl, dg, weights, stream, g, 5)
    s2 = stream.clone()
    out2, y2, _, _ = _run(wl, dg, weights, s2, g, 5, out=s2, want_y=False)
    assert out2.data_ptr() == s2.data_ptr() and y2 is None
    assert torch.equal(s2, ref_out)
    # stage by stage
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh)
    out3 = torch.empty_like(stream)
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    call = moe.ForwardCall(sh, dg["x"], dg["router_w"], None, weights, None, ids, w, ws,
                           residual=(stream, out3, g, EPS, 5))
    for i in range(len(moe.STAGES)):
        call.stage(i)
    torch.cuda.synchronize()
    assert torch.equal(out3, ref_out)


def test_residual_zero_output_keeps_scaled_stream():
    """Zero expert weights make the block's output exactly zero; with eps > 0
    the update is then exactly the kept stream, sqrt((k-1)/k) * stream, in
    FP32 (the product rounded once)."""
    wl = inputs.workload("tiny", T=64, H=256, I=128, x_dtype="f32", seed=5)
    dg = inputs.generate(wl, DEV)
    weights = {kk: torch.zeros_like(dg[kk], dtype=torch.bfloat16) for kk in ("gate", "up", "down")}
    stream, g = inputs.residual_inputs(wl, DEV)
    for k in (2, 105):
        out, y, _, _ = _run(wl, dg, weights, stream, g, k)
        assert torch.count_nonzero(y) == 0
        keep = torch.tensor(np.sqrt((k - 1) / k), dtype=torch.float32)
        assert torch.equal(out, stream * keep.to(DEV))


# ---------------------------------------------------------------------------
# full-size workloads: every token (decode, step 105) or sampled tokens and
# the near-ties
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,k,n_sample", [("decode", 105, None), ("decode", 2, 8), ("prefill", 40, 4)])
def test_residual_full_size(name, k, n_sample):
    wl = inputs.workload(name)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    stream, g = inputs.residual_inputs(wl, DEV)
    out, y, ids, w = _run(wl, dg, dg, stream, g, k, want_y=False)
    ref = oracle_route(dg)
    r = compare_routing(ids.cpu().numpy(), w.cpu().numpy(), ref)
    if n_sample is None:
        tok = np.arange(wl.T)
    else:
        rng = np.random.default_rng(wl.seed + k)
        tok = np.unique(np.concatenate([[0, wl.T - 1], rng.integers(0, wl.T, n_sample),
                                        np.nonzero(~r.safe)[0][:16]]))
    y_ref = oracle_y(dg, tok, r.ids[tok], r.weights[tok])
    out_ref = oracle.residual_update(y_ref, host_act(stream[torch.as_tensor(tok, device=DEV)]),
                                     g.cpu().numpy(), EPS, k)
    err = rel_err(out[torch.as_tensor(tok, device=DEV)].cpu().double().numpy(), out_ref)
    print(f"{name} k={k}: compared {len(tok)} tokens (near-ties {r.near_ties}); rel err {err:.3e}")
    assert err <= _tol(wl.x_dtype, wl.w_dtype), err
    del dg, out, stream
    gc.collect()
    torch.cuda.empty_cache()


def test_residual_maximum_token_count():
    """T = 2^20 at H = I = 128 (one CTA per row): the new stream of sampled
    tokens against the oracle."""
    T = 1 << 20
    wl = inputs.workload("prefill", T=T, H=128, I=128, seed=93)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    stream, g = inputs.residual_inputs(wl, DEV)
    out, _, ids, w = _run(wl, dg, dg, stream, g, 105, want_y=False)
    rng = np.random.default_rng(93)
    tok = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 2000)]))
    x_h = host_act(dg["x"])
    ref = oracle.route(x_h[tok], dg["router_w"].cpu().numpy(), None, want_scores=True)
    r = compare_routing(ids.cpu().numpy()[tok], w.cpu().numpy()[tok], ref)
    few = tok[:24]
    y_ref = oracle_y(dg, few, r.ids[:24], r.weights[:24])
    idx = torch.as_tensor(few, device=DEV)
    out_ref = oracle.residual_update(y_ref, host_act(stream[idx]), g.cpu().numpy(), EPS, 105)
    err = rel_err(out[idx].cpu().double().numpy(), out_ref)
    assert err <= _tol(wl.x_dtype, wl.w_dtype), err
    del dg, out, stream
    gc.collect()
    torch.cuda.empty_cache()
