"""GPU parity of the FP8 expert path (E4M3 weights with FP32 row scales,
activations quantised per row to E4M3 at run time, kind::f8f6f4 MMAs)
against the oracle's expert_ffn_fp8 on the same seeded inputs.  Rules as in
parity_helpers; the run-time codes of x are compared byte for byte."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import (Y_TOL, chunk_rows, compare_routing, full_size_tokens, host_act, oracle_route, oracle_y,
                            record_near_ties, rel_err)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from group_limited_routing_03_b300 import _build

    _build.build()
    moe.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _weights(d, layout, sh):
    w = {k: d[k] for k in ("gate", "up", "down", "gate_rs", "up_rs", "down_rs")}
    if layout == "tiled":
        w = moe.pack_weights(sh, w)
    return w


def _forward(wl, d, weights):
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh, "fp8")
    y = torch.empty((wl.T, wl.H), dtype=d["x"].dtype, device=DEV)
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_forward(sh, d["x"], d["router_w"], d.get("bias"), weights, y, ids, w, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, f"device status {code} where {where}"
    return y, ids, w, ws


# CTA pairs (T >= 256 routes per chunk, H % 512 == 0, I % 256 == 0), one CTA
# per unit with two-tile down units (H % 256 == 0), several k-blocks, both
# weight layouts, FP32 and BF16 x, a single token
@pytest.mark.parametrize("T,H,I,x_dtype,layout", [
    (128, 256, 128, "f32", "rows"), (33, 256, 256, "bf16", "rows"), (300, 512, 256, "bf16", "rows"),
    (300, 512, 256, "bf16", "tiled"), (1, 256, 128, "bf16", "tiled"), (600, 1024, 512, "bf16", "tiled"),
    (77, 512, 384, "bf16", "rows"), (257, 256, 256, "bf16", "rows")])
def test_fp8_small_all_tokens(T, H, I, x_dtype, layout):
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype=x_dtype, w_dtype="fp8", seed=T + H + 3)
    dc = inputs.generate(wl, "cpu")
    dg = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in dc.items()}
    sh = moe.shape(wl.T, wl.H, wl.I)
    y, ids, w, _ = _forward(wl, dg, _weights(dg, layout, sh))
    ref = oracle_route(dg)
    r = compare_routing(ids.cpu().numpy(), w.cpu().numpy(), ref)
    y_ref = oracle_y(dg, np.arange(wl.T), r.ids, r.weights)
    err = rel_err(y.cpu().double().numpy(), y_ref)
    assert err <= Y_TOL["fp8"], err


def test_fp8_activation_codes():
    """x's E4M3 codes and row scales in the workspace equal the oracle's
    quantisation of the same rows, byte for byte; h's codes follow the same
    rule (torch's cast of h / (amax / 448)) from the h the GPU stored."""
    wl = inputs.workload("tiny", T=200, H=512, I=256, x_dtype="bf16", w_dtype="fp8", seed=4)
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    _, _, _, ws = _forward(wl, dg, _weights(dg, "rows", sh))
    lay = moe.workspace_layout(sh, "fp8")
    R = wl.T * 8
    perm = ws[lay["perm"]:lay["perm"] + 4 * R].view(torch.int32).cpu().numpy()
    xq = ws[lay["xq"]:lay["xq"] + R * wl.H].view(R, wl.H).cpu().numpy()
    xs = ws[lay["xs"]:lay["xs"] + 4 * R].view(torch.float32).cpu().numpy()
    rows = host_act(dg["x"])[perm // 8]
    rows32 = (rows.astype(np.uint32) << 16).view(np.float32)
    codes, scales = oracle.quantize_e4m3_rows(rows32)
    np.testing.assert_array_equal(xq, codes)
    np.testing.assert_array_equal(xs, scales)
    # h: BF16 [R, I] in perm order, its codes in hq
    h = ws[lay["h"]:lay["h"] + 2 * R * wl.I].view(torch.bfloat16).view(R, wl.I).float()
    hq = ws[lay["hq"]:lay["hq"] + R * wl.I].view(R, wl.I)
    hs = ws[lay["hs"]:lay["hs"] + 4 * R].view(torch.float32)
    amax = h.abs().amax(1)
    # tensor / tensor: torch divides by a Python scalar through its reciprocal
    s = amax / torch.full_like(amax, 448.0)
    s = torch.where(s > 0, s, torch.ones_like(s))
    assert torch.equal(hs, s)
    want = (h / s[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(hq, want)
    xdt = moe.BEAM_BF16
    assert moe.beam_moe_stage_kernel_count(sh, 4, xdt, "fp8") == 2  # down: quantise h, then the GEMM
    assert moe.beam_moe_stage_kernel_count(sh, 4, xdt, "bf16") == 1
    assert moe.beam_moe_stage_kernel_count(sh, 4, xdt, "nvfp4") == 2  # down: h to FP16 rows, then the GEMM


@pytest.mark.parametrize("name", ["fp8_decode", "fp8"])
def test_fp8_full_size(name):
    """Routing of every token; outputs of every token at decode size, else of
    tokens covering every touched expert and every token chunk of the three
    most-loaded experts, plus the near-tie tokens (with the GPU's ids)."""
    wl = inputs.workload(name)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    y, ids, w, ws = _forward(wl, dg, _weights(dg, "tiled", sh))
    ref = oracle_route(dg)
    ids_h = ids.cpu().numpy()
    r = compare_routing(ids_h, w.cpu().numpy(), ref)
    tok = full_size_tokens(ids_h, chunk_rows(wl.T, wl.w_dtype), extra=np.nonzero(~r.safe)[0][:64])
    y_ref = oracle_y(dg, tok, r.ids[tok], r.weights[tok])
    err = rel_err(y.cpu()[tok].double().numpy(), y_ref)
    record_near_ties(name, wl.T, r, len(tok))
    print(f"{name}: near-ties {r.near_ties} of {wl.T}; compared {len(tok)} tokens; rel err {err:.3e}")
    assert err <= Y_TOL["fp8"], err
    del dg, y, ws
    gc.collect()
    torch.cuda.empty_cache()


def test_fp8_stages_equal_forward():
    """The FP8 forward issued stage by stage (the h quantisation inside the
    down stage) gives the bits of beam_moe_forward."""
    wl = inputs.workload("tiny", T=150, H=512, I=256, x_dtype="bf16", w_dtype="fp8", seed=8)
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    weights = _weights(dg, "tiled", sh)
    y, ids, w, _ = _forward(wl, dg, weights)
    ws = moe.alloc_workspace(sh, "fp8")
    y2 = torch.empty_like(y)
    ids2, w2 = torch.empty_like(ids), torch.empty_like(w)
    call = moe.ForwardCall(sh, dg["x"], dg["router_w"], None, weights, y2, ids2, w2, ws)
    for i in range(len(moe.STAGES)):
        call.stage(i)
    torch.cuda.synchronize()
    assert torch.equal(ids2, ids) and torch.equal(w2, w) and torch.equal(y2, y)


def test_fp8_maximum_token_count():
    """T = 2^20 (8M routes) at H = I = 128: routing and y of sampled tokens
    against the oracle, and the x codes of sampled route rows byte for byte."""
    T = 1 << 20
    wl = inputs.workload("fp8", T=T, H=128, I=128, seed=92)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    y, ids, w, ws = _forward(wl, dg, _weights(dg, "tiled", sh))
    rng = np.random.default_rng(92)
    tok = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 2000)]))
    x_h = host_act(dg["x"])
    ref = oracle.route(x_h[tok], dg["router_w"].cpu().numpy(), None, want_scores=True)
    r = compare_routing(ids.cpu().numpy()[tok], w.cpu().numpy()[tok], ref)
    few = tok[:24]
    y_ref = oracle_y(dg, few, r.ids[:24], r.weights[:24])
    err = rel_err(y.cpu()[few].double().numpy(), y_ref)
    assert err <= Y_TOL["fp8"], err
    # x codes of sampled route rows (perm order in the workspace)
    lay = moe.workspace_layout(sh, "fp8")
    R = T * 8
    rows = np.unique(np.concatenate([[0, R - 1], rng.integers(0, R, 3000)]))
    perm = ws[lay["perm"]:lay["perm"] + 4 * R].view(torch.int32)[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    xq = ws[lay["xq"]:lay["xq"] + R * wl.H].view(R, wl.H)[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    xs = ws[lay["xs"]:lay["xs"] + 4 * R].view(torch.float32)[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    rows32 = (x_h[perm // 8].astype(np.uint32) << 16).view(np.float32)
    codes, scales = oracle.quantize_e4m3_rows(rows32)
    np.testing.assert_array_equal(xq, codes)
    np.testing.assert_array_equal(xs, scales)
    del dg, y, ws
    gc.collect()
    torch.cuda.empty_cache()
