"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Rules are stated in parity_helpers."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import (Y_TOL, chunk_rows, compare_routing, full_size_tokens, host_act, oracle_route,
                            oracle_y, record_near_ties, rel_err, seeded_routing)

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


def _gpu_inputs(wl, *, cpu_gen=False):
    """Inputs on the GPU; for small workloads drawn on the CPU then copied."""
    if cpu_gen:
        d = inputs.generate(wl, "cpu")
        out = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        return out, d
    return inputs.generate(wl, DEV), None


def _bf16_weights(d):
    return {k: d[k].to(torch.bfloat16).contiguous() for k in ("gate", "up", "down")}


def _run_forward(wl, d, weights):
    sh = moe.shape(wl.T, wl.H, wl.I)
    ws = moe.alloc_workspace(sh, "nvfp4" if wl.w_dtype == "nvfp4" else "bf16")
    y = torch.empty((wl.T, wl.H), dtype=d["x"].dtype, device=DEV)
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_forward(sh, d["x"], d["router_w"], d.get("bias"), weights, y, ids, w, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, f"device status {code} where {where}"
    return y, ids, w, ws


# ---------------------------------------------------------------------------
# whole block, small shapes (every token compared)
# ---------------------------------------------------------------------------
def _small_forward_vs_oracle(wl, *, fp32_originals):
    """Forward of a small workload; routing checked on every token, y of every
    token (near-ties with the GPU's ids) against the oracle."""
    dg, dc = _gpu_inputs(wl, cpu_gen=True)
    weights = _bf16_weights(dg) if fp32_originals else dg
    y, ids, w, _ = _run_forward(wl, dg, weights)
    ref = oracle_route(dg)
    r = compare_routing(ids.cpu().numpy(), w.cpu().numpy(), ref)
    tok = np.arange(wl.T)
    # FP32 workloads: the oracle runs the FP32 originals (the GPU gets BF16 copies)
    ow = {k: dc[k].numpy() for k in ("gate", "up", "down")} if fp32_originals else None
    y_ref = oracle_y(dg, tok, r.ids, r.weights, oracle_weights=ow)
    err = rel_err(y.cpu().double().numpy(), y_ref)
    return r, err


def test_tiny_workload_as_specified():
    """The tiny layer exactly as specified: T=128, H=256, I=128, 256 experts,
    FP32 x / router / experts drawn with seed 0; every token compared."""
    wl = inputs.workload("tiny")
    assert (wl.T, wl.H, wl.I, wl.x_dtype, wl.w_dtype, wl.seed) == (128, 256, 128, "f32", "f32", 0)
    r, err = _small_forward_vs_oracle(wl, fp32_originals=True)
    record_near_ties("tiny", wl.T, r, wl.T)
    assert err <= Y_TOL["f32"], err


@pytest.mark.parametrize("T,H,I,x_dtype", [(128, 256, 128, "f32"), (1, 256, 128, "bf16"), (33, 256, 128, "bf16"),
                                           (300, 384, 256, "bf16"), (77, 1024, 512, "f32")])
def test_forward_small_all_tokens(T, H, I, x_dtype):
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype=x_dtype, seed=T + H)
    _, err = _small_forward_vs_oracle(wl, fp32_originals=True)
    assert err <= Y_TOL["bf16"], err


@pytest.mark.parametrize("T,H,I", [(300, 512, 256), (40, 256, 512), (1, 256, 256), (257, 256, 256)])
def test_forward_nvfp4_small_all_tokens(T, H, I):
    """NVFP4 experts (E2M1 codes, E4M3 block scales, FP32 global scale),
    expanded exactly to BF16 in TMEM, BF16 activations."""
    wl = inputs.workload("nvfp4", T=T, H=H, I=I, seed=31 + T)
    _, err = _small_forward_vs_oracle(wl, fp32_originals=False)
    assert err <= Y_TOL["nvfp4"], err


@pytest.mark.parametrize("name,T,H", [("prefill", 600, 1024), ("skew", 1536, 5120), ("prefill", 513, 256)])
def test_route_tensor_core_path(name, T, H):
    """T >= 512 BF16 tokens route on the tensor cores (three-term BF16 split
    of the FP32 router weight, FP32 accumulation); same parity rules."""
    wl = inputs.workload(name, T=T, H=H, seed=40 + T)
    d = inputs.generate(wl, DEV, experts=False)
    sh = moe.shape(T, H, 128)
    ws = moe.alloc_workspace(sh)
    ids = torch.empty((T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_route(sh, d["x"], d["router_w"], d.get("bias"), ids, w, ws)
    assert moe.beam_moe_read_device_status(ws)[0] == 0
    ref = oracle_route(d)
    bias = None if d.get("bias") is None else d["bias"].cpu().numpy()
    r = compare_routing(ids.cpu().numpy(), w.cpu().numpy(), ref, bias=bias)
    record_near_ties(f"{name} route T={T} H={H} (tensor-core router)", T, r, 0)
    # dispatch histograms written by the router agree with the ids
    moe.beam_moe_dispatch(sh, ids, ws)
    lay = moe.workspace_layout(sh)
    counts = ws[lay["counts"]:lay["counts"] + 1024].view(torch.int32).cpu().numpy()
    np.testing.assert_array_equal(counts, np.bincount(ids.cpu().numpy().reshape(-1), minlength=256))


def test_zero_input_exact():
    wl = inputs.workload("tiny", T=40, x_dtype="bf16")
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    dg["x"] = torch.zeros_like(dg["x"])
    y, ids, w, _ = _run_forward(wl, dg, _bf16_weights(dg))
    assert (ids.cpu() == torch.arange(8, dtype=torch.int32)).all()
    assert (w.cpu() == 2.5 / 8).all()
    assert (y.cpu() == 0).all()


# ---------------------------------------------------------------------------
# dispatch and experts with a routing drawn independently of the router
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,hot", [(1000, None), (3000, (5, 77, 200)), (1, None), (37, (0, 1, 2, 3, 4, 5, 6, 7))])
def test_dispatch_matches_oracle(T, hot):
    ids, _ = seeded_routing(T, seed=T, hot=hot)
    sh = moe.shape(T, 256, 128)
    ws = moe.alloc_workspace(sh)
    moe.beam_moe_dispatch(sh, ids.to(DEV), ws)
    lay = moe.workspace_layout(sh)
    torch.cuda.synchronize()
    R = T * 8

    def view(off, n):
        return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    ref = oracle.dispatch(ids.numpy())
    np.testing.assert_array_equal(view(lay["counts"], 256), ref["counts"])
    np.testing.assert_array_equal(view(lay["offsets"], 257), ref["offsets"])
    np.testing.assert_array_equal(view(lay["perm"], R), ref["perm"])
    np.testing.assert_array_equal(view(lay["pos"], R), ref["pos"])


@pytest.mark.parametrize("T,H,I,hot", [(600, 256, 128, (3, 77, 130, 131, 200, 201, 254, 255)),
                                       (300, 512, 256, (9,)), (17, 256, 384, None)])
def test_experts_given_routing(T, H, I, hot):
    """Experts + combine on a seeded routing; `hot` experts get every token,
    so they run several 256-token chunks."""
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype="bf16", seed=7 + T)
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    ids, w = seeded_routing(T, seed=T + 1, hot=hot)
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moe.beam_moe_experts(sh, dg["x"], _bf16_weights(dg), ids.to(DEV), w.to(DEV), y, ws)
    assert moe.beam_moe_read_device_status(ws)[0] == 0
    tok = np.arange(T)
    y_ref = oracle_y(dg, tok, ids.numpy(), w.numpy().astype(np.float64))
    assert rel_err(y.cpu().double().numpy(), y_ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("T,H,I,hot", [(600, 512, 512, None), (700, 512, 256, (4, 5, 6, 200)),
                                       (640, 1024, 256, (3, 250)), (256, 256, 768, None)])
def test_experts_cta_pair_path(T, H, I, hot):
    """Shapes that take the two-CTA (M=256 pair MMA) grouped GEMMs: BF16
    weights, 256-route chunks, H a multiple of 512 and I of 256 (the last
    shape checks the one-CTA fallback)."""
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype="bf16", seed=3 + T)
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    ids, w = seeded_routing(T, seed=T + 2, hot=hot)
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moe.beam_moe_experts(sh, dg["x"], dg, ids.to(DEV), w.to(DEV), y, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, (code, where)
    y_ref = oracle_y(dg, np.arange(T), ids.numpy(), w.numpy().astype(np.float64))
    assert rel_err(y.cpu().double().numpy(), y_ref) <= Y_TOL["bf16"]


def test_experts_nvfp4_given_routing():
    """NVFP4 experts on a seeded routing whose hot experts take every token
    (several chunks per expert)."""
    T, H, I = 520, 256, 256
    wl = inputs.workload("nvfp4", T=T, H=H, I=I, seed=77)
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    ids, w = seeded_routing(T, seed=5, hot=(1, 100, 255))
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh, "nvfp4")
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moe.beam_moe_experts(sh, dg["x"], dg, ids.to(DEV), w.to(DEV), y, ws)
    assert moe.beam_moe_read_device_status(ws)[0] == 0
    y_ref = oracle_y(dg, np.arange(T), ids.numpy(), w.numpy().astype(np.float64))
    assert rel_err(y.cpu().double().numpy(), y_ref) <= Y_TOL["nvfp4"]


def test_identical_experts_closed_form():
    """All experts share one weight set, so y = 2.5 * f(x) whatever the routing."""
    T, H, I = 200, 256, 256
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype="bf16", seed=99)
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    for k in ("gate", "up", "down"):
        dg[k] = dg[k][:1].expand_as(dg[k]).contiguous()
    y, ids, w, _ = _run_forward(wl, dg, dg)
    x = host_act(dg["x"])
    f = oracle.expert_ffn(x, *(host_act(dg[k][0]) for k in ("gate", "up", "down")))
    assert rel_err(y.cpu().double().numpy(), 2.5 * f) <= Y_TOL["bf16"]


def test_bounded_wait_reports_timeout_and_context_survives():
    sh = moe.shape(8, 256, 128)
    ws = moe.alloc_workspace(sh)
    moe.beam_moe_debug_timeout(ws, 2000)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == moe.BEAM_ERR_TIMEOUT and where == 9
    assert moe.beam_moe_read_device_status(ws)[0] == 0  # cleared
    wl = inputs.workload("tiny", T=8, x_dtype="bf16")
    dg, _ = _gpu_inputs(wl, cpu_gen=True)
    _run_forward(wl, dg, _bf16_weights(dg))  # the context is still usable


# ---------------------------------------------------------------------------
# full-size workloads: routing on every token, outputs on sampled tokens
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["decode", "prefill", "nvfp4", "skew", "nvfp4_dec"])
def test_full_size_workloads(name):
    """Routing of every token against the oracle; outputs of every token at
    decode sizes, else of tokens covering every touched expert and every
    unit of work (token chunk) of the three most-loaded experts, plus every
    near-tie token (with the GPU's ids)."""
    wl = inputs.workload(name)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    y, ids, w, ws = _run_forward(wl, dg, dg)
    ref = oracle_route(dg)
    bias = None if dg.get("bias") is None else dg["bias"].cpu().numpy()
    ids_h = ids.cpu().numpy()
    r = compare_routing(ids_h, w.cpu().numpy(), ref, bias=bias)
    counts = np.bincount(ids_h.reshape(-1), minlength=256)
    if name == "skew":
        assert counts.max() > 10 * counts.mean()
    tok = full_size_tokens(ids_h, chunk_rows(wl.T, wl.w_dtype), extra=np.nonzero(~r.safe)[0][:64])
    y_ref = oracle_y(dg, tok, r.ids[tok], r.weights[tok])
    err = rel_err(y.cpu()[tok].double().numpy(), y_ref)
    record_near_ties(name, wl.T, r, len(tok))
    print(f"{name}: near-ties {r.near_ties} of {wl.T}; compared {len(tok)} tokens "
          f"({int((counts > 0).sum())} experts touched); rel err {err:.3e}")
    assert err <= Y_TOL[wl.w_dtype], err
    del dg, y, ws
    gc.collect()
    torch.cuda.empty_cache()


def test_maximum_token_count():
    """T = 2^20, the largest token count the library takes (8M routes), at
    H = I = 128: the dispatch (per-expert counts, stable positions, their
    inverse) checked against the GPU's own ids in full, routing and y of
    sampled tokens against the oracle."""
    T = 1 << 20
    wl = inputs.workload("prefill", T=T, H=128, I=128, seed=91)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    y, ids, w, ws = _run_forward(wl, dg, dg)
    sh = moe.shape(wl.T, wl.H, wl.I)
    lay = moe.workspace_layout(sh)
    R = T * 8

    def ws_i32(off, n):
        return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    ids_h = ids.cpu().numpy()
    counts = ws_i32(lay["counts"], 256)
    np.testing.assert_array_equal(counts, np.bincount(ids_h.reshape(-1), minlength=256))
    offsets = ws_i32(lay["offsets"], 257)
    assert offsets[0] == 0 and offsets[-1] == R and (np.diff(offsets) == counts).all()
    perm = ws_i32(lay["perm"], R)
    pos = ws_i32(lay["pos"], R)
    np.testing.assert_array_equal(perm[pos], np.arange(R))
    # routes of each expert in ascending route index
    e_of_p = ids_h.reshape(-1)[perm]
    assert (np.diff(e_of_p) >= 0).all()
    same = np.diff(e_of_p) == 0
    assert (np.diff(perm)[same] > 0).all()
    del perm, pos, e_of_p, same
    # routing and outputs of sampled tokens
    rng = np.random.default_rng(91)
    tok = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 2000)]))
    x_h = host_act(dg["x"])
    bias = None if dg.get("bias") is None else dg["bias"].cpu().numpy()
    ref = oracle.route(x_h[tok], dg["router_w"].cpu().numpy(), bias, want_scores=True)
    r = compare_routing(ids_h[tok], w.cpu().numpy()[tok], ref, bias=bias)
    few = tok[:24]
    y_ref = oracle_y(dg, few, r.ids[:24], r.weights[:24])
    err = rel_err(y.cpu()[few].double().numpy(), y_ref)
    assert err <= Y_TOL["bf16"], err
    del dg, y, ws
    gc.collect()
    torch.cuda.empty_cache()


def test_cuda_graph_replay_matches_direct_calls():
    """A decode-size forward recorded in a CUDA graph and replayed on new
    inputs gives the bits of direct calls on the same inputs."""
    wl = inputs.workload("tiny", T=64, H=512, I=256, x_dtype="bf16", seed=17)
    dg = inputs.generate(wl, DEV)
    layer = moe.BeamMoE(dg["router_w"], None, _bf16_weights(dg), max_tokens=wl.T, pack=True)
    graphed = moe.GraphedForward(layer, wl.T)
    g = torch.Generator(device=DEV).manual_seed(5)
    for _ in range(3):
        x = torch.randn((wl.T, wl.H), generator=g, device=DEV).to(torch.bfloat16)
        y_g, ids_g, w_g = (t.clone() for t in graphed(x))
        torch.cuda.synchronize()
        y_d, ids_d, w_d = layer(x)
        torch.cuda.synchronize()
        assert torch.equal(ids_g, ids_d) and torch.equal(w_g, w_d) and torch.equal(y_g, y_d)
    code, where = moe.beam_moe_read_device_status(layer.workspace)
    assert code == 0, f"device status {code} where {where}"
