"""W4A4 (BEAM_NVFP4_A4): NVFP4 expert weights with every GEMM input row
quantised to NVFP4 at run time by the weights' recipe applied per row (the
library's reading of the NVFP4 checkpoint of the Beam launch post, section
"Mixture of Experts", for activations).

The quantiser is compared with the oracle's byte for byte (codes, block
scales, global scales) on rows of varied character, including rows built so
that elements fall exactly on the E2M1 rounding midpoints; inside a forward
the quantised x and h rows the GEMMs read are compared with the oracle
quantiser applied to the same inputs (x, and the GPU's own BF16 h), the down
GEMM with the oracle's decoders and a float64 matmul over those rows, and
the outputs with the oracle's W4A4 expert end to end."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import (Y_TOL, chunk_rows, full_size_tokens, host_act, host_expert, oracle_y, rel_err,
                            seeded_routing)

pytestmark = pytest.mark.gpu
DEV = "cuda"

E2M1 = np.array([oracle.decode_e2m1(c) for c in range(16)])
E4M3 = np.array([oracle.decode_e4m3(c) for c in range(256)])


@pytest.fixture(scope="module", autouse=True)
def _built():
    from group_limited_routing_03_b300 import _build

    _build.build()
    moe.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _values(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP16 bit patterns of e2m1 * e4m3 (exact in FP16) from the oracle's
    codes [n, K] and block scales [n, K/16]."""
    v = E2M1[codes] * E4M3[np.repeat(scales, 16, axis=1)]
    return v.astype(np.float16).view(np.uint16)


def _tie_row(K: int) -> np.ndarray:
    """A row whose first element (2688 = 6 * 448) makes its global scale
    exactly 1; then blocks with maximum 6 (block scale 1) and maximum 3
    (block scale 1/2), so that a / (s * g) is exact and lands on every E2M1
    rounding midpoint (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5), both signs."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    blk6 = [6.0] + mids + [-m for m in mids] + [0.1]
    blk3 = [3.0] + [m / 2 for m in mids] + [-m / 2 for m in mids] + [-0.0]
    row = [2688.0] + [0.0] * 15
    while len(row) < K:
        row += blk6 if (len(row) // 16) % 2 else blk3
    return np.array(row[:K], dtype=np.float32)


def _rows(n: int, K: int, seed: int) -> torch.Tensor:
    """FP32 rows: N(0,1); cubes of N(0,1) (heavy tails); N(0,1) * 2^-100
    (tiny, the global scale still a normal FP32 number); zero; N(0,1) with
    every 7th element * 2^20 (most block scales underflow to small E4M3
    subnormals or zero); N(0,1) on a grid of 1/4; and the midpoint row."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((n, K), generator=g)
    a[1::7] = a[1::7] ** 3
    a[2::7] *= 2.0 ** -100
    a[3::7] = 0.0
    a[4::7, ::7] *= 2.0 ** 20
    a[5::7] = torch.round(a[5::7] * 4) / 4
    a[6::7] = torch.from_numpy(_tie_row(K))
    return a


@pytest.mark.parametrize("K,dtype", [(256, torch.float32), (5120, torch.float32), (5120, torch.bfloat16),
                                     (2560, torch.bfloat16)])
def test_quantiser_matches_the_oracle_byte_for_byte(K, dtype):
    n = 49
    a = _rows(n, K, seed=K).to(dtype)
    codes = torch.empty((n, K), dtype=torch.uint8, device=DEV)
    scales = torch.empty((n, K // 16), dtype=torch.uint8, device=DEV)
    glob = torch.empty(n, dtype=torch.float32, device=DEV)
    values = torch.empty((n, K), dtype=torch.float16, device=DEV)
    moe.beam_debug_quantize_nvfp4(a.to(DEV), codes, scales, glob, values)
    torch.cuda.synchronize()
    oc, os_, og = oracle.quantize_nvfp4_rows(a.float().numpy())   # BF16 -> FP32 is exact
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy(), os_)
    np.testing.assert_array_equal(glob.cpu().numpy().view(np.uint32), og.view(np.uint32))
    np.testing.assert_array_equal(values.cpu().numpy().view(np.uint16), _values(oc, os_))
    # the midpoint rows did reach every midpoint
    e = a[6].float().numpy() / (E4M3[np.repeat(os_[6], 16)] * og[6])
    for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
        assert (np.abs(e) == m).any(), m


def oracle_y_w4a4(d: dict, tokens, ids, weights, *, want_h=False):
    """y_ref of the oracle's W4A4 experts for the listed tokens with the given
    routing (host arrays [n, 8]); with want_h also h [n, 8, I] before its
    BF16 rounding."""
    x = host_act(d["x"])[np.asarray(tokens)]
    n, K = ids.shape
    o = np.zeros((n, K, x.shape[1]))
    hs = None
    for e in np.unique(ids):
        rows, ks = np.nonzero(ids == e)
        mats, kw = host_expert(d, int(e))
        r = oracle.expert_ffn_w4a4(x[rows], *mats, **kw, want_h=want_h)
        if want_h:
            r, h = r
            if hs is None:
                hs = np.zeros((n, K, h.shape[1]))
            hs[rows, ks] = h
        o[rows, ks] = r
    y = oracle.combine(weights, o)
    return (y, hs) if want_h else y


def _layer(T, H, I, x_dtype, seed):
    wl = inputs.workload("nvfp4", T=T, H=H, I=I, x_dtype=x_dtype, seed=seed)
    dg = inputs.generate(wl, DEV)
    return dg, dict(dg, activations="nvfp4")


@pytest.mark.parametrize("T,H,I,x_dtype,hot", [(64, 512, 256, "bf16", (3, 200)), (200, 256, 512, "f32", None),
                                               (1, 256, 256, "bf16", None), (300, 1024, 256, "bf16", (7,))])
def test_w4a4_experts_against_the_oracle(T, H, I, x_dtype, hot):
    """Every token's output on a seeded routing against the oracle's W4A4
    experts to 3e-2 (as W4A16; the GPU's FP32 sums can flip a BF16 rounding
    of h and, rarely, one of its E2M1 codes), and far from the W4A16 output
    (the activations really are quantised)."""
    dg, wa4 = _layer(T, H, I, x_dtype, seed=70 + T)
    ids, w = seeded_routing(T, seed=T + 11, hot=hot)
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh, "nvfp4_a4")
    y = torch.empty((T, H), dtype=dg["x"].dtype, device=DEV)
    moe.beam_moe_experts(sh, dg["x"], wa4, ids.to(DEV), w.to(DEV), y, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, (code, where)
    yg = y.cpu().double().numpy()
    wts = w.numpy().astype(np.float64)
    y_ref = oracle_y_w4a4(dg, np.arange(T), ids.numpy(), wts)
    assert rel_err(yg, y_ref) <= Y_TOL["nvfp4"]
    if T >= 64:
        y16 = oracle_y(dg, np.arange(T), ids.numpy(), wts)
        assert rel_err(yg, y16) > 5e-2


def test_w4a4_intermediates_exact():
    """A whole forward stage by stage (router included): the gathered x rows
    the gate/up GEMM reads are the oracle quantiser's values of x bit for bit
    (row global scales beside them); h before its quantisation matches the
    oracle's W4A4 h to BF16 rounding; the rows the down GEMM reads are the
    oracle quantiser's values of the GPU's own BF16 h bit for bit; the output
    matches the down projection of those rows (oracle decoders, float64
    matmul) to BF16 rounding and the oracle's W4A4 layer to 3e-2."""
    T, H, I = 96, 512, 256
    dg, wa4 = _layer(T, H, I, "bf16", seed=501)
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh, "nvfp4_a4")
    lay = moe.workspace_layout(sh, "nvfp4_a4")
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((T, 8), dtype=torch.float32, device=DEV)
    call = moe.ForwardCall(sh, dg["x"], dg["router_w"], None, wa4, y, ids, w, ws)
    R = T * 8

    def region(off, count, dtype):
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).clone().cpu()

    for i in range(3):  # route, dispatch, gather
        call.stage(i)
    torch.cuda.synchronize()
    pos = region(lay["pos"], R, torch.int32).numpy().reshape(T, 8)
    xp = region(lay["xp"], R * H, torch.float16).numpy().reshape(R, H)
    xs = region(lay["xs"], R, torch.float32).numpy()
    oc, os_, og = oracle.quantize_nvfp4_rows(dg["x"].float().cpu().numpy())  # BF16 -> FP32 exact
    want = _values(oc, os_)
    for k in range(8):
        np.testing.assert_array_equal(xp[pos[:, k]].view(np.uint16), want)
        np.testing.assert_array_equal(xs[pos[:, k]], og)

    call.stage(3)  # gate/up: h in BF16
    torch.cuda.synchronize()
    h_bf16 = region(lay["h"], R * I, torch.bfloat16).float().numpy().reshape(R, I)
    call.stage(4)  # down: h quantised in place, then the GEMM
    call.stage(5)
    torch.cuda.synchronize()
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, (code, where)
    hq = region(lay["h"], R * I, torch.float16).numpy().reshape(R, I)
    hs = region(lay["hs"], R, torch.float32).numpy()
    hc, hsc, hg = oracle.quantize_nvfp4_rows(h_bf16)
    np.testing.assert_array_equal(hq.view(np.uint16), _values(hc, hsc))
    np.testing.assert_array_equal(hs, hg)

    ids_h, w_h = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    yg = y.cpu().double().numpy()
    y_ref, h_ref = oracle_y_w4a4(dg, np.arange(T), ids_h, w_h, want_h=True)
    # h of each route against the oracle's (before rounding): BF16 rounding
    # of values computed from the same quantised x
    h_gpu = h_bf16[pos.reshape(-1)].reshape(T, 8, I)
    scale = np.abs(h_ref).max(axis=2, keepdims=True)
    assert (np.abs(h_gpu - h_ref) <= 2.0 ** -7 * scale + 1e-30).all()
    # down GEMM over the GPU's quantised h rows: y = sum_k w_k Wd_e (hq g)
    o = np.zeros((T, 8, H))
    for e in np.unique(ids_h):
        mats, kw = host_expert(dg, int(e))
        packed, sd, gd = mats[2], kw["scales"][2], kw["global_scales"][2]
        codes = np.stack([packed & 0xF, packed >> 4], axis=2).reshape(H, I)
        wd = E2M1[codes] * E4M3[np.repeat(sd, 16, axis=1)] * gd
        rows, ks = np.nonzero(ids_h == e)
        r = pos[rows, ks]
        o[rows, ks] = (hq[r].astype(np.float64) * hs[r, None].astype(np.float64)) @ wd.T
    y_down = oracle.combine(w_h, o)
    assert rel_err(yg, y_down) <= 1e-2
    assert rel_err(yg, y_ref) <= Y_TOL["nvfp4"]


@pytest.mark.parametrize("T,H,I,pack", [(48, 512, 512, False), (300, 256, 512, True)])
def test_w4a4_dense_mlp(T, H, I, pack):
    """The dense SwiGLU MLP with W4A4 (one expert holding every row), both
    weight layouts: every row against the oracle's W4A4 expert."""
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype="nvfp4", seed=900 + T, E=1)
    dg = inputs.generate(wl, DEV)
    names = ("gate", "up", "down", "gate_sf", "up_sf", "down_sf", "gate_gs", "up_gs", "down_gs")
    wa4 = dict({k: dg[k] for k in names}, activations="nvfp4")
    mlp = moe.DenseMLP(wa4, max_tokens=T, pack=pack)
    y = mlp(dg["x"])
    code, where = moe.beam_moe_read_device_status(mlp.workspace)
    assert code == 0, (code, where)
    mats, kw = host_expert(dg, 0)
    y_ref = oracle.expert_ffn_w4a4(host_act(dg["x"]), *mats, **kw)
    assert rel_err(y.cpu().double().numpy(), y_ref) <= Y_TOL["nvfp4"]


def test_w4a4_full_size():
    """The W4A4 layer at the benchmark's size (nvfp4_a4: T=4096, the nvfp4
    layer's inputs, packed weights as the benchmark runs them): outputs of the
    tokens covering every touched expert and every chunk of the three most
    loaded experts against the oracle's W4A4 experts with the GPU's routing
    (the router, which does not see the expert format, is checked against the
    oracle on these same inputs by the nvfp4 full-size test)."""
    wl = inputs.workload("nvfp4_a4")
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    packed = dict(moe.pack_weights(sh, dg), activations="nvfp4")
    ws = moe.alloc_workspace(sh, "nvfp4_a4")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
    moe.beam_moe_forward(sh, dg["x"], dg["router_w"], None, packed, y, ids, w, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, (code, where)
    ids_h, w_h = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    tokens = full_size_tokens(ids_h, chunk_rows(wl.T, "nvfp4"))
    y_ref = oracle_y_w4a4(dg, tokens, ids_h[tokens], w_h[tokens])
    assert rel_err(y.cpu().double().numpy()[tokens], y_ref) <= Y_TOL["nvfp4"]
    print(f"w4a4 full size: {len(tokens)} outputs compared")
