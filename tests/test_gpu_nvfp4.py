"""NVFP4 expert weights on FP16 tensor cores: the converters' expansion of
every E2M1 x E4M3 product, and the exactness of the FP16 activations (a
power of two per row) on rows far from N(0, 1), both against the oracle."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import Y_TOL, oracle_y, seeded_routing

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


def test_expansion_of_every_code_pair_and_scale():
    """All 256 code bytes (two E2M1 elements each) under each of the 256 E4M3
    scales, expanded by the converters' device code, equal e2m1 * e4m3
    exactly (NaN for the two E4M3 NaN codes), the low nibble first."""
    codes = np.tile(np.arange(256, dtype=np.uint8), 256)            # 32 blocks of 8 bytes per scale
    scales = np.repeat(np.arange(256, dtype=np.uint8), 32)          # 8192 blocks
    out = torch.empty(16 * scales.size, dtype=torch.float16, device=DEV)
    moe.beam_debug_nvfp4_expand(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV), out)
    got = out.double().cpu().numpy().reshape(-1, 2)                 # (low nibble, high nibble) per byte
    e2m1 = np.array([oracle.decode_e2m1(c) for c in range(16)])
    e4m3 = np.array([oracle.decode_e4m3(c) for c in range(256)])
    s = e4m3[np.repeat(scales, 8)]
    want = np.stack([e2m1[codes & 0xF] * s, e2m1[codes >> 4] * s], axis=1)
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], want[~nan])
    # signs of zero products follow the code's sign bit times the scale's
    zero = (want == 0) & ~nan
    assert (np.signbit(got[zero]) == np.signbit(want[zero])).all()


def _rows_far_from_unit_scale(T, H, seed):
    """BF16 token rows: N(0,1); N(0,1) times 2^-30 (tiny values only: their
    h ~ 2^-65 stays a normal FP32 / BF16 number); times 2^40 (large values
    only, h ~ 2^80); N(0,1) with every other element times 2^-45 (a
    row spanning ~50 binades, more than FP16 holds after the row's power-of-two
    scale); and an all-zero row."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g)
    x[1::5] *= 2.0 ** -30
    x[2::5] *= 2.0 ** 40
    x[3::5, ::2] *= 2.0 ** -45
    x[4::5] = 0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,H,I", [(40, 256, 256), (300, 512, 256)])
def test_fp16_activation_rows_against_the_oracle(T, H, I):
    """Experts on a seeded routing with rows far from unit scale: each token's
    output against the oracle to 3e-2 of that token's own largest output (so
    the tiny rows are checked on their own scale, not hidden by the large
    ones); the all-zero rows give exactly zero."""
    wl = inputs.workload("nvfp4", T=T, H=H, I=I, seed=55 + T)
    dg = inputs.generate(wl, DEV)
    dg["x"] = _rows_far_from_unit_scale(T, H, seed=T).to(DEV)
    ids, w = seeded_routing(T, seed=T + 9, hot=(3, 200))
    sh = moe.shape(T, H, I)
    ws = moe.alloc_workspace(sh, "nvfp4")
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moe.beam_moe_experts(sh, dg["x"], dg, ids.to(DEV), w.to(DEV), y, ws)
    code, where = moe.beam_moe_read_device_status(ws)
    assert code == 0, (code, where)
    y_ref = oracle_y(dg, np.arange(T), ids.numpy(), w.numpy().astype(np.float64))
    yg = y.cpu().double().numpy()
    zero = np.arange(T) % 5 == 4
    assert (yg[zero] == 0).all()
    for t in np.nonzero(~zero)[0]:
        ref = np.abs(y_ref[t]).max()
        err = np.abs(yg[t] - y_ref[t]).max() / ref
        assert err <= Y_TOL["nvfp4"], (t, err, ref)


@pytest.mark.parametrize("T,H,I,hot", [(200, 512, 256, (3, 100)), (1, 256, 256, None), (96, 1024, 512, (7,)),
                                       (256, 256, 768, None)])
def test_tiled_weights_four_kblocks_per_stage(T, H, I, hot):
    """Few tokens (chunks of at most 32 routes) with packed weights: each
    pipeline stage carries four k-blocks (3-D boxes of consecutive tiles and
    of the chunk's activation rows).  Same bits as the row-major weights (one
    k-block per stage), and the oracle's output on a seeded routing whose hot
    experts take every token (several chunks of one expert)."""
    wl = inputs.workload("nvfp4", T=T, H=H, I=I, seed=300 + T)
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(T, H, I)
    packed = moe.pack_weights(sh, dg)
    ids, w = seeded_routing(T, seed=T + 3, hot=hot)
    ys = []
    for wts in (dg, packed):
        ws = moe.alloc_workspace(sh, "nvfp4")
        y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        moe.beam_moe_experts(sh, dg["x"], wts, ids.to(DEV), w.to(DEV), y, ws)
        code, where = moe.beam_moe_read_device_status(ws)
        assert code == 0, (code, where)
        ys.append(y)
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    y_ref = oracle_y(dg, np.arange(T), ids.numpy(), w.numpy().astype(np.float64))
    err = float(np.abs(ys[1].cpu().double().numpy() - y_ref).max() / np.abs(y_ref).max())
    assert err <= Y_TOL["nvfp4"], err


@pytest.mark.parametrize("name", ["nvfp4_dec", "nvfp4"])
def test_full_size_tiled_equals_rows(name):
    """The full-size NVFP4 layers as the benchmark runs them (packed weights)
    give the bits of the row-major weights, whose output the full-size parity
    test checks against the oracle."""
    wl = inputs.workload(name)
    torch.cuda.empty_cache()
    dg = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    packed = moe.pack_weights(sh, dg)
    outs = []
    for wts in (dg, packed):
        ws = moe.alloc_workspace(sh, "nvfp4")
        y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
        ids = torch.empty((wl.T, 8), dtype=torch.int32, device=DEV)
        w = torch.empty((wl.T, 8), dtype=torch.float32, device=DEV)
        moe.beam_moe_forward(sh, dg["x"], dg["router_w"], None, wts, y, ids, w, ws)
        code, where = moe.beam_moe_read_device_status(ws)
        assert code == 0, (code, where)
        outs.append((y, ids))
        del ws
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    del dg, packed, outs
    gc.collect()
    torch.cuda.empty_cache()
