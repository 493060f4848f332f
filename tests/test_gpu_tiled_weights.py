"""GPU: the tiled weight layout.  Packing is a pure regrouping of 16-byte
pieces (checked against torch reshape / permute of the row-major arrays), and
a forward with packed weights gives the same bits as with row-major weights."""
import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
from group_limited_routing_03_b300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from group_limited_routing_03_b300 import _build

    _build.build()
    moe.load()


def _tiled_reference(t: torch.Tensor, tile_row_bytes: int) -> torch.Tensor:
    """[E, N, ...] array as bytes [E*N, B], tiles of 128 rows x tile_row_bytes
    laid out tile after tile (rows of a tile contiguous)."""
    b = t.contiguous().view(torch.uint8).reshape(t.shape[0] * t.shape[1], -1)
    R, B = b.shape
    return b.reshape(R // 128, 128, B // tile_row_bytes, tile_row_bytes).permute(0, 2, 1, 3).contiguous().reshape(-1)


@pytest.mark.parametrize("w_dtype", ["bf16", "nvfp4"])
def test_pack_is_the_tile_regrouping(w_dtype):
    wl = inputs.workload("nvfp4" if w_dtype == "nvfp4" else "decode", T=64, H=512, I=256, seed=5)
    d = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    packed = moe.pack_weights(sh, d)
    torch.cuda.synchronize()
    wb = 32 if w_dtype == "nvfp4" else 128
    for name in ("gate", "up", "down"):
        got = packed[name].view(torch.uint8).reshape(-1)
        assert torch.equal(got, _tiled_reference(d[name], wb)), name
    if w_dtype == "nvfp4":
        for name in ("gate_sf", "up_sf", "down_sf"):
            assert torch.equal(packed[name].view(torch.uint8).reshape(-1), _tiled_reference(d[name], 16)), name
        for name in ("gate_gs", "up_gs", "down_gs"):
            assert packed[name].data_ptr() == d[name].data_ptr()
    assert packed["layout"] == "tiled"


@pytest.mark.parametrize("name,T,H,I", [("decode", 64, 512, 256), ("prefill", 600, 512, 512),
                                        ("nvfp4", 64, 512, 256), ("nvfp4", 700, 512, 256)])
def test_forward_same_bits_with_tiled_weights(name, T, H, I):
    """One CTA per unit (decode-sized), CTA pairs (600 tokens, H % 512 == 0)
    and both NVFP4 GEMMs, on row-major and on packed weights."""
    wl = inputs.workload(name, T=T, H=H, I=I, seed=17)
    d = inputs.generate(wl, DEV)
    sh = moe.shape(wl.T, wl.H, wl.I)
    packed = moe.pack_weights(sh, d)
    outs = []
    for wts in (d, packed):
        ws = moe.alloc_workspace(sh, "nvfp4" if wl.w_dtype == "nvfp4" else "bf16")
        y = torch.empty((T, H), dtype=d["x"].dtype, device=DEV)
        ids = torch.empty((T, 8), dtype=torch.int32, device=DEV)
        w = torch.empty((T, 8), dtype=torch.float32, device=DEV)
        moe.beam_moe_forward(sh, d["x"], d["router_w"], d.get("bias"), wts, y, ids, w, ws)
        code, where = moe.beam_moe_read_device_status(ws)
        assert code == 0, (code, where)
        outs.append((y, ids, w))
    (y0, i0, w0), (y1, i1, w1) = outs
    assert torch.equal(i0, i1) and torch.equal(w0, w1)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert torch.isfinite(y0.float()).all() and y0.float().abs().max() > 0
