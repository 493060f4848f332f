"""The seeded input generators: deterministic, and the storage encodings they
produce (NVFP4, FP8) decode back to values near the drawn ones.  No GPU."""
import numpy as np
import torch

from group_limited_routing_03_b300 import inputs


def test_generation_is_deterministic():
    wl = inputs.workload("tiny", T=16, H=256, I=128)
    a, b = inputs.generate(wl, "cpu"), inputs.generate(wl, "cpu")
    for k in ("x", "router_w", "gate", "up", "down"):
        assert torch.equal(a[k], b[k]), k
    s1, g1 = inputs.residual_inputs(wl, "cpu")
    s2, g2 = inputs.residual_inputs(wl, "cpu")
    assert torch.equal(s1, s2) and torch.equal(g1, g2)
    assert s1.shape == (16, 256) and g1.shape == (256,) and g1.dtype == torch.float32


def test_fp8_row_encoding_round_trip():
    g = torch.Generator().manual_seed(3)
    w = torch.randn((64, 256), generator=g) * 0.02
    w[5] = 0.0  # a zero row gets scale 1 and zero codes
    codes, scale = inputs.quantize_fp8_rows(w)
    assert codes.dtype == torch.float8_e4m3fn and scale.shape == (64,)
    assert scale[5] == 1.0 and torch.count_nonzero(codes[5].float()) == 0
    back = codes.float() * scale[:, None]
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 of each value, plus
    # the subnormal step 2^-9 * scale near zero
    err = (back - w).abs()
    bound = w.abs() * 2.0 ** -4 + scale[:, None] * 2.0 ** -10
    assert bool((err <= bound + 1e-12).all())
    # each row's largest magnitude maps to the largest code, 448
    amax_codes = codes.float().abs().amax(1)
    assert bool((amax_codes[torch.arange(64) != 5] == 448.0).all())


def test_nvfp4_encoding_round_trip():
    g = torch.Generator().manual_seed(4)
    w = torch.randn((32, 128), generator=g) * 0.02
    packed, sf, gs = inputs.quantize_nvfp4(w)
    assert packed.shape == (32, 64) and sf.shape == (32, 8)
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6])
    p = packed.numpy()
    codes = np.stack([p & 0xF, p >> 4], axis=-1).reshape(32, 128)
    scales = torch.from_numpy(sf.numpy()).view(torch.float8_e4m3fn).float().numpy()
    back = e2m1[codes] * np.repeat(scales, 16, axis=1) * gs
    # E2M1 steps are at most a third of a block's largest value
    blk_max = np.repeat(np.abs(w.numpy()).reshape(32, 8, 16).max(-1), 16, axis=1)
    assert np.all(np.abs(back - w.numpy()) <= blk_max / 3 + 1e-6)
