"""GPU parity of the dense SwiGLU MLP (the first layers of the model, run by
the block's grouped GEMMs as one expert that takes every row) against the
oracle's expert_ffn / expert_ffn_fp8 on the same seeded inputs; outputs within
the block's tolerances (parity_helpers)."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routing_03_b300 as moe
import oracle
from group_limited_routing_03_b300 import inputs
from parity_helpers import Y_TOL, host_act, host_expert, rel_err

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


def _dense_inputs(T, H, I, w_dtype, seed, device):
    wl = inputs.workload("tiny", T=T, H=H, I=I, x_dtype="bf16", w_dtype=w_dtype, seed=seed, E=1)
    d = inputs.generate(wl, device)
    if w_dtype == "f32":  # BF16 copies on the GPU, FP32 originals for the oracle
        d = dict(d, **{k + "_f32": d[k] for k in ("gate", "up", "down")})
        d.update({k: d[k].to(torch.bfloat16).contiguous() for k in ("gate", "up", "down")})
    return wl, d


def _oracle(d, rows):
    x = host_act(d["x"])[rows]
    if "gate_f32" in d:
        return oracle.expert_ffn(x, *(d[k + "_f32"][0].cpu().numpy() for k in ("gate", "up", "down")))
    mats, kw = host_expert(d, 0)
    if "fp8_rs" in kw:
        return oracle.expert_ffn_fp8(x, *mats, *kw["fp8_rs"])
    return oracle.expert_ffn(x, *mats, **kw)


def _weights(d):
    return {k: v for k, v in d.items() if k in ("gate", "up", "down", "gate_sf", "up_sf", "down_sf", "gate_gs",
                                                 "up_gs", "down_gs", "gate_rs", "up_rs", "down_rs")}


# one CTA per unit and CTA pairs (T >= 256, H % 512, I % 256), both layouts,
# FP8 with I > H (the dense workspace keeps h's codes apart), NVFP4, T = 1;
# K split across CTAs (few units: T <= 128 with enough k-blocks): 64 x 512 x
# 1024 (gate/up 2 parts, down 4), 100 x 768 x 512 (3 parts over a ragged chunk,
# down 2), FP8 48 x 1024 x 2048 (2 / 4 parts)
@pytest.mark.parametrize("T,H,I,w_dtype,pack", [
    (1, 256, 128, "f32", False), (33, 256, 384, "f32", True), (300, 512, 256, "f32", False),
    (600, 1024, 768, "f32", True), (300, 512, 1024, "fp8", False), (200, 256, 512, "fp8", True),
    (100, 512, 256, "nvfp4", False), (257, 512, 512, "nvfp4", True),
    (64, 512, 1024, "f32", False), (100, 768, 512, "f32", True), (48, 1024, 2048, "fp8", False)])
def test_dense_all_rows(T, H, I, w_dtype, pack):
    wl, d = _dense_inputs(T, H, I, w_dtype, T + I, "cpu")
    dg = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    mlp = moe.DenseMLP(_weights(dg), max_tokens=T, pack=pack)
    y = mlp(dg["x"])
    code, where = moe.beam_moe_read_device_status(mlp.workspace)
    assert code == 0, f"device status {code} where {where}"
    y_ref = _oracle(dg, np.arange(T))
    err = rel_err(y.cpu().double().numpy(), y_ref)
    tol = Y_TOL["nvfp4" if w_dtype == "nvfp4" else "bf16"]
    assert err <= tol, err


@pytest.mark.parametrize("name,n_sample", [("dense_dec", 6), ("dense", 4)])
def test_dense_full_size(name, n_sample):
    wl = inputs.workload(name)
    dg = inputs.generate(wl, DEV)
    mlp = moe.DenseMLP(_weights(dg), max_tokens=wl.T, pack=True)
    y = mlp(dg["x"])
    code, where = moe.beam_moe_read_device_status(mlp.workspace)
    assert code == 0, f"device status {code} where {where}"
    rng = np.random.default_rng(wl.seed)
    rows = np.unique(np.concatenate([[0, wl.T - 1], rng.integers(0, wl.T, n_sample)]))
    y_ref = _oracle(dg, rows)
    err = rel_err(y[torch.as_tensor(rows, device=DEV)].cpu().double().numpy(), y_ref)
    print(f"{name}: {len(rows)} rows, rel err {err:.3e}")
    assert err <= Y_TOL["bf16"], err
    del dg, y, mlp
    gc.collect()
    torch.cuda.empty_cache()


def test_dense_kernel_count():
    """K split after each GEMM at decode size (a finishing kernel each), none
    at prefill size (CTA pairs); FP8 adds the two row quantisations."""
    assert moe.dense_kernel_count(moe.dense_shape(64, 5120, 20480), "bf16") == 5
    assert moe.dense_kernel_count(moe.dense_shape(64, 5120, 20480), "fp8") == 7
    assert moe.dense_kernel_count(moe.dense_shape(8192, 5120, 20480), "bf16") == 3
    assert moe.dense_kernel_count(moe.dense_shape(64, 5120, 20480), "nvfp4") == 5  # + x and h to FP16 rows


def test_dense_fp8_with_fp32_x():
    """FP8 weights take FP32 x too (its first step re-encodes x as E4M3)."""
    wl = inputs.workload("tiny", T=70, H=512, I=768, x_dtype="f32", w_dtype="fp8", seed=31, E=1)
    dg = inputs.generate(wl, DEV)
    mlp = moe.DenseMLP(_weights(dg), max_tokens=wl.T)
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    moe.beam_dense_mlp_forward(moe.dense_shape(wl.T, wl.H, wl.I), dg["x"], mlp.weights, y, mlp.workspace)
    code, where = moe.beam_moe_read_device_status(mlp.workspace)
    assert code == 0, f"device status {code} where {where}"
    err = rel_err(y.cpu().double().numpy(), _oracle(dg, np.arange(wl.T)))
    assert err <= Y_TOL["fp8"], err
