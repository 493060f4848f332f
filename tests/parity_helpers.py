"""Helpers shared by the GPU parity tests: host copies of device inputs for
the oracle, oracle evaluation of sampled tokens, and the comparison rules.

Comparison rules (the same everywhere):
  * routing: ids must match the oracle exactly (as sets, and in order where
    the oracle's adjacent selection-score gaps exceed 1e-5) for every token
    whose oracle margin -- min(4th-5th group score gap, 8th-9th expert score
    gap) -- exceeds 1e-5; tokens at or below that margin are near-ties, which
    FP32 rounding may legitimately flip, and are counted, not compared;
  * weights: |w - w_ref| <= 1e-5 * |w_ref| + 1e-6 for the compared tokens;
  * outputs: max|y - y_ref| / max|y_ref| <= 1e-2 (BF16 and FP8 experts) or
    3e-2 (NVFP4 experts) over the compared tokens.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

MARGIN = 1e-5
Y_TOL = {"bf16": 1e-2, "f32": 1e-2, "nvfp4": 3e-2, "fp8": 1e-2}


def host_act(t: torch.Tensor) -> np.ndarray:
    """Exact host copy of activations: float32 array or uint16 BF16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def host_expert(d: dict, e: int):
    """Host copies of expert e's weights in a form oracle.expert_ffn takes
    (for FP8: the E4M3 codes as bytes and the row scales, oracle.expert_ffn_fp8)."""
    if d["gate"].dtype == torch.float8_e4m3fn:
        mats = [d[n][e].cpu().view(torch.uint8).numpy() for n in ("gate", "up", "down")]
        return mats, dict(fp8_rs=[d[n + "_rs"][e].cpu().numpy() for n in ("gate", "up", "down")])
    if d["gate"].dtype == torch.uint8:
        mats = [d[n][e].cpu().numpy() for n in ("gate", "up", "down")]
        scales = [d[n + "_sf"][e].cpu().numpy() for n in ("gate", "up", "down")]
        gs = [float(d[n + "_gs"][e]) for n in ("gate", "up", "down")]
        return mats, dict(scales=scales, global_scales=gs)
    return [host_act(d[n][e]) for n in ("gate", "up", "down")], {}


def oracle_route(d: dict):
    x = host_act(d["x"])
    b = None if d.get("bias") is None else d["bias"].cpu().numpy()
    return oracle.route(x, d["router_w"].cpu().numpy(), b, want_scores=True)


def oracle_y(d: dict, tokens, ids, weights, *, oracle_weights=None):
    """y_ref for the listed tokens with the given routing (ids / weights are
    host arrays [n, 8] for those tokens).  ``oracle_weights`` may override the
    expert weights with host arrays (e.g. the FP32 originals)."""
    x = host_act(d["x"])[np.asarray(tokens)]
    n, K = ids.shape
    H = x.shape[1]
    o = np.zeros((n, K, H))
    for e in np.unique(ids):
        rows, ks = np.nonzero(ids == e)
        if oracle_weights is not None:
            mats, kw = [oracle_weights[k][e] for k in ("gate", "up", "down")], {}
        else:
            mats, kw = host_expert(d, int(e))
        if "fp8_rs" in kw:
            o[rows, ks] = oracle.expert_ffn_fp8(x[rows], *mats, *kw["fp8_rs"])
        else:
            o[rows, ks] = oracle.expert_ffn(x[rows], *mats, **kw)
    return oracle.combine(weights, o)


def compare_routing(ids_gpu: np.ndarray, w_gpu: np.ndarray, ref: dict, bias=None):
    """Asserts the routing rules; returns the boolean mask of compared tokens."""
    safe = ref["margin"] > MARGIN
    assert safe.mean() > 0.5, f"too few tokens above the margin: {safe.mean():.3f}"
    ri, rw = ref["ids"], ref["weights"]
    bad = np.nonzero(safe & (np.sort(ids_gpu, 1) != np.sort(ri, 1)).any(1))[0]
    assert bad.size == 0, f"{bad.size} tokens with margin > {MARGIN} route differently, first {bad[:5]}"
    sel = ref["scores"] + (0.0 if bias is None else bias.astype(np.float64)[None, :])
    chosen = np.take_along_axis(sel, ri.astype(np.int64), 1)
    ordered = safe & (np.diff(chosen, axis=1) < -MARGIN).all(1)
    assert (ids_gpu[ordered] == ri[ordered]).all(), "order of chosen experts differs"
    # weights, aligned by expert id
    og = np.argsort(ids_gpu, 1)
    orf = np.argsort(ri, 1)
    wg = np.take_along_axis(w_gpu.astype(np.float64), og, 1)[safe]
    wr = np.take_along_axis(rw, orf, 1)[safe]
    np.testing.assert_allclose(wg, wr, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(w_gpu.astype(np.float64)[safe].sum(1), 2.5, rtol=2e-6)
    return safe


def rel_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> float:
    return float(np.abs(y_gpu - y_ref).max() / np.abs(y_ref).max())


def seeded_routing(T: int, seed: int, *, E=256, K=8, hot=None):
    """A routing drawn independently of the router: 8 distinct experts per
    token (uniform, or always including the experts in ``hot``), positive
    weights summing to 2.5.  Returns int32 ids [T,8], float32 w [T,8]."""
    g = torch.Generator().manual_seed(seed)
    keys = torch.rand((T, E), generator=g)
    if hot is not None:
        keys[:, list(hot)] += 10.0
    ids = torch.argsort(keys, dim=1, descending=True)[:, :K].to(torch.int32)
    w = torch.rand((T, K), generator=g) + 0.1
    w = (w / w.sum(1, keepdim=True) * 2.5).to(torch.float32)
    return ids.contiguous(), w.contiguous()
