"""Helpers shared by the GPU parity tests: host copies of device inputs for
the oracle, oracle evaluation of sampled tokens, the comparison rules and the
choice of tokens compared at full size.

Comparison rules (the same everywhere):
  * routing, tokens whose oracle margin -- min(4th-5th group score gap,
    8th-9th expert score gap) -- exceeds 1e-5: ids equal to the oracle's (as
    sets, and in order where the oracle's adjacent selection-score gaps exceed
    1e-5);
  * routing, the other tokens (near-ties, which FP32 rounding may flip): the
    GPU's ids must still be a valid answer within 1e-5 of the oracle's
    scores -- 8 distinct ids from at most 4 groups, each of those groups
    within 1e-5 of the oracle's 4th-best group score, and some completion of
    them to 4 such groups in which no unchosen expert beats the weakest chosen
    one by more than 1e-5, listed best first within 1e-5.  They are counted
    (near_ties) and reported per workload;
  * weights: for every token, w equals s[id] / sum_k s[id_k] * 2.5 with the
    oracle's scores s at the GPU's ids, |w - w_ref| <= 1e-5 * |w_ref| + 1e-6,
    and sum_k w = 2.5 to 2e-6;
  * outputs: max|y - y_ref| / max|y_ref| <= 1e-2 (BF16 and FP8 experts) or
    3e-2 (NVFP4 experts) over the compared tokens, y_ref being the oracle's
    block output for the routing the GPU chose (the oracle's own where the
    margin is clear, the GPU's ids with oracle weights at near-ties).
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass

import numpy as np
import torch

import oracle

MARGIN = 1e-5
Y_TOL = {"bf16": 1e-2, "f32": 1e-2, "nvfp4": 3e-2, "fp8": 1e-2}
N_GROUPS, GROUP_SIZE, GROUPS_KEPT, TOP_K, SCALE = 8, 32, 4, 8, 2.5

# (workload, tokens, near-tie tokens, compared outputs) of this session,
# printed in the terminal summary by conftest.py
NEAR_TIES: list = []


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


def group_scores(sel: np.ndarray) -> np.ndarray:
    """Sum of the two largest selection scores of each group of 32 contiguous
    experts: sel [n, 256] -> [n, 8]."""
    g = np.sort(sel.reshape(sel.shape[0], N_GROUPS, GROUP_SIZE), axis=2)
    return g[:, :, -1] + g[:, :, -2]


def valid_selection(ids, sel, tol=MARGIN):
    """None if the 8 ids are a valid group-limited top-8 of the selection
    scores `sel` [256] within `tol`, else the rule they break."""
    ids = np.asarray(ids, dtype=np.int64)
    if ids.shape != (TOP_K,) or ((ids < 0) | (ids >= N_GROUPS * GROUP_SIZE)).any():
        return "ids out of range"
    if np.unique(ids).size != TOP_K:
        return "repeated id"
    groups = set(int(j) for j in ids // GROUP_SIZE)
    if len(groups) > GROUPS_KEPT:
        return f"ids from {len(groups)} groups"
    g = group_scores(sel[None, :])[0]
    g4 = np.sort(g)[-GROUPS_KEPT]
    if any(g[j] < g4 - tol for j in groups):
        return "a chosen group is not among the best 4 groups"
    chosen = sel[ids]
    if (np.diff(chosen) > tol).any():
        return "ids not listed best first"
    weakest = chosen.min()
    others = [j for j in range(N_GROUPS) if j not in groups and g[j] >= g4 - tol]
    need = GROUPS_KEPT - len(groups)
    if need > len(others):
        return "fewer than 4 admissible groups"
    mask = np.zeros(sel.shape[0], bool)
    mask[ids] = True
    for extra in itertools.combinations(others, need):
        kept = sorted(groups) + list(extra)
        cand = np.concatenate([np.arange(j * GROUP_SIZE, (j + 1) * GROUP_SIZE) for j in kept])
        cand = cand[~mask[cand]]
        if cand.size == 0 or sel[cand].max() <= weakest + tol:
            return None
    return "an unchosen expert of the kept groups beats a chosen one"


@dataclass
class Routing:
    """Outcome of compare_routing: `safe` marks the tokens above the margin;
    `ids` / `weights` [T, 8] are the routing y_ref is evaluated with (the
    oracle's ids and weights where safe, else the GPU's ids with weights from
    the oracle's scores); `near_ties` counts the other tokens."""
    safe: np.ndarray
    ids: np.ndarray
    weights: np.ndarray
    near_ties: int


def compare_routing(ids_gpu: np.ndarray, w_gpu: np.ndarray, ref: dict, bias=None) -> Routing:
    """Asserts the routing rules (module docstring) on every token."""
    safe = ref["margin"] > MARGIN
    assert safe.mean() > 0.5, f"too few tokens above the margin: {safe.mean():.3f}"
    ri, rw = ref["ids"], ref["weights"]
    bad = np.nonzero(safe & (np.sort(ids_gpu, 1) != np.sort(ri, 1)).any(1))[0]
    assert bad.size == 0, f"{bad.size} tokens with margin > {MARGIN} route differently, first {bad[:5]}"
    scores = ref["scores"]
    sel = scores + (0.0 if bias is None else np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :])
    chosen = np.take_along_axis(sel, ri.astype(np.int64), 1)
    ordered = safe & (np.diff(chosen, axis=1) < -MARGIN).all(1)
    assert (ids_gpu[ordered] == ri[ordered]).all(), "order of chosen experts differs"
    near = np.nonzero(~safe)[0]
    for t in near:
        why = valid_selection(ids_gpu[t], sel[t])
        assert why is None, f"near-tie token {t}: GPU ids {ids_gpu[t].tolist()} invalid: {why}"
    # weights from the oracle's scores at the GPU's ids (the oracle's own
    # weights where the ids agree), for every token
    ids_y = np.where(safe[:, None], ri, ids_gpu).astype(np.int32)
    s_at = np.take_along_axis(scores, np.clip(ids_y, 0, scores.shape[1] - 1).astype(np.int64), 1)
    w_y = np.where(safe[:, None], rw, s_at / s_at.sum(1, keepdims=True) * SCALE)
    og = np.argsort(ids_gpu, 1)
    oy = np.argsort(ids_y, 1)
    wg = np.take_along_axis(w_gpu.astype(np.float64), og, 1)
    wr = np.take_along_axis(w_y, oy, 1)
    np.testing.assert_allclose(wg, wr, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(w_gpu.astype(np.float64).sum(1), SCALE, rtol=2e-6)
    return Routing(safe=safe, ids=ids_y, weights=w_y, near_ties=int(near.size))


def record_near_ties(label: str, T: int, r: Routing, compared: int):
    NEAR_TIES.append(dict(workload=label, tokens=int(T), near_ties=r.near_ties, outputs_compared=int(compared)))


def rel_err(y_gpu: np.ndarray, y_ref: np.ndarray) -> float:
    return float(np.abs(y_gpu - y_ref).max() / np.abs(y_ref).max())


def chunk_rows(T: int, w_dtype: str) -> int:
    """Routes per GEMM unit at most (the library's rule): a multiple of 32
    covering T, capped at 256 (NVFP4 weights: 160; 16 up to T = 256)."""
    if w_dtype == "nvfp4" and T <= 256:
        return 16
    cap = 160 if w_dtype == "nvfp4" else 256
    return min(cap, (T + 31) // 32 * 32)


def full_size_tokens(ids: np.ndarray, nmax: int, *, hot: int = 3, extra=(), all_below: int = 256) -> np.ndarray:
    """Tokens whose outputs are compared on a full-size workload, for the
    routing `ids` [T, 8] the GPU ran:
      * every token when T <= all_below;
      * else (1) tokens covering every unit of work of the `hot` most-loaded
        experts -- the library cuts an expert's n routes (ascending token
        order) into ceil(n / nmax) chunks whose sizes differ by at most one,
        each chunk a separate unit -- chosen greedily (a token routed to
        several hot experts covers one chunk of each); (2) greedily, tokens
        until every touched expert has at least one compared token; (3)
        tokens 0 and T-1 and `extra`."""
    T = ids.shape[0]
    if T <= all_below:
        return np.arange(T)
    counts = np.bincount(ids.reshape(-1), minlength=256)
    pick = {0, T - 1, *(int(t) for t in extra)}
    # (1) chunks of the hot experts: chunk index of each token, -1 if not routed there
    hot_e = np.argsort(-counts, kind="stable")[:hot]
    cidx = np.full((hot, T), -1, np.int64)
    covered = []
    for h, e in enumerate(hot_e):
        toks = np.nonzero((ids == e).any(1))[0]
        n = toks.size
        nch = max(1, -(-n // nmax))
        base, rem = divmod(n, nch)
        starts = np.array([c * base + min(c, rem) for c in range(nch)])
        cidx[h, toks] = np.searchsorted(starts, np.arange(n), side="right") - 1
        covered.append(np.zeros(nch, bool))
    for t in pick:
        for h in range(hot):
            if cidx[h, t] >= 0:
                covered[h][cidx[h, t]] = True
    while not all(c.all() for c in covered):
        gain = np.zeros(T, np.int64)
        for h in range(hot):
            ok = cidx[h] >= 0
            gain[ok] += ~covered[h][cidx[h, ok]]
        t = int(np.argmax(gain))
        pick.add(t)
        for h in range(hot):
            if cidx[h, t] >= 0:
                covered[h][cidx[h, t]] = True
    # (2) every touched expert
    uncovered = counts > 0
    for t in pick:
        uncovered[ids[t]] = False
    while uncovered.any():
        gain = uncovered[ids].sum(1)
        t = int(np.argmax(gain))
        pick.add(t)
        uncovered[ids[t]] = False
    return np.array(sorted(pick))


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
