"""The GPU parity rules themselves (parity_helpers), on the CPU: the
validity check that near-tie tokens must pass accepts the oracle's own
choices and every tie-flip within the margin, and rejects planted mistakes;
the token choice for full-size comparisons covers every touched expert and
every token chunk of the most-loaded experts."""
import numpy as np
import pytest

import oracle
from parity_helpers import (MARGIN, Routing, chunk_rows, compare_routing, full_size_tokens, group_scores,
                            valid_selection)


def _random_router(T, H=64, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H)).astype(np.float32)
    wr = (rng.standard_normal((256, H)) / np.sqrt(H)).astype(np.float32)
    return x, wr


def test_oracle_choices_are_valid():
    x, wr = _random_router(200)
    r = oracle.route(x, wr, None, want_scores=True)
    for t in range(200):
        assert valid_selection(r["ids"][t], r["scores"][t]) is None


def test_oracle_choices_with_bias_are_valid():
    x, wr = _random_router(100, seed=1)
    b = np.random.default_rng(2).uniform(0, 3, 256).astype(np.float32)
    r = oracle.route(x, wr, b, want_scores=True)
    sel = r["scores"] + b.astype(np.float64)[None, :]
    for t in range(100):
        assert valid_selection(r["ids"][t], sel[t]) is None


def _sel_with_groups():
    """Scores with clear gaps: the first two experts of group j score
    0.9 - 0.1 j and 0.899 - 0.1 j, the other thirty 0.05 - 0.0001 i (i the
    index inside the group), so groups 0..3 are kept and the top-8 are
    experts 0, 1, 32, 33, 64, 65, 96, 97, listed best first."""
    sel = np.array([0.9 - 0.1 * (e // 32) - 0.001 * (e % 32) if e % 32 < 2 else 0.05 - 0.0001 * (e % 32)
                    for e in range(256)])
    ids = np.array([0, 1, 32, 33, 64, 65, 96, 97])
    return sel, ids


def test_planted_mistakes_are_rejected():
    sel, ids = _sel_with_groups()
    assert valid_selection(ids, sel) is None
    bad = ids.copy()
    bad[-1] = 2  # a weaker expert of a kept group in place of expert 97
    assert valid_selection(bad, sel) is not None
    bad = ids.copy()
    bad[-1] = 128  # an expert of the 5th group (five groups)
    assert "groups" in valid_selection(bad, sel)
    bad = ids.copy()
    bad[-2:] = [128, 129]  # both of group 3's places to group 4: not a best-4 group
    assert "best 4 groups" in valid_selection(bad, sel)
    bad = ids.copy()
    bad[-1] = 0
    assert valid_selection(bad, sel) == "repeated id"
    assert valid_selection(ids[::-1], sel) == "ids not listed best first"
    bad = ids.copy()
    bad[0] = 256
    assert valid_selection(bad, sel) == "ids out of range"


def test_flips_within_the_margin_are_accepted():
    sel, ids = _sel_with_groups()
    # the 8th and 9th expert scores 1e-6 apart: either may be chosen
    sel2 = sel.copy()
    sel2[2] = sel2[97] - 1e-6
    alt = ids.copy()
    alt[-1] = 2
    assert valid_selection(ids, sel2) is None and valid_selection(alt, sel2) is None
    # ... but not 1e-4 apart
    sel3 = sel.copy()
    sel3[2] = sel3[97] - 1e-4
    assert valid_selection(alt, sel3) is not None
    # the 4th and 5th group scores 1e-6 apart: group 4 may replace group 3
    sel4 = sel.copy()
    sel4[128:160] = sel[96:128] - 1e-6 / 2
    alt4 = ids.copy()
    alt4[-2:] = [128, 129]
    assert valid_selection(alt4, sel4) is None
    g = group_scores(sel4[None, :])[0]
    assert abs(g[3] - g[4]) <= MARGIN


def test_compare_routing_accepts_the_oracle_and_rejects_a_flip():
    x, wr = _random_router(300, seed=3)
    ref = oracle.route(x, wr, None, want_scores=True)
    r = compare_routing(ref["ids"].copy(), ref["weights"].astype(np.float32), ref)
    assert isinstance(r, Routing) and r.near_ties == int((ref["margin"] <= MARGIN).sum())
    np.testing.assert_array_equal(r.ids, ref["ids"])
    t = int(np.nonzero(ref["margin"] > 1e-3)[0][0])
    ids = ref["ids"].copy()
    ids[t, -1] = next(e for e in range(256) if e not in ids[t] and e // 32 in set(ids[t] // 32))
    with pytest.raises(AssertionError):
        compare_routing(ids, ref["weights"].astype(np.float32), ref)


def test_near_tie_outputs_use_the_gpu_ids_with_oracle_weights():
    """A near-tie token routed differently (a valid flip) is evaluated with
    the GPU's ids and weights s[id] / sum s * 2.5 from the oracle's scores."""
    x, wr = _random_router(400, seed=4)
    ref = oracle.route(x, wr, None, want_scores=True)
    me = ref["margin_expert"]
    t = int(np.argmin(me))
    ids = ref["ids"].copy()
    sel = ref["scores"][t]
    kept = sorted(set(ids[t] // 32))
    cand = [e for j in kept for e in range(32 * j, 32 * j + 32) if e not in ids[t]]
    ninth = max(cand, key=lambda e: sel[e])
    flipped = ids[t].copy()
    flipped[-1] = ninth
    # make the flip a near-tie in the reference data (the test plants it in the oracle's output)
    ref = dict(ref)
    ref["margin"] = ref["margin"].copy()
    ref["margin"][t] = 0.0
    ref["scores"] = ref["scores"].copy()
    ref["scores"][t, ninth] = ref["scores"][t, ids[t, -1]] - 1e-7
    ids[t] = flipped
    s = ref["scores"][t, flipped]
    w = ref["weights"].astype(np.float32)
    w[t] = (s / s.sum() * 2.5).astype(np.float32)
    r = compare_routing(ids, w, ref)
    assert r.near_ties >= 1 and (r.ids[t] == flipped).all()
    np.testing.assert_allclose(r.weights[t], s / s.sum() * 2.5)


def test_full_size_tokens_cover_experts_and_hot_chunks():
    rng = np.random.default_rng(5)
    T = 20000
    keys = rng.random((T, 256))
    keys[:, [7, 100, 200]] += 10.0  # three experts take every token (79 chunks of <= 256)
    keys[:, 250] = -1.0            # one expert never chosen
    ids = np.argsort(-keys, 1)[:, :8].astype(np.int32)
    nmax = chunk_rows(T, "bf16")
    tok = full_size_tokens(ids, nmax)
    counts = np.bincount(ids.reshape(-1), minlength=256)
    assert set(np.unique(ids[tok])) == set(np.nonzero(counts)[0])
    for e in (7, 100, 200):
        routes = np.nonzero((ids == e).any(1))[0]
        chunks = np.array_split(routes, -(-routes.size // nmax))
        for c in chunks:
            assert np.isin(c, tok).any(), f"a chunk of expert {e} has no compared token"
    assert 0 in tok and T - 1 in tok
    assert len(tok) < 200
    # decode sizes: every token
    np.testing.assert_array_equal(full_size_tokens(ids[:64], 64), np.arange(64))


def test_chunk_rows_rule():
    assert chunk_rows(64, "bf16") == 64 and chunk_rows(8192, "bf16") == 256
    assert chunk_rows(4096, "nvfp4") == 160 and chunk_rows(64, "nvfp4") == 16 and chunk_rows(1, "fp8") == 32
    assert chunk_rows(257, "nvfp4") == 160 and chunk_rows(64, "bf16") == 64
