"""CPU oracle for the group-limited MoE block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library in
``group_limited_routing_03_b300``) never imports it, and the two share no
code: the arithmetic lives in ``beam_oracle.c`` (plain C, IEEE double),
written from the Beam launch post:

* "Willkommen Beam: ein offenes 501B-Modell ..." (spke.com), section
  "Mixture of Experts" -- sigmoid scores over 256 experts, 8 groups of 32,
  groups ranked by the sum of their two best scores, best 4 kept, top-8
  experts inside them, normalised weights times 2.5, no shared expert,
  SwiGLU experts (intermediate 2560, hidden 5120);
* the same post, section "Residual Stream" -- router and SwiGLU product in
  FP32 (the oracle uses double, the exact definition); the stream update
  sqrt((k-1)/k) * stream + output / sqrt(k) at step k, sublayer outputs
  normalised after the sublayer (read as RMSNorm, the norm the post names in
  section "Attention");
* the same post, section "Mixture of Experts", names an FP8 checkpoint
  beside BF16 and NVFP4 without its layout: read as E4M3 weights with an FP32
  scale per output row and activations quantised per row to E4M3 at run time
  (scale = row amax / 448) -- ``expert_ffn_fp8``;
* the Chinese translation "Reflection 发布 501B 开放模型 Beam ..."
  (sihot.dev), section 混合专家, says the same.

Every function here only marshals numpy arrays into the C library.

Parity status of each function (what pins it is in ``tests/test_oracle_*``):

* ``route``        pinned: brute force over all 70 group subsets and a full
                   sort of the candidates, closed-form designed scores, the
                   zero input, invariants, library matmul + expit for scores.
* ``expert_ffn``   pinned: numpy matmul on decoded weights, closed forms.
* ``combine``      pinned: identical-expert closed form, zero input.
* ``dispatch``     pinned: numpy stable argsort / bincount.
* ``residual_update`` pinned: the post's own statements -- the two weights'
                   squares sum to one (unit-RMS stream and normalised output on
                   disjoint supports keep unit RMS at every step), and after
                   the steps 2..105 the embedding and every normalised output
                   carry the same weight 1/sqrt(105); closed forms of RMSNorm
                   (constant rows, with and without eps).
* decoders         pinned: torch float8_e4m3fn conversion (all 256 codes),
                   the OCP E2M1 value table.
* ``encode_e4m3``  pinned: torch's float -> float8_e4m3fn cast (nearest, ties
                   to even) on every code value, every midpoint and random
                   values; saturation closed form.
* ``quantize_e4m3_rows`` pinned: closed forms (the row maximum encodes to
                   +-448, zero rows, power-of-two rows reconstruct exactly)
                   and torch's cast of a / (amax / 448).
* ``expert_ffn_fp8`` pinned: numpy matmuls on values decoded and quantised by
                   torch (float8_e4m3fn), independent of the oracle's encoder,
                   with h rounded to BF16 by torch.
* ``encode_e2m1``  pinned: brute-force nearest E2M1 magnitude with the
                   even-code tie rule, the generator's independent storage
                   encoder, saturation.
* ``quantize_nvfp4_rows`` pinned: scales against torch's E4M3 cast of the
                   FP32 block value, codes against a brute-force nearest
                   search, zero rows, error bounds.
* ``expert_ffn_w4a4`` pinned: numpy matmuls on weights decoded by the pinned
                   decoders and activations from the pinned quantiser (the
                   NVFP4-activation reading for a W4A4 path; no kernel yet).
* ``round_bf16``   pinned: torch's float32 -> bfloat16 cast on float inputs
                   (every tie of a random sample), closed forms on doubles.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "beam_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libbeam_oracle.so")

F32, BF16, NVFP4 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile beam_oracle.c into libbeam_oracle.so next to it (gcc -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_route.argtypes = [i64, i64, i32, i32, i32, i32, dbl, vp, i32, vp, vp, vp, vp, vp,
                                     vp, vp, vp, i32]
        lib.oracle_route.restype = i32
        lib.oracle_expert_ffn.argtypes = [i64, i64, i64, vp, i32, i32, vp, vp, vp, vp, vp, vp, dbl,
                                          dbl, dbl, vp, vp, i32]
        lib.oracle_expert_ffn.restype = i32
        lib.oracle_expert_ffn_fp8.argtypes = [i64, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        lib.oracle_expert_ffn_fp8.restype = i32
        lib.oracle_encode_e2m1.argtypes = [ctypes.c_float]
        lib.oracle_encode_e2m1.restype = ctypes.c_uint8
        lib.oracle_quantize_nvfp4_row.argtypes = [vp, i64, vp, vp, vp]
        lib.oracle_quantize_nvfp4_row.restype = None
        lib.oracle_expert_ffn_w4a4.argtypes = [i64, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp, dbl, dbl, dbl, vp, vp,
                                               i32]
        lib.oracle_expert_ffn_w4a4.restype = i32
        lib.oracle_round_bf16.argtypes = [dbl]
        lib.oracle_round_bf16.restype = ctypes.c_float
        lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.oracle_quantize_e4m3_row.argtypes = [vp, i64, vp, vp]
        lib.oracle_quantize_e4m3_row.restype = None
        lib.oracle_combine.argtypes = [i64, i32, i64, vp, vp, vp]
        lib.oracle_combine.restype = i32
        lib.oracle_residual_update.argtypes = [i64, i64, vp, vp, vp, dbl, i32, vp]
        lib.oracle_residual_update.restype = i32
        lib.oracle_dispatch.argtypes = [i64, i32, vp, vp, vp, vp, vp]
        lib.oracle_dispatch.restype = i32
        for name in ("oracle_decode_bf16", "oracle_decode_e4m3", "oracle_decode_e2m1"):
            getattr(lib, name).restype = dbl
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _act(x: np.ndarray):
    """Activations: float32 array, or uint16 array of BF16 bit patterns."""
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    raise TypeError(f"activations must be float32 or uint16 (bf16 bits), got {x.dtype}")


def route(x, router_w, bias=None, *, n_group=8, topk_group=4, top_k=8, scale=2.5,
          want_scores=False, want_logits=False, threads=None):
    """Group-limited routing of every row of x.

    Returns dict(ids int32[T,K], weights f64[T,K], margin f64[T] (min of the
    group and expert margins), margin_group, margin_expert, and optionally
    scores / logits f64[T,E]).
    """
    lib = _load()
    x, xd = _act(x)
    T, H = x.shape
    router_w = np.ascontiguousarray(router_w, dtype=np.float32)
    E = router_w.shape[0]
    assert router_w.shape == (E, H)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float64)
    mg = np.zeros(T, np.float64)
    me = np.zeros(T, np.float64)
    sc = np.zeros((T, E), np.float64) if want_scores else None
    lg = np.zeros((T, E), np.float64) if want_logits else None
    rc = lib.oracle_route(T, H, E, n_group, topk_group, top_k, scale, _ptr(x), xd, _ptr(router_w),
                          _ptr(b), _ptr(ids), _ptr(w), _ptr(mg), _ptr(me), _ptr(sc), _ptr(lg),
                          threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_route failed ({rc})")
    out = dict(ids=ids, weights=w, margin_group=mg, margin_expert=me, margin=np.minimum(mg, me))
    if want_scores:
        out["scores"] = sc
    if want_logits:
        out["logits"] = lg
    return out


def expert_ffn(x, wg, wu, wd, *, scales=None, global_scales=(1.0, 1.0, 1.0), want_h=False,
               threads=None):
    """One expert's SwiGLU MLP on the rows of x.

    Weights: float32 arrays, uint16 arrays (BF16 bits), or uint8 packed NVFP4
    ([rows, K/2]) with ``scales`` = (sg, su, sd) uint8 E4M3 arrays [rows, K/16]
    and ``global_scales`` = (gg, gu, gd).  Returns f64[n, H] (and h f64[n, I]).
    """
    lib = _load()
    x, xd = _act(x)
    n, H = x.shape
    if wg.dtype == np.float32:
        wdt = F32
    elif wg.dtype == np.uint16:
        wdt = BF16
    elif wg.dtype == np.uint8:
        wdt = NVFP4
    else:
        raise TypeError(f"unsupported weight dtype {wg.dtype}")
    I = wg.shape[0]
    kcols = H // 2 if wdt == NVFP4 else H
    assert wg.shape == (I, kcols) and wu.shape == (I, kcols), (wg.shape, wu.shape)
    assert wd.shape == (H, I // 2 if wdt == NVFP4 else I), wd.shape
    wg, wu, wd = (np.ascontiguousarray(a) for a in (wg, wu, wd))
    sg = su = sd = None
    if wdt == NVFP4:
        sg, su, sd = (np.ascontiguousarray(s, dtype=np.uint8) for s in scales)
        assert sg.shape == (I, H // 16) and su.shape == (I, H // 16) and sd.shape == (H, I // 16)
    out = np.zeros((n, H), np.float64)
    h = np.zeros((n, I), np.float64) if want_h else None
    gg, gu, gd = (float(v) for v in global_scales)
    rc = lib.oracle_expert_ffn(H, I, n, _ptr(x), xd, wdt, _ptr(wg), _ptr(wu), _ptr(wd), _ptr(sg),
                               _ptr(su), _ptr(sd), gg, gu, gd, _ptr(out), _ptr(h),
                               threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_expert_ffn failed ({rc})")
    return (out, h) if want_h else out


def combine(weights, o):
    """y[t] = sum_k weights[t,k] * o[t,k,:]; weights f64[n,K], o f64[n,K,H]."""
    lib = _load()
    weights = np.ascontiguousarray(weights, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    n, K = weights.shape
    H = o.shape[2]
    assert o.shape == (n, K, H)
    y = np.zeros((n, H), np.float64)
    rc = lib.oracle_combine(n, K, H, _ptr(weights), _ptr(o), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_combine failed ({rc})")
    return y


def residual_update(y, stream, w, eps, k):
    """The stream after the MoE sublayer at step k (section "Residual Stream"):
    sqrt((k-1)/k) * stream + RMSNorm(y) * w / sqrt(k), in double.  y f64[n,H];
    stream f64[n,H], f32, or uint16 BF16 bits; w f64/f32[H]."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    n, H = y.shape
    stream = np.asarray(stream)
    if stream.dtype == np.uint16:  # BF16 bits: the upper half of an FP32 pattern (exact)
        stream = (stream.astype(np.uint32) << 16).view(np.float32)
    stream = np.ascontiguousarray(stream, dtype=np.float64).reshape(n, H)
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(H)
    out = np.zeros((n, H), np.float64)
    rc = lib.oracle_residual_update(n, H, _ptr(y), _ptr(stream), _ptr(w), ctypes.c_double(eps), int(k), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_residual_update failed ({rc})")
    return out


def round_bf16(v: float) -> float:
    """The BF16 value nearest to the double v (ties to even)."""
    return float(_load().oracle_round_bf16(float(v)))


def encode_e4m3(v) -> int:
    """E4M3 code of one float32 value (nearest, ties to even, saturating)."""
    return int(_load().oracle_encode_e4m3(float(np.float32(v))))


def quantize_e4m3_rows(a):
    """Per-row E4M3 quantisation of float32 rows a [n, K]: (codes uint8 [n, K],
    scales float32 [n]) with scale = amax / 448 (1 for a zero row)."""
    lib = _load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    n, K = a.shape
    codes = np.zeros((n, K), np.uint8)
    scales = np.zeros(n, np.float32)
    for r in range(n):
        row = a[r]
        lib.oracle_quantize_e4m3_row(_ptr(row), K, _ptr(codes[r]), scales[r:r + 1].ctypes.data_as(ctypes.c_void_p))
    return codes, scales


def encode_e2m1(v) -> int:
    """E2M1 code (4 bits) of one float32 value: nearest, ties to even, saturating at 6."""
    return int(_load().oracle_encode_e2m1(float(np.float32(v))))


def quantize_nvfp4_rows(a):
    """Per-row NVFP4 quantisation of float32 rows a [n, K] (K % 16 == 0):
    (codes uint8 [n, K] one E2M1 code per byte, scales uint8 [n, K/16] E4M3
    bits, global float32 [n]) with global = amax / (6 * 448)."""
    lib = _load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    n, K = a.shape
    assert K % 16 == 0
    codes = np.zeros((n, K), np.uint8)
    scales = np.zeros((n, K // 16), np.uint8)
    glob = np.zeros(n, np.float32)
    for r in range(n):
        row = a[r]
        lib.oracle_quantize_nvfp4_row(_ptr(row), K, _ptr(codes[r]), _ptr(scales[r]),
                                      glob[r:r + 1].ctypes.data_as(ctypes.c_void_p))
    return codes, scales, glob


def expert_ffn_w4a4(x, wg, wu, wd, *, scales, global_scales, want_h=False, threads=None):
    """One expert with NVFP4 weights (as expert_ffn) whose GEMM inputs are
    quantised per row to NVFP4 (quantize_nvfp4_rows; h rounded to BF16
    first).  Returns f64[n, H] (and h f64[n, I] before rounding)."""
    lib = _load()
    x, xd = _act(x)
    n, H = x.shape
    I = wg.shape[0]
    assert wg.shape == (I, H // 2) and wu.shape == (I, H // 2) and wd.shape == (H, I // 2)
    wg, wu, wd = (np.ascontiguousarray(m, dtype=np.uint8) for m in (wg, wu, wd))
    sg, su, sd = (np.ascontiguousarray(m, dtype=np.uint8) for m in scales)
    gg, gu, gd = (float(v) for v in global_scales)
    out = np.zeros((n, H), np.float64)
    h = np.zeros((n, I), np.float64) if want_h else None
    rc = lib.oracle_expert_ffn_w4a4(H, I, n, _ptr(x), xd, _ptr(wg), _ptr(wu), _ptr(wd), _ptr(sg), _ptr(su),
                                    _ptr(sd), gg, gu, gd, _ptr(out), _ptr(h), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_expert_ffn_w4a4 failed ({rc})")
    return (out, h) if want_h else out


def expert_ffn_fp8(x, wg, wu, wd, rg, ru, rd, *, want_h=False, threads=None):
    """One expert with FP8 weights (E4M3 codes [I,H] / [H,I] uint8, FP32 row
    scales [I] / [H]) on the rows of x (float32 or BF16 bits); activations
    quantised per row to E4M3 before each GEMM.  Returns f64[n, H] (and the
    unquantised h f64[n, I])."""
    lib = _load()
    x, xd = _act(x)
    n, H = x.shape
    I = wg.shape[0]
    assert wg.shape == (I, H) and wu.shape == (I, H) and wd.shape == (H, I)
    wg, wu, wd = (np.ascontiguousarray(m, dtype=np.uint8) for m in (wg, wu, wd))
    rg, ru, rd = (np.ascontiguousarray(v, dtype=np.float32) for v in (rg, ru, rd))
    assert rg.shape == (I,) and ru.shape == (I,) and rd.shape == (H,)
    out = np.zeros((n, H), np.float64)
    h = np.zeros((n, I), np.float64) if want_h else None
    rc = lib.oracle_expert_ffn_fp8(H, I, n, _ptr(x), xd, _ptr(wg), _ptr(wu), _ptr(wd), _ptr(rg), _ptr(ru),
                                   _ptr(rd), _ptr(out), _ptr(h), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_expert_ffn_fp8 failed ({rc})")
    return (out, h) if want_h else out


def dispatch(ids, n_experts=256):
    """Per-expert route lists: counts[E], offsets[E+1], perm[R], pos[R]."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    R = ids.shape[0]
    counts = np.zeros(n_experts, np.int32)
    offsets = np.zeros(n_experts + 1, np.int32)
    perm = np.zeros(R, np.int32)
    pos = np.zeros(R, np.int32)
    rc = lib.oracle_dispatch(R, n_experts, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(perm),
                             _ptr(pos))
    if rc != 0:
        raise ValueError(f"oracle_dispatch failed ({rc})")
    return dict(counts=counts, offsets=offsets, perm=perm, pos=pos)


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)


def decode_e4m3(code: int) -> float:
    return _load().oracle_decode_e4m3(code)


def decode_e2m1(code: int) -> float:
    return _load().oracle_decode_e2m1(code)


def forward(x, router_w, bias, wg, wu, wd, *, scales=None, global_scales=None, n_group=8,
            topk_group=4, top_k=8, scale=2.5, tokens=None, threads=None):
    """Whole block for the tokens listed in ``tokens`` (all when None).

    wg/wu/wd are per-expert sequences (or stacked arrays) in any format
    ``expert_ffn`` accepts; ``scales[e]`` / ``global_scales[e]`` give the
    NVFP4 extras of expert e.  Routing runs on all tokens (it is cheap);
    the experts run only for the listed tokens, one expert at a time.
    Returns dict(route=..., tokens=idx, y=f64[len(idx), H]).
    """
    r = route(x, router_w, bias, n_group=n_group, topk_group=topk_group, top_k=top_k, scale=scale,
              threads=threads)
    T = x.shape[0]
    idx = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    H = x.shape[1]
    o = np.zeros((len(idx), top_k, H), np.float64)
    sub_ids = r["ids"][idx]
    for e in np.unique(sub_ids):
        rows, ks = np.nonzero(sub_ids == e)
        kw = {}
        if scales is not None:
            kw["scales"] = scales[e]
            kw["global_scales"] = global_scales[e]
        o[rows, ks] = expert_ffn(x[idx[rows]], wg[e], wu[e], wd[e], threads=threads, **kw)
    y = combine(r["weights"][idx], o)
    return dict(route=r, tokens=idx, y=y)
