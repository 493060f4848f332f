"""Seeded synthetic inputs for the MoE block (the only module both the CUDA
path's tests and the CPU oracle consume).

This module holds none of the block's arithmetic: it draws tensors with a
seeded ``torch.Generator`` and, for the NVFP4 workload, encodes the drawn
weights into the storage format (E2M1 codes, E4M3 block scales, FP32 global
scale).  Decoding that format is done independently by the CUDA kernels and
by the oracle.

Workloads (hidden H, intermediate I, 256 experts in 8 groups of 32, top-4
groups, top-8 experts, routed scale 2.5):

=========  ======  =====  =====  ============================================
name       T       H      I      storage
=========  ======  =====  =====  ============================================
tiny       128     256    128    FP32 x / router / experts (seed 0)
decode     64      5120   2560   BF16 x, BF16 experts (~20 GB), FP32 router
prefill    8192    5120   2560   same as decode, no router bias
nvfp4      4096    5120   2560   BF16 x, NVFP4 experts, FP32 router
nvfp4_dec  64      5120   2560   same as nvfp4 (decode)
nvfp4_a4   4096    5120   2560   the nvfp4 inputs (seed 3), W4A4 GEMMs
skew       32768   5120   2560   BF16, Zipf(1.1) router bias scaled to [0, 3]
fp8        8192    5120   2560   BF16 x, FP8 experts (E4M3 + row scales, ~10 GB)
fp8_decode 64      5120   2560   same as fp8
dense      8192    5120   20480  dense SwiGLU MLP (one "expert"), BF16 (0.63 GB)
dense_dec  64      5120   20480  same as dense
=========  ======  =====  =====  ============================================

The dense MLP's width is not given on the pages; 20480 = 8 x 2560 gives it
the per-token work of the MoE block's eight experts.

Distributions: x ~ N(0, 1) (a post-RMSNorm hidden state); router weight
~ N(0, variance 1/H), so logits are ~N(0, 1); expert weights ~ N(0, std 0.02).
Seeds: tiny 0, decode 1, prefill 2, nvfp4 3, skew 4, fp8 5, fp8_decode 6,
dense 7, dense_dec 8, nvfp4_dec 9.  Draw order: x, router
weight, bias, gate (expert by expert), up, down.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

N_EXPERTS = 256
N_GROUP = 8
TOPK_GROUP = 4
TOP_K = 8
ROUTED_SCALE = 2.5


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    x_dtype: str  # "f32" | "bf16"
    w_dtype: str  # "f32" | "bf16" | "nvfp4" | "fp8"
    seed: int
    bias: str  # "none" | "zipf"
    E: int = N_EXPERTS
    acts: str = "native"  # "nvfp4": the GEMM inputs quantised to NVFP4 at run time (W4A4, NVFP4 weights)

    @property
    def routes(self) -> int:
        return self.T * TOP_K


WORKLOADS = {
    "tiny": Workload("tiny", 128, 256, 128, "f32", "f32", 0, "none"),
    "decode": Workload("decode", 64, 5120, 2560, "bf16", "bf16", 1, "none"),
    "prefill": Workload("prefill", 8192, 5120, 2560, "bf16", "bf16", 2, "none"),
    "nvfp4": Workload("nvfp4", 4096, 5120, 2560, "bf16", "nvfp4", 3, "none"),
    "skew": Workload("skew", 32768, 5120, 2560, "bf16", "bf16", 4, "zipf"),
    "fp8": Workload("fp8", 8192, 5120, 2560, "bf16", "fp8", 5, "none"),
    "fp8_decode": Workload("fp8_decode", 64, 5120, 2560, "bf16", "fp8", 6, "none"),
    "nvfp4_dec": Workload("nvfp4_dec", 64, 5120, 2560, "bf16", "nvfp4", 9, "none"),
    # the nvfp4 layer's inputs (same seed) with W4A4 GEMMs
    "nvfp4_a4": Workload("nvfp4_a4", 4096, 5120, 2560, "bf16", "nvfp4", 3, "none", acts="nvfp4"),
    "dense": Workload("dense", 8192, 5120, 20480, "bf16", "bf16", 7, "none", E=1),
    "dense_dec": Workload("dense_dec", 64, 5120, 20480, "bf16", "bf16", 8, "none", E=1),
}


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller T)."""
    base = WORKLOADS[name]
    if not overrides:
        return base
    d = dict(base.__dict__)
    d.update(overrides)
    return Workload(**d)


# ---------------------------------------------------------------------------
# NVFP4 storage encoding (input preparation only)
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
E2M1_MAX = 6.0
# Magnitudes where round-to-nearest-even to the E2M1 grid
# {0, 0.5, 1, 1.5, 2, 3, 4, 6} moves up one code; ">" at midpoints whose lower
# neighbour has the even code, ">=" where the upper neighbour has it.
_E2M1_STEPS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False),
               (3.5, True), (5.0, False))


def _e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Round q to E2M1 (nearest, ties to even, saturating at +-6); 4-bit codes."""
    mag = q.abs()
    code = torch.zeros_like(mag, dtype=torch.uint8)
    for thr, inclusive in _E2M1_STEPS:
        code += (mag >= thr if inclusive else mag > thr).to(torch.uint8)
    sign = ((q < 0) & (code > 0)).to(torch.uint8) << 3
    return code | sign


def quantize_nvfp4(w: torch.Tensor):
    """Encode a float32 matrix [N, K] (K % 16 == 0) in NVFP4 storage.

    Common public recipe: global = amax / (6 * 448); block scale (16
    consecutive K) = E4M3(block_amax / 6 / global); element = E2M1(w /
    (scale * global)).  Returns (packed uint8 [N, K/2] with the even K index
    in the low nibble, scales uint8 [N, K/16] = E4M3 bits, global float).
    """
    N, K = w.shape
    assert K % 16 == 0
    w = w.float()
    amax = float(w.abs().max())
    g = amax / (E2M1_MAX * E4M3_MAX) if amax > 0 else 1.0
    blk = w.view(N, K // 16, 16)
    bamax = blk.abs().amax(-1)
    sc8 = (bamax / E2M1_MAX / g).clamp(max=E4M3_MAX).to(torch.float8_e4m3fn)
    step = sc8.to(torch.float32) * g
    safe = torch.where(step > 0, step, torch.ones_like(step))
    q = torch.where(step.unsqueeze(-1) > 0, blk / safe.unsqueeze(-1), torch.zeros_like(blk))
    codes = _e2m1_codes(q).view(N, K)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.contiguous(), sc8.view(torch.uint8).contiguous(), g


def quantize_fp8_rows(w: torch.Tensor):
    """Encode a float32 matrix [N, K] as FP8 with one scale per row: scale =
    row amax / 448 (1 for a zero row), codes = E4M3(w / scale) by torch's
    cast (nearest, ties to even).  Returns (codes float8_e4m3fn [N, K],
    scales float32 [N])."""
    w = w.float()
    amax = w.abs().amax(1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (w / scale[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes.contiguous(), scale.contiguous()


# ---------------------------------------------------------------------------
# Generation
# ---------------------------------------------------------------------------
def zipf_bias(E: int, gen: torch.Generator, device, s: float = 1.1, top: float = 3.0):
    """Per-expert bias from a Zipf(s) rank law scaled to [0, top]; ranks are a
    seeded permutation of the experts."""
    rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
    lo = E ** (-s)
    b = top * (rank.pow(-s) - lo) / (1.0 - lo)
    return b.to(torch.float32)


def _randn(shape, gen, device, std=1.0):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(std)


def generate(wl: Workload, device="cpu", *, experts=True):
    """Draw every input of workload ``wl`` on ``device``.

    Returns a dict with x [T,H], router_w [E,H] f32, bias [E] f32 or None and,
    when ``experts``: gate/up [E,I,H], down [E,H,I] (f32 or bf16) or, for
    NVFP4, gate/up/down packed uint8, gate_sf/up_sf/down_sf uint8 E4M3 and
    gate_gs/up_gs/down_gs float32 [E]; for FP8, gate/up/down float8_e4m3fn
    and gate_rs/up_rs/down_rs float32 row scales [E, I] / [E, H].
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    out = {}
    x = _randn((wl.T, wl.H), gen, device)
    out["x"] = x if wl.x_dtype == "f32" else x.to(torch.bfloat16)
    out["router_w"] = _randn((wl.E, wl.H), gen, device, std=math.sqrt(1.0 / wl.H))
    out["bias"] = zipf_bias(wl.E, gen, device) if wl.bias == "zipf" else None
    if not experts:
        return out
    shapes = {"gate": (wl.I, wl.H), "up": (wl.I, wl.H), "down": (wl.H, wl.I)}
    for name, (n, k) in shapes.items():
        if wl.w_dtype == "nvfp4":
            packed = torch.empty((wl.E, n, k // 2), dtype=torch.uint8, device=device)
            sf = torch.empty((wl.E, n, k // 16), dtype=torch.uint8, device=device)
            gs = torch.empty((wl.E,), dtype=torch.float32)
            for e in range(wl.E):
                p, s, g = quantize_nvfp4(_randn((n, k), gen, device, std=0.02))
                packed[e].copy_(p)
                sf[e].copy_(s)
                gs[e] = g
            out[name] = packed
            out[name + "_sf"] = sf
            out[name + "_gs"] = gs.to(device)
        elif wl.w_dtype == "fp8":
            codes = torch.empty((wl.E, n, k), dtype=torch.float8_e4m3fn, device=device)
            rs = torch.empty((wl.E, n), dtype=torch.float32, device=device)
            for e in range(wl.E):
                c, r = quantize_fp8_rows(_randn((n, k), gen, device, std=0.02))
                codes[e].copy_(c)
                rs[e].copy_(r)
            out[name] = codes
            out[name + "_rs"] = rs
        else:
            dt = torch.float32 if wl.w_dtype == "f32" else torch.bfloat16
            w = torch.empty((wl.E, n, k), dtype=dt, device=device)
            for e in range(wl.E):
                w[e].copy_(_randn((n, k), gen, device, std=0.02))
            out[name] = w
    return out


RESIDUAL_EPS = 1e-6  # RMSNorm eps of the post-norm (a common value; the post gives none)


def residual_inputs(wl: Workload, device="cpu", *, seed_offset=1000):
    """The residual stream entering the update and the post-norm's scale.

    stream [T,H] ~ N(0, 1) in x's dtype (the update keeps the stream at unit
    scale, so a unit-RMS stream is its steady state); norm_weight [H] f32
    ~ 1 + N(0, 0.1^2) (a learned scale near one).  Seed: the workload's seed
    plus ``seed_offset``, so the block's own inputs are unchanged."""
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed + seed_offset)
    s = _randn((wl.T, wl.H), gen, device)
    stream = s if wl.x_dtype == "f32" else s.to(torch.bfloat16)
    g = _randn((wl.H,), gen, device, std=0.1).add_(1.0)
    return stream, g


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
