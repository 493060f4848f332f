"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest
import torch

import group_limited_routing_03_b300 as moe
from group_limited_routing_03_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_moe.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("beam_moe_route", "beam_moe_forward", "beam_moe_experts", "beam_moe_dispatch",
                     "beam_moe_workspace_size", "beam_moe_workspace_layout", "beam_moe_read_device_status",
                     "beam_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in beam_moe.h but not exported"


def test_debug_build_exports_the_same_boundary(lib):
    """libbeam_moe_debug.so (device checks of every workspace index) exports
    every declared entry point too, and says which build it is."""
    _build.build(debug=True)
    dbg = moe.load_debug()
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} declared in beam_moe.h but not exported by the debug build"
    assert dbg.beam_moe_debug_build() == 1
    assert lib.beam_moe_debug_build() == 0


def test_status_strings(lib):
    for code in range(7):
        assert moe.beam_status_string(code)
    assert moe.beam_status_string(99) == "unknown status"


def _shape(**kw):
    base = dict(T=64, H=5120, I=2560)
    base.update(kw)
    return moe.shape(**base)


def test_workspace_size_and_layout(lib):
    sh = _shape()
    n = moe.workspace_size(sh)
    lay = moe.workspace_layout(sh)
    assert lay["total"] == n
    R = 64 * 8
    assert lay["xp"] + R * 5120 * 2 <= lay["h"]
    assert lay["h"] + R * 2560 * 2 <= lay["yr"]
    assert lay["yr"] + R * 5120 * 2 <= n
    for k in ("status", "counts", "offsets", "perm", "pos", "xp", "h", "yr"):
        assert lay[k] % 256 == 0
    assert lay["status"] == 0


@pytest.mark.parametrize("bad", [dict(E=128), dict(n_group=4), dict(topk_group=2), dict(top_k=6),
                                 dict(H=5000), dict(I=2500), dict(T=(1 << 20) + 1)])
def test_unsupported_shapes(lib, bad):
    assert moe.workspace_size(_shape(**bad)) == 0
    with pytest.raises(moe.BeamError) as ei:
        moe.workspace_layout(_shape(**bad))
    assert ei.value.code == moe.BEAM_ERR_UNSUPPORTED


def _route_raw(lib, sh, x=0x10000, xdt=moe.BEAM_BF16, wr=0x20000, bias=None, ids=0x30000, w=0x40000,
               ws=0x100000, nbytes=None):
    if nbytes is None:
        nbytes = moe.workspace_size(sh)
    return lib.beam_moe_route(ctypes.byref(sh), x, xdt, wr, bias, ids, w, ws, nbytes, None)


def test_route_argument_errors(lib):
    sh = _shape()
    assert _route_raw(lib, sh, x=None) == moe.BEAM_ERR_INVALID_ARG
    assert _route_raw(lib, sh, x=0x10008) == moe.BEAM_ERR_INVALID_ARG  # misaligned
    assert _route_raw(lib, sh, xdt=moe.BEAM_NVFP4) == moe.BEAM_ERR_UNSUPPORTED
    assert _route_raw(lib, sh, ws=None) == moe.BEAM_ERR_WORKSPACE
    assert _route_raw(lib, sh, ws=0x100080) == moe.BEAM_ERR_WORKSPACE  # not 256-aligned
    assert _route_raw(lib, sh, nbytes=1024) == moe.BEAM_ERR_WORKSPACE
    bad = _shape(T=0)
    assert _route_raw(lib, bad) == moe.BEAM_ERR_INVALID_ARG
    sh_nan = _shape(routed_scale=float("nan"))
    assert _route_raw(lib, sh_nan) == moe.BEAM_ERR_INVALID_ARG


def test_forward_weight_errors(lib):
    sh = _shape()
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_BF16
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, None
    n = moe.workspace_size(sh)
    rc = lib.beam_moe_forward(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, 0x20000, None, ctypes.byref(ew), 0x50000,
                              0x30000, 0x40000, 0x100000, n, None)
    assert rc == moe.BEAM_ERR_INVALID_ARG
    ew.down = 0x3000
    ew.gate_sf = 0x4000  # a scale pointer with BF16 weights
    rc = lib.beam_moe_forward(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, 0x20000, None, ctypes.byref(ew), 0x50000,
                              0x30000, 0x40000, 0x100000, n, None)
    assert rc == moe.BEAM_ERR_INVALID_ARG
    rc = lib.beam_moe_forward(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, 0x20000, None, None, 0x50000, 0x30000,
                              0x40000, 0x100000, n, None)
    assert rc == moe.BEAM_ERR_INVALID_ARG


def test_nvfp4_shape_and_pointer_rules(lib):
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_NVFP4
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, 0x3000
    ew.gate_sf, ew.up_sf, ew.down_sf = 0x4000, 0x5000, 0x6000
    ew.gate_gs, ew.up_gs, ew.down_gs = 0x7000, 0x8000, 0x9000
    for H, I, want in ((384, 256, moe.BEAM_ERR_UNSUPPORTED), (256, 384, moe.BEAM_ERR_UNSUPPORTED)):
        sh = _shape(T=16, H=H, I=I)
        n = moe.workspace_size(sh, "nvfp4")
        rc = lib.beam_moe_experts(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, ctypes.byref(ew), 0x30000, 0x40000,
                                  0x50000, 0x100000, n, None)
        assert rc == want
    sh = _shape(T=16, H=256, I=256)
    ew.up_sf = None
    rc = lib.beam_moe_experts(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, ctypes.byref(ew), 0x30000, 0x40000,
                              0x50000, 0x100000, moe.workspace_size(sh, "nvfp4"), None)
    assert rc == moe.BEAM_ERR_INVALID_ARG


def test_debug_timeout_argument_errors(lib):
    assert lib.beam_moe_debug_timeout(None, 4096, 100, None) == moe.BEAM_ERR_WORKSPACE
    assert lib.beam_moe_debug_timeout(0x100000, 4096, 0, None) == moe.BEAM_ERR_INVALID_ARG


def test_binding_refuses_host_tensors(lib):
    import torch

    with pytest.raises(ValueError):
        moe._ptr(torch.zeros(4))


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(moe, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(ImportError):
        moe.load()


def test_pack_weights_argument_errors(lib):
    sh = _shape(T=16, H=256, I=256)
    src = moe._ExpertWeights()
    src.dtype = moe.BEAM_BF16
    src.gate, src.up, src.down = 0x100000, 0x2000000, 0x4000000
    dst = moe._ExpertWeights()
    dst.dtype = moe.BEAM_BF16
    dst.gate, dst.up, dst.down = 0x10000000, 0x12000000, 0x14000000

    def call(s, d):
        return lib.beam_moe_pack_weights(ctypes.byref(sh), ctypes.byref(s), ctypes.byref(d), None)

    src.layout = moe.BEAM_LAYOUT_TILED  # the source must be row-major
    assert call(src, dst) == moe.BEAM_ERR_INVALID_ARG
    src.layout = moe.BEAM_LAYOUT_ROWS
    dst.dtype = moe.BEAM_NVFP4  # dtypes must agree
    assert call(src, dst) == moe.BEAM_ERR_INVALID_ARG
    dst.dtype = moe.BEAM_BF16
    dst.up = 0x100000 + 4096  # overlaps src.gate (256 x 256 x 256 x 2 bytes)
    assert call(src, dst) == moe.BEAM_ERR_INVALID_ARG
    src.layout = 7  # not a layout
    dst.up = 0x12000000
    assert call(src, dst) == moe.BEAM_ERR_INVALID_ARG


def test_forward_rejects_unknown_layout(lib):
    sh = _shape()
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_BF16
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, 0x3000
    ew.layout = 2
    n = moe.workspace_size(sh)
    rc = lib.beam_moe_forward(ctypes.byref(sh), 0x10000, moe.BEAM_BF16, 0x20000, None, ctypes.byref(ew), 0x50000,
                              0x30000, 0x40000, 0x100000, n, None)
    assert rc == moe.BEAM_ERR_INVALID_ARG


def test_forward_residual_argument_errors(lib):
    sh = _shape(T=64, H=256, I=256)
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_BF16
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, 0x3000
    n = moe.workspace_size(sh)
    row_bytes = 64 * 256 * 2  # the stream, BF16

    def call(stream, out, g, eps, step, y=None):
        r = moe._Residual(stream, out, g, eps, step)
        a = moe._Args(0x10000, moe.BEAM_BF16, 0x20000, None, ctypes.pointer(ew), y, 0x30000, 0x40000,
                      ctypes.pointer(r))
        return lib.beam_moe_forward_residual(ctypes.byref(sh), ctypes.byref(a), 0x100000, n, None)

    S, O, G = 0x1000000, 0x2000000, 0x3000000
    assert call(S, O, G, 1e-6, 1) == moe.BEAM_ERR_INVALID_ARG  # step < 2
    assert call(S, O, G, -1.0, 2) == moe.BEAM_ERR_INVALID_ARG  # eps < 0
    assert call(S, O, G, float("inf"), 2) == moe.BEAM_ERR_INVALID_ARG
    assert call(S, O, None, 1e-6, 2) == moe.BEAM_ERR_INVALID_ARG  # no norm weight
    assert call(S, O + 8, G, 1e-6, 2) == moe.BEAM_ERR_INVALID_ARG  # misaligned out
    assert call(S, S + 16, G, 1e-6, 2) == moe.BEAM_ERR_INVALID_ARG  # out overlaps the stream
    assert call(S, O, G, 1e-6, 2, y=O + row_bytes - 16) == moe.BEAM_ERR_INVALID_ARG  # y overlaps out
    # no residual at all: the entry point needs one
    a = moe._Args(0x10000, moe.BEAM_BF16, 0x20000, None, ctypes.pointer(ew), None, 0x30000, 0x40000, None)
    assert lib.beam_moe_forward_residual(ctypes.byref(sh), ctypes.byref(a), 0x100000, n, None) == \
        moe.BEAM_ERR_INVALID_ARG
    # without a residual, the plain stages still need y
    assert lib.beam_moe_forward_stage(ctypes.byref(sh), ctypes.byref(a), 0, 0x100000, n, None) == \
        moe.BEAM_ERR_INVALID_ARG


def test_fp8_weight_rules(lib):
    sh = _shape(T=16, H=256, I=256)
    n = moe.workspace_size(sh, "fp8")
    assert n == moe.workspace_size(sh, "bf16") > 0
    lay = moe.workspace_layout(sh, "fp8")
    R_pad = 16 * 8
    assert lay["xq"] == lay["xp"] and lay["hq"] >= lay["xq"] + R_pad * 256
    assert lay["hq"] + R_pad * 256 <= lay["xp"] + R_pad * 256 * 2  # h's codes fit in the BF16 row buffer
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_FP8
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, 0x3000
    ew.gate_rs, ew.up_rs, ew.down_rs = 0x4000, 0x5000, None

    def call(shape):
        return lib.beam_moe_experts(ctypes.byref(shape), 0x10000, moe.BEAM_BF16, ctypes.byref(ew), 0x30000,
                                    0x40000, 0x50000, 0x100000, moe.workspace_size(shape, "fp8"), None)

    assert call(sh) == moe.BEAM_ERR_INVALID_ARG  # a row-scale array missing
    ew.down_rs = 0x6000
    ew.gate_sf = 0x7000  # an NVFP4 array with FP8 weights
    assert call(sh) == moe.BEAM_ERR_INVALID_ARG
    ew.gate_sf = None
    assert call(_shape(T=16, H=256, I=384)) == moe.BEAM_ERR_UNSUPPORTED  # I > H
    ew.dtype = moe.BEAM_BF16  # row scales with BF16 weights
    assert call(sh) == moe.BEAM_ERR_INVALID_ARG


def test_dense_mlp_argument_errors(lib):
    sh = moe.dense_shape(64, 256, 512)
    n = moe.dense_workspace_size(sh, "bf16")
    assert n > 0 and moe.dense_workspace_size(moe.dense_shape(64, 200, 512)) == 0
    ew = moe._ExpertWeights()
    ew.dtype = moe.BEAM_BF16
    ew.gate, ew.up, ew.down = 0x1000, 0x2000, 0x3000

    def call(x, xdt, y, ws, nbytes):
        return lib.beam_dense_mlp_forward(ctypes.byref(sh), x, xdt, ctypes.byref(ew), y, ws, nbytes, None)

    assert call(None, moe.BEAM_BF16, 0x20000, 0x100000, n) == moe.BEAM_ERR_INVALID_ARG
    assert call(0x10008, moe.BEAM_BF16, 0x20000, 0x100000, n) == moe.BEAM_ERR_INVALID_ARG  # misaligned x
    assert call(0x10000, moe.BEAM_F32, 0x20000, 0x100000, n) == moe.BEAM_ERR_UNSUPPORTED  # FP32 x, BF16 weights
    assert call(0x10000, moe.BEAM_BF16, 0x20000, 0x100000, n - 1) == moe.BEAM_ERR_WORKSPACE
    assert call(0x10000, moe.BEAM_BF16, 0x20000, 0x100080, n) == moe.BEAM_ERR_WORKSPACE  # not 256-byte aligned
    assert lib.beam_dense_mlp_forward(None, 0x10000, moe.BEAM_BF16, ctypes.byref(ew), 0x20000, 0x100000, n,
                                      None) == moe.BEAM_ERR_INVALID_ARG


def test_pack_weights_fp8_row_scales_must_be_shared(lib):
    sh = _shape(T=16, H=256, I=256)
    src = moe._ExpertWeights()
    src.dtype = moe.BEAM_FP8
    src.gate, src.up, src.down = 0x100000, 0x2000000, 0x4000000
    src.gate_rs, src.up_rs, src.down_rs = 0x7000000, 0x7100000, 0x7200000
    dst = moe._ExpertWeights()
    dst.dtype = moe.BEAM_FP8
    dst.gate, dst.up, dst.down = 0x10000000, 0x12000000, 0x14000000
    dst.gate_rs, dst.up_rs, dst.down_rs = 0x7000000, 0x7100000, 0x7300000  # down_rs differs
    assert lib.beam_moe_pack_weights(ctypes.byref(sh), ctypes.byref(src), ctypes.byref(dst), None) == \
        moe.BEAM_ERR_INVALID_ARG
    dsh = moe.dense_shape(16, 256, 256)
    assert lib.beam_dense_pack_weights(None, ctypes.byref(src), ctypes.byref(dst), None) == moe.BEAM_ERR_INVALID_ARG
    assert lib.beam_dense_pack_weights(ctypes.byref(dsh), ctypes.byref(src), ctypes.byref(dst), None) == \
        moe.BEAM_ERR_INVALID_ARG


def test_dense_workspace_grows_with_k_split_planes(lib):
    """At decode sizes the dense workspace holds the K-split partial planes
    (parts x planes x T x N FP32); at prefill sizes none are needed."""
    small = moe.dense_workspace_size(moe.dense_shape(64, 5120, 20480))
    h_and_codes = 64 * 20480 * 2 + 64 * 5120 + 64 * 20480
    assert small > h_and_codes + 4 * 2 * 64 * 20480 * 4  # four gate/up parts, two planes
    big = moe.dense_workspace_size(moe.dense_shape(8192, 5120, 20480))
    assert big < 8192 * 20480 * 2 + 8192 * 5120 + 8192 * 20480 + (1 << 20)


def test_plain_c_program_uses_the_boundary(lib, tmp_path):
    """The header is C99 and the library is usable from a C program with no
    Python or torch: workspace sizing and argument errors, no GPU needed."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_boundary.c"
    src.write_text(r'''
#include <stdio.h>
#include "beam_moe.h"
int main(void) {
  beam_moe_shape_t s = {64, 5120, 2560, 256, 8, 4, 8, 2.5f};
  size_t n = beam_moe_workspace_size(&s, BEAM_BF16);
  size_t n8 = beam_moe_workspace_size(&s, BEAM_FP8);
  beam_dense_shape_t d = {64, 5120, 20480};
  size_t nd = beam_dense_workspace_size(&d, BEAM_BF16);
  beam_moe_shape_t bad = s;
  bad.E = 128;
  int rc = beam_moe_route(&bad, 0, BEAM_BF16, 0, 0, 0, 0, 0, 0, 0);
  printf("%zu %zu %zu %d %s\n", n, n8, nd, rc, beam_status_string((beam_status_t)rc));
  return (n == 0 || n8 != n || nd == 0 || rc != BEAM_ERR_UNSUPPORTED) ? 1 : 0;
}
''')
    exe = tmp_path / "use_boundary"
    libdir = os.path.dirname(moe.library_path())
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir,
                    "-lbeam_moe", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_w4a4_shares_the_nvfp4_arrays_and_workspace(lib):
    """BEAM_NVFP4_A4 (W4A4) takes the NVFP4 weight arrays and workspace; the
    binding selects it with "activations": "nvfp4"."""
    sh = _shape()
    assert moe.workspace_size(sh, "nvfp4_a4") == moe.workspace_size(sh, "nvfp4") > 0
    assert moe.workspace_layout(sh, "nvfp4_a4") == moe.workspace_layout(sh, "nvfp4")
    codes = torch.zeros((256, 4, 8), dtype=torch.uint8)
    assert moe._wdtype({"gate": codes}) == moe.BEAM_NVFP4
    assert moe._wdtype({"gate": codes, "activations": "nvfp4"}) == moe.BEAM_NVFP4_A4
    assert moe._wdtype("nvfp4_a4") == moe.BEAM_NVFP4_A4 == 4


def test_quantize_hook_checks_its_arguments(lib):
    """The W4A4 quantiser hook rejects bad arguments before any launch."""
    fake = ctypes.c_void_p(1 << 16)  # never dereferenced: every call below fails its checks
    call = lib.beam_debug_quantize_nvfp4
    assert call(None, moe.BEAM_BF16, 4, 64, fake, fake, fake, fake, None) == moe.BEAM_ERR_INVALID_ARG
    assert call(fake, moe.BEAM_BF16, 4, 40, fake, fake, fake, fake, None) == moe.BEAM_ERR_INVALID_ARG
    assert call(fake, moe.BEAM_BF16, 0, 64, fake, fake, fake, fake, None) == moe.BEAM_ERR_INVALID_ARG
    assert call(fake, moe.BEAM_FP8, 4, 64, fake, fake, fake, fake, None) == moe.BEAM_ERR_UNSUPPORTED
    assert call(ctypes.c_void_p((1 << 16) + 8), moe.BEAM_BF16, 4, 64, fake, fake, fake, fake, None) == \
        moe.BEAM_ERR_INVALID_ARG
