"""The Python binding's own argument checks (pure marshalling, no GPU): dtype
and shape errors are raised before any library call."""
import pytest
import torch

import group_limited_routing_03_b300 as moe


def test_activation_dtypes():
    assert moe._act_dtype(torch.zeros(2, dtype=torch.float32)) == moe.BEAM_F32
    assert moe._act_dtype(torch.zeros(2, dtype=torch.bfloat16)) == moe.BEAM_BF16
    with pytest.raises(TypeError):
        moe._act_dtype(torch.zeros(2, dtype=torch.float16))


def test_weight_dtypes_select_the_format():
    bf = {k: torch.zeros((1, 4, 4), dtype=torch.bfloat16) for k in ("gate", "up", "down")}
    f8 = {k: torch.zeros((1, 4, 4), dtype=torch.float8_e4m3fn) for k in ("gate", "up", "down")}
    u8 = {k: torch.zeros((1, 4, 2), dtype=torch.uint8) for k in ("gate", "up", "down")}
    assert moe._wdtype(bf) == moe.BEAM_BF16
    assert moe._wdtype(f8) == moe.BEAM_FP8
    assert moe._wdtype(u8) == moe.BEAM_NVFP4
    assert moe._wdtype("fp8") == moe.BEAM_FP8 and moe._wdtype(moe.BEAM_NVFP4) == moe.BEAM_NVFP4
    with pytest.raises(TypeError):
        moe._weights({k: torch.zeros((1, 4, 4), dtype=torch.float16) for k in ("gate", "up", "down")})


def test_residual_arguments_checked_before_marshalling():
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    g = torch.ones(128, dtype=torch.float32)
    with pytest.raises(ValueError):  # stream of another dtype
        moe._residual(x, torch.zeros((4, 128), dtype=torch.float32), x, g, 1e-6, 2)
    with pytest.raises(ValueError):  # out of another shape
        moe._residual(x, x, torch.zeros((4, 256), dtype=torch.bfloat16), g, 1e-6, 2)
    with pytest.raises(ValueError):  # norm weight not FP32 [H]
        moe._residual(x, x, x, g.to(torch.bfloat16), 1e-6, 2)
    with pytest.raises(ValueError):  # host tensors are refused when marshalled
        moe._residual(x, x, x, g, 1e-6, 2)


def _header_struct_fields(name):
    """Field names, in order, of `typedef struct { ... } name;` in the header."""
    import os
    import re

    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                             "beam_moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    m = re.search(r"typedef struct \{([^}]*)\}\s*" + name + r"\s*;", text)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        head, *rest = decl.split(",")
        fields.append(re.findall(r"\**(\w+)\s*$", head)[0])
        fields += [r.strip().lstrip("*") for r in rest]
    return fields


@pytest.mark.parametrize("cname,pyname", [
    ("beam_moe_shape_t", "Shape"), ("beam_expert_weights_t", "_ExpertWeights"), ("beam_moe_args_t", "_Args"),
    ("beam_ws_layout_t", "_WsLayout"), ("beam_residual_t", "_Residual"), ("beam_dense_shape_t", "DenseShape")])
def test_ctypes_structs_match_the_header(cname, pyname):
    assert [n for n, _ in getattr(moe, pyname)._fields_] == _header_struct_fields(cname)
