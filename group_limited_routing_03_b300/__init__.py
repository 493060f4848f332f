"""Group-limited Mixture-of-Experts block (Beam-shaped) on one B300.

Thin Python binding of the C ABI in ``include/beam_moe.h``: every function
here only marshals torch tensors (device memory, streams) into the calls of
``libbeam_moe.so``; every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: a missing or unloadable library raises.

The block (Beam launch post, "Willkommen Beam ..." (spke.com), section
"Mixture of Experts"): sigmoid router over 256 experts, 8 groups of 32 ranked
by the sum of their two best scores, best 4 groups kept, top-8 experts inside
them, weights normalised and scaled by 2.5, SwiGLU experts, no shared expert.
Expert weights in BF16, NVFP4 (W4A16) or FP8 (E4M3 with row scales, E4M3
activations); the block may be followed by the post-norm residual update of
section "Residual Stream" (``beam_moe_forward_residual``); the first layers'
dense SwiGLU MLP runs on the same GEMMs (``DenseMLP``); a decode-size forward
can be recorded in a CUDA graph (``GraphedForward``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "BeamError", "Shape", "shape", "workspace_size", "workspace_layout", "alloc_workspace",
    "beam_moe_route", "beam_moe_dispatch", "beam_moe_experts", "beam_moe_forward", "beam_moe_forward_stage",
    "ForwardCall", "STAGES", "beam_moe_stage_kernel_count", "beam_moe_route_noalloc", "pack_weights",
    "BEAM_LAYOUT_ROWS", "BEAM_LAYOUT_TILED",
    "beam_moe_read_device_status", "beam_moe_debug_timeout", "beam_debug_nvfp4_expand", "beam_status_string", "BeamMoE",
    "library_path", "load", "load_debug", "BEAM_F32", "BEAM_BF16", "BEAM_NVFP4", "BEAM_FP8", "BEAM_NVFP4_A4",
    "beam_debug_quantize_nvfp4",
    "beam_moe_forward_residual", "GraphedForward",
    "DenseShape", "dense_shape", "dense_workspace_size", "dense_kernel_count", "beam_dense_mlp_forward",
    "dense_pack_weights", "DenseMLP",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libbeam_moe.so")

BEAM_OK, BEAM_ERR_INVALID_ARG, BEAM_ERR_UNSUPPORTED, BEAM_ERR_WORKSPACE = 0, 1, 2, 3
BEAM_ERR_CUDA, BEAM_ERR_TIMEOUT, BEAM_ERR_DEVICE_CHECK = 4, 5, 6
BEAM_F32, BEAM_BF16, BEAM_NVFP4, BEAM_FP8, BEAM_NVFP4_A4 = 0, 1, 2, 3, 4


class BeamError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {beam_status_string(code)} (status {code})")


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("routed_scale", ctypes.c_float)]


class DenseShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32)]


class _ExpertWeights(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("gate_sf", ctypes.c_void_p), ("up_sf", ctypes.c_void_p),
                ("down_sf", ctypes.c_void_p), ("gate_gs", ctypes.c_void_p), ("up_gs", ctypes.c_void_p),
                ("down_gs", ctypes.c_void_p), ("layout", ctypes.c_int), ("gate_rs", ctypes.c_void_p),
                ("up_rs", ctypes.c_void_p), ("down_rs", ctypes.c_void_p)]


BEAM_LAYOUT_ROWS, BEAM_LAYOUT_TILED = 0, 1


class _Residual(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("out", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("step", ctypes.c_int32)]


class _Args(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("xdtype", ctypes.c_int), ("router_w", ctypes.c_void_p),
                ("router_bias", ctypes.c_void_p), ("weights", ctypes.POINTER(_ExpertWeights)),
                ("y", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("residual", ctypes.POINTER(_Residual))]


STAGES = ("route", "dispatch", "gather", "gate_up", "down", "combine")


class _WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "counts", "offsets", "perm", "pos", "xp", "h", "yr",
                                               "total", "xq", "hq", "xs", "hs")]


_lib = None


def library_path() -> str:
    return _LIB_PATH


_LIB_DEBUG_PATH = os.path.join(_PKG, "libbeam_moe_debug.so")
_lib_debug = None


def _configure(lib):
    vp, sz, i32, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    sp = ctypes.POINTER(Shape)
    lib.beam_moe_workspace_size.argtypes = [sp, i32]
    lib.beam_moe_workspace_size.restype = sz
    lib.beam_moe_workspace_layout.argtypes = [sp, i32, ctypes.POINTER(_WsLayout)]
    lib.beam_moe_route.argtypes = [sp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.beam_moe_dispatch.argtypes = [sp, vp, vp, sz, vp]
    lib.beam_moe_experts.argtypes = [sp, vp, i32, ctypes.POINTER(_ExpertWeights), vp, vp, vp, vp, sz, vp]
    lib.beam_moe_forward.argtypes = [sp, vp, i32, vp, vp, ctypes.POINTER(_ExpertWeights), vp, vp, vp, vp, sz, vp]
    lib.beam_moe_forward_stage.argtypes = [sp, ctypes.POINTER(_Args), i32, vp, sz, vp]
    lib.beam_moe_forward_residual.argtypes = [sp, ctypes.POINTER(_Args), vp, sz, vp]
    lib.beam_moe_read_device_status.argtypes = [vp, ctypes.POINTER(u32), vp]
    lib.beam_moe_route_noalloc.argtypes = [sp, vp, i32, vp, vp, vp, vp, vp]
    lib.beam_moe_route_noalloc.restype = i32
    lib.beam_moe_stage_kernel_count.argtypes = [sp, i32, i32, i32]
    lib.beam_moe_stage_kernel_count.restype = ctypes.c_int32
    lib.beam_moe_debug_timeout.argtypes = [vp, sz, u32, vp]
    lib.beam_debug_nvfp4_expand.argtypes = [vp, vp, i32, vp, vp]
    lib.beam_debug_quantize_nvfp4.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.beam_moe_debug_build.argtypes = []
    lib.beam_moe_debug_build.restype = ctypes.c_int32
    lib.beam_moe_pack_weights.argtypes = [sp, ctypes.POINTER(_ExpertWeights), ctypes.POINTER(_ExpertWeights), vp]
    dp = ctypes.POINTER(DenseShape)
    lib.beam_dense_workspace_size.argtypes = [dp, i32]
    lib.beam_dense_workspace_size.restype = sz
    lib.beam_dense_mlp_forward.argtypes = [dp, vp, i32, ctypes.POINTER(_ExpertWeights), vp, vp, sz, vp]
    lib.beam_dense_pack_weights.argtypes = [dp, ctypes.POINTER(_ExpertWeights), ctypes.POINTER(_ExpertWeights), vp]
    lib.beam_dense_kernel_count.argtypes = [dp, i32]
    lib.beam_dense_kernel_count.restype = ctypes.c_int32
    lib.beam_status_string.argtypes = [i32]
    lib.beam_status_string.restype = ctypes.c_char_p
    for n in ("beam_moe_workspace_layout", "beam_moe_route", "beam_moe_dispatch", "beam_moe_experts",
              "beam_moe_forward", "beam_moe_forward_stage", "beam_moe_forward_residual",
              "beam_moe_read_device_status",
              "beam_moe_debug_timeout", "beam_debug_nvfp4_expand", "beam_debug_quantize_nvfp4", "beam_dense_mlp_forward",
              "beam_dense_pack_weights"):
        getattr(lib, n).restype = i32
    return lib


def load():
    """Load libbeam_moe.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build the CUDA library first (__graft_entry__.build())")
    _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


def load_debug():
    """Load libbeam_moe_debug.so, the build with device-side checks of every
    workspace index (same C ABI; ``beam_moe_debug_build()`` returns 1)."""
    global _lib_debug
    if _lib_debug is not None:
        return _lib_debug
    if not os.path.exists(_LIB_DEBUG_PATH):
        raise ImportError(f"{_LIB_DEBUG_PATH} is missing: build it first (__graft_entry__.build())")
    _lib_debug = _configure(ctypes.CDLL(_LIB_DEBUG_PATH))
    return _lib_debug


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def shape(T, H, I, E=256, n_group=8, topk_group=4, top_k=8, routed_scale=2.5) -> Shape:
    return Shape(T, H, I, E, n_group, topk_group, top_k, routed_scale)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _act_dtype(t) -> int:
    if t.dtype == torch.float32:
        return BEAM_F32
    if t.dtype == torch.bfloat16:
        return BEAM_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _weights(w: dict) -> _ExpertWeights:
    ew = _ExpertWeights()
    if w["gate"].dtype == torch.bfloat16:
        ew.dtype = BEAM_BF16
    elif w["gate"].dtype == torch.uint8:
        # "activations": "nvfp4" asks for W4A4 (GEMM inputs quantised to NVFP4)
        ew.dtype = BEAM_NVFP4_A4 if w.get("activations") == "nvfp4" else BEAM_NVFP4
    elif w["gate"].dtype == torch.float8_e4m3fn:
        ew.dtype = BEAM_FP8
    else:
        raise TypeError(f"expert weights must be bfloat16, packed NVFP4 (uint8) or float8_e4m3fn, "
                        f"got {w['gate'].dtype}")
    for name in ("gate", "up", "down", "gate_sf", "up_sf", "down_sf", "gate_gs", "up_gs", "down_gs", "gate_rs",
                 "up_rs", "down_rs"):
        t = w.get(name)
        setattr(ew, name, None if t is None else _ptr(t).value)
    ew.layout = {"rows": BEAM_LAYOUT_ROWS, "tiled": BEAM_LAYOUT_TILED}[w.get("layout", "rows")]
    return ew


def _check(code: int, where: str):
    if code != BEAM_OK:
        raise BeamError(code, where)


def _wdtype(w) -> int:
    if isinstance(w, int):
        return w
    if isinstance(w, str):
        return {"bf16": BEAM_BF16, "nvfp4": BEAM_NVFP4, "fp8": BEAM_FP8, "nvfp4_a4": BEAM_NVFP4_A4}[w]
    if w["gate"].dtype == torch.float8_e4m3fn:
        return BEAM_FP8
    if w["gate"].dtype == torch.uint8:
        return BEAM_NVFP4_A4 if w.get("activations") == "nvfp4" else BEAM_NVFP4
    return BEAM_BF16


# --------------------------------------------------------------------------
# the C ABI, one function each
# --------------------------------------------------------------------------
def beam_status_string(code: int) -> str:
    return load().beam_status_string(int(code)).decode()


def workspace_size(sh: Shape, wdtype="bf16") -> int:
    return int(load().beam_moe_workspace_size(ctypes.byref(sh), _wdtype(wdtype)))


def workspace_layout(sh: Shape, wdtype="bf16") -> dict:
    lay = _WsLayout()
    _check(load().beam_moe_workspace_layout(ctypes.byref(sh), _wdtype(wdtype), ctypes.byref(lay)),
           "beam_moe_workspace_layout")
    return {n: int(getattr(lay, n)) for n, _ in _WsLayout._fields_}


def alloc_workspace(sh: Shape, wdtype="bf16", device="cuda") -> torch.Tensor:
    """Caller-side allocation of the workspace (the library allocates none)."""
    n = workspace_size(sh, wdtype)
    if n == 0:
        raise BeamError(BEAM_ERR_UNSUPPORTED, "workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def beam_moe_route(sh, x, router_w, router_bias, topk_ids, topk_w, workspace, stream=None):
    _check(load().beam_moe_route(ctypes.byref(sh), _ptr(x), _act_dtype(x), _ptr(router_w), _ptr(router_bias),
                                 _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "beam_moe_route")


def beam_moe_route_noalloc(sh, x, router_w, router_bias, topk_ids, topk_w, stream=None):
    """beam_moe_route without a workspace, for callers that cannot allocate
    device memory: scratch lives in a 6 MiB library-owned device buffer
    (T <= 65536).  Calls share that buffer, so calls that overlap on the GPU
    race; the first call on a device should come before any stream capture."""
    _check(load().beam_moe_route_noalloc(ctypes.byref(sh), _ptr(x), _act_dtype(x), _ptr(router_w),
                                         _ptr(router_bias), _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "beam_moe_route_noalloc")


def beam_moe_dispatch(sh, topk_ids, workspace, stream=None):
    _check(load().beam_moe_dispatch(ctypes.byref(sh), _ptr(topk_ids), _ptr(workspace), workspace.numel(),
                                    _stream(stream)), "beam_moe_dispatch")


def beam_moe_experts(sh, x, weights: dict, topk_ids, topk_w, y, workspace, stream=None):
    ew = _weights(weights)
    _check(load().beam_moe_experts(ctypes.byref(sh), _ptr(x), _act_dtype(x), ctypes.byref(ew), _ptr(topk_ids),
                                   _ptr(topk_w), _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "beam_moe_experts")


def beam_moe_forward(sh, x, router_w, router_bias, weights: dict, y, topk_ids, topk_w, workspace, stream=None):
    ew = _weights(weights)
    _check(load().beam_moe_forward(ctypes.byref(sh), _ptr(x), _act_dtype(x), _ptr(router_w), _ptr(router_bias),
                                   ctypes.byref(ew), _ptr(y), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "beam_moe_forward")


def _residual(x, resid, out, norm_weight, eps, step) -> _Residual:
    if resid.dtype != x.dtype or out.dtype != x.dtype or resid.shape != x.shape or out.shape != x.shape:
        raise ValueError("residual stream and out must have x's shape and dtype")
    if norm_weight.dtype != torch.float32 or norm_weight.shape != (x.shape[1],):
        raise ValueError("norm_weight must be float32 of shape [H]")
    return _Residual(_ptr(resid).value, _ptr(out).value, _ptr(norm_weight).value, float(eps), int(step))


class ForwardCall:
    """The marshalled arguments of one forward call, reusable across calls.

    ``stage(i)`` enqueues step i of the forward (``STAGES[i]``) through
    beam_moe_forward_stage; ``run()`` enqueues all of them through
    beam_moe_forward (beam_moe_forward_residual when ``residual`` =
    (stream, out, norm_weight, eps, step) is given; ``y`` may then be None).
    The tensors must stay alive while the object is used."""

    def __init__(self, sh, x, router_w, router_bias, weights: dict, y, topk_ids, topk_w, workspace, stream=None,
                 residual=None):
        self.sh = sh
        self._ew = _weights(weights)
        self._res = None if residual is None else _residual(x, *residual)
        self._args = _Args(_ptr(x).value, _act_dtype(x), _ptr(router_w).value,
                           None if router_bias is None else _ptr(router_bias).value, ctypes.pointer(self._ew),
                           None if y is None else _ptr(y).value, _ptr(topk_ids).value, _ptr(topk_w).value,
                           None if self._res is None else ctypes.pointer(self._res))
        self._keep = (x, router_w, router_bias, weights, y, topk_ids, topk_w, workspace, residual)
        self.weights = weights
        self._ws = _ptr(workspace)
        self._ws_bytes = workspace.numel()
        self._stream = _stream(stream)
        self._lib = load()

    def stage(self, i: int):
        _check(self._lib.beam_moe_forward_stage(ctypes.byref(self.sh), ctypes.byref(self._args), int(i), self._ws,
                                                self._ws_bytes, self._stream), f"beam_moe_forward_stage({i})")

    def run(self):
        a = self._args
        if self._res is not None:
            _check(self._lib.beam_moe_forward_residual(ctypes.byref(self.sh), ctypes.byref(a), self._ws,
                                                       self._ws_bytes, self._stream), "beam_moe_forward_residual")
            return
        _check(self._lib.beam_moe_forward(ctypes.byref(self.sh), a.x, a.xdtype, a.router_w, a.router_bias,
                                          a.weights, a.y, a.topk_ids, a.topk_w, self._ws, self._ws_bytes,
                                          self._stream), "beam_moe_forward")


def beam_moe_forward_stage(sh, stage: int, x, router_w, router_bias, weights: dict, y, topk_ids, topk_w,
                           workspace, stream=None):
    ForwardCall(sh, x, router_w, router_bias, weights, y, topk_ids, topk_w, workspace, stream).stage(stage)


def beam_moe_forward_residual(sh, x, router_w, router_bias, weights: dict, resid, out, norm_weight, eps, step,
                              topk_ids, topk_w, workspace, y=None, stream=None):
    """The block followed by the post-norm residual update at step ``step``:
    out = sqrt((k-1)/k) resid + RMSNorm(y) * norm_weight / sqrt(k).  ``out``
    may be ``resid`` (in place); ``y`` (optional) also receives the block's
    output."""
    ForwardCall(sh, x, router_w, router_bias, weights, y, topk_ids, topk_w, workspace, stream,
                residual=(resid, out, norm_weight, eps, step)).run()


def pack_weights(sh, weights: dict, stream=None) -> dict:
    """The expert weights regrouped into the library's tiled layout
    (beam_moe_pack_weights): new device arrays of the same shapes and dtypes
    for gate / up / down (and the NVFP4 block scales); the global scales are
    shared with ``weights``."""
    out = {k: v for k, v in weights.items()}
    for name in ("gate", "up", "down", "gate_sf", "up_sf", "down_sf"):
        if weights.get(name) is not None:
            out[name] = torch.empty_like(weights[name])
    src, dst = _weights(weights), _weights(out)
    _check(load().beam_moe_pack_weights(ctypes.byref(sh), ctypes.byref(src), ctypes.byref(dst), _stream(stream)),
           "beam_moe_pack_weights")
    out["layout"] = "tiled"
    return out


def beam_moe_stage_kernel_count(sh, stage: int, xdtype=BEAM_BF16, wdtype=BEAM_BF16) -> int:
    """Kernels the library launches for stage ``stage`` of a forward of ``sh``."""
    n = int(load().beam_moe_stage_kernel_count(ctypes.byref(sh), int(xdtype), _wdtype(wdtype), int(stage)))
    if n < 0:
        raise BeamError(BEAM_ERR_UNSUPPORTED, "beam_moe_stage_kernel_count")
    return n


def beam_moe_read_device_status(workspace, stream=None):
    """Synchronises the stream; returns (status code, where) and clears it."""
    where = ctypes.c_uint32(0)
    code = load().beam_moe_read_device_status(_ptr(workspace), ctypes.byref(where), _stream(stream))
    return int(code), int(where.value)


def beam_debug_nvfp4_expand(codes, scales, out, stream=None):
    """Expand NVFP4 blocks with the GEMM converters' device code: codes uint8
    [n_blocks * 8], scales uint8 [n_blocks] (E4M3), out int16/float16
    [n_blocks * 16] (FP16 bits)."""
    n_blocks = scales.numel()
    if codes.numel() != 8 * n_blocks or out.numel() != 16 * n_blocks:
        raise ValueError("codes must hold 8 bytes and out 16 values per block")
    _check(load().beam_debug_nvfp4_expand(_ptr(codes), _ptr(scales), n_blocks, _ptr(out), _stream(stream)),
           "beam_debug_nvfp4_expand")


def beam_debug_quantize_nvfp4(a, codes, scales, global_scale, values, stream=None):
    """Quantise rows of ``a`` (float32 or bfloat16 [rows, K]) with the W4A4
    forward's device code: codes uint8 [rows, K] (one E2M1 code per byte),
    scales uint8 [rows, K/16] (E4M3), global_scale float32 [rows], values
    int16/float16 [rows, K] (FP16 bits of e2m1 * e4m3)."""
    rows, K = a.shape
    if codes.numel() != rows * K or scales.numel() != rows * (K // 16) or global_scale.numel() != rows \
            or values.numel() != rows * K:
        raise ValueError("output sizes must match a's rows and K")
    _check(load().beam_debug_quantize_nvfp4(_ptr(a), _act_dtype(a), rows, K, _ptr(codes), _ptr(scales),
                                            _ptr(global_scale), _ptr(values), _stream(stream)),
           "beam_debug_quantize_nvfp4")


def beam_moe_debug_timeout(workspace, timeout_us: int, stream=None):
    _check(load().beam_moe_debug_timeout(_ptr(workspace), workspace.numel(), int(timeout_us), _stream(stream)),
           "beam_moe_debug_timeout")


class GraphedForward:
    """One forward of ``layer`` for a fixed token count, recorded once in a
    CUDA graph and replayed with one launch (a decode serving loop): the
    library's kernel launches, its tensor-map arguments and the workspace
    addresses are fixed at capture; each call copies x into the graph's
    static input and replays.  Shares ``layer.workspace``: do not run the
    layer and the graph at the same time."""

    def __init__(self, layer, T: int, dtype=torch.bfloat16):
        if T > layer.max_tokens:
            raise ValueError(f"{T} tokens > workspace capacity {layer.max_tokens}")
        dev = layer.router_w.device
        self.x = torch.zeros((T, layer.H), dtype=dtype, device=dev)
        self.y = torch.empty_like(self.x)
        self.ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
        self.w = torch.empty((T, 8), dtype=torch.float32, device=dev)
        sh = layer.shape(T)
        args = (sh, self.x, layer.router_w, layer.router_bias, layer.weights, self.y, self.ids, self.w,
                layer.workspace)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):  # warm-up outside the capture (kernel attributes, driver entry points)
            ForwardCall(*args, stream=side).run()
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._call = ForwardCall(*args, stream=torch.cuda.current_stream(dev))
            self._call.run()
        self.workspace = layer.workspace

    def __call__(self, x):
        self.x.copy_(x)
        self.graph.replay()
        return self.y, self.ids, self.w


# --------------------------------------------------------------------------
# dense SwiGLU MLP (the first layers of the model)
# --------------------------------------------------------------------------
def dense_shape(T, H, I) -> DenseShape:
    return DenseShape(T, H, I)


def dense_workspace_size(sh: DenseShape, wdtype="bf16") -> int:
    return int(load().beam_dense_workspace_size(ctypes.byref(sh), _wdtype(wdtype)))


def beam_dense_mlp_forward(sh: DenseShape, x, weights: dict, y, workspace, stream=None):
    """y = Wd (silu(Wg x) * (Wu x)) with one expert's worth of weights
    (gate/up [1, I, H], down [1, H, I] and the per-expert arrays)."""
    ew = _weights(weights)
    _check(load().beam_dense_mlp_forward(ctypes.byref(sh), _ptr(x), _act_dtype(x), ctypes.byref(ew), _ptr(y),
                                         _ptr(workspace), workspace.numel(), _stream(stream)),
           "beam_dense_mlp_forward")


def dense_kernel_count(sh: DenseShape, wdtype="bf16") -> int:
    """Kernels one beam_dense_mlp_forward launches for ``sh`` on this device."""
    n = int(load().beam_dense_kernel_count(ctypes.byref(sh), _wdtype(wdtype)))
    if n < 0:
        raise BeamError(BEAM_ERR_UNSUPPORTED, "beam_dense_kernel_count")
    return n


def dense_pack_weights(sh: DenseShape, weights: dict, stream=None) -> dict:
    """The dense MLP's weights regrouped into the tiled layout (new arrays)."""
    out = {k: v for k, v in weights.items()}
    for name in ("gate", "up", "down", "gate_sf", "up_sf", "down_sf"):
        if weights.get(name) is not None:
            out[name] = torch.empty_like(weights[name])
    src, dst = _weights(weights), _weights(out)
    _check(load().beam_dense_pack_weights(ctypes.byref(sh), ctypes.byref(src), ctypes.byref(dst), _stream(stream)),
           "beam_dense_pack_weights")
    out["layout"] = "tiled"
    return out


class DenseMLP:
    """One dense SwiGLU MLP with its weights and a workspace for up to
    ``max_tokens`` rows (caller-owned torch device tensors)."""

    def __init__(self, weights: dict, max_tokens: int, pack=False):
        self.I, self.H = weights["gate"].shape[1], weights["down"].shape[1]
        self.max_tokens = max_tokens
        if pack and weights.get("layout", "rows") == "rows":
            weights = dense_pack_weights(dense_shape(max_tokens, self.H, self.I), weights)
        self.weights = weights
        n = dense_workspace_size(dense_shape(max_tokens, self.H, self.I), _wdtype(weights))
        if n == 0:
            raise BeamError(BEAM_ERR_UNSUPPORTED, "beam_dense_workspace_size")
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=weights["gate"].device)

    def __call__(self, x, y=None, stream=None):
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError(f"{T} rows > workspace capacity {self.max_tokens}")
        y = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device) if y is None else y
        beam_dense_mlp_forward(dense_shape(T, self.H, self.I), x, self.weights, y, self.workspace, stream)
        return y


# --------------------------------------------------------------------------
# convenience: one layer with its weights and workspace
# --------------------------------------------------------------------------
class BeamMoE:
    """One MoE layer: router weight/bias, expert weights and a workspace sized
    for up to ``max_tokens`` tokens, all caller-owned torch device tensors.
    ``pack=True`` regroups row-major expert weights once into the tiled
    layout (a copy; the given arrays are not modified)."""

    def __init__(self, router_w, router_bias, weights: dict, max_tokens: int, routed_scale=2.5, pack=False):
        self.router_w, self.router_bias = router_w, router_bias
        self.E, self.H = router_w.shape
        self.I = weights["gate"].shape[1]
        self.routed_scale = routed_scale
        self.max_tokens = max_tokens
        if pack and weights.get("layout", "rows") == "rows":
            weights = pack_weights(self.shape(max_tokens), weights)
        self.weights = weights
        self.workspace = alloc_workspace(self.shape(max_tokens), _wdtype(weights), router_w.device)

    def shape(self, T):
        return shape(T, self.H, self.I, self.E, routed_scale=self.routed_scale)

    def __call__(self, x, y=None, topk_ids=None, topk_w=None, stream=None):
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError(f"{T} tokens > workspace capacity {self.max_tokens}")
        dev = x.device
        y = torch.empty_like(x) if y is None else y
        topk_ids = torch.empty((T, 8), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
        topk_w = torch.empty((T, 8), dtype=torch.float32, device=dev) if topk_w is None else topk_w
        beam_moe_forward(self.shape(T), x, self.router_w, self.router_bias, self.weights, y, topk_ids, topk_w,
                         self.workspace, stream)
        return y, topk_ids, topk_w

    def residual(self, x, resid, norm_weight, eps, step, out=None, y=None, topk_ids=None, topk_w=None,
                 stream=None):
        """The layer followed by the residual update at step ``step``; returns
        (new stream, topk_ids, topk_w).  ``out=resid`` updates in place."""
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError(f"{T} tokens > workspace capacity {self.max_tokens}")
        dev = x.device
        out = torch.empty_like(x) if out is None else out
        topk_ids = torch.empty((T, 8), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
        topk_w = torch.empty((T, 8), dtype=torch.float32, device=dev) if topk_w is None else topk_w
        beam_moe_forward_residual(self.shape(T), x, self.router_w, self.router_bias, self.weights, resid, out,
                                  norm_weight, eps, step, topk_ids, topk_w, self.workspace, y=y, stream=stream)
        return out, topk_ids, topk_w
