"""GB300-native Mixture-of-Experts FFN layer forward.

Thin Python binding (ctypes) over the C ABI of ``libmoe_gb300.so``
(``include/moe.h``).  The functions here only check and marshal arguments:
every step of the layer runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current CUDA stream.  If the library has not been
built, every call raises ``MoEError``; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["MoEError", "lib", "workspace_size", "alloc_workspace", "route", "permute", "forward",
           "read_status", "read_diagnostics", "LIB_PATH", "nvfp4_tc_scales", "nvfp4_quantize",
           "W4A4Weights", "w4a4_weights", "forward_w4a4", "forward_int8", "int8_struct"]

# MOE_GB300_LIB selects another build of the library (e.g. the index-checking
# MOE_DEBUG_BOUNDS build); the default is the in-tree libmoe_gb300.so.
LIB_PATH = os.environ.get("MOE_GB300_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                           "libmoe_gb300.so")

MOE_OK = 0


class MoEError(RuntimeError):
    pass


class _W4A4(ctypes.Structure):
    _fields_ = [("gu_codes", ctypes.c_void_p), ("gu_scales_tc", ctypes.c_void_p),
                ("gu_global", ctypes.c_void_p), ("dn_codes", ctypes.c_void_p),
                ("dn_scales_tc", ctypes.c_void_p), ("dn_global", ctypes.c_void_p),
                ("x_global", ctypes.c_void_p), ("h_global", ctypes.c_void_p)]


class _NVFP4(ctypes.Structure):
    _fields_ = [("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p),
                ("gu_global", ctypes.c_void_p), ("dn_codes", ctypes.c_void_p),
                ("dn_scales", ctypes.c_void_p), ("dn_global", ctypes.c_void_p)]


class _INT8(ctypes.Structure):
    _fields_ = [("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p),
                ("dn_codes", ctypes.c_void_p), ("dn_scales", ctypes.c_void_p)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, ctypes.POINTER(_NVFP4), _I, _I, _I, _I, _I, _P, _P, _P,
                         _P, _SZ, _P]),
    "moe_forward_profiled": (_I, [_P, _P, _P, _P, _P, ctypes.POINTER(_NVFP4), _I, _I, _I, _I, _I, _P,
                                  _P, _P, _P, _SZ, _P, ctypes.POINTER(_P),
                                  ctypes.POINTER(ctypes.c_int32)]),
    "moe_route_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_forward_w4a4": (_I, [_P, _P, _P, ctypes.POINTER(_W4A4), _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_w4a4_profiled": (_I, [_P, _P, _P, ctypes.POINTER(_W4A4), _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                       _SZ, _P, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_int32)]),
    "moe_forward_int8": (_I, [_P, _P, _P, ctypes.POINTER(_INT8), _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_int8_profiled": (_I, [_P, _P, _P, ctypes.POINTER(_INT8), _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                       _SZ, _P, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_int32)]),
    "moe_nvfp4_tc_scales": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "moe_nvfp4_quantize": (_I, [_P, _I, _I, ctypes.c_float, _P, _P, _P]),
    "moe_read_status": (_I, [_P, _P]),
    "moe_debug_force_wait_timeout": (_I, [_I]),
    "moe_read_diagnostics": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_error_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
}


def lib():
    """Load libmoe_gb300.so (raises MoEError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError(f"{LIB_PATH} is missing: build it with `python -m expert_layer_gb300._build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(rc: int, what: str):
    if rc != MOE_OK:
        msg = lib().moe_error_string(rc).decode()
        raise MoEError(f"{what} failed: {msg} ({rc})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _want(t: torch.Tensor, dtype, shape, name):
    if not isinstance(t, torch.Tensor):
        raise MoEError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise MoEError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MoEError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise MoEError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise MoEError(f"{name} must be contiguous")


def workspace_size(T: int, H: int, E: int, I: int, top_k: int) -> int:
    return int(lib().moe_workspace_size(T, H, E, I, top_k))


def alloc_workspace(T: int, H: int, E: int, I: int, top_k: int, device="cuda") -> torch.Tensor:
    n = workspace_size(T, H, E, I, top_k)
    if n == 0:
        raise MoEError("unsupported shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


def route(x, gate_w, bias, top_k, workspace=None, stream=None):
    """Router: returns (topk_idx int32 [T,k], topk_w fp32 [T,k])."""
    T, H = x.shape
    E = gate_w.shape[0]
    _want(x, torch.bfloat16, (T, H), "x")
    _want(gate_w, torch.bfloat16, (E, H), "gate_w")
    if bias is not None:
        _want(bias, torch.float32, (E,), "bias")
    if workspace is None:
        workspace = alloc_workspace(max(T, 1), H, E, 128, top_k, x.device)
    idx = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    rc = lib().moe_route(_ptr(x), _ptr(gate_w), _ptr(bias), T, H, E, top_k, _ptr(idx), _ptr(w),
                         _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_route")
    return idx, w


def permute(topk_idx, E, workspace=None, stream=None):
    """Grouping: returns (counts [E], offsets [E+1], perm [S], inv_perm [S]), int32."""
    T, k = topk_idx.shape
    _want(topk_idx, torch.int32, (T, k), "topk_idx")
    dev = topk_idx.device
    if workspace is None:
        workspace = alloc_workspace(max(T, 1), 128, E, 128, k, dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    rc = lib().moe_permute(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                           _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_permute")
    return counts, offsets, perm, inv


def forward(x, gate_w, bias, w_gate_up, w_down, top_k, nvfp4_gate_up=None, nvfp4_down=None,
            out=None, workspace=None, topk_idx=None, topk_w=None, stream=None):
    """The MoE layer forward; returns out bf16 [T, H].

    bf16 weights: w_gate_up [E, 2I, H], w_down [E, H, I].  NVFP4 weights: pass
    ``nvfp4_gate_up`` / ``nvfp4_down`` objects with ``codes`` (uint8),
    ``scales`` (uint8 e4m3) and ``glob`` (fp32 [E]) tensors and leave the bf16
    weights None.  ``topk_idx`` / ``topk_w`` optionally receive the routing."""
    T, H = x.shape
    E = gate_w.shape[0]
    _want(x, torch.bfloat16, (T, H), "x")
    _want(gate_w, torch.bfloat16, (E, H), "gate_w")
    if bias is not None:
        _want(bias, torch.float32, (E,), "bias")
    nv = None
    if nvfp4_gate_up is not None:
        if w_gate_up is not None or w_down is not None:
            raise MoEError("pass either bf16 or NVFP4 expert weights, not both")
        q, d = nvfp4_gate_up, nvfp4_down
        I = q.codes.shape[1] // 2
        _want(q.codes, torch.uint8, (E, 2 * I, H // 2), "gate_up codes")
        _want(q.scales, torch.uint8, (E, 2 * I, H // 16), "gate_up scales")
        _want(q.glob, torch.float32, (E,), "gate_up global")
        _want(d.codes, torch.uint8, (E, H, I // 2), "down codes")
        _want(d.scales, torch.uint8, (E, H, I // 16), "down scales")
        _want(d.glob, torch.float32, (E,), "down global")
        nv = _NVFP4(q.codes.data_ptr(), q.scales.data_ptr(), q.glob.data_ptr(), d.codes.data_ptr(),
                    d.scales.data_ptr(), d.glob.data_ptr())
    else:
        I = w_gate_up.shape[1] // 2
        _want(w_gate_up, torch.bfloat16, (E, 2 * I, H), "w_gate_up")
        _want(w_down, torch.bfloat16, (E, H, I), "w_down")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _want(out, torch.bfloat16, (T, H), "out")
    if topk_idx is not None:
        _want(topk_idx, torch.int32, (T, top_k), "topk_idx")
    if topk_w is not None:
        _want(topk_w, torch.float32, (T, top_k), "topk_w")
    if workspace is None:
        workspace = alloc_workspace(max(T, 1), H, E, I, top_k, x.device)
    rc = lib().moe_forward(_ptr(x), _ptr(gate_w), _ptr(bias), _ptr(w_gate_up), _ptr(w_down),
                           ctypes.byref(nv) if nv is not None else None, T, H, E, I, top_k,
                           _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
                           workspace.numel(), _stream(stream))
    _check(rc, "moe_forward")
    return out


def nvfp4_tc_scales(scales, gate_up: bool, stream=None):
    """NVFP4 block scales [E, rows, K/16] (uint8 e4m3) rearranged into the
    W4A4 tensor-core layout (a new uint8 tensor of the same size)."""
    E, rows, K16 = scales.shape
    _want(scales, torch.uint8, (E, rows, K16), "scales")
    out = torch.empty_like(scales)
    _check(lib().moe_nvfp4_tc_scales(_ptr(scales), E, rows, 16 * K16, 1 if gate_up else 0, _ptr(out),
                                     _stream(stream)), "moe_nvfp4_tc_scales")
    return out


def nvfp4_quantize(a, glob: float, stream=None):
    """NVFP4-encode bf16 rows a [R, K] with global scale glob: returns
    (codes uint8 [R, K/2], scales uint8 [R, K/16])."""
    R, K = a.shape
    _want(a, torch.bfloat16, (R, K), "a")
    codes = torch.empty((R, K // 2), dtype=torch.uint8, device=a.device)
    scales = torch.empty((R, K // 16), dtype=torch.uint8, device=a.device)
    _check(lib().moe_nvfp4_quantize(_ptr(a), R, K, float(glob), _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_nvfp4_quantize")
    return codes, scales


class W4A4Weights:
    """Expert weights of the W4A4 path: NVFP4 codes and globals, the block
    scales in the tensor-core layout, and the activations' globals."""

    def __init__(self, gate_up, down, x_global, h_global, stream=None):
        self.gu_codes, self.gu_global = gate_up.codes, gate_up.glob
        self.dn_codes, self.dn_global = down.codes, down.glob
        self.gu_scales_tc = nvfp4_tc_scales(gate_up.scales, True, stream)
        self.dn_scales_tc = nvfp4_tc_scales(down.scales, False, stream)
        self.x_global, self.h_global = x_global, h_global
        self.struct = _W4A4(*(t.data_ptr() for t in (self.gu_codes, self.gu_scales_tc, self.gu_global,
                                                     self.dn_codes, self.dn_scales_tc, self.dn_global,
                                                     self.x_global, self.h_global)))


def w4a4_weights(inp, stream=None) -> W4A4Weights:
    """W4A4Weights of a ``moe_inputs.MoEInputs`` bundle with NVFP4 weights and
    activation globals."""
    return W4A4Weights(inp.nvfp4_gate_up, inp.nvfp4_down, inp.x_global, inp.h_global, stream)


def forward_w4a4(x, gate_w, bias, weights: W4A4Weights, top_k, out=None, workspace=None, topk_idx=None,
                 topk_w=None, stream=None):
    """The MoE layer forward with NVFP4 weights and NVFP4 activations; returns
    out bf16 [T, H]."""
    T, H = x.shape
    E = gate_w.shape[0]
    I = weights.gu_codes.shape[1] // 2
    _want(x, torch.bfloat16, (T, H), "x")
    _want(gate_w, torch.bfloat16, (E, H), "gate_w")
    if bias is not None:
        _want(bias, torch.float32, (E,), "bias")
    _want(weights.gu_codes, torch.uint8, (E, 2 * I, H // 2), "gate_up codes")
    _want(weights.gu_scales_tc, torch.uint8, (E, 2 * I, H // 16), "gate_up scales")
    _want(weights.dn_codes, torch.uint8, (E, H, I // 2), "down codes")
    _want(weights.dn_scales_tc, torch.uint8, (E, H, I // 16), "down scales")
    for name in ("gu_global", "dn_global", "x_global", "h_global"):
        _want(getattr(weights, name), torch.float32, (E,), name)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _want(out, torch.bfloat16, (T, H), "out")
    if topk_idx is not None:
        _want(topk_idx, torch.int32, (T, top_k), "topk_idx")
    if topk_w is not None:
        _want(topk_w, torch.float32, (T, top_k), "topk_w")
    if workspace is None:
        workspace = alloc_workspace(max(T, 1), H, E, I, top_k, x.device)
    rc = lib().moe_forward_w4a4(_ptr(x), _ptr(gate_w), _ptr(bias), ctypes.byref(weights.struct), T, H, E, I,
                                top_k, _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "moe_forward_w4a4")
    return out


def int8_struct(gate_up, down):
    """The ``moe_int8_weights`` struct of two int8 block tensors (objects with
    ``codes`` int8 [E, R, K] and ``scales`` float16 [E, R, K/32])."""
    return _INT8(gate_up.codes.data_ptr(), gate_up.scales.data_ptr(), down.codes.data_ptr(),
                 down.scales.data_ptr())


def forward_int8(x, gate_w, bias, gate_up, down, top_k, out=None, workspace=None, topk_idx=None,
                 topk_w=None, stream=None):
    """The MoE layer forward with int8 block expert weights (W8A16); returns
    out bf16 [T, H].  ``gate_up`` / ``down``: objects with ``codes`` (int8
    [E, 2I, H] / [E, H, I]) and ``scales`` (float16, one per 32 elements
    along K)."""
    T, H = x.shape
    E = gate_w.shape[0]
    I = gate_up.codes.shape[1] // 2
    _want(x, torch.bfloat16, (T, H), "x")
    _want(gate_w, torch.bfloat16, (E, H), "gate_w")
    if bias is not None:
        _want(bias, torch.float32, (E,), "bias")
    _want(gate_up.codes, torch.int8, (E, 2 * I, H), "gate_up codes")
    _want(gate_up.scales, torch.float16, (E, 2 * I, H // 32), "gate_up scales")
    _want(down.codes, torch.int8, (E, H, I), "down codes")
    _want(down.scales, torch.float16, (E, H, I // 32), "down scales")
    st = int8_struct(gate_up, down)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _want(out, torch.bfloat16, (T, H), "out")
    if topk_idx is not None:
        _want(topk_idx, torch.int32, (T, top_k), "topk_idx")
    if topk_w is not None:
        _want(topk_w, torch.float32, (T, top_k), "topk_w")
    if workspace is None:
        workspace = alloc_workspace(max(T, 1), H, E, I, top_k, x.device)
    rc = lib().moe_forward_int8(_ptr(x), _ptr(gate_w), _ptr(bias), ctypes.byref(st), T, H, E, I, top_k,
                                _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                                _stream(stream))
    _check(rc, "moe_forward_int8")
    return out


def read_status(workspace, stream=None) -> int:
    """Synchronise and return the device status code of the last call."""
    return int(lib().moe_read_status(_ptr(workspace), _stream(stream)))


def read_diagnostics(workspace, stream=None) -> dict:
    buf = (ctypes.c_int32 * 4)()
    _check(lib().moe_read_diagnostics(_ptr(workspace), _stream(stream), buf), "moe_read_diagnostics")
    return dict(num_active=buf[0], num_large=buf[1], router_flagged=buf[2], router_fallback=buf[3])
