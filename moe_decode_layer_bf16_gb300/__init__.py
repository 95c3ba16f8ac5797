"""GB300-native (sm_103a) MoE decode layer: Python binding of libmoe_decode.so.

The binding only marshals arguments: every step of the decode path runs in
the library's CUDA kernels (include/moe_decode.h).  torch provides device
memory and streams.  There is no CPU fallback: if the library is not built,
every call raises.

Entry points (same names as the C ABI):
  moe_decode_workspace_size, moe_workspace_init, moe_decode_layer,
  splitk_gemm_workspace_size, splitk_gemm_bf16, rmsnorm_residual,
  moe_device_status, moe_debug_set_fault, moe_status_str
plus MoeDecodeLayer, a holder of one layer's weights and workspace.
"""

from __future__ import annotations

import ctypes
import os

from .dims import DSV3, TINY, LayerDims

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_decode.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_SCRATCH_LIMIT = 6

MOE_PATH_AUTO = 0
MOE_PATH_WARP_MMA = 1
MOE_PATH_TCGEN05 = 2



class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_status_str(status)} (status {status})")
        self.status = status


class _Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("routed_scaling", ctypes.c_float), ("swiglu_limit", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("e8m0", ctypes.c_int)]


_WEIGHT_FIELDS = ["router_w", "sel_bias", "w13", "w13_s", "w2", "w2_s", "sw13", "sw13_s", "sw2",
                  "sw2_s", "norm_gain"]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


_lib = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built (python -m moe_decode_layer_bf16_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_decode_workspace_size.argtypes = [ctypes.POINTER(_Dims), _i, ctypes.POINTER(_sz)]
        L.moe_workspace_init.argtypes = [_vp, _sz, _vp]
        L.moe_decode_layer.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights), _i, _vp, _vp, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.moe_decode_layer_traced.argtypes = L.moe_decode_layer.argtypes + [ctypes.POINTER(_vp)]
        L.moe_decode_layer_partial.argtypes = [ctypes.POINTER(_Dims), ctypes.POINTER(_Weights), _i, _vp, _vp,
                                               _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.moe_tp_boundary.argtypes = [_vp, _i, _vp, _vp, _i, _i, _f, _vp, _vp, _vp]
        L.splitk_gemm_workspace_size.argtypes = [_i, _i, _i, _i, ctypes.POINTER(_sz)]
        L.splitk_gemm_bf16.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
        L.splitk_gemm_bf16_noalloc.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
        L.moe_debug_fill_noalloc_scratch.argtypes = [_i, _vp]
        L.rmsnorm_residual.argtypes = [_vp, _vp, _vp, _i, _i, _f, _vp, _vp, _i, _vp, _vp, _vp, _vp]
        L.mtp_eh_front_workspace_size.argtypes = [_i, _i, ctypes.POINTER(_sz)]
        L.mtp_eh_front.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _f, _vp, _i, _i, _vp, _vp, _sz, _vp]
        L.moe_decode_layer_plan.argtypes = [ctypes.POINTER(_Dims), _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]
        L.moe_set_expert_path.argtypes = [_i]
        L.moe_device_status.argtypes = [_vp, _vp]
        L.moe_debug_set_fault.argtypes = [_vp, _i, _vp]
        L.moe_status_str.argtypes = [_i]
        L.moe_status_str.restype = ctypes.c_char_p
        for n in ("moe_decode_workspace_size", "moe_workspace_init", "moe_decode_layer", "moe_decode_layer_traced",
                  "splitk_gemm_workspace_size", "splitk_gemm_bf16", "splitk_gemm_bf16_noalloc", "rmsnorm_residual",
                  "moe_device_status", "moe_debug_set_fault", "moe_debug_fill_noalloc_scratch",
                  "moe_decode_layer_plan", "moe_set_expert_path", "moe_decode_layer_partial", "moe_tp_boundary",
                  "mtp_eh_front_workspace_size", "mtp_eh_front"):
            getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _dims(d: LayerDims) -> _Dims:
    return _Dims(d.hidden, d.inter, d.shared_inter, d.num_experts, d.top_k, d.routed_scaling,
                 d.swiglu_limit, d.rms_eps, 1 if d.e8m0 else 0)


def moe_status_str(status: int) -> str:
    return lib().moe_status_str(int(status)).decode()


def moe_decode_workspace_size(dims: LayerDims, max_tokens: int) -> int:
    n = _sz(0)
    _check(lib().moe_decode_workspace_size(ctypes.byref(_dims(dims)), int(max_tokens), ctypes.byref(n)),
           "moe_decode_workspace_size")
    return n.value


def moe_workspace_init(ws, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def moe_decode_layer(dims: LayerDims, weights: dict, x, residual, out, residual_out, workspace,
                     topk_ids=None, topk_w=None, sorted_routes=None, expert_offsets=None, stream=None):
    """One decode step (see include/moe_decode.h).  Tensors must be contiguous
    CUDA tensors of the documented dtypes; weights maps the moe_layer_weights
    field names (norm_gain may be given as 'gain') to tensors or None."""
    w = _Weights(*[_ptr(weights.get(n, weights.get("gain") if n == "norm_gain" else None))
                   for n in _WEIGHT_FIELDS])
    M = int(x.shape[0])
    rc = lib().moe_decode_layer(ctypes.byref(_dims(dims)), ctypes.byref(w), M, _ptr(x), _ptr(residual),
                                _ptr(out), _ptr(residual_out), _ptr(topk_ids), _ptr(topk_w),
                                _ptr(sorted_routes), _ptr(expert_offsets), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "moe_decode_layer")


def moe_decode_layer_traced(dims: LayerDims, weights: dict, x, residual, out, residual_out, workspace,
                            events, topk_ids=None, topk_w=None, sorted_routes=None, expert_offsets=None,
                            stream=None):
    """moe_decode_layer recording four torch.cuda.Event objects around its
    three kernels (before router, before experts, before boundary, after)."""
    w = _Weights(*[_ptr(weights.get(n, weights.get("gain") if n == "norm_gain" else None))
                   for n in _WEIGHT_FIELDS])
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event at its first record
            e.record()
    ev = (_vp * 4)(*[e.cuda_event for e in events])
    M = int(x.shape[0])
    rc = lib().moe_decode_layer_traced(ctypes.byref(_dims(dims)), ctypes.byref(w), M, _ptr(x),
                                       _ptr(residual), _ptr(out), _ptr(residual_out), _ptr(topk_ids),
                                       _ptr(topk_w), _ptr(sorted_routes), _ptr(expert_offsets),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream), ev)
    _check(rc, "moe_decode_layer_traced")


def moe_decode_layer_partial(dims: LayerDims, weights: dict, x, m_out, workspace, topk_ids=None, topk_w=None,
                             sorted_routes=None, expert_offsets=None, stream=None):
    """A tensor-parallel rank's share of the layer (see include/moe_decode.h):
    m_out (float32 [M, H]) = the weighted finalize of this rank's shard."""
    w = _Weights(*[_ptr(weights.get(n, weights.get("gain") if n == "norm_gain" else None))
                   for n in _WEIGHT_FIELDS])
    rc = lib().moe_decode_layer_partial(ctypes.byref(_dims(dims)), ctypes.byref(w), int(x.shape[0]), _ptr(x),
                                        _ptr(m_out), _ptr(topk_ids), _ptr(topk_w), _ptr(sorted_routes),
                                        _ptr(expert_offsets), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "moe_decode_layer_partial")


def moe_tp_boundary(partials, residual, gain, out, residual_out, eps: float, stream=None):
    """The boundary over G partial sums (float32 [G, M, H]): their sum plus the
    residual, then RMSNorm with the gain."""
    G, M, H = partials.shape
    rc = lib().moe_tp_boundary(_ptr(partials), int(G), _ptr(residual), _ptr(gain), int(M), int(H), float(eps),
                               _ptr(out), _ptr(residual_out), _stream(stream))
    _check(rc, "moe_tp_boundary")


def splitk_gemm_workspace_size(M: int, N: int, K: int, split_k: int = 0) -> int:
    n = _sz(0)
    _check(lib().splitk_gemm_workspace_size(int(M), int(N), int(K), int(split_k), ctypes.byref(n)),
           "splitk_gemm_workspace_size")
    return n.value


def splitk_gemm_bf16(A, W, C, workspace, alpha: float = 1.0, split_k: int = 0, stream=None):
    """C = alpha * A . W^T; C's dtype (bf16 or float32) selects the output form.
    split_k = 0 lets the library divide K over the whole GPU; S > 0 cuts every
    64-row tile into S K-segments (the workspace must be sized for that S)."""
    import torch
    M, K = A.shape
    N = W.shape[0]
    rc = lib().splitk_gemm_bf16(_ptr(A), _ptr(W), _ptr(C), 1 if C.dtype == torch.float32 else 0, M, N, K,
                                int(split_k), float(alpha), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "splitk_gemm_bf16")


def splitk_gemm_bf16_noalloc(A, W, C, alpha: float = 1.0, split_k: int = 0, stream=None):
    """splitk_gemm_bf16 with the library's static scratch instead of a caller
    workspace, for callers that cannot allocate device memory where they run
    the projection.  Calls that may overlap on the GPU must not share it."""
    import torch
    M, K = A.shape
    N = W.shape[0]
    rc = lib().splitk_gemm_bf16_noalloc(_ptr(A), _ptr(W), _ptr(C), 1 if C.dtype == torch.float32 else 0, M, N, K,
                                        int(split_k), float(alpha), _stream(stream))
    _check(rc, "splitk_gemm_bf16_noalloc")


def moe_debug_fill_noalloc_scratch(byte: int, stream=None):
    """Test hook: fill the no-allocation entry point's static scratch with `byte`."""
    _check(lib().moe_debug_fill_noalloc_scratch(int(byte), _stream(stream)), "moe_debug_fill_noalloc_scratch")


def mtp_eh_front_workspace_size(M: int, H: int) -> int:
    n = _sz(0)
    _check(lib().mtp_eh_front_workspace_size(int(M), int(H), ctypes.byref(n)), "mtp_eh_front_workspace_size")
    return n.value


def mtp_eh_front(input_ids, embed, hidden, enorm, hnorm, eps: float, eh_proj_w, out, workspace, stream=None):
    """out = [enorm(embed[input_ids]) | hnorm(hidden)] . eh_proj_w^T (the MTP
    layer's input projection); the concatenated input stays in the workspace
    at byte offset 256 as bf16 [M, 2H]."""
    M, H = hidden.shape
    rc = lib().mtp_eh_front(_ptr(input_ids), _ptr(embed), int(embed.shape[0]), _ptr(hidden), _ptr(enorm),
                            _ptr(hnorm), float(eps), _ptr(eh_proj_w), M, H, _ptr(out), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mtp_eh_front")


def rmsnorm_residual(residual, gain, out, residual_out, eps: float, x=None, rows=None, route_w=None,
                     shared=None, stream=None):
    M, H = residual.shape
    k = int(route_w.shape[1]) if route_w is not None else 0
    rc = lib().rmsnorm_residual(_ptr(x), _ptr(residual), _ptr(gain), M, H, float(eps), _ptr(rows),
                                _ptr(route_w), k, _ptr(shared), _ptr(out), _ptr(residual_out),
                                _stream(stream))
    _check(rc, "rmsnorm_residual")


def moe_decode_layer_plan(dims: LayerDims, M: int):
    """(expert kernel path, kernels launched) of a moe_decode_layer call of M tokens."""
    path, n = _i(0), _i(0)
    _check(lib().moe_decode_layer_plan(ctypes.byref(_dims(dims)), int(M), ctypes.byref(path), ctypes.byref(n)),
           "moe_decode_layer_plan")
    return path.value, n.value


def moe_set_expert_path(path: int):
    """Force the expert kernel of later calls (MOE_PATH_AUTO: the library's choice)."""
    _check(lib().moe_set_expert_path(int(path)), "moe_set_expert_path")


def moe_device_status(workspace, stream=None) -> int:
    return lib().moe_device_status(_ptr(workspace), _stream(stream))


def moe_debug_set_fault(workspace, fault: int, stream=None):
    _check(lib().moe_debug_set_fault(_ptr(workspace), int(fault), _stream(stream)), "moe_debug_set_fault")


class MoeDecodeLayer:
    """One MoE layer's weights (a dict of CUDA tensors) plus a zeroed workspace
    for up to max_tokens tokens."""

    def __init__(self, dims: LayerDims, weights: dict, max_tokens: int, device="cuda"):
        import torch
        self.dims = dims
        self.weights = weights
        self.max_tokens = int(max_tokens)
        n = moe_decode_workspace_size(dims, self.max_tokens)
        self.workspace = torch.empty(n, dtype=torch.uint8, device=device)
        moe_workspace_init(self.workspace)

    def __call__(self, x, residual, out=None, residual_out=None, topk_ids=None, topk_w=None,
                 sorted_routes=None, expert_offsets=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(x)
        if residual_out is None:
            residual_out = torch.empty_like(residual)
        moe_decode_layer(self.dims, self.weights, x, residual, out, residual_out, self.workspace,
                         topk_ids, topk_w, sorted_routes, expert_offsets, stream)
        return out, residual_out

    def status(self) -> int:
        return moe_device_status(self.workspace)
