"""BitLinear W1.58A8 forward for NVIDIA B300 (sm_103a).

Thin torch-facing binding over the C ABI in ``include/bitlinear.h``
(``libbitlinear.so``): it checks tensor devices, dtypes and layouts,
allocates outputs and workspaces with torch, and passes raw pointers and the
current CUDA stream to the library.  Every step of the computation runs in
the library's CUDA kernels.

    packed, gamma = bitlinear_pack_weights(W)            # W [N, K] fp32/bf16
    y = bitlinear_forward(packed, gamma, N, K, x)        # x [M, K] -> y [M, N] fp32
    xq, s = bitlinear_quant_act(x)                       # per-token int8 codes
    xq, s = bitlinear_rmsnorm_quant_act(x, g, eps)       # fused subln RMSNorm
    y = bitlinear_forward_q(packed, gamma, N, K, xq, s)
    acc = bitlinear_matmul_i32(packed, N, K, xq)         # exact int32 sums
"""
from __future__ import annotations

import ctypes

import torch

from . import capi
from .capi import BitLinearError

__all__ = [
    "BitLinearError", "BitLinear", "packed_row_bytes", "packed_bytes",
    "pack_workspace_bytes", "workspace_bytes", "bitlinear_pack_weights",
    "bitlinear_pack_weights_grouped", "bitlinear_quant_act", "bitlinear_relu2_quant_act",
    "bitlinear_rmsnorm_quant_act", "bitlinear_forward", "bitlinear_forward_ex",
    "bitlinear_forward_grouped", "bitlinear_forward_relu2", "bitlinear_forward_q",
    "bitlinear_matmul_i32", "bitlinear_forward_noalloc", "bitlinear_forward_chain",
    "set_launch_overlap", "get_launch_overlap", "device_error", "library_path",
]

_DTYPES = {torch.float32: capi.BL_F32, torch.bfloat16: capi.BL_BF16}


def library_path() -> str:
    capi.load()
    return capi.LIB_PATH


def _lib():
    return capi.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need_cuda(name: str, t: torch.Tensor, dtype=None, dim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name}: dtype {t.dtype} not supported")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must be {dim}-D")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------- sizes
def packed_row_bytes(K: int) -> int:
    out = ctypes.c_int64()
    capi.check(_lib().bitlinear_packed_row_bytes(K, ctypes.byref(out)), "packed_row_bytes")
    return out.value


def packed_bytes(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    capi.check(_lib().bitlinear_packed_bytes(N, K, ctypes.byref(out)), "packed_bytes")
    return out.value


def pack_workspace_bytes(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    capi.check(_lib().bitlinear_pack_workspace_bytes(N, K, ctypes.byref(out)),
               "pack_workspace_bytes")
    return out.value


def workspace_bytes(M: int, N: int, K: int) -> int:
    out = ctypes.c_size_t()
    capi.check(_lib().bitlinear_workspace_bytes(M, N, K, ctypes.byref(out)), "workspace_bytes")
    return out.value


def _workspace(nbytes: int, device, given):
    if nbytes == 0:
        return None
    if given is not None:
        _need_cuda("workspace", given)
        if given.numel() * given.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- ops
def bitlinear_pack_weights(W: torch.Tensor, packed: torch.Tensor | None = None,
                           gamma: torch.Tensor | None = None):
    """Absmean-ternarise and 2-bit-pack W [N, K] -> (packed uint8 [N, row_bytes], gamma [1])."""
    _need_cuda("W", W, (torch.float32, torch.bfloat16), 2)
    N, K = W.shape
    rb = packed_row_bytes(K)
    if packed is None:
        packed = torch.empty((N, rb), dtype=torch.uint8, device=W.device)
    if gamma is None:
        gamma = torch.empty((1,), dtype=torch.float32, device=W.device)
    ws = torch.empty(pack_workspace_bytes(N, K), dtype=torch.uint8, device=W.device)
    capi.check(_lib().bitlinear_pack_weights(
        _ptr(W), _DTYPES[W.dtype], N, K, _ptr(packed), _ptr(gamma), _ptr(ws), ws.numel(),
        _stream(W)), "bitlinear_pack_weights")
    return packed, gamma


def bitlinear_pack_weights_grouped(W: torch.Tensor, group_rows: int, packed: torch.Tensor | None = None,
                                   gamma: torch.Tensor | None = None):
    """Absmean-ternarise W [N, K] with one scale per group of group_rows output
    rows (a power of two dividing N; 1 = per output channel) ->
    (packed uint8 [N, row_bytes], gamma fp32 [N / group_rows])."""
    _need_cuda("W", W, (torch.float32, torch.bfloat16), 2)
    N, K = W.shape
    rb = packed_row_bytes(K)
    if packed is None:
        packed = torch.empty((N, rb), dtype=torch.uint8, device=W.device)
    if gamma is None:
        gamma = torch.empty((max(N // max(int(group_rows), 1), 1),), dtype=torch.float32, device=W.device)
    ws = torch.empty(pack_workspace_bytes(N, K), dtype=torch.uint8, device=W.device)
    capi.check(_lib().bitlinear_pack_weights_grouped(
        _ptr(W), _DTYPES[W.dtype], N, K, int(group_rows), _ptr(packed), _ptr(gamma), _ptr(ws), ws.numel(),
        _stream(W)), "bitlinear_pack_weights_grouped")
    return packed, gamma


def bitlinear_quant_act(x: torch.Tensor, xq: torch.Tensor | None = None,
                        scale: torch.Tensor | None = None):
    """Per-token absmax int8 codes of x [M, K] -> (xq int8 [M, K], s fp32 [M])."""
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    scale = torch.empty((M,), dtype=torch.float32, device=x.device) if scale is None else scale
    capi.check(_lib().bitlinear_quant_act(_ptr(x), _DTYPES[x.dtype], M, K, _ptr(xq),
                                          _ptr(scale), _stream(x)), "bitlinear_quant_act")
    return xq, scale


def bitlinear_relu2_quant_act(x: torch.Tensor, xq: torch.Tensor | None = None,
                              scale: torch.Tensor | None = None):
    """Per-token absmax int8 codes of relu2(x) = max(x, 0)^2 -> (xq, s)."""
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    scale = torch.empty((M,), dtype=torch.float32, device=x.device) if scale is None else scale
    capi.check(_lib().bitlinear_relu2_quant_act(_ptr(x), _DTYPES[x.dtype], M, K, _ptr(xq),
                                                _ptr(scale), _stream(x)), "bitlinear_relu2_quant_act")
    return xq, scale


def bitlinear_rmsnorm_quant_act(x: torch.Tensor, g: torch.Tensor | None = None,
                                eps: float = 1e-5, xq: torch.Tensor | None = None,
                                scale: torch.Tensor | None = None):
    """Fused subln RMSNorm (gain g [K] or None) + per-token absmax int8 codes."""
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M, K = x.shape
    if g is not None:
        _need_cuda("g", g, torch.float32, 1)
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    scale = torch.empty((M,), dtype=torch.float32, device=x.device) if scale is None else scale
    capi.check(_lib().bitlinear_rmsnorm_quant_act(
        _ptr(x), _DTYPES[x.dtype], _ptr(g), ctypes.c_float(eps), M, K, _ptr(xq), _ptr(scale),
        _stream(x)), "bitlinear_rmsnorm_quant_act")
    return xq, scale


def bitlinear_forward(packed: torch.Tensor, gamma: torch.Tensor, N: int, K: int,
                      x: torch.Tensor, y: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = BitLinear(x [M, K]) with the activation quantisation fused in."""
    _need_cuda("packed", packed, torch.uint8)
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    ws = _workspace(workspace_bytes(M, N, K), x.device, workspace)
    capi.check(_lib().bitlinear_forward(
        _ptr(packed), _ptr(gamma), N, K, _ptr(x), _DTYPES[x.dtype], M, _ptr(y), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(x)), "bitlinear_forward")
    return y


def bitlinear_forward_ex(packed: torch.Tensor, gamma: torch.Tensor, N: int, K: int,
                         x: torch.Tensor, y: torch.Tensor | None = None,
                         y_dtype: torch.dtype = torch.float32, residual: torch.Tensor | None = None,
                         act: int = 0, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] (fp32 or bf16) = BitLinear(act(x)) (+ residual, which may be y itself)."""
    _need_cuda("packed", packed, torch.uint8)
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    if y is None:
        y = torch.empty((M, N), dtype=y_dtype, device=x.device)
    _need_cuda("y", y, (torch.float32, torch.bfloat16), 2)
    if residual is not None:
        _need_cuda("residual", residual, y.dtype, 2)
    ws = _workspace(workspace_bytes(M, N, K), x.device, workspace)
    capi.check(_lib().bitlinear_forward_ex(
        _ptr(packed), _ptr(gamma), N, K, _ptr(x), _DTYPES[x.dtype], M, int(act), _ptr(y),
        _DTYPES[y.dtype], _ptr(residual), _ptr(ws), 0 if ws is None else ws.numel(), _stream(x)),
        "bitlinear_forward_ex")
    return y


def bitlinear_forward_grouped(packed: torch.Tensor, gamma: torch.Tensor, group_rows: int, N: int, K: int,
                              x: torch.Tensor, y: torch.Tensor | None = None,
                              y_dtype: torch.dtype = torch.float32, residual: torch.Tensor | None = None,
                              act: int = 0, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """bitlinear_forward_ex for weights packed with one scale per group of
    group_rows output rows (gamma fp32 [N / group_rows])."""
    _need_cuda("packed", packed, torch.uint8)
    _need_cuda("gamma", gamma, torch.float32)
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    if y is None:
        y = torch.empty((M, N), dtype=y_dtype, device=x.device)
    _need_cuda("y", y, (torch.float32, torch.bfloat16), 2)
    if residual is not None:
        _need_cuda("residual", residual, y.dtype, 2)
    ws = _workspace(workspace_bytes(M, N, K), x.device, workspace)
    capi.check(_lib().bitlinear_forward_grouped(
        _ptr(packed), _ptr(gamma), int(group_rows), N, K, _ptr(x), _DTYPES[x.dtype], M, int(act), _ptr(y),
        _DTYPES[y.dtype], _ptr(residual), _ptr(ws), 0 if ws is None else ws.numel(), _stream(x)),
        "bitlinear_forward_grouped")
    return y


def bitlinear_forward_relu2(packed: torch.Tensor, gamma: torch.Tensor, N: int, K: int,
                            x: torch.Tensor, y: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 = BitLinear(relu2(x)): a ReLU^2 FFN's down projection in one call."""
    _need_cuda("packed", packed, torch.uint8)
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    ws = _workspace(workspace_bytes(M, N, K), x.device, workspace)
    capi.check(_lib().bitlinear_forward_relu2(
        _ptr(packed), _ptr(gamma), N, K, _ptr(x), _DTYPES[x.dtype], M, _ptr(y), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(x)), "bitlinear_forward_relu2")
    return y


def bitlinear_forward_q(packed: torch.Tensor, gamma: torch.Tensor, N: int, K: int,
                        xq: torch.Tensor, scale: torch.Tensor, y: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp32 from pre-quantised activations (xq int8 [M, K], scale [M])."""
    _need_cuda("xq", xq, torch.int8, 2)
    _need_cuda("scale", scale, torch.float32)
    M = xq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=xq.device) if y is None else y
    ws = _workspace(workspace_bytes(M, N, K), xq.device, workspace)
    capi.check(_lib().bitlinear_forward_q(
        _ptr(packed), _ptr(gamma), N, K, _ptr(xq), _ptr(scale), M, _ptr(y), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(xq)), "bitlinear_forward_q")
    return y


def bitlinear_matmul_i32(packed: torch.Tensor, N: int, K: int, xq: torch.Tensor,
                         acc: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact int32 acc [M, N] = Wq @ xq^T (no rescale)."""
    _need_cuda("xq", xq, torch.int8, 2)
    M = xq.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=xq.device) if acc is None else acc
    ws = _workspace(workspace_bytes(M, N, K), xq.device, workspace)
    capi.check(_lib().bitlinear_matmul_i32(
        _ptr(packed), N, K, _ptr(xq), M, _ptr(acc), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(xq)), "bitlinear_matmul_i32")
    return acc


def bitlinear_forward_noalloc(packed: torch.Tensor, gamma: torch.Tensor, N: int, K: int,
                              x: torch.Tensor, y: torch.Tensor | None = None) -> torch.Tensor:
    """bitlinear_forward without a workspace: the library's fixed 8 MiB device
    scratch stands in for it (for callers that cannot allocate at call time).
    Calls share that scratch, so calls that may overlap on the GPU must be
    ordered.  Only y is allocated here, and only when not given."""
    _need_cuda("packed", packed, torch.uint8)
    _need_cuda("x", x, (torch.float32, torch.bfloat16), 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    capi.check(_lib().bitlinear_forward_noalloc(
        _ptr(packed), _ptr(gamma), N, K, _ptr(x), _DTYPES[x.dtype], M, _ptr(y), _stream(x)),
        "bitlinear_forward_noalloc")
    return y


def _chain_array(calls):
    calls = list(calls)
    if not calls:
        raise ValueError("empty chain")
    arr = (capi.ChainCall * len(calls))()
    for i, c in enumerate(calls):
        _need_cuda("packed", c["packed"], torch.uint8)
        _need_cuda("x", c["x"], (torch.float32, torch.bfloat16))
        _need_cuda("y", c["y"], torch.float32)
        arr[i] = capi.ChainCall(c["packed"].data_ptr(), c["gamma"].data_ptr(), c["x"].data_ptr(),
                                c["y"].data_ptr(), int(c["N"]), int(c["K"]), _DTYPES[c["x"].dtype],
                                int(c.get("act", capi.BL_ACT_NONE)), int(c.get("wait_prev", 0)),
                                int(c.get("M", c["x"].shape[0] if c["x"].dim() == 2 else 1)))
    return calls, arr


def chain_workspace_bytes(calls) -> int:
    """Device bytes bitlinear_forward_chain needs for these calls."""
    calls, arr = _chain_array(calls)
    n = ctypes.c_size_t()
    capi.check(_lib().bitlinear_chain_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(calls),
                                                      ctypes.byref(n)), "bitlinear_chain_workspace_bytes")
    return int(n.value)


def chain_workspace(calls, device) -> torch.Tensor:
    """A zero-filled workspace for this chain (keep it for later launches)."""
    return torch.zeros(chain_workspace_bytes(calls), dtype=torch.uint8, device=device)


def bitlinear_forward_chain(calls, workspace: torch.Tensor | None = None) -> None:
    """A decode chain of single-token forwards in one launch.

    calls: sequence of dicts with packed, gamma, x [M, K] (fp32 / bf16, M <= 16),
    y [M, N] fp32 (written), N, K and optionally act (capi.BL_ACT_RELU2 for relu2(x))
    and wait_prev (default 0: the library orders dependent calls itself).
    workspace: from chain_workspace (zero-filled before its first use; reuse it
    across launches); allocated when None."""
    calls, arr = _chain_array(calls)
    ws = workspace if workspace is not None else chain_workspace(calls, calls[0]["x"].device)
    capi.check(_lib().bitlinear_forward_chain(ctypes.cast(arr, ctypes.c_void_p), len(calls), _ptr(ws),
                                              ws.numel(),
                                              _stream(calls[0]["x"])), "bitlinear_forward_chain")


def set_launch_overlap(mode) -> None:
    """Launch overlap for forward kernels: 0 off, 1 (or True) prefetch weights
    while the previous kernel runs, 2 independent calls (see the C header)."""
    _lib().bitlinear_set_launch_overlap(int(mode))


def get_launch_overlap() -> int:
    return int(_lib().bitlinear_get_launch_overlap())


def device_error(clear: bool = True) -> int:
    """Device-side failure flags of the current device (0 = none).  Synchronous."""
    flags = ctypes.c_uint()
    st = _lib().bitlinear_device_error(ctypes.byref(flags), 1 if clear else 0)
    if st not in (capi.BL_OK, capi.BL_ERR_DEVICE):
        capi.check(st, "device_error")
    return flags.value


class BitLinear:
    """A bias-free BitLinear layer holding packed ternary weights.

    ``BitLinear.from_weight(W)`` packs W [out, in]; calling the object on x
    [tokens, in] (fp32 or bf16) returns fp32 [tokens, out].  A workspace is
    kept and reused across calls on the same stream.
    """

    def __init__(self, packed: torch.Tensor, gamma: torch.Tensor, out_features: int,
                 in_features: int):
        self.packed, self.gamma = packed, gamma
        self.out_features, self.in_features = out_features, in_features
        self._ws = None

    @classmethod
    def from_weight(cls, W: torch.Tensor) -> "BitLinear":
        packed, gamma = bitlinear_pack_weights(W.contiguous())
        return cls(packed, gamma, W.shape[0], W.shape[1])

    def _workspace_for(self, M: int):
        need = workspace_bytes(M, self.out_features, self.in_features)
        if need and (self._ws is None or self._ws.numel() < need):
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.packed.device)
        return self._ws if need else None

    def __call__(self, x: torch.Tensor) -> torch.Tensor:
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features).contiguous()
        y = bitlinear_forward(self.packed, self.gamma, self.out_features, self.in_features, x2,
                              workspace=self._workspace_for(x2.shape[0]))
        return y.reshape(*lead, self.out_features)
