"""CPU oracle for the BitLinear W1.58A8 forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product (``w1_a8_bitlinear_02_b300``) never
does, and the two share no code.

The arithmetic lives in ``bitlinear_oracle.c`` (plain C loops, one IEEE fp32
operation per step, fp64 where the definitions sum long series); this module
only builds it with gcc and marshals numpy arrays through ctypes.  Every
function documents the passage of the BitNet b1.58 pages it restates; see the
C file's header for the page titles.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlinear_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# No fast-math and no FMA contraction: each C expression is one IEEE op.
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
          "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    F = ctypes.c_float
    lib.bl_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.bl_oracle_get_threads.restype = ctypes.c_int
    lib.bl_oracle_row_bytes.argtypes = [I64]
    lib.bl_oracle_row_bytes.restype = I64
    lib.bl_oracle_abs_sum.argtypes = [P, I64, I64]
    lib.bl_oracle_abs_sum.restype = ctypes.c_double
    lib.bl_oracle_gamma.argtypes = [P, I64, I64]
    lib.bl_oracle_gamma.restype = F
    lib.bl_oracle_ternarize.argtypes = [P, I64, I64, F, P]
    lib.bl_oracle_pack.argtypes = [P, I64, I64, P]
    lib.bl_oracle_unpack.argtypes = [P, I64, I64, P]
    lib.bl_oracle_quant_act.argtypes = [P, I64, I64, P, P]
    lib.bl_oracle_relu2.argtypes = [P, I64, P]
    lib.bl_oracle_output.argtypes = [P, P, I64, ctypes.c_int, P, P]
    lib.bl_oracle_matmul_i32.argtypes = [P, P, I64, I64, I64, P]
    lib.bl_oracle_rescale.argtypes = [P, F, P, I64, I64, P]
    lib.bl_oracle_forward_packed.argtypes = [P, F, I64, I64, P, I64, P, P, P, P]
    lib.bl_oracle_rmsnorm_quant_act.argtypes = [P, P, F, I64, I64, P, P, P, P]
    lib.bl_oracle_gamma_groups.argtypes = [P, I64, I64, I64, P]
    lib.bl_oracle_ternarize_groups.argtypes = [P, I64, I64, I64, P, P]
    lib.bl_oracle_rescale_groups.argtypes = [P, P, I64, P, I64, I64, P]
    _lib = lib
    return lib


def _f32(a) -> np.ndarray:
    """fp32, C-contiguous.  bf16 inputs must already be widened (exactly) by
    the caller; float64 inputs are rejected so no silent rounding happens."""
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle expects float32 input, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def set_threads(n: int) -> None:
    _load().bl_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().bl_oracle_get_threads())


def row_bytes(K: int) -> int:
    """Bytes of one packed row: K rounded up to 64 weights, 2 bits each."""
    return int(_load().bl_oracle_row_bytes(int(K)))


def abs_sum(W) -> float:
    """fp64 sum of |W| in the fixed order row-major-within-row, then rows."""
    W = _f32(W)
    N, K = W.shape
    return float(_load().bl_oracle_abs_sum(_ptr(W), N, K))


def gamma(W) -> np.float32:
    """Per-tensor weight scale mean|W| + 1e-5 (absmean), as fp32."""
    W = _f32(W)
    N, K = W.shape
    return np.float32(_load().bl_oracle_gamma(_ptr(W), N, K))


def ternarize(W, g) -> np.ndarray:
    """clip(rne(fl32(W / gamma)), -1, 1) as int8 [N, K]."""
    W = _f32(W)
    N, K = W.shape
    q = np.empty((N, K), np.int8)
    _load().bl_oracle_ternarize(_ptr(W), N, K, ctypes.c_float(float(g)), _ptr(q))
    return q


def pack(q) -> np.ndarray:
    """Ternary int8 [N, K] -> packed uint8 [N, row_bytes(K)]."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    N, K = q.shape
    out = np.empty((N, row_bytes(K)), np.uint8)
    _load().bl_oracle_pack(_ptr(q), N, K, _ptr(out))
    return out


def unpack(packed, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    if packed.shape[1] != row_bytes(K):
        raise ValueError("packed row length does not match K")
    q = np.empty((N, K), np.int8)
    _load().bl_oracle_unpack(_ptr(packed), N, K, _ptr(q))
    return q


def pack_weights(W):
    """W fp32 [N, K] -> (packed uint8 [N, row_bytes(K)], gamma fp32)."""
    g = gamma(W)
    return pack(ternarize(W, g)), g


def quant_act(x):
    """x fp32 [M, K] -> (xq int8 [M, K], s fp32 [M]) per-token absmax."""
    x = _f32(x)
    M, K = x.shape
    xq = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().bl_oracle_quant_act(_ptr(x), M, K, _ptr(xq), _ptr(s))
    return xq, s


def relu2(x) -> np.ndarray:
    """Squared ReLU, elementwise: u = fl32(max(x, 0)^2)."""
    x = _f32(x)
    u = np.empty_like(x)
    _load().bl_oracle_relu2(_ptr(x), x.size, _ptr(u))
    return u


def relu2_quant_act(x):
    """Per-token absmax quantisation of relu2(x) -> (xq, s)."""
    return quant_act(relu2(x))


def forward_packed_relu2(packed, gamma: float, N: int, K: int, x) -> np.ndarray:
    """BitLinear forward of relu2(x) (the down projection of a ReLU^2 FFN)."""
    return forward_packed(packed, gamma, N, K, relu2(x))


def output(y, residual=None, bf16: bool = False) -> np.ndarray:
    """Forward output variants: fl32(y + residual) (residual fp32 values, e.g.
    widened bf16), then one RNE rounding to bf16 when bf16 (returned as the
    uint16 bit patterns); otherwise fp32."""
    y = _f32(y)
    r = None if residual is None else _f32(residual).reshape(y.shape)
    out_f = np.empty_like(y)
    out_b = np.empty(y.shape, np.uint16)
    _load().bl_oracle_output(_ptr(y), None if r is None else _ptr(r), y.size, 1 if bf16 else 0,
                             _ptr(out_f), _ptr(out_b))
    return out_b if bf16 else out_f


def matmul_i32(q, xq) -> np.ndarray:
    """acc[m, n] = sum_k q[n, k] * xq[m, k] (int32, exact)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    N, K = q.shape
    M, K2 = xq.shape
    if K != K2:
        raise ValueError("K mismatch")
    acc = np.empty((M, N), np.int32)
    _load().bl_oracle_matmul_i32(_ptr(q), _ptr(xq), M, N, K, _ptr(acc))
    return acc


def rescale(acc, g, s) -> np.ndarray:
    """y = fl32(float(acc) * fl32(gamma / s_m))."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M, N = acc.shape
    y = np.empty((M, N), np.float32)
    _load().bl_oracle_rescale(_ptr(acc), ctypes.c_float(float(g)), _ptr(s), M, N,
                              _ptr(y))
    return y


def forward_packed(packed, g, N: int, K: int, x) -> np.ndarray:
    """Whole forward from packed weights: quant x, unpack, contract, rescale."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.shape != (N, row_bytes(K)):
        raise ValueError("packed shape does not match (N, row_bytes(K))")
    x = _f32(x)
    M = x.shape[0]
    y = np.empty((M, N), np.float32)
    xq = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    acc = np.empty((M, N), np.int32)
    _load().bl_oracle_forward_packed(_ptr(packed), ctypes.c_float(float(g)), N, K,
                                     _ptr(x), M, _ptr(y), _ptr(xq), _ptr(s),
                                     _ptr(acc))
    return y


def forward(W, x):
    """Reference BitLinear forward from fp32 weights: returns (y, packed, gamma)."""
    packed, g = pack_weights(W)
    N, K = np.asarray(W).shape
    return forward_packed(packed, g, N, K, x), packed, g


def _check_groups(N: int, G: int) -> None:
    if G < 1 or N % G:
        raise ValueError("group_rows must be >= 1 and divide N")


def gamma_groups(W, G: int) -> np.ndarray:
    """One absmean scale per group of G consecutive output rows:
    gamma_g = fl32(fl32(S_g / (G*K)) + 1e-5), S_g the fp64 |W| sum of the
    group's rows (row sums in row order), fp32 [N / G]."""
    W = _f32(W)
    N, K = W.shape
    _check_groups(N, G)
    g = np.empty((N // G,), np.float32)
    _load().bl_oracle_gamma_groups(_ptr(W), N, K, G, _ptr(g))
    return g


def ternarize_groups(W, g, G: int) -> np.ndarray:
    """clip(rne(fl32(W[n] / gamma_{n / G})), -1, 1) as int8 [N, K]."""
    W = _f32(W)
    N, K = W.shape
    _check_groups(N, G)
    g = np.ascontiguousarray(g, dtype=np.float32)
    q = np.empty((N, K), np.int8)
    _load().bl_oracle_ternarize_groups(_ptr(W), N, K, G, _ptr(g), _ptr(q))
    return q


def pack_weights_groups(W, G: int):
    """W fp32 [N, K] -> (packed uint8 [N, row_bytes(K)], gamma fp32 [N / G])."""
    g = gamma_groups(W, G)
    return pack(ternarize_groups(W, g, G)), g


def rescale_groups(acc, g, G: int, s) -> np.ndarray:
    """y[m, n] = fl32(float(acc[m, n]) * fl32(gamma_{n / G} / s_m))."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    M, N = acc.shape
    _check_groups(N, G)
    y = np.empty((M, N), np.float32)
    _load().bl_oracle_rescale_groups(_ptr(acc), _ptr(g), G, _ptr(s), M, N, _ptr(y))
    return y


def forward_packed_groups(packed, g, G: int, N: int, K: int, x) -> np.ndarray:
    """Forward with grouped weight scales: quant x, unpack, contract, rescale
    each output row by its group's scale."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.shape != (N, row_bytes(K)):
        raise ValueError("packed shape does not match (N, row_bytes(K))")
    xq, s = quant_act(x)
    return rescale_groups(matmul_i32(unpack(packed, K), xq), g, G, s)


def rmsnorm_quant_act(x, gain=None, eps: float = 1e-5):
    """Fused subln RMSNorm + per-token absmax quant -> (xq, s, r)."""
    x = _f32(x)
    M, K = x.shape
    g = None if gain is None else _f32(gain).reshape(K)
    xq = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    r = np.empty((M,), np.float32)
    u = np.empty((K,), np.float32)
    _load().bl_oracle_rmsnorm_quant_act(
        _ptr(x), None if g is None else _ptr(g), ctypes.c_float(eps), M, K,
        _ptr(xq), _ptr(s), _ptr(r), _ptr(u))
    return xq, s, r
