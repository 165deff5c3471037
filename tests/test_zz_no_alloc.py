"""bitlinear_forward_noalloc: the forward for callers that cannot allocate device
memory when they call it (a serving engine's fixed pool, a plugin that may only
touch the tensors it is given, code that must not let cudaMalloc/cudaFree
synchronise the device).  Its scratch is a fixed array inside the library, so
its results must equal bitlinear_forward's with a caller-provided workspace.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.  It passes on its own in a
fresh process (the first call looks the scratch address up) and after the rest.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

REL_TOL = 1e-6


@pytest.fixture(scope="module")
def lib():
    from w1_a8_bitlinear_02_b300 import build, capi
    build.build()
    return capi.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """Checked on the host before anything is enqueued (no GPU needed)."""
    from w1_a8_bitlinear_02_b300 import capi
    fake = ctypes.c_void_p(0x10000)
    need = ctypes.c_size_t()
    assert lib.bitlinear_workspace_bytes(2048, 6912, 2560, ctypes.byref(need)) == 0
    assert need.value > 8 << 20
    st = lib.bitlinear_forward_noalloc(fake, fake, 6912, 2560, fake, capi.BL_BF16, 2048, fake, None)
    assert st == capi.BL_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(65, 2560, 2560), (130, 384, 1000), (200, 640, 512),
                                   (17, 384, 1000), (32, 2560, 2560), (33, 384, 1000),
                                   (64, 2560, 2560)])
def test_noalloc_matches_forward_twice(lib, M, N, K):
    """Two calls in a row through the C ABI: each result equals bitlinear_forward's
    (with a caller workspace) bit for bit, and the CPU oracle's."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    import w1_a8_bitlinear_02_b300 as bl
    from w1_a8_bitlinear_02_b300 import capi
    from w1_a8_bitlinear_02_b300 import workloads as wl
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    need = ctypes.c_size_t()
    assert lib.bitlinear_workspace_bytes(M, N, K, ctypes.byref(need)) == 0
    # M > 64 (tensor-core GEMM) uses the scratch; these few-token shapes run on
    # the few-token kernel (one wave of clusters), which needs none
    assert need.value <= 8 << 20
    assert (need.value > 0) == (M > 64)
    W = wl.weight(N, K, 0.02, 7 * N + K, "cpu")
    packed, gamma = bl.bitlinear_pack_weights(W.to(dev))
    p_ref, g_ref = oracle.pack_weights(W.numpy())
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    ws = torch.empty(max(need.value, 1), dtype=torch.uint8, device=dev)
    for call in range(2):  # two calls in a row share (and reuse) the fixed scratch
        xh = wl.activations(M, K, "outliers1pct", 100 * call + M, "cpu", torch.bfloat16)
        x = xh.to(dev)
        y_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert lib.bitlinear_forward(_ptr(packed), _ptr(gamma), N, K, _ptr(x), capi.BL_BF16, M,
                                     _ptr(y_ref), _ptr(ws), need.value, stream) == capi.BL_OK
        assert lib.bitlinear_forward_noalloc(_ptr(packed), _ptr(gamma), N, K, _ptr(x), capi.BL_BF16,
                                             M, _ptr(y), stream) == capi.BL_OK
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        got, ref = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= REL_TOL * np.abs(ref)).all(), f"call {call}"
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {call}"
        want = oracle.forward_packed(p_ref, g_ref, N, K, xh.float().numpy())
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f"call {call} vs oracle"
