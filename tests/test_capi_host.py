"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, sizes and the path planner behave, and invalid arguments
come back as status codes before anything touches a device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitlinear.h")


@pytest.fixture(scope="module")
def lib():
    from w1_a8_bitlinear_02_b300 import build, capi
    build.build()
    return capi.load()


def header_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BL_API[^;(]*?\b(bitlinear_\w+)\s*\(", text, re.S)))


def test_header_declares_the_api():
    syms = header_symbols()
    for name in ("bitlinear_pack_weights", "bitlinear_quant_act", "bitlinear_rmsnorm_quant_act",
                 "bitlinear_forward", "bitlinear_forward_q", "bitlinear_matmul_i32",
                 "bitlinear_workspace_bytes", "bitlinear_device_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from w1_a8_bitlinear_02_b300 import capi
    for name in header_symbols():
        assert hasattr(lib, name), name
        assert name in capi.SIGNATURES, f"{name} has no ctypes declaration"
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (bitlinear_\w+)", out))
    assert exported == set(header_symbols())


def test_library_targets_sm103a_only(lib):
    from w1_a8_bitlinear_02_b300 import capi
    out = subprocess.run(["/usr/local/cuda/bin/cuobjdump", "--list-elf", capi.LIB_PATH],
                         capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    arches = set(re.findall(r"sm_\w+", out.stdout))
    assert arches == {"sm_103a"}, arches


def test_version_and_status_strings(lib):
    assert lib.bitlinear_version() >= 100
    for s in range(9):
        assert lib.bitlinear_status_string(s)
    assert lib.bitlinear_status_string(99) == b"unknown status"


def test_row_bytes_and_sizes(lib):
    import w1_a8_bitlinear_02_b300 as bl
    assert bl.packed_row_bytes(1) == 16
    assert bl.packed_row_bytes(64) == 16
    assert bl.packed_row_bytes(65) == 32
    assert bl.packed_row_bytes(2560) == 640
    assert bl.packed_bytes(3840, 2560) == 3840 * 640
    assert bl.pack_workspace_bytes(100, 7) == 800
    # 30 layers of the ~2B shapes: 388 MB of packed weights
    tot = 30 * sum(bl.packed_bytes(n, k) for n, k in
                   ((3840, 2560), (2560, 2560), (6912, 2560), (2560, 6912)))
    assert tot == 388_300_800


def test_workspace_plan(lib):
    import w1_a8_bitlinear_02_b300 as bl
    # decode (M <= 4, GEMV) and batched decode (the few-token tensor-core
    # kernel, which quantises in shared memory, when its clusters cover the
    # weights in one wave of blocks) need no workspace
    for M in (1, 2, 3, 4, 8, 9, 16, 32, 33, 64):
        for N, K in ((2560, 6912), (3840, 2560), (6912, 2560), (2560, 2560)):
            if N == 6912 and M > 32:
                continue
            assert bl.workspace_bytes(M, N, K) == 0, (M, N, K)
    for M in (1, 2, 3, 4):
        assert bl.workspace_bytes(M, 28672, 8192) == 0, M
    for M in (1, 2):
        assert bl.workspace_bytes(M, 8192, 28672) == 0, M
    # more blocks than one wave (54 row tiles x 3 blocks at 33-64 tokens on
    # 6912 x 2560; the ~100B shapes from five tokens, 8192 x 28672 from three)
    # take the GEMM with its bf16 code buffer and scales
    for M, N, K in ((33, 6912, 2560), (64, 6912, 2560), (5, 28672, 8192), (64, 28672, 8192),
                    (3, 8192, 28672), (8, 8192, 28672)):
        need = bl.workspace_bytes(M, N, K)
        assert need >= M * bl.packed_row_bytes(K) * 4 * 2 + 4 * M, (M, N, K)
    # prefill (tensor-core GEMM) needs the bf16 code buffer and scales at least
    for M, N, K in ((65, 256, 512), (130, 2560, 2560), (2048, 6912, 2560), (2048, 2560, 6912)):
        need = bl.workspace_bytes(M, N, K)
        assert need >= M * bl.packed_row_bytes(K) * 4 * 2 + 4 * M
    # M = 1 with a K too large to hold in registers also takes the tensor-core path
    assert bl.workspace_bytes(1, 128, 131072) > 0


def test_invalid_arguments_return_status(lib):
    from w1_a8_bitlinear_02_b300 import capi
    sz = ctypes.c_size_t()
    i64 = ctypes.c_int64()
    assert lib.bitlinear_packed_bytes(1, 1, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_packed_row_bytes(0, ctypes.byref(i64)) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_packed_row_bytes(131073, ctypes.byref(i64)) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_workspace_bytes(0, 4, 4, ctypes.byref(sz)) == capi.BL_ERR_SHAPE
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: checks run first
    odd = ctypes.c_void_p(0x10008)
    # forward: NULL, shape, dtype, alignment
    assert lib.bitlinear_forward(None, fake, 4, 4, fake, 0, 1, fake, None, 0, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_forward(fake, fake, 4, 4, fake, 7, 1, fake, None, 0, None) == capi.BL_ERR_DTYPE
    assert lib.bitlinear_forward(fake, fake, 4, 0, fake, 0, 1, fake, None, 0, None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward(fake, fake, 4, 4, fake, 0, 0, fake, None, 0, None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward(odd, fake, 4, 4, fake, 0, 1, fake, None, 0, None) == capi.BL_ERR_ALIGN
    assert lib.bitlinear_forward_q(fake, fake, 4, 4, fake, None, 1, fake, None, 0, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_matmul_i32(fake, 4, 4, fake, 1, None, None, 0, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_quant_act(fake, 2, 1, 4, fake, fake, None) == capi.BL_ERR_DTYPE
    assert lib.bitlinear_rmsnorm_quant_act(fake, 0, None, ctypes.c_float(-1.0), 1, 4, fake, fake,
                                           None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_pack_weights(fake, 0, 4, 4, fake, fake, None, 0, None) == capi.BL_ERR_WORKSPACE
    assert lib.bitlinear_pack_weights(fake, 0, 4, 4, odd, fake, fake, 32, None) == capi.BL_ERR_ALIGN
    # grouped scales: group_rows must be a power of two dividing N
    for G in (0, 3, 8, -4):
        assert lib.bitlinear_pack_weights_grouped(fake, 0, 4, 4, G, fake, fake, fake, 32,
                                                  None) == capi.BL_ERR_SHAPE, G
        assert lib.bitlinear_forward_grouped(fake, fake, G, 4, 4, fake, 0, 1, 0, fake, 0, None, None, 0,
                                             None) == capi.BL_ERR_SHAPE, G
    assert lib.bitlinear_pack_weights_grouped(fake, 0, 4, 4, 2, fake, fake, None, 0,
                                              None) == capi.BL_ERR_WORKSPACE
    assert lib.bitlinear_forward_grouped(fake, None, 2, 4, 4, fake, 0, 1, 0, fake, 0, None, None, 0,
                                         None) == capi.BL_ERR_NULL
    assert lib.bitlinear_forward_grouped(fake, ctypes.c_void_p(0x10002), 2, 4, 4, fake, 0, 1, 0, fake, 0, None,
                                         None, 0, None) == capi.BL_ERR_ALIGN


def test_grid_limits_are_checked_before_launch(lib):
    """A token count whose GEMM grid would need more than 65535 token tiles is
    refused as a shape error, by the size query and by the forward, before
    anything is enqueued (fake pointers, never dereferenced)."""
    from w1_a8_bitlinear_02_b300 import capi
    sz = ctypes.c_size_t()
    fake = ctypes.c_void_p(0x10000)
    M = 20_000_000  # 78125 tiles of 256 tokens
    assert lib.bitlinear_workspace_bytes(M, 64, 64, ctypes.byref(sz)) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward(fake, fake, 64, 64, fake, capi.BL_BF16, M, fake, fake, 1 << 40,
                                 None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward_noalloc(fake, fake, 64, 64, fake, capi.BL_BF16, M, fake,
                                         None) == capi.BL_ERR_SHAPE
    # 65535 tiles of 256 tokens still plan
    assert lib.bitlinear_workspace_bytes(65535 * 256, 64, 64, ctypes.byref(sz)) == capi.BL_OK


def test_no_device_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from w1_a8_bitlinear_02_b300 import capi
    fake = ctypes.c_void_p(0x10000)
    st = lib.bitlinear_forward(fake, fake, 4, 4, fake, 0, 1, fake, None, 0, None)
    assert st in (capi.BL_ERR_CUDA, capi.BL_ERR_UNSUPPORTED)


def test_launch_overlap_switch(lib):
    import w1_a8_bitlinear_02_b300 as bl
    before = bl.get_launch_overlap()
    bl.set_launch_overlap(True)
    assert bl.get_launch_overlap()
    bl.set_launch_overlap(False)
    assert not bl.get_launch_overlap()
    bl.set_launch_overlap(before)


def test_chain_invalid_arguments_return_status(lib):
    """bitlinear_forward_chain checks every descriptor before touching the device."""
    from w1_a8_bitlinear_02_b300 import capi
    fake, odd = 0x10000, 0x10008  # never dereferenced
    ws = ctypes.c_void_p(fake)

    def chain(**kw):
        d = dict(packed=fake, gamma=fake, x=fake, y=fake, N=64, K=64, x_dtype=capi.BL_BF16,
                 act=capi.BL_ACT_NONE, wait_prev=1, M=1)
        d.update(kw)
        arr = (capi.ChainCall * 1)(capi.ChainCall(d["packed"], d["gamma"], d["x"], d["y"], d["N"],
                                                  d["K"], d["x_dtype"], d["act"], d["wait_prev"], d["M"]))
        return ctypes.cast(arr, ctypes.c_void_p), arr

    p, keep = chain(y=0x900000)
    assert lib.bitlinear_forward_chain(None, 1, ws, 256, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_forward_chain(p, 1, None, 256, None) == capi.BL_ERR_NULL
    assert lib.bitlinear_forward_chain(p, 0, ws, 256, None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward_chain(p, 241, ws, 256, None) == capi.BL_ERR_SHAPE
    assert lib.bitlinear_forward_chain(p, 1, ws, 255, None) == capi.BL_ERR_WORKSPACE
    assert lib.bitlinear_forward_chain(p, 1, ctypes.c_void_p(odd), 256, None) == capi.BL_ERR_ALIGN
    for kw, want in ((dict(y=0), capi.BL_ERR_NULL), (dict(K=32769), capi.BL_ERR_SHAPE),
                     (dict(N=0), capi.BL_ERR_SHAPE), (dict(x_dtype=7), capi.BL_ERR_DTYPE),
                     (dict(act=5), capi.BL_ERR_SHAPE), (dict(packed=odd), capi.BL_ERR_ALIGN),
                     (dict(y=fake + 64), capi.BL_ERR_SHAPE),  # y over its own x
                     (dict(M=17), capi.BL_ERR_SHAPE)):
        kw.setdefault("y", 0x900000)
        p2, keep2 = chain(**kw)
        assert lib.bitlinear_forward_chain(p2, 1, ws, 256, None) == want, kw


def _chain_record_bytes(K, M):
    """A record as the header describes it: a header (128 bytes for one token,
    64 + 64 M rounded up to 128 for more), then M x 64 code bytes per piece of
    every slab.  A row of ceil(K/64) pieces takes the fewest slabs of at most
    65 (one token), 31 (2-8) or 23 (9-16) pieces, split evenly, with an odd
    piece count per slab."""
    M = max(M, 1)
    pieces = -(-K // 64)
    cap = 65 if M == 1 else (31 if M <= 8 else 23)
    ns = -(-pieces // cap)
    P = -(-pieces // ns) | 1
    slabs = -(-pieces // P)
    assert P % 2 == 1 and P <= cap and slabs * P >= pieces and (slabs - 1) * cap < pieces
    head = 128 if M == 1 else -(-(64 + 64 * M) // 128) * 128
    return head + slabs * M * 64 * P


def test_chain_workspace_layout(lib):
    """bitlinear_chain_workspace_bytes adds up the parts its header lists: the
    control words, the call table, a record per call quantised before the chain
    and the output words of every call a later call reads -- and nothing for a
    call that waits or reads an earlier output."""
    from w1_a8_bitlinear_02_b300 import capi
    al = lambda b: -(-b // 256) * 256
    nxt = [0x10000000]

    def region(nbytes):  # disjoint fake device ranges, never dereferenced
        a = nxt[0]
        nxt[0] += al(nbytes) + 4096
        return a

    def call(N, K, M=1, x=None, dt=capi.BL_BF16, wait=0):
        M1 = max(M, 1)
        return capi.ChainCall(region(N * 16 * -(-K // 64)), region(4),
                              x if x is not None else region(M1 * K * 4), region(M1 * N * 4),
                              N, K, dt, capi.BL_ACT_NONE, wait, M)

    def need(calls):
        arr = (capi.ChainCall * len(calls))(*calls)
        sz = ctypes.c_size_t(0)
        st = lib.bitlinear_chain_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(calls), ctypes.byref(sz))
        return st, sz.value

    base = lambda n: 256 + al(88 * n)

    # independent calls of every token class, ragged and maximal K
    shapes = [(2560, 2560, 1), (6912, 2560, 0), (2560, 6912, 1), (640, 1000, 1), (64, 64, 1),
              (128, 32768, 1), (8192, 8192, 2), (28672, 8192, 8), (8192, 28672, 9),
              (333, 4160, 16), (777, 63, 4), (4096, 4095, 12)]
    calls = [call(N, K, M) for N, K, M in shapes]
    assert need(calls) == (capi.BL_OK, base(len(calls)) + sum(al(_chain_record_bytes(K, M)) for _, K, M in shapes))
    for N, K, M in shapes:
        assert _chain_record_bytes(K, M) >= max(M, 1) * K + 128

    # a dataflow chain: call 1 reads call 0's fp32 y, call 2 reads call 1's
    c0 = call(2560, 2560)
    c1 = call(6912, 2560, x=c0.y, dt=capi.BL_F32)
    c2 = call(2560, 6912, x=c1.y, dt=capi.BL_F32)
    assert need([c0, c1, c2]) == (capi.BL_OK, base(3) + al(_chain_record_bytes(2560, 1)) + al(8 * 2560) + al(8 * 6912))
    # a row inside a larger output still takes output words (offset x, shorter K)
    c3 = call(640, 1024, x=c1.y + 4 * 512, dt=capi.BL_F32)
    assert need([c0, c1, c3]) == (capi.BL_OK, base(3) + al(_chain_record_bytes(2560, 1)) + al(8 * 2560) + al(8 * 6912))

    # bf16 x over an earlier output, and wait_prev: a barrier, no record and no output words
    d0 = call(2560, 2560)
    d1 = call(2560, 1280, x=d0.y, dt=capi.BL_BF16)
    assert need([d0, d1]) == (capi.BL_OK, base(2) + al(_chain_record_bytes(2560, 1)))
    e0, e1 = call(2560, 2560), call(1024, 2560, wait=1)
    assert need([e0, e1]) == (capi.BL_OK, base(2) + al(_chain_record_bytes(2560, 1)))

    # several tokens whose x an earlier call writes: refused
    f0 = call(2560, 2560)
    f1 = call(640, 1280, M=2, x=f0.y, dt=capi.BL_F32)
    assert need([f0, f1])[0] == capi.BL_ERR_SHAPE
