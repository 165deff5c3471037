"""GPU parity: every C-ABI entry point against the CPU oracle, element by element.

Integers (packed codes, int8 activation codes, int32 sums) must match bit for
bit.  fp32 results (gamma, scales, y) are computed on both sides with the same
single-rounding IEEE steps, so they are compared bit for bit as well; the
contract's tolerance (relative 1e-6 on fp32 outputs) is checked as the weaker
statement alongside.  The one exception is the RMSNorm scale, whose mean of
squares is summed in a different order (documented in the header): it is held
to the 1e-6 relative tolerance while its codes stay bit-exact.

Sizes span several tiles and ragged tails and run in seconds on the oracle;
the last tests use the full workload shapes, whole outputs.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from w1_a8_bitlinear_02_b300 import workloads as wl

pytestmark = pytest.mark.gpu

REL_TOL = 1e-6


@pytest.fixture(scope="module")
def bl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import w1_a8_bitlinear_02_b300 as m
    m.capi.load()
    torch.cuda.set_device(0)
    return m


DEV = "cuda:0"
oracle.set_threads(min(16, os.cpu_count() or 1))


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_bits_equal(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.ascontiguousarray(got, np.float32)
    ref = np.ascontiguousarray(ref, np.float32)
    assert got.shape == ref.shape, what
    bad = got.view(np.uint32) != ref.view(np.uint32)
    if bad.any():
        i = np.argwhere(bad)[0]
        rel = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} differ; first at {tuple(i)}: "
                             f"{got[tuple(i)]!r} vs {ref[tuple(i)]!r}; max rel {rel:.3g}")
    denom = np.maximum(np.abs(ref), 1e-30)
    assert (np.abs(got - ref) <= REL_TOL * denom).all()


def pack_both(bl, N, K, std, seed, dtype=torch.float32):
    W = wl.weight(N, K, std, seed, "cpu", dtype)
    packed, gamma = bl.bitlinear_pack_weights(W.to(DEV))
    Wf = W.float().numpy()
    p_ref, g_ref = oracle.pack_weights(Wf)
    return packed, gamma, p_ref, g_ref


# ------------------------------------------------------------------ pack
@pytest.mark.parametrize("N,K,dtype", [
    (256, 512, torch.float32), (300, 100, torch.float32), (1, 1, torch.float32),
    (17, 65, torch.bfloat16), (129, 2560, torch.bfloat16), (1000, 333, torch.float32)])
def test_pack_weights(bl, N, K, dtype):
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, N * 7 + K, dtype)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.float32(gamma.item()).view(np.uint32) == np.float32(g_ref).view(np.uint32)


def test_pack_all_zero_and_ternary_weights(bl):
    W = torch.zeros((40, 70))
    W[3, 5] = 0.5
    W[7, 1] = -0.5
    packed, gamma = bl.bitlinear_pack_weights(W.to(DEV))
    p_ref, g_ref = oracle.pack_weights(W.numpy())
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert float(gamma.item()) == float(g_ref)
    Z = torch.zeros((3, 64))
    packed, gamma = bl.bitlinear_pack_weights(Z.to(DEV))
    assert (packed.cpu().numpy() == 0x55).all()


# ------------------------------------------------------------------ activations
@pytest.mark.parametrize("M,K,kind,dtype", [
    (4, 512, "outlier7", torch.float32), (3, 100, "normal", torch.float32),
    (1, 1, "normal", torch.float32), (5, 2560, "outliers1pct", torch.bfloat16),
    (2, 6912, "relu2", torch.bfloat16), (2, 64, "zeros", torch.bfloat16),
    (33, 1000, "normal", torch.bfloat16)])
def test_quant_act(bl, M, K, kind, dtype):
    x = wl.activations(M, K, kind, M + K, "cpu", dtype)
    xq, s = bl.bitlinear_quant_act(x.to(DEV))
    xq_ref, s_ref = oracle.quant_act(x.float().numpy())
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert_bits_equal(s.cpu().numpy(), s_ref, "scale")


@pytest.mark.parametrize("M,K,gain,dtype", [
    (4, 512, True, torch.float32), (3, 100, False, torch.float32),
    (6, 2560, True, torch.bfloat16), (2, 6912, False, torch.bfloat16), (1, 1, False, torch.float32)])
def test_rmsnorm_quant_act(bl, M, K, gain, dtype):
    x = wl.activations(M, K, "outliers1pct", 3 * K + M, "cpu", dtype)
    g = wl.rms_gain(K, K) if gain else None
    xq, s = bl.bitlinear_rmsnorm_quant_act(x.to(DEV), None if g is None else g.to(DEV), 1e-5)
    xq_ref, s_ref, _ = oracle.rmsnorm_quant_act(x.float().numpy(),
                                                None if g is None else g.numpy(), 1e-5)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    got = s.cpu().numpy()
    assert (np.abs(got - s_ref) <= REL_TOL * np.abs(s_ref)).all()


# ------------------------------------------------------------------ forward
SHAPES = [(256, 512), (300, 100), (130, 2560), (513, 1000)]
# 17-32 tokens take the few-token kernel's 32-token tile (bn = 32)
MS = [1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 24, 32, 33, 64, 65, 130, 257]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", MS)
def test_forward(bl, M, N, K):
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 11 * N + K)
    dtype = torch.float32 if M % 2 else torch.bfloat16
    x = wl.activations(M, K, "outliers1pct", 5 * M + K, "cpu", dtype)
    y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    y_ref = oracle.forward_packed(p_ref, g_ref, N, K, x.float().numpy())
    assert_bits_equal(y.cpu().numpy(), y_ref, f"y M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(256, 512), (300, 100), (513, 1000)])
@pytest.mark.parametrize("M", [1, 3, 4, 7, 17, 32, 64, 200])
def test_forward_q_and_matmul_i32(bl, M, N, K):
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 13 * N + K)
    x = wl.activations(M, K, "normal", 7 * M + K, "cpu", torch.float32)
    xq_ref, s_ref = oracle.quant_act(x.numpy())
    xq = torch.from_numpy(xq_ref).to(DEV)
    s = torch.from_numpy(s_ref).to(DEV)
    y = bl.bitlinear_forward_q(packed, gamma, N, K, xq, s)
    acc = bl.bitlinear_matmul_i32(packed, N, K, xq)
    torch.cuda.synchronize()
    q_ref = oracle.unpack(p_ref, K)
    acc_ref = oracle.matmul_i32(q_ref, xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_bits_equal(y.cpu().numpy(), oracle.rescale(acc_ref, g_ref, s_ref), "forward_q")


@pytest.mark.parametrize("M,K,dtype", [(1, 6912, torch.float32), (5, 1000, torch.bfloat16),
                                       (64, 6912, torch.float32), (300, 100, torch.bfloat16)])
def test_relu2_quant_act(bl, M, K, dtype):
    x = wl.activations(M, K, "normal", 19 * M + K, "cpu", dtype)
    xq, s = bl.bitlinear_relu2_quant_act(x.to(DEV))
    torch.cuda.synchronize()
    xq_ref, s_ref = oracle.relu2_quant_act(x.float().numpy())
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert_bits_equal(s.cpu().numpy(), s_ref, "relu2 scales")


# M = 1 (GEMV), 3 / 16 / 32 / 64 (few-token kernel), 130 (tensor-core GEMM)
@pytest.mark.parametrize("N,K", [(300, 100), (513, 1000), (2560, 6912)])
@pytest.mark.parametrize("M", [1, 3, 16, 32, 64, 130])
def test_forward_relu2(bl, M, N, K):
    """The down projection of a ReLU^2 FFN in one call: every path applies the
    squared ReLU where it quantises x, bit-exact with the oracle and with
    relu2_quant_act followed by forward_q."""
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 23 * N + K)
    dtype = torch.float32 if M % 2 else torch.bfloat16
    x = wl.activations(M, K, "normal", 29 * M + K, "cpu", dtype).to(DEV)
    y = bl.bitlinear_forward_relu2(packed, gamma, N, K, x)
    xq, s = bl.bitlinear_relu2_quant_act(x)
    y2 = bl.bitlinear_forward_q(packed, gamma, N, K, xq, s)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    y_ref = oracle.forward_packed_relu2(p_ref, g_ref, N, K, x.float().cpu().numpy())
    assert_bits_equal(y.cpu().numpy(), y_ref, f"forward_relu2 M={M} N={N} K={K}")
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


# M = 1, 2 (GEMV), 3, 24, 33, 64 (few-token kernel), 130 (tensor-core GEMM);
# the last shape also takes stream-K at M = 2048 (one case below)
@pytest.mark.parametrize("M,N,K", [(1, 513, 1000), (2, 300, 100), (3, 513, 1000), (24, 2560, 2560),
                                   (33, 2560, 2560),
                                   (64, 384, 768), (130, 300, 100), (2048, 2560, 320)])
@pytest.mark.parametrize("y_dtype,res,act", [(torch.float32, None, 0), (torch.bfloat16, None, 0),
                                             (torch.float32, "sep", 1), (torch.bfloat16, "inplace", 0),
                                             (torch.float32, "inplace", 1)])
def test_forward_ex_output_variants(bl, M, N, K, y_dtype, res, act):
    """bf16 / fp32 output, residual (separate or in place) and the squared-ReLU
    input, on every path, bit-exact with the oracle's output step."""
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 31 * N + K)
    x = wl.activations(M, K, "outliers1pct", 37 * M + K, "cpu", torch.bfloat16)
    r = (torch.randn((M, N), generator=torch.Generator().manual_seed(M + N)) * 2).to(y_dtype)
    y = torch.empty((M, N), dtype=y_dtype, device=DEV)
    residual = None
    if res == "sep":
        residual = r.to(DEV)
    elif res == "inplace":
        y.copy_(r.to(DEV))
        residual = y
    bl.bitlinear_forward_ex(packed, gamma, N, K, x.to(DEV), y=y, residual=residual, act=act)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    f = oracle.forward_packed_relu2 if act else oracle.forward_packed
    y32 = f(p_ref, g_ref, N, K, x.float().numpy())
    want = oracle.output(y32, None if res is None else r.float().numpy(), bf16=y_dtype == torch.bfloat16)
    got = y.cpu()
    if y_dtype == torch.bfloat16:
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), want)
    else:
        assert_bits_equal(got.numpy(), want, f"forward_ex M={M} N={N} K={K}")


def test_forward_equals_quant_then_forward_q(bl):
    N, K, M = 384, 768, 40
    packed, gamma, _, _ = pack_both(bl, N, K, 0.02, 5)
    x = wl.activations(M, K, "outliers1pct", 9, "cpu", torch.bfloat16).to(DEV)
    y1 = bl.bitlinear_forward(packed, gamma, N, K, x)
    xq, s = bl.bitlinear_quant_act(x)
    y2 = bl.bitlinear_forward_q(packed, gamma, N, K, xq, s)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_zero_activation_rows_give_zero(bl):
    N, K = 200, 300
    packed, gamma, _, _ = pack_both(bl, N, K, 0.02, 3)
    for M in (2, 9):
        x = wl.activations(M, K, "normal", 4, "cpu", torch.float32)
        x[0] = 0
        y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
        torch.cuda.synchronize()
        assert (y[0] == 0).all()


def test_launch_overlap_gives_same_results(bl):
    N, K = 640, 2560
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 21)
    xs = [wl.activations(M, K, "normal", 30 + M, "cpu", torch.bfloat16) for M in (1, 4, 64)]
    bl.set_launch_overlap(True)
    try:
        ys = [bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV)) for x in xs]
        torch.cuda.synchronize()
    finally:
        bl.set_launch_overlap(False)
    for x, y in zip(xs, ys):
        assert_bits_equal(y.cpu().numpy(), oracle.forward_packed(p_ref, g_ref, N, K,
                                                                  x.float().numpy()), "overlap")


def test_independent_calls_overlap_mode(bl):
    """Mode 2: a batch of independent calls (distinct inputs and outputs) may run
    concurrently; each result must still equal the oracle's."""
    shapes = [(384, 2560), (640, 512), (256, 6912)]
    mats = [pack_both(bl, N, K, 0.02, 40 + i) for i, (N, K) in enumerate(shapes)]
    xs = [wl.activations(M, K, "normal", 60 + M + K, "cpu", torch.bfloat16)
          for (N, K) in shapes for M in (1, 3, 8)]
    bl.set_launch_overlap(2)
    try:
        ys = []
        i = 0
        for j, (N, K) in enumerate(shapes):
            for M in (1, 3, 8):
                packed, gamma, _, _ = mats[j]
                ys.append(bl.bitlinear_forward(packed, gamma, N, K, xs[i].to(DEV)))
                i += 1
        torch.cuda.synchronize()
    finally:
        bl.set_launch_overlap(0)
    i = 0
    for j, (N, K) in enumerate(shapes):
        _, _, p_ref, g_ref = mats[j]
        for M in (1, 3, 8):
            assert_bits_equal(ys[i].cpu().numpy(),
                              oracle.forward_packed(p_ref, g_ref, N, K, xs[i].float().numpy()),
                              f"mode 2 N={N} K={K} M={M}")
            i += 1


# ------------------------------------------------------------------ decode chain
def test_chain_with_data_dependencies(bl):
    """Layers passing y to x inside one chain launch: o 2560->2560 (bf16 x),
    up 2560->6912 on o's fp32 output, down 6912->2560 on relu2(up's output),
    qkv 2560->3840 on down's output, and a ragged 300 x 1000 call.  Each step is
    checked against the oracle on the oracle's own previous output."""
    shapes = [(2560, 2560, 0), (6912, 2560, 0), (2560, 6912, 1), (3840, 2560, 0), (1000, 3840, 0)]
    mats = [pack_both(bl, N, K, 0.02, 300 + i) for i, (N, K, _) in enumerate(shapes)]
    x0 = wl.activations(1, 2560, "normal", 310, "cpu", torch.bfloat16)
    calls, ys = [], []
    x = x0.to(DEV)
    for (N, K, act), (packed, gamma, _, _) in zip(shapes, mats):
        y = torch.full((1, N), float("nan"), dtype=torch.float32, device=DEV)
        calls.append(dict(packed=packed, gamma=gamma, x=x, y=y, N=N, K=K, act=act))
        ys.append(y)
        x = y
    bl.bitlinear_forward_chain(calls)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    xr = x0.float().numpy()
    for i, ((N, K, act), (_, _, p_ref, g_ref)) in enumerate(zip(shapes, mats)):
        f = oracle.forward_packed_relu2 if act else oracle.forward_packed
        y_ref = f(p_ref, g_ref, N, K, xr)
        assert_bits_equal(ys[i].cpu().numpy(), y_ref, f"chain step {i}")
        xr = y_ref


@pytest.mark.parametrize("wait_prev", [1, 0])
def test_chain_equals_separate_calls(bl, wait_prev):
    """120 calls of the ~2B decode workload (independent inputs) in one chain:
    each output equals, bit for bit, a separate bitlinear_forward of the same call."""
    mats = wl.matrices("decode_2b", layers=3)
    calls, refs = [], []
    for mt in mats:
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, DEV)
        packed, gamma = bl.bitlinear_pack_weights(W)
        del W
        x = wl.activations(1, mt.K, mt.x_kind, mt.seed + 500, DEV, torch.bfloat16)
        y = torch.empty((1, mt.N), dtype=torch.float32, device=DEV)
        calls.append(dict(packed=packed, gamma=gamma, x=x, y=y, N=mt.N, K=mt.K, wait_prev=wait_prev))
        refs.append(bl.bitlinear_forward(packed, gamma, mt.N, mt.K, x))
    calls = calls * 10  # 120 calls (the same twelve matrices ten times)
    bl.bitlinear_forward_chain(calls)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    for c, r in zip(calls[:12], refs):
        assert torch.equal(c["y"].view(torch.int32), r.view(torch.int32))


def test_chain_subrange_inputs_and_long_rows(bl):
    """Inputs that are part of an earlier output (a prefix, an offset that keeps
    16-byte vectors, an odd offset read word by word), rows longer than one
    warp's 8192 weights (split over 2 and 4 warps), ReLU^2 on a chained input;
    the chain is launched three times on one workspace (each launch's tags are
    new) and every output is checked against the oracle each time."""
    # (N, K, src, offset into src's output, act)
    specs = [(3840, 2560, -1, 0, 0),      # x0 (bf16)
             (2560, 2560, 0, 0, 0),       # prefix of call 0's output
             (9000, 2560, 1, 0, 0),
             (2560, 9000, 2, 0, 1),       # K = 9000: rows over 2 warps; relu2
             (700, 2000, 0, 1280, 0),     # offset 1280 floats: 16-byte aligned words
             (333, 999, 0, 1, 0),         # odd offset, odd K: word by word
             (512, 20000, -1, 0, 0)]      # K = 20000 from x0's row: 4 warps per row
    mats = [pack_both(bl, N, K, 0.02, 700 + i) for i, (N, K, _, _, _) in enumerate(specs)]
    x0 = wl.activations(1, 20000, "normal", 710, "cpu", torch.bfloat16)
    xdev = x0.to(DEV)
    ys = [torch.full((1, N), float("nan"), dtype=torch.float32, device=DEV) for (N, *_ ) in specs]
    calls = []
    for i, ((N, K, src, off, act), (packed, gamma, _, _)) in enumerate(zip(specs, mats)):
        x = xdev[:, :K] if src < 0 else ys[src][:, off:off + K]
        calls.append(dict(packed=packed, gamma=gamma, x=x, y=ys[i], N=N, K=K, act=act))
    ws = bl.chain_workspace(calls, DEV)
    outs = []
    xr0 = x0.float().numpy()
    for (N, K, src, off, act), (_, _, p_ref, g_ref) in zip(specs, mats):
        xin = xr0[:, :K] if src < 0 else outs[src][:, off:off + K]
        f = oracle.forward_packed_relu2 if act else oracle.forward_packed
        outs.append(f(p_ref, g_ref, N, K, np.ascontiguousarray(xin, np.float32)))
    for launch in range(3):
        for y in ys:
            y.fill_(float("nan"))
        bl.bitlinear_forward_chain(calls, ws)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        for i, y in enumerate(ys):
            assert_bits_equal(y.cpu().numpy(), outs[i], f"launch {launch} call {i}")


def test_chain_many_tokens(bl):
    """Calls of 2 to 16 tokens (independent inputs, quantised ahead; stages of
    at most 31 or 23 pieces; 2-4 tokens on dp4a, 5-16 on the tensor cores) mixed with
    single-token calls, ragged N and K, bf16 and fp32 inputs, a squared-ReLU
    input, every ~2B projection at 8 tokens and a five-slab row at 6 tokens;
    the chain runs twice on one workspace and each output equals the oracle's."""
    specs = [(300, 1000, 2, torch.bfloat16, 0), (3840, 2560, 8, torch.bfloat16, 0), (2560, 2560, 8, torch.bfloat16, 0),
             (6912, 2560, 8, torch.bfloat16, 0), (2560, 6912, 8, torch.bfloat16, 1), (513, 100, 3, torch.float32, 0),
             (700, 2000, 1, torch.bfloat16, 0), (129, 4608, 5, torch.float32, 1), (1000, 64, 7, torch.bfloat16, 0),
             (4736, 9000, 6, torch.bfloat16, 0), (333, 512, 4, torch.bfloat16, 0),
             (2560, 6912, 16, torch.bfloat16, 1), (3840, 2560, 12, torch.bfloat16, 0), (777, 1000, 9, torch.float32, 0)]
    mats = [pack_both(bl, N, K, 0.02, 950 + i) for i, (N, K, _, _, _) in enumerate(specs)]
    calls, xs, ys = [], [], []
    for i, ((N, K, M, dt, act), (packed, gamma, _, _)) in enumerate(zip(specs, mats)):
        x = wl.activations(M, K, "outliers1pct", 960 + i, "cpu", dt)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        calls.append(dict(packed=packed, gamma=gamma, x=x.to(DEV), y=y, N=N, K=K, act=act))
        xs.append(x)
        ys.append(y)
    ws = bl.chain_workspace(calls, DEV)
    for launch in range(2):
        for y in ys:
            y.fill_(float("nan"))
        bl.bitlinear_forward_chain(calls, ws)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        for i, ((N, K, M, dt, act), (_, _, p_ref, g_ref)) in enumerate(zip(specs, mats)):
            f = oracle.forward_packed_relu2 if act else oracle.forward_packed
            assert_bits_equal(ys[i].cpu().numpy(), f(p_ref, g_ref, N, K, xs[i].float().numpy()),
                              f"launch {launch} call {i} M={M} N={N} K={K}")


def test_chain_write_after_read_and_write_after_write(bl):
    """Outputs that overwrite an earlier call's input buffer or output buffer:
    the library puts a grid barrier before such calls, so the results are those
    of running the calls one after another."""
    N, K = 2560, 2560
    mats = [pack_both(bl, N, K, 0.02, 800 + i) for i in range(4)]
    a0 = wl.activations(1, K, "normal", 810, "cpu", torch.float32)
    A = a0.to(DEV)
    B = torch.empty((1, N), dtype=torch.float32, device=DEV)
    C = torch.empty((1, N), dtype=torch.float32, device=DEV)
    # 0: A -> B;  1: B -> A (overwrites call 0's input);  2: A -> C;  3: B -> C (C again)
    plan = [(A, B), (B, A), (A, C), (B, C)]
    calls = [dict(packed=m[0], gamma=m[1], x=x, y=y, N=N, K=K) for m, (x, y) in zip(mats, plan)]
    bl.bitlinear_forward_chain(calls)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    ref = {"A": a0.numpy()}
    for i, (xn, yn) in enumerate((("A", "B"), ("B", "A"), ("A", "C"), ("B", "C"))):
        _, _, p_ref, g_ref = mats[i]
        ref[yn] = oracle.forward_packed(p_ref, g_ref, N, K, ref[xn])
    assert_bits_equal(A.cpu().numpy(), ref["A"], "A")
    assert_bits_equal(B.cpu().numpy(), ref["B"], "B")
    assert_bits_equal(C.cpu().numpy(), ref["C"], "C")


@pytest.mark.parametrize("N,K", [(50, 64), (333, 100), (4000, 448), (129, 512)])
def test_chain_short_rows(bl, N, K):
    """Rows shorter than one 128-byte box (the box reads zeros past the row),
    a row count that leaves a partial group in every block, chained twice."""
    mats = [pack_both(bl, N, K, 0.02, 900 + K), pack_both(bl, K, N, 0.02, 901 + K)]
    x0 = wl.activations(1, K, "normal", 902, "cpu", torch.bfloat16)
    y0 = torch.empty((1, N), dtype=torch.float32, device=DEV)
    y1 = torch.empty((1, K), dtype=torch.float32, device=DEV)
    calls = [dict(packed=mats[0][0], gamma=mats[0][1], x=x0.to(DEV), y=y0, N=N, K=K),
             dict(packed=mats[1][0], gamma=mats[1][1], x=y0, y=y1, N=K, K=N)]
    bl.bitlinear_forward_chain(calls)
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    r0 = oracle.forward_packed(mats[0][2], mats[0][3], N, K, x0.float().numpy())
    r1 = oracle.forward_packed(mats[1][2], mats[1][3], K, N, r0)
    assert_bits_equal(y0.cpu().numpy(), r0, "short rows 0")
    assert_bits_equal(y1.cpu().numpy(), r1, "short rows 1")


def test_chain_long_row_groups_alternating_teams(bl):
    """Row groups of many slabs (K = 28672: seven stages a group) next to
    groups of two, one-token and many-token: the warps of one team skip the
    other team's long group and must not take a ring slot's earlier phase
    for the stage they wait for.  Independent and dependent inputs; whole
    outputs against the oracle, repeated launches on one workspace."""
    specs = [(4736, 28672, -1, 1), (4736, 8192, -1, 1), (4736, 28672, -1, 1), (9472, 4736, 2, 1),
             (4736, 28672, -1, 3), (300, 9472, 3, 1)]
    mats = [pack_both(bl, N, K, 0.01, 1100 + i) for i, (N, K, _, _) in enumerate(specs)]
    xs, ys, calls = [], [], []
    for i, ((N, K, src, M), (packed, gamma, _, _)) in enumerate(zip(specs, mats)):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        if src < 0:
            x = wl.activations(M, K, "outliers1pct", 1110 + i, "cpu", torch.bfloat16)
            xd = x.to(DEV)
        else:
            x, xd = None, ys[src][:, :K]
        xs.append(x)
        ys.append(y)
        calls.append(dict(packed=packed, gamma=gamma, x=xd, y=y, N=N, K=K))
    ws = bl.chain_workspace(calls, DEV)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        bl.bitlinear_forward_chain(calls, ws)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        outs = []
        for i, ((N, K, src, M), (_, _, p_ref, g_ref)) in enumerate(zip(specs, mats)):
            xin = xs[i].float().numpy() if src < 0 else np.ascontiguousarray(outs[src][:, :K], np.float32)
            outs.append(oracle.forward_packed(p_ref, g_ref, N, K, xin))
            assert_bits_equal(ys[i].cpu().numpy(), outs[i], f"long groups call {i}")


def _independent_chain(bl, specs, seed, launches=1):
    """A chain of independent one-token calls (their own x, their own y): every
    call takes the fast form, so the producers hand row groups to the two
    teams through their queues.  Whole outputs against the oracle after each
    launch on one workspace."""
    calls, refs = [], []
    for i, (N, K, dtype, act) in enumerate(specs):
        packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, seed + i)
        x = wl.activations(1, K, "outliers1pct", seed + 500 + i, "cpu", dtype)
        y = torch.empty((1, N), dtype=torch.float32, device=DEV)
        calls.append(dict(packed=packed, gamma=gamma, x=x.to(DEV), y=y, N=N, K=K, act=act))
        f = oracle.forward_packed_relu2 if act else oracle.forward_packed
        refs.append(f(p_ref, g_ref, N, K, x.float().numpy()))
    ws = bl.chain_workspace(calls, DEV)
    for _ in range(launches):
        for c in calls:
            c["y"].fill_(float("nan"))
        bl.bitlinear_forward_chain(calls, ws)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        for i, (c, r) in enumerate(zip(calls, refs)):
            assert_bits_equal(c["y"].cpu().numpy(), r, f"independent chain call {i}")


def test_chain_independent_team_queues(bl):
    """Independent one-token calls of one, two and seven slabs a group; calls
    with fewer row groups than blocks (most blocks and one team idle) and with
    two groups a block; ragged N, bf16 and fp32 x, ReLU2 inputs and a K that is
    not a multiple of 8; three launches on one workspace."""
    bf, f32 = torch.bfloat16, torch.float32
    specs = [(64, 2560, bf, 0), (300, 6912, bf, 1), (9472, 2560, bf, 0), (640, 28672, bf, 0),
             (2560, 6912, f32, 0), (1000, 999, f32, 0), (4736, 8192, bf, 0), (33, 64, bf, 1)]
    _independent_chain(bl, specs, 1300, launches=3)


def test_chain_independent_most_calls(bl):
    """The most calls a chain takes (240), all independent and small: the
    blocks' per-call entries and the stage and group prefix sums over the
    whole call table."""
    shapes = [(64, 64), (96, 448), (200, 1000), (320, 2560), (37, 130)]
    specs = [(shapes[i % 5][0], shapes[i % 5][1], torch.bfloat16, i % 7 == 3) for i in range(240)]
    _independent_chain(bl, specs, 1400)


def test_chain_headline_step_full(bl):
    """The decode step the bench times, as it times it: the 30 layers' 120
    projections of the ~2B workload (391 MB of packed weights, each call its
    own x, drawn as the bench draws them), one chain launch on a reused
    workspace; every call's whole output against the oracle."""
    calls = []
    for mt in wl.matrices("decode_2b", layers=30):
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, DEV)
        packed, gamma = bl.bitlinear_pack_weights(W)
        del W
        x = wl.activations(1, mt.K, mt.x_kind, mt.seed + 500, DEV, torch.bfloat16)
        y = torch.empty((1, mt.N), dtype=torch.float32, device=DEV)
        calls.append(dict(packed=packed, gamma=gamma, x=x, y=y, N=mt.N, K=mt.K))
    assert len(calls) == 120
    ws = bl.chain_workspace(calls, DEV)
    for _ in range(2):
        for c in calls:
            c["y"].fill_(float("nan"))
        bl.bitlinear_forward_chain(calls, ws)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
    for i, c in enumerate(calls):
        ref = oracle.forward_packed(c["packed"].cpu().numpy(), float(c["gamma"].item()), c["N"], c["K"],
                                    c["x"].float().cpu().numpy())
        assert_bits_equal(c["y"].cpu().numpy(), ref, f"headline step call {i}")


def test_chain_100b_sweep_sampled(bl):
    """The 100B-class sweep the bench times: 80 layers' 160 calls (9.4 GB of
    packed weights resident), one chain launch at one token and one at eight;
    the first and last call of each shape (whole outputs) against the oracle
    (the oracle needs seconds per 100B-class call, so the rest is sampled)."""
    mats = wl.matrices("decode_100b")
    assert len(mats) == 160
    packs = []
    for mt in mats:
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, DEV)
        packs.append(bl.bitlinear_pack_weights(W))
        del W
    checked = [0, 1, len(mats) - 2, len(mats) - 1]
    for M in (1, 8):
        calls = []
        for mt, (packed, gamma) in zip(mats, packs):
            x = wl.activations(M, mt.K, mt.x_kind if M == 1 else "outliers1pct", mt.seed + 500 + M, DEV,
                               torch.bfloat16)
            y = torch.full((M, mt.N), float("nan"), dtype=torch.float32, device=DEV)
            calls.append(dict(packed=packed, gamma=gamma, x=x, y=y, N=mt.N, K=mt.K))
        bl.bitlinear_forward_chain(calls)
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        for i in (checked if M == 1 else checked[1:3]):
            c = calls[i]
            ref = oracle.forward_packed(c["packed"].cpu().numpy(), float(c["gamma"].item()), c["N"], c["K"],
                                        c["x"].float().cpu().numpy())
            assert_bits_equal(c["y"].cpu().numpy(), ref, f"100B sweep M={M} call {i}")
        for c in calls:
            assert not torch.isnan(c["y"]).any(), "an output left unwritten"
        del calls


@pytest.mark.parametrize("M", [8, 16, 64])
def test_chain_batched_step_sampled(bl, M):
    """Batched decode as the bench times it through the chain: the 30 layers'
    120 projections with M tokens (1 % outlier channels), the token rows in
    slices of 16 (each slice its own call), at most 240 calls a launch; the
    whole outputs of a sample of calls (every projection kind, first and last
    layers) against the oracle, every output written."""
    mats = wl.matrices("decode_2b", layers=30)
    items = []
    for mt in mats:
        W = wl.weight(mt.N, mt.K, mt.std, mt.seed, DEV)
        packed, gamma = bl.bitlinear_pack_weights(W)
        del W
        x = wl.activations(M, mt.K, "outliers1pct", mt.seed + 600 + M, DEV, torch.bfloat16)
        y = torch.full((M, mt.N), float("nan"), dtype=torch.float32, device=DEV)
        items.append(dict(packed=packed, gamma=gamma, x=x, y=y, N=mt.N, K=mt.K))
    calls = [dict(packed=it["packed"], gamma=it["gamma"], x=it["x"][h:h + 16], y=it["y"][h:h + 16],
                  N=it["N"], K=it["K"]) for it in items for h in range(0, M, 16)]
    for i in range(0, len(calls), 240):
        bl.bitlinear_forward_chain(calls[i:i + 240])
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    for i in (0, 1, 2, 3, len(items) - 4, len(items) - 3, len(items) - 2, len(items) - 1):
        it = items[i]
        ref = oracle.forward_packed(it["packed"].cpu().numpy(), float(it["gamma"].item()), it["N"], it["K"],
                                    it["x"].float().cpu().numpy())
        assert_bits_equal(it["y"].cpu().numpy(), ref, f"batched step M={M} projection {i}")
    for it in items:
        assert not torch.isnan(it["y"]).any(), "an output left unwritten"


def test_chain_unaligned_and_odd_k(bl):
    """K not a multiple of 8 and an input that starts off a 16-byte boundary
    take the element-by-element activation path."""
    N, K = 333, 999
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 77)
    xb = wl.activations(1, K + 1, "normal", 78, "cpu", torch.float32)
    xdev = xb.to(DEV)[:, 1:]  # 4-byte offset
    y = torch.empty((1, N), dtype=torch.float32, device=DEV)
    bl.bitlinear_forward_chain([dict(packed=packed, gamma=gamma, x=xdev, y=y, N=N, K=K)])
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    y_ref = oracle.forward_packed(p_ref, g_ref, N, K, xb.numpy()[:, 1:].copy())
    assert_bits_equal(y.cpu().numpy(), y_ref, "chain odd K")


# ------------------------------------------------------------------ full workload shapes
@pytest.mark.parametrize("name,N,K,kind", [(n, N, K, k) for n, N, K, k in wl.PROJ_2B])
def test_decode_2b_shapes_full(bl, name, N, K, kind):
    """One layer of the ~2B model at M = 1 (whole output) and M = 8 (whole output)."""
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, wl.weight_seed("decode_2b", 0, 0) + N)
    for M in (1, 8):
        x = wl.activations(M, K, kind, 77 + M, "cpu", torch.bfloat16)
        y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
        torch.cuda.synchronize()
        assert_bits_equal(y.cpu().numpy(), oracle.forward_packed(p_ref, g_ref, N, K,
                                                                  x.float().numpy()),
                          f"{name} M={M}")


@pytest.mark.parametrize("name,N,K,kind", [(n, N, K, k) for n, N, K, k in wl.PROJ_2B])
def test_batched_decode_2b_shapes_full(bl, name, N, K, kind):
    """Batched decode on one layer of the ~2B model: M = 3 (GEMV), 5, 8, 16, 17,
    24, 32, 33 and 64 tokens (the few-token kernel at its 16-, 32- and 64-token
    tiles, or the GEMM where that needs more than one wave) with 1 % outlier
    channels, whole outputs, through forward and forward_q."""
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, wl.weight_seed("decode_2b", 1, 0) + N)
    for M in (3, 5, 8, 16, 17, 24, 32, 33, 64):
        x = wl.activations(M, K, "outliers1pct", 91 + M, "cpu", torch.bfloat16)
        y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
        xq_ref, s_ref = oracle.quant_act(x.float().numpy())
        y_q = bl.bitlinear_forward_q(packed, gamma, N, K, torch.from_numpy(xq_ref).to(DEV),
                                     torch.from_numpy(s_ref).to(DEV))
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        y_ref = oracle.forward_packed(p_ref, g_ref, N, K, x.float().numpy())
        assert_bits_equal(y.cpu().numpy(), y_ref, f"{name} M={M}")
        assert_bits_equal(y_q.cpu().numpy(), y_ref, f"{name} M={M} forward_q")


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 320), (1900, 2500, 300), (2048, 2560, 6912),
                                   (8, 20480, 640), (24, 20480, 640), (40, 19000, 448),
                                   (8, 40960, 640), (24, 40960, 640), (40, 38000, 448)])
def test_streamk_tiles_full_output(bl, M, N, K):
    """Tile counts that fill the last wave poorly (149-160 tiles on 148 SMs) run
    stream-K: tiles are shared by two blocks whose int32 partials meet in the
    workspace.  Whole outputs (forward and matmul_i32) against the oracle; the
    third shape is the prefill down projection itself, checked in full; the
    rest have token tiles of 16, 32 and 64 (a few tokens on many rows), which
    run as whole tiles two blocks per SM (149-160 tiles in one wave, 297-320 in
    two) rather than stream-K."""
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 17 * N + K)
    x = wl.activations(M, K, "outliers1pct", 3 * M + K, "cpu", torch.bfloat16)
    y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
    xq_ref, s_ref = oracle.quant_act(x.float().numpy())
    acc = bl.bitlinear_matmul_i32(packed, N, K, torch.from_numpy(xq_ref).to(DEV))
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    acc_ref = oracle.matmul_i32(oracle.unpack(p_ref, K), xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_bits_equal(y.cpu().numpy(), oracle.rescale(acc_ref, g_ref, s_ref), f"stream-K M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K,kind", [(6912, 2560, "normal"), (2560, 6912, "relu2")])
def test_prefill_2048_full(bl, N, K, kind):
    """M = 2048 on the tensor-core path (up projection: whole 256-token tiles;
    down projection: stream-K), the whole output against the oracle."""
    M = 2048
    packed, gamma, p_ref, g_ref = pack_both(bl, N, K, 0.02, 4000 + N)
    x = wl.activations(M, K, kind, 4500 + K, "cpu", torch.bfloat16)
    y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    assert_bits_equal(y.cpu().numpy(), oracle.forward_packed(p_ref, g_ref, N, K, x.float().numpy()),
                      f"prefill {N}x{K}")


@pytest.mark.parametrize("N,K,Ms", [(28672, 8192, (1, 3, 8)), (8192, 28672, (1, 4, 8))])
def test_decode_100b_shape_full(bl, N, K, Ms):
    """The 100B-class matrices (28672 x 8192 and 8192 x 28672), packed on the
    GPU, whole outputs at one token, a few (GEMV or GEMM by fit) and eight
    (the GEMM: the few-token kernel would need more than one wave)."""
    W = wl.weight(N, K, 0.01, wl.weight_seed("decode_100b", 0, 0) + N, DEV)
    packed, gamma = bl.bitlinear_pack_weights(W)
    Wh = W.cpu().numpy()
    del W
    p_ref, g_ref = oracle.pack_weights(Wh)
    del Wh
    assert float(gamma.item()) == float(g_ref)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    for M in Ms:
        x = wl.activations(M, K, "normal", 5000 + M, "cpu", torch.bfloat16)
        y = bl.bitlinear_forward(packed, gamma, N, K, x.to(DEV))
        torch.cuda.synchronize()
        assert bl.device_error() == 0
        assert_bits_equal(y.cpu().numpy(), oracle.forward_packed(p_ref, g_ref, N, K,
                                                                  x.float().numpy()),
                          f"100b {N}x{K} M={M}")


# ------------------------------------------------- grouped weight scales
@pytest.mark.parametrize("N,K,G,dtype", [(256, 512, 1, torch.float32), (384, 1000, 128, torch.bfloat16),
                                         (6912, 2560, 128, torch.float32), (300, 70, 4, torch.float32)])
def test_pack_weights_grouped(bl, N, K, G, dtype):
    """One absmean scale per group of G output rows: codes and scales bit-exact."""
    W = wl.weight(N, K, 0.02, 41 * N + G, "cpu")
    W[: N // 2] *= 0.05  # groups of very different magnitude
    W = W.to(dtype)
    packed, gamma = bl.bitlinear_pack_weights_grouped(W.to(DEV), G)
    torch.cuda.synchronize()
    p_ref, g_ref = oracle.pack_weights_groups(W.float().numpy(), G)
    assert np.array_equal(gamma.cpu().numpy().view(np.uint32), g_ref.view(np.uint32))
    assert np.array_equal(packed.cpu().numpy(), p_ref)


# M = 1, 3 (GEMV), 16 / 32 / 64 (few-token kernel), 130 (GEMM), 2048 (stream-K)
@pytest.mark.parametrize("M,N,K", [(1, 384, 1000), (3, 2560, 2560), (16, 384, 1000), (32, 2560, 2560),
                                   (64, 2560, 2560),
                                   (130, 384, 1000), (2048, 2560, 320)])
@pytest.mark.parametrize("G", [1, 128])
def test_forward_grouped(bl, M, N, K, G):
    """Grouped-scale forward on every path, bit-exact with the oracle; the
    last case also through the bf16 output with an in-place residual."""
    W = wl.weight(N, K, 0.02, 43 * N + K, "cpu")
    W[N // 4: N // 2] *= 20.0
    packed, gamma = bl.bitlinear_pack_weights_grouped(W.to(DEV), G)
    p_ref, g_ref = oracle.pack_weights_groups(W.numpy(), G)
    x = wl.activations(M, K, "outliers1pct", 47 * M + K, "cpu", torch.bfloat16)
    y = bl.bitlinear_forward_grouped(packed, gamma, G, N, K, x.to(DEV))
    torch.cuda.synchronize()
    assert bl.device_error() == 0
    y_ref = oracle.forward_packed_groups(p_ref, g_ref, G, N, K, x.float().numpy())
    assert_bits_equal(y.cpu().numpy(), y_ref, f"grouped G={G} M={M} N={N} K={K}")
    if M == 2048:
        r = (torch.randn((M, N), generator=torch.Generator().manual_seed(G)) * 2).to(torch.bfloat16)
        yb = r.to(DEV)
        bl.bitlinear_forward_grouped(packed, gamma, G, N, K, x.to(DEV), y=yb, residual=yb, act=1)
        torch.cuda.synchronize()
        y2 = oracle.forward_packed_groups(p_ref, g_ref, G, N, K, oracle.relu2(x.float().numpy()))
        want = oracle.output(y2, r.float().numpy(), bf16=True)
        assert np.array_equal(yb.cpu().view(torch.int16).numpy().view(np.uint16), want)
