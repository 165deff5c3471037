"""Pins for the CPU oracle: checks against things other than the oracle itself.

- a hand-worked example whose every value was derived by hand (golden file);
- the packed layout on hand-derived one-hot bytes (golden file);
- exact rational arithmetic (Python Fractions / ints) on tiny random shapes;
- a library routine (numpy int64 matmul) for the integer contraction;
- a closed form (fraction of zero codes for Gaussian weights);
- invariants and degenerate cases.

Sources of the definitions: the 2B4T report translation on
blog.csdn.net/soaring_casia ("原生1.58bit大模型"), section 2 "BitLinear层"
items 1-3 (absmean ternary weights, per-token absmax int8 activations, subln);
"BitNet b1.58 深度解析" (chenxutan.com) section 2.3(2) for the rescale.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

F32_EPS = Fraction(1, 2 ** 23)
# y = fl32(acc * fl32(gamma / s)): two roundings of at most 2^-24 relative each
Y_REL = Fraction(2, 2 ** 24) + Fraction(1, 2 ** 47)


# ---------------------------------------------------------------- helpers
def fl32(fr: Fraction) -> np.float32:
    """Round an exact rational to the nearest binary32, ties to even."""
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f,
             np.nextafter(f, np.float32(np.inf))]
    best, bestd = None, None
    for c in cands:
        d = abs(Fraction(float(c)) - fr)
        if bestd is None or d < bestd or (
                d == bestd and (np.array(c).view(np.uint32) & 1) == 0):
            best, bestd = c, d
    return np.float32(best)


def rne(fr: Fraction) -> int:
    fl = math.floor(fr)
    diff = fr - fl
    if diff > Fraction(1, 2):
        return fl + 1
    if diff < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def near_half(fr: Fraction, rel=Fraction(1, 2 ** 22)) -> bool:
    """True if fr is within a couple of fp32 ulps of a rounding boundary."""
    d = abs(fr - math.floor(fr) - Fraction(1, 2))
    return d <= abs(fr) * rel + Fraction(1, 2 ** 40)


FEPS = fl32(Fraction(1, 100000))  # the fp32 constant 1e-5f


# ---------------------------------------------------------------- pin-1
def test_hand_example(golden_dir):
    with open(os.path.join(golden_dir, "hand_example.json")) as f:
        gd = json.load(f)
    W = np.array(gd["W"], np.float32)
    x = np.array(gd["x"], np.float32)
    g = oracle.gamma(W)
    assert Fraction(float(W.__abs__().sum())) / W.size == Fraction(gd["mean_abs_W"])
    assert g == fl32(Fraction(gd["mean_abs_W"]) + Fraction(float(FEPS)))
    q = oracle.ternarize(W, g)
    assert q.tolist() == gd["Wq"]
    xq, s = oracle.quant_act(x)
    assert s.tolist() == gd["s"]
    assert xq.tolist() == gd["xq"]
    acc = oracle.matmul_i32(q, xq)
    assert acc.tolist() == gd["acc"]
    packed = oracle.pack(q)
    assert [bytes(r).hex() for r in packed] == gd["packed_rows_hex"]
    y = oracle.forward_packed(packed, g, 2, 4, x)
    for m in range(2):
        c = fl32(Fraction(float(g)) / Fraction(gd["s"][m]))  # the token's scale gamma/s
        for n in range(2):
            a = gd["acc"][m][n]
            assert y[m, n] == fl32(a * Fraction(float(c)))
            e = a * Fraction(float(g)) / Fraction(gd["s"][m])
            assert abs(Fraction(float(y[m, n])) - e) <= abs(e) * Y_REL


def test_weight_ties_round_half_to_even(golden_dir):
    with open(os.path.join(golden_dir, "weight_tie_example.json")) as f:
        gd = json.load(f)
    W = np.array([[float.fromhex(v) for v in row] for row in gd["W_hex"]], np.float32)
    g = oracle.gamma(W)
    assert float(g) == float.fromhex(gd["gamma_hex"])
    assert Fraction(float(W[0, 0])) / Fraction(float(g)) == Fraction(1, 2)
    assert oracle.ternarize(W, g).tolist() == gd["Wq"]


def test_pack_layout_onehot(golden_dir):
    with open(os.path.join(golden_dir, "pack_layout_onehot.json")) as f:
        gd = json.load(f)
    K = gd["K"]
    assert oracle.row_bytes(K) == gd["row_bytes"]
    for c in gd["cases"]:
        q = np.zeros((1, K), np.int8)
        q[0, c["k"]] = c["q"]
        p = oracle.pack(q)[0]
        expect = np.full(gd["row_bytes"], 0x55, np.uint8)
        expect[c["byte"]] = int(c["value"], 16)
        assert p.tolist() == expect.tolist(), c
        assert oracle.unpack(p[None, :], K).tolist() == q.tolist()


@pytest.mark.parametrize("K", [1, 15, 16, 63, 64, 65, 100, 512])
def test_pack_roundtrip_and_padding(K):
    rng = np.random.default_rng(K)
    q = rng.integers(-1, 2, size=(5, K)).astype(np.int8)
    p = oracle.pack(q)
    assert p.shape == (5, 16 * ((K + 63) // 64))
    assert oracle.unpack(p, K).tolist() == q.tolist()
    # no code 3 anywhere; padded weights decode to 0
    bits = np.unpackbits(p, bitorder="little").reshape(5, -1, 2)
    codes = bits[..., 0] + 2 * bits[..., 1]
    assert codes.max() <= 2
    Kp = 4 * p.shape[1]
    qp = oracle.unpack(p, Kp)
    assert (qp[:, K:] == 0).all()


# ---------------------------------------------------------------- pin-3 brute force
@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_rational(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 24))
    K = int(rng.integers(1, 48))
    M = int(rng.integers(1, 5))
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    if seed % 2:
        x[:, 0] *= 20
    # gamma: exact rational mean, one rounding, then + 1e-5f with one rounding
    S = sum(Fraction(abs(float(w))) for w in W.ravel())
    g = oracle.gamma(W)
    assert g == fl32(Fraction(float(fl32(S / (N * K)))) + Fraction(float(FEPS)))
    # codes: exact rational round of W/gamma, except within ~1 ulp of a tie
    q = oracle.ternarize(W, g)
    G = Fraction(float(g))
    skipped = 0
    for (n, k), w in np.ndenumerate(W):
        r = Fraction(float(w)) / G
        if near_half(r):
            skipped += 1
            continue
        assert q[n, k] == max(-1, min(1, rne(r)))
    assert skipped <= 1
    # activations
    xq, s = oracle.quant_act(x)
    for m in range(M):
        amax = max(abs(Fraction(float(v))) for v in x[m])
        assert s[m] == fl32(Fraction(127) / max(amax, Fraction(float(FEPS))))
        S_ = Fraction(float(s[m]))
        for k in range(K):
            p = Fraction(float(x[m, k])) * S_
            if near_half(p):
                continue
            assert xq[m, k] == max(-128, min(127, rne(p)))
    # contraction: Python ints and numpy's int64 matmul
    acc = oracle.matmul_i32(q, xq)
    for m in range(M):
        for n in range(N):
            assert acc[m, n] == sum(int(q[n, k]) * int(xq[m, k]) for k in range(K))
    assert (acc == xq.astype(np.int64) @ q.astype(np.int64).T).all()
    # y within two roundings of the exact rational acc * gamma / s
    y = oracle.rescale(acc, g, s)
    for m in range(M):
        # the token's scale c = fl32(gamma / s): a true division, one rounding
        c = fl32(G / Fraction(float(s[m])))
        for n in range(N):
            e = int(acc[m, n]) * G / Fraction(float(s[m]))
            assert abs(Fraction(float(y[m, n])) - e) <= abs(e) * Y_REL
            # the definition's two single roundings, evaluated exactly
            assert y[m, n] == fl32(int(acc[m, n]) * Fraction(float(c)))
    # forward from packed == the pieces
    y2 = oracle.forward_packed(oracle.pack(q), g, N, K, x)
    assert (y2.view(np.uint32) == y.view(np.uint32)).all()


# ---------------------------------------------------------------- pin-4 closed form
def test_zero_fraction_closed_form():
    """For W ~ N(0, s^2), gamma ~ E|W| = s*sqrt(2/pi); a weight rounds to 0 iff
    |W| < gamma/2, so P(0) = erf(sqrt(2/pi)/2/sqrt(2)) = 0.3101.  The
    threshold-at-mean rule printed in the 深度解析 page's snippet (section 2.2)
    would give erf(1/sqrt(pi)) = 0.5751 instead: this pins the round rule."""
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((1024, 1024)) * 0.02).astype(np.float32)
    q = oracle.ternarize(W, oracle.gamma(W))
    p0 = float((q == 0).mean())
    expect = math.erf(math.sqrt(2 / math.pi) / 2 / math.sqrt(2))
    assert abs(expect - 0.3101) < 1e-4
    assert abs(p0 - expect) < 0.004
    assert abs(float((q == 1).mean()) - (1 - expect) / 2) < 0.004
    assert abs(p0 - math.erf(1 / math.sqrt(math.pi))) > 0.2


# ---------------------------------------------------------------- pin-2 invariants
@pytest.mark.parametrize("density", [0.05, 0.5, 1.0])
def test_ternary_representable_weights(density):
    rng = np.random.default_rng(int(density * 100))
    c = np.float32(0.037)
    sign = rng.choice([-1, 1], size=(16, 96))
    mask = rng.random((16, 96)) < density
    mask[0, 0] = True
    W = (sign * mask * c).astype(np.float32)
    q = oracle.ternarize(W, oracle.gamma(W))
    assert (q == np.sign(W).astype(np.int8)).all()


def test_activation_invariants():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 333)).astype(np.float32)
    xq, s = oracle.quant_act(x)
    assert np.abs(xq.astype(int)).max() <= 127
    for m in range(8):
        i = int(np.argmax(np.abs(x[m])))
        assert abs(int(xq[m, i])) == 127
    # scaling a token by 2^e leaves its codes unchanged and scales s by 2^-e
    for e in (-3, 5):
        xq2, s2 = oracle.quant_act((x * np.float32(2.0 ** e)).astype(np.float32))
        assert (xq2 == xq).all()
        assert (s2 == (s * np.float32(2.0 ** -e))).all()


def test_integer_activations_amax_127():
    """Integer x with max|x| = 127: s = 1, xq = x, y = fl32(acc * gamma)."""
    rng = np.random.default_rng(11)
    x = rng.integers(-127, 128, size=(3, 200)).astype(np.float32)
    x[:, 5] = 127
    W = (rng.standard_normal((40, 200)) * 0.02).astype(np.float32)
    y, packed, g = oracle.forward(W, x)
    xq, s = oracle.quant_act(x)
    assert (s == 1).all() and (xq == x).all()
    q = oracle.unpack(packed, 200)
    acc = x.astype(np.int64) @ q.astype(np.int64).T
    c = fl32(Fraction(float(g)))  # gamma / 1
    for (m, n), a in np.ndenumerate(acc):
        assert y[m, n] == fl32(int(a) * Fraction(float(c)))


def test_power_of_two_scaling_of_x_scales_y_exactly():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((64, 128)) * 0.02).astype(np.float32)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    y, packed, g = oracle.forward(W, x)
    y4 = oracle.forward_packed(packed, g, 64, 128, (x * np.float32(4)).astype(np.float32))
    assert (y4 == y * np.float32(4)).all()


def test_token_rows_are_independent():
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((32, 64)) * 0.02).astype(np.float32)
    x = rng.standard_normal((6, 64)).astype(np.float32)
    y, packed, g = oracle.forward(W, x)
    perm = rng.permutation(6)
    yp = oracle.forward_packed(packed, g, 32, 64, np.ascontiguousarray(x[perm]))
    assert (yp == y[perm]).all()


# ---------------------------------------------------------------- pin-5 special cases
def test_single_weight_single_input():
    W = np.array([[-0.3]], np.float32)
    x = np.array([[0.75], [-2.0]], np.float32)
    y, packed, g = oracle.forward(W, x)
    assert g == fl32(Fraction(float(np.float32(0.3))) + Fraction(float(FEPS)))
    assert oracle.unpack(packed, 1).tolist() == [[-1]]
    xq, s = oracle.quant_act(x)
    assert xq.tolist() == [[127], [-127]]
    for m in range(2):
        a = -int(xq[m, 0])
        e = a * Fraction(float(g)) / Fraction(float(s[m]))
        assert abs(Fraction(float(y[m, 0])) - e) <= abs(e) * Y_REL
    assert abs(float(y[0, 0]) - (-0.3 * 0.75)) < 1e-4


def test_all_zero_weights_and_inputs():
    W = np.zeros((3, 70), np.float32)
    g = oracle.gamma(W)
    assert g == FEPS
    packed, _ = oracle.pack_weights(W)
    assert (packed == 0x55).all()
    x = np.zeros((2, 70), np.float32)
    x[1, 3] = 1.5
    y, _, _ = oracle.forward(W, x)
    assert (y == 0).all()
    xq, s = oracle.quant_act(x)
    assert s[0] == fl32(Fraction(127) / Fraction(float(FEPS)))
    assert (xq[0] == 0).all()
    W2 = np.random.default_rng(1).standard_normal((3, 70)).astype(np.float32)
    y2, _, _ = oracle.forward(W2, x)
    assert (y2[0] == 0).all()


def test_outputs_are_order_free_in_threads():
    rng = np.random.default_rng(2)
    q = rng.integers(-1, 2, size=(300, 257)).astype(np.int8)
    xq = rng.integers(-127, 128, size=(3, 257)).astype(np.int8)
    oracle.set_threads(1)
    a1 = oracle.matmul_i32(q, xq)
    oracle.set_threads(4)
    a4 = oracle.matmul_i32(q, xq)
    oracle.set_threads(1)
    assert (a1 == a4).all()


# ---------------------------------------------------------------- subln RMSNorm
def test_rmsnorm_scale_against_high_precision():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((5, 300)).astype(np.float32)
    x[2] *= 1e-3
    gain = (1 + 0.1 * rng.random(300)).astype(np.float32)
    eps = 1e-5
    xq, s, r = oracle.rmsnorm_quant_act(x, gain, eps)
    for m in range(5):
        ms = sum(Fraction(float(v)) ** 2 for v in x[m]) / 300
        exact_r = 1.0 / math.sqrt(float(ms) + eps)
        assert abs(float(r[m]) - exact_r) <= 3 * 2 ** -24 * exact_r
    # codes are those of u = x * g (absmax quant is invariant under r_t > 0)
    u = (x * gain).astype(np.float32)
    xq_u, s_u = oracle.quant_act(u)
    assert (xq == xq_u).all()
    assert (s == (s_u / r).astype(np.float32)).all()
    # the literal "normalise, then quantise" form agrees up to rounding
    v = ((x * r[:, None]).astype(np.float32) * gain).astype(np.float32)
    xq_v, s_v = oracle.quant_act(v)
    diff = np.abs(xq_v.astype(int) - xq.astype(int))
    assert diff.max() <= 1 and (diff > 0).mean() <= 0.001
    assert np.allclose(s_v, s, rtol=1e-6, atol=0)


def test_rmsnorm_constant_row_closed_form():
    """x = c everywhere: r = 1/sqrt(c^2 + eps), every code is sign(c)*127."""
    x = np.full((2, 64), 0.5, np.float32)
    x[1] = -3.0
    xq, s, r = oracle.rmsnorm_quant_act(x, None, 1e-5)
    assert (xq[0] == 127).all() and (xq[1] == -127).all()
    for m, c in enumerate((0.5, -3.0)):
        assert abs(float(r[m]) - 1 / math.sqrt(c * c + 1e-5)) <= 2 ** -23 / abs(c)
        s_u = np.float32(127) / np.float32(abs(c))
        assert s[m] == np.float32(s_u / r[m])


# ------------------------------------------------------------------ squared ReLU
def test_relu2_closed_form_on_exact_values():
    """relu2 of multiples of 1/8 is exact: max(x, 0)^2 = k^2 / 64 for x = k / 8 > 0,
    and 0 for x <= 0 (including -0.0)."""
    k = np.arange(-200, 201, dtype=np.int64)
    x = (k / 8.0).astype(np.float32)
    u = oracle.relu2(x)
    want = np.where(k > 0, (k * k) / 64.0, 0.0).astype(np.float32)
    assert np.array_equal(u, want)
    assert oracle.relu2(np.array([-0.0], np.float32))[0] == 0.0


def test_relu2_is_the_correctly_rounded_square():
    """For x > 0, fl32(x * x) equals the fp64 product (exact for two binary32
    factors) rounded once to binary32: an independent evaluation path."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1.0, 30.0], 20000)).astype(np.float32)
    u = oracle.relu2(x)
    exact = np.where(x > 0, x.astype(np.float64) * x.astype(np.float64), 0.0).astype(np.float32)
    assert np.array_equal(u, exact)


def test_relu2_quant_act_invariants():
    """Codes of a squared-ReLU input are never negative; every token with a
    positive entry has a code 127; all-negative tokens give all-zero codes."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 700)).astype(np.float32)
    x[5] = -np.abs(x[5])  # a token with no positive entry
    xq, s = oracle.relu2_quant_act(x)
    assert xq.min() >= 0
    for m in range(16):
        if m == 5:
            assert (xq[m] == 0).all() and s[m] == np.float32(127.0) / np.float32(1e-5)
        else:
            assert xq[m].max() == 127
    # it is the plain quantisation applied to the activation values
    xq2, s2 = oracle.quant_act(oracle.relu2(x))
    assert np.array_equal(xq, xq2) and np.array_equal(s, s2)


def test_forward_relu2_equals_forward_of_squared_relu_values():
    """On integer-valued inputs whose positive squares stay below 128 the
    activation scale is 127 / amax and the exact integer dot product of the
    squares is recovered: y = fl32(acc * fl32(gamma / s))."""
    rng = np.random.default_rng(11)
    N, K = 24, 96
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    packed, g = oracle.pack_weights(W)
    x = rng.integers(-11, 12, size=(3, K)).astype(np.float32)
    x[:, 0] = 11.0  # amax of the squares is 121 in every token
    y = oracle.forward_packed_relu2(packed, g, N, K, x)
    u = np.where(x > 0, x * x, 0.0)
    s = np.float32(127.0) / np.float32(121.0)
    xq = np.clip(np.rint((u.astype(np.float32) * s).astype(np.float32)), -128, 127).astype(np.int64)
    q = oracle.unpack(packed, K).astype(np.int64)
    acc = xq @ q.T
    c = np.float32(np.float32(g) / s)
    assert np.array_equal(y, (acc.astype(np.float32) * c).astype(np.float32))


# ------------------------------------------------------------------ output variants
def test_output_bf16_rounding_pins():
    """bf16 output rounding against values whose bf16 neighbours are known:
    exact values pass through, halfway cases go to the even neighbour, and the
    result is the nearest bf16 (checked against an fp64 nearest search)."""
    exact = np.array([1.0, -2.5, 0.0, 3.140625, 65280.0], np.float32)
    assert np.array_equal(oracle.output(exact, bf16=True),
                          (exact.view(np.uint32) >> 16).astype(np.uint16))
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: to even (1.0); 1 + 3 * 2^-8 -> 1 + 2^-6
    half = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], np.float32)
    assert oracle.output(half, bf16=True).tolist() == [0x3F80, 0x3F82, 0xBF80]
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(5000) * 100).astype(np.float32)
    b = oracle.output(v, bf16=True)
    up = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    lo = ((b.astype(np.uint32) - 1) << 16).view(np.float32).astype(np.float64)
    hi = ((b.astype(np.uint32) + 1) << 16).view(np.float32).astype(np.float64)
    d = np.abs(up - v.astype(np.float64))
    assert (d <= np.abs(lo - v) + 0).all() and (d <= np.abs(hi - v)).all()


def test_output_residual_is_one_fp32_add():
    """With a residual the output is the correctly rounded fp32 sum (the exact
    fp64 sum of two binary32 values rounded once)."""
    rng = np.random.default_rng(9)
    y = (rng.standard_normal(4000) * 3).astype(np.float32)
    r = (rng.standard_normal(4000) * 1000).astype(np.float32)
    out = oracle.output(y, r)
    assert np.array_equal(out, (y.astype(np.float64) + r.astype(np.float64)).astype(np.float32))
    assert np.array_equal(oracle.output(y), y)


# ------------------------------------------------- grouped weight scales
# "BitNet b1.58 深度解析" (chenxutan.com) section 5.2 groups the weight's
# output rows by 128 for its scales, section 2.2 keeps one scale per output
# row; the absmean-round quantiser is kept, only the mean's support narrows.

def test_groups_of_all_rows_are_the_per_tensor_scale():
    """G = N is the per-tensor case: same scale, same codes, same outputs."""
    rng = np.random.default_rng(11)
    for N, K in ((256, 512), (96, 100), (1, 7)):
        W = rng.normal(0, 0.02, (N, K)).astype(np.float32)
        p1, g1 = oracle.pack_weights(W)
        p2, g2 = oracle.pack_weights_groups(W, N)
        assert g2.shape == (1,) and g2[0] == g1
        assert np.array_equal(p1, p2)
        x = rng.normal(0, 1, (3, K)).astype(np.float32)
        y1 = oracle.forward_packed(p1, g1, N, K, x)
        y2 = oracle.forward_packed_groups(p2, g2, N, N, K, x)
        assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_groups_hand_worked_per_row_example():
    """Two rows, one scale each (G = 1), every value derived by hand.
    Row 0 = [0.5, -0.5, 0.25, 0]: mean|w| = 1.25 / 4 = 0.3125, w / gamma =
    [1.6, -1.6, 0.8, 0] -> rne, clip -> [1, -1, 1, 0].  Row 1 = [4, -2, 0, 1]:
    mean 7 / 4 = 1.75, w / gamma = [2.29, -1.14, 0, 0.57] -> [1, -1, 0, 1].
    (One scale for both rows, mean 8.25 / 8 = 1.03125, would zero row 0.)
    Token [1, 2, 3, 4]: s = 127 / 4 = 31.75, x s = [31.75, 63.5, 95.25, 127]
    -> [32, 64, 95, 127] (63.5 rounds to even); acc = [32 - 64 + 95,
    32 - 64 + 127] = [63, 95]; y_n = acc_n * gamma_n / 31.75."""
    W = np.array([[0.5, -0.5, 0.25, 0.0], [4.0, -2.0, 0.0, 1.0]], np.float32)
    g = oracle.gamma_groups(W, 1)
    assert g[0] == fl32(Fraction(5, 16) + Fraction(float(np.float32(1e-5))))
    assert g[1] == fl32(Fraction(7, 4) + Fraction(float(np.float32(1e-5))))
    q = oracle.ternarize_groups(W, g, 1)
    assert q.tolist() == [[1, -1, 1, 0], [1, -1, 0, 1]]
    assert oracle.ternarize(W, oracle.gamma(W)).tolist()[0] == [0, 0, 0, 0]
    packed, g2 = oracle.pack_weights_groups(W, 1)
    assert np.array_equal(g, g2)
    x = np.array([[1.0, 2.0, 3.0, 4.0]], np.float32)
    xq, s = oracle.quant_act(x)
    assert xq.tolist() == [[32, 64, 95, 127]] and s[0] == np.float32(31.75)
    y = oracle.forward_packed_groups(packed, g, 1, 2, 4, x)
    for n, acc in enumerate((63, 95)):
        exact = Fraction(acc) * Fraction(float(g[n])) / Fraction(127, 4)
        assert abs(Fraction(float(y[0, n])) - exact) <= Y_REL * abs(exact)


def test_groups_are_the_per_tensor_scale_of_each_row_block():
    """G = 128 on three blocks of rows with magnitudes 1e-3, 1 and 30: each
    block's codes and scale are the per-tensor ones of that block alone."""
    rng = np.random.default_rng(12)
    K = 200
    W = np.concatenate([rng.normal(0, a, (128, K)) for a in (1e-3, 1.0, 30.0)]).astype(np.float32)
    packed, g = oracle.pack_weights_groups(W, 128)
    assert g.shape == (3,)
    for b in range(3):
        pb, gb = oracle.pack_weights(W[128 * b:128 * (b + 1)])
        assert g[b] == gb
        assert np.array_equal(packed[128 * b:128 * (b + 1)], pb)
    # the small block survives its own scale (about a third zeros), and
    # would not survive one scale for the whole tensor
    q = oracle.unpack(packed, K)
    assert 0.25 < np.mean(q[:128] == 0) < 0.45
    assert np.all(oracle.ternarize(W, oracle.gamma(W))[:128] == 0)


def test_groups_per_row_closed_form():
    """W[n] = a_n t_n with t ternary and exactly a quarter zeros per row: the
    row's absmean is 0.75 a_n, so W / gamma_n = +-1.33 or 0 and the codes are
    t itself for scales a_n over five decades; y against exact rationals."""
    rng = np.random.default_rng(13)
    N, K, M = 40, 64, 3
    t = np.zeros((N, K), np.int8)
    for n in range(N):
        nz = rng.permutation(K)[:48]
        t[n, nz] = rng.choice(np.array([-1, 1], np.int8), 48)
    a = (10.0 ** rng.uniform(-3, 2, N)).astype(np.float32)
    W = (t.astype(np.float32) * a[:, None]).astype(np.float32)
    packed, g = oracle.pack_weights_groups(W, 1)
    assert np.array_equal(oracle.unpack(packed, K), t)
    x = rng.normal(0, 1, (M, K)).astype(np.float32)
    y = oracle.forward_packed_groups(packed, g, 1, N, K, x)
    xq, s = oracle.quant_act(x)
    for m in range(M):
        for n in range(N):
            acc = int(np.dot(t[n].astype(np.int64), xq[m].astype(np.int64)))
            exact = Fraction(acc) * Fraction(float(g[n])) / Fraction(float(s[m]))
            assert abs(Fraction(float(y[m, n])) - exact) <= Y_REL * abs(exact)


@pytest.mark.parametrize("seed", range(6))
def test_groups_random_shapes_match_per_tensor_of_each_group(seed):
    """For random N, K and group sizes G dividing N, every group's scale and
    codes equal the per-tensor oracle applied to that group's rows alone, and
    the grouped rescale of each group's rows equals the per-tensor rescale."""
    rng = np.random.default_rng(100 + seed)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    N = G * int(rng.integers(1, 6))
    K = int(rng.integers(1, 150))
    W = (rng.normal(0, 1, (N, K)) * (10.0 ** rng.uniform(-3, 1, (N, 1)))).astype(np.float32)
    packed, g = oracle.pack_weights_groups(W, G)
    x = rng.normal(0, 1, (3, K)).astype(np.float32)
    y = oracle.forward_packed_groups(packed, g, G, N, K, x)
    for b in range(N // G):
        rows = slice(b * G, (b + 1) * G)
        pb, gb = oracle.pack_weights(W[rows])
        assert g[b] == gb
        assert np.array_equal(packed[rows], pb)
        yb = oracle.forward_packed(pb, gb, G, K, x)
        assert np.array_equal(y[:, rows].view(np.uint32), yb.view(np.uint32))
