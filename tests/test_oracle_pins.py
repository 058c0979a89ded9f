"""Pins for the CPU oracle: each check fixes the oracle to something other than
itself -- the format specifications' printed values (``tests/golden``), a
library float8 decoder/encoder (torch ``float8_e4m3fn``), brute force on tiny
inputs, closed forms and invariants of the quantisation recipe.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
from conftest import read_golden

GRID = {int(c): float(v) for c, v in read_golden("e2m1_grid.txt")}
FACTS = {r[0]: (r[1], float(r[2])) for r in read_golden("e4m3_facts.txt")}
DIV = FACTS["tensor_scale_divisor"][1]


def e2m1_from_grid(code):
    """Independent E2M1 decode: the printed grid plus the sign bit."""
    v = GRID[code & 7]
    return -v if code & 8 else v


def e4m3_from_torch(codes):
    """Independent E4M3 decode: torch's float8_e4m3fn reinterpretation."""
    t = torch.as_tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def deq_independent(q, s, g):
    """Dequantise with the independent decoders above, in FP64."""
    rows, half = q.shape
    k = half * 2
    codes = np.empty((rows, k), np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    lut = np.array([e2m1_from_grid(c) for c in range(16)])
    sc = e4m3_from_torch(s.reshape(-1)).reshape(s.shape)
    return lut[codes] * np.repeat(sc, 16, axis=1) * float(np.float32(g))


# ---- element formats ---------------------------------------------------------

def test_e2m1_value_grid():
    for c in range(16):
        assert oracle.e2m1_value(c) == e2m1_from_grid(c)
        # sign of the zero code survives
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_e4m3_decode_all_256_codes_match_torch():
    ref = e4m3_from_torch(np.arange(256))
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), hex(c)
        else:
            assert v == ref[c], hex(c)
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_printed_facts():
    for name, (code, value) in FACTS.items():
        if code == "-":
            continue
        assert oracle.e4m3_value(int(code, 16)) == value, name
    assert DIV == 6.0 * 448.0


def test_e2m1_tie_table():
    for inp, code, val in read_golden("e2m1_ties.txt"):
        assert oracle.e2m1_encode(float(inp)) == int(code), inp
        assert oracle.e2m1_encode(-float(inp)) == int(code) | 8, inp
        assert GRID[int(code)] == float(val)


def test_e2m1_encode_is_nearest_brute_force():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), np.linspace(-6.5, 6.5, 2601)]).astype(np.float32)
    grid = np.array([e2m1_from_grid(c) for c in range(16)])
    for v in vals:
        c = oracle.e2m1_encode(float(v))
        d = np.abs(grid - float(v))
        # nearest among all 16 codes (saturating beyond 6 is "nearest" too)
        assert d[c] == d.min(), (v, c)
        if v != 0:
            assert (c >> 3) == (1 if v < 0 else 0)


def test_e2m1_saturation_and_signed_zero():
    assert oracle.e2m1_encode(1e30) == 7
    assert oracle.e2m1_encode(-1e30) == 15
    assert oracle.e2m1_encode(float("inf")) == 7
    assert oracle.e2m1_encode(-0.0) == 8
    assert oracle.e2m1_encode(-0.2) == 8
    assert oracle.e2m1_encode(0.0) == 0


def test_e4m3_encode_matches_torch_cast_in_range():
    """torch rounds to nearest even with subnormals but does not saturate
    (480 -> NaN), so compare only below the 448/480 midpoint."""
    rng = np.random.default_rng(2)
    mids = [(e4m3_from_torch([c])[0] + e4m3_from_torch([c + 1])[0]) / 2 for c in range(0, 0x7E)]
    vals = np.concatenate([
        np.exp2(rng.uniform(-14, 8.8, 6000)),
        np.array(mids),                       # every tie
        np.nextafter(np.array(mids, np.float32), np.float32(0)),
        np.nextafter(np.array(mids, np.float32), np.float32(1e9)),
        [0.0, 2.0 ** -10, 2.0 ** -9, 448.0, 464.0],
    ]).astype(np.float32)
    vals = vals[vals <= 464.0]
    ref = torch.as_tensor(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        assert oracle.e4m3_encode(float(v)) == int(r), v


def test_e4m3_encode_saturates():
    for v in (448.0, 464.0, 464.1, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E


# ---- quantisation recipe -------------------------------------------------------

def test_global_scale_definition():
    t = synthetic.activations(3, 256, seed=4)
    g = oracle.global_scale(t)
    assert g == np.float32(np.abs(t).max()) / np.float32(DIV)


def test_round_trip_exact_on_grid_blocks():
    """Blocks built from grid values times a power-of-two scale, with each
    block's largest magnitude 6, dequantise back exactly."""
    rng = np.random.default_rng(5)
    rows, k = 4, 128
    codes = rng.integers(0, 16, size=(rows, k))
    codes[:, ::16] = 7                                   # a +6 in every block
    vals = np.array([e2m1_from_grid(c) for c in codes.ravel()]).reshape(rows, k)
    gains = np.exp2(rng.integers(-6, 3, size=(rows, k // 16)).astype(np.float64))
    t = (vals * np.repeat(gains, 16, axis=1)).astype(np.float32)
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    back = deq_independent(q, s, g)
    # the E4M3 block scale is exact here only if bmax/(6g) is; check the
    # invariant that matters instead: every element is recovered to within
    # the scale's rounding and the +6 element lands on code 7.
    assert np.all((q[:, ::8] & 15) == 7)
    np.testing.assert_allclose(back, t, rtol=2 ** -4, atol=0)


def test_round_trip_exact_when_scale_exact():
    """With g a power of two times 1/2688 chosen so that bmax/(6g) is a
    representable E4M3 value, quantise->dequantise is the identity."""
    rng = np.random.default_rng(6)
    k = 64
    codes = rng.integers(0, 16, size=(2, k))
    codes[:, ::16] = 7
    vals = np.array([e2m1_from_grid(c) for c in codes.ravel()]).reshape(2, k)
    t = vals.astype(np.float32)           # block max 6 everywhere
    g = np.float32(0.25)                  # 6g = 1.5 ; s = 6/1.5 = 4 exact ; S = 1
    q, s = oracle.quantize(t, g)
    assert np.all(s == 0x48)              # E4M3 4.0 = 0 1001 000
    np.testing.assert_array_equal(deq_independent(q, s, g), t.astype(np.float64))


def test_block_max_maps_to_six_when_scale_normal():
    t = synthetic.log_uniform_blocks(16, 512, seed=7, lo_exp=-3, hi_exp=3)
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    codes = np.empty(t.shape, np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    blocks = np.abs(t).reshape(16, -1, 16)
    arg = blocks.argmax(axis=2)
    cb = codes.reshape(16, -1, 16)
    for r in range(16):
        for b in range(blocks.shape[1]):
            if s[r, b] >= 0x08:                     # normal E4M3 scale
                assert cb[r, b, arg[r, b]] & 7 == 7


def test_dequant_error_bound():
    """|deq - t| <= half the local E2M1 step times S, and at most S*0.5 for
    the saturating top interval only when the scale itself rounded down."""
    t = synthetic.log_uniform_blocks(8, 1024, seed=8)
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    back = deq_independent(q, s, g)
    S = np.repeat(e4m3_from_torch(s.reshape(-1)).reshape(s.shape) * float(g), 16, axis=1)
    err = np.abs(back - t.astype(np.float64))
    v = np.abs(t.astype(np.float64)) / np.where(S > 0, S, 1)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    ok = (S == 0) | (err <= 0.5 * step * S * (1 + 1e-6)) | (v > 6)
    assert ok.all()
    # saturated elements dequantise to exactly +-6 S
    sat = (S > 0) & (v > 6)
    np.testing.assert_allclose(np.abs(back[sat]), 6 * S[sat], rtol=1e-12)


def test_zero_tensor_and_zero_blocks():
    t = np.zeros((2, 64), np.float32)
    g = oracle.global_scale(t)
    assert g == 0
    q, s = oracle.quantize(t, g)
    assert not q.any() and not s.any()
    # negative zeros keep their sign bit
    t[1, 3] = -0.0
    q, s = oracle.quantize(t, g)
    assert q[1, 1] == 0x80
    # a zero block inside a non-zero tensor
    t = synthetic.activations(1, 64, seed=9, outliers=False)
    t[0, 16:32] = 0
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    assert s[0, 1] == 0 and not q[0, 8:16].any() and s[0, 0] != 0


def test_tiny_blocks_underflow_to_zero_scale():
    """A block far below the tensor amax rounds its E4M3 scale to 0."""
    t = np.ones((1, 32), np.float32)
    t[0, 16:] = 1e-7
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    assert s[0, 1] == 0 and not q[0, 8:].any()


def test_pack_low_nibble_first():
    t = np.zeros((1, 16), np.float32)
    t[0, 0] = 6.0      # code 7, element 0 -> low nibble of byte 0
    t[0, 1] = -3.0     # code 13, element 1 -> high nibble of byte 0
    g = np.float32(0.25)  # S = 1 with bmax 6
    q, s = oracle.quantize(t, g)
    assert q[0, 0] == (13 << 4) | 7


def test_pack_weight_matches_quantize_with_own_scale():
    w = synthetic.weights(8, 64, 0.02, seed=10)
    q, s, g = oracle.pack_weight(w)
    q2, s2 = oracle.quantize(w, oracle.global_scale(w))
    assert g == oracle.global_scale(w)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)


def test_dequantize_matches_independent_decoders():
    t = synthetic.log_uniform_blocks(5, 256, seed=11)
    g = oracle.global_scale(t)
    q, s = oracle.quantize(t, g)
    np.testing.assert_array_equal(oracle.dequantize(q, s, g), deq_independent(q, s, g))


# ---- GEMM ------------------------------------------------------------------------

@pytest.mark.parametrize("m,k,n", [(1, 16, 1), (2, 32, 3), (8, 48, 17), (3, 256, 5), (8, 256, 33)])
def test_gemm_equals_dense_fp64_matmul(m, k, n):
    x = synthetic.activations(m, k, seed=20 + k)
    w = synthetic.weights(n, k, 0.02, seed=30 + n)
    gx = oracle.global_scale(x)
    xq, xs = oracle.quantize(x, gx)
    wq, ws, gw = oracle.pack_weight(w)
    dense = deq_independent(xq, xs, gx) @ deq_independent(wq, ws, gw).T
    y = oracle.gemm(xq, xs, gx, wq, ws, gw)
    np.testing.assert_allclose(y, dense, rtol=1e-13, atol=1e-300)


def test_gemm_closed_form_all_ones():
    """X = W = 1: every block's scale saturates to 448, every code is 6, so
    y = K * (6*448*gX) * (6*448*gW) with gX = gW = fl32(1/2688)."""
    k, n = 64, 3
    x = np.ones((2, k), np.float32)
    w = np.ones((n, k), np.float32)
    gx = oracle.global_scale(x)
    xq, xs = oracle.quantize(x, gx)
    wq, ws, gw = oracle.pack_weight(w)
    assert np.all(xs == 0x7E) and np.all(xq == 0x77)
    y = oracle.gemm(xq, xs, gx, wq, ws, gw)
    expect = k * (2688.0 * float(gx)) * (2688.0 * float(gw))
    np.testing.assert_array_equal(y, np.full((2, n), expect))


def test_gemm_single_block_closed_form():
    """One non-zero 16-block per row: y is that block's products alone."""
    k = 64
    x = np.zeros((1, k), np.float32)
    w = np.zeros((1, k), np.float32)
    x[0, 32:48] = np.array([6, -3, 2, 0.5] * 4, np.float32)
    w[0, 32:48] = np.array([1.5, 4, -6, 1] * 4, np.float32)
    gx = oracle.global_scale(x)
    gw = oracle.global_scale(w)
    xq, xs = oracle.quantize(x, gx)
    wq, ws = oracle.quantize(w, gw)
    y = oracle.gemm(xq, xs, gx, wq, ws, gw)[0, 0]
    sx = e4m3_from_torch([xs[0, 2]])[0] * float(gx)
    sw = e4m3_from_torch([ws[0, 2]])[0] * float(gw)
    xv = [e2m1_from_grid(int(oracle.e2m1_encode(np.float32(v) / np.float32(sx)))) for v in x[0, 32:48]]
    wv = [e2m1_from_grid(int(oracle.e2m1_encode(np.float32(v) / np.float32(sw)))) for v in w[0, 32:48]]
    assert y == pytest.approx(sx * sw * float(np.dot(xv, wv)), rel=1e-15)
    # and a closed form that needs no encoder: values are exactly on the grid
    # times S when S is exact; the product pattern sums to 4*(9-12-12+0.5).
    assert float(np.dot(xv, wv)) == pytest.approx(4 * (6 * 1.5 - 3 * 4 - 2 * 6 + 0.5 * 1), rel=0.2)


def test_gemm_sampled_matches_full():
    m, k, n = 4, 512, 40
    x = synthetic.activations(m, k, seed=40)
    w = synthetic.weights(n, k, 0.02, seed=41)
    gx = oracle.global_scale(x)
    xq, xs = oracle.quantize(x, gx)
    wq, ws, gw = oracle.pack_weight(w)
    y = oracle.gemm(xq, xs, gx, wq, ws, gw)
    ms = np.array([0, 3, 2, 1, 3])
    ns = np.array([0, 39, 7, 20, 0])
    np.testing.assert_array_equal(oracle.gemm_sampled(xq, xs, gx, wq, ws, gw, ms, ns), y[ms, ns])


# ---- BF16 conversions (production activation / output dtype) ----------------

def test_bf16_golden_facts():
    """Hand-derived values (tests/golden/bf16_facts.txt: IEEE 754 binary32
    layout, BF16 = its upper 16 bits, round to nearest even)."""
    vals, bits = [], []
    for row in read_golden("bf16_facts.txt"):
        v, b = row[0], row[1]
        vals.append(float(v))
        bits.append(int(b, 16))
    got = oracle.f32_to_bf16(np.array(vals, np.float32))
    np.testing.assert_array_equal(got, np.array(bits, np.uint16))
    np.testing.assert_array_equal(oracle.bf16_to_f32(np.array(bits, np.uint16)),
                                  oracle.bf16_to_f32(got))


def test_bf16_widen_is_upper_half_of_binary32():
    """Every finite BF16 pattern widens to the binary32 with those 16 bits on
    top and zeros below (closed form, checked on the bit patterns)."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    w = oracle.bf16_to_f32(b)
    np.testing.assert_array_equal(w.view(np.uint32), b.astype(np.uint32) << 16)


def test_bf16_round_matches_torch_and_round_trips():
    """Narrowing equals torch's BF16 cast (a library rounding routine) on
    random values over many decades, on every exact tie between neighbours
    near 1, 2^-100 and 2^100, and one binary32 ulp either side of each; and
    narrowing a widened BF16 gives it back."""
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.uniform(-60, 60, 20000))).astype(np.float32)
    ties = []
    for e in (0, -100, 100):
        j = np.arange(0, 128)
        lo = (1.0 + j / 128.0) * 2.0 ** e
        mid = (lo + 2.0 ** e / 256.0).astype(np.float32)            # exact halfway points
        ties += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf))]
    v = np.concatenate([v, *ties, -np.concatenate(ties)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16(v), want)
    b = np.arange(0, 0x7F80, dtype=np.uint16)                     # every finite positive
    np.testing.assert_array_equal(oracle.f32_to_bf16(oracle.bf16_to_f32(b)), b)
