"""Pins of the oracle's MXFP4-weight variant (E2M1 codes, 1x32 UE8M0 scales), CPU only.

OCP Microscaling Formats (MX) v1.0 fixes the element format (section 5.3.3,
FP4 E2M1: largest normal 6.0, smallest normal 1.0, the one subnormal 0.5, no
infinities or NaN) and the shared exponent X = floor(log2(amax)) - 2
(section 6.3; 2 = the exponent of 6.0 = 1.5 * 2^2).  These tests check the
oracle's E2M1 table against those printed values, its encoder against an
exhaustive nearest-value search over all 16 codes, the quantiser against
closed forms and the half-spacing bound, the weight packing layout, and the
layer (MXFP4 weights, MXFP8 activations) against a dequantise-first brute
force with plain fp64 matmuls.
"""
import numpy as np
import pytest

import oracle
from test_oracle_mx_pins import mx_dequant
from test_oracle_pins import _router_inputs, bf16_bits, f32

# OCP MX v1.0, section 5.3.3: the eight non-negative FP4 E2M1 values (codes 0-7;
# codes 8-15 are their negatives, code 8 being -0).
E2M1_PRINTED = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_table():
    return np.array([oracle.e2m1_decode(c) for c in range(16)])


def mx4_dequant(q, s):
    return e2m1_table()[q] * np.repeat(np.exp2(s.astype(np.float64) - 127.0), 32, axis=-1)


def nearest_even_e2m1(v: float) -> int:
    """Exhaustive search: the code whose value is nearest to v (|v| clipped to 6),
    ties to the code with an even mantissa bit; the sign of v is kept."""
    a = min(abs(v), 6.0)
    best, dbest = None, None
    for c in range(8):
        d = abs(E2M1_PRINTED[c] - a)
        if best is None or d < dbest or (d == dbest and c % 2 == 0):
            best, dbest = c, d
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_table_is_the_printed_format():
    t = e2m1_table()
    assert list(t[:8]) == E2M1_PRINTED
    assert list(-t[8:]) == E2M1_PRINTED and np.signbit(t[8])


def test_e2m1_encoder_matches_exhaustive_search():
    grid = np.arange(-8.0, 8.0 + 1e-9, 1.0 / 64.0)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near = np.concatenate([ties, np.nextafter(ties.astype(np.float32), np.float32(0)),
                           np.nextafter(ties.astype(np.float32), np.float32(10))]).astype(np.float64)
    rng = np.random.default_rng(2)
    vals = np.concatenate([grid, near, -near, rng.uniform(-10, 10, 2000), [0.0, -0.0, 1e-30, -1e-30, 1e30, -1e30]])
    vals = vals.astype(np.float32)
    got = np.array([oracle.e2m1_encode(float(v)) for v in vals])
    want = np.array([nearest_even_e2m1(float(v)) for v in vals])
    bad = np.nonzero(got != want)[0]
    assert len(bad) == 0, [(float(vals[i]), int(got[i]), int(want[i])) for i in bad[:8]]


def test_mx4_scale_closed_forms():
    rows = np.zeros((7, 128), np.float32)
    rows[0, :32] = 6.0 * 2.0 ** 3            # amax = 6 * 2^3: X = 3, the amax element is code 7 (6.0)
    rows[1, :32] = 2.0 ** -4                 # amax = 2^-4: X = -6, elements 4.0 (code 6)
    rows[2, :32] = 7.5 * 2.0 ** 10           # top binade above 6: X = 10, saturates to 6.0
    rows[3, 32:64] = -0.0                    # all-zero group of signed zeros: byte 0, codes +0
    rows[4, :32] = 2.0 ** -130               # amax below 2^-125: X clamped to -127
    rows[5, :32] = 3.0e38                    # floor(log2(3e38)) = 127: X = 125
    rows[6, :32] = np.linspace(-1.0, 1.0, 32)  # amax = 1: X = -2, the ends scale to +-4.0 (code 6, 14)
    q, s = oracle.mx4_quant_rows_f32(rows)
    assert s[0, 0] == 127 + 3 and np.all(q[0, :32] == 7)
    assert s[1, 0] == 127 - 6 and np.all(q[1, :32] == 6)
    assert s[2, 0] == 127 + 10 and np.all(q[2, :32] == 7)
    assert s[3, 1] == 0 and np.all(q[3, 32:64] == 0)
    assert s[4, 0] == 0  # X = -127: 2^-130 / 2^-127 = 0.125 rounds to 0
    assert np.all(q[4, :32] == 0)
    assert s[5, 0] == 127 + 125
    assert s[6, 0] == 127 - 2 and q[6, 31] == 6 and q[6, 0] == 14
    assert np.all(s[:, 3] == 0)


def test_mx4_round_trip_within_half_spacing():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((32, 256)) * np.exp2(rng.uniform(-20, 20, (32, 1)))).astype(np.float32)
    q, s = oracle.mx4_quant_rows_f32(x)
    d = mx4_dequant(q, s)
    scale = np.repeat(np.exp2(s.astype(np.float64) - 127.0), 32, axis=-1)
    a = np.abs(x.astype(np.float64)) / scale          # |v| / 2^X, in [0, 8)
    # spacing of E2M1 around a: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]; above 6: saturated
    spacing = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    inrange = a <= 6.0
    err = np.abs(d - x) / scale
    assert np.all(err[inrange] <= spacing[inrange] / 2 + 1e-12)
    assert np.all(np.abs(d[~inrange]) / scale[~inrange] == 6.0)
    # every group's amax lands in the top binade [4, 8) of the scaled range
    amax = np.abs(x).reshape(32, 8, 32).max(axis=2) / np.exp2(s.astype(np.float64) - 127.0)
    assert np.all((amax >= 4.0) & (amax < 8.0))


def test_mx4_weight_pack_layout_and_padding():
    E, H, I = 2, 100, 70
    rng = np.random.default_rng(10)
    w13 = rng.standard_normal((E, 2 * I, H)).astype(np.float32)
    w2 = rng.standard_normal((E, H, I)).astype(np.float32)
    q13, s13 = oracle.mx4_pack_w13(w13)
    q2, s2 = oracle.mx4_pack_w2(w2)
    Ip = 128
    for e in range(E):
        qg, sg = oracle.mx4_quant_rows_f32(w13[e, :I])
        qu, su = oracle.mx4_quant_rows_f32(w13[e, I:])
        assert np.array_equal(q13[e, :I], qg) and np.array_equal(s13[e, :I], sg)
        assert np.array_equal(q13[e, Ip:Ip + I], qu) and np.array_equal(s13[e, Ip:Ip + I], su)
        assert not q13[e, I:Ip].any() and not q13[e, Ip + I:].any() and not s13[e, I:Ip].any()
        qd, sd = oracle.mx4_quant_rows_f32(w2[e])
        assert np.array_equal(q2[e, :H], qd) and np.array_equal(s2[e, :H], sd) and not q2[e, H:].any()
    assert q13.max() <= 15 and q2.max() <= 15


def _mx4_brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I):
    """Dequantise everything first (E2M1 weights and e4m3 activations, times
    2^(byte-127) per 32-group), then plain fp64 matmuls; h is requantised with
    the oracle's MXFP8 quantiser."""
    T, H = x.shape
    Ip = w2q.shape[2]
    r = oracle.router(x, rw, rb, k)
    xq, sx = oracle.mx_quant_rows_bf16(x)
    xd = mx_dequant(xq, sx)
    W13 = mx4_dequant(w13q, s13)
    W2 = mx4_dequant(w2q, s2)
    out = np.zeros((T, H))
    ys = np.zeros((T, k, H))
    for t in range(T):
        for j in range(k):
            e = r["idx"][t, j]
            gu = W13[e] @ xd[t]
            g = gu[:I] + f32(b13[e, :I])
            u = gu[Ip:Ip + I] + f32(b13[e, I:])
            h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
            hq, sh = oracle.mx_quant_rows_f32(h[None, :])
            y = W2[e, :H] @ mx_dequant(hq, sh)[0] + f32(b2[e])
            ys[t, j] = y
            out[t] += f32(r["w_bf16"][t, j]).astype(np.float64) * y
    return out, ys


@pytest.mark.parametrize("T,H,I,E,k", [(5, 128, 128, 4, 2), (6, 200, 136, 5, 3)])
def test_mx4_layer_matches_dequantise_first_brute_force(T, H, I, E, k):
    rng = np.random.default_rng(T * 91 + H)
    x, rw, rb = _router_inputs(T, H, E, seed=T + 5 * H)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    b13 = bf16_bits((rng.standard_normal((E, 2 * I)) * 0.1).astype(np.float32))
    b2 = bf16_bits((rng.standard_normal((E, H)) * 0.1).astype(np.float32))
    w13q, s13 = oracle.mx4_pack_w13(w13)
    w2q, s2 = oracle.mx4_pack_w2(w2)
    out, inter = oracle.mx4_forward(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, want_intermediates=True)
    ref, ys = _mx4_brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I)
    assert np.allclose(inter["y"].reshape(T, k, H), ys, rtol=1e-10, atol=1e-12)
    assert np.array_equal(out, oracle.bf16_from_f64(ref))
    # the FP4 weights change the result: a plain MXFP8-weight layer differs
    w13q8, s138 = oracle.mx_pack_w13(w13)
    w2q8, s28 = oracle.mx_pack_w2(w2)
    out8 = oracle.mx_forward(x, rw, rb, w13q8, s138, b13, w2q8, s28, b2, k)
    assert not np.array_equal(out, out8)
