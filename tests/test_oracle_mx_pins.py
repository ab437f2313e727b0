"""Pins of the oracle's MXFP8 variant (1x32 power-of-two UE8M0 scales), CPU only.

The MX scale of a 32-value group is defined by the OCP Microscaling (MX)
specification v1.0, section 6.3: X = floor(log2(amax)) - 8 for e4m3 (whose
largest normal is 1.75 * 2^8), stored as the byte X + 127; the codes are
e4m3(v / 2^X).  These tests check that definition against closed forms,
against numpy's frexp with PyTorch's float8_e4m3fn conversion (a library
routine) on values in range, and the layer against a dequantise-first brute
force with plain fp64 matmuls.
"""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import _router_inputs, bf16_bits, f32


def mx_dequant(q, s):
    tab = oracle.e4m3_decode_table()
    return tab[q] * np.repeat(np.exp2(s.astype(np.float64) - 127.0), 32, axis=-1)


def test_mx_scale_closed_forms():
    rows = np.zeros((6, 128), np.float32)
    rows[0, :32] = 1.75 * 2.0 ** 5          # amax = 1.75 * 2^5: X = 5 - 8, element = 448 exactly
    rows[1, :32] = 1.9 * 2.0 ** 5           # top binade above 448: saturates to 448
    rows[2, :32] = 2.0 ** np.arange(-16, 16)  # powers of two 2^-16 .. 2^15: X = 7, codes exact from 2^-9 up
    rows[3, 32:64] = -0.0                    # all-zero group (signed zeros): byte 0, codes +0
    rows[4, :32] = 2.0 ** -140              # amax below 2^-127 * 2^8: X clamped to -127
    rows[5, :32] = 3.0e38                   # floor(log2(3e38)) = 127: X = 119
    q, s = oracle.mx_quant_rows_f32(rows)
    assert s[0, 0] == 127 - 3 and np.all(q[0, :32] == 0x7E)
    assert s[1, 0] == 127 - 3 and np.all(q[1, :32] == 0x7E)
    assert s[2, 0] == 127 + 7
    d = mx_dequant(q[2:3], s[2:3])[0, :32]
    exact = 2.0 ** np.arange(-16, 16)
    ok = exact >= 2.0 ** 7 * 2.0 ** -9  # values down to the smallest e4m3 subnormal times 2^X are exact
    assert np.array_equal(d[ok], exact[ok])
    assert s[3, 1] == 0 and np.all(q[3, 32:64] == 0)
    assert s[4, 0] == 0 and np.all(q[4, :32] == oracle.e4m3_encode(np.float32([2.0 ** -13]))[0])
    assert s[5, 0] == 127 + 119
    assert np.all(s[:, 3] == 0)  # untouched trailing groups


def test_mx_matches_frexp_and_torch_float8_in_range():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    q, s = oracle.mx_quant_rows_f32(x)
    g = x.reshape(64, 8, 32)
    amax = np.abs(g).max(axis=2)
    _, e = np.frexp(amax.astype(np.float64))
    X = e - 1 - 8
    assert np.array_equal(s.astype(np.int64) - 127, X)
    scaled = (g.astype(np.float64) * np.exp2(-X)[..., None]).astype(np.float32)
    inrange = np.abs(scaled) <= 448.0
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qq = q.reshape(64, 8, 32)
    assert np.array_equal(qq[inrange], ref[inrange])
    assert np.all(qq[~inrange] & 0x7F == 0x7E)  # the rest saturate to +-448


def test_mx_weight_pack_layout_and_padding():
    E, H, I = 2, 100, 70
    rng = np.random.default_rng(9)
    w13 = rng.standard_normal((E, 2 * I, H)).astype(np.float32)
    w2 = rng.standard_normal((E, H, I)).astype(np.float32)
    q13, s13 = oracle.mx_pack_w13(w13)
    q2, s2 = oracle.mx_pack_w2(w2)
    Hp, Ip = 128, 128
    for e in range(E):
        qg, sg = oracle.mx_quant_rows_f32(w13[e, :I])
        qu, su = oracle.mx_quant_rows_f32(w13[e, I:])
        assert np.array_equal(q13[e, :I], qg) and np.array_equal(s13[e, :I], sg)
        assert np.array_equal(q13[e, Ip:Ip + I], qu) and np.array_equal(s13[e, Ip:Ip + I], su)
        assert not q13[e, I:Ip].any() and not s13[e, I:Ip].any()
        assert not q13[e, Ip + I:].any() and not s13[e, Ip + I:].any()
        qd, sd = oracle.mx_quant_rows_f32(w2[e])
        assert np.array_equal(q2[e, :H], qd) and np.array_equal(s2[e, :H], sd) and not q2[e, H:].any()
    assert s13.shape == (E, 2 * Ip, Hp // 32) and s2.shape == (E, Hp, Ip // 32)


def _mx_brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I):
    """Dequantise everything first (codes x 2^(byte-127) per 32-group), then
    plain fp64 matmuls; h is requantised with the oracle's MX quantiser."""
    T, H = x.shape
    Ip = w2q.shape[2]
    r = oracle.router(x, rw, rb, k)
    xq, sx = oracle.mx_quant_rows_bf16(x)
    xd = mx_dequant(xq, sx)
    W13 = mx_dequant(w13q, s13)
    W2 = mx_dequant(w2q, s2)
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
def test_mx_layer_matches_dequantise_first_brute_force(T, H, I, E, k):
    rng = np.random.default_rng(T * 77 + H)
    x, rw, rb = _router_inputs(T, H, E, seed=T + 3 * H)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    b13 = bf16_bits((rng.standard_normal((E, 2 * I)) * 0.1).astype(np.float32))
    b2 = bf16_bits((rng.standard_normal((E, H)) * 0.1).astype(np.float32))
    w13q, s13 = oracle.mx_pack_w13(w13)
    w2q, s2 = oracle.mx_pack_w2(w2)
    out, inter = oracle.mx_forward(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, want_intermediates=True)
    ref, ys = _mx_brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I)
    assert np.allclose(inter["y"].reshape(T, k, H), ys, rtol=1e-10, atol=1e-12)
    assert np.array_equal(out, oracle.bf16_from_f64(ref))
