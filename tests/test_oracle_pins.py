"""Pins for the oracle: each check ties it to something other than itself.

- e4m3 table / encoder: the format definition's special values, PyTorch's own
  float8_e4m3fn conversion (a library routine), and an exhaustive comparison of
  the bisection encoder with the scanning encoder.
- quantisers: the half-ulp round-trip bound and closed forms for constant blocks.
- router: brute force with numpy (full sort, textbook softmax).
- permutation: invariants and a numpy stable sort.
- expert GEMMs and the whole layer: a dequantise-first numpy path (fp64 matmul
  of decoded weights) on tiny shapes, and the hand-worked 1-token / 2-expert
  example under tests/golden/.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (numpy, independent of the oracle)."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def f32(b: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f32(np.asarray(b, np.uint16))


# ---------------------------------------------------------------- e4m3 ----
def test_e4m3_table_matches_format_definition_special_values():
    t = oracle.e4m3_decode_table()
    assert t[0x7E] == 448.0  # largest finite
    assert t[0x01] == 2.0 ** -9  # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9  # largest subnormal
    assert t[0x08] == 2.0 ** -6  # smallest normal
    assert t[0x38] == 1.0
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.sum(np.isnan(t)) == 2
    assert np.all(t[0x80:0xFF] == -t[0x00:0x7F])
    assert np.all(np.diff(t[0x00:0x7F]) > 0)  # monotone: bisection is valid


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = oracle.e4m3_decode_table()
    both_nan = np.isnan(ref) & np.isnan(t)
    assert np.all(both_nan | (ref == t))


def _tie_points():
    t = oracle.e4m3_decode_table()[:0x7F]
    mids = (t[:-1] + t[1:]) / 2  # exact in fp64 and in fp32
    m32 = mids.astype(np.float32)
    assert np.all(m32.astype(np.float64) == mids)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    pts = np.concatenate([m32, up, dn, t.astype(np.float32)])
    return np.concatenate([pts, -pts]).astype(np.float32)


def test_e4m3_bisection_equals_scan_exhaustive_bf16_and_ties():
    allbf = synth.bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    allbf = allbf[~np.isnan(allbf)]
    v = np.concatenate([allbf, _tie_points(), np.float32([1e30, -1e30, 448.0, 449.0, 463.99, 464.0, 470.0])])
    a = oracle.e4m3_encode(v)
    b = oracle.e4m3_encode(v, scan=True)
    assert np.array_equal(a, b)


def test_e4m3_encoder_matches_torch_in_range():
    allbf = synth.bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    v = np.concatenate([allbf, _tie_points()]).astype(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 464.0)]  # torch does not saturate above the 448/480 midpoint
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_and_keeps_sign():
    got = oracle.e4m3_encode(np.float32([465.0, 1e6, 3e38, -1e6, -465.0, -1e-9, 1e-9, 0.0]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x00, 0x00]
    # ties to even: 2^-10 lies halfway between 0 and 2^-9 -> 0; 1.5*2^-9 -> 2*2^-9 (code 2)
    got = oracle.e4m3_encode(np.float32([2.0 ** -10, 1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9, 1.0625, 1.1875]))
    assert list(got) == [0x00, 0x02, 0x02, 0x38, 0x3A]


def test_bf16_from_f64_single_rounding():
    ulp = 2.0 ** -7  # spacing in [1, 2)
    vals = np.array([1.0 + ulp / 2, 1.0 + 1.5 * ulp, 1.0 + ulp / 2 + 1e-12, -(1.0 + ulp / 2), 0.0, 1.2882890])
    got = oracle.bf16_from_f64(vals)
    want = np.array([0x3F80, 0x3F82, 0x3F81, 0xBF80, 0x0000, 0x3FA5], np.uint16)  # 1.2890625 = 0x3FA5
    assert np.array_equal(got, want)
    # double rounding through fp32 would round 1 + ulp/2 + 2^-30 down; one step rounds it up
    assert oracle.bf16_from_f64(np.array([1.0 + ulp / 2 + 2.0 ** -30]))[0] == 0x3F81


# ---------------------------------------------------------- quantisers ----
def _e4m3_half_ulp(a: np.ndarray) -> np.ndarray:
    """Half the e4m3 spacing at magnitude a (format definition: 3 mantissa bits, min exponent -6)."""
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * 2.0 ** (e - 3)


def test_activation_quant_roundtrip_half_ulp():
    rng = np.random.default_rng(0)
    x = bf16_bits(rng.standard_normal((16, 300)).astype(np.float32) * np.float32(3.0))
    q, s = oracle.quant_rows_bf16(x)
    assert q.shape == (16, 384) and s.shape == (16, 3)
    tab = oracle.e4m3_decode_table()
    xv = f32(x).astype(np.float64)
    deq = tab[q[:, :300]] * np.repeat(s.astype(np.float64), 128, axis=1)[:, :300]
    scaled = np.abs(xv) / np.repeat(s.astype(np.float64), 128, axis=1)[:, :300]
    bound = (_e4m3_half_ulp(scaled) * (1 + 1e-6) + 1e-6) * np.repeat(s, 128, axis=1)[:, :300]
    assert np.all(np.abs(deq - xv) <= bound)
    assert np.all(q[:, 300:] == 0)  # pad columns
    # each group's largest element encodes to +-448 (s = amax/448)
    for g in range(3):
        blk = np.abs(xv[:, g * 128:min(300, g * 128 + 128)])
        arg = np.argmax(blk, axis=1)
        codes = q[np.arange(16), g * 128 + arg] & 0x7F
        assert np.all(codes == 0x7E)
        assert np.array_equal(s[:, g], (blk.max(axis=1).astype(np.float32) / np.float32(448.0)))


def test_zero_group_gives_unit_scale_and_zero_codes():
    x = np.zeros((2, 256), np.float32)
    x[1, 128:] = 1.0
    q, s = oracle.quant_rows_f32(x)
    assert np.all(q[0] == 0) and np.all(s[0] == 1.0) and s[1, 0] == 1.0 and np.all(q[1, :128] == 0)
    assert np.all(q[1, 128:] == 0x7E) and s[1, 1] == np.float32(1.0) / np.float32(448.0)


def test_weight_blocks_closed_form_and_layout():
    H, I = 200, 130  # padded to 256 / 256: ragged in both
    w13 = np.zeros((1, 2 * I, H), np.float32)
    w13[0, :I, :] = 2.0 ** -7  # gate: one constant
    w13[0, I:, :] = -3.0  # up
    w13[0, 5, 7] = 2.0 ** -5  # raises amax of gate block (0,0)
    q, s = oracle.pack_w13(w13)
    assert q.shape == (1, 512, 256) and s.shape == (1, 4, 2)
    Ip = 256
    # gate block (0,0): amax = 2^-5, the constant 2^-7 encodes to 448/4 = 112 = 1.75 * 2^6 (0x6E)
    assert s[0, 0, 0] == np.float32(2.0 ** -5) / np.float32(448.0)
    assert q[0, 5, 7] == 0x7E and q[0, 0, 0] == 0x6E
    # up rows live at [Ip, Ip+I), negative codes, 448 at full scale
    assert np.all(q[0, Ip:Ip + I, :H] == 0xFE) and s[0, 2, 0] == np.float32(3.0) / np.float32(448.0)
    # padding: rows [I, Ip) and [Ip+I, 2Ip), columns [H, Hp) are zero codes; empty blocks have scale 1
    assert np.all(q[0, I:Ip] == 0) and np.all(q[0, Ip + I:] == 0) and np.all(q[0, :, H:] == 0)
    assert s[0, 3, 1] == np.float32(3.0) / np.float32(448.0)  # up rows 128..129 of the second block
    w2 = np.full((1, H, I), 0.5, np.float32)
    q2, s2 = oracle.pack_w2(w2)
    assert q2.shape == (1, 256, 256) and np.all(q2[0, :H, :I] == 0x7E) and np.all(q2[0, H:] == 0)
    assert s2[0, 1, 1] == np.float32(0.5) / np.float32(448.0)


def test_weight_blocks_roundtrip_half_ulp_random():
    rng = np.random.default_rng(1)
    w2 = (rng.standard_normal((2, 300, 260)) * 0.02).astype(np.float32)
    q, s = oracle.pack_w2(w2)
    tab = oracle.e4m3_decode_table()
    S = np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)[:, :300, :260].astype(np.float64)
    deq = tab[q[:, :300, :260]] * S
    bound = (_e4m3_half_ulp(np.abs(w2) / S) * (1 + 1e-6) + 1e-6) * S
    assert np.all(np.abs(deq - w2) <= bound)


# -------------------------------------------------------------- router ----
def _router_inputs(T, H, E, seed=3, rb_scale=0.1):
    rng = np.random.default_rng(seed)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    rw = bf16_bits((rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32))
    rb = bf16_bits((rng.standard_normal(E) * rb_scale).astype(np.float32))
    return x, rw, rb


def test_router_matches_brute_force_sort_and_textbook_softmax():
    T, H, E, k = 40, 96, 12, 3
    x, rw, rb = _router_inputs(T, H, E)
    r = oracle.router(x, rw, rb, k, want_logits=True)
    logits = f32(x).astype(np.float64) @ f32(rw).astype(np.float64).T + f32(rb).astype(np.float64)
    assert np.allclose(r["logits"], logits, rtol=0, atol=1e-12)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))  # descending logit, then ascending index
        sel = np.sort(order[:k])
        assert np.array_equal(r["idx"][t], sel)
        z = np.exp(logits[t, sel] - logits[t, sel].max())
        w = z / z.sum()
        assert np.allclose(r["w_f32"][t], w, rtol=1e-6, atol=0)
        assert abs(r["w_f32"][t].astype(np.float64).sum() - 1.0) < 1e-6
        assert abs(f32(r["w_bf16"][t]).astype(np.float64).sum() - 1.0) <= k * 2.0 ** -9
        assert np.isclose(r["margin"][t], logits[t, order[k - 1]] - logits[t, order[k]], rtol=0, atol=1e-12)
    assert np.array_equal(r["w_bf16"], bf16_bits(r["w_f32"]))


def test_router_softmax_is_over_selected_experts_only():
    # two experts selected out of four: weights must not see the unselected logits
    x = bf16_bits(np.ones((1, 8), np.float32))
    rw = np.zeros((4, 8), np.uint16)
    rb = bf16_bits(np.float32([2.0, -1.0, 1.0, -3.0]))
    r = oracle.router(x, rw, rb, 2)
    assert list(r["idx"][0]) == [0, 2]
    e = np.exp(1.0)
    assert np.allclose(r["w_f32"][0], [e / (e + 1), 1 / (e + 1)], rtol=1e-7)


def test_router_ties_go_to_lower_expert():
    x = bf16_bits(np.ones((3, 16), np.float32))
    rw = np.zeros((6, 16), np.uint16)
    rb = np.zeros(6, np.uint16)
    r = oracle.router(x, rw, rb, 3)
    assert np.all(r["idx"] == [0, 1, 2])
    assert np.all(r["margin"] == 0.0)
    rb = bf16_bits(np.float32([0, 1, 1, 0, 1, 1]))
    r = oracle.router(x, rw, rb, 3)
    assert np.all(r["idx"] == [1, 2, 4])


# --------------------------------------------------------- permutation ----
def test_permutation_invariants_and_stable_sort():
    rng = np.random.default_rng(4)
    T, E, k = 50, 7, 3
    idx = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(T)]).astype(np.int32)
    p = oracle.permute(idx, E)
    assert np.array_equal(p["count"], np.bincount(idx.ravel(), minlength=E))
    assert p["offset"][0] == 0 and np.array_equal(np.diff(p["offset"]), p["count"])
    flat_e = idx.ravel()
    order = np.lexsort((np.arange(T * k) // k, flat_e))  # by expert, then token
    assert np.array_equal(p["perm"], order)
    assert np.array_equal(np.sort(p["perm"]), np.arange(T * k))  # each (t, j) exactly once
    assert np.all(np.bincount(p["perm"] // k, minlength=T) == k)  # each token k times
    assert np.array_equal(p["inv"][p["perm"]], np.arange(T * k))


# ------------------------------------------------ layer vs brute force ----
def _decode_blocks(q, s):
    tab = oracle.e4m3_decode_table()
    S = np.repeat(np.repeat(s.astype(np.float64), 128, axis=-2), 128, axis=-1)
    return tab[q] * S


def _brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I):
    """Dequantise everything first, then plain fp64 matmuls (numpy)."""
    T, H = x.shape
    Hp = w13q.shape[2]
    Ip = w2q.shape[2]
    tab = oracle.e4m3_decode_table()
    r = oracle.router(x, rw, rb, k)
    xq, sx = oracle.quant_rows_bf16(x)
    xd = tab[xq] * np.repeat(sx.astype(np.float64), 128, axis=1)  # [T, Hp]
    W13 = _decode_blocks(w13q, s13)  # [E, 2Ip, Hp]
    W2 = _decode_blocks(w2q, s2)  # [E, Hp, Ip]
    out = np.zeros((T, H))
    ys = np.zeros((T, k, H))
    for t in range(T):
        for j in range(k):
            e = r["idx"][t, j]
            gu = W13[e] @ xd[t]
            g = gu[:I] + f32(b13[e, :I])
            u = gu[Ip:Ip + I] + f32(b13[e, I:])
            h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
            hq, sh = oracle.quant_rows_f32(h[None, :])
            hd = tab[hq[0]] * np.repeat(sh[0].astype(np.float64), 128)
            y = W2[e, :H] @ hd + f32(b2[e])
            ys[t, j] = y
            out[t] += f32(r["w_bf16"][t, j]).astype(np.float64) * y
    return out, ys


@pytest.mark.parametrize("T,H,I,E,k", [(5, 128, 128, 4, 2), (6, 200, 136, 5, 3), (3, 256, 384, 3, 3)])
def test_layer_matches_dequantise_first_brute_force(T, H, I, E, k):
    rng = np.random.default_rng(T * 1000 + H)
    x, rw, rb = _router_inputs(T, H, E, seed=T + H)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    b13 = bf16_bits((rng.standard_normal((E, 2 * I)) * 0.1).astype(np.float32))
    b2 = bf16_bits((rng.standard_normal((E, H)) * 0.1).astype(np.float32))
    w13q, s13 = oracle.pack_w13(w13)
    w2q, s2 = oracle.pack_w2(w2)
    out, inter = oracle.forward(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, want_intermediates=True)
    ref, ys = _brute_force_layer(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, I)
    assert np.allclose(inter["y"].reshape(T, k, H), ys, rtol=1e-10, atol=1e-12)
    assert np.array_equal(out, oracle.bf16_from_f64(ref))
    # a token subset gives the same rows
    sub = np.array([T - 1, 0], np.int32)
    out_sub = oracle.forward(x, rw, rb, w13q, s13, b13, w2q, s2, b2, k, tokens=sub)
    assert np.array_equal(out_sub, out[sub])


# ------------------------------------------------- hand-worked example ----
def _hand_example(b2_0: float):
    H = I = 128
    x = bf16_bits(np.ones((1, H), np.float32))
    rw = np.zeros((2, H), np.uint16)
    rb = bf16_bits(np.float32([1.0, 0.0]))
    w13 = np.zeros((2, 2 * I, H), np.float32)
    w13[0, :I] = 2.0 ** -7
    w13[0, I:] = 2.0 ** -6
    w13[1, :I] = -2.0 ** -7
    w13[1, I:] = 2.0 ** -6
    w2 = np.full((2, H, I), 2.0 ** -7, np.float32)
    b13 = np.zeros((2, 2 * I), np.uint16)
    b2 = np.zeros((2, H), np.uint16)
    b2[0, :] = bf16_bits(np.float32([b2_0]))[0]
    w13q, s13 = oracle.pack_w13(w13)
    w2q, s2 = oracle.pack_w2(w2)
    return oracle.forward(x, rw, rb, w13q, s13, b13, w2q, s2, b2, 2, want_intermediates=True)


def test_hand_worked_one_token_two_experts():
    with open(os.path.join(GOLDEN, "hand_example_1tok_2exp.json")) as f:
        g = json.load(f)
    out, inter = _hand_example(g["b2_expert0"])
    assert np.all(out == bf16_bits(np.float32([g["out_bf16"]]))[0])
    assert np.allclose(inter["y"][0], g["y_expert0"], rtol=1e-6)
    assert np.allclose(inter["y"][1], g["y_expert1"], rtol=1e-6)
    out0, _ = _hand_example(0.0)
    assert np.all(out0 == bf16_bits(np.float32([g["out_bf16_b2_zero"]]))[0])
    # the routing-weight reading: fp32 weights would have given a different output
    assert g["out_bf16_b2_zero_if_fp32_weights"] != g["out_bf16_b2_zero"]
    r = oracle.router(bf16_bits(np.ones((1, 128), np.float32)), np.zeros((2, 128), np.uint16),
                      bf16_bits(np.float32([1.0, 0.0])), 2)
    assert np.allclose(f32(r["w_bf16"][0]), g["weights_bf16"], rtol=0, atol=0)
