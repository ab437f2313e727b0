"""Parity of the CUDA path (through the C ABI) with the oracle, on the GPU.

Bit-exact: router indices, the permutation (counts, offsets, rows), the FP8
codes and scales of x, the packed weights and the stand-alone quantiser.
Within tolerance: routing weights (one bf16 step), requantised h (>= 99.9 %
identical codes, the rest neighbours) and the bf16 output
(max|d| <= 2e-2 max|oracle|, mean|d| <= 2e-3 mean|oracle|).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import Layer, bf16_bits, check_codes_close, check_output, sample_tokens, torch_bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def margin_safe_x(cfg, rw, rb, x=None):
    """Draw x for an ad-hoc layer shape, redrawing rows whose top-k margin is below 1e-3."""
    att = np.zeros(cfg.T, np.uint32)
    x = synth.x_rows(cfg, att) if x is None else x
    rows = np.arange(cfg.T)
    while len(rows):
        m = oracle.router(np.ascontiguousarray(x[rows]), rw, rb, cfg.top_k)["margin"]
        rows = rows[m < 1e-3]
        att[rows] += 1
        if len(rows):
            x[rows] = synth.x_rows(cfg, att, rows=rows)
    return x


def full_check(moe, layer: Layer, n_sample: int | None = None, upload: bool = True):
    T, k, E = layer.T, layer.k, layer.E
    if upload:
        layer.to_device()
    out, v, ws = layer.run_gpu()
    assert moe.read_device_status(ws) == 0
    r = layer.oracle_router()
    # routing: bit-exact indices, weights within one bf16 step
    assert np.array_equal(v["topk_idx"].cpu().numpy(), r["idx"])
    # fp32 softmax weights: |dw|/w <= 2*|d logit|; the GPU logits (fp32 FMA or tensor-core
    # accumulation of H bf16 products) are within ~2.5e-5 of the fp64 ones for H <= 4096
    w_gpu = v["topk_w"].cpu().numpy()
    wrel = np.abs(w_gpu - r["w_f32"]) / r["w_f32"]
    print(f"routing weight max rel diff {wrel.max():.3g}")
    assert wrel.max() <= 5e-5
    wb_gpu = v["topk_wb"].cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int32)
    assert np.all(np.abs(wb_gpu - r["w_bf16"].astype(np.int32)) <= 1)
    # grouping by expert: bit-exact
    p = oracle.permute(r["idx"], E)
    for key in ("count", "offset", "perm", "inv"):
        assert np.array_equal(v[key].cpu().numpy(), p[key]), key
    # GEMM tile lists cover every expert's rows
    st = v["status"].cpu().numpy()
    decode = T * k <= 64 * E  # decode-sized batches: 32-row token tiles, 128-feature n-tiles
    bm = 32 if decode else 128
    assert st[3] == bm
    mt = (p["count"] + bm - 1) // bm
    # down GEMM: 256-feature tiles (two w2 row blocks) at prefill; at decode P of the RB n-tiles
    # of an m-tile pair two row blocks and RB - 2P take one (P chosen at launch, 0 <= P <= RB/2)
    RB = layer.Hp // 128
    assert st[1] == mt.sum() * (layer.Ip // 128)
    if decode:
        assert st[2] % mt.sum() == 0 and RB - RB // 2 <= st[2] // mt.sum() <= RB
    else:
        assert st[2] == mt.sum() * ((RB + 1) // 2)
    # x quantisation: bit-exact codes and scales in every permuted row
    xq, sx = oracle.quant_rows_bf16(layer.x)
    tok_of_row = p["perm"] // k
    assert np.array_equal(v["xq"].cpu().numpy(), xq[tok_of_row])
    assert np.array_equal(v["sx"].cpu().numpy(), sx[tok_of_row])
    # layer output (all tokens, or a sample including the most/least loaded experts)
    tokens = (np.arange(T, dtype=np.int32) if n_sample is None else
              sample_tokens(r["idx"], E, n_sample, perm=p["perm"], offset=p["offset"], bm=bm))
    o_out, inter = layer.oracle_forward(tokens, r["idx"])
    rel = check_output(torch_bf16_to_np(out)[tokens], o_out)
    # requantised h of the same (token, slot) rows
    rows = p["inv"][(tokens[:, None] * k + np.arange(k)[None, :]).ravel()]
    frac = check_codes_close(v["hq"].cpu().numpy()[rows], inter["hq"])
    assert np.allclose(v["sh"].cpu().numpy()[rows], inter["sh"], rtol=2e-3, atol=0)
    return out, rel, frac


def test_bounded_wait_returns_instead_of_hanging(moe):
    assert moe.test_bounded_wait(10 ** 9, 1) == 1
    assert moe.test_bounded_wait(2 * 10 ** 6, 0) == 2  # nothing arrives: gives up after 2 ms


def test_quantize_rows_bit_exact(moe):
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((33, 300)) * np.exp(rng.uniform(-8, 8, (33, 1)))).astype(np.float32)
    v[3] = 0.0
    v[5, 128:256] = 0.0
    v[6, :7] = np.float32([448.0, -448.0, 1e-30, -1e-30, 2.0 ** -9, 3.0, -0.0])
    v[7, :5] = np.float32([-0.0, 1e-39, -1e-39, 2.0 ** -100, -(2.0 ** -110)])  # signed zero, subnormals, tiny
    v[8, :128] = np.float32(2.0 ** -120) * np.linspace(-1, 1, 128, dtype=np.float32)  # a whole group of tiny values
    # groups at the edge of the branch-free division's range (amax = 2^-64 and just below), with values
    # under 2^-96 and signed zeros inside them, and a group of negative zeros only
    v[9, :128] = np.float32(2.0 ** -64) * np.linspace(-1, 1, 128, dtype=np.float32)
    v[9, :6] = np.float32([2.0 ** -64, 2.0 ** -97, -(2.0 ** -97), -0.0, 1e-45, -1e-45])
    v[9, 128:256] = np.float32(np.nextafter(np.float32(2.0 ** -64), np.float32(0))) * np.linspace(-1, 1, 128,
                                                                                                 dtype=np.float32)
    v[10, 256:] = -0.0
    v[11, :4] = np.float32([3e38, -3e38, 1e-40, -2.0 ** -96])
    q, s = moe.quantize_rows(torch.from_numpy(v).cuda())
    qo, so = oracle.quant_rows_f32(v)
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != qo)
    assert len(bad) == 0, [(int(r), int(c), float(v[r, c]) if c < v.shape[1] else None, int(qg[r, c]), int(qo[r, c]))
                           for r, c in bad[:8]]
    assert np.array_equal(s.cpu().numpy(), so)


@pytest.mark.parametrize("H,I,E", [(256, 256, 2), (200, 130, 3), (2880, 2880, 1)])
def test_pack_weights_bit_exact(moe, H, I, E):
    rng = np.random.default_rng(H + I)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    w13[0, :128, :128] = 0.0  # an all-zero block
    q13, s13, q2, s2 = moe.pack_weights(torch.from_numpy(w13).cuda(), torch.from_numpy(w2).cuda())
    oq13, os13 = oracle.pack_w13(w13)
    oq2, os2 = oracle.pack_w2(w2)
    # the library stores each 128x128 block contiguously; compare in row-major order
    assert np.array_equal(moe.unblock(q13).cpu().numpy(), oq13) and np.array_equal(s13.cpu().numpy(), os13)
    assert np.array_equal(moe.unblock(q2).cpu().numpy(), oq2) and np.array_equal(s2.cpu().numpy(), os2)


def test_tiny_layer_all_tokens(moe):
    out, rel, frac = full_check(moe, Layer(synth.config("tiny")))
    assert rel[0] < 2e-2


def _adhoc(name, T, H, I, E, k, seed=11, rb=None, rw_zero=False):
    """An ad-hoc layer shape from the generator; rb (float) overrides the router bias."""
    cfg = synth.LayerConfig(name, T, H, I, E, k, seed, "normal", "normal")
    rw, rb_gen = synth.router(cfg)
    if rw_zero:
        rw = np.zeros_like(rw)
    rb = rb_gen if rb is None else bf16_bits(np.asarray(rb, np.float32))
    x = synth.x_rows(cfg) if rw_zero else margin_safe_x(cfg, rw, rb)
    return Layer(cfg, x=x, rw=rw, rb=rb)


def test_single_token(moe):
    full_check(moe, _adhoc("one_token", 1, 256, 256, 8, 2))


def test_ragged_hidden_and_intermediate(moe):
    full_check(moe, _adhoc("ragged", 37, 200, 136, 5, 3))


# Decode-sized batches whose one-block down tiles would outnumber the SMs: the
# down GEMM takes two w2 row blocks (j and j + RB/2) per tile; with an even
# block count every tile is paired, with an odd one each m-tile also has one
# one-block tile, listed after all the paired ones.
PAIRED_DOWN_SHAPES = [("paired_even_blocks", 48, 256, 128), ("paired_odd_blocks", 32, 384, 64)]


@pytest.mark.parametrize("name,T,H,E", PAIRED_DOWN_SHAPES, ids=lambda v: v if isinstance(v, str) else None)
def test_decode_paired_down_tiles(moe, name, T, H, E):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert min(E, T * 4) * ((H + 127) // 128) > sms  # the shape takes the paired tiles
    full_check(moe, _adhoc(name, T, H, 256, E, 4))


def test_all_tokens_to_two_experts_multi_tile(moe):
    # experts 0 and 1 get every token (3 M tiles each: 128 + 128 + 44 rows); experts 2..7 get none
    rb = np.array([8.0, 8.0, 0, 0, 0, 0, 0, 0], np.float32)
    layer = _adhoc("skewed", 300, 256, 256, 8, 2, rb=rb)
    full_check(moe, layer)


def test_top_k_equals_E(moe):
    full_check(moe, _adhoc("k_eq_E", 20, 256, 384, 4, 4))


def test_equal_logits_pick_lowest_experts(moe):
    layer = _adhoc("ties", 16, 256, 256, 8, 3, rb=np.zeros(8, np.float32), rw_zero=True)
    layer.to_device()
    _, v, _ = layer.run_gpu()
    assert np.all(v["topk_idx"].cpu().numpy() == [0, 1, 2])
    w = v["topk_w"].cpu().numpy()
    assert np.allclose(w, 1.0 / 3.0, rtol=1e-6)


def test_many_tokens_router_scan_and_blocked_permute(moe):
    # T >= 512: the router's last CTA scans the histogram; T > 2048: 8 tokens per permutation CTA;
    # T >= 2048: 128-token router tiles, 20 of them (the last holds 68 tokens), clusters of 4 CTAs
    # with one K chunk each
    full_check(moe, _adhoc("many_tokens", 2500, 256, 256, 8, 2), n_sample=48)


def test_router_scan_with_small_token_tiles(moe):
    # 512 <= T < 2048: the router's last CTA scans, 32-token tiles (32 of them, the last holds 8)
    full_check(moe, _adhoc("mid_tokens", 1000, 256, 256, 8, 2), n_sample=32)


def test_large_router_tile_with_unaligned_rows(moe):
    # 128-token router tiles fed by element-wise loads (H not a multiple of 8), a ragged last tile
    full_check(moe, _adhoc("many_odd", 2100, 196, 136, 6, 2), n_sample=32)


@pytest.mark.parametrize("E,k", [(64, 8), (200, 8)])
def test_router_expert_paddings(moe, E, k):
    # the tensor-core router pads the experts to 64 and 256 columns (zero-filled weight rows)
    full_check(moe, _adhoc(f"experts_{E}", 2100, 256, 128, E, k), n_sample=16)


def test_equal_logits_pick_lowest_experts_large_batch(moe):
    layer = _adhoc("ties_large", 2048, 256, 128, 16, 4, rb=np.zeros(16, np.float32), rw_zero=True)
    layer.to_device()
    _, v, _ = layer.run_gpu()
    assert np.all(v["topk_idx"].cpu().numpy() == [0, 1, 2, 3])
    assert np.allclose(v["topk_w"].cpu().numpy(), 0.25, rtol=1e-6)


def test_hidden_size_not_multiple_of_8(moe):
    # rows of x and of the router weights are not 16-byte aligned: element-wise router loads
    full_check(moe, _adhoc("odd_hidden", 19, 196, 136, 6, 2))


def test_graphed_layer_matches_eager(moe):
    layer = Layer(synth.config("tiny")).to_device()
    ml = moe.MoeLayer(layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
                      layer.d_b2, layer.k)
    g = ml.graphed(layer.T)
    for x in (layer.d_x, torch.flip(layer.d_x, dims=[0]).contiguous()):  # two batches through one graph
        ref = ml(x)
        g.x.copy_(x)
        got = g()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name,T,H,E,k", [("graph_decode", 48, 256, 128, 4), ("graph_prefill", 600, 384, 4, 2)],
                         ids=lambda v: v if isinstance(v, str) else None)
def test_graphed_layer_matches_eager_both_regimes(moe, name, T, H, E, k):
    # decode-sized (paired down tiles) and prefill-sized (two MMA issuers) batches through one graph
    cfg = synth.LayerConfig(name, T, H, 256, E, k, 11, "normal", "normal")
    layer = Layer(cfg, x=synth.x_rows(cfg)).to_device()  # no oracle here: any ties resolve alike
    ml = moe.MoeLayer(layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
                      layer.d_b2, layer.k)
    g = ml.graphed(layer.T)
    for x in (layer.d_x, torch.flip(layer.d_x, dims=[0]).contiguous()):
        ref = ml(x)
        g.x.copy_(x)
        got = g()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_repeated_calls_are_bit_identical(moe):
    layer = Layer(synth.config("tiny")).to_device()
    a, _, ws = layer.run_gpu()
    b, _, _ = layer.run_gpu(workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name,n_sample", [("oss20b_decode", None), ("oss120b_decode", 64),
                                           ("oss120b_prefill", 128), ("qwen235b_prefill", 128)])
def test_layer_shapes_full_size(moe, name, n_sample):
    full_check(moe, Layer(synth.config(name)), n_sample=n_sample)
    torch.cuda.empty_cache()


def _tiny_token_layer(name, T, E, k, tiny_t):
    """A layer whose token tiny_t has x scaled by 2^-40 and zero gate/up biases, so
    that its h = silu(g) * u has a group amax far below 2^-64 (the quantiser's IEEE
    division range); the router bias alone routes it (distinct biases, margin 0.1)."""
    cfg = synth.LayerConfig(name, T, 256, 256, E, k, 13, "normal", "zero")
    rw, _ = synth.router(cfg)
    rb = bf16_bits(np.float32(0.1) * np.arange(E, 0, -1, dtype=np.float32))
    x = synth.x_rows(cfg)
    xt = synth.bf16_to_f32(x[tiny_t]) * np.float32(2.0 ** -40)  # exact: a power of two
    x[tiny_t] = bf16_bits(xt)
    x = margin_safe_x(cfg, rw, rb, x)
    b13, b2 = synth.expert_biases(cfg)
    layer = Layer(cfg, x=x, rw=rw, rb=rb, b13=np.zeros_like(b13), b2=b2)
    assert np.array_equal(layer.x[tiny_t], x[tiny_t])  # the tiny row kept its draw
    return layer


@pytest.mark.parametrize("T,E,k", [(16, 4, 2), (600, 4, 2)], ids=["decode_tile", "prefill_tile"])
def test_requant_of_a_token_with_tiny_h(moe, T, E, k):
    # decode tiles: the token's lane makes its whole warp take IEEE division;
    # prefill tiles: the token's row thread takes it alone
    tiny_t = 5
    layer = _tiny_token_layer(f"tiny_h_{T}", T, E, k, tiny_t)
    out, _, _ = full_check(moe, layer)
    _, v, _ = layer.run_gpu()
    rows = v["inv"].cpu().numpy()[tiny_t * k:(tiny_t + 1) * k]
    sh = v["sh"].cpu().numpy()[rows]
    assert np.all(sh < np.float32(2.0 ** -64 / 448)) and np.all(sh > 0), sh  # amax < 2^-64: the slow path ran


@pytest.mark.parametrize("name,T,H,I,E,k", [
    ("max_experts_topk", 48, 256, 256, 256, 8),       # E and top_k at their limits (router pads 256 experts)
    ("max_hidden_decode", 8, 16384, 128, 4, 2),        # H at its limit: 128 K blocks in the gate/up GEMM
    ("max_hidden_prefill", 600, 16384, 128, 4, 2),     # the same through the 128-row tile GEMMs
    ("max_inter_prefill", 600, 128, 16384, 4, 2),      # I at its limit: 128 h blocks, 128 K blocks in the down GEMM
], ids=lambda v: v if isinstance(v, str) else None)
def test_size_limits(moe, name, T, H, I, E, k):
    full_check(moe, _adhoc(name, T, H, I, E, k), n_sample=None if T <= 64 else 48)
    torch.cuda.empty_cache()
