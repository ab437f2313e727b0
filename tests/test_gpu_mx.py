"""Parity of the MXFP8 variant (through the C ABI) with the oracle, on the GPU.

Bit-exact: router indices, the permutation, the MX codes and scale bytes of x
(every permuted row), the packed weights and scale atoms, and the stand-alone
1x32 quantiser.  Within tolerance: the bf16 output (same bounds as the 128x128
variant) and the requantised h: the scale byte of a group may differ by one
where fp32 and fp64 SwiGLU values fall on either side of a power of two
(<= 1 % of groups), and in groups with equal bytes >= 99.9 % of the codes are
identical, the rest neighbours.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import Layer, bf16_bits, check_codes_close, check_output, mx_row_scales, sample_tokens, torch_bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def margin_safe_x(cfg, rw, rb):
    att = np.zeros(cfg.T, np.uint32)
    x = synth.x_rows(cfg, att)
    rows = np.arange(cfg.T)
    while len(rows):
        m = oracle.router(np.ascontiguousarray(x[rows]), rw, rb, cfg.top_k)["margin"]
        rows = rows[m < 1e-3]
        att[rows] += 1
        if len(rows):
            x[rows] = synth.x_rows(cfg, att, rows=rows)
    return x


def adhoc(name, T, H, I, E, k, seed=11, rb=None):
    cfg = synth.LayerConfig(name, T, H, I, E, k, seed, "normal", "normal")
    rw, rb_gen = synth.router(cfg)
    rb = rb_gen if rb is None else bf16_bits(np.asarray(rb, np.float32))
    return Layer(cfg, x=margin_safe_x(cfg, rw, rb), rw=rw, rb=rb, mx=True)


def full_check_mx(moe, layer: Layer, n_sample: int | None = None, upload: bool = True):
    T, k, E, Hp, Ip = layer.T, layer.k, layer.E, layer.Hp, layer.Ip
    if upload:
        layer.to_device()
    out, v, ws = layer.run_gpu()
    assert moe.read_device_status(ws) == 0
    r = layer.oracle_router()
    assert np.array_equal(v["topk_idx"].cpu().numpy(), r["idx"])
    wb_gpu = v["topk_wb"].cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int32)
    assert np.all(np.abs(wb_gpu - r["w_bf16"].astype(np.int32)) <= 1)
    p = oracle.permute(r["idx"], E)
    for key in ("count", "offset", "perm", "inv"):
        assert np.array_equal(v[key].cpu().numpy(), p[key]), key
    bm = moe.m_tile_rows(T, E, k)
    assert int(v["status"].cpu().numpy()[3]) == bm
    tiles1 = v["tiles1"].cpu().numpy()
    # x: MX codes and scale bytes of every permuted row, bit-exact
    xq, sx = oracle.mx_quant_rows_bf16(layer.x)
    tok_of_row = p["perm"] // k
    assert np.array_equal(v["xq"].cpu().numpy(), xq[tok_of_row])
    sx_gpu = mx_row_scales(v["sx"].cpu().numpy(), p["count"], p["offset"], tiles1, Ip // 128, bm)
    assert np.array_equal(sx_gpu, sx[tok_of_row])
    # output rows (all tokens or a sample with the most/least loaded experts)
    tokens = np.arange(T, dtype=np.int32) if n_sample is None else sample_tokens(r["idx"], E, n_sample)
    o_out, inter = layer.oracle_forward(tokens, r["idx"])
    rel = check_output(torch_bf16_to_np(out)[tokens], o_out)
    # requantised h of the same (token, slot) rows
    rows = p["inv"][(tokens[:, None] * k + np.arange(k)[None, :]).ravel()]
    sh_gpu = mx_row_scales(v["sh"].cpu().numpy(), p["count"], p["offset"], tiles1, Ip // 128, bm)[rows]
    sh_ref = inter["sh"]
    dbyte = sh_gpu.astype(np.int32) - sh_ref.astype(np.int32)
    assert np.abs(dbyte).max() <= 1, "an h scale byte differs by more than one binade"
    same = dbyte == 0
    assert same.mean() >= 0.99, f"only {same.mean():.4f} of h scale bytes identical"
    hq_gpu = v["hq"].cpu().numpy()[rows].reshape(len(rows), Ip // 32, 32)
    hq_ref = inter["hq"].reshape(len(rows), Ip // 32, 32)
    frac = check_codes_close(hq_gpu[same], hq_ref[same])
    return out, rel, frac


def test_mx_quantize_rows_bit_exact(moe):
    rng = np.random.default_rng(17)
    v = (rng.standard_normal((40, 300)) * np.exp(rng.uniform(-8, 8, (40, 1)))).astype(np.float32)
    v[3] = 0.0                                            # all-zero row: byte 0, +0 codes
    v[5, 32:64] = -0.0                                    # a group of negative zeros only
    v[6, :8] = np.float32([448.0, -448.0, 1e-30, -1e-30, 2.0 ** -9, 3.0, -0.0, 1.0])
    v[7, :5] = np.float32([-0.0, 1e-39, -1e-39, 2.0 ** -100, -(2.0 ** -110)])  # subnormals, tiny values
    v[8, :32] = np.float32(2.0 ** -125) * np.linspace(-1, 1, 32, dtype=np.float32)  # amax below the clamp
    v[9, :32] = np.float32(2.0 ** -119)                   # amax exactly at the clamp edge
    v[9, 32:64] = np.float32(np.nextafter(np.float32(2.0 ** -119), np.float32(0)))
    v[10, :32] = np.linspace(-1, 1, 32, dtype=np.float32) * np.float32(np.nextafter(np.float32(2.0), np.float32(0)))
    v[10, 32:64] = np.linspace(-2, 2, 32, dtype=np.float32)  # amax exactly a power of two
    v[11, :4] = np.float32([3e38, -3e38, 1e-40, -2.0 ** -96])  # near fp32 max
    v[12, :32] = np.float32(500.0) * np.linspace(-1, 1, 32, dtype=np.float32)  # top binade saturates to 448
    v[13, :32] = np.float32(1e-45)                        # subnormal amax
    v[14, :3] = np.float32([464.0, 479.0, 481.0])         # ties and saturation around e4m3's largest normal
    q, s = moe.quantize_rows_mx(torch.from_numpy(v).cuda())
    qo, so = oracle.mx_quant_rows_f32(v)
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != qo)
    assert len(bad) == 0, [(int(r), int(c), float(v[r, c]) if c < v.shape[1] else None, int(qg[r, c]), int(qo[r, c]))
                           for r, c in bad[:8]]
    assert np.array_equal(s.cpu().numpy(), so)


@pytest.mark.parametrize("H,I,E", [(256, 256, 2), (200, 130, 3), (2880, 2880, 1)])
def test_mx_pack_weights_bit_exact(moe, H, I, E):
    rng = np.random.default_rng(H + I + 1)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.02 * np.exp(rng.uniform(-4, 4, (E, H, 1)))).astype(np.float32)
    w13[0, :3, :32] = 0.0   # all-zero groups
    w13[0, 5, 64:96] = -0.0
    q13, s13, q2, s2 = moe.pack_weights_mx(torch.from_numpy(w13).cuda(), torch.from_numpy(w2).cuda())
    oq13, os13 = oracle.mx_pack_w13(w13)
    oq2, os2 = oracle.mx_pack_w2(w2)
    assert np.array_equal(moe.unblock(q13).cpu().numpy(), oq13)
    assert np.array_equal(moe.unblock_scales_mx(s13).cpu().numpy(), os13)
    assert np.array_equal(moe.unblock(q2).cpu().numpy(), oq2)
    assert np.array_equal(moe.unblock_scales_mx(s2).cpu().numpy(), os2)


def test_mx_tiny_layer_all_tokens(moe):
    full_check_mx(moe, Layer(synth.config("tiny"), mx=True))


def test_mx_single_token(moe):
    full_check_mx(moe, adhoc("one_token", 1, 256, 256, 8, 2))


def test_mx_ragged_hidden_and_intermediate(moe):
    full_check_mx(moe, adhoc("ragged", 37, 200, 136, 5, 3))


def test_mx_hidden_size_not_multiple_of_8(moe):
    full_check_mx(moe, adhoc("odd_hidden", 19, 196, 136, 6, 2))


def test_mx_top_k_equals_E(moe):
    full_check_mx(moe, adhoc("k_eq_E", 20, 256, 384, 4, 4))


def test_mx_prefill_tiles_skewed(moe):
    # 128-row tile kernels (R = 600 > 64 E): experts 0 and 1 get every token (3 m-tiles: 128 + 128 + 44)
    rb = np.array([8.0, 8.0, 0, 0, 0, 0, 0, 0], np.float32)
    full_check_mx(moe, adhoc("skewed", 300, 256, 256, 8, 2, rb=rb))


def test_mx_prefill_odd_block_count(moe):
    # Hp / 128 = 3: the down GEMM's last 256-wide tile has one w2 block; ragged I
    full_check_mx(moe, adhoc("odd_blocks", 600, 384, 200, 4, 2), n_sample=64)


@pytest.mark.parametrize("name,T,H,E", [("paired_even_blocks", 48, 256, 128), ("paired_odd_blocks", 32, 384, 64)],
                         ids=lambda v: v if isinstance(v, str) else None)
def test_mx_decode_paired_down_tiles(moe, name, T, H, E):
    # the decode down GEMM's paired w2 row blocks (RB even: every tile; RB odd: plus one one-block tile)
    full_check_mx(moe, adhoc(name, T, H, 256, E, 4))


def test_mx_many_tokens_router_scan(moe):
    full_check_mx(moe, adhoc("many_tokens", 2500, 256, 256, 8, 2), n_sample=48)


@pytest.mark.parametrize("fp4", [False, True], ids=["mxfp8", "mxfp4"])
@pytest.mark.parametrize("name,T,H,E", [("graph_decode", 48, 256, 128), ("graph_prefill", 600, 384, 4)],
                         ids=lambda v: v if isinstance(v, str) else None)
def test_mx_graphed_layer_matches_eager(moe, name, T, H, E, fp4):
    # one CUDA-graph replay (the five kernels with their programmatic dependencies) gives the
    # eager call's bits, for decode-sized (paired down tiles) and prefill-sized batches
    cfg = synth.LayerConfig(name, T, H, 256, E, 4 if E > 4 else 2, 11, "normal", "normal")
    layer = Layer(cfg, x=synth.x_rows(cfg), mx=True, fp4=fp4).to_device()  # no oracle here
    ml = moe.MoeLayer(layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
                      layer.d_b2, layer.k)
    g = ml.graphed(layer.T)
    for x in (layer.d_x, torch.flip(layer.d_x, dims=[0]).contiguous()):
        ref = ml(x)
        g.x.copy_(x)
        got = g()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_mx_repeated_calls_are_bit_identical(moe):
    layer = Layer(synth.config("tiny"), mx=True).to_device()
    a, _, ws = layer.run_gpu()
    b, _, _ = layer.run_gpu(workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name,n_sample", [("oss20b_decode", None), ("oss120b_decode", 32),
                                           ("oss120b_prefill", 24), ("qwen235b_prefill", 24)])
def test_mx_layer_shapes_full_size(moe, name, n_sample):
    full_check_mx(moe, Layer(synth.config(name), mx=True), n_sample=n_sample)
    torch.cuda.empty_cache()
