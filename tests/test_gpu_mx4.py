"""Parity of the MXFP4-weight variant (through the C ABI) with the oracle, on the GPU.

Weights are E2M1 codes with 1x32 UE8M0 scales (OCP MX v1.0), two codes per
byte; x and h are MXFP8 as in the MXFP8 variant.  Bit-exact: routing, the
permutation, the x codes and scale bytes, and the packed weight codes and
scale atoms.  Within the layer tolerance: the bf16 output; the requantised h
as in the MXFP8 tests (scale bytes within one binade, >= 99 % identical;
codes >= 99.9 % identical, the rest neighbours).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import Layer, bf16_bits
from test_gpu_mx import full_check_mx, margin_safe_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def adhoc4(name, T, H, I, E, k, seed=11, rb=None):
    cfg = synth.LayerConfig(name, T, H, I, E, k, seed, "normal", "normal")
    rw, rb_gen = synth.router(cfg)
    rb = rb_gen if rb is None else bf16_bits(np.asarray(rb, np.float32))
    return Layer(cfg, x=margin_safe_x(cfg, rw, rb), rw=rw, rb=rb, fp4=True)


@pytest.mark.parametrize("H,I,E", [(256, 256, 2), (200, 130, 3), (2880, 2880, 1)])
def test_mx4_pack_weights_bit_exact(moe, H, I, E):
    rng = np.random.default_rng(H + I + 7)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.02 * np.exp(rng.uniform(-4, 4, (E, H, 1)))).astype(np.float32)
    w13[0, :3, :32] = 0.0                      # all-zero groups: byte 0, +0 codes
    w13[0, 5, 64:96] = -0.0
    # exact midpoints of the scaled grid (amax 6 * 2^-3 -> X = -3): ties go to the even code
    w13[0, 6, :8] = np.float32([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]) * np.float32(2.0 ** -3)
    w13[0, 6, 8:16] = -w13[0, 6, :8]
    w13[0, 7, :32] = np.float32(7.9 * 2.0 ** -5)  # top binade above 6: saturates to code 7
    w13[0, 7, 1] = np.float32(-1e-12)         # rounds to -0 (code 8)
    q13, s13, q2, s2 = moe.pack_weights_mxfp4(torch.from_numpy(w13).cuda(), torch.from_numpy(w2).cuda())
    oq13, os13 = oracle.mx4_pack_w13(w13)
    oq2, os2 = oracle.mx4_pack_w2(w2)
    assert np.array_equal(moe.unblock_fp4(q13).cpu().numpy(), oq13)
    assert np.array_equal(moe.unblock_scales_mx(s13).cpu().numpy(), os13)
    assert np.array_equal(moe.unblock_fp4(q2).cpu().numpy(), oq2)
    assert np.array_equal(moe.unblock_scales_mx(s2).cpu().numpy(), os2)
    assert oq13[0, 6, :16].tolist() == [7, 0, 2, 2, 4, 4, 6, 6, 15, 8, 10, 10, 12, 12, 14, 14]
    assert oq13[0, 7, 1] == 8


def test_mx4_tiny_layer_all_tokens(moe):
    full_check_mx(moe, Layer(synth.config("tiny"), fp4=True))


@pytest.mark.parametrize("name,T,H,E", [("paired_even_blocks", 48, 256, 128), ("paired_odd_blocks", 32, 384, 64)],
                         ids=lambda v: v if isinstance(v, str) else None)
def test_mx4_decode_paired_down_tiles(moe, name, T, H, E):
    # the decode down GEMM's paired w2 row blocks with E2M1 weight boxes
    full_check_mx(moe, adhoc4(name, T, H, 256, E, 4))


def test_mx4_single_token(moe):
    full_check_mx(moe, adhoc4("one_token", 1, 256, 256, 8, 2))


def test_mx4_ragged_hidden_and_intermediate(moe):
    full_check_mx(moe, adhoc4("ragged", 37, 200, 136, 5, 3))


def test_mx4_top_k_equals_E(moe):
    full_check_mx(moe, adhoc4("k_eq_E", 20, 256, 384, 4, 4))


def test_mx4_prefill_tiles_skewed(moe):
    # 128-row tile kernels (R = 600 > 64 E): experts 0 and 1 get every token (3 m-tiles: 128 + 128 + 44)
    rb = np.array([8.0, 8.0, 0, 0, 0, 0, 0, 0], np.float32)
    full_check_mx(moe, adhoc4("skewed", 300, 256, 256, 8, 2, rb=rb))


def test_mx4_prefill_odd_block_count(moe):
    # Hp / 128 = 3: the down GEMM's last 256-wide tile has one w2 block; ragged I
    full_check_mx(moe, adhoc4("odd_blocks", 600, 384, 200, 4, 2), n_sample=64)


def test_mx4_repeated_calls_are_bit_identical(moe):
    layer = Layer(synth.config("tiny"), fp4=True).to_device()
    a, _, ws = layer.run_gpu()
    b, _, _ = layer.run_gpu(workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mx4_rejects_weights_not_32_byte_aligned(moe):
    layer = Layer(synth.config("tiny"), fp4=True).to_device()
    E, H, I, T, k = layer.E, layer.H, layer.I, layer.T, layer.k
    buf = torch.empty(layer.d_w13.numel() + 16, dtype=torch.uint8, device="cuda")
    w13 = buf[16:16 + layer.d_w13.numel()].view(layer.d_w13.shape)
    w13.copy_(layer.d_w13)
    with pytest.raises(moe.MoeError) as err:
        moe.forward(layer.d_x, layer.d_rw, layer.d_rb, w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
                    layer.d_b2, k)
    assert err.value.code == 2


def test_mx4_halves_the_weight_bytes(moe):
    E, H, I = 4, 2880, 2880
    assert np.prod(moe.w13_shape_fp4(E, H, I)) * 2 == np.prod(moe.w13_shape(E, H, I))
    assert np.prod(moe.w2_shape_fp4(E, H, I)) * 2 == np.prod(moe.w2_shape(E, H, I))


@pytest.mark.parametrize("name,n_sample", [("oss20b_decode", None), ("oss120b_decode", 32),
                                           ("oss120b_prefill", 24), ("qwen235b_prefill", 24)])
def test_mx4_layer_shapes_full_size(moe, name, n_sample):
    full_check_mx(moe, Layer(synth.config(name), fp4=True), n_sample=n_sample)
    torch.cuda.empty_cache()
