"""The boundary calls beside the forward, through the C ABI, on the GPU.

moe_route_debug: the routing steps alone ("GPT-OSS on Day 0", MoE section: the
routing kernel -- top-k, then softmax over the selected experts -- kept apart
from the expert GEMMs) into caller buffers; indices, offsets, the permutation
and the 1x128 FP8 codes and scales of x must equal the oracle's bit for bit.

moe_block_weights: row-major FP8 codes (the layout of the layer statement,
128x128 block scales from "GPT-OSS on Day 0", infrastructure decisions) into
the blocked layout the GEMMs read; codes packed by the oracle and converted
must equal the library packer's output, and a forward on them must give the
same output bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import Layer, bf16_np_to_torch, torch_bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("name", ["oss20b_decode", "oss120b_prefill"])
def test_route_debug_bit_exact(moe, name):
    cfg = synth.config(name)
    layer = Layer(cfg)  # host arrays only: routing needs no expert weights
    x, rw, rb = bf16_np_to_torch(layer.x), bf16_np_to_torch(layer.rw), bf16_np_to_torch(layer.rb)
    got = moe.route_debug(x, rw, rb, cfg.top_k)
    torch.cuda.synchronize()
    r = layer.oracle_router()
    assert np.array_equal(got["topk_idx"].cpu().numpy(), r["idx"])
    wrel = np.abs(got["topk_w"].cpu().numpy() - r["w_f32"]) / r["w_f32"]
    assert wrel.max() <= 5e-5  # fp32 logits within ~2.5e-5 of the fp64 ones for H <= 4096
    p = oracle.permute(r["idx"], cfg.E)
    assert np.array_equal(got["offset"].cpu().numpy(), p["offset"])
    assert np.array_equal(got["perm"].cpu().numpy(), p["perm"])
    xq, sx = oracle.quant_rows_bf16(layer.x)
    tok = p["perm"] // cfg.top_k
    assert np.array_equal(got["xq"].cpu().numpy(), xq[tok])
    assert np.array_equal(got["sx"].cpu().numpy(), sx[tok])


@pytest.mark.parametrize("H,I,E", [(200, 130, 3), (2880, 2880, 2)])
def test_block_weights_equal_the_packer(moe, H, I, E):
    rng = np.random.default_rng(H * 7 + I)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    oq13, _ = oracle.pack_w13(w13)  # row-major codes [E, 2Ip, Hp]
    oq2, _ = oracle.pack_w2(w2)  # [E, Hp, Ip]
    b13, b2 = moe.block_weights(torch.from_numpy(oq13).cuda(), torch.from_numpy(oq2).cuda(), H, I)
    q13, _, q2, _ = moe.pack_weights(torch.from_numpy(w13).cuda(), torch.from_numpy(w2).cuda())
    torch.cuda.synchronize()
    assert torch.equal(b13, q13) and torch.equal(b2, q2)
    assert np.array_equal(moe.unblock(b13).cpu().numpy(), oq13)


def test_forward_on_converted_row_major_codes(moe):
    layer = Layer(synth.config("tiny")).to_device()
    ref, _, _ = layer.run_gpu()
    q13, s13, q2, s2 = layer.oracle_weights(range(layer.E))  # oracle-packed, row-major
    b13, b2 = moe.block_weights(torch.from_numpy(q13).cuda(), torch.from_numpy(q2).cuda(), layer.H, layer.I)
    out = moe.forward(layer.d_x, layer.d_rw, layer.d_rb, b13, torch.from_numpy(s13).cuda(), layer.d_b13, b2,
                      torch.from_numpy(s2).cuda(), layer.d_b2, layer.k)
    torch.cuda.synchronize()
    assert np.array_equal(torch_bf16_to_np(out), torch_bf16_to_np(ref))
