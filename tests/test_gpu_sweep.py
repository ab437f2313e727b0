"""Small-batch decode on the full-size expert shapes, against the oracle (the
layer as stated, and the MXFP8 and MXFP4-weight variants).

"Hosting Qwen on Blackwell" (sections "Decoders" and "MoE GEMM") measures the
decode MoE GEMM with few tokens and with every expert given one token; here
the gpt-oss-20b- and 120b-shaped layers run with T = 1, 4 and 16 tokens of
their workload (a prefix of its rows) and with a batch that routes exactly one
row to every expert.  Routing, permutation and x codes bit-exact; output
within the layer tolerance on every token.
"""
import dataclasses
import os
import sys

import numpy as np
import pytest
import torch

import synth
from harness import Layer, bf16_np_to_torch
from test_gpu_layer import full_check
from test_gpu_mx import full_check_mx

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402  (the one-row-per-expert batch the bench sweeps)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


_BASE = {}


def base_layer(name: str, fmt: str = "block128") -> Layer:
    """The workload's layer with its weights packed on the device in the format
    (kept for the module)."""
    key = (name, fmt)
    if key not in _BASE:
        _BASE.clear()
        torch.cuda.empty_cache()
        lay = Layer(synth.config(name), mx=fmt == "mx", fp4=fmt == "mxfp4").to_device()
        lay.oracle_weights([])  # create the oracle's weight cache so that the batches below share it
        _BASE[key] = lay
    return _BASE[key]


def with_batch(base: Layer, T: int, x=None, rw=None, rb=None) -> Layer:
    """A batch of T tokens through the base layer's experts (same packed weights)."""
    cfg = dataclasses.replace(base.cfg, T=T)
    lay = Layer(cfg, x=base.x[:T].copy() if x is None else x, rw=base.rw if rw is None else rw,
                rb=base.rb if rb is None else rb, b13=base.b13, b2=base.b2, mx=base.mx, fp4=base.fp4)
    for a in ("d_w13", "d_s13", "d_w2", "d_s2", "d_b13", "d_b2"):
        setattr(lay, a, getattr(base, a))
    lay.d_x, lay.d_rw, lay.d_rb = bf16_np_to_torch(lay.x), bf16_np_to_torch(lay.rw), bf16_np_to_torch(lay.rb)
    lay._oq = base._oq
    return lay


CASES = [(name, T) for name in ("oss20b_decode", "oss120b_decode") for T in (1, 4, 16, "one_per_expert")]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}-T{t}" for n, t in CASES])
def test_small_batch_full_shape(moe, name, T):
    base = base_layer(name)
    if T == "one_per_expert":
        cfg = dataclasses.replace(base.cfg, T=base.E // base.k)
        x, rw, rb = bench.one_per_expert_inputs(cfg)
        lay = with_batch(base, cfg.T, x=x, rw=rw, rb=rb)
    else:
        lay = with_batch(base, T)
    full_check(moe, lay, upload=False)
    if T == "one_per_expert":
        _, v, _ = lay.run_gpu()
        assert np.all(v["count"].cpu().numpy() == 1)


MX_CASES = [(fmt, T) for fmt in ("mx", "mxfp4") for T in (1, 4, "one_per_expert")]


@pytest.mark.parametrize("fmt,T", MX_CASES, ids=[f"oss20b_decode-{f}-T{t}" for f, t in MX_CASES])
def test_small_batch_mx_formats(moe, fmt, T):
    base = base_layer("oss20b_decode", fmt)
    if T == "one_per_expert":
        cfg = dataclasses.replace(base.cfg, T=base.E // base.k)
        x, rw, rb = bench.one_per_expert_inputs(cfg)
        lay = with_batch(base, cfg.T, x=x, rw=rw, rb=rb)
    else:
        lay = with_batch(base, T)
    full_check_mx(moe, lay, upload=False)
