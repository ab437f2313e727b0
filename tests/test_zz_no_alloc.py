"""The forward entry point that allocates nothing (moe_forward_static_scratch).

It is meant for callers that may not call cudaMalloc/cudaFree themselves --
plugins whose device memory belongs to a host framework's allocator or a
serving engine's fixed pool, or code that keeps allocation out of its latency
path -- so its scratch is a 32 MiB device array inside the library instead of
a caller-provided workspace.  Called through the C ABI, it must give the same
layer output as moe_forward (the entry point with a workspace), bit for bit, on
two calls in a row (the second call finds the first call's leftovers in the
shared array), with the array's status word reading MOE_OK after each call, on
a decode-sized batch (the weight-streaming GEMMs) and on a prefill-sized one
(the 128-row tile GEMMs), and must refuse sizes whose scratch would not fit.
"""
import numpy as np
import pytest
import torch

import synth
from harness import Layer, check_output, torch_bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def _call_static(moe, layer, out):
    L = moe.lib()
    ptrs = [layer.d_x, layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
            layer.d_b2]
    return L.moe_forward_static_scratch(*[t.data_ptr() for t in ptrs], layer.T, layer.H, layer.I, layer.E, layer.k,
                                        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _prefill_sized_layer():
    # 1024 tokens x top-2 over 8 experts: 2048 rows > 64 rows per expert, so the
    # 128-row tile GEMMs run; its workspace is a few MiB
    cfg = synth.LayerConfig("static_prefill", 1024, 256, 256, 8, 2, 5, "normal", "normal")
    return Layer(cfg, x=synth.x_rows(cfg))  # GPU against GPU: no margin redraws needed


@pytest.mark.parametrize("make", [lambda: Layer(synth.config("oss20b_decode")), _prefill_sized_layer],
                         ids=["decode_oss20b", "prefill_tiny"])
def test_static_scratch_forward_matches_workspace_forward(moe, make):
    layer = make().to_device()
    R = layer.T * layer.k
    assert moe.workspace_size(layer.T, layer.H, layer.I, layer.E, layer.k) <= (32 << 20)
    ref, _, ws = layer.run_gpu()  # moe_forward with a caller-provided workspace
    assert moe.read_device_status(ws) == 0
    ref_np = torch_bf16_to_np(ref)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        code = _call_static(moe, layer, out)
        assert code == 0, f"call {call}: moe_forward_static_scratch returned {code}"
        assert moe.read_static_scratch_status() == 0, f"call {call}: a device wait timed out"
        got = torch_bf16_to_np(out)
        check_output(got, ref_np)
        assert np.array_equal(got, ref_np), f"call {call}: differs from moe_forward (R={R})"


def test_static_scratch_rejects_sizes_beyond_its_array(moe):
    layer = Layer(synth.config("tiny")).to_device()
    L = moe.lib()
    big_T = 8192  # workspace of T=8192, H=I=2880, E=128, k=4 is far above 32 MiB
    assert L.moe_workspace_size(big_T, 2880, 2880, 128, 4) > (32 << 20)
    out = torch.empty((1, 1), dtype=torch.bfloat16, device="cuda")
    ptrs = [layer.d_x, layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
            layer.d_b2]
    code = L.moe_forward_static_scratch(*[t.data_ptr() for t in ptrs], big_T, 2880, 2880, 128, 4, out.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert code == 3  # MOE_ERR_WORKSPACE, before anything is launched
    torch.cuda.synchronize()
