"""The forward entry point that allocates nothing (moe_forward_static_scratch).

It is meant for callers that may not call cudaMalloc/cudaFree themselves --
plugins whose device memory belongs to a host framework's allocator or a
serving engine's fixed pool, or code that keeps allocation out of its latency
path -- so its scratch is a 32 MiB device array inside the library instead of
a caller-provided workspace.  Called through the C ABI, it must give the same
layer output as moe_forward (the entry point with a workspace), on two calls in
a row (the second call finds the first call's leftovers in the shared array),
and must refuse sizes whose scratch would not fit.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from harness import Layer, check_output, torch_bf16_to_np

pytestmark = pytest.mark.gpu


def _call_static(moe, layer, out):
    L = moe.lib()
    ptrs = [layer.d_x, layer.d_rw, layer.d_rb, layer.d_w13, layer.d_s13, layer.d_b13, layer.d_w2, layer.d_s2,
            layer.d_b2]
    return L.moe_forward_static_scratch(*[t.data_ptr() for t in ptrs], layer.T, layer.H, layer.I, layer.E, layer.k,
                                        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_static_scratch_forward_matches_workspace_forward():
    import sparse_moe_layer_gb300 as moe
    moe.build()
    layer = Layer(synth.config("oss20b_decode")).to_device()
    ref, _, _ = layer.run_gpu()  # moe_forward with a caller-provided workspace
    ref_np = torch_bf16_to_np(ref)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        code = _call_static(moe, layer, out)
        assert code == 0, f"call {call}: moe_forward_static_scratch returned {code}"
        torch.cuda.synchronize()
        got = torch_bf16_to_np(out)
        check_output(got, ref_np)
        assert np.array_equal(got, ref_np), f"call {call}: differs from moe_forward"


def test_static_scratch_rejects_sizes_beyond_its_array():
    import sparse_moe_layer_gb300 as moe
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
