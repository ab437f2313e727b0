"""The C-ABI library: it loads, exports every entry point the header declares,
checks arguments on the host, and contains none of the oracle.  No GPU needed."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def moe():
    import sparse_moe_layer_gb300 as m
    m.build()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("moe_forward", "moe_workspace_size", "moe_get_workspace_layout", "moe_pack_weights",
              "moe_quantize_rows", "moe_read_device_status", "moe_status_str"):
        assert f in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(moe_[a-z_0-9]+)\b", out))
    assert set(declared_functions()) <= exported
    assert "oracle_" not in out and "synth_" not in out


def test_host_argument_checks(moe):
    L = moe.lib()
    assert L.moe_workspace_size(0, 256, 256, 8, 2) == 0
    assert L.moe_workspace_size(64, 256, 256, 8, 9) == 0  # top_k > 8
    assert L.moe_workspace_size(64, 256, 256, 2, 3) == 0  # top_k > E
    assert L.moe_workspace_size(64, 256, 256, 300, 2) == 0  # E > 256
    assert L.moe_workspace_size(64, 256, 256, 8, 2) > 0
    lay = moe.workspace_layout(64, 2880, 2880, 32, 4)
    offs = [lay[k] for k in ("status", "hist", "count", "offset", "chunk_base", "tiles1", "tiles2", "topk_idx",
                             "topk_w", "topk_wb", "perm", "inv", "xq", "sx", "hq", "sh", "part")]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay["total_bytes"] >= lay["part"] + 256 * 2944 * 4
    # null pointers are rejected before any CUDA call
    args = [None] * 9 + [64, 256, 256, 8, 2, None, None, 0, None]
    assert L.moe_forward(*args) == 1
    assert L.moe_pack_weights(None, None, 256, 256, 8, None, None, None, None, None) == 1
    assert L.moe_quantize_rows(None, 4, 4, 4, None, None, None) == 1
    assert L.moe_status_str(5) == b"a bounded device-side wait timed out"


def test_mx_host_argument_checks_and_layout(moe):
    L = moe.lib()
    for f in ("moe_forward_mx", "moe_forward_mx_profiled", "moe_pack_weights_mx", "moe_quantize_rows_mx",
              "moe_workspace_size_mx", "moe_get_workspace_layout_mx"):
        assert f in declared_functions()
    assert L.moe_workspace_size_mx(0, 256, 256, 8, 2) == 0
    args = [None] * 9 + [64, 256, 256, 8, 2, None, None, 0, None]
    assert L.moe_forward_mx(*args) == 1
    assert L.moe_pack_weights_mx(None, None, 256, 256, 8, None, None, None, None, None) == 1
    assert L.moe_quantize_rows_mx(None, 4, 4, 4, None, None, None) == 1
    # scale atoms: one 512-byte atom per (m-tile, K block); m-tiles <= E + ceil(R / bm)
    for T, E, k, bm in ((64, 32, 4, 32), (8192, 128, 4, 128)):
        R, Hp, Ip = T * k, 2944, 2944
        lay = moe.workspace_layout(T, 2880, 2880, E, k, mx=True)
        mtb = E + (R + bm - 1) // bm
        assert moe.m_tile_rows(T, E, k) == bm
        assert lay["xq"] + R * Hp <= lay["sx"] and lay["sx"] + mtb * (Hp // 128) * 512 <= lay["hq"]
        assert lay["hq"] + R * Ip <= lay["sh"] and lay["sh"] + mtb * (Ip // 128) * 512 <= lay["part"]
        assert all(lay[f] % 256 == 0 for f in ("sx", "sh", "part"))
        assert moe.workspace_size(T, 2880, 2880, E, k, mx=True) == lay["total_bytes"]


def test_mx_scale_atom_unblocking(moe):
    import torch
    s = (torch.arange(2 * 3 * 2 * 512) % 251).to(torch.uint8).reshape(2, 3, 2, 512)
    u = moe.unblock_scales_mx(s)
    assert tuple(u.shape) == (2, 3 * 128, 2 * 4)
    for e, rb, kb, r, g in ((0, 0, 0, 0, 0), (1, 2, 1, 77, 3), (0, 1, 0, 127, 2), (1, 0, 1, 33, 1)):
        assert int(u[e, rb * 128 + r, kb * 4 + g]) == int(s[e, rb, kb, (r % 32) * 16 + (r // 32) * 4 + g])


def test_product_sources_do_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_layer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle/" not in text and "liboracle" not in text, f


def test_static_scratch_limits_on_the_host(moe):
    """The entry point without a workspace checks its pointers first, then refuses
    invalid sizes and sizes whose scratch exceeds its 32 MiB array, all before any
    CUDA call; the decode shapes fit."""
    L = moe.lib()
    nul = [None] * 9
    fake = [16 * (i + 1) for i in range(9)]  # non-null, never dereferenced: every check runs on the host first
    assert L.moe_forward_static_scratch(*nul, 8192, 2880, 2880, 128, 4, None, None) == 1  # null pointers first
    assert L.moe_forward_static_scratch(*fake, 8192, 2880, 2880, 128, 4, 16, None) == 3  # MOE_ERR_WORKSPACE
    assert L.moe_forward_static_scratch(*fake, 0, 2880, 2880, 128, 4, 16, None) == 1  # MOE_ERR_INVALID_ARG
    for T, E in ((64, 32), (256, 128)):
        assert 0 < L.moe_workspace_size(T, 2880, 2880, E, 4) <= (32 << 20)
    assert L.moe_workspace_size(8192, 2880, 2880, 128, 4) > (32 << 20)


def test_route_debug_and_block_weights_host_checks(moe):
    L = moe.lib()
    for f in ("moe_route_debug", "moe_route_workspace_size", "moe_block_weights", "moe_read_static_scratch_status"):
        assert f in declared_functions()
    assert L.moe_route_workspace_size(0, 256, 8, 2) == 0
    assert L.moe_route_workspace_size(64, 256, 8, 9) == 0
    assert L.moe_route_workspace_size(64, 256, 8, 2) > 0
    fake = [16 * (i + 1) for i in range(3)]
    outs = [256 * (i + 1) for i in range(6)]
    assert L.moe_route_debug(None, None, None, 64, 256, 8, 2, *([None] * 6), None, 0, None) == 1
    assert L.moe_route_debug(*fake, 0, 256, 8, 2, *outs, 4096, 1 << 20, None) == 1  # T < 1
    assert L.moe_route_debug(*fake, 64, 256, 8, 2, *outs, 4096 + 8, 1 << 20, None) == 2  # workspace not 256-aligned
    assert L.moe_route_debug(*fake, 64, 256, 8, 2, *outs, 4096, 16, None) == 3  # short workspace
    assert L.moe_block_weights(None, None, 256, 256, 8, None, None, None) == 1
    assert L.moe_block_weights(16, None, 256, 256, 8, None, None, None) == 1  # w13 output missing
    assert L.moe_block_weights(17, None, 256, 256, 8, 32, None, None) == 2  # misaligned input
