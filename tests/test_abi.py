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


def test_product_sources_do_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_layer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle/" not in text and "liboracle" not in text, f
