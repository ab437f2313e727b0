"""The Python binding's host side on the CPU: it refuses anything but CUDA
tensors (there is no CPU fallback), checks the packed weight shapes before
calling the library, tells the weight formats apart, and its layout helpers
agree with the library's tile rule."""
import pytest
import torch

import sparse_moe_layer_gb300 as moe


def _layer_tensors(E=4, H=256, I=256, device="cpu", fmt="block128"):
    bf = torch.bfloat16
    x = torch.zeros((8, H), dtype=bf, device=device)
    rw = torch.zeros((E, H), dtype=bf, device=device)
    rb = torch.zeros((E,), dtype=bf, device=device)
    b13 = torch.zeros((E, 2 * I), dtype=bf, device=device)
    b2 = torch.zeros((E, H), dtype=bf, device=device)
    if fmt == "block128":
        w13 = torch.zeros(moe.w13_shape(E, H, I), dtype=torch.uint8, device=device)
        w2 = torch.zeros(moe.w2_shape(E, H, I), dtype=torch.uint8, device=device)
        s13 = torch.ones((E, 2 * moe.pad128(I) // 128, moe.pad128(H) // 128), device=device)
        s2 = torch.ones((E, moe.pad128(H) // 128, moe.pad128(I) // 128), device=device)
    else:
        shp13, shp2 = ((moe.w13_shape_fp4, moe.w2_shape_fp4) if fmt == "mxfp4" else (moe.w13_shape, moe.w2_shape))
        w13 = torch.zeros(shp13(E, H, I), dtype=torch.uint8, device=device)
        w2 = torch.zeros(shp2(E, H, I), dtype=torch.uint8, device=device)
        s13 = torch.zeros(moe.s13_mx_shape(E, H, I), dtype=torch.uint8, device=device)
        s2 = torch.zeros(moe.s2_mx_shape(E, H, I), dtype=torch.uint8, device=device)
    return x, rw, rb, w13, s13, b13, w2, s2, b2


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()


@pytest.mark.parametrize("fmt", ["block128", "mxfp8", "mxfp4"])
def test_forward_refuses_host_tensors(fmt):
    args = _layer_tensors(fmt=fmt)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    out = torch.zeros((8, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        moe.forward(*args, 2, out=out, workspace=ws)


def test_forward_checks_packed_shapes_before_the_library():
    x, rw, rb, w13, s13, b13, w2, s2, b2 = _layer_tensors()
    with pytest.raises(ValueError, match="packed weight shapes"):
        moe.forward(x, rw, rb, w13[:, :1], s13, b13, w2, s2, b2, 2)
    with pytest.raises(ValueError, match="block scale shapes"):
        moe.forward(x, rw, rb, w13, s13[:, :1], b13, w2, s2, b2, 2)
    x, rw, rb, w13, s13, b13, w2, s2, b2 = _layer_tensors(fmt="mxfp8")
    with pytest.raises(ValueError, match="MX scale atom shapes"):
        moe.forward(x, rw, rb, w13, s13[:, :1], b13, w2, s2, b2, 2)


def test_weight_format_from_scale_dtype_and_row_width():
    for fmt in ("block128", "mxfp8", "mxfp4"):
        _, _, _, w13, s13, _, _, _, _ = _layer_tensors(fmt=fmt)
        assert moe.weight_format(w13, s13) == fmt


def test_m_tile_rows_follows_the_decode_rule():
    # decode-sized (at most 64 rows per expert on average): 32-row tiles; else 128
    assert moe.m_tile_rows(64, 32, 4) == 32
    assert moe.m_tile_rows(512, 32, 4) == 32  # 2048 rows = 64 per expert
    assert moe.m_tile_rows(513, 32, 4) == 128
    assert moe.m_tile_rows(8192, 128, 4) == 128


def test_unblock_is_the_blocked_layout_inverse():
    E, RB, KB = 2, 3, 2
    rows = torch.arange(E * RB * 128 * KB * 128, dtype=torch.int64).reshape(E, RB * 128, KB * 128)
    blocked = rows.reshape(E, RB, 128, KB, 128).permute(0, 1, 3, 2, 4).contiguous()
    assert torch.equal(moe.unblock(blocked), rows)
    # element (row r, column c) of expert e lives in block (r // 128, c // 128) at (r % 128, c % 128)
    e, r, c = 1, 300, 200
    assert int(blocked[e, r // 128, c // 128, r % 128, c % 128]) == int(rows[e, r, c])
