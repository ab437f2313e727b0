"""Shared helpers for the parity tests: build one layer's inputs for the CUDA
path (device tensors, weights packed by the library) and for the oracle
(numpy arrays, weights packed by the oracle), and compare the two."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import synth

TOL_MAX = 2e-2  # max|gpu - oracle| <= TOL_MAX * max|oracle|
TOL_MEAN = 2e-3  # mean|gpu - oracle| <= TOL_MEAN * mean|oracle|


def threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_np_to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def torch_bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Layer:
    """Inputs of one layer shape: host arrays (bf16 as uint16 bits) plus device tensors."""

    def __init__(self, cfg: synth.LayerConfig, x: np.ndarray | None = None, rw=None, rb=None, b13=None, b2=None,
                 w13_master=None, w2_master=None, mx: bool = False, fp4: bool = False):
        self.cfg = cfg
        self.mx = mx or fp4  # MX variant (1x32 UE8M0 scales) instead of 128x128 / 1x128 fp32 scales
        self.fp4 = fp4  # MXFP4 weights (E2M1 codes), MXFP8 activations
        self.T, self.H, self.I, self.E, self.k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
        self.Hp, self.Ip = cfg.Hp, cfg.Ip
        self.x = synth.layer_x(cfg) if x is None else x
        if rw is None:
            rw, rb = synth.router(cfg)
        self.rw, self.rb = rw, rb
        if b13 is None:
            b13, b2 = synth.expert_biases(cfg)
        self.b13, self.b2 = b13, b2
        self._w13_master, self._w2_master = w13_master, w2_master  # explicit masters (edge-case tests)
        self._oq = None

    # ---- master weights (fp32), per expert range ----
    def w13_master(self, first: int, count: int) -> np.ndarray:
        if self._w13_master is not None:
            return np.ascontiguousarray(self._w13_master[first:first + count])
        return synth.w13_master(self.cfg, first, count)

    def w2_master(self, first: int, count: int) -> np.ndarray:
        if self._w2_master is not None:
            return np.ascontiguousarray(self._w2_master[first:first + count])
        return synth.w2_master(self.cfg, first, count)

    # ---- CUDA side ----
    def to_device(self, chunk_experts: int = 8):
        import sparse_moe_layer_gb300 as moe
        E, H, I, Hp, Ip = self.E, self.H, self.I, self.Hp, self.Ip
        dev = "cuda"
        self.d_x = bf16_np_to_torch(self.x)
        self.d_rw = bf16_np_to_torch(self.rw)
        self.d_rb = bf16_np_to_torch(self.rb)
        self.d_b13 = bf16_np_to_torch(self.b13)
        self.d_b2 = bf16_np_to_torch(self.b2)
        q13_shape, q2_shape = ((moe.w13_shape_fp4, moe.w2_shape_fp4) if self.fp4 else (moe.w13_shape, moe.w2_shape))
        self.d_w13 = torch.empty(q13_shape(E, H, I), dtype=torch.uint8, device=dev)
        self.d_w2 = torch.empty(q2_shape(E, H, I), dtype=torch.uint8, device=dev)
        if self.mx:
            self.d_s13 = torch.empty(moe.s13_mx_shape(E, H, I), dtype=torch.uint8, device=dev)
            self.d_s2 = torch.empty(moe.s2_mx_shape(E, H, I), dtype=torch.uint8, device=dev)
        else:
            self.d_s13 = torch.empty((E, 2 * Ip // 128, Hp // 128), dtype=torch.float32, device=dev)
            self.d_s2 = torch.empty((E, Hp // 128, Ip // 128), dtype=torch.float32, device=dev)
        pack = (moe.pack_weights_into_mxfp4 if self.fp4 else
                moe.pack_weights_into_mx if self.mx else moe.pack_weights_into)
        for e0 in range(0, E, chunk_experts):
            n = min(chunk_experts, E - e0)
            m13 = torch.from_numpy(self.w13_master(e0, n)).to(dev)
            m2 = torch.from_numpy(self.w2_master(e0, n)).to(dev)
            pack(m13, m2, H, I, n, self.d_w13[e0:e0 + n], self.d_s13[e0:e0 + n], self.d_w2[e0:e0 + n],
                 self.d_s2[e0:e0 + n])
            torch.cuda.synchronize()
            del m13, m2
        return self

    def run_gpu(self, workspace=None):
        import sparse_moe_layer_gb300 as moe
        if workspace is None:
            workspace = moe.new_workspace(self.T, self.H, self.I, self.E, self.k, mx=self.mx)
        out = moe.forward(self.d_x, self.d_rw, self.d_rb, self.d_w13, self.d_s13, self.d_b13, self.d_w2, self.d_s2,
                          self.d_b2, self.k, workspace=workspace)
        torch.cuda.synchronize()
        views = moe.workspace_views(workspace, self.T, self.H, self.I, self.E, self.k, mx=self.mx)
        return out, views, workspace

    # ---- oracle side ----
    def oracle_weights(self, experts) -> tuple:
        """Oracle-packed codes/scales as full [E, ...] arrays with only `experts` filled."""
        E, Hp, Ip = self.E, self.Hp, self.Ip
        if self._oq is None:
            if self.mx:
                self._oq = (np.zeros((E, 2 * Ip, Hp), np.uint8), np.zeros((E, 2 * Ip, Hp // 32), np.uint8),
                            np.zeros((E, Hp, Ip), np.uint8), np.zeros((E, Hp, Ip // 32), np.uint8), set())
            else:
                self._oq = (np.zeros((E, 2 * Ip, Hp), np.uint8), np.ones((E, 2 * Ip // 128, Hp // 128), np.float32),
                            np.zeros((E, Hp, Ip), np.uint8), np.ones((E, Hp // 128, Ip // 128), np.float32), set())
        q13, s13, q2, s2, done = self._oq
        todo = sorted(set(int(e) for e in experts) - done)
        p13, p2 = ((oracle.mx4_pack_w13, oracle.mx4_pack_w2) if self.fp4 else
                   (oracle.mx_pack_w13, oracle.mx_pack_w2) if self.mx else (oracle.pack_w13, oracle.pack_w2))

        def one(e):
            p13(self.w13_master(e, 1), q13[e:e + 1], s13[e:e + 1])
            p2(self.w2_master(e, 1), q2[e:e + 1], s2[e:e + 1])

        with ThreadPoolExecutor(max_workers=threads()) as ex:
            list(ex.map(one, todo))
        done.update(todo)
        return q13, s13, q2, s2

    def oracle_router(self):
        rows = np.array_split(np.arange(self.T), max(1, min(self.T, 4 * threads())))
        rows = [r for r in rows if len(r)]

        def one(r):
            return oracle.router(np.ascontiguousarray(self.x[r]), self.rw, self.rb, self.k)

        with ThreadPoolExecutor(max_workers=threads()) as ex:
            parts = list(ex.map(one, rows))
        return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}

    def oracle_forward(self, tokens, idx_all=None):
        tokens = np.asarray(tokens, np.int32)
        if idx_all is None:
            idx_all = self.oracle_router()["idx"]
        q13, s13, q2, s2 = self.oracle_weights(np.unique(idx_all[tokens]))
        chunks = [c for c in np.array_split(tokens, max(1, min(len(tokens), threads()))) if len(c)]

        fwd = oracle.mx4_forward if self.fp4 else oracle.mx_forward if self.mx else oracle.forward

        def one(c):
            return fwd(self.x, self.rw, self.rb, q13, s13, self.b13, q2, s2, self.b2, self.k, tokens=c,
                       want_intermediates=True)

        with ThreadPoolExecutor(max_workers=threads()) as ex:
            parts = list(ex.map(one, chunks))
        out = np.concatenate([p[0] for p in parts])
        inter = {key: np.concatenate([p[1][key] for p in parts]) for key in parts[0][1]}
        return out, inter


def mx_row_scales(atoms: np.ndarray, count: np.ndarray, offset: np.ndarray, tiles: np.ndarray, nt: int,
                  bm: int) -> np.ndarray:
    """Activation scale atoms [m-tiles, KB, 512] -> UE8M0 bytes [R, KB*4] by permuted row.
    Row r of expert e sits in m-tile tiles[e]/nt + (r - offset[e]) // bm at row
    m = (r - offset[e]) % bm of that tile; the atom byte of (m, group g) is
    (m % 32) * 16 + (m // 32) * 4 + g."""
    KB = atoms.shape[1]
    R = int(offset[-1])
    out = np.zeros((R, KB * 4), np.uint8)
    for e in range(len(count)):
        for r in range(int(offset[e]), int(offset[e]) + int(count[e])):
            local = r - int(offset[e])
            mt, m = int(tiles[e]) // nt + local // bm, local % bm
            byte = (m % 32) * 16 + (m // 32) * 4
            out[r] = atoms[mt, :, byte:byte + 4].reshape(-1)
    return out


def sample_tokens(idx: np.ndarray, E: int, n: int, seed: int = 0, perm: np.ndarray | None = None,
                  offset: np.ndarray | None = None, bm: int = 128) -> np.ndarray:
    """Tokens for sampled output checks: first, last, the tokens of the most- and
    least-loaded (non-empty) experts, and seeded random others up to n; with the
    permutation (perm, offset) also the tokens in the first and last row of every
    expert's last bm-row GEMM tile (the partial M tile of the grouped GEMMs)."""
    T, k = idx.shape
    if T <= n:
        return np.arange(T, dtype=np.int32)
    counts = np.bincount(idx.ravel(), minlength=E)
    nz = np.nonzero(counts)[0]
    most, least = nz[np.argmax(counts[nz])], nz[np.argmin(counts[nz])]
    pick = {0, T - 1}
    for e in (most, least):
        ts = np.nonzero((idx == e).any(axis=1))[0]
        pick.update(int(t) for t in ts[:2])
        pick.add(int(ts[-1]))
    if perm is not None and offset is not None:
        for e in nz:
            lo, hi = int(offset[e]), int(offset[e + 1])
            last_tile = lo + (hi - lo - 1) // bm * bm
            pick.add(int(perm[last_tile]) // k)
            pick.add(int(perm[hi - 1]) // k)
    rng = np.random.default_rng(seed)
    while len(pick) < n:
        pick.add(int(rng.integers(T)))
    return np.array(sorted(pick), dtype=np.int32)


def check_output(gpu_rows: np.ndarray, oracle_rows: np.ndarray):
    g = synth.bf16_to_f32(gpu_rows).astype(np.float64)
    o = synth.bf16_to_f32(oracle_rows).astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    d = np.abs(g - o)
    max_ok = d.max() <= TOL_MAX * np.abs(o).max()
    mean_ok = d.mean() <= TOL_MEAN * np.abs(o).mean()
    assert max_ok and mean_ok, (f"out mismatch: max|d|={d.max():.4g} (limit {TOL_MAX * np.abs(o).max():.4g}), "
                                f"mean|d|={d.mean():.4g} (limit {TOL_MEAN * np.abs(o).mean():.4g})")
    return d.max() / np.abs(o).max(), d.mean() / np.abs(o).mean()


def check_codes_close(gpu: np.ndarray, ref: np.ndarray, min_equal: float = 0.999):
    """e4m3 codes from fp32 inputs that differ in rounding: almost all equal,
    the rest neighbours (same sign, magnitude code +-1, or both near zero)."""
    eq = gpu == ref
    frac = eq.mean()
    assert frac >= min_equal, f"only {frac:.5f} of codes identical"
    a, b = gpu[~eq].astype(np.int32), ref[~eq].astype(np.int32)
    ma, mb = a & 0x7F, b & 0x7F
    ok = ((a >> 7) == (b >> 7)) & (np.abs(ma - mb) <= 1) | ((ma <= 1) & (mb <= 1))
    assert ok.all(), f"{(~ok).sum()} codes differ by more than one step"
    return frac
