"""Seeded synthetic inputs for the sparse MoE layer (shared by tests and bench).

The numbers come from ``synth.c`` (SplitMix64 streams + Box-Muller, identical
bits on x86-64 and aarch64).  This module only draws and shapes inputs; it
holds none of the layer's arithmetic.  Weight tensors are drawn as fp32
"master" weights; turning them into FP8 codes and block scales is the job of
the library's packer (and, independently, of the oracle).

Workloads (the five layer shapes this project measures; gpt-oss-20b/120b and a
Qwen3-235B-shaped layer, from the "GPT-OSS on Day 0" and "Hosting Qwen on
Blackwell" posts):

  tiny           T=64    H=256  I=256  E=8   k=2  seed 0
  oss20b_decode  T=64    H=2880 I=2880 E=32  k=4  seed 1  router_b = 0
  oss120b_decode T=256   H=2880 I=2880 E=128 k=4  seed 2  Zipf router_b
  oss120b_prefill T=8192 H=2880 I=2880 E=128 k=4  seed 3  router_b = 0
  qwen235b_prefill T=16384 H=4096 I=1536 E=128 k=8 seed 4 Zipf router_b, zero expert biases

Distributions (std-dev sigma unless noted): x ~ N(0,1) bf16; router_w ~ N(0, 1/H)
read as variance (sigma = 1/sqrt(H)) bf16; router_b ~ N(0, 0.1) bf16 for the
tiny layer, 0 or Zipf 0.5*ln(1/(e+1)) otherwise; w13 [E,2I,H], w2 [E,H,I] ~
N(0, 0.02) fp32 masters; b13 [E,2I], b2 [E,H] ~ N(0, 0.01) bf16 (zero for the
Qwen-shaped layer).  Row t of x may be redrawn (attempt > 0) so that its
top-k margin is at least 1e-3; the attempts per row are data passed in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

TAG_X, TAG_RW, TAG_RB, TAG_W13, TAG_B13, TAG_W2, TAG_B2 = 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
    """Compile libsynth.so (plain C, no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-pthread", "-o", _LIB, _SRC, "-lm"])
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, u32, i32, dbl, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.synth_stream_key.argtypes = [u64, u32, u64, u32]
        L.synth_stream_key.restype = u64
        L.synth_draw_u64.argtypes = [u64, u64]
        L.synth_draw_u64.restype = u64
        L.synth_ln.argtypes = [dbl]
        L.synth_ln.restype = dbl
        L.synth_normal_at.argtypes = [u64, u64]
        L.synth_normal_at.restype = dbl
        L.synth_tensor.argtypes = [u64, u32, u64, u64, u64, vp, dbl, vp, vp, i32]
        L.synth_tensor.restype = None
        L.synth_zipf_bias_bf16.argtypes = [i32, dbl, vp]
        L.synth_zipf_bias_bf16.restype = None
        _lib = L
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    seed: int
    router_b: str  # "normal" (sigma 0.1), "zero" or "zipf"
    expert_bias: str  # "normal" (sigma 0.01) or "zero"

    @property
    def Hp(self) -> int:
        return (self.H + 127) // 128 * 128

    @property
    def Ip(self) -> int:
        return (self.I + 127) // 128 * 128

    @property
    def R(self) -> int:
        return self.T * self.top_k


CONFIGS = [
    LayerConfig("tiny", 64, 256, 256, 8, 2, 0, "normal", "normal"),
    LayerConfig("oss20b_decode", 64, 2880, 2880, 32, 4, 1, "zero", "normal"),
    LayerConfig("oss120b_decode", 256, 2880, 2880, 128, 4, 2, "zipf", "normal"),
    LayerConfig("oss120b_prefill", 8192, 2880, 2880, 128, 4, 3, "zero", "normal"),
    LayerConfig("qwen235b_prefill", 16384, 4096, 1536, 128, 8, 4, "zipf", "zero"),
]
BY_NAME = {c.name: c for c in CONFIGS}


def config(name_or_index) -> LayerConfig:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    return BY_NAME[name_or_index]


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def tensor(seed: int, tag: int, majors: int, per_major: int, sigma: float, dtype: str,
           major_base: int = 0, attempts: np.ndarray | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """[majors, per_major] values sigma*N(0,1); dtype 'f32' -> float32, 'bf16' -> uint16 bit patterns."""
    np_dtype = np.float32 if dtype == "f32" else np.uint16
    if out is None:
        out = np.empty((majors, per_major), dtype=np_dtype)
    assert out.dtype == np_dtype and out.flags.c_contiguous and out.size == majors * per_major
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.uint32)
        assert att.shape == (majors,)
    lib().synth_tensor(seed, tag, major_base, majors, per_major, None if att is None else _ptr(att), float(sigma),
                       _ptr(out) if dtype == "f32" else None, _ptr(out) if dtype == "bf16" else None, _threads())
    return out


_REDRAWS = os.path.join(os.path.dirname(_HERE), "tests", "golden", "margin_redraws.json")


def margin_attempts(cfg: LayerConfig) -> np.ndarray:
    """Per-row redraw counts of x for this layer shape (a stored data table)."""
    import json
    with open(_REDRAWS) as f:
        table = json.load(f)
    if cfg.name not in table:
        raise KeyError(f"no redraw table for {cfg.name}; regenerate tests/golden/margin_redraws.json")
    att = np.zeros(cfg.T, np.uint32)
    for t, a in table[cfg.name].items():
        if int(t) < cfg.T:  # a shape with fewer tokens uses a prefix of the rows
            att[int(t)] = a
    return att


def x_rows(cfg: LayerConfig, attempts: np.ndarray | None = None, rows: np.ndarray | None = None) -> np.ndarray:
    """x [T,H] bf16 bits.  Row t uses stream (seed, x, t, attempts[t])."""
    if rows is None:
        return tensor(cfg.seed, TAG_X, cfg.T, cfg.H, 1.0, "bf16", attempts=attempts)
    out = np.empty((len(rows), cfg.H), dtype=np.uint16)
    for i, t in enumerate(rows):
        a = 0 if attempts is None else int(attempts[t])
        tensor(cfg.seed, TAG_X, 1, cfg.H, 1.0, "bf16", major_base=int(t),
               attempts=np.array([a], dtype=np.uint32), out=out[i:i + 1])
    return out


def router(cfg: LayerConfig):
    """router_w [E,H] bf16 bits (sigma 1/sqrt(H)), router_b [E] bf16 bits."""
    rw = tensor(cfg.seed, TAG_RW, cfg.E, cfg.H, 1.0 / np.sqrt(float(cfg.H)), "bf16")
    if cfg.router_b == "normal":
        rb = tensor(cfg.seed, TAG_RB, 1, cfg.E, 0.1, "bf16").reshape(cfg.E)
    elif cfg.router_b == "zero":
        rb = np.zeros(cfg.E, dtype=np.uint16)
    elif cfg.router_b == "zipf":
        rb = np.empty(cfg.E, dtype=np.uint16)
        lib().synth_zipf_bias_bf16(cfg.E, 0.5, _ptr(rb))
    else:
        raise ValueError(cfg.router_b)
    return rw, rb


def expert_biases(cfg: LayerConfig):
    """b13 [E, 2I] (gate then up) and b2 [E, H], bf16 bits."""
    if cfg.expert_bias == "zero":
        return np.zeros((cfg.E, 2 * cfg.I), np.uint16), np.zeros((cfg.E, cfg.H), np.uint16)
    b13 = tensor(cfg.seed, TAG_B13, cfg.E, 2 * cfg.I, 0.01, "bf16")
    b2 = tensor(cfg.seed, TAG_B2, cfg.E, cfg.H, 0.01, "bf16")
    return b13, b2


def w13_master(cfg: LayerConfig, first: int = 0, count: int | None = None, out=None) -> np.ndarray:
    """fp32 w13 [count, 2I, H] for experts [first, first+count): rows [0,I) gate, [I,2I) up."""
    count = cfg.E - first if count is None else count
    o = tensor(cfg.seed, TAG_W13, count, 2 * cfg.I * cfg.H, 0.02, "f32", major_base=first,
               out=None if out is None else out.reshape(count, -1))
    return o.reshape(count, 2 * cfg.I, cfg.H)


def w2_master(cfg: LayerConfig, first: int = 0, count: int | None = None, out=None) -> np.ndarray:
    """fp32 w2 [count, H, I] for experts [first, first+count)."""
    count = cfg.E - first if count is None else count
    o = tensor(cfg.seed, TAG_W2, count, cfg.H * cfg.I, 0.02, "f32", major_base=first,
               out=None if out is None else out.reshape(count, -1))
    return o.reshape(count, cfg.H, cfg.I)


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def layer_x(cfg: LayerConfig) -> np.ndarray:
    """x [T,H] bf16 bits of the layer workload, margin redraws applied."""
    return x_rows(cfg, margin_attempts(cfg))
