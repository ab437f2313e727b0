#!/usr/bin/env python
"""MoE-layer tokens/s on one GB300 (sparse gpt-oss-style MoE MLP forward).

One step = one call of the whole layer (router, top-k + softmax, grouping by
expert + FP8 quantisation of x, gate/up GEMM + SwiGLU + requant, down GEMM +
routing-weight scale, combine) over one batch of T synthetic tokens whose
inputs are resident in HBM.  L2 is flushed before every step (a 256 MiB write,
then a 256 MiB read, so that the step neither finds its inputs in L2 nor has to
write back the flush's dirty lines) and the step is timed with CUDA events on
the launching stream; the flush is outside the events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
                  [--format block128|mx|mxfp4]

--format mx runs the MXFP8 variant (1x32 UE8M0 scales on both operands,
block-scaled tensor-core MMA) on the same workload; --format mxfp4 the same
with MXFP4 weights (E2M1 codes, two per byte) and MXFP8 activations; the
default is the layer with 128x128 weight / 1x128 activation block scales.

Multi-GPU: one process per GPU (torchrun), each an independent replica of the
same workload (the layer has no exchange step on one GPU): weak scaling,
value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; % of HBM (decode) / FP8 TC peak (prefill)"
WEIGHTS = {"block128": "FP8 e4m3 128x128 block scales (x, h: 1x128), packed on device by moe_pack_weights",
           "mx": "MXFP8: e4m3 with 1x32 UE8M0 scales on weights, x and h, packed on device by moe_pack_weights_mx",
           "mxfp4": "MXFP4 weights (E2M1, two per byte, 1x32 UE8M0 scales; packed on device by "
                    "moe_pack_weights_mxfp4) x MXFP8 activations (x, h)"}
DEFAULT_CONFIG = "qwen235b_prefill"
FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]), bf16_sust=float(p["bf16_tflops_sustained"]),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


def workload_str(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top_k={cfg.top_k} seed={cfg.seed} "
            f"router_b={cfg.router_b} expert_bias={cfg.expert_bias}")


def algorithmic(cfg, counts: np.ndarray, mx: bool = False, fp4: bool = False) -> dict:
    """Algorithmic bytes / FLOPs (unpadded; activated experts only).  Scales:
    fp32 per 128x128 weight block and per 1x128 activation group, or (mx) one
    byte per 32 values of every weight row and activation row.  Weight codes:
    one byte each, or half a byte (fp4: MXFP4 weights)."""
    H, I, T, k, E = cfg.H, cfg.I, cfg.T, cfg.top_k, cfg.E
    R = T * k
    act = int((counts > 0).sum())
    hb, ib = -(-H // 128), -(-I // 128)
    if mx:
        hg, ig = -(-H // 32), -(-I // 32)
        cb = 0.5 if fp4 else 1.0  # bytes per weight code
        w13 = int(act * (cb * 2 * I * H + 2 * I * hg + 2 * 2 * I))
        w2 = int(act * (cb * H * I + H * ig + 2 * H))
        sxb, shb = R * hg, R * ig
    else:
        w13 = act * (2 * I * H + 4 * 2 * ib * hb + 2 * 2 * I)
        w2 = act * (H * I + 4 * hb * ib + 2 * H)
        sxb, shb = 4 * R * hb, 4 * R * ib
    gemm1_bytes = w13 + R * H + sxb + R * I + shb
    gemm2_bytes = w2 + R * I + shb + 4 * R * H
    step_bytes = w13 + w2 + E * H * 2 + E * 2 + T * H * 2 + T * H * 2
    return dict(active=act, gemm1_bytes=gemm1_bytes, gemm2_bytes=gemm2_bytes, step_bytes=step_bytes,
                gemm1_flops=2 * R * 2 * I * H, gemm2_flops=2 * R * H * I, router_flops=2 * T * E * H)


def source_digest(mx: bool = False, decode: bool | None = None) -> str:
    """Digest of a GEMM kernel's sources (ncu traffic is valid only for the source it
    was taken on): the file of the kernel (MX kernels; the 128x128 prefill or
    decode kernels; both 128x128 files when `decode` is None) and the shared headers."""
    h = hashlib.sha256()
    if mx:
        files = ("moe_gemm_mx.cu",)
    elif decode is None:
        files = ("moe_gemm.cu", "moe_gemm_decode.cu")
    else:
        files = ("moe_gemm_decode.cu",) if decode else ("moe_gemm.cu",)
    for f in files + ("moe_device.cuh", "moe_internal.h"):
        with open(os.path.join(ROOT, "sparse_moe_layer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, cfg_name: str, mx: bool = False, decode: bool | None = None):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)
        rec = t.get(f"{kernel}@{cfg_name}")
        if rec and rec.get("source_digest") == source_digest(mx, None if mx else decode):
            return int(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms in a child process."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.proc = None
        self.lines = []
        sel = [f"--id={gpu_uuid}"] if gpu_uuid else []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l.strip() for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=mx, reasons=sorted(reasons), samples=0)
        loaded = [s for s in sm if s > 0.5 * (mx or max(sm))] or sm
        return dict(sm_mhz=statistics.median(loaded), sm_max_mhz=mx, reasons=sorted(reasons), samples=len(sm))


def one_per_expert_inputs(cfg):
    """x and router of a batch that sends exactly one row to every expert
    (T = E / top_k): token t's logit is 1 for experts [t*k, t*k+k) and 0 else
    (x[t] = e_t, router_w[e] = e_{e//k}, router_b = 0), bf16 bits."""
    one = np.uint16(0x3F80)  # bf16 1.0
    x = np.zeros((cfg.T, cfg.H), np.uint16)
    x[np.arange(cfg.T), np.arange(cfg.T)] = one
    rw = np.zeros((cfg.E, cfg.H), np.uint16)
    rw[np.arange(cfg.E), np.arange(cfg.E) // cfg.top_k] = one
    return x, rw, np.zeros(cfg.E, np.uint16)


def build_layer(cfg, device, routing="synthetic", mx=False, fp4=False):
    """Inputs of the workload resident on the device; weights packed by the library
    (mx: MXFP8 codes and scale atoms; fp4: MXFP4 weight codes and scale atoms)."""
    import torch
    import sparse_moe_layer_gb300 as moe

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    if routing == "one_per_expert":
        x, rw, rb = one_per_expert_inputs(cfg)
    else:
        x = synth.layer_x(cfg)
        rw, rb = synth.router(cfg)
    b13, b2 = synth.expert_biases(cfg)
    E, H, I, Hp, Ip = cfg.E, cfg.H, cfg.I, cfg.Hp, cfg.Ip
    q13_shape, q2_shape = (moe.w13_shape_fp4, moe.w2_shape_fp4) if fp4 else (moe.w13_shape, moe.w2_shape)
    w13 = torch.empty(q13_shape(E, H, I), dtype=torch.uint8, device=device)
    w2 = torch.empty(q2_shape(E, H, I), dtype=torch.uint8, device=device)
    if mx or fp4:
        s13 = torch.empty(moe.s13_mx_shape(E, H, I), dtype=torch.uint8, device=device)
        s2 = torch.empty(moe.s2_mx_shape(E, H, I), dtype=torch.uint8, device=device)
    else:
        s13 = torch.empty((E, 2 * Ip // 128, Hp // 128), dtype=torch.float32, device=device)
        s2 = torch.empty((E, Hp // 128, Ip // 128), dtype=torch.float32, device=device)
    pack = moe.pack_weights_into_mxfp4 if fp4 else moe.pack_weights_into_mx if mx else moe.pack_weights_into
    chunk = 8
    for e0 in range(0, E, chunk):
        n = min(chunk, E - e0)
        m13 = torch.from_numpy(synth.w13_master(cfg, e0, n)).to(device)
        m2 = torch.from_numpy(synth.w2_master(cfg, e0, n)).to(device)
        pack(m13, m2, H, I, n, w13[e0:e0 + n], s13[e0:e0 + n], w2[e0:e0 + n], s2[e0:e0 + n])
        torch.cuda.synchronize()
        del m13, m2
    layer = moe.MoeLayer(bf16(rw), bf16(rb), w13, s13, bf16(b13), w2, s2, bf16(b2), cfg.top_k)
    return layer, bf16(x), x


def oracle_format(cfg, mx: bool, fp4: bool = False):
    """Empty oracle weight arrays of the format, its per-expert packer and its layer forward."""
    import oracle
    E, Hp, Ip = cfg.E, cfg.Hp, cfg.Ip
    if mx or fp4:
        arrs = (np.zeros((E, 2 * Ip, Hp), np.uint8), np.zeros((E, 2 * Ip, Hp // 32), np.uint8),
                np.zeros((E, Hp, Ip), np.uint8), np.zeros((E, Hp, Ip // 32), np.uint8))
        p13, p2, fwd = ((oracle.mx4_pack_w13, oracle.mx4_pack_w2, oracle.mx4_forward) if fp4 else
                        (oracle.mx_pack_w13, oracle.mx_pack_w2, oracle.mx_forward))
    else:
        arrs = (np.zeros((E, 2 * Ip, Hp), np.uint8), np.ones((E, 2 * Ip // 128, Hp // 128), np.float32),
                np.zeros((E, Hp, Ip), np.uint8), np.ones((E, Hp // 128, Ip // 128), np.float32))
        p13, p2, fwd = oracle.pack_w13, oracle.pack_w2, oracle.forward
    q13, s13, q2, s2 = arrs

    def pack(e):
        p13(synth.w13_master(cfg, int(e), 1), q13[e:e + 1], s13[e:e + 1])
        p2(synth.w2_master(cfg, int(e), 1), q2[e:e + 1], s2[e:e + 1])

    return arrs, pack, fwd


def sample_for_baseline(idx: np.ndarray, E: int, n: int, seed: int = 1234) -> tuple[np.ndarray, str]:
    """A bounded token sample of the batch for the CPU baseline: up to n/4 tokens
    of the least-loaded non-empty expert, up to n/4 of the most-loaded one, the
    rest a seeded random draw of the batch (n tokens in all, at most T).
    Returns (sorted token indices, description)."""
    T = idx.shape[0]
    n = int(min(T, max(1, n)))
    counts = np.bincount(idx.ravel(), minlength=E)
    nz = np.nonzero(counts)[0]
    most, least = int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])
    pick: list[int] = []
    seen = set()
    for e in (least, most):
        for t in np.nonzero((idx == e).any(axis=1))[0][:max(1, n // 4)]:
            if len(pick) < n and int(t) not in seen:
                pick.append(int(t))
                seen.add(int(t))
    for t in np.random.default_rng(seed).permutation(T):
        if len(pick) >= n:
            break
        if int(t) not in seen:
            pick.append(int(t))
            seen.add(int(t))
    desc = (f"{len(pick)} of {T} tokens: tokens of the least-loaded expert {least} ({counts[least]} rows) and of "
            f"the most-loaded expert {most} ({counts[most]} rows), the rest a seeded random draw")
    return np.array(sorted(pick), dtype=np.int32), desc


def cpu_oracle_leg(cfg, seconds: float, mx: bool = False, fp4: bool = False):
    """Time the oracle (single thread) on a bounded sample of the workload:
    about `seconds` of CPU work -- a token sample that includes tokens of the
    most- and least-loaded experts (sample_for_baseline; the whole batch when it
    fits the budget), the full layer per token, repeated if one pass is short.
    The oracle's routing of the batch (to find those experts) and its weight
    packing are untimed.  Returns (tokens per second, sample description, seconds)."""
    import oracle
    x = synth.layer_x(cfg)
    rw, rb = synth.router(cfg)
    b13, b2 = synth.expert_biases(cfg)
    k = cfg.top_k
    (q13, s13, q2, s2), pack, fwd = oracle_format(cfg, mx, fp4)
    packed = set()
    from concurrent.futures import ThreadPoolExecutor
    nthreads = max(1, min(16, os.cpu_count() or 1))

    def route(rows):
        return oracle.router(np.ascontiguousarray(x[rows]), rw, rb, k)["idx"]

    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        idx = np.concatenate(list(ex.map(route, [c for c in np.array_split(np.arange(cfg.T), 4 * nthreads)
                                                 if len(c)])))

    def pack_for(tokens):  # weight conversion is offline for both sides: untimed
        todo = [int(e) for e in np.unique(idx[tokens]) if int(e) not in packed]
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(pack, todo))
        packed.update(todo)

    # calibrate on a few tokens, then size the sample to the time budget
    probe = np.arange(min(2, cfg.T), dtype=np.int32)
    pack_for(probe)
    t0 = time.perf_counter()
    fwd(x, rw, rb, q13, s13, b13, q2, s2, b2, k, tokens=probe)
    per_token = max((time.perf_counter() - t0) / len(probe), 1e-6)
    tokens, sdesc = sample_for_baseline(idx, cfg.E, int(seconds / per_token))
    n = len(tokens)
    passes = max(1, int(seconds / (n * per_token)))
    pack_for(tokens)
    t0 = time.perf_counter()
    for _ in range(passes):
        fwd(x, rw, rb, q13, s13, b13, q2, s2, b2, k, tokens=tokens)
    dt = time.perf_counter() - t0
    desc = (f"{sdesc}; x {passes} pass(es) ({len(packed)} experts packed), full layer per token, "
            f"single-threaded fp64 oracle" + (" (MXFP4-weight variant)" if fp4 else " (MXFP8 variant)" if mx else ""))
    return passes * n / dt, desc, dt


def flush_l2(wbuf, rbuf, i: int) -> None:
    """Leave L2 cold and clean before a timed step: writing `wbuf` (larger than
    L2) evicts whatever the previous step left there, and reading `rbuf` (also
    larger than L2) then evicts the dirty lines of that write, so their
    write-back happens here instead of inside the step's first kernels."""
    wbuf.fill_(i & 0xFF)
    rbuf.sum()


def max_over_ranks(ms: float, pg, device) -> float:
    """The slowest rank's time (every rank receives it); the value itself on one rank."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, T: int, ms: float) -> float:
    """Whole-job throughput: every rank's T tokens over the slowest rank's step time."""
    return world * T / (ms * 1e-3)


def run_reference(args, cfg, rank):
    """The oracle as the reference arm: K steps, each a bounded sample (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    x = synth.layer_x(cfg)
    rw, rb = synth.router(cfg)
    b13, b2 = synth.expert_biases(cfg)
    k = cfg.top_k
    rng = np.random.default_rng(99)
    tokens_all = rng.permutation(cfg.T).astype(np.int32)
    r = oracle.router(np.ascontiguousarray(x[tokens_all]), rw, rb, k)
    mx, fp4 = args.format == "mx", args.format == "mxfp4"
    (q13, s13, q2, s2), pack, fwd = oracle_format(cfg, mx, fp4)
    from concurrent.futures import ThreadPoolExecutor
    needed = np.unique(r["idx"])
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(pack, needed))
    # one token per step, cycling through a seeded permutation of the batch
    def step(i):
        t = tokens_all[i % len(tokens_all)]
        fwd(x, rw, rb, q13, s13, b13, q2, s2, b2, k, tokens=np.array([t], np.int32))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = dict(metric=METRIC, value=value, unit="tokens/s", n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                ms_per_step=dt * 1e3 / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=workload_str(cfg), step="one token of the batch through the whole layer",
                            weights=WEIGHTS[args.format]),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=1, kind="oracle",
                                  sample=f"{args.steps} tokens, one per step, single-threaded fp64 C oracle"),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=[c.name for c in synth.CONFIGS])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--format", default="block128", choices=["block128", "mx", "mxfp4"],
                    help="mx: the MXFP8 variant (moe_forward_mx); mxfp4: MXFP4 weights (moe_forward_mxfp4)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work in the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="batch size T instead of the workload's (small-batch decode sweep; same weights)")
    ap.add_argument("--routing", default="synthetic", choices=["synthetic", "one_per_expert"],
                    help="one_per_expert: T = E/top_k tokens routed so that every expert gets exactly one row")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = synth.config(args.config)
    if args.routing == "one_per_expert":
        if cfg.E % cfg.top_k or cfg.E // cfg.top_k > cfg.H:
            ap.error("one_per_expert needs top_k | E and E/top_k <= H")
        cfg = dataclasses.replace(cfg, T=cfg.E // cfg.top_k)
    elif args.tokens:
        cfg = dataclasses.replace(cfg, T=args.tokens)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    import sparse_moe_layer_gb300 as moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    fp4 = args.format == "mxfp4"
    mx = args.format == "mx" or fp4
    layer, x_dev, x_host_np = build_layer(cfg, dev, args.routing, mx, fp4)
    T, H = cfg.T, cfg.H
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush_l2(flush, flush_rd, 1)
        layer(x_dev, out=out)
    torch.cuda.synchronize()
    ws = layer.workspace(T)
    assert moe.read_device_status(ws) == 0, "device wait timed out during warm-up"
    counts = moe.workspace_views(ws, T, cfg.H, cfg.I, cfg.E, cfg.top_k, mx=mx)["count"].cpu().numpy()
    alg = algorithmic(cfg, counts, mx, fp4)

    K = args.steps
    # Timed region 1 (the value): the step replayed as a CUDA graph (one memset
    # node + five kernels with programmatic dependencies), events around each replay.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.forward(x_dev, layer.router_w, layer.router_b, layer.w13, layer.s13, layer.b13, layer.w2, layer.s2,
                    layer.b2, cfg.top_k, out=out, workspace=ws)
    for _ in range(args.warmup):
        flush_l2(flush, flush_rd, 1)
        graph.replay()
    torch.cuda.synchronize()
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    time.sleep(0.25)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2(flush, flush_rd, i)
        ev_s[i].record(stream)
        graph.replay()
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if pg:
        pg.barrier()
    step_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(K)]
    # the median step (robust to a stray slow replay); the mean is reported beside it
    ms = max_over_ranks(statistics.median(step_ms), pg, dev)
    ms_mean = max_over_ranks(statistics.fmean(step_ms), pg, dev)
    # Timed region 2 (per-kernel time): the same K steps launched directly with
    # moe_forward_profiled, whose events are recorded on the launching stream
    # between the five kernels.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for row in ev:  # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2(flush, flush_rd, i)
        # a ~0.1 ms spin kernel lets the host enqueue the whole step before its
        # first event, so no stage time contains host launch latency
        torch.cuda._sleep(200_000)
        moe.forward(x_dev, layer.router_w, layer.router_b, layer.w13, layer.s13, layer.b13, layer.w2, layer.s2,
                    layer.b2, cfg.top_k, out=out, workspace=ws, events=ev[i])
    torch.cuda.synchronize()
    sampler.stop()
    status = moe.read_device_status(ws)
    stage_ms = {s: statistics.median(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K))
                for j, s in enumerate(moe.STAGES)}
    eager_ms = statistics.median(ev[i][0].elapsed_time(ev[i][5]) for i in range(K))

    # end to end through the public API with host buffers: H2D of x into the
    # graphed layer's input, the layer (one graph launch), D2H of its output
    x_host = torch.from_numpy(np.ascontiguousarray(x_host_np).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    glayer = layer.graphed(T)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(min(args.warmup, 5)):
        glayer.x.copy_(x_host, non_blocking=True)
        out_host.copy_(glayer(), non_blocking=True)
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2(flush, flush_rd, i)
        e2e_ev[i][0].record(stream)
        glayer.x.copy_(x_host, non_blocking=True)
        out_host.copy_(glayer(), non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in e2e_ev), pg, dev)
    out = glayer.out
    assert torch.equal(out_host.view(torch.int16), out.cpu().view(torch.int16))

    pk = peaks()
    # the library runs the swap-AB decode GEMMs (weight streaming, HBM-bound) when the
    # batch has at most 64 rows per expert on average, else the 128x256-tile prefill GEMMs
    prefill = T * cfg.top_k > 64 * cfg.E
    g1_s = stage_ms["gemm_gateup"] * 1e-3
    if prefill:
        # FP8 dense = 2 x bf16 dense (nominal ratio); the GEMM is timed inside back-to-back
        # layer steps, so against the sustained (power-capped) bf16 figure
        fp8_peak = 2.0 * pk["bf16_sust"]
        roof = dict(bound="tensor", achieved=alg["gemm1_flops"] / g1_s / 1e12, peak=fp8_peak, unit="TFLOP/s")
    else:
        roof = dict(bound="hbm", achieved=alg["gemm1_bytes"] / g1_s / 1e9, peak=pk["hbm"], unit="GB/s")
    roof["frac"] = roof["achieved"] / roof["peak"]
    # a record holds for the named workload itself, not for a --tokens / --routing variant of it
    own_workload = args.tokens == 0 and args.routing == "synthetic"
    roof["traffic"] = (recorded_traffic("gemm_gateup_mx4" if fp4 else "gemm_gateup_mx" if mx else "gemm_gateup",
                                        cfg.name, mx, decode=not prefill) if own_workload else None)
    if fp4:
        roof["kernel"] = ("moe_gemm_mx_kernel<true, FP4W> (block-scaled e4m3 x e2m1 gate/up GEMM + SwiGLU + MX "
                          "requant)" if prefill else
                          "moe_gemm_mx_decode_kernel<true, FP4W> (swap-AB block-scaled e2m1 x e4m3 gate/up GEMM + "
                          "SwiGLU + MX requant)")
    elif mx:
        roof["kernel"] = ("moe_gemm_mx_kernel<true> (block-scaled gate/up GEMM + SwiGLU + MX requant)" if prefill else
                          "moe_gemm_mx_decode_kernel<true> (swap-AB block-scaled gate/up GEMM + SwiGLU + MX requant)")
    else:
        roof["kernel"] = ("moe_gemm_kernel<true> (gate/up GEMM + SwiGLU + requant)" if prefill else
                          "moe_gemm_decode_kernel<true> (swap-AB gate/up GEMM + SwiGLU + requant)")
    roof["peak_source"] = pk["source"] + (" (hbm_gbs)" if not prefill else " (2 x bf16_tflops_sustained)")
    roof["algorithmic_per_launch"] = alg["gemm1_bytes"] if not prefill else alg["gemm1_flops"]

    value = job_tokens_per_s(world, T, ms)
    line = dict(metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=K, warmup=args.warmup,
                ms_per_step=ms, ms_per_step_mean=ms_mean, timing="median of the K timed steps (mean beside it)",
                higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="e2m1 x e4m3" if fp4 else "e4m3",
                data="synthetic",
                config=dict(workload=workload_str(cfg) + ("" if args.routing == "synthetic" else
                                                          " routing=one row per expert (T = E/top_k)"),
                            parallelism=f"replicas{world}",
                            l2="flushed before every step (256 MiB write, then 256 MiB read so no dirty line is left; "
                               "outside the timed events)",
                            weights=WEIGHTS[args.format]),
                roofline=roof,
                step=dict(ms_per_stage=stage_ms, active_experts=alg["active"],
                          gemm_down_achieved=(alg["gemm2_flops"] / (stage_ms["gemm_down"] * 1e-3) / 1e12 if prefill
                                              else alg["gemm2_bytes"] / (stage_ms["gemm_down"] * 1e-3) / 1e9),
                          step_GBps=alg["step_bytes"] / (ms * 1e-3) / 1e9,
                          step_hbm_frac=alg["step_bytes"] / (ms * 1e-3) / 1e9 / pk["hbm"],
                          gemm_tflops=(alg["gemm1_flops"] + alg["gemm2_flops"]) / (ms * 1e-3) / 1e12,
                          wall_s=wall, device_status=status,
                          launch="CUDA graph replay of " + ("moe_forward_mxfp4" if fp4 else "moe_forward_mx" if mx
                                                            else "moe_forward"),
                          eager_ms_per_step=eager_ms),
                e2e=dict(value=job_tokens_per_s(world, T, e2e_ms), unit="tokens/s", h2d_bytes_per_step=T * H * 2,
                         d2h_bytes_per_step=T * H * 2, ms_per_step=e2e_ms,
                         api="MoeLayer.graphed(T): x copied in from pinned host memory, one graph replay, "
                             "out copied back"),
                gpu_launches=5 * K,
                clocks=sampler.summary())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, dt = cpu_oracle_leg(cfg, args.cpu_seconds, mx, fp4)
        line["cpu_baseline"] = dict(value=v, unit="tokens/s", cores=1, kind="oracle", sample=desc, seconds=dt)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
