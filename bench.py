#!/usr/bin/env python3
"""Throughput of the routed FP8 MoE FFN layer forward (Kimi K2 shapes) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload all|decode|prefill|skewed|skewed40|dense] [--impl ours|reference]

One step = one forward of the whole layer over one batch of T tokens already
resident in HBM: router GEMM + top-k, x quantisation, permutation, grouped
gate/up and down FP8 GEMMs, combine. The headline workload is the decode batch
(T=256, d=7168, 384 routed experts top-8 + 1 shared, expert hidden 2048). By
default (--workload all) the same run then measures the prefill batch (T=4096),
the two skewed batches (T=16384) and the dense FFN of the first block
(T=8192, H=18432) and reports each under "workloads". Under torchrun each rank
runs an independent replica on its own batch (weak scaling; no collective on
the data path).

Prints one JSON line (rank 0). Besides the throughput each workload reports the
roofline of its dominant kernel (the gate/up grouped GEMM, timed with CUDA
events inside the timed region; the whole FFN for the dense workload) against
the measured and the nominal peaks, the end-to-end throughput through the
one-call API with pinned host buffers, the CPU oracle timed on a token sample,
and the SM clocks sampled during its timed region.
"""
from __future__ import annotations

import os

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import moe_synth as S  # noqa: E402

METRIC = "MoE-layer tokens/s (d7168, 384e top-8, FP8) + % of HBM / FP8-TC roofline"
# decode_e64: the decode layer with 64 routed experts and 48 tokens (about 6 rows per
# expert, as at T=256 with 384 experts; 2.9 GB of weights): a profiling case of a few GB
DECODE_E64 = S.MoEShape("kimi_k2_moe_decode_e64_t48", T=48, d=7168, E=64, topk=8, H=2048)
# prefill_e64: 64 routed experts and 768 tokens (96 rows per expert, the 128-token
# tile path of the prefill batch; 2.9 GB of weights)
PREFILL_E64 = S.MoEShape("kimi_k2_moe_prefill_e64_t768", T=768, d=7168, E=64, topk=8, H=2048)
WORKLOADS = {"decode": S.DECODE, "prefill": S.PREFILL, "skewed": S.SKEWED, "skewed40": S.SKEWED40,
             "dense": S.DENSE, "toy": S.TOY,
             "decode_e64": DECODE_E64, "prefill_e64": PREFILL_E64}
DATA = ("synthetic, seeded: x ~ N(0,1) bf16; W_g ~ N(0,0.02) bf16; bias ~ N(0,0.01) fp32 (+0.5 on 16 hot "
        "experts for the skewed workload, +0.18 for skewed40); expert weights ~ N(0,0.02) stored e4m3 with "
        "128x128 fp32 scales")

# DRAM bytes (read + write) per launch of the decode gate/up kernel, from one ncu
# capture of the same kernel on the decode-like case of a few GB (decode_e64:
# 1.9183 GB of traffic for 1.9092 GB of algorithmic and 4.1 MB of implementation
# bytes). Traffic grows with the touched experts' weights, so the full launch's
# figure is this ratio times its algorithmic plus implementation bytes. Keyed by the
# hash of the kernel sources at capture time: once the sources change, the figure no
# longer applies (null).
NCU_TRAFFIC = {"ratio": 1.0026, "src": "5081a4644fcb33b5", "case": "decode_e64"}
# The same for the token-major gate/up kernel in the one-tile-per-expert regime of
# the prefill batch (prefill_e64: 96 rows per routed expert, so one 128-token tile;
# 1.9723 GB of traffic for 1.9146 GB of algorithmic and 65.7 MB of implementation
# bytes), applied to workloads without hot experts and with at most 128 rows per
# routed expert.
NCU_TRAFFIC_WIDE = {"ratio": 0.9960, "src": "5081a4644fcb33b5", "case": "prefill_e64"}


def kernel_src_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "routed_fp8_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def expert_bn_is_decode(shape) -> bool:
    """The decode regime (fused gate/up kernel, 32-token tiles) that the capture covers."""
    return shape.topk * shape.T / shape.E <= 12.0


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def init_group(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

_CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                 "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                 "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            except Exception:
                pass
            cmd = ["nvidia-smi", "--query-gpu=" + ",".join(_CLOCK_FIELDS), "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.5)   # first sample lands before the timed region starts
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(_CLOCK_FIELDS):
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                n += 1
                for name, v in zip(names, parts[3:]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ------------------------------------------------------------------ CPU oracle timing

def oracle_tokens_per_s(x_rows, wg, bias, experts_host, shape, n_rep=1):
    """Times the CPU oracle's layer forward on the given token rows; tokens/s."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    for _ in range(n_rep):
        O.moe_layer(x_rows, wg, bias, experts_host, shape.topk, shape.route_scale, n_shared=shape.n_shared)
    dt = time.perf_counter() - t0
    return x_rows.shape[0] * n_rep / dt, dt


def experts_for(idx_rows, shape):
    return sorted(set(np.asarray(idx_rows).ravel().tolist()) | {shape.E + s for s in range(shape.n_shared)})


def host_experts_from_device(ex_dev, need, shape):
    host = S.ExpertWeights(*(torch.zeros((shape.E + shape.n_shared,) + t.shape[1:], dtype=t.dtype)
                             for t in (ex_dev.w13, ex_dev.w13_s, ex_dev.w2, ex_dev.w2_s)))
    for e in need:
        host.w13[e].copy_(ex_dev.w13[e].cpu())
        host.w13_s[e].copy_(ex_dev.w13_s[e].cpu())
        host.w2[e].copy_(ex_dev.w2[e].cpu())
        host.w2_s[e].copy_(ex_dev.w2_s[e].cpu())
    return host


def sample_tokens(T, n, seed=0):
    return np.sort(np.random.default_rng(seed).choice(T, size=min(n, T), replace=False))


# ------------------------------------------------------------------ reference arm

def run_reference(args, shape):
    """The CPU oracle as the reference implementation, on bounded token samples."""
    from oracle import moe_oracle as O
    rank, _, world = dist_env()
    if rank != 0:
        return None
    n_tok = args.ref_tokens
    dense = isinstance(shape, S.DenseShape)
    if dense:
        x = S.gen_x(shape.T, shape.d, seed=args.seed, name="x_dense")
        toks = sample_tokens(shape.T, n_tok, seed=args.seed)
        w13, w13_s, w2, w2_s = S.gen_expert(0, shape.d, shape.H, seed=args.seed, name="dense")

        def step():
            O.dense_swiglu(x[toks], w13, w13_s, w2, w2_s)
        sample_desc = f"{len(toks)} of {shape.T} tokens per step through the dense FFN (fp64 oracle)"
    else:
        x = S.gen_x(shape.T, shape.d, seed=args.seed)
        wg, b = S.gen_router(shape, seed=args.seed)
        toks = sample_tokens(shape.T, n_tok, seed=args.seed)
        r = O.route(x[toks].float().numpy(), wg.float().numpy(), b.double().numpy(), shape.topk, shape.route_scale)
        ex = S.gen_experts(shape.E + shape.n_shared, shape.d, shape.H, seed=args.seed,
                           only=experts_for(r["idx"], shape))

        def step():
            O.moe_layer(x[toks], wg, b, ex, shape.topk, shape.route_scale, n_shared=shape.n_shared)
        sample_desc = (f"{len(toks)} of {shape.T} tokens per step (routing, permutation, quantisation and the "
                       f"experts those tokens use; fp64 oracle)")
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    tps = len(toks) * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": workload_config(shape),
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": _CORES, "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def workload_config(shape) -> dict:
    if isinstance(shape, S.DenseShape):
        return {"workload": shape.name, "T": shape.T, "d": shape.d, "H": shape.H,
                "l2": "inputs larger than L2 (0.40 GB of FP8 weights + 59 MB of activations per step)"}
    cfg = {"workload": shape.name, "T": shape.T, "d": shape.d, "E": shape.E, "topk": shape.topk, "H": shape.H,
           "n_shared": shape.n_shared, "route_scale": shape.route_scale,
           "weight_layout": "tiled 128x128 (moe_pack_weights_fp8, once before timing)",
           "l2": f"inputs larger than L2 ({(shape.E + shape.n_shared) * 3 * shape.d * shape.H / 1e9:.2f} GB of "
                 f"FP8 expert weights per step)"}
    if shape.hot_experts:
        cfg["hot_experts"] = len(shape.hot_experts)
        cfg["hot_bias"] = shape.hot_bias
    return cfg


# ------------------------------------------------------------------ rooflines

NOMINAL_HBM_GBS = 8000.0       # GB300 HBM3e, vendor figure (about 8 TB/s)
NOMINAL_FP8_TFLOPS = 4500.0    # GB300 dense FP8 tensor, vendor figure


def roofline(kernel, alg_bytes, alg_flops, ms, peaks, traffic=None, impl_bytes=None):
    """The launch's binding roofline: whichever of its algorithmic HBM bytes and its
    FP8 FLOPs takes longer at the measured peak. Fractions against the measured
    peak (frac; for FP8 2 x the measured bf16 burst, and frac_sustained against 2 x
    the sustained figure) and against the vendor's nominal figure (frac_nominal)."""
    fp8_peak = 2 * peaks["bf16_tflops"]
    tensor = alg_flops / (fp8_peak * 1e12) > alg_bytes / (peaks["hbm_gbs"] * 1e9)
    out = {"kernel": kernel, "alg_bytes_per_launch": alg_bytes, "alg_flops_per_launch": alg_flops, "launch_ms": ms}
    if impl_bytes is not None:
        out["impl_bytes_per_launch"] = impl_bytes
    if tensor:
        a = alg_flops / (ms * 1e-3) / 1e12
        out.update({"bound": "tensor", "achieved": a, "peak": fp8_peak, "unit": "TFLOP/s", "frac": a / fp8_peak,
                    "frac_sustained": a / (2 * peaks["bf16_tflops_sustained"]), "frac_nominal": a / NOMINAL_FP8_TFLOPS,
                    "traffic": traffic,
                    "peak_source": peaks["source"] + " bf16 burst x 2 (nominal fp8/bf16 ratio); frac_nominal against "
                                   f"{NOMINAL_FP8_TFLOPS:.0f} TFLOP/s"})
    else:
        a = alg_bytes / (ms * 1e-3) / 1e9
        out.update({"bound": "hbm", "achieved": a, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": a / peaks["hbm_gbs"], "frac_nominal": a / NOMINAL_HBM_GBS, "traffic": traffic,
                    "peak_source": peaks["source"] + " hbm_gbs copy bandwidth; frac_nominal against "
                                   f"{NOMINAL_HBM_GBS:.0f} GB/s"})
    return out


# ------------------------------------------------------------------ our arm

def pipelined_e2e(dev, steps, warmup, x_src, out_shape, call, world):
    """End to end through the public API with each step's input copied in from pinned
    host memory and its output copied out, as a serving loop runs it: the copies go on
    two streams of their own (host to device, device to host) and double buffers let
    step i's input copy run during step i-1's compute and its output copy during step
    i+1's. Events order every copy after the compute that frees or fills its buffer.
    Returns (ms for `steps` steps, the last output on the device)."""
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    x_host = [x_src.cpu().pin_memory() for _ in range(2)]
    y_host = [torch.empty(out_shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x_src) for _ in range(2)]
    yd = [torch.empty(out_shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            s = i % 2
            h2d.wait_event(comp_done[s])        # step i-2's compute is done with xd[s]
            with torch.cuda.stream(h2d):
                xd[s].copy_(x_host[s], non_blocking=True)
            in_ready[s].record(h2d)
            comp.wait_event(in_ready[s])
            comp.wait_event(out_done[s])        # step i-2's output copy is done with yd[s]
            call(xd[s], yd[s])
            comp_done[s].record(comp)
            d2h.wait_event(comp_done[s])
            with torch.cuda.stream(d2h):
                y_host[s].copy_(yd[s], non_blocking=True)
            out_done[s].record(d2h)
        return (n - 1) % 2

    run(max(1, warmup))
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_event(e0)
    last = run(steps)
    comp.wait_event(out_done[0])
    comp.wait_event(out_done[1])
    e1.record(comp)
    torch.cuda.synchronize(dev)
    barrier(world)
    return e0.elapsed_time(e1), yd[last]


def cpu_baseline_moe(shape, x, wg, b, ex, idx, n_tokens, seed):
    """The fp64 oracle on a bounded token sample of the workload (host cores)."""
    toks = sample_tokens(shape.T, n_tokens, seed=seed)
    host = host_experts_from_device(ex, experts_for(idx.cpu().numpy()[toks], shape), shape)
    tps, dt = oracle_tokens_per_s(x.cpu()[toks], wg.cpu(), b.cpu(), host, shape)
    return {"value": tps, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{len(toks)} of {shape.T} tokens through the fp64 oracle ({dt:.1f} s)"}


def run_moe(args, shape, rank, local, world, dev, peaks, ex=None, ext=None):
    """ex: the expert weights (row-major; the CPU baseline decodes them); ext: the
    same weights in the tiled layout, which every GPU call of the step reads."""
    import routed_fp8_expert_gb300 as moe
    cfg = moe.cfg_of(shape, w_tiled=True)
    T, d, H, k, E, Sh = shape.T, shape.d, shape.H, shape.topk, shape.E, shape.n_shared
    R = (k + Sh) * T
    if ex is None:
        ex = S.gen_experts(E + Sh, d, H, seed=args.seed, device=dev)
    if ext is None:
        # the one-time weight preparation, before any timing
        ext = S.ExpertWeights(moe.pack_weights_fp8(ex.w13), ex.w13_s, moe.pack_weights_fp8(ex.w2), ex.w2_s)
        torch.cuda.synchronize(dev)
    x = S.gen_x(T, d, seed=args.seed + rank, device=dev)
    wg, b = S.gen_router(shape, seed=args.seed, device=dev)
    ws = moe.workspace(cfg, T, dev)
    # persistent buffers of the step
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_tok = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv_pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    xq_perm = torch.empty((R, d), dtype=torch.uint8, device=dev)
    sx_perm = torch.empty((d // 128, R), dtype=torch.float32, device=dev)
    hq = torch.empty((R, H), dtype=torch.uint8, device=dev)
    hs = torch.empty((H // 128, R), dtype=torch.float32, device=dev)
    o = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    L = moe.load()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    cref = ctypes.byref(cfg)
    nws = ws.numel()

    def call(rc):
        if rc != 0:
            raise RuntimeError(L.moe_last_error_string().decode())
        return L.moe_last_launch_count()

    names = ["route", "quant_permute", "gateup", "down", "combine"]

    def step(ev=None, marks=range(6)):
        """One layer forward through the split calls; ev[j] is recorded at mark j
        (before the calls, then after each one) for the marks listed."""
        n = 0

        def mark(j):
            if ev is not None and j in marks:
                ev[j].record()
        mark(0)
        n += call(L.moe_route(P(x), P(wg), P(b), cref, T, P(idx), P(w), None, P(ws), nws, st))
        mark(1)
        n += call(L.moe_quant_permute_fp8(P(idx), P(x), cref, T, P(offsets), P(sorted_tok), P(inv_pos),
                                          P(xq_perm), P(sx_perm), P(ws), nws, st))
        mark(2)
        n += call(L.moe_expert_gateup_fp8(P(xq_perm), P(sx_perm), P(offsets), P(ext.w13), P(ext.w13_s), cref, T,
                                          P(hq), P(hs), P(ws), nws, st))
        mark(3)
        n += call(L.moe_expert_down_fp8(P(hq), P(hs), P(offsets), P(ext.w2), P(ext.w2_s), cref, T, P(o), P(ws), nws,
                                        st))
        mark(4)
        n += call(L.moe_combine(P(o), P(w), P(inv_pos), cref, T, P(y), st))
        mark(5)
        return n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    moe.check_device_error(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index or 0)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    launches = 0
    # the timed steps carry events around the gate/up call only (the roofline kernel):
    # an event between two calls keeps the second call's kernels from launching
    # during the first's tail, which cost ~20 us per decode step with all five marked
    t0.record()
    for i in range(args.steps):
        launches += step(evs[i], marks=(2, 3))
    t1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    moe.check_device_error(dev)
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    gu_ms_live = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    # every call's time from a pass of its own after the timed steps, all marks set
    n_per = min(args.steps, 20)
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n_per)]
    for i in range(n_per):
        step(evp[i])
    torch.cuda.synchronize(dev)
    per = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evp) for j, n in enumerate(names)}

    # routing statistics of the last step
    counts = torch.diff(offsets).cpu().numpy()
    touched = int((counts > 0).sum()) + Sh
    # one gate/up launch: algorithmic bytes are the touched experts' gate+up weights
    # and scales and the step's activation codes read once; the permuted copies read
    # and the h codes written are the implementation's own traffic, kept apart
    gu_bytes = touched * (2 * H * d + 2 * (H // 128) * (d // 128) * 4) + T * (d + (d // 128) * 4)
    gu_impl = R * d + R * (d // 128) * 4 + R * H + R * (H // 128) * 4
    gu_ms = gu_ms_live
    gu_flops = 4 * R * H * d
    traffic_val = None
    if NCU_TRAFFIC and NCU_TRAFFIC.get("src") == kernel_src_hash() and expert_bn_is_decode(shape):
        traffic_val = NCU_TRAFFIC["ratio"] * (gu_bytes + gu_impl)
    elif (NCU_TRAFFIC_WIDE and NCU_TRAFFIC_WIDE.get("src") == kernel_src_hash() and not shape.hot_experts
          and shape.topk * shape.T / shape.E <= 128):
        traffic_val = NCU_TRAFFIC_WIDE["ratio"] * (gu_bytes + gu_impl)
    gu_kernel = ("grouped_gemm_kernel<GateUp, 32>" if expert_bn_is_decode(shape) else
                 "grouped_gemm_wide_kernel<GateUpWide, 128>")
    layer_weight_bytes = touched * (3 * H * d + 3 * (H // 128) * (d // 128) * 4) + E * d * 2
    flops = T * (2 * E * d) + (T * k + T * Sh) * 6 * d * H
    ms_step = ms_total / args.steps
    tokens_total = sum_over_ranks(T * args.steps, world, dev)
    value = tokens_total / (ms_total * 1e-3)

    # end to end through the one-call API, each step's x copied in from pinned host
    # memory and its y copied out, overlapped with the neighbouring steps' compute
    e2e_ms, yd = pipelined_e2e(dev, args.steps, args.warmup, x, (T, d),
                               lambda xi, yo: moe.layer_forward(xi, wg, b, ext, cfg, ws=ws, y=yo), world)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = tokens_total / (e2e_ms * 1e-3)
    same = torch.equal(yd, y)
    pieces = time_block_pieces(L, x, o, w, inv_pos, cfg, shape, dev, st, peaks)
    pieces["moe_block_ffn_forward"] = time_block_call(moe, x, wg, b, ext, cfg, ws, dev, n=max(3, min(args.steps, 20)))
    step_bytes = layer_weight_bytes + 2 * T * d * 2

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": DATA, "config": workload_config(shape),
        "roofline": roofline(gu_kernel, gu_bytes, gu_flops, gu_ms, peaks, traffic_val, gu_impl),
        "layer": {"alg_weight_bytes": layer_weight_bytes, "alg_bytes_whole_step": step_bytes,
                  "hbm_frac_whole_step": step_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "hbm_frac_nominal_whole_step": step_bytes / (ms_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                  "tflops": flops / (ms_step * 1e-3) / 1e12, "fp8_peak_tflops": 2 * peaks["bf16_tflops"],
                  "fp8_frac_whole_step": flops / (ms_step * 1e-3) / 1e12 / (2 * peaks["bf16_tflops"]),
                  "touched_experts": touched, "max_rows_per_expert": int(counts.max()),
                  **({"hot_share": float(counts[list(shape.hot_experts)].sum() / counts[:E].sum())}
                     if shape.hot_experts else {}),
                  "kernels_ms": per,
                  "kernels_ms_pass": f"{n_per} steps after the timed ones, an event between every two calls; the "
                                     f"roofline's gate/up time comes from the timed steps themselves"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * d * 2, "api": "moe_layer_forward", "matches_step_output": bool(same),
                "copies": "pinned host buffers; copy-in and copy-out streams overlapped with the neighbouring "
                          "steps' compute (double buffers)"},
        "gpu_launches": launches,
        "clocks": clk,
        "block_pieces": pieces,
    }
    return line, (x, wg, b, ex, idx, ext)


def time_block_pieces(L, x, o, w, inv_pos, cfg, shape, dev, st, peaks, n=50):
    """The block's kernels next to the layer, timed apart from the step with CUDA
    events on the step's own tensors (x as the residual stream, o and the routing of
    the last step): RMSNorm + quantise of the layer input, and the combine fused with
    the residual addition and the next block's RMSNorm. HBM-bound: algorithmic bytes
    (reads + writes) over the time, against the measured copy bandwidth."""
    import ctypes
    T, d, k, Sh = shape.T, shape.d, shape.topk, shape.n_shared
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    gamma = S.gen_norm_weight(d, seed=0, device=dev)
    xb = torch.empty_like(x)
    xq = torch.empty((T, d), dtype=torch.uint8, device=dev)
    sx = torch.empty((T, d // 128), dtype=torch.float32, device=dev)
    h_out = torch.empty_like(x)
    x_next = torch.empty_like(x)
    eps = ctypes.c_float(1e-6)
    calls = {
        "rmsnorm_quant_kernel": (lambda: L.moe_rmsnorm_quant_fp8(P(x), P(gamma), eps, T, d, P(xb), P(xq), P(sx), 0, st),
                                 T * d * 2 + d * 2 + T * d * 2 + T * d + T * (d // 128) * 4),
        "combine_residual_rmsnorm_kernel": (
            lambda: L.moe_combine_residual_rmsnorm(P(o), P(w), P(inv_pos), ctypes.byref(cfg), T, P(x), P(gamma), eps,
                                                   P(h_out), P(x_next), st),
            (k + Sh) * T * d * 2 + T * k * 8 + T * d * 2 + d * 2 + 2 * T * d * 2),
    }
    out = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            if fn() != 0:
                raise RuntimeError(L.moe_last_error_string().decode())
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / n
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "alg_bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"]}
    return out


def time_block_call(moe, x, wg, b, ex, cfg, ws, dev, n=20):
    """The FFN half of the block in one call (RMSNorm_post with the fused
    quantisation, the layer, residual addition and RMSNorm_next) against the
    one-call layer on the same inputs (x as the residual stream), and the one-call
    layer captured in a CUDA graph and replayed: CUDA events, n calls each after
    three warm-up calls."""
    g_post = S.gen_norm_weight(x.shape[1], seed=1, name="norm_post", device=dev)
    g_next = S.gen_norm_weight(x.shape[1], seed=1, name="norm_next", device=dev)
    h_out = torch.empty_like(x)
    x_next = torch.empty_like(x)
    y = torch.empty_like(x)
    calls = {"block_ms": lambda: moe.block_ffn_forward(x, g_post, wg, b, ex, cfg, gamma_next=g_next, ws=ws,
                                                        h_out=h_out, x_next=x_next),
             "layer_ms": lambda: moe.layer_forward(x, wg, b, ex, cfg, ws=ws, y=y)}
    out = {}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        out[name] = e0.elapsed_time(e1) / n
    out["extra_ms"] = out["block_ms"] - out["layer_ms"]
    # the one-call layer captured once in a CUDA graph and replayed (same inputs)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        calls["layer_ms"]()
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls["layer_ms"]()
    for _ in range(3):
        graph.replay()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    out["layer_graph_ms"] = e0.elapsed_time(e1) / n
    return out


def run_dense(args, shape, rank, world, dev, peaks, want_cpu=False):
    import routed_fp8_expert_gb300 as moe
    T, d, H = shape.T, shape.d, shape.H
    inp = S.gen_dense_inputs(shape, seed=args.seed, device=dev)
    ws = moe.dense_workspace(d, H, T, dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        moe.dense_swiglu_fp8(inp.x, inp.w13, inp.w13_s, inp.w2, inp.w2_s, ws=ws, y=y)
        return moe.last_launch_count()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(dev.index or 0)
    barrier(world)
    clocks.start()
    launches = 0
    for i in range(args.steps):
        flush.zero_()   # evict the 0.4 GB of weights from L2 between steps
        ev[i][0].record()
        launches += step()
        ev[i][1].record()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    moe.check_device_error(dev)
    total = sum(a.elapsed_time(b_) for a, b_ in ev)
    ms_total = max_over_ranks(total, world, dev)
    flops = 6.0 * T * d * H
    ms = ms_total / args.steps
    tokens_total = sum_over_ranks(T * args.steps, world, dev)
    w_bytes = 3 * H * d + 3 * (H // 128) * (d // 128) * 4

    # end to end through dense_swiglu_fp8: each step's x copied in from pinned host
    # memory and its y copied out, overlapped with the neighbouring steps' compute
    # (no L2 flush needed: the copies pass 0.23 GB through it)
    e2e_ms, _ = pipelined_e2e(dev, args.steps, args.warmup, inp.x, (T, d),
                              lambda xi, yo: moe.dense_swiglu_fp8(xi, inp.w13, inp.w13_s, inp.w2, inp.w2_s, ws=ws,
                                                                  y=yo), world)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    line = {
        "metric": METRIC, "value": tokens_total / (ms_total * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": DATA,
        "config": dict(workload_config(shape), l2="L2 flushed between steps (256 MB write)"),
        "roofline": roofline("dense_swiglu_fp8 (quantise + GateUpWide + DownWide)", w_bytes + 2 * T * d * 2, flops,
                             ms, peaks),
        "e2e": {"value": tokens_total / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * d * 2, "api": "dense_swiglu_fp8",
                "copies": "pinned host buffers; copy-in and copy-out streams overlapped with the neighbouring "
                          "steps' compute (double buffers)"},
        "gpu_launches": launches, "clocks": clk,
    }
    if want_cpu:
        toks = sample_tokens(T, args.cpu_tokens, seed=args.seed)
        from oracle import moe_oracle as O
        w13, w13_s, w2, w2_s = inp.w13.cpu(), inp.w13_s.cpu(), inp.w2.cpu(), inp.w2_s.cpu()
        xs = inp.x.cpu()[toks]
        t0 = time.perf_counter()
        O.dense_swiglu(xs, w13, w13_s, w2, w2_s)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": len(toks) / dt, "unit": "tokens/s", "cores": _CORES, "kind": "oracle",
                                "sample": f"{len(toks)} of {T} tokens through the fp64 oracle ({dt:.1f} s)"}
    return line


# the workloads a default run measures besides the decode headline
EXTRA_WORKLOADS = ("prefill", "skewed", "skewed40", "dense")
SUMMARY_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "roofline", "layer", "e2e",
                "cpu_baseline", "gpu_launches", "clocks", "block_pieces")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", choices=["all"] + sorted(WORKLOADS), default="all",
                    help="all (default): the decode line plus every other workload under 'workloads'")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-tokens", type=int, default=4, help="tokens in the oracle's timed sample")
    ap.add_argument("--ref-tokens", type=int, default=1, help="tokens per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    shape = WORKLOADS["decode" if args.workload == "all" else args.workload]
    rank, local, world = dist_env()

    if args.impl == "reference":
        line = run_reference(args, shape)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_group(world, "nccl")
    peaks = measured_peaks()
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if isinstance(shape, S.DenseShape):
        line = run_dense(args, shape, rank, world, dev, peaks, want_cpu=want_cpu)
    else:
        line, extra = run_moe(args, shape, rank, local, world, dev, peaks)
        if want_cpu:
            x, wg, b, ex, idx, _ = extra
            line["cpu_baseline"] = cpu_baseline_moe(shape, x, wg, b, ex, idx, args.cpu_tokens, args.seed)
        if args.workload == "all":
            # every other workload, each with its own roofline, clocks, end-to-end figure
            # and oracle sample; the MoE batches reuse the step's 16.96 GB of weights
            ex, ext = extra[3], extra[5]
            wl = {}
            for name in EXTRA_WORKLOADS:
                wshape = WORKLOADS[name]
                if isinstance(wshape, S.DenseShape):
                    wline = run_dense(args, wshape, rank, world, dev, peaks, want_cpu=want_cpu)
                else:
                    wline, wextra = run_moe(args, wshape, rank, local, world, dev, peaks, ex=ex, ext=ext)
                    if want_cpu:
                        x, wg, b, _, idx, _ = wextra
                        wline["cpu_baseline"] = cpu_baseline_moe(wshape, x, wg, b, ex, idx, max(1, args.cpu_tokens // 2),
                                                                 args.seed)
                    del wextra
                wl[name] = {key: wline[key] for key in SUMMARY_KEYS if key in wline}
            line["workloads"] = wl
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
