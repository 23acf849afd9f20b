"""Benchmark of the expert-attention hot path on GB300.

Default workload: one 64-layer Euler step of the action expert's attention (64 independent
layers, S = 4700 valid cache rows, Smax = 8192, bf16 KV caches of [8, 8192, 128] per layer,
2.15 GB in total), run as one ``expert_attn_layers`` call per step. Prints ONE JSON line with
the metric in microseconds per layer, the achieved HBM bandwidth and roofline fraction of the
dominant (attention) kernel, an end-to-end number through the C ABI with host buffers, and the
fp64 CPU oracle timed on the host cores as a reported baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    torchrun --nproc-per-node N bench.py --gpus N ...   (N independent replicas, weak scaling)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_attention_long_gb300._lib import kernels_per_call  # noqa: E402
from gqa_attention_long_gb300.inputs import config_seed, layer_inputs, layer_inputs_on_device  # noqa: E402

METRIC = "µs/layer & achieved HBM GB/s (% roofline), expert attention, S=4700 Smax=8192"
CLOCK_WINDOW_S = 1.5
HQ, HKV, D, T = 16, 8, 128, 64


def algo_bytes_per_layer(S: int, b: int = 2) -> int:
    """Algorithmic HBM bytes of one layer: live cache K/V rows, own K/V rows written and read
    back, raw q/k/v read, output written."""
    return 2 * HKV * S * D * b + 2 * (2 * HKV * T * D * b) + (HQ + 2 * HKV) * T * D * 2 + HQ * T * D * 2


def layer_bytes(S: int, hidden: int = 1536, inter: int = 6144) -> int:
    """Algorithmic HBM bytes of one whole decoder layer: its bf16 weights (wqkv, wo, w1, w3, w2
    and the norm gains), the live cache K/V rows, the own K/V rows written and read back, and
    the residual stream read and written (the activations between the steps are intermediates)."""
    weights = 2 * (4096 * hidden + hidden * 2048 + 3 * inter * hidden + 2 * hidden + 2 * D)
    cache = 2 * HKV * S * D * 2 + 2 * (2 * HKV * T * D * 2)
    return weights + cache + 2 * (2 * T * hidden)


def algo_bytes_per_layer_fp8(S: int) -> int:
    """As algo_bytes_per_layer for an e4m3 cache (1-byte K/V codes; block scales negligible)."""
    return 2 * HKV * S * D + 2 * (2 * HKV * T * D) + (HQ + 2 * HKV) * T * D * 2 + HQ * T * D * 2


def launches_per_call(n_layers: int, S: int, sm_count: int, kv_dtype: int = 0) -> int:
    """Kernels one expert_attn_layers call launches (the library's own plan, mirrored on the
    host: the attention kernel per 64 layers, which merges its split units itself; an e4m3
    cache adds the prologue kernel)."""
    return kernels_per_call(n_layers, S, sm_count, kv_dtype)


def decode_bytes_per_layer(pos: int) -> int:
    """Algorithmic HBM bytes of one text-model decode step of one layer: cache K/V rows 0..pos
    read (row pos after it is written), the new k/v row written, raw q/k/v read, output written."""
    return 2 * HKV * (pos + 1) * D * 2 + 2 * HKV * D * 2 + (64 + 2 * HKV) * D * 2 + 64 * D * 2


def flops_per_layer(S: int) -> int:
    return 4 * (2 * T) * D * (S + T) * HKV


def attention_traffic(S: int, Smax: int, n: int):
    """DRAM bytes per attention launch from the committed ncu capture, or None when the capture
    was taken on another workload or on a different version of the kernel source."""
    import hashlib
    tfile = os.path.join(ROOT, "profiles", "attention_kernel_traffic.json")
    if not os.path.exists(tfile):
        return None
    tj = json.load(open(tfile))
    h = hashlib.sha256()
    for f in tj["source_files"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if h.hexdigest()[:16] != tj["source_sha256_16"]:
        return None
    if (tj.get("S"), tj.get("Smax"), tj.get("layers")) != (S, Smax, n):
        return None
    return tj["bytes_per_launch"]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling (every 50 ms) while the measured steps run. The raw
    samples go to a CSV file in $EA_CLOCKS_DIR (default: the system temporary directory); the
    summary keeps only the samples taken between two marks of the host clock (the window of
    back-to-back steps around the timed region)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(os.environ.get("EA_CLOCKS_DIR") or tempfile.gettempdir(),
                                 f"clocks_gpu{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    @staticmethod
    def _when(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self, t0: float | None = None, t1: float | None = None) -> dict:
        """Median SM clock, highest max clock and active throttle reasons of the samples taken
        in [t0, t1] (host time.time() marks; all samples when no marks are given)."""
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            w = self._when(f[0])
            if t0 is not None and (w is None or w < t0 or w > t1):
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
               "samples": len(sm)}
        if t0 is not None:
            out["window_s"] = round(t1 - t0, 3)
        return out


def oracle_sample(S: int, Smax: int, n_layers: int, min_seconds: float) -> dict:
    """The fp64 CPU oracle, as it stands, on n_layers distinct layers of the workload, repeated
    until min_seconds of oracle time; returns microseconds per layer."""
    import oracle
    f = lambda t: t.double().numpy()  # noqa: E731
    arrays = []
    for l in range(n_layers):
        x = layer_inputs(config_seed(4, l), S, Smax)
        arrays.append([f(v) for v in (x.q_raw, x.k_raw, x.v_raw, x.q_gamma, x.k_gamma, x.k_cache, x.v_cache)])
    done, spent = 0, 0.0
    while spent < min_seconds or done == 0:
        for a in arrays:
            t0 = time.perf_counter()
            oracle.expert_attention_layer(*a, S, Smax, 0)
            spent += time.perf_counter() - t0
            done += 1
    return {"us_per_layer": spent / done * 1e6, "layers": done, "seconds": spent}


def time_calls(fn, warmup: int, reps: int, stream) -> float:
    """Milliseconds per call of fn (launches on `stream`), CUDA events around reps back-to-back
    calls after warmup untimed ones."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, rank: int, world: int) -> None:
    """Reference arm: the fp64 CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    S, Smax = args.S, args.Smax
    for _ in range(args.warmup):
        oracle_sample(S, Smax, 1, 0.0)
    times = []
    for _ in range(args.steps):
        times.append(oracle_sample(S, Smax, 1, 0.0)["us_per_layer"])
    us = statistics.mean(times)
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/layer", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us * 1e-3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args),
            "cpu_baseline": {"value": us, "unit": "us/layer", "cores": cores, "kind": "oracle",
                             "sample": "one layer of the workload per step (fp64 numpy oracle, BLAS threads = all cores)"},
            "e2e": {"value": us, "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_e4m3_step(args, ea, dev, rank: int, world: int) -> None:
    """The step over e4m3 caches alone (caches quantised on the device by the library): warm-up,
    then K timed steps; prints a short JSON line. A target for profilers, not the bench line."""
    S, Smax, n = args.S, args.Smax, args.layers
    ncol = Smax // 128 + 1
    L8 = []
    for l in range(n):
        x = layer_inputs_on_device(config_seed(4, l) + 100000 * rank, S, Smax, dev)
        kq = torch.empty(HKV, Smax, D, dtype=torch.uint8, device=dev)
        vq = torch.empty(HKV, Smax, D, dtype=torch.uint8, device=dev)
        ks = torch.empty(HKV, ncol, dtype=torch.float32, device=dev)
        vs = torch.empty(HKV, ncol, dtype=torch.float32, device=dev)
        ea.expert_attn_quantize_cache(x.k_cache, S, Smax, kq, ks)
        ea.expert_attn_quantize_cache(x.v_cache, S, Smax, vq, vs)
        L8.append(ea.LayerBuffers(q_raw=x.q_raw, k_raw=x.k_raw, v_raw=x.v_raw, q_gamma=x.q_gamma,
                                  k_gamma=x.k_gamma, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs,
                                  out=torch.empty(HQ, T, D, dtype=torch.bfloat16, device=dev)))
        del x
    ws8 = ea.alloc_workspace(n, Smax, ea.EA_KV_FP8_E4M3)
    arr8 = ea.make_args(L8, Smax, ea.EA_KV_FP8_E4M3)
    ea.expert_attn_set_splits(args.splits)
    stream = torch.cuda.current_stream()
    ms = time_calls(lambda: ea.expert_attn_layers(L8, S, Smax, 0, ea.EA_KV_FP8_E4M3, ws8, stream, _arr=arr8),
                    args.warmup, args.steps, stream)
    st, bits = ea.expert_attn_read_status(ws8)
    if st != 0:
        raise RuntimeError(f"e4m3 kernel status bits {bits:#x}")
    b8 = algo_bytes_per_layer_fp8(S) * n
    if rank == 0:
        print(json.dumps({"workload": f"{n}-layer step, S={S}, Smax={Smax}, e4m3 cache", "us_per_layer": ms * 1e3 / n,
                          "ms_per_step": ms, "step_hbm_gbs": b8 / (ms * 1e-3) / 1e9}), flush=True)


def workload_config(args) -> dict:
    return {"workload": f"{args.layers}-layer Euler step of expert attention, S={args.S}, Smax={args.Smax}, bf16 KV cache",
            "layers": args.layers, "S": args.S, "Smax": args.Smax, "q_heads": HQ, "kv_heads": HKV,
            "head_dim": D, "tokens": T, "global_batch": 1,
            "l2": "inputs larger than L2 (distinct caches of all layers, no flush)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--S", type=int, default=4700)
    ap.add_argument("--Smax", type=int, default=8192)
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the FP8 and single-layer extras")
    ap.add_argument("--splits", type=int, default=0, help="attention CTAs (0 = one per SM)")
    ap.add_argument("--kv", choices=["bf16", "e4m3"], default="bf16",
                    help="e4m3: time only the step over e4m3 caches (a profiling target; no extras)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import gqa_attention_long_gb300 as ea
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    S, Smax, n = args.S, args.Smax, args.layers
    if args.kv == "e4m3":
        run_e4m3_step(args, ea, dev, rank, world)
        return
    xs = [layer_inputs_on_device(config_seed(4, l) + 100000 * rank, S, Smax, dev) for l in range(n)]
    # the step's activations (raw q, k, v of every layer) and outputs live in one buffer each, so
    # that the end-to-end path moves them with one host->device and one device->host copy
    act = torch.empty(n, HQ + 2 * HKV, T, D, dtype=torch.bfloat16, device=dev)
    outs = torch.empty(n, HQ, T, D, dtype=torch.bfloat16, device=dev)
    for l, x in enumerate(xs):
        act[l, :HQ].copy_(x.q_raw)
        act[l, HQ:HQ + HKV].copy_(x.k_raw)
        act[l, HQ + HKV:].copy_(x.v_raw)
    Ls = [ea.LayerBuffers(q_raw=act[l, :HQ], k_raw=act[l, HQ:HQ + HKV], v_raw=act[l, HQ + HKV:],
                          q_gamma=x.q_gamma, k_gamma=x.k_gamma, k_cache=x.k_cache, v_cache=x.v_cache,
                          out=outs[l]) for l, x in enumerate(xs)]
    ws = ea.alloc_workspace(n, Smax)
    arr = ea.make_args(Ls, Smax, ea.EA_KV_BF16)
    ea.expert_attn_set_splits(args.splits)
    stream = torch.cuda.current_stream()

    def step():
        ea.expert_attn_layers(Ls, S, Smax, 0, ea.EA_KV_BF16, ws, stream, _arr=arr)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, device time with CUDA events on the launching stream. The
    # clocks are sampled over a window of at least CLOCK_WINDOW_S seconds of the same step run
    # back to back (untimed), which ends with the timed steps themselves, so that the reported
    # clock is the one the timed steps ran at even when they last only milliseconds.
    with ClockSampler(local) as clk:
        t_win0 = time.time()
        while time.time() - t_win0 < CLOCK_WINDOW_S:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_win1 = time.time()
        barrier(world)
        time.sleep(0.1)  # let the sampler write its last line of the window
    clocks = clk.summary(t_win0, t_win1)
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    st, bits = ea.expert_attn_read_status(ws)
    if st != 0:
        raise RuntimeError(f"kernel status bits {bits:#x}")
    ms_step = ms_total / args.steps
    us_layer = ms_step * 1e3 / (n * world)

    # ---- dominant kernel (attention) timed on its own with events between the kernels; with a
    # bf16 cache it is the whole layer (no prologue kernel, and it merges its split units
    # itself), so its algorithmic bytes are the layer's
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e in evs:  # torch creates the CUDA event on first record
        for x in e:
            x.record(stream)
    for i in range(args.steps):
        ea.expert_attn_layers_profiled(Ls, S, Smax, 0, ea.EA_KV_BF16, ws, evs[i], stream, _arr=arr)
    torch.cuda.synchronize()
    k2 = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    peaks = load_peaks()
    k2_bytes = algo_bytes_per_layer(S) * n
    achieved = k2_bytes / (k2 * 1e-3) / 1e9
    traffic = attention_traffic(S, Smax, n)

    # ---- end to end through the C ABI with host buffers: every step copies its raw q/k/v in from
    # pinned host memory, runs the step and copies its outputs back. Two device buffer sets and
    # three streams (host->device copy, compute, device->host copy) let consecutive steps
    # overlap, as a serving loop would; events keep a buffer set from being refilled before the
    # step that reads it, and its outputs from being overwritten before they are copied out.
    h_act = act.cpu().pin_memory()
    h_out = [torch.empty(outs.shape, dtype=outs.dtype).pin_memory() for _ in range(2)]
    act_b = [act, torch.empty_like(act)]
    outs_b = [outs, torch.empty_like(outs)]
    Ls_b = [Ls, [ea.LayerBuffers(q_raw=act_b[1][l, :HQ], k_raw=act_b[1][l, HQ:HQ + HKV],
                                 v_raw=act_b[1][l, HQ + HKV:], q_gamma=x.q_gamma, k_gamma=x.k_gamma,
                                 k_cache=x.k_cache, v_cache=x.v_cache, out=outs_b[1][l])
                 for l, x in enumerate(xs)]]
    arr_b = [arr, ea.make_args(Ls_b[1], Smax, ea.EA_KV_BF16)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}

    def e2e_steps(k_steps):
        for i in range(k_steps):
            b = i % 2
            if i >= 2:  # buffer set b is free once step i-2 has computed from it
                s_in.wait_event(ev["comp"][b])
            with torch.cuda.stream(s_in):
                act_b[b].copy_(h_act, non_blocking=True)
            ev["in"][b].record(s_in)
            stream.wait_event(ev["in"][b])
            if i >= 2:  # its outputs of step i-2 have been copied out
                stream.wait_event(ev["out"][b])
            ea.expert_attn_layers(Ls_b[b], S, Smax, 0, ea.EA_KV_BF16, ws, stream, _arr=arr_b[b])
            ev["comp"][b].record(stream)
            s_out.wait_event(ev["comp"][b])
            with torch.cuda.stream(s_out):
                h_out[b].copy_(outs_b[b], non_blocking=True)
            ev["out"][b].record(s_out)

    e2e_steps(4)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    s_in.wait_stream(stream)
    e2e_steps(args.steps)
    stream.wait_stream(s_out)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world) / args.steps
    h2d = h_act.numel() * h_act.element_size()
    d2h = h_out[0].numel() * h_out[0].element_size()

    # ---- FP8 (e4m3) cache variant of the same step: caches quantised on the device by the library
    fp8 = None
    if not args.no_extras:
        ncol = Smax // 128 + 1
        L8 = []
        for x, L in zip(xs, Ls):
            kq = torch.empty(HKV, Smax, D, dtype=torch.uint8, device=dev)
            vq = torch.empty(HKV, Smax, D, dtype=torch.uint8, device=dev)
            ks = torch.empty(HKV, ncol, dtype=torch.float32, device=dev)
            vs = torch.empty(HKV, ncol, dtype=torch.float32, device=dev)
            ea.expert_attn_quantize_cache(x.k_cache, S, Smax, kq, ks)
            ea.expert_attn_quantize_cache(x.v_cache, S, Smax, vq, vs)
            L8.append(ea.LayerBuffers(q_raw=L.q_raw, k_raw=L.k_raw, v_raw=L.v_raw, q_gamma=L.q_gamma,
                                      k_gamma=L.k_gamma, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs,
                                      out=L.out))
        ws8 = ea.alloc_workspace(n, Smax, ea.EA_KV_FP8_E4M3)
        arr8 = ea.make_args(L8, Smax, ea.EA_KV_FP8_E4M3)
        for _ in range(args.warmup):
            ea.expert_attn_layers(L8, S, Smax, 0, ea.EA_KV_FP8_E4M3, ws8, stream, _arr=arr8)
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            ea.expert_attn_layers(L8, S, Smax, 0, ea.EA_KV_FP8_E4M3, ws8, stream, _arr=arr8)
        g1.record(stream)
        torch.cuda.synchronize()
        st8, bits8 = ea.expert_attn_read_status(ws8)
        if st8 != 0:
            raise RuntimeError(f"fp8 kernel status bits {bits8:#x}")
        ms8 = g0.elapsed_time(g1) / args.steps
        b8 = algo_bytes_per_layer_fp8(S) * n
        fp8 = {"workload": f"{n}-layer step, S={S}, Smax={Smax}, e4m3 cache", "us_per_layer": ms8 * 1e3 / n,
               "ms_per_step": ms8, "step_hbm_gbs": b8 / (ms8 * 1e-3) / 1e9,
               "step_roofline_frac": b8 / (ms8 * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        if n >= 8:  # one layer per call (the e4m3 single-layer configuration), 8 layers rotated
            ws81 = ea.alloc_workspace(1, Smax, ea.EA_KV_FP8_E4M3)
            arr81 = [ea.make_args([L8[l]], Smax, ea.EA_KV_FP8_E4M3) for l in range(8)]
            k81 = [0]

            def one8():
                ea.expert_attn_layers([L8[k81[0] % 8]], S, Smax, 0, ea.EA_KV_FP8_E4M3, ws81, stream,
                                      _arr=arr81[k81[0] % 8])
                k81[0] += 1
            us81 = time_calls(one8, 8, 8 * max(4, args.steps // 2), stream) * 1e3
            st81, bits81 = ea.expert_attn_read_status(ws81)
            if st81 != 0:
                raise RuntimeError(f"fp8 one-layer kernel status bits {bits81:#x}")
            fp8["one_layer_per_call_us"] = us81
            fp8["one_layer_hbm_gbs"] = algo_bytes_per_layer_fp8(S) / (us81 * 1e-6) / 1e9
            del ws81
        del L8, ws8

    # ---- the 64-layer step over the S sweep (S in {1024, 2048, 4700, 8128}, Smax 8192) and with
    # the tighter cache (Smax 5120, S 4700): time should track S + 64, not Smax
    sweep = tight = None
    if not args.no_extras and n == 64 and Smax == 8192 and S <= 4700:
        # rows [S, Smax - 64) of the caches above hold the hidden-row fill; for the larger S of the
        # sweep they are live rows, so they get N(0, 1) values (still hidden at S = 4700)
        g7 = torch.Generator(device=dev).manual_seed(config_seed(4, 999))
        for x in xs:
            for c in (x.k_cache, x.v_cache):
                c[:, S:Smax - T].copy_(torch.randn(HKV, Smax - T - S, D, generator=g7, device=dev))
        sweep = {}
        for S_ in (1024, 2048, 4700, 8128):
            ms_ = ms_step if S_ == S else time_calls(
                lambda: ea.expert_attn_layers(Ls, S_, Smax, 0, ea.EA_KV_BF16, ws, stream, _arr=arr),
                args.warmup, args.steps, stream)
            b_ = algo_bytes_per_layer(S_) * n
            sweep[f"S={S_}"] = {"us_per_layer": ms_ * 1e3 / n, "ms_per_step": ms_,
                                "step_hbm_gbs": b_ / (ms_ * 1e-3) / 1e9,
                                "step_roofline_frac": b_ / (ms_ * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                "roofline_us_per_step_at_8tbs": b_ / 8e12 * 1e6,
                                "frac_of_8tbs_roofline": b_ / 8e12 / (ms_ * 1e-3)}
        st_, bits_ = ea.expert_attn_read_status(ws)
        if st_ != 0:
            raise RuntimeError(f"sweep kernel status bits {bits_:#x}")
        Smax2 = 5120
        xs2 = [layer_inputs_on_device(config_seed(2, l), S, Smax2, dev) for l in range(n)]
        Ls2 = [ea.LayerBuffers(q_raw=L.q_raw, k_raw=L.k_raw, v_raw=L.v_raw, q_gamma=x2.q_gamma,
                               k_gamma=x2.k_gamma, k_cache=x2.k_cache, v_cache=x2.v_cache, out=L.out)
               for L, x2 in zip(Ls, xs2)]
        ws2 = ea.alloc_workspace(n, Smax2)
        arr2 = ea.make_args(Ls2, Smax2, ea.EA_KV_BF16)
        ms2 = time_calls(lambda: ea.expert_attn_layers(Ls2, S, Smax2, 0, ea.EA_KV_BF16, ws2, stream, _arr=arr2),
                         args.warmup, args.steps, stream)
        st2, bits2 = ea.expert_attn_read_status(ws2)
        if st2 != 0:
            raise RuntimeError(f"Smax 5120 kernel status bits {bits2:#x}")
        b2 = algo_bytes_per_layer(S) * n
        tight = {"workload": f"{n}-layer step, S={S}, Smax={Smax2}, bf16 cache", "us_per_layer": ms2 * 1e3 / n,
                 "ms_per_step": ms2, "step_hbm_gbs": b2 / (ms2 * 1e-3) / 1e9,
                 "step_roofline_frac": b2 / (ms2 * 1e-3) / 1e9 / peaks["hbm_gbs"],
                 "ratio_to_smax_8192": ms2 / ms_step}
        del xs2, Ls2, ws2

    # ---- one layer per call (the pages' per-layer measurement), rotating over 8 distinct layers
    single = None
    if not args.no_extras and n >= 8:
        ws1 = ea.alloc_workspace(1, Smax)
        arrs = [ea.make_args([Ls[l]], Smax, ea.EA_KV_BF16) for l in range(8)]
        for l in range(8):
            ea.expert_attn_layers([Ls[l]], S, Smax, 0, ea.EA_KV_BF16, ws1, stream, _arr=arrs[l])
        torch.cuda.synchronize()
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 8 * max(4, args.steps // 2)
        h0.record(stream)
        for k in range(reps):
            ea.expert_attn_layers([Ls[k % 8]], S, Smax, 0, ea.EA_KV_BF16, ws1, stream, _arr=arrs[k % 8])
        h1.record(stream)
        torch.cuda.synchronize()
        us1 = h0.elapsed_time(h1) * 1e3 / reps
        single = {"workload": f"one layer per call, S={S}, Smax={Smax}, bf16 cache, 8 layers rotated (> L2)",
                  "us_per_layer": us1, "hbm_gbs": algo_bytes_per_layer(S) / (us1 * 1e-6) / 1e9}

    # ---- the sequential chain: 64 dependent layers (layer i+1's raw q is layer i's output, a
    # stand-in for the wo/MLP between them), one expert_attn_layer call per layer, replayed as a
    # CUDA graph; latency per layer
    chain = None
    if not args.no_extras:
        Lc = [ea.LayerBuffers(q_raw=(outs[l - 1] if l > 0 else act[0, :HQ]), k_raw=act[l, HQ:HQ + HKV],
                              v_raw=act[l, HQ + HKV:], q_gamma=Ls[l].q_gamma, k_gamma=Ls[l].k_gamma,
                              k_cache=Ls[l].k_cache, v_cache=Ls[l].v_cache, out=outs[l]) for l in range(n)]
        wsc = ea.alloc_workspace(1, Smax)
        arrc = [ea.make_args([Lc[l]], Smax, ea.EA_KV_BF16) for l in range(n)]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for l in range(n):  # warm-up outside the capture (tensor maps, attributes)
                ea.expert_attn_layers([Lc[l]], S, Smax, 0, ea.EA_KV_BF16, wsc, side, _arr=arrc[l])
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for l in range(n):
                ea.expert_attn_layers([Lc[l]], S, Smax, 0, ea.EA_KV_BF16, wsc, side, _arr=arrc[l])
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(side)
        with torch.cuda.stream(side):
            for _ in range(args.steps):
                graph.replay()
        c1.record(side)
        torch.cuda.synchronize()
        stc, bitsc = ea.expert_attn_read_status(wsc)
        if stc != 0:
            raise RuntimeError(f"chain kernel status bits {bitsc:#x}")
        msc = c0.elapsed_time(c1) / args.steps
        chain = {"workload": f"{n} dependent layers (layer i+1's raw q = layer i's output), one expert_attn_layer "
                             f"call each, replayed as a CUDA graph; S={S}, Smax={Smax}, bf16 cache",
                 "us_per_layer": msc * 1e3 / n, "ms_per_chain": msc,
                 "launches_per_layer": launches_per_call(1, S, torch.cuda.get_device_properties(dev).multi_processor_count)}

    # ---- the whole decoder layer with synthetic weights: 8 distinct layers
    # chained (layer i+1's input is layer i's output), one expert_decoder_layer call each,
    # replayed as a CUDA graph; the weights (75.5 MB per layer) and caches of the 8 layers exceed
    # L2, so every replay streams them from HBM
    dlayer = None
    if not args.no_extras and n >= 8:
        from gqa_attention_long_gb300.inputs import expert_layer_weights_on_device
        H, I, NL = 1536, 6144, 8
        Wl = [expert_layer_weights_on_device(config_seed(5, l), dev) for l in range(NL)]
        g5 = torch.Generator(device=dev).manual_seed(config_seed(5, 99))
        xb = [torch.randn(T, H, generator=g5, device=dev).to(torch.bfloat16) for _ in range(NL + 1)]
        wsl = ea.alloc_decoder_layer_workspace(H, I)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())

        def layer_chain():
            for l in range(NL):
                ea.expert_decoder_layer(xb[l], xb[l + 1], Wl[l], xs[l].k_cache, xs[l].v_cache, S, Smax, 0,
                                        wsl, stream=side)
        with torch.cuda.stream(side):
            layer_chain()  # warm-up outside the capture (tensor maps, attributes)
        torch.cuda.synchronize()
        graph_l = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_l, stream=side):
            layer_chain()
        for _ in range(args.warmup):
            graph_l.replay()
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(side)
        with torch.cuda.stream(side):
            for _ in range(args.steps):
                graph_l.replay()
        d1.record(side)
        torch.cuda.synchronize()
        stl, bitsl = ea.expert_attn_read_status(wsl)
        if stl != 0:
            raise RuntimeError(f"decoder layer status bits {bitsl:#x}")
        msl = d0.elapsed_time(d1) / args.steps
        lb = layer_bytes(S, H, I)
        dlayer = {"workload": f"{NL} chained decoder layers (hidden {H}, inter {I}, synthetic bf16 weights "
                              f"75.5 MB per layer), S={S}, Smax={Smax}, bf16 cache, one expert_decoder_layer call "
                              f"each, replayed as a CUDA graph",
                  "us_per_layer": msl * 1e3 / NL, "bytes_per_layer": lb,
                  "hbm_gbs": lb * NL / (msl * 1e-3) / 1e9,
                  "roofline_frac": lb * NL / (msl * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "launches_per_layer": 4 + launches_per_call(1, S, torch.cuda.get_device_properties(dev).multi_processor_count)}
        del Wl, wsl

    # ---- the text model's single-token decode attention over the same caches:
    # the decode token at row pos = S of every layer's cache (the expert never reads that row).
    # All 64 layers in one call (throughput), and one layer per call rotating over 8 layers
    # (the latency of one layer of a decode step)
    tdec = None
    if not args.no_extras:
        g6 = torch.Generator(device=dev).manual_seed(config_seed(6, 0))
        rb = lambda *shape: torch.randn(*shape, generator=g6, device=dev).to(torch.bfloat16)  # noqa: E731
        Ld = [ea.DecodeBuffers(q_raw=rb(64, D), k_raw=rb(HKV, D), v_raw=rb(HKV, D), q_gamma=x.q_gamma,
                               k_gamma=x.k_gamma, k_cache=x.k_cache, v_cache=x.v_cache,
                               out=torch.empty(64, D, dtype=torch.bfloat16, device=dev)) for x in xs]
        wsd = ea.alloc_decode_workspace(n)
        arrd = ea.make_decode_args(Ld, Smax)
        for _ in range(args.warmup):
            ea.text_decode_attention(Ld, S, Smax, 0, wsd, stream, _arr=arrd)
        torch.cuda.synchronize()
        t0d, t1d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0d.record(stream)
        for _ in range(args.steps):
            ea.text_decode_attention(Ld, S, Smax, 0, wsd, stream, _arr=arrd)
        t1d.record(stream)
        torch.cuda.synchronize()
        msd = t0d.elapsed_time(t1d) / args.steps
        ws1d = ea.alloc_decode_workspace(1)
        arr1 = [ea.make_decode_args([Ld[l]], Smax) for l in range(8)]
        for l in range(8):
            ea.text_decode_attention([Ld[l]], S, Smax, 0, ws1d, stream, _arr=arr1[l])
        torch.cuda.synchronize()
        reps = 8 * max(4, args.steps // 2)
        t2d, t3d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t2d.record(stream)
        for k in range(reps):
            ea.text_decode_attention([Ld[k % 8]], S, Smax, 0, ws1d, stream, _arr=arr1[k % 8])
        t3d.record(stream)
        torch.cuda.synchronize()
        us1d = t2d.elapsed_time(t3d) * 1e3 / reps
        for w_ in (wsd, ws1d):
            std, bitsd = ea.expert_attn_read_status(w_)
            if std != 0:
                raise RuntimeError(f"decode kernel status bits {bitsd:#x}")
        bd = decode_bytes_per_layer(S)
        tdec = {"workload": f"text-model decode attention, 64 q heads / 8 kv heads, pos={S}, Smax={Smax}, "
                            f"bf16 cache; {n} layers per call, and one layer per call over 8 layers",
                "us_per_layer": msd * 1e3 / n, "bytes_per_layer": bd,
                "hbm_gbs": bd * n / (msd * 1e-3) / 1e9,
                "roofline_frac": bd * n / (msd * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "one_layer_per_call_us": us1d, "one_layer_hbm_gbs": bd / (us1d * 1e-6) / 1e9,
                "launches_per_call": 1}
        del Ld, wsd, ws1d

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        smp = oracle_sample(S, Smax, 8, 10.0)
        cpu = {"value": smp["us_per_layer"], "unit": "us/layer", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{smp['layers']} layer evaluations over 8 distinct layers of the workload "
                         f"({smp['seconds']:.1f} s, fp64 numpy oracle, BLAS threads = all cores)"}

    if rank == 0:
        step_bytes = algo_bytes_per_layer(S) * n
        line = {
            "metric": METRIC, "value": us_layer, "unit": "us/layer", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(args),
            "step_hbm_gbs": step_bytes / (ms_step * 1e-3) / 1e9 * world,
            "step_roofline_frac": step_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "attention_kernel", "peak_src": peaks["src"],
                         "bytes_per_launch": k2_bytes, "ms_per_launch": k2},
            "kernels_ms": {"attention": k2},
            "clocks": clocks,
            "e2e": {"value": e2e_ms * 1e3 / (n * world), "unit": "us/layer", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "pipelining": "two device buffer sets; host->device copy, step and device->host "
                                  "copy on three streams, consecutive steps overlapping"},
            "gpu_launches": args.steps * launches_per_call(n, S, torch.cuda.get_device_properties(dev).multi_processor_count),
            "cpu_baseline": cpu,
            "fp8_step": fp8,
            "sweep_S": sweep,
            "tight_cache": tight,
            "single_layer": single,
            "sequential_chain": chain,
            "decoder_layer": dlayer,
            "text_decode": tdec,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
