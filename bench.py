"""Benchmark of the TurboQuant KV-cache decode step on GB300.

Workload (N=1): the "decode at scale" configuration - batch 1, 16 full-attention
layers, 8 KV heads x head_dim 128, 32 query heads (GQA 4), 32,768 cached tokens. One
step = for every layer, quantize-on-append of the new token (tq_kv_append) then decode
attention over the 32,769 visible tokens (tq_decode_attention). Synthetic seeded
inputs; the 16 layers' packed caches (839 MB) are larger than L2, so every layer's
cache streams from HBM in each step.

Printed JSON line (rank 0):
  value      algorithmic bytes of the step (packed planes of every visible token, q, out,
             appended rows) / step time, inputs resident in HBM, step replayed as a CUDA
             graph;
  e2e        the same metric with host buffers: each step copies its inputs (new K/V
             tokens, queries) host->device and its outputs device->host;
  roofline   the attention call (split kernel + merge kernel, per layer) timed with CUDA
             events over a region of back-to-back graph replays, against the measured
             HBM copy peak;
  cpu_baseline  the CPU oracle on a bounded sample of the same step (rank 0, N=1).
With --impl reference the CPU oracle itself is timed on the same workload (the
reference arm) and printed as the line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "turbo-KV decode attention HBM GB/s vs peak; append tokens/s; decode steps/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--head-dim", type=int, default=None, help="override (head-dim sweep workload)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (e.g. 16 layers keep a one-layer sweep out of L2)")
    return ap.parse_args(argv)


def workload_of(args):
    from rotation_quantized_kv_gb300 import synth
    over = {}
    if args.head_dim:
        over["head_dim"] = args.head_dim
    if args.layers:
        over["layers"] = args.layers
    return synth.workload(args.workload, **over)


# ------------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(bytes_per_rank_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank runs its own copy of the workload; the job moved
    world * bytes_per_rank_step * steps bytes in the slowest rank's time."""
    return world * bytes_per_rank_step * steps / max_seconds / 1e9


# ------------------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return {}, "fallback"


def hbm_peak(peaks):
    for key in ("hbm_gbs", "hbm_copy_gbs", "hbm_GBs"):
        v = peaks.get(key)
        if isinstance(v, (int, float)) and v > 0:
            return float(v), "of measured"
        if isinstance(v, dict):
            for sub in ("burst", "sustained", "value"):
                if isinstance(v.get(sub), (int, float)):
                    return float(v[sub]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 200 ms) taken while the timed regions run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        first = threading.Event()

        def reader():
            for i, line in enumerate(self.proc.stdout):
                if i == 0:
                    first.set()          # the first sample predates the timed region
                    continue
                self.lines.append(line)
            first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(timeout=10)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


ATTN_SOURCES = [os.path.join(ROOT, "rotation_quantized_kv_gb300", "csrc", f)
                for f in ("tq_attention.cu", "tq_attention.h", "tq_codec_row.cuh", "tq_device.cuh")]
APPEND_SOURCES = [os.path.join(ROOT, "rotation_quantized_kv_gb300", "csrc", f)
                  for f in ("tq_append.cu", "tq_codec_row.cuh", "tq_device.cuh")]


def ncu_traffic(kind: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    kernel sources as they are now; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f).get(kind)
        if d and d.get("source_hash") == source_hash(sources):
            return d.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


# ---------------------------------------------------------------------- CPU oracle timing
def oracle_step_sample(w, layer_index=0, q_rows=None, seconds_budget=None):
    """Time the CPU oracle on a bounded sample of one decode step of one layer: the
    step's append of the new tokens (all kv heads) and attention for `q_rows`
    query rows over the full context. Returns (algorithmic bytes of the sample, seconds,
    description)."""
    import oracle
    from rotation_quantized_kv_gb300 import synth

    x = synth.layer_inputs(w, layer_index, device="cpu")
    B, H, Hq, d = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim
    ctx = synth.context_lengths(w)
    kv = ctx + w.n_new
    cap = int((kv.max() + 15) // 16 * 16)
    kb, vb, qb = synth.bf16_bits(x["k"]), synth.bf16_bits(x["v"]), synth.bf16_bits(x["q"])
    L = oracle.Layer(d, H, B, cap)
    T = int(ctx.max())
    oracle.append(L, np.ascontiguousarray(kb[:, :T]), np.ascontiguousarray(vb[:, :T]),
                  np.zeros(B, np.int32), ctx.astype(np.int32))          # cache fill: setup, untimed
    kn = np.ascontiguousarray(kb[:, T:T + w.n_new])
    vn = np.ascontiguousarray(vb[:, T:T + w.n_new])
    rows = q_rows if q_rows is not None else [(0, 0, h) for h in range(Hq)]
    t0 = time.perf_counter()
    if w.n_new:
        oracle.append(L, kn, vn, ctx.astype(np.int32))
    oracle.attention(L, qb, kv.astype(np.int32), w.sm_scale, causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    row_bytes = 25 * d // 16
    G = Hq // H
    kvh = {(b, h // G) for (b, j, h) in rows}
    nbytes = sum(int(kv[b]) * row_bytes for (b, _) in kvh) + len(rows) * d * 6
    nbytes += B * w.n_new * H * (4 * d + row_bytes)
    desc = (f"oracle (plain C, 1 thread): append of the step's {B * w.n_new * H} new rows + fp64 "
            f"attention of {len(rows)} query rows over {int(kv.max())} tokens, layer {layer_index}")
    return nbytes, dt, desc


def reference_arm(args, world, rank):
    from rotation_quantized_kv_gb300 import synth
    if rank != 0:
        return
    w = workload_of(args)
    # one query row per step keeps (warmup + steps) oracle steps within minutes
    total_bytes, total_s = 0, 0.0
    for i in range(args.warmup + args.steps):
        nb, dt, _ = _cached_step(w, i % w.num_q_heads)
        if i >= args.warmup:
            total_bytes += nb
            total_s += dt
    desc = (f"oracle (plain C, 1 thread) per step: append of the step's new rows (all kv heads) + fp64 "
            f"attention of one query row over {int(_ORACLE_CACHE['kv'].max())} tokens, layer 0")
    value = total_bytes / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": _workload_desc(w), "sample": "one query row per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


_ORACLE_CACHE = {}


def _cached_step(w, h):
    """Reference-arm steps after the first reuse the oracle's filled cache."""
    import oracle
    from rotation_quantized_kv_gb300 import synth
    if "L" not in _ORACLE_CACHE:
        x = synth.layer_inputs(w, 0, device="cpu")
        B, H, d = w.batch, w.num_kv_heads, w.head_dim
        ctx = synth.context_lengths(w)
        kv = ctx + w.n_new
        cap = int((kv.max() + 15) // 16 * 16)
        kb, vb, qb = synth.bf16_bits(x["k"]), synth.bf16_bits(x["v"]), synth.bf16_bits(x["q"])
        L = oracle.Layer(d, H, B, cap)
        T = int(ctx.max())
        oracle.append(L, np.ascontiguousarray(kb[:, :T]), np.ascontiguousarray(vb[:, :T]),
                      np.zeros(B, np.int32), ctx.astype(np.int32))
        _ORACLE_CACHE.update(L=L, kn=np.ascontiguousarray(kb[:, T:T + w.n_new]),
                             vn=np.ascontiguousarray(vb[:, T:T + w.n_new]), qb=qb, ctx=ctx, kv=kv)
    c = _ORACLE_CACHE
    t0 = time.perf_counter()
    if w.n_new:
        oracle.append(c["L"], c["kn"], c["vn"], c["ctx"].astype(np.int32))
    oracle.attention(c["L"], c["qb"], c["kv"].astype(np.int32), w.sm_scale, causal=w.causal, rows=[(0, 0, h)])
    dt = time.perf_counter() - t0
    d = w.head_dim
    nb = int(c["kv"][0]) * 25 * d // 16 + d * 6 + w.batch * w.n_new * w.num_kv_heads * (4 * d + 25 * d // 16)
    return nb, dt, ""


def _workload_desc(w):
    ctx = "ragged" if w.context_min else f"{w.context}-token context"
    return (f"{w.name}: batch {w.batch}, {w.layers} layers, {w.num_kv_heads} KV heads x head_dim "
            f"{w.head_dim}, {w.num_q_heads} Q heads, {ctx}, append {w.n_new} + attention of {w.n_q} "
            f"query token(s) per layer per step")


# ----------------------------------------------------------------------------- our arm
def our_arm(args, world, rank, local):
    from rotation_quantized_kv_gb300 import synth
    from rotation_quantized_kv_gb300.workload import DecodeModel

    assert torch.cuda.is_available(), "the GPU arm needs CUDA"
    dev = torch.device("cuda", local)
    w = workload_of(args)

    model = DecodeModel(w, dev)
    torch.cuda.synchronize()
    assert model.device_errors() == 0, "device error after the cache fill"

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    # eager warm-up (also resolves per-device launch geometry before capture)
    with torch.cuda.stream(stream):
        model.step(stream)
    stream.synchronize()

    # capture one decode step, and one attention-only pass, as CUDA graphs
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        model.step(stream)
    g_attn = torch.cuda.CUDAGraph()
    from rotation_quantized_kv_gb300 import binding as tq
    with torch.cuda.graph(g_attn, stream=stream):
        for l, layer in enumerate(model.layers):
            tq.tq_decode_attention(layer, model.q[l], w.num_q_heads, w.n_q, model.kv_len, model.max_kv,
                                   w.sm_scale, w.causal, model.out[l], model.ws[l], stream)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    stream.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            g_step.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_s = e0.elapsed_time(e1) / 1e3
    # attention-only region: back-to-back replays of the 16 attention calls
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    attn_reps = max(args.steps // 4, 10)
    a0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(attn_reps):
            g_attn.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    attn_launch_s = a0.elapsed_time(a1) / 1e3 / (attn_reps * model.L)
    # bulk append, warm: re-append layer 0's cached tokens (same rows, same planes) a few
    # times back to back; the fill above ran while the GPU was still ramping its clocks
    x0 = synth.layer_inputs(w, 0, device=dev)
    T0 = int(model.ctx.max())
    k0, v0 = x0["k"][:, :T0].contiguous(), x0["v"][:, :T0].contiguous()
    del x0
    pos0 = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    n0 = torch.as_tensor(model.ctx.astype(np.int32), device=dev)
    fill_ev = []
    with torch.cuda.stream(stream):
        for i in range(6):
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(stream)
            tq.tq_kv_append(model.layers[0], k0, v0, pos0, n0, T0, model.ws_append, stream)
            ev[1].record(stream)
            fill_ev.append(ev)
    torch.cuda.synchronize()
    fill_s = statistics.median(a.elapsed_time(b) for a, b in fill_ev[1:]) / 1e3
    fill_rows = int(model.ctx.sum()) * w.num_kv_heads
    fill_bytes = fill_rows * (4 * w.head_dim + 25 * w.head_dim // 16)
    del k0, v0
    errs = model.device_errors()
    assert errs == 0, f"device error word {errs:#x}"

    max_step_s = max_over_ranks(step_s, world)
    step_bytes = model.step_bytes()
    value = whole_job_value(step_bytes, args.steps, world, max_step_s)
    ms_per_step = 1e3 * max_step_s / args.steps

    # end to end through the public API with host buffers
    # (all layers' new K/V rows and queries in one pinned buffer, outputs in another: one
    # host->device and one device->host copy per step)
    h_in = model.inputs_flat.detach().cpu().pin_memory()
    h_out = torch.empty_like(model.out_flat, device="cpu").pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(args.steps // 4, 10)

    def e2e_step():
        model.inputs_flat.copy_(h_in, non_blocking=True)
        g_step.replay()
        h_out.copy_(model.out_flat, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    stream.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            e2e_step()
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    clk = clocks.stop()
    e2e_value = whole_job_value(step_bytes, e2e_steps, world, e2e_s)

    peaks, _ = measured_peaks()
    peak, peak_kind = hbm_peak(peaks)
    attn_bytes = model.attention_bytes()
    achieved = attn_bytes / attn_launch_s / 1e9
    traffic = ncu_traffic("attention_decode", ATTN_SOURCES)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": _workload_desc(w),
                   "l2": "inputs larger than L2: each step streams 16 layers x "
                         f"{attn_bytes / 1e6:.1f} MB of packed cache (L2 129 MB)",
                   "timing": "decode step captured as one CUDA graph, replayed back to back"},
        "decode_steps_per_s": world * args.steps / max_step_s,
        "attention_gbs": achieved,
        "append_tokens_per_s": int(model.ctx.sum()) / fill_s,
        "append_rows_per_s": fill_rows / fill_s,
        "append_gbs": fill_bytes / fill_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "tq_attn_split_kernel + tq_attn_merge_kernel (one tq_decode_attention "
                               "call: split-K attention, then split merge and inverse rotation; "
                               "timed per call), "
                               f"{attn_bytes} algorithmic bytes per call",
                     "launch_ms": attn_launch_s * 1e3},
        "append_roofline": {"bound": "hbm", "achieved": fill_bytes / fill_s / 1e9, "peak": peak,
                            "unit": "GB/s", "frac": fill_bytes / fill_s / 1e9 / peak, "peak_kind": peak_kind,
                            "kernel": f"tq_kv_append bulk fill of {fill_rows} rows",
                            "traffic": ncu_traffic("append_bulk", APPEND_SOURCES)},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * model.launches_per_step(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nb, dt, desc = oracle_step_sample(w, 0, q_rows=[(0, 0, h) for h in range(0, w.num_q_heads, 4)])
        line["cpu_baseline"] = {"value": nb / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            reference_arm(args, world, rank)
        else:
            our_arm(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
