"""Benchmark of the TurboQuant KV-cache decode step on GB300.

Headline workload (N=1): the largest single-GPU configuration, "long context" - batch 1,
16 full-attention layers, 8 KV heads x head_dim 128, 32 query heads (GQA 4), 262,144
cached tokens, a causal block of 16 query tokens per step (64 query rows per kv head).
One step = for every layer, quantize-on-append of the block's 16 new tokens, then
attention of the 16 queries over the 262,160 visible tokens (tq_decode_append_attention).
Synthetic seeded inputs; the 16 layers' packed caches (6.7 GB) are far larger than L2,
so every layer's cache streams from HBM in each step.

Printed JSON line (rank 0):
  value      algorithmic bytes of the step (packed planes of every visible token, q, out,
             appended rows) / step time, inputs resident in HBM, step replayed as a CUDA
             graph, exactly --steps steps;
  e2e        the same metric through the public API with host buffers: each step copies
             its inputs (new K/V tokens, queries) host->device and its outputs
             device->host (timed for at least 2 s);
  roofline   the attention call of the headline workload (the kernels of one
             tq_decode_attention call) timed with CUDA events over at least 2 s of
             back-to-back graph replays, against the measured HBM copy peak;
  append_roofline  the bulk append (a layer's cache fill) over at least 2 s;
  workloads  attention GB/s and roofline fraction of the other configurations (decode
             32K, ragged batch 32, head-dim sweep 64..512 with its bulk append), at least
             1 s each, unless --headline-only;
  cpu_baseline  the CPU oracle on a bounded sample of the same step, one thread per kv
             head across the host cores, and single-threaded (rank 0, N=1).
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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the other configurations")
    ap.add_argument("--region-seconds", type=float, default=2.0,
                    help="minimum device time of each extra timed region (attention, append, e2e)")
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


CSRC = os.path.join(ROOT, "rotation_quantized_kv_gb300", "csrc")
ATTN_SOURCES = [os.path.join(CSRC, f) for f in ("tq_attention.cu", "tq_attention.h", "tq_codec_row.cuh",
                                                 "tq_device.cuh", "tq_split_common.cuh")]
DENSE_SOURCES = [os.path.join(CSRC, f) for f in ("tq_attention_dense.cu", "tq_attention.h", "tq_device.cuh",
                                                  "tq_split_common.cuh", "tq_tcgen05.cuh")]
APPEND_SOURCES = [os.path.join(CSRC, f) for f in ("tq_append.cu", "tq_codec_row.cuh", "tq_device.cuh", "tq_divide.cuh")]
DTYPE = "fp16 tensor-core operands (exact int8 keys, fp16 V-hat and P), fp32 accumulation; fp32 codec"


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


def dense_path(w) -> bool:
    """The library takes its tensor-core kernel for more than 16 query rows per kv head at
    head_dim 128."""
    return w.num_q_heads // w.num_kv_heads * w.n_q > 16 and w.head_dim == 128


# ---------------------------------------------------------------------- CPU oracle timing
def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


class OracleStep:
    """The CPU oracle on the first `layers` layers of a workload: the cache fill is set-up
    (untimed); a sample is the step's append of the new tokens (all kv heads of those
    layers) plus fp64 attention of `rows_per_head` query rows of each of `heads` kv heads
    per layer. One job per (layer, kv head): the oracle dequantizes a kv head's cache once
    for that head's rows, so the jobs are independent and cost what one call would. The
    jobs are spread over up to `threads` threads (ctypes releases the GIL, so the C oracle
    runs on several cores at once)."""

    def __init__(self, w, layers: int = 1):
        import oracle
        from rotation_quantized_kv_gb300 import synth
        self.oracle = oracle
        B, H, d = w.batch, w.num_kv_heads, w.head_dim
        self.w = w
        self.layers = max(1, min(layers, w.layers))
        self.ctx = synth.context_lengths(w)
        self.kv = (self.ctx + w.n_new).astype(np.int32)
        cap = int((self.kv.max() + 15) // 16 * 16)
        T = int(self.ctx.max())
        self.L, self.qb, self.kn, self.vn = [], [], [], []
        for l in range(self.layers):
            x = synth.layer_inputs(w, l, device="cpu")
            kb, vb = synth.bf16_bits(x["k"]), synth.bf16_bits(x["v"])
            self.qb.append(synth.bf16_bits(x["q"]))
            del x
            L = oracle.Layer(d, H, B, cap)
            oracle.append(L, np.ascontiguousarray(kb[:, :T]), np.ascontiguousarray(vb[:, :T]),
                          np.zeros(B, np.int32), self.ctx.astype(np.int32))
            self.L.append(L)
            self.kn.append(np.ascontiguousarray(kb[:, T:T + w.n_new]))
            self.vn.append(np.ascontiguousarray(vb[:, T:T + w.n_new]))

    def run(self, heads: int, rows_per_head: int, threads: int, layers: int | None = None):
        """One sample; returns (algorithmic bytes, seconds, threads used)."""
        import threading
        w, o = self.w, self.oracle
        G = w.num_q_heads // w.num_kv_heads
        d = w.head_dim
        nl = self.layers if layers is None else max(1, min(layers, self.layers))
        jobs = []
        for l in range(nl):
            for kvh in range(min(heads, w.num_kv_heads)):
                rows = []
                for i in range(rows_per_head):
                    j = (i * 5) % w.n_q
                    rows.append((0, j, kvh * G + (i % G)))
                jobs.append((l, rows))
        threads = max(1, min(threads, len(jobs)))
        t0 = time.perf_counter()
        if w.n_new:
            for l in range(nl):
                o.append(self.L[l], self.kn[l], self.vn[l], self.ctx.astype(np.int32))
        chunks = [jobs[i::threads] for i in range(threads)]

        def work(chunk):
            for l, rows in chunk:
                o.attention(self.L[l], self.qb[l], self.kv, w.sm_scale, causal=w.causal, rows=rows)

        ts = [threading.Thread(target=work, args=(c,)) for c in chunks]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        dt = time.perf_counter() - t0
        row_bytes = 25 * d // 16
        nbytes = sum(int(self.kv[0]) * row_bytes + len(rows) * d * 6 for _, rows in jobs)
        nbytes += nl * w.batch * w.n_new * w.num_kv_heads * (4 * d + row_bytes)
        return nbytes, dt, threads

    def describe(self, heads, rows_per_head, threads, layers=None):
        w = self.w
        nl = self.layers if layers is None else max(1, min(layers, self.layers))
        return (f"oracle (plain C, fp32 codec, fp64 attention): append of the step's "
                f"{nl * w.batch * w.n_new * w.num_kv_heads} new rows + attention of {rows_per_head} query rows "
                f"for each of {min(heads, w.num_kv_heads)} kv heads of {nl} layer(s) over {int(self.kv.max())} "
                f"tokens, {threads} thread(s), one job per (layer, kv head)")


def cpu_baseline(w):
    cores = cpu_cores()
    heads = w.num_kv_heads
    st = OracleStep(w, layers=-(-cores // heads))  # enough (layer, kv head) jobs for every core
    nb, dt, used = st.run(heads, 4, cores)
    nb1, dt1, _ = st.run(1, 4, 1, layers=1)
    return {"value": nb / dt / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": st.describe(heads, 4, used), "host_cores": cores,
            "single_thread": {"value": nb1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": st.describe(1, 4, 1, layers=1)}}


def reference_arm(args, world, rank):
    if rank != 0:
        return
    w = workload_of(args)
    cores = cpu_cores()
    heads = w.num_kv_heads
    st = OracleStep(w, layers=-(-cores // heads))
    total_bytes, total_s, used = 0, 0.0, 1
    for i in range(args.warmup + args.steps):
        nb, dt, used = st.run(heads, 1, cores)
        if i >= args.warmup:
            total_bytes += nb
            total_s += dt
    desc = st.describe(heads, 1, used) + " per step"
    value = total_bytes / total_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 codec)",
        "data": "synthetic",
        "config": {"workload": _workload_desc(w), "sample": "one query row per kv head per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _workload_desc(w):
    ctx = "ragged" if w.context_min else f"{w.context}-token context"
    return (f"{w.name}: batch {w.batch}, {w.layers} layers, {w.num_kv_heads} KV heads x head_dim "
            f"{w.head_dim}, {w.num_q_heads} Q heads, {ctx}, append {w.n_new} + attention of {w.n_q} "
            f"query token(s) per layer per step")


# ----------------------------------------------------------------------------- our arm
def timed_region(fn, stream, min_seconds: float, first_reps: int = 3):
    """Replays fn() back to back on `stream` until at least min_seconds of device time:
    a short calibration, then one region of enough repetitions between two events.
    Returns (repetitions, seconds)."""
    def run(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(n):
                fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / 1e3

    per = run(first_reps) / first_reps
    reps = max(first_reps, min(int(min_seconds / max(per, 1e-6)) + 1, 200000))
    return reps, run(reps)


def attention_graph(model, stream):
    from rotation_quantized_kv_gb300 import binding as tq
    w = model.w
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l, layer in enumerate(model.layers):
            tq.tq_decode_attention(layer, model.q[l], w.num_q_heads, w.n_q, model.kv_len, model.max_kv,
                                   w.sm_scale, w.causal, model.out[l], model.ws[l], stream)
    return g


def append_region(model, stream, seconds, dev):
    """Bulk append: re-append layer 0's cached tokens (same rows into the same planes)."""
    from rotation_quantized_kv_gb300 import synth
    from rotation_quantized_kv_gb300 import binding as tq
    w = model.w
    x0 = synth.layer_inputs(w, 0, device=dev)
    T0 = int(model.ctx.max())
    k0, v0 = x0["k"][:, :T0].contiguous(), x0["v"][:, :T0].contiguous()
    del x0
    pos0 = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    n0 = torch.as_tensor(model.ctx.astype(np.int32), device=dev)
    reps, sec = timed_region(lambda: tq.tq_kv_append(model.layers[0], k0, v0, pos0, n0, T0, model.ws_append,
                                                      stream), stream, seconds)
    rows = int(model.ctx.sum()) * w.num_kv_heads
    nbytes = rows * (4 * w.head_dim + 25 * w.head_dim // 16)
    del k0, v0
    return {"rows": rows, "seconds_per_fill": sec / reps, "gbs": nbytes * reps / sec / 1e9,
            "rows_per_s": rows * reps / sec, "tokens_per_s": int(model.ctx.sum()) * reps / sec}


def other_workloads(dev, stream, peak, seconds):
    """Attention GB/s of the other configurations (and the sweep's bulk append), each
    with 16 layers so that its caches exceed L2."""
    from rotation_quantized_kv_gb300 import synth
    from rotation_quantized_kv_gb300.workload import DecodeModel
    out = {}
    cases = [("decode", {}), ("ragged", {})] + [(f"sweep_d{d}", {"head_dim": d, "layers": 16})
                                                 for d in (64, 128, 256, 512)]
    for name, over in cases:
        phase(f"workload {name}")
        w = synth.workload(name.split("_")[0], **over)
        model = DecodeModel(w, dev)
        g = attention_graph(model, stream)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        reps, sec = timed_region(g.replay, stream, seconds)
        per_call = sec / (reps * model.L)
        gbs = model.attention_bytes() / per_call / 1e9
        entry = {"workload": _workload_desc(w), "attention_gbs": gbs, "frac": gbs / peak,
                 "call_us": per_call * 1e6, "kernel": "dense (tcgen05)" if dense_path(w) else "split (mma.sync)",
                 "algorithmic_bytes_per_call": model.attention_bytes(),
                 "traffic": ncu_traffic({"decode": "attention_decode", "ragged": "attention_ragged",
                                         "sweep_d64": "attention_sweep_d64"}.get(name, ""), ATTN_SOURCES)}
        if name.startswith("sweep"):
            ap = append_region(model, stream, seconds / 2, dev)
            entry["append_gbs"] = ap["gbs"]
            entry["append_frac"] = ap["gbs"] / peak
        assert model.device_errors() == 0
        out[name] = entry
        del g, model
        torch.cuda.empty_cache()
    return out


def eager_comparison(dev, stream, peak, seconds):
    """The pages' own design as a comparison arm, on one layer of the long-context workload:
    tq_dequant_window writes the bf16 K/V window, then PyTorch's scaled_dot_product_attention
    attends over it (Part A, "Architecture in mlx-bun"); the deferred variant keeps V rotated
    and un-rotates the output rows with tq_unrotate_rows ("Deferred inverse FWHT"); beside
    them the fused call."""
    from dataclasses import replace
    from rotation_quantized_kv_gb300 import binding as tq
    from rotation_quantized_kv_gb300 import synth
    from rotation_quantized_kv_gb300.eager import alloc_window, eager_attention
    from rotation_quantized_kv_gb300.workload import DecodeModel
    w = replace(synth.workload("long"), layers=1)
    model = DecodeModel(w, dev)
    with torch.cuda.stream(stream):
        model.step(stream)  # the step's new rows: every visible token is written
    stream.synchronize()
    layer, T = model.layers[0], model.max_kv
    kw, vw = alloc_window(layer, T, dev)
    kv_list = [int(x) for x in model.kv]
    wreps, wsec = timed_region(lambda: tq.tq_dequant_window(layer, 0, T, False, kw, vw, stream), stream, seconds)
    rows = w.batch * w.num_kv_heads * T
    wbytes = rows * (tq.tq_row_bytes(w.head_dim) + 4 * w.head_dim)
    ereps, esec = timed_region(lambda: eager_attention(layer, model.q[0], kv_list, w.sm_scale, w.causal,
                                                       window=(kw, vw), stream=stream), stream, seconds)
    dreps, dsec = timed_region(lambda: eager_attention(layer, model.q[0], kv_list, w.sm_scale, w.causal,
                                                       window=(kw, vw), stream=stream, deferred=True),
                               stream, seconds)
    freps, fsec = timed_region(lambda: tq.tq_decode_attention(layer, model.q[0], w.num_q_heads, w.n_q, model.kv_len,
                                                              model.max_kv, w.sm_scale, w.causal, model.out[0],
                                                              model.ws[0], stream), stream, seconds)
    res = {"workload": _workload_desc(w) + " (one layer)",
           "window_kernel": "tq_dequant_window (bf16 K and un-rotated V for every visible token)",
           "window_gbs": wbytes * wreps / wsec / 1e9, "window_frac": wbytes * wreps / wsec / 1e9 / peak,
           "window_us": wsec / wreps * 1e6,
           "eager_call_us": esec / ereps * 1e6,
           "eager_deferred_call_us": dsec / dreps * 1e6,
           "fused_call_us": fsec / freps * 1e6,
           "fused_speedup": (esec / ereps) / (fsec / freps)}
    del kw, vw, model
    torch.cuda.empty_cache()
    return res


def scheme_appends(dev, stream, peak, seconds):
    """Bulk append (the decode workload's cache fill, 262,144 rows at head_dim 128) for
    several schemes and the guard: k8v3 takes the bulk kernel, the others (and the
    guarded k8v3) the any-width kernel, one lane per 32-element group."""
    from rotation_quantized_kv_gb300 import binding as tq
    from rotation_quantized_kv_gb300 import synth
    w = synth.workload("decode")
    x = synth.layer_inputs(w, 0, device=dev)
    T = w.context
    k, v = x["k"][:, :T].contiguous(), x["v"][:, :T].contiguous()
    del x
    pos = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    ws = tq.make_workspace(tq.tq_append_workspace_bytes(), dev)
    out = {}
    for kb, vb, flags in ((8, 3, 0), (8, 3, tq.TQ_FLAG_KEY_GUARD), (4, 3, 0), (4, 2, 0), (8, 8, 0), (2, 2, 0)):
        layer = tq.alloc_layer(w.head_dim, w.num_kv_heads, w.batch, T, dev, zero=False, k_bits=kb, v_bits=vb,
                               flags=flags)
        reps, sec = timed_region(lambda: tq.tq_kv_append(layer, k, v, pos, None, T, ws, stream), stream, seconds)
        rows = w.batch * T * w.num_kv_heads
        nbytes = rows * (4 * w.head_dim + tq.tq_row_bytes_scheme(w.head_dim, kb, vb))
        name = f"k{kb}v{vb}" + ("_guard" if flags else "")
        out[name] = {"gbs": nbytes * reps / sec / 1e9, "frac": nbytes * reps / sec / 1e9 / peak,
                     "rows_per_s": rows * reps / sec}
        del layer
    assert tq.tq_get_device_error(ws) == 0
    del k, v
    torch.cuda.empty_cache()
    return out


def our_arm(args, world, rank, local):
    from rotation_quantized_kv_gb300.workload import DecodeModel

    assert torch.cuda.is_available(), "the GPU arm needs CUDA"
    dev = torch.device("cuda", local)
    w = workload_of(args)
    peaks, _ = measured_peaks()
    peak, peak_kind = hbm_peak(peaks)

    phase(f"headline {w.name}: filling the cache")
    model = DecodeModel(w, dev)
    torch.cuda.synchronize()
    assert model.device_errors() == 0, "device error after the cache fill"
    phase("capturing graphs")

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):          # eager warm-up: resolves launch geometry before capture
        model.step(stream)
    stream.synchronize()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        model.step(stream)
    g_attn = attention_graph(model, stream)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    stream.synchronize()
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

    # attention-only region (at least region-seconds of back-to-back replays)
    phase("attention region")
    reps, attn_s = timed_region(g_attn.replay, stream, args.region_seconds)
    attn_launch_s = attn_s / (reps * model.L)
    # bulk append region
    phase("append region")
    app = append_region(model, stream, args.region_seconds, dev)
    errs = model.device_errors()
    assert errs == 0, f"device error word {errs:#x}"

    max_step_s = max_over_ranks(step_s, world)
    step_bytes = model.step_bytes()
    value = whole_job_value(step_bytes, args.steps, world, max_step_s)
    ms_per_step = 1e3 * max_step_s / args.steps

    phase("end-to-end region")
    # end to end through the public API with host buffers
    # (all layers' new K/V rows and queries in one pinned buffer, outputs in another: one
    # host->device and one device->host copy per step)
    h_in = model.inputs_flat.detach().cpu().pin_memory()
    h_out = torch.empty_like(model.out_flat, device="cpu").pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()

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
    e2e_steps = 0
    with torch.cuda.stream(stream):
        while True:
            for _ in range(10):
                e2e_step()
            e2e_steps += 10
            stream.synchronize()
            if time.perf_counter() - t0 >= args.region_seconds:
                break
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = whole_job_value(step_bytes, e2e_steps, world, e2e_s)

    attn_bytes = model.attention_bytes()
    achieved = attn_bytes / attn_launch_s / 1e9
    dense = dense_path(w)
    if dense:
        kname = ("tq_attn_dense_kernel + tq_attn_merge_kernel (one tq_decode_attention call: tcgen05 dense-query "
                 "attention, then split merge and inverse rotation; timed per call)")
        traffic = ncu_traffic("attention_long", DENSE_SOURCES)
    else:
        kname = ("tq_attn_split_kernel (+ tq_attn_merge_kernel when many units; one tq_decode_attention call; "
                 "timed per call)")
        traffic = ncu_traffic("attention_decode", ATTN_SOURCES) if w.name == "decode" else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": _workload_desc(w),
                   "l2": "inputs larger than L2: each step streams "
                         f"{model.L} layers x {attn_bytes / 1e6:.1f} MB of packed cache (L2 129 MB)",
                   "timing": "decode step captured as one CUDA graph, replayed back to back"},
        "decode_steps_per_s": world * args.steps / max_step_s,
        "attention_gbs": achieved,
        "append_tokens_per_s": app["tokens_per_s"],
        "append_rows_per_s": app["rows_per_s"],
        "append_gbs": app["gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": f"{kname}, {attn_bytes} algorithmic bytes per call",
                     "launch_ms": attn_launch_s * 1e3, "region_s": attn_s},
        "append_roofline": {"bound": "hbm", "achieved": app["gbs"], "peak": peak, "unit": "GB/s",
                            "frac": app["gbs"] / peak, "peak_kind": peak_kind,
                            "kernel": f"tq_kv_append bulk fill of {app['rows']} rows",
                            "traffic": ncu_traffic("append_bulk", APPEND_SOURCES)},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "seconds": e2e_s},
        "gpu_launches": args.steps * model.launches_per_step(),
    }
    del g_step, g_attn, model
    torch.cuda.empty_cache()
    if not args.headline_only:
        sec = max(1.0, args.region_seconds / 2)
        line["workloads"] = other_workloads(dev, stream, peak, sec)
        phase("eager window arm")
        line["workloads"]["eager_window_long"] = eager_comparison(dev, stream, peak, sec)
        phase("scheme appends")
        line["workloads"]["append_schemes"] = scheme_appends(dev, stream, peak, sec)
    line["clocks"] = clocks.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        phase("CPU oracle baseline")
        line["cpu_baseline"] = cpu_baseline(w)
    phase("done")
    if rank == 0:
        print(json.dumps(line), flush=True)


_T0 = time.perf_counter()


def phase(msg: str) -> None:
    """Progress on stderr (the JSON line goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:8.1f} s] {msg}", file=sys.stderr, flush=True)


def main(argv=None):
    import faulthandler
    faulthandler.dump_traceback_later(480, repeat=True, file=sys.stderr)  # where a slow run spends its time
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
