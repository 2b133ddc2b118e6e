"""Decode-attention benchmark over a two-D compressed KV cache.

Workload: the 128K-context batch-8 Llama-3.1-8B-shaped attention layer
(8 KV heads, 32 query heads, head dim 128, segment 128, c = 40, tau = 0.85,
top-k 4096), 32 independently seeded layers.  One step = one decode step of
every layer (mkv_decode per layer, layers cycled so that the 674 MB of packed
keys each layer streams never sit in the 129 MB L2).  Inputs are synthetic
(seeded generators; no model weights or datasets).

Metric: context tokens attended per second = layers * B * T / step time.
Prints one JSON line.  With torchrun (N > 1) each rank runs the whole workload
on its own GPU (weak scaling, no data-path collective); the step time is the
maximum over ranks.

--impl reference times the CPU oracle (fp64 NumPy) on a bounded sample of the
same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from two_compressed_kv_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attention ctx-tokens/s (128K, bs8) and achieved HBM GB/s vs 8 TB/s"
UNIT = "ctx-tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = os.environ.get("MKV_DIST_BACKEND") or ("nccl" if torch.cuda.is_available()
                                                          else "gloo")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(ms_local: float, steps: int, units_per_rank_step: float, ws: int, device):
    """Whole-job throughput: every rank runs the same per-rank work (weak
    scaling); the step time is the slowest rank's.  Returns (ms per step,
    units per second over all ranks)."""
    ms = _max_over_ranks(ms_local, ws, device)
    ms_step = ms / steps
    return ms_step, ws * units_per_rank_step / (ms_step / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def committed_traffic(kernel_file: str, summary: str):
    """DRAM bytes per launch of the score kernel from a committed ncu summary,
    or None when the summary is missing or was taken on a different source."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    src = open(os.path.join(ROOT, "two_compressed_kv_gb300", "csrc", kernel_file), "rb").read()
    sha = hashlib.sha256(src).hexdigest()
    vals = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxes.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


# ---------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_prepare(w: W.Workload, K=None, V=None, q=None):
    """Compresses stream (b=0, h=0) of layer 0 with the oracle (not timed) and
    returns what the timed oracle decode needs."""
    from oracle import mosaickv as O
    if K is None:
        K, V = W.draw_kv(w, layer=0, device="cpu", streams=1)
        q = W.draw_queries(w, K)
    Kn = K[0, 0].cpu().numpy()
    Vn = V[0, 0].cpu().numpy()
    qn = q[0, :w.group].cpu().numpy()
    ck = O.compress_stream(Kn, w.segment, w.c, w.tau)
    cv = O.compress_stream(Vn, w.segment, w.c, w.tau)
    hk, pk = O.pack_stream(ck)
    hv, pv = O.pack_stream(cv)
    return {"T": Kn.shape[0], "q": qn, "ck": ck, "cv": cv, "hk": hk, "pk": pk, "hv": hv, "pv": pv}


def oracle_decode_sample(w: W.Workload, seconds: float, prep):
    """Times the oracle's decode (unpack the packed stream + scores + top-k +
    attention) of the prepared stream, repeated for about `seconds` (at least
    once).  Returns (ctx-tokens/s, repetitions, median seconds per decode).
    A context token has one stream per KV head, so the rate is T over the time
    of n_kv_heads such decodes (one stream timed, scaled)."""
    from oracle import mosaickv as O
    T = prep["T"]
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        Kh = O.unpack_stream(prep["hk"], prep["pk"], T, w.segment, w.c)
        Vh = O.unpack_stream(prep["hv"], prep["pv"], T, w.segment, w.c)
        O.decode_stream(prep["q"], prep["ck"].R, prep["cv"].R, Kh, Vh, w.top_k)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end:
            break
    per = statistics.median(times)
    return T / (per * w.n_kv_heads), len(times), per


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def host_cpu() -> dict:
    """Host CPU description for the CPU-baseline record: logical CPU count and
    model name (the "model name" line on x86, "CPU implementer/part" codes on
    Arm, else the platform string)."""
    import platform
    model = ""
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        model = fields.get("model name") or fields.get("Model name") or ""
        if not model and "CPU implementer" in fields:
            model = f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    except OSError:
        pass
    return {"cpu_count": os.cpu_count() or 1,
            "cpu_model": model or platform.processor() or platform.machine()}


def workload_config(w: W.Workload, layers: int, k_bytes: float = None) -> dict:
    if k_bytes is None:
        l2 = "inputs larger than L2 (129 MB), layers cycled"
    else:
        l2 = (f"inputs larger than L2 (129 MB): each layer streams {k_bytes / 1e6:.0f} MB of "
              f"packed keys, {layers} layers cycled")
    return {
        "workload": f"{w.name}: batch {w.batch}, {w.n_kv_heads} KV / {w.n_q_heads} query heads, "
                    f"head dim 128, context {w.ctx}, {layers} layers, segment {w.segment}, "
                    f"c {w.c}, tau {w.tau}, top-k {w.top_k}",
        "batch": w.batch, "ctx": w.ctx, "layers": layers, "n_kv_heads": w.n_kv_heads,
        "n_q_heads": w.n_q_heads, "head_dim": 128, "segment": w.segment, "c": w.c,
        "tau": w.tau, "top_k": w.top_k, "storage": "fp16 values, uint8 channel indices",
        "l2": l2,
    }


def one_thread_oracle(workload: str, seconds: float) -> dict:
    """The same oracle decode sample in a child process whose BLAS and OpenMP
    pools have one thread (the pool size is fixed when numpy loads)."""
    import subprocess
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from two_compressed_kv_gb300 import workloads as W; "
            "w = W.WORKLOADS[%r]; v, reps, per = bench.oracle_decode_sample(w, %r, "
            "bench.oracle_prepare(w)); print(json.dumps({'value': v, 'reps': reps}))"
            % (ROOT, workload, float(seconds)))
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, timeout=900,
                           stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": d["value"], "unit": UNIT, "cores": 1, "repetitions": d["reps"]}
    except Exception as e:   # the all-core figure stands on its own
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def run_reference(args, w: W.Workload, ws: int, rank: int):
    if rank != 0:
        return
    cfg = workload_config(w, 1)
    cfg["sample"] = "stream (b=0, h=0) of layer 0"
    # each step is a bounded sample of the oracle's decode; the whole run stays
    # within about 90 s of oracle time whatever --steps is
    per_step = max(0.25, min(args.ref_seconds, 90.0 / (args.warmup + args.steps)))
    vals = []
    n = 0
    prep = oracle_prepare(w)
    for i in range(args.warmup + args.steps):
        v, reps, per = oracle_decode_sample(w, per_step, prep)
        if i >= args.warmup:
            vals.append(v)
            n += reps
    value = statistics.median(vals)
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.ctx / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         **host_cpu(),
                         "sample": f"oracle decode (unpack + score + top-k + attention) of one "
                                   f"{w.ctx}-token stream of layer 0, {n} timed repetitions, "
                                   f"scaled to the {w.n_kv_heads} KV heads of a token"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if not args.no_one_thread:
        line["cpu_baseline"]["one_thread"] = one_thread_oracle(args.workload, 5.0)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def capture_steps(step, n: int, dev):
    """n CUDA graphs, each holding one call of step()."""
    out = []
    for _ in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        out.append(g)
    torch.cuda.synchronize(dev)
    return out


def kernel_times(ctxs, step, flags: int, n: int, dev, base_flags: int = 0) -> dict:
    """Per-kernel device time of n decode steps run with the given timing
    flags (events are recorded when a graph is captured, so the timers are
    reset after a warm-up graph has run and each timed graph runs exactly
    once before they are read).  Returns {kernel name: (total ms, launches)}."""
    from two_compressed_kv_gb300 import mkv as M
    for m in ctxs:
        M.mkv_set_flags(m.ctx, flags)
    try:
        for g in capture_steps(step, 1, dev):
            g.replay()
        torch.cuda.synchronize(dev)
        for m in ctxs:
            for kid in range(len(M.KERNEL_NAMES)):
                M.mkv_kernel_time(m.ctx, kid, reset=True)
        for g in capture_steps(step, n, dev):
            g.replay()
        torch.cuda.synchronize(dev)
        out = {}
        for kid, name in enumerate(M.KERNEL_NAMES):
            tot, cnt = 0.0, 0
            for m in ctxs:
                a, b = M.mkv_kernel_time(m.ctx, kid, reset=True)
                tot, cnt = tot + a, cnt + b
            if cnt:
                out[name] = (tot, cnt)
        return out
    finally:
        for m in ctxs:
            M.mkv_set_flags(m.ctx, base_flags)


def fused_step_ms(ctxs, qs, outs, steps: int, dev, stream) -> float:
    """Device time of one step decoded with mkv_decode_layers (all layers, up
    to 64 per call, one launch of each decode kernel per call), timed like the
    headline: CUDA-graph replays, 3 warm-up steps, CUDA events."""
    from two_compressed_kv_gb300 import mkv as M
    groups = [range(i, min(i + M.MKV_MAX_FUSED_LAYERS, len(ctxs)))
              for i in range(0, len(ctxs), M.MKV_MAX_FUSED_LAYERS)]

    def fstep():
        for gr in groups:
            M.mkv_decode_layers([ctxs[i].ctx for i in gr], [qs[i] for i in gr],
                                [outs[i] for i in gr])

    fstep()
    torch.cuda.synchronize(dev)
    graphs = capture_steps(fstep, steps + 3, dev)
    for g in graphs[:3]:
        g.replay()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for g in graphs[3:]:
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    for m in ctxs:
        if M.mkv_check_device(m.ctx) != M.MKV_OK:
            raise RuntimeError("a device-side check fired during the fused timing")
    return ev0.elapsed_time(ev1) / steps


def gathered_bytes(m, M, sel: np.ndarray, w: W.Workload) -> float:
    """Bytes of the K and V rows (plus shared masks) that the selected tokens
    read, counted from the packed layout of every stream."""
    c = w.c
    total = 0
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            for x in range(2):
                hdr = M.mkv_export_headers(m.ctx, b, h, x, m.n_segments())
                segs = sel[b, h] // w.segment
                st = hdr["strategy"][segs]
                row = np.select([st == 0, st == 1, st == 3], [2 * c, 3 * c, 2 * c + 16], 256)
                total += int(row.sum())
                sm_segs = np.unique(segs[st == 0])
                total += len(sm_segs) * ((c + 15) // 16 * 16)
    return float(total)


def run_gpu(args, w: W.Workload, ws: int, rank: int, local: int):
    from two_compressed_kv_gb300 import mkv as M
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    L = args.layers
    base_flags = M.MKV_FLAG_NO_PDL if args.no_pdl else 0
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, w.segment, w.c, w.tau,
                        w.top_k, flags=base_flags, device=local)
    ctxs, qs, outs = [], [], []
    comp_ms = []
    cpu_args = None
    for layer in range(L):
        K, V = W.draw_kv(w, layer=layer, device=dev)
        q = W.draw_queries(w, K, layer=layer)
        if layer == 0 and rank == 0 and ws == 1 and not args.no_cpu_baseline:
            cpu_args = (K[:1, :1].cpu(), V[:1, :1].cpu(), q[:1].cpu())
        m = M.Mkv(cfg)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        m.compress(K, V)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        comp_ms.append(e0.elapsed_time(e1))
        ctxs.append(m)
        qs.append(q)
        outs.append(torch.empty(q.shape, dtype=torch.float32, device=dev))
        del K, V
    torch.cuda.empty_cache()
    st0 = ctxs[0].stats()
    kk = min(w.top_k, w.ctx)
    sel0 = torch.empty(w.batch, w.n_kv_heads, kk, dtype=torch.int32, device=dev)

    def step():
        # the binding launches on torch's current stream: the capture stream
        # while a graph is being captured
        for m, q, o in zip(ctxs, qs, outs):
            M.mkv_decode(m.ctx, q, o, None, None)

    # One CUDA graph per step (all layers): replays have no host launch gaps.
    # The timed graphs hold no events: each decode kernel may start while the
    # one before it finishes (programmatic dependent launch).
    def capture(n):
        return capture_steps(step, n, dev)

    l0 = sum(m.stats()["kernel_launches"] for m in ctxs)
    step()
    torch.cuda.synchronize(dev)
    per_step_launches = sum(m.stats()["kernel_launches"] for m in ctxs) - l0
    use_graph = not args.no_graph
    warm = capture(args.warmup) if use_graph else []
    for i in range(args.warmup):
        warm[i].replay() if use_graph else step()
    torch.cuda.synchronize(dev)
    timed = capture(args.steps) if use_graph else []
    if use_graph:              # re-warm after the capture pause
        timed[0].replay()
        timed[min(1, args.steps - 1)].replay()
        torch.cuda.synchronize(dev)
    launches0 = sum(m.stats()["kernel_launches"] for m in ctxs)

    def run(i):
        if use_graph:
            timed[i].replay()
        else:
            step()

    clocks = ClockSampler(local)
    _barrier(ws)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        run(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    _barrier(ws)
    clk = clocks.stop()
    for m in ctxs:
        if M.mkv_check_device(m.ctx) != M.MKV_OK:
            raise RuntimeError("a device-side wait gave up during the timed region")
    if use_graph:   # kernels are counted when captured: one step's worth per graph
        launches = per_step_launches * args.steps
    else:
        launches = sum(m.stats()["kernel_launches"] for m in ctxs) - launches0
    units_step = L * w.batch * w.ctx
    ms_step, value = _job_value(ev0.elapsed_time(ev1), args.steps, units_step, ws, dev)
    fused_ms = fused_step_ms(ctxs, qs, outs, args.steps, dev, stream) if use_graph else None

    # per-kernel device time: the same steps again, with events around every
    # kernel (which launches them one after another), then around the score
    # kernel alone
    ktimes = kernel_times(ctxs, step, M.MKV_FLAG_KERNEL_TIMING, min(args.steps, 10), dev,
                          base_flags)
    ktimes["score"] = kernel_times(ctxs, step, M.MKV_FLAG_SCORE_TIMING, min(args.steps, 10),
                                   dev, base_flags)["score"]

    # algorithmic bytes of one layer-step (layer 0), counted from its layout
    M.mkv_decode(ctxs[0].ctx, qs[0], outs[0], sel0, stream)
    torch.cuda.synchronize(dev)
    score_bytes = float(st0["payload_bytes"][0] + st0["header_bytes"] // 2)
    gath = gathered_bytes(ctxs[0], M, sel0.cpu().numpy(), w)
    small = (w.batch * w.n_q_heads * 128 * (2 + 4) + 2 * w.streams * 128 * 128 * 4)
    alg_layer = score_bytes + gath + small
    hbm_gbs = alg_layer * L / (ms_step / 1e3) / 1e9

    peak, peak_kind = measured_peaks()
    s_ms, s_n = ktimes["score"]
    score_avg_s = s_ms / max(1, s_n) / 1e3
    roof = {"kernel": "score_kernel", "bound": "hbm",
            "achieved": score_bytes / score_avg_s / 1e9, "peak": peak, "unit": "GB/s",
            "frac": score_bytes / score_avg_s / 1e9 / peak, "peak_kind": peak_kind,
            "traffic": committed_traffic("k_score.cu", "score_kernel_headline_128k.txt"),
            "algorithmic_bytes_per_launch": score_bytes,
            "avg_launch_us": score_avg_s * 1e6}

    # end to end through the public API with host buffers: per step, one copy
    # of every layer's queries from pinned host memory, mkv_decode of each
    # layer (launched from the host, not captured), one copy of every
    # layer's output back
    q_host = torch.stack([q.cpu() for q in qs]).pin_memory()
    q_dev = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev)
    out_dev = torch.empty((L,) + tuple(outs[0].shape), dtype=torch.float32, device=dev)
    out_host = torch.empty(out_dev.shape, dtype=torch.float32).pin_memory()
    h2d = q_host.numel() * q_host.element_size()
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        q_dev.copy_(q_host, non_blocking=True)
        for layer, m in enumerate(ctxs):
            M.mkv_decode(m.ctx, q_dev[layer], out_dev[layer], None, stream)
        out_host.copy_(out_dev, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    _barrier(ws)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    t_e2e = time.perf_counter() - t0
    _barrier(ws)
    t_e2e = _max_over_ranks(t_e2e, ws, dev)
    e2e_value = ws * units_step * args.steps / t_e2e

    cpu = None
    if cpu_args is not None:
        cv, reps, per = oracle_decode_sample(w, args.cpu_seconds, oracle_prepare(w, *cpu_args))
        cpu = {"value": cv, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", **host_cpu(),
               "sample": f"oracle decode (unpack + score + top-k + attention) of one "
                         f"{w.ctx}-token stream (b=0, h=0) of layer 0, {reps} repetitions, "
                         f"median {per * 1e3:.0f} ms, scaled to the {w.n_kv_heads} KV heads "
                         f"of a token"}

    comp_kernels = None
    side = {}
    if rank == 0:
        for c in ctxs:
            c.close()
        ctxs = []
        torch.cuda.empty_cache()
        comp_kernels = compress_kernel_ms(w, dev)
    if rank == 0 and not args.no_side:
        for name, layers in ((W.MILLION_1M.name, 1), (W.MIXED_256K.name, 1),
                             (W.LAYER_32K.name, 32)):
            side[name] = side_workload(W.WORKLOADS[name], layers, max(5, args.steps), dev, stream)
            torch.cuda.empty_cache()
        # the headline shape with bitmask-indexed per-vector segments (4 layers)
        from two_compressed_kv_gb300 import mkv as M
        side[w.name + "+bitmask-pv"] = side_workload(w, 4, max(5, args.steps), dev, stream,
                                                     M.MKV_FLAG_BITMASK_PV)
        torch.cuda.empty_cache()

    if rank == 0:
        cfgd = workload_config(w, L, score_bytes)
        cfgd["parallelism"] = f"replicas x{ws}" if ws > 1 else "single GPU"
        tok = L * w.batch * w.ctx
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": cfgd,
            "hbm_gbs": hbm_gbs, "hbm_frac_of_measured": hbm_gbs / peak,
            "hbm_frac_of_nominal_8tbs": hbm_gbs / NOMINAL_HBM_GBS,
            "algorithmic_bytes_per_layer_step": alg_layer,
            "roofline": roof,
            "score_kernel_us_per_layer": ktimes["score"][0] / max(1, ktimes["score"][1]) * 1e3,
            "kernel_us_per_layer_standalone": {k: v[0] / max(1, v[1]) * 1e3
                                               for k, v in ktimes.items()},
            "pdl": not args.no_pdl,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "cuda_graph": use_graph,
            "clocks": clk,
            "prefill": {"value": w.batch * w.ctx / (statistics.median(comp_ms) / 1e3),
                        "unit": "prefill-tokens/s per layer (K and V)",
                        "ms_per_layer_median": statistics.median(comp_ms)},
            "compression": {"payload_bytes_K": st0["payload_bytes"][0],
                            "payload_bytes_V": st0["payload_bytes"][1],
                            "uncompressed_bytes": st0["uncompressed_bytes"],
                            "ratio": st0["uncompressed_bytes"] / (st0["payload_bytes"][0] +
                                                                  st0["payload_bytes"][1]),
                            "strategies_K": st0["strategy_count"][0],
                            "strategies_V": st0["strategy_count"][1]},
            "ctx_tokens_per_step": tok,
        }
        if fused_ms:
            line["fused_layers"] = {
                "api": f"mkv_decode_layers (all {L} layers in one call: one launch of each "
                       f"decode kernel per step)",
                "ms_per_step": fused_ms, "value": ws * tok / (fused_ms / 1e3), "unit": UNIT,
                "hbm_frac_of_measured": alg_layer * L / (fused_ms / 1e3) / 1e9 / peak}
        line["prefill"].update(prefill_roofline(w, statistics.median(comp_ms), st0, peak))
        line["prefill"]["kernel_ms_per_layer"] = comp_kernels
        if side:
            line["other_workloads"] = side
        print(json.dumps(line), flush=True)
    for m in ctxs:
        m.close()


def compress_kernel_ms(w: W.Workload, dev) -> dict:
    """Device time of each compression step for layer 0 (a fresh ctx with
    kernel timing on; the layer is compressed twice, the second is read)."""
    from two_compressed_kv_gb300 import mkv as M
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, w.segment, w.c, w.tau,
                        w.top_k, flags=M.MKV_FLAG_KERNEL_TIMING, device=dev.index or 0)
    K, V = W.draw_kv(w, layer=0, device=dev)
    out = {}
    with M.Mkv(cfg) as m:
        m.compress(K, V)
        torch.cuda.synchronize(dev)
        for kid in range(5, 10):
            M.mkv_kernel_time(m.ctx, kid, reset=True)
        m.compress(K, V)
        torch.cuda.synchronize(dev)
        for kid, name in enumerate(M.COMPRESS_KERNEL_NAMES, start=5):
            out[name] = M.mkv_kernel_time(m.ctx, kid)[0]
    del K, V
    torch.cuda.empty_cache()
    return out


def prefill_roofline(w: W.Workload, ms: float, st: dict, peak_gbs: float) -> dict:
    """mkv_compress against its bounds.  Algorithmic bytes: K and V read twice
    (the Gram pass, then the rotation pass, which needs the finished basis)
    plus the packed cache written.  Tensor work: the Gram (2 T d^2 per stream)
    and the rotation (2 T d^2 per stream and pass, two fp16 parts of R, two
    passes), all fp16 with fp32 accumulation; peak = the measured bf16 GEMM
    rate (the fp16 dense rate is the same)."""
    streams = 2 * w.batch * w.n_kv_heads
    x_bytes = streams * w.ctx * 128 * 2
    alg = 2 * x_bytes + st["payload_bytes"][0] + st["payload_bytes"][1] + st["header_bytes"]
    flops = streams * w.ctx * 128 * 128 * 2 * (1 + 2 * 2)
    tf_peak = None
    pth = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pth):
        with open(pth) as f:
            tf_peak = float(json.load(f).get("bf16_tflops", 0.0)) or None
    gbs = alg / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    return {"algorithmic_bytes_per_layer": alg, "hbm_gbs": gbs, "hbm_frac_of_measured": gbs / peak_gbs,
            "tensor_flops_per_layer": flops, "tensor_tflops": tfs,
            "tensor_frac_of_measured_bf16": (tfs / tf_peak) if tf_peak else None}


def side_workload(w: W.Workload, layers: int, steps: int, dev, stream, flags: int = 0) -> dict:
    """One more workload, timed like the headline (CUDA-graph replays of a
    decode of every layer, 3 warm-up steps, CUDA events on the launching
    stream) plus its mkv_compress time per layer."""
    from two_compressed_kv_gb300 import mkv as M
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, w.segment, w.c, w.tau,
                        w.top_k, flags=flags, device=dev.index or 0)
    ctxs, qs, outs, comp = [], [], [], []
    for layer in range(layers):
        K, V = W.draw_kv(w, layer=layer, device=dev)
        q = W.draw_queries(w, K, layer=layer)
        m = M.Mkv(cfg)
        m.compress(K, V)          # first compression of a shape: not timed
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        m.compress(K, V)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        comp.append(e0.elapsed_time(e1))
        ctxs.append(m)
        qs.append(q)
        outs.append(torch.empty(q.shape, dtype=torch.float32, device=dev))
        del K, V
    st0 = ctxs[0].stats()

    def step():
        for m, q, o in zip(ctxs, qs, outs):
            M.mkv_decode(m.ctx, q, o, None, None)

    step()
    torch.cuda.synchronize(dev)
    graphs = capture_steps(step, steps + 3, dev)
    for g in graphs[:3]:
        g.replay()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for g in graphs[3:]:
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms_step = ev0.elapsed_time(ev1) / steps
    for m in ctxs:
        if M.mkv_check_device(m.ctx) != M.MKV_OK:
            raise RuntimeError("a device-side check fired during the timed region")
    fused_ms = fused_step_ms(ctxs, qs, outs, steps, dev, stream) if layers > 1 else None
    kt = kernel_times(ctxs, step, flags | M.MKV_FLAG_KERNEL_TIMING, 5, dev, flags)
    s_ms, s_n = kernel_times(ctxs, step, flags | M.MKV_FLAG_SCORE_TIMING, 5, dev, flags)["score"]
    kk = min(w.top_k, w.ctx)
    sel0 = torch.empty(w.batch, w.n_kv_heads, kk, dtype=torch.int32, device=dev)
    M.mkv_decode(ctxs[0].ctx, qs[0], outs[0], sel0, stream)
    torch.cuda.synchronize(dev)
    score_bytes = float(st0["payload_bytes"][0] + st0["header_bytes"] // 2)
    small = (w.batch * w.n_q_heads * 128 * (2 + 4) + 2 * w.streams * 128 * 128 * 4)
    alg = score_bytes + gathered_bytes(ctxs[0], M, sel0.cpu().numpy(), w) + small
    peak, kind = measured_peaks()
    score_us = s_ms / max(1, s_n) * 1e3
    res = {"config": workload_config(w, layers, score_bytes), "ms_per_step": ms_step,
           "value": layers * w.batch * w.ctx / (ms_step / 1e3), "unit": UNIT,
           "algorithmic_bytes_per_layer_step": alg,
           "hbm_gbs": alg * layers / (ms_step / 1e3) / 1e9,
           "hbm_frac_of_measured": alg * layers / (ms_step / 1e3) / 1e9 / peak,
           "score_kernel_us": score_us,
           "score_kernel_frac_of_measured": score_bytes / (score_us / 1e6) / 1e9 / peak,
           "prefill": {"value": w.batch * w.ctx / (statistics.median(comp) / 1e3),
                       "unit": "prefill-tokens/s per layer (K and V)",
                       "ms_per_layer_median": statistics.median(comp)},
           "kernel_us_per_layer_standalone": {k: v[0] / max(1, v[1]) * 1e3 for k, v in kt.items()},
           "strategies_K": st0["strategy_count"][0], "strategies_V": st0["strategy_count"][1],
           "payload_bytes_K": st0["payload_bytes"][0], "payload_bytes_V": st0["payload_bytes"][1]}
    if fused_ms:
        res["fused_layers"] = {"api": f"mkv_decode_layers ({layers} layers in one call)",
                               "ms_per_step": fused_ms,
                               "value": layers * w.batch * w.ctx / (fused_ms / 1e3),
                               "hbm_frac_of_measured":
                                   alg * layers / (fused_ms / 1e3) / 1e9 / peak}
    if flags & M.MKV_FLAG_BITMASK_PV:
        res["config"]["strategies"] = "SM, PV, PVB (bitmask-indexed per-vector), D"
    res["prefill"].update(prefill_roofline(w, statistics.median(comp), st0, peak))
    for m in ctxs:
        m.close()
    ctxs = []
    res["prefill"]["kernel_ms_per_layer"] = compress_kernel_ms(w, dev)
    return res


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--workload", default=W.HEADLINE_128K.name, choices=list(W.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-one-thread", action="store_true",
                    help="reference arm: skip the extra one-thread oracle timing")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling runs)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch the decode kernels without programmatic dependent launch")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the 1M-context and mixed-256K lines added to the headline line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = W.WORKLOADS[args.workload]
    if args.batch:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch, name=f"{w.name}-batch{args.batch}")
    ws, rank, local = _dist()
    try:
        if args.impl == "reference":
            run_reference(args, w, ws, rank)
        else:
            run_gpu(args, w, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
