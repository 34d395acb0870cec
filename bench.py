"""Benchmark: streaming chunk attention at the Wan-1.3B shape on GB300.

One step = one streamed chunk of the Wan-1.3B-shaped world model: 4 denoise
steps x 30 layers of chunk attention (B=1, H=12, D=128, 1536 tokens per
chunk, queries attend to their own chunk plus the 2 cached chunks of a 2-slot
ring: 4608 keys in steady state), then the 30 ring appends of the chunk's KV.
``value`` is chunks/s of the whole job (all ranks), inputs resident in HBM;
``e2e`` repeats the measurement with the step's inputs copied from pinned host
memory and its outputs copied back inside the timed region.

``--impl reference`` times the CPU oracle (plain fp64 numpy) on the same
metric, one sampled attention call per step, scaled to chunks/s.

Multi-GPU: the path has no exchange step, so N ranks run N independent
streams (weak scaling); value = chunks of all ranks / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "chunk-attention TFLOP/s & chunks/s at Wan-1.3B shape; % of roofline"
# DRAM bytes (read + write) of one attention launch of this workload, from an
# ncu capture of the same kernel build (dram__bytes_read.sum +
# dram__bytes_write.sum, small case of one layer); None once the kernel has
# changed since that capture.
ATTN_DRAM_BYTES_PER_LAUNCH = 33_106_432 + 2_048
ATTN_DRAM_BYTES_SOURCE = ("ncu --set full capture of chunk_attn_kh_kernel<128,0,0>, one Wan-1.3B call "
                          "(python bench.py --attn-only 6 --splits 0), same kernel build")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region.

    nvidia-smi starts before the warm-up and is waited for until its first
    sample arrives; it then polls every ``period_ms``.  Each sample is stamped
    with the host time it arrived, and only samples inside [begin(), end()]
    (end() is called after the closing synchronize) are summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.idx = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.t_begin = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(2.5 * self.period_ms / 1000.0)  # let the sample in flight arrive
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo = self.t_begin if self.t_begin is not None else -1e30
        hi = (self.t_end if self.t_end is not None else 1e30) + 1.5 * self.period_ms / 1000.0
        for t, ln in list(self.lines):
            if not (lo <= t <= hi):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "period_ms": self.period_ms}


def max_over_ranks(pg, values, device):
    """Each timing maxed over the ranks (the slowest rank decides the job's
    time); ``pg`` is torch.distributed or None for one process."""
    if pg is None:
        return [float(x) for x in values]
    import torch

    t = torch.tensor([float(x) for x in values], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, world, ms):
    """Units of all ranks per second over the (max-over-ranks) time ``ms``."""
    return units_per_rank * world / (ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    sab.library()
    w = synth.workload("wan13b")
    L, S = w.layers, w.steps
    B, H, D, Lc = w.B, w.H, w.D, w.Lc
    stream = torch.cuda.current_stream()
    # inputs for every (denoise step, layer), generated on the device (seeded)
    g = synth.generator(w.seed + 7919 * rank, device=str(dev))
    shape = (B, Lc, H, D)
    Q = [[synth.randn_bf16(g, shape, str(dev), rms_norm=True) for _ in range(L)] for _ in range(S)]
    Kc = [[synth.randn_bf16(g, shape, str(dev), rms_norm=True) for _ in range(L)] for _ in range(S)]
    Vc = [[synth.randn_bf16(g, shape, str(dev)) for _ in range(L)] for _ in range(S)]
    O = [[torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(L)] for _ in range(S)]
    LSE = [[torch.empty((B, H, Lc), dtype=torch.float32, device=dev) for _ in range(L)] for _ in range(S)]
    ring = sab.KVRing(L, B, H, D, Lc, w.R, device=dev)
    work = ring.workspace(args.splits) if args.splits != 1 else None
    save = max(0, S - 2)  # KV of the penultimate denoise step goes to the cache
    launches = [0]

    def chunk_step(c, ev=None, bufs=None):
        # ev: (start, end) event lists; one pair brackets the 30 back-to-back
        # attention launches of each denoise step (per-launch events would
        # themselves cost device time), so the attention kernel's average
        # launch duration is measured live, on its own stream.
        q_, k_, v_, o_, l_ = bufs if bufs is not None else (Q, Kc, Vc, O, LSE)
        for s in range(S):
            if ev is not None:
                ev[0].append(torch.cuda.Event(enable_timing=True))
                ev[1].append(torch.cuda.Event(enable_timing=True))
                ev[0][-1].record(stream)
            for l in range(L):
                sab.chunk_attention(ring.handle, l, c, q_[s][l], k_[s][l], v_[s][l], w.W, False, args.splits,
                                    w.scale, o_[s][l], l_[s][l], work, stream)
                launches[0] += 1
            if ev is not None:
                ev[1][-1].record(stream)
        for l in range(L):
            sab.kv_ring_append(ring.handle, l, c, k_[save][l], v_[save][l], stream)
            launches[0] += 1

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    chunk = 0
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            chunk_step(chunk)
            chunk += 1
        assert chunk >= 2, "warm-up must reach the steady-state window (>= 2 chunks)"
        barrier()
        launches[0] = 0
        ev = ([], [])
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        clk.begin()
        t0.record(stream)
        for _ in range(args.steps):
            chunk_step(chunk, ev)
            chunk += 1
        t1.record(stream)
        barrier()
        clk.end()
    ms = t0.elapsed_time(t1)
    gpu_launches = launches[0]
    attn_ms = [a.elapsed_time(b) / L for a, b in zip(*ev)]  # per launch
    status = sab.get_last_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device error {sab.status_string(status)}")

    # ---------------- end to end: pinned host inputs in, outputs out, per step
    # Every step copies its inputs from pinned host memory and its outputs
    # back.  The copies run on their own streams into double-buffered device
    # sets, so step i+1's inputs upload and step i-1's outputs download while
    # step i computes (the pages' asynchronous I/O); ordering is by events.
    # One contiguous pinned block per direction and per device set, so each
    # step moves its inputs in one host->device copy and its outputs in two
    # device->host copies (fewer, larger copies keep the copy engines busy).
    hQKV = torch.empty((S, L, 3) + shape, dtype=torch.bfloat16).pin_memory()
    for s_ in range(S):
        for l_ in range(L):
            hQKV[s_, l_, 0].copy_(Q[s_][l_].cpu())
            hQKV[s_, l_, 1].copy_(Kc[s_][l_].cpu())
            hQKV[s_, l_, 2].copy_(Vc[s_][l_].cpu())
    hO = torch.empty((S, L) + shape, dtype=torch.bfloat16).pin_memory()
    hL = torch.empty((S, L, B, H, Lc), dtype=torch.float32).pin_memory()
    sets = []
    for _ in range(2):
        qkv = torch.empty((S, L, 3) + shape, dtype=torch.bfloat16, device=dev)
        od = torch.empty((S, L) + shape, dtype=torch.bfloat16, device=dev)
        ld = torch.empty((S, L, B, H, Lc), dtype=torch.float32, device=dev)
        views = ([[qkv[s_, l_, 0] for l_ in range(L)] for s_ in range(S)],
                 [[qkv[s_, l_, 1] for l_ in range(L)] for s_ in range(S)],
                 [[qkv[s_, l_, 2] for l_ in range(L)] for s_ in range(S)],
                 [[od[s_, l_] for l_ in range(L)] for s_ in range(S)],
                 [[ld[s_, l_] for l_ in range(L)] for s_ in range(S)])
        sets.append((qkv, od, ld, views))
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(first_chunk, nsteps):
        comp, d2h_done = [], []
        for i in range(nsteps):
            qkv, od, ld, views = sets[i % 2]
            if i >= 2:
                up.wait_event(comp[i - 2])  # set i%2 inputs no longer read
            with torch.cuda.stream(up):
                qkv.copy_(hQKV, non_blocking=True)
            h2d_ev = torch.cuda.Event()
            h2d_ev.record(up)
            stream.wait_event(h2d_ev)
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])  # set i%2 outputs downloaded
            chunk_step(first_chunk + i, bufs=views)
            ce = torch.cuda.Event()
            ce.record(stream)
            comp.append(ce)
            down.wait_event(ce)
            with torch.cuda.stream(down):
                hO.copy_(od, non_blocking=True)
                hL.copy_(ld, non_blocking=True)
            de = torch.cuda.Event()
            de.record(down)
            d2h_done.append(de)
        stream.wait_event(d2h_done[-1])

    e2e_run(chunk, 2)
    chunk += 2
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    e2e_run(chunk, args.steps)
    chunk += args.steps
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    h2d = S * L * 3 * B * Lc * H * D * 2
    d2h = S * L * (B * Lc * H * D * 2 + B * H * Lc * 4)

    # ---------------- graph replay: one chunk step captured once with the
    # device-indexed calls (chunk index in device memory), replayed per chunk
    graph = None
    if not args.no_graph:
        d_chunk = torch.full((1,), chunk, dtype=torch.int64, device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            gs = torch.cuda.current_stream()
            for s in range(S):
                for l in range(L):
                    sab.chunk_attention_dev(ring.handle, l, d_chunk, Q[s][l], Kc[s][l], Vc[s][l], w.W, False,
                                            args.splits, w.scale, O[s][l], LSE[s][l], work, gs)
            for l in range(L):
                sab.kv_ring_append_dev(ring.handle, l, d_chunk, Kc[save][l], Vc[save][l], gs)
            sab.chunk_counter_add(d_chunk, 1, gs)
        for _ in range(max(3, args.warmup)):
            g.replay()
        barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        barrier()
        g_ms = g0.elapsed_time(g1)
        status = sab.get_last_device_error(stream)
        if status != 0:
            raise RuntimeError(f"device error {sab.status_string(status)}")
        graph = {"value": round(args.steps * ws / (g_ms / 1e3), 3), "unit": "chunks/s",
                 "ms_per_step": round(g_ms / args.steps, 4), "kernels_per_replay": S * L + L + 1}

    ms, e2e_ms = max_over_ranks(pg, [ms, e2e_ms], dev)
    nkeys = Lc * (w.W + 1)
    flops_call = 4.0 * B * H * D * Lc * nkeys
    calls = S * L * args.steps
    value = whole_job_rate(args.steps, ws, ms)
    tflops = flops_call * calls * ws / (ms / 1e3) / 1e12
    attn_avg_s = statistics.mean(attn_ms) / 1e3
    peaks, src = _peaks()
    # the kernel is timed in groups of 30 back-to-back launches (about 1 ms),
    # not in a seconds-long loop: the burst peak is its denominator
    peak = peaks["bf16_tflops"]
    achieved = flops_call / attn_avg_s / 1e12
    configs = None
    if rank == 0 and not args.no_configs:
        configs = config_records(peaks, src, stream)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        base = oracle_baselines()
        calls_per_chunk = S * L
        hb = base.pop("wan13b")
        cpu = {"value": round(hb["value"] / calls_per_chunk, 6), "unit": "chunks/s", "cores": hb["cores"],
               "kind": "oracle", "sample": hb["sample"] + f"; x{calls_per_chunk} calls per chunk",
               "single_thread": {"value": round(hb["single_thread"]["value"] / calls_per_chunk, 6),
                                 "unit": "chunks/s", "cores": 1,
                                 "sample": hb["single_thread"]["sample"] + f"; x{calls_per_chunk} calls per chunk"}}
        if configs is not None:
            for name, b in base.items():
                if name in configs:
                    configs[name]["cpu_baseline"] = b
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "chunks/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "wan13b streaming: B1 H12 D128, 1536 tokens/chunk, ring 2 slots, window current+2 "
                               "(4608 keys), 4 denoise steps x 30 layers per chunk + 30 ring appends",
                   "global_batch": ws, "seq_len": Lc, "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (30-layer ring 566 MB + 1.7 GB of per-call Q/K/V per step)"},
        "tflops": round(tflops, 2), "attention_us_per_call": round(attn_avg_s * 1e6, 2),
        "gpu_launches": gpu_launches,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": ATTN_DRAM_BYTES_PER_LAUNCH,
                     "traffic_source": ATTN_DRAM_BYTES_SOURCE,
                     "peak_source": f"bf16 dense burst, {src}"},
        "e2e": {"value": round(whole_job_rate(args.steps, ws, e2e_ms), 3), "unit": "chunks/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clk.summary(),
    }
    if graph is not None:
        line["graph_replay"] = graph
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if configs is not None:
        line["configs"] = configs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ------------------------------------------------------ per-config records
# Every workload besides the headline one, timed the way the headline is:
# CUDA events around groups of back-to-back calls on the launching stream
# (median over groups), the library's own launch choice (num_splits = 0).
# Streaming workloads rotate over enough layers that one call's inputs and
# ring rows are out of L2 when its turn comes again; the full-sequence
# workloads move more than 4x L2 per call.

def _group_us(calls, per_group, groups, stream):
    import torch

    n = len(calls)
    i = 0
    for _ in range(3 * per_group):  # warm-up
        calls[i % n]()
        i += 1
    res = []
    for _ in range(groups):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(per_group):
            calls[i % n]()
            i += 1
        b.record(stream)
        res.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) * 1e3 / per_group for x, y in res)


def _stream_setup(name, layers, sab, synth, torch):
    """A ring of ``layers`` layers filled up to the first chunk whose window
    is full, the queries (and current K/V) of that chunk per layer."""
    w = synth.workload(name)
    kv = (sab.KV_INT8K_FP8V if w.kv_int8k else sab.KV_FP8_E4M3) if w.kv_fp8 else sab.KV_BF16
    ring = sab.KVRing(layers, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=kv)
    g = synth.generator(w.seed + 17, device="cuda")
    if w.sink:
        for l in range(layers):
            ring.set_sink(l, *synth.sink_kv(w, g, "cuda"))
    steady = w.R - 1 if not w.kcur_separate else w.W
    cur = [None] * layers
    for c in range(steady + 1):
        for l in range(layers):
            q, k, v = synth.chunk_qkv(w, g, "cuda")
            if not w.kcur_separate or c < steady:
                ring.append(l, c, k, v)
            cur[l] = (q, k, v)
    return w, ring, steady, cur


def config_records(peaks, src, stream):
    import torch

    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    bf16_peak = peaks["bf16_tflops"]
    out = {}

    def rec(name, workload, us, flops, extra=None, peak=None, peak_note=None):
        tf = flops / (us * 1e-6) / 1e12
        pk = bf16_peak if peak is None else peak
        r = {"workload": workload, "us_per_call": round(us, 2), "calls_per_s": round(1e6 / us, 1),
             "tflops": round(tf, 1), "gflop_per_call": round(flops / 1e9, 3),
             "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": pk, "unit": "TFLOP/s",
                          "frac": round(tf / pk, 4),
                          "peak_source": peak_note or f"bf16 dense burst, {src}"}}
        if extra:
            r.update(extra)
        out[name] = r

    # streaming workloads: tiny (launch-bound), the long window with sink in
    # bf16, E4M3 and INT8-key caches, and the E4M3-product variant
    for name, layers in (("tiny", 1), ("long_sink", 4), ("fp8_kv", 8), ("int8k_kv", 8)):
        w, ring, c, cur = _stream_setup(name, layers, sab, synth, torch)
        nkeys = w.Lc * (w.W + 1) + (w.Lc if w.sink else 0)
        flops = 4.0 * w.B * w.H * w.D * w.Lc * nkeys
        O = [torch.empty_like(cur[l][0]) for l in range(layers)]
        L = [torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda") for _ in range(layers)]
        ws = ring.workspace(0)

        def make(l, splits, work):
            q, k, v = cur[l]
            kc, vc = (k, v) if w.kcur_separate else (None, None)
            return lambda: sab.chunk_attention(ring.handle, l, c, q, kc, vc, w.W, w.sink, splits, w.scale, O[l],
                                               L[l], work, stream)

        us = _group_us([make(l, 0, ws) for l in range(layers)], 20, 8, stream)
        desc = (f"B{w.B} H{w.H} D{w.D}, {w.Lc} tokens/chunk, {'sink + ' if w.sink else ''}ring {w.R} slots, "
                f"window current+{w.W} ({nkeys} keys)"
                + (", E4M3 K/V cache" if w.kv_fp8 and not w.kv_int8k else "")
                + (", INT8 K / E4M3 V cache" if w.kv_int8k else "")
                + f"; {layers} layer(s) rotated")
        extra = {"keys": nkeys, "splits": "library choice (0)"}
        if w.splits > 1:  # the split count the workload names, merged by LSE in-kernel
            ws8 = ring.workspace(w.splits)
            extra[f"us_per_call_splits{w.splits}"] = round(
                _group_us([make(l, w.splits, ws8) for l in range(layers)], 20, 8, stream), 2)
        rec(name, desc, us, flops, extra)
        if name == "fp8_kv":
            def make8(l, splits):
                q = cur[l][0]
                return lambda: sab.chunk_attention_fp8mma(ring.handle, l, c, q, w.W, w.sink, w.scale, O[l], L[l],
                                                          stream, num_splits=splits, workspace=ws)

            us8 = _group_us([make8(l, 0) for l in range(layers)], 20, 8, stream)
            us8_1 = _group_us([make8(l, 1) for l in range(layers)], 20, 8, stream)
            rec("fp8_kv_e4m3_mma", desc + "; Q and P rounded to E4M3, kind::f8f6f4 products", us8, flops,
                {"keys": nkeys, "splits": "library choice (0)", "us_per_call_unsplit": round(us8_1, 2)},
                peak=2 * bf16_peak, peak_note=f"fp8 dense = 2 x bf16 dense burst (nominal ratio), {src}")
        del ring, cur, O, L
        torch.cuda.empty_cache()

    # block-causal full sequence (training shape) and its gradients
    w = synth.workload("block_causal")
    g = synth.generator(w.seed, device="cuda")
    q, k, v = synth.full_sequence_qkv(w, g, "cuda")
    Lt = w.seq_chunks * w.Lc
    O = torch.empty_like(q)
    L = torch.empty((w.B, w.H, Lt), dtype=torch.float32, device="cuda")
    flops = 4.0 * w.D * _visible_pairs_block_causal(w)
    us = _group_us([lambda: sab.block_causal_attention(q, k, v, w.Lc, w.W, 0, w.scale, O, L, None, stream)], 3, 5,
                   stream)
    desc = f"B{w.B} x {Lt} tokens ({w.seq_chunks} chunks of {w.Lc}), H{w.H} D{w.D}, window {w.W}"
    rec("block_causal", desc, us, flops, {"tokens": Lt})
    do = synth.randn_bf16(g, tuple(q.shape), "cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(sab.block_causal_attention_backward_workspace(w.B, Lt, w.H), dtype=torch.uint8, device="cuda")
    us = _group_us([lambda: sab.block_causal_attention_backward(q, k, v, O, do, L, w.Lc, w.W, w.scale, dq, dk, dv,
                                                                bws, stream)], 2, 5, stream)
    rec("block_causal_backward", desc + "; dQ, dK, dV (algorithmic 10 D flops per visible pair)", us, 2.5 * flops,
        {"tokens": Lt})
    del q, k, v, O, L, do, dq, dk, dv, bws
    torch.cuda.empty_cache()

    # memory prefix (compressed-memory training shape), forward and gradients
    w = synth.workload("memory_prefix")
    q, k, v = synth.full_sequence_qkv(w, g, "cuda")
    Lt = q.shape[1]
    ml = torch.tensor(w.mem_lens, dtype=torch.int32, device="cuda")
    O = torch.empty_like(q)
    L = torch.empty((w.B, w.H, Lt), dtype=torch.float32, device="cuda")
    pairs = sum(P * P + sum(w.Lc * (P + w.Lc * (min(c, w.W) + 1)) for c in range(w.seq_chunks)) for P in w.mem_lens)
    flops = 4.0 * w.H * w.D * pairs
    desc = (f"B{w.B} x {Lt} tokens: memory of {w.mem_pad} positions ({w.mem_lens} real) + {w.seq_chunks} chunks of "
            f"{w.Lc}, H{w.H} D{w.D}, window {w.W}")
    us = _group_us([lambda: sab.memory_prefix_attention(q, k, v, w.mem_pad, ml, w.Lc, w.W, w.scale, O, L, stream)],
                   5, 5, stream)
    rec("memory_prefix", desc, us, flops, {"tokens": Lt})
    do = synth.randn_bf16(g, tuple(q.shape), "cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(sab.block_causal_attention_backward_workspace(w.B, Lt, w.H), dtype=torch.uint8, device="cuda")
    us = _group_us([lambda: sab.memory_prefix_attention_backward(q, k, v, O, do, L, w.mem_pad, ml, w.Lc, w.W, w.scale,
                                                                 dq, dk, dv, bws, stream)], 3, 5, stream)
    rec("memory_prefix_backward", desc + "; gradients", us, 2.5 * flops, {"tokens": Lt})
    del q, k, v, O, L, do, dq, dk, dv, bws
    torch.cuda.empty_cache()

    # fused Q/K RMSNorm + rotary embedding + BF16 ring append (HBM-bound)
    w = synth.workload("wan13b")
    shape = (w.B, w.Lc, w.H, w.D)
    nsets = 16  # 16 x 18.9 MB of inputs rotate: every call reads from HBM
    sets = [tuple(synth.randn_bf16(g, shape, "cuda") for _ in range(3)) for _ in range(nsets)]
    qouts = [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(nsets)]
    ring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R)
    rope = sab.RopeDesc(2, 24, 32, 44, 42, 42, 10000.0, 1e-6)
    state = {"c": 0}

    def producer(i):
        def f():
            q_, k_, v_ = sets[i]
            sab.qk_norm_rope(ring.handle, 0, state["c"], q_, k_, v_, rope, qouts[i], append=True, stream=stream)
            state["c"] += 1
        return f

    us = _group_us([producer(i) for i in range(nsets)], 32, 5, stream)
    nbytes = 6 * w.B * w.Lc * w.H * w.D * 2  # read q, k, v; write q', ring k', ring v
    gbs = nbytes / (us * 1e-6) / 1e9
    out["qk_norm_rope_append"] = {
        "workload": "one Wan-1.3B chunk (B1 H12 D128, 1536 tokens, latent grid 2x24x32, rotary bands 44/42/42), "
                    "fused append into a BF16 ring", "us_per_call": round(us, 2),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm copy, {src}"},
        "bytes_per_call": nbytes}
    del sets, qouts, ring

    # ring append alone: BF16 copy (Wan-1.3B chunk) and E4M3 absmax
    # quantisation (long-window chunk); 16 layers and 16 input sets rotate, so
    # reads and writes both leave L2
    for name, wname, kvd in (("ring_append_bf16", "wan13b", sab.KV_BF16),
                             ("ring_append_fp8", "fp8_kv", sab.KV_FP8_E4M3)):
        w = synth.workload(wname)
        shape = (w.B, w.Lc, w.H, w.D)
        sets = [tuple(synth.randn_bf16(g, shape, "cuda") for _ in range(2)) for _ in range(nsets)]
        ring = sab.KVRing(nsets, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=kvd)
        chunk = [0] * nsets

        def appender(i):
            def f():
                k_, v_ = sets[i]
                sab.kv_ring_append(ring.handle, i, chunk[i], k_, v_, stream)
                chunk[i] += 1
            return f

        us = _group_us([appender(i) for i in range(nsets)], 32, 5, stream)
        elems = 2 * w.B * w.Lc * w.H * w.D
        nbytes = elems * 2 + elems * (2 if kvd == sab.KV_BF16 else 1)  # read bf16 K, V; write the ring's codes
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {
            "workload": f"B{w.B} H{w.H} D{w.D}, {w.Lc} tokens/chunk, token-major K, V -> head-major ring slot"
                        + ("" if kvd == sab.KV_BF16 else ", E4M3 codes + per-(b, h) scales"),
            "us_per_call": round(us, 2),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm copy, {src}"},
            "bytes_per_call": nbytes}
        del sets, ring
    assert sab.get_last_device_error(stream) == 0
    return out


def run_attn_only(args):
    """Small profiling case: one layer of the Wan-1.3B stream at chunk 2
    (4608 keys), N back-to-back attention calls over 4 input sets; with
    ``--case fp8_kv_e4m3_mma`` / ``fp8_kv`` / ``int8k_kv`` N calls over the
    long-window 8-bit workload (sink + 20 slots, 8505 keys), with
    ``--case ring_append`` N BF16 and N E4M3 ring appends."""
    import torch

    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    if args.case in ("fp8_kv_e4m3_mma", "fp8_kv", "int8k_kv"):
        return run_attn_only_fp8mma(args)
    if args.case == "ring_append":
        return run_attn_only_append(args)
    if args.case == "block_causal_backward":
        return run_attn_only_backward(args)
    dev = torch.device("cuda", 0)
    w = synth.workload("wan13b")
    g = synth.generator(w.seed, device="cuda")
    shape = (w.B, w.Lc, w.H, w.D)
    sets = [tuple(synth.randn_bf16(g, shape, "cuda", rms_norm=(i < 2)) for i in range(3)) for _ in range(4)]
    ring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R, device=dev)
    ring.append(0, 0, sets[0][1], sets[0][2])
    ring.append(0, 1, sets[1][1], sets[1][2])
    ws = ring.workspace(args.splits) if args.splits != 1 else None
    O = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    LSE = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(args.attn_only):
        q, k, v = sets[i % 4]
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sab.chunk_attention(ring.handle, 0, 2, q, k, v, w.W, False, args.splits, w.scale, O, LSE, ws, stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in times]
    flops = 4.0 * w.B * w.H * w.D * w.Lc * w.Lc * (w.W + 1)
    tail = us[min(3, len(us) - 1):]
    print(json.dumps({"attn_only_calls": len(us), "us_median": statistics.median(tail),
                      "tflops_median": flops / (statistics.median(tail) * 1e-6) / 1e12, "splits": args.splits}))
    assert sab.get_last_device_error(stream) == 0


def run_attn_only_backward(args):
    """One sample of the training shape (30720 tokens, H12, D128, window 2):
    one forward, then N backward calls (delta, key-tile and query-tile
    kernels each)."""
    import torch

    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    w = synth.workload("block_causal", B=1)
    g = synth.generator(w.seed, device="cuda")
    q, k, v = synth.full_sequence_qkv(w, g, "cuda")
    do = synth.randn_bf16(g, tuple(q.shape), "cuda")
    Lt = q.shape[1]
    O = torch.empty_like(q)
    LSE = torch.empty((w.B, w.H, Lt), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sab.block_causal_attention(q, k, v, w.Lc, w.W, 0, w.scale, O, LSE, None, stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(sab.block_causal_attention_backward_workspace(w.B, Lt, w.H), dtype=torch.uint8, device="cuda")
    times = []
    for _ in range(args.attn_only):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sab.block_causal_attention_backward(q, k, v, O, do, LSE, w.Lc, w.W, w.scale, dq, dk, dv, ws, stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in times]
    tail = us[min(1, len(us) - 1):]
    print(json.dumps({"attn_only_calls": len(us), "case": args.case, "us_median": statistics.median(tail)}))
    assert sab.get_last_device_error(stream) == 0


def run_attn_only_append(args):
    """``--case ring_append``: N BF16 appends of a Wan-1.3B chunk, then N E4M3
    appends of a long-window chunk, each into its own layer of a 16-layer ring
    from 16 rotating input sets (reads and writes leave L2)."""
    import torch

    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    stream = torch.cuda.current_stream()
    g = synth.generator(7, device="cuda")
    res = {}
    for name, wname, kvd in (("bf16", "wan13b", sab.KV_BF16), ("fp8", "fp8_kv", sab.KV_FP8_E4M3)):
        w = synth.workload(wname)
        shape = (w.B, w.Lc, w.H, w.D)
        sets = [tuple(synth.randn_bf16(g, shape, "cuda") for _ in range(2)) for _ in range(16)]
        ring = sab.KVRing(16, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink, kv_dtype=kvd)
        times = []
        for i in range(args.attn_only):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sab.kv_ring_append(ring.handle, i % 16, i // 16, *sets[i % 16], stream)
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        us = [a.elapsed_time(b) * 1e3 for a, b in times]
        res[name] = statistics.median(us[min(3, len(us) - 1):])
        del sets, ring
    print(json.dumps({"attn_only_calls": args.attn_only, "case": args.case, "us_median": res}))
    assert sab.get_last_device_error(stream) == 0


def run_attn_only_fp8mma(args):
    """``--case fp8_kv_e4m3_mma``: the E4M3-product entry; ``--case fp8_kv``
    / ``int8k_kv``: the 8-bit cache through the fp16-expansion path; the
    library's split choice, over the first chunk with a full window."""
    import torch

    import streaming_attention_block_gb300 as sab
    from streaming_attention_block_gb300 import synth

    w = synth.workload("int8k_kv" if args.case == "int8k_kv" else "fp8_kv")
    g = synth.generator(w.seed, device="cuda")
    ring = sab.KVRing(1, w.B, w.H, w.D, w.Lc, w.R, has_sink=w.sink,
                      kv_dtype=sab.KV_INT8K_FP8V if args.case == "int8k_kv" else sab.KV_FP8_E4M3)
    sk, sv = synth.sink_kv(w, g, "cuda")
    ring.set_sink(0, sk, sv)
    for c in range(w.W + 1):  # first chunk with a full window
        q, k, v = synth.chunk_qkv(w, g, "cuda")
        ring.append(0, c, k, v)
    O = torch.empty_like(q)
    LSE = torch.empty((w.B, w.H, w.Lc), dtype=torch.float32, device="cuda")
    ws = ring.workspace(0)
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(args.attn_only):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if args.case == "fp8_kv_e4m3_mma":
            sab.chunk_attention_fp8mma(ring.handle, 0, w.W, q, w.W, w.sink, w.scale, O, LSE, stream, num_splits=0,
                                       workspace=ws)
        else:
            sab.chunk_attention(ring.handle, 0, w.W, q, None, None, w.W, w.sink, 0, w.scale, O, LSE, ws, stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in times]
    tail = us[min(3, len(us) - 1):]
    print(json.dumps({"attn_only_calls": len(us), "case": args.case, "us_median": statistics.median(tail)}))
    assert sab.get_last_device_error(stream) == 0


def run_sweep(args):
    """One JSON line per workload (the per-config records of the bench line,
    without the oracle timings)."""
    import torch

    peaks, src = _peaks()
    for name, r in config_records(peaks, src, torch.cuda.current_stream()).items():
        print(json.dumps(dict(sweep=name, **r)), flush=True)


# ------------------------------------------------------------------ oracle
# The CPU baseline: the oracle as it stands, timed on the host cores on a
# bounded sample of each workload (query rows are independent, so a subset of
# rows scaled by the visible query-key pairs of a full call gives its time).
# Run in child processes so that the BLAS thread count can be fixed before
# numpy loads: once with every core the process may use, once with 1 thread.

def _cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def _visible_pairs_block_causal(w):
    return w.B * w.H * sum(w.Lc * w.Lc * (min(c, w.W) + 1) for c in range(w.seq_chunks))


def _timed_rows(fn, n_rows, frac):
    """Seconds of one full oracle call whose cost grows with the query rows.
    ``fn(r)`` runs the call on the first r rows.  frac >= 1: the full call is
    timed.  Otherwise r = frac * n_rows and 2r rows are timed and the full
    call is extrapolated linearly (fixed cost per call + cost per row)."""
    if frac >= 1.0:
        t = time.perf_counter()
        fn(n_rows)
        return time.perf_counter() - t, f"all {n_rows} query rows"
    r = max(4, int(n_rows * frac))
    t = time.perf_counter()
    fn(r)
    t1 = time.perf_counter() - t
    t = time.perf_counter()
    fn(2 * r)
    t2 = time.perf_counter() - t
    slope = max(0.0, (t2 - t1) / r)
    fixed = max(0.0, t1 - slope * r)
    return fixed + slope * n_rows, f"{r} and {2 * r} of {n_rows} query rows, extrapolated linearly"


def oracle_samples(frac):
    """Seconds per full call of every workload's oracle ({name: {"seconds",
    "sample"}}); ``frac`` < 1 samples that fraction of the query rows."""
    import numpy as np

    from oracle import attention as OA
    from oracle import backward as OB
    from oracle import fp8 as OF
    from oracle import fp8mma as OM
    from oracle import int8 as OI
    from oracle.ring import ListRing
    from streaming_attention_block_gb300 import synth

    def bhld(t):
        return np.ascontiguousarray(np.transpose(t.float().numpy().astype(np.float64), (0, 2, 1, 3)))

    def deq(t, int8=False):
        x = t.float().numpy()
        if int8:
            c, sc = OI.quantize_chunk_bhld(x)
            return c.astype(np.float64) * sc.astype(np.float64)[:, :, None, None], sc
        c, sc = OF.quantize_chunk_bhld(x)
        return OF.e4m3_decode(c) * sc.astype(np.float64)[:, :, None, None], sc

    out = {}
    # Wan-1.3B streaming call at chunk 2 (4608 keys: 2 cached chunks + the current one)
    w = synth.workload("wan13b")
    gen = synth.generator(w.seed)
    ring = ListRing(w.R)
    for c in range(2):
        _, k, v = synth.chunk_qkv(w, gen)
        ring.append(c, bhld(k), bhld(v))
    q, k, v = (bhld(x) for x in synth.chunk_qkv(w, gen))
    sec, how = _timed_rows(lambda r: OA.streaming_chunk_attention(q[:, :, :r], ring, 2, k, v, w.W, False, w.scale),
                           w.Lc, frac)
    out["wan13b"] = {"seconds": sec, "sample": f"one call at chunk 2 (12 heads x 4608 keys): {how}"}
    # tiny: the whole 6-chunk stream
    w = synth.workload("tiny")
    gen = synth.generator(w.seed)
    ring = ListRing(w.R)
    el = 0.0
    for c in range(w.chunks):
        q, k, v = (bhld(x) for x in synth.chunk_qkv(w, gen))
        t = time.perf_counter()
        OA.streaming_chunk_attention(q, ring, c, k, v, w.W, False, w.scale)
        el += time.perf_counter() - t
        ring.append(c, k, v)
    out["tiny"] = {"seconds": el / w.chunks, "sample": "the whole 6-chunk stream, averaged per call"}
    # long window with sink (bf16, E4M3 and INT8-key caches): the first chunk with a full window
    for name in ("long_sink", "fp8_kv", "int8k_kv"):
        w = synth.workload(name)
        gen = synth.generator(w.seed)
        ring = ListRing(w.R)
        vsc = {}
        sk, sv = synth.sink_kv(w, gen)
        if w.kv_fp8:
            (ksd, _), (svd, vss) = deq(sk, w.kv_int8k), deq(sv)
            ring.set_sink(ksd, svd)
            vsc[OA.SINK_CHUNK] = vss
        else:
            ring.set_sink(bhld(sk), bhld(sv))
        for c in range(w.R):
            q, k, v = synth.chunk_qkv(w, gen)
            if w.kv_fp8:
                (kd, _), (vd, vss) = deq(k, w.kv_int8k), deq(v)
                ring.append(c, kd, vd)
                vsc[c] = vss
            else:
                ring.append(c, bhld(k), bhld(v))
        qb = bhld(q)
        c = w.R - 1
        sec, how = _timed_rows(lambda r: OA.streaming_chunk_attention(qb[:, :, :r], ring, c, None, None, w.W, True,
                                                                      w.scale), w.Lc, frac)
        out[name] = {"seconds": sec, "sample": f"one call at chunk {c} ({w.H} heads x 8505 keys"
                                               + (", dequantised cache" if w.kv_fp8 else "") + f"): {how}"}
        if name == "fp8_kv":  # E4M3 products: the oracle of that variant on the same cache
            K, V, kid, ksink = OA.streaming_key_set(ring, c, None, None, w.W, True)
            vs_keys = [np.array([vsc[int(i)][b, h] for i in kid], dtype=np.float64)
                       for b in range(w.B) for h in range(w.H)]

            def f8(r):
                mask = OA.chunk_visibility(np.full(r, c), kid, w.W, ksink)
                for b in range(w.B):
                    for h in range(w.H):
                        OM.head_attention(qb[b, h, :r].astype(np.float32), K[b, h], V[b, h], mask, w.scale,
                                          vs_keys[b * w.H + h])

            sec, how = _timed_rows(f8, w.Lc, frac)
            out["fp8_kv_e4m3_mma"] = {"seconds": sec, "sample": f"one call at chunk {c} (24 heads x 8505 keys, "
                                                                f"with the rounding bound): {how}"}
    # block-causal full sequence: the third chunk of a 3-chunk sequence has
    # the steady-state key set (4608 keys); scaled by visible pairs
    w = synth.workload("block_causal")
    w3 = synth.workload("block_causal", B=1, seq_chunks=3)
    q, k, v = synth.full_sequence_qkv(w3, synth.generator(w.seed))
    qf, kf, vf = (x.float().numpy() for x in (q, k, v))
    rows = np.arange(2 * w.Lc, 3 * w.Lc)
    sec, how = _timed_rows(lambda r: OA.block_causal_attention(qf, kf, vf, w.Lc, w.W, w.scale, rows=rows[:r]),
                           w.Lc, frac)
    pairs = w.H * w.Lc * 3 * w.Lc
    out["block_causal"] = {"seconds": sec * _visible_pairs_block_causal(w) / pairs,
                           "sample": f"the 1536 rows of one steady-state chunk x 12 heads x 4608 keys ({how}), "
                                     f"scaled by visible pairs to B2 x 30720 tokens"}
    # gradients: one head of a 3-chunk sequence, chunk by chunk over the keys
    # each chunk sees; scaled by visible pairs
    do = synth.randn_bf16(synth.generator(w.seed + 1), tuple(q.shape)).float().numpy()
    n_tok = 3 * w.Lc
    t = time.perf_counter()
    OB.block_causal_attention_backward_rows(qf, kf, vf, do, w.Lc, w.W, w.scale, 0, 0, np.arange(n_tok),
                                            np.arange(n_tok))
    el = time.perf_counter() - t
    pairs = w.Lc * w.Lc * (1 + 2 + 3)
    out["block_causal_backward"] = {"seconds": el * _visible_pairs_block_causal(w) / pairs,
                                    "sample": f"dQ, dK, dV of every row of one head of a {n_tok}-token sequence, "
                                              f"scaled by visible pairs to B2 x 30720 tokens x 12 heads"}
    return out


def oracle_baselines(seconds_budget_hint=None):
    """All-core and single-thread oracle timings ({name: cpu_baseline dict}),
    each from a child process with its BLAS thread count fixed."""
    res = {}
    ncores = _cpu_threads()
    runs = []
    for threads, frac in ((ncores, 1.0), (1, 0.125)):
        env = dict(os.environ)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[var] = str(threads)
        env["CUDA_VISIBLE_DEVICES"] = ""
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-samples", str(frac)], env=env,
                           capture_output=True, text=True, timeout=900)
        if r.returncode != 0:
            raise RuntimeError(f"oracle sample run failed:\n{r.stderr[-2000:]}")
        runs.append((threads, json.loads(r.stdout.strip().splitlines()[-1])))
    (nc, full), (_, single) = runs
    for name, d in full.items():
        one = single[name]
        res[name] = {"value": round(1.0 / d["seconds"], 6), "unit": "calls/s", "cores": nc, "kind": "oracle",
                     "sample": d["sample"] + " (numpy fp64; BLAS threads = cores, elementwise numpy single-threaded)",
                     "single_thread": {"value": round(1.0 / one["seconds"], 6), "unit": "calls/s", "cores": 1,
                                       "sample": one["sample"]}}
    return res


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    from oracle import attention as OA
    from oracle.ring import ListRing
    from streaming_attention_block_gb300 import synth

    w = synth.workload("wan13b")
    gen = synth.generator(w.seed)
    ring = ListRing(w.R)
    data = []
    for c in range(3):
        q, k, v = synth.chunk_qkv(w, gen)
        data.append(tuple(np.transpose(x.float().numpy().astype(np.float64), (0, 2, 1, 3)) for x in (q, k, v)))
    ring.append(0, data[0][1], data[0][2])
    ring.append(1, data[1][1], data[1][2])
    q, k, v = data[2]
    # each step: a quarter of the query rows of one steady-state attention
    # call (rows are independent), i.e. 1/480 of a chunk
    rows = w.Lc // 4
    sub = [q[:, :, i * rows:(i + 1) * rows] for i in range(4)]
    for i in range(args.warmup):
        OA.streaming_chunk_attention(sub[i % 4][:, :, :16], ring, 2, k, v, w.W, False, w.scale)
    t = time.perf_counter()
    for i in range(args.steps):
        OA.streaming_chunk_attention(sub[i % 4], ring, 2, k, v, w.W, False, w.scale)
    el = time.perf_counter() - t
    per_step = el / args.steps
    per_chunk = per_step * 4 * w.steps * w.layers
    value = 1.0 / per_chunk
    cpu = {"value": round(value, 6), "unit": "chunks/s", "cores": _cpu_threads(), "kind": "oracle",
           "sample": f"{args.steps} steps of 384 query rows x 12 heads x 4608 keys (fp64), {per_step:.2f} s each; "
                     f"scaled x{4 * w.steps * w.layers} to one chunk (4 steps x 30 layers x 1536 rows)"}
    line = {"metric": METRIC, "value": round(value, 6), "unit": "chunks/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "wan13b streaming: B1 H12 D128, 1536 tokens/chunk, ring 2 slots, window current+2 "
                                   "(4608 keys); oracle sample per step, scaled to chunks/s",
                       "global_batch": 1, "seq_len": w.Lc, "parallelism": "cpu"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "chunks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config records")
    ap.add_argument("--oracle-samples", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--no-graph", action="store_true", help="skip the graph-replay measurement")
    ap.add_argument("--splits", type=int, default=0, help="KV splits per attention call (0: library's choice)")
    ap.add_argument("--sweep", action="store_true", help="time one attention call of every workload")
    ap.add_argument("--case", default="wan13b",
                    choices=["wan13b", "fp8_kv_e4m3_mma", "fp8_kv", "int8k_kv", "ring_append", "block_causal_backward"],
                    help="workload of --attn-only")
    ap.add_argument("--attn-only", type=int, default=0, metavar="N",
                    help="profiling case: N steady-state attention calls on one layer, then exit")
    args = ap.parse_args()
    if args.oracle_samples is not None:  # child process of oracle_baselines()
        print(json.dumps(oracle_samples(args.oracle_samples)), flush=True)
        return
    if args.attn_only:
        return run_attn_only(args)
    if args.sweep:
        return run_sweep(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
