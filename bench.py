#!/usr/bin/env python
"""Benchmark of the CSA2 FP4 compressed global KV cache decode step on B300.

Default workload: 64 sequences x 131072 context tokens, 4-layer mode schedule
Full -> Reindex -> Reuse -> Reuse, candidate pool 8192, top-K 2048, one decode query
per sequence.  Metric: decode queries/s per layer (query tokens x layers / time), with
the achieved HBM bandwidth of the dominant kernel against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU; ranks are independent replicas of the
workload (weak scaling, no collective on the data path).  `--impl reference` times the
CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 FP4-KV decode queries/s per layer; achieved HBM GB/s vs B300 peak"
UNIT = "queries/s per layer"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


# ------------------------------------------------------------------ helpers ------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms while running; each sample
    is stamped on arrival, and the summary keeps the samples between mark() and stop()
    (the timed loops), or all of them when mark() was not called."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None
        self._mark = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self):
        """Start of the timed loops: samples before this are not summarised."""
        self._mark = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        t_end = time.monotonic()
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t_lo = self._mark if self._mark is not None else -1e30
        for ts, ln in self.lines:
            if ts < t_lo or ts > t_end:
                continue
            parts = [p.strip() for p in ln.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("CSA2_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def flush_l2(buf, k):
    """Evict L2 before a timed call: write a 256 MB buffer (larger than the 126 MB L2), then
    read it back, so that L2 holds only clean lines of the buffer and the timed call pays
    no write-back of the flush's own dirty lines."""
    import torch
    buf.fill_(k & 0xFF)
    buf.view(torch.int64).sum()


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def shard_sequences(num_seqs: int, world: int, rank: int, scaling: str = "weak"):
    """Sequences this rank serves.  Weak scaling: every rank serves a full, independent
    replica of the batch.  Strong scaling: the batch is split into contiguous shards."""
    if scaling == "weak" or world == 1:
        return np.arange(num_seqs)
    per = (num_seqs + world - 1) // world
    return np.arange(rank * per, min(num_seqs, (rank + 1) * per))


# ------------------------------------------------------------------ algorithmic bytes --

def decode_config(wl, mx: bool, world: int, schedule: str = "parallel") -> dict:
    """The `config` of a decode-workload line; the reference arm prints the same one."""
    return {"workload": wl.name + ("_mxfp4" if mx else ""), "num_seqs": int(len(wl.seq_lens)),
            "context_tokens": int(wl.seq_lens.max()), "query_tokens": wl.num_q,
            "layers": len(wl.schedule), "schedule": "".join("FRU"[m] for m in wl.schedule),
            "pool": wl.pool_size, "topk": wl.topk,
            "l2": "no flush: every step streams %.2f GB of indexer keys (> 126 MB L2)"
                  % (full_index_bytes(wl) / 1e9),
            "launch": ("CUDA graph of the step's libcsa2 calls, index calls in layer order "
                       "and attention calls on 4 side branches after their source layer's "
                       "index call" if schedule == "parallel" else
                       "CUDA graph of the step's libcsa2 calls in layer order")
                      + "; per-mode times from per-call graphs",
            "parallelism": f"replicas x{world}"}


def write_config(ww, world: int) -> dict:
    """The `config` of a write-path line (prefill write or decode-time append)."""
    append = ww.T <= 128
    l2 = ("flushed before every call (256 MB written, then read back): the %.0f MB of weights fit in L2"
          % (ww.n_out * ww.d_model * 2 / 1e6)) if append else \
        "no flush: H is %.0f MB (> 126 MB L2)" % (ww.T * ww.d_model * 2 / 1e6)
    return {"workload": ww.name, "tokens": ww.T, "d_model": ww.d_model,
            "latent_projections": ww.n_kv_proj, "key_projections": ww.n_idx_proj,
            "l2": l2, "parallelism": f"replicas x{world}"}


def pages_config(world: int, n: int = 16384, rec: int = 34816) -> dict:
    """The `config` of the page-export line (every page of the 64 x 16384-token cache)."""
    return {"workload": "page_export_64x16384", "pages": n, "record_bytes": rec,
            "l2": "no flush: %.0f MB of pages per step (> 126 MB L2)" % (n * rec / 1e6),
            "parallelism": f"replicas x{world}"}


def host_cpu() -> dict:
    """CPU model and logical core count of this host (for every CPU timing)."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"cpu_model": model, "nproc": os.cpu_count() or 1}


def full_index_bytes(wl) -> int:
    """Bytes a Full-layer index step must move: every context key row (256 B) of every
    query's sequence (read once per sequence), the indexer queries, top-K and pool."""
    per_seq = wl.seq_lens.astype(np.int64) * 256
    return int(per_seq.sum() + wl.num_q * (4 * 128 * 2 + 4 * wl.topk + 4 * wl.pool_size))


def reindex_bytes(wl) -> int:
    return int(wl.num_q * (wl.pool_size * (4 + 256) + 4 * 128 * 2 + 4 * wl.topk))


def attn_bytes(wl) -> int:
    """Selected FP4 rows (256 B codes + 32 B scales), q, indices, out and lse."""
    return int(wl.num_q * (wl.topk * (288 + 4) + 16 * 512 * 2 + 16 * 512 * 4 + 16 * 4))


# ------------------------------------------------------------------ ours ---------

def run_ours(args, world, rank, local):
    import torch
    import csa2_inputs as gen
    import fp4_compressed_sparse_03_b300 as csa2
    from fp4_compressed_sparse_03_b300.decode import DecodeStep
    from fp4_compressed_sparse_03_b300.workload import all_queries_host, fill_decode_cache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of(args.workload)
    mx = args.workload.endswith("_mx")  # the MXFP4 variant of the cache and read path
    cache = fill_decode_cache(wl, device=dev, mx=mx)
    q_idx_h, q_h = all_queries_host(wl)
    q_idx = torch.from_numpy(q_idx_h.view(np.int16)).to(dev)
    q = torch.from_numpy(q_h.view(np.int16)).to(dev)
    mq = int(wl.q_per_seq.max())
    step = DecodeStep(cache, wl.q_seq, wl.schedule, wl.pool_size, wl.topk, mq)
    L = len(wl.schedule)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        step.run(q_idx, q)
    torch.cuda.synchronize(dev)
    status, bits = csa2.csa2_read_status(step.dev_status)
    if status != csa2.CSA2_OK:
        raise RuntimeError(f"device status {bits:#x} after warm-up")

    # The step is replayed as a CUDA graph of the same libcsa2 launches, so the device
    # time is not paced by per-call host work (about 12 calls per step).  In the parallel
    # schedule a layer's attention call overlaps the next layers' index calls.
    par = args.step_schedule == "parallel"
    g_step = step.capture(q_idx, q, parallel=par)
    g_call = step.capture_calls(q_idx, q)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    full_layers = [l for l, m in enumerate(wl.schedule) if m == csa2.CSA2_FULL]
    re_layers = [l for l, m in enumerate(wl.schedule) if m == csa2.CSA2_REINDEX]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        g_step.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    # per-call times: the per-call graphs with events between them, on the same stream
    K1 = max(1, min(K, 50))
    ev = {(k, l, w): torch.cuda.Event(enable_timing=True)
          for k in range(K1) for l in range(L) for w in ("i0", "i1", "a1")}
    for k in range(K1):
        for l in range(L):
            ev[(k, l, "i0")].record(stream)
            if (l, "index") in g_call:
                g_call[(l, "index")].replay()
            ev[(k, l, "i1")].record(stream)
            g_call[(l, "attn")].replay()
            ev[(k, l, "a1")].record(stream)
    torch.cuda.synchronize(dev)
    # per-layer attention with L2 flushed before each layer (a 256 MB buffer written and read): the
    # Reuse layers' attention otherwise re-reads rows the previous layer just gathered
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    K3 = max(1, min(K, 20))
    evc = {(k, l, w): torch.cuda.Event(enable_timing=True)
           for k in range(K3) for l in range(L) for w in (0, 1)}
    for k in range(K3):
        for l in range(L):
            flush_l2(flush, k * L + l)
            evc[(k, l, 0)].record(stream)
            g_call[(l, "attn")].replay()
            evc[(k, l, 1)].record(stream)
    torch.cuda.synchronize(dev)
    del flush
    barrier(world)
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_step = reduce_max(ms_total / K, world, dev)
    status, bits = csa2.csa2_read_status(step.dev_status)
    if status != csa2.CSA2_OK:
        raise RuntimeError(f"device status {bits:#x} after timed steps")

    def avg(l, a, b):
        return float(np.mean([ev[(k, l, a)].elapsed_time(ev[(k, l, b)]) for k in range(K1)]))

    full_ms = float(np.mean([avg(l, "i0", "i1") for l in full_layers]))
    re_ms = float(np.mean([avg(l, "i0", "i1") for l in re_layers])) if re_layers else 0.0
    attn_ms = float(np.mean([avg(l, "i1", "a1") for l in range(L)]))
    attn_layer_ms = [round(avg(l, "i1", "a1"), 4) for l in range(L)]
    attn_cold_ms = [round(float(np.mean([evc[(k, l, 0)].elapsed_time(evc[(k, l, 1)]) for k in range(K3)])), 4)
                    for l in range(L)]
    units = wl.num_q * L * world
    value = units / (ms_step / 1e3)

    hbm_peak, tc_peak, peak_src = load_peaks()
    fb = full_index_bytes(wl)
    achieved = fb / (full_ms / 1e3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        t = tj.get(args.workload)
        if t and t.get("kernel_hash") == kernel_hash():
            traffic = t.get("bytes_per_launch")

    # ---- end to end: every step's queries go up from pinned host memory and its outputs
    # come back to pinned host memory.  Two buffer sets (two DecodeSteps over the same
    # cache) and separate upload / download streams let the copies of neighbouring steps
    # overlap the compute of this one. ----
    q_idx_pin = torch.from_numpy(q_idx_h.view(np.int16)).pin_memory()
    q_pin = torch.from_numpy(q_h.view(np.int16)).pin_memory()
    idx_layers = [l for l, m in enumerate(wl.schedule) if m != csa2.CSA2_REUSE]
    step_b = DecodeStep(cache, wl.q_seq, wl.schedule, wl.pool_size, wl.topk, mq)
    q_idx_b, q_b = q_idx.clone(), q.clone()
    step_b.run(q_idx_b, q_b)
    torch.cuda.synchronize(dev)
    sets = [(step, q_idx, q, g_step), (step_b, q_idx_b, q_b, step_b.capture(q_idx_b, q_b, parallel=par))]
    out_pin = [torch.empty(step.out.shape, dtype=torch.float32).pin_memory() for _ in sets]
    lse_pin = [torch.empty(step.lse.shape, dtype=torch.float32).pin_memory() for _ in sets]
    h2d = sum(q_idx_pin[l].numel() * 2 for l in idx_layers) + q_pin.numel() * 2
    d2h = out_pin[0].numel() * 4 + lse_pin[0].numel() * 4
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_done = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]
    K2 = max(1, min(K, args.e2e_steps))
    barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for k in range(K2):
        sk = k % 2
        st_k, qi_k, q_k, g_k = sets[sk]
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(ev_done[sk])  # step k - 2 has finished reading these inputs
            for l in idx_layers:
                qi_k[l].copy_(q_idx_pin[l], non_blocking=True)
            q_k.copy_(q_pin, non_blocking=True)
            ev_in[sk].record(up)
        stream.wait_event(ev_in[sk])
        if k >= 2:
            stream.wait_event(ev_out[sk])  # step k - 2's outputs have been copied out
        g_k.replay()
        ev_done[sk].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[sk])
            out_pin[sk].copy_(st_k.out, non_blocking=True)
            lse_pin[sk].copy_(st_k.lse, non_blocking=True)
            ev_out[sk].record(down)
    e1.record(down)
    torch.cuda.synchronize(dev)
    wall_e2e = (time.perf_counter() - w0) / K2 * 1e3
    barrier(world)
    ms_e2e = reduce_max(max(e0.elapsed_time(e1) / K2, wall_e2e), world, dev)
    for st_k, *_ in sets:
        status, bits = csa2.csa2_read_status(st_k.dev_status)
        if status != csa2.CSA2_OK:
            raise RuntimeError(f"device status {bits:#x} after end-to-end steps")
    e2e_value = units / (ms_e2e / 1e3)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_sample, mx)

    launches_per_step = count_launches(wl, step)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("fp4-e2m1/e8m0-per-32 (MXFP4) kv" if mx else "fp4-e2m1/e4m3 kv") +
                 ", bf16 keys+queries, f32 accumulate",
        "data": "synthetic (seeded counter-based generator)",
        "config": decode_config(wl, mx, world, args.step_schedule),
        "per_mode_ms": {"full_index": round(full_ms, 4), "reindex": round(re_ms, 4),
                        "attention": round(attn_ms, 4), "attention_per_layer": attn_layer_ms,
                        "attention_cold_per_layer": attn_cold_ms,
                        "attention_cold_note": "each layer's attention replayed alone after a "
                                               "256 MB L2 flush (written, then read back)"},
        "roofline": {"bound": "hbm", "kernel": "csa2_index(FULL) call: group_prefix_kernel + score_pages_kernel + select_cta_kernel",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": fb, "traffic": traffic},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": K2,
                "pipelining": "two buffer sets; uploads and downloads of neighbouring steps "
                              "overlap the compute"},
        "gpu_launches": int(launches_per_step * K),
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_write(args, world, rank, local):
    """The CED write path alone: one csa2_kv_write per step.
    ced_write: the whole prefill write (H [32768, 4096] bf16 times 20 latent + 20
    indexer-key projections, quantised on write); roofline the tensor pipe, 2 T d n_out
    flops per call.
    decode_append: the new token of each of 64 sequences through the same projections;
    roofline HBM, the 105 MB of projection weights streamed per call.  The weights fit
    in L2, so L2 is flushed (a 256 MB buffer written, then read) before every timed call, and each
    call is timed by its own events."""
    import torch
    import csa2_inputs as gen
    import fp4_compressed_sparse_03_b300 as csa2
    from fp4_compressed_sparse_03_b300.workload import fill_write_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    append = args.workload == "decode_append"
    ww = gen.config_append() if append else gen.config_write()
    H, Wt, slots = fill_write_inputs(ww, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if append else None
    num_slots = ww.num_pages * 64
    codes = torch.empty((ww.n_kv_proj, num_slots, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((ww.n_kv_proj, num_slots, 32), dtype=torch.uint8, device=dev)
    keys = torch.empty((ww.n_idx_proj, num_slots, 128), dtype=torch.int16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(h=H, sl=slots):
        csa2.check(csa2.csa2_kv_write(h, Wt, codes, scales, keys, ww.T, ww.d_model, ww.n_kv_proj,
                                      ww.n_idx_proj, sl, num_slots, st, stream))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(K):
        if flush is not None:
            flush_l2(flush, k)
        evs[k][0].record(stream)
        call()
        evs[k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    status, bits = csa2.csa2_read_status(st)
    if status != csa2.CSA2_OK:
        raise RuntimeError(f"device status {bits:#x} after timed steps")
    per_call = np.array([a.elapsed_time(b) for a, b in evs])
    kern_ms = float(np.mean(per_call))
    # with L2 flushes between calls the step is the call itself
    ms_step = reduce_max(kern_ms if append else t0.elapsed_time(t1) / K, world, dev)
    units = ww.T * world
    value = units / (ms_step / 1e3)
    flops = 2.0 * ww.T * ww.d_model * ww.n_out
    hbm_peak, tc_peak, peak_src = load_peaks()
    achieved = flops / (kern_ms / 1e3) / 1e12
    # algorithmic bytes of one call: weights and H read, codes + scales + keys written
    out_row = ww.n_kv_proj * (256 + 32) + ww.n_idx_proj * 128 * 2
    abytes = ww.n_out * ww.d_model * 2 + ww.T * ww.d_model * 2 + ww.T * (out_row + 4)
    achieved_gbs = abytes / (kern_ms / 1e3) / 1e9

    # end to end: H from pinned host memory in, every code, scale and key back out (for
    # decode_append the step's result is the new rows only: gathered, then read back)
    H_pin = torch.empty(H.shape, dtype=H.dtype).pin_memory()
    H_pin.copy_(H)
    rows = ww.T if append else codes.shape[1]
    c_pin = torch.empty((codes.shape[0], rows, 256), dtype=codes.dtype).pin_memory()
    s_pin = torch.empty((scales.shape[0], rows, 32), dtype=scales.dtype).pin_memory()
    k_pin = torch.empty((keys.shape[0], rows, 128), dtype=keys.dtype).pin_memory()
    H_dev = torch.empty_like(H)
    sl_long = slots.long()
    if append:  # first use of the gathers outside the timed region
        c_pin.copy_(codes.index_select(1, sl_long))
    K2 = max(1, min(K, args.e2e_steps, 10))
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for _ in range(K2):
        if flush is not None:
            flush_l2(flush, 7)
        H_dev.copy_(H_pin, non_blocking=True)
        call(H_dev)
        if append:
            c_pin.copy_(codes.index_select(1, sl_long), non_blocking=True)
            s_pin.copy_(scales.index_select(1, sl_long), non_blocking=True)
            k_pin.copy_(keys.index_select(1, sl_long), non_blocking=True)
        else:
            c_pin.copy_(codes, non_blocking=True)
            s_pin.copy_(scales, non_blocking=True)
            k_pin.copy_(keys, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = (time.perf_counter() - w0) / K2 * 1e3
    ms_e2e = reduce_max(max(e0.elapsed_time(e1) / K2, wall), world, dev)
    h2d = H.numel() * 2
    d2h = c_pin.numel() + s_pin.numel() + k_pin.numel() * 2

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_write(ww, args.cpu_sample)
    if append:
        roof = {"bound": "hbm", "kernel": "csa2_kv_write: kv_write_kernel",
                "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm_peak, 4), "peak_source": peak_src + " HBM copy",
                "algorithmic_bytes_per_launch": int(abytes), "traffic": None}
    else:
        roof = {"bound": "tensor", "kernel": "csa2_kv_write: kv_write_kernel",
                "achieved": round(achieved, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tc_peak, 4), "peak_source": peak_src + " bf16 burst",
                "algorithmic_flops_per_launch": flops, "traffic": None}
    cfg = write_config(ww, world)
    if append:  # the mean is the reported time; the spread of the per-call event times beside it
        cfg["per_call_us"] = {"mean": round(float(np.mean(per_call)) * 1e3, 2),
                              "median": round(float(np.median(per_call)) * 1e3, 2),
                              "min": round(float(np.min(per_call)) * 1e3, 2)}
    line = {
        "metric": ("decode-time append: new tokens/s projected and quantised into the paged cache"
                   if append else "CED write path: tokens/s projected and quantised on write"),
        "value": round(value, 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 operands, f32 accumulate, fp4-e2m1/e4m3 + bf16 out",
        "data": "synthetic (seeded counter-based generator)",
        "config": cfg,
        "roofline": roof,
        "e2e": {"value": round(units / (ms_e2e / 1e3), 1), "unit": "tokens/s",
                "l2_flush": ("each timed step includes the 256 MB L2 flush (written and read back, about 80 us)"
                             if append else "none"),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": K2},
        "gpu_launches": K,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_pages(args, world, rank, local):
    """Persistent KV tier: export every page of the 64 x 16384-token cache (16384 pages of
    34816 B: codes, scales, keys) per step with csa2_export_pages.  The roofline is HBM:
    each record is read once and written once.  End to end adds the copy of the packed
    pages into pinned host memory (the host tier)."""
    import torch
    import fp4_compressed_sparse_03_b300 as csa2
    from fp4_compressed_sparse_03_b300.workload import fill_decode_cache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of("decode_short")
    cache = fill_decode_cache(wl, device=dev)
    lay = wl.layout
    ids = np.concatenate([lay.page_table[b, :-(-int(n) // 64)] for b, n in enumerate(lay.seq_lens)])
    ids_d = torch.as_tensor(ids.astype(np.int32), device=dev)
    n = len(ids)
    rec = csa2.csa2_page_export_bytes(32)
    packed = torch.empty(n * rec, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        csa2.check(csa2.csa2_export_pages(cache.codes[0], cache.scales[0], cache.keys[0], 32,
                                          cache.num_pages, ids_d, n, packed, st, stream))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    K = args.steps
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        call()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    status, bits = csa2.csa2_read_status(st)
    if status != csa2.CSA2_OK:
        raise RuntimeError(f"device status {bits:#x} after timed steps")
    ms_step = reduce_max(t0.elapsed_time(t1) / K, world, dev)
    tokens = n * 64 * world
    value = tokens / (ms_step / 1e3)
    hbm_peak, _, peak_src = load_peaks()
    abytes = 2 * n * rec + n * 4
    achieved = abytes / (t0.elapsed_time(t1) / K / 1e3) / 1e9
    host_buf = torch.empty(n * rec, dtype=torch.uint8).pin_memory()
    K2 = max(1, min(K, args.e2e_steps, 5))
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for _ in range(K2):
        call()
        host_buf.copy_(packed, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = reduce_max(max(e0.elapsed_time(e1) / K2, (time.perf_counter() - w0) / K2 * 1e3),
                        world, dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_pages(args.cpu_sample)
    line = {
        "metric": "persistent KV tier: tokens/s of cache pages exported (codes, scales, keys)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8 (byte copy)",
        "data": "synthetic (seeded counter-based generator)",
        "config": pages_config(world, n, rec),
        "roofline": {"bound": "hbm", "kernel": "csa2_export_pages: page_copy_kernel",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src + " HBM copy",
                     "algorithmic_bytes_per_launch": int(abytes), "traffic": None},
        "e2e": {"value": round(tokens / (ms_e2e / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": int(n * rec), "steps": K2},
        "gpu_launches": K,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


CHUNK_METRIC = ("multi-query sparse attention: query tokens/s, 4 draft queries per sequence "
                "with their own top-K")
CHUNK_SHARED = 0.75  # default fraction of each draft query's selection common to its chunk


def chunk_inputs(shared=CHUNK_SHARED):
    """The draft-token chunk workload: the 64 x 16384-token cache, 4 draft queries per
    sequence, each with top-2048 entries of which `shared` (75 % by default) are common to
    the sequence's four (host arrays: q bf16 bits [256, 16, 512], idx int32 [256, 2048],
    q_seq int32 [256])."""
    import csa2_inputs as gen
    wl = workload_of("decode_short")
    B, G, K = len(wl.seq_lens), 4, wl.topk
    idx = np.concatenate([gen.overlapping_index_sets(wl.seed, b, int(wl.seq_lens[b]), K, G,
                                                     shared) for b in range(B)])
    q = gen.q_rows(wl.seed, 7, np.arange(B * G))
    q_seq = np.repeat(np.arange(B, dtype=np.int32), G)
    return wl, q, idx, q_seq, G, K


def run_chunk(args, world, rank, local):
    """Multi-query sparse attention in dense-contraction form: the union of each chunk's
    selections gathered and dequantised once for its 4 queries (csa2_sparse_attn_chunked),
    timed per call with L2 flushed before each (the selected rows, ~66 MB, fit in L2); the
    per-query path on the same arguments is timed the same way for comparison.  Roofline:
    HBM, on the distinct rows the chunks select plus q, indices and outputs."""
    import torch
    import fp4_compressed_sparse_03_b300 as csa2
    from fp4_compressed_sparse_03_b300.workload import fill_decode_cache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl, q, idx, q_seq, G, K = chunk_inputs(args.shared)
    cache = fill_decode_cache(wl, device=dev)
    nq = len(q_seq)
    q_d = torch.as_tensor(q.view(np.int16), device=dev)
    idx_d = torch.as_tensor(idx, device=dev)
    qs_d = torch.as_tensor(q_seq, device=dev)
    out = torch.empty((nq, 16, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((nq, 16), dtype=torch.float32, device=dev)
    ws = torch.empty(csa2.csa2_chunk_attn_workspace_size(nq, G, K), dtype=torch.uint8, device=dev)
    ws_pq = torch.empty(max(16, csa2.csa2_attn_workspace_size(nq, K)), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    scale = float(np.float32(1.0 / np.sqrt(512.0)))

    def chunked(qa=q_d, ia=idx_d):
        csa2.check(csa2.csa2_sparse_attn_chunked(qa, cache.codes[0], cache.scales[0], ia,
                                                 cache.pages, out, lse, nq, qs_d, G, K, scale, ws,
                                                 None, st, stream), "chunked attention")

    def per_query():
        csa2.check(csa2.csa2_sparse_attn(q_d, cache.codes[0], cache.scales[0], idx_d, cache.pages,
                                         out, lse, nq, qs_d, K, scale, ws_pq, None, st, stream),
                   "attention")

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for k in range(n):
            flush_l2(flush, k)
            evs[k][0].record(stream)
            fn()
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    for _ in range(args.warmup):
        chunked()
        per_query()
    torch.cuda.synchronize(dev)
    Kst = args.steps
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    ms_call = timed(chunked, Kst)
    ms_pq = timed(per_query, Kst)
    barrier(world)
    clk = clocks.stop()
    status, bits = csa2.csa2_read_status(st)
    if status != csa2.CSA2_OK:
        raise RuntimeError(f"device status {bits:#x} after timed steps")
    ms_step = reduce_max(ms_call, world, dev)
    value = nq * world / (ms_step / 1e3)
    # distinct rows the chunks select (the union per sequence), and what every query moves
    union = sum(np.unique(idx[c * G:(c + 1) * G][idx[c * G:(c + 1) * G] >= 0]).size
                for c in range(nq // G))
    abytes = union * 288 + nq * (16 * 512 * 2 + K * 4 + 16 * 512 * 4 + 16 * 4)
    hbm_peak, _, peak_src = load_peaks()
    achieved = abytes / (ms_call / 1e3) / 1e9

    # end to end: q and indices from pinned host memory in, outputs and lse back out
    q_pin = torch.empty(q_d.shape, dtype=q_d.dtype).pin_memory()
    q_pin.copy_(q_d)
    i_pin = torch.empty(idx_d.shape, dtype=idx_d.dtype).pin_memory()
    i_pin.copy_(idx_d)
    o_pin = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    l_pin = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_dev, i_dev = torch.empty_like(q_d), torch.empty_like(idx_d)
    K2 = max(1, min(Kst, args.e2e_steps, 20))
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for _ in range(K2):
        flush_l2(flush, 3)
        q_dev.copy_(q_pin, non_blocking=True)
        i_dev.copy_(i_pin, non_blocking=True)
        chunked(q_dev, i_dev)
        o_pin.copy_(out, non_blocking=True)
        l_pin.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = reduce_max(max(e0.elapsed_time(e1) / K2, (time.perf_counter() - w0) / K2 * 1e3),
                        world, dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_chunk(args.cpu_sample, args.shared)
    line = {
        "metric": CHUNK_METRIC, "value": round(value, 1), "unit": "queries/s", "n_gpus": world,
        "steps": Kst, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4-e2m1/e4m3 kv, bf16 queries, f16 operands, f32 accumulate",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": "draft_chunk_64x4x16384", "num_seqs": len(wl.seq_lens),
                   "queries_per_chunk": G, "context_tokens": int(wl.seq_lens.max()), "topk": K,
                   "shared_fraction": args.shared, "union_rows": int(union),
                   "l2": "flushed before every call (256 MB written, then read back): the selected rows fit in L2",
                   "per_query_path_ms": round(ms_pq, 4), "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": "csa2_sparse_attn_chunked call: chunk_union_kernel + "
                               "chunk_attn_kernel + attn_combine_kernel",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src + " HBM copy",
                     "algorithmic_bytes_per_launch": int(abytes), "traffic": None},
        "e2e": {"value": round(nq * world / (ms_e2e / 1e3), 1), "unit": "queries/s",
                "l2_flush": "each timed step includes the 256 MB L2 flush (written and read back, about 80 us)",
                "h2d_bytes_per_step": int(q_d.numel() * 2 + idx_d.numel() * 4),
                "d2h_bytes_per_step": int(out.numel() * 4 + lse.numel() * 4), "steps": K2},
        "gpu_launches": 3 * Kst,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def cpu_baseline_chunk(sample_queries: int, shared: float = CHUNK_SHARED):
    """The oracle (gather, dequantise, double-precision attention per query) on the first
    `sample_queries` draft queries of the chunk workload; the cache rows of their
    sequences are generated and quantised before the clock starts."""
    import csa2_inputs as gen
    import oracle
    from csa2_inputs import native
    wl, q, idx, q_seq, G, K = chunk_inputs(shared)
    n = max(1, min(sample_queries, len(q_seq)))
    gains = gen.latent_gains(wl.seed, 0)
    rows = {}
    for b in sorted(set(int(x) for x in q_seq[:n])):
        rows[b] = oracle.quantize(native.latent_rows_host(wl.seed, 0, b, 0, int(wl.seq_lens[b]), gains))
    scale = float(np.float32(1.0 / np.sqrt(512.0)))
    t0 = time.perf_counter()
    for i in range(n):
        c, s = rows[int(q_seq[i])]
        oracle.attention_over_cache(q[i], c, s, idx[i], scale)
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": "queries/s", "cores": 1, "kind": "oracle", **host_cpu(),
            "sample": f"{n} of {len(q_seq)} queries of draft_chunk_64x4x16384, {dt:.1f} s on 1 thread"}


def cpu_baseline_pages(sample_pages: int, repeats: int = 200):
    """The oracle's page-record layout (numpy) on `sample_pages` pages of the first
    sequence of the 64 x 16384 cache, packed `repeats` times."""
    import csa2_inputs as gen
    import oracle
    from csa2_inputs import native
    wl = workload_of("decode_short")
    n = min(sample_pages, 256) * 64
    gains = gen.latent_gains(wl.seed, 0)
    codes, scales = oracle.quantize(native.latent_rows_host(wl.seed, 0, 0, 0, n, gains))
    keys = native.key_rows_host(wl.seed, 0, 0, 0, n)
    ids = np.arange(n // 64)
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.pack_pages(codes, scales, keys, ids)
    dt = time.perf_counter() - t0
    return {"value": round(repeats * n / dt, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle", **host_cpu(),
            "sample": f"{n // 64} pages of page_export_64x16384 packed {repeats} times, "
                      f"{dt:.1f} s on 1 thread"}


def cpu_baseline_write(ww, sample_rows: int):
    """The oracle's write path (double-accumulated projection, then quantise / round) on
    `sample_rows` token rows, one host thread per row."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cores = os.cpu_count() or 1
    rows = np.linspace(0, ww.T - 1, max(1, sample_rows)).astype(np.int64)
    Wt = ww.w_rows(np.arange(ww.n_out))
    Hs = [ww.h_rows(np.array([r])) for r in rows]
    threads = min(cores, len(Hs))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda h: oracle.kv_write_rows(h, Wt, ww.n_kv_proj, ww.n_idx_proj), Hs))
    dt = time.perf_counter() - t0
    return {"value": round(len(Hs) / dt, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle", **host_cpu(),
            "sample": f"{len(Hs)} of {ww.T} token rows x {ww.n_out} output columns of {ww.name}, "
                      f"{dt:.1f} s wall on {threads} threads"}


def workload_of(name: str):
    import csa2_inputs as gen
    if name.endswith("_mx"):  # the same workload over an MXFP4 cache
        return workload_of(name[:-3])
    if name == "decode_batch16":   # the decode batch with 16 of its 64 sequences (profiling size)
        wl = gen.config_decode_batch()
        return gen.DecodeWorkload("decode_batch_16x131072", wl.seed, wl.seq_lens[:16],
                                  wl.q_per_seq[:16], wl.schedule, wl.pool_size, wl.topk)
    if name == "decode_short":     # the decode batch's 64 queries over 16384-token contexts:
        wl = gen.config_decode_batch()   # the attention launch shape at profiling size
        return gen.DecodeWorkload("decode_batch_64x16384", wl.seed,
                                  np.full(len(wl.seq_lens), 16384, np.int32), wl.q_per_seq,
                                  wl.schedule, wl.pool_size, wl.topk)
    return {"decode_batch": gen.config_decode_batch, "long_context": gen.config_long_context,
            "ragged": gen.config_ragged, "tiny": gen.config_tiny}[name]()


def count_launches(wl, step) -> int:
    """Kernels libcsa2 launches per decode step.  Full index call: the run-list kernel, the
    page scorer and one selection kernel (three, filter / resolve / emit, beyond 2^18
    tokens of context); Reindex: the gather scorer and one selection kernel; Reuse: none;
    attention: over the E4M3 cache the query-term kernel and the attention kernel, over the
    MXFP4 cache the attention kernel; either plus the split combine when the selected set
    spans more than one 128-entry tile (it is then split)."""
    import fp4_compressed_sparse_03_b300 as csa2
    wide = step.cache.page_table.shape[1] * 64 > (1 << 18)
    n = 0
    for m in wl.schedule:
        if m == csa2.CSA2_FULL:
            n += 2 + (3 if wide else 1)
        elif m == csa2.CSA2_REINDEX:
            n += 2
    per_attn = (1 if step.cache.mx else 2) + (1 if step.topk > 128 else 0)
    return n + len(wl.schedule) * per_attn


# Sources of the Full index call's kernels (the roofline line's kernels)
INDEX_SOURCES = ("index.cu", "async.cuh", "common.cuh")


def kernel_hash() -> str:
    """Hash of the code (comments and blank space removed) of the sources the Full index
    call's kernels are built from; its traffic counters are only reported for this exact
    code."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_compressed_sparse_03_b300", "csrc")
    for f in INDEX_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _code_only(src: str) -> str:
    """C++ source without // and /* */ comments and with runs of blank space collapsed
    (string literals holding comment markers are not expected in these kernels)."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


# ------------------------------------------------------------------ CPU oracle ---

def _oracle_query_step(wl, qi, keys, codes, scales, q_idx_h, q_h, scale, mx=False):
    """The whole layer schedule for one query on the CPU oracle."""
    import csa2_inputs as gen
    import oracle
    idx, pool = {}, None
    src = wl.index_source()
    n = keys.shape[0]
    for l, m in enumerate(wl.schedule):
        if m == gen.FULL:
            i, pool, _ = oracle.index_full(q_idx_h[l][qi], keys, wl.topk, wl.pool_size)
            idx[l] = i
        elif m == gen.REINDEX:
            idx[l], _ = oracle.index_reindex(q_idx_h[l][qi], keys, pool, wl.topk)
        else:
            idx[l] = oracle.index_reuse(idx[src[l]])
        oracle.attention_over_cache(q_h[l][qi], codes, scales, idx[src[l]], scale, mx=mx)
    return n


_PREP = {}  # (workload, mx, query) -> the query's resident inputs, generated once


def cpu_baseline(wl, sample_queries: int, mx: bool = False, first: int | None = None):
    """Time the oracle, as it stands, on a bounded sample of the workload: the full layer
    schedule for `sample_queries` queries (spread over the batch, or `first`, first + 1, ...
    when given), one host thread per query.  Generating a query's inputs is not timed, and
    is done once per query per process."""
    from concurrent.futures import ThreadPoolExecutor

    import csa2_inputs as gen
    import oracle
    from csa2_inputs import native
    from csa2_inputs.native import layer_queries_host

    cores = os.cpu_count() or 1
    if first is None:
        qs = np.linspace(0, wl.num_q - 1, min(sample_queries, wl.num_q)).astype(int)
    else:
        qs = [(first + i) % wl.num_q for i in range(min(sample_queries, wl.num_q))]
    L = len(wl.schedule)
    qh = [layer_queries_host(wl, l) for l in range(L)]
    q_idx_h = np.stack([a for a, _ in qh])
    q_h = np.stack([b for _, b in qh])
    gains = gen.latent_gains(wl.seed, 0)

    def prep(qi):  # resident inputs: keys and the quantised latent of the query's sequence
        key = (wl.name, mx, int(qi))
        if key in _PREP:
            return _PREP[key]
        b = int(wl.q_seq[qi])
        n = int(wl.seq_lens[b])
        keys = native.key_rows_host(wl.seed, 0, b, 0, n)
        quant = oracle.mx_quantize if mx else oracle.quantize
        codes, scales = quant(native.latent_rows_host(wl.seed, 0, b, 0, n, gains))
        _PREP[key] = (int(qi), keys, codes, scales)
        return _PREP[key]

    with ThreadPoolExecutor(max_workers=cores) as ex:
        inputs = list(ex.map(prep, qs))
    scale = float(np.float32(1.0 / math.sqrt(512.0)))
    threads = min(cores, len(inputs))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda a: _oracle_query_step(wl, a[0], a[1], a[2], a[3], q_idx_h, q_h, scale,
                                                 mx), inputs))
    dt = time.perf_counter() - t0
    return {"value": round(len(inputs) * L / dt, 3), "unit": UNIT, "cores": threads,
            "kind": "oracle", **host_cpu(),
            "sample": f"{len(inputs)} of {wl.num_q} queries x {L} layers of {wl.name}, "
                      f"{dt:.1f} s wall on {threads} threads"}


def run_reference(args, world, rank):
    """The oracle as the reference arm, on the same workload, metric and unit."""
    import csa2_inputs as gen
    if rank != 0:
        return
    if args.workload in ("ced_write", "decode_append"):
        return run_reference_write(args, world)
    if args.workload == "draft_chunk":
        per_step = max(1, args.cpu_sample // max(1, args.steps))
        t0 = time.perf_counter()
        vals = [cpu_baseline_chunk(per_step, args.shared) for _ in range(args.steps)]
        dt = time.perf_counter() - t0
        cb = dict(vals[-1])
        cb["value"] = round(float(np.mean([c["value"] for c in vals])), 3)
        cb["sample"] = f"{args.steps} steps x {per_step} queries of draft_chunk_64x4x16384"
        line = {"impl": "reference", "metric": CHUNK_METRIC, "value": cb["value"],
                "unit": "queries/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
                "data": "synthetic (seeded counter-based generator)",
                "config": {"workload": "draft_chunk_64x4x16384"}, "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "queries/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.workload == "page_export":
        cb = cpu_baseline_pages(args.cpu_sample)
        line = {"impl": "reference",
                "metric": "persistent KV tier: tokens/s of cache pages exported (codes, scales, keys)",
                "value": cb["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup,
                # a step exports the cache's 16384 pages (1048576 tokens)
                "ms_per_step": round(1048576 / cb["value"] * 1e3, 2), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8 (CPU oracle, numpy)",
                "data": "synthetic (seeded counter-based generator)",
                "config": pages_config(world), "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    wl = workload_of(args.workload)
    per_step = max(1, args.cpu_sample // max(1, args.steps))
    mx = args.workload.endswith("_mx")
    # steps cycle over a few queries whose inputs are generated once, before the clock
    # starts, so a step is the oracle's own work on one bounded sample
    distinct = max(1, min(8, wl.num_q // per_step))
    for i in range(distinct):
        cpu_baseline(wl, per_step, mx, first=i * per_step)
    vals = []
    t0 = time.perf_counter()
    for k in range(args.steps):
        vals.append(cpu_baseline(wl, per_step, mx, first=(k % distinct) * per_step))
    dt = time.perf_counter() - t0
    v = float(np.mean([c["value"] for c in vals]))
    cb = dict(vals[-1])
    cb["value"] = round(v, 3)
    cb["sample"] = f"{args.steps} steps x {per_step} queries x {len(wl.schedule)} layers of {wl.name}"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
            "data": "synthetic (seeded counter-based generator)",
            "config": decode_config(wl, args.workload.endswith("_mx"), world,
                                    args.step_schedule),
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_write(args, world):
    import csa2_inputs as gen
    append = args.workload == "decode_append"
    ww = gen.config_append() if append else gen.config_write()
    per_step = max(1, args.cpu_sample // max(1, args.steps))
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline_write(ww, per_step))
    dt = time.perf_counter() - t0
    v = float(np.mean([c["value"] for c in vals]))
    cb = dict(vals[-1])
    cb["value"] = round(v, 3)
    cb["sample"] = f"{args.steps} steps x {per_step} token rows of {ww.name}"
    line = {"impl": "reference",
            "metric": ("decode-time append: new tokens/s projected and quantised into the paged cache"
                       if append else "CED write path: tokens/s projected and quantised on write"),
            "value": round(v, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (CPU oracle)", "data": "synthetic (seeded counter-based generator)",
            "config": write_config(ww, world),
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_batch",
                    choices=["decode_batch", "decode_batch16", "decode_short", "long_context", "ragged", "tiny",
                             "ced_write", "decode_append", "decode_batch_mx", "decode_short_mx",
                             "page_export", "draft_chunk"])
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--step-schedule", choices=["parallel", "serial"], default="parallel",
                    help="decode step graph: attention calls on side branches, or every "
                         "call in layer order on one stream")
    ap.add_argument("--cpu-sample", type=int, default=None,
                    help="queries (decode) or token rows (write workloads) timed on the oracle; "
                         "default 32 queries / 256 rows (all 64 for decode_append), about "
                         "10-30 s of CPU work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shared", type=float, default=CHUNK_SHARED,
                    help="draft_chunk: fraction of each query's selection common to its chunk")
    args = ap.parse_args()
    if args.cpu_sample is None:
        args.cpu_sample = {"ced_write": 256, "decode_append": 64,
                           "page_export": 256}.get(args.workload, 32)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload in ("ced_write", "decode_append"):
        args.warmup = max(3, args.warmup)
        run_write(args, world, rank, local)
    elif args.workload == "page_export":
        args.warmup = max(3, args.warmup)
        run_pages(args, world, rank, local)
    elif args.workload == "draft_chunk":
        args.warmup = max(3, args.warmup)
        run_chunk(args, world, rank, local)
    else:
        args.warmup = max(3, args.warmup)
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
