"""Benchmark of the compressed-KV write/read hot path on GB300.

One step = one long-prefill batch through the whole path:
  1. dsv4kv_compress_store: 64 requests (~262k tokens, lognormal lengths),
     ratio-2 softmax pair pooling of the fused | kv | score | rows, RMSNorm,
     RoPE, V41 quantization, paged store (page size 64);
  2. the sparse-prefill read of each request's top-2048 compressed ids: 4
     layers share the source; the first get_with_head_topk runs the fused
     top-k -> slot -> gather-dequant kernel, the other three are reuse hits.
value = (rows stored + real rows gathered) / step time, inputs resident in
        HBM; the top-k list's -1 padding (requests with fewer than 2048
        compressed rows) yields zero rows that are not counted.
e2e   = the same step through host buffers: pinned host -> device copy of
        the step's inputs and device -> host copy of the gathered rows inside
        the timed region (request chunks, copies overlapped with the kernels,
        the same store + 1 dequant + 3 reuse hits per chunk).

Besides the headline line's timed region, the run measures (each reported
in the same JSON line): the store and the gather of the step one launch at
a time (medians of >= 50 event pairs, the roofline's durations); each of
the five workloads on its own (`configs`: µs and rows/s, L2 flushed before
each launch, and warm where the working set fits in L2; the 1 Mi-row
gather as 4 dequant launches against 1 dequant + 3 reuse hits); the other
layouts' store-only, gather and fake-quantization launches (`cold_l2`); the
decode / verify ring steps; the CPU oracle per workload on one core and on
all cores (`cpu_baseline`, `oracle_per_config`).  nvidia-smi clocks are
sampled across the whole run.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed-KV rows/s (store, gather-dequant) and achieved HBM GB/s vs 8 TB/s"
LAYERS = 4
KERNEL_SAMPLES = 100   # launches of the store / gather timed one by one (median)
CONFIG_REPS = 50       # timed launches per workload leg (median), after 5 warm-ups
E2E_CHUNKS = 4
# algorithmic bytes per unit (what the method must move)
STORE_BYTES_PER_ROW = 2 * (1024 + 1024) + 256 + 528   # 2 x (kv + score) bf16, RoPE row, V41 row
GATHER_BYTES_PER_ROW = 528 + 4 + 1024                  # V41 row + id, bf16 row out
PAD_BYTES_PER_ROW = 4 + 1024                           # a -1 id: read the id, write a zero row

_CSRC = os.path.join("deepseek_v4_compressed_c2_gb300", "csrc")
STORE_SOURCES = [os.path.join(_CSRC, f) for f in
                 ("compress_store.cu", "compress_row.cuh", "quant.cuh", "tma.cuh", "layout.cuh",
                  "internal.cuh")]


def _profiled_traffic(name, sources):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since that capture (hash mismatch)."""
    import hashlib
    try:
        h = hashlib.sha256()
        for f in sources:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        fields = {}
        with open(os.path.join(ROOT, "profiles", name + ".md")) as fh:
            for line in fh:
                if ":" in line and not line.startswith("|"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip().split()[0] if v.strip() else ""
        if fields.get("source_sha256") != h.hexdigest()[:16]:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, one query every ~`period` s on
    a host thread for the whole run (a one-shot query per sample, so nothing
    is lost to output buffering).  `busy(name)` brackets GPU work: the
    reported median SM clock is taken over samples inside those windows."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, period=0.02):
        self.idx, self.period = gpu_index, period
        self.samples = []           # (t_mid, sm, max, reasons)
        self.windows = []           # (name, t0, t1)
        self._stop = threading.Event()
        self._t = None

    def start(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _run(self):
        cmd = ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits"]
        while not self._stop.is_set():
            t0 = time.monotonic()
            try:
                out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout
            except Exception:
                return
            t1 = time.monotonic()
            parts = [p.strip() for p in out.strip().split(",")]
            if len(parts) >= 7:
                try:
                    sm, mx = float(parts[0]), float(parts[1])
                    reasons = {n for n, v in zip(self.NAMES, parts[3:7]) if v.lower() == "active"}
                    self.samples.append(((t0 + t1) / 2, sm, mx, reasons))
                except ValueError:
                    pass
            self._stop.wait(self.period)

    class _Window:
        def __init__(self, s, name):
            self.s, self.name = s, name

        def __enter__(self):
            self.t0 = time.monotonic()

        def __exit__(self, *exc):
            self.s.windows.append((self.name, self.t0, time.monotonic()))

    def busy(self, name):
        return ClockSampler._Window(self, name)

    def stop(self):
        self._stop.set()
        if self._t is not None:
            self._t.join(timeout=10)
        inside = [s for s in self.samples if any(t0 <= s[0] <= t1 for _, t0, t1 in self.windows)]
        use = inside or self.samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for s in use:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in use),
                "sm_max_mhz": max(s[2] for s in use), "reasons": sorted(reasons),
                "samples": len(self.samples), "samples_during_gpu_work": len(inside),
                "sm_mhz_min_during_gpu_work": min(s[1] for s in use),
                "gpu_work_windows": [n for n, _, _ in self.windows],
                "period_s": self.period}


def set_l2_fetch_granularity(nbytes):
    """The serving process's L2 fetch granularity (cudaLimitMaxL2FetchGranularity,
    a limit of this process's CUDA context: it ends with the process).  The
    step's read is a gather of random 288-584 B rows, and a whole 128-byte
    line fetched per partly wanted line is DRAM traffic the gather does not
    need; 0 leaves the context's default.  Returns the limit read back."""
    import ctypes
    import torch
    torch.zeros(1, device="cuda")                 # the context exists
    lib = None
    for cand in (os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so"),
                 "libcudart.so.13", "libcudart.so"):
        try:
            lib = ctypes.CDLL(cand)
            break
        except OSError:
            continue
    if lib is None:
        return None
    limit = 0x05                                  # cudaLimitMaxL2FetchGranularity
    if nbytes:
        if lib.cudaDeviceSetLimit(limit, ctypes.c_size_t(nbytes)) != 0:
            return None
    v = ctypes.c_size_t(0)
    return int(v.value) if lib.cudaDeviceGetLimit(ctypes.byref(v), limit) == 0 else None


def max_over_ranks(values, world, device="cpu"):
    """Element-wise max of per-rank floats over the process group (the bench
    reports the slowest rank's time); identity when world == 1."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, world, slowest_ms):
    """Weak scaling: every rank processes its own batch of `units_per_rank`;
    the job's rate is all units over the slowest rank's time."""
    return units_per_rank * world / (slowest_ms / 1e3)


def make_inputs(seed=7):
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    return W.cfg5_long_prefill(seed=seed)


def gather_rows_valid(cfg):
    """real rows of the step's gather: the top-k ids >= 0"""
    return int((cfg["topk"] >= 0).sum())


def headline_config(cfg, world, l2_fetch):
    """The `config` both arms print for the long-prefill step (l2_fetch: the
    GPU arm's L2 fetch granularity setting, bytes)."""
    n_tok, k = cfg["topk"].shape
    return {"workload": cfg["name"], "requests": len(cfg["lengths"]),
            "tokens": int(sum(cfg["lengths"])), "store_rows": int(cfg["n_out"]),
            "gather_rows_valid": gather_rows_valid(cfg), "gather_id_slots": int(n_tok * k),
            "layers_reading_source": LAYERS, "layout": "V41", "ratio": 2, "page_size": 64,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (fused rows %d MB per step)"
                  % (cfg["rows"].nbytes // 10 ** 6),
            "l2_fetch_granularity_bytes": l2_fetch}


# ------------------------------------------------------------------ oracle
def cpu_info():
    """(cores this process may run on, CPU model string)"""
    cores = len(os.sched_getaffinity(0))
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu model")):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return cores, model or "unknown"


def _split(a, parts):
    return [c for c in np.array_split(a, parts) if len(c)]


def _run_parts(fn, chunks, threads):
    """fn over the chunks, on `threads` host threads (the oracle's C calls
    release the interpreter lock); returns wall seconds"""
    t0 = time.perf_counter()
    if threads <= 1:
        for c in chunks:
            fn(c)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fn, chunks))
    return time.perf_counter() - t0


class OracleStep:
    """The oracle as it stands on a bounded sample of the long-prefill step:
    the store of the batch's first m compressed rows (ratio-2 compress,
    RMSNorm, RoPE, V41 quantize, paged store) and the gather of the same
    fraction of the step's real top-k rows (the oracle's own slots), with the
    rows split over `threads` host threads."""

    def __init__(self, cfg):
        import oracle
        self.o, self.cfg = oracle, cfg
        self.pool = np.zeros(cfg["pool_rows"] * 528, np.uint8)
        slots, _, _ = oracle.topk_to_slots(cfg["topk"], cfg["token_to_req"], cfg["page_table"],
                                           cfg["page_bits"])
        self.slots = slots.reshape(-1)[slots.reshape(-1) >= 0].astype(np.int32)

    def rows_for(self, m):
        g = int(round(m * len(self.slots) / self.cfg["n_out"]))
        return m, g

    def run(self, m, threads):
        cfg, o = self.cfg, self.o
        m, g = self.rows_for(m)

        def store(which):
            o.compress_store(1, 2, cfg["rows"], cfg["ext"], page_table=cfg["page_table"],
                             page_bits=cfg["page_bits"], norm_w=cfg["norm_w"], eps=cfg["eps"],
                             freqs=cfg["freqs"], n_out=cfg["n_out"], which=which,
                             pool=self.pool, pool_rows=cfg["pool_rows"], want_f64=False,
                             want_f32=False, want_latent=False)

        def gather(ids):
            o.dequant_gather(1, self.pool, cfg["pool_rows"], ids)

        t = _run_parts(store, _split(np.arange(m, dtype=np.int64), threads), threads)
        t += _run_parts(gather, _split(self.slots[:g], threads), threads)
        return m + g, t

    def size_for(self, budget_s, threads):
        """compressed rows per sample so that one sample takes ~budget_s"""
        probe = min(512, self.cfg["n_out"])
        units, t = self.run(probe, threads)
        return int(min(self.cfg["n_out"], max(16, probe * budget_s / max(t, 1e-6))))


def cpu_baseline(cfg, budget_s=6.0):
    """The oracle on the long-prefill step, timed on the host cores: one core
    and all cores (threads over rows), each on a sample of ~budget_s."""
    cores, model = cpu_info()
    step = OracleStep(cfg)
    res = {}
    for threads in (1, cores):
        m = step.size_for(budget_s, threads)
        units, t = step.run(m, threads)
        res[threads] = (units, t, m)
    units, t, m = res[cores]
    u1, t1, m1 = res[1]
    return {"value": units / t, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "cpu_model": model,
            "sample": f"first {m} of {cfg['n_out']} compressed rows of the batch (ratio-2 "
                      f"compress, RMSNorm, RoPE, V41 store) + the same fraction of the real "
                      f"top-k rows gathered, rows split over {cores} threads, {t:.2f} s",
            "single_thread": {"value": u1 / t1, "unit": "rows/s", "cores": 1,
                              "sample": f"first {m1} compressed rows + the same fraction of "
                                        f"the gathered rows, {t1:.2f} s"}}


def oracle_per_config(cfgs, budget_s=2.0):
    """The oracle on each workload, one core and then all cores (threads over
    rows), the store and the gather / dequant timed apart: each on a bounded
    sample (~budget_s on one core) of the workload's store rows and of its
    ids (cfg1, cfg3: the written slots; cfg4: the 262,144 ids, whose rows the
    oracle stores first, untimed; cfg2 has no read)."""
    import oracle
    cores, model = cpu_info()
    out = {"cores": cores, "cpu_model": model}
    for key, c in cfgs.items():
        layout = c["layout"]
        pool = np.zeros(c["pool_rows"] * oracle.row_bytes(layout), np.uint8)
        p = oracle.plan(c["ratio"], c["ext"], c["page_table"], c["page_bits"])

        def store(which, c=c, pool=pool, layout=layout):
            oracle.compress_store(layout, c["ratio"], c["rows"], c["ext"],
                                  page_table=c["page_table"], page_bits=c["page_bits"],
                                  norm_w=c["norm_w"], eps=c["eps"], freqs=c["freqs"],
                                  n_out=c["n_out"], which=which, pool=pool,
                                  pool_rows=c["pool_rows"], want_f64=False, want_f32=False,
                                  want_latent=False)

        def gather(ids, c=c, pool=pool, layout=layout):
            oracle.dequant_gather(layout, pool, c["pool_rows"], ids)

        if "ids" in c:                       # gather only; its rows stored first, untimed
            rows, ids = np.zeros(0, np.int64), np.asarray(c["ids"], np.int32)
            _run_parts(store, _split(ids.astype(np.int64) - (1 << c["page_bits"]), cores), cores)
        elif c["ratio"] == 1:                # store, then dequant of the written slots
            rows, ids = np.arange(p["total"], dtype=np.int64), p["slot"][p["slot"] > 0].astype(np.int32)
        else:                                # store only
            rows, ids = np.arange(p["total"], dtype=np.int64), np.zeros(0, np.int32)
        entry = {"name": c["name"]}
        for part, fn, items, probe in (("store", store, rows, 256), ("gather", gather, ids, 4096)):
            if not len(items):
                continue
            k0 = min(probe, len(items))
            t = _run_parts(fn, [items[:k0]], 1)
            n = int(min(len(items), max(k0, k0 * budget_s / max(t, 1e-6))))
            d = {"sample_rows": n, "of_rows": int(len(items))}
            for threads in (1, cores):
                t = _run_parts(fn, _split(items[:n], threads), threads)
                d["rows_per_s_1core" if threads == 1 else "rows_per_s_all_cores"] = n / t
            entry[part] = d
        out[key] = entry
    return out


def run_reference(args, rank):
    """The reference arm: the CPU oracle on all host cores, on rank 0 only,
    each step a bounded sample sized so that warm-up + steps take about two
    minutes in all."""
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    cfg = make_inputs()
    cores, model = cpu_info()
    step = OracleStep(cfg)
    step.run(64, 1)                          # the oracle's tables, built on one thread
    per_step = max(0.005, 120.0 / (args.steps + args.warmup))
    m = step.size_for(per_step, cores)
    for _ in range(args.warmup):
        step.run(m, cores)
    runs = [step.run(m, cores) for _ in range(args.steps)]
    t = statistics.median(r[1] for r in runs)
    v = runs[0][0] / t
    sample = (f"first {m} of {cfg['n_out']} compressed rows (ratio-2 compress, RMSNorm, RoPE, "
              f"V41 store) + the same fraction of the real top-k rows gathered per step, rows "
              f"split over {cores} threads, median {t * 1e3:.1f} ms")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(cfg, world, args.l2_fetch_granularity or None),
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "cpu_model": model, "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU legs
class Flusher:
    """Before a timed launch: write `flush` (512 MB, 4x the L2), then read
    `scrub` (256 MB), which evicts the write's dirty lines, so the launch
    starts from an L2 that holds neither its inputs nor lines still to be
    written back."""

    def __init__(self, dev):
        import torch
        self.flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.scrub = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
        self.i = 0

    def __call__(self, clean=True):
        self.i += 1
        self.flush.fill_(self.i & 0xFF)
        if clean:
            self.scrub.max()


def _timed(fn, stream, reps, flusher=None, clean=True, warm=5):
    """median and count of CUDA-event times (ms) of fn() on `stream`; with a
    flusher the L2 is flushed before every launch, else the launches run back
    to back (the working set stays wherever the previous launch left it)"""
    import torch
    times = []
    with torch.cuda.stream(stream):
        for i in range(reps + warm):
            if flusher is not None:
                flusher(clean)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in times[warm:])


def _graph_us(fn, stream, reps=50):
    """device time per launch (us) of fn() captured `reps` times in one CUDA
    graph: median of 5 replays; the launch-bound legs' serving-loop figure"""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            fn()
    times = []
    with torch.cuda.stream(stream):
        for i in range(8):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    del g
    return statistics.median(a.elapsed_time(b) for a, b in times[3:]) * 1e3 / reps


def _leg(ms, units, bytes_per_unit=None, peak=None, **extra):
    d = {"us": ms * 1e3, "rows": units, "rows_per_s": units / (ms / 1e3)}
    if bytes_per_unit is not None:
        gbs = bytes_per_unit * units / (ms / 1e3) / 1e9
        d.update(gbs=gbs, bytes_per_row=bytes_per_unit)
        if peak is not None:
            d.update(frac=gbs / peak, frac_of_8000=gbs / 8000.0)
    d.update(extra)
    return d


def config_legs(B, dev, stream, flusher, cfg4, peak):
    """Each workload on its own, with the L2 flushed before every launch
    ("cold"), and back to back ("warm") where the working set fits in L2."""
    import torch
    from deepseek_v4_compressed_c2_gb300 import workloads as W

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    err = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {}

    def store_call(c, pool):
        stream.wait_stream(torch.cuda.current_stream(dev))   # the pool's zero fill first
        return B.prepare_compress_store(
            c["layout"], c["ratio"], bf(c["rows"]), t(c["ext"]), pool, page_table=t(c["page_table"]),
            page_bits=c["page_bits"], rmsnorm_w=None if c["norm_w"] is None else bf(c["norm_w"]),
            eps=c["eps"], freqs_cis=t(c["freqs"]), n_out=c["n_out"], err_word=err, stream=stream)

    # cfg1: V41 ratio-1 store of 256 rows, then dequant of the 256 slots
    c1 = W.cfg1_v41_roundtrip()
    pool = torch.zeros(c1["pool_rows"] * 528, dtype=torch.uint8, device=dev)
    st = store_call(c1, pool)
    ids = torch.arange(64, 64 + 256, dtype=torch.int32, device=dev)
    out = torch.empty((256, 512), dtype=torch.bfloat16, device=dev)
    ga = B.prepare_dequant_gather(1, pool, ids, out, err_word=err, stream=stream)
    res["cfg1_" + c1["name"]] = {
        "store_cold": _leg(_timed(st, stream, CONFIG_REPS, flusher), 256),
        "store_warm": _leg(_timed(st, stream, CONFIG_REPS), 256),
        "store_in_graph": _leg(_graph_us(st, stream) / 1e3, 256),
        "dequant_cold": _leg(_timed(ga, stream, CONFIG_REPS, flusher), 256),
        "dequant_warm": _leg(_timed(ga, stream, CONFIG_REPS), 256),
        "dequant_in_graph": _leg(_graph_us(ga, stream) / 1e3, 256),
        "note": "0.4 MB each way: launch-latency bound, no roofline claim; *_in_graph = "
                "device time per launch inside a CUDA graph of 50 launches"}

    # cfg2: ratio-2 V41 compressor, 4 requests (1809 rows of 2048 output rows)
    c2 = W.cfg2_ratio2_small()
    pool = torch.zeros(c2["pool_rows"] * 528, dtype=torch.uint8, device=dev)
    st = store_call(c2, pool)
    n2 = int(sum(n // 2 for n in c2["lengths"]))
    res["cfg2_" + c2["name"]] = {
        "store_cold": _leg(_timed(st, stream, CONFIG_REPS, flusher), n2, STORE_BYTES_PER_ROW),
        "store_warm": _leg(_timed(st, stream, CONFIG_REPS), n2, STORE_BYTES_PER_ROW),
        "store_in_graph": _leg(_graph_us(st, stream) / 1e3, n2, STORE_BYTES_PER_ROW),
        "note": "8.8 MB of algorithmic bytes: L2-resident and launch-latency bound, "
                "no roofline claim"}

    # cfg3: FP4 ratio-1 store of 32768 rows, then the full dequant
    c3 = W.cfg3_fp4_store()
    pool = torch.zeros(c3["pool_rows"] * 288, dtype=torch.uint8, device=dev)
    st = store_call(c3, pool)
    ids = torch.arange(128, 128 + 32768, dtype=torch.int32, device=dev)
    out = torch.empty((32768, 512), dtype=torch.bfloat16, device=dev)
    ga = B.prepare_dequant_gather(2, pool, ids, out, err_word=err, stream=stream)
    res["cfg3_" + c3["name"]] = {
        "store_cold": _leg(_timed(st, stream, CONFIG_REPS, flusher), 32768, 1024 + 288, peak),
        "store_warm": _leg(_timed(st, stream, CONFIG_REPS), 32768, 1024 + 288),
        "store_in_graph": _leg(_graph_us(st, stream) / 1e3, 32768, 1024 + 288),
        "dequant_cold": _leg(_timed(ga, stream, CONFIG_REPS, flusher), 32768, 288 + 4 + 1024, peak),
        "dequant_warm": _leg(_timed(ga, stream, CONFIG_REPS), 32768, 288 + 4 + 1024),
        "dequant_in_graph": _leg(_graph_us(ga, stream) / 1e3, 32768, 288 + 4 + 1024),
        "note": "43 MB each way: fits in L2, so warm launches read L2; *_in_graph = device "
                "time per launch inside a CUDA graph of 50 launches (warm)"}

    # cfg4: 1 Mi-row V41 pool, 262,144 ids, read by 4 layers
    pool = torch.zeros(cfg4["pool_rows"] * 528, dtype=torch.uint8, device=dev)
    rows4 = bf(cfg4["rows"])
    stream.wait_stream(torch.cuda.current_stream(dev))
    fill = B.prepare_compress_store(1, 1, rows4, t(cfg4["ext"]), pool,
                                    page_table=t(cfg4["page_table"]), page_bits=cfg4["page_bits"],
                                    n_out=cfg4["n_out"], err_word=err, stream=stream)
    ms_fill = _timed(fill, stream, max(5, CONFIG_REPS // 5), flusher)
    ids = t(cfg4["ids"])
    n_ids = ids.numel()
    kv = B.SparsePrefillKVBuffer(torch.empty((n_ids, 512), dtype=torch.bfloat16, device=dev))
    ga = B.prepare_dequant_gather(1, pool, ids, kv.storage, err_word=err, stream=stream)
    gwh = B.prepare_get_with_head(kv, 1, pool, ids, err_word=err, stream=stream)
    ms_one = _timed(ga, stream, CONFIG_REPS, flusher)

    def no_reuse():
        for _ in range(LAYERS):
            ga()

    hits = []

    def with_reuse():
        kv.dsv4kv_kvbuf_begin_forward()
        hits[:] = [gwh() for _ in range(LAYERS)]

    ms_4 = _timed(no_reuse, stream, CONFIG_REPS, flusher)
    ms_r = _timed(with_reuse, stream, CONFIG_REPS, flusher)
    assert hits == [False] + [True] * (LAYERS - 1)
    res["cfg4_" + cfg4["name"]] = {
        "store_fill_cold": _leg(ms_fill, cfg4["n_out"], 1024 + 528, peak),
        "gather_cold": _leg(ms_one, n_ids, GATHER_BYTES_PER_ROW, peak),
        "four_layers_without_reuse": {"us": ms_4 * 1e3, "dequant_launches": LAYERS,
                                      "rows_per_s": LAYERS * n_ids / (ms_4 / 1e3)},
        "four_layers_with_reuse": {"us": ms_r * 1e3, "dequant_launches": 1, "reuse_hits": 3,
                                   "rows_per_s": LAYERS * n_ids / (ms_r / 1e3)},
        "reuse_speedup": ms_4 / ms_r,
        "note": "L2 flushed before each timed group; rows_per_s of the 4-layer legs counts "
                "the rows every layer reads"}
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return res, pool, rows4, ids


def cold_paths(B, dev, stream, flusher, cfg4, rows4, ids, peak):
    """The other layouts on the 1 Mi-row workload, each launch timed alone
    with a cold L2: the ratio-1 store-only fill (1,048,512 rows of the same
    bf16 latents) and the gather of the same 262,144 ids in the V41_FP4 and
    V4 layouts; the fake quantization of the latents in every layout; on the
    V41 pool the short-context gather (128 tokens of one request, lengths
    uniform in [1, 2048], numpy seed 5) and the gather after a write-only
    flush (dirty L2)."""
    import torch
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ext = torch.from_numpy(cfg4["ext"]).to(dev)
    pt = torch.from_numpy(cfg4["page_table"]).to(dev)
    n_rows, n_ids = cfg4["n_out"], ids.numel()
    out = torch.empty((n_ids, 512), dtype=torch.bfloat16, device=dev)
    fq_out = torch.empty((n_rows, 512), dtype=torch.bfloat16, device=dev)
    res = {}
    for layout, name, rb in ((1, "v41", 528), (2, "fp4", 288), (0, "v4", 584)):
        pool = torch.zeros(cfg4["pool_rows"] * rb, dtype=torch.uint8, device=dev)
        stream.wait_stream(torch.cuda.current_stream(dev))
        store = B.prepare_compress_store(layout, 1, rows4, ext, pool, page_table=pt,
                                         page_bits=cfg4["page_bits"], n_out=n_rows, err_word=err,
                                         stream=stream)
        gather = B.prepare_dequant_gather(layout, pool, ids, out, err_word=err, stream=stream)
        ms_s = _timed(store, stream, max(5, CONFIG_REPS // 5), flusher)
        ms_g = _timed(gather, stream, CONFIG_REPS, flusher)
        res[f"store_ratio1_{name}_{n_rows}rows"] = _leg(ms_s, n_rows, 1024 + rb, peak)
        res[f"gather_{name}_{n_ids}_of_{cfg4['pool_rows']}"] = _leg(ms_g, n_ids, rb + 4 + 1024, peak)
        ms_f = _timed(lambda: B.dsv4kv_fake_quant(layout, rows4, fq_out, stream=stream), stream,
                      max(5, CONFIG_REPS // 5), flusher)
        res[f"fake_quant_{name}_{n_rows}rows"] = _leg(ms_f, n_rows, 2048, peak)
        if layout == 1:
            n_tok, k = 128, 2048
            lens_in = torch.from_numpy(np.random.default_rng(5).integers(1, k + 1, n_tok)
                                       .astype(np.int32)).to(dev)
            ttr = torch.zeros(n_tok, dtype=torch.int32, device=dev)
            ms_a = _timed(lambda: B.dsv4kv_dequant_gather_all(1, pool, lens_in, k, ttr, pt,
                                                              cfg4["page_bits"], out[:n_tok * k],
                                                              err_word=err, stream=stream),
                          stream, CONFIG_REPS, flusher)
            ms_gd = _timed(gather, stream, CONFIG_REPS, flusher, clean=False)
            res[f"gather_v41_{n_ids}_of_{cfg4['pool_rows']}_dirty_l2"] = _leg(
                ms_gd, n_ids, GATHER_BYTES_PER_ROW, peak,
                note="L2 flushed by the 512 MB write alone; ~129 MB of its dirty lines are "
                     "written back during the gather")
            res["gather_all_v41_128tok_2048"] = _leg(
                ms_a, n_tok * k, None, None, selected_rows=int(lens_in.sum().item()),
                out_gbs=1024 * n_tok * k / (ms_a / 1e3) / 1e9,
                note="every token of one request re-reads the same <= 2048 compressed rows "
                     "(L2-resident after the first); bound by the 1 KB/row output")
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        del pool
    res["peak_kind"] = _peaks()[1]
    return res


def c1_leg(B, dev, stream, flusher, cfg, rows, peak):
    """The full c1 form of the compressor on the long-prefill batch: ratio 1
    with RMSNorm and RoPE, one V41 row per token (the same 262,144 fused rows,
    already on the device, their kv half read), into a pool paged by
    `workloads.c1_page_table`; each launch timed alone with a cold L2."""
    import torch
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    pt_h, pool_rows = W.c1_page_table(cfg["lengths"], page_bits=cfg["page_bits"])
    n = int(sum(cfg["lengths"]))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pool = torch.zeros(pool_rows * 528, dtype=torch.uint8, device=dev)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    store = B.prepare_compress_store(1, 1, rows, torch.from_numpy(cfg["ext"]).to(dev), pool,
                                     page_table=torch.from_numpy(pt_h).to(dev),
                                     page_bits=cfg["page_bits"], rmsnorm_w=bf(cfg["norm_w"]),
                                     eps=cfg["eps"], freqs_cis=torch.from_numpy(cfg["freqs"]).to(dev),
                                     n_out=n, err_word=err, stream=stream)
    ms = _timed(store, stream, max(5, CONFIG_REPS // 5), flusher)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {f"store_ratio1_v41_norm_rope_{n}rows": _leg(ms, n, 1024 + 256 + 528, peak,
                                                         note="1808 B/row: kv row, RoPE row, V41 row")}


def decode_verify_steps(B, dev, stream, reps=50, max_prefix=4096):
    """The ring form of the compressor on decode-shaped steps (one new token
    per request; 1 + 3 draft tokens per request; a small decode step; a
    chunked-prefill step of 16 requests x 200 tokens).  These are small,
    latency-bound launches (working set in L2).  The serving loop runs them
    inside a CUDA graph whose offsets are refreshed in place, so the device
    time per launch is taken from a captured graph of `reps` launches; the
    eager figure (one prepared C-ABI call per launch from Python) is kept
    beside it and includes the host's launch cost."""
    import torch
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    res = {}
    for name, n_req, n_new in (("decode_4096req_1tok", 4096, 1), ("verify_1024req_4tok", 1024, 4),
                               ("decode_512req_1tok", 512, 1), ("chunked_16req_200tok", 16, 200)):
        cfg = W.decode_verify(seed=13, n_req=n_req, n_new=n_new, ring_size=4,
                              max_prefix=max_prefix)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
        ring = bf(cfg["ring"])
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        rows = bf(cfg["rows"])
        ext = torch.from_numpy(cfg["ext"]).to(dev)
        stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(stream):
            call = B.prepare_compress_store(
                1, 2, rows, ext, pool, page_table=torch.from_numpy(cfg["page_table"]).to(dev),
                page_bits=6, rmsnorm_w=bf(cfg["norm_w"]), eps=cfg["eps"],
                freqs_cis=torch.from_numpy(cfg["freqs"]).to(dev), n_out=cfg["n_out"],
                err_word=err, stream=stream, start_pos=torch.from_numpy(cfg["start_pos"]).to(dev),
                ring=ring)
            for _ in range(5):
                call()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        eager_us = a.elapsed_time(b) * 1e3 / reps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(reps):
                call()
        graph_us = []
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graph.replay()
                b.record(stream)
                graph_us.append((a, b))
        torch.cuda.synchronize(dev)
        assert int(err.item()) == 0
        us = statistics.median(a.elapsed_time(b) for a, b in graph_us) * 1e3 / reps
        res[name] = {"us_per_launch": us, "eager_us_per_launch": eager_us, "rows": cfg["n_out"],
                     "tokens": n_req * n_new, "rows_per_s": cfg["n_out"] / (us / 1e6),
                     "timing": f"median of 5 replays of a graph of {reps} launches"}
        del graph
    return res


PROFILE_LEGS = ("store_long_prefill", "step_gather", "gather_v41", "gather_fp4", "gather_v4",
                "store_fp4_1m", "decode", "verify", "store_c1")


def profile_leg(name):
    """One leg's launches alone, for an ncu capture (three launches, the L2
    flushed before each): the long-prefill store; the step's fused top-k
    gather (after one store); the cold gather of the 262,144 cfg4 ids from
    the 1 Mi-row pool in a layout (the pool filled by one store-only launch
    first); the FP4 store-only fill of that pool; the decode (4096 x 1) or
    verify (1024 x 4) ring step; the full c1 form on the long-prefill tokens.
    Prints one JSON line; times nothing."""
    import torch
    from deepseek_v4_compressed_c2_gb300 import binding as B
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    B.lib()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)    # allocations and launches in one order
    flusher = Flusher(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    if name in ("store_long_prefill", "step_gather"):
        cfg = make_inputs()
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
        call = B.prepare_compress_store(1, 2, bf(cfg["rows"]), t(cfg["ext"]), pool,
                                        page_table=t(cfg["page_table"]), page_bits=6,
                                        rmsnorm_w=bf(cfg["norm_w"]), eps=cfg["eps"],
                                        freqs_cis=t(cfg["freqs"]), n_out=cfg["n_out"],
                                        err_word=err, stream=stream)
        if name == "step_gather":
            n_tok, k = cfg["topk"].shape
            out = torch.empty((n_tok * k, 512), dtype=torch.bfloat16, device=dev)
            call = B.prepare_dequant_gather_topk(1, pool, t(cfg["topk"]), t(cfg["token_to_req"]),
                                                 t(cfg["page_table"]), 6, out, err_word=err,
                                                 stream=stream)
    elif name == "store_c1":
        cfg = W.c1_long_prefill()
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
        call = B.prepare_compress_store(1, 1, bf(cfg["rows"]), t(cfg["ext"]), pool,
                                        page_table=t(cfg["page_table"]), page_bits=cfg["page_bits"],
                                        rmsnorm_w=bf(cfg["norm_w"]), eps=cfg["eps"],
                                        freqs_cis=t(cfg["freqs"]), n_out=cfg["n_out"],
                                        err_word=err, stream=stream)
    elif name == "store_fp4_1m":
        cfg = W.cfg4_gather()
        pool = torch.zeros(cfg["pool_rows"] * 288, dtype=torch.uint8, device=dev)
        call = B.prepare_compress_store(2, 1, bf(cfg["rows"]), t(cfg["ext"]), pool,
                                        page_table=t(cfg["page_table"]), page_bits=cfg["page_bits"],
                                        n_out=cfg["n_out"], err_word=err, stream=stream)
    elif name.startswith("gather_"):
        layout, rb = {"gather_v41": (1, 528), "gather_fp4": (2, 288), "gather_v4": (0, 584)}[name]
        cfg = W.cfg4_gather()
        pool = torch.zeros(cfg["pool_rows"] * rb, dtype=torch.uint8, device=dev)
        B.dsv4kv_compress_store(layout, 1, bf(cfg["rows"]), t(cfg["ext"]), pool,
                                page_table=t(cfg["page_table"]), page_bits=cfg["page_bits"],
                                n_out=cfg["n_out"], err_word=err, stream=stream)
        ids = t(cfg["ids"])
        out = torch.empty((ids.numel(), 512), dtype=torch.bfloat16, device=dev)
        call = B.prepare_dequant_gather(layout, pool, ids, out, err_word=err, stream=stream)
    else:
        n_req, n_new = (4096, 1) if name == "decode" else (1024, 4)
        cfg = W.decode_verify(seed=13, n_req=n_req, n_new=n_new, ring_size=4, max_prefix=4096)
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
        call = B.prepare_compress_store(1, 2, bf(cfg["rows"]), t(cfg["ext"]), pool,
                                        page_table=t(cfg["page_table"]), page_bits=6,
                                        rmsnorm_w=bf(cfg["norm_w"]), eps=cfg["eps"],
                                        freqs_cis=t(cfg["freqs"]), n_out=cfg["n_out"],
                                        err_word=err, stream=stream,
                                        start_pos=t(cfg["start_pos"]), ring=bf(cfg["ring"]))
    for _ in range(3):
        flusher()
        call()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, f"{int(err.item())} device faults"
    print(json.dumps({"profile_leg": name, "launches": 3 + (name.endswith("gather") or name.startswith("gather_"))}), flush=True)


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    from deepseek_v4_compressed_c2_gb300 import binding as B
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    B.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    l2_fetch = set_l2_fetch_granularity(args.l2_fetch_granularity)
    clocks = ClockSampler(local)
    clocks.start()
    cfg = make_inputs()

    def to_dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    rows = to_dev_bf16(cfg["rows"])
    ext = torch.from_numpy(cfg["ext"]).to(dev)
    pt = torch.from_numpy(cfg["page_table"]).to(dev)
    w = to_dev_bf16(cfg["norm_w"])
    freqs = torch.from_numpy(cfg["freqs"]).to(dev)
    topk = torch.from_numpy(cfg["topk"]).to(dev)
    ttr = torch.from_numpy(cfg["token_to_req"]).to(dev)
    n_store = cfg["n_out"]
    n_tok, k = cfg["topk"].shape
    n_slots = n_tok * k
    n_valid = gather_rows_valid(cfg)
    pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvbuf = B.SparsePrefillKVBuffer(torch.empty((n_slots, 512), dtype=torch.bfloat16, device=dev))
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))   # the zero fills before any launch
    launches = [0]
    store = B.prepare_compress_store(1, 2, rows, ext, pool, page_table=pt, page_bits=6,
                                     rmsnorm_w=w, eps=cfg["eps"], freqs_cis=freqs, n_out=n_store,
                                     err_word=err, stream=stream)
    gwh = B.prepare_get_with_head_topk(kvbuf, 1, pool, topk, ttr, pt, 6, err_word=err,
                                       stream=stream)

    def read_layers():
        kvbuf.dsv4kv_kvbuf_begin_forward()
        hits = [gwh() for _layer in range(LAYERS)]
        assert hits == [False] + [True] * (LAYERS - 1)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        store()
        if ev is not None:
            ev[1].record(stream)
        read_layers()
        if ev is not None:
            ev[2].record(stream)
        launches[0] += 2

    def barrier():
        if world > 1:
            dist.barrier()

    with clocks.busy("warmup"), torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, "device faults during warm-up"

    # ---- the timed region: K steps back to back, inputs resident in HBM
    # (537 MB of fused rows per step, larger than the L2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    launches[0] = 0
    with clocks.busy("timed_region"):
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(args.steps):
                step()
            t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    n_launch = launches[0]
    elapsed_ms = t0.elapsed_time(t1)

    # ---- per-kernel durations: KERNEL_SAMPLES more steps with events around
    # the store and around the gather (the events sit between the kernels, so
    # these steps do not overlap one launch's tail with the next's start)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KERNEL_SAMPLES)]
    with clocks.busy("per_kernel"), torch.cuda.stream(stream):
        for e in evs:
            step(e)
        torch.cuda.synchronize(dev)
    store_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    gather_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)

    # ---- end to end through host buffers (pinned host -> device -> host).
    # The batch is split into request chunks whose rows are contiguous; chunk
    # c's rows travel host -> device while chunk c-1 is stored and read, and
    # gathered rows travel back on a third stream.  Each chunk runs the same
    # sequence as the device-resident step: the store, then 4 layers' reads
    # through a reuse buffer (1 dequant + 3 hits) over its slice of the
    # output.  Each step moves every input row in and every gathered row out.
    n_req = len(cfg["lengths"])
    bounds = np.linspace(0, n_req, E2E_CHUNKS + 1).astype(int)
    first, counts = cfg["ext"][0].astype(np.int64), cfg["ext"][1].astype(np.int64)
    h_rows = torch.from_numpy(cfg["rows"].view(np.int16)).view(torch.bfloat16).pin_memory()
    d_rows = rows.clone()
    d_out = torch.empty((n_slots, 512), dtype=torch.bfloat16, device=dev)
    h_out = torch.empty((n_slots, 512), dtype=torch.bfloat16).pin_memory()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    chunks, h2d = [], 0
    for c in range(E2E_CHUNKS):
        r0, r1 = int(bounds[c]), int(bounds[c + 1])
        if r1 <= r0:
            continue
        row0, row1 = int(first[r0]), int(first[r1 - 1] + counts[r1 - 1])
        meta = {"ext": np.ascontiguousarray(cfg["ext"][:, r0:r1]),
                "pt": np.ascontiguousarray(cfg["page_table"][r0:r1]),
                "topk": np.ascontiguousarray(cfg["topk"][r0:r1]),
                "ttr": np.arange(r1 - r0, dtype=np.int32)}
        h_meta = {k2: torch.from_numpy(v).pin_memory() for k2, v in meta.items()}
        d_meta = {k2: v.to(dev) for k2, v in h_meta.items()}
        n_out_c = int((counts[r0:r1] // 2).sum())
        store_c = B.prepare_compress_store(1, 2, d_rows, d_meta["ext"], pool,
                                           page_table=d_meta["pt"], page_bits=6, rmsnorm_w=w,
                                           eps=cfg["eps"], freqs_cis=freqs, n_out=n_out_c,
                                           err_word=err, stream=stream)
        kv_c = B.SparsePrefillKVBuffer(d_out[r0 * k:r1 * k])
        gwh_c = B.prepare_get_with_head_topk(kv_c, 1, pool, d_meta["topk"], d_meta["ttr"],
                                             d_meta["pt"], 6, err_word=err, stream=stream)
        h2d += (row1 - row0) * rows.stride(0) * 2 + sum(v.numel() * v.element_size()
                                                         for v in h_meta.values())
        chunks.append(dict(rows=(row0, row1), out=(r0 * k, r1 * k), h=h_meta, d=d_meta,
                           store=store_c, kv=kv_c, gwh=gwh_c,
                           ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event(),
                           ev_out=torch.cuda.Event()))
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(3, min(args.steps, 30))

    def e2e_step():
        for ch in chunks:                          # inputs in
            with torch.cuda.stream(s_in):
                s_in.wait_event(ch["ev_done"])     # the previous step is done with them
                for k2 in ch["h"]:
                    ch["d"][k2].copy_(ch["h"][k2], non_blocking=True)
                a, b = ch["rows"]
                d_rows[a:b].copy_(h_rows[a:b], non_blocking=True)
                ch["ev_in"].record(s_in)
        for ch in chunks:                          # store + 4 layers' reads
            stream.wait_event(ch["ev_in"])
            stream.wait_event(ch["ev_out"])        # d_out chunk copied out by the last step
            ch["store"]()
            ch["kv"].dsv4kv_kvbuf_begin_forward()
            hits = [ch["gwh"]() for _layer in range(LAYERS)]
            assert hits == [False] + [True] * (LAYERS - 1)
            ch["ev_done"].record(stream)
        for ch in chunks:                          # gathered rows out
            with torch.cuda.stream(s_out):
                s_out.wait_event(ch["ev_done"])
                a, b = ch["out"]
                h_out[a:b].copy_(d_out[a:b], non_blocking=True)
                ch["ev_out"].record(s_out)
        launches[0] += 2 * len(chunks)

    torch.cuda.synchronize(dev)          # the chunks' device buffers are in place
    with clocks.busy("e2e"):
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        e0.record(s_in)
        for _ in range(e2e_steps):
            e2e_step()
        s_out.wait_event(chunks[-1]["ev_out"])
        e1.record(s_out)
        torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    assert int(err.item()) == 0, "device faults during the timed region"
    # the host copy of the gathered rows equals the device-resident step's
    assert torch.equal(h_out.view(torch.int16), kvbuf.storage[:n_slots].cpu().view(torch.int16))
    del d_rows, chunks

    # ---- the five workloads one by one, the other layouts, decode / verify
    peak, peak_kind = _peaks()
    configs = cold = decode = None
    cfg4 = None
    if not args.no_cold_gather:
        cfg4 = W.cfg4_gather()
        flusher = Flusher(dev)
        with clocks.busy("configs"):
            configs, _pool4, rows4, ids4 = config_legs(B, dev, stream, flusher, cfg4, peak)
            del _pool4
            cold = cold_paths(B, dev, stream, flusher, cfg4, rows4, ids4, peak)
            del rows4, ids4
            cold.update(c1_leg(B, dev, stream, flusher, cfg, rows, peak))
            del flusher
            torch.cuda.empty_cache()
        with clocks.busy("decode_verify"):
            decode = decode_verify_steps(B, dev, stream, max_prefix=args.decode_prefix)
    clk = clocks.stop()

    # ---- max over ranks
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)
    if rank != 0:
        return
    ms_per_step = elapsed_ms / args.steps
    units = n_store + n_valid
    value = whole_job_rate(units, world, ms_per_step)
    store_gbs = STORE_BYTES_PER_ROW * n_store / (store_ms / 1e3) / 1e9
    gather_bytes = GATHER_BYTES_PER_ROW * n_valid + PAD_BYTES_PER_ROW * (n_slots - n_valid)
    gather_gbs = gather_bytes / (gather_ms / 1e3) / 1e9
    traffic = _profiled_traffic("compress_store_long_prefill", STORE_SOURCES)
    step_bytes = STORE_BYTES_PER_ROW * n_store + gather_bytes
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": headline_config(cfg, world, l2_fetch),
        "roofline": {"bound": "hbm", "achieved": store_gbs, "peak": peak, "unit": "GB/s",
                     "frac": store_gbs / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "compress_store_kernel<V41, ratio 2, norm, rope>",
                     "bytes_per_row": STORE_BYTES_PER_ROW, "frac_of_8000": store_gbs / 8000.0,
                     "duration": f"median of {KERNEL_SAMPLES} in-step launches, CUDA events"},
        # the whole step against the same peak: both kernels' algorithmic bytes
        # over the step time (the gathered rows are written with evict-first
        # stores, so part of their write-back lands in the next store's time)
        "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "peak_kind": peak_kind,
                          "bytes_per_step": step_bytes},
        "kernels": {
            "compress_store": {"ms": store_ms, "rows_per_s": n_store / (store_ms / 1e3),
                               "gbs": store_gbs, "samples": KERNEL_SAMPLES},
            "dequant_gather_topk_x1_plus_3_hits": {"ms": gather_ms,
                                                  "rows_per_s": n_valid / (gather_ms / 1e3),
                                                  "gbs": gather_gbs, "samples": KERNEL_SAMPLES,
                                                  "bytes": gather_bytes}},
        "configs": configs,
        "cold_l2": cold,
        "decode_verify_ring": decode,
        "e2e": {"value": whole_job_rate(units, world, e2e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "sequence": f"{E2E_CHUNKS} request chunks, each: store, then {LAYERS} layers' "
                            f"reads through a reuse buffer (1 dequant + {LAYERS - 1} hits); "
                            "copies on two more streams"},
        "gpu_launches": n_launch,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
        if cfg4 is not None:
            line["oracle_per_config"] = oracle_per_config(
                {"cfg1": W.cfg1_v41_roundtrip(), "cfg2": W.cfg2_ratio2_small(),
                 "cfg3": W.cfg3_fp4_store(), "cfg4": cfg4})
            line["oracle_per_config"]["cfg5"] = {
                "name": cfg["name"],
                "store_and_gather": {
                    "rows_per_s_1core": line["cpu_baseline"]["single_thread"]["value"],
                    "rows_per_s_all_cores": line["cpu_baseline"]["value"],
                    "sample": line["cpu_baseline"]["sample"]}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cold-gather", action="store_true",
                    help="skip the per-workload, other-layout and decode / verify legs")
    ap.add_argument("--decode-only", action="store_true",
                    help="diagnostic: only the decode / verify ring-form launches, one JSON line")
    ap.add_argument("--decode-prefix", type=int, default=4096,
                    help="cached prefix bound of the decode / verify requests (sizes their pool)")
    ap.add_argument("--l2-fetch-granularity", type=int, default=32, choices=[0, 32, 64, 128],
                    help="this process's L2 fetch granularity in bytes (0: the context default)")
    ap.add_argument("--profile-leg", choices=PROFILE_LEGS,
                    help="diagnostic for ncu: one leg's three launches (L2 flushed before each), "
                         "no timing")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.profile_leg:
        profile_leg(args.profile_leg)
        return
    if args.decode_only:
        import torch
        from deepseek_v4_compressed_c2_gb300 import binding as B
        B.lib()
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        res = decode_verify_steps(B, dev, torch.cuda.Stream(device=dev),
                                  max_prefix=args.decode_prefix)
        if rank == 0:
            print(json.dumps({"decode_verify_ring": res, "decode_prefix": args.decode_prefix}),
                  flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
