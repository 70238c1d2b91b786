"""Benchmark of the compressed-KV write/read hot path on GB300.

One step = one long-prefill batch through the whole path:
  1. dsv4kv_compress_store: 64 requests (~262k tokens, lognormal lengths),
     ratio-2 softmax pair pooling of the fused | kv | score | rows, RMSNorm,
     RoPE, V41 quantization, paged store (page size 64);
  2. the sparse-prefill read of each request's top-2048 compressed ids: 4
     layers share the source; the first get_with_head_topk runs the fused
     top-k -> slot -> gather-dequant kernel, the other three are reuse hits.
value = (rows stored + rows gathered) / step time, inputs resident in HBM.
e2e   = the same through host buffers: pinned host -> device copy of the
        step's inputs and device -> host copy of the gathered rows inside the
        timed region (request chunks, copies overlapped with the kernels).

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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compressed-KV rows/s (store, gather-dequant) and achieved HBM GB/s vs 8 TB/s"
LAYERS = 4
EVENT_EVERY = 10     # steps between per-kernel event samples in the timed region
E2E_CHUNKS = 8
# algorithmic bytes per unit (what the method must move)
STORE_BYTES_PER_ROW = 2 * (1024 + 1024) + 256 + 528   # 2 x (kv + score) bf16, RoPE row, V41 row
GATHER_BYTES_PER_ROW = 528 + 4 + 1024                  # V41 row + id, bf16 row out


_CSRC = os.path.join("deepseek_v4_compressed_c2_gb300", "csrc")
STORE_SOURCES = [os.path.join(_CSRC, f) for f in
                 ("compress_store.cu", "quant.cuh", "tma.cuh", "layout.cuh", "internal.cuh")]


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
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
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
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def make_inputs(seed=7):
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    return W.cfg5_long_prefill(seed=seed)


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


def _oracle_sample(cfg, m):
    """The oracle as it stands, single-threaded: the batch's first m
    compressed rows (ratio-2 compress, RMSNorm, RoPE, V41 store) and m
    gathered rows.  Returns seconds."""
    import oracle
    n = cfg["n_out"]
    pool = np.zeros(cfg["pool_rows"] * 528, np.uint8)
    which = np.arange(m, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.compress_store(1, 2, cfg["rows"], cfg["ext"], page_table=cfg["page_table"],
                          page_bits=cfg["page_bits"], norm_w=cfg["norm_w"], eps=cfg["eps"],
                          freqs=cfg["freqs"], n_out=n, which=which, pool=pool,
                          pool_rows=cfg["pool_rows"], want_f64=False, want_f32=False,
                          want_latent=False)
    oracle.dequant_gather(1, pool, cfg["pool_rows"], np.arange(64, 64 + m, dtype=np.int32))
    return time.perf_counter() - t0


def _sample_rows(cfg, budget_s):
    """rows per oracle sample so that one sample takes about budget_s"""
    probe = min(256, cfg["n_out"])
    t = _oracle_sample(cfg, probe)
    return int(min(cfg["n_out"], max(16, probe * budget_s / max(t, 1e-6))))


def cpu_baseline(cfg, budget_s=10.0):
    """The oracle timed on the host cores on a bounded sample (~budget_s) of
    the same workload."""
    m = _sample_rows(cfg, budget_s)
    t = _oracle_sample(cfg, m)
    return {"value": 2 * m / t, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"first {m} of {cfg['n_out']} compressed rows of the batch (ratio-2 "
                      f"compress, RMSNorm, RoPE, V41 store) + {m} gathered rows, {t:.2f} s"}


def run_reference(args, rank):
    """The reference arm: the CPU oracle, on rank 0 only, each step a bounded
    sample sized so that warm-up + steps take about two minutes in all."""
    if rank != 0:
        return
    cfg = make_inputs()
    per_step = max(0.005, 120.0 / (args.steps + args.warmup))
    m = _sample_rows(cfg, per_step)
    for _ in range(args.warmup):
        _oracle_sample(cfg, m)
    secs = [_oracle_sample(cfg, m) for _ in range(args.steps)]
    t = statistics.median(secs)
    v = 2 * m / t
    sample = (f"first {m} of {cfg['n_out']} compressed rows (ratio-2 compress, RMSNorm, RoPE, "
              f"V41 store) + {m} gathered rows per step, median {t * 1e3:.1f} ms")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg["name"], "sample": sample},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _timed(fn, flush, stream, reps, scrub=None):
    """median CUDA-event time of fn() in ms, L2 flushed before each launch:
    a write of `flush` (512 MB, 4x the L2); with `scrub`, then a read of it
    (256 MB), which evicts the dirty lines of the write, so the timed kernel
    starts from a cold L2 that holds neither its inputs nor lines still to be
    written back"""
    import torch
    times = []
    with torch.cuda.stream(stream):
        for i in range(reps + 3):
            flush.fill_(i & 0xFF)
            if scrub is not None:
                scrub.max()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in times[3:])


def cold_gather(B, dev, stream, reps):
    """The store-only fill and the gather, each timed alone with a cold L2:
    1,048,576-row pools (page 0 reserved) in the V41, V41_FP4 and V4 layouts,
    filled by the ratio-1 store from bf16 N(0,1) latents (torch generator,
    seed 4); 262,144 unique row ids (numpy seed 4); between launches a 512 MB
    buffer written and a 256 MB one read (see _timed).  Also, per layout, the
    fake quantization of the same 1,048,512 latent rows (bf16 in, bf16 out),
    and on the V41 pool the short-context gather: 128 tokens of one request,
    each selecting every compressed row it sees (lengths uniform in
    [1, 2048], numpy seed 5)."""
    import torch
    pool_rows, n_ids = 1 << 20, 1 << 18
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    lat = torch.randn((pool_rows - 64, 512), generator=g, device=dev).to(torch.bfloat16)
    ext = torch.tensor([[0], [pool_rows - 64]], dtype=torch.int32, device=dev)
    pt = torch.arange(1, pool_rows // 64, dtype=torch.int32, device=dev).view(1, -1)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(4)
    ids = torch.from_numpy((rng.choice(pool_rows - 64, n_ids, replace=False) + 64)
                           .astype(np.int32)).to(dev)
    out = torch.empty((n_ids, 512), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    scrub = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
    peak, kind = _peaks()
    res = {}
    fq_out = torch.empty((pool_rows - 64, 512), dtype=torch.bfloat16, device=dev)
    for layout, name, rb in ((1, "v41", 528), (2, "fp4", 288), (0, "v4", 584)):
        pool = torch.zeros(pool_rows * rb, dtype=torch.uint8, device=dev)
        store = B.prepare_compress_store(layout, 1, lat, ext, pool, page_table=pt, page_bits=6,
                                         n_out=pool_rows - 64, err_word=err, stream=stream)
        gather = B.prepare_dequant_gather(layout, pool, ids, out, err_word=err, stream=stream)
        ms_s = _timed(store, flush, stream, max(3, reps // 5), scrub)
        ms_g = _timed(gather, flush, stream, reps, scrub)
        assert int(err.item()) == 0
        sb, gb = 1024 + rb, rb + 4 + 1024
        res[f"store_ratio1_{name}_1048512rows"] = {
            "ms": ms_s, "rows_per_s": (pool_rows - 64) / (ms_s / 1e3),
            "gbs": sb * (pool_rows - 64) / (ms_s / 1e3) / 1e9,
            "frac": sb * (pool_rows - 64) / (ms_s / 1e3) / 1e9 / peak, "bytes_per_row": sb}
        res[f"gather_{name}_262144_of_1048576"] = {
            "ms": ms_g, "rows_per_s": n_ids / (ms_g / 1e3), "gbs": gb * n_ids / (ms_g / 1e3) / 1e9,
            "frac": gb * n_ids / (ms_g / 1e3) / 1e9 / peak, "frac_of_8000": gb * n_ids / (ms_g / 1e3) / 8e12,
            "bytes_per_row": gb}
        ms_f = _timed(lambda: B.dsv4kv_fake_quant(layout, lat, fq_out, stream=stream), flush,
                      stream, max(3, reps // 5), scrub)
        res[f"fake_quant_{name}_1048512rows"] = {
            "ms": ms_f, "rows_per_s": (pool_rows - 64) / (ms_f / 1e3),
            "gbs": 2048 * (pool_rows - 64) / (ms_f / 1e3) / 1e9,
            "frac": 2048 * (pool_rows - 64) / (ms_f / 1e3) / 1e9 / peak, "bytes_per_row": 2048}
        if layout == 1:
            n_tok, k = 128, 2048
            lens_in = torch.from_numpy(np.random.default_rng(5).integers(1, k + 1, n_tok)
                                       .astype(np.int32)).to(dev)
            ttr = torch.zeros(n_tok, dtype=torch.int32, device=dev)
            ms_a = _timed(lambda: B.dsv4kv_dequant_gather_all(1, pool, lens_in, k, ttr, pt, 6,
                                                              out[:n_tok * k], err_word=err,
                                                              stream=stream),
                          flush, stream, reps, scrub)
            n_rows = int(lens_in.sum().item())
            # the same gather after the write-only flush: it also pays the
            # write-back of the flush's dirty lines
            ms_gd = _timed(gather, flush, stream, reps)
            res["gather_v41_262144_of_1048576_dirty_l2"] = {
                "ms": ms_gd, "gbs": 1556 * n_ids / (ms_gd / 1e3) / 1e9,
                "frac": 1556 * n_ids / (ms_gd / 1e3) / 1e9 / peak,
                "note": "L2 flushed by the 512 MB write alone; ~129 MB of its dirty lines are "
                        "written back during the gather"}
            res["gather_all_v41_128tok_2048"] = {
                "ms": ms_a, "rows": n_tok * k, "selected_rows": n_rows,
                "rows_per_s": n_tok * k / (ms_a / 1e3),
                "out_gbs": 1024 * n_tok * k / (ms_a / 1e3) / 1e9,
                "note": "every token of one request re-reads the same <= 2048 compressed rows "
                        "(L2-resident after the first); bound by the 1 KB/row output"}
        assert int(err.item()) == 0
        del pool
    res["peak_kind"] = kind
    return res


def decode_verify_steps(B, dev, stream, reps=50, max_prefix=4096):
    """The ring form of the compressor on decode-shaped steps (one new token
    per request; 1 + 3 draft tokens per request).  These are small,
    latency-bound launches (working set in L2).  The serving loop runs them
    inside a CUDA graph whose offsets are refreshed in place, so the device
    time per launch is taken from a captured graph of `reps` launches; the
    eager figure (one prepared C-ABI call per launch from Python) is kept
    beside it and includes the host's launch cost."""
    import torch
    from deepseek_v4_compressed_c2_gb300 import workloads as W
    res = {}
    for name, n_req, n_new in (("decode_4096req_1tok", 4096, 1), ("verify_1024req_4tok", 1024, 4)):
        cfg = W.decode_verify(seed=13, n_req=n_req, n_new=n_new, ring_size=4,
                              max_prefix=max_prefix)
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
        ring = bf(cfg["ring"])
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        rows = bf(cfg["rows"])
        ext = torch.from_numpy(cfg["ext"]).to(dev)
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
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        assert int(err.item()) == 0
        us = a.elapsed_time(b) * 1e3 / reps
        res[name] = {"us_per_launch": us, "eager_us_per_launch": eager_us, "rows": cfg["n_out"],
                     "tokens": n_req * n_new, "rows_per_s": cfg["n_out"] / (us / 1e6)}
        del graph
    return res


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    from deepseek_v4_compressed_c2_gb300 import binding as B
    B.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
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
    n_gather = n_tok * k
    pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvbuf = B.SparsePrefillKVBuffer(torch.empty((n_gather, 512), dtype=torch.bfloat16, device=dev))
    stream = torch.cuda.Stream(device=dev)
    launches = [0]

    def prepared(rows_t, ext_t, pt_t, topk_t, ttr_t):
        """the step's three C-ABI calls, marshalled once"""
        store = B.prepare_compress_store(1, 2, rows_t, ext_t, pool, page_table=pt_t, page_bits=6,
                                         rmsnorm_w=w, eps=cfg["eps"], freqs_cis=freqs,
                                         n_out=n_store, err_word=err, stream=stream)
        gwh = B.prepare_get_with_head_topk(kvbuf, 1, pool, topk_t, ttr_t, pt_t, 6, err_word=err,
                                           stream=stream)
        return store, gwh

    resident = prepared(rows, ext, pt, topk, ttr)

    def step(ev=None, calls=resident):
        store, gwh = calls
        if ev is not None:
            ev[0].record(stream)
        store()
        if ev is not None:
            ev[1].record(stream)
        kvbuf.dsv4kv_kvbuf_begin_forward()
        hits = [gwh() for _layer in range(LAYERS)]
        if ev is not None:
            ev[2].record(stream)
        assert hits == [False] + [True] * (LAYERS - 1)
        launches[0] += 2
        return kvbuf.storage

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, "device faults during warm-up"

    # ---- device-resident timing.  The per-kernel durations come from CUDA
    # events around the store and the gather on every EVENT_EVERY-th step of
    # the timed region: each event record costs ~2 us of stream time, so
    # events on every step would lengthen the step by ~4 %.
    ev_steps = list(range(0, args.steps, EVENT_EVERY))
    evs = {i: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for i in ev_steps}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    launches[0] = 0
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            step(evs.get(i))
        t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    n_launch = launches[0]
    elapsed_ms = t0.elapsed_time(t1)
    store_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs.values())
    gather_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs.values())

    # ---- end to end through host buffers (pinned host -> device -> host).
    # The batch is split into request chunks whose rows are contiguous; chunk
    # c's rows travel host -> device while chunk c-1 is stored and gathered,
    # and gathered rows travel back on a third stream.  Each step still moves
    # every input row in and every gathered row out.
    n_req = len(cfg["lengths"])
    bounds = np.linspace(0, n_req, E2E_CHUNKS + 1).astype(int)
    first, counts = cfg["ext"][0].astype(np.int64), cfg["ext"][1].astype(np.int64)
    h_rows = torch.from_numpy(cfg["rows"].view(np.int16)).view(torch.bfloat16).pin_memory()
    d_rows = rows.clone()
    d_out = torch.empty((n_gather, 512), dtype=torch.bfloat16, device=dev)
    h_out = torch.empty((n_gather, 512), dtype=torch.bfloat16).pin_memory()
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
        k_tok = cfg["topk"].shape[1]
        store_c = B.prepare_compress_store(1, 2, d_rows, d_meta["ext"], pool, page_table=d_meta["pt"],
                                           page_bits=6, rmsnorm_w=w, eps=cfg["eps"],
                                           freqs_cis=freqs, n_out=n_out_c, err_word=err,
                                           stream=stream)
        gather_c = B.prepare_dequant_gather_topk(1, pool, d_meta["topk"], d_meta["ttr"],
                                                 d_meta["pt"], 6, d_out[r0 * k_tok:r1 * k_tok],
                                                 err_word=err, stream=stream)
        h2d += (row1 - row0) * rows.stride(0) * 2 + sum(v.numel() * v.element_size()
                                                         for v in h_meta.values())
        chunks.append(dict(rows=(row0, row1), out=(r0 * k_tok, r1 * k_tok), h=h_meta, d=d_meta,
                           store=store_c, gather=gather_c,
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
        for ch in chunks:                          # store + gather
            stream.wait_event(ch["ev_in"])
            stream.wait_event(ch["ev_out"])        # d_out chunk copied out by the last step
            ch["store"]()
            ch["gather"]()
            ch["ev_done"].record(stream)
        for ch in chunks:                          # gathered rows out
            with torch.cuda.stream(s_out):
                s_out.wait_event(ch["ev_done"])
                a, b = ch["out"]
                h_out[a:b].copy_(d_out[a:b], non_blocking=True)
                ch["ev_out"].record(s_out)
        launches[0] += 2 * len(chunks)

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
    assert torch.equal(h_out.view(torch.int16), kvbuf.storage[:n_gather].cpu().view(torch.int16))

    # ---- the gather alone on a cold L2: a 1 Mi-row V41 pool (553 MB), 262,144
    # unique random ids, L2 flushed (a 512 MB write) before every launch
    cold = None
    if not args.no_cold_gather:
        cold = cold_gather(B, dev, stream, max(5, min(args.steps, 50)))
        decode = decode_verify_steps(B, dev, stream, max_prefix=args.decode_prefix)
    else:
        decode = None

    # ---- max over ranks
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)
    if rank != 0:
        return
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(n_store + n_gather, world, ms_per_step)
    peak, peak_kind = _peaks()
    store_gbs = STORE_BYTES_PER_ROW * n_store / (store_ms / 1e3) / 1e9
    gather_gbs = GATHER_BYTES_PER_ROW * n_gather / (gather_ms / 1e3) / 1e9
    traffic = _profiled_traffic("compress_store_long_prefill", STORE_SOURCES)
    step_bytes = STORE_BYTES_PER_ROW * n_store + GATHER_BYTES_PER_ROW * n_gather
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "requests": len(cfg["lengths"]),
                   "tokens": int(sum(cfg["lengths"])), "store_rows": n_store,
                   "gather_rows": n_gather, "layers_reading_source": LAYERS, "layout": "V41",
                   "ratio": 2, "page_size": 64, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (fused rows %d MB per step)"
                         % (cfg["rows"].nbytes // 10 ** 6)},
        "roofline": {"bound": "hbm", "achieved": store_gbs, "peak": peak, "unit": "GB/s",
                     "frac": store_gbs / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "compress_store_kernel<V41, ratio 2, norm, rope>",
                     "bytes_per_row": STORE_BYTES_PER_ROW, "frac_of_8000": store_gbs / 8000.0},
        # the whole step against the same peak: both kernels' algorithmic bytes
        # over the step time (the gathered rows are written with evict-first
        # stores, so part of their write-back lands in the next store's time)
        "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "peak_kind": peak_kind,
                          "bytes_per_step": step_bytes},
        "kernels": {
            "compress_store": {"ms": store_ms, "rows_per_s": n_store / (store_ms / 1e3),
                               "gbs": store_gbs},
            "dequant_gather_topk_x1_plus_3_hits": {"ms": gather_ms,
                                              "rows_per_s": n_gather / (gather_ms / 1e3),
                                              "gbs": gather_gbs}},
        "cold_l2": cold,
        "decode_verify_ring": decode,
        "e2e": {"value": whole_job_rate(n_store + n_gather, world, e2e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": n_launch,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cold-gather", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="diagnostic: only the decode / verify ring-form launches, one JSON line")
    ap.add_argument("--decode-prefix", type=int, default=4096,
                    help="cached prefix bound of the decode / verify requests (sizes their pool)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
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
