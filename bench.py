#!/usr/bin/env python
"""Benchmark of the block-paged KV-cache hot path on GB300.

One step = one pass of the path over the decode-sized gather batch (fp16 pool of
10000 pages x 16 slots x 32 heads x 128 dims, 64 sequences of U[512, 4096] tokens,
uint32 block tables from a shuffled free list): hp_plan (device validation of the
descriptor + ragged prefix sums) then hp_gather_planned (the page-span copy), both
through the C ABI.  The metric is effective HBM GB/s (algorithmic bytes read and
written per step / step time).

Printed: one JSON line (rank 0) with the headline value, the roofline of the copy
kernel, the CPU oracle timed on a bounded sample, an end-to-end figure through host
buffers, and per-operation measurements of the other rows of the path (append,
prefix sharing, dequantising gather, per-lane layout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Under torchrun each rank runs its own replica of the batch on its own GPU (no
collective on the data path); the time is the max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (bytes read+written) of paged gather/scatter, % of roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_hp_gb300", "csrc", f)
                  for f in ("hp_bulk.cu", "hp_resolve.cuh")]


# ----------------------------------------------------------------------------- helpers
def peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(paths):
    m = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            m.update(f.read())
    return m.hexdigest()[:16]


def recorded_traffic(kernel_key, units_now):
    """DRAM bytes per launch from a committed ncu summary, scaled to this launch's
    units, or None when the summary is absent or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key]
    except Exception:
        return None
    srcs = [os.path.join(ROOT, p) for p in rec.get("source", [])]
    if not srcs or rec.get("source_sha256_16") != source_hash(srcs):
        return None
    return rec["dram_bytes_per_unit"] * units_now


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 7:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[3:7]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def idx_tensor(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    v = a.view(np.int32) if a.dtype == np.uint32 else a.astype(np.uint64).view(np.int64)
    return torch.from_numpy(v.copy()).to(dev)


def gather_bytes(w, lens=None):
    """Algorithmic bytes of one gather of the batch: every valid row read once and
    written once, plus one block-table entry per page span."""
    lens = (w.lens if lens is None else lens).astype(np.int64)
    T = int(lens.sum())
    spans = int((-(-lens // w.page_size)).sum())
    ib = 4 if w.index_dtype == np.uint32 else 8
    return 2 * T * w.row_bytes + spans * ib, spans


def validate_bytes(w):
    ib = 4 if w.index_dtype == np.uint32 else 8
    return len(w.table) * ib + (2 * w.num_seqs + 1) * ib


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(step_bytes, steps, world, total_ms):
    """Every rank moves step_bytes per step (weak scaling); the job's time is the
    slowest rank's."""
    return world * step_bytes * steps / (total_ms * 1e-3) / 1e9


# ----------------------------------------------------------------------------- device arm
class GatherStep:
    """Resident device buffers of one gather batch and the two C-ABI calls of a step."""

    def __init__(self, w, dev, hp, inputs):
        import torch
        self.w, self.hp = w, hp
        self.pool = inputs.device_pool(w, dev)
        self.table = idx_tensor(w.table, dev)
        self.seq_ptr = idx_tensor(w.seq_ptr, dev)
        self.lens = idx_tensor(w.lens, dev)
        self.scales = inputs.device_scales(w, dev) if w.scales_seed is not None else None
        self.dequant = self.scales is not None
        self.desc = hp.PagedDesc(self.pool, self.table, self.seq_ptr, self.lens,
                                 num_pages=w.num_pages, page_size=w.page_size,
                                 num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype,
                                 index_type=0 if w.index_dtype == np.uint32 else 1,
                                 scales=self.scales, flags=hp.HAS_QUANT if self.dequant else 0)
        self.ws = hp.workspace_for(self.desc, dev)
        self.T = w.total_tokens
        ob = self.T * w.num_heads * w.head_dim * (2 if self.dequant else inputs.ELEM_BYTES[w.dtype])
        self.out = torch.empty(ob, dtype=torch.uint8, device=dev)
        self.status = torch.full((1,), -12345, dtype=torch.int32, device=dev)

    def plan(self, stream):
        rc = self.hp.hp_plan(self.desc, self.T, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def copy(self, stream):
        f = self.hp.hp_gather_dequant_planned if self.dequant else self.hp.hp_gather_planned
        rc = f(self.desc, self.out, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def check_status(self):
        st = int(self.status.item())
        assert st == 0, self.hp.status_name(st)


def time_steps(step, steps, warmup, stream, dist=None):
    """Warm-up, then `steps` timed steps (plan + copy, nothing between them) bracketed
    by barrier + synchronize.  Returns (per-step ms list, wall seconds)."""
    import torch
    for _ in range(warmup):
        step.plan(stream)
        step.copy(stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for e0, e1 in ev:
        e0.record(stream)
        step.plan(stream)
        step.copy(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    step.check_status()
    return [a.elapsed_time(b) for a, b in ev], wall


def time_copy_kernel(step, launches, stream):
    """The copy kernel alone, each launch between its own pair of events on the
    launching stream (the plan of the last step stays valid)."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(launches)]
    torch.cuda.synchronize()
    for e0, e1 in ev:
        e0.record(stream)
        step.copy(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    step.check_status()
    return [a.elapsed_time(b) for a, b in ev]


def e2e_host_buffers(w, dev, inputs):
    """The end-to-end measurement's pinned host buffers: the pool (filled from the seeded
    device pool) and two output buffers, shared by every e2e_gather call."""
    import torch
    pool_dev = inputs.device_pool(w, dev)
    h_pool = torch.empty(pool_dev.shape, dtype=torch.uint8, pin_memory=True)
    h_pool.copy_(pool_dev)
    del pool_dev
    n = w.total_tokens * w.row_bytes
    return dict(pool=h_pool, outs=[torch.empty(n, dtype=torch.uint8, pin_memory=True)
                                   for _ in range(2)])


def e2e_gather(w, dev, hp, inputs, steps, upload_pool=True, host=None):
    """The same step through host buffers: every step uploads the pool and index buffers
    from pinned host memory, gathers through the C ABI and downloads the gathered tensor
    to pinned host memory.  Steps are pipelined over two device buffer sets and three
    streams (upload, gather, download), so step k+1's upload overlaps step k's download;
    a buffer set is reused only after the gather that read it and the download that read
    its output have finished.  upload_pool=False keeps the pool resident on the device
    (uploaded once, before the timed steps) and uploads only the index buffers."""
    import torch
    if host is None:
        host = e2e_host_buffers(w, dev, inputs)
    h_pool = host["pool"]
    host_idx = [torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).pin_memory()
                for a in (w.table, w.seq_ptr, w.lens)]
    T = w.total_tokens
    sets = []
    for i in range(2):
        d_pool = torch.empty(h_pool.shape, dtype=torch.uint8, device=dev)
        d_idx = [torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_idx]
        desc = hp.PagedDesc(d_pool, d_idx[0], d_idx[1], d_idx[2], num_pages=w.num_pages,
                            page_size=w.page_size, num_heads=w.num_heads,
                            head_dim=w.head_dim, dtype=w.dtype, index_type=0)
        sets.append(dict(pool=d_pool, idx=d_idx, desc=desc, ws=hp.workspace_for(desc, dev),
                         status=torch.zeros(1, dtype=torch.int32, device=dev),
                         out=torch.empty(T * w.row_bytes, dtype=torch.uint8, device=dev),
                         h_out=host["outs"][i],
                         gathered=None, downloaded=None))
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def one(k, first=False):
        b = sets[k % 2]
        with torch.cuda.stream(up):
            if b["gathered"] is not None:
                up.wait_event(b["gathered"])  # the last gather through this set is done
            if upload_pool or first:
                b["pool"].copy_(h_pool, non_blocking=True)
            for d, h in zip(b["idx"], host_idx):
                d.copy_(h, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(up)
        comp.wait_event(uploaded)
        if b["downloaded"] is not None:
            comp.wait_event(b["downloaded"])  # its output buffer has been read back
        rc = hp.hp_gather(b["desc"], b["out"], T, b["ws"], b["status"], stream=comp)
        assert rc == 0
        b["gathered"] = torch.cuda.Event()
        b["gathered"].record(comp)
        down.wait_event(b["gathered"])
        with torch.cuda.stream(down):
            b["h_out"].copy_(b["out"], non_blocking=True)
            b["downloaded"] = torch.cuda.Event()
            b["downloaded"].record(down)

    for k in range(2):
        one(k, first=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for k in range(steps):
        one(k)
    main = torch.cuda.current_stream()
    main.wait_stream(down)
    e1.record(main)
    torch.cuda.synchronize()
    assert all(int(b["status"].item()) == 0 for b in sets)
    ms = e0.elapsed_time(e1) / steps
    h2d = (h_pool.numel() if upload_pool else 0) + sum(h.numel() * h.element_size()
                                                       for h in host_idx)
    return ms, h2d, T * w.row_bytes


def e2e_gather_in_place(w, dev, hp, inputs, steps, host):
    """The same steps with the pool left in pinned host memory and the output written
    straight into pinned host memory: every step uploads only its index buffers, and the
    gather reads the live pages over the host link and writes the rows back over it (the
    library routes host-resident memory to its register copy engine).  Two index and
    output buffer sets alternate, as in e2e_gather."""
    import torch
    h_pool = host["pool"]
    host_idx = [torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).pin_memory()
                for a in (w.table, w.seq_ptr, w.lens)]
    T = w.total_tokens
    stream = torch.cuda.current_stream()
    sets = []
    for i in range(2):
        d_idx = [torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_idx]
        desc = hp.PagedDesc(h_pool, d_idx[0], d_idx[1], d_idx[2], num_pages=w.num_pages,
                            page_size=w.page_size, num_heads=w.num_heads,
                            head_dim=w.head_dim, dtype=w.dtype, index_type=0,
                            flags=hp.HOST_MEMORY)
        sets.append(dict(idx=d_idx, desc=desc, ws=hp.workspace_for(desc, dev),
                         status=torch.zeros(1, dtype=torch.int32, device=dev),
                         h_out=host["outs"][i]))

    def one(k):
        b = sets[k % 2]
        for d, h in zip(b["idx"], host_idx):
            d.copy_(h, non_blocking=True)
        assert hp.hp_gather(b["desc"], b["h_out"], T, b["ws"], b["status"], stream=stream) == 0

    for k in range(2):
        one(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        one(k)
    e1.record(stream)
    torch.cuda.synchronize()
    assert all(int(b["status"].item()) == 0 for b in sets)
    ms = e0.elapsed_time(e1) / steps
    live = int((-(-w.lens.astype(np.int64) // w.page_size)).sum())  # spans read
    h2d = T * w.row_bytes + sum(h.numel() * h.element_size() for h in host_idx)
    return ms, h2d, T * w.row_bytes, live


# ----------------------------------------------------------------------------- oracle arm
def _oracle_desc_for(w, host_pool, seqs_upto, tokens_cap, oracle_mod):
    lens = w.lens.astype(np.int64)[:seqs_upto].copy()
    if tokens_cap is not None:
        c = np.cumsum(lens)
        k = int(np.searchsorted(c, tokens_cap))
        lens = lens[:k + 1].copy()
        prev = int(c[k - 1]) if k > 0 else 0
        lens[-1] = max(1, min(int(lens[-1]), tokens_cap - prev))
    n = len(lens)
    sp = w.seq_ptr[:n + 1].astype(w.index_dtype)
    table = w.table[:int(sp[-1])]
    d = oracle_mod.Desc(host_pool, table, sp, lens.astype(w.index_dtype), num_pages=w.num_pages,
                        page_size=w.page_size, num_heads=w.num_heads, head_dim=w.head_dim,
                        dtype=w.dtype, index_type=0 if w.index_dtype == np.uint32 else 1)
    return d, lens


def time_oracle(w, host_pool, oracle_mod, budget_s, max_tokens=None):
    """Oracle gather on a prefix of the batch sized to take about budget_s seconds."""
    tokens = 256
    while True:
        d, lens = _oracle_desc_for(w, host_pool, w.num_seqs, tokens, oracle_mod)
        t0 = time.perf_counter()
        d.gather()
        dt = time.perf_counter() - t0
        T = int(lens.sum())
        if dt >= budget_s * 0.5 or T >= w.total_tokens or (max_tokens and T >= max_tokens):
            break
        scale = max(2.0, min(16.0, budget_s / max(dt, 1e-4)))
        tokens = int(min(w.total_tokens, tokens * scale))
        if max_tokens:
            tokens = min(tokens, max_tokens)
    b, _ = gather_bytes(w, lens)
    return b / dt / 1e9, dt, T, lens


class OracleThreads:
    """The oracle gather, as it stands, on nthreads host threads over the first
    `tokens_cap` tokens of the batch (all of it when None): the sequences are cut into
    nthreads contiguous groups, each gathered by one call through its own sub-descriptor
    (ctypes releases the GIL during the call)."""

    def __init__(self, w, host_pool, oracle_mod, nthreads, tokens_cap=None):
        from concurrent.futures import ThreadPoolExecutor
        _, lens = _oracle_desc_for(w, host_pool, w.num_seqs, tokens_cap, oracle_mod)
        lens = lens.astype(np.int64)
        n = len(lens)
        cuts = np.linspace(0, n, min(nthreads, n) + 1).astype(int)
        self.descs, self.outs = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            if b <= a:
                continue
            sp = (w.seq_ptr[a:b + 1].astype(np.int64) - int(w.seq_ptr[a])).astype(w.index_dtype)
            table = w.table[int(w.seq_ptr[a]):int(w.seq_ptr[b])]
            d = oracle_mod.Desc(host_pool, table, sp, lens[a:b].astype(w.index_dtype),
                                num_pages=w.num_pages, page_size=w.page_size,
                                num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype,
                                index_type=0 if w.index_dtype == np.uint32 else 1)
            self.descs.append(d)
            self.outs.append(np.zeros((d.total_tokens(), w.row_bytes), dtype=np.uint8))
        self.pool = ThreadPoolExecutor(max(1, len(self.descs)))
        self.tokens = int(lens.sum())
        self.bytes, _ = gather_bytes(w, lens)
        self.threads = len(self.descs)

    def step(self):
        faults = list(self.pool.map(lambda i: self.descs[i].gather(self.outs[i])[2],
                                    range(len(self.descs))))
        assert all(f == "OK" for f in faults), faults

    def close(self):
        self.pool.shutdown()


def host_threads():
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def time_oracle_threads(w, host_pool, oracle_mod, nthreads):
    """The threaded oracle gather of the whole batch: (GB/s, seconds, threads used)."""
    r = OracleThreads(w, host_pool, oracle_mod, nthreads)
    r.step()  # page in
    t0 = time.perf_counter()
    r.step()
    dt = time.perf_counter() - t0
    r.close()
    return r.bytes / dt / 1e9, dt, r.threads


# ----------------------------------------------------------------------------- ops
def release_device_memory():
    """Return cached blocks to the driver, then give it time to clear what was freed: for
    a few milliseconds after a release of tens of GB, that clearing competes with the next
    kernel for HBM (a copy then ran 0.55 ms instead of 0.41 ms for its first eight calls)."""
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    time.sleep(0.2)


def median_ms(fn, stream, n=20, warm=3, between=None):
    """Median of n CUDA-event timings of fn() on `stream`, after `warm` untimed calls;
    `between` (untimed) runs before each timed call, e.g. an L2 scrub.  A spin kernel of
    about 0.1 ms (no memory traffic) precedes each timed call, so the launches of fn() are
    queued by the time the first event fires: the time is the device's, as in a loop that
    keeps the queue full, not the host's launch latency."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(n):
        if between is not None:
            between()
        if hasattr(torch.cuda, "_sleep"):
            with torch.cuda.stream(stream):
                torch.cuda._sleep(200000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def rate_entry(bytes_, ms, peak, **kw):
    gbps = bytes_ / (ms * 1e-3) / 1e9
    return dict(ms=round(ms, 4), gbps=round(gbps, 1), frac=round(gbps / peak, 4), **kw)


def attention_only(scale, dev, hp, inputs, peak, reps, host_kv=False):
    """Decode attention alone on the decode-append batch at `scale` ("full": 256 sequences
    of 1K-32K tokens; "mid": 32 of them, about 2.5 GB on the device, the profiler's case;
    "short": 2048 sequences of 16-1024 tokens); host_kv: K and V in page-locked host
    memory."""
    import torch
    w = inputs.config("decode_append", scale)
    pool = inputs.device_pool(w, dev)
    hk = None
    if host_kv:
        hk = torch.empty(pool.shape, dtype=pool.dtype, pin_memory=True)
        hk.copy_(pool)
        pool = hk
    d_k = hp.PagedDesc(pool, idx_tensor(w.table, dev), idx_tensor(w.seq_ptr, dev),
                       idx_tensor(w.lens, dev), num_pages=w.num_pages, page_size=w.page_size,
                       num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype, index_type=0)
    stream = torch.cuda.current_stream()
    res = attention_measurement(dev, hp, inputs, w, d_k, peak,
                                lambda b, ms, **kw: rate_entry(b, ms, peak, **kw),
                                lambda fn, n: median_ms(fn, stream, n), reps=reps, host_kv=hk)
    res.update(op="decode_attention", workload=w.name, num_seqs=w.num_seqs,
               total_tokens=w.total_tokens, num_heads=w.num_heads, head_dim=w.head_dim,
               kv_memory="page-locked host" if host_kv else "device")
    return res


def lane_only(dev, hp, inputs, peak, reps):
    """The per-lane snapshot gather of the lane_synthetic layout ([512, 32, 8, 16, 128]
    bf16, 256 lanes of about 6,555 rows)."""
    import torch
    lw = inputs.lane_synthetic()
    g = torch.Generator(device=dev)
    g.manual_seed(lw.seed)
    lpool = torch.randn(lw.pool_shape, generator=g, device=dev).to(torch.bfloat16)
    lt = torch.from_numpy(lw.table.view(np.int64).copy()).to(dev)
    lo = torch.empty((lw.batch, lw.kv_heads, lw.n, lw.width), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    ms = median_ms(lambda: hp.hp_lane_gather(lpool, lt, lw.capacity, lw.page_tokens, lw.batch,
                                             lw.kv_heads, lw.width, "bf16", lw.n, lo, status),
                   stream, reps)
    assert int(status.item()) == 0
    res = rate_entry(2 * lw.lanes * lw.n * lw.width * 2 + lw.pages * 8, ms, peak)
    res.update(op="lane_gather", lanes=lw.lanes, rows=lw.n)
    # the same 4 KiB runs (every lane's pages, in the snapshot's order) gathered by torch's
    # index_select over the pool seen as 4 KiB rows: the access pattern's own rate on this
    # GPU, for reading the fraction above
    used = -(-lw.n // lw.page_tokens)
    pg = torch.from_numpy(lw.table[:used].astype(np.int64)).to(dev)
    lane_ids = torch.arange(lw.batch * lw.kv_heads, device=dev)
    idx = (pg[None, :] * (lw.batch * lw.kv_heads) + lane_ids[:, None]).reshape(-1)
    rows = lpool.view(-1, lw.page_tokens * lw.width)
    dst = torch.empty((idx.numel(), rows.shape[1]), dtype=rows.dtype, device=dev)
    ms_t = median_ms(lambda: torch.index_select(rows, 0, idx, out=dst), stream, reps)
    res["torch_index_select_same_runs"] = rate_entry(2 * dst.numel() * 2 + idx.numel() * 8,
                                                     ms_t, peak)
    return res


def decode_step_only(dev, hp, inputs, steps):
    """The decode append step alone (one new row for each of 256 sequences of the
    decode_append batch), validated and permissive, issued back to back; then the
    zeroing of the grown batch's dead slots."""
    import torch
    w = inputs.config("decode_append")
    pool = inputs.device_pool(w, dev)
    table, sp = idx_tensor(w.table, dev), idx_tensor(w.seq_ptr, dev)
    before, new_ptr = idx_tensor(w.lens_before, dev), idx_tensor(w.new_ptr, dev)
    new = inputs.device_new_rows(w, dev)
    kw = dict(num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
              head_dim=w.head_dim, dtype=w.dtype, index_type=0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    res = {"op": "decode_append_step", "rows": w.total_new}
    for flags, name in ((0, "validated"), (1, "permissive")):
        d = hp.PagedDesc(pool, table, sp, before, flags=flags, **kw)
        ws = hp.workspace_for(d, dev)
        one = lambda: hp.hp_scatter_append(d, new, new_ptr, w.total_new, ws, status)
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            one()
        b.record(stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, hp.status_name(int(status.item()))
        res[name + "_us_back_to_back"] = round(a.elapsed_time(b) / steps * 1e3, 2)
    # zeroing the slots past every sequence's count after the step (273k table entries)
    d = hp.PagedDesc(pool, table, sp, idx_tensor(w.lens, dev), **kw)
    ws = hp.workspace_for(d, dev)
    rc, nsc = hp.hp_zero_tails_scratch_bytes(d)
    scratch = torch.empty(nsc, dtype=torch.uint8, device=dev)
    for _ in range(3):
        hp.hp_zero_tails(d, ws, scratch, status)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        hp.hp_zero_tails(d, ws, scratch, status)
    b.record(stream)
    torch.cuda.synchronize()
    res["zero_tails_us_back_to_back"] = round(a.elapsed_time(b) / steps * 1e3, 2)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    return res


def transpose_only(dev, hp, peak, reps, nb=10000, bsz=16, H=32, D=128, x=8):
    """Both cache layout conversions on a [nb, bs, H, D] fp16 cache (1.31 GB each way)."""
    import torch
    stream = torch.cuda.current_stream()
    kin = torch.empty(nb * bsz * H * D * 2, dtype=torch.uint8, device=dev)
    kout = torch.empty_like(kin)
    res = {"op": "cache_layout_conversions", "shape": [nb, bsz, H, D], "x": x, "dtype": "f16"}
    ms = median_ms(lambda: hp.hp_from_kernel_layout(kin, kout, nb, bsz, H, D, x, "f16"), stream, reps)
    res["kernel_layout_to_interchange"] = rate_entry(2 * kin.numel(), ms, peak)
    ms = median_ms(lambda: hp.hp_to_kernel_layout(kout, kin, nb, bsz, H, D, x, "f16"), stream, reps)
    res["interchange_to_kernel_layout"] = rate_entry(2 * kin.numel(), ms, peak)
    return res


def attention_measurement(dev, hp, inputs, w, d_k, peak, entry, med_ms, Hq=32, reps=10,
                          host_kv=None):
    """hp_attention_decode over batch w (K pool and descriptor d_k; a V pool of the same
    geometry is drawn here): Hq query heads, bytes = K and V rows once + q + out.
    host_kv: a page-locked host copy of the K pool; then d_k reads it and V is copied to
    page-locked host memory too (an offloaded cache read over the host link)."""
    import torch
    wv = inputs.Workload(**{**w.__dict__, "pool_seed": w.pool_seed + 77})
    vpool = inputs.device_pool(wv, dev)
    if host_kv is not None:
        vh = torch.empty(vpool.shape, dtype=vpool.dtype, pin_memory=True)
        vh.copy_(vpool)
        vpool = vh
    gq = torch.Generator(device=dev)
    gq.manual_seed(11)
    qd = torch.randn((w.num_seqs, Hq, w.head_dim), generator=gq, device=dev).to(torch.bfloat16)
    ao = torch.empty((w.num_seqs, Hq, w.head_dim), dtype=torch.float32, device=dev)
    rc, nws = hp.hp_attention_decode_workspace_bytes(d_k, Hq)
    assert rc == 0
    aws = torch.zeros(nws, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ms = med_ms(lambda: hp.hp_attention_decode(d_k, vpool, qd, Hq, 1 / np.sqrt(w.head_dim), ao,
                                               aws, status), n=reps)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    kv_bytes = 2 * w.total_tokens * w.row_bytes
    nbytes = kv_bytes + qd.numel() * 2 + ao.numel() * 4
    res = entry(nbytes, ms,
                note="K and V rows read once; %d query heads, GQA %d" % (Hq, Hq // w.num_heads))
    # the per-layer cost when one plan serves every layer of a decode step: the planned
    # call alone (attention kernel only)
    assert hp.hp_attention_plan(d_k, Hq, aws, status) == 0
    ms_p = med_ms(lambda: hp.hp_attention_decode_planned(d_k, vpool, qd, Hq,
                                                         1 / np.sqrt(w.head_dim), ao, aws,
                                                         status), n=reps)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    res["planned_call"] = entry(nbytes, ms_p, note="hp_attention_decode_planned after one "
                                "hp_attention_plan (per layer of a decode step)")
    del vpool, aws
    release_device_memory()
    return res


def dequant_measurements(dev, hp, inputs, entry, med_ms):
    """The dequantising gathers on the quantized_pool batch (int8 codes -> bf16): per-slot
    scales, then the other schemes of [HF] Per-scheme composition with zero points."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    w = inputs.config("quantized_pool")
    st = GatherStep(w, dev, hp, inputs)
    T = w.total_tokens
    spans = int((-(-w.lens.astype(np.int64) // w.page_size)).sum())
    b = T * (w.num_heads * w.head_dim * 3 + 4) + spans * 8
    st.plan(stream)
    ms = med_ms(lambda: st.copy(stream), n=10)
    out["quantized_pool_dequant_gather"] = entry(b, ms)
    st.check_status()
    g = torch.Generator(device=dev)
    g.manual_seed(w.scales_seed + 1)
    for name, tag, axis, count in (("per_tensor", 0x01, 0, 1),
                                   ("per_channel_heads", 0x02, 1, w.num_heads),
                                   ("per_channel_head_dim", 0x02, 2, w.head_dim),
                                   ("per_slot_affine", 0x03, 0, w.num_pages * w.page_size)):
        sc = torch.rand(count, generator=g, device=dev) * 0.049 + 0.001
        zp = torch.randint(-20, 21, (count,), generator=g, device=dev,
                           dtype=torch.int8).view(torch.uint8)
        q = hp.quant_desc(tag, sc, zp, axis=axis, block_size=w.page_size if tag == 3 else 0)
        ms = med_ms(lambda: hp.hp_gather_dequant_q_planned(st.desc, q, st.out, st.ws, st.status),
                    n=5)
        # b counts a 4-byte scale per row; per-slot zero points add one byte per row, the
        # other schemes' parameters are a few hundred bytes read from cache
        nbytes = b + T if tag == 3 else b - 4 * T
        out["quantized_pool_dequant_" + name + "_zp"] = entry(nbytes, ms)
        st.check_status()
    del st
    release_device_memory()
    return out


def decode_step_layers(dev, hp, inputs, entry, med_ms, layers=4, Hq=32):
    """A decode step of a `layers`-layer model on the 32-sequence decode-append batch:
    one append plan and one attention plan serve every layer, and each layer appends its
    new K and V rows and runs attention through the shared block table.  Bytes: each
    layer's K and V rows read once by attention, plus its appended rows (read + written)."""
    import torch
    w = inputs.config("decode_append", "mid")
    kw = dict(num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
              head_dim=w.head_dim, dtype=w.dtype, index_type=0)
    table, sp = idx_tensor(w.table, dev), idx_tensor(w.seq_ptr, dev)
    before, after = idx_tensor(w.lens_before, dev), idx_tensor(w.lens, dev)
    new_ptr = idx_tensor(w.new_ptr, dev)
    new = inputs.device_new_rows(w, dev)
    pools = []
    for l in range(layers):
        kp = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 2000 + 2 * l}), dev)
        vp = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 2001 + 2 * l}), dev)
        pools.append((kp, vp, hp.PagedDesc(kp, table, sp, before, **kw),
                      hp.PagedDesc(vp, table, sp, before, **kw),
                      hp.PagedDesc(kp, table, sp, after, **kw)))
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    q = torch.randn((w.num_seqs, Hq, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((w.num_seqs, Hq, w.head_dim), dtype=torch.float32, device=dev)
    d_before, d_after = pools[0][2], pools[0][4]
    ws_a = hp.workspace_for(d_before, dev)
    rc, nws = hp.hp_attention_decode_workspace_bytes(d_after, Hq)
    ws_t = torch.zeros(nws, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1 / np.sqrt(w.head_dim)

    def step():
        hp.hp_append_plan(d_before, new_ptr, w.total_new, ws_a, status)
        for kp, vp, dk, dv, _ in pools:
            hp.hp_scatter_append_planned(dk, new, new_ptr, w.total_new, ws_a, status)
            hp.hp_scatter_append_planned(dv, new, new_ptr, w.total_new, ws_a, status)
        hp.hp_attention_plan(d_after, Hq, ws_t, status)
        for kp, vp, _, _, dka in pools:
            hp.hp_attention_decode_planned(dka, vp, q, Hq, scale, out, ws_t, status)

    ms = med_ms(step, n=10)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    nbytes = layers * (2 * w.total_tokens * w.row_bytes + q.numel() * 2 + out.numel() * 4 +
                       2 * 2 * w.total_new * w.row_bytes)
    res = entry(nbytes, ms, note="%d layers of %d sequences: per step 1 append plan, %d "
                "planned appends, 1 attention plan, %d planned attention calls" %
                (layers, w.num_seqs, 2 * layers, layers))
    del pools
    return res


def ops_measurements(dev, hp, inputs, peak, reps=20):
    """The other rows of the path at their own configurations (bytes as in
    gather_bytes; medians over reps, inputs larger than L2 except where noted)."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()

    def med_ms(fn, n=reps, warm=3, between=None):
        return median_ms(fn, stream, n, warm, between)

    # L2-cold timings write a 256 MB buffer (twice the 129 MB L2) before each timed call
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def cold():
        scrub.fill_(1)

    def step_us(fn, n=300):
        """Steps issued back to back, as a decode loop issues them: (issue-bound) time
        per step, and the same step captured once in a CUDA graph and replayed."""
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        loop = a.elapsed_time(b) / n * 1e3
        graph = None
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                fn()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                fn()
            for _ in range(5):
                g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(n):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            graph = round(a.elapsed_time(b) / n * 1e3, 2)
        except Exception as e:  # report, do not hide, a capture failure
            graph = "capture failed: %s" % str(e).splitlines()[0][:80]
        return {"us_per_step_back_to_back": round(loop, 2), "us_per_step_graph": graph}

    def entry(bytes_, ms, **kw):
        return rate_entry(bytes_, ms, peak, **kw)

    # tiny prefix-sharing gather: latency
    w = inputs.tiny_prefix_gather()
    st = GatherStep(w, dev, hp, inputs)
    # stream=None: the binding uses torch's current stream, the capture stream inside a graph
    out["tiny_prefix_gather"] = step_us(lambda: (st.plan(None), st.copy(None)))
    out["tiny_prefix_gather"]["us_per_step_l2_cold"] = round(
        1e3 * med_ms(lambda: (st.plan(stream), st.copy(stream)), between=cold), 2)
    st.check_status()
    # the same gather as one hp_gather call: a small validated batch takes the one-launch
    # path (plan, table check and copy in one kernel)
    out["tiny_prefix_gather_one_call"] = step_us(
        lambda: hp.hp_gather(st.desc, st.out, st.T, st.ws, st.status))
    st.check_status()
    del st

    # prefix sharing at scale
    w = inputs.config("prefix_sharing")
    st = GatherStep(w, dev, hp, inputs)
    b, spans = gather_bytes(w)
    st.plan(stream)
    ms = med_ms(lambda: st.copy(stream))
    out["prefix_sharing_gather"] = entry(b, ms, note="logical bytes; the 128 shared pages are "
                                         "read from L2 after their first use")
    ms = med_ms(lambda: st.copy(stream), between=cold)
    out["prefix_sharing_gather_l2_cold"] = entry(
        b, ms, note="logical bytes, L2 scrubbed (256 MB write) before each call")
    st.check_status()
    del st

    out.update(dequant_measurements(dev, hp, inputs, entry, med_ms))

    # decode step: append one row per sequence, then gather the grown batch
    w = inputs.config("decode_append")
    pool = inputs.device_pool(w, dev)
    table, sp = idx_tensor(w.table, dev), idx_tensor(w.seq_ptr, dev)
    before, after = idx_tensor(w.lens_before, dev), idx_tensor(w.lens, dev)
    new_ptr = idx_tensor(w.new_ptr, dev)
    new = inputs.device_new_rows(w, dev)
    kw = dict(num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
              head_dim=w.head_dim, dtype=w.dtype, index_type=0)
    d_app = hp.PagedDesc(pool, table, sp, before, **kw)
    ws = hp.workspace_for(d_app, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out["decode_append_step"] = dict(
        step_us(lambda: hp.hp_scatter_append(d_app, new, new_ptr, w.total_new, ws, status)),
        rows=w.total_new, bytes=2 * w.total_new * w.row_bytes)
    # the same step with HP_PERMISSIVE (the caller vouches for the descriptor): one kernel,
    # one warp per sequence, no plan and no block-table check
    d_app_p = hp.PagedDesc(pool, table, sp, before, flags=1, **kw)
    out["decode_append_step_permissive"] = dict(
        step_us(lambda: hp.hp_scatter_append(d_app_p, new, new_ptr, w.total_new, ws, status)),
        rows=w.total_new, bytes=2 * w.total_new * w.row_bytes)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    d_g = hp.PagedDesc(pool, table, sp, after, **kw)
    T = w.total_tokens
    o = torch.empty(T * w.row_bytes, dtype=torch.uint8, device=dev)
    assert hp.hp_plan(d_g, T, ws, status) == 0
    b, _ = gather_bytes(w)
    ms = med_ms(lambda: hp.hp_gather_planned(d_g, o, ws, status), n=10)
    out["decode_append_gather"] = entry(b, ms)
    # bulk (prefill-style) scatter of every row of the batch into its pages
    zeros = torch.zeros(w.num_seqs, dtype=torch.int32, device=dev)
    d_bulk = hp.PagedDesc(pool, table, sp, zeros, **kw)
    np_bulk = idx_tensor(np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))]).astype(np.uint32), dev)
    assert hp.hp_append_plan(d_bulk, np_bulk, T, ws, status) == 0
    ms = med_ms(lambda: hp.hp_scatter_append_planned(d_bulk, o, np_bulk, T, ws, status), n=10)
    out["bulk_scatter_append"] = entry(b, ms)
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    # writer side: copy-on-write copies of 20,000 pages into free pages, and zeroing the
    # slots past every sequence's count (the pool's partial last pages)
    rng = np.random.default_rng(9)
    used = np.unique(w.table.astype(np.int64))
    free = np.setdiff1d(np.arange(w.num_pages), used)
    src = rng.choice(used, 20000, replace=False).astype(np.uint32)
    dst = rng.choice(free, 20000, replace=False).astype(np.uint32)
    sd, dd = idx_tensor(src, dev), idx_tensor(dst, dev)
    page_bytes = w.page_size * w.row_bytes
    ms = med_ms(lambda: hp.hp_copy_pages(pool, w.num_pages, page_bytes, 0, sd, dd, 20000,
                                         status), n=10)
    out["copy_pages_cow"] = entry(2 * 20000 * page_bytes + 2 * 20000 * 4, ms)
    # the same 20,000 source pages gathered into a contiguous buffer by torch's
    # index_select (random 32 KiB reads, sequential writes): the pattern's rate at this size
    pages = pool.view(w.num_pages, page_bytes)
    tmp = torch.empty((20000, page_bytes), dtype=torch.uint8, device=dev)
    sl = sd.long()
    ms = med_ms(lambda: torch.index_select(pages, 0, sl, out=tmp), n=10)
    out["copy_pages_cow_torch_index_select_same_pages"] = entry(2 * 20000 * page_bytes, ms)
    del tmp
    rc, nsc = hp.hp_zero_tails_scratch_bytes(d_g)
    scratch = torch.empty(nsc, dtype=torch.uint8, device=dev)
    out["zero_tails_step"] = step_us(lambda: hp.hp_zero_tails(d_g, ws, scratch, status))
    assert int(status.item()) == 0, hp.status_name(int(status.item()))
    # decode attention over the grown batch: 32 query heads on the 8 K/V heads, reading
    # every key and value row once through the block table
    del o
    release_device_memory()
    out["decode_attention"] = attention_measurement(dev, hp, inputs, w, d_g, peak, entry, med_ms)
    del pool, new
    release_device_memory()

    out["decode_step_4_layers"] = decode_step_layers(dev, hp, inputs, entry, med_ms)
    release_device_memory()

    # kernel-internal [nb, H, D/x, bs, x] -> interchange [nb, bs, H, D], decode-gather pool
    nb, bsz, H, D = 10000, 16, 32, 128
    kin = torch.empty(nb * bsz * H * D * 2, dtype=torch.uint8, device=dev)
    kout = torch.empty_like(kin)
    ms = med_ms(lambda: hp.hp_from_kernel_layout(kin, kout, nb, bsz, H, D, 8, "f16"), n=10)
    out["kernel_layout_to_interchange"] = entry(2 * kin.numel(), ms)
    ms = med_ms(lambda: hp.hp_to_kernel_layout(kout, kin, nb, bsz, H, D, 8, "f16"), n=10)
    out["interchange_to_kernel_layout"] = entry(2 * kin.numel(), ms)
    del kin, kout

    # per-lane [N, B, H_kv, P, d] layout
    lw = inputs.lane_synthetic()
    g = torch.Generator(device=dev)
    g.manual_seed(lw.seed)
    lpool = torch.randn(lw.pool_shape, generator=g, device=dev).to(torch.bfloat16)
    lt = torch.from_numpy(lw.table.view(np.int64).copy()).to(dev)
    lo = torch.empty((lw.batch, lw.kv_heads, lw.n, lw.width), dtype=torch.bfloat16, device=dev)
    ms = med_ms(lambda: hp.hp_lane_gather(lpool, lt, lw.capacity, lw.page_tokens, lw.batch,
                                          lw.kv_heads, lw.width, "bf16", lw.n, lo, status))
    out["lane_gather"] = entry(2 * lw.lanes * lw.n * lw.width * 2 + lw.pages * 8, ms)
    lnew = torch.randn((lw.batch, lw.kv_heads, 1, lw.width), device=dev).to(torch.bfloat16)
    out["lane_append_step"] = step_us(
        lambda: hp.hp_lane_append(lpool, lt, lw.capacity, lw.page_tokens, lw.batch, lw.kv_heads,
                                  lw.width, "bf16", lw.n, 1, lnew, status))
    assert int(status.item()) == 0
    return out


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-ops", action="store_true", help="skip the per-operation measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--workload", default="decode_gather",
                    choices=["decode_gather", "decode_append", "prefix_sharing", "quantized_pool",
                             "quantized_pool_mid"],
                    help="batch the timed steps gather (default: the decode-sized gather)")
    ap.add_argument("--attention", choices=["full", "mid", "short"],
                    help="time only hp_attention_decode on the decode-append batch at this "
                         "scale (warm-up calls, then --steps timed calls) and print its line")
    ap.add_argument("--decode-layers", action="store_true",
                    help="only the 4-layer decode step through the planned calls (32 "
                         "sequences) and print its line")
    ap.add_argument("--host-kv", action="store_true",
                    help="with --attention: K and V pools in page-locked host memory")
    ap.add_argument("--transpose", action="store_true",
                    help="time only the two cache layout conversions (kernel-internal "
                         "[10000, 32, 16, 16, 8] <-> interchange [10000, 16, 32, 128], fp16) "
                         "and print their line")
    ap.add_argument("--dequant", action="store_true",
                    help="only the dequantising gathers (every scheme) on quantized_pool")
    ap.add_argument("--lane", action="store_true",
                    help="time only the per-lane snapshot gather (256 lanes of the "
                         "lane_synthetic layout) and print its line")
    ap.add_argument("--decode-step", action="store_true",
                    help="issue --steps decode append steps (256 rows into the decode_append "
                         "pool), validated and then permissive, and print their timing")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.lane:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp, inputs
        build.build()
        hp.lib()
        print(json.dumps(lane_only("cuda", hp, inputs, peak_hbm()[0], args.steps)))
        return
    if args.decode_layers:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp, inputs
        build.build()
        hp.lib()
        peak = peak_hbm()[0]
        stream = torch.cuda.current_stream()
        print(json.dumps(decode_step_layers(
            "cuda", hp, inputs, lambda b, ms, **kw: rate_entry(b, ms, peak, **kw),
            lambda fn, n=10: median_ms(fn, stream, n))))
        return
    if args.dequant:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp, inputs
        build.build()
        hp.lib()
        peak = peak_hbm()[0]
        stream = torch.cuda.current_stream()
        print(json.dumps(dequant_measurements(
            "cuda", hp, inputs, lambda b, ms, **kw: rate_entry(b, ms, peak, **kw),
            lambda fn, n=args.steps: median_ms(fn, stream, n))))
        return
    if args.decode_step:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp, inputs
        build.build()
        hp.lib()
        print(json.dumps(decode_step_only("cuda", hp, inputs, args.steps)))
        return
    if args.transpose:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp
        build.build()
        hp.lib()
        print(json.dumps(transpose_only("cuda", hp, peak_hbm()[0], args.steps)))
        return
    if args.attention:
        import torch
        from paged_kv_cache_hp_gb300 import build, hp, inputs
        build.build()
        hp.lib()
        print(json.dumps(attention_only(args.attention, "cuda", hp, inputs, peak_hbm()[0],
                                        args.steps, host_kv=args.host_kv)))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from paged_kv_cache_hp_gb300 import inputs
    if args.workload == "quantized_pool_mid":
        w = inputs.config("quantized_pool", "mid")
    else:
        w = inputs.config(args.workload)
    T = w.total_tokens
    step_bytes_copy, spans = gather_bytes(w)
    if w.scales_seed is not None:  # int8 in, 4-byte scale per row, bf16 out
        step_bytes_copy = T * (w.num_heads * w.head_dim * 3 + 4) + spans * 8
    step_bytes = step_bytes_copy + validate_bytes(w)
    config = {"workload": w.name, "num_pages": w.num_pages, "page_size": w.page_size,
              "num_heads": w.num_heads, "head_dim": w.head_dim, "pool_dtype": w.dtype,
              "num_seqs": w.num_seqs, "total_tokens": T,
              "index": "u32" if w.index_dtype == np.uint32 else "u64",
              "bytes_per_step": step_bytes, "l2": "inputs larger than L2 (%.2f GB per step)"
              % (step_bytes / 1e9), "parallelism": "replicas x%d" % args.gpus}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        host_pool = inputs.host_pool(w) if w.pool_bytes <= (64 << 20) else None
        if host_pool is None:
            import torch
            host_pool = inputs.device_pool(w, "cpu", force_device_rng=True).numpy() \
                if not torch.cuda.is_available() else inputs.device_pool(w, "cuda").cpu().numpy()
        # each step: the threaded oracle over a prefix of the batch sized so that the
        # whole --steps/--warmup run takes about two minutes of host time
        per_step = max(0.002, 120.0 / (args.steps + args.warmup))
        nthr = host_threads()
        full = OracleThreads(w, host_pool, oracle, nthr)
        full.step()
        t0 = time.perf_counter()
        full.step()
        dt_full = time.perf_counter() - t0
        full.close()
        cap = None if dt_full <= per_step else max(256, int(w.total_tokens * per_step / dt_full))
        run = OracleThreads(w, host_pool, oracle, nthr, cap)
        for _ in range(args.warmup):
            run.step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run.step()
        el = time.perf_counter() - t0
        run.close()
        value = run.bytes * args.steps / el / 1e9
        sample = ("oracle gather of the first %d of %d tokens per step on %d host threads "
                  "(one contiguous group of sequences each)" % (run.tokens, w.total_tokens,
                                                                 run.threads))
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": round(value, 3),
                          "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": w.dtype, "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": round(value, 3), "unit": UNIT,
                                           "cores": run.threads, "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": round(value, 3), "unit": UNIT,
                                  "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    import torch
    from paged_kv_cache_hp_gb300 import build, hp
    build.build()
    hp.lib()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = "cuda:%d" % (local if world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    step = GatherStep(w, dev, hp, inputs)
    with ClockSampler(local) as clk:
        step_ms, wall = time_steps(step, args.steps, args.warmup, stream, dist)
        copy_ms = time_copy_kernel(step, min(args.steps, 500), stream)
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    value = whole_job_gbps(step_bytes, args.steps, world, total_ms)
    peak, peak_kind = peak_hbm()
    copy_mean = statistics.mean(copy_ms)
    achieved = step_bytes_copy / (copy_mean * 1e-3) / 1e9

    # a same-bytes device-to-device copy as the practical ceiling
    a = torch.empty(T * w.row_bytes, dtype=torch.uint8, device=dev)
    bb = torch.empty_like(a)
    for _ in range(3):
        bb.copy_(a)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(20):
        bb.copy_(a)
    e1.record(stream)
    torch.cuda.synchronize()
    d2d_gbps = 2 * a.numel() / (e0.elapsed_time(e1) / 20 * 1e-3) / 1e9
    del a, bb

    traffic = recorded_traffic("gather_" + w.name, spans)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; pool ~N(0,1) drawn on the device)", "config": config,
        "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if traffic is None else int(traffic),
                     "kernel": ("copy_kernel<dequant> (hp_gather_dequant_planned)"
                                if step.dequant else "bulk_kernel<gather> (hp_gather_planned)"),
                     "kernel_timing": "CUDA events around each of %d copy-only launches "
                                      "after the timed steps" % len(copy_ms),
                     "peak_kind": peak_kind + " (hbm_gbs, copy)",
                     "algorithmic_bytes_per_launch": step_bytes_copy,
                     "launch_ms_mean": round(copy_mean, 4),
                     "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                     "d2d_copy_same_bytes_gbps": round(d2d_gbps, 1)},
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_e2e and args.workload == "decode_gather":
        # the host link shows occasional slow stretches (a whole run of steps at about
        # half speed, seen with either kind of pinned memory): three runs of 8 steps, the
        # median run reported and every run listed
        host = e2e_host_buffers(w, dev, inputs)
        runs = [e2e_gather(w, dev, hp, inputs, steps=8, host=host) for _ in range(3)]
        ms, h2d, d2h = sorted(runs)[1]
        result["e2e"] = {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(ms, 3),
                         "runs_ms_per_step": [round(r[0], 3) for r in runs],
                         "note": "pinned host buffers; uploads, gathers and downloads "
                                 "pipelined over two buffer sets; median of three runs of "
                                 "8 steps"}
        runs = [e2e_gather(w, dev, hp, inputs, steps=8, upload_pool=False, host=host)
                for _ in range(3)]
        ms_r, h2d_r, d2h_r = sorted(runs)[1]
        for o in host["outs"]:
            o[:1 << 20].fill_(0xEE)  # so that the check below sees the in-place gather's rows
        runs_z = [e2e_gather_in_place(w, dev, hp, inputs, steps=8, host=host)
                  for _ in range(3)]
        ms_z, h2d_z, d2h_z, _ = sorted(runs_z)[1]
        # the output must be the gather's: compare one buffer with a device gather
        check = host["outs"][0][:1 << 20].clone()
        del host
        result["e2e"]["resident_pool"] = {
            "value": round(step_bytes / (ms_r * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d_r, "d2h_bytes_per_step": d2h_r,
            "ms_per_step": round(ms_r, 3),
            "runs_ms_per_step": [round(r[0], 3) for r in runs],
            "note": "the pool stays on the device (a resident cache); every step uploads "
                    "its index buffers and downloads the gathered tensor"}
        assert torch.equal(check.to(dev), step.out[:1 << 20]), "in-place gather differs"
        result["e2e"]["pool_in_host_memory"] = {
            "value": round(step_bytes / (ms_z * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d_z, "d2h_bytes_per_step": d2h_z,
            "ms_per_step": round(ms_z, 3),
            "runs_ms_per_step": [round(r[0], 3) for r in runs_z],
            "note": "the pool stays in pinned host memory and the gather writes its rows "
                    "into pinned host memory: each step uploads its index buffers; the "
                    "kernel reads the live pages and writes the output over the host link"}
    if rank == 0 and world == 1 and not args.no_cpu and w.scales_seed is None:
        import oracle
        oracle.build()
        host_pool = step.pool.cpu().numpy()
        gbps, dt, Ts, lens = time_oracle(w, host_pool, oracle, budget_s=12.0)
        gbps_mt, dt_mt, used = time_oracle_threads(w, host_pool, oracle, host_threads())
        result["cpu_baseline"] = {
            "value": round(gbps_mt, 3), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "oracle gather of the whole batch (%d tokens) on %d threads, one "
                      "contiguous group of sequences each, %.2f s" % (T, used, dt_mt),
            "single_thread": {"value": round(gbps, 3), "cores": 1,
                              "sample": "oracle gather (one thread) of the first %d of %d "
                                        "tokens, %.1f s" % (Ts, T, dt)}}
    if rank == 0 and world == 1 and not args.no_ops:
        del step
        release_device_memory()
        result["ops"] = ops_measurements(dev, hp, inputs, peak)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


if __name__ == "__main__":
    main()
