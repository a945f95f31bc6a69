#!/usr/bin/env python
"""Benchmark of the block-paged KV-cache hot path on GB300.

One step = one pass of the path over the decode-step batch (bf16 GQA pool of 300,000
pages x 16 slots x 8 K/V heads x 128 dims, 256 sequences of U[1024, 32768] tokens,
uint32 block tables from a shuffled free list), all through the C ABI:
hp_scatter_append of one new row per sequence at its token count (validated on the
device: plan, table check, one warp per sequence), then hp_plan (device validation of
the grown batch + ragged prefix sums) and hp_gather_planned (the page-span copy of all
4.37M tokens).  The metric is effective HBM GB/s (algorithmic bytes read and written
per step / step time).

Printed: one JSON line (rank 0) with the headline value, the roofline of the gather's
copy kernel, the CPU oracle timed on the same step, an end-to-end figure through pinned
host buffers, and per-operation measurements: the other benchmark configurations (tiny
prefix gather, decode-sized gather, prefix sharing, int8 dequantising gather), each with
its roofline fraction, DRAM traffic record and CPU oracle baseline, and the other rows of
the path (append, schemes, lane layout, writer side, attention, layout conversions).

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


# Workloads whose DRAM traffic record comes from a smaller capture of the same kernel on
# the same length distribution (the full size is above the profiler's size rule): the
# record's bytes per unit (page span) times this launch's units.
TRAFFIC_FROM = {"gather_decode_append": "gather_decode_append_mid",
                "gather_quantized_pool": "gather_quantized_pool_mid"}


def recorded_traffic(kernel_key, units_now):
    """DRAM bytes per launch from a committed ncu summary, scaled to this launch's
    units, or None when the summary is absent or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    kernel_key = TRAFFIC_FROM.get(kernel_key, kernel_key)
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


def dequant_bytes(w, lens=None):
    """Algorithmic bytes of one dequantising gather: per row the int8 codes read, the bf16
    row written and its 4-byte scale; 8 bytes of block table per page span."""
    lens = (w.lens if lens is None else lens).astype(np.int64)
    T = int(lens.sum())
    spans = int((-(-lens // w.page_size)).sum())
    return T * (w.num_heads * w.head_dim * 3 + 4) + spans * 8, spans


def append_bytes(w):
    """Algorithmic bytes of the decode-step append: every new row read and written once,
    one block-table entry per row, the new_ptr offsets."""
    ib = 4 if w.index_dtype == np.uint32 else 8
    return 2 * w.total_new * w.row_bytes + w.total_new * ib + (w.num_seqs + 1) * ib


def unique_gather_bytes(w):
    """The bytes a gather must move from and to DRAM at least: each physical page's live
    rows once however many sequences read them (the prefix pages of a shared prompt
    once), the output rows, the block table."""
    ib = 4 if w.index_dtype == np.uint32 else 8
    lens = w.lens.astype(np.int64)
    return (int(w.live_slots().sum()) + int(lens.sum())) * w.row_bytes + len(w.table) * ib


def physical_rows(w):
    """The pool row (page * P + slot) of every output token, in output order."""
    lens = w.lens.astype(np.int64)
    sp = w.seq_ptr.astype(np.int64)
    seq = np.repeat(np.arange(len(lens)), lens)
    t = np.arange(int(lens.sum())) - np.repeat(np.cumsum(lens) - lens, lens)
    pages = w.table.astype(np.int64)[sp[seq] + t // w.page_size]
    return pages * w.page_size + t % w.page_size


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

    launches = 3  # plan, table check, copy
    kernel = "bulk_kernel<gather> (hp_gather_planned)"

    def plan(self, stream):
        rc = self.hp.hp_plan(self.desc, self.T, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def copy(self, stream):
        f = self.hp.hp_gather_dequant_planned if self.dequant else self.hp.hp_gather_planned
        rc = f(self.desc, self.out, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def run(self, stream):
        self.plan(stream)
        self.copy(stream)

    def check_status(self):
        st = int(self.status.item())
        assert st == 0, self.hp.status_name(st)


class DecodeAppendStep:
    """Resident device buffers of the decode-step batch and the three C-ABI calls of one
    step: hp_scatter_append of one new row per sequence at its count (validated: plan,
    table check, row kernel), then hp_plan and hp_gather_planned of the grown batch.  The
    counts are not advanced between steps, so every step appends the same rows at the same
    slots and gathers the same tokens: identical work each time."""

    launches = 6  # append plan, table check, row kernel; gather plan, table check, copy
    kernel = "bulk_kernel<gather> (hp_gather_planned)"

    def __init__(self, w, dev, hp, inputs):
        import torch
        self.w, self.hp = w, hp
        self.pool = inputs.device_pool(w, dev)
        self.table = idx_tensor(w.table, dev)
        self.seq_ptr = idx_tensor(w.seq_ptr, dev)
        self.before = idx_tensor(w.lens_before, dev)
        self.after = idx_tensor(w.lens, dev)
        self.new_ptr = idx_tensor(w.new_ptr, dev)
        self.new = inputs.device_new_rows(w, dev)
        kw = dict(num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
                  head_dim=w.head_dim, dtype=w.dtype,
                  index_type=0 if w.index_dtype == np.uint32 else 1)
        self.d_app = hp.PagedDesc(self.pool, self.table, self.seq_ptr, self.before, **kw)
        self.desc = hp.PagedDesc(self.pool, self.table, self.seq_ptr, self.after, **kw)
        self.ws_a = hp.workspace_for(self.d_app, dev)
        self.ws = hp.workspace_for(self.desc, dev)
        self.T = w.total_tokens
        self.out = torch.empty(self.T * w.row_bytes, dtype=torch.uint8, device=dev)
        self.st_a = torch.full((1,), -12345, dtype=torch.int32, device=dev)
        self.status = torch.full((1,), -12345, dtype=torch.int32, device=dev)

    def append(self, stream):
        rc = self.hp.hp_scatter_append(self.d_app, self.new, self.new_ptr, self.w.total_new,
                                       self.ws_a, self.st_a, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def copy(self, stream):
        rc = self.hp.hp_gather_planned(self.desc, self.out, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)

    def run(self, stream):
        self.append(stream)
        rc = self.hp.hp_plan(self.desc, self.T, self.ws, self.status, stream=stream)
        assert rc == 0, self.hp.status_name(rc)
        self.copy(stream)

    def check_status(self):
        for t in (self.st_a, self.status):
            st = int(t.item())
            assert st == 0, self.hp.status_name(st)


def time_steps(step, steps, warmup, stream, dist=None):
    """Warm-up, then `steps` timed steps (all of a step's calls, nothing between them)
    bracketed by barrier + synchronize.  Returns (per-step ms list, wall seconds)."""
    import torch
    for _ in range(warmup):
        step.run(stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for e0, e1 in ev:
        e0.record(stream)
        step.run(stream)
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


def _pinned_index(a):
    import torch
    a = np.ascontiguousarray(a)
    v = a.view(np.int32) if a.dtype == np.uint32 else a.astype(np.uint64).view(np.int64)
    return torch.from_numpy(v.copy()).pin_memory()


def e2e_host_buffers(w, dev, inputs):
    """Pinned host buffers of an end-to-end measurement, shared by its runs: the pool
    (filled from the seeded device pool, as it is before any append), the index buffers,
    the new rows of a decode step, and two output buffers."""
    import torch
    pool_dev = inputs.device_pool(w, dev)
    h_pool = torch.empty(pool_dev.shape, dtype=torch.uint8, pin_memory=True)
    h_pool.copy_(pool_dev)
    del pool_dev
    n = w.total_tokens * w.row_bytes
    host = dict(pool=h_pool, outs=[torch.empty(n, dtype=torch.uint8, pin_memory=True)
                                   for _ in range(2)])
    if w.new_ptr is not None:
        host["idx"] = [_pinned_index(a) for a in (w.table, w.seq_ptr, w.lens_before, w.lens,
                                                  w.new_ptr)]
        host["new"] = torch.from_numpy(inputs.host_new_rows(w).reshape(-1).copy()).pin_memory()
    else:
        host["idx"] = [_pinned_index(a) for a in (w.table, w.seq_ptr, w.lens)]
    return host


def e2e_steps(w, dev, hp, steps, host, upload_pool=True):
    """The step through host buffers: every step uploads its inputs from pinned host
    memory (the pool unless upload_pool is False, the index buffers, a decode step's new
    rows), runs the step's C-ABI calls (a decode step: hp_scatter_append, hp_plan,
    hp_gather_planned; a gather: hp_gather) and downloads the gathered tensor to pinned
    host memory.  Steps are pipelined over two device buffer sets and three streams
    (upload, compute, download), so step k+1's upload overlaps step k's download; a buffer
    set is reused only after the step that read it and the download of its output are
    done.  Returns (ms per step, h2d bytes, d2h bytes)."""
    import torch
    h_pool, host_idx, h_new = host["pool"], host["idx"], host.get("new")
    decode = h_new is not None
    T = w.total_tokens
    it = 0 if w.index_dtype == np.uint32 else 1
    kw = dict(num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
              head_dim=w.head_dim, dtype=w.dtype, index_type=it)
    sets = []
    for i in range(2):
        d_pool = torch.empty(h_pool.shape, dtype=torch.uint8, device=dev)
        d_idx = [torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_idx]
        b = dict(pool=d_pool, idx=d_idx, status=torch.zeros(1, dtype=torch.int32, device=dev),
                 st_a=torch.zeros(1, dtype=torch.int32, device=dev),
                 out=torch.empty(T * w.row_bytes, dtype=torch.uint8, device=dev),
                 h_out=host["outs"][i], gathered=None, downloaded=None)
        if decode:
            b["new"] = torch.empty(h_new.shape, dtype=h_new.dtype, device=dev)
            b["d_app"] = hp.PagedDesc(d_pool, d_idx[0], d_idx[1], d_idx[2], **kw)
            b["desc"] = hp.PagedDesc(d_pool, d_idx[0], d_idx[1], d_idx[3], **kw)
            b["ws_a"] = hp.workspace_for(b["d_app"], dev)
        else:
            b["desc"] = hp.PagedDesc(d_pool, d_idx[0], d_idx[1], d_idx[2], **kw)
        b["ws"] = hp.workspace_for(b["desc"], dev)
        sets.append(b)
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def one(k, first=False):
        b = sets[k % 2]
        with torch.cuda.stream(up):
            if b["gathered"] is not None:
                up.wait_event(b["gathered"])  # the last step through this set is done
            if upload_pool or first:
                b["pool"].copy_(h_pool, non_blocking=True)
            for d, h in zip(b["idx"], host_idx):
                d.copy_(h, non_blocking=True)
            if decode:
                b["new"].copy_(h_new, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(up)
        comp.wait_event(uploaded)
        if b["downloaded"] is not None:
            comp.wait_event(b["downloaded"])  # its output buffer has been read back
        if decode:
            assert hp.hp_scatter_append(b["d_app"], b["new"], b["idx"][4], w.total_new,
                                        b["ws_a"], b["st_a"], stream=comp) == 0
            assert hp.hp_plan(b["desc"], T, b["ws"], b["status"], stream=comp) == 0
            assert hp.hp_gather_planned(b["desc"], b["out"], b["ws"], b["status"],
                                        stream=comp) == 0
        else:
            assert hp.hp_gather(b["desc"], b["out"], T, b["ws"], b["status"], stream=comp) == 0
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
    assert all(int(b["status"].item()) == 0 and int(b["st_a"].item()) == 0 for b in sets)
    ms = e0.elapsed_time(e1) / steps
    h2d = (h_pool.numel() if upload_pool else 0) + sum(h.numel() * h.element_size()
                                                       for h in host_idx)
    if decode:
        h2d += h_new.numel()
    return ms, h2d, T * w.row_bytes


def e2e_measurement(w, dev, hp, inputs, step_bytes, check_out):
    """Three runs of 8 pipelined steps through pinned host buffers (the host link shows
    occasional slow stretches, a whole run at about half speed): the median run, every
    run listed, and the same with the pool resident on the device.  The downloaded rows
    are compared with the device-resident step's output (check_out)."""
    import torch
    host = e2e_host_buffers(w, dev, inputs)
    runs = [e2e_steps(w, dev, hp, 8, host) for _ in range(3)]
    ms, h2d, d2h = sorted(runs)[1]
    n = min(1 << 20, check_out.numel())
    for o in host["outs"]:
        assert torch.equal(o[:n].to(dev), check_out[:n]), "end-to-end output differs"
        assert torch.equal(o[-n:].to(dev), check_out[-n:]), "end-to-end output differs"
    res = {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
           "runs_ms_per_step": [round(r[0], 3) for r in runs],
           "note": "pinned host buffers; every step uploads the pool, the index buffers%s and "
                   "downloads the gathered tensor; pipelined over two buffer sets; median of "
                   "three runs of 8 steps" % (" and the new rows" if w.new_ptr is not None
                                              else "")}
    runs = [e2e_steps(w, dev, hp, 8, host, upload_pool=False) for _ in range(3)]
    ms_r, h2d_r, d2h_r = sorted(runs)[1]
    res["resident_pool"] = {
        "value": round(step_bytes / (ms_r * 1e-3) / 1e9, 1), "unit": UNIT,
        "h2d_bytes_per_step": h2d_r, "d2h_bytes_per_step": d2h_r,
        "ms_per_step": round(ms_r, 3), "runs_ms_per_step": [round(r[0], 3) for r in runs],
        "note": "the pool stays on the device (a resident cache); every step uploads its "
                "index buffers%s and downloads the gathered tensor"
                % (" and new rows" if w.new_ptr is not None else "")}
    del host
    return res


# ----------------------------------------------------------------------------- oracle arm
def _prefix_lens(w, tokens_cap):
    """Token counts of the first tokens_cap tokens of the batch (the whole batch when
    None): whole sequences, the last one cut short."""
    lens = w.lens.astype(np.int64).copy()
    if tokens_cap is None or tokens_cap >= int(lens.sum()):
        return lens
    c = np.cumsum(lens)
    k = int(np.searchsorted(c, tokens_cap))
    lens = lens[:k + 1].copy()
    prev = int(c[k - 1]) if k > 0 else 0
    lens[-1] = max(1, min(int(lens[-1]), tokens_cap - prev))
    return lens


def _oracle_sub(w, host_pool, oracle_mod, a, b, lens, scales=None):
    """An oracle descriptor over sequences a..b-1 (re-based slices), counts `lens`."""
    sp = (w.seq_ptr[a:b + 1].astype(np.int64) - int(w.seq_ptr[a])).astype(w.index_dtype)
    table = w.table[int(w.seq_ptr[a]):int(w.seq_ptr[b])]
    return oracle_mod.Desc(host_pool, table, sp, np.asarray(lens).astype(w.index_dtype),
                           num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
                           head_dim=w.head_dim, dtype=w.dtype,
                           index_type=0 if w.index_dtype == np.uint32 else 1, scales=scales,
                           flags=0 if scales is None else oracle_mod.HAS_QUANT)


class OracleThreads:
    """The oracle's gather (its dequantising gather when `scales` is given), as it stands,
    on nthreads host threads over the first `tokens_cap` tokens of the batch (all of it
    when None): the sequences are cut into nthreads contiguous groups, each gathered by
    one call through its own sub-descriptor (ctypes releases the GIL during the call).
    For a decode-step batch each step first runs the oracle's append of the new rows
    (one call, on the calling thread)."""

    def __init__(self, w, host_pool, oracle_mod, nthreads, tokens_cap=None, scales=None,
                 append=False):
        from concurrent.futures import ThreadPoolExecutor
        lens = _prefix_lens(w, tokens_cap)
        n = len(lens)
        cuts = np.linspace(0, n, min(nthreads, n) + 1).astype(int)
        self.descs, self.outs = [], []
        E = w.num_heads * w.head_dim
        for a, b in zip(cuts[:-1], cuts[1:]):
            if b <= a:
                continue
            d = _oracle_sub(w, host_pool, oracle_mod, a, b, lens[a:b], scales)
            self.descs.append(d)
            T = int(lens[a:b].sum())
            self.outs.append(np.zeros((T, w.row_bytes), dtype=np.uint8) if scales is None
                             else np.zeros((T, E), dtype=np.uint16))
        self.dequant = scales is not None
        self.pool = ThreadPoolExecutor(max(1, len(self.descs)))
        self.tokens = int(lens.sum())
        self.bytes = (dequant_bytes if self.dequant else gather_bytes)(w, lens)[0]
        self.threads = len(self.descs)
        self.append = None
        if append:
            self.append = (_oracle_sub(w, host_pool, oracle_mod, 0, w.num_seqs, w.lens_before),
                           inputs_new_rows(w), w.new_ptr)
            self.bytes += append_bytes(w)

    def step(self):
        if self.append is not None:
            d, rows, new_ptr = self.append
            assert d.scatter_append(rows, new_ptr) == "OK"
        if self.dequant:
            f = lambda i: self.descs[i].gather_dequant(self.outs[i])[2]
        else:
            f = lambda i: self.descs[i].gather(self.outs[i])[2]
        faults = list(self.pool.map(f, range(len(self.descs))))
        assert all(x == "OK" for x in faults), faults

    def close(self):
        self.pool.shutdown()


def inputs_new_rows(w):
    from paged_kv_cache_hp_gb300 import inputs
    return inputs.host_new_rows(w)


def host_threads():
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def time_oracle_run(w, host_pool, oracle_mod, nthreads, budget_s, scales=None, append=False):
    """The oracle on nthreads threads over as much of the batch (a prefix of it) as takes
    about budget_s seconds a step: a probe of 65,536 tokens sets the size.  Returns
    (GB/s, seconds, tokens, threads used)."""
    probe = OracleThreads(w, host_pool, oracle_mod, nthreads, tokens_cap=1 << 16, scales=scales)
    probe.step()
    t0 = time.perf_counter()
    probe.step()
    rate = probe.tokens / max(time.perf_counter() - t0, 1e-6)
    probe.close()
    cap = int(rate * budget_s)
    run = OracleThreads(w, host_pool, oracle_mod, nthreads,
                        tokens_cap=None if cap >= w.total_tokens else cap, scales=scales,
                        append=append)
    run.step()  # page in
    t0 = time.perf_counter()
    run.step()
    dt = time.perf_counter() - t0
    run.close()
    return run.bytes / dt / 1e9, dt, run.tokens, run.threads


def cpu_baseline_entry(w, host_pool, oracle_mod, scales=None, append=False, budget_s=8.0,
                       single_budget_s=6.0):
    """The oracle as it stands timed on this host: on every host thread (the whole batch
    when it takes under budget_s, else a prefix), and on one thread (a prefix of about
    single_budget_s)."""
    what = "dequantising gather" if scales is not None else "gather"
    if append:
        what = "append of the %d new rows + %s" % (w.total_new, what)
    gbps, dt, tok, used = time_oracle_run(w, host_pool, oracle_mod, host_threads(), budget_s,
                                          scales, append)
    g1, dt1, tok1, _ = time_oracle_run(w, host_pool, oracle_mod, 1, single_budget_s, scales,
                                       append)
    span = "the whole batch (%d tokens)" % tok if tok >= w.total_tokens else \
        "the first %d of %d tokens" % (tok, w.total_tokens)
    span1 = "the whole batch" if tok1 >= w.total_tokens else \
        "the first %d of %d tokens" % (tok1, w.total_tokens)
    return {"value": round(gbps, 3), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "oracle %s of %s on %d threads, one contiguous group of sequences each, "
                      "%.2f s" % (what, span, used, dt),
            "single_thread": {"value": round(g1, 3), "cores": 1,
                              "sample": "oracle %s (one thread) of %s, %.2f s"
                                        % (what, span1, dt1)}}


def host_pool_for(w, dev=None):
    """The pool's bytes on the host: the seeded device pool copied back when a GPU is
    present (the bytes every GPU measurement reads); on a host without one, small pools
    from numpy and large ones zero-filled (a byte copy's time does not depend on the
    bytes)."""
    from paged_kv_cache_hp_gb300 import inputs
    if w.pool_bytes <= (64 << 20):
        return inputs.host_pool(w).reshape(-1), "seeded"
    import torch
    if torch.cuda.is_available():
        return inputs.device_pool(w, dev or "cuda").cpu().numpy().reshape(-1), "seeded"
    return np.zeros(w.pool_bytes, dtype=np.uint8), "zero-filled (no GPU on this host)"


def host_scales_for(w, dev=None):
    from paged_kv_cache_hp_gb300 import inputs
    import torch
    if w.scales_seed is None:
        return None
    n = w.num_pages * w.page_size
    if n * 4 <= (64 << 20) or not torch.cuda.is_available():
        return inputs.host_scales(w) if n * 4 <= (64 << 20) else \
            np.full(n, 0.01, dtype=np.float32)
    return inputs.device_scales(w, dev or "cuda").cpu().numpy()


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


def attention_only(scale, dev, hp, inputs, peak, reps, host_kv=False, kernel="auto",
                   heads=(8, 4, 128)):
    """Decode attention alone on the decode-append batch at `scale` ("full": 256 sequences
    of 1K-32K tokens; "mid": 32 of them, about 2.5 GB on the device, the profiler's case;
    "short": 2048 sequences of 16-1024 tokens); host_kv: K and V in page-locked host
    memory (HP_HOST_MEMORY); kernel: "auto" (the library's choice), "tensor" or "cuda";
    heads: (K/V heads, query heads per K/V head, head_dim) -- the same token counts and
    page tables with another head layout."""
    import torch
    w = inputs.config("decode_append", scale)
    hkv, g, hd = heads
    if (hkv, hd) != (w.num_heads, w.head_dim):
        lo, hi = (16, 1024) if scale == "short" else (1024, 32768)
        w = inputs.decode_append(num_pages=w.num_pages, num_seqs=w.num_seqs, len_lo=lo,
                                 len_hi=hi, num_heads=hkv, head_dim=hd, name=w.name)
    pool = inputs.device_pool(w, dev)
    hk = None
    if host_kv:
        hk = torch.empty(pool.shape, dtype=pool.dtype, pin_memory=True)
        hk.copy_(pool)
        pool = hk
    flags = {"auto": 0, "tensor": hp.ATTN_TENSOR_CORES, "cuda": hp.ATTN_CUDA_CORES}[kernel]
    if host_kv:
        flags |= hp.HOST_MEMORY
    d_k = hp.PagedDesc(pool, idx_tensor(w.table, dev), idx_tensor(w.seq_ptr, dev),
                       idx_tensor(w.lens, dev), num_pages=w.num_pages, page_size=w.page_size,
                       num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype, index_type=0,
                       flags=flags)
    stream = torch.cuda.current_stream()
    res = attention_measurement(dev, hp, inputs, w, d_k, peak,
                                lambda b, ms, **kw: rate_entry(b, ms, peak, **kw),
                                lambda fn, n: median_ms(fn, stream, n), Hq=hkv * g, reps=reps,
                                host_kv=hk)
    res.update(op="decode_attention", workload=w.name, num_seqs=w.num_seqs,
               total_tokens=w.total_tokens, num_heads=w.num_heads, head_dim=w.head_dim,
               kv_memory="page-locked host" if host_kv else "device", kernel=kernel)
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
    # one contiguous copy of the snapshot's bytes: the ceiling of a launch this size
    cg = d2d_copy_gbps(lw.lanes * lw.n * lw.width * 2, dev, stream)
    res["d2d_copy_same_bytes"] = {"gbps": round(cg, 1), "frac": round(cg / peak, 4)}
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


def dequant_measurements(dev, hp, inputs, entry, med_ms, oracle_mod=None):
    """The dequantising gathers on the quantized_pool batch (int8 codes -> bf16): per-slot
    scales (the benchmark configuration, with its traffic record and, given the oracle,
    its CPU baseline), then the other schemes of [HF] Per-scheme composition with zero
    points."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    w = inputs.config("quantized_pool")
    st = GatherStep(w, dev, hp, inputs)
    T = w.total_tokens
    b, spans = dequant_bytes(w)
    st.plan(stream)
    ms = med_ms(lambda: st.copy(stream), n=10)
    e = entry(b, ms, workload=w.name, tokens=T, units=spans, kernel="copy_kernel<dequant>")
    traffic = recorded_traffic("gather_" + w.name, spans)
    e["traffic"] = None if traffic is None else int(traffic)
    if traffic is not None:
        e["traffic_source"] = traffic_source("gather_" + w.name)
    out["quantized_pool_dequant_gather"] = e
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
    if oracle_mod is not None:
        host_pool = st.pool.cpu().numpy().reshape(-1)
        scales = st.scales.cpu().numpy()
        del st
        release_device_memory()
        e["cpu_baseline"] = cpu_baseline_entry(w, host_pool, oracle_mod, scales=scales)
        del host_pool
    else:
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


def config_entry(dev, hp, inputs, w, peak, med_ms, oracle_mod, cold=None, e2e=False):
    """One benchmark configuration's gather (dequantising for an int8 pool): the copy
    kernel's median time after one plan and the whole step's (plan, table check, copy),
    the fraction of the peak, the DRAM traffic record, and the oracle's baseline.  With
    prefix sharing, also the bytes a gather must move at least (each shared page once)
    and their fraction: the logical bytes count a shared page once per reader, and those
    reads after the first come from L2."""
    import torch
    stream = torch.cuda.current_stream()
    st = GatherStep(w, dev, hp, inputs)
    b, spans = (dequant_bytes if st.dequant else gather_bytes)(w)
    st.run(stream)
    ms = med_ms(lambda: st.copy(stream), n=10)
    ms_step = med_ms(lambda: st.run(stream), n=10)
    st.check_status()
    e = rate_entry(b, ms, peak, workload=w.name, tokens=w.total_tokens, units=spans,
                   kernel="copy_kernel<dequant>" if st.dequant else "bulk_kernel<gather>")
    e["step"] = rate_entry(b + validate_bytes(w), ms_step, peak,
                           note="hp_plan + copy (plan, table check, copy kernels)")
    traffic = recorded_traffic("gather_" + w.name, spans)
    e["traffic"] = None if traffic is None else int(traffic)
    if traffic is not None:
        e["traffic_source"] = traffic_source("gather_" + w.name)
    if w.name.startswith("prefix_sharing"):
        ub = unique_gather_bytes(w)
        e["note"] = "logical bytes: each shared prefix page counted once per sequence"
        e["unique_bytes"] = ub
        e["gbps_unique"] = round(ub / (ms * 1e-3) / 1e9, 1)
        e["frac_unique"] = round(ub / (ms * 1e-3) / 1e9 / peak, 4)
        if traffic is not None:
            e["traffic_over_unique"] = round(traffic / ub, 4)
        # the same rows through a generic gather (torch index_select over the pool's rows),
        # for reading frac_unique
        rows = st.pool.view(w.num_pages * w.page_size, -1)
        it = torch.from_numpy(physical_rows(w)).to(dev)
        dst = torch.empty((it.numel(), rows.shape[1]), dtype=rows.dtype, device=dev)
        ms_i = med_ms(lambda: torch.index_select(rows, 0, it, out=dst), n=10)
        e["torch_index_select_same_rows"] = {
            "ms": round(ms_i, 4), "frac_unique": round(ub / (ms_i * 1e-3) / 1e9 / peak, 4)}
        del dst, it
        if cold is not None:
            ms_c = med_ms(lambda: st.copy(stream), n=10, between=cold)
            e["l2_cold"] = rate_entry(b, ms_c, peak, note="L2 scrubbed (256 MB write) before "
                                      "each call; logical bytes")
            e["l2_cold"]["frac_unique"] = round(ub / (ms_c * 1e-3) / 1e9 / peak, 4)
    if e2e and not st.dequant:
        e["e2e"] = e2e_measurement(w, dev, hp, inputs, b + validate_bytes(w), st.out)
    if oracle_mod is not None:
        host_pool = st.pool.cpu().numpy().reshape(-1)
        scales = st.scales.cpu().numpy() if st.dequant else None
        del st
        release_device_memory()
        e["cpu_baseline"] = cpu_baseline_entry(w, host_pool, oracle_mod, scales=scales)
        del host_pool
    return e


def ops_measurements(dev, hp, inputs, peak, oracle_mod=None, reps=20):
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
        per step, and the same step captured once in a CUDA graph and replayed.  About
        50 ms of the step first: after the seconds of host work the CPU baselines take, the
        GPU's clocks need that long to come back up (a 256-row append then replayed in
        10 us instead of 8.2)."""
        t_end = time.perf_counter() + 0.05
        while time.perf_counter() < t_end:
            for _ in range(20):
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

    # tiny prefix-sharing gather (28 tokens): latency
    w = inputs.tiny_prefix_gather()
    st = GatherStep(w, dev, hp, inputs)
    # stream=None: the binding uses torch's current stream, the capture stream inside a graph
    out["tiny_prefix_gather"] = step_us(lambda: (st.plan(None), st.copy(None)))
    out["tiny_prefix_gather"]["us_per_step_l2_cold"] = round(
        1e3 * med_ms(lambda: (st.plan(stream), st.copy(stream)), between=cold), 2)
    st.check_status()
    if oracle_mod is not None:
        d = _oracle_sub(w, inputs.host_pool(w).reshape(-1), oracle_mod, 0, w.num_seqs, w.lens)
        d.gather()
        t0 = time.perf_counter()
        for _ in range(2000):
            d.gather()
        out["tiny_prefix_gather"]["cpu_baseline"] = {
            "us_per_call": round((time.perf_counter() - t0) / 2000 * 1e6, 2), "cores": 1,
            "kind": "oracle", "sample": "oracle gather of the whole batch, one thread, mean "
                                        "of 2000 calls (each allocating its output)"}
    # the same gather as one hp_gather call: a small validated batch takes the one-launch
    # path (plan, table check and copy in one kernel)
    out["tiny_prefix_gather_one_call"] = step_us(
        lambda: hp.hp_gather(st.desc, st.out, st.T, st.ws, st.status))
    st.check_status()
    del st

    # decode-sized gather (64 sequences, 8 KiB rows) and prefix sharing (128 sequences on
    # one 2048-token prompt): each configuration with its traffic record and CPU baseline
    w = inputs.config("decode_gather")
    out["decode_gather"] = config_entry(dev, hp, inputs, w, peak, med_ms, oracle_mod,
                                        e2e=True)
    release_device_memory()
    w = inputs.config("prefix_sharing")
    out["prefix_sharing_gather"] = config_entry(dev, hp, inputs, w, peak, med_ms, oracle_mod,
                                                cold=cold)
    release_device_memory()

    out.update(dequant_measurements(dev, hp, inputs, entry, med_ms, oracle_mod))

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
    ap.add_argument("--workload", default="decode_append",
                    choices=["decode_append", "decode_append_mid", "decode_gather",
                             "prefix_sharing", "quantized_pool", "quantized_pool_mid"],
                    help="batch of the timed steps (default: the decode step, append then "
                         "gather, at its stated size; *_mid: the profiler's smaller case)")
    ap.add_argument("--attention", choices=["full", "mid", "short"],
                    help="time only hp_attention_decode on the decode-append batch at this "
                         "scale (warm-up calls, then --steps timed calls) and print its line")
    ap.add_argument("--decode-layers", action="store_true",
                    help="only the 4-layer decode step through the planned calls (32 "
                         "sequences) and print its line")
    ap.add_argument("--host-kv", action="store_true",
                    help="with --attention: K and V pools in page-locked host memory")
    ap.add_argument("--attention-kernel", default="auto", choices=["auto", "tensor", "cuda"],
                    help="with --attention: the library's choice of kernel, or force one")
    ap.add_argument("--attention-heads", default="8,4,128",
                    help="with --attention: K/V heads, query heads per K/V head and head_dim "
                         "(the same sequences with another head layout)")
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
        heads = tuple(int(x) for x in args.attention_heads.split(","))
        print(json.dumps(attention_only(args.attention, "cuda", hp, inputs, peak_hbm()[0],
                                        args.steps, host_kv=args.host_kv,
                                        kernel=args.attention_kernel, heads=heads)))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from paged_kv_cache_hp_gb300 import inputs
    w = workload(inputs, args.workload)
    T = w.total_tokens
    decode = w.new_ptr is not None
    dequant = w.scales_seed is not None
    copy_bytes, spans = (dequant_bytes if dequant else gather_bytes)(w)
    step_bytes = copy_bytes + validate_bytes(w)
    if decode:  # the append, and its own plan's reads
        step_bytes += append_bytes(w) + validate_bytes(w)
    config = {"workload": w.name, "num_pages": w.num_pages, "page_size": w.page_size,
              "num_heads": w.num_heads, "head_dim": w.head_dim, "pool_dtype": w.dtype,
              "num_seqs": w.num_seqs, "total_tokens": T,
              "index": "u32" if w.index_dtype == np.uint32 else "u64",
              "bytes_per_step": step_bytes, "l2": "inputs larger than L2 (%.2f GB per step)"
              % (step_bytes / 1e9), "parallelism": "replicas x%d" % args.gpus}
    if decode:
        config.update(new_rows_per_step=w.total_new, step=(
            "hp_scatter_append (validated: plan, table check, one warp per sequence) of one "
            "new row per sequence at its count, then hp_plan + hp_gather_planned of the "
            "grown batch; the counts are not advanced between steps (identical work)"),
            num_pages_note="300,000 pages: the stated 60,000 cannot hold 256 sequences of "
                           "U[1024, 32768] tokens (about 270,000 pages needed)"
            if w.name == "decode_append" else None)
    else:
        config["step"] = ("hp_plan + hp_gather_dequant_planned" if dequant
                          else "hp_plan + hp_gather_planned")

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, w, config, decode)
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

    step = DecodeAppendStep(w, dev, hp, inputs) if decode else GatherStep(w, dev, hp, inputs)
    with ClockSampler(local) as clk:
        step_ms, wall = time_steps(step, args.steps, args.warmup, stream, dist)
        copy_ms = time_copy_kernel(step, min(args.steps, 500), stream)
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    value = whole_job_gbps(step_bytes, args.steps, world, total_ms)
    peak, peak_kind = peak_hbm()
    copy_mean = statistics.mean(copy_ms)
    achieved = copy_bytes / (copy_mean * 1e-3) / 1e9
    d2d_gbps = d2d_copy_gbps(T * w.row_bytes, dev, stream)

    traffic = recorded_traffic("gather_" + w.name, spans)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; pool ~N(0,1) drawn on the device)", "config": config,
        "gpu_launches": step.launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if traffic is None else int(traffic),
                     "kernel": ("copy_kernel<dequant> (hp_gather_dequant_planned)"
                                if dequant else step.kernel),
                     "kernel_timing": "CUDA events around each of %d copy-only launches "
                                      "after the timed steps" % len(copy_ms),
                     "peak_kind": peak_kind + " (hbm_gbs, copy)",
                     "algorithmic_bytes_per_launch": copy_bytes,
                     "units_per_launch": spans,
                     "launch_ms_mean": round(copy_mean, 4),
                     "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                     "d2d_copy_same_bytes_gbps": round(d2d_gbps, 1)},
        "clocks": clk.summary(),
    }
    if traffic is not None:
        result["roofline"]["traffic_source"] = traffic_source("gather_" + w.name)
    if rank == 0 and world == 1 and not args.no_e2e and not dequant:
        result["e2e"] = e2e_measurement(w, dev, hp, inputs, step_bytes, step.out)
        release_device_memory()
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        # (for a decode step the pool already holds the new rows; the oracle's append
        # writes the same rows over them, the same work as on the pool before the step)
        host_pool = step.pool.cpu().numpy().reshape(-1)
        scales = step.scales.cpu().numpy() if dequant else None
        result["cpu_baseline"] = cpu_baseline_entry(w, host_pool, oracle, scales=scales,
                                                    append=decode)
        del host_pool
    if rank == 0 and world == 1 and not args.no_ops:
        del step
        release_device_memory()
        result["ops"] = ops_measurements(dev, hp, inputs, peak,
                                         None if args.no_cpu else load_oracle())
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def load_oracle():
    import oracle
    oracle.build()
    return oracle


def workload(inputs, name):
    if name.endswith("_mid"):
        return inputs.config(name[:-4], "mid")
    return inputs.config(name)


def traffic_source(key):
    src = TRAFFIC_FROM.get(key, key)
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)[src]
        how = "captured on this workload" if src == key else \
            "captured on %s, scaled by page spans" % src[len("gather_"):]
        return "%s, %s" % (rec.get("capture"), how)
    except Exception:
        return None


def d2d_copy_gbps(nbytes, dev, stream):
    """A same-bytes device-to-device copy (torch copy_), the practical ceiling."""
    import torch
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
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
    del a, bb
    return 2 * nbytes / (e0.elapsed_time(e1) / 20 * 1e-3) / 1e9


def reference_arm(args, w, config, decode):
    """The CPU oracle as it stands, on every host thread, each step over a prefix of the
    batch sized so that the whole --steps/--warmup run takes about two minutes (for a
    decode step: the oracle's append of the new rows, then the gather of the prefix)."""
    import oracle
    oracle.build()
    host_pool, fill = host_pool_for(w)
    scales = host_scales_for(w)
    per_step = max(0.002, 120.0 / (args.steps + args.warmup))
    nthr = host_threads()
    probe = OracleThreads(w, host_pool, oracle, nthr, tokens_cap=1 << 16, scales=scales)
    probe.step()
    t0 = time.perf_counter()
    probe.step()
    rate = probe.tokens / max(time.perf_counter() - t0, 1e-6)
    probe.close()
    cap = int(rate * per_step)
    run = OracleThreads(w, host_pool, oracle, nthr, None if cap >= w.total_tokens else max(256, cap),
                        scales=scales, append=decode)
    for _ in range(args.warmup):
        run.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run.step()
    el = time.perf_counter() - t0
    run.close()
    value = run.bytes * args.steps / el / 1e9
    what = ("append of the %d new rows, then gather" % w.total_new) if decode else \
        ("dequantising gather" if scales is not None else "gather")
    sample = ("oracle %s of the first %d of %d tokens per step on %d host threads (one "
              "contiguous group of sequences each); pool %s" % (what, run.tokens, w.total_tokens,
                                                               run.threads, fill))
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


if __name__ == "__main__":
    main()
