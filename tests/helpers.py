"""Test plumbing: puts one seeded workload in front of both the CUDA library and
the CPU oracle.  Only marshalling -- no lookup arithmetic lives here."""
import numpy as np

from paged_kv_cache_hp_gb300 import inputs

# library status name <- oracle rule name
def lib_name(oracle_name: str) -> str:
    return "HP_OK" if oracle_name == "OK" else "HP_ERR_" + oracle_name


def index_tensor(arr, device):
    """numpy uint32/uint64 -> torch int32/int64 tensor with the same bytes."""
    import torch
    a = np.ascontiguousarray(arr)
    view = a.view(np.int32) if a.dtype == np.uint32 else a.astype(np.uint64).view(np.int64)
    return torch.from_numpy(view.copy()).to(device)


class Batch:
    """Device tensors + an hp descriptor + an oracle descriptor for one workload."""

    def __init__(self, w: inputs.Workload, device="cuda", pool=None, host_pool=None, flags=0,
                 lens=None, **desc_overrides):
        import torch
        from paged_kv_cache_hp_gb300 import hp
        import oracle
        self.w = w
        it = 0 if w.index_dtype == np.uint32 else 1
        self.it = it
        self.lens_host = np.ascontiguousarray(w.lens if lens is None else lens, dtype=w.index_dtype)
        if pool is None:
            pool = inputs.device_pool(w, device)
        self.pool = pool
        self.table = index_tensor(w.table, device) if len(w.table) else None
        self.seq_ptr = index_tensor(w.seq_ptr, device)
        self.lens = index_tensor(self.lens_host, device)
        self.scales = None
        if w.scales_seed is not None:
            self.scales = inputs.device_scales(w, device)
            flags |= hp.HAS_QUANT
        self.flags = flags
        self.desc = hp.PagedDesc(self.pool, self.table, self.seq_ptr, self.lens,
                                 num_pages=w.num_pages, page_size=w.page_size,
                                 num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype,
                                 index_type=it, scales=self.scales, flags=flags, **desc_overrides)
        self.ws = hp.workspace_for(self.desc, device)
        self.status = torch.full((1,), 12345, dtype=torch.int32, device=device)
        self._host_pool = host_pool

    def host_pool(self):
        if self._host_pool is None:
            self._host_pool = self.pool.cpu().numpy()
        return self._host_pool

    def oracle_desc(self, pool_host=None, lens=None, **overrides):
        import oracle
        w = self.w
        sc = None if self.scales is None else self.scales.cpu().numpy()
        return oracle.Desc(self.host_pool() if pool_host is None else pool_host,
                           w.table if len(w.table) else None, w.seq_ptr,
                           self.lens_host if lens is None else lens,
                           num_pages=w.num_pages, page_size=w.page_size, num_heads=w.num_heads,
                           head_dim=w.head_dim, dtype=w.dtype, scales=sc, flags=self.flags,
                           index_type=self.it,
                           addrs={"pool": self.pool.data_ptr(),
                                  "table": 0 if self.table is None else self.table.data_ptr(),
                                  "seq_ptr": self.seq_ptr.data_ptr(),
                                  "lens": self.lens.data_ptr(),
                                  "scales": 0 if self.scales is None else self.scales.data_ptr()},
                           **overrides)

    def status_value(self):
        return int(self.status.item())


def sub_batch(w: inputs.Workload, seqs, lens=None):
    """The CSR slices of a few sequences, re-based: (table, seq_ptr, lens) numpy arrays
    describing just those sequences, in the given order."""
    lens = w.lens if lens is None else lens
    sp = w.seq_ptr.astype(np.int64)
    tables = [w.table[sp[s]:sp[s + 1]] for s in seqs]
    seq_ptr = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(w.index_dtype)
    table = np.concatenate(tables).astype(w.index_dtype) if tables else np.zeros(0, w.index_dtype)
    return table, seq_ptr, np.asarray([lens[s] for s in seqs], dtype=w.index_dtype)


# --------------------------------------------------------------- whole-output comparisons
def host_threads():
    import os
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def sequence_groups(lens, group_tokens):
    """Contiguous groups of sequences of about group_tokens tokens each (at least one
    sequence per group): a list of (s0, s1, row0, row1), rows in the gathered tensor."""
    lens = np.asarray(lens, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lens)])
    groups, s0 = [], 0
    S = len(lens)
    while s0 < S:
        s1 = int(np.searchsorted(off, off[s0] + group_tokens, side="right")) - 1
        s1 = min(S, max(s1, s0 + 1))
        groups.append((s0, s1, int(off[s0]), int(off[s1])))
        s0 = s1
    return groups


def oracle_group(oracle, w, host_pool, lens, s0, s1, pool_exec, scales=None):
    """The oracle's gather (or, with per-slot `scales`, its dequantising gather) of
    sequences s0..s1-1, each worker thread gathering one contiguous share of them
    through a re-based sub-descriptor into its rows of one output array.  Returns the
    rows: uint8 [T, row_bytes], or uint16 bf16 codes [T, H*D] when dequantising."""
    lens = np.asarray(lens, dtype=np.int64)
    sp = w.seq_ptr.astype(np.int64)
    T = int(lens[s0:s1].sum())
    if scales is None:
        out = np.empty((T, w.row_bytes), dtype=np.uint8)
    else:
        out = np.empty((T, w.num_heads * w.head_dim), dtype=np.uint16)
    n = s1 - s0
    parts = max(1, min(n, pool_exec._max_workers))
    cuts = np.linspace(s0, s1, parts + 1).astype(np.int64)
    base = int(lens[:s0].sum())
    it = 0 if w.index_dtype == np.uint32 else 1

    def one(k):
        a, b = int(cuts[k]), int(cuts[k + 1])
        if b <= a:
            return "OK"
        r0 = int(lens[:a].sum()) - base
        r1 = r0 + int(lens[a:b].sum())
        d = oracle.Desc(host_pool, w.table[sp[a]:sp[b]], (sp[a:b + 1] - sp[a]).astype(w.index_dtype),
                        lens[a:b].astype(w.index_dtype), num_pages=w.num_pages,
                        page_size=w.page_size, num_heads=w.num_heads, head_dim=w.head_dim,
                        dtype=w.dtype, index_type=it, scales=scales,
                        flags=0 if scales is None else oracle.HAS_QUANT)
        if scales is None:
            return d.gather(out[r0:r1])[2]
        return d.gather_dequant(out[r0:r1])[2]

    faults = list(pool_exec.map(one, range(parts)))
    assert all(f == "OK" for f in faults), faults
    return out


def compare_whole_gather(oracle, w, host_pool, lens, got_rows, group_tokens=1 << 19,
                         scales=None):
    """Every row of a gathered tensor against the oracle, group by group of sequences.
    got_rows(row0, row1) returns the library's rows [row1 - row0, ...] as a host array of
    the oracle's shape.  Returns the number of rows compared."""
    from concurrent.futures import ThreadPoolExecutor
    rows = 0
    with ThreadPoolExecutor(host_threads()) as ex:
        for s0, s1, r0, r1 in sequence_groups(lens, group_tokens):
            want = oracle_group(oracle, w, host_pool, lens, s0, s1, ex, scales=scales)
            got = got_rows(r0, r1)
            if not np.array_equal(got, want):
                bad = np.nonzero((got != want).reshape(len(want), -1).any(axis=1))[0]
                raise AssertionError("rows differ: %d of sequences %d..%d, first at row %d"
                                     % (len(bad), s0, s1 - 1, r0 + int(bad[0])))
            rows += r1 - r0
    return rows
