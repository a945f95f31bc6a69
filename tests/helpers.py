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
