"""Test infrastructure only: the CPU oracle for the block-paged KV-cache path.

This package wraps ``hp_oracle.c`` (a plain, slow CPU restatement of the
Element Lookup, the storage-invariant checks, the per-lane layout of the
"Keep token order across cache pages" chapter and its payload counts) with
ctypes.  Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import it; the library under
``paged_kv_cache_hp_gb300`` never does, and the two share no code.

All arguments are plain numpy arrays.  Nothing here touches a GPU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hp_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# element types, by name, with the oracle's own numbering
DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3, "u8": 4, "f64": 5}
PERMISSIVE = 1
HAS_QUANT = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile hp_oracle.c into liboracle.so beside it (gcc, ISO C11, no fast-math)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


class OrDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in
                ("rank", "paged_axis", "has_shard", "flags", "dtype", "index_type")] + \
               [(n, ctypes.c_uint64) for n in
                ("num_pages", "page_size", "num_heads", "head_dim", "num_seqs",
                 "table_len", "scales_len")] + \
               [("page_pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("seq_ptr", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("scales", ctypes.c_void_p)] + \
               [(n, ctypes.c_uint64) for n in
                ("addr_pool", "addr_table", "addr_seq_ptr", "addr_lens", "addr_scales")]


class OrQuant(ctypes.Structure):
    _fields_ = [("scheme_tag", ctypes.c_uint32), ("axis", ctypes.c_uint32),
                ("block_size", ctypes.c_uint64), ("count", ctypes.c_uint64),
                ("scales", ctypes.c_void_p), ("zero_points", ctypes.c_void_p),
                ("addr_scales", ctypes.c_uint64), ("addr_zero_points", ctypes.c_uint64)]


PER_TENSOR, PER_CHANNEL, PER_BLOCK_AFFINE = 0x01, 0x02, 0x03


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            u64, vp, i32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int
            P = ctypes.POINTER
            L.or_code_name.restype = ctypes.c_char_p
            L.or_code_name.argtypes = [i32]
            L.or_elem_size.restype = u64
            L.or_elem_size.argtypes = [ctypes.c_uint32]
            L.or_validate.restype = i32
            L.or_validate.argtypes = [P(OrDesc), P(u64)]
            L.or_validate_append.restype = i32
            L.or_validate_append.argtypes = [P(OrDesc), vp, u64, P(u64)]
            L.or_total_tokens.restype = u64
            L.or_total_tokens.argtypes = [P(OrDesc), P(i32)]
            L.or_lookup.restype = i32
            L.or_lookup.argtypes = [P(OrDesc), u64, u64, u64, u64, vp]
            L.or_lookup_dequant.restype = i32
            L.or_lookup_dequant.argtypes = [P(OrDesc), u64, u64, u64, u64, P(ctypes.c_uint16)]
            L.or_gather.restype = i32
            L.or_gather.argtypes = [P(OrDesc), vp, vp]
            L.or_gather_dequant.restype = i32
            L.or_gather_dequant.argtypes = [P(OrDesc), vp, vp]
            L.or_scatter_append.restype = i32
            L.or_scatter_append.argtypes = [P(OrDesc), vp, vp, u64]
            L.or_bf16_rne.restype = ctypes.c_uint16
            L.or_bf16_rne.argtypes = [ctypes.c_double]
            L.or_lane_new.restype = i32
            L.or_lane_new.argtypes = [u64, u64, vp, u64, P(u64)]
            L.or_lane_address.restype = i32
            L.or_lane_address.argtypes = [u64, u64, vp, u64, P(u64)]
            L.or_lane_row_start.restype = u64
            L.or_lane_row_start.argtypes = [u64, u64, vp, u64, u64, u64, u64]
            L.or_lane_physical_row_start.restype = i32
            L.or_lane_physical_row_start.argtypes = [u64, u64, vp, u64, u64, u64, u64, u64, u64, P(u64)]
            L.or_lane_gather.restype = None
            L.or_lane_gather.argtypes = [vp, u64, u64, vp, u64, u64, u64, u64, u64, vp]
            L.or_lane_append.restype = i32
            L.or_lane_append.argtypes = [vp, u64, u64, vp, u64, u64, u64, u64, u64, u64, vp]
            Q = P(OrQuant)
            L.or_validate_quant.restype = i32
            L.or_validate_quant.argtypes = [P(OrDesc), Q]
            L.or_lookup_dequant_q.restype = i32
            L.or_lookup_dequant_q.argtypes = [P(OrDesc), Q, u64, u64, u64, u64,
                                              P(ctypes.c_uint16)]
            L.or_gather_dequant_q.restype = i32
            L.or_gather_dequant_q.argtypes = [P(OrDesc), Q, vp, vp]
            L.or_copy_pages.restype = i32
            L.or_copy_pages.argtypes = [vp, u64, u64, ctypes.c_uint32, vp, vp, u64]
            L.or_zero_tails.restype = None
            L.or_zero_tails.argtypes = [P(OrDesc), vp]
            L.or_from_kernel_layout.restype = None
            L.or_from_kernel_layout.argtypes = [vp, vp, u64, u64, u64, u64, u64, u64]
            L.or_to_kernel_layout.restype = None
            L.or_to_kernel_layout.argtypes = [vp, vp, u64, u64, u64, u64, u64, u64]
            L.or_padded_to_csr.restype = i32
            L.or_padded_to_csr.argtypes = [vp, vp, u64, u64, u64, ctypes.c_uint32, vp, u64, vp,
                                           P(u64)]
            L.or_csr_to_padded.restype = i32
            L.or_csr_to_padded.argtypes = [vp, vp, u64, u64, u64, ctypes.c_uint32, vp, P(u64)]
            L.or_f16_to_double.restype = ctypes.c_double
            L.or_f16_to_double.argtypes = [ctypes.c_uint16]
            L.or_bf16_to_double.restype = ctypes.c_double
            L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.or_attention_decode.restype = None
            L.or_attention_decode.argtypes = [P(OrDesc), vp, vp, u64, ctypes.c_double, vp]
            L.or_payload.restype = i32
            L.or_payload.argtypes = [u64, u64, u64, u64, u64, u64, P(u64)]
            _lib = L
    return _lib


def code_name(code: int) -> str:
    return lib().or_code_name(code).decode()


def _ptr(a):
    return None if a is None else a.ctypes.data


class Desc:
    """A block-paged descriptor over host numpy arrays, held alive with it.

    ``pool`` is a numpy array whose raw bytes are the page pool
    [num_pages, page_size, num_heads, head_dim] in element type ``dtype``.
    ``table``, ``seq_ptr`` and ``lens`` are uint32 or uint64 arrays (the index
    type follows ``table``'s dtype unless ``index_type`` is given).  ``addrs``
    overrides the buffer addresses the structural checks see (for example the
    device addresses of the same buffers); by default the host addresses are
    used, with a 64-byte-aligned stand-in for each present buffer.
    """

    def __init__(self, pool, table, seq_ptr, lens, *, num_pages, page_size, num_heads,
                 head_dim, dtype, scales=None, index_type=None, flags=0, rank=3,
                 paged_axis=0, has_shard=0, table_len=None, num_seqs=None,
                 scales_len=None, addrs=None):
        if index_type is None:
            index_type = 0 if np.asarray(seq_ptr).dtype == np.uint32 else 1
        it = np.uint32 if index_type == 0 else np.uint64
        self.pool = pool
        self.table = None if table is None else np.ascontiguousarray(table, dtype=it)
        self.seq_ptr = np.ascontiguousarray(seq_ptr, dtype=it)
        self.lens = np.ascontiguousarray(lens, dtype=it)
        self.scales = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
        d = OrDesc()
        d.rank, d.paged_axis, d.has_shard, d.flags = rank, paged_axis, has_shard, flags
        d.dtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
        d.index_type = index_type
        d.num_pages, d.page_size, d.num_heads, d.head_dim = num_pages, page_size, num_heads, head_dim
        d.num_seqs = len(self.lens) if num_seqs is None else num_seqs
        d.table_len = (0 if self.table is None else len(self.table)) if table_len is None else table_len
        d.scales_len = (0 if self.scales is None else len(self.scales)) if scales_len is None else scales_len
        d.page_pool = _ptr(pool)
        d.block_table = _ptr(self.table)
        d.seq_ptr = _ptr(self.seq_ptr)
        d.seq_lens = _ptr(self.lens)
        d.scales = _ptr(self.scales)
        present = {"pool": pool is not None, "table": self.table is not None and d.table_len > 0,
                   "seq_ptr": True, "lens": True, "scales": self.scales is not None}
        a = {k: (64 * (i + 1) if v else 0) for i, (k, v) in enumerate(present.items())}
        if addrs:
            a.update(addrs)
        d.addr_pool, d.addr_table, d.addr_seq_ptr = a["pool"], a["table"], a["seq_ptr"]
        d.addr_lens, d.addr_scales = a["lens"], a["scales"]
        self.c = d
        self.es = lib().or_elem_size(d.dtype)

    # -- checks ------------------------------------------------------------
    def validate(self):
        first = ctypes.c_uint64(0)
        c = lib().or_validate(ctypes.byref(self.c), ctypes.byref(first))
        return code_name(c), first.value

    def validate_append(self, new_ptr, total_new):
        first = ctypes.c_uint64(0)
        npt = np.ascontiguousarray(new_ptr, dtype=self.seq_ptr.dtype)
        c = lib().or_validate_append(ctypes.byref(self.c), _ptr(npt), total_new, ctypes.byref(first))
        return code_name(c), first.value

    def total_tokens(self):
        ok = ctypes.c_int(0)
        t = lib().or_total_tokens(ctypes.byref(self.c), ctypes.byref(ok))
        return t if ok.value else None

    # -- lookups -----------------------------------------------------------
    def lookup(self, s, t, h, d):
        buf = np.zeros(self.es, dtype=np.uint8)
        c = lib().or_lookup(ctypes.byref(self.c), s, t, h, d, _ptr(buf))
        return code_name(c), buf

    def lookup_dequant(self, s, t, h, d):
        v = ctypes.c_uint16(0)
        c = lib().or_lookup_dequant(ctypes.byref(self.c), s, t, h, d, ctypes.byref(v))
        return code_name(c), v.value

    def gather(self, out=None):
        """Returns (out bytes as uint8 [T, H*D*es], rows_written mask, fault name)."""
        T = self.total_tokens()
        row_bytes = self.c.num_heads * self.c.head_dim * self.es
        if out is None:
            out = np.zeros((T, row_bytes), dtype=np.uint8)
        written = np.zeros(max(T, 1), dtype=np.uint8)
        c = lib().or_gather(ctypes.byref(self.c), _ptr(out), _ptr(written))
        return out, written[:T].astype(bool), code_name(c)

    def gather_dequant(self, out=None):
        """Returns (out uint16 bf16 codes [T, H*D], rows_written mask, fault name)."""
        T = self.total_tokens()
        if out is None:
            out = np.zeros((T, self.c.num_heads * self.c.head_dim), dtype=np.uint16)
        written = np.zeros(max(T, 1), dtype=np.uint8)
        c = lib().or_gather_dequant(ctypes.byref(self.c), _ptr(out), _ptr(written))
        return out, written[:T].astype(bool), code_name(c)

    # -- quantization schemes ----------------------------------------------
    @staticmethod
    def quant(scheme_tag, scales, zero_points=None, axis=0, block_size=0, count=None,
              addrs=None):
        """An OrQuant over host arrays (kept alive on the returned object's `keep`)."""
        sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
        zp = None if zero_points is None else np.ascontiguousarray(zero_points)
        q = OrQuant()
        q.scheme_tag, q.axis, q.block_size = scheme_tag, axis, block_size
        q.count = (0 if sc is None else len(sc)) if count is None else count
        q.scales, q.zero_points = _ptr(sc), _ptr(zp)
        a = {"scales": 64 * 8 if sc is not None else 0, "zero_points": 64 * 9 if zp is not None else 0}
        if addrs:
            a.update(addrs)
        q.addr_scales, q.addr_zero_points = a["scales"], a["zero_points"]
        q.keep = (sc, zp)
        return q

    def validate_quant(self, q):
        return code_name(lib().or_validate_quant(ctypes.byref(self.c), ctypes.byref(q)))

    def lookup_dequant_q(self, q, s, t, h, d):
        v = ctypes.c_uint16(0)
        c = lib().or_lookup_dequant_q(ctypes.byref(self.c), ctypes.byref(q), s, t, h, d,
                                      ctypes.byref(v))
        return code_name(c), v.value

    def gather_dequant_q(self, q, out=None):
        """Returns (out uint16 bf16 codes [T, H*D], rows_written mask, fault name)."""
        T = self.total_tokens()
        if out is None:
            out = np.zeros((T, self.c.num_heads * self.c.head_dim), dtype=np.uint16)
        written = np.zeros(max(T, 1), dtype=np.uint8)
        c = lib().or_gather_dequant_q(ctypes.byref(self.c), ctypes.byref(q), _ptr(out),
                                      _ptr(written))
        return out, written[:T].astype(bool), code_name(c)

    # -- writer side ----------------------------------------------------------
    def copy_pages(self, src, dst):
        """Copies page src[i] over page dst[i] in self.pool, in place; returns the code."""
        it = self.seq_ptr.dtype
        a = np.ascontiguousarray(src, dtype=it)
        b = np.ascontiguousarray(dst, dtype=it)
        pb = self.c.page_size * self.c.num_heads * self.c.head_dim * self.es
        return code_name(lib().or_copy_pages(_ptr(self.pool), self.c.num_pages, pb,
                                             self.c.index_type, _ptr(a), _ptr(b), len(a)))

    def zero_tails(self):
        """Zeroes the slots no sequence reads, in self.pool; returns the per-page live counts."""
        live = np.zeros(max(self.c.num_pages, 1), dtype=np.uint64)
        lib().or_zero_tails(ctypes.byref(self.c), _ptr(live))
        return live[:self.c.num_pages]

    def attention_decode(self, v_pool, q, num_q_heads, scale):
        """Decode attention over this descriptor's K pool and v_pool (same geometry);
        q [num_seqs, Hq, D] of the pool's element type.  Returns float64 [S, Hq, D]."""
        vp_ = np.ascontiguousarray(v_pool)
        q_ = np.ascontiguousarray(q)
        out = np.zeros((self.c.num_seqs, num_q_heads, self.c.head_dim), np.float64)
        lib().or_attention_decode(ctypes.byref(self.c), _ptr(vp_), _ptr(q_), num_q_heads,
                                  float(scale), _ptr(out))
        return out

    def scatter_append(self, new_rows, new_ptr, total_new=None):
        """Writes into self.pool in place; returns the fault name.  total_new is the
        number of rows new_rows holds (by default, its byte size over one row's)."""
        npt = np.ascontiguousarray(new_ptr, dtype=self.seq_ptr.dtype)
        nr = np.ascontiguousarray(new_rows)
        if total_new is None:
            row_bytes = self.c.num_heads * self.c.head_dim * self.es
            total_new = nr.nbytes // row_bytes if row_bytes else 0
        return code_name(lib().or_scatter_append(ctypes.byref(self.c), _ptr(nr), _ptr(npt),
                                                 int(total_new)))


def bf16_rne(x: float) -> int:
    return lib().or_bf16_rne(float(x))


# -- per-lane layout ----------------------------------------------------------
def lane_new(capacity, page_tokens, table):
    t = np.ascontiguousarray(table, dtype=np.uint64)
    det = (ctypes.c_uint64 * 2)()
    c = lib().or_lane_new(capacity, page_tokens, _ptr(t) if len(t) else None, len(t), det)
    return code_name(c), (det[0], det[1])


def lane_address(capacity, page_tokens, table, position):
    t = np.ascontiguousarray(table, dtype=np.uint64)
    o = (ctypes.c_uint64 * 3)()
    if lib().or_lane_address(capacity, page_tokens, _ptr(t), position, o):
        return None
    return (o[0], o[1], o[2])


def lane_physical_row_start(capacity, page_tokens, table, batch_size, heads, width,
                            batch, head, position):
    t = None if table is None else np.ascontiguousarray(table, dtype=np.uint64)
    o = ctypes.c_uint64(0)
    if lib().or_lane_physical_row_start(capacity, page_tokens, _ptr(t), batch_size, heads,
                                        width, batch, head, position, ctypes.byref(o)):
        return None
    return o.value


def lane_gather(pool, capacity, page_tokens, table, batch_size, heads, width, n):
    """pool: numpy array holding [N, B, H, P, d]; returns out [B, H, n, d] (same dtype)."""
    t = None if table is None else np.ascontiguousarray(table, dtype=np.uint64)
    out = np.zeros((batch_size, heads, n, width), dtype=pool.dtype)
    lib().or_lane_gather(_ptr(np.ascontiguousarray(pool)), capacity, page_tokens, _ptr(t),
                         batch_size, heads, width, pool.dtype.itemsize, n, _ptr(out))
    return out


def lane_append(pool, capacity, page_tokens, table, batch_size, heads, width, n, new_rows):
    """Appends new_rows [B, H, m, d] at positions n..n+m-1 in place; returns the code name."""
    t = None if table is None else np.ascontiguousarray(table, dtype=np.uint64)
    nr = np.ascontiguousarray(new_rows)
    assert pool.flags.c_contiguous
    m = nr.shape[2]
    c = lib().or_lane_append(_ptr(pool), capacity, page_tokens, _ptr(t), batch_size, heads,
                             width, pool.dtype.itemsize, n, m, _ptr(nr))
    return code_name(c)


def from_kernel_layout(src, nb, bs, H, D, x):
    """Kernel-internal [nb, H, D/x, bs, x] (numpy array of any element type) ->
    interchange [nb, bs, H, D]."""
    src = np.ascontiguousarray(src)
    out = np.empty((nb, bs, H, D), dtype=src.dtype)
    lib().or_from_kernel_layout(_ptr(src), _ptr(out), nb, bs, H, D, x, src.dtype.itemsize)
    return out


def to_kernel_layout(src, nb, bs, H, D, x):
    """Interchange [nb, bs, H, D] -> kernel-internal [nb, H, D/x, bs, x]."""
    src = np.ascontiguousarray(src)
    out = np.empty((nb, H, D // x, bs, x), dtype=src.dtype)
    lib().or_to_kernel_layout(_ptr(src), _ptr(out), nb, bs, H, D, x, src.dtype.itemsize)
    return out


def padded_to_csr(padded, lens, page_size, table_cap=None):
    """padded [batch, max_blocks], lens [batch] (uint32 or uint64) -> (code, first,
    table, seq_ptr)."""
    padded = np.ascontiguousarray(padded)
    it = 0 if padded.dtype == np.uint32 else 1
    lens = np.ascontiguousarray(lens, dtype=padded.dtype)
    batch, mb = padded.shape
    cap = batch * mb if table_cap is None else table_cap
    table = np.zeros(max(cap, 1), dtype=padded.dtype)
    sp = np.zeros(batch + 1, dtype=padded.dtype)
    first = ctypes.c_uint64(0)
    c = lib().or_padded_to_csr(_ptr(padded), _ptr(lens), batch, mb, page_size, it, _ptr(table),
                               cap, _ptr(sp), ctypes.byref(first))
    name = code_name(c)
    return name, first.value, (table[:int(sp[-1])] if name == "OK" else None), sp


def csr_to_padded(table, seq_ptr, max_blocks, pad):
    seq_ptr = np.ascontiguousarray(seq_ptr)
    it = 0 if seq_ptr.dtype == np.uint32 else 1
    table = np.ascontiguousarray(table, dtype=seq_ptr.dtype)
    batch = len(seq_ptr) - 1
    out = np.zeros((batch, max_blocks), dtype=seq_ptr.dtype)
    first = ctypes.c_uint64(0)
    c = lib().or_csr_to_padded(_ptr(table) if len(table) else None, _ptr(seq_ptr), batch,
                               max_blocks, pad, it, _ptr(out), ctypes.byref(first))
    return code_name(c), first.value, out


PAYLOAD_FIELDS = ("reserved_pages", "active_pages", "allocated_scalar_slots",
                  "live_scalar_slots", "unused_scalar_slots",
                  "active_page_tail_scalar_slots", "inactive_page_scalar_slots",
                  "allocated_payload_bytes", "live_payload_bytes", "unused_payload_bytes",
                  "active_page_tail_payload_bytes", "inactive_page_payload_bytes")


def payload(capacity, page_tokens, length, batch, kv_heads, width):
    o = (ctypes.c_uint64 * 12)()
    c = lib().or_payload(capacity, page_tokens, length, batch, kv_heads, width, o)
    if c:
        return code_name(c)
    return dict(zip(PAYLOAD_FIELDS, list(o)))
