"""Seeded synthetic workloads for the block-paged KV cache, and the host block allocator.

This module builds inputs only: block tables, ``seq_ptr`` offsets, token counts
and page-pool contents.  It holds none of the lookup arithmetic, so the CUDA
library and the CPU oracle can both be fed from it without sharing code.

* ``BlockAllocator`` / ``RequestState`` follow the free-list allocator of
  "Visualize PagedAttention block layout" (sections "The block allocator" and
  "Block tables: the page table equivalent").  The printed trace hands out the
  lowest free block first (A gets [0, 1, 2] out of 20 free blocks), so that is
  the default order here; an explicit order (a shuffled free list) may be given
  instead, consumed front to back.
* The workload builders reproduce the five benchmark configurations (tiny
  prefix-sharing gather, decode-sized gather, decode append then gather, prefix
  sharing at scale, int8 pool with per-slot scales) plus scaled-down versions
  for exhaustive checks, and the per-lane layout of "Keep token order across
  cache pages".

Index structures always come from ``numpy.random.default_rng(seed)`` (PCG64),
which gives the same numbers on every platform.  Pool contents come from numpy
for small pools and from a seeded ``torch.Generator`` on the pool's device for
large ones; either way the same bytes go to every consumer.  Slots that hold no
live token (the tail of a partial last page, wholly unused pages) are filled
with the byte 0x7F so that a reader that strays into them produces a visible
mismatch.
"""
from __future__ import annotations

import dataclasses
import heapq
from collections import deque
from typing import Optional

import numpy as np

SENTINEL = 0x7F

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1, "u8": 1, "f64": 8}


# --------------------------------------------------------------------------- allocator
class BlockAllocator:
    """Free list of physical block IDs with reference counts for copy-on-write sharing.

    ``allocate`` takes the next free block (lowest ID first by default, or the
    next entry of ``order``) and sets its count to 1; ``free`` drops a reference
    and returns the block to the free list at zero; ``share`` adds a reference.
    Raises ``RuntimeError("Out of KV cache blocks")`` when nothing is free.
    """

    def __init__(self, num_blocks: int, block_size: int = 16, order=None):
        self.block_size = block_size
        self.ref_counts = [0] * num_blocks
        if order is None:
            self._heap = list(range(num_blocks))
            heapq.heapify(self._heap)
            self._fifo = None
        else:
            order = [int(b) for b in order]
            if sorted(order) != list(range(num_blocks)):
                raise ValueError("order must be a permutation of the block IDs")
            self._heap = None
            self._fifo = deque(order)

    def allocate(self) -> int:
        if self.num_free == 0:
            raise RuntimeError("Out of KV cache blocks")
        block_id = heapq.heappop(self._heap) if self._fifo is None else self._fifo.popleft()
        self.ref_counts[block_id] = 1
        return block_id

    def free(self, block_id: int) -> None:
        if self.ref_counts[block_id] <= 0:
            raise ValueError("block %d is not allocated" % block_id)
        self.ref_counts[block_id] -= 1
        if self.ref_counts[block_id] == 0:
            if self._fifo is None:
                heapq.heappush(self._heap, block_id)
            else:
                self._fifo.append(block_id)

    def share(self, block_id: int) -> None:
        if self.ref_counts[block_id] <= 0:
            raise ValueError("block %d is not allocated" % block_id)
        self.ref_counts[block_id] += 1

    def cow(self, block_id: int) -> int:
        """Copy-on-write: the block a request may modify in place.  A block it holds
        alone is returned as is; a shared one loses this reference and a fresh block is
        allocated, which the caller fills with a copy of the old one before writing."""
        if self.ref_counts[block_id] <= 0:
            raise ValueError("block %d is not allocated" % block_id)
        if self.ref_counts[block_id] == 1:
            return block_id
        fresh = self.allocate()
        self.ref_counts[block_id] -= 1
        return fresh

    @property
    def num_free(self) -> int:
        return len(self._heap) if self._fifo is None else len(self._fifo)


class RequestState:
    """A request's share of the cache: its token count and, in logical order, the
    physical blocks holding those tokens.  The invariant kept is that the table has
    exactly ceil(num_tokens / block_size) blocks: admission sizes it for the prompt,
    and a token that opens a new block draws one more from the allocator (the trace of
    "Visualizing the layout": a 4-block request grows to 4 + 1 blocks when its 10 new
    tokens cross one boundary).  Releasing hands every block back, first to last."""

    def __init__(self, request_id, prompt_len: int, allocator: BlockAllocator):
        self.request_id = request_id
        self.allocator = allocator
        self.block_table = []
        self.num_tokens = 0
        self._grow_to(prompt_len)

    def _grow_to(self, tokens: int) -> None:
        self.num_tokens = tokens
        bs = self.allocator.block_size
        while len(self.block_table) * bs < tokens:
            self.block_table.append(self.allocator.allocate())

    def append_token(self) -> None:
        self._grow_to(self.num_tokens + 1)

    def release(self) -> None:
        held, self.block_table = self.block_table, []
        for block_id in held:
            self.allocator.free(block_id)


# --------------------------------------------------------------------------- workloads
@dataclasses.dataclass
class Workload:
    """A block-paged batch: pool geometry, index buffers and how to fill the pool."""
    name: str
    num_pages: int
    page_size: int
    num_heads: int
    head_dim: int
    dtype: str                    # element type of the page pool
    index_dtype: type             # np.uint32 or np.uint64
    table: np.ndarray             # block_table, concatenated per-sequence slices
    seq_ptr: np.ndarray           # num_seqs + 1 offsets into table
    lens: np.ndarray              # per-sequence token counts the batch is read with
    pool_seed: int
    pool_dist: str                # "uniform(-1,1)", "normal", "randint(-127,127)"
    scales_seed: Optional[int] = None   # int8 pools: fp32 per-slot scales U[0.001, 0.05]
    # decode append (when present): counts before the append, CSR of the new rows
    lens_before: Optional[np.ndarray] = None
    new_ptr: Optional[np.ndarray] = None
    new_seed: Optional[int] = None

    @property
    def num_seqs(self) -> int:
        return len(self.lens)

    @property
    def row_bytes(self) -> int:
        return self.num_heads * self.head_dim * ELEM_BYTES[self.dtype]

    @property
    def total_tokens(self) -> int:
        return int(np.sum(self.lens.astype(np.uint64)))

    @property
    def pool_bytes(self) -> int:
        return self.num_pages * self.page_size * self.row_bytes

    @property
    def total_new(self) -> int:
        return 0 if self.new_ptr is None else int(self.new_ptr[-1])

    def live_slots(self, lens=None) -> np.ndarray:
        """Per physical page, how many leading slots hold a live token of some
        sequence (tokens fill a page from slot 0)."""
        lens = self.lens if lens is None else lens
        live = np.zeros(self.num_pages, dtype=np.int64)
        P = self.page_size
        for s in range(self.num_seqs):
            lo, hi = int(self.seq_ptr[s]), int(self.seq_ptr[s + 1])
            n = int(lens[s])
            pages = self.table[lo:hi].astype(np.int64)
            k = np.minimum(np.maximum(n - P * np.arange(hi - lo), 0), P)
            np.maximum.at(live, pages, k)
        return live


def _slices(tables, index_dtype):
    seq_ptr = np.zeros(len(tables) + 1, dtype=np.uint64)
    seq_ptr[1:] = np.cumsum([len(t) for t in tables])
    table = np.concatenate([np.asarray(t, dtype=np.uint64) for t in tables]) if tables else \
        np.zeros(0, dtype=np.uint64)
    return table.astype(index_dtype), seq_ptr.astype(index_dtype)


def _need(n, P):
    return -(-int(n) // P)


def _draw_lens(rng, num_seqs, lo, hi, P, num_pages, extra=0):
    """Token counts ~ U[lo, hi] (inclusive); redrawn from the same stream while
    the batch's pages (plus ``extra`` per-sequence slack) exceed the pool."""
    for _ in range(1000):
        lens = rng.integers(lo, hi, size=num_seqs, endpoint=True)
        need = int(np.sum(-(-(lens.astype(np.int64) + extra) // P)))
        if need <= num_pages:
            return lens
    raise ValueError("%d pages cannot hold %d sequences of U[%d, %d] tokens"
                     % (num_pages, num_seqs, lo, hi))


def tiny_prefix_gather() -> Workload:
    """16 fp32 pages of 4 slots x 2 heads x 4 dims ~ U(-1,1) (seed 0); two
    sequences with slices [12,5,7,9] (15 tokens) and [12,5,7,3] (13 tokens),
    the prefix-sharing example of the Hurray specification, uint32 indices."""
    table = np.array([12, 5, 7, 9, 12, 5, 7, 3], dtype=np.uint32)
    return Workload("tiny_prefix_gather", 16, 4, 2, 4, "f32", np.uint32, table,
                    np.array([0, 4, 8], dtype=np.uint32), np.array([15, 13], dtype=np.uint32),
                    pool_seed=0, pool_dist="uniform(-1,1)")


def decode_gather(seed=2, num_pages=10000, page_size=16, num_heads=32, head_dim=128,
                  num_seqs=64, len_lo=512, len_hi=4096, dtype="f16",
                  index_dtype=np.uint32, name="decode_gather") -> Workload:
    """fp16 K pool ~N(0,1); token counts ~U[len_lo, len_hi]; each sequence takes
    ceil(len/P) pages, in order, from one shuffled free list."""
    rng = np.random.default_rng(seed)
    lens = _draw_lens(rng, num_seqs, len_lo, len_hi, page_size, num_pages)
    alloc = BlockAllocator(num_pages, page_size, order=rng.permutation(num_pages))
    tables = [RequestState(s, int(n), alloc).block_table for s, n in enumerate(lens)]
    table, seq_ptr = _slices(tables, index_dtype)
    return Workload(name, num_pages, page_size, num_heads, head_dim, dtype, index_dtype,
                    table, seq_ptr, lens.astype(index_dtype), pool_seed=seed, pool_dist="normal")


def decode_append(seed=3, num_pages=300000, page_size=16, num_heads=8, head_dim=128,
                  num_seqs=256, len_lo=1024, len_hi=32768, new_per_seq=1, dtype="bf16",
                  index_dtype=np.uint32, name="decode_append") -> Workload:
    """bf16 GQA pool ~N(0,1).  Each sequence holds len ~U[len_lo, len_hi] tokens,
    then appends ``new_per_seq`` rows ~N(0,1) at positions len, len+1, ...; a
    sequence takes a new page from the shuffled free list whenever a new token
    lands at a page boundary (len % P == 0), after every sequence's initial
    pages.  ``lens`` is the count after the append (what the gather reads);
    ``lens_before`` the count the append starts from."""
    rng = np.random.default_rng(seed)
    lens = _draw_lens(rng, num_seqs, len_lo, len_hi, page_size, num_pages, extra=new_per_seq)
    alloc = BlockAllocator(num_pages, page_size, order=rng.permutation(num_pages))
    reqs = [RequestState(s, int(n), alloc) for s, n in enumerate(lens)]
    for r in reqs:
        for _ in range(new_per_seq):
            r.append_token()
    table, seq_ptr = _slices([r.block_table for r in reqs], index_dtype)
    after = np.array([r.num_tokens for r in reqs], dtype=np.uint64)
    new_ptr = (np.arange(num_seqs + 1, dtype=np.uint64) * new_per_seq).astype(index_dtype)
    return Workload(name, num_pages, page_size, num_heads, head_dim, dtype, index_dtype,
                    table, seq_ptr, after.astype(index_dtype), pool_seed=seed,
                    pool_dist="normal", lens_before=lens.astype(index_dtype), new_ptr=new_ptr,
                    new_seed=seed + 1000)


def prefix_sharing(seed=4, num_pages=16384, page_size=16, num_heads=8, head_dim=128,
                   num_seqs=128, prompt_tokens=2048, suf_lo=64, suf_hi=1024, dtype="bf16",
                   index_dtype=np.uint32, name="prefix_sharing") -> Workload:
    """All sequences alias the same ceil(prompt/P) physical pages (the first IDs
    of the shuffled free list, shared by reference count) for a common prompt,
    then take fresh pages for a unique suffix ~U[suf_lo, suf_hi]."""
    rng = np.random.default_rng(seed)
    alloc = BlockAllocator(num_pages, page_size, order=rng.permutation(num_pages))
    prompt = RequestState("prompt", prompt_tokens, alloc)
    suffix = rng.integers(suf_lo, suf_hi, size=num_seqs, endpoint=True)
    tables = []
    for n in suffix:
        for b in prompt.block_table:
            alloc.share(b)
        own = RequestState(None, int(n), alloc).block_table
        tables.append(list(prompt.block_table) + own)
    table, seq_ptr = _slices(tables, index_dtype)
    lens = (suffix + prompt_tokens).astype(index_dtype)
    return Workload(name, num_pages, page_size, num_heads, head_dim, dtype, index_dtype,
                    table, seq_ptr, lens, pool_seed=seed, pool_dist="normal")


def quantized_pool(seed=5, num_pages=400000, page_size=32, num_heads=8, head_dim=128,
                   num_seqs=1024, len_lo=256, len_hi=8192, index_dtype=np.uint64,
                   name="quantized_pool") -> Workload:
    """int8 symmetric pool ~U[-127,127] with fp32 per-slot scales ~U[0.001,0.05]
    (num_pages*page_size of them), uint64 table and offsets."""
    rng = np.random.default_rng(seed)
    lens = _draw_lens(rng, num_seqs, len_lo, len_hi, page_size, num_pages)
    alloc = BlockAllocator(num_pages, page_size, order=rng.permutation(num_pages))
    tables = [RequestState(s, int(n), alloc).block_table for s, n in enumerate(lens)]
    table, seq_ptr = _slices(tables, index_dtype)
    return Workload(name, num_pages, page_size, num_heads, head_dim, "i8", index_dtype,
                    table, seq_ptr, lens.astype(index_dtype), pool_seed=seed,
                    pool_dist="randint(-127,127)", scales_seed=seed + 2000)


# Full-size configurations and scaled-down versions the CPU oracle checks whole.
def config(name: str, scale: str = "full") -> Workload:
    if name == "tiny_prefix_gather":
        return tiny_prefix_gather()
    small = scale == "small"
    if name == "decode_gather":
        return decode_gather(num_pages=600, num_seqs=7, len_lo=1, len_hi=700,
                             name="decode_gather_small") if small else decode_gather()
    if name == "decode_append":
        if scale == "mid":  # 32 sequences, about 2.5 GB of K and V pools
            return decode_append(num_pages=40000, num_seqs=32, name="decode_append_mid")
        if scale == "short":  # 2048 short sequences (16 to 1024 tokens), about 4.4 GB read
            return decode_append(num_pages=80000, num_seqs=2048, len_lo=16, len_hi=1024,
                                 name="decode_append_short")
        return decode_append(num_pages=2000, num_seqs=9, len_lo=1, len_hi=2000,
                             name="decode_append_small") if small else decode_append()
    if name == "prefix_sharing":
        return prefix_sharing(num_pages=700, num_seqs=6, prompt_tokens=200, suf_lo=1,
                              suf_hi=300, name="prefix_sharing_small") if small else prefix_sharing()
    if name == "quantized_pool":
        if scale == "mid":  # about 2.5 GB moved: small enough for a full profiler capture
            return quantized_pool(num_pages=50000, num_seqs=128, name="quantized_pool_mid")
        return quantized_pool(num_pages=1500, num_seqs=11, len_lo=1, len_hi=900,
                              name="quantized_pool_small") if small else quantized_pool()
    raise KeyError(name)


CONFIG_NAMES = ("tiny_prefix_gather", "decode_gather", "decode_append", "prefix_sharing",
                "quantized_pool")


# --------------------------------------------------------------------------- pool contents
def _host_values(dist, seed, count, dtype):
    rng = np.random.default_rng(seed)
    if dist == "uniform(-1,1)":
        v = rng.uniform(-1.0, 1.0, count)
    elif dist == "normal":
        v = rng.standard_normal(count, dtype=np.float32)
    elif dist == "randint(-127,127)":
        return rng.integers(-127, 127, size=count, endpoint=True).astype(np.int8).view(np.uint8)
    else:
        raise ValueError(dist)
    return _to_bytes(np.asarray(v), dtype)


def _to_bytes(v, dtype):
    if dtype in ("i8", "u8"):  # a normal draw on an integer pool: 32 steps per unit, clipped
        return np.clip(np.rint(v * 32), -127, 127).astype(np.int8).view(np.uint8)
    if dtype == "f32":
        return v.astype(np.float32).view(np.uint8)
    if dtype == "f64":
        return v.astype(np.float64).view(np.uint8)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint8)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.uint16).numpy().view(np.uint8)
    raise ValueError(dtype)


def host_pool(w: Workload) -> np.ndarray:
    """Pool bytes as a numpy uint8 array [num_pages, page_size, row_bytes] with
    the non-live slots set to the sentinel byte (small workloads)."""
    n = w.num_pages * w.page_size * w.num_heads * w.head_dim
    raw = _host_values(w.pool_dist, w.pool_seed, n, w.dtype)
    pool = np.ascontiguousarray(raw).reshape(w.num_pages, w.page_size, w.row_bytes).copy()
    live = w.live_slots()
    dead = np.arange(w.page_size)[None, :] >= live[:, None]
    pool[dead] = SENTINEL
    return pool


def host_scales(w: Workload) -> np.ndarray:
    rng = np.random.default_rng(w.scales_seed)
    return rng.uniform(0.001, 0.05, w.num_pages * w.page_size).astype(np.float32)


def host_new_rows(w: Workload) -> np.ndarray:
    """The append's new rows, ~N(0,1), as uint8 [total_new, row_bytes]."""
    rng = np.random.default_rng(w.new_seed)
    v = rng.standard_normal(w.total_new * w.num_heads * w.head_dim, dtype=np.float32)
    return np.ascontiguousarray(_to_bytes(v, w.dtype)).reshape(w.total_new, w.row_bytes)


_TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16", "i8": "int8",
             "u8": "uint8", "f64": "float64"}


def device_pool(w: Workload, device, *, force_device_rng: bool = False):
    """Pool as a torch uint8 tensor [num_pages, page_size, row_bytes] on ``device``.

    Small pools reuse the numpy bytes of ``host_pool``; large ones (over 64 MiB,
    or when ``force_device_rng``) are drawn on the device with a seeded
    ``torch.Generator`` -- the same distribution, different bytes, identical for
    every consumer of the returned tensor."""
    import torch
    if w.pool_bytes <= (64 << 20) and not force_device_rng:
        return torch.from_numpy(host_pool(w)).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.pool_seed)
    shape = (w.num_pages, w.page_size, w.num_heads * w.head_dim)
    dt = getattr(torch, _TORCH_DT[w.dtype])
    if w.pool_dist == "normal":
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32 if dt in (
            torch.float16, torch.bfloat16) else dt)
        t = t.to(dt)
    elif w.pool_dist == "uniform(-1,1)":
        t = torch.rand(shape, generator=g, device=device, dtype=dt) * 2 - 1
    elif w.pool_dist == "randint(-127,127)":
        t = torch.randint(-127, 128, shape, generator=g, device=device, dtype=torch.int8)
    else:
        raise ValueError(w.pool_dist)
    pool = t.view(torch.uint8).view(w.num_pages, w.page_size, w.row_bytes)
    live = torch.from_numpy(w.live_slots()).to(device)
    dead = torch.arange(w.page_size, device=device)[None, :] >= live[:, None]
    pool.masked_fill_(dead[:, :, None], SENTINEL)
    return pool


def device_scales(w: Workload, device, *, force_device_rng: bool = False):
    import torch
    n = w.num_pages * w.page_size
    if n * 4 <= (64 << 20) and not force_device_rng:
        return torch.from_numpy(host_scales(w)).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.scales_seed)
    return torch.rand(n, generator=g, device=device, dtype=torch.float32) * 0.049 + 0.001


def device_new_rows(w: Workload, device):
    import torch
    return torch.from_numpy(host_new_rows(w)).to(device)


# --------------------------------------------------------------------------- per-lane layout
@dataclasses.dataclass
class LaneWorkload:
    """The [N, B, H_kv, P, d] layout of "Keep token order across cache pages":
    capacity C, P positions per page, a permutation table T of N = ceil(C/P)
    pages, B batch lanes, H_kv shared heads, d features, n live rows."""
    name: str
    capacity: int
    page_tokens: int
    table: np.ndarray
    batch: int
    kv_heads: int
    width: int
    dtype: str
    n: int
    seed: int

    @property
    def pages(self) -> int:
        return _need(self.capacity, self.page_tokens)

    @property
    def lanes(self) -> int:
        return self.batch * self.kv_heads

    @property
    def pool_shape(self):
        return (self.pages, self.batch, self.kv_heads, self.page_tokens, self.width)

    @property
    def es(self) -> int:
        return ELEM_BYTES[self.dtype]


def lane_worked_example() -> LaneWorkload:
    """Capacity 12, 3 positions per page, T = (2, 0, 3, 1), one batch lane, two
    shared K/V heads of two f64 features, seven live positions."""
    return LaneWorkload("lane_worked_example", 12, 3, np.array([2, 0, 3, 1], dtype=np.uint64),
                        1, 2, 2, "f64", 7, seed=20)


def lane_synthetic(seed=6, capacity=8192, page_tokens=16, batch=32, kv_heads=8, width=128,
                   dtype="bf16", n=None, name="lane_synthetic") -> LaneWorkload:
    rng = np.random.default_rng(seed)
    pages = _need(capacity, page_tokens)
    table = rng.permutation(pages).astype(np.uint64)
    if n is None:
        n = int(rng.integers(capacity // 2, capacity - 1, endpoint=True))
    return LaneWorkload(name, capacity, page_tokens, table, batch, kv_heads, width, dtype, n,
                        seed=seed)


def lane_host_pool(w: LaneWorkload) -> np.ndarray:
    count = int(np.prod(w.pool_shape))
    raw = _host_values("normal", w.seed, count, w.dtype)
    return np.ascontiguousarray(raw).reshape(*w.pool_shape[:-1], w.width * w.es).copy()


def lane_host_new_rows(w: LaneWorkload, m: int) -> np.ndarray:
    rng = np.random.default_rng(w.seed + 1000)
    v = rng.standard_normal(w.lanes * m * w.width, dtype=np.float32)
    return np.ascontiguousarray(_to_bytes(v, w.dtype)).reshape(w.batch, w.kv_heads, m,
                                                                w.width * w.es)
