"""Host-side logic: the block allocator and the seeded workload builders."""
import numpy as np
import pytest

from conftest import golden_kv, golden_lines
from paged_kv_cache_hp_gb300 import inputs


def test_allocator_trace():
    """"Visualize PagedAttention block layout", section "Visualizing the layout"."""
    g = golden_kv("allocator_trace.txt")
    alloc = inputs.BlockAllocator(int(g["blocks"][0]), int(g["block_size"][0]))
    reqs = {}
    for ln in golden_lines("allocator_trace.txt"):
        if ln[0] == "admit":
            _, name, n, _, table, _, free = ln
            reqs[name] = inputs.RequestState(name, int(n), alloc)
            assert reqs[name].block_table == [int(x) for x in table.split(",")]
            assert alloc.num_free == int(free)
        elif ln[0] == "append":
            _, name, n, _, table = ln
            for _ in range(int(n)):
                reqs[name].append_token()
            assert reqs[name].block_table == [int(x) for x in table.split(",")]
        elif ln[0] == "release":
            _, name, _, _, free = ln
            reqs[name].release()
            assert alloc.num_free == int(free)
    # the two released blocks are handed out again, lowest first
    assert alloc.allocate() == 3 and alloc.allocate() == 4


def test_allocator_sharing_and_exhaustion():
    """Copy-on-write sharing: a shared block returns to the free list only when
    its last reference is dropped; an empty free list raises."""
    alloc = inputs.BlockAllocator(3, 16)
    sys_blocks = [alloc.allocate(), alloc.allocate()]
    d_table = sys_blocks + [alloc.allocate()]
    for b in sys_blocks:
        alloc.share(b)
    assert alloc.ref_counts[:2] == [2, 2] and alloc.num_free == 0
    with pytest.raises(RuntimeError, match="Out of KV cache blocks"):
        alloc.allocate()
    for b in d_table:
        alloc.free(b)
    assert alloc.num_free == 1
    for b in sys_blocks:
        alloc.free(b)
    assert alloc.num_free == 3


def test_block_bytes_context():
    """"The block abstraction": 16 tokens x 32 heads x 128 dims of fp16, K and V,
    is 262,144 bytes per block per layer -- the decode-gather pool's page is one
    such K (or V) half."""
    g = golden_kv("block_bytes.txt")
    w = inputs.decode_gather(num_pages=64, num_seqs=2, len_lo=16, len_hi=64)
    assert (w.page_size, w.num_heads, w.head_dim) == tuple(
        int(g[k][0]) for k in ("block_size", "num_heads", "head_dim"))
    assert 2 * w.page_size * w.row_bytes == int(g["bytes_per_block_per_layer"][0])
    assert 2 * w.page_size * w.row_bytes * int(g["layers"][0]) == \
        int(g["bytes_per_block_all_layers"][0])


def _check_structure(w, lens=None):
    lens = w.lens if lens is None else lens
    sp = w.seq_ptr.astype(np.int64)
    assert sp[0] == 0 and np.all(np.diff(sp) >= 0) and sp[-1] == len(w.table)
    assert np.all(w.table.astype(np.int64) < w.num_pages)
    need = -(-lens.astype(np.int64) // w.page_size)
    assert np.all(need <= np.diff(sp))
    assert w.table.dtype == w.index_dtype and w.seq_ptr.dtype == w.index_dtype
    assert w.lens.dtype == w.index_dtype


@pytest.mark.parametrize("name", inputs.CONFIG_NAMES)
def test_full_size_recipes(name):
    w = inputs.config(name, "full")
    _check_structure(w)
    if name == "tiny_prefix_gather":
        assert w.total_tokens == 28 and list(w.seq_ptr) == [0, 4, 8]
    elif name == "decode_gather":
        assert (w.num_pages, w.page_size, w.num_heads, w.head_dim, w.dtype) == \
            (10000, 16, 32, 128, "f16")
        assert w.num_seqs == 64 and w.lens.min() >= 512 and w.lens.max() <= 4096
        assert len(set(w.table.tolist())) == len(w.table)  # drawn without replacement
    elif name == "decode_append":
        assert (w.page_size, w.num_heads, w.head_dim, w.dtype) == (16, 8, 128, "bf16")
        assert w.num_seqs == 256
        before = w.lens_before.astype(np.int64)
        assert before.min() >= 1024 and before.max() <= 32768
        assert np.array_equal(w.lens.astype(np.int64), before + 1)
        # a sequence whose new token starts a page has exactly one more page
        slices = np.diff(w.seq_ptr.astype(np.int64))
        assert np.array_equal(slices, -(-(before + 1) // 16))
        assert len(set(w.table.tolist())) == len(w.table)
        _check_structure(w, w.lens_before)
    elif name == "prefix_sharing":
        sp = w.seq_ptr.astype(np.int64)
        first = w.table[sp[0]:sp[0] + 128]
        for s in range(w.num_seqs):
            assert np.array_equal(w.table[sp[s]:sp[s] + 128], first)
        suffix = w.lens.astype(np.int64) - 2048
        assert suffix.min() >= 64 and suffix.max() <= 1024
        own = np.concatenate([w.table[sp[s] + 128:sp[s + 1]] for s in range(w.num_seqs)])
        assert len(set(own.tolist())) == len(own) and not set(own.tolist()) & set(first.tolist())
    elif name == "quantized_pool":
        assert (w.num_pages, w.page_size, w.dtype, w.index_dtype) == (400000, 32, "i8", np.uint64)
        assert w.num_seqs == 1024 and w.lens.min() >= 256 and w.lens.max() <= 8192


def test_host_pool_sentinel_and_determinism():
    w = inputs.config("decode_gather", "small")
    a, b = inputs.host_pool(w), inputs.host_pool(w)
    assert np.array_equal(a, b)
    live = w.live_slots()
    for p in range(w.num_pages):
        assert (a[p, live[p]:] == inputs.SENTINEL).all()
    # live slots hold data (an all-sentinel row of N(0,1) draws is vanishingly unlikely)
    rows = a[live > 0, 0]
    assert not (rows == inputs.SENTINEL).all(axis=1).any()


def test_lane_recipes():
    w = inputs.lane_worked_example()
    assert (w.capacity, w.page_tokens, list(w.table), w.batch, w.kv_heads, w.width, w.n) == \
        (12, 3, [2, 0, 3, 1], 1, 2, 2, 7)
    s = inputs.lane_synthetic()
    assert sorted(s.table.tolist()) == list(range(s.pages))
    assert 0 < s.n <= s.capacity


def test_whole_output_comparison_catches_one_wrong_byte(oracle):
    """The group-by-group comparison the full-size GPU tests use: on a small batch, rows
    built by numpy's own indexing pass, and the same rows with one byte changed (in any
    group) fail, naming the first bad row."""
    from helpers import compare_whole_gather, sequence_groups
    w = inputs.config("decode_gather", "small")
    pool = inputs.host_pool(w)
    P = w.page_size
    rows = []
    for s in range(w.num_seqs):
        lo = int(w.seq_ptr[s])
        for t in range(int(w.lens[s])):
            rows.append(pool[int(w.table[lo + t // P]), t % P])
    want = np.stack(rows)
    groups = sequence_groups(w.lens, 300)
    assert len(groups) > 2 and groups[-1][3] == len(want)
    assert compare_whole_gather(oracle, w, pool, w.lens, lambda a, b: want[a:b],
                                group_tokens=300) == len(want)
    for bad_row in (0, len(want) // 2, len(want) - 1):
        wrong = want.copy()
        wrong[bad_row, 5] ^= 1
        with pytest.raises(AssertionError, match="first at row %d" % bad_row):
            compare_whole_gather(oracle, w, pool, w.lens, lambda a, b: wrong[a:b],
                                 group_tokens=300)


@pytest.mark.parametrize("name", ["prefix_sharing", "decode_gather"])
def test_bench_physical_rows_brute_force(name):
    """The pool row of every output token that the bench's generic-gather comparison reads
    (bench.physical_rows) equals the Element Lookup taken token by token: page
    block_table[seq_ptr[s] + t / P], slot t % P, for the small version of each batch."""
    import bench
    w = inputs.config(name, "small")
    got = bench.physical_rows(w)
    want = []
    for s in range(w.num_seqs):
        for t in range(int(w.lens[s])):
            page = int(w.table[int(w.seq_ptr[s]) + t // w.page_size])
            want.append(page * w.page_size + t % w.page_size)
    assert got.tolist() == want
