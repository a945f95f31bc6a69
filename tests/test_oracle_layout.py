"""Pins the oracle's layout conversion ([HF] Framework Compliance: the kernel-internal
[num_blocks, num_kv_heads, head_dim/x, block_size, x] key-cache layout versus the
interchange [num_blocks, block_size, num_kv_heads, head_dim]) to numpy's transpose."""
import numpy as np
import pytest


@pytest.mark.parametrize("nb,bs,H,D,x,dt", [(3, 4, 2, 8, 8, np.float16), (2, 16, 3, 16, 8, np.uint16),
                                            (4, 5, 1, 6, 3, np.int8), (2, 3, 2, 4, 1, np.float32),
                                            (1, 16, 8, 128, 8, np.float16), (2, 2, 2, 2, 2, np.float64)])
def test_matches_numpy_transpose(oracle, nb, bs, H, D, x, dt):
    rng = np.random.default_rng(nb * 1000 + bs * 10 + x)
    internal = rng.integers(0, 100, (nb, H, D // x, bs, x)).astype(dt)
    want = internal.transpose(0, 3, 1, 2, 4).reshape(nb, bs, H, D)
    got = oracle.from_kernel_layout(internal, nb, bs, H, D, x)
    assert np.array_equal(got, want)
    back = oracle.to_kernel_layout(got, nb, bs, H, D, x)
    assert np.array_equal(back, internal)


def test_x_one_is_the_value_cache_layout(oracle):
    """With x = 1 the internal layout is [num_blocks, H, D, block_size]."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((2, 3, 4, 5)).astype(np.float32)  # [nb, H, D, bs]
    got = oracle.from_kernel_layout(v.reshape(2, 3, 4, 5, 1), 2, 5, 3, 4, 1)
    assert np.array_equal(got, v.transpose(0, 3, 1, 2))


def test_padded_tables_from_the_allocator_trace(oracle):
    """[VA] "Visualizing the layout": after A grows to 50 tokens, A's table is
    [0, 1, 2, 9] and C's [5, 6, 7, 8] (50 tokens each, block size 16)."""
    from conftest import golden_lines
    tables = {}
    for ln in golden_lines("allocator_trace.txt"):
        if ln[0] in ("admit", "append") and "->" in ln:
            tables[ln[1]] = [int(x) for x in ln[ln.index("->") + 1].split(",")]
    padded = np.array([tables["A"], tables["C"]], dtype=np.uint32)
    name, first, table, sp = oracle.padded_to_csr(padded, [50, 50], 16)
    assert name == "OK" and list(table) == [0, 1, 2, 9, 5, 6, 7, 8] and list(sp) == [0, 4, 8]
    # fewer valid tokens use fewer leading entries
    name, first, table, sp = oracle.padded_to_csr(padded, [33, 1], 16)
    assert list(table) == [0, 1, 2, 5] and list(sp) == [0, 3, 4]
    name, first, back = oracle.csr_to_padded(np.array([0, 1, 2, 9, 5, 6, 7, 8], np.uint32),
                                             np.array([0, 4, 8], np.uint32), 4, 99)
    assert name == "OK" and np.array_equal(back, padded)


def test_block_example_round_trip(oracle):
    """[HF] Example: seq_ptr [0,2,3], table [0,1,0] (6 and 3 tokens, page_size 4)."""
    name, first, padded = oracle.csr_to_padded(np.array([0, 1, 0], np.uint64),
                                               np.array([0, 2, 3], np.uint64), 2, 7)
    assert name == "OK" and padded.tolist() == [[0, 1], [0, 7]]
    name, first, table, sp = oracle.padded_to_csr(padded, np.array([6, 3], np.uint64), 4)
    assert name == "OK" and list(table) == [0, 1, 0] and list(sp) == [0, 2, 3]


def test_padded_csr_errors(oracle):
    name, first, _, _ = oracle.padded_to_csr(np.zeros((3, 2), np.uint32), [8, 9, 1], 4)
    assert (name, first) == ("LEN", 1)                     # 9 tokens need 3 pages of 4
    name, first, _, _ = oracle.padded_to_csr(np.zeros((2, 2), np.uint32), [8, 8], 4, table_cap=3)
    assert name == "OUT_SIZE"
    name, first, _ = oracle.csr_to_padded(np.zeros(5, np.uint32), np.array([0, 2, 5], np.uint32),
                                          2, 0)
    assert (name, first) == ("LEN", 1)


@pytest.mark.parametrize("seed", range(10))
def test_padded_csr_random_round_trip(oracle, seed):
    rng = np.random.default_rng(seed)
    B, MB, P = int(rng.integers(1, 9)), int(rng.integers(1, 7)), int(rng.integers(1, 5))
    padded = rng.integers(0, 1000, (B, MB)).astype(np.uint64)
    lens = rng.integers(0, MB * P + 1, B).astype(np.uint64)
    name, first, table, sp = oracle.padded_to_csr(padded, lens, P)
    assert name == "OK"
    for s in range(B):
        need = -(-int(lens[s]) // P)
        assert list(table[sp[s]:sp[s + 1]]) == list(padded[s, :need])
    name, first, back = oracle.csr_to_padded(table, sp, MB, 12345)
    for s in range(B):
        need = -(-int(lens[s]) // P)
        assert list(back[s, :need]) == list(padded[s, :need])
        assert (back[s, need:] == 12345).all()
