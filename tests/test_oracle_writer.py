"""Writer side: trailing-slot zeroing ([HF] Partial trailing page) and the copy-on-write
page copy ([VA] Copy-on-write for beam search and prefix sharing), oracle and allocator."""
import numpy as np
import pytest

from conftest import golden_kv
from paged_kv_cache_hp_gb300 import inputs


def ints(xs):
    return [int(x) for x in xs]


def test_zero_tails_block_example(oracle):
    """[HF] Example: page 1's slots 2-3 (tokens 6-7 of sequence 0) are zeroed; page 0's
    slot 3 is undefined for sequence 1 but holds token 3 of sequence 0, so it stays;
    pages no slice names stay."""
    g = golden_kv("block_example.txt")
    P, N, H, D = (int(g[k][0]) for k in ("page_size", "num_pages", "num_heads", "head_dim"))
    pool = (np.arange(N * P * H * D) + 1).astype(np.float16)
    before = pool.copy().reshape(N, P, H, D)
    d = oracle.Desc(pool, ints(g["block_table"]), ints(g["seq_ptr"]), ints(g["lens"]),
                    num_pages=N, page_size=P, num_heads=H, head_dim=D, dtype="f16", index_type=0)
    live = d.zero_tails()
    after = pool.reshape(N, P, H, D)
    assert list(live[:2]) == [4, 2]
    zeroed = ints(g["undefined_page1_slots"])
    for slot in range(P):
        if slot in zeroed:
            assert (after[1, slot] == 0).all()
        else:
            assert np.array_equal(after[1, slot], before[1, slot])
    assert int(g["seq1_undefined_page0_slot"][0]) == 3
    assert np.array_equal(after[0], before[0])
    assert np.array_equal(after[2:], before[2:])


def test_zero_tails_prefix_sharing_config(oracle):
    w = inputs.tiny_prefix_gather()   # slices [12,5,7,9] (15 tokens) and [12,5,7,3] (13)
    pool = inputs.host_pool(w)
    before = pool.copy()
    d = oracle.Desc(pool, w.table, w.seq_ptr, w.lens, num_pages=16, page_size=4, num_heads=2,
                    head_dim=4, dtype="f32")
    d.zero_tails()
    for page in (12, 5, 7):
        assert np.array_equal(pool[page], before[page])
    assert np.array_equal(pool[9, :3], before[9, :3]) and (pool[9, 3:] == 0).all()
    assert np.array_equal(pool[3, :1], before[3, :1]) and (pool[3, 1:] == 0).all()
    untouched = [p for p in range(16) if p not in (12, 5, 7, 9, 3)]
    assert np.array_equal(pool[untouched], before[untouched])


@pytest.mark.parametrize("seed", range(25))
def test_zero_tails_keeps_every_readable_row(oracle, seed):
    """Random batches with aliasing: the gather is unchanged, zeroing again changes
    nothing, and every zeroed slot is one no sequence reads."""
    rng = np.random.default_rng(seed)
    N, P, H, D = 9, int(rng.integers(1, 5)), 2, 3
    S = int(rng.integers(1, 5))
    lens, table, sp = [], [], [0]
    for _ in range(S):
        n = int(rng.integers(0, 3 * P + 1))
        k = -(-n // P) + int(rng.integers(0, 2))
        table += [int(x) for x in rng.integers(0, N, k)]
        sp.append(len(table))
        lens.append(n)
    pool = rng.integers(1, 256, (N, P, H, D, 4), dtype=np.uint8)
    d = oracle.Desc(pool, table if table else None, sp, lens, num_pages=N, page_size=P,
                    num_heads=H, head_dim=D, dtype="f32", index_type=1)
    assert d.validate() == ("OK", 0)
    g0 = d.gather()[0]
    before = pool.copy()
    d.zero_tails()
    assert np.array_equal(d.gather()[0], g0)
    once = pool.copy()
    d.zero_tails()
    assert np.array_equal(pool, once)
    readable = np.zeros((N, P), bool)
    for s in range(S):
        for t in range(lens[s]):
            readable[table[sp[s] + t // P], t % P] = True
    changed = (pool != before).any(axis=(2, 3, 4))
    assert not (changed & readable).any()
    referenced = np.zeros(N, bool)
    referenced[table] = True
    # every slot that was not readable in a referenced page is zero now
    assert (pool[referenced][~readable[referenced]] == 0).all()


def test_copy_pages_and_cow(oracle):
    """[VA]: requests D and E share two system-prompt blocks; D is about to write into
    the second one, so it gets a private copy and E's view does not change."""
    alloc = inputs.BlockAllocator(8, 4)
    sys_blocks = [alloc.allocate(), alloc.allocate()]
    d_table = sys_blocks + [alloc.allocate()]
    for b in sys_blocks:
        alloc.share(b)
    e_table = sys_blocks + [alloc.allocate()]
    assert alloc.ref_counts[sys_blocks[1]] == 2
    fresh = alloc.cow(sys_blocks[1])
    assert fresh not in d_table + e_table and alloc.ref_counts[sys_blocks[1]] == 1
    assert alloc.cow(d_table[2]) == d_table[2]           # not shared: written in place
    rng = np.random.default_rng(0)
    pool = rng.integers(0, 256, (8, 4, 2, 2, 2), dtype=np.uint8)
    before = pool.copy()
    desc = oracle.Desc(pool, d_table + e_table, [0, 3, 6], [12, 12], num_pages=8, page_size=4,
                       num_heads=2, head_dim=2, dtype="f16", index_type=0)
    assert desc.copy_pages([sys_blocks[1]], [fresh]) == "OK"
    assert np.array_equal(pool[fresh], before[sys_blocks[1]])
    others = [p for p in range(8) if p != fresh]
    assert np.array_equal(pool[others], before[others])
    # out-of-range pairs are skipped and reported
    assert desc.copy_pages([0, 9], [5, 6]) == "PAGE_ID"
    assert np.array_equal(pool[5], before[0]) and np.array_equal(pool[6], before[6])


@pytest.mark.parametrize("seed", range(10))
def test_copy_pages_random(oracle, seed):
    rng = np.random.default_rng(seed)
    N = 12
    pool = rng.integers(0, 256, (N, 3, 5), dtype=np.uint8)
    perm = rng.permutation(N)
    k = int(rng.integers(0, N // 2 + 1))
    src, dst = perm[:k], perm[k:2 * k]
    want = pool.copy()
    want[dst] = pool[src]
    d = oracle.Desc(pool, None, [0], np.zeros(0, np.uint64), num_pages=N, page_size=3,
                    num_heads=1, head_dim=5, dtype="u8", index_type=1)
    assert d.copy_pages(src, dst) == "OK"
    assert np.array_equal(pool, want)
