"""Brute force on tiny random inputs: the oracle against numpy's own N-d indexing.

The expected values come from indexing a numpy array of shape
[num_pages, page_size, num_heads, head_dim] (or [N, B, H_kv, P, d] for the
per-lane layout) with (page, slot, head, dim) tuples -- numpy's row-major
definition -- so a transposed axis, a dropped term or a wrong stride in the
oracle's flat-index arithmetic shows up here.
"""
import itertools

import numpy as np
import pytest

ES = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1, "f64": 8}


def random_batch(rng, alias=True):
    S = int(rng.integers(0, 5))
    P = int(rng.integers(1, 6))
    H = int(rng.integers(1, 4))
    D = int(rng.integers(1, 4))
    N = int(rng.integers(1, 13))
    lens, tables = [], []
    free = list(rng.permutation(N))
    for _ in range(S):
        n = int(rng.integers(0, 3 * P + 1))
        need = -(-n // P)
        extra = int(rng.integers(0, 2))  # slices may reserve an unused page
        k = need + extra
        if alias:
            tables.append([int(x) for x in rng.integers(0, N, k)])
        else:
            if len(free) < k:
                n, k = 0, 0
            tables.append([int(free.pop()) for _ in range(k)])
        lens.append(n)
    seq_ptr = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int64)
    table = [x for t in tables for x in t]
    return S, P, H, D, N, lens, table, seq_ptr


@pytest.mark.parametrize("seed", range(60))
def test_gather_matches_ndarray_indexing(oracle, seed):
    rng = np.random.default_rng(seed)
    S, P, H, D, N, lens, table, seq_ptr = random_batch(rng)
    dtype = ["f32", "f16", "bf16", "i8", "f64"][seed % 5]
    es = ES[dtype]
    pool = rng.integers(0, 256, (N, P, H, D, es), dtype=np.uint8)
    it = seed % 2
    desc = oracle.Desc(pool, table if table else None, seq_ptr, lens, num_pages=N, page_size=P,
                       num_heads=H, head_dim=D, dtype=dtype, index_type=it)
    assert desc.validate() == ("OK", 0)
    out, written, fault = desc.gather()
    assert fault == "OK" and written.all()
    out = out.reshape(-1, H, D, es)
    row = 0
    for s in range(S):
        for t in range(lens[s]):
            page = table[seq_ptr[s] + t // P]
            for h, d in itertools.product(range(H), range(D)):
                assert np.array_equal(out[row, h, d], pool[page, t % P, h, d])
            row += 1
    assert row == out.shape[0]


@pytest.mark.parametrize("seed", range(40))
def test_append_matches_ndarray_indexing(oracle, seed):
    rng = np.random.default_rng(100 + seed)
    S, P, H, D, N, full, table, seq_ptr = random_batch(rng, alias=False)
    # split each sequence's count into "before" and "new"
    before = [int(rng.integers(0, n + 1)) for n in full]
    new_n = [f - b for f, b in zip(full, before)]
    new_ptr = np.concatenate([[0], np.cumsum(new_n)]).astype(np.int64)
    pool = rng.integers(0, 256, (N, P, H, D, 2), dtype=np.uint8)
    ref = pool.copy()
    new = rng.integers(0, 256, (int(new_ptr[-1]), H, D, 2), dtype=np.uint8)
    desc = oracle.Desc(pool, table if table else None, seq_ptr, before, num_pages=N, page_size=P,
                       num_heads=H, head_dim=D, dtype="f16", index_type=1)
    assert desc.validate_append(new_ptr, int(new_ptr[-1])) == ("OK", 0)
    assert desc.scatter_append(new, new_ptr) == "OK"
    for s in range(S):
        for i in range(new_n[s]):
            t = before[s] + i
            ref[table[seq_ptr[s] + t // P], t % P] = new[new_ptr[s] + i]
    assert np.array_equal(pool, ref)


@pytest.mark.parametrize("seed", range(20))
def test_permissive_append_reads_no_row_past_total_new(oracle, seed):
    """A permissive append whose new_ptr runs backwards or past total_new: those
    sequences contribute no rows (the first such pair's code is returned), the others
    land as numpy indexing puts them, and no input row at or past total_new is read (the
    input buffer is cut to exactly total_new rows, so a read past it would take bytes
    from a guard that the reference never writes)."""
    rng = np.random.default_rng(300 + seed)
    S, P, H, D, N, full, table, seq_ptr = random_batch(rng, alias=False)
    if S < 2:
        return
    before = [int(rng.integers(0, n + 1)) for n in full]
    new_n = [f - b for f, b in zip(full, before)]
    new_ptr = np.concatenate([[0], np.cumsum(new_n)]).astype(np.int64)
    total_new = int(new_ptr[-1])
    starts = [s for s in range(S) if new_ptr[s] > 0]
    if seed % 2 == 0 or not starts:  # the last pair ends past total_new
        new_ptr[S] = total_new + 1 + int(rng.integers(0, 3))
    else:  # one pair runs backwards
        bad = starts[int(rng.integers(0, len(starts)))]
        new_ptr[bad + 1] = new_ptr[bad] - 1
    pool = rng.integers(0, 256, (N, P, H, D, 2), dtype=np.uint8)
    ref = pool.copy()
    guard = np.full((total_new + 8, H, D, 2), 0xEE, dtype=np.uint8)
    guard[:total_new] = rng.integers(0, 256, (total_new, H, D, 2), dtype=np.uint8)
    new = guard[:total_new]
    desc = oracle.Desc(pool, table if table else None, seq_ptr, before, num_pages=N, page_size=P,
                       num_heads=H, head_dim=D, dtype="f16", index_type=1, flags=1)
    code = desc.scatter_append(new, new_ptr, total_new)
    skipped = set()
    first = "OK"
    for s in range(S):
        a, b = int(new_ptr[s]), int(new_ptr[s + 1])
        if b < a or b > total_new:
            skipped.add(s)
            if first == "OK":
                first = "NEW_PTR_ORDER" if b < a else "NEW_PTR_END"
            continue
        for i in range(b - a):
            t = before[s] + i
            if t // P >= seq_ptr[s + 1] - seq_ptr[s]:
                if first == "OK":
                    first = "LEN"
                continue
            ref[table[seq_ptr[s] + t // P], t % P] = new[a + i]
    assert code == first and skipped
    assert np.array_equal(pool, ref)


@pytest.mark.parametrize("seed", range(20))
def test_dequant_gather_matches_ndarray_indexing(oracle, seed):
    import torch
    rng = np.random.default_rng(200 + seed)
    S, P, H, D, N, lens, table, seq_ptr = random_batch(rng)
    pool = rng.integers(-127, 127, (N, P, H, D), endpoint=True).astype(np.int8)
    scales = rng.uniform(0.001, 0.05, (N, P)).astype(np.float32)
    desc = oracle.Desc(pool, table if table else None, seq_ptr, lens, num_pages=N, page_size=P,
                       num_heads=H, head_dim=D, dtype="i8", scales=scales.reshape(-1), flags=2,
                       index_type=1)
    assert desc.validate() == ("OK", 0)
    out, written, fault = desc.gather_dequant()
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = got.reshape(-1, H, D)
    row = 0
    for s in range(S):
        for t in range(lens[s]):
            page = table[seq_ptr[s] + t // P]
            exact = pool[page, t % P].astype(np.float64) * float(scales[page, t % P])
            # within half a bfloat16 ulp of the exact product (one rounding)
            ulp = 2.0 ** (np.floor(np.log2(np.abs(exact), where=exact != 0,
                                           out=np.zeros_like(exact))) - 7)
            assert np.all(np.abs(got[row] - exact) <= ulp / 2)
            row += 1


@pytest.mark.parametrize("seed", range(40))
def test_lane_gather_append_match_ndarray_indexing(oracle, seed):
    rng = np.random.default_rng(300 + seed)
    P = int(rng.integers(1, 5))
    C = int(rng.integers(1, 14))
    N = -(-C // P)
    T = rng.permutation(N).astype(np.uint64)
    B, H, W = (int(x) for x in rng.integers(1, 4, 3))
    n = int(rng.integers(0, C + 1))
    pool = rng.standard_normal((N, B, H, P, W))
    out = oracle.lane_gather(pool, C, P, T, B, H, W, n)
    for b, h, p, f in itertools.product(range(B), range(H), range(n), range(W)):
        assert out[b, h, p, f] == pool[T[p // P], b, h, p % P, f]
    m = int(rng.integers(0, C - n + 1))
    new = rng.standard_normal((B, H, m, W))
    ref = pool.copy()
    assert oracle.lane_append(pool, C, P, T, B, H, W, n, new) == "OK"
    for b, h, i in itertools.product(range(B), range(H), range(m)):
        p = n + i
        ref[T[p // P], b, h, p % P] = new[b, h, i]
    assert np.array_equal(pool, ref)
    if C - n + 1 <= C:
        too_many = rng.standard_normal((B, H, C - n + 1, W))
        assert oracle.lane_append(pool, C, P, T, B, H, W, n, too_many) == "LENGTH"


def _all_lookups_ok(desc, lens):
    for s, n in enumerate(lens):
        for t in range(n):
            if desc.lookup(s, t, 0, 0)[0] != "OK":
                return False
    return True


def test_validator_enumeration(oracle):
    """Every seq_ptr of length 1..4 over {0..3}, with tables and counts drawn at
    random: whenever the strict verdict is OK every token's lookup stays inside
    its slice, the table and the pool; a failed verdict names a rule whose
    condition really fails at the reported index; permissive mode accepts all."""
    rng = np.random.default_rng(5)
    P, H, D = 2, 1, 1
    seen = set()
    for L in range(1, 5):
        for seq_ptr in itertools.product(range(4), repeat=L):
            S = L - 1
            for k in range(4):
                tlen = int(seq_ptr[-1]) if k % 2 else int(rng.integers(0, 4))
                N = int(rng.integers(1, 4))
                table = [int(x) for x in rng.integers(0, N + 1, tlen)]
                lens = [int(x) for x in rng.integers(0, 5, S)]
                pool = np.zeros((N, P, H, D, 2), np.uint8)
                mk = lambda flags: oracle.Desc(pool, table if tlen else None, list(seq_ptr), lens,
                                               num_pages=N, page_size=P, num_heads=H, head_dim=D,
                                               dtype="f16", index_type=0, table_len=tlen,
                                               flags=flags)
                code, i = mk(0).validate()
                seen.add(code)
                assert mk(1).validate() == ("OK", 0)
                if code == "OK":
                    assert _all_lookups_ok(mk(0), lens)
                elif code == "SEQ_PTR_START":
                    assert seq_ptr[0] != 0
                elif code == "SEQ_PTR_ORDER":
                    assert seq_ptr[i] > seq_ptr[i + 1] and seq_ptr[0] == 0
                elif code == "SEQ_PTR_END":
                    assert seq_ptr[S] != tlen and list(seq_ptr) == sorted(seq_ptr)
                elif code == "PAGE_ID":
                    assert table[i] >= N and all(x < N for x in table[:i])
                elif code == "LEN":
                    assert lens[i] > (seq_ptr[i + 1] - seq_ptr[i]) * P
                    assert all(x < N for x in table)
                else:
                    raise AssertionError(code)
    assert seen == {"OK", "SEQ_PTR_START", "SEQ_PTR_ORDER", "SEQ_PTR_END", "PAGE_ID", "LEN"}


def test_permissive_gather_skips_unreadable_rows(oracle):
    """In permissive mode a lookup that leaves its slice, the table or the pool
    reads nothing: its output row keeps its previous bytes."""
    P, H, D, N = 2, 1, 2, 3
    pool = np.arange(N * P * H * D, dtype=np.float32)
    # seq 0: 3 tokens but a 1-page slice; seq 1: page id 7 out of range
    desc = oracle.Desc(pool, [1, 7], [0, 1, 2], [3, 2], num_pages=N, page_size=P, num_heads=H,
                       head_dim=D, dtype="f32", index_type=0, flags=1)
    assert desc.validate() == ("OK", 0)
    out = np.full((5, H * D * 4), 0xEE, np.uint8)
    out, written, fault = desc.gather(out)
    assert list(written) == [True, True, False, False, False]
    assert fault == "LEN"
    assert (out[2:] == 0xEE).all()
    assert np.array_equal(out[0].view(np.float32), pool.reshape(N, P, D)[1, 0])
