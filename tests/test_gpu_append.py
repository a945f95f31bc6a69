"""GPU parity: hp_scatter_append against the CPU oracle -- the whole pool after the
append, byte for byte."""
import numpy as np
import pytest

from helpers import Batch, index_tensor, lib_name, sub_batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def append_case(hp, oracle, w, lens_before, new_ptr, new_rows_host, it=None):
    """Runs the device append and the oracle append on copies of the same pool;
    returns (device pool bytes, oracle pool bytes, status name)."""
    import torch
    b = Batch(w, lens=lens_before)
    host = b.host_pool().copy()
    new_dev = torch.from_numpy(np.ascontiguousarray(new_rows_host)).to("cuda")
    np_dev = index_tensor(np.asarray(new_ptr, dtype=w.index_dtype), "cuda")
    total = int(new_ptr[-1])
    rc = hp.hp_scatter_append(b.desc, new_dev, np_dev, total, b.ws, b.status)
    torch.cuda.synchronize()
    assert hp.status_name(rc) == "HP_OK"
    o = b.oracle_desc(pool_host=host, lens=np.asarray(lens_before, dtype=w.index_dtype))
    assert o.validate_append(new_ptr, total) == ("OK", 0)
    assert o.scatter_append(new_rows_host, new_ptr) == "OK"
    return b.pool.cpu().numpy(), host, hp.status_name(b.status_value()), b


def test_decode_step_append_small(hp, oracle):
    w = inputs.config("decode_append", "small")
    got, want, st, _ = append_case(hp, oracle, w, w.lens_before, w.new_ptr, inputs.host_new_rows(w))
    assert st == "HP_OK"
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seed", range(6))
def test_multi_row_append_crossing_pages(hp, oracle, seed):
    """Several rows per sequence, starting anywhere in a page and crossing page
    boundaries; some sequences append nothing."""
    rng = np.random.default_rng(seed)
    P = [1, 3, 16, 5, 16, 7][seed]
    w = inputs.decode_gather(seed=50 + seed, num_pages=900, page_size=P, num_heads=2,
                             head_dim=[8, 16, 4, 3, 64, 5][seed], num_seqs=7, len_lo=0,
                             len_hi=90, dtype=["bf16", "f32", "i8", "f16", "f16", "f64"][seed],
                             index_dtype=np.uint64 if seed % 2 else np.uint32)
    full = w.lens.astype(np.int64)
    before = np.array([rng.integers(0, n + 1) for n in full])
    new_n = full - before
    new_n[rng.integers(0, len(new_n))] = 0
    before = full - new_n
    new_ptr = np.concatenate([[0], np.cumsum(new_n)]).astype(w.index_dtype)
    rows = np.random.default_rng(seed + 7).integers(0, 256, (int(new_ptr[-1]), w.row_bytes),
                                                    dtype=np.uint8)
    got, want, st, b = append_case(hp, oracle, w, before.astype(w.index_dtype), new_ptr, rows)
    assert st == "HP_OK"
    assert np.array_equal(got, want)


def test_bulk_append_then_gather_round_trip(hp, oracle):
    """Prefill-style: every row of the batch appended into empty slices, then gathered
    back -- the gather returns the appended rows."""
    import torch
    w = inputs.config("prefix_sharing", "small")
    # give every sequence private pages (appending into shared pages is undefined)
    w = inputs.decode_gather(seed=77, num_pages=700, num_heads=8, head_dim=128, num_seqs=6,
                             len_lo=1, len_hi=300, dtype="bf16")
    T = w.total_tokens
    rows = np.random.default_rng(1).integers(0, 256, (T, w.row_bytes), dtype=np.uint8)
    new_ptr = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))]).astype(np.uint32)
    zeros = np.zeros(w.num_seqs, dtype=np.uint32)
    got, want, st, b = append_case(hp, oracle, w, zeros, new_ptr, rows)
    assert st == "HP_OK" and np.array_equal(got, want)
    g = Batch(w, pool=b.pool)
    out = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(g.desc, out, T, g.ws, g.status) == 0
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().reshape(T, -1), rows)


def test_full_size_decode_step_then_gather(hp, oracle):
    """The decode step at full size (256 sequences, one new row each, a new page
    where the row starts one), then the gather of the grown batch; sampled checks."""
    import torch
    w = inputs.config("decode_append", "full")
    b = Batch(w, lens=w.lens_before)
    new = inputs.device_new_rows(w, "cuda")
    np_dev = index_tensor(w.new_ptr, "cuda")
    rc = hp.hp_scatter_append(b.desc, new, np_dev, w.total_new, b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0 and b.status_value() == 0
    # every new row sits where the oracle's Element Lookup puts token len_before[s]
    o = b.oracle_desc(pool_host=b.pool.cpu().numpy(), lens=w.lens)
    new_h = new.cpu().numpy()
    es = 2
    rng = np.random.default_rng(3)
    for s in range(w.num_seqs):
        t = int(w.lens_before[s])
        for h, d in zip(rng.integers(0, 8, 6), rng.integers(0, 128, 6)):
            code, v = o.lookup(s, t, int(h), int(d))
            assert code == "OK"
            k = (int(h) * 128 + int(d)) * es
            assert np.array_equal(v, new_h[s, k:k + es])
    # the grown batch gathers consistently with the oracle
    g = Batch(w, pool=b.pool)
    T = w.total_tokens
    out = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(g.desc, out, T, g.ws, g.status) == 0
    torch.cuda.synchronize()
    assert g.status_value() == 0
    got = out.cpu().numpy().reshape(T, -1)
    tok_off = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))])
    last_rows = tok_off[1:] - 1
    assert np.array_equal(got[last_rows], new_h)
    seqs = [0, 100, 255]
    table, seq_ptr, lens = sub_batch(w, seqs)
    sub = oracle.Desc(o.pool, table, seq_ptr, lens, num_pages=w.num_pages, page_size=16,
                      num_heads=8, head_dim=128, dtype="bf16", index_type=0)
    want = sub.gather()[0]
    rows = np.concatenate([np.arange(tok_off[s], tok_off[s + 1]) for s in seqs])
    assert np.array_equal(got[rows], want)


@pytest.mark.parametrize("case,want", [
    ({}, ("OK", 0)),
    ({"new_ptr": [1, 1, 2]}, ("NEW_PTR_START", 0)),
    ({"new_ptr": [0, 2, 1]}, ("NEW_PTR_ORDER", 1)),
    ({"total_new": 3}, ("NEW_PTR_END", 2)),
    ({"lens": [8, 2]}, ("CAPACITY", 0)),
    ({"lens": [7, 3]}, ("OK", 0)),
    ({"lens": [5, 4]}, ("CAPACITY", 1)),
    ({"table": [0, 9, 2]}, ("PAGE_ID", 1)),
    ({"seq_ptr": [0, 3, 2]}, ("SEQ_PTR_ORDER", 1)),
])
@pytest.mark.parametrize("it", [0, 1])
def test_append_verdicts(hp, oracle, case, want, it):
    import torch
    dt = np.uint32 if it == 0 else np.uint64
    table = case.get("table", [0, 1, 2])
    seq_ptr = case.get("seq_ptr", [0, 2, 3])
    lens = case.get("lens", [5, 2])
    new_ptr = case.get("new_ptr", [0, 1, 2])
    total = case.get("total_new", 2)
    pool = torch.full((4 * 4 * 8,), 0x33, dtype=torch.uint8, device="cuda")
    d = hp.PagedDesc(pool, index_tensor(np.asarray(table, dt), "cuda"),
                     index_tensor(np.asarray(seq_ptr, dt), "cuda"),
                     index_tensor(np.asarray(lens, dt), "cuda"), num_pages=4, page_size=4,
                     num_heads=2, head_dim=2, dtype="f16", index_type=it)
    ws = hp.workspace_for(d)
    npd = index_tensor(np.asarray(new_ptr, dt), "cuda")
    rc, first = hp.hp_validate_append(d, npd, total, ws)
    o = oracle.Desc(pool.cpu().numpy(), table, seq_ptr, lens, num_pages=4, page_size=4,
                    num_heads=2, head_dim=2, dtype="f16", index_type=it)
    assert o.validate_append(new_ptr, total) == want
    assert (hp.status_name(rc), first) == (lib_name(want[0]), want[1])
    if want[0] != "OK":
        st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        rows = torch.full((max(total, 3) * 8,), 0x44, dtype=torch.uint8, device="cuda")
        assert hp.hp_scatter_append(d, rows, npd, total, ws, st) == 0
        torch.cuda.synchronize()
        assert hp.status_name(st.item()) == lib_name(want[0])
        assert (pool.cpu().numpy() == 0x33).all()  # nothing written


def test_permissive_append_skips_unwritable_rows(hp, oracle):
    import torch
    w = inputs.decode_gather(seed=31, num_pages=200, num_heads=2, head_dim=8, num_seqs=5,
                             len_lo=1, len_hi=60)
    full = w.lens.astype(np.int64)
    before = full // 2
    new_n = full - before
    new_n[1] += 3 * w.page_size  # runs past its slice
    new_ptr = np.concatenate([[0], np.cumsum(new_n)]).astype(np.uint32)
    rows = np.random.default_rng(5).integers(0, 256, (int(new_ptr[-1]), w.row_bytes),
                                             dtype=np.uint8)
    b = Batch(w, flags=1, lens=before.astype(np.uint32))
    host = b.host_pool().copy()
    rc = hp.hp_scatter_append(b.desc, torch.from_numpy(rows).to("cuda"),
                              index_tensor(new_ptr, "cuda"), int(new_ptr[-1]), b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0
    o = b.oracle_desc(pool_host=host, lens=before.astype(np.uint32))
    assert o.scatter_append(rows, new_ptr) == "LEN"
    assert np.array_equal(b.pool.cpu().numpy(), host)
    assert hp.status_name(b.status_value()) == "HP_ERR_LEN"


def test_planned_append_steps_equal_one_call(hp, oracle):
    """hp_append_plan + hp_scatter_append_planned on one stream is hp_scatter_append."""
    import torch
    w = inputs.config("decode_append", "small")
    b1 = Batch(w, lens=w.lens_before)
    b2 = Batch(w, lens=w.lens_before, pool=b1.pool.clone())
    new = inputs.device_new_rows(w, "cuda")
    npd = index_tensor(w.new_ptr, "cuda")
    assert hp.hp_scatter_append(b1.desc, new, npd, w.total_new, b1.ws, b1.status) == 0
    assert hp.hp_append_plan(b2.desc, npd, w.total_new, b2.ws, b2.status) == 0
    assert hp.hp_scatter_append_planned(b2.desc, new, npd, w.total_new, b2.ws, b2.status) == 0
    torch.cuda.synchronize()
    assert b1.status_value() == 0 and b2.status_value() == 0
    assert torch.equal(b1.pool, b2.pool)


def _permissive_case(hp, oracle, w, before, new_ptr, rows, pool=None):
    import torch
    b = Batch(w, flags=1, lens=np.asarray(before, dtype=w.index_dtype), pool=pool)
    host = b.host_pool().copy()
    rc = hp.hp_scatter_append(b.desc, torch.from_numpy(np.ascontiguousarray(rows)).to("cuda"),
                              index_tensor(np.asarray(new_ptr, dtype=w.index_dtype), "cuda"),
                              int(new_ptr[-1]), b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0
    o = b.oracle_desc(pool_host=host, lens=np.asarray(before, dtype=w.index_dtype))
    want = o.scatter_append(rows, np.asarray(new_ptr, dtype=w.index_dtype))
    return b.pool.cpu().numpy(), host, want, hp.status_name(b.status_value())


@pytest.mark.parametrize("case", ["decode", "u64", "narrow", "wide", "few_rows"])
def test_permissive_decode_step_matches_oracle(hp, oracle, case):
    """HP_PERMISSIVE with fewer new rows than one page per sequence: the one-kernel path
    (one warp per sequence, no plan) writes exactly what the oracle writes."""
    rng = np.random.default_rng(len(case))
    geo = {"decode": (16, 8, 128, "bf16", np.uint32), "u64": (16, 4, 64, "f16", np.uint64),
           "narrow": (5, 3, 7, "f16", np.uint32), "wide": (8, 8, 256, "bf16", np.uint64),
           "few_rows": (16, 2, 64, "f32", np.uint32)}[case]
    P, H, D, dt, it = geo
    w = inputs.decode_gather(seed=90 + len(case), num_pages=3000, page_size=P, num_heads=H,
                             head_dim=D, num_seqs=40, len_lo=1, len_hi=400, dtype=dt,
                             index_dtype=it)
    full = w.lens.astype(np.int64)
    new_n = np.minimum(full, rng.integers(0, 4 if case == "few_rows" else 2, w.num_seqs))
    before = full - new_n
    new_ptr = np.concatenate([[0], np.cumsum(new_n)])
    rows = rng.integers(0, 256, (int(new_ptr[-1]), w.row_bytes), dtype=np.uint8)
    got, want_pool, code, st = _permissive_case(hp, oracle, w, before, new_ptr, rows)
    assert code == "OK" and st == "HP_OK"
    assert np.array_equal(got, want_pool)


def test_permissive_decode_step_full_size(hp, oracle):
    import torch
    w = inputs.config("decode_append", "full")
    b = Batch(w, flags=1, lens=w.lens_before)
    new = inputs.device_new_rows(w, "cuda")
    rc = hp.hp_scatter_append(b.desc, new, index_tensor(w.new_ptr, "cuda"), w.total_new, b.ws,
                              b.status)
    torch.cuda.synchronize()
    assert rc == 0 and b.status_value() == 0
    g = Batch(w, pool=b.pool)
    T = w.total_tokens
    out = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(g.desc, out, T, g.ws, g.status) == 0
    torch.cuda.synchronize()
    tok_off = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))])
    got = out.cpu().numpy().reshape(T, -1)
    assert np.array_equal(got[tok_off[1:] - 1], new.cpu().numpy())


@pytest.mark.parametrize("fault", ["LEN", "PAGE_ID"])
def test_permissive_decode_step_skips_unwritable_rows(hp, oracle, fault):
    rng = np.random.default_rng(7)
    w = inputs.decode_gather(seed=61, num_pages=800, page_size=8, num_heads=2, head_dim=16,
                             num_seqs=12, len_lo=1, len_hi=90, dtype="f16")
    full = w.lens.astype(np.int64)
    new_n = np.ones(w.num_seqs, np.int64)
    before = full - 1
    table = w.table.copy()
    if fault == "LEN":  # sequence 3 appends at a token past its slice
        span = int(w.seq_ptr[4] - w.seq_ptr[3])
        before[3] = span * w.page_size
    else:  # the page sequence 5's new row lands in is not in the pool
        k = int(w.seq_ptr[5]) + int(before[5]) // w.page_size
        table[k] = w.num_pages + 3
    w2 = inputs.Workload(**{**w.__dict__, "table": table})
    new_ptr = np.concatenate([[0], np.cumsum(new_n)])
    rows = rng.integers(0, 256, (int(new_ptr[-1]), w.row_bytes), dtype=np.uint8)
    got, want_pool, code, st = _permissive_case(hp, oracle, w2, before, new_ptr, rows,
                                                pool=inputs.device_pool(w, "cuda"))
    assert code == fault and st == "HP_ERR_" + fault
    assert np.array_equal(got, want_pool)


def test_one_append_plan_serves_the_pools_of_several_layers(hp, oracle):
    """hp_append_plan once (a decode step: one row per sequence), then the planned append
    into two pools (a layer's K and V) through descriptors that differ only in
    page_pool: each pool matches the oracle's append into it."""
    import torch
    w = inputs.config("decode_append", "small")
    b = Batch(w, lens=w.lens_before)
    np_dev = index_tensor(w.new_ptr, "cuda")
    assert hp.hp_append_plan(b.desc, np_dev, w.total_new, b.ws, b.status) == 0
    for layer in range(2):
        pl = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 950 + layer}),
                                "cuda")
        host = pl.cpu().numpy().copy()
        rows = np.random.default_rng(layer).integers(0, 256, (w.total_new, w.row_bytes),
                                                     dtype=np.uint8)
        dl = hp.PagedDesc(pl, b.table, b.seq_ptr, b.lens, num_pages=w.num_pages,
                          page_size=w.page_size, num_heads=w.num_heads, head_dim=w.head_dim,
                          dtype=w.dtype, index_type=b.it)
        new = torch.from_numpy(rows.reshape(-1).copy()).to("cuda")
        assert hp.hp_scatter_append_planned(dl, new, np_dev, w.total_new, b.ws, b.status) == 0
        torch.cuda.synchronize()
        assert b.status_value() == 0
        o = b.oracle_desc(pool_host=host, lens=w.lens_before)
        assert o.scatter_append(rows, w.new_ptr) == "OK"
        assert np.array_equal(pl.cpu().numpy(), host)


@pytest.mark.parametrize("fault", ["NEW_PTR_END", "NEW_PTR_ORDER"])
def test_permissive_decode_step_reads_no_row_past_total_new(hp, oracle, fault):
    """HP_PERMISSIVE with a new_ptr that ends past total_new (or runs backwards): the
    one-kernel decode path skips that sequence, reports the rule, reads no row outside
    the total_new rows given, and writes exactly what the oracle writes."""
    import torch
    rng = np.random.default_rng(11)
    w = inputs.decode_gather(seed=71, num_pages=900, page_size=16, num_heads=8, head_dim=128,
                             num_seqs=20, len_lo=2, len_hi=200, dtype="bf16")
    full = w.lens.astype(np.int64)
    before = full - 1
    if fault == "NEW_PTR_END":  # one row each; the last sequence claims rows past the buffer
        new_ptr = np.arange(w.num_seqs + 1, dtype=np.int64)
        total_new = w.num_seqs
        new_ptr[-1] = total_new + 3
    else:  # sequence 7's pair is (7, 6): backwards; every other pair holds one row
        new_ptr = np.concatenate([np.arange(8), np.arange(6, w.num_seqs - 1)]).astype(np.int64)
        total_new = int(new_ptr[-1])
    rows = rng.integers(0, 256, (total_new, w.row_bytes), dtype=np.uint8)
    # the device buffer holds exactly total_new rows, followed by a page of other bytes
    dev = torch.full(((total_new + 16) * w.row_bytes,), 0xEE, dtype=torch.uint8, device="cuda")
    dev[:total_new * w.row_bytes] = torch.from_numpy(rows.reshape(-1)).to("cuda")
    b = Batch(w, flags=1, lens=before.astype(np.uint32))
    host = b.host_pool().copy()
    rc = hp.hp_scatter_append(b.desc, dev, index_tensor(new_ptr.astype(np.uint32), "cuda"),
                              total_new, b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0
    o = b.oracle_desc(pool_host=host, lens=before.astype(np.uint32))
    assert o.scatter_append(rows, new_ptr.astype(np.uint32), total_new) == fault
    assert hp.status_name(b.status_value()) == "HP_ERR_" + fault
    got = b.pool.cpu().numpy()
    assert np.array_equal(got, host)
