"""GPU parity: hp_gather / hp_validate against the CPU oracle, element by element.

Bit-exact: a gather copies bytes, so every output byte must equal the oracle's.
"""
import numpy as np
import pytest

from conftest import guarded, guards_intact
from helpers import Batch, index_tensor, lib_name, sub_batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu

GATHER_CONFIGS = ("tiny_prefix_gather", "decode_gather", "decode_append", "prefix_sharing")


def run_gather(hp, b, out_tokens=None, **kw):
    import torch
    T = b.w.total_tokens if out_tokens is None else out_tokens
    nbytes = T * b.w.row_bytes
    buf, out = guarded(nbytes)
    rc = hp.hp_gather(b.desc, out, T, b.ws, b.status, **kw)
    torch.cuda.synchronize()
    return rc, buf, out, nbytes


@pytest.mark.parametrize("name", GATHER_CONFIGS)
def test_gather_matches_oracle_small(hp, oracle, name):
    w = inputs.config(name, "small")
    b = Batch(w)
    rc, buf, out, nbytes = run_gather(hp, b)
    assert hp.status_name(rc) == "HP_OK"
    assert hp.status_name(b.status_value()) == "HP_OK"
    want, written, fault = b.oracle_desc().gather()
    assert fault == "OK" and written.all()
    got = out.cpu().numpy().reshape(want.shape)
    assert np.array_equal(got, want)
    assert guards_intact(buf, nbytes)


def test_tiny_prefix_config_rows(hp, oracle):
    """Slices [12,5,7,9] / [12,5,7,3]: the shared prefix reads pages 12, 5, 7 for
    both sequences; rows 12-14 come from page 9, row 27 from page 3."""
    w = inputs.tiny_prefix_gather()
    b = Batch(w)
    rc, buf, out, nbytes = run_gather(hp, b)
    assert rc == 0 and b.status_value() == 0
    got = out.cpu().numpy().reshape(28, 32)
    pool = b.host_pool()
    assert np.array_equal(got[15:27], got[0:12])
    assert np.array_equal(got[12:15], pool[9, :3]) and np.array_equal(got[27], pool[3, 0])
    assert np.array_equal(got, b.oracle_desc().gather()[0])


def _check_sampled(hp, oracle, b, got, n_seq=4, n_elem=3000, seed=0):
    """Whole sequences (first, last and random ones) through the oracle's gather of
    their re-based slices, plus random single elements through its Element Lookup."""
    import torch
    w = b.w
    rng = np.random.default_rng(seed)
    S = w.num_seqs
    seqs = sorted(set([0, S - 1] + list(rng.integers(0, S, n_seq))))
    table, seq_ptr, lens = sub_batch(w, seqs, b.lens_host)
    host = b.host_pool()
    sub = oracle.Desc(host, table, seq_ptr, lens, num_pages=w.num_pages, page_size=w.page_size,
                      num_heads=w.num_heads, head_dim=w.head_dim, dtype=w.dtype,
                      index_type=b.it)
    want, written, fault = sub.gather()
    assert fault == "OK"
    tok_off = np.concatenate([[0], np.cumsum(b.lens_host.astype(np.int64))])
    rows = np.concatenate([np.arange(tok_off[s], tok_off[s + 1]) for s in seqs])
    assert np.array_equal(got[rows], want)
    # random elements anywhere in the batch
    full = b.oracle_desc()
    es = inputs.ELEM_BYTES[w.dtype]
    H, D = w.num_heads, w.head_dim
    for _ in range(n_elem):
        s = int(rng.integers(0, S))
        n = int(b.lens_host[s])
        if n == 0:
            continue
        t, h, d = int(rng.integers(0, n)), int(rng.integers(0, H)), int(rng.integers(0, D))
        code, val = full.lookup(s, t, h, d)
        assert code == "OK"
        row = tok_off[s] + t
        assert np.array_equal(got[row, (h * D + d) * es:(h * D + d + 1) * es], val)


@pytest.mark.parametrize("name", ["decode_gather", "prefix_sharing", "decode_append"])
def test_gather_full_size_sampled(hp, oracle, name):
    import torch
    w = inputs.config(name, "full")
    b = Batch(w)
    rc, buf, out, nbytes = run_gather(hp, b)
    assert rc == 0 and b.status_value() == 0
    got = out.cpu().numpy().reshape(w.total_tokens, w.row_bytes)
    assert guards_intact(buf, nbytes)
    _check_sampled(hp, oracle, b, got)
    # no row of the output is a sentinel-filled (never written / undefined) slot
    assert not (got[:, :16] == inputs.SENTINEL).all(axis=1).any()


@pytest.mark.parametrize("H,D,dtype", [(1, 1, "i8"), (1, 3, "f16"), (3, 1, "f32"), (1, 5, "f64"),
                                       (2, 3, "bf16"), (5, 7, "i8"), (1, 4, "f16"),
                                       (3, 4, "f32")])
@pytest.mark.parametrize("P", [1, 3, 16])
def test_gather_narrow_rows(hp, oracle, H, D, dtype, P):
    """Rows whose byte length is not a multiple of 16 take the narrower vector paths."""
    w = inputs.decode_gather(seed=H * 100 + D * 10 + P, num_pages=300, page_size=P,
                             num_heads=H, head_dim=D, dtype=dtype, num_seqs=6, len_lo=0,
                             len_hi=40, index_dtype=np.uint64 if P == 3 else np.uint32)
    b = Batch(w)
    rc, buf, out, nbytes = run_gather(hp, b)
    assert rc == 0 and b.status_value() == 0
    want = b.oracle_desc().gather()[0]
    assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)
    assert guards_intact(buf, nbytes)


def test_gather_u64_indices_and_zero_lengths(hp, oracle):
    w = inputs.decode_gather(seed=9, num_pages=400, num_heads=4, head_dim=64, num_seqs=9,
                             len_lo=0, len_hi=300, index_dtype=np.uint64)
    lens = w.lens.copy()
    lens[[0, 4, 8]] = 0  # empty sequences keep their (unread) slices
    b = Batch(w, lens=lens)
    rc, buf, out, nbytes = run_gather(hp, b, out_tokens=int(lens.sum()))
    assert rc == 0 and b.status_value() == 0
    want = b.oracle_desc().gather()[0]
    assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)


def test_empty_batch(hp, oracle):
    """num_seqs = 0, block_table NULL, seq_ptr = [0]."""
    import torch
    seq_ptr = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = torch.zeros(4 * 4 * 16, dtype=torch.uint8, device="cuda")
    d = hp.PagedDesc(pool, None, seq_ptr, None, num_pages=4, page_size=4, num_heads=2, head_dim=4,
                     dtype="f16", index_type=0)
    ws = hp.workspace_for(d)
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    assert hp.hp_gather(d, None, 0, ws, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    assert hp.hp_validate(d, ws) == (0, 0)
    bad = torch.ones(1, dtype=torch.int32, device="cuda")  # seq_ptr[0] = 1
    d2 = hp.PagedDesc(pool, None, bad, None, num_pages=4, page_size=4, num_heads=2, head_dim=4,
                      dtype="f16", index_type=0)
    assert hp.status_name(hp.hp_validate(d2, ws)[0]) == "HP_ERR_SEQ_PTR_START"


def test_out_size_mismatch_writes_nothing(hp, oracle):
    w = inputs.config("decode_gather", "small")
    b = Batch(w)
    rc, buf, out, nbytes = run_gather(hp, b, out_tokens=w.total_tokens - 1)
    assert rc == 0
    assert hp.status_name(b.status_value()) == "HP_ERR_OUT_SIZE"
    assert (out.cpu().numpy() == 0xEE).all() and guards_intact(buf, nbytes)


# ----------------------------------------------------------------------- validation
def _mk(hp, pool, table, seq_ptr, lens, it=0, **kw):
    import torch
    dt = np.uint32 if it == 0 else np.uint64
    tt = index_tensor(np.asarray(table, dt), "cuda") if len(table) else None
    return hp.PagedDesc(pool, tt, index_tensor(np.asarray(seq_ptr, dt), "cuda"),
                        index_tensor(np.asarray(lens, dt), "cuda"), index_type=it, **kw)


@pytest.mark.parametrize("kw,want", [
    ({}, ("OK", 0)),
    ({"seq_ptr": [1, 2, 3]}, ("SEQ_PTR_START", 0)),
    ({"seq_ptr": [0, 3, 2, 3], "lens": [1, 1, 1]}, ("SEQ_PTR_ORDER", 1)),
    ({"seq_ptr": [0, 2, 2]}, ("SEQ_PTR_END", 2)),
    ({"seq_ptr": [0, 2, 4]}, ("SEQ_PTR_END", 2)),
    ({"table": [0, 4, 2]}, ("PAGE_ID", 1)),
    ({"table": [7, 4, 2]}, ("PAGE_ID", 0)),
    ({"lens": [9, 4]}, ("LEN", 0)),
    ({"lens": [8, 5]}, ("LEN", 1)),
    ({"lens": [8, 4]}, ("OK", 0)),
    ({"seq_ptr": [1, 0, 3], "table": [9, 9, 9]}, ("SEQ_PTR_START", 0)),
    ({"seq_ptr": [0, 3, 2], "table": [9, 9, 9]}, ("SEQ_PTR_ORDER", 1)),
    ({"table": [9, 9, 9], "lens": [99, 99]}, ("PAGE_ID", 0)),
    ({"table": [1, 1, 1], "lens": [8, 4]}, ("OK", 0)),
    ({"flags": 1, "seq_ptr": [1, 0, 3], "table": [9, 9, 9]}, ("OK", 0)),
    ({"rank": 2}, ("RANK", 0)),
    ({"has_shard": 1}, ("SHARD", 0)),
])
@pytest.mark.parametrize("it", [0, 1])
def test_validate_verdicts(hp, oracle, kw, want, it):
    import torch
    pool = torch.zeros(4 * 4 * 2 * 2 * 2, dtype=torch.uint8, device="cuda")
    args = dict(table=[0, 1, 2], seq_ptr=[0, 2, 3], lens=[5, 4])
    extra = {k: kw[k] for k in ("flags", "rank", "has_shard") if k in kw}
    args.update({k: v for k, v in kw.items() if k in args})
    d = _mk(hp, pool, args["table"], args["seq_ptr"], args["lens"], it=it, num_pages=4,
            page_size=4, num_heads=2, head_dim=2, dtype="f16", **extra)
    ws = hp.workspace_for(d)
    rc, first = hp.hp_validate(d, ws)
    o = oracle.Desc(pool.cpu().numpy(), args["table"], args["seq_ptr"], args["lens"],
                    num_pages=4, page_size=4, num_heads=2, head_dim=2, dtype="f16",
                    index_type=it, **extra).validate()
    assert o == want
    assert (hp.status_name(rc), first) == (lib_name(want[0]), want[1])
    # the gather reaches the same verdict on the device and writes nothing
    if not extra or extra == {"flags": 1}:
        st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        T = int(sum(args["lens"]))
        buf, out = guarded(T * 8)
        assert hp.hp_gather(d, out, T, ws, st) == 0
        torch.cuda.synchronize()
        if want[0] == "OK" and not extra:
            assert st.item() == 0
        elif want[0] != "OK":
            assert hp.status_name(st.item()) == lib_name(want[0])
            assert (buf.cpu().numpy() == 0xEE).all()


def test_validate_random_parity(hp, oracle):
    """Random small descriptors, valid and invalid: the device verdict (rule and
    first index) equals the oracle's."""
    import torch
    rng = np.random.default_rng(21)
    pool = torch.zeros(64, dtype=torch.uint8, device="cuda")
    seen = set()
    for trial in range(300):
        S = int(rng.integers(0, 6))
        tlen = int(rng.integers(0, 8))
        N = int(rng.integers(1, 6))
        if S == 0:
            seq_ptr = np.array([0 if trial % 2 else tlen])
        else:
            inner = np.sort(rng.integers(0, tlen + 1, S - 1))
            seq_ptr = np.concatenate([[0], inner, [tlen]])
        if trial % 3 == 0:
            seq_ptr = rng.integers(0, 5, S + 1)
        table = rng.integers(0, N + (trial % 4 == 0), tlen)
        slices = np.maximum(np.diff(seq_ptr), 0)
        lens = np.array([rng.integers(0, 2 * k + 2) for k in slices], dtype=np.int64)
        it = trial % 2
        kw = dict(num_pages=N, page_size=2, num_heads=1, head_dim=4, dtype="i8")
        d = _mk(hp, pool, list(table), list(seq_ptr), list(lens), it=it, **kw)
        ws = hp.workspace_for(d)
        rc, first = hp.hp_validate(d, ws)
        o = oracle.Desc(pool.cpu().numpy(), list(table) if tlen else None, list(seq_ptr),
                        list(lens), index_type=it, **kw).validate()
        seen.add(o[0])
        assert (hp.status_name(rc), first) == (lib_name(o[0]), o[1]), (seq_ptr, table, lens)
    assert {"OK", "SEQ_PTR_START", "SEQ_PTR_ORDER", "SEQ_PTR_END", "PAGE_ID", "LEN"} <= seen


def test_validate_large_table_first_index(hp, oracle):
    """Invariant (3) over a 270k-entry table: the first bad entry is found however
    the CTAs race."""
    import torch
    w = inputs.config("decode_append", "full")
    table = w.table.copy()
    bad = [200_000, 123_457, 250_001]
    for k in bad:
        table[k] = w.num_pages + k
    pool = torch.zeros(64, dtype=torch.uint8, device="cuda")
    d = hp.PagedDesc(pool, index_tensor(table, "cuda"), index_tensor(w.seq_ptr, "cuda"),
                     index_tensor(w.lens, "cuda"), num_pages=w.num_pages, page_size=16,
                     num_heads=8, head_dim=128, dtype="bf16", index_type=0)
    ws = hp.workspace_for(d)
    rc, first = hp.hp_validate(d, ws)
    assert (hp.status_name(rc), first) == ("HP_ERR_PAGE_ID", min(bad))


def test_permissive_gather_skips_unreadable_rows(hp, oracle):
    """Permissive mode: rows whose lookup leaves the slice, the table or the pool are
    not written; the readable rows equal the oracle's; d_status names a fault the
    oracle also met."""
    import torch
    w = inputs.config("decode_gather", "small")
    table = w.table.copy()
    table[3] = w.num_pages + 5                      # a page outside the pool
    lens = w.lens.copy()
    lens[2] += 3 * w.page_size                      # reads past its slice
    w2 = inputs.Workload(**{**w.__dict__, "table": table})
    b = Batch(w2, pool=inputs.device_pool(w, "cuda"), flags=1, lens=lens)
    T = int(lens.astype(np.int64).sum())
    rc, buf, out, nbytes = run_gather(hp, b, out_tokens=T)
    assert rc == 0
    want = np.full((T, w.row_bytes), 0xEE, np.uint8)
    want, written, fault = b.oracle_desc().gather(want)
    assert not written.all()
    got = out.cpu().numpy().reshape(T, w.row_bytes)
    assert np.array_equal(got, want)
    assert hp.status_name(b.status_value()) in {"HP_ERR_LEN", "HP_ERR_PAGE_ID"}
    assert guards_intact(buf, nbytes)


def test_planned_steps_equal_one_call(hp, oracle):
    """hp_plan + hp_gather_planned on one stream is hp_gather."""
    import torch
    w = inputs.config("prefix_sharing", "small")
    b = Batch(w)
    T = w.total_tokens
    out1 = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    out2 = torch.empty_like(out1)
    assert hp.hp_gather(b.desc, out1, T, b.ws, b.status) == 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ws2 = hp.workspace_for(b.desc)
        assert hp.hp_plan(b.desc, T, ws2, None, stream=s) == 0
        assert hp.hp_gather_planned(b.desc, out2, ws2, None, stream=s) == 0
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_one_launch_gather_random_verdicts_and_rows(hp, oracle):
    """Small validated batches take the one-launch gather: on random small descriptors,
    valid and invalid, its status is the oracle's rule, the verdict key it leaves in the
    workspace names the oracle's first failing index, and a valid batch gathers the
    oracle's rows."""
    import torch
    rng = np.random.default_rng(33)
    ranks = {"SEQ_PTR_START": 1, "SEQ_PTR_ORDER": 2, "SEQ_PTR_END": 3, "PAGE_ID": 4, "LEN": 5}
    seen = set()
    for trial in range(200):
        S = int(rng.integers(0, 6))
        tlen = int(rng.integers(0, 8))
        N = int(rng.integers(1, 6))
        if S == 0:
            seq_ptr = np.array([0 if trial % 2 else tlen])
        else:
            inner = np.sort(rng.integers(0, tlen + 1, S - 1))
            seq_ptr = np.concatenate([[0], inner, [tlen]])
        if trial % 3 == 0:
            seq_ptr = rng.integers(0, 5, S + 1)
        table = rng.integers(0, N + (trial % 4 == 0), tlen)
        slices = np.maximum(np.diff(seq_ptr), 0)
        lens = np.array([rng.integers(0, 2 * k + 2) for k in slices], dtype=np.int64)
        it = trial % 2
        pool_h = rng.integers(0, 256, N * 2 * 4, dtype=np.uint8)
        pool = torch.from_numpy(pool_h).to("cuda")
        kw = dict(num_pages=N, page_size=2, num_heads=1, head_dim=4, dtype="i8")
        d = _mk(hp, pool, list(table), list(seq_ptr), list(lens), it=it, **kw)
        ws = hp.workspace_for(d)
        T = int(lens.sum())
        buf, out = guarded(T * 4)
        st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        assert hp.hp_gather(d, out, T, ws, st) == 0
        torch.cuda.synchronize()
        od = oracle.Desc(pool_h, list(table) if tlen else None, list(seq_ptr), list(lens),
                         index_type=it, **kw)
        code, first = od.validate()
        seen.add(code)
        assert hp.status_name(st.item()) == lib_name(code), (seq_ptr, table, lens)
        key = int(ws[:8].cpu().numpy().view(np.uint64)[0])
        if code == "OK":
            assert key == (1 << 64) - 1
            want = od.gather()[0].reshape(-1)
            assert np.array_equal(out.cpu().numpy()[:T * 4], want)
        else:
            assert (key >> 58, key & ((1 << 58) - 1)) == (ranks[code], first)
            assert (buf.cpu().numpy() == 0xEE).all()
    assert {"OK", "SEQ_PTR_START", "SEQ_PTR_ORDER", "SEQ_PTR_END", "PAGE_ID", "LEN"} <= seen


def test_one_plan_serves_the_pools_of_several_layers(hp, oracle):
    """hp_plan once, then hp_gather_planned through descriptors that differ only in
    page_pool (one pool per layer): each output equals that pool's one-call gather."""
    import torch
    w = inputs.config("decode_gather", "small")
    b = Batch(w)
    assert hp.hp_plan(b.desc, w.total_tokens, b.ws, b.status) == 0
    for layer in range(3):
        pl = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 900 + layer}),
                                "cuda")
        dl = hp.PagedDesc(pl, b.table, b.seq_ptr, b.lens, num_pages=w.num_pages,
                          page_size=w.page_size, num_heads=w.num_heads, head_dim=w.head_dim,
                          dtype=w.dtype, index_type=b.it)
        got = torch.empty(w.total_tokens * w.row_bytes, dtype=torch.uint8, device="cuda")
        assert hp.hp_gather_planned(dl, got, b.ws, b.status) == 0
        torch.cuda.synchronize()
        assert b.status_value() == 0
        want = b.oracle_desc(pool_host=pl.cpu().numpy()).gather()[0]
        assert np.array_equal(got.cpu().numpy().reshape(want.shape), want)
