"""GPU parity for the per-lane [N, B, H_kv, P, d] layout ("Keep token order across
cache pages"): hp_lane_gather / hp_lane_append against the oracle, byte for byte."""
import numpy as np
import pytest

from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def test_worked_example_positions(hp, oracle):
    """f64 pool whose values are their own scalar indices: the snapshot of lane
    (batch 0, head 0), feature 0 reads 24, 26, 28, 0, 2, 4, 36 for positions 0..6."""
    import torch
    w = inputs.lane_worked_example()
    pool = np.arange(np.prod(w.pool_shape), dtype=np.float64).reshape(w.pool_shape)
    out = torch.zeros((w.batch, w.kv_heads, w.n, w.width), dtype=torch.float64, device="cuda")
    st = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    rc = hp.hp_lane_gather(_dev(pool), _dev(w.table.view(np.int64)), w.capacity, w.page_tokens,
                           w.batch, w.kv_heads, w.width, "f64", w.n, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    got = out.cpu().numpy()
    assert list(got[0, 0, :, 0].astype(int)) == [24, 26, 28, 0, 2, 4, 36]
    assert got[0, 1, 0, 0] == 30
    want = oracle.lane_gather(pool, w.capacity, w.page_tokens, w.table, w.batch, w.kv_heads,
                              w.width, w.n)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seed", range(12))
def test_lane_gather_append_random(hp, oracle, seed):
    import torch
    rng = np.random.default_rng(400 + seed)
    P = int(rng.integers(1, 20))
    C = int(rng.integers(1, 300))
    B, H = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    W = int(rng.choice([1, 3, 8, 64, 128]))
    dtype = ["bf16", "f32", "f64", "i8"][seed % 4]
    es = inputs.ELEM_BYTES[dtype]
    N = -(-C // P)
    T = rng.permutation(N).astype(np.uint64)
    n = int(rng.integers(0, C + 1))
    pool = rng.integers(0, 256, (N, B, H, P, W * es), dtype=np.uint8)
    npdt = {"bf16": np.uint16, "f32": np.float32, "f64": np.float64, "i8": np.int8}[dtype]
    pool_t = pool.view(npdt).reshape(N, B, H, P, W)
    dpool = _dev(pool)
    dT = _dev(T.view(np.int64))
    st = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    out = torch.full((B * H * n * W * es + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    rc = hp.hp_lane_gather(dpool, dT, C, P, B, H, W, dtype, n, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    want = oracle.lane_gather(pool_t, C, P, T, B, H, W, n)
    o = out.cpu().numpy()
    # compare bytes: random bit patterns include NaNs
    assert np.array_equal(o[:B * H * n * W * es], np.ascontiguousarray(want).view(np.uint8).reshape(-1))
    assert (o[B * H * n * W * es:] == 0xEE).all()
    m = int(rng.integers(0, C - n + 1))
    new = rng.integers(0, 256, (B, H, m, W * es), dtype=np.uint8)
    rc = hp.hp_lane_append(dpool, dT, C, P, B, H, W, dtype, n, m, _dev(new), st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    host = pool_t.copy()
    assert oracle.lane_append(host, C, P, T, B, H, W, n, new.view(npdt).reshape(B, H, m, W)) == "OK"
    assert np.array_equal(dpool.cpu().numpy().reshape(-1), host.view(np.uint8).reshape(-1))


def test_lane_length_and_table_errors(hp, oracle):
    import torch
    w = inputs.lane_worked_example()
    pool = torch.zeros(w.pool_shape, dtype=torch.float64, device="cuda")
    T = _dev(w.table.view(np.int64))
    out = torch.zeros((1, 2, 13, 2), dtype=torch.float64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hp.hp_lane_gather(pool, T, 12, 3, 1, 2, 2, "f64", 13, out, st)
    assert hp.status_name(rc) == "HP_ERR_LENGTH"
    new = torch.zeros((1, 2, 6, 2), dtype=torch.float64, device="cuda")
    assert hp.status_name(hp.hp_lane_append(pool, T, 12, 3, 1, 2, 2, "f64", 7, 6, new, st)) == \
        "HP_ERR_LENGTH"
    assert hp.status_name(hp.hp_lane_gather(pool, T, 0, 3, 1, 2, 2, "f64", 0, out, st)) == \
        "HP_ERR_ZERO_CAPACITY"
    assert hp.status_name(hp.hp_lane_gather(pool, T, 12, 0, 1, 2, 2, "f64", 0, out, st)) == \
        "HP_ERR_ZERO_PAGE_SIZE"
    # an entry outside the pool skips its rows and is reported
    bad = _dev(np.array([2, 0, 7, 1], dtype=np.int64))
    out.fill_(-1.0)
    rc = hp.hp_lane_gather(pool, bad, 12, 3, 1, 2, 2, "f64", 9, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and hp.status_name(st.item()) == "HP_ERR_PHYSICAL_PAGE"
    assert (out.cpu().numpy()[0, :, 6:9] == -1.0).all()


def test_lane_synthetic_full_size_sampled(hp, oracle):
    """The benchmark's per-lane workload (32 x 8 lanes, 8192 positions of 128 bf16
    features): lanes sampled whole against the oracle."""
    import torch
    w = inputs.lane_synthetic()
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    pool = torch.randn(w.pool_shape, generator=g, device="cuda").to(torch.bfloat16)
    T = _dev(w.table.view(np.int64))
    out = torch.empty((w.batch, w.kv_heads, w.n, w.width), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hp.hp_lane_gather(pool, T, w.capacity, w.page_tokens, w.batch, w.kv_heads, w.width,
                           "bf16", w.n, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    host = pool.view(torch.int16).cpu().numpy()
    got = out.view(torch.int16).cpu().numpy()
    rng = np.random.default_rng(2)
    for b, h in zip(rng.integers(0, w.batch, 4), rng.integers(0, w.kv_heads, 4)):
        # the oracle on a one-lane slice of the pool
        one = np.ascontiguousarray(host[:, b:b + 1, h:h + 1])
        want = oracle.lane_gather(one, w.capacity, w.page_tokens, w.table, 1, 1, w.width, w.n)
        assert np.array_equal(got[b, h], want[0, 0])


@pytest.mark.parametrize("B,H,P,W,dtype", [(3, 3, 16, 128, "bf16"), (1, 5, 8, 128, "f32"),
                                           (2, 3, 4, 256, "bf16"), (1, 1, 16, 64, "bf16"),
                                           (5, 7, 32, 32, "bf16"), (2, 2, 2, 512, "bf16"),
                                           (4, 8, 16, 256, "bf16")])
def test_lane_gather_run_sizes(hp, oracle, B, H, P, W, dtype):
    """(lane, page) runs of 2-16 KiB: odd lane counts, live lengths that end in a partial
    page, one row, the whole capacity; then one page ID outside the pool, whose rows are
    skipped and reported while every other row still lands."""
    import torch
    rng = np.random.default_rng(B * 100 + H * 10 + P)
    es = inputs.ELEM_BYTES[dtype]
    C = int(rng.integers(3 * P, 60 * P))
    N = -(-C // P)
    T = rng.permutation(N).astype(np.uint64)
    pool = rng.integers(0, 256, (N, B, H, P, W * es), dtype=np.uint8)
    dpool = _dev(pool)
    st = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    for n in (1, P + 1, C - 1, C, int(rng.integers(1, C + 1))):
        nbytes = B * H * n * W * es
        out = torch.full((nbytes + 64,), 0xEE, dtype=torch.uint8, device="cuda")
        rc = hp.hp_lane_gather(dpool, _dev(T.view(np.int64)), C, P, B, H, W, dtype, n, out, st)
        torch.cuda.synchronize()
        assert rc == 0 and st.item() == 0
        want = oracle.lane_gather(pool, C, P, T, B, H, W * es, n)
        o = out.cpu().numpy()
        assert np.array_equal(o[:nbytes], want.reshape(-1)), n
        assert (o[nbytes:] == 0xEE).all()
    bad = T.copy()
    k = int(rng.integers(0, N))
    bad[k] = N + 3
    n = C
    nbytes = B * H * n * W * es
    out = torch.full((nbytes,), 0xEE, dtype=torch.uint8, device="cuda")
    rc = hp.hp_lane_gather(dpool, _dev(bad.view(np.int64)), C, P, B, H, W, dtype, n, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and hp.status_name(st.item()) == "HP_ERR_PHYSICAL_PAGE"
    o = out.cpu().numpy().reshape(B * H, n, W * es)
    good = oracle.lane_gather(pool, C, P, T, B, H, W * es, n).reshape(B * H, n, W * es)
    rows = np.arange(n) // P == k
    assert (o[:, rows] == 0xEE).all()
    assert np.array_equal(o[:, ~rows], good[:, ~rows])
