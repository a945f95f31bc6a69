"""GPU parity of the writer side: hp_copy_pages (copy-on-write page copy) and hp_zero_tails
(zeroing the slots no sequence reads) against the oracle, whole pools byte for byte."""
import numpy as np
import pytest

from helpers import Batch, index_tensor
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("page_bytes,it", [(32768, 0), (131072, 1), (4096, 0), (12, 1),
                                           (2048, 1), (20000, 0)])
def test_copy_pages_matches_oracle(hp, oracle, page_bytes, it):
    import torch
    rng = np.random.default_rng(page_bytes + it)
    N = 64
    pool = rng.integers(0, 256, (N, page_bytes), dtype=np.uint8)
    perm = rng.permutation(N)
    k = 20
    src, dst = perm[:k], perm[k:2 * k]
    dt = np.uint32 if it == 0 else np.uint64
    dpool = torch.from_numpy(pool).to("cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    rc = hp.hp_copy_pages(dpool, N, page_bytes, it, index_tensor(src.astype(dt), "cuda"),
                          index_tensor(dst.astype(dt), "cuda"), k, st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    d = oracle.Desc(pool, None, np.zeros(1, dt), np.zeros(0, dt), num_pages=N, page_size=1,
                    num_heads=1, head_dim=page_bytes, dtype="u8", index_type=it)
    assert d.copy_pages(src, dst) == "OK"
    assert np.array_equal(dpool.cpu().numpy(), pool)


def test_copy_pages_out_of_range_pair(hp, oracle):
    import torch
    N, pb = 8, 4096
    pool = np.random.default_rng(1).integers(0, 256, (N, pb), dtype=np.uint8)
    dpool = torch.from_numpy(pool).to("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    src, dst = np.array([0, 9, 2], np.uint32), np.array([5, 6, 7], np.uint32)
    assert hp.hp_copy_pages(dpool, N, pb, 0, index_tensor(src, "cuda"), index_tensor(dst, "cuda"),
                            3, st) == 0
    torch.cuda.synchronize()
    assert hp.status_name(st.item()) == "HP_ERR_PAGE_ID"
    d = oracle.Desc(pool, None, np.zeros(1, np.uint32), np.zeros(0, np.uint32), num_pages=N,
                    page_size=1, num_heads=1, head_dim=pb, dtype="u8", index_type=0)
    assert d.copy_pages(src, dst) == "PAGE_ID"
    assert np.array_equal(dpool.cpu().numpy(), pool)


def _zero_tails(hp, b):
    import torch
    rc, n = hp.hp_zero_tails_scratch_bytes(b.desc)
    scratch = torch.empty(max(n, 4), dtype=torch.uint8, device="cuda")
    return hp.hp_zero_tails(b.desc, b.ws, scratch, b.status)


@pytest.mark.parametrize("name", ["tiny_prefix_gather", "decode_gather", "decode_append",
                                  "prefix_sharing"])
def test_zero_tails_matches_oracle(hp, oracle, name):
    import torch
    w = inputs.config(name, "small")
    b = Batch(w)
    host = b.host_pool().copy()
    assert _zero_tails(hp, b) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    b.oracle_desc(pool_host=host).zero_tails()
    assert np.array_equal(b.pool.cpu().numpy(), host)


@pytest.mark.parametrize("H,D,dtype", [(1, 3, "f16"), (2, 5, "i8"), (4, 8, "f32")])
def test_zero_tails_narrow_rows_and_aliasing(hp, oracle, H, D, dtype):
    """Random aliasing (several sequences naming one page) and rows that are not a
    multiple of 16 bytes."""
    import torch
    rng = np.random.default_rng(H * D)
    N, P = 40, 5
    lens, table, sp = [], [], [0]
    for _ in range(12):
        n = int(rng.integers(0, 4 * P))
        k = -(-n // P) + int(rng.integers(0, 2))
        table += [int(x) for x in rng.integers(0, N, k)]
        sp.append(len(table))
        lens.append(n)
    w = inputs.Workload("alias", N, P, H, D, dtype, np.uint64, np.array(table, np.uint64),
                        np.array(sp, np.uint64), np.array(lens, np.uint64), 3, "normal")
    pool = rng.integers(1, 256, (N, P, w.row_bytes), dtype=np.uint8)
    b = Batch(w, pool=torch.from_numpy(pool).to("cuda"))
    assert _zero_tails(hp, b) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    host = pool.copy()
    b.oracle_desc(pool_host=host).zero_tails()
    assert np.array_equal(b.pool.cpu().numpy(), host)


def test_zero_tails_rejects_invalid_descriptors_even_if_permissive(hp, oracle):
    import torch
    w = inputs.config("decode_gather", "small")
    table = w.table.copy()
    table[2] = w.num_pages + 1
    w2 = inputs.Workload(**{**w.__dict__, "table": table})
    b = Batch(w2, pool=inputs.device_pool(w, "cuda"), flags=1)  # HP_PERMISSIVE asked
    before = b.pool.clone()
    assert _zero_tails(hp, b) == 0
    torch.cuda.synchronize()
    assert hp.status_name(b.status_value()) == "HP_ERR_PAGE_ID"
    assert torch.equal(b.pool, before)


def test_zero_tails_full_size_keeps_the_gather(hp, oracle):
    """After the decode step's batch (4.37M tokens, 273k pages) is zeroed past its counts,
    gathering it returns exactly what it returned before, and the partial pages' tails
    are zero."""
    import torch
    w = inputs.config("decode_append", "full")
    b = Batch(w)
    T = w.total_tokens
    out0 = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(b.desc, out0, T, b.ws, b.status) == 0
    assert _zero_tails(hp, b) == 0
    out1 = torch.empty_like(out0)
    assert hp.hp_gather(b.desc, out1, T, b.ws, b.status) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    assert torch.equal(out0, out1)
    sp = w.seq_ptr.astype(np.int64)
    for s in range(0, w.num_seqs, 17):
        n = int(w.lens[s])
        if n % 16:
            page = int(w.table[sp[s] + n // 16])
            tail = b.pool[page, n % 16:].cpu().numpy()
            assert (tail == 0).all()
