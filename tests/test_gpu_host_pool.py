"""GPU parity of the operations on a page pool (or an output) in page-locked host memory:
the kernels read and write it in place over the host link (the caller sets HP_HOST_MEMORY,
which sends the copies to the register engine; the TMA engine is kept to device memory).
Bit-exact against the oracle, like every copy."""
import numpy as np
import pytest

from helpers import Batch, index_tensor
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _pinned_copy(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


@pytest.mark.parametrize("out_on_host", [False, True])
@pytest.mark.parametrize("name", ["decode_gather", "prefix_sharing"])
def test_gather_from_a_host_pool(hp, oracle, name, out_on_host):
    """128 KiB (decode_gather) and 32 KiB (prefix_sharing) page runs, which a device pool
    sends through the TMA engine; the output in device or in host memory."""
    import torch
    w = inputs.config(name, "small")
    dev = Batch(w)
    host_pool = _pinned_copy(dev.pool)
    b = Batch(w, pool=host_pool, flags=hp.HOST_MEMORY)
    T = w.total_tokens
    if out_on_host:
        out = torch.full((T * w.row_bytes,), 0xEE, dtype=torch.uint8, pin_memory=True)
    else:
        out = torch.full((T * w.row_bytes,), 0xEE, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(b.desc, out, T, b.ws, b.status) == 0
    torch.cuda.synchronize()
    assert hp.status_name(b.status_value()) == "HP_OK"
    want, written, fault = dev.oracle_desc().gather()
    assert fault == "OK" and written.all()
    assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)


def test_bulk_append_into_a_host_pool_then_gather(hp, oracle):
    """Prefill-style append of every row into empty slices of a host-resident pool, then
    the gather back: the rows come back, and no other byte of the pool changed."""
    import torch
    w = inputs.decode_gather(seed=78, num_pages=300, num_heads=8, head_dim=128, num_seqs=5,
                             len_lo=1, len_hi=300, dtype="bf16")
    T = w.total_tokens
    pool = _pinned_copy(inputs.device_pool(w, "cuda"))
    before = pool.numpy().copy()
    rows = np.random.default_rng(2).integers(0, 256, (T, w.row_bytes), dtype=np.uint8)
    new = torch.from_numpy(rows.reshape(-1)).to("cuda")
    new_ptr = index_tensor(np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))])
                           .astype(np.uint32), "cuda")
    zeros = np.zeros(w.num_seqs, dtype=np.uint32)
    a = Batch(w, pool=pool, lens=zeros, flags=hp.HOST_MEMORY)
    assert hp.hp_scatter_append(a.desc, new, new_ptr, T, a.ws, a.status) == 0
    torch.cuda.synchronize()
    assert a.status_value() == 0
    # the oracle's append on a copy of the pool as it was gives the same bytes
    want_pool = before.copy()
    o = a.oracle_desc(pool_host=want_pool, lens=zeros)
    np_host = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))]).astype(np.uint32)
    assert o.scatter_append(rows, np_host) == "OK"
    assert np.array_equal(pool.numpy(), want_pool)
    g = Batch(w, pool=pool, flags=hp.HOST_MEMORY)
    out = torch.empty(T * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(g.desc, out, T, g.ws, g.status) == 0
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().reshape(T, -1), rows)


def test_copy_pages_in_a_host_pool(hp, oracle):
    import torch
    pages, page_bytes = 64, 32768
    rng = np.random.default_rng(5)
    host = rng.integers(0, 256, pages * page_bytes, dtype=np.uint8)
    pool = torch.from_numpy(host.copy()).pin_memory()
    src = rng.choice(32, 20, replace=False).astype(np.uint32)
    dst = (32 + rng.choice(32, 20, replace=False)).astype(np.uint32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hp.hp_copy_pages(pool, pages, page_bytes, 0, index_tensor(src, "cuda"),
                          index_tensor(dst, "cuda"), 20, st, flags=hp.HOST_MEMORY)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    want = host.reshape(pages, page_bytes).copy()
    want[dst] = want[src]
    assert np.array_equal(pool.numpy().reshape(pages, page_bytes), want)


@pytest.mark.parametrize("out_on_host", [False, True])
def test_dequant_gather_from_a_host_pool(hp, oracle, out_on_host):
    """The dequantising gather (int8 codes x per-slot scales -> bf16) on a pool in
    page-locked host memory, the output in device or host memory: the same bits as the
    oracle's single rounding."""
    import torch
    w = inputs.config("quantized_pool", "small")
    dev = Batch(w)
    b = Batch(w, pool=_pinned_copy(dev.pool), flags=hp.HOST_MEMORY)
    T = w.total_tokens
    n = T * w.num_heads * w.head_dim
    kw = dict(pin_memory=True) if out_on_host else dict(device="cuda")
    out = torch.full((n,), -1, dtype=torch.int16, **kw)
    assert hp.hp_gather_dequant(b.desc, out, T, b.ws, b.status) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    want, written, fault = dev.oracle_desc().gather_dequant()
    assert fault == "OK" and written.all()
    got = out.cpu().numpy().view(np.uint16).reshape(want.shape)
    assert np.array_equal(got, want)


def test_lane_gather_and_append_on_a_host_pool(hp, oracle):
    """[N, B, H_kv, P, d] lane layout with 16 KiB (lane, page) runs, which a device pool
    sends through the TMA engine, in page-locked host memory: snapshot, then append."""
    import torch
    rng = np.random.default_rng(9)
    C, P, B, H, W = 1000, 64, 2, 3, 128
    N = -(-C // P)
    T = rng.permutation(N).astype(np.uint64)
    pool = rng.integers(0, 256, (N, B, H, P, W * 2), dtype=np.uint8)
    hpool = torch.from_numpy(pool.copy()).pin_memory()
    dT = torch.from_numpy(T.view(np.int64).copy()).to("cuda")
    st = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    n = 777
    out = torch.full((B * H * n * W * 2,), 0xEE, dtype=torch.uint8, pin_memory=True)
    assert hp.hp_lane_gather(hpool, dT, C, P, B, H, W, "bf16", n, out, st,
                             flags=hp.HOST_MEMORY) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    pool_t = pool.view(np.uint16).reshape(N, B, H, P, W)
    want = oracle.lane_gather(pool_t, C, P, T, B, H, W, n)
    assert np.array_equal(out.numpy(), np.ascontiguousarray(want).view(np.uint8).reshape(-1))
    m = 150
    new = rng.integers(0, 256, (B, H, m, W * 2), dtype=np.uint8)
    hnew = torch.from_numpy(new.copy()).pin_memory()
    assert hp.hp_lane_append(hpool, dT, C, P, B, H, W, "bf16", n, m, hnew, st,
                             flags=hp.HOST_MEMORY) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    host = pool_t.copy()
    assert oracle.lane_append(host, C, P, T, B, H, W, n,
                              new.view(np.uint16).reshape(B, H, m, W)) == "OK"
    assert np.array_equal(hpool.numpy().reshape(-1), host.view(np.uint8).reshape(-1))


def test_decode_attention_on_host_resident_k_and_v(hp, oracle):
    """K and V pools in page-locked host memory (an offloaded cache, HP_HOST_MEMORY): the
    CUDA-core kernel's cp.async loads read them over the host link; the result is bit for
    bit the one the same kernel gives from device pools (HP_HOST_MEMORY set there too, which
    keeps the call off the tensor-core kernel), and matches the oracle."""
    import torch
    w = inputs.decode_gather(seed=61, num_pages=400, page_size=16, num_heads=2, head_dim=128,
                             num_seqs=4, len_lo=1, len_hi=1500, dtype="bf16")
    b = Batch(w, flags=hp.HOST_MEMORY)
    vdev = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 62}), "cuda")
    khost, vhost = _pinned_copy(b.pool), _pinned_copy(vdev)
    dh = hp.PagedDesc(khost, b.table, b.seq_ptr, b.lens, num_pages=w.num_pages, page_size=16,
                      num_heads=2, head_dim=128, dtype="bf16", index_type=b.it,
                      flags=hp.HOST_MEMORY)
    g = torch.Generator(device="cuda")
    g.manual_seed(63)
    q = torch.randn((w.num_seqs, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, 8)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    want = torch.full((w.num_seqs, 8, 128), float("nan"), dtype=torch.float32, device="cuda")
    got = torch.full_like(want, float("nan"))
    assert hp.hp_attention_decode(b.desc, vdev, q, 8, 0.09, want, ws, b.status) == 0
    assert hp.hp_attention_decode(dh, vhost, q, 8, 0.09, got, ws, b.status) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    ref = b.oracle_desc().attention_decode(vdev.cpu().numpy(),
                                           q.view(torch.int16).cpu().numpy().view(np.uint16), 8,
                                           0.09)
    vmax = float(vdev.view(torch.bfloat16).float().abs().max())
    assert np.abs(got.cpu().numpy() - ref).max() <= 1e-4 * vmax + 1e-6
