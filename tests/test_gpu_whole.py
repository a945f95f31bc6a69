"""GPU parity at the benchmark configurations' stated sizes, on every output byte.

The sampled full-size checks in the other files are the quick variants.  These compare
the whole gathered tensor of the decode-sized batch, the decode step (the whole pool after
the append, then the whole gather of the grown batch), the prefix-sharing batch and the
int8 pool's dequantising gather with the CPU oracle, one group of sequences at a time so
that host memory stays bounded (the oracle's rows of a group are built on every host
thread, then compared with the same rows copied back from the device).

Bars: bit-exact for the copies ("Block-Paged Layout -- Hurray Format Specification",
Element Lookup); for the dequantising gather (Per-page-slot parameters) |gpu - oracle| <=
2^-8 |oracle| per element, and no bit may differ, since the kernel rounds the exact
product once as the oracle does.  The per-lane snapshot ("Keep token order across cache
pages") and decode attention at full size are compared whole too, attention within the
bound derived in test_gpu_attention.py.
"""
import numpy as np
import pytest

from helpers import Batch, compare_whole_gather, host_threads, index_tensor, oracle_group, \
    sequence_groups
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _device_rows(out, row_bytes, dtype=np.uint8, width=None):
    """A got_rows callback over a flat device tensor of rows."""
    def rows(r0, r1):
        h = out[r0 * row_bytes:r1 * row_bytes].cpu().numpy()
        return h.view(dtype).reshape(r1 - r0, -1 if width is None else width)
    return rows


def _gather_whole(hp, oracle, w, b, host_pool):
    import torch
    T = w.total_tokens
    nbytes = T * w.row_bytes
    out = torch.full((nbytes + 256,), 0xEE, dtype=torch.uint8, device="cuda")
    rc = hp.hp_gather(b.desc, out, T, b.ws, b.status)
    torch.cuda.synchronize()
    assert hp.status_name(rc) == "HP_OK" and hp.status_name(b.status_value()) == "HP_OK"
    assert (out[nbytes:].cpu().numpy() == 0xEE).all()  # nothing past the output
    n = compare_whole_gather(oracle, w, host_pool, b.lens_host, _device_rows(out, w.row_bytes))
    assert n == T
    return out


@pytest.mark.parametrize("name", ["decode_gather", "prefix_sharing"])
def test_whole_gather(hp, oracle, name):
    """The decode-sized gather (64 sequences, 154,680 tokens of 8 KiB) and the
    prefix-sharing batch (128 sequences sharing 128 pages), every byte."""
    w = inputs.config(name, "full")
    b = Batch(w)
    _gather_whole(hp, oracle, w, b, b.host_pool())


def test_whole_decode_step_append_then_gather(hp, oracle):
    """The decode step at its stated size: 256 sequences of 1K-32K tokens each append one
    row (a new page when the count is a multiple of 16), validated.  The whole pool after
    the append equals the oracle's append on a host copy of the pool as it was; then the
    whole gather of the grown batch (4.37M tokens) equals the oracle's gather."""
    import torch
    w = inputs.config("decode_append", "full")
    b = Batch(w, lens=w.lens_before)
    host = b.pool.cpu().numpy()  # the pool before the append; the oracle appends into it
    rows = inputs.host_new_rows(w)
    rc = hp.hp_scatter_append(b.desc, torch.from_numpy(rows).to("cuda"),
                              index_tensor(w.new_ptr, "cuda"), w.total_new, b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0 and hp.status_name(b.status_value()) == "HP_OK"
    o = b.oracle_desc(pool_host=host, lens=w.lens_before)
    assert o.validate_append(w.new_ptr, w.total_new) == ("OK", 0)
    assert o.scatter_append(rows, w.new_ptr) == "OK"
    step = 16384  # pages per comparison (512 MiB)
    for p0 in range(0, w.num_pages, step):
        p1 = min(w.num_pages, p0 + step)
        assert np.array_equal(b.pool[p0:p1].cpu().numpy(), host[p0:p1]), (p0, p1)
    del o
    g = Batch(w, pool=b.pool)
    _gather_whole(hp, oracle, w, g, host)


def test_whole_dequant_gather(hp, oracle):
    """The int8 pool (400,000 pages of 32 slots, 13.1 GB) with fp32 per-slot scales,
    1024 sequences of 256-8192 tokens, u64 indices: all 4.24M bf16 rows."""
    import torch
    w = inputs.config("quantized_pool", "full")
    b = Batch(w)
    T = w.total_tokens
    E = w.num_heads * w.head_dim
    out = torch.full((T * E + 128,), -1, dtype=torch.int16, device="cuda")
    rc = hp.hp_gather_dequant(b.desc, out, T, b.ws, b.status)
    torch.cuda.synchronize()
    assert rc == 0 and hp.status_name(b.status_value()) == "HP_OK"
    assert (out[T * E:].cpu().numpy() == -1).all()
    host = b.pool.cpu().numpy()
    scales = b.scales.cpu().numpy()
    stats = {"rows": 0}

    def got_rows(r0, r1):
        g = out[r0 * E:r1 * E].cpu().numpy().view(np.uint16).reshape(r1 - r0, E)
        stats["rows"] += r1 - r0
        return g

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(host_threads()) as ex:
        for s0, s1, r0, r1 in sequence_groups(b.lens_host, 1 << 19):
            want = oracle_group(oracle, w, host, b.lens_host, s0, s1, ex, scales=scales)
            got = got_rows(r0, r1)
            gf = (got.astype(np.uint32) << 16).view(np.float32)
            wf = (want.astype(np.uint32) << 16).view(np.float32)
            assert np.all(np.abs(gf.astype(np.float64) - wf) <= 2.0 ** -8 * np.abs(wf)), (s0, s1)
            assert np.count_nonzero(got != want) == 0, (s0, s1)
    assert stats["rows"] == T


def test_whole_lane_snapshot(hp, oracle):
    """The per-lane workload (32 x 8 lanes of 8192 positions, 128 bf16 features, a
    random permutation table): every lane of the snapshot against the oracle."""
    import torch
    w = inputs.lane_synthetic()
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    pool = torch.randn(w.pool_shape, generator=g, device="cuda").to(torch.bfloat16)
    T = torch.from_numpy(w.table.view(np.int64).copy()).to("cuda")
    out = torch.empty((w.batch, w.kv_heads, w.n, w.width), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = hp.hp_lane_gather(pool, T, w.capacity, w.page_tokens, w.batch, w.kv_heads, w.width,
                           "bf16", w.n, out, st)
    torch.cuda.synchronize()
    assert rc == 0 and st.item() == 0
    host = pool.view(torch.int16).cpu().numpy()
    got = out.view(torch.int16).cpu().numpy()
    want = oracle.lane_gather(host, w.capacity, w.page_tokens, w.table, w.batch, w.kv_heads,
                              w.width, w.n)
    assert np.array_equal(got, want)


def test_whole_decode_attention(hp, oracle):
    """Decode attention over the decode step's grown batch (256 sequences, 32 query heads on
    8 K/V heads, bf16): every (sequence, query head) against the oracle's float64
    attention, each host thread taking one contiguous share of the sequences."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    w = inputs.config("decode_append", "full")
    Hq, D = 32, w.head_dim
    scale = 1.0 / np.sqrt(D)
    b = Batch(w)
    wv = inputs.Workload(**{**w.__dict__, "pool_seed": w.pool_seed + 77})
    vpool = inputs.device_pool(wv, "cuda")
    rng = np.random.default_rng(3)
    qt = torch.from_numpy(rng.standard_normal((w.num_seqs, Hq, D)).astype(np.float32)).to(
        torch.bfloat16)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, Hq)
    ws = torch.full((nws,), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full((w.num_seqs, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    rc = hp.hp_attention_decode(b.desc, vpool, qt.to("cuda"), Hq, scale, out, ws, b.status)
    torch.cuda.synchronize()
    assert hp.status_name(rc) == "HP_OK" and b.status_value() == 0
    got = out.cpu().numpy()
    # the tolerance's scale: the largest |V| among the value rows the batch reads
    live = torch.from_numpy(w.live_slots()).to("cuda")
    vmax = 0.0
    for p0 in range(0, w.num_pages, 20000):
        p1 = min(w.num_pages, p0 + 20000)
        v = vpool[p0:p1].view(torch.bfloat16).float().abs()
        keep = torch.arange(w.page_size, device="cuda")[None, :] < live[p0:p1, None]
        vmax = max(vmax, float((v * keep[:, :, None]).max()))
    kh = b.pool.cpu().numpy()
    vh = vpool.cpu().numpy()
    qh = qt.view(torch.int16).numpy().view(np.uint16)
    sp = w.seq_ptr.astype(np.int64)
    S = w.num_seqs
    cuts = np.linspace(0, S, min(S, host_threads() * 4) + 1).astype(np.int64)

    def one(k):
        a, c = int(cuts[k]), int(cuts[k + 1])
        if c <= a:
            return None
        sub = oracle.Desc(kh, w.table[sp[a]:sp[c]], (sp[a:c + 1] - sp[a]).astype(w.index_dtype),
                          w.lens[a:c], num_pages=w.num_pages, page_size=w.page_size,
                          num_heads=w.num_heads, head_dim=D, dtype=w.dtype, index_type=0)
        return a, c, sub.attention_decode(vh, np.ascontiguousarray(qh[a:c]), Hq, scale)

    tol = 1e-4 * vmax + 1e-6
    with ThreadPoolExecutor(host_threads()) as ex:
        for r in ex.map(one, range(len(cuts) - 1)):
            if r is None:
                continue
            a, c, want = r
            err = np.abs(got[a:c] - want)
            assert np.all(np.isfinite(got[a:c])) and err.max() <= tol, (a, c, err.max(), tol)
