"""GPU parity of hp_attention_decode (decode attention through the block table) against the
oracle's float64 attention.

Tolerance, derived from the fp32 path: each output is a convex combination of value rows,
so |out| <= max|V|; the kernel's errors come from fp32 dot products of head_dim terms,
a base-2 exponential with relative error below 2^-22, and fp32 accumulation over the
weighted rows of each sequence segment plus the merge of the segments' records -- a
relative error well under 1e-4 of max|V| (about n * 2^-24 for n terms in the worst
case; measured on GB300: 1e-8 to 3e-8 of max|V|, 2e-6 with a peaked softmax).  The bar is
|gpu - oracle| <= 1e-4 * max|V| + 1e-6 per element."""
import numpy as np
import pytest

from helpers import Batch, sub_batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu

KF = 0  # the kernel the current test asks for (HP_ATTN_TENSOR_CORES or HP_ATTN_CUDA_CORES)


@pytest.fixture(autouse=True, params=["tensor_cores", "cuda_cores"])
def attn_kernel(request, hp):
    """Every test here runs once on each kernel: the tensor-core kernel (where the shape
    allows it: head_dim 128, 1, 2, 4 or 8 K/V heads, at most 32 query heads, pages of 8 to
    128 / H_kv slots; the others fall back to the CUDA cores) and the CUDA-core kernel."""
    global KF
    KF = hp.ATTN_TENSOR_CORES if request.param == "tensor_cores" else hp.ATTN_CUDA_CORES
    yield request.param


def _run(hp, oracle, w, Hq, seed, scale=None):
    import torch
    D = w.head_dim
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    b = Batch(w, flags=KF)
    wv = inputs.Workload(**{**w.__dict__, "pool_seed": w.pool_seed + 77})
    vpool = inputs.device_pool(wv, "cuda")
    rng = np.random.default_rng(seed)
    qf = rng.standard_normal((w.num_seqs, Hq, D)).astype(np.float32)
    if w.dtype == "bf16":
        qt = torch.from_numpy(qf).to(torch.bfloat16)
    else:
        qt = torch.from_numpy(qf.astype(np.float16))
    q = qt.to("cuda")
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, Hq)
    # the workspace holds no state between calls: start from garbage, then reuse it
    ws = torch.full((nws,), 0xFF, dtype=torch.uint8, device="cuda")
    results = []
    for _ in range(2):
        out = torch.full((w.num_seqs, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        rc = hp.hp_attention_decode(b.desc, vpool, q, Hq, scale, out, ws, b.status)
        torch.cuda.synchronize()
        assert hp.status_name(rc) == "HP_OK" and b.status_value() == 0
        results.append(out.cpu().numpy())
    # the segments are merged in a fixed order, whichever warp finishes last
    assert np.array_equal(results[0].view(np.uint32), results[1].view(np.uint32))
    return b, vpool, qt, results[0], scale


def _check(got, want, vmax):
    tol = 1e-4 * vmax + 1e-6
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)) and err.max() <= tol, (err.max(), tol)


@pytest.mark.parametrize("dtype,Hkv,G,D,P,scale", [
    ("bf16", 8, 4, 128, 16, None), ("f16", 8, 4, 128, 16, None), ("bf16", 2, 1, 64, 8, None),
    ("bf16", 4, 2, 256, 5, None), ("f16", 3, 8, 128, 3, None), ("bf16", 12, 1, 128, 32, None),
    ("bf16", 2, 8, 256, 16, None), ("f16", 2, 8, 64, 16, None), ("f16", 1, 4, 64, 1, None),
    ("bf16", 8, 4, 128, 16, 1.5),  # peaked softmax: a few tokens carry the weight
    # the tensor-core kernel's other shapes: its steps are 128 / H_kv tokens of every K/V
    # head, so these have 8, 1, 1, 2 and 1 pages per step and 1, 2, 4 or 8 heads
    ("bf16", 2, 8, 128, 8, None), ("f16", 2, 2, 128, 64, None), ("bf16", 1, 1, 128, 128, None),
    ("bf16", 4, 8, 128, 8, None), ("f16", 4, 2, 128, 32, None), ("bf16", 1, 8, 128, 16, None),
    ("bf16", 8, 2, 128, 8, None),  # 8 K/V heads on pages of 8 slots: two pages per step
])
def test_attention_matches_oracle(hp, oracle, dtype, Hkv, G, D, P, scale):
    # lengths up to ~1300 tokens: small pages move the 32-page window many times
    w = inputs.decode_gather(seed=Hkv * 10 + G + D + P, num_pages=4000, page_size=P,
                             num_heads=Hkv, head_dim=D, num_seqs=5, len_lo=0, len_hi=1300,
                             dtype=dtype, index_dtype=np.uint32 if P % 2 == 0 else np.uint64)
    Hq = Hkv * G
    b, vpool, qt, got, scale = _run(hp, oracle, w, Hq, seed=P, scale=scale)
    kh = b.host_pool()
    vh = vpool.cpu().numpy()
    od = b.oracle_desc(pool_host=kh)
    qh = qt.view(torch_int16()).numpy().view(np.uint16)
    want = od.attention_decode(vh, qh, Hq, scale)
    _check(got, want, _vmax_read(od, vh, dtype))
    for s in range(w.num_seqs):
        if int(w.lens[s]) == 0:
            assert (got[s] == 0).all()


def _tc_shapes():
    """Every shape the tensor-core kernel takes: 1, 2, 4 or 8 K/V heads, G in {1, 2, 4, 8}
    with at most 32 query heads, pages of a power of two from 8 to 128 / H_kv slots."""
    out = []
    for hkv in (1, 2, 4, 8):
        for g in (1, 2, 4, 8):
            if hkv * g > 32:
                continue
            p = 8
            while p <= 128 // hkv:
                out.append((hkv, g, p))
                p *= 2
    return out


def _tc_pair_shapes():
    """Head_dim 64 shapes the tensor-core kernel takes in pairs of K/V heads: 2, 4, 8 or 16
    K/V heads, G in {1, 2, 4} with at most 32 query heads, pages from 8 to 256 / H_kv."""
    out = []
    for hkv in (2, 4, 8, 16):
        for g in (1, 2, 4):
            if hkv * g > 32:
                continue
            p = 8
            while p <= 256 // hkv:
                out.append((hkv, g, p))
                p *= 2
    return out


@pytest.mark.parametrize("Hkv,G,P", _tc_pair_shapes())
def test_attention_every_head_dim_64_pair_shape(hp, oracle, Hkv, G, P):
    """Head_dim 64 on each shape the tensor-core kernel takes as pairs of K/V heads (and on
    the CUDA-core kernel), small ragged batches, element type and index width alternating."""
    import torch
    dtype = "bf16" if (Hkv + G + P) % 2 == 0 else "f16"
    index_dtype = np.uint64 if (Hkv * G + P // 8) % 2 == 1 else np.uint32
    w = inputs.decode_gather(seed=Hkv * 100 + G * 10 + P + 7, num_pages=1200, page_size=P,
                             num_heads=Hkv, head_dim=64, num_seqs=4, len_lo=0, len_hi=600,
                             dtype=dtype, index_dtype=index_dtype)
    Hq = Hkv * G
    b, vpool, qt, got, scale = _run(hp, oracle, w, Hq, seed=P + G + 1)
    kh = b.host_pool()
    vh = vpool.cpu().numpy()
    od = b.oracle_desc(pool_host=kh)
    want = od.attention_decode(vh, qt.view(torch_int16()).numpy().view(np.uint16), Hq, scale)
    _check(got, want, _vmax_read(od, vh, dtype))


@pytest.mark.parametrize("Hkv,G,D,P", [
    (8, 8, 128, 16), (16, 4, 128, 8), (16, 8, 128, 16), (32, 2, 128, 16),
    (16, 4, 64, 16), (32, 2, 64, 8), (8, 8, 64, 16),
])
def test_attention_more_than_32_query_heads(hp, oracle, Hkv, G, D, P):
    """More than 32 query heads: the tensor-core kernel runs once per group of K/V heads with
    at most 32 query heads (2 or 4 groups here; head_dim 64 in pairs first), each launch on
    its heads' slice of the pool rows, the queries and the output (head_dim 64 at G = 8 stays
    on the CUDA cores).  Small ragged batches against the oracle."""
    import torch
    dtype = "bf16" if (Hkv + G) % 2 == 0 else "f16"
    w = inputs.decode_gather(seed=Hkv * 10 + G + D + P, num_pages=2000, page_size=P,
                             num_heads=Hkv, head_dim=D, num_seqs=5, len_lo=0, len_hi=700,
                             dtype=dtype, index_dtype=np.uint64 if G == 2 else np.uint32)
    Hq = Hkv * G
    b, vpool, qt, got, scale = _run(hp, oracle, w, Hq, seed=Hq + P)
    kh = b.host_pool()
    vh = vpool.cpu().numpy()
    od = b.oracle_desc(pool_host=kh)
    want = od.attention_decode(vh, qt.view(torch_int16()).numpy().view(np.uint16), Hq, scale)
    _check(got, want, _vmax_read(od, vh, dtype))


@pytest.mark.parametrize("Hkv,G,P", _tc_shapes())
def test_attention_every_tensor_core_shape(hp, oracle, Hkv, G, P):
    """Each supported (K/V heads, query heads per K/V head, page size) on a small ragged
    batch (lengths 0 to about 600, so partial last steps and empty sequences), element
    type and index width alternating, on whichever kernel the fixture asks for: the
    tensor-core kernel takes every one of these shapes."""
    import torch
    dtype = "bf16" if (Hkv + G + P) % 2 == 0 else "f16"
    index_dtype = np.uint64 if (Hkv * G + P // 8) % 2 == 1 else np.uint32
    w = inputs.decode_gather(seed=Hkv * 100 + G * 10 + P, num_pages=1200, page_size=P,
                             num_heads=Hkv, head_dim=128, num_seqs=4, len_lo=0, len_hi=600,
                             dtype=dtype, index_dtype=index_dtype)
    Hq = Hkv * G
    b, vpool, qt, got, scale = _run(hp, oracle, w, Hq, seed=P + G)
    kh = b.host_pool()
    vh = vpool.cpu().numpy()
    od = b.oracle_desc(pool_host=kh)
    want = od.attention_decode(vh, qt.view(torch_int16()).numpy().view(np.uint16), Hq, scale)
    _check(got, want, _vmax_read(od, vh, dtype))


def torch_int16():
    import torch
    return torch.int16


def _vmax_read(od, vh, dtype):
    """Largest |V| among the value rows the batch reads (the oracle's gather of V)."""
    import torch
    keep = od.pool
    od.pool = vh
    od.c.page_pool = vh.ctypes.data
    rows = od.gather()[0]
    od.pool = keep
    od.c.page_pool = keep.ctypes.data
    if rows.size == 0:
        return 0.0
    t = torch.from_numpy(rows.reshape(-1).view(np.int16).copy())
    f = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).float().numpy()
    return float(np.abs(f).max())


def test_attention_single_token_and_empty(hp, oracle):
    """A one-token sequence returns its value row (the weight is 1); an empty one zeros."""
    import torch
    w = inputs.decode_gather(seed=5, num_pages=50, page_size=16, num_heads=2, head_dim=128,
                             num_seqs=3, len_lo=1, len_hi=40, dtype="bf16")
    lens = w.lens.copy()
    lens[0], lens[2] = 1, 0
    w = inputs.Workload(**{**w.__dict__, "lens": lens})
    b, vpool, qt, got, scale = _run(hp, oracle, w, 4, seed=1)
    page = int(w.table[0])
    vrow = torch.from_numpy(vpool.cpu().numpy()[page, 0].view(np.int16).copy()).view(
        torch.bfloat16).float().numpy().reshape(2, 128)
    for qh in range(4):
        np.testing.assert_allclose(got[0, qh], vrow[qh // 2], rtol=0, atol=1e-6)
    assert (got[2] == 0).all()


def test_attention_full_size_sampled(hp, oracle):
    """The decode step's grown batch (256 sequences up to 32k tokens, 8 K/V heads, 32 query
    heads, bf16): a few whole sequences against the oracle."""
    import torch
    w = inputs.config("decode_append", "full")
    b, vpool, qt, got, scale = _run(hp, oracle, w, 32, seed=3)
    seqs = [0, 77, 255]
    table, seq_ptr, lens = sub_batch(w, seqs)
    kh = b.pool.cpu().numpy()
    vh = vpool.cpu().numpy()
    sub = oracle.Desc(kh, table, seq_ptr, lens, num_pages=w.num_pages, page_size=16,
                      num_heads=8, head_dim=128, dtype="bf16", index_type=0)
    qh = qt.view(torch.int16).numpy().view(np.uint16)[seqs]
    want = sub.attention_decode(vh, qh, 32, scale)
    _check(got[seqs], want, _vmax_read(sub, vh, "bf16"))


def test_attention_rejections(hp, oracle):
    import torch
    w = inputs.config("decode_gather", "small")   # 32 heads of 128, fp16
    b = Batch(w, flags=KF)
    rc, n = hp.hp_attention_decode_workspace_bytes(b.desc, 32)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    q = torch.zeros((w.num_seqs, 48, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((w.num_seqs, 48, 128), dtype=torch.float32, device="cuda")
    assert hp.status_name(hp.hp_attention_decode(b.desc, b.pool, q, 48, 1.0, out, ws)) == \
        "HP_ERR_ARG"   # 48 query heads over 32 K/V heads
    assert hp.status_name(hp.hp_attention_decode(b.desc, b.pool, q, 32, 1.0, out, ws[:100])) == \
        "HP_ERR_WORKSPACE"


def test_attention_one_long_sequence_split_over_many_warps(hp, oracle):
    """One sequence of 30,000 tokens: the step space is shared by every CTA, so the
    sequence is cut into hundreds of segments whose records the last warp to finish merges."""
    import torch
    table = np.random.default_rng(3).permutation(2000)[:1875].astype(np.uint32)
    w = inputs.Workload("long", 2000, 16, 2, 128, "bf16", np.uint32, table,
                        np.array([0, 1875], np.uint32), np.array([30000], np.uint32), 5, "normal")
    b, vpool, qt, got, scale = _run(hp, oracle, w, 8, seed=4)
    od = b.oracle_desc()
    want = od.attention_decode(vpool.cpu().numpy(), qt.view(torch.int16).numpy().view(np.uint16),
                               8, scale)
    _check(got, want, _vmax_read(od, vpool.cpu().numpy(), "bf16"))


@pytest.mark.parametrize("D", [64, 128])
def test_attention_mostly_empty_batch(hp, oracle, D):
    """600 sequences, all but three empty (the first and the last nine among them): empty
    ones give zeros, the others match (head_dim 128 reaches the tensor-core kernel)."""
    import torch
    rng = np.random.default_rng(8)
    lens = np.zeros(600, np.uint32)
    lens[[5, 300, 590]] = [17, 700, 1]
    pages = -(-lens.astype(np.int64) // 16)
    sp = np.concatenate([[0], np.cumsum(pages)]).astype(np.uint32)
    table = rng.permutation(400)[:int(sp[-1])].astype(np.uint32)
    w = inputs.Workload("sparse", 400, 16, 4, D, "f16", np.uint32, table, sp, lens, 6, "normal")
    b, vpool, qt, got, scale = _run(hp, oracle, w, 8, seed=5)
    od = b.oracle_desc()
    want = od.attention_decode(vpool.cpu().numpy(), qt.view(torch.int16).numpy().view(np.uint16),
                               8, scale)
    _check(got, want, _vmax_read(od, vpool.cpu().numpy(), "f16"))
    assert (got[lens == 0] == 0).all()


@pytest.mark.parametrize("fault", ["page_id", "len"])
def test_attention_validates_permissive_descriptors(hp, oracle, fault):
    """HP_PERMISSIVE does not reach decode attention: a block-table entry naming a page
    outside the pool, or a token count beyond the slice, is rejected by the validation
    (the rule's code in the status word) and nothing is read or written."""
    import torch
    w = inputs.decode_gather(seed=12, num_pages=200, page_size=16, num_heads=2, head_dim=64,
                             num_seqs=4, len_lo=20, len_hi=300, dtype="bf16")
    pool = inputs.device_pool(w, "cuda")  # drawn from the well-formed batch
    table, lens = w.table.copy(), w.lens.copy()
    if fault == "page_id":
        table[int(w.seq_ptr[2])] = w.num_pages + 7
    else:
        lens[1] = (int(w.seq_ptr[2]) - int(w.seq_ptr[1])) * 16 + 1
    w = inputs.Workload(**{**w.__dict__, "table": table, "lens": lens})
    b = Batch(w, pool=pool, flags=hp.PERMISSIVE | KF)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, 4)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    q = torch.zeros((w.num_seqs, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((w.num_seqs, 4, 64), float("nan"), dtype=torch.float32, device="cuda")
    rc = hp.hp_attention_decode(b.desc, b.pool, q, 4, 0.125, out, ws, b.status)
    torch.cuda.synchronize()
    assert hp.status_name(rc) == "HP_OK"
    want = "HP_ERR_PAGE_ID" if fault == "page_id" else "HP_ERR_LEN"
    assert hp.status_name(b.status_value()) == want
    assert torch.isnan(out).all()


@pytest.mark.parametrize("dtype,Hkv,G,D", [("bf16", 4, 4, 128), ("f16", 2, 8, 256),
                                           ("bf16", 8, 1, 64), ("f16", 12, 2, 128)])
def test_planned_attention_over_layers(hp, oracle, dtype, Hkv, G, D):
    """One hp_attention_plan, then planned calls for three "layers" (their own K and V
    pools and queries through the same table): each equals the one-call result bit for
    bit, so the segment counts are back at zero after every planned call."""
    import torch
    w = inputs.decode_gather(seed=31 + D + G, num_pages=3000, page_size=16, num_heads=Hkv,
                             head_dim=D, num_seqs=6, len_lo=0, len_hi=2500, dtype=dtype)
    Hq = Hkv * G
    b = Batch(w, flags=KF)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, Hq)
    ws_plan = torch.full((nws,), 0xFF, dtype=torch.uint8, device="cuda")
    ws_one = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    layers = []
    for layer in range(3):
        kl = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 500 + layer}), "cuda")
        vl = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": 600 + layer}), "cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(700 + layer)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        ql = torch.randn((w.num_seqs, Hq, D), generator=g, device="cuda").to(tdt)
        layers.append((kl, vl, ql))
    assert hp.hp_attention_plan(b.desc, Hq, ws_plan, b.status) == 0
    for kl, vl, ql in layers:
        dl = hp.PagedDesc(kl, b.table, b.seq_ptr, b.lens, num_pages=w.num_pages, page_size=16,
                          num_heads=Hkv, head_dim=D, dtype=dtype, index_type=b.it, flags=KF)
        got = torch.full((w.num_seqs, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        want = torch.full_like(got, float("nan"))
        assert hp.hp_attention_decode_planned(dl, vl, ql, Hq, 0.09, got, ws_plan, b.status) == 0
        assert hp.hp_attention_decode(dl, vl, ql, Hq, 0.09, want, ws_one, b.status) == 0
        torch.cuda.synchronize()
        assert b.status_value() == 0
        assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    # and the last layer against the oracle
    od = oracle.Desc(kl.cpu().numpy(), w.table, w.seq_ptr, w.lens, num_pages=w.num_pages,
                     page_size=16, num_heads=Hkv, head_dim=D, dtype=dtype, index_type=b.it)
    vh = vl.cpu().numpy()
    wantd = od.attention_decode(vh, ql.view(torch.int16).cpu().numpy().view(np.uint16), Hq, 0.09)
    _check(got.cpu().numpy(), wantd, _vmax_read(od, vh, dtype))


def test_planned_attention_after_a_failed_plan_writes_nothing(hp, oracle):
    import torch
    w = inputs.decode_gather(seed=32, num_pages=200, page_size=16, num_heads=2, head_dim=64,
                             num_seqs=3, len_lo=20, len_hi=300, dtype="bf16")
    pool = inputs.device_pool(w, "cuda")
    table = w.table.copy()
    table[0] = w.num_pages
    w = inputs.Workload(**{**w.__dict__, "table": table})
    b = Batch(w, pool=pool, flags=KF)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, 4)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    q = torch.zeros((w.num_seqs, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((w.num_seqs, 4, 64), float("nan"), dtype=torch.float32, device="cuda")
    assert hp.hp_attention_plan(b.desc, 4, ws, b.status) == 0
    assert hp.hp_attention_decode_planned(b.desc, pool, q, 4, 0.125, out, ws, b.status) == 0
    torch.cuda.synchronize()
    assert hp.status_name(b.status_value()) == "HP_ERR_PAGE_ID"
    assert torch.isnan(out).all()
