"""GPU parity of hp_gather_dequant_q ([HF] Per-scheme composition: per-tensor,
per-channel on num_heads or head_dim, per-block-affine = per page slot; symmetric or with
zero points; int8 or uint8 codes) against the oracle.  Bar: |Δ| <= 2^-8 |ref| and no
bit differences expected (both sides round the exact product once)."""
import zlib

import numpy as np
import pytest

from helpers import Batch
from paged_kv_cache_hp_gb300 import inputs
from test_gpu_dequant import check_close

pytestmark = pytest.mark.gpu

SCHEMES = {"tensor": (0x01, 0), "head": (0x02, 1), "dim": (0x02, 2), "slot": (0x03, 0)}


def _params(rng, w, scheme, asym, dtype):
    count = {"tensor": 1, "head": w.num_heads, "dim": w.head_dim,
             "slot": w.num_pages * w.page_size}[scheme]
    scales = rng.uniform(0.001, 0.05, count).astype(np.float32)
    zp = None
    if asym:
        lo, hi = (-30, 30) if dtype == "i8" else (90, 170)
        zp = rng.integers(lo, hi, count).astype(np.int8 if dtype == "i8" else np.uint8)
    return scales, zp


def _run(hp, oracle, w, scheme, asym, dtype, seed):
    import torch
    rng = np.random.default_rng(seed)
    b = Batch(w)
    if dtype == "u8":  # same bytes, read as unsigned codes
        b.desc.c.dtype = hp.DTYPES["u8"]
    scales, zp = _params(rng, w, scheme, asym, dtype)
    tag, axis = SCHEMES[scheme]
    bs = w.page_size if scheme == "slot" else 0
    sd = torch.from_numpy(scales).to("cuda")
    zd = None if zp is None else torch.from_numpy(zp.view(np.uint8)).to("cuda")
    q = hp.quant_desc(tag, sd, zd, axis=axis, block_size=bs)
    T = w.total_tokens
    E = w.num_heads * w.head_dim
    out = torch.full((T * E + 64,), -1, dtype=torch.int16, device="cuda")
    rc = hp.hp_gather_dequant_q(b.desc, q, out, T, b.ws, b.status)
    torch.cuda.synchronize()
    assert hp.status_name(rc) == "HP_OK" and b.status_value() == 0
    o = out.cpu().numpy().view(np.uint16)
    assert (o[T * E:] == 0xFFFF).all()
    od = b.oracle_desc()
    od.c.dtype = 3 if dtype == "i8" else 4
    oq = oracle.Desc.quant(tag, scales, zp, axis=axis, block_size=bs)
    assert od.validate_quant(oq) == "OK"
    want, written, fault = od.gather_dequant_q(oq)
    assert fault == "OK" and written.all()
    return o[:T * E].reshape(T, E), want


@pytest.mark.parametrize("scheme", list(SCHEMES))
@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("dtype", ["i8", "u8"])
def test_schemes_small(hp, oracle, scheme, asym, dtype):
    w = inputs.config("quantized_pool", "small")
    seed = zlib.crc32(repr((scheme, asym, dtype)).encode())
    got, want = _run(hp, oracle, w, scheme, asym, dtype, seed)
    assert check_close(got, want) == 0


@pytest.mark.parametrize("H,D,P", [(3, 5, 4), (2, 12, 3), (4, 8, 1), (1, 24, 7), (3, 16, 4),
                                   (6, 32, 5), (5, 48, 3), (2, 16, 8), (8, 256, 32)])
@pytest.mark.parametrize("scheme", list(SCHEMES))
def test_schemes_shapes(hp, oracle, H, D, P, scheme):
    """Rows or heads that do not split into groups of 8 take the element-wise path, the
    others 8-code groups -- with per-channel parameters read once per thread when a row's
    group count divides the CTA's 256 threads (4 and 256 groups) and per group
    otherwise (6, 24 and 30 groups)."""
    w = inputs.quantized_pool(seed=H * 100 + D + P, num_pages=400, page_size=P, num_heads=H,
                              head_dim=D, num_seqs=5, len_lo=0, len_hi=60,
                              index_dtype=np.uint32 if P % 2 else np.uint64)
    got, want = _run(hp, oracle, w, scheme, True, "i8", H * D * P)
    assert check_close(got, want) == 0


def test_per_channel_full_size_sampled(hp, oracle):
    """The full int8 pool (400,000 pages, 1024 sequences, u64) under per-channel
    head_dim scales with zero points: random elements against the oracle's lookup."""
    import torch
    w = inputs.config("quantized_pool", "full")
    rng = np.random.default_rng(77)
    b = Batch(w)
    scales, zp = _params(rng, w, "dim", True, "i8")
    q = hp.quant_desc(0x02, torch.from_numpy(scales).to("cuda"),
                      torch.from_numpy(zp.view(np.uint8)).to("cuda"), axis=2)
    T, E = w.total_tokens, w.num_heads * w.head_dim
    out = torch.empty(T * E, dtype=torch.int16, device="cuda")
    assert hp.hp_gather_dequant_q(b.desc, q, out, T, b.ws, b.status) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    got = out.view(T, E)
    od = b.oracle_desc()
    oq = oracle.Desc.quant(0x02, scales, zp, axis=2)
    tok_off = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))])
    rows, cols, wants = [], [], []
    for _ in range(4000):
        s = int(rng.integers(0, w.num_seqs))
        t = int(rng.integers(0, int(w.lens[s])))
        e = int(rng.integers(0, E))
        code, v = od.lookup_dequant_q(oq, s, t, e // w.head_dim, e % w.head_dim)
        assert code == "OK"
        rows.append(tok_off[s] + t)
        cols.append(e)
        wants.append(v)
    g = got[torch.tensor(rows, device="cuda"), torch.tensor(cols, device="cuda")]
    assert check_close(g.cpu().numpy().view(np.uint16), np.array(wants, np.uint16)) == 0


@pytest.mark.parametrize("kw,want", [
    (dict(scheme_tag=0x03, axis=1, block_size=32, count=48000), "HP_ERR_QUANT_BLOCK"),
    (dict(scheme_tag=0x03, axis=0, block_size=16, count=48000), "HP_ERR_QUANT_BLOCK"),
    (dict(scheme_tag=0x03, axis=0, block_size=32, count=47999), "HP_ERR_SCALES"),
    (dict(scheme_tag=0x02, axis=0, count=8), "HP_ERR_QUANT_SCHEME"),
    (dict(scheme_tag=0x02, axis=1, count=9), "HP_ERR_SCALES"),
    (dict(scheme_tag=0x05, count=1), "HP_ERR_QUANT_SCHEME"),
    (dict(scheme_tag=0x01, count=1), "HP_OK"),
])
def test_scheme_rules_match_oracle(hp, oracle, kw, want):
    import torch
    w = inputs.config("quantized_pool", "small")
    b = Batch(w)
    sc = torch.ones(max(kw["count"], 1), dtype=torch.float32, device="cuda")
    q = hp.quant_desc(kw["scheme_tag"], sc, None, axis=kw.get("axis", 0),
                      block_size=kw.get("block_size", 0), count=kw["count"])
    T = w.total_tokens
    out = torch.empty(T * w.num_heads * w.head_dim, dtype=torch.int16, device="cuda")
    rc = hp.hp_gather_dequant_q(b.desc, q, out, T, b.ws, b.status)
    assert hp.status_name(rc) == want
    oq = oracle.Desc.quant(kw["scheme_tag"], sc.cpu().numpy(), None, axis=kw.get("axis", 0),
                           block_size=kw.get("block_size", 0), count=kw["count"])
    name = b.oracle_desc().validate_quant(oq)
    assert want == ("HP_OK" if name == "OK" else "HP_ERR_" + name)
