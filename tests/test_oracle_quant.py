"""Pins the oracle's quantization schemes ([HF] Quantization Compatibility, Per-scheme
composition) to the specification's sentences and to exact rational arithmetic."""
import itertools
import zlib
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_pins import _exact_bf16


def _batch(rng, dtype="i8", N=6, P=4, H=3, D=5):
    lens = [7, 0, 11, 4]
    table, sp = [], [0]
    free = list(rng.permutation(N))
    for n in lens:
        k = -(-n // P)
        table += [int(free.pop()) for _ in range(k)] if len(free) >= k else [0] * k
        sp.append(len(table))
    lo, hi = (-128, 127) if dtype == "i8" else (0, 255)
    npdt = np.int8 if dtype == "i8" else np.uint8
    pool = rng.integers(lo, hi, (N, P, H, D), endpoint=True).astype(npdt)
    return pool, table, sp, lens


def _desc(oracle, pool, table, sp, lens, dtype):
    N, P, H, D = pool.shape
    return oracle.Desc(pool, table, sp, lens, num_pages=N, page_size=P, num_heads=H, head_dim=D,
                       dtype=dtype, index_type=0)


@pytest.mark.parametrize("kw,want", [
    (dict(scheme_tag=0x03, axis=0, block_size=4, count=24), "OK"),
    (dict(scheme_tag=0x03, axis=1, block_size=4, count=24), "QUANT_BLOCK"),  # axis must be 0
    (dict(scheme_tag=0x03, axis=2, block_size=4, count=24), "QUANT_BLOCK"),
    (dict(scheme_tag=0x03, axis=0, block_size=8, count=24), "QUANT_BLOCK"),  # != page_size
    (dict(scheme_tag=0x03, axis=0, block_size=4, count=6), "SCALES"),   # shape/block_size: no
    (dict(scheme_tag=0x01, count=1), "OK"),
    (dict(scheme_tag=0x01, count=2), "SCALES"),
    (dict(scheme_tag=0x02, axis=1, count=3), "OK"),                      # num_heads channels
    (dict(scheme_tag=0x02, axis=2, count=5), "OK"),                      # head_dim channels
    (dict(scheme_tag=0x02, axis=2, count=3), "SCALES"),
    (dict(scheme_tag=0x02, axis=0, count=24), "QUANT_SCHEME"),           # paged axis: never
    (dict(scheme_tag=0x02, axis=3, count=5), "QUANT_SCHEME"),
    (dict(scheme_tag=0x00, count=1), "QUANT_SCHEME"),
    (dict(scheme_tag=0x04, count=1), "QUANT_SCHEME"),
    (dict(scheme_tag=0x01, count=1, addrs={"scales": 0}), "NULL"),
    (dict(scheme_tag=0x01, count=1, addrs={"scales": 64 + 4}), "ALIGN"),
    (dict(scheme_tag=0x01, count=1, zp=True, addrs={"zero_points": 64 + 1}), "ALIGN"),
])
def test_scheme_rules(oracle, kw, want):
    rng = np.random.default_rng(0)
    pool, table, sp, lens = _batch(rng)
    d = _desc(oracle, pool, table, sp, lens, "i8")
    kw = dict(kw)
    n = kw["count"]
    zp = np.zeros(max(n, 1), np.int8) if kw.pop("zp", False) else None
    q = oracle.Desc.quant(kw.pop("scheme_tag"), np.ones(max(n, 1), np.float32), zp, **kw)
    assert d.validate_quant(q) == want


def test_scheme_needs_an_8bit_pool(oracle):
    rng = np.random.default_rng(0)
    pool, table, sp, lens = _batch(rng)
    d = _desc(oracle, pool.astype(np.float16), table, sp, lens, "f16")
    q = oracle.Desc.quant(0x01, np.ones(1, np.float32))
    assert d.validate_quant(q) == "DTYPE"


@pytest.mark.parametrize("dtype", ["i8", "u8"])
@pytest.mark.parametrize("scheme", ["tensor", "head", "dim", "slot"])
@pytest.mark.parametrize("asym", [False, True])
def test_scheme_values_are_the_exact_affine_product_rounded_once(oracle, dtype, scheme, asym):
    """Each element equals the bfloat16 nearest (q - zp) * scale, computed with exact
    rationals; the parameter entry comes from numpy broadcasting over the [T, H, D]
    output (tensor: one; head: axis 1; dim: axis 2; slot: the row's page slot)."""
    rng = np.random.default_rng(zlib.crc32(repr((dtype, scheme, asym)).encode()))
    pool, table, sp, lens = _batch(rng, dtype)
    N, P, H, D = pool.shape
    d = _desc(oracle, pool, table, sp, lens, dtype)
    count = {"tensor": 1, "head": H, "dim": D, "slot": N * P}[scheme]
    scales = rng.uniform(0.001, 0.05, count).astype(np.float32)
    npdt = pool.dtype
    zp = None
    if asym:
        lo, hi = (-20, 20) if dtype == "i8" else (100, 150)
        zp = rng.integers(lo, hi, count).astype(npdt)
    tag, axis, bs = {"tensor": (1, 0, 0), "head": (2, 1, 0), "dim": (2, 2, 0),
                     "slot": (3, 0, P)}[scheme]
    q = oracle.Desc.quant(tag, scales, zp, axis=axis, block_size=bs)
    assert d.validate_quant(q) == "OK"
    out, written, fault = d.gather_dequant_q(q)
    assert fault == "OK" and written.all()
    got = (out.astype(np.uint32) << 16).view(np.float32).reshape(-1, H, D)
    # the (page, slot) of each output row, then each element's parameter index
    rows = [(table[sp[s] + t // P], t % P) for s, n in enumerate(lens) for t in range(n)]
    T = len(rows)
    assert got.shape[0] == T
    for r, (page, slot) in enumerate(rows):
        for h, e in itertools.product(range(H), range(D)):
            k = {"tensor": 0, "head": h, "dim": e, "slot": page * P + slot}[scheme]
            z = 0 if zp is None else int(zp[k])
            exact = (int(pool[page, slot, h, e]) - z) * Fraction(float(scales[k]))
            assert got[r, h, e] == _exact_bf16(exact), (r, h, e)


def test_per_block_affine_symmetric_is_the_per_slot_dequant(oracle):
    """With axis 0, block_size = page_size and no zero points the scheme is the
    per-page-slot dequantisation of [HF] Per-page-slot parameters."""
    rng = np.random.default_rng(5)
    pool, table, sp, lens = _batch(rng)
    N, P, H, D = pool.shape
    scales = rng.uniform(0.001, 0.05, N * P).astype(np.float32)
    d = oracle.Desc(pool, table, sp, lens, num_pages=N, page_size=P, num_heads=H, head_dim=D,
                    dtype="i8", scales=scales, flags=oracle.HAS_QUANT, index_type=0)
    q = oracle.Desc.quant(0x03, scales, None, axis=0, block_size=P)
    assert np.array_equal(d.gather_dequant_q(q)[0], d.gather_dequant()[0])


def test_uint8_with_midpoint_zero_point_and_unit_scale(oracle):
    """uint8 codes with zero point 128 and scale 1 give the integers q - 128, exactly."""
    rng = np.random.default_rng(6)
    pool, table, sp, lens = _batch(rng, "u8")
    N, P, H, D = pool.shape
    d = _desc(oracle, pool, table, sp, lens, "u8")
    q = oracle.Desc.quant(0x01, np.ones(1, np.float32), np.full(1, 128, np.uint8))
    out = d.gather_dequant_q(q)[0]
    got = (out.astype(np.uint32) << 16).view(np.float32).reshape(-1, H, D)
    rows = [(table[sp[s] + t // P], t % P) for s, n in enumerate(lens) for t in range(n)]
    want = np.stack([pool[p, sl].astype(np.int32) - 128 for p, sl in rows])
    assert np.array_equal(got, want.astype(np.float32))
