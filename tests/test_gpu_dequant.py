"""GPU parity: hp_gather_dequant (int8 pool, fp32 per-page-slot scales -> bf16).

Bar: |gpu - oracle| <= 2^-8 * |oracle| per element.  The oracle rounds the exact
product once; the kernel computes the same correctly rounded value, so the tests
also count elements that differ at all and expect none.
"""
import numpy as np
import pytest

from helpers import Batch, sub_batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def bf16_to_f64(u16):
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def check_close(got_u16, want_u16):
    g, w = bf16_to_f64(got_u16), bf16_to_f64(want_u16)
    assert np.all(np.abs(g - w) <= 2.0 ** -8 * np.abs(w)), "outside 2^-8 |ref|"
    return int(np.count_nonzero(got_u16 != want_u16))


def run_dequant(hp, b, out_tokens=None):
    import torch
    w = b.w
    T = w.total_tokens if out_tokens is None else out_tokens
    out = torch.full((T * w.num_heads * w.head_dim + 128,), -1, dtype=torch.int16, device="cuda")
    rc = hp.hp_gather_dequant(b.desc, out, T, b.ws, b.status)
    torch.cuda.synchronize()
    o = out.cpu().numpy().view(np.uint16)
    assert (o[T * w.num_heads * w.head_dim:] == 0xFFFF).all()  # nothing past the output
    return rc, o[:T * w.num_heads * w.head_dim].reshape(T, -1)


def test_dequant_small_config(hp, oracle):
    w = inputs.config("quantized_pool", "small")
    b = Batch(w)
    rc, got = run_dequant(hp, b)
    assert rc == 0 and b.status_value() == 0
    want, written, fault = b.oracle_desc().gather_dequant()
    assert fault == "OK" and written.all()
    assert check_close(got, want) == 0


@pytest.mark.parametrize("H,D,P", [(1, 3, 4), (3, 5, 2), (2, 8, 7), (1, 16, 1), (4, 32, 32),
                                   (8, 256, 32), (32, 512, 4), (32, 1024, 2), (3, 48, 5)])
def test_dequant_shapes(hp, oracle, H, D, P):
    """Rows that are not a multiple of 8 elements take the element-wise path, the others
    8-code groups; copy units from 3 rows of 3 codes to 64 KiB pages (8 heads of 256 codes
    x 32 slots, 32 heads of 512 x 4) and rows of 32 KiB."""
    w = inputs.quantized_pool(seed=H * 10 + D + P, num_pages=500, page_size=P, num_heads=H,
                              head_dim=D, num_seqs=5, len_lo=0, len_hi=70,
                              index_dtype=np.uint32 if P % 2 else np.uint64)
    b = Batch(w)
    rc, got = run_dequant(hp, b)
    assert rc == 0 and b.status_value() == 0
    want = b.oracle_desc().gather_dequant()[0]
    assert check_close(got, want) == 0


def _tie_scales(rng, n, oracle):
    """(q, scale) pairs whose binary32 product is exactly a bfloat16 midpoint while the
    exact product is not, chosen so that rounding that binary32 midpoint to even goes
    the other way from rounding the exact product: the cases where rounding twice is
    off by one unit."""
    import torch
    out = []
    while len(out) < n:
        q = int(rng.integers(2, 128)) * (1 if rng.integers(0, 2) else -1)
        code = int(rng.integers(0x3B00, 0x40C0))           # |m| in about [0.002, 6]
        m = float(np.array([(code << 16) | 0x8000], np.uint32).view(np.float32)[0])
        s0 = np.float32(abs(m / q))
        for k in range(-64, 65):
            s = np.float32(s0 + np.float32(k) * np.spacing(s0))
            p = np.float32(np.float32(q) * s)
            if abs(float(p)) != m or q * float(s) == float(p):
                continue
            exact = oracle.bf16_rne(q * float(s))
            naive = int(torch.tensor([float(p)], dtype=torch.float32).to(torch.bfloat16)
                        .view(torch.int16).item()) & 0xFFFF
            if exact != naive:
                out.append((q, s))
            break
    return out


def test_dequant_double_rounding_cases(hp, oracle):
    """Products whose binary32 rounding is a bfloat16 tie: the kernel must follow
    the exact product, like the oracle."""
    import torch
    rng = np.random.default_rng(8)
    cases = _tie_scales(rng, 64, oracle)
    P, H, D = 4, 1, 16
    N = len(cases)
    pool = np.zeros((N, P, H * D), np.int8)
    scales = np.zeros((N, P), np.float32)
    for i, (q, s) in enumerate(cases):
        pool[i, :, :] = q
        scales[i, :] = s
    w = inputs.Workload("ties", N, P, H, D, "i8", np.uint32, np.arange(N, dtype=np.uint32),
                        np.arange(N + 1, dtype=np.uint32), np.full(N, P, np.uint32), 0,
                        "randint(-127,127)", scales_seed=0)
    b = Batch(w, pool=torch.from_numpy(pool.view(np.uint8)).to("cuda"))
    b.scales.copy_(torch.from_numpy(scales.reshape(-1)))
    rc, got = run_dequant(hp, b)
    assert rc == 0 and b.status_value() == 0
    want = b.oracle_desc().gather_dequant()[0]
    # the naive double rounding differs from the oracle on every one of these
    naive = torch.from_numpy((pool.astype(np.float32) * scales[:, :, None]).reshape(N * P, -1))
    naive = naive.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.count_nonzero(naive != want) == want.size
    assert check_close(got, want) == 0


def test_dequant_full_size_sampled(hp, oracle):
    """400,000 int8 pages, 1024 sequences, uint64 indices: whole sampled sequences
    through the oracle, plus random single elements."""
    import torch
    w = inputs.config("quantized_pool", "full")
    b = Batch(w)
    rc, got = run_dequant(hp, b)
    assert rc == 0 and b.status_value() == 0
    host = b.host_pool()
    sc = b.scales.cpu().numpy()
    rng = np.random.default_rng(4)
    seqs = sorted(set([0, w.num_seqs - 1] + list(rng.integers(0, w.num_seqs, 4))))
    table, seq_ptr, lens = sub_batch(w, seqs)
    sub = oracle.Desc(host, table, seq_ptr, lens, num_pages=w.num_pages, page_size=w.page_size,
                      num_heads=w.num_heads, head_dim=w.head_dim, dtype="i8", scales=sc,
                      flags=oracle.HAS_QUANT, index_type=1)
    want = sub.gather_dequant()[0]
    tok_off = np.concatenate([[0], np.cumsum(w.lens.astype(np.int64))])
    rows = np.concatenate([np.arange(tok_off[s], tok_off[s + 1]) for s in seqs])
    assert check_close(got[rows], want) == 0
    full = b.oracle_desc()
    for _ in range(3000):
        s = int(rng.integers(0, w.num_seqs))
        t = int(rng.integers(0, int(w.lens[s])))
        e = int(rng.integers(0, w.num_heads * w.head_dim))
        code, v = full.lookup_dequant(s, t, e // w.head_dim, e % w.head_dim)
        assert code == "OK" and got[tok_off[s] + t, e] == v


def test_dequant_rejects_wrong_pool_type(hp, oracle):
    import torch
    w = inputs.config("decode_gather", "small")
    b = Batch(w)
    out = torch.empty(w.total_tokens * w.num_heads * w.head_dim, dtype=torch.int16, device="cuda")
    rc = hp.hp_gather_dequant(b.desc, out, w.total_tokens, b.ws, b.status)
    assert hp.status_name(rc) == "HP_ERR_DTYPE"
