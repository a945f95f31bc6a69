"""Pins the oracle's decode attention over a block-paged K/V cache: element conversions
against numpy, closed forms (one token, uniform weights, empty sequences) and a numpy
float64 softmax-attention over K/V gathered with numpy indexing."""
import numpy as np
import pytest


def test_f16_and_bf16_conversions(oracle):
    codes = np.arange(1 << 16, dtype=np.uint16)
    f16 = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.lib().or_f16_to_double(int(c)) for c in codes])
    finite = np.isfinite(f16)
    assert np.array_equal(got[finite], f16[finite])
    assert np.array_equal(np.isnan(got), np.isnan(f16)) and np.array_equal(np.isinf(got), np.isinf(f16))
    with np.errstate(invalid="ignore"):  # signalling NaN codes become quiet NaNs
        bf = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gotb = np.array([oracle.lib().or_bf16_to_double(int(c)) for c in codes[::7]])
    fin = np.isfinite(bf[::7])
    assert np.array_equal(gotb[fin], bf[::7][fin])
    assert np.array_equal(np.isnan(gotb), np.isnan(bf[::7]))
    assert np.array_equal(np.isinf(gotb), np.isinf(bf[::7]))


def _batch(rng, dtype, S=3, N=12, P=4, H=2, D=8, lens=None):
    lens = list(rng.integers(0, 3 * P + 1, S)) if lens is None else lens
    table, sp = [], [0]
    free = list(rng.permutation(N))
    for n in lens:
        k = -(-int(n) // P)
        table += [int(free.pop()) for _ in range(k)]
        sp.append(len(table))
    npdt = np.float16 if dtype == "f16" else np.float32
    K = rng.standard_normal((N, P, H, D)).astype(npdt)
    V = rng.standard_normal((N, P, H, D)).astype(npdt)
    return K, V, table, sp, [int(x) for x in lens]


def _desc(oracle, K, table, sp, lens, dtype):
    N, P, H, D = K.shape
    return oracle.Desc(K, table if table else None, sp, lens, num_pages=N, page_size=P,
                       num_heads=H, head_dim=D, dtype=dtype, index_type=0)


@pytest.mark.parametrize("dtype,Hq", [("f16", 2), ("f16", 4), ("f32", 8), ("f32", 2)])
@pytest.mark.parametrize("seed", range(4))
def test_matches_numpy_softmax_attention(oracle, dtype, Hq, seed):
    rng = np.random.default_rng(seed * 10 + Hq)
    K, V, table, sp, lens = _batch(rng, dtype)
    N, P, H, D = K.shape
    q = rng.standard_normal((len(lens), Hq, D)).astype(K.dtype)
    scale = 1 / np.sqrt(D)
    got = _desc(oracle, K, table, sp, lens, dtype).attention_decode(V, q, Hq, scale)
    G = Hq // H
    for s, n in enumerate(lens):
        rows = [(table[sp[s] + t // P], t % P) for t in range(n)]
        for qh in range(Hq):
            if n == 0:
                assert (got[s, qh] == 0).all()
                continue
            Ks = np.array([K[p, sl, qh // G] for p, sl in rows], np.float64)
            Vs = np.array([V[p, sl, qh // G] for p, sl in rows], np.float64)
            sc = scale * Ks @ q[s, qh].astype(np.float64)
            w = np.exp(sc - sc.max())
            w /= w.sum()
            np.testing.assert_allclose(got[s, qh], w @ Vs, rtol=1e-12, atol=1e-12)


def test_closed_forms(oracle):
    rng = np.random.default_rng(1)
    K, V, table, sp, lens = _batch(rng, "f32", S=3, lens=[1, 7, 0])
    N, P, H, D = K.shape
    d = _desc(oracle, K, table, sp, lens, "f32")
    q = rng.standard_normal((3, 2, D)).astype(np.float32)
    out = d.attention_decode(V, q, 2, 0.3)
    # one token: its value row, whatever the score
    assert np.array_equal(out[0, 0], V[table[0], 0, 0].astype(np.float64))
    # a zero query weighs every token equally: the mean of the value rows
    q0 = np.zeros_like(q)
    out0 = d.attention_decode(V, q0, 2, 0.3)
    rows = [(table[sp[1] + t // P], t % P) for t in range(7)]
    mean = np.mean([V[p, sl, 1].astype(np.float64) for p, sl in rows], axis=0)
    np.testing.assert_allclose(out0[1, 1], mean, rtol=1e-13)
    # an empty sequence gives zeros
    assert (out[2] == 0).all()
