"""GPU parity of the layout conversions: kernel-internal <-> interchange cache layout
([HF] Framework Compliance) and padded <-> CSR block tables, against the oracle."""
import numpy as np
import pytest

from helpers import index_tensor

pytestmark = pytest.mark.gpu

NPDT = {"f16": np.float16, "bf16": np.uint16, "f32": np.float32, "i8": np.int8, "f64": np.float64}


@pytest.mark.parametrize("nb,bs,H,D,x,dtype", [
    (37, 16, 8, 128, 8, "f16"),   # the older key-cache reshape, 16-byte chunks
    (20, 16, 4, 64, 1, "bf16"),   # x = 1: the [nb, H, D, bs] value-cache form
    (9, 5, 3, 12, 3, "i8"),
    (11, 7, 2, 8, 4, "f32"),
    (5, 3, 2, 6, 2, "f64"),
    (64, 32, 2, 256, 8, "f16"),
    (13, 8, 3, 32, 4, "f32"),     # 16-byte chunks, block_size 8: swizzled staging
    (7, 24, 2, 64, 8, "bf16"),    # block_size a multiple of 8 but not a power of two
    (6, 12, 2, 64, 8, "f16"),     # 16-byte chunks, block_size not a multiple of 8: plain
])
def test_transpose_matches_oracle(hp, oracle, nb, bs, H, D, x, dtype):
    import torch
    rng = np.random.default_rng(nb * bs + x)
    es = np.dtype(NPDT[dtype]).itemsize
    internal = rng.integers(0, 256, (nb, H, D // x, bs, x * es), dtype=np.uint8)
    src = torch.from_numpy(internal).to("cuda")
    dst = torch.full((nb * bs * H * D * es + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    assert hp.hp_from_kernel_layout(src, dst, nb, bs, H, D, x, dtype) == 0
    back = torch.full_like(src, 0x11)
    assert hp.hp_to_kernel_layout(dst, back, nb, bs, H, D, x, dtype) == 0
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    assert (got[nb * bs * H * D * es:] == 0xEE).all()
    want = oracle.from_kernel_layout(internal.view(NPDT[dtype]).reshape(nb, H, D // x, bs, x),
                                     nb, bs, H, D, x)
    assert np.array_equal(got[:nb * bs * H * D * es], want.view(np.uint8).reshape(-1))
    assert torch.equal(back, src)


def test_transpose_rejections(hp, oracle):
    import torch
    a = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    assert hp.status_name(hp.hp_from_kernel_layout(a, a, 1, 16, 1, 10, 4, "f16")) == "HP_ERR_ARG"
    assert hp.status_name(hp.hp_from_kernel_layout(a, a, 1, 256, 1, 128, 8, "f32")) == \
        "HP_ERR_ARG"   # 128 KiB per (block, head)
    assert hp.status_name(hp.hp_from_kernel_layout(a, a, 1, 16, 1, 8, 0, "f16")) == \
        "HP_ERR_ZERO_DIM"


def test_transpose_decode_pool_round_trip(hp, oracle):
    """The decode-gather pool (10,000 blocks x 16 slots x 32 heads x 128 fp16): out and
    back is the identity, and sampled blocks equal the oracle's transpose."""
    import torch
    nb, bs, H, D, x = 10000, 16, 32, 128, 8
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    internal = torch.randint(0, 256, (nb * bs * H * D * 2,), generator=g, dtype=torch.uint8,
                             device="cuda")
    inter = torch.empty_like(internal)
    back = torch.empty_like(internal)
    assert hp.hp_from_kernel_layout(internal, inter, nb, bs, H, D, x, "f16") == 0
    assert hp.hp_to_kernel_layout(inter, back, nb, bs, H, D, x, "f16") == 0
    torch.cuda.synchronize()
    assert torch.equal(back, internal)
    blk = bs * H * D * 2
    for b in (0, 4567, nb - 1):
        src = internal[b * blk:(b + 1) * blk].cpu().numpy().view(np.float16)
        want = oracle.from_kernel_layout(src.reshape(1, H, D // x, bs, x), 1, bs, H, D, x)
        got = inter[b * blk:(b + 1) * blk].cpu().numpy()
        assert np.array_equal(got, want.view(np.uint8).reshape(-1))  # bytes: NaN patterns


@pytest.mark.parametrize("seed", range(6))
def test_padded_csr_match_oracle(hp, oracle, seed):
    import torch
    rng = np.random.default_rng(seed)
    it = seed % 2
    dt = np.uint32 if it == 0 else np.uint64
    B, MB, P = int(rng.integers(1, 3000)), int(rng.integers(1, 40)), int(rng.integers(1, 17))
    padded = rng.integers(0, 1 << 20, (B, MB)).astype(dt)
    lens = rng.integers(0, MB * P + 1, B).astype(dt)
    rc, wsb = hp.hp_table_workspace_bytes(B)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    cap = B * MB
    tab = torch.zeros(cap, dtype=torch.int32 if it == 0 else torch.int64, device="cuda")
    sp = torch.zeros(B + 1, dtype=tab.dtype, device="cuda")
    assert hp.hp_padded_to_csr(index_tensor(padded, "cuda"), index_tensor(lens, "cuda"), B, MB,
                               P, it, tab, cap, sp, ws, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    name, first, want_t, want_sp = oracle.padded_to_csr(padded, lens, P)
    assert name == "OK"
    got_sp = sp.cpu().numpy().view(dt)
    assert np.array_equal(got_sp, want_sp)
    assert np.array_equal(tab.cpu().numpy().view(dt)[:len(want_t)], want_t)
    out = torch.zeros(B * MB, dtype=tab.dtype, device="cuda")
    assert hp.hp_csr_to_padded(tab, int(want_sp[-1]), sp, B, MB, 7, it, out, ws, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    name, first, want_p = oracle.csr_to_padded(want_t, want_sp, MB, 7)
    assert np.array_equal(out.cpu().numpy().view(dt).reshape(B, MB), want_p)


def test_padded_csr_errors_write_nothing(hp, oracle):
    import torch
    padded = np.zeros((3, 2), np.uint32)
    lens = np.array([8, 9, 1], np.uint32)
    rc, wsb = hp.hp_table_workspace_bytes(3)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tab = torch.full((6,), -1, dtype=torch.int32, device="cuda")
    sp = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    assert hp.hp_padded_to_csr(index_tensor(padded, "cuda"), index_tensor(lens, "cuda"), 3, 2, 4, 0,
                               tab, 6, sp, ws, st) == 0
    torch.cuda.synchronize()
    assert hp.status_name(st.item()) == "HP_ERR_LEN"
    assert (tab.cpu().numpy() == -1).all() and (sp.cpu().numpy() == -1).all()
    assert oracle.padded_to_csr(padded, lens, 4)[:2] == ("LEN", 1)
    lens = np.array([8, 8, 1], np.uint32)
    assert hp.hp_padded_to_csr(index_tensor(padded, "cuda"), index_tensor(lens, "cuda"), 3, 2, 4, 0,
                               tab, 4, sp, ws, st) == 0
    torch.cuda.synchronize()
    assert hp.status_name(st.item()) == "HP_ERR_OUT_SIZE"
    out = torch.full((6,), -1, dtype=torch.int32, device="cuda")
    spn = index_tensor(np.array([0, 2, 5, 5], np.uint32), "cuda")
    assert hp.hp_csr_to_padded(tab, 6, spn, 3, 2, 0, 0, out, ws, st) == 0
    torch.cuda.synchronize()
    assert hp.status_name(st.item()) == "HP_ERR_LEN"
    assert (out.cpu().numpy() == -1).all()
