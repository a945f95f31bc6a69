"""Pins the CPU oracle to values the pages print and to closed forms.

Every expected value here comes from a golden fixture (with its source) or from
an independent route -- numpy's own row-major indexing, torch's bfloat16
conversion, exact rational arithmetic -- never from the oracle's own formula.
"""
from fractions import Fraction

import numpy as np
import pytest

from conftest import golden_kv, golden_lines
from paged_kv_cache_hp_gb300 import inputs


def ints(xs):
    return [int(x) for x in xs]


# ------------------------------------------------------------------ Element Lookup
def test_block_example_element_lookup(oracle):
    """Hurray spec, section Example: seq_ptr [0,2,3], table [0,1,0], P=4, 5 pages,
    2 heads x 8 dims, fp16.  Pool values are their own flat positions, so each
    lookup returns the row-major index numpy assigns to (page, slot, head, dim)."""
    g = golden_kv("block_example.txt")
    P, N, H, D = (int(g[k][0]) for k in ("page_size", "num_pages", "num_heads", "head_dim"))
    assert N * P * H * D == int(g["pool_values"][0]) == 320
    pool = np.arange(N * P * H * D, dtype=np.float16)  # exact up to 2048
    desc = oracle.Desc(pool, ints(g["block_table"]), ints(g["seq_ptr"]), ints(g["lens"]),
                       num_pages=N, page_size=P, num_heads=H, head_dim=D, dtype="f16",
                       index_type=0)
    assert desc.validate() == ("OK", 0)
    pages = {0: ints(g["seq0_page_of_tokens"]), 1: ints(g["seq1_page_of_tokens"])}
    slots = {0: ints(g["seq0_slot_of_tokens"]), 1: [0, 1, 2]}
    for s, lens in ((0, 6), (1, 3)):
        for t in range(lens):
            for h in range(H):
                for d in range(D):
                    code, b = desc.lookup(s, t, h, d)
                    assert code == "OK"
                    want = np.ravel_multi_index((pages[s][t], slots[s][t], h, d), (N, P, H, D))
                    assert b.view(np.float16)[0] == want
    # token 5 of sequence 0 is slot 1 of page 1: head 1, dim 7 sits at position 95
    assert desc.lookup(0, 5, 1, 7)[1].view(np.float16)[0] == 95
    out, written, fault = desc.gather()
    assert fault == "OK" and written.all() and out.shape == (9, H * D * 2)
    # sequence 1 aliases page 0: its three rows are sequence 0's first three, bit for bit
    assert np.array_equal(out[6:9], out[0:3])


def test_prefix_sharing_tiny_config(oracle):
    """Hurray spec, section Prefix Sharing: slices [12,5,7,9] and [12,5,7,3]
    (15 and 13 tokens, P=4, fp32, 2 heads x 4 dims)."""
    g = golden_kv("prefix_sharing.txt")
    w = inputs.tiny_prefix_gather()
    assert list(w.table[:4]) == ints(g["seq0_slice"]) and list(w.table[4:]) == ints(g["seq1_slice"])
    pool = inputs.host_pool(w)  # [16, 4, 32 bytes]
    desc = oracle.Desc(pool, w.table, w.seq_ptr, w.lens, num_pages=16, page_size=4,
                       num_heads=2, head_dim=4, dtype="f32")
    assert desc.validate() == ("OK", 0)
    out, written, fault = desc.gather()
    assert fault == "OK" and written.all() and out.shape == (28, 32)
    # seq 0 rows 0-11 come from pages 12, 5, 7 in order; rows 12-14 from page 9 slots 0-2
    for k, page in enumerate((12, 5, 7)):
        assert np.array_equal(out[4 * k:4 * k + 4], pool[page])
    assert np.array_equal(out[12:15], pool[9, :3])
    # seq 1 (rows 15-27): shares the first 12 rows, then page 3 slot 0
    assert np.array_equal(out[15:27], out[0:12])
    assert np.array_equal(out[27], pool[3, 0])
    # no sentinel slot was read
    assert not (out == inputs.SENTINEL).all(axis=1).any()


def test_identity_table_is_a_prefix_copy(oracle):
    """One sequence whose slice is 0, 1, 2, ...: the gather is the pool's first
    len rows, a plain memcpy."""
    rng = np.random.default_rng(1)
    N, P, H, D = 6, 5, 3, 2
    pool = rng.integers(0, 256, N * P * H * D * 2, dtype=np.uint8)
    for length in (1, 4, 5, 17, 30):
        need = -(-length // P)
        desc = oracle.Desc(pool, np.arange(need), [0, need], [length], num_pages=N, page_size=P,
                           num_heads=H, head_dim=D, dtype="bf16", index_type=1)
        out, _, fault = desc.gather()
        assert fault == "OK"
        assert np.array_equal(out.reshape(-1), pool[:length * H * D * 2])


def test_empty_batch_form(oracle):
    """Hurray spec, Buffer Table note: num_seqs = 0, block_table empty (may be
    null), seq_ptr = [0]."""
    desc = oracle.Desc(np.zeros(64, np.uint8), None, [0], np.zeros(0, np.uint32), num_pages=2,
                       page_size=4, num_heads=2, head_dim=4, dtype="f16", index_type=0)
    assert desc.validate() == ("OK", 0)
    assert desc.total_tokens() == 0
    out, written, fault = desc.gather()
    assert out.shape == (0, 16) and fault == "OK"


# ------------------------------------------------------------------ validation
def _desc(oracle, **kw):
    base = dict(pool=np.zeros(4 * 4 * 2 * 2 * 2, np.uint8), table=[0, 1, 2], seq_ptr=[0, 2, 3],
                lens=[5, 4], num_pages=4, page_size=4, num_heads=2, head_dim=2, dtype="f16",
                index_type=0)
    base.update(kw)
    return oracle.Desc(base.pop("pool"), base.pop("table"), base.pop("seq_ptr"),
                       base.pop("lens"), **base)


@pytest.mark.parametrize("kw,want", [
    ({}, ("OK", 0)),
    ({"rank": 2}, ("RANK", 0)),                      # Description: rank must be 3
    ({"rank": 4}, ("RANK", 0)),
    ({"paged_axis": 1}, ("PAGED_AXIS", 0)),          # invariant (6)
    ({"has_shard": 1}, ("SHARD", 0)),                # Sharding
    ({"index_type": 2}, ("INDEX_TYPE", 0)),          # only 0x00 / 0x01
    ({"num_pages": (1 << 32) + 1, "pool": np.zeros(8, np.uint8)}, ("INDEX_TYPE", 0)),
    ({"dtype": 9}, ("DTYPE", 0)),
    ({"page_size": 0}, ("ZERO_DIM", 0)),
    ({"num_heads": 0}, ("ZERO_DIM", 0)),
    ({"head_dim": 0}, ("ZERO_DIM", 0)),
    ({"flags": 2}, ("SCALES", 0)),                   # HAS_QUANT without scales
    ({"flags": 2, "scales": np.ones(15, np.float32)}, ("SCALES", 0)),  # wants 4*4 = 16
    ({"flags": 2, "scales": np.ones(16, np.float32)}, ("OK", 0)),
    ({"addrs": {"pool": 0}}, ("NULL", 0)),
    ({"addrs": {"table": 0}}, ("NULL", 0)),
    ({"addrs": {"seq_ptr": 0}}, ("NULL", 0)),
    ({"addrs": {"lens": 0}}, ("NULL", 0)),
    ({"addrs": {"pool": 64 + 32}}, ("ALIGN", 0)),     # Alignment: at least 64 bytes
    ({"addrs": {"lens": 64 * 5 + 8}}, ("ALIGN", 0)),
    ({"num_pages": 1 << 44, "page_size": 1 << 20, "index_type": 1}, ("OVERFLOW", 0)),
    ({"seq_ptr": [1, 2, 3]}, ("SEQ_PTR_START", 0)),   # invariant (1)
    ({"seq_ptr": [0, 3, 2, 3], "lens": [1, 1, 1]}, ("SEQ_PTR_ORDER", 1)),  # invariant (2)
    ({"seq_ptr": [0, 2, 2]}, ("SEQ_PTR_END", 2)),     # seq_ptr[S] != table length
    ({"seq_ptr": [0, 2, 4]}, ("SEQ_PTR_END", 2)),
    ({"table": [0, 4, 2]}, ("PAGE_ID", 1)),           # invariant (3): < num_pages
    ({"table": [7, 4, 2]}, ("PAGE_ID", 0)),
    ({"lens": [9, 4]}, ("LEN", 0)),                   # 9 tokens in 2 pages of 4
    ({"lens": [8, 5]}, ("LEN", 1)),
    ({"lens": [8, 4]}, ("OK", 0)),
    # several violations: the first rule in order wins
    ({"seq_ptr": [1, 0, 3], "table": [9, 9, 9]}, ("SEQ_PTR_START", 0)),
    ({"seq_ptr": [0, 3, 2], "table": [9, 9, 9]}, ("SEQ_PTR_ORDER", 1)),
    ({"table": [9, 9, 9], "lens": [99, 99]}, ("PAGE_ID", 0)),
    # permissive mode skips invariants (1)-(3) and the count rule, not the structure
    ({"flags": 1, "seq_ptr": [1, 0, 3], "table": [9, 9, 9]}, ("OK", 0)),
    ({"flags": 1, "rank": 2}, ("RANK", 0)),
])
def test_validate_rules(oracle, kw, want):
    assert _desc(oracle, **kw).validate() == want


def test_aliasing_is_not_validated(oracle):
    """Hurray spec, Storage Invariants: aliased page IDs are expressible, not
    validated -- a table naming one page three times is valid."""
    assert _desc(oracle, table=[1, 1, 1], lens=[8, 4]).validate() == ("OK", 0)


# ------------------------------------------------------------------ per-lane layout
def test_lane_worked_positions(oracle):
    g = golden_kv("lane_positions.txt")
    C, P = int(g["capacity"][0]), int(g["page_tokens"][0])
    T = ints(g["table"])
    B, H, W = int(g["batch"][0]), int(g["kv_heads"][0]), int(g["width"][0])
    got = [oracle.lane_physical_row_start(C, P, T, B, H, W, 0, 0, p) for p in ints(g["positions"])]
    assert got == ints(g["indices"])
    # head 1 begins 6 scalars further into the page
    assert oracle.lane_physical_row_start(C, P, T, B, H, W, 0, 1, 0) == \
        ints(g["indices"])[0] + int(g["head1_offset"][0])
    # every logical page starts at T[q] * (scalar slots per page)
    spp = int(g["slots_per_page"][0])
    for q in range(len(T)):
        assert oracle.lane_physical_row_start(C, P, T, B, H, W, 0, 0, q * P) == T[q] * spp
    # reserved positions 9..11 are addressable in physical page 1
    for p in ints(g["reserved_positions"]):
        assert oracle.lane_address(C, P, T, p)[1] == int(g["reserved_physical_page"][0])
    # out of range: position >= C, batch >= B, head >= H_kv
    assert oracle.lane_address(C, P, T, C) is None
    assert oracle.lane_physical_row_start(C, P, T, B, H, W, 0, 0, C) is None
    assert oracle.lane_physical_row_start(C, P, T, B, H, W, 1, 0, 0) is None
    assert oracle.lane_physical_row_start(C, P, T, B, H, W, 0, 2, 0) is None
    # the address triple of position 6: logical page 2, physical page 3, offset 0
    assert oracle.lane_address(C, P, T, 6) == (2, 3, 0)


@pytest.mark.parametrize("C,P,T,want", [
    (12, 3, [2, 0, 3, 1], ("OK", (0, 0))),
    (12, 3, [2, 0, 2, 1], ("ALIASED_PAGE", (2, 0))),
    (12, 3, [2, 0, 4, 1], ("PHYSICAL_PAGE", (2, 4))),
    (0, 3, [], ("ZERO_CAPACITY", (0, 0))),
    (12, 0, [], ("ZERO_PAGE_SIZE", (0, 0))),
    (12, 3, [2, 0, 3], ("PAGE_COUNT", (4, 3))),
    (10, 3, [2, 0, 3, 1], ("OK", (0, 0))),            # ceil(10/3) = 4 pages
    (10, 3, [2, 0, 3, 1, 4], ("PAGE_COUNT", (4, 5))),
    ((1 << 64) - 1, 1 << 63, [0, 1], ("LANE_OVERFLOW", (0, 0))),  # 2 pages * 2^63 = 2^64
    (12, 3, [4, 0, 0, 1], ("PHYSICAL_PAGE", (0, 4))),  # the first failing entry wins
    (12, 3, [0, 0, 9, 1], ("ALIASED_PAGE", (0, 0))),
])
def test_lane_constructor_rules(oracle, C, P, T, want):
    assert oracle.lane_new(C, P, T) == want


def test_lane_single_lane_identity_is_contiguous(oracle):
    """With one lane and the identity table the paged row start reduces to the
    contiguous layout (lane*C + p)*width of the same chapter."""
    for C, P, W in ((12, 3, 2), (10, 4, 5), (7, 7, 1), (9, 1, 3)):
        T = list(range(-(-C // P)))
        for p in range(C):
            assert oracle.lane_physical_row_start(C, P, T, 1, 1, W, 0, 0, p) == \
                oracle.lane_physical_row_start(C, P, None, 1, 1, W, 0, 0, p) == p * W


def test_payload_counts(oracle):
    g = {}
    for ln in golden_lines("payload.txt"):
        for kv in ln[1:]:
            if "=" in kv:
                k, v = kv.split("=")
                g.setdefault(ln[0], {})[k] = v
    m = g["main"]
    got = oracle.payload(*(int(m[k]) for k in ("capacity", "page_tokens", "length", "batch",
                                               "kv_heads", "width")))
    for k, v in m.items():
        if k in got:
            assert got[k] == int(v), k
    assert 2 * got["allocated_payload_bytes"] == int(golden_kv("payload.txt")["two_layers_allocated_bytes"][0])
    # conservation: live + tail + inactive = allocated
    assert got["live_scalar_slots"] + got["active_page_tail_scalar_slots"] + \
        got["inactive_page_scalar_slots"] == got["allocated_scalar_slots"]
    r = g["rounding"]
    C, P, B, H, W = (int(r[k]) for k in ("capacity", "page_tokens", "batch", "kv_heads", "width"))
    got = oracle.payload(C, P, int(r["length"]), B, H, W)
    assert got["allocated_scalar_slots"] == int(r["allocated_scalar_slots"])
    assert got["unused_scalar_slots"] == got["allocated_scalar_slots"]  # n = 0
    # contiguous K and V arrays: one past the last contiguous row start, twice
    contiguous = 2 * (oracle.lane_physical_row_start(C, P, None, B, H, W, B - 1, H - 1, C - 1) + W)
    assert contiguous == int(r["contiguous_scalar_slots"])
    extra = got["allocated_scalar_slots"] - contiguous
    assert extra == int(r["extra_slots"]) and extra * 8 == int(r["extra_bytes"])
    for p in (int(x) for x in r["inaccessible_positions"].split(",")):
        assert oracle.lane_address(C, P, [2, 0, 3, 1], p) is None
    assert oracle.payload(C, P, C + 1, B, H, W) == "LENGTH"


# ------------------------------------------------------------------ bfloat16 rounding
def test_bf16_rne_known_codes(oracle):
    cases = [(1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000), (0.1, 0x3DCD),
             (1 + 2 ** -8, 0x3F80),            # tie, to even
             (1 + 3 * 2 ** -8, 0x3F82),        # tie, to even (upwards)
             (1 + 2 ** -8 + 2 ** -30, 0x3F81),  # just above the tie
             (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
             (3.0e38, 0x7F62), (3.4e38, 0x7F80),  # past the largest finite value: inf
             (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (3 * 2.0 ** -134, 0x0002),
             (2.0 ** -126, 0x0080)]
    for x, code in cases:
        assert oracle.bf16_rne(x) == code, (x, hex(oracle.bf16_rne(x)))
    assert oracle.bf16_rne(float("nan")) & 0x7FFF > 0x7F80


def test_bf16_rne_matches_torch_on_binary32(oracle):
    """For binary32 inputs the single rounding equals torch's float32->bfloat16
    conversion (round to nearest even)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    bits = np.concatenate([
        rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32),
        (rng.integers(0, 1 << 16, 4000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000,  # ties
        rng.integers(0, 1 << 23, 2000, dtype=np.uint64).astype(np.uint32),  # subnormals
    ])
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(x)) for x in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def _exact_bf16(x: Fraction) -> float:
    """Nearest bfloat16 to a rational, ties to even, by search over the binade."""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # |x| = a * 2^e, 1 <= a < 2; 8 significant bits -> steps of 2^-7
    steps = a * 128
    lo = int(steps)
    frac = steps - lo
    n = lo + (1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and lo % 2) else 0)
    return sign * n * 2.0 ** (e - 7)


def test_dequant_lookup_is_the_exact_product_rounded_once(oracle):
    rng = np.random.default_rng(11)
    N, P, H, D = 3, 4, 2, 8
    pool = rng.integers(-127, 127, N * P * H * D, endpoint=True).astype(np.int8)
    for scales in (rng.uniform(0.001, 0.05, N * P).astype(np.float32),
                   np.ones(N * P, np.float32),
                   (2.0 ** rng.integers(-20, 20, N * P)).astype(np.float32)):
        desc = oracle.Desc(pool, [2, 0, 1], [0, 3], [11], num_pages=N, page_size=P,
                           num_heads=H, head_dim=D, dtype="i8", scales=scales, flags=2,
                           index_type=0)
        assert desc.validate() == ("OK", 0)
        out, written, fault = desc.gather_dequant()
        assert fault == "OK" and written.all()
        import torch
        got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).float().numpy()
        for t in range(11):
            phys, off = [2, 0, 1][t // P], t % P
            for e in range(H * D):
                q = int(pool.reshape(N, P, H * D)[phys, off, e])
                s = Fraction(float(scales[phys * P + off]))
                assert got[t, e] == _exact_bf16(q * s), (t, e)
        if np.all(scales == 1):
            # integers |q| <= 127 are exact in bfloat16
            assert np.array_equal(got, pool.reshape(N, P, H * D)[[2, 2, 2, 2, 0, 0, 0, 0, 1, 1, 1],
                                                                  [0, 1, 2, 3] * 2 + [0, 1, 2]])


# ------------------------------------------------------------------ append
def test_append_then_gather_round_trip(oracle):
    """Appending every row of a batch into empty slices and gathering it back
    returns the appended rows."""
    rng = np.random.default_rng(3)
    N, P, H, D = 12, 3, 2, 3
    lens = [7, 1, 9]
    table = [5, 0, 11, 3, 7, 2, 9]  # 3 + 1 + 3 pages
    seq_ptr = [0, 3, 4, 7]
    pool = np.full(N * P * H * D * 4, 0x55, np.uint8)
    new = rng.integers(0, 256, (sum(lens), H * D * 4), dtype=np.uint8)
    empty = oracle.Desc(pool, table, seq_ptr, [0, 0, 0], num_pages=N, page_size=P, num_heads=H,
                        head_dim=D, dtype="f32", index_type=1)
    new_ptr = np.concatenate([[0], np.cumsum(lens)])
    assert empty.validate_append(new_ptr, sum(lens)) == ("OK", 0)
    assert empty.scatter_append(new, new_ptr) == "OK"
    full = oracle.Desc(pool, table, seq_ptr, lens, num_pages=N, page_size=P, num_heads=H,
                       head_dim=D, dtype="f32", index_type=1)
    out, _, fault = full.gather()
    assert fault == "OK" and np.array_equal(out, new)
    # the appended rows landed at numpy's (page, slot) positions; nothing else changed
    pool4 = pool.reshape(N, P, H * D * 4)
    touched = np.zeros((N, P), bool)
    row = 0
    for s in range(3):
        for t in range(lens[s]):
            page = table[seq_ptr[s] + t // P]
            assert np.array_equal(pool4[page, t % P], new[row])
            touched[page, t % P] = True
            row += 1
    assert (pool4[~touched] == 0x55).all()


@pytest.mark.parametrize("kw,want", [
    ({}, ("OK", 0)),
    ({"new_ptr": [1, 1, 2]}, ("NEW_PTR_START", 0)),
    ({"new_ptr": [0, 2, 1]}, ("NEW_PTR_ORDER", 1)),
    ({"total_new": 3}, ("NEW_PTR_END", 2)),
    ({"lens": [8, 2]}, ("CAPACITY", 0)),        # 8 + 1 > 2 pages * 4 slots
    ({"lens": [7, 3]}, ("OK", 0)),
    ({"lens": [5, 4]}, ("CAPACITY", 1)),        # 4 + 1 > 1 page * 4 slots
    ({"table": [0, 9, 2]}, ("PAGE_ID", 1)),     # storage invariants come first
])
def test_validate_append_rules(oracle, kw, want):
    new_ptr = kw.pop("new_ptr", [0, 1, 2])
    total = kw.pop("total_new", 2)
    d = _desc(oracle, lens=kw.pop("lens", [5, 2]), **kw)
    assert d.validate_append(new_ptr, total) == want
