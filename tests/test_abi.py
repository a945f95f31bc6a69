"""The C ABI without a GPU: the library loads, exports exactly the entry points
include/hp.h declares, and its host-side checks agree with the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def hpc():
    from paged_kv_cache_hp_gb300 import build, hp
    build.build()
    hp.lib()
    return hp


def declared():
    with open(os.path.join(ROOT, "include", "hp.h")) as f:
        text = f.read()
    return set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(hp_\w+)\s*\(", text, re.M))


def test_exports_match_header(hpc):
    names = declared()
    assert {"hp_validate", "hp_gather", "hp_gather_dequant", "hp_scatter_append",
            "hp_lane_validate", "hp_lane_gather", "hp_lane_append"} <= names
    out = subprocess.check_output(["nm", "-D", "--defined-only", hpc.LIB_PATH], text=True)
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    hp_exports = {n for n in exported if n.startswith("hp_")}
    assert hp_exports == names
    lib = ctypes.CDLL(hpc.LIB_PATH)
    for n in names:
        assert getattr(lib, n)


def test_status_names(hpc):
    assert hpc.status_name(0) == "HP_OK"
    assert hpc.status_name(-1) == "HP_ERR_RANK"
    assert hpc.status_name(-31) == "HP_ERR_CUDA"
    assert hpc.status_name(5) == "HP_ERR_UNKNOWN"
    # every code the header defines has its own name
    with open(os.path.join(ROOT, "include", "hp.h")) as f:
        codes = dict((m[0], int(m[1])) for m in re.findall(r"(HP_ERR_\w+)\s*=\s*(-\d+)", f.read()))
    for name, value in codes.items():
        assert hpc.status_name(value) == name


def fake_desc(hpc, **kw):
    """A descriptor over made-up, 64-byte-aligned addresses: only host-side checks
    may run on it (each case below fails one before any launch)."""
    d = hpc.HpPagedDesc()
    f = dict(rank=3, paged_axis=0, has_shard=0, flags=0, dtype=1, index_type=0, num_pages=4,
             page_size=4, num_heads=2, head_dim=2, num_seqs=2, table_len=3, scales_len=0,
             page_pool=0x10000, block_table=0x20000, seq_ptr=0x30000, seq_lens=0x40000,
             scales=0)
    f.update(kw)
    for k, v in f.items():
        setattr(d, k, v)

    class W:
        c = d
        ref = ctypes.byref(d)
    return W, f


STRUCTURAL = [
    dict(rank=2), dict(rank=0), dict(paged_axis=1), dict(has_shard=1), dict(index_type=2),
    dict(num_pages=(1 << 32) + 1), dict(dtype=17), dict(page_size=0), dict(num_heads=0),
    dict(head_dim=0), dict(flags=2), dict(flags=2, scales=0x50000, scales_len=15),
    dict(page_pool=0), dict(block_table=0), dict(seq_ptr=0), dict(seq_lens=0),
    dict(page_pool=0x10020), dict(block_table=0x20008), dict(seq_ptr=0x30004),
    dict(seq_lens=0x40010), dict(flags=2, scales=0x50008, scales_len=16),
    dict(num_pages=1 << 44, page_size=1 << 20, index_type=1),
    dict(rank=2, has_shard=1, page_pool=0),
]


@pytest.mark.parametrize("kw", STRUCTURAL)
def test_structural_checks_match_oracle(hpc, oracle, kw):
    W, f = fake_desc(hpc, **kw)
    first = ctypes.c_uint64(7)
    ws = ctypes.c_void_p(0x60000)
    rc = hpc.lib().hp_validate(W.ref, ws, 1 << 20, ctypes.byref(first), None)
    o = oracle.OrDesc()
    for k in ("rank", "paged_axis", "has_shard", "flags", "dtype", "index_type", "num_pages",
              "page_size", "num_heads", "head_dim", "num_seqs", "table_len", "scales_len"):
        setattr(o, k, f[k])
    o.addr_pool, o.addr_table, o.addr_seq_ptr = f["page_pool"], f["block_table"], f["seq_ptr"]
    o.addr_lens, o.addr_scales = f["seq_lens"], f["scales"]
    ofirst = ctypes.c_uint64(0)
    oc = oracle.lib().or_validate(ctypes.byref(o), ctypes.byref(ofirst))
    name = oracle.code_name(oc)
    assert name != "OK"
    assert hpc.status_name(rc) == "HP_ERR_" + name
    assert first.value == 0
    # every entry point applies the same checks before enqueueing anything
    for call in (lambda: hpc.lib().hp_plan(W.ref, 2, ws, 1 << 20, None, None),
                 lambda: hpc.lib().hp_gather(W.ref, ctypes.c_void_p(0x70000), 2, ws, 1 << 20,
                                             None, None),
                 lambda: hpc.lib().hp_scatter_append(W.ref, ctypes.c_void_p(0x70000),
                                                     ctypes.c_void_p(0x80000), 2, ws, 1 << 20,
                                                     None, None)):
        assert hpc.status_name(call()) == "HP_ERR_" + name


def test_workspace_checks(hpc):
    W, f = fake_desc(hpc, num_seqs=100)
    n = ctypes.c_uint64(0)
    assert hpc.lib().hp_workspace_bytes(W.ref, ctypes.byref(n)) == 0
    assert n.value == 256 + 2 * 1024  # 8 * 101 bytes rounded to 256, twice
    for ws, size in ((0, 1 << 20), (0x60010, 1 << 20), (0x60000, n.value - 1)):
        rc = hpc.lib().hp_gather(W.ref, ctypes.c_void_p(0x70000), 5, ctypes.c_void_p(ws), size,
                                 None, None)
        assert hpc.status_name(rc) == "HP_ERR_WORKSPACE"


def test_lane_validate_matches_oracle(hpc, oracle):
    rng = np.random.default_rng(0)
    cases = [(12, 3, [2, 0, 3, 1]), (12, 3, [2, 0, 2, 1]), (12, 3, [2, 0, 4, 1]), (0, 3, []),
             (12, 0, []), (12, 3, [2, 0, 3]), (10, 3, [2, 0, 3, 1]),
             ((1 << 64) - 1, 1 << 63, [0, 1])]
    for _ in range(300):
        C, P = int(rng.integers(1, 40)), int(rng.integers(1, 9))
        N = -(-C // P)
        T = list(rng.permutation(N))
        k = int(rng.integers(0, 4))
        if k == 1 and N > 1:
            T[int(rng.integers(0, N))] = T[int(rng.integers(0, N))]
        elif k == 2:
            T[int(rng.integers(0, N))] = N + int(rng.integers(0, 3))
        elif k == 3:
            T = T[:-1] if rng.integers(0, 2) else T + [0]
        cases.append((C, P, T))
    for C, P, T in cases:
        rc, det = hpc.hp_lane_validate(C, P, np.asarray(T, dtype=np.uint64))
        name, odet = oracle.lane_new(C, P, T)
        assert hpc.status_name(rc) == ("HP_OK" if name == "OK" else "HP_ERR_" + name)
        assert det == odet


def test_lane_host_checks(hpc):
    L = hpc.lib()
    pool, table, out = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    assert hpc.status_name(L.hp_lane_gather(pool, table, 12, 3, 1, 2, 2, 5, 13, out, 0, None, None)) \
        == "HP_ERR_LENGTH"
    assert hpc.status_name(L.hp_lane_gather(pool, table, 12, 3, 0, 2, 2, 5, 1, out, 0, None, None)) \
        == "HP_ERR_ZERO_DIM"
    assert hpc.status_name(L.hp_lane_gather(pool, table, 12, 3, 1, 2, 2, 9, 1, out, 0, None, None)) \
        == "HP_ERR_DTYPE"
    assert hpc.status_name(L.hp_lane_append(pool, table, 12, 3, 1, 2, 2, 5, 7, 6, out, 0,
                                            None, None)) == "HP_ERR_LENGTH"
    assert hpc.status_name(L.hp_lane_gather(pool, table, 1 << 62, 1, 1 << 10, 2, 2, 5, 1, out,
                                            0, None, None)) == "HP_ERR_LANE_OVERFLOW"


@pytest.mark.parametrize("num_seqs,num_heads,G,D", [
    (256, 8, 4, 128), (32, 8, 4, 128), (0, 8, 4, 128), (1, 1, 8, 64), (2048, 2, 2, 256),
    (7, 3, 1, 64), (100, 12, 2, 128), (5, 16, 1, 256),
])
def test_attention_workspace_bound(hpc, num_seqs, num_heads, G, D):
    """hp_attention_decode_workspace_bytes = the plan's workspace + fp32 records (max, sum,
    acc[D], 128 accumulators for D = 64) of every query head for (num_seqs + 512 * R) *
    num_heads segments, R = 8 / num_heads below 8 K/V heads, else 1, a 4-byte count per
    (sequence, K/V head), and for D = 64 the padded queries (256 bytes per query head) with
    256 bytes of alignment room."""
    W, f = fake_desc(hpc, num_seqs=num_seqs, table_len=3, num_heads=num_heads, head_dim=D,
                     num_pages=4)
    plan = ctypes.c_uint64(0)
    assert hpc.lib().hp_workspace_bytes(W.ref, ctypes.byref(plan)) == 0
    R = 8 // num_heads if num_heads < 8 else 1
    rc, n = hpc.hp_attention_decode_workspace_bytes(W, G * num_heads)
    assert rc == 0
    rd = 128 if D == 64 else D
    qpad = num_seqs * num_heads * G * 256 + 256 if D == 64 else 0
    assert n == (plan.value + (num_seqs + 512 * R) * num_heads * G * (rd + 2) * 4
                 + 4 * num_seqs * num_heads + qpad)
