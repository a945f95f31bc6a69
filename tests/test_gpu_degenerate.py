"""Degenerate sizes on the GPU: empty batches, batches whose sequences are all empty, zero
blocks or pairs.  Every call returns HP_OK, stores HP_OK in the status word and writes
nothing it should not."""
import numpy as np
import pytest

from helpers import Batch, index_tensor
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _empty_desc(hp, dtype="bf16", num_pages=8):
    import torch
    pool = torch.zeros(num_pages * 16 * 2 * 64 * 2, dtype=torch.uint8, device="cuda")
    sp = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = hp.PagedDesc(pool, None, sp, None, num_pages=num_pages, page_size=16, num_heads=2,
                     head_dim=64, dtype=dtype, index_type=0)
    return d, pool


def test_attention_on_an_empty_batch(hp, oracle):
    import torch
    d, pool = _empty_desc(hp)
    rc, nws = hp.hp_attention_decode_workspace_bytes(d, 4)
    assert rc == 0
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    assert hp.hp_attention_decode(d, pool, None, 4, 0.1, None, ws, st) == 0
    assert hp.hp_attention_plan(d, 4, ws, st) == 0
    assert hp.hp_attention_decode_planned(d, pool, None, 4, 0.1, None, ws, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0


def test_attention_when_every_sequence_is_empty(hp, oracle):
    """Sequences with slices but no tokens: there is no step at all, and every output
    is zero."""
    import torch
    w = inputs.decode_gather(seed=41, num_pages=100, page_size=16, num_heads=2, head_dim=64,
                             num_seqs=5, len_lo=1, len_hi=40, dtype="bf16")
    b = Batch(w, lens=np.zeros(w.num_seqs, dtype=np.uint32))
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, 8)
    ws = torch.full((nws,), 0xFF, dtype=torch.uint8, device="cuda")
    q = torch.ones((w.num_seqs, 8, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((w.num_seqs, 8, 64), float("nan"), dtype=torch.float32, device="cuda")
    assert hp.hp_attention_decode(b.desc, b.pool, q, 8, 0.1, out, ws, b.status) == 0
    torch.cuda.synchronize()
    assert b.status_value() == 0
    assert (out == 0).all()


def test_zero_tails_on_an_empty_batch(hp, oracle):
    import torch
    d, pool = _empty_desc(hp)
    ws = hp.workspace_for(d)
    rc, n = hp.hp_zero_tails_scratch_bytes(d)
    scratch = torch.zeros(max(n, 4), dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    before = pool.clone()
    assert hp.hp_zero_tails(d, ws, scratch, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(pool, before)  # pages no slice names are left alone


def test_zero_block_transposes_and_zero_pair_copies(hp, oracle):
    import torch
    a = torch.full((4096,), 0x5A, dtype=torch.uint8, device="cuda")
    b = torch.full((4096,), 0xA5, dtype=torch.uint8, device="cuda")
    assert hp.hp_from_kernel_layout(a, b, 0, 16, 2, 64, 8, "f16") == 0
    assert hp.hp_to_kernel_layout(a, b, 0, 16, 2, 64, 8, "f16") == 0
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    idx = index_tensor(np.zeros(1, np.uint32), "cuda")
    assert hp.hp_copy_pages(a, 4, 1024, 0, idx, idx, 0, st) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    assert (a == 0x5A).all() and (b == 0xA5).all()
