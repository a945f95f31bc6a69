"""hp_gather_noalloc: the gather for callers that cannot allocate device memory.

Some callers have no way to allocate device memory -- a plugin inside a framework that
owns the device's memory budget, or a latency-critical loop that must not call
cudaMalloc/cudaFree.  hp_gather_noalloc serves them with a workspace array the library
carries in its own device memory.  These tests call it through the C ABI and check that
its output equals hp_gather's and the CPU oracle's gather (bit for bit, the gather's bar)
on consecutive calls that share that array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from helpers import Batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_SEQS = 16384  # HP_NOALLOC_MAX_SEQS


def _both(hp, b, T):
    import torch
    ref = torch.full((T * b.w.row_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    out = torch.full_like(ref, 0xCD)
    st_ref = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    assert hp.hp_gather(b.desc, ref, T, b.ws, st_ref) == 0
    assert hp.status_name(hp.hp_gather_noalloc(b.desc, out, T, st)) == "HP_OK"
    torch.cuda.synchronize()
    assert st_ref.item() == 0 and st.item() == 0
    return ref, out


def test_noalloc_equals_gather_on_consecutive_calls(hp, oracle):
    # several calls in a row, on different batches: each must be independent of what the
    # previous one left in the shared array
    for name in ("prefix_sharing", "decode_gather", "prefix_sharing"):
        w = inputs.config(name, "small")
        b = Batch(w)
        want, written, fault = b.oracle_desc().gather()
        assert fault == "OK" and written.all()
        ref, out = _both(hp, b, w.total_tokens)
        assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())
        assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)
        # and once more on the same batch
        ref2, out2 = _both(hp, b, w.total_tokens)
        assert np.array_equal(out2.cpu().numpy(), ref.cpu().numpy())
        assert np.array_equal(out2.cpu().numpy().reshape(want.shape), want)


def test_noalloc_at_its_sequence_limit(hp, oracle):
    """Exactly HP_NOALLOC_MAX_SEQS short sequences (some empty) fit; one more is refused
    with HP_ERR_NOALLOC_LIMIT before any work is enqueued."""
    import torch
    w = inputs.decode_gather(seed=12, num_pages=20000, page_size=4, num_heads=2, head_dim=8,
                             num_seqs=MAX_SEQS, len_lo=0, len_hi=2)
    b = Batch(w)
    ref, out = _both(hp, b, w.total_tokens)
    assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())
    want = b.oracle_desc().gather()[0]
    assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)
    big = hp.HpPagedDesc()
    ctypes.memmove(ctypes.byref(big), b.desc.ref, ctypes.sizeof(big))
    big.num_seqs = MAX_SEQS + 1

    class D:
        ref = ctypes.byref(big)
    assert hp.status_name(hp.hp_gather_noalloc(D, out, w.total_tokens)) == "HP_ERR_NOALLOC_LIMIT"


def test_noalloc_reports_device_verdicts(hp, oracle):
    """A batch the plan rejects leaves the output untouched and names the rule, as
    hp_gather does."""
    import torch
    w = inputs.config("decode_gather", "small")
    b = Batch(w)
    T = w.total_tokens
    out = torch.full((T * w.row_bytes,), 0xEE, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    assert hp.hp_gather_noalloc(b.desc, out, T - 1, st) == 0
    torch.cuda.synchronize()
    assert hp.status_name(st.item()) == "HP_ERR_OUT_SIZE"
    assert (out.cpu().numpy() == 0xEE).all()
