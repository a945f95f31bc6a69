"""The bounded waits of the TMA copy engine, exercised without a GPU fault: with the
HP_TEST_STALL test hook every CTA arms a load it never issues, its wait runs out after
about 2 s, the call stores HP_ERR_TIMEOUT in the status word and returns; the context is
still usable and the next gather matches the oracle."""
import time

import numpy as np
import pytest

from helpers import Batch
from paged_kv_cache_hp_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads", [32, 8])
def test_stalled_bulk_gather_times_out_and_the_context_survives(hp, oracle, heads):
    """32 heads: rows of 8 KiB, 128 KiB copy units (the one-thread producer with 8 KiB
    stages); 8 heads: rows of 2 KiB, 32 KiB units (loader and storer threads with 16 KiB
    stages).  Both batches are too large for the one-launch path."""
    import torch
    w = inputs.decode_gather(seed=12, num_pages=1200, num_heads=heads, head_dim=128,
                             num_seqs=9, len_lo=400, len_hi=1400, dtype="f16")
    b = Batch(w, flags=hp.TEST_STALL)
    out = torch.full((w.total_tokens * w.row_bytes,), 0xEE, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    assert hp.hp_gather(b.desc, out, w.total_tokens, b.ws, b.status) == 0
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert hp.status_name(b.status_value()) == "HP_ERR_TIMEOUT"
    assert 1.0 < waited < 30.0
    # the same batch without the hook, on the same context
    g = Batch(w, pool=b.pool)
    out2 = torch.empty(w.total_tokens * w.row_bytes, dtype=torch.uint8, device="cuda")
    assert hp.hp_gather(g.desc, out2, w.total_tokens, g.ws, g.status) == 0
    torch.cuda.synchronize()
    assert g.status_value() == 0
    want = g.oracle_desc().gather()[0]
    assert np.array_equal(out2.cpu().numpy().reshape(want.shape), want)
