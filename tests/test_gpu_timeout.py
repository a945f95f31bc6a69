"""The bounded waits of the TMA copy engine and of the tensor-core attention kernel,
exercised without a GPU fault: with the HP_TEST_STALL test hook every CTA arms a load it
never issues, its wait runs out after about 2 s, the call stores HP_ERR_TIMEOUT in the
status word and returns; the context is still usable and the next call matches the
oracle."""
import time

import numpy as np
import pytest

from helpers import Batch
from test_gpu_attention import _vmax_read
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


def test_stalled_tensor_core_attention_times_out_and_the_context_survives(hp, oracle):
    """Decode attention on the tensor cores with HP_TEST_STALL: each CTA's K loader arms its
    first step's loads without issuing them, so the score issuer's wait runs out, then the
    other roles' (the softmax threads stop together at their step barrier); the call stores
    HP_ERR_TIMEOUT and the kernel returns.  The same batch without the hook, on the same
    context, matches the oracle."""
    import torch
    w = inputs.decode_gather(seed=21, num_pages=3000, page_size=16, num_heads=8, head_dim=128,
                             num_seqs=8, len_lo=200, len_hi=2000, dtype="bf16")
    Hq, scale = 32, 1.0 / np.sqrt(128)
    vpool = inputs.device_pool(inputs.Workload(**{**w.__dict__, "pool_seed": w.pool_seed + 5}),
                               "cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(21)
    q = torch.randn((w.num_seqs, Hq, 128), generator=gen, device="cuda").to(torch.bfloat16)
    b = Batch(w, flags=hp.TEST_STALL | hp.ATTN_TENSOR_CORES)
    rc, nws = hp.hp_attention_decode_workspace_bytes(b.desc, Hq)
    assert rc == 0
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    out = torch.zeros((w.num_seqs, Hq, 128), dtype=torch.float32, device="cuda")
    t0 = time.time()
    assert hp.hp_attention_decode(b.desc, vpool, q, Hq, scale, out, ws, b.status) == 0
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert hp.status_name(b.status_value()) == "HP_ERR_TIMEOUT"
    assert 1.0 < waited < 30.0
    g = Batch(w, pool=b.pool, flags=hp.ATTN_TENSOR_CORES)
    out2 = torch.full((w.num_seqs, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert hp.hp_attention_decode(g.desc, vpool, q, Hq, scale, out2, ws, g.status) == 0
    torch.cuda.synchronize()
    assert g.status_value() == 0
    vh = vpool.cpu().numpy()
    od = g.oracle_desc()
    want = od.attention_decode(vh, q.view(torch.int16).cpu().numpy().view(np.uint16), Hq, scale)
    got = out2.cpu().numpy()
    vmax = _vmax_read(od, vh, "bf16")
    assert np.all(np.isfinite(got)) and np.abs(got - want).max() <= 1e-4 * vmax + 1e-6
