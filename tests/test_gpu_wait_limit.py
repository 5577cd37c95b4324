"""The failure path of the bounded waits, made on purpose without a fault:
with the test hook pka_test_skip_copies on, the decode and prefill kernels
issue no copy and publish no work, so the first wait of every CTA runs out
after its 2 s limit.  Nothing is in flight when a CTA winds down (no copy and
no MMA was issued), so the GPU is never left with work aimed at a CTA that has
exited.  The test checks that pka_check_status reports the expired wait, then
that a normal forward on the same context gives the oracle's rows."""
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", ["decodes", "prefills"])
def test_expired_wait_is_reported_and_the_context_stays_usable(oracle, kind):
    import torch

    import paged_kv_attention_33_gb300 as pka

    if kind == "decodes":
        sp = W.BatchSpec("wait_d", 8, 2, 64, 16, decode_ctx=[40, 300, 7])
    else:
        sp = W.BatchSpec("wait_p", 8, 2, 64, 16, prefill=[(130, 0), (40, 20)])
    b = W.make_batch(sp, seed=9700)
    dev = "cuda"
    cache = G.to_dev(b.cache, dev)
    pka.reshape_and_cache(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                          torch.from_numpy(b.slot_mapping).to(dev))
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes, dev)
    q = G.to_dev(b.query, dev)
    out = torch.full_like(q, float("nan"))
    pka.test_skip_copies(True)
    try:
        pka.paged_attn_forward(q, cache, meta, out, scale=sp.softmax_scale)
    finally:
        pka.test_skip_copies(False)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5 and "wait timed out" in str(e.value)
    assert torch.isnan(out.float()).all()  # no row was written
    pka.check_status()  # the error word was cleared
    # the same context, a normal forward: the oracle's rows
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(b.key, b.value, want, b.slot_mapping)
    _, out2, lse2 = G.run_library(b)
    import numpy as np

    rows = np.arange(b.num_tokens * sp.num_heads, dtype=np.int64)
    o_ref, l_ref = G.oracle_expected(oracle, b, want, rows=rows)
    G.assert_close(G.compare(out2, lse2, o_ref, l_ref, rows, sp.num_heads), kind)
