"""Parity at the largest sizes the workloads reach and beyond: decode contexts
of 128K-256K keys (16K stages and 16K block-table columns per sequence, pieces
spread over the whole grid) over bf16 and fp8 pools, and a 32K-token causal
prompt with prior context (4K work items); device-generated inputs, checked
against the fp64 oracle on every decode row and, for the prompts, one row of
every (128-query tile, head) plus the last ragged tile of one head."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_decode_very_long_contexts(oracle):
    sp = W.BatchSpec("long_decode", 32, 8, 128, 16, decode_ctx=[0, 131071, 262143, 77777])
    b = W.make_batch(sp, seed=9100, device="cuda")
    G.check_batch(oracle, b, label="256K-key decodes", threads=16)


def test_fp8_decode_very_long_contexts(oracle):
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("long_decode8", 32, 8, 128, 16, decode_ctx=[0, 131071, 262143, 77777])
    b = W.make_batch(sp, seed=9101, device="cuda")
    pool = W.random_fp8_pool(b, seed=9102)
    want = pool.cpu().numpy()
    del b.cache
    torch.cuda.empty_cache()
    ks, vs = 4.0 / 448, 4.0 / 448
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              "cuda", kv_dtype="fp8", k_scale=ks, v_scale=vs)
    out = torch.empty_like(b.query)
    lse = torch.empty(b.query.shape[:2], dtype=torch.float32, device="cuda")
    pka.paged_attn_forward_fused(b.query, b.key, b.value, torch.from_numpy(b.slot_mapping).cuda(),
                                 pool, meta, out, lse, scale=sp.softmax_scale)
    pka.check_status()
    key, value, query = (W.to_host_bits(x) for x in (b.key, b.value, b.query))
    oracle.reshape_and_cache_fp8(key, value, want, b.slot_mapping, ks, vs)
    assert np.array_equal(want, pool.cpu().numpy())
    rows = np.arange(b.num_tokens * sp.num_heads, dtype=np.int64)
    o_ref, l_ref = oracle.paged_attention_fp8(query, want, ks, vs, b.query_start_loc, b.seq_lens,
                                              b.block_table, sp.softmax_scale, rows=rows,
                                              threads=16)
    G.assert_close(G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows,
                             sp.num_heads), "256K-key fp8 decodes")


def test_prefill_32k_prompt_with_context(oracle):
    sp = W.BatchSpec("long_prefill", 32, 8, 128, 64, decode_ctx=[5000],
                     prefill=[(32768, 3000), (300, 0)])
    b = W.make_batch(sp, seed=9200, device="cuda")
    rows = G.tile_cover_rows(b, seed=11)
    G.check_batch(oracle, b, rows=rows, label="32K-token prompt", threads=16)
