"""Full-size parity of the five workloads in the benchmark's launch
configuration: one paged_attn_forward_fused call (the cache write inside the
decode launch) with a workspace of pka_workspace_size bytes, the same seeded
batch the benchmark times, compared with the fp64 oracle.

Complete where the oracle finishes in seconds, dense where it does not:
  * decode_heavy (4,096 rows) and cascade (16,384 rows): every row, bf16 and
    fp8 pools, plus the whole pool byte for byte;
  * prefill, mixed and a 32K-token prompt: every decode row, one row of every
    (128-query tile, head) of every prefill sequence -- every work item of the
    tensor-core pass and both of its softmax tiles -- and every row of each
    prefill sequence's last, ragged tile for one head.
The oracle's inputs are the generator's arrays only: it writes the step's new
rows into its own host copy of the generated pool and attends over that copy.
fp8 pools: the prior context is a seeded draw of e4m3 codes (the oracle's
exhaustive encoder is too slow for a pool of a gigabyte); the step's new rows
are quantised by both sides from the same bf16 K/V.
"""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FP8_SCALE = 4.0 / 448  # |x| <= 4 fills the e4m3 range


def _bench_batch(name):
    return W.make_batch(W.named_spec(name), seed=W.NAMED_SEEDS[name], device="cuda")


def _check_bf16(oracle, name, rows_of=None):
    b = _bench_batch(name)
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(G.host_bits(b.key), G.host_bits(b.value), want, b.slot_mapping)
    pool, out, lse = G.run_fused(b)
    del b.cache
    assert np.array_equal(want, W.to_host_bits(pool)), f"{name}: cache write differs"
    del pool
    H = b.spec.num_heads
    rows = np.arange(b.num_tokens * H, dtype=np.int64) if rows_of is None else rows_of(b)
    o_ref, l_ref = G.oracle_expected(oracle, b, want, rows=rows, threads=16)
    res = G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, H)
    G.assert_close(res, f"{name} ({len(rows)} rows)")
    return res


def _check_fp8(oracle, name, rows_of=None, seed=0):
    import torch

    b = _bench_batch(name)
    pool = W.random_fp8_pool(b, seed=W.NAMED_SEEDS[name] + 10 + seed)
    want = pool.cpu().numpy()
    del b.cache
    torch.cuda.empty_cache()
    key, value, query = (W.to_host_bits(x) for x in (b.key, b.value, b.query))
    pool, out, lse = G.run_fused(b, pool=pool, k_scale=FP8_SCALE, v_scale=FP8_SCALE)
    oracle.reshape_and_cache_fp8(key, value, want, b.slot_mapping, FP8_SCALE, FP8_SCALE)
    assert np.array_equal(want, pool.cpu().numpy()), f"{name} fp8: cache write differs"
    del pool
    H = b.spec.num_heads
    rows = np.arange(b.num_tokens * H, dtype=np.int64) if rows_of is None else rows_of(b)
    # a cascade is by definition the plain attention over the whole table
    o_ref, l_ref = oracle.paged_attention_fp8(query, want, FP8_SCALE, FP8_SCALE,
                                              b.query_start_loc, b.seq_lens, b.block_table,
                                              b.spec.softmax_scale, rows=rows, threads=16)
    res = G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, H)
    G.assert_close(res, f"{name} fp8 ({len(rows)} rows)")
    return res


def test_decode_heavy_every_row(oracle):
    _check_bf16(oracle, "decode_heavy")


def test_decode_heavy_fp8_every_row(oracle):
    _check_fp8(oracle, "decode_heavy")


def test_cascade_every_row(oracle):
    _check_bf16(oracle, "cascade")


def test_cascade_fp8_every_row(oracle):
    _check_fp8(oracle, "cascade")


def test_prefill_every_tile(oracle):
    _check_bf16(oracle, "prefill", rows_of=lambda b: G.tile_cover_rows(b, seed=21))


def test_mixed_every_tile(oracle):
    _check_bf16(oracle, "mixed", rows_of=lambda b: G.tile_cover_rows(b, seed=22))


def test_mixed_fp8_every_tile(oracle):
    _check_fp8(oracle, "mixed", rows_of=lambda b: G.tile_cover_rows(b, seed=23))


def test_tiny_decode_every_row(oracle):
    _check_bf16(oracle, "tiny_decode")
