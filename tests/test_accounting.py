"""Work accounting against the figures the pages print (tests/golden)."""
import json
import os

from paged_kv_attention_33_gb300 import accounting as A
from paged_kv_attention_33_gb300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def test_cascade_read_example():
    g = GOLD["cascade_prefix_reads"]
    naive, casc = A.cascade_prefix_token_reads(g["num_requests"], g["prefix_len"], [0] * 50)
    assert naive == g["naive_prefix_token_reads"]
    assert casc == g["cascade_prefix_token_reads"]


def test_decode_intensity_page_counting():
    g = GOLD["decode_intensity"]
    assert A.decode_intensity_page_counting(g["bytes_per_element"]) == g["flop_per_byte"]


def test_generated_pool_has_the_page_shape():
    g = GOLD["kv_cache_shape"]
    b = W.make_batch(W.named_spec("tiny_decode"), seed=1)
    sp = b.spec
    assert b.cache.shape == (b.num_blocks, 2, sp.block_size, sp.num_kv_heads, sp.head_size)
    assert len(g["axes"]) == b.cache.ndim and sp.block_size % g["block_size_multiple"] == 0


def test_admitted_pairs_bruteforce():
    for q, c, lo in [(1, 0, 0), (5, 0, 0), (7, 3, 0), (4, 10, 6), (9, 2, 5), (3, 1, 8)]:
        want = sum(1 for i in range(q) for j in range(c + q) if j <= c + i and j >= lo)
        assert A.admitted_pairs(q, c, True, lo) == want
        assert A.admitted_pairs(q, c, False, lo) == q * max(0, c + q - lo)


def test_named_workload_sizes():
    dh = W.named_spec("decode_heavy")
    assert dh.num_decodes == 128 and min(dh.decode_ctx) >= 512 and max(dh.decode_ctx) <= 8192
    gb = A.decode_kv_bytes(dh) / 1e9
    assert 1.5 < gb < 3.0
    pf = W.named_spec("prefill")
    tf = A.prefill_flops(pf) / 1e12
    assert 0.5 < tf < 3.5
    cs = W.named_spec("cascade")
    naive, casc = A.cascade_prefix_token_reads(256, 4096, [L - 4096 for L in cs.seq_lens])
    assert naive > 5 * casc
