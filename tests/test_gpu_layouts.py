"""GPU parity of the two physical pool layouts (NHD and HND, the "FlashAttention
y FlashInfer" page, "Resumen en una frase") and of the large pages FlashInfer
serves on Blackwell with GQA (block sizes 256-1024, the same page's
get_supported_kernel_block_sizes listing): cache write bit exact, decode,
prefill and cascade rows against the fp64 oracle on the logical pool."""
import dataclasses

import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("bs", [16, 64, 256, 512, 1024])
def test_decode_layout_and_page_size(oracle, layout, bs):
    ctx = [1, 15, 200, 511, 1023, 1500, 2047, 3000]
    sp = W.BatchSpec(f"d_{layout}_{bs}", 32, 8, 128, bs, decode_ctx=ctx, kv_layout=layout)
    b = W.make_batch(sp, seed=7000 + bs)
    G.check_batch(oracle, b, label=f"decode {layout} bs={bs}")
    G.check_batch(oracle, b, split_kv_tokens=64, label=f"decode {layout} bs={bs} split 64")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("bs,D", [(16, 128), (256, 128), (1024, 64), (512, 128)])
def test_prefill_layout_and_page_size(oracle, layout, bs, D):
    sp = W.BatchSpec(f"p_{layout}_{bs}", 16, 4, D, bs, decode_ctx=[300, 5],
                     prefill=[(130, 0), (257, 600), (1, 1030)], kv_layout=layout)
    b = W.make_batch(sp, seed=7100 + bs + D)
    G.check_batch(oracle, b, label=f"mixed {layout} bs={bs} D={D}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_cascade_hnd_large_pages(oracle, layout):
    P = 1024
    sp = W.BatchSpec(f"c_{layout}", 64, 8, 128, 256, decode_ctx=[P + 3, P + 300, P + 1000],
                     prefill=[(40, P), (200, P + 20)], common_prefix_len=P, kv_layout=layout)
    b = W.make_batch(sp, seed=7200)
    G.check_batch(oracle, b, label=f"cascade {layout} bs=256")


def test_unknown_layout_is_rejected():
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("bad", 8, 2, 64, 16, decode_ctx=[10])
    b = W.make_batch(sp, seed=7300)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, 1, "cuda")
    meta.kv_layout = 7
    q = G.to_dev(b.query, "cuda")
    with pytest.raises(pka.PkaError) as e:
        pka.paged_attn_forward(q, G.to_dev(b.cache, "cuda"), meta, torch.empty_like(q))
    assert e.value.status == -1
