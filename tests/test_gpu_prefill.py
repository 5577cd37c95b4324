"""GPU parity of the tcgen05 prefill path (varlen causal prefill, chunked
prefill over cached context, mixed decode-first batches) against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_prefill_single_tile(oracle):
    sp = W.BatchSpec("p1", 4, 4, 64, 16, prefill=[(128, 0)])
    G.check_batch(oracle, W.make_batch(sp, seed=3001), label="one full tile")


@pytest.mark.parametrize("H,Hkv,D,bs", [
    (8, 2, 64, 16),
    (32, 8, 128, 16),
    (8, 8, 128, 32),
    (16, 2, 128, 64),
    (8, 1, 64, 128),
])
def test_prefill_ragged(oracle, H, Hkv, D, bs):
    # lengths 1, one below / at / above a 128-row tile, and a few tiles with a tail
    sp = W.BatchSpec("pr", H, Hkv, D, bs, prefill=[(1, 0), (127, 0), (128, 0), (129, 0),
                                                    (300, 0), (17, 0)], table_pad=2)
    G.check_batch(oracle, W.make_batch(sp, seed=3100 + H + D + bs), label=f"{H},{Hkv},{D},{bs}")


@pytest.mark.parametrize("bs", [16, 64, 128])
def test_chunked_prefill_with_context(oracle, bs):
    sp = W.BatchSpec("pc", 16, 4, 128, bs, prefill=[(200, 37), (64, 256), (1, 500), (130, 128),
                                                    (257, 1)])
    G.check_batch(oracle, W.make_batch(sp, seed=3200 + bs), label=f"chunked bs={bs}")


def test_mixed_decode_first_batch(oracle):
    sp = W.BatchSpec("mx", 32, 8, 128, 64, decode_ctx=[0, 100, 1000, 4095],
                     prefill=[(150, 300), (256, 0), (5, 700)])
    G.check_batch(oracle, W.make_batch(sp, seed=3300), label="mixed")


def test_non_causal_prefill(oracle):
    sp = W.BatchSpec("nc", 8, 2, 64, 16, prefill=[(70, 0), (130, 45)], causal=False)
    G.check_batch(oracle, W.make_batch(sp, seed=3400), label="non-causal")
