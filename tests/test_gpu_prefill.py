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


@pytest.mark.parametrize("gain", [6.0, 40.0])
def test_prefill_logits_rising_past_the_first_tile(oracle, gain):
    """Keys of a later tile scaled by `gain` raise the logits there (log2
    units) by ~12 at gain 6 and by ~100 at gain 40 above the first tile's max:
    the softmax's reference max moves (past its threshold) and O, already
    holding the earlier tiles' PV, is rescaled; at gain 40 the earlier tiles'
    weights underflow to nothing."""
    sp = W.BatchSpec("rise", 8, 2, 128, 16, prefill=[(512, 0), (300, 40)])
    b = W.make_batch(sp, seed=3600)
    k = W.bf16_bits_to_f32(b.key)
    q0, q1 = int(b.query_start_loc[0]), int(b.query_start_loc[1])
    k[q0 + 256:q0 + 384] *= gain  # keys 256..383 of the first prompt (its third tile)
    k[q1 + 120:q1 + 200] *= gain  # keys 160..239 of the second (40 cached keys first)
    b.key = W.f32_to_bf16_bits(k)
    G.check_batch(oracle, b, label=f"rising logits x{gain}")


def test_many_prefill_sequences(oracle):
    """600 short prefill chunks with cached context beside two decodes: the
    prefill kernel maps its work items to sequences through a per-CTA prefix
    table of super-tiles; every row matches the oracle."""
    rng = np.random.default_rng(3700)
    prefill = [(int(q), int(c)) for q, c in zip(rng.integers(1, 40, 600),
                                                 rng.integers(0, 60, 600))]
    sp = W.BatchSpec("many", 8, 2, 64, 16, decode_ctx=[10, 300], prefill=prefill)
    G.check_batch(oracle, W.make_batch(sp, seed=3701), label="600 prefill sequences")


def test_decodes_with_a_long_prompt(oracle):
    """Two decodes beside a 16K-token prompt: the forward's plan runs the decode
    and the prefill pass one after the other here (the prompt's work dwarfs the
    decode's), where smaller mixed batches run them side by side.  One row of
    every 128-query tile and head, and every decode row, against the oracle."""
    sp = W.BatchSpec("long_prompt", 16, 2, 64, 16, decode_ctx=[10, 3000],
                     prefill=[(16384, 0)])
    b = W.make_batch(sp, seed=3800)
    G.check_batch(oracle, b, rows=G.tile_cover_rows(b, seed=3801), label="long prompt")


def test_non_causal_prefill(oracle):
    sp = W.BatchSpec("nc", 8, 2, 64, 16, prefill=[(70, 0), (130, 45)], causal=False)
    G.check_batch(oracle, W.make_batch(sp, seed=3400), label="non-causal")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_small_pages_reblocked_and_direct(oracle, layout):
    """A bf16 pool of 16-key pages under query-heavy prefills: with the
    workspace pka_workspace_size asks for, the prefill pass reads a copy of
    its sequences' keys in 128-key blocks; with pka_workspace_size_min it reads
    the pages as they are.  Both match the oracle on every row, and each other
    bit for bit."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("reblock", 16, 4, 128, 16, decode_ctx=[100, 1000],
                     prefill=[(300, 0), (700, 37), (257, 1000), (129, 5)], table_pad=2,
                     kv_layout=layout)
    b = W.make_batch(sp, seed=3500)
    dev = "cuda"
    cache = W.to_layout(G.to_dev(b.cache, dev), layout)
    pka.reshape_and_cache(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                          torch.from_numpy(b.slot_mapping).to(dev), kv_layout=layout)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes, dev,
                              kv_layout=layout)
    T, H, D = b.num_tokens, sp.num_heads, sp.head_size
    full = pka.workspace_size(meta, T, H, sp.num_kv_heads, D, sp.block_size)
    small = pka.workspace_size_min(meta, T, H, sp.num_kv_heads, D, sp.block_size)
    assert full > small > 0  # the copy is planned
    q = G.to_dev(b.query, dev)
    results = []
    for nbytes in (full, small):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
        pka.paged_attn_forward(q, cache, meta, out, lse, scale=sp.softmax_scale, workspace=ws)
        pka.check_status()
        results.append((out, lse))
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(b.key, b.value, want, b.slot_mapping)
    rows = np.arange(T * H, dtype=np.int64)
    o_ref, l_ref = G.oracle_expected(oracle, b, want, rows=rows)
    for label, (out, lse) in zip(("re-blocked", "direct"), results):
        G.assert_close(G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, H),
                       f"{layout} {label}")
    assert torch.equal(results[0][0].view(torch.int16), results[1][0].view(torch.int16))
    assert torch.equal(results[0][1], results[1][1])
