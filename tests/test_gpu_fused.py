"""GPU parity of pka_paged_attn_forward_fused: the cache write folded into the
forward (the "FlashAttention y FlashInfer" page, "Responsabilidades": the FA
kernel writes the KV cache itself).  The pool must come out byte for byte as
the oracle's write leaves it, the attention rows within tolerance of the
oracle, and both bit-identical to the two-call path (write, then forward)."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _run(batch, fused: bool):
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = "cuda"
    sp = batch.spec
    q = G.to_dev(batch.query, dev)
    k = G.to_dev(batch.key, dev)
    v = G.to_dev(batch.value, dev)
    cache = W.to_layout(G.to_dev(batch.cache, dev), sp.kv_layout)
    slots = torch.from_numpy(batch.slot_mapping).to(dev)
    meta = pka.Meta.from_host(batch.query_start_loc, batch.seq_lens, batch.block_table,
                              sp.num_decodes, dev, common_prefix_len=sp.common_prefix_len,
                              kv_layout=sp.kv_layout)
    T = batch.num_tokens
    out = torch.full((T, sp.num_heads, sp.head_size), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((T, sp.num_heads), float("nan"), dtype=torch.float32, device=dev)
    if fused:
        pka.paged_attn_forward_fused(q, k, v, slots, cache, meta, out, lse,
                                     scale=sp.softmax_scale, causal=sp.causal)
    else:
        pka.reshape_and_cache(k, v, cache, slots, kv_layout=sp.kv_layout)
        pka.paged_attn_forward(q, cache, meta, out, lse, scale=sp.softmax_scale,
                               causal=sp.causal)
    pka.check_status()
    return (W.to_host_bits(W.from_layout(cache, sp.kv_layout)), W.to_host_bits(out),
            lse.cpu().numpy())


CASES = {
    "decodes": dict(H=32, Hkv=8, D=128, bs=16, decode_ctx=[0, 15, 16, 17, 300, 2000]),
    "decodes_g4_d64": dict(H=8, Hkv=2, D=64, bs=64, decode_ctx=[1, 63, 64, 65, 700]),
    "mixed": dict(H=32, Hkv=8, D=128, bs=64, decode_ctx=[100, 1000],
                  prefill=[(70, 0), (129, 300)]),
    "prefill_only": dict(H=16, Hkv=4, D=128, bs=16, decode_ctx=[], prefill=[(40, 10), (130, 0)]),
    "cascade": dict(H=64, Hkv=8, D=128, bs=128, decode_ctx=[256, 300, 900],
                    prefill=[(50, 256)], common_prefix_len=256),
    "hnd_large_pages": dict(H=32, Hkv=8, D=128, bs=256, decode_ctx=[10, 255, 256, 1500],
                            prefill=[(200, 100)], kv_layout="HND"),
    # 16-key pages under query-heavy prefills with prior context that ends inside a
    # 128-key tile: the context's blocks go through the re-blocking copy, the tiles
    # of this step's keys come from the step's rows
    "small_pages_context": dict(H=16, Hkv=4, D=128, bs=16, decode_ctx=[5, 300],
                                prefill=[(400, 0), (300, 70), (300, 200), (129, 37)]),
    "hnd_small_pages_context": dict(H=16, Hkv=4, D=64, bs=16, decode_ctx=[40],
                                    prefill=[(400, 130), (300, 0), (300, 255)],
                                    kv_layout="HND"),
    # batches the mixed plan runs side by side: the decode on part of the SMs,
    # the prefill pass as its programmatic dependent on the rest
    "mixed_side_by_side": dict(H=32, Hkv=8, D=128, bs=16,
                               decode_ctx=[2000 + 250 * k for k in range(16)],
                               prefill=[(256, 1000), (256, 1500)]),
    "hnd_mixed_side_by_side": dict(H=32, Hkv=8, D=128, bs=64,
                                   decode_ctx=[6000 - 230 * k for k in range(16)],
                                   prefill=[(256, 1400), (200, 900)], kv_layout="HND"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_matches_oracle_and_two_calls(oracle, case):
    kw = dict(CASES[case])
    H, Hkv, D, bs = kw.pop("H"), kw.pop("Hkv"), kw.pop("D"), kw.pop("bs")
    sp = W.BatchSpec(f"fused_{case}", H, Hkv, D, bs, **kw)
    b = W.make_batch(sp, seed=9000 + len(case))
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(G.host_bits(b.key), G.host_bits(b.value), want, b.slot_mapping)
    cache_f, out_f, lse_f = _run(b, fused=True)
    assert np.array_equal(cache_f, want), "fused cache write differs from the oracle's"
    o_ref, l_ref = G.oracle_expected(oracle, b, want)
    rows = np.arange(b.num_tokens * H, dtype=np.int64)
    G.assert_close(G.compare(out_f, lse_f, o_ref, l_ref, rows, H), case)
    cache_2, out_2, lse_2 = _run(b, fused=False)
    assert np.array_equal(cache_f, cache_2)
    assert np.array_equal(out_f, out_2), "fused output differs from the two-call path"
    assert np.array_equal(lse_f, lse_2)
