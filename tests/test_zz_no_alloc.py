"""The allocation-free forward entry point (pka_paged_attn_forward_noalloc).

It serves callers that cannot allocate device memory -- an engine that gave
nearly all of HBM to its KV pool, a plugin host that only passes input and
output pointers, a loop that must not call cudaMalloc -- by keeping the
partial results in a scratch buffer built into the library.  Here its output
is checked against the regular entry point (which takes a workspace) on the
same inputs, for two calls in a row, so the second call also runs over the
first call's leftovers.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import paged_kv_attention_33_gb300 as pka
from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G


def _run_both(spec, seed, split):
    import torch

    dev = "cuda"
    b = W.make_batch(spec, seed=seed)
    cache = G.to_dev(b.cache, dev)
    pka.reshape_and_cache(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                          torch.from_numpy(b.slot_mapping).to(dev))
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, spec.num_decodes,
                              dev, common_prefix_len=spec.common_prefix_len,
                              split_kv_tokens=split)
    need = pka.workspace_size(meta, b.num_tokens, spec.num_heads, spec.num_kv_heads,
                              spec.head_size, spec.block_size)
    assert 0 < need <= 16 << 20
    q = G.to_dev(b.query, dev)
    T, H = q.shape[:2]
    ref = torch.empty_like(q)
    ref_lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    pka.paged_attn_forward(q, cache, meta, ref, ref_lse, scale=spec.softmax_scale)
    results = []
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
        pka.paged_attn_forward_noalloc(q, cache, meta, out, lse, scale=spec.softmax_scale)
        results.append((out, lse))
    pka.check_status()
    return ref, ref_lse, results


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["decode_splits", "cascade_mixed"])
def test_noalloc_matches_workspace_entry_point(case):
    if case == "decode_splits":
        rng = np.random.Generator(np.random.PCG64(11))
        spec = W.BatchSpec("na1", 32, 8, 128, 16,
                           decode_ctx=rng.integers(1, 3000, size=24).tolist())
        split = 256
    else:
        spec = W.BatchSpec("na2", 32, 8, 128, 64, decode_ctx=[128, 300, 1000],
                           prefill=[(100, 128), (70, 200)], common_prefix_len=128)
        split = 64
    ref, ref_lse, results = _run_both(spec, seed=5001, split=split)
    import torch

    # the same plan, kernels and split layout as the workspace entry point, so
    # the rows agree bit for bit; a partial-slot mix-up or a stale leftover of
    # the first call would show in the second
    for k, (out, lse) in enumerate(results):
        assert torch.isfinite(out).all() and torch.isfinite(lse).all(), f"call {k}"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {k}"
        assert torch.equal(lse, ref_lse), f"call {k}"


def test_noalloc_rejects_batches_above_its_scratch():
    """A batch whose partials need more than the built-in 16 MiB is refused
    with PKA_ERR_WORKSPACE before anything is enqueued."""
    lib = pka.load_library()
    # a cascade over 8192 prefill tokens: the shared-prefix partials alone are
    # 8192 x 32 heads x 128 x 4 bytes
    m = pka._CMeta(16, 16, 16, 1024, 2, 0, 4096, 16384, 16, 0)
    # the smallest workspace the forward accepts (no optional prefill copy)
    need = lib.pka_workspace_size_min(ctypes.byref(m), 8192, 32, 8, 128, 16)
    assert 16 << 20 < need <= lib.pka_workspace_size(ctypes.byref(m), 8192, 32, 8, 128, 16)
    rc = lib.pka_paged_attn_forward_noalloc(256, 512, ctypes.byref(m), 1024, None, 8192, 32, 8,
                                            128, 16, 100000, 0.088, 1, None)
    assert rc == -3
    msg = lib.pka_last_error().decode()
    assert "16777216" in msg and str(need) in msg


@pytest.mark.gpu
def test_noalloc_over_an_fp8_pool(oracle):
    """An fp8 mixed batch small enough that its partials and the bf16 copy of
    its prefill blocks fit the built-in scratch: the same rows as the
    workspace entry point, twice in a row."""
    import torch

    spec = W.BatchSpec("na8", 16, 4, 128, 16, decode_ctx=[40, 700], prefill=[(64, 100)])
    b = W.make_batch(spec, seed=5002)
    c = G.host_bits(b.cache)
    p8 = np.empty(c.shape, dtype=np.uint8)
    p8[:, 0] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 0]), 0.05)
    p8[:, 1] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 1]), 0.03)
    dev = "cuda"
    pool = torch.from_numpy(p8).to(dev)
    pka.reshape_and_cache_fp8(G.to_dev(b.key, dev), G.to_dev(b.value, dev), pool,
                              torch.from_numpy(b.slot_mapping).to(dev), 0.05, 0.03)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, spec.num_decodes,
                              dev, kv_dtype="fp8", k_scale=0.05, v_scale=0.03)
    need = pka.workspace_size(meta, b.num_tokens, spec.num_heads, spec.num_kv_heads,
                              spec.head_size, spec.block_size)
    assert 0 < need <= 16 << 20
    q = G.to_dev(b.query, dev)
    ref = torch.empty_like(q)
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    pka.paged_attn_forward(q, pool, meta, ref, ref_lse, scale=spec.softmax_scale)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
        pka.paged_attn_forward_noalloc(q, pool, meta, out, lse, scale=spec.softmax_scale)
        pka.check_status()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(lse, ref_lse)
