"""Shared helpers of the GPU parity tests: run a batch through the C ABI and
compare with the fp64 oracle element by element.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output) against the fp64
oracle: output max-abs <= 2e-2 and mean-abs <= 2e-3, lse abs <= 1e-3;
the cache write is compared byte for byte.
"""
from __future__ import annotations

import numpy as np

from paged_kv_attention_33_gb300 import workloads as W

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def device():
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("GPU test run without a CUDA device")
    return "cuda"


def to_dev(x, dev):
    import torch

    if isinstance(x, np.ndarray):
        if x.dtype == np.uint16:
            return W.to_device(x, dev)
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return x.to(dev)


def run_library(batch: W.Batch, split_kv_tokens: int = 0, causal: bool | None = None,
                with_lse: bool = True):
    """reshape_and_cache then paged_attn_forward on the GPU.
    Returns host copies: cache bits, out bits [T,H,D], lse [T,H] (or None)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = device()
    sp = batch.spec
    q = to_dev(batch.query, dev)
    k = to_dev(batch.key, dev)
    v = to_dev(batch.value, dev)
    cache = to_dev(batch.cache, dev)
    if not isinstance(batch.cache, np.ndarray):
        cache = cache.clone()  # keep the generated pool untouched
    cache = W.to_layout(cache, sp.kv_layout)  # the pool in the batch's physical order
    slots = torch.from_numpy(batch.slot_mapping).to(dev)
    pka.reshape_and_cache(k, v, cache, slots, kv_layout=sp.kv_layout)
    meta = pka.Meta.from_host(batch.query_start_loc, batch.seq_lens, batch.block_table,
                              sp.num_decodes, dev, common_prefix_len=sp.common_prefix_len,
                              split_kv_tokens=split_kv_tokens, kv_layout=sp.kv_layout)
    T = batch.num_tokens
    out = torch.full((T, sp.num_heads, sp.head_size), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((T, sp.num_heads), float("nan"), dtype=torch.float32, device=dev) \
        if with_lse else None
    pka.paged_attn_forward(q, cache, meta, out, lse, scale=sp.softmax_scale,
                           causal=sp.causal if causal is None else causal)
    pka.check_status()
    return (W.to_host_bits(W.from_layout(cache, sp.kv_layout)), W.to_host_bits(out),
            None if lse is None else lse.cpu().numpy())


def compare(out_bits, lse, o_ref, l_ref, rows, H):
    """Errors of GPU rows `rows` (r = t*H + h) against the oracle."""
    t = rows // H
    h = rows % H
    o = W.bf16_bits_to_f32(out_bits[t, h]).astype(np.float64)
    err = np.abs(o - o_ref)
    res = {"out_max_abs": float(np.max(err)) if err.size else 0.0,
           "out_mean_abs": float(np.mean(err)) if err.size else 0.0,
           "finite": bool(np.all(np.isfinite(o)))}
    if lse is not None:
        le = np.abs(lse[t, h].astype(np.float64) - l_ref)
        res["lse_max_abs"] = float(np.max(le)) if le.size else 0.0
        res["finite"] = res["finite"] and bool(np.all(np.isfinite(lse[t, h])))
    return res


def assert_close(res, label=""):
    assert res["finite"], f"{label}: non-finite output {res}"
    assert res["out_max_abs"] <= OUT_MAX_ABS, f"{label}: {res}"
    assert res["out_mean_abs"] <= OUT_MEAN_ABS, f"{label}: {res}"
    if "lse_max_abs" in res:
        assert res["lse_max_abs"] <= LSE_ABS, f"{label}: {res}"


def oracle_expected(oracle, batch: W.Batch, cache_bits, rows=None, threads=8):
    sp = batch.spec
    if sp.common_prefix_len > 0:
        return oracle.cascade_attention(host_bits(batch.query), cache_bits,
                                        batch.query_start_loc, batch.seq_lens, batch.block_table,
                                        sp.softmax_scale, sp.common_prefix_len, sp.causal,
                                        rows=rows, threads=threads)
    return oracle.paged_attention(host_bits(batch.query), cache_bits, batch.query_start_loc, batch.seq_lens,
                                  batch.block_table, sp.softmax_scale, sp.causal, rows=rows,
                                  threads=threads)


def host_bits(x):
    return x if isinstance(x, np.ndarray) else W.to_host_bits(x)


def check_batch(oracle, batch: W.Batch, split_kv_tokens=0, rows=None, label="", threads=8):
    """Full parity check of one batch: the cache bytes, then attention rows.

    The oracle's inputs are the generator's arrays only: it writes the new rows
    into its own host copy of the generated pool and attends over that copy."""
    want = host_bits(batch.cache).copy()
    oracle.reshape_and_cache(host_bits(batch.key), host_bits(batch.value), want,
                             batch.slot_mapping)
    cache_gpu, out, lse = run_library(batch, split_kv_tokens)
    assert np.array_equal(want, cache_gpu), f"{label}: cache write differs"
    del cache_gpu
    H = batch.spec.num_heads
    if rows is None:
        rows = np.arange(batch.num_tokens * H, dtype=np.int64)
    o_ref, l_ref = oracle_expected(oracle, batch, want, rows=rows, threads=threads)
    res = compare(out, lse, o_ref, l_ref, rows, H)
    assert_close(res, label)
    return res


def tile_cover_rows(batch: W.Batch, seed: int, tile: int = 128) -> np.ndarray:
    """Rows r = t*H + h for a dense check of a batch too large to check whole:
    every decode row (all heads); one random row of every (128-query tile,
    head) of every prefill sequence, i.e. of every work item of the
    tensor-core pass and each of its two softmax tiles; and every row of each
    prefill sequence's last, ragged tile for one random head."""
    H = batch.spec.num_heads
    nd = batch.spec.num_decodes
    qsl = np.asarray(batch.query_start_loc, dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(seed))
    heads = np.arange(H, dtype=np.int64)
    rows = [np.arange(qsl[nd] * H, dtype=np.int64)]
    for s in range(nd, len(qsl) - 1):
        t0, n = int(qsl[s]), int(qsl[s + 1] - qsl[s])
        for a in range(0, n, tile):
            t = t0 + rng.integers(a, min(n, a + tile), size=H)
            rows.append(t * H + heads)
        if n > 0:
            last = (n - 1) // tile * tile
            rows.append(np.arange(t0 + last, t0 + n, dtype=np.int64) * H + rng.integers(0, H))
    return np.unique(np.concatenate(rows))


def run_fused(batch: W.Batch, pool=None, k_scale=None, v_scale=None):
    """One step as the benchmark makes it: paged_attn_forward_fused (the cache
    write inside the decode launch) with a workspace of pka_workspace_size
    bytes, over the batch's pool (a clone of it) or over `pool` (an fp8 pool of
    uint8 codes when k_scale is given), updated in place.  Returns the pool
    (device), out and lse (device)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = device()
    sp = batch.spec
    fp8 = k_scale is not None
    if pool is None:
        pool = to_dev(batch.cache, dev)
        if not isinstance(batch.cache, np.ndarray):
            pool = pool.clone()
    meta = pka.Meta.from_host(batch.query_start_loc, batch.seq_lens, batch.block_table,
                              sp.num_decodes, dev, common_prefix_len=sp.common_prefix_len,
                              kv_dtype="fp8" if fp8 else "bf16",
                              k_scale=k_scale if fp8 else 1.0,
                              v_scale=v_scale if fp8 else 1.0)
    T = batch.num_tokens
    need = pka.workspace_size(meta, T, sp.num_heads, sp.num_kv_heads, sp.head_size,
                              sp.block_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out = torch.full((T, sp.num_heads, sp.head_size), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((T, sp.num_heads), float("nan"), dtype=torch.float32, device=dev)
    pka.paged_attn_forward_fused(to_dev(batch.query, dev), to_dev(batch.key, dev),
                                 to_dev(batch.value, dev),
                                 torch.from_numpy(batch.slot_mapping).to(dev), pool, meta, out,
                                 lse, scale=sp.softmax_scale, causal=sp.causal, workspace=ws)
    pka.check_status()
    return pool, out, lse

