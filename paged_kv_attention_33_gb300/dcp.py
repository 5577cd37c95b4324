"""Decode context parallelism (DCP): the keys of every decode sequence are
sharded over the ranks of a group; each rank attends its query rows over its
own shard and the partial results are combined by log-sum-exp.

The "FlashAttention y FlashInfer" page ("Limites y fallos") names the DCP
combine branch (an all-gather of the lse with a reduce of the outputs, or an
all-to-all) and warns that the wrong choice breaks the softmax combine across
shards; the "AttentionBackend" page ("Limites y fallos", lse_base_on_e) adds
that the combine must use the lse base the partials were made in.  Here:

  * shard: page n of a sequence (keys [n*bs, (n+1)*bs)) lives on rank
    n % world; a rank's local sequence is its pages in order, so only its last
    page can be partial and the ordinary paged kernels read it unchanged.  A
    rank may hold no key of a short sequence: its partial is lse = -inf, out 0.
  * step: local partial (out, lse) of the rank -> all-gather over the group ->
    pka_merge_partials of the world's partials in rank order.
  * lse base: the forward reports natural-log lse; the merge takes the base as
    an argument (LSE_BASE_E, or LSE_BASE_2 for partials in log2 units).

This module holds the integer sharding and the collective calls only: every
step of the arithmetic (the local attention, an empty shard's out = 0 and
lse = -inf, the merge) runs in the library's kernels.

Only decodes are sharded (the name's "decode"): a prefill query's causal limit
is a global key position, which a rank-local sequence does not carry.
"""
from __future__ import annotations

import math

import numpy as np


def shard_decode_metadata(seq_lens, block_table, block_size: int, rank: int, world: int):
    """(local seq_lens int32 [S], local block_table int32 [S, W]) of `rank`:
    pages n = rank, rank + world, ... of each sequence, in order."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    block_table = np.asarray(block_table)
    S = seq_lens.shape[0]
    pages = [list(range(rank, math.ceil(int(L) / block_size), world)) for L in seq_lens]
    width = max([len(p) for p in pages] + [1])
    table = np.full((S, width), -1, dtype=np.int32)
    lens = np.zeros(S, dtype=np.int32)
    for s, ps in enumerate(pages):
        L = int(seq_lens[s])
        for i, n in enumerate(ps):
            table[s, i] = block_table[s, n]
            lens[s] += min(block_size, L - n * block_size)
    return lens, table


def dcp_decode_step(local_partial, merge, group=None):
    """One rank's DCP step.  `local_partial()` -> (out [T, H, D], lse [T, H]) of
    this rank's shard; the partials of all ranks are gathered (rank order) and
    `merge(outs [P, T, H, D], lses [P, T, H])` combines them.  Returns what
    `merge` returns.  With no process group (or world size 1) the local
    partial is the whole result's only part."""
    import torch
    import torch.distributed as dist

    out, lse = local_partial()
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return merge(out.unsqueeze(0), lse.unsqueeze(0))
    world = dist.get_world_size(group)
    outs = [torch.empty_like(out) for _ in range(world)]
    lses = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(outs, out.contiguous(), group=group)
    dist.all_gather(lses, lse.contiguous(), group=group)
    return merge(torch.stack(outs), torch.stack(lses))


def gpu_local_partial(query, kv_cache, local_meta, scale=None, workspace=None):
    """The rank's partial on its GPU through the library: (out bf16, lse fp32 ln).
    A shard with no key of some (or every) sequence is served by the library
    too: those rows come back as out = 0, lse = -inf, the merge's identity."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    T, H, D = query.shape
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=query.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=query.device)
    pka.paged_attn_forward(query, kv_cache, local_meta, out, lse, scale=scale, causal=True,
                           workspace=workspace)
    return out, lse


def gpu_merge(outs, lses, lse_base=0):
    """pka_merge_partials on the GPU: (out bf16 [T, H, D], lse fp32 [T, H])."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    P, T, H, D = outs.shape
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=outs.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=outs.device)
    pka.merge_partials(outs.contiguous(), lses.contiguous(), out, lse, lse_base=lse_base)
    return out, lse
