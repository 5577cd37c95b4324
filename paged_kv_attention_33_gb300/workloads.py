"""Seeded synthetic batches for the paged-KV attention forward.

This module only draws inputs: sequence lengths, block tables, slot mappings,
queries, new K/V rows and the prior-context part of the paged pool.  It holds
none of the attention arithmetic and imports neither the CUDA binding nor the
oracle; both sides of every parity test receive the very same arrays from
here.

Conventions (the batch layout the pages describe):
 * query [num_tokens, num_heads, head_size] ("FlashAttention y FlashInfer"
   page, "Flujo de datos"), decode requests first, then prefill requests
   (same page, "Responsabilidades": decode-first order);
 * pool [num_blocks, 2, block_size, num_kv_heads, head_size], NHD, K at
   index 0 and V at index 1 (same page, get_kv_cache_shape);
 * query_start_loc [S+1], seq_lens [S], block_table [S, max_blocks] padded
   with -1 ("AttentionBackend" page, "Archivos clave": CommonAttentionMetadata);
 * seq_lens counts the whole KV length including this step's new tokens; the
   new K/V rows are written by reshape_and_cache through slot_mapping
   (slot = block * block_size + offset) before attention reads them;
 * every slot of the pool that no sequence uses, including the tail of each
   sequence's last block, holds a bf16 NaN so that any read of it shows.

Bulk values are N(0,1) drawn in fp32 and rounded to bf16 (round to nearest
even).  Small batches are drawn with numpy's PCG64; large ones can be drawn
directly on a CUDA device with a seeded torch generator (``device="cuda"``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = 0x7FC0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


@dataclass
class BatchSpec:
    """Shape of one attention step: which requests, how long, which heads."""
    name: str
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    decode_ctx: list = field(default_factory=list)   # prior context of each decode (q = 1)
    prefill: list = field(default_factory=list)      # (query_len, prior_ctx) of each prefill
    common_prefix_len: int = 0                       # shared prefix tokens (cascade)
    pool_blocks: int | None = None                   # None: exactly the blocks in use
    scale: float | None = None                       # None: 1/sqrt(head_size)
    causal: bool = True
    table_pad: int = 0                               # extra -1 columns in block_table
    kv_layout: str = "NHD"                           # physical pool order: "NHD" or "HND"

    @property
    def num_decodes(self) -> int:
        return len(self.decode_ctx)

    @property
    def query_lens(self) -> list:
        return [1] * len(self.decode_ctx) + [q for q, _ in self.prefill]

    @property
    def seq_lens(self) -> list:
        return [c + 1 for c in self.decode_ctx] + [q + c for q, c in self.prefill]

    @property
    def num_tokens(self) -> int:
        return sum(self.query_lens)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_size)


# Seeds of the five workloads: the lengths of named_spec(name) are drawn from
# NAMED_SEEDS[name], and the benchmark draws the batch's values with the same
# seed (make_batch(named_spec(name), seed=NAMED_SEEDS[name])).
NAMED_SEEDS = {"tiny_decode": 1001, "decode_heavy": 1002, "prefill": 1003, "mixed": 1004,
               "cascade": 1005}


def named_spec(name: str, seed: int | None = None) -> BatchSpec:
    """The five synthetic workloads of the method (lengths drawn from `seed`).

    tiny_decode   4 decodes, L ~ U[1,200], H=8, Hkv=2, D=64, bs=16, pool of 64 blocks
    decode_heavy  128 decodes, prior context ~ U[512,8192], H=32, Hkv=8, D=128, bs=16
    prefill       8 prompts, N ~ U[1024,8192], no prior context, H=32, Hkv=8, D=128, bs=16
    mixed         64 decodes (context ~ U[1024,16384]) then 4 chunks of 2048 queries over
                  prior context ~ U[0,16384]; H=32, Hkv=8, D=128, bs=64
    cascade       256 decodes sharing a 4096-token prefix, private suffix ~ U[64,1024]
                  (the new token included); H=64, Hkv=8, D=128, bs=128
    """
    rng = np.random.Generator(np.random.PCG64(NAMED_SEEDS[name] if seed is None else seed))
    if name == "tiny_decode":
        lens = rng.integers(1, 200, size=4, endpoint=True)
        return BatchSpec(name, 8, 2, 64, 16, decode_ctx=[int(x) - 1 for x in lens],
                         pool_blocks=64, scale=1.0 / 8.0)
    if name == "decode_heavy":
        ctx = rng.integers(512, 8192, size=128, endpoint=True)
        return BatchSpec(name, 32, 8, 128, 16, decode_ctx=[int(x) for x in ctx])
    if name == "prefill":
        n = rng.integers(1024, 8192, size=8, endpoint=True)
        return BatchSpec(name, 32, 8, 128, 16, prefill=[(int(x), 0) for x in n])
    if name == "mixed":
        ctx = rng.integers(1024, 16384, size=64, endpoint=True)
        pc = rng.integers(0, 16384, size=4, endpoint=True)
        return BatchSpec(name, 32, 8, 128, 64, decode_ctx=[int(x) for x in ctx],
                         prefill=[(2048, int(c)) for c in pc])
    if name == "cascade":
        suf = rng.integers(64, 1024, size=256, endpoint=True)
        return BatchSpec(name, 64, 8, 128, 128, decode_ctx=[4096 + int(s) - 1 for s in suf],
                         common_prefix_len=4096)
    raise KeyError(name)


NAMED = ("tiny_decode", "decode_heavy", "prefill", "mixed", "cascade")


@dataclass
class Batch:
    """One step's inputs.  Bulk tensors are numpy uint16 (bf16 bits) on the host
    path and torch bfloat16 tensors on the device path; metadata is numpy."""
    spec: BatchSpec
    query: object            # [T, H, D]
    key: object              # [T, Hkv, D]   new rows of this step
    value: object            # [T, Hkv, D]
    cache: object            # [NB, 2, bs, Hkv, D] prior context filled, new slots poisoned
    slot_mapping: np.ndarray  # [T] int64
    query_start_loc: np.ndarray  # [S+1] int32
    seq_lens: np.ndarray     # [S] int32
    block_table: np.ndarray  # [S, max_blocks] int32, -1 padded
    num_blocks: int

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])


def _layout(spec: BatchSpec, rng: np.random.Generator):
    """Block tables, slot mapping and the list of prior-context slots to fill."""
    bs = spec.block_size
    P = spec.common_prefix_len
    qlens = spec.query_lens
    lens = spec.seq_lens
    S = len(lens)
    if P % bs != 0:
        raise ValueError("common_prefix_len must be a multiple of block_size")
    n_shared = P // bs
    need = [math.ceil(L / bs) for L in lens]
    private = [n - n_shared for n in need]
    if P > 0 and min(private) < 0:
        raise ValueError("a sequence is shorter than the shared prefix")
    used = n_shared + sum(private)
    nb = spec.pool_blocks if spec.pool_blocks is not None else used
    if nb < used:
        raise ValueError("pool too small")
    perm = rng.permutation(nb).astype(np.int64)
    shared = perm[:n_shared]
    width = max(need) + spec.table_pad
    table = np.full((S, max(width, 1)), -1, dtype=np.int32)
    cur = n_shared
    for s in range(S):
        table[s, :n_shared] = shared
        table[s, n_shared:need[s]] = perm[cur:cur + private[s]]
        cur += private[s]
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(qlens)
    T = int(qsl[-1])
    slots = np.empty(T, dtype=np.int64)
    ctx_slots = []
    for s in range(S):
        c = lens[s] - qlens[s]
        pos = np.arange(c, lens[s], dtype=np.int64)
        slots[qsl[s]:qsl[s + 1]] = table[s, pos // bs].astype(np.int64) * bs + pos % bs
        start = 0 if s == 0 else min(P, c)   # the shared prefix is filled once
        pos = np.arange(start, c, dtype=np.int64)
        ctx_slots.append(table[s, pos // bs].astype(np.int64) * bs + pos % bs)
    ctx_slots = np.concatenate(ctx_slots) if ctx_slots else np.zeros(0, np.int64)
    return nb, table, qsl, np.asarray(lens, dtype=np.int32), slots, ctx_slots


def make_batch(spec: BatchSpec, seed: int, device: str = "cpu") -> Batch:
    """Draw one batch.  device="cpu": numpy arrays; otherwise torch tensors on
    `device` drawn by a torch generator seeded with `seed`."""
    rng = np.random.Generator(np.random.PCG64(seed))
    nb, table, qsl, lens, slots, ctx_slots = _layout(spec, rng)
    T = int(qsl[-1])
    H, Hkv, D, bs = spec.num_heads, spec.num_kv_heads, spec.head_size, spec.block_size
    if device == "cpu":
        def normal(*shape):
            return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))

        query = normal(T, H, D)
        key = normal(T, Hkv, D)
        value = normal(T, Hkv, D)
        cache = np.full((nb, 2, bs, Hkv, D), BF16_NAN, dtype=np.uint16)
        blk, off = ctx_slots // bs, ctx_slots % bs
        cache[blk, 0, off] = normal(len(ctx_slots), Hkv, D)
        cache[blk, 1, off] = normal(len(ctx_slots), Hkv, D)
    else:
        import torch

        g = torch.Generator(device=device)
        g.manual_seed(seed)

        def normal(*shape):
            return torch.randn(shape, generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16)

        query = normal(T, H, D)
        key = normal(T, Hkv, D)
        value = normal(T, Hkv, D)
        cache = torch.full((nb, 2, bs, Hkv, D), float("nan"), device=device,
                           dtype=torch.bfloat16)
        cs = torch.from_numpy(ctx_slots).to(device)
        blk, off = cs // bs, cs % bs
        n = len(ctx_slots)
        # fill in slabs so the fp32 temporaries stay small
        step = 1 << 18
        for a in range(0, n, step):
            b = min(n, a + step)
            cache[blk[a:b], 0, off[a:b]] = normal(b - a, Hkv, D)
            cache[blk[a:b], 1, off[a:b]] = normal(b - a, Hkv, D)
    return Batch(spec, query, key, value, cache, slots, qsl, lens, table, nb)


E4M3_NAN = 0x7F


def random_fp8_pool(batch: Batch, seed: int, max_code: int = 0x48):
    """A seeded e4m3 pool shaped like batch.cache: every slot the bf16 pool fills
    holds a random finite code of magnitude code <= max_code (0x48 = 4.0), every
    slot it leaves NaN holds the e4m3 NaN code.  Codes are drawn directly (no
    quantisation): numpy for a host batch, a seeded torch generator on the
    batch's device otherwise.  Returns an array / tensor of uint8."""
    if isinstance(batch.cache, np.ndarray):
        rng = np.random.Generator(np.random.PCG64(seed))
        mag = rng.integers(0, max_code + 1, size=batch.cache.shape, dtype=np.uint8)
        sign = rng.integers(0, 2, size=batch.cache.shape, dtype=np.uint8) << 7
        codes = mag | sign
        codes[(batch.cache & 0x7FFF) > 0x7F80] = E4M3_NAN
        return codes
    import torch

    dev = batch.cache.device
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    mag = torch.randint(0, max_code + 1, batch.cache.shape, generator=g, device=dev,
                        dtype=torch.uint8)
    sign = torch.randint(0, 2, batch.cache.shape, generator=g, device=dev,
                         dtype=torch.uint8) * 128
    codes = mag | sign
    codes[torch.isnan(batch.cache)] = E4M3_NAN
    return codes


def to_layout(cache, kv_layout: str):
    """The pool in physical order `kv_layout`: NHD is the logical
    [NB, 2, bs, Hkv, D] itself, HND swaps the slot and head axes to
    [NB, 2, Hkv, bs, D] (numpy array or torch tensor, contiguous)."""
    if kv_layout.upper() == "NHD":
        return cache
    if isinstance(cache, np.ndarray):
        return np.ascontiguousarray(np.swapaxes(cache, 2, 3))
    return cache.transpose(2, 3).contiguous()


def from_layout(pool, kv_layout: str):
    """Inverse of to_layout: the logical [NB, 2, bs, Hkv, D] pool."""
    return to_layout(pool, kv_layout)  # swapping the two axes again undoes it


def to_host_bits(x) -> np.ndarray:
    """uint16 bf16 bits of a numpy array or a (device) torch bf16 tensor."""
    if isinstance(x, np.ndarray):
        return x
    import torch

    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_device(x: np.ndarray, device: str):
    """torch bf16 tensor on `device` holding the uint16 bits `x`."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)


def sample_rows(batch: Batch, n: int, seed: int) -> np.ndarray:
    """n distinct (token, head) rows r = t*H + h, always including the first and
    last token of every sequence (the ends of the causal range)."""
    H = batch.spec.num_heads
    T = batch.num_tokens
    rng = np.random.Generator(np.random.PCG64(seed))
    must = []
    q = batch.query_start_loc
    for s in range(len(q) - 1):
        if q[s + 1] > q[s]:
            must += [q[s], q[s + 1] - 1]
    must = np.unique(np.asarray(must, dtype=np.int64))
    rows = set((must * H + rng.integers(0, H, size=len(must))).tolist())
    total = T * H
    n = min(n, total)
    while len(rows) < n:
        rows.update(rng.integers(0, total, size=n - len(rows)).tolist())
    return np.asarray(sorted(rows)[: max(n, len(must))], dtype=np.int64)
