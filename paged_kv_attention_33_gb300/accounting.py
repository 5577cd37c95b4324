"""Algorithmic work of one attention step, for throughput and roofline figures.

Counting rules:
 * decode: the K and V rows each decode reads, once per kv head (the query
   heads of a kv head share the read), bf16: sum_s (L_s - kv_begin) * Hkv * D
   * 2 (K and V) * 2 bytes.  Queries, outputs and metadata are not counted.
 * prefill: 4 * D flops per query head per admitted (query, key) pair (one
   multiply-add for Q.K and one for P.V per dimension); masked pairs that the
   kernel skips are not counted.
 * cascade: prefix tokens are read once for the whole batch instead of once
   per request (the blog post "El especialista del plato estrella",
   "Que aporta FlashInfer: JIT y cascade attention").
"""
from __future__ import annotations

from .workloads import BatchSpec

BF16 = 2


def decode_kv_bytes(spec: BatchSpec, kv_begin: int = 0, elem_bytes: int = BF16) -> int:
    """K and V bytes the decodes read (elem_bytes 1 for an fp8 e4m3 pool)."""
    row = spec.num_kv_heads * spec.head_size * 2 * elem_bytes
    return sum(max(0, L - kv_begin) for L in spec.seq_lens[: spec.num_decodes]) * row


def admitted_pairs(q_len: int, ctx: int, causal: bool = True, key_lo: int = 0) -> int:
    """Number of (query, key) pairs with key >= key_lo that the mask admits for a
    sequence of q_len queries after ctx prior tokens."""
    total = 0
    L = ctx + q_len
    if not causal:
        return q_len * max(0, L - key_lo)
    # query i admits keys [key_lo, ctx + i]
    for_i0 = ctx - key_lo + 1
    if for_i0 >= 1:
        total = q_len * for_i0 + q_len * (q_len - 1) // 2
    else:
        for i in range(q_len):
            total += max(0, ctx + i + 1 - key_lo)
    return total


def prefill_flops(spec: BatchSpec, key_lo: int = 0) -> int:
    pairs = sum(admitted_pairs(q, c, spec.causal, key_lo) for q, c in spec.prefill)
    return 4 * spec.head_size * spec.num_heads * pairs


def decode_flops(spec: BatchSpec, kv_begin: int = 0) -> int:
    keys = sum(max(0, L - kv_begin) for L in spec.seq_lens[: spec.num_decodes])
    return 4 * spec.head_size * spec.num_heads * keys


def cascade_prefix_token_reads(num_requests: int, prefix_len: int, suffix_lens) -> tuple:
    """(naive, cascade) token reads for R requests sharing a P-token prefix:
    naive reads the prefix once per request, sum_i (P + s_i); the cascade
    reads it once, P + sum_i s_i."""
    s = sum(suffix_lens)
    return num_requests * prefix_len + s, prefix_len + s


def decode_intensity_page_counting(bytes_per_element: int) -> float:
    """Decode arithmetic intensity the way the blog post counts it: about L*d
    operations over L*d*s bytes, i.e. 1/s."""
    return 1.0 / bytes_per_element
