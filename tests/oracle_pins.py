"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin takes an ``Oracle`` (the real one, or a planted-mistake variant) and
returns ``(ok, detail)``.  The pins are chosen so that a plausible mistake in
any step of the oracle (a dropped scale, a wrong sign, the wrong kv head, an
off-by-one on the causal diagonal, K and V swapped, a wrong in-page offset, a
wrong logarithm base, a merge term dropped, a wrong cache slot) fails at least
one of them; tests/test_oracle_mutants.py proves that for each such mistake.

What they compare against:
 * dense_bruteforce: the textbook dense softmax(scale*Q K^T + causal mask) V
   with scipy's softmax/logsumexp on contiguous K/V gathered independently
   with numpy fancy indexing;
 * closed forms: one key (out = V_0, lse = scale*<q,K_0>), a zero query
   (out = mean of the admitted V rows, lse = ln #admitted), constant V rows;
 * invariances the paged layout must have: any permutation of the physical
   blocks, any block_size;
 * exact re-association: split-KV and prefix/suffix (cascade) merges equal the
   unsplit result; a decode equals the last row of the matching prefill;
 * the cache write as a closed-form byte copy.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import logsumexp, softmax

from paged_kv_attention_33_gb300 import workloads as W

TOL = 1e-12


def _values(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def write_new_rows_numpy(batch: W.Batch) -> np.ndarray:
    """Cache with this step's rows placed by plain numpy indexing."""
    cache = batch.cache.copy()
    bs = batch.spec.block_size
    s = batch.slot_mapping
    keep = s >= 0
    cache[s[keep] // bs, 0, s[keep] % bs] = batch.key[keep]
    cache[s[keep] // bs, 1, s[keep] % bs] = batch.value[keep]
    return cache


def dense_reference(batch: W.Batch, cache: np.ndarray):
    """Textbook attention per sequence on contiguous K/V; returns out [T*H, D], lse [T*H]."""
    sp = batch.spec
    H, Hkv, D, bs = sp.num_heads, sp.num_kv_heads, sp.head_size, sp.block_size
    g = H // Hkv
    T = batch.num_tokens
    q = _values(batch.query)
    out = np.zeros((T, H, D))
    lse = np.zeros((T, H))
    for s in range(len(batch.seq_lens)):
        L = int(batch.seq_lens[s])
        t0, t1 = int(batch.query_start_loc[s]), int(batch.query_start_loc[s + 1])
        nq = t1 - t0
        if nq == 0:
            continue
        ctx = L - nq
        blocks = batch.block_table[s, : math.ceil(L / bs)]
        K = _values(cache[blocks, 0]).reshape(-1, Hkv, D)[:L]
        V = _values(cache[blocks, 1]).reshape(-1, Hkv, D)[:L]
        i = np.arange(nq)[:, None]
        j = np.arange(L)[None, :]
        allowed = (j <= ctx + i) if sp.causal else np.ones((nq, L), bool)
        for h in range(H):
            kv = h // g
            logits = sp.softmax_scale * (q[t0:t1, h] @ K[:, kv].T)
            logits = np.where(allowed, logits, -np.inf)
            out[t0:t1, h] = softmax(logits, axis=1) @ V[:, kv]
            lse[t0:t1, h] = logsumexp(logits, axis=1)
    return out.reshape(T * H, D), lse.reshape(T * H)


def run_oracle(oracle, batch: W.Batch, cache: np.ndarray, **kw):
    sp = batch.spec
    return oracle.paged_attention(batch.query, cache, batch.query_start_loc, batch.seq_lens,
                                  batch.block_table, sp.softmax_scale, sp.causal, **kw)


def _close(a, b, tol=TOL):
    a = np.asarray(a)
    b = np.asarray(b)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    err = np.where(same_inf, 0.0, np.abs(a - b))
    err = np.where(np.isnan(err), np.inf, err)
    worst = float(np.max(err)) if err.size else 0.0
    return bool(np.all(np.isfinite(err)) and worst <= tol), worst


def tiny_specs():
    """Small shapes covering decode, prefill with and without context, GQA 1/4,
    block sizes 16 and 32, lengths 1, exact multiples of the block size and
    ragged tails."""
    return [
        W.BatchSpec("t_decode", 8, 2, 64, 16, decode_ctx=[0, 15, 16, 40, 199]),
        W.BatchSpec("t_prefill", 4, 4, 64, 16, prefill=[(1, 0), (17, 0), (32, 0)]),
        W.BatchSpec("t_chunked", 8, 2, 64, 32, decode_ctx=[5, 63],
                    prefill=[(9, 23), (40, 64)], table_pad=2),
        W.BatchSpec("t_gqa8", 16, 2, 128, 16, decode_ctx=[30], prefill=[(12, 7)]),
    ]


# --------------------------------------------------------------------------- pins

def pin_dense_bruteforce(oracle):
    worst = 0.0
    for k, sp in enumerate(tiny_specs()):
        b = W.make_batch(sp, seed=100 + k)
        cache = write_new_rows_numpy(b)
        o_ref, l_ref = dense_reference(b, cache)
        o, l = run_oracle(oracle, b, cache)
        ok1, e1 = _close(o, o_ref)
        ok2, e2 = _close(l, l_ref)
        worst = max(worst, e1, e2)
        if not (ok1 and ok2):
            return False, f"{sp.name}: out err {e1:.3g}, lse err {e2:.3g}"
    return True, f"max err {worst:.3g}"


def pin_single_key(oracle):
    """L = 1: out = V_0 and lse = scale * <q, K_0>."""
    sp = W.BatchSpec("one", 4, 2, 64, 16, decode_ctx=[0, 0, 0])
    b = W.make_batch(sp, seed=7)
    cache = write_new_rows_numpy(b)
    o, l = run_oracle(oracle, b, cache)
    q = _values(b.query)
    k = _values(b.key)
    v = _values(b.value)
    g = sp.num_heads // sp.num_kv_heads
    for t in range(3):
        for h in range(sp.num_heads):
            r = t * sp.num_heads + h
            want_l = sp.softmax_scale * float(np.dot(q[t, h], k[t, h // g]))
            if not (_close(o[r], v[t, h // g])[0] and abs(l[r] - want_l) <= TOL):
                return False, f"token {t} head {h}"
    return True, "ok"


def pin_zero_query(oracle):
    """q = 0: all admitted keys weigh the same -> mean of V, lse = ln(#admitted)."""
    sp = W.BatchSpec("zq", 4, 1, 64, 16, decode_ctx=[20], prefill=[(6, 10)])
    b = W.make_batch(sp, seed=8)
    b.query[:] = 0
    cache = write_new_rows_numpy(b)
    o, l = run_oracle(oracle, b, cache)
    H, bs = sp.num_heads, sp.block_size
    for s in range(2):
        L = int(b.seq_lens[s])
        t0, t1 = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
        ctx = L - (t1 - t0)
        blocks = b.block_table[s, : math.ceil(L / bs)]
        V = _values(cache[blocks, 1]).reshape(-1, 1, 64)[:L, 0]
        for i in range(t1 - t0):
            n = ctx + i + 1
            for h in range(H):
                r = (t0 + i) * H + h
                if not (_close(o[r], V[:n].mean(axis=0), 1e-12)[0]
                        and abs(l[r] - math.log(n)) <= TOL):
                    return False, f"seq {s} query {i}"
    return True, "ok"


def pin_constant_v(oracle):
    """All V rows equal -> out is that row for every query, whatever the weights."""
    sp = W.BatchSpec("cv", 8, 2, 64, 16, decode_ctx=[50], prefill=[(20, 5)])
    b = W.make_batch(sp, seed=9)
    row = b.value[0].copy()
    cache = write_new_rows_numpy(b)
    cache[:, 1] = row[None, None]
    o, _ = run_oracle(oracle, b, cache)
    g = sp.num_heads // sp.num_kv_heads
    want = _values(row)
    for r in range(o.shape[0]):
        h = r % sp.num_heads
        if not _close(o[r], want[h // g], 1e-12)[0]:
            return False, f"row {r}"
    return True, "ok"


def _repage(batch: W.Batch, cache: np.ndarray, new_bs: int, seed: int):
    """Same logical K/V stored at another block size, blocks shuffled anew."""
    sp = batch.spec
    Hkv, D = sp.num_kv_heads, sp.head_size
    lens = [int(x) for x in batch.seq_lens]
    need = [math.ceil(L / new_bs) for L in lens]
    nb = sum(need)
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(nb)
    table = np.full((len(lens), max(need)), -1, np.int32)
    new = np.full((nb, 2, new_bs, Hkv, D), W.BF16_NAN, np.uint16)
    cur = 0
    for s, L in enumerate(lens):
        table[s, : need[s]] = perm[cur: cur + need[s]]
        cur += need[s]
        old = batch.block_table[s, : math.ceil(L / sp.block_size)]
        for kv in range(2):
            rows = cache[old, kv].reshape(-1, Hkv, D)[:L]
            flat = np.full((need[s] * new_bs, Hkv, D), W.BF16_NAN, np.uint16)
            flat[:L] = rows
            new[table[s, : need[s]], kv] = flat.reshape(need[s], new_bs, Hkv, D)
    sp2 = W.BatchSpec(sp.name, sp.num_heads, Hkv, D, new_bs, sp.decode_ctx, sp.prefill,
                      scale=sp.scale, causal=sp.causal)
    return W.Batch(sp2, batch.query, batch.key, batch.value, new, batch.slot_mapping,
                   batch.query_start_loc, batch.seq_lens, table, nb), new


def pin_block_size_invariance(oracle):
    sp = W.BatchSpec("bsi", 8, 2, 64, 16, decode_ctx=[3, 100], prefill=[(33, 40)])
    b = W.make_batch(sp, seed=10)
    cache = write_new_rows_numpy(b)
    o0, l0 = run_oracle(oracle, b, cache)
    worst = 0.0
    for k, nbs in enumerate((16, 32, 64, 128)):
        b2, c2 = _repage(b, cache, nbs, seed=50 + k)
        o, l = run_oracle(oracle, b2, c2)
        ok1, e1 = _close(o, o0)
        ok2, e2 = _close(l, l0)
        worst = max(worst, e1, e2)
        if not (ok1 and ok2):
            return False, f"block_size {nbs}: {e1:.3g} {e2:.3g}"
    return True, f"max err {worst:.3g}"


def pin_block_permutation(oracle):
    sp = W.BatchSpec("perm", 8, 2, 64, 16, decode_ctx=[70, 9], prefill=[(25, 31)])
    b = W.make_batch(sp, seed=11)
    cache = write_new_rows_numpy(b)
    o0, l0 = run_oracle(oracle, b, cache)
    rng = np.random.Generator(np.random.PCG64(12))
    for _ in range(3):
        pi = rng.permutation(b.num_blocks)          # new physical id of old block x: pi[x]
        new = np.empty_like(cache)
        new[pi] = cache
        table = np.where(b.block_table >= 0, pi[np.maximum(b.block_table, 0)], -1)
        b2 = W.Batch(sp, b.query, b.key, b.value, new, b.slot_mapping, b.query_start_loc,
                     b.seq_lens, table.astype(np.int32), b.num_blocks)
        o, l = run_oracle(oracle, b2, new)
        if not (_close(o, o0)[0] and _close(l, l0)[0]):
            return False, "output changed under a block permutation"
    return True, "ok"


def pin_split_merge(oracle):
    """Attention over [0,m) merged with [m,L) by log-sum-exp equals [0,L)."""
    sp = W.BatchSpec("split", 8, 2, 64, 16, decode_ctx=[150, 40], prefill=[(30, 20)])
    b = W.make_batch(sp, seed=13)
    cache = write_new_rows_numpy(b)
    o0, l0 = run_oracle(oracle, b, cache)
    worst = 0.0
    for m in (1, 16, 37, 64, 200):
        oa, la = run_oracle(oracle, b, cache, key_lo=0, key_hi=m)
        ob, lb = run_oracle(oracle, b, cache, key_lo=m, key_hi=-1)
        o, l = oracle.lse_merge(oa, la, ob, lb)
        ok1, e1 = _close(o, o0, 1e-11)
        ok2, e2 = _close(l, l0, 1e-11)
        worst = max(worst, e1, e2)
        if not (ok1 and ok2):
            return False, f"split at {m}: {e1:.3g} {e2:.3g}"
    return True, f"max err {worst:.3g}"


def pin_cascade_equals_plain(oracle):
    """Shared-prefix cascade (prefix once + suffix, merged) equals plain attention."""
    sp = W.BatchSpec("casc", 8, 2, 64, 16, decode_ctx=[64 + 5, 64 + 40, 64],
                     prefill=[(10, 70)], common_prefix_len=64)
    b = W.make_batch(sp, seed=14)
    cache = write_new_rows_numpy(b)
    o0, l0 = run_oracle(oracle, b, cache)
    o, l = oracle.cascade_attention(b.query, cache, b.query_start_loc, b.seq_lens,
                                    b.block_table, sp.softmax_scale, 64, sp.causal)
    ok1, e1 = _close(o, o0, 1e-11)
    ok2, e2 = _close(l, l0, 1e-11)
    if not (ok1 and ok2):
        return False, f"{e1:.3g} {e2:.3g}"
    # and the shared blocks really are shared
    if not np.all(b.block_table[:, :4] == b.block_table[0, :4]):
        return False, "prefix blocks not shared"
    return True, f"max err {max(e1, e2):.3g}"


def pin_merge_identity(oracle):
    rng = np.random.Generator(np.random.PCG64(15))
    o = rng.standard_normal((6, 8))
    l = rng.standard_normal(6)
    empty_o = np.zeros((6, 8))
    empty_l = np.full(6, -np.inf)
    m1, ml1 = oracle.lse_merge(o, l, empty_o, empty_l)
    m2, ml2 = oracle.lse_merge(empty_o, empty_l, o, l)
    m3, ml3 = oracle.lse_merge(empty_o, empty_l, empty_o, empty_l)
    ok = (_close(m1, o)[0] and _close(ml1, l)[0] and _close(m2, o)[0] and _close(ml2, l)[0]
          and np.all(m3 == 0) and np.all(np.isneginf(ml3)))
    # two equal halves: lse grows by ln 2, output unchanged
    m4, ml4 = oracle.lse_merge(o, l, o, l)
    ok = ok and _close(m4, o)[0] and _close(ml4, l + math.log(2.0))[0]
    return bool(ok), "ok" if ok else "merge identity broken"


def pin_decode_is_last_prefill_row(oracle):
    """A decode over L tokens equals the last query row of a causal prefill of
    the same L tokens (same K/V, same last query)."""
    Lp = 45
    sp_p = W.BatchSpec("pf", 8, 2, 64, 16, prefill=[(Lp, 0)])
    bp = W.make_batch(sp_p, seed=16)
    cache = write_new_rows_numpy(bp)
    op, lp = run_oracle(oracle, bp, cache)
    sp_d = W.BatchSpec("dc", 8, 2, 64, 16, decode_ctx=[Lp - 1])
    bd = W.Batch(sp_d, bp.query[Lp - 1:], bp.key[Lp - 1:], bp.value[Lp - 1:], cache,
                 bp.slot_mapping[Lp - 1:], np.array([0, 1], np.int32),
                 np.array([Lp], np.int32), bp.block_table, bp.num_blocks)
    od, ld = run_oracle(oracle, bd, cache)
    H = sp_p.num_heads
    ok1, e1 = _close(od, op[(Lp - 1) * H:])
    ok2, e2 = _close(ld, lp[(Lp - 1) * H:])
    return ok1 and ok2, f"{e1:.3g} {e2:.3g}"


def pin_cache_write(oracle):
    """Cache write is the closed-form byte copy; padding slots are skipped and
    every other byte of the pool is unchanged."""
    sp = W.BatchSpec("cw", 4, 2, 64, 16, decode_ctx=[3, 17], prefill=[(21, 10)], pool_blocks=12)
    b = W.make_batch(sp, seed=17)
    slots = b.slot_mapping.copy()
    slots[2] = -1                       # a padding token
    before = b.cache.copy()
    cache = b.cache.copy()
    oracle.reshape_and_cache(b.key, b.value, cache, slots)
    want = before.copy()
    bs = sp.block_size
    for t, s in enumerate(slots):
        if s < 0:
            continue
        want[s // bs, 0, s % bs] = b.key[t]
        want[s // bs, 1, s % bs] = b.value[t]
    if not np.array_equal(cache, want):
        return False, f"{int((cache != want).sum())} elements differ"
    bad = slots.copy()
    bad[0] = b.num_blocks * bs          # one past the pool
    try:
        oracle.reshape_and_cache(b.key, b.value, cache.copy(), bad)
        return False, "out-of-pool slot accepted"
    except ValueError:
        pass
    return True, "ok"


ALL_PINS = [
    pin_dense_bruteforce,
    pin_single_key,
    pin_zero_query,
    pin_constant_v,
    pin_block_size_invariance,
    pin_block_permutation,
    pin_split_merge,
    pin_cascade_equals_plain,
    pin_merge_identity,
    pin_decode_is_last_prefill_row,
    pin_cache_write,
]
