"""GPU parity of the cache write and the stream-K split-KV decode path against
the fp64 oracle (all calls go through the C ABI).  split_kv_tokens sets the
keys per CTA: small values spread a sequence over many CTAs (fused merge of
many pieces), 1 << 30 puts the whole batch on one CTA (every sequence one
piece)."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _spec(H, Hkv, D, bs, ctx, **kw):
    return W.BatchSpec(f"d_{H}_{Hkv}_{D}_{bs}", H, Hkv, D, bs, decode_ctx=list(ctx), **kw)


def test_tiny_decode_named(oracle):
    b = W.make_batch(W.named_spec("tiny_decode"), seed=2001)
    G.check_batch(oracle, b, label="tiny_decode")


@pytest.mark.parametrize("split", [0, 64, 128, 192, 1 << 30])
def test_tiny_decode_forced_splits(oracle, split):
    b = W.make_batch(W.named_spec("tiny_decode"), seed=2002)
    G.check_batch(oracle, b, split_kv_tokens=split, label=f"split {split}")


# lengths 1, one short of / exactly / one past a 16-key slice and a block
EDGE_CTX = [0, 14, 15, 16, 31, 32, 63, 64, 65, 127, 128, 129, 200, 511]


@pytest.mark.parametrize("H,Hkv,D,bs", [
    (8, 2, 64, 16),     # group 4, two kv heads (4 slices per stage)
    (32, 8, 128, 16),   # the decode-heavy shape
    (8, 1, 128, 32),    # group 8, one kv head
    (8, 4, 64, 64),     # group 2
    (8, 8, 128, 128),   # group 1
    (64, 8, 128, 128),  # group 8, the cascade shape
])
def test_decode_edges(oracle, H, Hkv, D, bs):
    b = W.make_batch(_spec(H, Hkv, D, bs, EDGE_CTX, table_pad=3), seed=2100 + H + Hkv + bs)
    for split in (0, 16 * (8 // Hkv), 48 * (8 // Hkv), 1 << 30):
        G.check_batch(oracle, b, split_kv_tokens=split, label=f"split {split}")


# A small batch (at most one 16*(8/Hkv)-key stage per SM) whose longest
# sequence has at most 8 stages is divided one sequence per CTA; one more stage
# (or more stages than SMs) and it is divided evenly again, its sequences split
# over CTAs.  Both sides of each boundary, for one, two and eight kv heads.
@pytest.mark.parametrize("H,Hkv,D,bs", [(8, 2, 64, 16), (32, 8, 128, 16), (8, 1, 128, 32)])
@pytest.mark.parametrize("stages", [8, 9])
def test_decode_small_batch_division(oracle, H, Hkv, D, bs, stages):
    sk = 16 * (8 // Hkv)  # keys per stage
    ctx = [stages * sk - 1, 3 * sk, sk - 1, 0, 2 * sk + 5]  # L = ctx + 1
    b = W.make_batch(_spec(H, Hkv, D, bs, ctx), seed=2300 + Hkv + stages)
    G.check_batch(oracle, b, label=f"longest {stages} stages")


@pytest.mark.parametrize("n", [152, 153])
def test_decode_one_stage_per_sm(oracle, n):
    """n one-stage decodes: one per SM (each CTA one sequence), or one more than
    the SMs (divided evenly)."""
    rng = np.random.Generator(np.random.PCG64(n))
    ctx = rng.integers(0, 16, size=n).tolist()
    b = W.make_batch(_spec(32, 8, 128, 16, ctx), seed=2400 + n)
    G.check_batch(oracle, b, label=f"{n} one-stage decodes")


# A decode-only batch of a few long decodes (at least four SMs per decode):
# every decode spreads over many CTAs and their pieces are merged by a launch
# over the whole GPU after the decode's.
@pytest.mark.parametrize("H,Hkv,D,bs", [(32, 8, 128, 16), (8, 2, 64, 64), (8, 1, 128, 32)])
def test_decode_few_long_decodes(oracle, H, Hkv, D, bs):
    ctx = [6000, 4097, 2500, 31, 5111]  # one of them inside a single CTA
    b = W.make_batch(_spec(H, Hkv, D, bs, ctx), seed=2500 + Hkv + D)
    G.check_batch(oracle, b, label="few long decodes")
    G.check_batch(oracle, b, split_kv_tokens=4096, label="few long decodes, 4096 keys per CTA")


def test_small_batch_longer_than_max_seq_len_is_flagged(oracle):
    """A decode-only batch that max_seq_len says the kernel divides one
    sequence per CTA skips the counter reset.  A decode longer than
    max_seq_len (too long for that division) is flagged, nothing is computed,
    and the next call is served."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = _spec(8, 2, 64, 16, [1000, 9, 30])  # 1,001 keys: 16 stages of 64 keys
    b = W.make_batch(sp, seed=2320)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, 3, "cuda")
    meta.max_seq_len = 64  # understated: one stage per decode by this bound
    q = G.to_dev(b.query, "cuda")
    out = torch.empty_like(q)
    pka.paged_attn_forward(q, G.to_dev(b.cache, "cuda"), meta, out, scale=sp.softmax_scale)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5
    pka.check_status()
    G.check_batch(oracle, b, label="the true max_seq_len")


def test_one_sequence_per_cta_ignores_counter_leftovers(oracle):
    """A workspace whose counters hold a split batch's piece counts serves a
    small batch divided one sequence per CTA (its counters are not reset)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = "cuda"
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device=dev)
    for ctx, seed in (([3000, 2000, 1500, 700], 2321), ([40, 100, 7, 0], 2322)):
        b = W.make_batch(_spec(32, 8, 128, 16, ctx), seed=seed)
        sp = b.spec
        want = G.host_bits(b.cache).copy()
        oracle.reshape_and_cache(G.host_bits(b.key), G.host_bits(b.value), want, b.slot_mapping)
        cache = G.to_dev(b.cache, dev)
        pka.reshape_and_cache(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                              torch.from_numpy(b.slot_mapping).to(dev))
        meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table,
                                  sp.num_decodes, dev)
        T = b.num_tokens
        out = torch.full((T, sp.num_heads, sp.head_size), float("nan"), dtype=torch.bfloat16,
                         device=dev)
        lse = torch.full((T, sp.num_heads), float("nan"), dtype=torch.float32, device=dev)
        pka.paged_attn_forward(G.to_dev(b.query, dev), cache, meta, out, lse,
                               scale=sp.softmax_scale, workspace=ws)
        pka.check_status()
        rows = np.arange(T * sp.num_heads, dtype=np.int64)
        o_ref, l_ref = G.oracle_expected(oracle, b, want, rows=rows)
        res = G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows,
                        sp.num_heads)
        G.assert_close(res, f"ctx {ctx}")


def test_decode_many_splits_ragged(oracle):
    rng = np.random.Generator(np.random.PCG64(5))
    ctx = rng.integers(1, 3000, size=24).tolist()
    b = W.make_batch(_spec(32, 8, 128, 16, ctx), seed=2200)
    G.check_batch(oracle, b, split_kv_tokens=64, label="64 keys per CTA")
    G.check_batch(oracle, b, split_kv_tokens=1000, label="1000 keys per CTA")
    G.check_batch(oracle, b, label="auto")


def test_out_of_pool_slot_is_flagged():
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = _spec(8, 2, 64, 16, [5, 9], pool_blocks=4)
    b = W.make_batch(sp, seed=2300)
    cache = G.to_dev(b.cache, "cuda")
    slots = b.slot_mapping.copy()
    slots[1] = 4 * 16          # one past the pool: skipped and flagged
    before = cache.clone()
    pka.reshape_and_cache(G.to_dev(b.key, "cuda"), G.to_dev(b.value, "cuda"), cache,
                          torch.from_numpy(slots).cuda())
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5
    pka.check_status()         # the error word was cleared
    # the good token landed, nothing else changed
    assert int((cache.view(torch.int16) != before.view(torch.int16)).sum()) > 0


def test_out_of_pool_block_is_flagged():
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = _spec(8, 2, 64, 16, [40, 9])
    b = W.make_batch(sp, seed=2301)
    table = b.block_table.copy()
    table[0, 1] = b.num_blocks + 7   # outside the pool
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, table, 2, "cuda")
    q = G.to_dev(b.query, "cuda")
    out = torch.empty_like(q)
    pka.paged_attn_forward(q, G.to_dev(b.cache, "cuda"), meta, out, scale=sp.softmax_scale)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5
    pka.check_status()


def test_cascade_merge_kernel(oracle):
    """pka_cascade_merge against the oracle's merge on the same bf16 inputs,
    including rows where one or both sides are empty (lse = -inf)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    rng = np.random.Generator(np.random.PCG64(9))
    T, H, D = 37, 8, 128
    oa = W.f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32))
    ob = W.f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32))
    la = (rng.standard_normal((T, H)) * 3).astype(np.float32)
    lb = (rng.standard_normal((T, H)) * 3).astype(np.float32)
    la[0, :] = -np.inf
    lb[1, :] = -np.inf
    la[2, :] = -np.inf
    lb[2, :] = -np.inf
    dev = "cuda"
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lo = torch.empty((T, H), dtype=torch.float32, device=dev)
    pka.cascade_merge(W.to_device(oa, dev), torch.from_numpy(la).to(dev), W.to_device(ob, dev),
                      torch.from_numpy(lb).to(dev), out, lo)
    pka.check_status()
    f = lambda x: W.bf16_bits_to_f32(x).astype(np.float64).reshape(T * H, D)
    o_ref, l_ref = oracle.lse_merge(f(oa), la.astype(np.float64).ravel(), f(ob),
                                    lb.astype(np.float64).ravel())
    got = W.bf16_bits_to_f32(W.to_host_bits(out)).astype(np.float64).reshape(T * H, D)
    assert np.max(np.abs(got - o_ref)) <= 2e-2
    lg = lo.cpu().numpy().astype(np.float64).ravel()
    both = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[both]))
    assert np.all(got[both] == 0)
    assert np.max(np.abs(lg[~both] - l_ref[~both])) <= 1e-3
    # in place (out aliases out_a)
    a = W.to_device(oa, dev)
    la_t = torch.from_numpy(la).to(dev)
    pka.cascade_merge(a, la_t, W.to_device(ob, dev), torch.from_numpy(lb).to(dev), a, la_t)
    pka.check_status()
    assert torch.equal(a.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("fused", [False, True])
def test_decode_batch_above_one_launch(oracle, fused):
    """More decodes than one decode launch takes (4096): the batch runs as two
    launches that reuse the partial slots and counters, the fused write's
    substitution happening in each; every row checked."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    rng = np.random.Generator(np.random.PCG64(2400))
    ctx = [int(x) for x in rng.integers(0, 40, size=4500)]
    sp = _spec(8, 2, 64, 16, ctx)
    b = W.make_batch(sp, seed=2401)
    if not fused:
        G.check_batch(oracle, b, label="4500 decodes")
        return
    dev = "cuda"
    cache = G.to_dev(b.cache, dev)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes, dev)
    q = G.to_dev(b.query, dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    pka.paged_attn_forward_fused(q, G.to_dev(b.key, dev), G.to_dev(b.value, dev),
                                 torch.from_numpy(b.slot_mapping).to(dev), cache, meta, out, lse,
                                 scale=sp.softmax_scale)
    pka.check_status()
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(b.key, b.value, want, b.slot_mapping)
    assert np.array_equal(want, W.to_host_bits(cache))
    o_ref, l_ref = oracle.paged_attention(b.query, want, b.query_start_loc, b.seq_lens,
                                          b.block_table, sp.softmax_scale, threads=8)
    rows = np.arange(b.num_tokens * sp.num_heads, dtype=np.int64)
    G.assert_close(G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows,
                             sp.num_heads), "4500 decodes fused")
