"""GPU parity of the fp8 (e4m3) KV pool (the "FlashAttention y FlashInfer"
page, "Resumen en una frase" and "Limites y fallos": an fp8 e4m3 KV cache;
one fp32 scale per tensor for K and for V).

The starting pool is the generated bf16 pool quantised by the oracle (the
prior context as earlier steps' writes would have left it; unused slots hold
bf16 NaN, i.e. the e4m3 NaN code, which no admitted key may touch).  The cache
write must match the oracle's codes byte for byte; attention rows are compared
with the oracle's fp64 attention over the dequantised pool at the bf16 path's
tolerances (the kernel computes on the exact code values, so quantisation
adds no error between the two sides).
"""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def fp8_pool(oracle, batch, k_scale, v_scale):
    c = G.host_bits(batch.cache)
    p8 = np.empty(c.shape, dtype=np.uint8)
    p8[:, 0] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 0]), k_scale)
    p8[:, 1] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 1]), v_scale)
    return p8


def run_fp8(batch, pool8, k_scale, v_scale, split_kv_tokens=0, fused=False, query=None,
            causal=True):
    """The fp8 write and forward through the C ABI; host copies of the logical
    pool codes, the output bits and the lse."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = G.device()
    sp = batch.spec
    q = G.to_dev(batch.query if query is None else query, dev)
    k = G.to_dev(batch.key, dev)
    v = G.to_dev(batch.value, dev)
    cache = W.to_layout(torch.from_numpy(pool8).to(dev), sp.kv_layout)
    slots = torch.from_numpy(batch.slot_mapping).to(dev)
    meta = pka.Meta.from_host(batch.query_start_loc, batch.seq_lens, batch.block_table,
                              sp.num_decodes, dev, split_kv_tokens=split_kv_tokens,
                              common_prefix_len=sp.common_prefix_len,
                              kv_layout=sp.kv_layout, kv_dtype="fp8", k_scale=k_scale,
                              v_scale=v_scale)
    T = batch.num_tokens
    out = torch.full((T, sp.num_heads, sp.head_size), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((T, sp.num_heads), float("nan"), dtype=torch.float32, device=dev)
    if fused:
        pka.paged_attn_forward_fused(q, k, v, slots, cache, meta, out, lse,
                                     scale=sp.softmax_scale, causal=causal)
    else:
        pka.reshape_and_cache_fp8(k, v, cache, slots, k_scale, v_scale, kv_layout=sp.kv_layout)
        pka.paged_attn_forward(q, cache, meta, out, lse, scale=sp.softmax_scale, causal=causal)
    pka.check_status()
    return (W.from_layout(cache, sp.kv_layout).cpu().numpy(), W.to_host_bits(out),
            lse.cpu().numpy())


# The kernel's scores are exact products (K codes and the prescaled Q are exact
# in f16) summed in fp32: their error is at most ~head_size * 2^-24 = 2^-17 of
# max_j scale * sum_i |K_ji q_i| (the usual bound of an fp32 sum of 128 terms).
ACCUM_REL = 2.0 ** -17


def score_bound(oracle, batch, pool8, k_scale, query):
    """Per row (t*H + h): max over the row's keys j of scale * sum_i |K_ji q_i|."""
    sp = batch.spec
    table = oracle.e4m3_value(np.arange(256, dtype=np.uint8))
    q = np.abs(W.bf16_bits_to_f32(query).astype(np.float64))  # [T, H, D]
    g = sp.num_heads // sp.num_kv_heads
    out = np.zeros(batch.num_tokens * sp.num_heads)
    for s_ in range(len(batch.seq_lens)):
        L = int(batch.seq_lens[s_])
        keys = np.arange(L)
        blk = batch.block_table[s_][keys // sp.block_size]
        kabs = np.abs(table[pool8[blk, 0, keys % sp.block_size]]) * k_scale  # [L, Hkv, D]
        for t in range(int(batch.query_start_loc[s_]), int(batch.query_start_loc[s_ + 1])):
            for h in range(sp.num_heads):
                out[t * sp.num_heads + h] = sp.softmax_scale * np.max(kabs[:, h // g] @ q[t, h])
    return out


def check_fp8(oracle, batch, k_scale, v_scale, split_kv_tokens=0, fused=False, label="",
              query=None, lse_rel_bound=0.0, causal=True):
    pool = fp8_pool(oracle, batch, k_scale, v_scale)
    want = pool.copy()
    oracle.reshape_and_cache_fp8(batch.key, batch.value, want, batch.slot_mapping, k_scale,
                                 v_scale)
    got_pool, out, lse = run_fp8(batch, pool, k_scale, v_scale, split_kv_tokens, fused, query,
                                 causal)
    assert np.array_equal(want, got_pool), f"{label}: fp8 cache write differs"
    sp = batch.spec
    qh = batch.query if query is None else query
    o_ref, l_ref = oracle.paged_attention_fp8(qh, want, k_scale, v_scale, batch.query_start_loc,
                                              batch.seq_lens, batch.block_table,
                                              sp.softmax_scale, causal=causal, threads=8)
    rows = np.arange(batch.num_tokens * sp.num_heads, dtype=np.int64)
    res = G.compare(out, None, o_ref, l_ref, rows, sp.num_heads)
    G.assert_close(res, label)
    t, h = rows // sp.num_heads, rows % sp.num_heads
    le = np.abs(lse[t, h].astype(np.float64) - l_ref)
    tol = G.LSE_ABS
    if lse_rel_bound:
        tol = tol + lse_rel_bound * score_bound(oracle, batch, want, k_scale, qh)[rows]
    assert np.all(np.isfinite(lse[t, h])) and np.all(le <= tol), \
        f"{label}: lse error {le.max()}"
    return out, lse, got_pool


def _decode_spec(name, H, Hkv, bs, ctx, layout="NHD"):
    return W.BatchSpec(name, H, Hkv, 128, bs, decode_ctx=ctx, kv_layout=layout)


@pytest.mark.parametrize("Hkv,g", [(8, 1), (8, 2), (8, 3), (8, 4), (4, 8), (2, 8), (1, 8), (1, 5)])
def test_fp8_decode_heads(oracle, Hkv, g):
    # lengths around the 16-key boxes and the 32-key units (L = ctx + 1)
    ctx = [0, 1, 14, 15, 16, 17, 30, 31, 32, 62, 63, 64, 100, 255, 256, 1000, 2047, 3001]
    sp = _decode_spec(f"fp8_{Hkv}_{g}", Hkv * g, Hkv, 16, ctx)
    b = W.make_batch(sp, seed=8000 + 10 * Hkv + g)
    check_fp8(oracle, b, 0.0625, 0.03125, label=f"Hkv={Hkv} g={g}")
    check_fp8(oracle, b, 0.0371, 0.0173, split_kv_tokens=48,
              label=f"Hkv={Hkv} g={g} split 48, non-power-of-two scales")


@pytest.mark.parametrize("Hkv,g", [(8, 4), (2, 8)])
@pytest.mark.parametrize("stages", [8, 9])
def test_fp8_decode_small_batch_division(oracle, Hkv, g, stages):
    """Both sides of the small-batch boundary (one sequence per CTA while the
    longest has at most 8 stages of 32*(8/Hkv) keys) over an fp8 pool."""
    sk = 32 * (8 // Hkv)
    ctx = [stages * sk - 1, 3 * sk, sk - 1, 0, 2 * sk + 5]  # L = ctx + 1
    sp = _decode_spec(f"fp8_small_{Hkv}_{g}_{stages}", Hkv * g, Hkv, 16, ctx)
    b = W.make_batch(sp, seed=8500 + 10 * Hkv + stages)
    check_fp8(oracle, b, 0.0625, 0.03125, label=f"Hkv={Hkv} longest {stages} stages")


@pytest.mark.parametrize("fused", [False, True])
def test_fp8_few_long_decodes(oracle, fused):
    """A few long decodes over an fp8 pool: their pieces merged by the launch
    after the decode's."""
    sp = _decode_spec("fp8_few_long", 32, 8, 16, [7000, 3001, 12, 4500])
    b = W.make_batch(sp, seed=8600)
    check_fp8(oracle, b, 0.0625, 0.03125, fused=fused, label=f"few long decodes fused={fused}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("bs", [16, 64, 256, 1024])
def test_fp8_decode_layouts_and_pages(oracle, layout, bs):
    ctx = [3, 200, 511, 1023, 1500, 4000]
    sp = _decode_spec(f"fp8_{layout}_{bs}", 32, 8, bs, ctx, layout)
    b = W.make_batch(sp, seed=8100 + bs)
    check_fp8(oracle, b, 0.05, 0.02, label=f"{layout} bs={bs}")
    check_fp8(oracle, b, 0.05, 0.02, split_kv_tokens=64, label=f"{layout} bs={bs} split 64")


def test_fp8_saturating_scale(oracle):
    """A scale small enough that many |x|/scale exceed 448: those codes clamp
    to +-448 in both the write and the oracle."""
    sp = _decode_spec("fp8_sat", 16, 4, 16, [40, 300])
    b = W.make_batch(sp, seed=8200)
    check_fp8(oracle, b, 1.0 / 256, 1.0 / 300, label="saturating")


@pytest.mark.parametrize("shift", [-24, -12, 12, 18])
@pytest.mark.parametrize("Hkv,g", [(8, 4), (4, 8)])
def test_fp8_query_far_from_unit_scale(oracle, shift, Hkv, g):
    """The kernel takes Q to f16 with a power-of-two prescale per head (bf16
    reaches past f16's range); queries scaled by 2^shift (past f16's largest
    value at +18, into its subnormals at -24) must give the oracle's rows.
    At +18 the logits are ~1e6 with heavy cancellation, where no fp32 sum
    resolves 1e-3: the lse may differ by the fp32 accumulation bound."""
    sp = _decode_spec(f"fp8_q{shift}_{g}", Hkv * g, Hkv, 16, [5, 77, 1000])
    b = W.make_batch(sp, seed=8300 + shift + g)
    q = W.f32_to_bf16_bits(W.bf16_bits_to_f32(b.query) * np.float32(2.0 ** shift))
    check_fp8(oracle, b, 0.0625, 0.0625, query=q, label=f"q x 2^{shift} g={g}",
              lse_rel_bound=ACCUM_REL)


@pytest.mark.parametrize("Hkv,g", [(8, 4), (8, 2), (4, 8)])
def test_fp8_lse_bound_is_inside_the_tolerance(oracle, Hkv, g):
    """At ordinary scale the accumulation bound itself is far inside the lse
    tolerance, for every group size."""
    sp = _decode_spec(f"fp8_bound_{g}", Hkv * g, Hkv, 16, [300, 1000, 2500])
    b = W.make_batch(sp, seed=8350 + g)
    pool = fp8_pool(oracle, b, 0.0625, 0.0625)
    want = pool.copy()
    oracle.reshape_and_cache_fp8(b.key, b.value, want, b.slot_mapping, 0.0625, 0.0625)
    bound = score_bound(oracle, b, want, 0.0625, b.query)
    assert np.max(bound) * ACCUM_REL < G.LSE_ABS / 10
    check_fp8(oracle, b, 0.0625, 0.0625, label=f"accumulation bound g={g}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_fused_write_matches_two_calls(oracle, layout):
    """pka_paged_attn_forward_fused on an fp8 pool: the decode launch quantises
    each new row into its staged tile and its slot; pool bytes equal to the
    oracle's, rows equal to the oracle's, and bit-identical to the two calls."""
    sp = _decode_spec(f"fp8_fused_{layout}", 32, 8, 16, [0, 15, 16, 31, 500, 2000], layout)
    b = W.make_batch(sp, seed=8400)
    o1, l1, p1 = check_fp8(oracle, b, 0.04, 0.03, fused=True, label=f"fused {layout}")
    o2, l2, p2 = check_fp8(oracle, b, 0.04, 0.03, fused=False, label=f"two-call {layout}")
    assert np.array_equal(p1, p2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("layout,bs", [("NHD", 16), ("HND", 16), ("NHD", 64), ("HND", 256)])
def test_fp8_mixed_decode_and_prefill(oracle, layout, bs, fused):
    """Decodes and prefill chunks (with and without prior context, ragged 128-row
    tiles) over one fp8 pool: the decodes read the codes, the prefills run on
    the workspace's bf16 copy of their blocks; one call or two."""
    sp = W.BatchSpec(f"fp8_mixed_{layout}_{bs}", 32, 8, 128, bs, decode_ctx=[0, 17, 600],
                     prefill=[(1, 0), (130, 0), (257, 300), (64, 1100)], kv_layout=layout)
    b = W.make_batch(sp, seed=8600 + bs + (1 if layout == "HND" else 0))
    check_fp8(oracle, b, 0.04, 0.03, fused=fused, label=f"mixed {layout} bs={bs} fused={fused}")


def test_fp8_prefill_only_and_non_causal(oracle):
    """A batch of prefills alone over an fp8 pool (the fused call writes first,
    then attends), causal and not."""
    sp = W.BatchSpec("fp8_prefill", 16, 4, 128, 16, prefill=[(200, 0), (40, 70), (129, 512)])
    b = W.make_batch(sp, seed=8700)
    check_fp8(oracle, b, 0.06, 0.02, fused=True, label="prefill only, fused")
    check_fp8(oracle, b, 0.06, 0.02, label="prefill only, non-causal", causal=False)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("kind", ["decodes", "mixed", "prefills"])
def test_fp8_cascade(oracle, layout, kind):
    """A shared-prefix cascade over an fp8 pool: the prefix pass and the
    prefill suffixes run on bf16 copies of their blocks (the prefix read through
    row 0: a decode's blocks copied for it, or a prefill's own copy), the decode
    suffixes read the codes and merge the prefix partials in the kernel."""
    P = 256
    dec = {"decodes": [P + 3, P + 40, P + 700, P + 33], "mixed": [P + 10, P + 500],
           "prefills": []}[kind]
    pre = {"decodes": [], "mixed": [(40, P), (150, P + 20)], "prefills": [(60, P), (129, P + 5)]}[kind]
    sp = W.BatchSpec(f"fp8_casc_{kind}_{layout}", 32, 8, 128, 16, decode_ctx=dec, prefill=pre,
                     common_prefix_len=P, kv_layout=layout)
    b = W.make_batch(sp, seed=8950 + len(dec) + len(pre))
    check_fp8(oracle, b, 0.05, 0.04, label=f"cascade {kind} {layout}")
    check_fp8(oracle, b, 0.05, 0.04, fused=True, label=f"cascade {kind} {layout} fused")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_mixed_side_by_side(oracle, layout):
    """A mixed batch the plan runs side by side over an fp8 pool: the prefill
    blocks' bf16 copy, the decode over the codes on part of the SMs, the
    prefill pass as its programmatic dependent on the rest."""
    ctx = [2000 + 250 * k for k in range(16)]
    sp = W.BatchSpec(f"fp8_mixed_sbs_{layout}", 32, 8, 128, 64, decode_ctx=ctx,
                     prefill=[(256, 1000), (256, 1500)], kv_layout=layout)
    b = W.make_batch(sp, seed=8995)
    check_fp8(oracle, b, 0.05, 0.04, label=f"mixed side by side {layout}")
    check_fp8(oracle, b, 0.05, 0.04, fused=True, label=f"mixed side by side {layout} fused")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_cascade_side_by_side(oracle, layout):
    """A cascade the plan runs side by side over an fp8 pool: the prefix blocks'
    bf16 copy, the prefix pass as that copy's programmatic dependent, the
    suffix decode (over the codes) as the pass's, then the combine."""
    P = 1024
    rng = np.random.Generator(np.random.PCG64(7))
    ctx = (P + rng.integers(64, 800, size=48)).tolist()
    sp = W.BatchSpec(f"fp8_casc_sbs_{layout}", 32, 8, 128, 64, decode_ctx=ctx,
                     common_prefix_len=P, kv_layout=layout)
    b = W.make_batch(sp, seed=8990)
    check_fp8(oracle, b, 0.05, 0.04, label=f"cascade side by side {layout}")
    check_fp8(oracle, b, 0.05, 0.04, fused=True, label=f"cascade side by side {layout} fused")


def test_fp8_unserved_batches_are_refused(oracle):
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("fp8_d64", 16, 4, 64, 16, decode_ctx=[40, 50], prefill=[(20, 35)])
    b = W.make_batch(sp, seed=8500)
    dev = G.device()
    pool = torch.from_numpy(fp8_pool(oracle, b, 0.1, 0.1)).to(dev)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              dev, kv_dtype="fp8", k_scale=0.1, v_scale=0.1)
    q = G.to_dev(b.query, dev)
    with pytest.raises(pka.PkaError) as e:
        pka.paged_attn_forward(q, pool, meta, torch.empty_like(q))
    assert e.value.status == -2
    before = pool.clone()
    with pytest.raises(pka.PkaError) as e:
        pka.paged_attn_forward_fused(q, G.to_dev(b.key, dev), G.to_dev(b.value, dev),
                                     torch.from_numpy(b.slot_mapping).to(dev), pool, meta,
                                     torch.empty_like(q))
    assert e.value.status == -2
    torch.cuda.synchronize()
    assert torch.equal(before, pool)  # nothing was written


def test_fp8_decode_batch_above_one_launch(oracle):
    """4500 fp8 decodes: two decode launches, the fused write in each."""
    rng = np.random.Generator(np.random.PCG64(8800))
    ctx = [int(x) for x in rng.integers(0, 40, size=4500)]
    sp = _decode_spec("fp8_4500", 4, 1, 16, ctx)  # one kv head keeps the pool small
    b = W.make_batch(sp, seed=8801)
    check_fp8(oracle, b, 0.05, 0.05, fused=True, label="4500 fp8 decodes")


@pytest.mark.parametrize("which", ["decode", "prefill"])
def test_fp8_out_of_pool_block_is_flagged(oracle, which):
    """A block-table entry outside an fp8 pool is never read: the decode kernel
    (or, for a prefill, the block copy) skips it and flags it, and
    check_status reports PKA_ERR_DEVICE_CHECK once."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec(f"fp8_oob_{which}", 8, 1, 128, 16, decode_ctx=[40], prefill=[(20, 30)])
    b = W.make_batch(sp, seed=8900)
    table = b.block_table.copy()
    row = 0 if which == "decode" else 1
    table[row, 1] = b.num_blocks + 5
    dev = "cuda"
    pool = torch.from_numpy(fp8_pool(oracle, b, 0.05, 0.05)).to(dev)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, table, sp.num_decodes, dev,
                              kv_dtype="fp8", k_scale=0.05, v_scale=0.05)
    q = G.to_dev(b.query, dev)
    pka.paged_attn_forward(q, pool, meta, torch.empty_like(q), scale=sp.softmax_scale)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5
    pka.check_status()  # the error word was cleared
