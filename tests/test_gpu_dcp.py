"""GPU parity of decode context parallelism and of pka_merge_partials.

The ranks of a context-parallel group are run one after another on one GPU
(each an ordinary forward over its shard of the keys, no rank waits on
another), their partials merged by pka_merge_partials and compared with the
fp64 oracle's unsharded attention; the lse-base flag is checked both ways
(the "AttentionBackend" page, "Limites y fallos": a wrong base breaks the
softmax denominator across shards)."""
import math

import numpy as np
import pytest

from paged_kv_attention_33_gb300 import dcp
from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G


# lse unit changes of the base-flag checks (test-side only: the library takes
# the base as an argument and converts nothing in Python)
_LN2 = math.log(2.0)


def _ln_to_log2(lse):
    return lse / _LN2


def _log2_to_ln(lse):
    return lse * _LN2


pytestmark = pytest.mark.gpu


def _partials(b, world, dev):
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = b.spec
    q = G.to_dev(b.query, dev)
    cache = G.to_dev(b.cache, dev)
    pka.reshape_and_cache(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                          torch.from_numpy(b.slot_mapping).to(dev))
    outs, lses = [], []
    for r in range(world):
        lens, table = dcp.shard_decode_metadata(b.seq_lens, b.block_table, sp.block_size, r,
                                                world)
        meta = pka.Meta.from_host(b.query_start_loc, lens, table, sp.num_decodes, dev)
        o, l = dcp.gpu_local_partial(q, cache, meta, scale=sp.softmax_scale)
        outs.append(o)
        lses.append(l)
    pka.check_status()
    return torch.stack(outs), torch.stack(lses)


def _reference(oracle, b):
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(G.host_bits(b.key), G.host_bits(b.value), want, b.slot_mapping)
    return G.oracle_expected(oracle, b, want)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
@pytest.mark.parametrize("H,Hkv,D,bs", [(32, 8, 128, 16), (8, 2, 64, 64)])
def test_dcp_decode_matches_unsharded(oracle, world, H, Hkv, D, bs):
    # lengths below, at and above world*bs, so that some ranks hold nothing
    ctx = [0, 5, bs - 1, bs, 2 * bs + 3, 4 * bs, 300, 1000, 2500]
    sp = W.BatchSpec(f"dcp{world}", H, Hkv, D, bs, decode_ctx=ctx)
    b = W.make_batch(sp, seed=8000 + world + bs)
    outs, lses = _partials(b, world, "cuda")
    out, lse = dcp.gpu_merge(outs, lses)
    o_ref, l_ref = _reference(oracle, b)
    rows = np.arange(b.num_tokens * H, dtype=np.int64)
    res = G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, H)
    G.assert_close(res, f"dcp world={world}")


def test_dcp_lse_base_flag():
    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("dcp_base", 32, 8, 128, 16, decode_ctx=[100, 700, 3000, 33])
    b = W.make_batch(sp, seed=8100)
    outs, lses = _partials(b, 3, "cuda")
    o_e, l_e = dcp.gpu_merge(outs, lses, lse_base=pka.LSE_BASE_E)
    o_2, l_2 = dcp.gpu_merge(outs, _ln_to_log2(lses), lse_base=pka.LSE_BASE_2)
    diff = (o_e.float() - o_2.float()).abs().max().item()
    assert diff <= 1e-2, diff
    assert (_log2_to_ln(l_2) - l_e).abs().max().item() <= 1e-4
    # log2 partials merged as if natural-log: visibly wrong
    o_bad, _ = dcp.gpu_merge(outs, _ln_to_log2(lses), lse_base=pka.LSE_BASE_E)
    assert (o_bad.float() - o_e.float()).abs().max().item() > 5e-2


def test_merge_partials_kernel_against_oracle(oracle):
    import torch

    import paged_kv_attention_33_gb300 as pka

    rng = np.random.Generator(np.random.PCG64(12))
    P, T, H, D = 5, 13, 8, 128
    outs = W.f32_to_bf16_bits(rng.standard_normal((P, T, H, D), dtype=np.float32))
    lses = (rng.standard_normal((P, T, H)) * 3).astype(np.float32)
    lses[0, 0] = -np.inf
    lses[:, 1] = -np.inf          # a row with no keys anywhere
    lses[1:, 2] = -np.inf         # a row with keys in one part only
    dev = "cuda"
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    pka.merge_partials(W.to_device(outs, dev), torch.from_numpy(lses).to(dev), out, lse)
    pka.check_status()
    f = lambda x: W.bf16_bits_to_f32(x).astype(np.float64).reshape(T * H, D)
    o_ref, l_ref = f(outs[0]), lses[0].astype(np.float64).ravel()
    for p in range(1, P):
        o_ref, l_ref = oracle.lse_merge(o_ref, l_ref, f(outs[p]), lses[p].astype(np.float64).ravel())
    got = W.bf16_bits_to_f32(W.to_host_bits(out)).astype(np.float64).reshape(T * H, D)
    assert np.max(np.abs(got - o_ref)) <= 2e-2
    lg = lse.cpu().numpy().astype(np.float64).ravel()
    empty = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[empty])) and np.all(got[empty] == 0)
    assert np.max(np.abs(lg[~empty] - l_ref[~empty])) <= 1e-3
    # out may not alias the partials
    with pytest.raises(pka.PkaError):
        o = W.to_device(outs, dev)
        pka.merge_partials(o, torch.from_numpy(lses).to(dev), o[2], None)


@pytest.mark.parametrize("world", [1, 2, 4])
def test_dcp_over_an_fp8_pool(oracle, world):
    """The same sharding over an fp8 e4m3 pool (per-tensor scales): every rank
    runs the fp8 decode on its shard (some shards empty), the partials merge to
    the oracle's unsharded fp8 attention."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec(f"dcp8_{world}", 32, 8, 128, 16, decode_ctx=[0, 5, 15, 16, 35, 300, 2500])
    b = W.make_batch(sp, seed=8200 + world)
    ks, vs = 0.05, 0.04
    c = G.host_bits(b.cache)
    pool = np.empty(c.shape, dtype=np.uint8)
    pool[:, 0] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 0]), ks)
    pool[:, 1] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 1]), vs)
    dev = "cuda"
    cache = torch.from_numpy(pool).to(dev)
    pka.reshape_and_cache_fp8(G.to_dev(b.key, dev), G.to_dev(b.value, dev), cache,
                              torch.from_numpy(b.slot_mapping).to(dev), ks, vs)
    q = G.to_dev(b.query, dev)
    outs, lses = [], []
    for r in range(world):
        lens, table = dcp.shard_decode_metadata(b.seq_lens, b.block_table, sp.block_size, r,
                                                world)
        meta = pka.Meta.from_host(b.query_start_loc, lens, table, sp.num_decodes, dev,
                                  kv_dtype="fp8", k_scale=ks, v_scale=vs)
        o, l = dcp.gpu_local_partial(q, cache, meta, scale=sp.softmax_scale)
        outs.append(o)
        lses.append(l)
    pka.check_status()
    out, lse = dcp.gpu_merge(torch.stack(outs), torch.stack(lses))
    oracle.reshape_and_cache_fp8(b.key, b.value, pool, b.slot_mapping, ks, vs)
    o_ref, l_ref = oracle.paged_attention_fp8(b.query, pool, ks, vs, b.query_start_loc,
                                              b.seq_lens, b.block_table, sp.softmax_scale)
    rows = np.arange(b.num_tokens * sp.num_heads, dtype=np.int64)
    res = G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, sp.num_heads)
    G.assert_close(res, f"dcp fp8 world={world}")


@pytest.mark.parametrize("H,Hkv,D,bs", [(32, 8, 128, 16), (8, 2, 64, 64)])
def test_dcp_shard_without_any_key(oracle, H, Hkv, D, bs):
    """Every sequence fits in one page, so ranks 1 and 2 hold no key at all
    (their max_seq_len is 0): the library itself returns out = 0, lse = -inf
    for those shards (one kv head per warp, and several warps per kv head),
    and the merge gives the unsharded result."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("dcp_empty", H, Hkv, D, bs, decode_ctx=[0, 3, bs - 1])
    b = W.make_batch(sp, seed=8200 + bs)
    outs, lses = _partials(b, 3, "cuda")
    for r in (1, 2):
        lens, _ = dcp.shard_decode_metadata(b.seq_lens, b.block_table, bs, r, 3)
        assert int(lens.max()) == 0
        assert torch.all(outs[r].float() == 0) and torch.all(torch.isneginf(lses[r]))
    out, lse = dcp.gpu_merge(outs, lses)
    pka.check_status()
    o_ref, l_ref = _reference(oracle, b)
    rows = np.arange(b.num_tokens * H, dtype=np.int64)
    G.assert_close(G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows, H),
                   "dcp empty shards")


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_merges_flag_a_non_finite_lse(bad):
    """A partial whose lse is +inf or NaN is no attention result (a corrupt
    input): both merge kernels report it through the device error word
    instead of spreading NaN unnoticed; -inf (an empty part) stays valid."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    T, H, D = 5, 4, 64
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(8300)
    outs = torch.randn((2, T, H, D), generator=g, device=dev).to(torch.bfloat16)
    lses = torch.randn((2, T, H), generator=g, device=dev)
    lses[0, 1, 2] = float("-inf")
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    pka.merge_partials(outs, lses, out, lse)
    pka.cascade_merge(outs[0], lses[0], outs[1], lses[1], out, lse)
    pka.check_status()  # -inf is an empty part, not an error
    lses[1, 3, 0] = bad
    pka.merge_partials(outs, lses, out, lse)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5 and "+inf or NaN" in str(e.value)
    pka.cascade_merge(outs[0], lses[0], outs[1], lses[1], out, lse)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5
    pka.check_status()  # the error word was cleared
