"""Decode context parallelism (the "FlashAttention y FlashInfer" page, "Limites
y fallos": the DCP combine across shards; the "AttentionBackend" page, "Limites
y fallos": the lse base of that combine).

Host part (no GPU): the key sharding, and a world-size-2 gloo run of the rank
step with the fp64 oracle as each rank's local attention, merged in fp64 --
equal to the oracle's unsharded result; merging log2 partials as if they were
natural-log ones gives a wrong result (the failure the page warns about)."""
import os
import socket
import math
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from paged_kv_attention_33_gb300 import dcp
from paged_kv_attention_33_gb300 import workloads as W


# lse unit changes of the base-flag checks (test-side only: the library takes
# the base as an argument and converts nothing in Python)
_LN2 = math.log(2.0)


def _ln_to_log2(lse):
    return lse / _LN2


def _log2_to_ln(lse):
    return lse * _LN2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_shards_partition_every_sequence(world):
    rng = np.random.Generator(np.random.PCG64(3))
    bs = 16
    lens = np.array([1, 15, 16, 17, 40, 100, 257, 1000])
    width = int(np.ceil(lens.max() / bs))
    table = rng.permutation(len(lens) * width).reshape(len(lens), width).astype(np.int32)
    seen = {s: [] for s in range(len(lens))}
    total = np.zeros(len(lens), dtype=np.int64)
    for r in range(world):
        ll, lt = dcp.shard_decode_metadata(lens, table, bs, r, world)
        total += ll
        for s in range(len(lens)):
            npages = int(np.ceil(ll[s] / bs))
            assert np.all(lt[s, npages:] == -1)
            owned = [n for n in range(int(np.ceil(lens[s] / bs))) if n % world == r]
            assert list(lt[s, :npages]) == [table[s, n] for n in owned]
            # every local page but the last is full
            assert ll[s] == sum(min(bs, lens[s] - n * bs) for n in owned)
            seen[s] += owned
    assert np.array_equal(total, lens)
    for s in range(len(lens)):
        assert sorted(seen[s]) == list(range(int(np.ceil(lens[s] / bs))))


def _merge64(outs, lses, base_e=True):
    """fp64 log-sum-exp merge of P partials (test reference), lse in ln or log2."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    scale = 1.0 if base_e else np.log(2.0)
    m = np.max(lses, axis=0)
    fin = np.isfinite(m)
    w = np.where(np.isfinite(lses), np.exp((lses - np.where(fin, m, 0.0)) * scale), 0.0)
    ws = w.sum(axis=0)
    out = np.where(ws[..., None] > 0, (w[..., None] * outs).sum(axis=0) /
                   np.where(ws > 0, ws, 1.0)[..., None], 0.0)
    lse = np.where(ws > 0, np.where(fin, m, 0.0) + np.log(np.where(ws > 0, ws, 1.0)) / scale,
                   -np.inf)
    return out, lse


def _spec():
    return W.BatchSpec("dcp", 8, 2, 64, 16, decode_ctx=[5, 40, 100, 250, 16])


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    from oracle import Oracle
    from paged_kv_attention_33_gb300 import dcp as D
    from paged_kv_attention_33_gb300 import workloads as WW

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sp = _spec()
    b = WW.make_batch(sp, seed=31)
    orc = Oracle()
    cache = b.cache.copy()
    orc.reshape_and_cache(b.key, b.value, cache, b.slot_mapping)
    lens, table = D.shard_decode_metadata(b.seq_lens, b.block_table, sp.block_size, rank, world)
    T, H = b.num_tokens, sp.num_heads

    def local():
        # rows of sequences this rank holds keys of; the others attend an
        # empty key set: out 0, lse -inf
        rows = np.array([t * H + h for s in range(len(lens)) if lens[s] > 0
                         for t in range(b.query_start_loc[s], b.query_start_loc[s + 1])
                         for h in range(H)], dtype=np.int64)
        o = np.zeros((T * H, sp.head_size))
        l = np.full(T * H, -np.inf)
        if rows.size:
            o[rows], l[rows] = orc.paged_attention(b.query, cache, b.query_start_loc, lens,
                                                   table, sp.softmax_scale, True, rows=rows)
        return (torch.from_numpy(o.reshape(T, H, -1)), torch.from_numpy(l.reshape(T, H)))

    def merge(outs, lses):
        return _merge64(outs.numpy(), lses.numpy())

    out, lse = D.dcp_decode_step(local, merge)
    # the same partials in log2 units, merged with the log2 base and (wrongly) with ln
    out2, lse2 = D.dcp_decode_step(
        lambda: (local()[0], torch.from_numpy(_ln_to_log2(local()[1].numpy()))),
        lambda o, l: _merge64(o.numpy(), l.numpy(), base_e=False))
    bad, _ = D.dcp_decode_step(
        lambda: (local()[0], torch.from_numpy(_ln_to_log2(local()[1].numpy()))),
        lambda o, l: _merge64(o.numpy(), l.numpy(), base_e=True))
    full_o, full_l = orc.paged_attention(b.query, cache, b.query_start_loc, b.seq_lens,
                                         b.block_table, sp.softmax_scale, True)
    q.put((rank, float(np.max(np.abs(out.reshape(T * H, -1) - full_o))),
           float(np.max(np.abs(lse.reshape(-1) - full_l))),
           float(np.max(np.abs(out2.reshape(T * H, -1) - full_o))),
           float(np.max(np.abs(_log2_to_ln(lse2.reshape(-1)) - full_l))),
           float(np.max(np.abs(bad.reshape(T * H, -1) - full_o)))))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_dcp_step_two_gloo_ranks_equals_unsharded():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, e_out, e_lse, e_out2, e_lse2, e_bad in res:
        assert e_out < 1e-12 and e_lse < 1e-12, (rank, e_out, e_lse)
        assert e_out2 < 1e-12 and e_lse2 < 1e-12, (rank, e_out2, e_lse2)
        assert e_bad > 1e-3, (rank, e_bad)  # the wrong base is visibly wrong


def test_merge_reference_against_oracle_pairwise_fold(oracle):
    """The fp64 test merge equals folding the oracle's two-way merge."""
    rng = np.random.Generator(np.random.PCG64(11))
    P, n, d = 4, 9, 16
    outs = rng.standard_normal((P, n, d))
    lses = rng.standard_normal((P, n)) * 4
    lses[1, 0] = -np.inf
    lses[:, 1] = -np.inf
    o, l = outs[0], lses[0]
    for p in range(1, P):
        o, l = oracle.lse_merge(o, l, outs[p], lses[p])
    mo, ml = _merge64(outs, lses)
    assert np.allclose(mo, o, atol=1e-12)
    # rows with no key on every rank have lse = -inf on both sides
    assert np.array_equal(np.isneginf(ml), np.isneginf(l))
    fin = np.isfinite(l)
    assert np.all(np.abs(ml[fin] - l[fin]) < 1e-12)
