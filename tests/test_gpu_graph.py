"""The forward is a sequence of asynchronous launches on the caller's stream
with no host synchronisation, so a serving loop can capture a step in a CUDA
graph and replay it (the "El especialista del plato estrella" blog, "Como se
conecta con el resto del stack": attention kernels are captured in CUDA
graphs; the "FlashAttention y FlashInfer" page, "Resumen en una frase": the
backends' levels of cudagraph support).  A fused step captured and replayed
must give, bit for bit, the eager step's output, lse and pool."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _eager_and_replayed(b, pool, meta, sp):
    import torch

    import paged_kv_attention_33_gb300 as pka

    dev = "cuda"
    q, k, v = (G.to_dev(x, dev) for x in (b.query, b.key, b.value))
    slots = torch.from_numpy(b.slot_mapping).to(dev)
    T = b.num_tokens
    need = pka.workspace_size(meta, T, sp.num_heads, sp.num_kv_heads, sp.head_size,
                              sp.block_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def step(out, lse, p):
        pka.paged_attn_forward_fused(q, k, v, slots, p, meta, out, lse, scale=sp.softmax_scale,
                                     workspace=ws)

    pool_e = pool.clone()
    out_e = torch.empty_like(q)
    lse_e = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    step(out_e, lse_e, pool_e)
    pka.check_status()

    pool_g = pool.clone()
    out_g = torch.full_like(q, float("nan"))
    lse_g = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(out_g, lse_g, pool_g)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):  # the writes are idempotent: replays agree with one eager step
        graph.replay()
    torch.cuda.synchronize()
    pka.check_status()
    return (out_e, lse_e, pool_e), (out_g, lse_g, pool_g)


def test_graph_replay_of_a_mixed_fused_step():
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("graph_mixed", 32, 8, 128, 16, decode_ctx=[5, 300, 2000],
                     prefill=[(130, 0), (64, 700)])
    b = W.make_batch(sp, seed=9300)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              "cuda")
    (oe, le, pe), (og, lg, pg) = _eager_and_replayed(b, G.to_dev(b.cache, "cuda"), meta, sp)
    assert torch.equal(oe.view(torch.int16), og.view(torch.int16))
    assert torch.equal(le, lg)
    assert torch.equal(pe.view(torch.int16), pg.view(torch.int16))


def test_graph_replay_over_an_fp8_pool(oracle):
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("graph_fp8", 32, 8, 128, 16, decode_ctx=[5, 300, 2000],
                     prefill=[(130, 0)])
    b = W.make_batch(sp, seed=9301)
    c = G.host_bits(b.cache)
    p8 = np.empty(c.shape, dtype=np.uint8)
    p8[:, 0] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 0]), 0.05)
    p8[:, 1] = oracle.quantize_e4m3(np.ascontiguousarray(c[:, 1]), 0.04)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              "cuda", kv_dtype="fp8", k_scale=0.05, v_scale=0.04)
    (oe, le, pe), (og, lg, pg) = _eager_and_replayed(b, torch.from_numpy(p8).cuda(), meta, sp)
    assert torch.equal(oe.view(torch.int16), og.view(torch.int16))
    assert torch.equal(le, lg)
    assert torch.equal(pe, pg)


def test_graph_replay_of_a_cascade_step():
    """A shared-prefix cascade whose prefix pass and suffix decode run side by
    side (the decode a programmatic dependent launch) is captured and replayed
    with the same results as eager, bit for bit."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    P = 2048
    sp = W.BatchSpec("graph_cascade", 64, 8, 128, 128,
                     decode_ctx=[P + 3, P + 100, P + 700, P + 1023, P + 64, P + 300],
                     common_prefix_len=P)
    b = W.make_batch(sp, seed=9302)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              "cuda", common_prefix_len=P)
    (oe, le, pe), (og, lg, pg) = _eager_and_replayed(b, G.to_dev(b.cache, "cuda"), meta, sp)
    assert torch.equal(oe.view(torch.int16), og.view(torch.int16))
    assert torch.equal(le, lg)
    assert torch.equal(pe.view(torch.int16), pg.view(torch.int16))


def test_graph_replay_of_a_few_long_decodes():
    """A decode-only batch of a few long decodes: the decode launch and the
    merge launch of its split decodes (its programmatic dependent) captured
    together."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("graph_few_long", 32, 8, 128, 16, decode_ctx=[6000, 3500, 20, 4100])
    b = W.make_batch(sp, seed=9400)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, sp.num_decodes,
                              "cuda")
    (oe, le, pe), (og, lg, pg) = _eager_and_replayed(b, G.to_dev(b.cache, "cuda"), meta, sp)
    assert torch.equal(oe.view(torch.int16), og.view(torch.int16))
    assert torch.equal(le, lg)
    assert torch.equal(pe.view(torch.int16), pg.view(torch.int16))
