"""GPU parity of the shared-prefix cascade: prefix attended once on the tensor
cores, per-sequence suffixes by the decode / prefill kernels, merged by
log-sum-exp; compared with the oracle's cascade and with plain attention."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_cascade_small_decodes(oracle):
    sp = W.BatchSpec("c1", 16, 2, 128, 16, decode_ctx=[64, 65, 100, 200, 64 + 15],
                     common_prefix_len=64)
    G.check_batch(oracle, W.make_batch(sp, seed=4001), label="cascade decodes")


@pytest.mark.parametrize("bs,P", [(16, 128), (64, 256), (128, 128)])
def test_cascade_with_prefill_chunks(oracle, bs, P):
    sp = W.BatchSpec("c2", 32, 8, 128, bs, decode_ctx=[P, P + 7, P + 300],
                     prefill=[(40, P), (130, P + 50), (1, P + 1)], common_prefix_len=P)
    G.check_batch(oracle, W.make_batch(sp, seed=4100 + bs), label=f"cascade bs={bs}")


@pytest.mark.parametrize("H,Hkv,D,bs,P", [
    (16, 2, 64, 16, 1008),    # 8 key tiles, the last one ragged: 2 chunks
    (32, 8, 128, 64, 2048),   # 16 key tiles: 4 chunks
    (64, 8, 128, 128, 4096),  # the cascade workload's shape: 2 chunks
])
def test_cascade_split_prefix(oracle, H, Hkv, D, bs, P):
    """Prefixes long enough that the shared-prefix pass cuts its keys into
    chunks (few work items, so the chunks fill the grid): one partial per
    chunk, merged with the decode pieces and with the prefill suffixes."""
    sp = W.BatchSpec("c5", H, Hkv, D, bs, decode_ctx=[P + 1, P + 17, P + 300, P + 129],
                     prefill=[(33, P), (200, P + 40)], common_prefix_len=P)
    b = W.make_batch(sp, seed=4300 + P)
    G.check_batch(oracle, b, label=f"cascade split P={P}")
    G.check_batch(oracle, b, split_kv_tokens=64, label=f"cascade split P={P}, 64 keys/CTA")


@pytest.mark.parametrize("layout,bs", [("NHD", 16), ("HND", 128)])
def test_cascade_side_by_side(oracle, layout, bs):
    """A batch the cascade plan runs side by side (48 decodes sharing a
    1024-token prefix: the prefix pass on part of the SMs, the suffix decode as
    its dependent on the rest, then the combine), in both pool layouts."""
    P = 1024
    rng = np.random.Generator(np.random.PCG64(bs))
    ctx = (P + rng.integers(64, 800, size=48)).tolist()
    sp = W.BatchSpec(f"c_sbs_{layout}", 32, 8, 128, bs, decode_ctx=ctx, common_prefix_len=P,
                     kv_layout=layout)
    b = W.make_batch(sp, seed=4400 + bs)
    G.check_batch(oracle, b, label=f"cascade side by side {layout} bs={bs}")


def test_cascade_equals_plain(oracle):
    """The same batch with and without the cascade gives the same rows (both
    within tolerance of the oracle's plain attention)."""
    sp = W.BatchSpec("c3", 64, 8, 128, 128, decode_ctx=[256 + k * 37 for k in range(12)],
                     common_prefix_len=256)
    b = W.make_batch(sp, seed=4200)
    res_c = G.check_batch(oracle, b, label="cascade")
    sp0 = W.BatchSpec("c3p", 64, 8, 128, 128, decode_ctx=sp.decode_ctx)
    b0 = W.Batch(sp0, b.query, b.key, b.value, b.cache, b.slot_mapping, b.query_start_loc,
                 b.seq_lens, b.block_table, b.num_blocks)
    res_p = G.check_batch(oracle, b0, label="plain")
    assert res_c["out_max_abs"] <= 2e-2 and res_p["out_max_abs"] <= 2e-2


def test_cascade_precondition_is_flagged():
    """A prefill chunk whose queries start inside the shared prefix breaks the
    cascade's premise; the kernel flags it instead of computing garbage."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    sp = W.BatchSpec("c4", 8, 2, 64, 16, decode_ctx=[40], prefill=[(20, 40)],
                     common_prefix_len=32)
    b = W.make_batch(sp, seed=4300)
    meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table, 1, "cuda",
                              common_prefix_len=48)   # 48 > ctx of... decode ctx 40
    q = G.to_dev(b.query, "cuda")
    out = torch.empty_like(q)
    pka.paged_attn_forward(q, G.to_dev(b.cache, "cuda"), meta, out, scale=sp.softmax_scale)
    with pytest.raises(pka.PkaError) as e:
        pka.check_status()
    assert e.value.status == -5


def test_cascade_small_pages_prefix_off_the_tile_grid(oracle):
    """A cascade over 16-key pages whose shared prefix (80 keys) is not a
    multiple of 128, with query-heavy prefill suffixes: the suffix pass reads
    the 128-key re-blocked copy from key 80, so its TMA boxes shrink to
    gcd(16, 128, 80) = 16 rows and never straddle a copied block."""
    P = 80
    sp = W.BatchSpec("casc_reblock", 16, 4, 128, 16, decode_ctx=[P + 5, P + 300],
                     prefill=[(300, P), (400, P + 50)], common_prefix_len=P)
    G.check_batch(oracle, W.make_batch(sp, seed=4400), label="cascade re-blocked suffix")
