"""Seeded random batches over every axis the forward serves, each compared
with the fp64 oracle on every row (and the pool byte for byte).

Each case draws: head_size 64 or 128; 1, 2, 4 or 8 kv heads; a query-head
group of 1-8 (up to 16 without decodes); block size 16-256; NHD or HND; up to
six decodes and three prefill chunks with prior context; causal or not; a
shared-prefix cascade in a third of the cases (the prefix a multiple of the
block size that every sequence's context covers); an fp8 e4m3 pool in a third
of the head_size-128 cases; and, for NHD bf16 pools, the fused call in half of
the cases.  Sizes stay small enough for the oracle to check everything."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W
from tests import gpu_util as G
from tests.test_gpu_fp8 import check_fp8

pytestmark = pytest.mark.gpu

N_CASES = 40


def random_case(i):
    rng = np.random.Generator(np.random.PCG64(7000 + i))
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    has_dec = rng.random() < 0.8
    g = int(rng.integers(1, 9)) if has_dec else int(rng.choice([1, 2, 4, 8, 16]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    layout = str(rng.choice(["NHD", "HND"]))
    P = bs * int(rng.integers(1, 4)) if rng.random() < 1 / 3 else 0
    nd = int(rng.integers(1, 7)) if has_dec else 0
    npf = int(rng.integers(0, 4)) if has_dec else int(rng.integers(1, 4))
    dctx = [P + int(rng.integers(0, 600)) for _ in range(nd)]
    pf = [(int(rng.integers(1, 300)), P + int(rng.integers(0, 400))) for _ in range(npf)]
    spec = W.BatchSpec(f"rand{i}", Hkv * g, Hkv, D, bs, decode_ctx=dctx, prefill=pf,
                       common_prefix_len=P, causal=bool(rng.random() < 0.85),
                       kv_layout=layout, table_pad=int(rng.integers(0, 3)))
    fp8 = D == 128 and rng.random() < 1 / 3
    fused = layout == "NHD" and rng.random() < 0.5
    return spec, fp8, fused, int(rng.integers(1 << 30))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_batch_matches_the_oracle(oracle, i):
    spec, fp8, fused, seed = random_case(i)
    b = W.make_batch(spec, seed=seed)
    label = (f"case {i}: H={spec.num_heads} Hkv={spec.num_kv_heads} D={spec.head_size} "
             f"bs={spec.block_size} {spec.kv_layout} P={spec.common_prefix_len} "
             f"decodes={spec.num_decodes} prefills={spec.prefill} causal={spec.causal} "
             f"fp8={fp8} fused={fused}")
    if fp8:
        check_fp8(oracle, b, 0.05, 0.04, fused=fused, label=label, causal=spec.causal)
        return
    if not fused:
        G.check_batch(oracle, b, label=label)
        return
    want = G.host_bits(b.cache).copy()
    oracle.reshape_and_cache(b.key, b.value, want, b.slot_mapping)
    pool, out, lse = G.run_fused(b)
    assert np.array_equal(want, W.to_host_bits(pool)), f"{label}: cache write differs"
    rows = np.arange(b.num_tokens * spec.num_heads, dtype=np.int64)
    o_ref, l_ref = G.oracle_expected(oracle, b, want, rows=rows)
    G.assert_close(G.compare(W.to_host_bits(out), lse.cpu().numpy(), o_ref, l_ref, rows,
                             spec.num_heads), label)
