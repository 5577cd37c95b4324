"""Pins of the oracle's fp8 (e4m3) KV pool, checked against what the format
definition fixes (the OCP 8-bit floating-point format E4M3: bias 7, 3 mantissa
bits, no infinities, largest finite 448, subnormals m/8 * 2^-6) and against the
already pinned bf16 oracle.  The pages name an fp8 e4m3 KV cache (the
"FlashAttention y FlashInfer" page, "Resumen en una frase" and "Limites y
fallos"); the quantisation reading (per-tensor scale, fp32 x/scale, round to
nearest even, saturate) is stated in the oracle's source."""
import numpy as np
import pytest

from paged_kv_attention_33_gb300 import workloads as W


def _bf16(values):
    return W.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


# (value, code): worked encodings from the format definition
WORKED = [
    (0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (2.0, 0x40), (0.5, 0x30), (1.125, 0x39),
    (448.0, 0x7E), (-448.0, 0xFE), (240.0, 0x77), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
    (7 * 2.0 ** -9, 0x07),                    # largest subnormal
    (1000.0, 0x7E), (-1e6, 0xFE),             # saturation
    (464.0, 0x7E),                            # halfway to a value past 448: saturates
    (1.0625, 0x38), (1.1875, 0x3A),           # ties go to the even code
    (3 * 2.0 ** -10, 0x02), (2.0 ** -10, 0x00),  # ties among subnormals
    (0.3, 0x2A), (-0.3, 0xAA),                # bf16(0.3) = 0.30078125: 0.3125 is nearer than 0.28125
]


def test_worked_encodings(oracle):
    vals = [v for v, _ in WORKED]
    got = oracle.quantize_e4m3(_bf16(vals), 1.0)
    for (v, want), g in zip(WORKED, got):
        assert g == want, (v, hex(g), hex(want))
    assert oracle.quantize_e4m3(_bf16([-0.0]), 1.0)[0] == 0x80  # the sign of zero is kept


def test_values_and_round_trip_of_every_finite_code(oracle):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_value(codes)
    # closed form of the format: (1 + m/8) 2^(e-7), subnormals m/8 2^-6
    for c, v in zip(codes, vals):
        c = int(c)
        e, m, s = (c >> 3) & 15, c & 7, -1.0 if c >> 7 else 1.0
        want = s * (m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
        assert v == want
    assert np.isnan(oracle.e4m3_value([0x7F, 0xFF])).all()
    # every finite e4m3 value is exact in bf16, and encodes back to its code
    back = oracle.quantize_e4m3(_bf16(vals), 1.0)
    assert np.array_equal(back, codes)


def test_scale_divides_before_rounding(oracle):
    """code(x, s) is the code of the fp32 quotient x / s."""
    rng = np.random.Generator(np.random.PCG64(5))
    x = _bf16(rng.standard_normal(4096, dtype=np.float32) * 3)
    for s in (0.5, 0.037, 2.5, 1 / 3):
        q = (W.bf16_bits_to_f32(x).astype(np.float32) / np.float32(s)).astype(np.float32)
        # q itself is not a bf16 value in general: compare through the brute-force
        # nearest-value rule on the exact quotient
        codes = oracle.quantize_e4m3(x, s)
        table = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
        for qi, ci in zip(q[:512], codes[:512]):
            a = min(abs(float(qi)), 448.0)
            d = np.abs(table - a)
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
            want |= 0x80 if np.signbit(qi) else 0
            assert ci == want, (qi, hex(ci), hex(want))


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 0.25), (2.0, 0.125)])
def test_fp8_attention_equals_bf16_attention_on_the_dequantised_pool(oracle, k_scale, v_scale):
    """With power-of-two scales every dequantised value is exact in bf16: the
    fp8 attention must equal, bit for bit, the bf16 oracle on a pool holding
    those values (same fp64 sum, same order)."""
    sp = W.BatchSpec("fp8pin", 8, 2, 64, 16, decode_ctx=[3, 40, 100],
                     prefill=[(20, 7)])
    b = W.make_batch(sp, seed=61)
    cache = b.cache.copy()
    oracle.reshape_and_cache(b.key, b.value, cache, b.slot_mapping)
    cache[np.isnan(W.bf16_bits_to_f32(cache))] = 0  # unused slots: any finite value
    codes = np.empty(cache.shape, dtype=np.uint8)
    codes[:, 0] = oracle.quantize_e4m3(cache[:, 0], k_scale)
    codes[:, 1] = oracle.quantize_e4m3(cache[:, 1], v_scale)
    deq = np.empty(cache.shape, dtype=np.float64)
    deq[:, 0] = oracle.e4m3_value(codes[:, 0]) * k_scale
    deq[:, 1] = oracle.e4m3_value(codes[:, 1]) * v_scale
    as_bf16 = W.f32_to_bf16_bits(deq.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(as_bf16).astype(np.float64), deq)
    o8, l8 = oracle.paged_attention_fp8(b.query, codes, k_scale, v_scale, b.query_start_loc,
                                        b.seq_lens, b.block_table, sp.softmax_scale)
    ob, lb = oracle.paged_attention(b.query, as_bf16, b.query_start_loc, b.seq_lens,
                                    b.block_table, sp.softmax_scale)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_fp8_cache_write_is_the_quantised_row(oracle):
    sp = W.BatchSpec("fp8w", 8, 2, 64, 16, decode_ctx=[3, 40])
    b = W.make_batch(sp, seed=62)
    cache8 = np.zeros(b.cache.shape, dtype=np.uint8)
    oracle.reshape_and_cache_fp8(b.key, b.value, cache8, b.slot_mapping, 0.75, 1.5)
    for t, slot in enumerate(b.slot_mapping):
        blk, off = slot // sp.block_size, slot % sp.block_size
        assert np.array_equal(cache8[blk, 0, off], oracle.quantize_e4m3(b.key[t], 0.75))
        assert np.array_equal(cache8[blk, 1, off], oracle.quantize_e4m3(b.value[t], 1.5))
    # nothing else written
    mask = np.zeros(cache8.shape[:3], dtype=bool)
    for slot in b.slot_mapping:
        mask[slot // sp.block_size, :, slot % sp.block_size] = True
    assert not cache8[~mask].any()


@pytest.mark.parametrize("k_scale,v_scale", [(0.0371, 0.0173), (1.3, 0.77)])
def test_fp8_attention_equals_dense_softmax_with_any_scale(oracle, k_scale, v_scale):
    """With scales that are not powers of two the dequantised values are not
    bf16 values; the fp8 attention must still be the dense softmax over
    code_value * scale (gathered through the block table, causal), computed
    here in numpy float64 from the codes."""
    sp = W.BatchSpec("fp8dense", 4, 2, 128, 16, decode_ctx=[7, 33], prefill=[(5, 20)])
    b = W.make_batch(sp, seed=63)
    cache = b.cache.copy()
    oracle.reshape_and_cache(b.key, b.value, cache, b.slot_mapping)
    cache[np.isnan(W.bf16_bits_to_f32(cache))] = 0
    codes = np.empty(cache.shape, dtype=np.uint8)
    codes[:, 0] = oracle.quantize_e4m3(cache[:, 0], k_scale)
    codes[:, 1] = oracle.quantize_e4m3(cache[:, 1], v_scale)
    o8, l8 = oracle.paged_attention_fp8(b.query, codes, k_scale, v_scale, b.query_start_loc,
                                        b.seq_lens, b.block_table, sp.softmax_scale)
    table = oracle.e4m3_value(np.arange(256, dtype=np.uint8))
    q = W.bf16_bits_to_f32(b.query).astype(np.float64)
    H, Hkv, D, bs = sp.num_heads, sp.num_kv_heads, sp.head_size, sp.block_size
    g = H // Hkv
    for s in range(len(b.seq_lens)):
        L = int(b.seq_lens[s])
        t0, t1 = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
        keys = np.arange(L)
        blk = b.block_table[s][keys // bs]
        K = table[codes[blk, 0, keys % bs]] * np.float64(np.float32(k_scale))  # [L, Hkv, D]
        V = table[codes[blk, 1, keys % bs]] * np.float64(np.float32(v_scale))
        for i, t in enumerate(range(t0, t1)):
            allowed = L - (t1 - t0) + i + 1  # bottom-right causal
            for h in range(H):
                x = sp.softmax_scale * (K[:allowed, h // g] @ q[t, h])
                m = x.max()
                w = np.exp(x - m)
                lse = m + np.log(w.sum())
                out = (w / w.sum()) @ V[:allowed, h // g]
                r = t * H + h
                assert abs(l8[r] - lse) <= 1e-12 * max(1.0, abs(lse))
                assert np.max(np.abs(o8[r] - out)) <= 1e-12
