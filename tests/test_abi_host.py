"""Host-side checks of the C ABI: the library builds, loads and exports every
entry point include/pka.h declares, and argument errors are reported before
any GPU work (these calls return before touching a device)."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_attention_33_gb300 as pka
from paged_kv_attention_33_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pka.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pka_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return pka.load_library()


def test_header_declares_the_three_operations():
    syms = declared_symbols()
    for name in ("pka_reshape_and_cache", "pka_paged_attn_forward", "pka_cascade_merge"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(pka_[a-z_]+)\b", out))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing
    for s in declared_symbols():
        assert hasattr(lib, s)


def test_library_is_built_for_sm103a_only():
    """Every translation unit and the link step take exactly one target,
    sm_103a machine code (no PTX to be compiled for another GPU at load)."""
    assert pbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    cmds = pbuild.commands()
    assert cmds and all(c.count("-gencode") == 1 and "arch=compute_103a,code=sm_103a" in c
                        for c in cmds)


def _meta(**kw):
    m = pka._CMeta()
    m.query_start_loc = 16
    m.seq_lens = 16
    m.block_table = 16
    m.block_table_stride = 8
    m.num_seqs = 2
    m.num_decodes = 2
    m.max_query_len = 1
    m.max_seq_len = 100
    m.common_prefix_len = 0
    m.split_kv_tokens = 0
    for k, v in kw.items():
        setattr(m, k, v)
    return m


def _fwd(lib, meta, T=2, H=8, Hkv=2, D=64, bs=16, query=256, cache=512, out=1024, scale=0.125,
         ws=None, ws_bytes=0):
    return lib.pka_paged_attn_forward(query, cache, ctypes.byref(meta), out, None, T, H, Hkv, D,
                                      bs, 64, scale, 1, ws, ws_bytes, None)


@pytest.mark.parametrize("bs", [0, 8, 24, 40])
def test_block_size_must_be_multiple_of_16(lib, bs):
    rc = _fwd(lib, _meta(), bs=bs)
    assert rc == -1
    assert b"multiple of 16" in lib.pka_last_error()
    rc = lib.pka_reshape_and_cache(16, 16, 16, 16, 4, 2, 64, bs, 64, None)
    assert rc == -1


def test_head_size_rules(lib):
    assert _fwd(lib, _meta(), D=60) == -1          # not a multiple of 8
    assert _fwd(lib, _meta(), D=264) == -1         # above 256
    assert _fwd(lib, _meta(), D=96) == -2          # valid but not built


def test_group_rules(lib):
    assert _fwd(lib, _meta(), H=6, Hkv=4) == -1    # not a multiple
    assert _fwd(lib, _meta(), H=48, Hkv=3) == -2   # kv heads not built
    assert _fwd(lib, _meta(), H=32, Hkv=2) == -2   # decode group 16 not built


def test_inconsistent_sizes(lib):
    assert _fwd(lib, _meta(num_decodes=3)) == -1
    assert _fwd(lib, _meta(max_seq_len=-1)) == -1
    # 0 bounds a decode-only batch whose decodes hold no key, not a prefill
    assert _fwd(lib, _meta(num_decodes=1, max_query_len=1, max_seq_len=0)) == -1
    assert _fwd(lib, _meta(block_table_stride=2)) == -1
    assert _fwd(lib, _meta(common_prefix_len=8)) == -1
    assert _fwd(lib, _meta(common_prefix_len=100)) == -1


def test_null_and_alias(lib):
    assert _fwd(lib, _meta(), query=0) == -1
    assert _fwd(lib, _meta(), query=256, out=256) == -1
    assert _fwd(lib, _meta(), query=8) == -1      # misaligned
    assert _fwd(lib, _meta(), scale=float("nan")) == -1


def test_workspace_size_and_missing_workspace(lib):
    m = _meta(split_kv_tokens=64, max_seq_len=1000, block_table_stride=64)
    need = lib.pka_workspace_size(ctypes.byref(m), 2, 8, 2, 64, 16)
    # 2 decodes x ceil(1000/64)=16 splits x 8 heads x (64 fp32 + 1 fp32)
    assert need >= 2 * 16 * 8 * 65 * 4
    assert _fwd(lib, m) == -3
    assert lib.pka_workspace_size(ctypes.byref(_meta()), 2, 8, 2, 60, 16) == 0


def test_cascade_merge_arguments(lib):
    assert lib.pka_cascade_merge(16, 16, 16, 16, 16, None, 4, 8, 60, None) == -1
    assert lib.pka_cascade_merge(None, 16, 16, 16, 16, None, 4, 8, 64, None) == -1
    assert lib.pka_cascade_merge(16, 16, 16, 16, 16, None, 0, 8, 64, None) == 0


def test_unknown_kv_layout_is_rejected(lib):
    """The pool layout is one of the two the pages name (NHD, HND)."""
    assert _fwd(lib, _meta(kv_layout=2)) == -1
    assert lib.pka_workspace_size(ctypes.byref(_meta(kv_layout=-1)), 2, 8, 2, 64, 16) == 0
    assert lib.pka_reshape_and_cache_ex(16, 16, 16, 16, 1, 2, 64, 16, 4, 3, None) == -1
    # a zero-initialised meta is NHD
    assert pka._CMeta().kv_layout == pka.LAYOUT_NHD


def test_hnd_pool_is_the_slot_head_transpose():
    """The HND pool holds row (block b, kv, slot o, head k) at [b][kv][k][o]:
    the logical [NB, 2, bs, Hkv, D] pool with the slot and head axes swapped
    (checked element by element on a pool of distinct values), and the
    conversion back is exact."""
    import numpy as np

    from paged_kv_attention_33_gb300 import workloads as W

    nb, bs, hkv, d = 3, 4, 5, 6
    logical = np.arange(nb * 2 * bs * hkv * d, dtype=np.uint16).reshape(nb, 2, bs, hkv, d)
    hnd = W.to_layout(logical, "HND")
    assert hnd.shape == (nb, 2, hkv, bs, d) and hnd.flags["C_CONTIGUOUS"]
    for b in range(nb):
        for kv in range(2):
            for o in range(bs):
                for k in range(hkv):
                    assert np.array_equal(hnd[b, kv, k, o], logical[b, kv, o, k])
    # head k's page is one contiguous run of bs*d elements
    flat = hnd.reshape(-1)
    start = ((1 * 2 + 1) * hkv + 2) * bs * d
    assert np.array_equal(flat[start:start + bs * d].reshape(bs, d), logical[1, 1, :, 2])
    assert np.array_equal(W.from_layout(hnd, "HND"), logical)
    assert W.to_layout(logical, "NHD") is logical


def test_merge_partials_arguments(lib):
    assert lib.pka_merge_partials(16, 16, 0, 4096, None, 4, 8, 64, 0, None) == -1    # no parts
    assert lib.pka_merge_partials(16, 16, 2, 4096, None, 4, 8, 60, 0, None) == -1    # head_size
    assert lib.pka_merge_partials(16, 16, 2, 65536, None, 4, 8, 64, 7, None) == -1   # base
    assert lib.pka_merge_partials(None, 16, 2, 65536, None, 4, 8, 64, 0, None) == -1
    assert lib.pka_merge_partials(16, 16, 2, 16 + 4 * 8 * 64 * 2, None, 4, 8, 64, 0, None) == -1  # alias
    assert lib.pka_merge_partials(16, 16, 2, 16, None, 0, 8, 64, 0, None) == 0       # empty


def test_fused_forward_arguments(lib):
    m = _meta()
    fused = lib.pka_paged_attn_forward_fused
    # null / misaligned new rows or slots
    assert fused(256, None, 256, 256, 512, ctypes.byref(m), 1024, None, 2, 8, 2, 64, 16, 64,
                 0.125, 1, None, 0, None) == -1
    assert fused(256, 256, 256, 4, 512, ctypes.byref(m), 1024, None, 2, 8, 2, 64, 16, 64,
                 0.125, 1, None, 0, None) == -1
    # the forward's own checks still apply (block size)
    assert fused(256, 256, 256, 256, 512, ctypes.byref(m), 1024, None, 2, 8, 2, 64, 24, 64,
                 0.125, 1, None, 0, None) == -1


def test_fp8_pool_arguments(lib):
    """kv_dtype is one of the two pool element types; an fp8 pool needs
    positive finite scales and is served at head_size 128 (UNSUPPORTED
    otherwise, before any work)."""
    fp8 = dict(kv_dtype=pka.KV_FP8_E4M3, k_scale=0.5, v_scale=2.0)
    assert pka._CMeta().kv_dtype == pka.KV_BF16  # a zero-initialised meta is bf16
    assert _fwd(lib, _meta(kv_dtype=2)) == -1
    assert lib.pka_workspace_size(ctypes.byref(_meta(kv_dtype=-1)), 2, 8, 2, 128, 16) == 0
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert _fwd(lib, _meta(**{**fp8, "k_scale": bad}), D=128) == -1
        assert _fwd(lib, _meta(**{**fp8, "v_scale": bad}), D=128) == -1
    assert _fwd(lib, _meta(**fp8), D=64) == -2                        # head_size 64
    # a cascade over fp8 is served: its shared prefix gets a bf16 copy too
    casc8 = _meta(common_prefix_len=16, **fp8)
    w_c8 = lib.pka_workspace_size(ctypes.byref(casc8), 2, 8, 2, 128, 16)
    w_c16 = lib.pka_workspace_size(ctypes.byref(_meta(common_prefix_len=16)), 2, 8, 2, 128, 16)
    assert w_c8 - w_c16 >= 1 * 2 * 16 * 2 * 128 * 2  # one prefix block
    assert lib.pka_workspace_size(ctypes.byref(_meta(**fp8)), 2, 8, 2, 64, 16) == 0
    # a bf16 meta ignores the scales
    assert lib.pka_workspace_size(ctypes.byref(_meta(k_scale=-1.0)), 2, 8, 2, 64, 16) > 0
    # prefills over an fp8 pool are served through a bf16 copy of their blocks in
    # the workspace: ceil(max_seq_len / bs) blocks of 2*bs*Hkv*D bf16 per prefill
    mixed8 = _meta(num_decodes=1, max_query_len=4, **fp8)
    mixed16 = _meta(num_decodes=1, max_query_len=4)
    w8 = lib.pka_workspace_size(ctypes.byref(mixed8), 5, 8, 2, 128, 16)
    w16 = lib.pka_workspace_size(ctypes.byref(mixed16), 5, 8, 2, 128, 16)
    blocks = -(-100 // 16)  # max_seq_len 100
    assert w8 - w16 >= blocks * 2 * 16 * 2 * 128 * 2 + 2 * blocks * 4
    assert _fwd(lib, mixed8, T=5, D=128) == -3  # served, but needs that workspace
    # the fused entry refuses an unserved fp8 batch before writing anything
    m = _meta(num_decodes=0, max_query_len=4, **fp8)
    assert lib.pka_paged_attn_forward_fused(256, 256, 256, 256, 512, ctypes.byref(m), 1024, None,
                                            5, 8, 2, 64, 16, 64, 0.125, 1, None, 0, None) == -2


def test_fp8_cache_write_arguments(lib):
    w = lib.pka_reshape_and_cache_fp8
    assert w(16, 16, 16, 16, 1, 2, 128, 16, 4, 0, 0.0, 1.0, None) == -1   # scale
    assert w(16, 16, 16, 16, 1, 2, 128, 16, 4, 0, 1.0, float("nan"), None) == -1
    assert w(16, 16, 16, 16, 1, 2, 128, 16, 4, 5, 1.0, 1.0, None) == -1   # layout
    assert w(16, 16, 16, 16, 1, 2, 128, 24, 4, 0, 1.0, 1.0, None) == -1   # block size
    assert w(16, 16, 16, 16, 1, 2, 72, 16, 4, 0, 1.0, 1.0, None) == -2    # head_size % 16
    assert w(None, 16, 16, 16, 1, 2, 128, 16, 4, 0, 1.0, 1.0, None) == -1  # null
    assert w(16, 16, 16, 16, 0, 2, 128, 16, 4, 0, 1.0, 1.0, None) == 0     # nothing to do
