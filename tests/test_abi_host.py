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


def test_library_is_built_for_sm103a():
    out = subprocess.run(["cuobjdump", "--list-elf", pbuild.LIB], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


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
    assert _fwd(lib, _meta(max_seq_len=0)) == -1
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
