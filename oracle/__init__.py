"""Test infrastructure: ctypes front end of the plain fp64 CPU oracle.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg import this package.  It shares no code with the CUDA path: the
oracle is the single C file ``pka_oracle.c`` next to this module, compiled
with gcc into ``oracle/_build/``.

All arrays crossing into the oracle are numpy arrays: bf16 tensors are passed
as their uint16 bit patterns, results come back as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pka_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(mutant: int = 0, out_dir: str | None = None) -> str:
    """Compile the oracle (or a planted-mistake variant) and return the .so path."""
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "libpka_oracle.so" if mutant == 0 else f"libpka_oracle_m{mutant}.so"
    path = os.path.join(out_dir, name)
    if (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORACLE_MUTANT={mutant}",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_reshape_and_cache.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64]
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    att = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
           ctypes.c_int]
    lib.oracle_paged_attention.argtypes = att + [_I64, _I64, _P, _I64, _P, _P]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_cascade_attention.argtypes = att + [_I64, _P, _I64, _P, _P]
    lib.oracle_cascade_attention.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [_P, _P, _P, _P, _I64, _I64, _P, _P]
    lib.oracle_lse_merge.restype = None
    lib.oracle_quantize_e4m3.argtypes = [_P, _I64, ctypes.c_float, _P]
    lib.oracle_quantize_e4m3.restype = None
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64,
                                                 ctypes.c_float, ctypes.c_float]
    lib.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
    lib.oracle_paged_attention_fp8.argtypes = [_P, _P, ctypes.c_double, ctypes.c_double, _P,
                                               _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                               ctypes.c_double, ctypes.c_int, _P, _I64, _P, _P]
    lib.oracle_paged_attention_fp8.restype = ctypes.c_int
    return lib


def load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant not in _LIBS:
            _LIBS[mutant] = _declare(ctypes.CDLL(build(mutant)))
        return _LIBS[mutant]


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle's four entry points, bound to one compiled variant."""

    def __init__(self, mutant: int = 0):
        self.lib = load(mutant)

    # -- cache write ---------------------------------------------------------
    def reshape_and_cache(self, key, value, cache, slot_mapping):
        """In-place byte copy of key/value rows into the uint16 pool `cache`."""
        key = _c(key, np.uint16)
        value = _c(value, np.uint16)
        assert cache.dtype == np.uint16 and cache.flags.c_contiguous
        slots = _c(slot_mapping, np.int64)
        nb, two, bs, hkv, d = cache.shape
        assert two == 2
        rc = self.lib.oracle_reshape_and_cache(
            _ptr(key), _ptr(value), _ptr(cache), _ptr(slots), slots.shape[0], hkv, d, bs, nb)
        if rc != 0:
            raise ValueError(f"oracle reshape_and_cache failed ({rc})")

    # -- attention -----------------------------------------------------------
    def _attn_args(self, query, cache, qsl, seq_lens, block_table):
        query = _c(query, np.uint16)
        cache = _c(cache, np.uint16)
        qsl = _c(qsl, np.int32)
        seq_lens = _c(seq_lens, np.int32)
        block_table = _c(block_table, np.int32)
        return query, cache, qsl, seq_lens, block_table

    def paged_attention(self, query, cache, qsl, seq_lens, block_table, scale, causal=True,
                        key_lo=0, key_hi=-1, rows=None, threads=1):
        """fp64 (out [R, D], lse [R]) for rows r = t*H + h (all rows when rows is None)."""
        query, cache, qsl, seq_lens, block_table = self._attn_args(
            query, cache, qsl, seq_lens, block_table)
        T, H, D = query.shape
        nb, _, bs, hkv, _ = cache.shape
        if rows is None:
            rows = np.arange(T * H, dtype=np.int64)
        rows = _c(rows, np.int64)
        n = rows.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        S = seq_lens.shape[0]

        def run(lo, hi):
            if hi <= lo:
                return 0
            return self.lib.oracle_paged_attention(
                _ptr(query), _ptr(cache), _ptr(qsl), _ptr(seq_lens), _ptr(block_table),
                block_table.shape[1], S, H, hkv, D, bs, nb, float(scale), int(bool(causal)),
                int(key_lo), int(key_hi), _ptr(rows[lo:hi]), hi - lo,
                out[lo:hi].ctypes.data_as(ctypes.c_void_p),
                lse[lo:hi].ctypes.data_as(ctypes.c_void_p))

        self._parallel(run, n, threads)
        return out, lse

    def cascade_attention(self, query, cache, qsl, seq_lens, block_table, scale,
                          common_prefix_len, causal=True, rows=None, threads=1):
        query, cache, qsl, seq_lens, block_table = self._attn_args(
            query, cache, qsl, seq_lens, block_table)
        T, H, D = query.shape
        nb, _, bs, hkv, _ = cache.shape
        if rows is None:
            rows = np.arange(T * H, dtype=np.int64)
        rows = _c(rows, np.int64)
        n = rows.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        S = seq_lens.shape[0]

        def run(lo, hi):
            if hi <= lo:
                return 0
            return self.lib.oracle_cascade_attention(
                _ptr(query), _ptr(cache), _ptr(qsl), _ptr(seq_lens), _ptr(block_table),
                block_table.shape[1], S, H, hkv, D, bs, nb, float(scale), int(bool(causal)),
                int(common_prefix_len), _ptr(rows[lo:hi]), hi - lo,
                out[lo:hi].ctypes.data_as(ctypes.c_void_p),
                lse[lo:hi].ctypes.data_as(ctypes.c_void_p))

        self._parallel(run, n, threads)
        return out, lse

    @staticmethod
    def _parallel(run, n, threads):
        threads = max(1, int(threads))
        if threads == 1 or n < 2 * threads:
            rcs = [run(0, n)]
        else:
            # ctypes drops the GIL inside the C call, so plain threads run the
            # single-threaded oracle on disjoint row ranges side by side.
            bounds = np.linspace(0, n, threads + 1).astype(np.int64)
            with ThreadPoolExecutor(threads) as ex:
                rcs = list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])),
                                  range(threads)))
        for rc in rcs:
            if rc != 0:
                raise ValueError(f"oracle attention failed ({rc})")

    # -- fp8 (e4m3) pool -----------------------------------------------------
    def quantize_e4m3(self, x_bits, scale):
        """uint8 e4m3 codes of the bf16 values `x_bits` divided by `scale` (fp32)."""
        x = _c(x_bits, np.uint16)
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.oracle_quantize_e4m3(_ptr(x), x.size, float(np.float32(scale)), _ptr(out))
        return out

    def e4m3_value(self, codes):
        """Exact value (float64) of each e4m3 code."""
        codes = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.oracle_e4m3_value(int(c)) for c in codes.ravel()],
                        dtype=np.float64).reshape(codes.shape)

    def reshape_and_cache_fp8(self, key, value, cache8, slot_mapping, k_scale, v_scale):
        """Quantise key/value rows into the uint8 e4m3 pool `cache8` in place."""
        key = _c(key, np.uint16)
        value = _c(value, np.uint16)
        assert cache8.dtype == np.uint8 and cache8.flags.c_contiguous
        slots = _c(slot_mapping, np.int64)
        nb, two, bs, hkv, d = cache8.shape
        rc = self.lib.oracle_reshape_and_cache_fp8(
            _ptr(key), _ptr(value), _ptr(cache8), _ptr(slots), slots.shape[0], hkv, d, bs, nb,
            float(np.float32(k_scale)), float(np.float32(v_scale)))
        if rc != 0:
            raise ValueError(f"oracle reshape_and_cache_fp8 failed ({rc})")

    def paged_attention_fp8(self, query, cache8, k_scale, v_scale, qsl, seq_lens, block_table,
                            scale, causal=True, rows=None, threads=1):
        """paged_attention over an e4m3 pool (K = code*k_scale, V = code*v_scale)."""
        query = _c(query, np.uint16)
        cache8 = _c(cache8, np.uint8)
        qsl = _c(qsl, np.int32)
        seq_lens = _c(seq_lens, np.int32)
        block_table = _c(block_table, np.int32)
        T, H, D = query.shape
        nb, _, bs, hkv, _ = cache8.shape
        if rows is None:
            rows = np.arange(T * H, dtype=np.int64)
        rows = _c(rows, np.int64)
        n = rows.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        S = seq_lens.shape[0]

        def run(lo, hi):
            if hi <= lo:
                return 0
            return self.lib.oracle_paged_attention_fp8(
                _ptr(query), _ptr(cache8), float(np.float32(k_scale)), float(np.float32(v_scale)),
                _ptr(qsl), _ptr(seq_lens), _ptr(block_table), block_table.shape[1], S, H, hkv, D,
                bs, nb, float(scale), int(bool(causal)), _ptr(rows[lo:hi]), hi - lo,
                out[lo:hi].ctypes.data_as(ctypes.c_void_p),
                lse[lo:hi].ctypes.data_as(ctypes.c_void_p))

        self._parallel(run, n, threads)
        return out, lse

    # -- merge ---------------------------------------------------------------
    def lse_merge(self, o_a, lse_a, o_b, lse_b):
        o_a = _c(o_a, np.float64)
        o_b = _c(o_b, np.float64)
        lse_a = _c(lse_a, np.float64)
        lse_b = _c(lse_b, np.float64)
        n, d = o_a.shape
        o = np.zeros_like(o_a)
        lse = np.zeros_like(lse_a)
        self.lib.oracle_lse_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), n, d,
                                  _ptr(o), _ptr(lse))
        return o, lse


def cpu_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
