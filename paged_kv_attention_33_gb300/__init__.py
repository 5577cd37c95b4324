"""GB300-native paged-KV attention forward: Python binding of libpka.so.

Thin ctypes marshalling over the C ABI declared in include/pka.h: tensor
shapes become size arguments, tensors become device pointers, the current
torch CUDA stream becomes the stream argument.  Every step of the attention
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
every call raises if the library cannot be loaded.

Entry points (same names as the C ABI without the ``pka_`` prefix):
    reshape_and_cache(key, value, kv_cache, slot_mapping)
    paged_attn_forward(query, kv_cache, meta, out, lse=None, scale=None, causal=True)
    cascade_merge(out_a, lse_a, out_b, lse_b, out, lse_out=None)
    workspace_size(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size)
    check_status()
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

__all__ = ["Meta", "PkaError", "LAYOUT_NHD", "LAYOUT_HND", "KV_BF16", "KV_FP8_E4M3",
           "reshape_and_cache", "reshape_and_cache_fp8", "paged_attn_forward", "cascade_merge",
           "paged_attn_forward_noalloc", "paged_attn_forward_fused", "workspace_size",
           "workspace_size_min",
           "merge_partials", "LSE_BASE_E",
           "LSE_BASE_2", "check_status", "set_kernel_events", "kernel_launches",
           "load_library", "test_skip_copies",
           "library_path", "KERNEL_DECODE", "KERNEL_PREFILL"]

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_lock = threading.Lock()
_lib = None

STATUS = {0: "PKA_OK", -1: "PKA_ERR_INVALID_ARG", -2: "PKA_ERR_UNSUPPORTED",
          -3: "PKA_ERR_WORKSPACE", -4: "PKA_ERR_CUDA", -5: "PKA_ERR_DEVICE_CHECK"}


class PkaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class _CMeta(ctypes.Structure):
    _fields_ = [("query_start_loc", _P), ("seq_lens", _P), ("block_table", _P),
                ("block_table_stride", _I32), ("num_seqs", _I32), ("num_decodes", _I32),
                ("max_query_len", _I32), ("max_seq_len", _I32), ("common_prefix_len", _I32),
                ("split_kv_tokens", _I32), ("kv_layout", _I32), ("kv_dtype", _I32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]

# Physical pool layouts (pka_kv_layout): the logical shape is always
# [num_blocks, 2, block_size, num_kv_heads, head_size]; HND stores it as
# [num_blocks, 2, num_kv_heads, block_size, head_size].
LAYOUT_NHD = 0
LAYOUT_HND = 1


# Element types of the pool (pka_kv_dtype): bf16, or fp8 e4m3 codes with one
# fp32 dequantisation scale per tensor for K and for V.
KV_BF16 = 0
KV_FP8_E4M3 = 1


def _kv_dtype(kv_dtype) -> int:
    if isinstance(kv_dtype, str):
        return {"BF16": KV_BF16, "FP8": KV_FP8_E4M3, "FP8_E4M3": KV_FP8_E4M3,
                "E4M3": KV_FP8_E4M3}[kv_dtype.upper()]
    return int(kv_dtype)


def _layout(kv_layout) -> int:
    if isinstance(kv_layout, str):
        return {"NHD": LAYOUT_NHD, "HND": LAYOUT_HND}[kv_layout.upper()]
    return int(kv_layout)


def _pool_dims(kv_cache, kv_layout):
    """(num_blocks, block_size, num_kv_heads, head_size) of a pool tensor."""
    nb, _, a, b, d = kv_cache.shape
    return (nb, b, a, d) if _layout(kv_layout) == LAYOUT_HND else (nb, a, b, d)


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpka.so (building it first if asked and it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libpka.so not built ({path}); run "
                                   "paged_kv_attention_33_gb300.build.build()")
            path = _build.build()
        lib = ctypes.CDLL(path)
        lib.pka_reshape_and_cache.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I64, _P]
        lib.pka_reshape_and_cache.restype = ctypes.c_int
        lib.pka_reshape_and_cache_ex.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I64,
                                                 _I32, _P]
        lib.pka_reshape_and_cache_ex.restype = ctypes.c_int
        lib.pka_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I64,
                                                  _I32, ctypes.c_float, ctypes.c_float, _P]
        lib.pka_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.pka_workspace_size.argtypes = [ctypes.POINTER(_CMeta), _I32, _I32, _I32, _I32, _I32]
        lib.pka_workspace_size.restype = ctypes.c_size_t
        lib.pka_workspace_size_min.argtypes = [ctypes.POINTER(_CMeta), _I32, _I32, _I32, _I32,
                                               _I32]
        lib.pka_workspace_size_min.restype = ctypes.c_size_t
        lib.pka_paged_attn_forward.argtypes = [_P, _P, ctypes.POINTER(_CMeta), _P, _P, _I32,
                                               _I32, _I32, _I32, _I32, _I64, ctypes.c_float,
                                               _I32, _P, ctypes.c_size_t, _P]
        lib.pka_paged_attn_forward.restype = ctypes.c_int
        lib.pka_paged_attn_forward_noalloc.argtypes = [_P, _P, ctypes.POINTER(_CMeta), _P, _P,
                                                       _I32, _I32, _I32, _I32, _I32, _I64,
                                                       ctypes.c_float, _I32, _P]
        lib.pka_paged_attn_forward_noalloc.restype = ctypes.c_int
        lib.pka_cascade_merge.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P]
        lib.pka_merge_partials.argtypes = [_P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P]
        lib.pka_paged_attn_forward_fused.argtypes = [_P, _P, _P, _P, _P, ctypes.POINTER(_CMeta),
                                                     _P, _P, _I32, _I32, _I32, _I32, _I32,
                                                     _I64, ctypes.c_float, _I32, _P,
                                                     ctypes.c_size_t, _P]
        lib.pka_paged_attn_forward_fused.restype = ctypes.c_int
        lib.pka_merge_partials.restype = ctypes.c_int
        lib.pka_cascade_merge.restype = ctypes.c_int
        lib.pka_set_kernel_events.argtypes = [_I32, _P, _P]
        lib.pka_set_kernel_events.restype = ctypes.c_int
        lib.pka_test_skip_copies.argtypes = [_I32]
        lib.pka_test_skip_copies.restype = ctypes.c_int
        lib.pka_kernel_launches.argtypes = []
        lib.pka_kernel_launches.restype = ctypes.c_uint64
        lib.pka_check_status.argtypes = [_P]
        lib.pka_check_status.restype = ctypes.c_int
        lib.pka_last_error.argtypes = []
        lib.pka_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        msg = load_library().pka_last_error().decode(errors="replace")
        raise PkaError(rc, msg)


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Meta:
    """Batch metadata: device tensors plus the host-side sizes the plan needs.

    query_start_loc int32 [S+1], seq_lens int32 [S], block_table int32
    [S, stride] live on the device; num_decodes, max_query_len, max_seq_len,
    common_prefix_len, split_kv_tokens and kv_layout (LAYOUT_NHD / LAYOUT_HND,
    or "NHD" / "HND") are host values, and so are kv_dtype (KV_BF16, or
    KV_FP8_E4M3 / "fp8" for a pool of e4m3 codes) with its scales k_scale and
    v_scale.
    """

    def __init__(self, query_start_loc, seq_lens, block_table, num_decodes, max_query_len,
                 max_seq_len, common_prefix_len=0, split_kv_tokens=0, kv_layout=LAYOUT_NHD,
                 kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0):
        self.query_start_loc = query_start_loc
        self.seq_lens = seq_lens
        self.block_table = block_table
        self.num_decodes = int(num_decodes)
        self.max_query_len = int(max_query_len)
        self.max_seq_len = int(max_seq_len)
        self.common_prefix_len = int(common_prefix_len)
        self.split_kv_tokens = int(split_kv_tokens)
        self.kv_layout = _layout(kv_layout)
        self.kv_dtype = _kv_dtype(kv_dtype)
        self.k_scale = float(k_scale)
        self.v_scale = float(v_scale)

    @classmethod
    def from_host(cls, query_start_loc, seq_lens, block_table, num_decodes, device,
                  common_prefix_len=0, split_kv_tokens=0, kv_layout=LAYOUT_NHD,
                  kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0):
        """Build from host (numpy) arrays, copying them to `device`."""
        import numpy as np
        import torch

        qsl = np.asarray(query_start_loc, dtype=np.int32)
        sl = np.asarray(seq_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        ql = np.diff(qsl)
        nd = int(num_decodes)
        max_q = int(ql[nd:].max()) if len(ql) > nd else 1
        max_s = int(sl.max()) if len(sl) else 1
        return cls(torch.from_numpy(qsl).to(device), torch.from_numpy(sl).to(device),
                   torch.from_numpy(bt).to(device), nd, max_q, max_s, common_prefix_len,
                   split_kv_tokens, kv_layout, kv_dtype, k_scale, v_scale)

    def _c(self) -> _CMeta:
        return _CMeta(self.query_start_loc.data_ptr(), self.seq_lens.data_ptr(),
                      self.block_table.data_ptr(), self.block_table.shape[1],
                      self.seq_lens.shape[0], self.num_decodes, self.max_query_len,
                      self.max_seq_len, self.common_prefix_len, self.split_kv_tokens,
                      self.kv_layout, self.kv_dtype, self.k_scale, self.v_scale)


def reshape_and_cache(key, value, kv_cache, slot_mapping, stream=None,
                      kv_layout=LAYOUT_NHD) -> None:
    """Scatter key/value [T, Hkv, D] rows into kv_cache at slot_mapping; the pool
    is [NB, 2, bs, Hkv, D] (NHD) or [NB, 2, Hkv, bs, D] (HND)."""
    lib = load_library()
    nb, bs, hkv, d = _pool_dims(kv_cache, kv_layout)
    _check(lib.pka_reshape_and_cache_ex(_ptr(key), _ptr(value), _ptr(kv_cache),
                                        _ptr(slot_mapping), key.shape[0], hkv, d, bs, nb,
                                        _layout(kv_layout), _stream(stream)))


def reshape_and_cache_fp8(key, value, kv_cache, slot_mapping, k_scale, v_scale, stream=None,
                          kv_layout=LAYOUT_NHD) -> None:
    """Quantise key/value [T, Hkv, D] (bf16) rows into an e4m3 pool (uint8 or
    float8_e4m3fn, [NB, 2, bs, Hkv, D] NHD or [NB, 2, Hkv, bs, D] HND):
    code = e4m3(x / scale), ties to even, clamped to +-448."""
    lib = load_library()
    if kv_cache.element_size() != 1:
        raise ValueError("an fp8 pool has one byte per element")
    nb, bs, hkv, d = _pool_dims(kv_cache, kv_layout)
    _check(lib.pka_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(kv_cache),
                                         _ptr(slot_mapping), key.shape[0], hkv, d, bs, nb,
                                         _layout(kv_layout), float(k_scale), float(v_scale),
                                         _stream(stream)))


def workspace_size(meta: Meta, num_tokens, num_heads, num_kv_heads, head_size, block_size) -> int:
    lib = load_library()
    cm = meta._c()
    return int(lib.pka_workspace_size(ctypes.byref(cm), num_tokens, num_heads, num_kv_heads,
                                      head_size, block_size))


def workspace_size_min(meta: Meta, num_tokens, num_heads, num_kv_heads, head_size,
                       block_size) -> int:
    """The smallest workspace the forward accepts (pka_workspace_size_min)."""
    lib = load_library()
    cm = meta._c()
    return int(lib.pka_workspace_size_min(ctypes.byref(cm), num_tokens, num_heads,
                                          num_kv_heads, head_size, block_size))


def paged_attn_forward(query, kv_cache, meta: Meta, out, lse=None, scale=None, causal=True,
                       workspace=None, stream=None) -> None:
    """out[T, H, D] (bf16) and lse[T, H] (fp32, ln) of the paged attention forward."""
    import torch

    lib = load_library()
    T, H, D = query.shape
    nb, bs, hkv, _ = _pool_dims(kv_cache, meta.kv_layout)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    cm = meta._c()
    need = int(lib.pka_workspace_size(ctypes.byref(cm), T, H, hkv, D, bs))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pka_paged_attn_forward(_ptr(query), _ptr(kv_cache), ctypes.byref(cm), _ptr(out),
                                      _ptr(lse), T, H, hkv, D, bs, nb, float(scale),
                                      1 if causal else 0, _ptr(workspace), ws_bytes,
                                      _stream(stream)))


def paged_attn_forward_fused(query, key, value, slot_mapping, kv_cache, meta: Meta, out,
                             lse=None, scale=None, causal=True, workspace=None,
                             stream=None) -> None:
    """reshape_and_cache(key, value, kv_cache, slot_mapping) then paged_attn_forward,
    with the cache write folded into the forward's decode launch."""
    import torch

    lib = load_library()
    T, H, D = query.shape
    nb, bs, hkv, _ = _pool_dims(kv_cache, meta.kv_layout)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    cm = meta._c()
    need = int(lib.pka_workspace_size(ctypes.byref(cm), T, H, hkv, D, bs))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pka_paged_attn_forward_fused(_ptr(query), _ptr(key), _ptr(value),
                                            _ptr(slot_mapping), _ptr(kv_cache), ctypes.byref(cm),
                                            _ptr(out), _ptr(lse), T, H, hkv, D, bs, nb,
                                            float(scale), 1 if causal else 0, _ptr(workspace),
                                            ws_bytes, _stream(stream)))


def paged_attn_forward_noalloc(query, kv_cache, meta: Meta, out, lse=None, scale=None,
                               causal=True, stream=None) -> None:
    """paged_attn_forward without a workspace: for callers that cannot allocate
    device memory, the library's built-in 16 MiB scratch holds the partial
    results.  Batches that need more raise PkaError (PKA_ERR_WORKSPACE).
    Calls that overlap on the GPU share that scratch and must be serialised."""
    lib = load_library()
    T, H, D = query.shape
    nb, bs, hkv, _ = _pool_dims(kv_cache, meta.kv_layout)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    cm = meta._c()
    _check(lib.pka_paged_attn_forward_noalloc(_ptr(query), _ptr(kv_cache), ctypes.byref(cm),
                                              _ptr(out), _ptr(lse), T, H, hkv, D, bs, nb,
                                              float(scale), 1 if causal else 0, _stream(stream)))


def cascade_merge(out_a, lse_a, out_b, lse_b, out, lse_out=None, stream=None) -> None:
    """Log-sum-exp merge of two partial attentions ([T, H, D] bf16 + [T, H] fp32 ln)."""
    lib = load_library()
    T, H, D = out_a.shape
    _check(lib.pka_cascade_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out),
                                 _ptr(lse_out), T, H, D, _stream(stream)))


# Units of a log-sum-exp (pka_lse_base)
LSE_BASE_E = 0
LSE_BASE_2 = 1


def merge_partials(outs, lses, out, lse_out=None, lse_base=LSE_BASE_E, stream=None) -> None:
    """Log-sum-exp merge of P partial attentions over disjoint key sets:
    outs [P, T, H, D] bf16, lses [P, T, H] fp32 in base lse_base (LSE_BASE_E:
    natural log, LSE_BASE_2: log2) -> out [T, H, D] bf16, lse_out [T, H] in the
    same base."""
    lib = load_library()
    P, T, H, D = outs.shape
    _check(lib.pka_merge_partials(_ptr(outs), _ptr(lses), P, _ptr(out), _ptr(lse_out), T, H, D,
                                  int(lse_base), _stream(stream)))


KERNEL_DECODE = 0
KERNEL_PREFILL = 1


def set_kernel_events(kernel: int, start=None, stop=None) -> None:
    """Record torch CUDA events `start`/`stop` around the named kernel in every
    later forward on this thread (None turns it off)."""
    def raw(e):
        return None if e is None else ctypes.c_void_p(e.cuda_event)

    _check(load_library().pka_set_kernel_events(kernel, raw(start), raw(stop)))


def test_skip_copies(on: bool) -> None:
    """Failure-path test hook (pka_test_skip_copies): while on, the kernels of
    later forwards on this thread issue no copies, so their first bounded wait
    runs out and check_status() raises PKA_ERR_DEVICE_CHECK.  Tests only."""
    _check(load_library().pka_test_skip_copies(1 if on else 0))


def kernel_launches() -> int:
    """Kernels the library has launched from this thread so far."""
    return int(load_library().pka_kernel_launches())


def check_status(stream=None) -> None:
    """Synchronise the stream and raise if a device-side check failed."""
    _check(load_library().pka_check_status(_stream(stream)))
