"""Python binding of the pkvqk C ABI (``include/pkvqk.h``).

Argument marshalling only: the ``pkvqk_*`` functions below have the C names
and C arguments (integers for pointers, ints, floats); the short-named
helpers (``norm_rope_append``, ``paged_decode``, ``paged_prefill``,
``lse_combine``) take torch
tensors, read their data pointers and strides and call the C entry point on
the current CUDA stream.  All computation happens in the library's kernels;
if ``libpkvqk.so`` is missing or fails to load, importing this module raises.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkvqk.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} not found: build it with `python -m paged_kv_cache_qk_gb300.build` "
        "(there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

c_i32, c_i64, c_f32, c_size, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

PKVQK_OK = 0
PKVQK_ERR_INVALID_ARG = 1
PKVQK_ERR_UNSUPPORTED = 2
PKVQK_ERR_WORKSPACE_TOO_SMALL = 3
PKVQK_ERR_POINTER_RESIDENCY = 4
PKVQK_ERR_CUDA = 5
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL",
                4: "POINTER_RESIDENCY", 5: "CUDA"}

FLAG_BAD_SLOT = 0x1
FLAG_BAD_BLOCK_ID = 0x2
FLAG_WAIT_TIMEOUT = 0x4


class CacheLayout(ctypes.Structure):
    """Mirror of ``pkvqk_cache_layout``."""
    _fields_ = [
        ("num_blocks", c_i64),
        ("block_size", c_i32),
        ("num_kv_heads", c_i32),
        ("head_dim", c_i32),
        ("reserved", c_i32),
        ("block_stride", c_i64),
        ("slot_stride", c_i64),
        ("head_stride", c_i64),
    ]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


pkvqk_last_error = _sig("pkvqk_last_error", ctypes.c_char_p, [])
pkvqk_abi_version = _sig("pkvqk_abi_version", c_i32, [])
pkvqk_norm_rope_append = _sig("pkvqk_norm_rope_append", ctypes.c_int, [
    c_vp, c_i64, c_i64,                 # q, strides
    c_vp, c_i64, c_i64,                 # k
    c_vp, c_i64, c_i64,                 # v
    c_vp, c_vp,                         # positions, slot_mapping
    c_vp, c_vp,                         # gamma_q, gamma_k
    c_f32, c_f32,                       # theta, eps
    c_i32, c_i32,                       # num_tokens, num_q_heads
    c_vp, c_vp, ctypes.POINTER(CacheLayout),
    c_vp, c_vp])                        # status_flags, stream
pkvqk_rope_table_bytes = _sig("pkvqk_rope_table_bytes", c_size, [c_i32])
pkvqk_rope_table_build = _sig("pkvqk_rope_table_build", ctypes.c_int, [c_vp, c_i32, c_f32, c_vp])
pkvqk_norm_rope_append_cached = _sig("pkvqk_norm_rope_append_cached", ctypes.c_int, [
    c_vp, c_i64, c_i64,                 # q, strides
    c_vp, c_i64, c_i64,                 # k
    c_vp, c_i64, c_i64,                 # v
    c_vp, c_vp,                         # positions, slot_mapping
    c_vp, c_vp,                         # gamma_q, gamma_k
    c_f32, c_f32,                       # theta, eps
    c_i32, c_i32,                       # num_tokens, num_q_heads
    c_vp, c_vp, ctypes.POINTER(CacheLayout),
    c_vp, c_i32,                        # rope_table, table_positions
    c_vp, c_vp])                        # status_flags, stream
pkvqk_choose_num_splits = _sig("pkvqk_choose_num_splits", c_i32,
                               [c_i32, c_i32, c_i32, c_i32, c_i64, c_i32, c_i32])
pkvqk_decode_workspace_bytes = _sig("pkvqk_decode_workspace_bytes", c_size,
                                    [c_i32, c_i32, c_i32, c_i32, c_i32])
_decode_args = [
    c_vp, c_i64, c_i64,                 # q, strides
    c_vp, c_vp, ctypes.POINTER(CacheLayout),
    c_vp, c_i32,                        # block_tables, max_blocks_per_seq
    c_vp,                               # seq_lens
    c_i32, c_i32, c_i32,                # batch, q_len, num_q_heads
    c_i32, c_i32, c_f32,                # num_splits, max_seq_len_hint, scale
]
pkvqk_paged_decode = _sig("pkvqk_paged_decode", ctypes.c_int,
                          _decode_args + [c_vp, c_vp, c_vp, c_size, c_vp, c_vp])
pkvqk_paged_decode_partials = _sig("pkvqk_paged_decode_partials", ctypes.c_int,
                                   _decode_args + [c_vp, c_size, c_vp, c_vp])
pkvqk_lse_combine = _sig("pkvqk_lse_combine", ctypes.c_int,
                         [c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp])
pkvqk_paged_decode_static_ws = _sig("pkvqk_paged_decode_static_ws", ctypes.c_int,
                                    _decode_args + [c_vp, c_vp, c_vp, c_vp])
pkvqk_static_workspace_capacity = _sig("pkvqk_static_workspace_capacity", c_size, [])
pkvqk_choose_prefill_splits = _sig("pkvqk_choose_prefill_splits", c_i32,
                                   [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32])
pkvqk_prefill_workspace_bytes = _sig("pkvqk_prefill_workspace_bytes", c_size,
                                     [c_i32, c_i32, c_i32, c_i32, c_i32])
pkvqk_paged_prefill = _sig("pkvqk_paged_prefill", ctypes.c_int,
                           _decode_args + [c_vp, c_vp, c_vp, c_size, c_vp, c_vp])
pkvqk_paged_prefill_varlen = _sig("pkvqk_paged_prefill_varlen", ctypes.c_int, [
    c_vp, c_i64, c_i64,                 # q, strides
    c_vp, c_i32, c_i64,                 # cu_seqlens_q, max_q_len, total_q
    c_vp, c_vp, ctypes.POINTER(CacheLayout),
    c_vp, c_i32, c_vp,                  # block_tables, max_blocks_per_seq, seq_lens
    c_i32, c_i32,                       # batch, num_q_heads
    c_i32, c_i32, c_f32,                # num_splits, max_seq_len_hint, scale
    c_vp, c_vp, c_vp, c_size, c_vp, c_vp])

EXPORTED = [
    "pkvqk_last_error", "pkvqk_abi_version", "pkvqk_norm_rope_append",
    "pkvqk_choose_num_splits", "pkvqk_decode_workspace_bytes", "pkvqk_paged_decode",
    "pkvqk_paged_decode_partials", "pkvqk_lse_combine", "pkvqk_paged_decode_static_ws",
    "pkvqk_static_workspace_capacity", "pkvqk_choose_prefill_splits",
    "pkvqk_prefill_workspace_bytes", "pkvqk_paged_prefill", "pkvqk_paged_prefill_varlen",
    "pkvqk_rope_table_bytes", "pkvqk_rope_table_build", "pkvqk_norm_rope_append_cached",
]


class PkvqkError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"pkvqk status {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status):
    if status != PKVQK_OK:
        raise PkvqkError(status, pkvqk_last_error().decode(errors="replace"))
    return status


# ---------------------------------------------------------- torch helpers

def _torch():
    import torch
    return torch


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def cache_layout(k_cache) -> CacheLayout:
    """Layout of a [num_blocks, block_size, num_kv_heads, head_dim] (strided) cache view."""
    nb, bs, hkv, d = k_cache.shape
    s = k_cache.stride()
    if s[3] != 1:
        raise ValueError("head_dim must be the contiguous axis")
    return CacheLayout(nb, bs, hkv, d, 0, s[0], s[1], s[2])


def norm_rope_append(q, k, v, positions, slot_mapping, gamma_q, gamma_k, theta, eps,
                     k_cache, v_cache, status_flags=None, stream=None):
    """q [T, Hq, D] (in place), k/v [T, Hkv, D], caches [NB, bs, Hkv, D] views."""
    T, Hq, D = q.shape
    lay = cache_layout(k_cache)
    if tuple(v_cache.stride()) != tuple(k_cache.stride()) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share one layout")
    check(pkvqk_norm_rope_append(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1),
        _ptr(positions), _ptr(slot_mapping), _ptr(gamma_q), _ptr(gamma_k),
        float(theta), float(eps), T, Hq,
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(status_flags), _stream(stream)))


def rope_table_bytes(max_positions):
    return int(pkvqk_rope_table_bytes(max_positions))


def rope_table_build(table, max_positions, theta, stream=None):
    """table: device tensor of at least rope_table_bytes(max_positions) bytes."""
    if max_positions > 0 and table.numel() * table.element_size() < rope_table_bytes(max_positions):
        raise ValueError("rope table too small")
    check(pkvqk_rope_table_build(_ptr(table), max_positions, float(theta), _stream(stream)))


def norm_rope_append_cached(q, k, v, positions, slot_mapping, gamma_q, gamma_k, theta, eps,
                            k_cache, v_cache, rope_table, table_positions, status_flags=None,
                            stream=None):
    """norm_rope_append with the angles of positions < table_positions read from a
    table built by rope_table_build (same theta)."""
    T, Hq, D = q.shape
    lay = cache_layout(k_cache)
    if tuple(v_cache.stride()) != tuple(k_cache.stride()) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share one layout")
    check(pkvqk_norm_rope_append_cached(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1),
        _ptr(positions), _ptr(slot_mapping), _ptr(gamma_q), _ptr(gamma_k),
        float(theta), float(eps), T, Hq,
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(rope_table), int(table_positions),
        _ptr(status_flags), _stream(stream)))


def decode_workspace_bytes(batch, q_len, num_q_heads, head_dim, num_splits):
    return int(pkvqk_decode_workspace_bytes(batch, q_len, num_q_heads, head_dim, num_splits))


def choose_num_splits(batch, num_kv_heads, rows_per_kv_head, max_seq_len, total_tokens,
                      block_size, sm_count=0):
    return int(pkvqk_choose_num_splits(batch, num_kv_heads, rows_per_kv_head, max_seq_len,
                                       total_tokens, block_size, sm_count))


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, out, *, q_len=1, num_splits=1,
                 max_seq_len_hint=0, scale=0.0, lse_out=None, workspace=None,
                 status_flags=None, stream=None):
    """q [B*q_len, Hq, D]; out [B, q_len, Hq, D] (or [B*q_len, Hq, D]) contiguous bf16."""
    Tq, Hq, D = q.shape
    B = Tq // q_len
    lay = cache_layout(k_cache)
    if tuple(v_cache.stride()) != tuple(k_cache.stride()) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share one layout")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(pkvqk_paged_decode(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        B, q_len, Hq, int(num_splits), int(max_seq_len_hint), float(scale),
        _ptr(out), _ptr(lse_out), _ptr(workspace), ws_bytes,
        _ptr(status_flags), _stream(stream)))


def paged_decode_partials(q, k_cache, v_cache, block_tables, seq_lens, workspace, *, q_len=1,
                          num_splits=2, max_seq_len_hint=0, scale=0.0, status_flags=None,
                          stream=None):
    Tq, Hq, D = q.shape
    B = Tq // q_len
    lay = cache_layout(k_cache)
    ws_bytes = workspace.numel() * workspace.element_size()
    check(pkvqk_paged_decode_partials(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        B, q_len, Hq, int(num_splits), int(max_seq_len_hint), float(scale),
        _ptr(workspace), ws_bytes, _ptr(status_flags), _stream(stream)))


def lse_combine(ws_o, ws_lse, rows, num_splits, out, lse_out=None, stream=None):
    check(pkvqk_lse_combine(_ptr(ws_o), _ptr(ws_lse), int(rows), 128, int(num_splits),
                            _ptr(out), _ptr(lse_out), _stream(stream)))


def choose_prefill_splits(batch, num_kv_heads, q_len, group, max_seq_len, sm_count=0):
    return int(pkvqk_choose_prefill_splits(batch, num_kv_heads, q_len, group, max_seq_len,
                                           sm_count))


def prefill_workspace_bytes(batch, q_len, num_q_heads, head_dim, num_splits):
    return int(pkvqk_prefill_workspace_bytes(batch, q_len, num_q_heads, head_dim, num_splits))


def paged_prefill(q, k_cache, v_cache, block_tables, seq_lens, out, *, q_len, num_splits=1,
                  max_seq_len_hint=0, scale=0.0, lse_out=None, workspace=None,
                  status_flags=None, stream=None):
    """Causal multi-query attention on the tensor cores.

    q [B*q_len, Hq, D]; out [B, q_len, Hq, D] (or [B*q_len, Hq, D]) contiguous bf16.
    """
    Tq, Hq, D = q.shape
    B = Tq // q_len
    lay = cache_layout(k_cache)
    if tuple(v_cache.stride()) != tuple(k_cache.stride()) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share one layout")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(pkvqk_paged_prefill(
        _ptr(q), q.stride(0), q.stride(1),
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        B, q_len, Hq, int(num_splits), int(max_seq_len_hint), float(scale),
        _ptr(out), _ptr(lse_out), _ptr(workspace), ws_bytes,
        _ptr(status_flags), _stream(stream)))


def paged_prefill_varlen(q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables, seq_lens,
                         out, *, num_splits=1, max_seq_len_hint=0, scale=0.0, lse_out=None,
                         workspace=None, status_flags=None, stream=None):
    """Varlen causal multi-query attention on the tensor cores.

    q [total_q, Hq, D] packed rows, cu_seqlens_q int32 [B + 1] on the device,
    max_q_len a host int; out [total_q, Hq, D] contiguous bf16.
    """
    total_q, Hq, D = q.shape
    B = cu_seqlens_q.shape[0] - 1
    lay = cache_layout(k_cache)
    if tuple(v_cache.stride()) != tuple(k_cache.stride()) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must share one layout")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(pkvqk_paged_prefill_varlen(
        _ptr(q), q.stride(0), q.stride(1), _ptr(cu_seqlens_q), int(max_q_len), int(total_q),
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(lay),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        B, Hq, int(num_splits), int(max_seq_len_hint), float(scale),
        _ptr(out), _ptr(lse_out), _ptr(workspace), ws_bytes,
        _ptr(status_flags), _stream(stream)))
