"""ctypes front end of the plain-C fp64 oracle (oracle/pagedkv_oracle.c).

TEST INFRASTRUCTURE ONLY: used by tests/, the smoke check and the benchmark's
CPU-baseline leg; the product path never imports it.  Inputs are CPU torch
tensors (or numpy arrays) in their storage dtype; the C code decodes the
16-bit formats itself, exactly, and computes in fp64.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import build as _build

_lib = None

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.float64: 3}
_NP_DT = {np.dtype(np.float16): 0, np.dtype(np.float32): 2, np.dtype(np.float64): 3}

_p = C.c_void_p
_i32 = C.c_int32
_i64 = C.c_int64
_d = C.c_double


def lib():
    global _lib
    if _lib is None:
        # PKV_ORACLE_LIB points the oracle at another build of the same C
        # source (the mutation tests use it to plant mistakes).
        path = os.environ.get("PKV_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        L.orc_f16_bits_to_double.restype = _d
        L.orc_f16_bits_to_double.argtypes = [C.c_uint16]
        L.orc_bf16_bits_to_double.restype = _d
        L.orc_bf16_bits_to_double.argtypes = [C.c_uint16]
        L.orc_decode_elements.restype = None
        L.orc_decode_elements.argtypes = [_p, _p, C.c_size_t, C.c_int]
        L.orc_kv_cache_bytes.restype = C.c_uint64
        L.orc_kv_cache_bytes.argtypes = [C.c_uint64] * 6
        L.orc_paged_decode_two_pass.restype = C.c_int
        L.orc_paged_decode_two_pass.argtypes = [_p, _p, _p, _p, C.c_int, _p, C.c_int, _p, _p,
                                                C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                                C.c_int, C.c_int, _d]
        L.orc_paged_decode_online.restype = C.c_int
        L.orc_paged_decode_online.argtypes = [_p, _p, _p, _p, _p, _p, C.c_int, _p, C.c_int, _p,
                                              _p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                              C.c_int, C.c_int, _d, C.c_int, C.c_int, C.c_int]
        L.orc_paged_multi_query.restype = C.c_int
        L.orc_paged_multi_query.argtypes = [_p, _p, _p, _p, C.c_int, _p, C.c_int, _p, _p, C.c_int,
                                            C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _d]
        L.orc_merge_states.restype = None
        L.orc_merge_states.argtypes = [_p, _p, _p, _p, C.c_int, C.c_int]
        L.orc_kv_append.restype = C.c_int
        L.orc_kv_append.argtypes = [_p, _p, _p, _p, C.c_int, _p, C.c_int, C.c_int, C.c_int,
                                    C.c_int, _i64]
        L.orc_swap_blocks.restype = _i64
        L.orc_swap_blocks.argtypes = [_p, _p, _i64, _p, _i64, _i64, _i64]
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _cpu(t):
    """Contiguous CPU tensor view (numpy arrays are wrapped without copy)."""
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(t))
    if t.device.type != "cpu":
        raise OracleError("the oracle reads host memory only")
    return t.contiguous()


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t.numel() else C.c_void_p(0)


def kv_cache_bytes(n_layers, n_heads, d_head, seq_len, batch, elem_bytes=2) -> int:
    return int(lib().orc_kv_cache_bytes(n_layers, n_heads, d_head, seq_len, batch, elem_bytes))


def decode_elements(bits: torch.Tensor, dtype: torch.dtype) -> np.ndarray:
    """Decode a buffer of `dtype` elements to float64 with the oracle's own
    decoders (bits: any tensor whose bytes are the elements)."""
    t = _cpu(bits).view(dtype)
    out = np.empty(t.numel(), dtype=np.float64)
    lib().orc_decode_elements(out.ctypes.data, _ptr(t), t.numel(), _DT[dtype])
    return out.reshape(tuple(t.shape))


def _decode_args(q, k_pool, v_pool, block_tables, context_lens, seq_ids):
    q, k_pool, v_pool = _cpu(q), _cpu(k_pool), _cpu(v_pool)
    if not (q.dtype == k_pool.dtype == v_pool.dtype):
        raise OracleError("q, k_pool and v_pool must share one dtype")
    bt = _cpu(block_tables).to(torch.int32).contiguous()
    cl = _cpu(context_lens).to(torch.int32).contiguous()
    S, H, D = q.shape
    nb, B, Hk, D2 = k_pool.shape
    if D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise OracleError("pool shapes disagree")
    if seq_ids is None:
        sel = torch.arange(S, dtype=torch.int32)
    else:
        sel = torch.as_tensor(seq_ids, dtype=torch.int32).contiguous()
    return q, k_pool, v_pool, bt, cl, sel, (S, H, Hk, D, B, nb)


def decode_two_pass(q, k_pool, v_pool, block_tables, context_lens, scale, seq_ids=None):
    """fp64 softmax(q K^T * scale) V over the logically gathered context of
    each selected sequence.  Returns float64 ndarray [n_sel, H, D]."""
    q, k, v, bt, cl, sel, (S, H, Hk, D, B, nb) = _decode_args(q, k_pool, v_pool, block_tables,
                                                              context_lens, seq_ids)
    out = np.zeros((sel.numel(), H, D), dtype=np.float64)
    rc = lib().orc_paged_decode_two_pass(out.ctypes.data, _ptr(q), _ptr(k), _ptr(v), _DT[q.dtype],
                                         _ptr(bt), bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl),
                                         _ptr(sel), sel.numel(), S, H, Hk, D, B, nb, float(scale))
    if rc != 0:
        raise OracleError(f"orc_paged_decode_two_pass failed with code {rc}")
    return out


def decode_online(q, k_pool, v_pool, block_tables, context_lens, scale, tile_tokens, seq_ids=None,
                  t_begin=0, t_end=-1, return_state=False):
    """The pages' one-pass recurrence with tiles of `tile_tokens` keys over
    logical tokens [t_begin, t_end).  Returns O (and (M, L) if asked)."""
    q, k, v, bt, cl, sel, (S, H, Hk, D, B, nb) = _decode_args(q, k_pool, v_pool, block_tables,
                                                              context_lens, seq_ids)
    out = np.zeros((sel.numel(), H, D), dtype=np.float64)
    m = np.zeros((sel.numel(), H), dtype=np.float64)
    l_ = np.zeros((sel.numel(), H), dtype=np.float64)
    rc = lib().orc_paged_decode_online(out.ctypes.data, m.ctypes.data, l_.ctypes.data, _ptr(q),
                                       _ptr(k), _ptr(v), _DT[q.dtype], _ptr(bt),
                                       bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl), _ptr(sel),
                                       sel.numel(), S, H, Hk, D, B, nb, float(scale),
                                       int(tile_tokens), int(t_begin), int(t_end))
    if rc != 0:
        raise OracleError(f"orc_paged_decode_online failed with code {rc}")
    return (out, m, l_) if return_state else out


def multi_query(q, k_pool, v_pool, block_tables, context_lens, q_start, scale):
    """fp64 causal attention of each sequence's last q_len tokens over its
    paged context.  q [total_q, H, D], q_start int32 [S + 1].  Returns
    float64 ndarray [total_q, H, D]."""
    q, k, v = _cpu(q), _cpu(k_pool), _cpu(v_pool)
    if not (q.dtype == k.dtype == v.dtype):
        raise OracleError("q, k_pool and v_pool must share one dtype")
    bt = _cpu(block_tables).to(torch.int32).contiguous()
    cl = _cpu(context_lens).to(torch.int32).contiguous()
    qs = _cpu(q_start).to(torch.int32).contiguous()
    T, H, D = q.shape
    nb, B, Hk, _ = k.shape
    S = cl.numel()
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = lib().orc_paged_multi_query(out.ctypes.data, _ptr(q), _ptr(k), _ptr(v), _DT[q.dtype],
                                     _ptr(bt), bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl),
                                     _ptr(qs), S, H, Hk, D, B, nb, float(scale))
    if rc != 0:
        raise OracleError(f"orc_paged_multi_query failed with code {rc}")
    return out


def merge_states(m, l_, o):
    """Merge partial states of one output row: m, l [P], o [P, D]."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l_ = np.ascontiguousarray(l_, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    out = np.zeros(o.shape[1], dtype=np.float64)
    lib().orc_merge_states(out.ctypes.data, m.ctypes.data, l_.ctypes.data, o.ctypes.data,
                           o.shape[0], o.shape[1])
    return out


def kv_append(k_pool, v_pool, k_new, v_new, slot_mapping):
    """In place on CPU tensors: pools [nb, B, Hk, D], k_new/v_new [S, Hk, D],
    slot_mapping int64 [S] (-1 skips)."""
    for t in (k_pool, v_pool):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise OracleError("pools must be contiguous CPU tensors (written in place)")
    kn, vn = _cpu(k_new), _cpu(v_new)
    sm = _cpu(slot_mapping).to(torch.int64).contiguous()
    nb, B, Hk, D = k_pool.shape
    rc = lib().orc_kv_append(_ptr(k_pool), _ptr(v_pool), _ptr(kn), _ptr(vn), k_pool.element_size(),
                             _ptr(sm), sm.numel(), Hk, D, B, nb)
    if rc != 0:
        raise OracleError(f"orc_kv_append failed with code {rc}")


def swap_blocks(dst_pool, src_pool, pairs) -> int:
    """In place: dst_pool[j] = src_pool[i] for each (i, j) row of `pairs`
    (int64 [n, 2]).  Returns the count of out-of-range pairs skipped."""
    if dst_pool.device.type != "cpu" or not dst_pool.is_contiguous():
        raise OracleError("dst_pool must be a contiguous CPU tensor")
    src = _cpu(src_pool)
    pr = _cpu(pairs).to(torch.int64).contiguous()
    bb = dst_pool[0].numel() * dst_pool.element_size() if dst_pool.shape[0] else 0
    if src.shape[0] and src[0].numel() * src.element_size() != bb:
        raise OracleError("source and destination blocks differ in size")
    return int(lib().orc_swap_blocks(_ptr(dst_pool), _ptr(src), bb, _ptr(pr), pr.shape[0],
                                     src.shape[0], dst_pool.shape[0]))
