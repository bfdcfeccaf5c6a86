"""torch-facing binding of the C ABI: the same entry points as include/pagedkv.h,
taking tensors and doing argument marshalling only (shapes, dtypes, pointers,
the current CUDA stream).  Every step of the computation runs in the library's
CUDA kernels; torch provides device memory and streams.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _lib
from ._lib import check, lib

_DT = {torch.float16: _lib.PKV_F16, torch.bfloat16: _lib.PKV_BF16, torch.float32: _lib.PKV_F32}


# The current stream's raw handle without building a Stream object (a few
# microseconds per call); the public call where torch lacks the shortcut.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    if stream is not None:
        return C.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        return C.c_void_p(_raw_stream(torch.cuda.current_device()))
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return C.c_void_p(t.data_ptr()) if t is not None and t.numel() else C.c_void_p(0)


def _need_cuda(name: str, t: torch.Tensor):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_all_cuda(names, tensors) -> None:
    """_need_cuda over several tensors; the per-name pass runs only when one
    fails (the decode calls sit on a serving loop's critical path)."""
    for t in tensors:
        if not (t.is_cuda and t.is_contiguous()):
            for name, u in zip(names, tensors):
                _need_cuda(name, u)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    """_stream_ptr as a plain integer (ctypes converts it for a void* argument)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _addr(t: Optional[torch.Tensor]) -> int:
    """_ptr as a plain integer."""
    return t.data_ptr() if t is not None and t.numel() else 0


_DECODE_NAMES = ("out", "q", "k_pool", "v_pool", "block_tables", "context_lens")
_APPEND_NAMES = _DECODE_NAMES + ("k_new", "v_new", "slot_mapping")


def set_tuning(**knobs) -> None:
    """Override launch shapes for tests and tuning sweeps, e.g.
    ``set_tuning(decode_hpc=2, mq_tc=0)``; a value of None restores the
    automatic choice.  Names: the pkv_tune_knob names of pagedkv.h in lower
    case without the PKV_TUNE_ prefix.  Process-wide."""
    for name, value in knobs.items():
        if name not in _lib.TUNE_KNOBS:
            raise ValueError(f"unknown tuning knob {name!r}")
        v = _lib.TUNE_AUTO if value is None else int(value)
        check(lib().pkv_set_tuning(_lib.TUNE_KNOBS[name], v), "pkv_set_tuning")


def get_tuning(name: str) -> Optional[int]:
    """Current override of one knob, None when it holds the automatic choice."""
    v = int(lib().pkv_get_tuning(_lib.TUNE_KNOBS[name]))
    return None if v == _lib.TUNE_AUTO else v


def reset_tuning() -> None:
    """Every knob back to the automatic choice."""
    set_tuning(**{name: None for name in _lib.TUNE_KNOBS})


def decode_workspace_bytes(num_seqs: int, n_heads: int, n_kv_heads: int, head_dim: int,
                           block_size: int, max_context_len: int, split_tokens: int = 0) -> int:
    return int(lib().pkv_decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim,
                                                block_size, max_context_len, split_tokens))


def decode_split_tokens(num_seqs: int, n_heads: int, n_kv_heads: int, head_dim: int,
                        block_size: int, max_context_len: int) -> int:
    return int(lib().pkv_decode_split_tokens(num_seqs, n_heads, n_kv_heads, head_dim, block_size,
                                             max_context_len))


class _Shape(C.Structure):
    """pkv_decode_shape of include/pagedkv.h."""
    _fields_ = [("kernel", C.c_int), ("split_tokens", C.c_int), ("max_splits", C.c_int),
                ("heads_per_cta", C.c_int), ("stages", C.c_int), ("warps_per_token", C.c_int),
                ("threads", C.c_int), ("stream_ctas", C.c_int), ("smem_bytes", C.c_size_t)]


_KERNELS = ("cuda_core", "tensor_core", "streaming")


def decode_launch_shape(num_seqs: int, n_heads: int, n_kv_heads: int, head_dim: int,
                        block_size: int, max_context_len: int, split_tokens: int = 0,
                        sm_count: int = 152, smem_optin: int = 232448,
                        smem_per_sm: int = 233472) -> dict:
    """The launch shape the automatic choice takes for a decode problem on a
    device with these facts (default: GB300's), by host arithmetic only --
    kernel ("cuda_core", "tensor_core" or "streaming"), split_tokens,
    max_splits, heads_per_cta, stages, warps_per_token, threads,
    stream_ctas, smem_bytes."""
    sh = _Shape()
    check(lib().pkv_decode_launch_shape(num_seqs, n_heads, n_kv_heads, head_dim, block_size,
                                        max_context_len, split_tokens, sm_count, smem_optin,
                                        smem_per_sm, C.byref(sh)), "pkv_decode_launch_shape")
    out = {name: getattr(sh, name) for name, _ in _Shape._fields_}
    out["kernel"] = _KERNELS[sh.kernel]
    return out


def alloc_decode_workspace(q: torch.Tensor, k_pool: torch.Tensor, max_context_len: int,
                           split_tokens: int = 0) -> Optional[torch.Tensor]:
    S, H, D = q.shape
    _, B, Hk, _ = k_pool.shape
    n = decode_workspace_bytes(S, H, Hk, D, B, max_context_len, split_tokens)
    if n == 0:
        return None
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def paged_attn_decode(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                      v_pool: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, max_context_len: int,
                      split_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[s,h] = softmax(scale * q[s,h] . K^T) V over the paged context of s.
    Shapes: q/out [S, H, D], pools [num_blocks, B, Hk, D], block_tables int32
    [S, max_blocks], context_lens int32 [S]."""
    _need_all_cuda(_DECODE_NAMES, (out, q, k_pool, v_pool, block_tables, context_lens))
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    S, H, D = q.shape
    nb, B, Hk, D2 = k_pool.shape
    if (D2 != D or v_pool.shape != k_pool.shape or out.shape != q.shape
            or q.dtype != k_pool.dtype or v_pool.dtype != k_pool.dtype
            or block_tables.dim() != 2 or block_tables.shape[0] != S
            or context_lens.shape != (S,)):
        raise ValueError("inconsistent shapes or dtypes")
    if workspace is None:
        workspace = alloc_decode_workspace(q, k_pool, max_context_len, split_tokens)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().paged_attn_decode(out.data_ptr(), _DT[out.dtype], q.data_ptr(), _addr(k_pool),
                                 _addr(v_pool), _DT[k_pool.dtype], block_tables.data_ptr(),
                                 block_tables.shape[1], context_lens.data_ptr(), S, H, Hk, D, B,
                                 nb, float(scale), int(max_context_len), int(split_tokens),
                                 _addr(workspace), ws_bytes, _stream_handle(stream))
    check(st, "paged_attn_decode")
    return out


def _append_args(out, q, k_pool, v_pool, block_tables, context_lens, scale, max_context_len,
                 k_new, v_new, slot_mapping, split_tokens, workspace, stream) -> tuple:
    """Checked C arguments of paged_attn_decode_append (its order)."""
    _need_all_cuda(_APPEND_NAMES, (out, q, k_pool, v_pool, block_tables, context_lens, k_new,
                                   v_new, slot_mapping))
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    S, H, D = q.shape
    nb, B, Hk, D2 = k_pool.shape
    if (D2 != D or v_pool.shape != k_pool.shape or out.shape != q.shape
            or q.dtype != k_pool.dtype or v_pool.dtype != k_pool.dtype
            or block_tables.dim() != 2 or block_tables.shape[0] != S
            or context_lens.shape != (S,) or k_new.shape != (S, Hk, D)
            or k_new.shape != v_new.shape or k_new.dtype != k_pool.dtype
            or v_new.dtype != k_pool.dtype or slot_mapping.shape != (S,)):
        raise ValueError("inconsistent shapes or dtypes")
    if workspace is None:
        workspace = alloc_decode_workspace(q, k_pool, max_context_len, split_tokens)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return (out.data_ptr(), _DT[out.dtype], q.data_ptr(), _addr(k_pool), _addr(v_pool),
            _DT[k_pool.dtype], block_tables.data_ptr(), block_tables.shape[1],
            context_lens.data_ptr(), S, H, Hk, D, B, nb, float(scale), int(max_context_len),
            int(split_tokens), _addr(workspace), ws_bytes, k_new.data_ptr(), v_new.data_ptr(),
            slot_mapping.data_ptr(), _stream_handle(stream))


def paged_attn_decode_append(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                             v_pool: torch.Tensor, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, scale: float, max_context_len: int,
                             k_new: torch.Tensor, v_new: torch.Tensor,
                             slot_mapping: torch.Tensor, split_tokens: int = 0,
                             workspace: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """kv_append(k_pool, v_pool, k_new, v_new, slot_mapping) then
    paged_attn_decode(...) in one launch; context_lens counts the appended
    token.  No other sequence of the call may read a page that holds a slot."""
    st = lib().paged_attn_decode_append(
        *_append_args(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                      max_context_len, k_new, v_new, slot_mapping, split_tokens, workspace,
                      stream))
    check(st, "paged_attn_decode_append")
    return out


class _Copy(C.Structure):
    """pkv_copy of include/pagedkv.h."""
    _fields_ = [("host", C.c_void_p), ("device", C.c_void_p), ("bytes", C.c_size_t)]


class HostStep:
    """A serving step from host memory, prepared once: every
    (host tensor, device tensor) pair of `copies` is copied host to device
    (the host tensor's bytes; pinned memory copies asynchronously), then
    paged_attn_decode_append runs on the device tensors, then `out` is
    copied back into `out_host` (a CPU tensor of the same shape and dtype),
    and with `synchronize` the step returns once the stream is idle -- one
    library call (paged_attn_decode_append_host) per run().  The arguments
    are checked and marshalled here, so run() issues the copies at once.
    Between runs the tensors' contents may change (the step's inputs, the
    pools, the lengths), not their addresses; max_context_len must bound
    every context of every run.  `stream` is fixed here (None: the current
    stream now)."""

    def __init__(self, copies, out_host: torch.Tensor, out: torch.Tensor, q: torch.Tensor,
                 k_pool: torch.Tensor, v_pool: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, scale: float, max_context_len: int,
                 k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                 split_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None, synchronize: bool = True):
        _need_all_cuda(_APPEND_NAMES, (out, q, k_pool, v_pool, block_tables, context_lens, k_new,
                                       v_new, slot_mapping))
        if workspace is None:
            workspace = alloc_decode_workspace(q, k_pool, max_context_len, split_tokens)
        args = _append_args(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                            max_context_len, k_new, v_new, slot_mapping, split_tokens, workspace,
                            stream)
        pairs = list(copies)
        arr = (_Copy * max(1, len(pairs)))()
        for i, (h, d) in enumerate(pairs):
            if h.is_cuda or not d.is_cuda:
                raise ValueError("each copy is a (host tensor, device tensor) pair")
            nbytes = h.numel() * h.element_size()
            if not (h.is_contiguous() and d.is_contiguous()) or \
                    d.numel() * d.element_size() < nbytes:
                raise ValueError("copies need contiguous tensors and room on the device")
            arr[i].host, arr[i].device, arr[i].bytes = h.data_ptr(), d.data_ptr(), nbytes
        if out_host.is_cuda or out_host.shape != out.shape or out_host.dtype != out.dtype or \
                not out_host.is_contiguous():
            raise ValueError("out_host must be a contiguous CPU tensor shaped like out")
        # the tensors stay referenced while the step may run
        self._keep = (pairs, out_host, out, q, k_pool, v_pool, block_tables, context_lens,
                      k_new, v_new, slot_mapping, workspace)
        self._fn = lib().paged_attn_decode_append_host
        self._args = (arr, len(pairs), out_host.data_ptr(), out.numel() * out.element_size(),
                      1 if synchronize else 0) + args
        self.out_host = out_host

    def run(self) -> torch.Tensor:
        check(self._fn(*self._args), "paged_attn_decode_append_host")
        return self.out_host


def paged_attn_decode_append_host(copies, out_host: torch.Tensor, out: torch.Tensor,
                                  q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  scale: float, max_context_len: int, k_new: torch.Tensor,
                                  v_new: torch.Tensor, slot_mapping: torch.Tensor,
                                  split_tokens: int = 0,
                                  workspace: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None,
                                  synchronize: bool = True) -> torch.Tensor:
    """One HostStep, prepared and run once (see HostStep)."""
    return HostStep(copies, out_host, out, q, k_pool, v_pool, block_tables, context_lens, scale,
                    max_context_len, k_new, v_new, slot_mapping, split_tokens, workspace, stream,
                    synchronize).run()


class _Problem(C.Structure):
    """pkv_decode_problem of include/pagedkv.h."""
    _fields_ = [("out", C.c_void_p), ("q", C.c_void_p), ("k_pool", C.c_void_p),
                ("v_pool", C.c_void_p), ("block_tables", C.c_void_p),
                ("context_lens", C.c_void_p), ("k_new", C.c_void_p), ("v_new", C.c_void_p),
                ("slot_mapping", C.c_void_p), ("num_seqs", C.c_int), ("num_blocks", C.c_int),
                ("max_blocks_per_seq", C.c_int)]


class _Plan(C.Structure):
    _fields_ = [("opaque", C.c_uint64 * 16)]


class DecodeBatch:
    """Independent decode problems (each with its own pools, tables, lengths,
    queries and outputs, optionally a fused append) planned once and run in
    one launch.  `problems` is a list of dicts with the keys out, q, k_pool,
    v_pool, block_tables, context_lens and optionally k_new, v_new,
    slot_mapping (as paged_attn_decode_append).  The plan stays valid while
    those tensors keep their storage and every context stays within
    max_context_len; run() reads their current contents."""

    def __init__(self, problems, scale: float, max_context_len: int, split_tokens: int = 0,
                 stream: Optional[torch.cuda.Stream] = None):
        if not problems:
            raise ValueError("no problems")
        ref = problems[0]
        _, H, D = ref["q"].shape
        _, B, Hk, _ = ref["k_pool"].shape
        kv_dt, out_dt = ref["k_pool"].dtype, ref["out"].dtype
        arr = (_Problem * len(problems))()
        for i, pr in enumerate(problems):
            for name in ("out", "q", "k_pool", "v_pool", "block_tables", "context_lens"):
                _need_cuda(name, pr[name])
            q, kp = pr["q"], pr["k_pool"]
            S = q.shape[0]
            if (tuple(q.shape[1:]) != (H, D) or tuple(kp.shape[1:]) != (B, Hk, D)
                    or pr["v_pool"].shape != kp.shape or tuple(pr["out"].shape) != (S, H, D)
                    or q.dtype != kv_dt or kp.dtype != kv_dt or pr["v_pool"].dtype != kv_dt
                    or pr["out"].dtype != out_dt
                    or pr["block_tables"].dtype != torch.int32
                    or pr["context_lens"].dtype != torch.int32
                    or pr["block_tables"].shape[0] != S or pr["context_lens"].shape != (S,)):
                raise ValueError(f"problem {i}: inconsistent shapes or dtypes")
            sm = pr.get("slot_mapping")
            if sm is not None:
                for name in ("k_new", "v_new", "slot_mapping"):
                    _need_cuda(name, pr[name])
                if (sm.dtype != torch.int64 or sm.shape != (S,)
                        or tuple(pr["k_new"].shape) != (S, Hk, D)
                        or pr["v_new"].shape != pr["k_new"].shape
                        or pr["k_new"].dtype != kv_dt or pr["v_new"].dtype != kv_dt):
                    raise ValueError(f"problem {i}: inconsistent append rows")
            arr[i] = _Problem(pr["out"].data_ptr(), q.data_ptr(), kp.data_ptr(),
                              pr["v_pool"].data_ptr(), pr["block_tables"].data_ptr(),
                              pr["context_lens"].data_ptr(),
                              pr["k_new"].data_ptr() if sm is not None else None,
                              pr["v_new"].data_ptr() if sm is not None else None,
                              sm.data_ptr() if sm is not None else None, S, kp.shape[0],
                              pr["block_tables"].shape[1])
        self._problems = list(problems)      # keeps the tensors alive
        ws_bytes = int(lib().pkv_decode_batched_workspace_bytes(
            C.addressof(arr), len(problems), H, Hk, D, B, int(max_context_len),
            int(split_tokens)))
        if ws_bytes == 0:
            raise ValueError("unsupported batch (head counts, head_dim, block size)")
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=ref["q"].device)
        self._plan = _Plan()
        st = lib().pkv_decode_batched_plan(
            C.addressof(self._plan), C.addressof(arr), len(problems), _DT[out_dt], _DT[kv_dt], H,
            Hk, D, B, float(scale), int(max_context_len), int(split_tokens),
            _ptr(self.workspace), ws_bytes, _stream_ptr(stream))
        check(st, "pkv_decode_batched_plan")

    def run(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        check(lib().paged_attn_decode_batched(C.addressof(self._plan), _stream_ptr(stream)),
              "paged_attn_decode_batched")


def paged_attn_multi_query(out: torch.Tensor, q: torch.Tensor, q_start: torch.Tensor,
                           k_pool: torch.Tensor, v_pool: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           max_q_len: int, max_context_len: int,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Causal attention of each sequence's last q_len tokens (rows
    q_start[s] .. q_start[s+1]-1 of q [total_q, H, D]) over its paged context."""
    for name, t in (("out", out), ("q", q), ("q_start", q_start), ("k_pool", k_pool),
                    ("v_pool", v_pool), ("block_tables", block_tables),
                    ("context_lens", context_lens)):
        _need_cuda(name, t)
    if q_start.dtype != torch.int32 or block_tables.dtype != torch.int32 or \
            context_lens.dtype != torch.int32:
        raise ValueError("q_start, block_tables and context_lens must be int32")
    T, H, D = q.shape
    nb, B, Hk, D2 = k_pool.shape
    S = context_lens.shape[0]
    if (D2 != D or tuple(out.shape) != (T, H, D) or tuple(v_pool.shape) != tuple(k_pool.shape)
            or q.dtype != k_pool.dtype or v_pool.dtype != k_pool.dtype
            or q_start.shape != (S + 1,) or block_tables.shape[0] != S):
        raise ValueError("inconsistent shapes or dtypes")
    st = lib().paged_attn_multi_query(_ptr(out), _DT[out.dtype], _ptr(q), _ptr(q_start), T,
                                      int(max_q_len), _ptr(k_pool), _ptr(v_pool),
                                      _DT[k_pool.dtype], _ptr(block_tables), block_tables.shape[1],
                                      _ptr(context_lens), S, H, Hk, D, B, nb, float(scale),
                                      int(max_context_len), _stream_ptr(stream))
    check(st, "paged_attn_multi_query")
    return out


def kv_append(k_pool: torch.Tensor, v_pool: torch.Tensor, k_new: torch.Tensor,
              v_new: torch.Tensor, slot_mapping: torch.Tensor,
              stream: Optional[torch.cuda.Stream] = None) -> None:
    """k_pool.view(-1, Hk, D)[slot_mapping[s]] = k_new[s] (same for V);
    slot -1 skips."""
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool), ("k_new", k_new), ("v_new", v_new),
                    ("slot_mapping", slot_mapping)):
        _need_cuda(name, t)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    nb, B, Hk, D = k_pool.shape
    S = k_new.shape[0]
    if (tuple(k_new.shape) != (S, Hk, D) or k_new.shape != v_new.shape
            or v_pool.shape != k_pool.shape or slot_mapping.shape != (S,)
            or len({k_pool.dtype, v_pool.dtype, k_new.dtype, v_new.dtype}) != 1):
        raise ValueError("inconsistent shapes or dtypes")
    st = lib().kv_append(_ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new), _DT[k_pool.dtype],
                         _ptr(slot_mapping), S, Hk, D, B, nb, _stream_ptr(stream))
    check(st, "kv_append")


def swap_blocks(dst_pool: torch.Tensor, src_pool: torch.Tensor, pairs: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """dst_pool[j] = src_pool[i] for each (i, j) row of `pairs` (int64 [n, 2]).
    src_pool and pairs may live in pinned host memory."""
    _need_cuda("dst_pool", dst_pool)
    for name, t in (("src_pool", src_pool), ("pairs", pairs)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [n, 2]")
    bb = dst_pool[0].numel() * dst_pool.element_size() if dst_pool.shape[0] else 0
    if src_pool.shape[0] and src_pool[0].numel() * src_pool.element_size() != bb:
        raise ValueError("source and destination blocks differ in size")
    st = lib().swap_blocks(_ptr(dst_pool), _ptr(src_pool), bb, _ptr(pairs), pairs.shape[0],
                           src_pool.shape[0], dst_pool.shape[0], _stream_ptr(stream))
    check(st, "swap_blocks")


def swap_blocks_kv(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor,
                   src_v: torch.Tensor, pairs: torch.Tensor,
                   stream: Optional[torch.cuda.Stream] = None) -> None:
    """swap_blocks on the Key and the Value cache in one launch (same pairs)."""
    for name, t in (("dst_k", dst_k), ("dst_v", dst_v)):
        _need_cuda(name, t)
    for name, t in (("src_k", src_k), ("src_v", src_v), ("pairs", pairs)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [n, 2]")
    if dst_k.shape != dst_v.shape or src_k.shape != src_v.shape:
        raise ValueError("Key and Value pools must have the same shapes")
    bb = dst_k[0].numel() * dst_k.element_size() if dst_k.shape[0] else 0
    if src_k.shape[0] and src_k[0].numel() * src_k.element_size() != bb:
        raise ValueError("source and destination blocks differ in size")
    st = lib().swap_blocks_kv(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v), bb, _ptr(pairs),
                              pairs.shape[0], src_k.shape[0], dst_k.shape[0], _stream_ptr(stream))
    check(st, "swap_blocks_kv")


def device_errors(clear: bool = True) -> int:
    """PKV_DEVERR_* bits raised by kernels on the current device (synchronises)."""
    v = C.c_uint32(0)
    check(lib().pkv_device_errors(C.byref(v), 1 if clear else 0), "pkv_device_errors")
    return int(v.value)


class BlockManager:
    """Host block manager of the library (lowest free id first, reference
    counts).  Wraps pkv_block_manager_*; arrays are CPU int32/int64 tensors."""

    def __init__(self, num_blocks: int, block_size: int, free_ids=None):
        L = lib()
        if free_ids is None:
            h = L.pkv_block_manager_create(num_blocks, block_size)
        else:
            ids = torch.as_tensor(list(free_ids), dtype=torch.int32).contiguous()
            h = L.pkv_block_manager_create_with_free(num_blocks, block_size, _ptr(ids), ids.numel())
        if not h:
            raise ValueError("pkv_block_manager_create failed (bad arguments)")
        self._h = C.c_void_p(h)
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib._lib is not None:
            _lib._lib.pkv_block_manager_destroy(h)
            self._h = None

    def allocate(self) -> int:
        b = C.c_int32(-1)
        check(lib().pkv_block_allocate(self._h, C.byref(b)), "pkv_block_allocate")
        return int(b.value)

    def free(self, block_id: int) -> None:
        check(lib().pkv_block_free(self._h, block_id), "pkv_block_free")

    def add_reference(self, block_id: int) -> None:
        check(lib().pkv_block_add_reference(self._h, block_id), "pkv_block_add_reference")

    def free_count(self) -> int:
        return int(lib().pkv_block_free_count(self._h))

    def ref_count(self, block_id: int) -> int:
        return int(lib().pkv_block_ref_count(self._h, block_id))

    def free_ids(self) -> list:
        n = lib().pkv_block_free_ids(self._h, None, 0)
        buf = torch.empty(max(n, 1), dtype=torch.int32)
        lib().pkv_block_free_ids(self._h, _ptr(buf), n)
        return buf[:n].tolist()

    def append_slots(self, block_tables: torch.Tensor, context_lens: torch.Tensor,
                     slot_mapping: torch.Tensor) -> int:
        """In place on CPU tensors (int32 tables/lengths, int64 slots).
        Returns the status (PKV_OK or PKV_ERR_NO_BLOCKS) instead of raising,
        since a failed sequence is reported through slot -1."""
        for t, dt in ((block_tables, torch.int32), (context_lens, torch.int32),
                      (slot_mapping, torch.int64)):
            if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != dt:
                raise ValueError("append_slots takes contiguous CPU int32/int32/int64 tensors")
        S = context_lens.shape[0]
        st = lib().pkv_append_slots(self._h, _ptr(block_tables), block_tables.shape[1],
                                    _ptr(context_lens), S, _ptr(slot_mapping))
        if st not in (_lib.PKV_OK, _lib.PKV_ERR_NO_BLOCKS):
            check(st, "pkv_append_slots")
        return int(st)

    def append_slots_cow(self, block_tables: torch.Tensor, context_lens: torch.Tensor,
                         slot_mapping: torch.Tensor):
        """append_slots with copy-on-write of shared pages.  Returns (status,
        copy_pairs int64 [n, 2]) -- copy those pairs before kv_append."""
        for t, dt in ((block_tables, torch.int32), (context_lens, torch.int32),
                      (slot_mapping, torch.int64)):
            if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != dt:
                raise ValueError("append_slots_cow takes contiguous CPU int32/int32/int64 tensors")
        S = context_lens.shape[0]
        pairs = torch.empty(max(S, 1), 2, dtype=torch.int64)
        n = C.c_int(0)
        st = lib().pkv_append_slots_cow(self._h, _ptr(block_tables), block_tables.shape[1],
                                        _ptr(context_lens), S, _ptr(slot_mapping), _ptr(pairs),
                                        C.byref(n))
        if st not in (_lib.PKV_OK, _lib.PKV_ERR_NO_BLOCKS):
            check(st, "pkv_append_slots_cow")
        return int(st), pairs[:n.value].clone()


def _defrag(self, block_tables: torch.Tensor):
    """Plan a compaction (used blocks to [0, n)); updates this manager and the
    CPU int32 tables in place and returns the int64 [n, 2] pairs to copy."""
    if block_tables.device.type != "cpu" or block_tables.dtype != torch.int32 or \
            not block_tables.is_contiguous():
        raise ValueError("defrag takes a contiguous CPU int32 block table")
    cap = self.num_blocks
    pairs = torch.empty(max(cap, 1), 2, dtype=torch.int64)
    n = C.c_int(0)
    check(lib().pkv_defrag(self._h, _ptr(block_tables), block_tables.shape[1],
                           block_tables.shape[0], _ptr(pairs), cap, C.byref(n)), "pkv_defrag")
    return pairs[:n.value].clone()


BlockManager.defrag = _defrag


class DeviceBlockManager:
    """The block manager's state in device memory, driven by kernels (same
    semantics as BlockManager).  ref_counts / free_ids / state are CUDA int32
    tensors owned by this object."""

    def __init__(self, ref_counts, block_size: int, device="cuda"):
        rc = torch.as_tensor(ref_counts, dtype=torch.int32).to(device).contiguous()
        self.num_blocks = rc.numel()
        self.block_size = block_size
        self.ref_counts = rc
        self.free_ids = torch.empty(max(1, self.num_blocks), dtype=torch.int32, device=device)
        self.state = torch.zeros(4, dtype=torch.int32, device=device)
        check(lib().pkv_device_rebuild_free_list(_ptr(self.ref_counts), _ptr(self.free_ids),
                                                 _ptr(self.state), self.num_blocks,
                                                 _stream_ptr(None)),
              "pkv_device_rebuild_free_list")

    def append_slots(self, block_tables: torch.Tensor, context_lens: torch.Tensor,
                     slot_mapping: torch.Tensor, stream=None) -> None:
        for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                        ("slot_mapping", slot_mapping)):
            _need_cuda(name, t)
        if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or \
                slot_mapping.dtype != torch.int64:
            raise ValueError("int32 tables and lengths, int64 slots")
        check(lib().pkv_device_append_slots(_ptr(self.ref_counts), _ptr(self.free_ids),
                                            _ptr(self.state), _ptr(block_tables),
                                            block_tables.shape[1], _ptr(context_lens),
                                            context_lens.shape[0], self.block_size,
                                            self.num_blocks, _ptr(slot_mapping),
                                            _stream_ptr(stream)),
              "pkv_device_append_slots")

    def free(self, block_ids: torch.Tensor, stream=None) -> None:
        _need_cuda("block_ids", block_ids)
        ids = block_ids.to(torch.int32).contiguous()
        check(lib().pkv_device_free_blocks(_ptr(self.ref_counts), _ptr(self.free_ids),
                                           _ptr(self.state), _ptr(ids), ids.numel(),
                                           self.num_blocks, _stream_ptr(stream)),
              "pkv_device_free_blocks")

    def free_list(self) -> list:
        st = self.state.tolist()
        return self.free_ids[st[0]:st[0] + st[1]].tolist()

    def failed_last_append(self) -> int:
        return int(self.state[2].item())
