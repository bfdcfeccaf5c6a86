"""Seeded synthetic inputs for paged-KV decode: context lengths, block tables,
query, K/V pools, new-token rows and block-copy pairs.

This module holds input construction only -- no attention, append or copy
arithmetic -- so that both the CUDA path and the CPU oracle can be fed the
same bytes.  Everything is drawn on the host from ``numpy.random.default_rng``
(PCG64, identical on x86_64 and aarch64) and rounded to the storage dtype by
torch's round-to-nearest-even conversion.

The five workloads (sizes as the decode problem states them):
  1 tiny          4 seqs, 8 q = 8 kv heads, d=64, B=16, lens U[1,200],
                  pool 64 blocks, fp16 in / fp32 out, + 8 block-copy pairs
  2 llama7b_mha   64 seqs, 32 heads MHA, d=128, B=16, lens U[512,4096],
                  pool = needed blocks + 10 %, bf16
  3 gqa_prefix    128 seqs, 32 q / 8 kv heads, d=128, B=16, lens
                  log-uniform [128,32768]; groups of 8 seqs share their first
                  64 physical blocks (whole blocks only), bf16
  4 long_context  16 seqs x 32768 tokens, 32 heads MHA, d=128, B=32, bf16,
                  pool = exactly the needed blocks, randomly permuted (8 GiB)
  5 continuous    256 seqs, Pareto(1.5) lens clipped [16,16384], 32 q / 8 kv
                  heads, d=128, B=16, bf16; one appended token per seq, then
                  1024 device-to-device and 1024 host-to-device block pairs
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

CONFIGS = {
    1: dict(name="tiny", S=4, H=8, Hk=8, D=64, B=16, dtype=torch.float16, out_dtype=torch.float32,
            lens=("uniform", 1, 200), pool_blocks=64, swap_pairs=8),
    2: dict(name="llama7b_mha", S=64, H=32, Hk=32, D=128, B=16, dtype=torch.bfloat16,
            out_dtype=torch.bfloat16, lens=("uniform", 512, 4096), pool_extra=0.10),
    3: dict(name="gqa_prefix", S=128, H=32, Hk=8, D=128, B=16, dtype=torch.bfloat16,
            out_dtype=torch.bfloat16, lens=("loguniform", 128, 32768), pool_extra=0.10,
            share_group=8, share_blocks=64),
    4: dict(name="long_context", S=16, H=32, Hk=32, D=128, B=32, dtype=torch.bfloat16,
            out_dtype=torch.bfloat16, lens=("const", 32768), pool_extra=0.0),
    5: dict(name="continuous", S=256, H=32, Hk=8, D=128, B=16, dtype=torch.bfloat16,
            out_dtype=torch.bfloat16, lens=("pareto", 1.5, 16, 16384), pool_extra=0.10,
            append=True, d2d_pairs=1024, h2d_pairs=1024, host_pool_blocks=2048),
}


@dataclasses.dataclass
class DecodeCase:
    """One synthetic decode problem.  All tensors are on the host (CPU)."""
    name: str
    S: int
    H: int
    Hk: int
    D: int
    B: int
    dtype: torch.dtype
    out_dtype: torch.dtype
    scale: float
    context_lens: torch.Tensor          # int32 [S] (lengths before any append)
    block_tables: torch.Tensor          # int32 [S, max_blocks]; unused entries -1
    q: torch.Tensor                     # [S, H, D]
    k_pool: torch.Tensor                # [num_blocks, B, Hk, D]
    v_pool: torch.Tensor                # [num_blocks, B, Hk, D]
    free_ids: list                      # sorted ids no table references
    seed: int
    # block-copy companions (optional)
    swap_src_k: Optional[torch.Tensor] = None   # source pools of the copy
    swap_src_v: Optional[torch.Tensor] = None
    swap_dst_k: Optional[torch.Tensor] = None   # destination pools of the copy
    swap_dst_v: Optional[torch.Tensor] = None
    swap_pairs: Optional[torch.Tensor] = None   # int64 [n, 2] (src, dst)
    # append companions (optional)
    k_new: Optional[torch.Tensor] = None        # [S, Hk, D]
    v_new: Optional[torch.Tensor] = None
    # continuous-batching extras (optional)
    d2d_pairs: Optional[torch.Tensor] = None    # int64 [n, 2] within the pools
    h2d_pairs: Optional[torch.Tensor] = None    # int64 [n, 2] host pool -> pools
    host_k_pool: Optional[torch.Tensor] = None  # [host_blocks, B, Hk, D]
    host_v_pool: Optional[torch.Tensor] = None

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.S else 0

    def row_bytes(self) -> int:
        """Bytes of one token's K (or V) row for all kv heads."""
        return self.Hk * self.D * torch.tensor([], dtype=self.dtype).element_size()


def _lens(rng, spec, S):
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=S)
    if kind == "loguniform":
        lo, hi = math.log(spec[1]), math.log(spec[2])
        return np.floor(np.exp(rng.uniform(lo, hi, size=S))).astype(np.int64).clip(spec[1], spec[2])
    if kind == "const":
        return np.full(S, spec[1], dtype=np.int64)
    if kind == "pareto":
        a, xm, hi = spec[1], spec[2], spec[3]
        # classical Pareto(a, x_m): x_m * (1 + Lomax(a)); numpy's pareto() is Lomax.
        return np.floor(xm * (1.0 + rng.pareto(a, size=S))).astype(np.int64).clip(xm, hi)
    raise ValueError(kind)


_CHUNK = 1 << 24


def _normal(rng, shape, dtype, chunk_elems=_CHUNK):
    """N(0,1) drawn as float32 and rounded to `dtype`.  Large tensors are
    drawn in fixed-size chunks, each from its own generator spawned from one
    seed taken from `rng`, so the values do not depend on how many threads
    draw them."""
    import concurrent.futures as cf
    import os
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype)
    children = np.random.SeedSequence(int(rng.integers(0, 2 ** 63))).spawn(
        (n + chunk_elems - 1) // chunk_elems)

    def fill(k):
        a = k * chunk_elems
        b = min(n, a + chunk_elems)
        g = np.random.Generator(np.random.PCG64(children[k]))
        out[a:b] = torch.from_numpy(g.standard_normal(b - a, dtype=np.float32)).to(dtype)

    if len(children) <= 1:
        for k in range(len(children)):
            fill(k)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(len(children))))
    return out.view(*shape)


def make_case(config: int, seed: Optional[int] = None, S: Optional[int] = None,
              lens: Optional[tuple] = None, poison: bool = False,
              lens_override: Optional[list] = None, **over) -> DecodeCase:
    """Build workload `config` (1..5).  `S`, `lens` (a length spec such as
    ("uniform", lo, hi)), `lens_override` (explicit list) and any key of the
    config dict override the stated sizes for small parity cases.

    poison=True fills every pool row that no sequence's context covers
    (unused blocks and the tail rows of each last page) with NaN, so that a
    read outside the context shows up in the output."""
    spec = dict(CONFIGS[config])
    spec.update(over)
    if S is not None:
        spec["S"] = S
    if lens is not None:
        spec["lens"] = lens
    seed = (config - 1) if seed is None else seed
    rng = np.random.default_rng(seed)
    S, H, Hk, D, B = spec["S"], spec["H"], spec["Hk"], spec["D"], spec["B"]
    dtype = spec["dtype"]

    if lens_override is not None:
        n = np.asarray(lens_override, dtype=np.int64)
        S = spec["S"] = len(n)
    else:
        n = _lens(rng, spec["lens"], S)
    nblk = (n + B - 1) // B
    appending = bool(spec.get("append"))
    # one more table column where an append may open a new page
    need_cols = (n + 1 + B - 1) // B if appending else nblk
    max_blocks = int(max(1, need_cols.max() if S else 1))

    # --- physical placement -------------------------------------------------
    group = spec.get("share_group")
    shared_per_group = spec.get("share_blocks", 0)
    n_groups = (S + group - 1) // group if group else 0
    shared_needed = n_groups * shared_per_group
    private = []
    for s in range(S):
        sh = min(shared_per_group, int(n[s]) // B) if group else 0
        private.append(int(nblk[s]) - sh)
    used = shared_needed + sum(private)
    if "pool_blocks" in spec:
        num_blocks = int(spec["pool_blocks"])
    else:
        num_blocks = int(math.ceil(used * (1.0 + spec.get("pool_extra", 0.0))))
    reserve = 0
    if appending:
        reserve = S + spec.get("d2d_pairs", 0) + spec.get("h2d_pairs", 0)
        num_blocks = max(num_blocks, used) + reserve
    if num_blocks < used:
        raise ValueError("pool too small for the drawn lengths")
    perm = rng.permutation(num_blocks)
    cursor = 0
    shared_ids = []
    for g in range(n_groups):
        shared_ids.append(perm[cursor:cursor + shared_per_group])
        cursor += shared_per_group
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    for s in range(S):
        sh = min(shared_per_group, int(n[s]) // B) if group else 0
        if sh:
            bt[s, :sh] = shared_ids[s // group][:sh]
        k = private[s]
        bt[s, sh:sh + k] = perm[cursor:cursor + k]
        cursor += k
    referenced = set(int(x) for x in bt[bt >= 0].ravel())
    free_ids = sorted(set(range(num_blocks)) - referenced)

    scale = 1.0 / math.sqrt(D)
    q = _normal(rng, (S, H, D), dtype)
    k_pool = _normal(rng, (num_blocks, B, Hk, D), dtype)
    v_pool = _normal(rng, (num_blocks, B, Hk, D), dtype)

    case = DecodeCase(name=spec["name"], S=S, H=H, Hk=Hk, D=D, B=B, dtype=dtype,
                      out_dtype=spec["out_dtype"], scale=scale,
                      context_lens=torch.from_numpy(n.astype(np.int32)),
                      block_tables=torch.from_numpy(bt), q=q, k_pool=k_pool, v_pool=v_pool,
                      free_ids=free_ids, seed=seed)

    if spec.get("swap_pairs"):
        m = int(spec["swap_pairs"])
        src = rng.choice(num_blocks, size=m, replace=False)
        dst = rng.choice(num_blocks, size=m, replace=False)
        case.swap_pairs = torch.from_numpy(np.stack([src, dst], axis=1).astype(np.int64))
        case.swap_src_k, case.swap_src_v = k_pool, v_pool
        case.swap_dst_k = _normal(rng, (num_blocks, B, Hk, D), dtype)
        case.swap_dst_v = _normal(rng, (num_blocks, B, Hk, D), dtype)

    if appending:
        case.k_new = _normal(rng, (S, Hk, D), dtype)
        case.v_new = _normal(rng, (S, Hk, D), dtype)
        # Copy targets come from the free ids above the lowest S, which the
        # append step may hand out (lowest id first).
        pickable = np.array(free_ids[S:], dtype=np.int64)
        n_d2d, n_h2d = int(spec.get("d2d_pairs", 0)), int(spec.get("h2d_pairs", 0))
        targets = rng.choice(pickable, size=n_d2d + n_h2d, replace=False)
        d2d_dst, h2d_dst = targets[:n_d2d], targets[n_d2d:]
        others = np.setdiff1d(np.arange(num_blocks), targets)
        d2d_src = rng.choice(others, size=n_d2d, replace=False)
        case.d2d_pairs = torch.from_numpy(np.stack([d2d_src, d2d_dst], axis=1).astype(np.int64))
        hb = int(spec.get("host_pool_blocks", n_h2d))
        case.host_k_pool = _normal(rng, (hb, B, Hk, D), dtype)
        case.host_v_pool = _normal(rng, (hb, B, Hk, D), dtype)
        h2d_src = rng.choice(hb, size=n_h2d, replace=False)
        case.h2d_pairs = torch.from_numpy(np.stack([h2d_src, h2d_dst], axis=1).astype(np.int64))

    if poison:
        poison_pools(case)
    return case


def covered_rows(case: DecodeCase, lens=None, tables=None) -> np.ndarray:
    """Boolean [num_blocks, B]: True where some sequence's context (of the
    given lengths and tables, default the case's) covers that pool row."""
    lens = case.context_lens.numpy() if lens is None else np.asarray(lens)
    cov = np.zeros((case.num_blocks, case.B), dtype=bool)
    bt = case.block_tables.numpy() if tables is None else np.asarray(tables)
    for s in range(case.S):
        ns = int(lens[s])
        for j in range((ns + case.B - 1) // case.B):
            rows = min(case.B, ns - j * case.B)
            cov[bt[s, j], :rows] = True
    return cov


def poison_pools(case: DecodeCase) -> None:
    """Fill every uncovered pool row with NaN (in place)."""
    cov = torch.from_numpy(covered_rows(case))
    nan = torch.tensor(float("nan"), dtype=case.dtype)
    for pool in (case.k_pool, case.v_pool):
        pool[~cov] = nan


def kv_bytes(case: DecodeCase, lens=None, tables=None) -> tuple[int, int]:
    """(logical, unique) K+V bytes a decode step reads: logical counts every
    sequence's context rows; unique counts each physical pool row once."""
    lens = case.context_lens.numpy() if lens is None else np.asarray(lens)
    row = case.row_bytes()
    logical = int(np.sum(lens)) * row * 2
    unique = int(covered_rows(case, lens, tables).sum()) * row * 2
    return logical, unique


def sampled_seqs(case: DecodeCase, k: int, seed: int = 1234) -> list:
    """k sequence indices for sampled full-size checks: the longest, the
    shortest and k-2 drawn at random (sorted)."""
    lens = case.context_lens.numpy()
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    rng = np.random.default_rng(seed)
    rest = [s for s in rng.permutation(case.S).tolist() if s not in pick]
    pick.update(rest[:max(0, k - len(pick))])
    return sorted(pick)[:max(k, 2)]


def multi_query_inputs(case: DecodeCase, q_len_spec, seed: int = 77):
    """Query rows for attention of several new tokens per sequence (a prefill
    chunk, or tokens to verify): sequence s gets q_len_s <= context_lens[s]
    rows, its last q_len_s tokens.  q_len_spec is ("const", n) or ("uniform",
    lo, hi) (clipped to the context).  Returns (q [total, H, D] in the case's
    dtype, q_start int32 [S + 1])."""
    rng = np.random.default_rng(seed)
    lens = case.context_lens.numpy()
    if q_len_spec[0] == "const":
        ql = np.full(case.S, q_len_spec[1], dtype=np.int64)
    else:
        ql = rng.integers(q_len_spec[1], q_len_spec[2] + 1, size=case.S)
    ql = np.minimum(ql, lens)
    q_start = np.zeros(case.S + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(ql)
    q = _normal(rng, (int(q_start[-1]), case.H, case.D), case.dtype)
    return q, torch.from_numpy(q_start)
