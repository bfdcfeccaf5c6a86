"""The fp64 decode oracle run on many host cores at once.

TEST INFRASTRUCTURE ONLY: used by tests/ (whole-output parity at the full
workload sizes) and by the benchmark's CPU-baseline and reference legs,
never by the product path.

The arithmetic is the oracle's own (oracle.decode_two_pass, the plain
two-pass definition); this module only cuts the work into independent
pieces and runs them on a thread pool.  The C oracle is called through
ctypes, which releases the interpreter lock for the call, so the pieces run
in parallel.  A piece is one sequence with all its heads, or, when there
are too few sequences to keep every thread busy, one sequence with a
contiguous range of kv heads (and their query heads): that piece's blocks
and heads are first gathered into a compact pool of its own.  Attention
rows of different sequences and heads do not interact, so the result is the
one a single call over everything gives, element for element.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

from . import oracle as orc


def host_threads() -> int:
    """Threads to use: the cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def _pieces(lens, seq_ids, Hk, threads):
    """(sequence, kv head begin, kv head end) pieces, longest first: whole
    sequences when there are at least 4 per thread, else sequences cut into
    kv-head ranges (a divisor of Hk) until there are."""
    seqs = sorted(seq_ids, key=lambda s: -int(lens[s]))
    cut = 1
    while len(seqs) * cut < 4 * threads and cut < Hk:
        cut *= 2
    while Hk % cut:
        cut //= 2
    step = Hk // cut
    return [(s, h0, h0 + step) for s in seqs for h0 in range(0, Hk, step)], cut


def decode_two_pass(q, k_pool, v_pool, block_tables, context_lens, scale, seq_ids=None,
                    threads=None):
    """oracle.decode_two_pass over the selected sequences (all by default),
    computed on `threads` host threads.  Returns float64 [n_sel, H, D]."""
    q = q.contiguous()
    S, H, D = q.shape
    nb, B, Hk, _ = k_pool.shape
    G = H // Hk
    lens = context_lens.to(torch.int64).tolist()
    sel = list(range(S)) if seq_ids is None else [int(s) for s in seq_ids]
    pos = {s: i for i, s in enumerate(sel)}
    threads = threads or host_threads()
    pieces, cut = _pieces(lens, sel, Hk, threads)
    out = np.zeros((len(sel), H, D), dtype=np.float64)
    bt = block_tables.to(torch.int32)

    def run(piece):
        s, h0, h1 = piece
        n = lens[s]
        if cut == 1 or n <= 0:
            whole = orc.decode_two_pass(q, k_pool, v_pool, bt, context_lens, scale,
                                        seq_ids=[s])[0]
            out[pos[s], h0 * G:h1 * G] = whole[h0 * G:h1 * G]
            return
        nblk = (n + B - 1) // B
        ids = bt[s, :nblk].to(torch.int64)
        # a compact pool holding only this sequence's blocks and kv heads
        k_sub = k_pool[ids][:, :, h0:h1].contiguous()
        v_sub = v_pool[ids][:, :, h0:h1].contiguous()
        q_sub = q[s:s + 1, h0 * G:h1 * G].contiguous()
        bt_sub = torch.arange(max(nblk, 1), dtype=torch.int32).view(1, -1)
        l_sub = torch.tensor([n], dtype=torch.int32)
        out[pos[s], h0 * G:h1 * G] = orc.decode_two_pass(q_sub, k_sub, v_sub, bt_sub, l_sub,
                                                         scale)[0]

    if threads == 1:
        for p in pieces:
            run(p)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            for f in [ex.submit(run, p) for p in pieces]:
                f.result()
    return out
