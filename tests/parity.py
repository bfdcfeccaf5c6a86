"""Shared parity helpers of the GPU tests: run the library on a workload case
and compare against the fp64 oracle with the stated tolerance.

Tolerance (attention output vs the fp64 oracle, N(0,1) inputs):
  * max |err| <= 4e-3 and mean |err| <= 5e-4, where an element above 4e-3
    is accepted only if it is rounding-limited: |oracle| >= 2 (where one
    half-ulp of bf16 is 7.8e-3) and |err| <= half an ulp of the output type
    at |oracle| + 1e-5; likewise the mean bound is rounding-limited where
    the correctly rounded oracle itself exceeds it (rows that see a handful
    of keys, e.g. the first tokens of a prefill from scratch, have |O| near
    |V| and a bf16 mean rounding error near 5e-4): then the bound is that
    rounded oracle's own mean error + 10 % (reported as mean_bound);
  * and, tighter, every element is within one ulp of the oracle rounded to
    the output type plus 2e-6 absolute (fp32 output: |err| <= 2e-5 +
    1e-5 |oracle|), which bounds the fp32 accumulation error of the kernel
    itself.  The absolute floor covers outputs that cancel to nearly zero,
    where a relative ulp is smaller than fp32 rounding of the summands.
    Where the caller passes the attention of |V| (sum_t w_t |V_t|, same
    weights), the one-ulp bound also admits the rounding of the softmax
    weights that the tensor-core kernels feed to the P V product as a hi +
    lo pair of 16-bit numbers: each weight keeps a relative error of at most
    2^-18 (bf16: hi rounded to 8 bits, lo to 8 bits of the remainder) or
    2^-22 (fp16), so the output may move by that times sum_t w_t |V_t|; the
    bound takes twice that (2^-17, 2^-21) to cover the fp32 rounding of the
    weights themselves.  A row attending to a few keys whose values cancel
    (output near 0, sum |w V| near 1) reaches a few 1e-6.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 4e-3
MEAN_ABS = 5e-4

_MANT = {torch.bfloat16: 7, torch.float16: 10}


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of `dtype` numbers at |x| (normal range; subnormal floor)."""
    m = _MANT[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** (-14 if dtype == torch.float16 else -126))
    return np.exp2(np.floor(np.log2(ax)) - m)


_SPLIT = {torch.bfloat16: 2.0 ** -17, torch.float16: 2.0 ** -21}


def attention_errors(got: torch.Tensor, ref: np.ndarray, out_dtype: torch.dtype,
                     abs_weighted=None, kv_dtype: torch.dtype = torch.bfloat16) -> dict:
    g = got.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "mean_abs": float(err.mean()) if err.size else 0.0,
             "n": int(err.size), "finite": bool(np.all(np.isfinite(g)))}
    over = err > MAX_ABS
    if out_dtype in _MANT:
        half = 0.5 * ulp(ref, out_dtype)
        limited = over & (np.abs(ref) >= 2.0) & (err <= half + 1e-5)
        stats["rounding_limited"] = int(limited.sum())
        stats["violations"] = int((over & ~limited).sum())
        r = torch.from_numpy(ref).to(out_dtype).to(torch.float64).numpy()
        bound = ulp(r, out_dtype) * 1.0001 + 2e-6
        beyond = np.abs(g - r) > bound
        if beyond.any() and abs_weighted is not None:
            aw = abs_weighted() if callable(abs_weighted) else abs_weighted
            beyond = np.abs(g - r) > bound + _SPLIT[kv_dtype] * np.asarray(aw)
        stats["beyond_one_ulp"] = int(beyond.sum())
        rounded_mean = float(np.abs(r - ref).mean()) if ref.size else 0.0
        stats["mean_bound"] = max(MEAN_ABS, 1.1 * rounded_mean)
        if beyond.any():
            i = np.unravel_index(np.argmax(np.abs(g - r) * beyond), g.shape)
            stats["worst"] = {"index": [int(x) for x in i], "got": float(g[i]),
                              "oracle": float(ref[i]), "oracle_rounded": float(r[i])}
    else:
        stats["rounding_limited"] = 0
        stats["violations"] = int(over.sum())
        beyond = err > 2e-5 + 1e-5 * np.abs(ref)
        if beyond.any() and abs_weighted is not None:
            aw = abs_weighted() if callable(abs_weighted) else abs_weighted
            beyond = err > 2e-5 + 1e-5 * np.abs(ref) + _SPLIT[kv_dtype] * np.asarray(aw)
        stats["beyond_one_ulp"] = int(beyond.sum())
    return stats


def assert_attention_close(got, ref, out_dtype, what="", abs_weighted=None,
                           kv_dtype=torch.bfloat16):
    """abs_weighted: sum_t w_t |V_t| per output element (an array, or a
    callable computing it on demand), see the module docstring."""
    st = attention_errors(got, ref, out_dtype, abs_weighted, kv_dtype)
    assert st["finite"], f"{what}: non-finite output"
    assert st["violations"] == 0, f"{what}: {st}"
    assert st["mean_abs"] <= st.get("mean_bound", MEAN_ABS), f"{what}: {st}"
    assert st["beyond_one_ulp"] == 0, f"{what}: {st}"
    return st


def to_device(case, device="cuda"):
    d = {}
    for name in ("q", "k_pool", "v_pool", "block_tables", "context_lens"):
        d[name] = getattr(case, name).to(device).contiguous()
    return d


def run_decode(case, split_tokens=0, dev=None, lens=None, tables=None, out_dtype=None,
               max_context_len=None):
    """Library decode on the GPU; returns the output on the device."""
    import paged_kv_decode_26_gb300 as pkv
    dev = dev if dev is not None else to_device(case)
    lens_t = dev["context_lens"] if lens is None else lens
    bt = dev["block_tables"] if tables is None else tables
    od = out_dtype or case.out_dtype
    out = torch.empty(case.S, case.H, case.D, dtype=od, device="cuda")
    mcl = int(lens_t.max().item()) if max_context_len is None else max_context_len
    pkv.paged_attn_decode(out, dev["q"], dev["k_pool"], dev["v_pool"], bt, lens_t, case.scale,
                          mcl, split_tokens=split_tokens)
    return out
