"""Shared parity helpers of the GPU tests: run the library on a workload case
and compare against the fp64 oracle with the stated tolerance.

Tolerance (attention output vs the fp64 oracle, N(0,1) inputs):
  * max |err| <= 4e-3 and mean |err| <= 5e-4, where an element above 4e-3
    is accepted only if it is rounding-limited: |oracle| >= 2 (where one
    half-ulp of bf16 is 7.8e-3) and |err| <= half an ulp of the output type
    at |oracle| + 1e-5;
  * and, tighter, every element is within one ulp of the oracle rounded to
    the output type plus 2e-6 absolute (fp32 output: |err| <= 2e-5 +
    1e-5 |oracle|), which bounds the fp32 accumulation error of the kernel
    itself.  The absolute floor covers outputs that cancel to nearly zero,
    where a relative ulp is smaller than fp32 rounding of the summands.
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


def attention_errors(got: torch.Tensor, ref: np.ndarray, out_dtype: torch.dtype) -> dict:
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
        beyond = np.abs(g - r) > ulp(r, out_dtype) * 1.0001 + 2e-6
        stats["beyond_one_ulp"] = int(beyond.sum())
        if beyond.any():
            i = np.unravel_index(np.argmax(np.abs(g - r) * beyond), g.shape)
            stats["worst"] = {"index": [int(x) for x in i], "got": float(g[i]),
                              "oracle": float(ref[i]), "oracle_rounded": float(r[i])}
    else:
        stats["rounding_limited"] = 0
        stats["violations"] = int(over.sum())
        stats["beyond_one_ulp"] = int((err > 2e-5 + 1e-5 * np.abs(ref)).sum())
    return stats


def assert_attention_close(got, ref, out_dtype, what=""):
    st = attention_errors(got, ref, out_dtype)
    assert st["finite"], f"{what}: non-finite output"
    assert st["violations"] == 0, f"{what}: {st}"
    assert st["mean_abs"] <= MEAN_ABS, f"{what}: {st}"
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
