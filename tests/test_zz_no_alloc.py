"""paged_attn_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (it keeps split partials in a scratch array built
into the library instead of a caller workspace): called through the C ABI,
its output must match paged_attn_decode's on two calls in a row, and a
problem too large for the built-in scratch must be refused before launch.

This file is named to be collected last."""
import ctypes as C

import pytest
import torch

from paged_kv_decode_26_gb300 import workloads as wl
from tests.parity import assert_attention_close, to_device

pytestmark = pytest.mark.gpu

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_26_gb300 import build
    build.build()
    import paged_kv_decode_26_gb300 as m
    m.device_errors(clear=True)
    return m


def _noalloc(pkv, case, dev, out, split, max_ctx):
    L = pkv.lib()
    ptr = lambda t: C.c_void_p(t.data_ptr())
    return L.paged_attn_decode_noalloc(
        ptr(out), _DT[out.dtype], ptr(dev["q"]), ptr(dev["k_pool"]), ptr(dev["v_pool"]),
        _DT[case.dtype], ptr(dev["block_tables"]), case.max_blocks_per_seq,
        ptr(dev["context_lens"]), case.S, case.H, case.Hk, case.D, case.B, case.num_blocks,
        case.scale, max_ctx, split, C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _reference(pkv, case, dev, split, max_ctx):
    out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    pkv.paged_attn_decode(out, dev["q"], dev["k_pool"], dev["v_pool"], dev["block_tables"],
                          dev["context_lens"], case.scale, max_ctx, split_tokens=split)
    return out


def test_matches_workspace_entry_point_on_two_calls(pkv):
    # two different problems back to back: the second call must not be
    # affected by what the first left in the shared scratch
    cases = [
        (wl.make_case(2, S=6, lens=("uniform", 300, 2500), seed=41), 128),
        (wl.make_case(3, S=10, lens=("loguniform", 1, 3000), share_blocks=4, seed=42), 0),
    ]
    for case, split in cases:
        dev = to_device(case)
        max_ctx = case.max_context_len
        assert pkv.decode_workspace_bytes(case.S, case.H, case.Hk, case.D, case.B, max_ctx,
                                          split) > 0  # the scratch is really used
        ref = _reference(pkv, case, dev, split, max_ctx)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(pkv, case, dev, out, split, max_ctx) == 0
        torch.cuda.synchronize()
        assert_attention_close(out, ref.double().cpu().numpy(), case.out_dtype, case.name)
        assert torch.equal(out, ref)
    assert pkv.device_errors(clear=True) == 0


def test_rejects_problem_larger_than_scratch(pkv):
    case = wl.make_case(2, S=4, lens=("const", 64), H=4, Hk=4, seed=43)
    dev = to_device(case)
    out = torch.zeros(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    # claim a huge maximum context at the smallest split: the partials would
    # need far more than the built-in scratch
    big = 1 << 20
    need = pkv.decode_workspace_bytes(case.S, case.H, case.Hk, case.D, case.B, big, 16)
    assert need > 16 * 1024 * 1024
    assert _noalloc(pkv, case, dev, out, 16, big) == 4  # PKV_ERR_WORKSPACE
    assert b"16 MiB" in pkv.lib().pkv_last_error_detail()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing was launched
