"""The tensor-core decode run as resident CTAs that each take an exactly equal
share of the pages (paged_decode_mma_stream_kernel plus its boundary merge,
selected by the decode_stream tuning knob or automatically for short
contexts): through the C ABI, against the fp64 oracle, with empty contexts,
ragged tails, runs cut by many share boundaries, fewer pages than CTAs,
fused appends and bad block ids.  Its results depend only on the inputs and
the device (the shares follow from the lengths and the grid), so repeated
calls agree bit for bit."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle import parallel
from paged_kv_decode_26_gb300 import workloads as wl
from tests.parity import assert_attention_close, run_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_26_gb300 import build
    build.build()
    import paged_kv_decode_26_gb300 as pkv
    pkv.device_errors(clear=True)
    yield pkv


def _bits(t):
    return t.contiguous().view(torch.int16) if t.element_size() == 2 else \
        t.contiguous().view(torch.int32)


def _abs_v(case, seq_ids=None):
    """sum_t w_t |V_t| per output element, on demand (the tensor-core
    consumer's hi + lo weight rounding term of the parity bound)."""
    return lambda: parallel.decode_two_pass(case.q, case.k_pool, case.v_pool.abs(),
                                            case.block_tables, case.context_lens, case.scale,
                                            seq_ids=seq_ids)


def _stream(tuning, case, dev=None, **kw):
    """Two stream decodes of the case (automatic split): asserted bit-equal,
    the first returned."""
    dev = dev if dev is not None else to_device(case)
    tuning(decode_stream=1)
    a = run_decode(case, split_tokens=0, dev=dev, **kw)
    b = run_decode(case, split_tokens=0, dev=dev, **kw)
    torch.cuda.synchronize()
    assert torch.equal(_bits(a), _bits(b)), "stream decode not repeatable"
    return a


def _check(lib, case, got, what):
    ref = parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale)
    assert_attention_close(got, ref, case.out_dtype, what, abs_weighted=_abs_v(case),
                           kv_dtype=case.dtype)
    assert lib.device_errors(clear=True) == 0


@pytest.mark.parametrize("D,B", [(128, 16), (64, 16), (128, 32), (64, 32)])
@pytest.mark.parametrize("H,Hk", [(32, 8), (16, 2), (8, 1)])
def test_stream_matches_oracle(lib, tuning, D, B, H, Hk):
    lens = [0, 1, 15, 16, 17, 33, 0, 70, 2 * B * 8 + 3, 5, 300, 1, 64, 0, 129, 31]
    case = wl.make_case(5, lens_override=lens, H=H, Hk=Hk, D=D, B=B, d2d_pairs=0,
                        h2d_pairs=0, host_pool_blocks=1, poison=True, seed=D + B + H)
    out = _stream(tuning, case)
    _check(lib, case, out, f"D={D} B={B} {H}/{Hk}")


@pytest.mark.parametrize("lens,H,Hk", [
    ([20000], 32, 8),                 # one long context cut by every share boundary
    ([9000, 3, 0, 4100, 17], 8, 1),   # long runs next to short ones
    ([16, 1, 31], 32, 8),             # fewer pages than CTAs: one share per page
    ([0, 0, 0], 32, 4),               # no pages at all: zero rows only
    ([1] * 700, 16, 2),               # one-page runs only: no workspace, no merge
])
def test_stream_share_boundaries(lib, tuning, lens, H, Hk):
    case = wl.make_case(5, lens_override=lens, H=H, Hk=Hk, D=128, B=16, d2d_pairs=0,
                        h2d_pairs=0, host_pool_blocks=1, poison=True, seed=len(lens) + H)
    out = _stream(tuning, case)
    if max(lens) <= 16:
        assert lib.decode_workspace_bytes(case.S, H, Hk, 128, 16, max(lens), 0) == 0
    _check(lib, case, out, f"lens {lens[:5]}")


def test_stream_ignores_workspace_contents(lib, tuning):
    """The partial states are written before the merge reads them: a
    workspace full of NaN gives the same bits as a zeroed one."""
    import paged_kv_decode_26_gb300 as pkv
    case = wl.make_case(5, S=64, lens=("pareto", 1.5, 16, 4000), d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, seed=5)
    dev = to_device(case)
    tuning(decode_stream=1)
    mcl = int(case.context_lens.max())
    outs = []
    for fill in (0.0, float("nan")):
        ws = pkv.alloc_decode_workspace(dev["q"], dev["k_pool"], mcl)
        assert ws is not None and ws.numel() > 0
        ws.view(torch.float32)[: ws.numel() // 4].fill_(fill)
        out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_decode(out, dev["q"], dev["k_pool"], dev["v_pool"], dev["block_tables"],
                              dev["context_lens"], case.scale, mcl, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(_bits(outs[0]), _bits(outs[1]))
    _check(lib, case, outs[0], "workspace contents")


def test_explicit_split_runs_the_per_unit_kernel(lib, tuning):
    """An explicit split length is honoured: the per-unit kernel runs (its
    bits with the knob on and off agree)."""
    case = wl.make_case(5, S=40, lens=("pareto", 1.5, 16, 3000), d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, seed=9)
    dev = to_device(case)
    outs = []
    for mode in (0, 1):
        tuning(decode_stream=mode)
        outs.append(run_decode(case, split_tokens=64, dev=dev))
    torch.cuda.synchronize()
    assert torch.equal(_bits(outs[0]), _bits(outs[1]))
    _check(lib, case, outs[1], "explicit split")


@pytest.mark.parametrize("config,extra", [
    (5, dict(S=300, lens=("pareto", 1.5, 16, 2000))),
    (5, dict(S=64, lens=("pareto", 1.5, 16, 16384))),
    (3, dict(S=40, lens=("loguniform", 1, 3000), share_blocks=8)),
    (5, dict(S=2048, lens=("uniform", 0, 40))),          # the most sequences the kernel takes
    (5, dict(S=2049, lens=("uniform", 0, 40))),          # one more: the per-unit kernel runs
])
def test_stream_workload_mixes(lib, tuning, config, extra):
    if config == 5:
        extra = dict(extra, d2d_pairs=0, h2d_pairs=0, host_pool_blocks=1)
    case = wl.make_case(config, poison=True, seed=17, **extra)
    out = _stream(tuning, case)
    if case.S > 2048:
        tuning(decode_stream=0)
        ref_bits = run_decode(case, split_tokens=0)
        assert torch.equal(_bits(out), _bits(ref_bits))
    _check(lib, case, out, f"config {config} S={case.S}")


@pytest.mark.parametrize("H,Hk,D", [(32, 8, 128), (8, 8, 128), (8, 8, 64)])
def test_stream_fused_append_equals_two_calls(lib, tuning, H, Hk, D):
    """paged_attn_decode_append on the stream kernel gives the pools and the
    output of kv_append followed by paged_attn_decode, bit for bit; a slot
    of -1 appends nothing, a slot past the pool is skipped and flagged, an
    empty context still receives its row.  Groups of 4 and MHA (the
    tensor-core consumer forced; a three-page ring at head_dim 128)."""
    import paged_kv_decode_26_gb300 as pkv
    tuning(decode_mma=1, decode_stream=1)
    case = wl.make_case(5, S=24, lens=("pareto", 1.5, 16, 600), H=H, Hk=Hk, D=D, d2d_pairs=0,
                        h2d_pairs=0, host_pool_blocks=1, poison=True, seed=31 + H + D)
    S = case.S
    bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    bt = case.block_tables.clone()
    need = int(((case.context_lens + 1 + case.B - 1) // case.B).max())
    if need > bt.shape[1]:
        bt = torch.cat([bt, torch.full((S, need - bt.shape[1]), -1, dtype=torch.int32)], 1)
    lens = case.context_lens.clone()
    slots = torch.empty(S, dtype=torch.int64)
    assert bm.append_slots(bt, lens, slots) == 0
    slots_used = slots.clone()
    slots_used[0] = -1
    lens[0] -= 1
    slots_used[2] = case.num_blocks * case.B + 5
    lens[2] -= 1
    lens[4] = 0                     # an empty context whose slot still gets the row
    d = {k: v.cuda() for k, v in (("q", case.q), ("bt", bt), ("lens", lens),
                                  ("slots", slots_used), ("kn", case.k_new), ("vn", case.v_new))}
    results = []
    for fused in (False, True):
        kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
        out = torch.zeros(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        if fused:
            pkv.paged_attn_decode_append(out, d["q"], kp, vp, d["bt"], d["lens"], case.scale,
                                         int(lens.max()), d["kn"], d["vn"], d["slots"])
        else:
            pkv.kv_append(kp, vp, d["kn"], d["vn"], d["slots"])
            pkv.paged_attn_decode(out, d["q"], kp, vp, d["bt"], d["lens"], case.scale,
                                  int(lens.max()))
        torch.cuda.synchronize()
        assert pkv.device_errors(clear=True) & 0x4
        results.append((out.cpu(), kp.cpu(), vp.cpu()))
    (o1, k1, v1), (o2, k2, v2) = results
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    assert torch.equal(_bits(o1), _bits(o2))
    ref = orc.decode_two_pass(case.q, k1, v1, bt, lens, case.scale)
    assert_attention_close(o2, ref, case.out_dtype, "fused append", kv_dtype=case.dtype,
                           abs_weighted=lambda: orc.decode_two_pass(case.q, k1, v1.abs(), bt,
                                                                    lens, case.scale))


def test_stream_bad_block_ids_are_flagged(lib, tuning):
    case = wl.make_case(3, S=6, lens=("const", 100), H=16, Hk=4, seed=3)
    bt = case.block_tables.clone()
    bt[1, 2] = case.num_blocks + 5
    bt[1, 3] = -7
    dev = to_device(case)
    keep = [0, 2, 3, 4, 5]
    ref = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale, seq_ids=keep)
    for mode in (0, 1):
        tuning(decode_stream=mode)
        out = run_decode(case, split_tokens=0, dev=dev, tables=bt.cuda())
        torch.cuda.synchronize()
        assert lib.device_errors(clear=True) & 0x1
        assert torch.isfinite(out.float()).all()
        assert_attention_close(out[keep], ref, case.out_dtype, f"mode {mode}",
                               kv_dtype=case.dtype, abs_weighted=_abs_v(case, keep))


def test_stream_workspace_does_not_grow_with_sequences(lib, tuning):
    """Two partial-state slots per CTA: the workspace of a short-context
    decode does not grow with the number of sequences and fits the no-alloc
    entry point's built-in scratch, whose output then equals the workspace
    call's bit for bit."""
    import ctypes as C
    tuning(decode_stream=1)
    ws = {S: lib.decode_workspace_bytes(S, 32, 8, 128, 16, 200, 0) for S in (64, 512, 2048)}
    # (64 sequences take two kv heads per CTA and more CTAs per SM: other slots)
    assert 0 < ws[2048] == ws[512] <= ws[64] <= 16 << 20   # PKV_NOALLOC_SCRATCH_BYTES
    case = wl.make_case(5, S=2048, lens=("uniform", 1, 200), d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, seed=77)
    dev = to_device(case)
    mcl = int(case.context_lens.max())
    ref = run_decode(case, split_tokens=0, dev=dev)
    out = torch.empty_like(ref)
    ptr = lambda t: C.c_void_p(t.data_ptr())
    dt = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
    st = lib.lib().paged_attn_decode_noalloc(
        ptr(out), dt[out.dtype], ptr(dev["q"]), ptr(dev["k_pool"]), ptr(dev["v_pool"]),
        dt[case.dtype], ptr(dev["block_tables"]), case.max_blocks_per_seq,
        ptr(dev["context_lens"]), case.S, case.H, case.Hk, case.D, case.B, case.num_blocks,
        case.scale, mcl, 0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref))
    _check(lib, case, out, "2048 short contexts")


def test_stream_repeated_calls_on_one_workspace(lib, tuning):
    """The same decode 300 times on one workspace (its partial states and
    boundary records overwritten every call) gives the first call's bits
    every time."""
    import paged_kv_decode_26_gb300 as pkv
    tuning(decode_stream=1)
    case = wl.make_case(5, S=48, lens=("pareto", 1.5, 16, 3000), d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, seed=13)
    dev = to_device(case)
    mcl = int(case.context_lens.max())
    ws = pkv.alloc_decode_workspace(dev["q"], dev["k_pool"], mcl)
    first = None
    outs = []
    for i in range(300):
        out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_decode(out, dev["q"], dev["k_pool"], dev["v_pool"], dev["block_tables"],
                              dev["context_lens"], case.scale, mcl, workspace=ws)
        if i == 0:
            first = out
        elif i % 50 == 0 or i == 299:
            outs.append(out)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(_bits(o), _bits(first))
    _check(lib, case, first, "300 calls")


def test_stream_calls_on_two_streams(lib, tuning):
    """Two stream decodes in flight at once (two CUDA streams, own
    workspaces, each with its boundary merge as a dependent launch): each
    equals its own single-stream result."""
    import paged_kv_decode_26_gb300 as pkv
    tuning(decode_stream=1)
    cases = [wl.make_case(5, S=S, lens=("pareto", 1.5, 16, 2500), d2d_pairs=0, h2d_pairs=0,
                          host_pool_blocks=1, seed=seed) for S, seed in ((96, 21), (64, 22))]
    devs = [to_device(c) for c in cases]
    alone = [run_decode(c, split_tokens=0, dev=d) for c, d in zip(cases, devs)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    wss = []
    for c, d in zip(cases, devs):
        mcl = int(c.context_lens.max())
        wss.append(pkv.alloc_decode_workspace(d["q"], d["k_pool"], mcl))
        outs.append(torch.empty(c.S, c.H, c.D, dtype=c.out_dtype, device="cuda"))
    torch.cuda.synchronize()
    for rep in range(20):
        for c, d, st, o, ws in zip(cases, devs, streams, outs, wss):
            with torch.cuda.stream(st):
                pkv.paged_attn_decode(o, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                                      d["context_lens"], c.scale, int(c.context_lens.max()),
                                      workspace=ws)
    torch.cuda.synchronize()
    for a, o in zip(alone, outs):
        assert torch.equal(_bits(a), _bits(o))
    assert lib.device_errors(clear=True) == 0


@pytest.mark.parametrize("dtype,out_dtype", [(torch.float16, torch.float32),
                                             (torch.float16, torch.float16),
                                             (torch.bfloat16, torch.float32)])
@pytest.mark.parametrize("D", [64, 128])
def test_stream_dtypes(lib, tuning, dtype, out_dtype, D):
    """fp16 and bf16 K/V with fp16, bf16 and fp32 outputs, including
    contexts whose last block is at most half full (half-block loads)."""
    lens = [1, 7, 8, 9, 16, 17, 24, 25, 40, 300, 0, 129]
    case = wl.make_case(5, lens_override=lens, D=D, dtype=dtype, out_dtype=out_dtype,
                        d2d_pairs=0, h2d_pairs=0, host_pool_blocks=1, poison=True, seed=D + 3)
    out = _stream(tuning, case)
    _check(lib, case, out, f"{dtype} -> {out_dtype}, D={D}")


def test_stream_group_of_two_forced(lib, tuning):
    """Groups of 2 take the tensor-core consumer only when forced
    (decode_mma=1); the streaming decode then handles them too."""
    lens = [0, 5, 16, 17, 33, 300, 1000, 9, 64]
    case = wl.make_case(5, lens_override=lens, H=16, Hk=8, d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, poison=True, seed=2)
    tuning(decode_mma=1)
    out = _stream(tuning, case)
    _check(lib, case, out, "groups of 2, forced tensor-core consumer")


@pytest.mark.parametrize("D", [64, 128])
def test_stream_one_head_per_kv_head_forced(lib, tuning, D):
    """One query head per kv head (MHA) on the tensor-core consumer (forced):
    the streaming decode and the per-unit kernel, against the oracle."""
    lens = [0, 5, 16, 17, 33, 300, 1000, 9, 64, 1, 2049, 128]
    case = wl.make_case(5, lens_override=lens, H=8, Hk=8, D=D, d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, poison=True, seed=11 + D)
    tuning(decode_mma=1)
    out = _stream(tuning, case)
    _check(lib, case, out, f"MHA D={D}, streaming tensor-core decode")
    tuning(decode_stream=0)
    for split in (0, 64):
        got = run_decode(case, split_tokens=split)
        _check(lib, case, got, f"MHA D={D}, per-unit tensor-core decode, split {split}")


@pytest.mark.parametrize("H,Hk,lens,D,B", [
    (8, 8, ("pareto", 1.5, 16, 16384), 128, 16),    # MHA, a long tail
    (8, 8, ("pareto", 1.5, 16, 16384), 64, 32),     # ... head_dim 64, 32-token blocks
    (16, 8, ("uniform", 1, 600), 128, 16),          # groups of 2
    (16, 4, ("pareto", 1.2, 16, 20000), 128, 16),   # groups of 4 past 4096 tokens
])
def test_many_sequences_stream_automatically(lib, tuning, H, Hk, lens, D, B):
    """From 256 sequences the automatic choice is the streaming decode for
    any group size and context length: its output equals the forced
    streaming tensor-core decode bit for bit and the oracle's within the
    tolerance."""
    case = wl.make_case(5, S=300, lens=lens, H=H, Hk=Hk, D=D, B=B, d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, poison=True, seed=H + Hk + D)
    dev = to_device(case)
    auto = run_decode(case, split_tokens=0, dev=dev)
    tuning(decode_mma=1, decode_stream=1)
    forced = run_decode(case, split_tokens=0, dev=dev)
    torch.cuda.synchronize()
    assert torch.equal(_bits(auto), _bits(forced))
    _check(lib, case, auto, f"{H}/{Hk} heads, 300 sequences, {lens}")
