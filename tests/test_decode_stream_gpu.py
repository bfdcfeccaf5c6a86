"""The tensor-core decode run as resident CTAs streaming the work units
(paged_decode_mma_stream_kernel, selected by the decode_stream tuning knob):
through the C ABI, against the fp64 oracle and bit for bit against the
one-CTA-per-unit kernel (the arithmetic of a unit is the same), with empty
contexts, ragged tails, splits, fused appends and bad block ids."""
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


def _abs_v(case):
    """sum_t w_t |V_t| per output element, on demand (the tensor-core
    consumer's hi + lo weight rounding term of the parity bound)."""
    return lambda: parallel.decode_two_pass(case.q, case.k_pool, case.v_pool.abs(),
                                            case.block_tables, case.context_lens, case.scale)


def _both(lib, tuning, case, split, **kw):
    """(per-unit kernel output, stream kernel output) of one decode with the
    same split length (split 0: the stream kernel's automatic one, which the
    per-unit kernel is then given explicitly), plus the stream kernel's
    output with the automatic split."""
    dev = to_device(case)
    tuning(decode_stream=1)
    auto = None
    if split == 0:
        auto = run_decode(case, split_tokens=0, dev=dev, **kw)
        split = lib.decode_split_tokens(case.S, case.H, case.Hk, case.D, case.B,
                                        int(case.context_lens.max()))
    b = run_decode(case, split_tokens=split, dev=dev, **kw)
    tuning(decode_stream=0)
    a = run_decode(case, split_tokens=split, dev=dev, **kw)
    torch.cuda.synchronize()
    if auto is not None:
        assert torch.equal(_bits(auto), _bits(b))
    return a, b


@pytest.mark.parametrize("D,B", [(128, 16), (64, 16), (128, 32), (64, 32)])
@pytest.mark.parametrize("H,Hk", [(32, 8), (16, 2), (8, 1)])
@pytest.mark.parametrize("split", [0, 2, 8])
def test_stream_equals_per_unit_kernel(lib, tuning, D, B, H, Hk, split):
    lens = [0, 1, 15, 16, 17, 33, 0, 70, 2 * B * 8 + 3, 5, 300, 1, 64, 0, 129, 31]
    case = wl.make_case(5, lens_override=lens, H=H, Hk=Hk, D=D, B=B, d2d_pairs=0,
                        h2d_pairs=0, host_pool_blocks=1, poison=True, seed=D + B + H + split)
    a, b = _both(lib, tuning, case, split * B)
    assert torch.equal(_bits(a), _bits(b))
    ref = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    assert_attention_close(b, ref, case.out_dtype, f"D={D} B={B} {H}/{Hk} split {split}",
                           abs_weighted=_abs_v(case), kv_dtype=case.dtype)
    assert lib.device_errors(clear=True) == 0


@pytest.mark.parametrize("config,extra", [
    (5, dict(S=300, lens=("pareto", 1.5, 16, 2000))),
    (3, dict(S=40, lens=("loguniform", 1, 3000), share_blocks=8)),
    (5, dict(S=2048, lens=("uniform", 0, 40))),          # the most sequences the kernel takes
    (5, dict(S=2049, lens=("uniform", 0, 40))),          # one more: the per-unit kernel runs
])
def test_stream_workload_mixes(lib, tuning, config, extra):
    if config == 5:
        extra = dict(extra, d2d_pairs=0, h2d_pairs=0, host_pool_blocks=1)
    case = wl.make_case(config, poison=True, seed=17, **extra)
    for split in (0, 64):
        a, b = _both(lib, tuning, case, split)
        assert torch.equal(_bits(a), _bits(b))
    ref = parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale)
    assert_attention_close(b, ref, case.out_dtype, f"config {config}",
                           abs_weighted=_abs_v(case), kv_dtype=case.dtype)
    assert lib.device_errors(clear=True) == 0


def test_stream_fused_append_equals_two_calls(lib, tuning):
    """paged_attn_decode_append on the stream kernel gives the pools and the
    output of kv_append followed by paged_attn_decode, bit for bit; a slot
    of -1 appends nothing, a slot past the pool is skipped and flagged, an
    empty context still receives its row."""
    import paged_kv_decode_26_gb300 as pkv
    tuning(decode_stream=1)
    case = wl.make_case(5, S=24, lens=("pareto", 1.5, 16, 600), d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, poison=True, seed=31)
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
    outs = []
    for mode in (0, 1):
        tuning(decode_stream=mode)
        outs.append(run_decode(case, split_tokens=32, dev=dev, tables=bt.cuda()))
        torch.cuda.synchronize()
        assert lib.device_errors(clear=True) & 0x1
    keep = [0, 2, 3, 4, 5]
    assert torch.equal(_bits(outs[0]), _bits(outs[1]))
    ref = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale, seq_ids=keep)
    assert_attention_close(outs[1][keep], ref, case.out_dtype, kv_dtype=case.dtype,
                           abs_weighted=lambda: orc.decode_two_pass(
                               case.q, case.k_pool, case.v_pool.abs(), case.block_tables,
                               case.context_lens, case.scale, seq_ids=keep))
