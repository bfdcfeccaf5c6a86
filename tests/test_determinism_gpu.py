"""Repeated calls on the same inputs give bit-identical outputs: the
kernels reduce in a fixed order (no atomics on data, split partials merged
in split order, tensor-core products issued in a fixed sequence)."""
import pytest
import torch

from paged_kv_decode_26_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_26_gb300 import build
    build.build()
    import paged_kv_decode_26_gb300 as m
    m.device_errors(clear=True)
    return m


@pytest.mark.parametrize("config,split", [(2, 0), (2, 64), (3, 0), (1, 0)])
def test_decode_repeats_bitwise(pkv, config, split):
    case = wl.make_case(config, S=8 if config != 1 else None, poison=True)
    d = {k: getattr(case, k).cuda() for k in ("q", "k_pool", "v_pool", "block_tables",
                                            "context_lens")}
    outs = []
    for _ in range(5):
        out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_decode(out, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                              d["context_lens"], case.scale, case.max_context_len,
                              split_tokens=split)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16) if o.element_size() == 2 else o.view(torch.int32),
                           outs[0].view(torch.int16) if o.element_size() == 2
                           else outs[0].view(torch.int32))
    assert pkv.device_errors(clear=True) == 0


@pytest.mark.parametrize("mode", ["0", "1"])
def test_multi_query_repeats_bitwise(pkv, tuning, mode):
    tuning(mq_tc=mode)
    case = wl.make_case(3, S=6, lens=("uniform", 200, 900), poison=True, seed=4)
    q, qs = wl.multi_query_inputs(case, ("uniform", 60, 300), seed=5)
    args = [q.cuda(), qs.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
            case.block_tables.cuda(), case.context_lens.cuda()]
    max_q = int((qs[1:] - qs[:-1]).max())
    outs = []
    for _ in range(5):
        out = torch.empty(q.shape[0], case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_multi_query(out, *args[:2], *args[2:], case.scale, max_q,
                                   case.max_context_len)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert pkv.device_errors(clear=True) == 0


def _bits(o):
    return o.view(torch.int16) if o.element_size() == 2 else o.view(torch.int32)


@pytest.mark.parametrize("config,S,split,lens", [
    (2, 40, 64, None),                                   # MHA consumer, many splits
    (3, 24, 0, None),                                    # GQA tensor-core consumer
    (4, 5, 256, [0, 1, 256, 257, 4000]),                 # block size 32, exact multiples
    (2, 70, 16, [0] * 30 + [16 * k + 3 for k in range(40)]),  # many empty contexts
])
def test_dense_order_matches_grid_order(pkv, tuning, config, S, split, lens):
    """CTAs taking units from the dense list (full splits first, short last
    splits after) or in grid order with the head group fastest compute the
    same partials as CTAs taking them by grid coordinates: the outputs agree
    bit for bit."""
    over = {"pool_extra": 0.5} if config == 4 else {}
    case = wl.make_case(config, S=S, poison=True, seed=11, lens_override=lens, **over)
    d = {k: getattr(case, k).cuda() for k in ("q", "k_pool", "v_pool", "block_tables",
                                            "context_lens")}
    outs = {}
    for mode in ("0", "1", "2"):
        tuning(decode_order=mode)
        out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_decode(out, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                              d["context_lens"], case.scale, case.max_context_len,
                              split_tokens=split)
        outs[mode] = out
    torch.cuda.synchronize()
    assert torch.equal(_bits(outs["0"]), _bits(outs["1"]))
    assert torch.equal(_bits(outs["0"]), _bits(outs["2"]))
    assert pkv.device_errors(clear=True) == 0


def test_multi_query_longest_first_matches_index_order(pkv, tuning):
    """The tcgen05 multi-query kernel's CTAs taking sequences longest context
    first compute what CTAs taking them in index order compute: bit for bit,
    with lengths spread over orders of magnitude, equal lengths (the tie
    order) and several query tiles per sequence."""
    tuning(mq_tc="1")
    lens = [900, 150, 4000, 150, 2600, 300, 4000, 700, 1200, 260]
    case = wl.make_case(3, S=len(lens), lens_override=lens, poison=True, seed=13)
    q, qs = wl.multi_query_inputs(case, ("uniform", 100, 600), seed=14)
    args = [q.cuda(), qs.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
            case.block_tables.cuda(), case.context_lens.cuda()]
    max_q = int((qs[1:] - qs[:-1]).max())
    outs = {}
    for mode in ("0", "1"):
        tuning(mq_lpt=mode)
        out = torch.empty(q.shape[0], case.H, case.D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_multi_query(out, *args[:2], *args[2:], case.scale, max_q,
                                   case.max_context_len)
        outs[mode] = out
    torch.cuda.synchronize()
    assert torch.equal(outs["0"].view(torch.int16), outs["1"].view(torch.int16))
    assert pkv.device_errors(clear=True) == 0
