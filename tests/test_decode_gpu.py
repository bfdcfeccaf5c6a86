"""Parity of the CUDA decode path (through the C ABI) with the fp64 oracle on
the five workloads: small cases compared element by element, the full-size
workloads compared on every output element in the benchmark's launch
configuration (the oracle threaded over the host cores), plus edge cases
and the kernels' own index checks."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
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


def _oracle(case, seq_ids=None, lens=None, tables=None, k=None, v=None):
    return orc.decode_two_pass(case.q, case.k_pool if k is None else k,
                               case.v_pool if v is None else v,
                               case.block_tables if tables is None else tables,
                               case.context_lens if lens is None else lens, case.scale,
                               seq_ids=seq_ids)


def _abs_v(case, **kw):
    """sum_t w_t |V_t| per output element (the oracle's attention with |V|),
    on demand: the tensor-core consumer's hi + lo weight rounding term of
    the parity bound."""
    return lambda: _oracle(case, **dict(kw, v=kw.get("v", case.v_pool).abs()))


def _no_device_errors(pkv):
    assert pkv.device_errors(clear=True) == 0


# ----------------------------------------------------------- small cases

SMALL = {
    1: dict(),                                                    # the tiny workload itself
    2: dict(S=6, lens=("uniform", 1, 700)),
    3: dict(S=16, lens=("loguniform", 1, 2000), share_blocks=8),
    4: dict(S=2, lens=("const", 3000)),
    5: dict(S=24, lens=("pareto", 1.5, 16, 600), d2d_pairs=8, h2d_pairs=8, host_pool_blocks=16),
}


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("split", [0, 16, 64, 512])
def test_small_case_matches_oracle(lib, config, split):
    case = wl.make_case(config, poison=True, **SMALL[config])
    if split % case.B:
        pytest.skip("split must be a multiple of the block size")
    got = run_decode(case, split_tokens=split)
    ref = _oracle(case)
    assert_attention_close(got, ref, case.out_dtype, f"config {config} split {split}",
                           abs_weighted=_abs_v(case), kv_dtype=case.dtype)
    _no_device_errors(lib)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("dtype,out_dtype", [(torch.bfloat16, torch.bfloat16),
                                             (torch.float16, torch.float16),
                                             (torch.float16, torch.float32),
                                             (torch.bfloat16, torch.float32)])
def test_shape_matrix(lib, D, B, H, Hk, dtype, out_dtype):
    case = wl.make_case(2, S=3, lens=("uniform", 1, 300), H=H, Hk=Hk, D=D, B=B, dtype=dtype,
                        out_dtype=out_dtype, poison=True, seed=D + B + H + Hk)
    for split in (0, 4 * B):
        got = run_decode(case, split_tokens=split)
        assert_attention_close(got, _oracle(case), out_dtype, f"{D} {B} {H}/{Hk} split {split}",
                               abs_weighted=_abs_v(case), kv_dtype=dtype)
    _no_device_errors(lib)


@pytest.mark.parametrize("knobs", [
    {"decode_wpt": 2},
    {"decode_wpt": 2, "decode_stages": 4},
    {"decode_wpt": 4, "decode_hpc": 2},
    {"decode_hpc": 1, "decode_stages": 6},
    {"decode_hpc": 2, "decode_stages": 2},
    {"decode_qpw": 2},
    {"decode_qpw": 1, "decode_hpc": 2},
    {"decode_mma": 0},
    {"decode_mma": 1, "decode_hpc": 2, "decode_stages": 4},
], ids=lambda e: ",".join(f"{k[7:]}={v}" for k, v in e.items()))
@pytest.mark.parametrize("config", [1, 2, 3, 4])
def test_launch_configurations(lib, tuning, config, knobs):
    """Every tuning choice of the launch (kv heads per CTA, ring depth, warps
    taking turns on pages, query heads per warp) computes the same result."""
    tuning(**knobs)
    case = wl.make_case(config, poison=True, **SMALL[config])
    for split in (0, 2 * case.B * 4):
        try:
            got = run_decode(case, split_tokens=split)
        except lib.PagedKVError as e:
            # a combination whose ring does not fit in shared memory is refused
            assert e.status == 2 and "shared memory" in str(e)
            pytest.skip(f"{knobs} does not fit: {e}")
        assert_attention_close(got, _oracle(case), case.out_dtype, f"{knobs} split {split}",
                               abs_weighted=_abs_v(case), kv_dtype=case.dtype)
    _no_device_errors(lib)


@pytest.mark.parametrize("mma", ["0", "1"])
@pytest.mark.parametrize("D,B", [(64, 16), (128, 16), (64, 32), (128, 32)])
@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("dtype,out_dtype", [(torch.bfloat16, torch.bfloat16),
                                             (torch.float16, torch.float32)])
def test_grouped_heads_both_paths(lib, tuning, mma, D, B, H, Hk, dtype, out_dtype):
    """One query head per kv head and groups of 2, 4 and 8 on the CUDA-core
    and the tensor-core consumer, ragged tails and NaN padding included."""
    tuning(decode_mma=mma)
    case = wl.make_case(3, S=4, lens=("uniform", 1, 400), H=H, Hk=Hk, D=D, B=B, dtype=dtype,
                        out_dtype=out_dtype, share_blocks=2, poison=True, seed=H + D + B)
    for split in (0, 2 * B):
        got = run_decode(case, split_tokens=split)
        assert_attention_close(got, _oracle(case), out_dtype, f"mma={mma} split {split}",
                               abs_weighted=_abs_v(case), kv_dtype=dtype)
    _no_device_errors(lib)


@pytest.mark.parametrize("S,H,Hk,B,max_ctx,expect", [
    (64, 32, 32, 16, 4097, 512),     # llama7b_mha: 4K contexts keep 512-token splits
    (128, 32, 8, 16, 32075, 1024),   # gqa_prefix: 32K contexts, 256 (seq, head-group) units
    (16, 32, 32, 32, 32769, 1024),   # long_context (2 kv heads per CTA: 256 units)
    (255, 32, 8, 16, 16385, 512),    # 510 units, more than 2 x SMs: 512 tokens
    (256, 32, 8, 16, 1235, 1248),    # continuous as generated (longest 1235): streaming decode,
                                     # no split (the whole page-rounded context)
    (128, 32, 8, 16, 4096, 4096),    # GQA up to 4K tokens: streaming decode
    (128, 32, 8, 16, 4104, 512),     # GQA past 4K tokens: one CTA per unit
    (1, 32, 8, 16, 4096, 512),       # one sequence: one CTA per unit
    (128, 32, 8, 16, 8192, 1024),    # 8K tokens, few units: longer splits
    (256, 32, 8, 16, 20000, 20000),  # 256 sequences or more: streaming at any length
    (256, 32, 32, 16, 4096, 4096),   # ... and for MHA
    (255, 32, 32, 16, 4096, 512),    # one fewer MHA sequence: one CTA per unit
    (4, 8, 8, 16, 201, 208),         # tiny: one split of the whole (page-rounded) context
    (4096, 32, 8, 16, 4096, 4096),   # many units: no split at all
])
def test_automatic_split_length(lib, S, H, Hk, B, max_ctx, expect):
    """The automatic split length: 512 tokens; 1024 when the longest
    context is 8K tokens or more and there are at most 2 x SMs (sequence,
    head-group) units; the whole context when the units fill the GPU 16
    times over (sizes for GB300's 152 SMs); the whole context for the
    streaming tensor-core decode (groups of 4 or 8, 2 to 2048 sequences,
    longest context at most 4096; any group and length from 256 to 2048
    sequences), which cuts the work at its CTAs' shares instead of splits."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("unit thresholds are stated for 152 SMs")
    assert lib.decode_split_tokens(S, H, Hk, 128, B, max_ctx) == expect


def test_split_invariance(lib):
    case = wl.make_case(2, S=4, lens=("uniform", 900, 2000), out_dtype=torch.float32)
    outs = [run_decode(case, split_tokens=s) for s in (16, 48, 256, 1024, 2048)]
    for o in outs[1:]:
        assert torch.allclose(o, outs[0], rtol=1e-5, atol=2e-6)
    _no_device_errors(lib)


def test_physical_placement_invariance(lib):
    case = wl.make_case(3, S=8, lens=("uniform", 1, 400), share_blocks=4)
    a = run_decode(case, split_tokens=64)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(case.num_blocks))
    k2 = torch.empty_like(case.k_pool)
    v2 = torch.empty_like(case.v_pool)
    k2[perm] = case.k_pool
    v2[perm] = case.v_pool
    bt = case.block_tables.clone()
    bt[bt >= 0] = perm.to(torch.int32)[bt[bt >= 0].long()]
    case.k_pool, case.v_pool, case.block_tables = k2, v2, bt
    b = run_decode(case, split_tokens=64)
    assert torch.equal(a, b)
    _no_device_errors(lib)


# ----------------------------------------------------------- edge cases

def test_context_one_and_empty(lib):
    case = wl.make_case(2, lens_override=[1, 0, 1, 17, 0, 16], H=8, Hk=8)
    got = run_decode(case, split_tokens=16)
    G = case.H // case.Hk
    for s in (0, 2):
        p = int(case.block_tables[s, 0])
        for h in range(case.H):
            assert torch.equal(got[s, h].cpu(), case.v_pool[p, 0, h // G])
    assert torch.count_nonzero(got[1]) == 0 and torch.count_nonzero(got[4]) == 0
    assert_attention_close(got, _oracle(case), case.out_dtype)
    _no_device_errors(lib)


def test_all_empty_batch(lib):
    case = wl.make_case(2, lens_override=[0, 0, 0], H=4, Hk=4)
    got = run_decode(case, max_context_len=0)
    assert torch.count_nonzero(got) == 0
    _no_device_errors(lib)


def test_dominant_key(lib):
    case = wl.make_case(2, lens_override=[300], H=2, Hk=2, out_dtype=torch.float32)
    t = 123
    p = int(case.block_tables[0, t // case.B])
    case.q[:] = 1.0
    case.k_pool[p, t % case.B] = 8.0  # score 8*128/sqrt(128) ~ 90 above the rest
    got = run_decode(case, split_tokens=64)
    for h in range(case.H):
        assert torch.allclose(got[0, h].cpu(), case.v_pool[p, t % case.B, h].float(), atol=1e-6)
    _no_device_errors(lib)


def test_maximum_split_and_max_pages(lib):
    """One split covering 4096 pages (the per-split maximum) and a context
    of 32768 tokens at block size 16."""
    case = wl.make_case(2, lens_override=[32768, 5], H=2, Hk=2)
    got = run_decode(case, split_tokens=4096 * 16)
    assert_attention_close(got, _oracle(case), case.out_dtype)
    _no_device_errors(lib)


def test_workspace_too_small_is_rejected(lib):
    case = wl.make_case(2, S=2, lens=("const", 2000), H=4, Hk=4)
    dev = to_device(case)
    out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.PagedKVError, match="WORKSPACE"):
        lib.paged_attn_decode(out, dev["q"], dev["k_pool"], dev["v_pool"], dev["block_tables"],
                              dev["context_lens"], case.scale, 2000, split_tokens=64,
                              workspace=ws)


def test_out_of_range_block_id_is_flagged_not_read(lib):
    case = wl.make_case(2, S=3, lens=("const", 100), H=4, Hk=4)
    bt = case.block_tables.clone()
    bt[1, 2] = case.num_blocks + 5
    bt[1, 3] = -7
    dev = to_device(case)
    got = run_decode(case, split_tokens=32, dev=dev, tables=bt.cuda())
    assert lib.device_errors(clear=True) & 0x1
    ref = _oracle(case, seq_ids=[0, 2])
    assert_attention_close(got[[0, 2]], ref, case.out_dtype)
    assert torch.isfinite(got[1].float()).all()


def test_context_beyond_bound_is_flagged(lib):
    case = wl.make_case(2, S=2, lens=("const", 100), H=4, Hk=4)
    got = run_decode(case, split_tokens=32, max_context_len=40)
    assert lib.device_errors(clear=True) & 0x2
    assert torch.isfinite(got.float()).all()


# ------------------------------------------------- full sizes (every element)

@pytest.mark.parametrize("config", [2, 3, 4, 5])
def test_full_size_step_whole_output(lib, config):
    """The benchmark's step at the stated full size of the workload: one new
    token per sequence (slots from the host manager, checked against the
    oracle's allocator), then the append and the decode in one
    paged_attn_decode_append call with the automatic launch shape.  Both
    pools are compared bit for bit with the oracle's appends, and every
    output element with the fp64 oracle on the appended state."""
    import paged_kv_decode_26_gb300 as pkv
    from oracle import parallel
    from oracle.block_manager import append_slots
    case = wl.make_case(config, **({"pool_extra": 0.01} if config == 4 else {}))
    S = case.S
    if case.k_new is None:
        case.k_new = wl._normal(np.random.default_rng(case.seed + 7), (S, case.Hk, case.D),
                                case.dtype)
        case.v_new = wl._normal(np.random.default_rng(case.seed + 8), (S, case.Hk, case.D),
                                case.dtype)
    bt = case.block_tables.clone()
    need = int(((case.context_lens + 1 + case.B - 1) // case.B).max())
    if need > bt.shape[1]:
        bt = torch.cat([bt, torch.full((S, need - bt.shape[1]), -1, dtype=torch.int32)], 1)
    lens = case.context_lens.clone()
    slots = torch.empty(S, dtype=torch.int64)
    bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    assert bm.append_slots(bt, lens, slots) == 0
    tables = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    o_tables, o_lens, o_slots, _ = append_slots(tables, case.context_lens.tolist(), case.B,
                                                case.free_ids, case.num_blocks)
    assert slots.tolist() == o_slots and lens.tolist() == o_lens
    for s in range(S):
        assert bt[s][bt[s] >= 0].tolist() == o_tables[s]

    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    out = torch.empty(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    pkv.paged_attn_decode_append(out, case.q.cuda(), dk, dv, bt.cuda(), lens.cuda(), case.scale,
                                 int(lens.max()), case.k_new.cuda(), case.v_new.cuda(),
                                 slots.cuda())
    torch.cuda.synchronize()
    _no_device_errors(lib)

    k, v = case.k_pool, case.v_pool          # the oracle appends in place
    orc.kv_append(k, v, case.k_new, case.v_new, slots)
    assert torch.equal(dk.cpu().view(torch.int16), k.view(torch.int16))
    assert torch.equal(dv.cpu().view(torch.int16), v.view(torch.int16))
    del dk, dv
    ref = parallel.decode_two_pass(case.q, k, v, bt, lens, case.scale)
    st = assert_attention_close(
        out, ref, case.out_dtype, f"config {config}", kv_dtype=case.dtype,
        abs_weighted=lambda: parallel.decode_two_pass(case.q, k, v.abs(), bt, lens, case.scale))
    print(f"config {config}: {st['n']} elements, max |err| {st['max_abs']:.3g}, "
          f"mean {st['mean_abs']:.3g}, rounding-limited {st['rounding_limited']}")


# ------------------------------------------------- fused append + decode

@pytest.mark.parametrize("config,split", [(1, 0), (2, 0), (2, 64), (3, 0), (5, 0)])
def test_decode_append_equals_two_calls(lib, config, split):
    """paged_attn_decode_append gives the pools and the output of
    kv_append followed by paged_attn_decode, bit for bit (the same kernels'
    arithmetic), including sequences whose slot is -1 and a slot outside the
    pool (skipped and flagged by both)."""
    import paged_kv_decode_26_gb300 as pkv
    extra = {"d2d_pairs": 8, "h2d_pairs": 8, "host_pool_blocks": 16} if config == 5 else {}
    case = wl.make_case(config, S=8 if config != 1 else None, poison=True, seed=config + 40,
                        **extra)
    S = case.S
    bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    bt = case.block_tables.clone()
    need = int(((case.context_lens + 1 + case.B - 1) // case.B).max())
    if need > bt.shape[1]:
        bt = torch.cat([bt, torch.full((S, need - bt.shape[1]), -1, dtype=torch.int32)], 1)
    lens = case.context_lens.clone()
    slots = torch.empty(S, dtype=torch.int64)
    bm.append_slots(bt, lens, slots)
    gen = torch.Generator().manual_seed(config)
    k_new = torch.randn(S, case.Hk, case.D, generator=gen).to(case.dtype)
    v_new = torch.randn(S, case.Hk, case.D, generator=gen).to(case.dtype)
    slots_used = slots.clone()
    # sequence 0 appends nothing; sequence 2's slot lies outside the pool
    # (skipped and flagged): neither context counts the new token
    for s_, bad in ((0, -1), (2, case.num_blocks * case.B + 5)):
        if s_ < S and int(slots[s_]) >= 0:
            slots_used[s_] = bad
            lens[s_] -= 1
    max_ctx = int(lens.max())
    d = {k: v.cuda() for k, v in (("q", case.q), ("bt", bt), ("lens", lens),
                                  ("slots", slots_used), ("kn", k_new), ("vn", v_new))}
    results = []
    for fused in (False, True):
        kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
        out = torch.zeros(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        if fused:
            pkv.paged_attn_decode_append(out, d["q"], kp, vp, d["bt"], d["lens"], case.scale,
                                         max_ctx, d["kn"], d["vn"], d["slots"],
                                         split_tokens=split)
        else:
            pkv.kv_append(kp, vp, d["kn"], d["vn"], d["slots"])
            pkv.paged_attn_decode(out, d["q"], kp, vp, d["bt"], d["lens"], case.scale, max_ctx,
                                  split_tokens=split)
        torch.cuda.synchronize()
        flags = pkv.device_errors(clear=True)
        assert (flags & 0x4) == (0x4 if S > 2 and int(slots[2]) >= 0 else 0)
        results.append((out.cpu(), kp.cpu(), vp.cpu()))
    (o1, k1, v1), (o2, k2, v2) = results
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    iv = torch.int16 if o1.element_size() == 2 else torch.int32
    assert torch.equal(o1.view(iv), o2.view(iv))
    # and against the oracle for the appended state
    ref = _oracle(case, lens=lens, tables=bt, k=k1, v=v1)
    assert_attention_close(o2, ref, case.out_dtype, f"config {config}", kv_dtype=case.dtype,
                           abs_weighted=_abs_v(case, lens=lens, tables=bt, k=k1, v=v1))


@pytest.mark.parametrize("config", [1, 2, 5])
def test_host_step_equals_device_call(lib, config):
    """paged_attn_decode_append_host (the step's inputs packed in one pinned
    host buffer, copied in, appended and decoded, the output copied back,
    the stream synchronised) leaves the same pools and output, bit for bit,
    as copying the inputs and calling paged_attn_decode_append; out_host
    holds the device output."""
    import paged_kv_decode_26_gb300 as pkv
    extra = {"d2d_pairs": 0, "h2d_pairs": 0, "host_pool_blocks": 1} if config == 5 else {}
    case = wl.make_case(config, S=8 if config != 1 else None, poison=True, seed=config + 60,
                        **extra)
    S = case.S
    bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    bt = case.block_tables.clone()
    need = int(((case.context_lens + 1 + case.B - 1) // case.B).max())
    if need > bt.shape[1]:
        bt = torch.cat([bt, torch.full((S, need - bt.shape[1]), -1, dtype=torch.int32)], 1)
    lens = case.context_lens.clone()
    slots = torch.empty(S, dtype=torch.int64)
    bm.append_slots(bt, lens, slots)
    gen = torch.Generator().manual_seed(config + 60)
    k_new = torch.randn(S, case.Hk, case.D, generator=gen).to(case.dtype)
    v_new = torch.randn(S, case.Hk, case.D, generator=gen).to(case.dtype)
    max_ctx = int(lens.max())
    # one pinned staging buffer and its device twin, each input at a 256-byte offset
    parts = [case.q, k_new, v_new, bt, lens, slots]
    offs, o = [], 0
    for t in parts:
        offs.append(o)
        o += (t.numel() * t.element_size() + 255) // 256 * 256
    hbuf = torch.zeros(o, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(o, dtype=torch.uint8, device="cuda")

    def views(buf):
        return [buf[a:a + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for a, t in zip(offs, parts)]
    for hv, t in zip(views(hbuf), parts):
        hv.copy_(t)
    q_d, kn_d, vn_d, bt_d, lens_d, slots_d = views(dbuf)
    results = []
    for host_call in (False, True):
        kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
        out = torch.zeros(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
        out_h = torch.full((S, case.H, case.D), float("nan"), dtype=case.out_dtype).pin_memory()
        dbuf.zero_()
        torch.cuda.synchronize()
        if host_call:
            pkv.paged_attn_decode_append_host([(hbuf, dbuf)], out_h, out, q_d, kp, vp, bt_d,
                                              lens_d, case.scale, max_ctx, kn_d, vn_d, slots_d)
        else:
            dbuf.copy_(hbuf)
            pkv.paged_attn_decode_append(out, q_d, kp, vp, bt_d, lens_d, case.scale, max_ctx,
                                         kn_d, vn_d, slots_d)
            out_h.copy_(out)
        torch.cuda.synchronize()
        assert pkv.device_errors(clear=True) == 0
        results.append((out_h.clone(), kp.cpu(), vp.cpu(), out.cpu()))
    (o1, k1, v1, _), (o2, k2, v2, dev2) = results
    iv = torch.int16 if o1.element_size() == 2 else torch.int32
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    assert torch.equal(o1.view(iv), o2.view(iv))
    assert torch.equal(o2.view(iv), dev2.view(iv))
    ref = _oracle(case, lens=lens, tables=bt, k=k2, v=v2)
    assert_attention_close(o2, ref, case.out_dtype, f"host step, config {config}",
                           kv_dtype=case.dtype,
                           abs_weighted=_abs_v(case, lens=lens, tables=bt, k=k2, v=v2))
    # prepared once, run twice with new host inputs in between: each run
    # equals the device call on the inputs of that run (the append writes
    # the same rows again, so the pools stay as they are)
    kp, vp = k2.cuda(), v2.cuda()
    out = torch.zeros(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    out_h = torch.empty(S, case.H, case.D, dtype=case.out_dtype).pin_memory()
    step = pkv.HostStep([(hbuf, dbuf)], out_h, out, q_d, kp, vp, bt_d, lens_d, case.scale,
                        max_ctx, kn_d, vn_d, slots_d)
    q_h = views(hbuf)[0]
    for sign in (1.0, -1.0):
        q_h.copy_(case.q * sign)
        got = step.run().clone()
        ref_out = torch.zeros_like(out)
        pkv.paged_attn_decode(ref_out, q_d, kp, vp, bt_d, lens_d, case.scale, max_ctx)
        torch.cuda.synchronize()
        assert torch.equal(got.view(iv), ref_out.cpu().view(iv)), f"HostStep run, sign {sign}"
    assert pkv.device_errors(clear=True) == 0
