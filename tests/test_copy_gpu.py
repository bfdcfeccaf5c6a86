"""Bit-exact parity of the append and block-copy kernels (through the C ABI)
with the oracle's plain loops, and the whole continuous-batching step
(allocate -> append -> decode -> copy device-to-device and host-to-device)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle.block_manager import append_slots
from paged_kv_decode_26_gb300 import workloads as wl
from tests.parity import assert_attention_close, run_decode

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
    return t.contiguous().view(torch.int16) if t.element_size() == 2 else t.contiguous().view(torch.int32)


def test_swap_tiny_workload(lib):
    case = wl.make_case(1)
    dk, dv = case.swap_dst_k.cuda(), case.swap_dst_v.cuda()
    sk, sv = case.swap_src_k.cuda(), case.swap_src_v.cuda()
    pairs = case.swap_pairs.cuda()
    lib.swap_blocks(dk, sk, pairs)
    lib.swap_blocks(dv, sv, pairs)
    rk, rv = case.swap_dst_k.clone(), case.swap_dst_v.clone()
    assert orc.swap_blocks(rk, case.swap_src_k, case.swap_pairs) == 0
    assert orc.swap_blocks(rv, case.swap_src_v, case.swap_pairs) == 0
    assert torch.equal(_bits(dk.cpu()), _bits(rk)) and torch.equal(_bits(dv.cpu()), _bits(rv))
    assert lib.device_errors() == 0


def test_swap_page_mock_example(lib, golden):
    g = golden("swap_mock_example.json")
    src = torch.randn(g["num_src_blocks"], 32, 64, 16)
    dst = torch.zeros(g["num_dst_blocks"], 32, 64, 16)
    pairs = torch.tensor([[i, j] for i, j in enumerate(g["mapping"])], dtype=torch.int64)
    d = dst.cuda()
    lib.swap_blocks(d, src.cuda(), pairs.cuda())
    assert lib.device_errors() & 0x8          # target 5 does not exist
    orc.swap_blocks(dst, src, pairs)
    assert torch.equal(d.cpu(), dst)
    assert int((d.sum(dim=[1, 2, 3]) != 0).sum()) == g["filled_blocks"]


@pytest.mark.parametrize("block_bytes", [16, 48, 4096, 32768, 40976])
def test_swap_sizes_and_untouched_bytes(lib, block_bytes):
    rng = np.random.default_rng(block_bytes)
    ns, nd, n = 37, 41, 23
    src = torch.from_numpy(rng.integers(0, 255, size=(ns, block_bytes), dtype=np.uint8))
    dst = torch.from_numpy(rng.integers(0, 255, size=(nd, block_bytes), dtype=np.uint8))
    si = rng.choice(ns, n, replace=False)
    di = rng.choice(nd, n, replace=False)
    pairs = torch.from_numpy(np.stack([si, di], 1).astype(np.int64))
    pairs[3] = torch.tensor([-1, 5])
    d = dst.cuda()
    lib.swap_blocks(d, src.cuda(), pairs.cuda())
    orc.swap_blocks(dst, src, pairs)
    assert torch.equal(d.cpu(), dst)
    assert lib.device_errors() == 0


@pytest.mark.parametrize("block_bytes,n", [(16, 300), (48, 23), (4096, 100), (40976, 23),
                                          (131072, 9)])
@pytest.mark.parametrize("knobs", [
    {},                                                    # the default (16-byte loads/stores)
    {"swap_bulk": 1},                                      # bulk copies, automatic launch shape
    {"swap_bulk": 1, "swap_chunk": 16, "swap_stages": 2, "swap_ctas": 1},  # several batches per CTA
    {"swap_bulk": 1, "swap_chunk": 4096, "swap_stages": 8, "swap_ctas": 4},
    {"swap_bulk": 1, "swap_chunk": 65536, "swap_stages": 8},  # stages cut to fit shared memory
    {"swap_bulk": 1, "swap_chunk": 24, "swap_stages": 3},  # rounded down to 16 bytes
    {"swap_bulk": 1, "swap_hint": 0, "swap_chunk": 8192},  # no L2 cache hints
], ids=lambda k: ",".join(f"{a[5:]}={b}" for a, b in k.items()) or "default")
def test_swap_bulk_launch_shapes(lib, tuning, knobs, block_bytes, n):
    """Both device-to-device copy kernels: the 16-byte load/store one and the
    bulk-copy one for every chunk size (a block in one copy, in several, with
    a shorter last chunk), ring depth and CTAs per SM, with skipped and
    out-of-range pairs, bit-exact against the oracle's loop, K and V in one
    launch and the untouched bytes kept."""
    tuning(**knobs)
    rng = np.random.default_rng(block_bytes + n)
    ns, nd = n + 9, n + 13
    src = [torch.from_numpy(rng.integers(0, 255, size=(ns, block_bytes), dtype=np.uint8))
           for _ in range(2)]
    dst = [torch.from_numpy(rng.integers(0, 255, size=(nd, block_bytes), dtype=np.uint8))
           for _ in range(2)]
    si = rng.choice(ns, n, replace=False)
    di = rng.choice(nd, n, replace=False)
    pairs = torch.from_numpy(np.stack([si, di], 1).astype(np.int64))
    pairs[min(3, n - 1)] = torch.tensor([-1, int(di[min(3, n - 1)])])
    d = [x.cuda() for x in dst]
    s = [x.cuda() for x in src]
    lib.swap_blocks_kv(d[0], d[1], s[0], s[1], pairs.cuda())
    torch.cuda.synchronize()
    for k in range(2):
        orc.swap_blocks(dst[k], src[k], pairs)
        assert torch.equal(d[k].cpu(), dst[k])
    assert lib.device_errors() == 0
    bad = pairs.clone()
    bad[0, 0] = ns                                         # source past its pool
    expect = dst[0].clone()
    lib.swap_blocks(d[0], s[0], bad.cuda())
    assert lib.device_errors(clear=True) & 0x8
    assert orc.swap_blocks(expect, src[0], bad) == 1
    assert torch.equal(d[0].cpu(), expect)


def test_swap_within_one_pool(lib):
    """Device-to-device inside one pool (disjoint sources and targets), as
    the copy-on-write and defragmentation moves use it."""
    case = wl.make_case(5, S=256, lens=("uniform", 16, 64), d2d_pairs=200, h2d_pairs=4,
                        host_pool_blocks=8)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    pairs = case.d2d_pairs
    lib.swap_blocks_kv(dk, dv, dk, dv, pairs.cuda())
    rk, rv = case.k_pool.clone(), case.v_pool.clone()
    orc.swap_blocks(rk, rk.clone(), pairs)
    orc.swap_blocks(rv, rv.clone(), pairs)
    assert torch.equal(_bits(dk.cpu()), _bits(rk)) and torch.equal(_bits(dv.cpu()), _bits(rv))
    assert lib.device_errors() == 0


def test_swap_from_pinned_host(lib):
    case = wl.make_case(5, S=8, lens=("uniform", 16, 64), d2d_pairs=4, h2d_pairs=32,
                        host_pool_blocks=64)
    hk = case.host_k_pool.pin_memory()
    pairs_host = case.h2d_pairs.pin_memory()
    dk = case.k_pool.cuda()
    lib.swap_blocks(dk, hk, pairs_host)          # source and pairs in pinned host memory
    ref = case.k_pool.clone()
    orc.swap_blocks(ref, case.host_k_pool, case.h2d_pairs)
    assert torch.equal(_bits(dk.cpu()), _bits(ref))
    assert lib.device_errors() == 0


@pytest.mark.parametrize("pinned_source", [False, True])
def test_swap_kv_one_launch_matches_two_calls(lib, pinned_source):
    case = wl.make_case(5, S=8, lens=("uniform", 16, 64), d2d_pairs=4, h2d_pairs=40,
                        host_pool_blocks=64)
    pairs = case.h2d_pairs.clone()
    pairs[7, 0] = -1                           # a skipped pair
    if pinned_source:
        sk, sv, pr = case.host_k_pool.pin_memory(), case.host_v_pool.pin_memory(), pairs.pin_memory()
    else:
        sk, sv, pr = case.host_k_pool.cuda(), case.host_v_pool.cuda(), pairs.cuda()
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    lib.swap_blocks_kv(dk, dv, sk, sv, pr)
    rk, rv = case.k_pool.clone(), case.v_pool.clone()
    orc.swap_blocks(rk, case.host_k_pool, pairs)
    orc.swap_blocks(rv, case.host_v_pool, pairs)
    assert torch.equal(_bits(dk.cpu()), _bits(rk)) and torch.equal(_bits(dv.cpu()), _bits(rv))
    assert lib.device_errors() == 0
    bad = pairs.clone()
    bad[0, 1] = case.num_blocks                # destination past the pool
    lib.swap_blocks_kv(dk, dv, sk, sv, bad.cuda() if not pinned_source else bad.pin_memory())
    assert lib.device_errors() & 0x8


def test_append_matches_oracle_and_flags_bad_slots(lib):
    case = wl.make_case(5, S=40, lens=("uniform", 1, 70), d2d_pairs=4, h2d_pairs=4,
                        host_pool_blocks=8)
    tables = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    _, _, slots, _ = append_slots(tables, case.context_lens.tolist(), case.B, case.free_ids,
                                  case.num_blocks)
    slots = torch.tensor(slots, dtype=torch.int64)
    slots[5] = -1
    k, v = case.k_pool.clone(), case.v_pool.clone()
    orc.kv_append(k, v, case.k_new, case.v_new, slots)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    lib.kv_append(dk, dv, case.k_new.cuda(), case.v_new.cuda(), slots.cuda())
    assert torch.equal(_bits(dk.cpu()), _bits(k)) and torch.equal(_bits(dv.cpu()), _bits(v))
    assert lib.device_errors() == 0
    bad = slots.clone()
    bad[0] = case.num_blocks * case.B          # one past the pool
    lib.kv_append(dk, dv, case.k_new.cuda(), case.v_new.cuda(), bad.cuda())
    assert lib.device_errors() & 0x4
    assert torch.equal(_bits(dk.cpu()), _bits(k))


def test_append_f32_and_fp16_rows(lib):
    for dtype, D in ((torch.float32, 4), (torch.float16, 64)):
        k = torch.randn(6, 16, 2, D).to(dtype)
        v = torch.randn(6, 16, 2, D).to(dtype)
        kn = torch.randn(3, 2, D).to(dtype)
        vn = torch.randn(3, 2, D).to(dtype)
        slots = torch.tensor([95, 0, 17])
        dk, dv = k.cuda(), v.cuda()
        lib.kv_append(dk, dv, kn.cuda(), vn.cuda(), slots.cuda())
        orc.kv_append(k, v, kn, vn, slots)
        assert torch.equal(dk.cpu(), k) and torch.equal(dv.cpu(), v)
    assert lib.device_errors() == 0


def _continuous_step(lib, case):
    """Library side of one continuous-batching step."""
    bm = lib.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    bt = case.block_tables.clone()
    lens = case.context_lens.clone()
    slots = torch.empty(case.S, dtype=torch.int64)
    assert bm.append_slots(bt, lens, slots) == 0
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    q = case.q.cuda()
    lib.kv_append(dk, dv, case.k_new.cuda(), case.v_new.cuda(), slots.cuda())
    out = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    lib.paged_attn_decode(out, q, dk, dv, bt.cuda(), lens.cuda(), case.scale,
                          int(lens.max()))
    d2d = case.d2d_pairs.cuda()
    lib.swap_blocks(dk, dk, d2d)
    lib.swap_blocks(dv, dv, d2d)
    hk, hv = case.host_k_pool.pin_memory(), case.host_v_pool.pin_memory()
    h2d = case.h2d_pairs.pin_memory()
    lib.swap_blocks_kv(dk, dv, hk, hv, h2d)
    torch.cuda.synchronize()
    return bt, lens, slots, out, dk.cpu(), dv.cpu()


def _continuous_oracle(case):
    tables = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    new_tables, new_lens, slots, _ = append_slots(tables, case.context_lens.tolist(), case.B,
                                                  case.free_ids, case.num_blocks)
    k, v = case.k_pool.clone(), case.v_pool.clone()
    orc.kv_append(k, v, case.k_new, case.v_new, torch.tensor(slots))
    bt = torch.full_like(case.block_tables, -1)
    for s, row in enumerate(new_tables):
        bt[s, :len(row)] = torch.tensor(row, dtype=torch.int32)
    lens = torch.tensor(new_lens, dtype=torch.int32)
    out = orc.decode_two_pass(case.q, k, v, bt, lens, case.scale)
    # sum_t w_t |V_t| on the appended state (the hi + lo weight term of the bound)
    out_abs = lambda: orc.decode_two_pass(case.q, k0, v0.abs(), bt, lens, case.scale)  # noqa: E731
    k0, v0 = k.clone(), v.clone()
    for pool in (k, v):
        assert orc.swap_blocks(pool, pool.clone(), case.d2d_pairs) == 0
    assert orc.swap_blocks(k, case.host_k_pool, case.h2d_pairs) == 0
    assert orc.swap_blocks(v, case.host_v_pool, case.h2d_pairs) == 0
    return bt, lens, slots, out, k, v, out_abs


@pytest.mark.parametrize("small", [True, False])
def test_continuous_batching_step(lib, small):
    if small:
        case = wl.make_case(5, S=48, lens=("pareto", 1.5, 16, 700), d2d_pairs=32, h2d_pairs=32,
                            host_pool_blocks=64, poison=True)
    else:
        case = wl.make_case(5)            # the stated workload at full size
    bt, lens, slots, out, k, v = _continuous_step(lib, case)
    rbt, rlens, rslots, rout, rk, rv, rabs = _continuous_oracle(case)
    assert slots.tolist() == rslots
    assert torch.equal(lens, rlens)
    assert torch.equal(bt, rbt)
    assert torch.equal(_bits(k), _bits(rk)) and torch.equal(_bits(v), _bits(rv))
    assert_attention_close(out, rout, case.out_dtype, "continuous step", kv_dtype=case.dtype,
                           abs_weighted=rabs)
    assert lib.device_errors() == 0


def test_copy_on_write_step(lib):
    """Forked sequences share their parent's blocks (partly filled last pages
    included).  One step: copy-on-write bookkeeping (native manager), copy of
    the shared pages (swap_blocks_kv), append, decode -- against the oracle's
    allocator, copy, append and decode.  Parents must keep their own pages."""
    from oracle.block_manager import append_slots_cow
    lens = [20, 37, 5, 50, 20, 37, 37]           # seqs 4..6 fork seqs 0, 1, 1
    parents = {4: 0, 5: 1, 6: 1}
    case = wl.make_case(5, lens_override=lens, H=8, Hk=2, D=64, d2d_pairs=0, h2d_pairs=0,
                        host_pool_blocks=1, poison=False)
    for c, p in parents.items():
        case.block_tables[c] = case.block_tables[p]
    nb, B, S = case.num_blocks, case.B, case.S
    refs = [0] * nb
    for row in case.block_tables.tolist():
        for b in row:
            if b >= 0:
                refs[b] += 1
    free_ids = sorted(b for b in range(nb) if refs[b] == 0)
    tables = [[x for x in row if x >= 0] for row in case.block_tables.tolist()]

    # ---- library
    bm = lib.BlockManager(nb, B, free_ids=free_ids)
    for b in range(nb):
        for _ in range(refs[b] - 1):
            bm.add_reference(b)
    bt, lt = case.block_tables.clone(), case.context_lens.clone()
    slots = torch.empty(S, dtype=torch.int64)
    st, pairs = bm.append_slots_cow(bt, lt, slots)
    assert st == 0 and pairs.shape[0] == 3       # each child's shared partial page
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    lib.swap_blocks_kv(dk, dv, dk, dv, pairs.cuda())
    lib.kv_append(dk, dv, case.k_new.cuda(), case.v_new.cuda(), slots.cuda())
    out = torch.empty(S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    lib.paged_attn_decode(out, case.q.cuda(), dk, dv, bt.cuda(), lt.cuda(), case.scale,
                          int(lt.max()))
    torch.cuda.synchronize()

    # ---- oracle
    new_tables, new_lens, ref_slots, ref_pairs, _, _ = append_slots_cow(
        tables, lens, B, free_ids, nb, refs)
    assert slots.tolist() == ref_slots and [tuple(x) for x in pairs.tolist()] == ref_pairs
    k, v = case.k_pool.clone(), case.v_pool.clone()
    pr = torch.tensor(ref_pairs, dtype=torch.int64)
    orc.swap_blocks(k, k.clone(), pr)
    orc.swap_blocks(v, v.clone(), pr)
    orc.kv_append(k, v, case.k_new, case.v_new, torch.tensor(ref_slots))
    rbt = torch.full_like(case.block_tables, -1)
    for s, row in enumerate(new_tables):
        rbt[s, :len(row)] = torch.tensor(row, dtype=torch.int32)
    assert torch.equal(bt, rbt)
    ref = orc.decode_two_pass(case.q, k, v, rbt, torch.tensor(new_lens, dtype=torch.int32),
                              case.scale)
    assert torch.equal(_bits(dk.cpu()), _bits(k)) and torch.equal(_bits(dv.cpu()), _bits(v))
    assert_attention_close(out, ref, case.out_dtype, "copy-on-write step")
    # whichever of a parent and its child wrote first into their shared page
    # got a private copy: afterwards they no longer share the page they wrote
    for c, p in parents.items():
        assert bt[c, lens[c] // B] != bt[p, lens[p] // B]
    assert lib.device_errors() == 0


def test_defragmentation_keeps_decode_identical(lib):
    """Compact the pool (used blocks to the lowest ids) with the planner and
    one swap_blocks_kv, then decode: bit-identical to the decode before."""
    case = wl.make_case(3, S=12, lens=("uniform", 1, 300), share_blocks=3, pool_extra=1.5)
    nb, B = case.num_blocks, case.B
    refs = [0] * nb
    for row in case.block_tables.tolist():
        for b in row:
            if b >= 0:
                refs[b] += 1
    free_ids = [b for b in range(nb) if refs[b] == 0]
    bm = lib.BlockManager(nb, B, free_ids=free_ids)
    for b in range(nb):
        for _ in range(refs[b] - 1):
            bm.add_reference(b)
    dk, dv = case.k_pool.cuda(), case.v_pool.cuda()
    before = torch.empty(case.S, case.H, case.D, dtype=case.out_dtype, device="cuda")
    lib.paged_attn_decode(before, case.q.cuda(), dk, dv, case.block_tables.cuda(),
                          case.context_lens.cuda(), case.scale, case.max_context_len)
    bt = case.block_tables.clone()
    pairs = bm.defrag(bt)
    assert pairs.shape[0] > 0
    lib.swap_blocks_kv(dk, dv, dk, dv, pairs.cuda())
    after = torch.empty_like(before)
    lib.paged_attn_decode(after, case.q.cuda(), dk, dv, bt.cuda(), case.context_lens.cuda(),
                          case.scale, case.max_context_len)
    assert torch.equal(before, after)
    n_used = sum(1 for r in refs if r > 0)
    assert int(bt.max()) == n_used - 1 and bm.free_ids() == list(range(n_used, nb))
    assert lib.device_errors() == 0
