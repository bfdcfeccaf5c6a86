"""Pins of the fp64 CPU oracle against things other than itself: library
routines (numpy, scipy, torch), closed forms, invariants, and the examples the
pages print (tests/golden/).  CPU only."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle as orc
from oracle import block_manager as bm
from oracle.block_manager import append_slots
from paged_kv_decode_26_gb300 import workloads as wl


# ---------------------------------------------------------------- decoders

def test_f16_decoder_all_bit_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    got = orc.decode_elements(bits, torch.float16)
    ref = bits.numpy().view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_bf16_decoder_all_bit_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    got = orc.decode_elements(bits, torch.bfloat16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


# ---------------------------------------------------------------- helpers

def _contiguous_case(S, H, Hk, D, B, lens, dtype=torch.float64, seed=0):
    """Sequences stored back to back: seq s owns blocks s*mb .. s*mb+mb-1, so
    that the pool reshaped to [S, mb*B, Hk, D] is each sequence's logical
    context with no table arithmetic needed to read it."""
    g = torch.Generator().manual_seed(seed)
    mb = max(1, max((n + B - 1) // B for n in lens))
    nb = S * mb
    k = torch.randn(nb, B, Hk, D, generator=g, dtype=torch.float64).to(dtype)
    v = torch.randn(nb, B, Hk, D, generator=g, dtype=torch.float64).to(dtype)
    q = torch.randn(S, H, D, generator=g, dtype=torch.float64).to(dtype)
    bt = torch.arange(nb, dtype=torch.int32).view(S, mb)
    cl = torch.tensor(lens, dtype=torch.int32)
    return q, k, v, bt, cl, mb


def _logical(pool, S, mb, B, Hk, D):
    return pool.to(torch.float64).reshape(S, mb * B, Hk, D)


# ------------------------------------------------- attention vs libraries

@pytest.mark.parametrize("H,Hk", [(4, 4), (8, 2)])
def test_two_pass_matches_scipy_softmax(H, Hk):
    S, D, B = 3, 16, 4
    lens = [1, 9, 16]
    q, k, v, bt, cl, mb = _contiguous_case(S, H, Hk, D, B, lens)
    scale = 0.37
    got = orc.decode_two_pass(q, k, v, bt, cl, scale)
    K = _logical(k, S, mb, B, Hk, D).numpy()
    V = _logical(v, S, mb, B, Hk, D).numpy()
    G = H // Hk
    for s in range(S):
        for h in range(H):
            n = lens[s]
            x = scale * K[s, :n, h // G, :] @ q[s, h].numpy()
            w = scipy.special.softmax(x)
            ref = w @ V[s, :n, h // G, :]
            np.testing.assert_allclose(got[s, h], ref, rtol=1e-13, atol=1e-14)


def test_two_pass_matches_torch_sdpa_gqa():
    """GQA with contiguous groups equals torch's SDPA on KV heads repeated
    with repeat_interleave (query head h uses kv head h // G)."""
    S, H, Hk, D, B = 2, 8, 2, 32, 8
    lens = [13, 24]
    q, k, v, bt, cl, mb = _contiguous_case(S, H, Hk, D, B, lens, seed=3)
    scale = 1 / math.sqrt(D)
    got = orc.decode_two_pass(q, k, v, bt, cl, scale)
    K = _logical(k, S, mb, B, Hk, D)
    V = _logical(v, S, mb, B, Hk, D)
    for s in range(S):
        n = lens[s]
        Ks = K[s, :n].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)  # [H, n, D]
        Vs = V[s, :n].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[s].unsqueeze(1), Ks, Vs, scale=scale).squeeze(1)
        np.testing.assert_allclose(got[s], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_tiny_brute_force_by_hand():
    """d=2, two keys, values chosen so the result is known in closed form:
    scores 0 and ln 3 give weights 1/4 and 3/4."""
    q = torch.tensor([[[1.0, 0.0]]], dtype=torch.float64)
    k = torch.tensor([[[[0.0, 5.0]], [[math.log(3.0), -2.0]]]], dtype=torch.float64)  # [1,2,1,2]
    v = torch.tensor([[[[4.0, 8.0]], [[0.0, -4.0]]]], dtype=torch.float64)
    out = orc.decode_two_pass(q, k, v, torch.tensor([[0]]), torch.tensor([2]), 1.0)
    np.testing.assert_allclose(out[0, 0], [1.0, -1.0], rtol=0, atol=1e-15)
    # only the first key: weight 1
    out1 = orc.decode_two_pass(q, k, v, torch.tensor([[0]]), torch.tensor([1]), 1.0)
    assert out1[0, 0].tolist() == [4.0, 8.0]


# ------------------------------------------------------ closed forms

def test_context_one_gives_v_exactly():
    case = wl.make_case(1, S=4, lens=("const", 1))
    out = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    G = case.H // case.Hk
    for s in range(case.S):
        p = int(case.block_tables[s, 0])
        for h in range(case.H):
            ref = case.v_pool[p, 0, h // G].to(torch.float64).numpy()
            assert np.array_equal(out[s, h], ref)


def test_constant_v_gives_v():
    case = wl.make_case(1, S=3)
    c = torch.linspace(-2, 2, case.D).to(case.dtype)
    case.v_pool[:] = c
    out = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    ref = c.to(torch.float64).numpy()
    for s in range(case.S):
        for h in range(case.H):
            np.testing.assert_allclose(out[s, h], ref, rtol=1e-14, atol=1e-15)


def test_dominant_key_selects_its_value():
    S, H, Hk, D, B = 1, 2, 1, 8, 4
    q, k, v, bt, cl, mb = _contiguous_case(S, H, Hk, D, B, [7], seed=5)
    q[:] = 1.0
    k[:] = 0.0
    k[1, 2, 0, :] = 100.0  # logical token 6 (block 1, row 2) dominates by 800
    out = orc.decode_two_pass(q, k, v, bt, cl, 1.0)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], v[1, 2, 0].numpy(), rtol=0, atol=1e-300)


def test_empty_context_is_zero():
    case = wl.make_case(1, S=3, lens_override=[0, 5, 0])
    out = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[1])) and np.any(out[1] != 0)


def test_scores_use_the_scale():
    """Doubling the scale equals doubling q (the scores are scale * q.k)."""
    case = wl.make_case(1, S=2, dtype=torch.float64)
    a = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                            case.context_lens, 2 * case.scale)
    b = orc.decode_two_pass(case.q * 2, case.k_pool, case.v_pool, case.block_tables,
                            case.context_lens, case.scale)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------ invariants

def _replace_placement(case, new_ids_of):
    """Move every block to a new physical id (a bijection) and rewrite the tables."""
    nb = case.num_blocks
    perm = np.asarray(new_ids_of)
    k2 = torch.empty_like(case.k_pool)
    v2 = torch.empty_like(case.v_pool)
    k2[torch.from_numpy(perm)] = case.k_pool
    v2[torch.from_numpy(perm)] = case.v_pool
    bt = case.block_tables.numpy().copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    assert sorted(perm.tolist()) == list(range(nb))
    return k2, v2, torch.from_numpy(bt)


@pytest.mark.parametrize("config", [1, 3])
def test_physical_permutation_invariance(config):
    case = wl.make_case(config, S=6, lens=("uniform", 1, 70) if config == 1 else ("uniform", 1, 90),
                        share_blocks=2)
    base = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                               case.context_lens, case.scale)
    perm = np.random.default_rng(9).permutation(case.num_blocks)
    k2, v2, bt2 = _replace_placement(case, perm)
    moved = orc.decode_two_pass(case.q, k2, v2, bt2, case.context_lens, case.scale)
    assert np.array_equal(base, moved)


def test_page_block_table_example(golden):
    """The pages' example tables ([5,12,8], [3,7], [9,14,16,20]) hold the same
    logical data as a contiguous layout: identical outputs."""
    tables = golden("block_table_example.json")["tables"]
    B, H, Hk, D = 4, 4, 2, 8
    lens = [len(t) * B - 1 for t in tables]  # a ragged last page each
    S = len(tables)
    q, k, v, bt_c, cl, mb = _contiguous_case(S, H, Hk, D, B, lens, seed=11)
    base = orc.decode_two_pass(q, k, v, bt_c, cl, 0.3)
    nb = 21
    k2 = torch.full((nb, B, Hk, D), float("nan"), dtype=torch.float64)
    v2 = k2.clone()
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        for j, p in enumerate(t):
            k2[p] = k[s * mb + j]
            v2[p] = v[s * mb + j]
            bt[s, j] = p
    # rows past each context in the last page are never read: poison them
    for s, t in enumerate(tables):
        k2[t[-1], lens[s] % B or B:] = float("nan")
        v2[t[-1], lens[s] % B or B:] = float("nan")
    got = orc.decode_two_pass(q, k2, v2, bt, cl, 0.3)
    assert np.array_equal(base, got)


def test_masking_poisoned_rows_not_read():
    clean = wl.make_case(1, S=4)
    dirty = wl.make_case(1, S=4, poison=True)
    a = orc.decode_two_pass(clean.q, clean.k_pool, clean.v_pool, clean.block_tables,
                            clean.context_lens, clean.scale)
    b = orc.decode_two_pass(dirty.q, dirty.k_pool, dirty.v_pool, dirty.block_tables,
                            dirty.context_lens, dirty.scale)
    assert np.all(np.isfinite(b))
    assert np.array_equal(a, b)


def test_mha_with_replicated_kv_equals_gqa():
    """[SWAP] MQA/GQA: sharing a KV head by indexing equals replicating it."""
    case = wl.make_case(3, S=3, lens=("uniform", 1, 80), share_blocks=1)
    G = case.H // case.Hk
    gqa = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    k_rep = case.k_pool.repeat_interleave(G, dim=2).contiguous()
    v_rep = case.v_pool.repeat_interleave(G, dim=2).contiguous()
    mha = orc.decode_two_pass(case.q, k_rep, v_rep, case.block_tables, case.context_lens,
                              case.scale)
    assert np.array_equal(gqa, mha)


def test_out_of_range_block_is_rejected():
    case = wl.make_case(1, S=2, lens_override=[20, 3])
    case.block_tables[0, 1] = case.num_blocks
    with pytest.raises(orc.OracleError):
        orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                            case.context_lens, case.scale)


# ------------------------------------------- online recurrence and merge

@pytest.mark.parametrize("tile", [1, 3, 16, 17, 1000])
def test_online_recurrence_equals_two_pass(tile):
    case = wl.make_case(3, S=5, lens=("uniform", 1, 120), share_blocks=2)
    a = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                            case.context_lens, case.scale)
    b = orc.decode_online(case.q, case.k_pool, case.v_pool, case.block_tables,
                          case.context_lens, case.scale, tile)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


def test_online_state_is_log_partition():
    """Final (M, L) of the recurrence: M is the maximum score and
    M + ln L = logsumexp of the scores (scipy)."""
    q, k, v, bt, cl, mb = _contiguous_case(1, 2, 2, 16, 4, [11], seed=2)
    out, m, l_ = orc.decode_online(q, k, v, bt, cl, 0.5, 4, return_state=True)
    K = _logical(k, 1, mb, 4, 2, 16).numpy()
    for h in range(2):
        x = 0.5 * K[0, :11, h, :] @ q[0, h].numpy()
        np.testing.assert_allclose(m[0, h], x.max(), rtol=1e-14)
        np.testing.assert_allclose(m[0, h] + math.log(l_[0, h]), scipy.special.logsumexp(x),
                                   rtol=1e-14)


@pytest.mark.parametrize("cuts", [[0, 50], [0, 7, 33, 34], [0, 1000]])
def test_merge_of_split_states_equals_two_pass(cuts):
    case = wl.make_case(2, S=3, lens=("uniform", 40, 90), H=4, Hk=4, D=32)
    full = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                               case.context_lens, case.scale)
    edges = cuts + [10 ** 6]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        parts.append(orc.decode_online(case.q, case.k_pool, case.v_pool, case.block_tables,
                                       case.context_lens, case.scale, 16, t_begin=a, t_end=b,
                                       return_state=True))
    for s in range(case.S):
        for h in range(case.H):
            m = np.array([p[1][s, h] for p in parts])
            l_ = np.array([p[2][s, h] for p in parts])
            o = np.stack([p[0][s, h] for p in parts])
            got = orc.merge_states(m, l_, o)
            np.testing.assert_allclose(got, full[s, h], rtol=1e-12, atol=1e-13)


# ------------------------------------------------ byte accounting (golden)

def test_kv_cache_bytes_worked_example(golden):
    g = golden("kv_cache_bytes.json")
    got = orc.kv_cache_bytes(g["n_layers"], g["n_heads"], g["d_head"], g["seq_len"], g["batch"],
                             g["elem_bytes"])
    assert got == g["bytes"] == 274877906944
    # one layer of the long-context workload: 16 seqs x 32768 tokens x 32 heads x 128 = 8 GiB
    assert orc.kv_cache_bytes(1, 32, 128, 32768, 16, 2) == 8 * 2 ** 30


# ---------------------------------------------------------- block copy

def test_swap_page_mock_example(golden):
    g = golden("swap_mock_example.json")
    src = torch.randn(g["num_src_blocks"], 32, 64, 16)
    dst = torch.zeros(g["num_dst_blocks"], 32, 64, 16)
    pairs = torch.tensor([[i, j] for i, j in enumerate(g["mapping"])], dtype=torch.int64)
    skipped = orc.swap_blocks(dst, src, pairs)
    assert skipped == 1  # target 5 does not exist
    for d, s in g["expected_dst_from_src"].items():
        assert torch.equal(dst[int(d)], src[s])
    for d in g["untouched_dst"]:
        assert torch.count_nonzero(dst[d]) == 0
    assert int((dst.sum(dim=[1, 2, 3]) != 0).sum()) == g["filled_blocks"]


def test_swap_matches_torch_indexing():
    g = np.random.default_rng(4)
    src = torch.randn(50, 4, 2, 8).to(torch.bfloat16)
    dst = torch.randn(40, 4, 2, 8).to(torch.bfloat16)
    si = torch.from_numpy(g.choice(50, 17, replace=False))
    di = torch.from_numpy(g.choice(40, 17, replace=False))
    ref = dst.clone()
    ref[di] = src[si]
    orc.swap_blocks(dst, src, torch.stack([si, di], 1))
    assert torch.equal(dst.view(torch.int16), ref.view(torch.int16))


def test_swap_skips_invalid_pairs():
    src = torch.arange(5 * 6, dtype=torch.float32).view(5, 6)
    dst = torch.zeros(3, 6)
    pairs = torch.tensor([[-1, 0], [1, -1], [7, 1], [2, 9], [4, 2]])
    assert orc.swap_blocks(dst, src, pairs) == 2
    assert torch.count_nonzero(dst[:2]) == 0
    assert torch.equal(dst[2], src[4])


# -------------------------------------------------------------- append

def test_kv_append_matches_torch_indexing():
    case = wl.make_case(5, S=20, lens=("uniform", 1, 60), d2d_pairs=4, h2d_pairs=4,
                        host_pool_blocks=8)
    tables = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    _, _, slots, _ = append_slots(tables, case.context_lens.tolist(), case.B, case.free_ids,
                                  case.num_blocks)
    slots = torch.tensor(slots, dtype=torch.int64)
    slots[3] = -1  # a skipped sequence
    k, v = case.k_pool.clone(), case.v_pool.clone()
    orc.kv_append(k, v, case.k_new, case.v_new, slots)
    rk, rv = case.k_pool.clone(), case.v_pool.clone()
    keep = slots >= 0
    rk.view(-1, case.Hk, case.D)[slots[keep]] = case.k_new[keep]
    rv.view(-1, case.Hk, case.D)[slots[keep]] = case.v_new[keep]
    assert torch.equal(k.view(torch.int16), rk.view(torch.int16))
    assert torch.equal(v.view(torch.int16), rv.view(torch.int16))


def test_kv_append_rejects_slot_past_pool():
    k = torch.zeros(2, 4, 1, 8)
    v = torch.zeros(2, 4, 1, 8)
    with pytest.raises(orc.OracleError):
        orc.kv_append(k, v, torch.ones(1, 1, 8), torch.ones(1, 1, 8), torch.tensor([8]))
    assert torch.count_nonzero(k) == 0


# ---------------------------------------------------------- allocator

def test_allocator_walkthrough(golden):
    """The two-request walkthrough of [LAYOUT] section 三: register A (20
    tokens) and B (10), append 13 tokens to A, finish B."""
    g = golden("allocator_walkthrough.json")
    B = g["block_size"]
    refs = bm.make_pool(g["num_blocks"])
    assert len(bm.free_list(refs)) == g["free_at_start"]
    a = bm.admit(refs, g["req_A"]["prompt_len"], B)
    b = bm.admit(refs, g["req_B"]["prompt_len"], B)
    assert a == g["req_A"]["blocks"] and b == g["req_B"]["blocks"]
    assert len(bm.free_list(refs)) == g["free_after_register"]
    n = g["req_A"]["prompt_len"]
    opened_at = None
    for i in range(g["appends_A"]):
        before = len(a)
        slot, n_new = bm.add_token(refs, a, n, B)
        assert slot >= 0 and n_new == n + 1
        assert slot == a[n // B] * B + n % B
        n = n_new
        if len(a) > before:
            assert opened_at is None
            opened_at = i + 1
    assert opened_at == g["new_block_on_append_number"]
    assert a[-1] == g["new_block_id"]
    assert a == g["A_blocks_after_appends"]
    assert n == g["A_tokens_after_appends"]
    assert len(bm.free_list(refs)) == g["free_after_appends"]
    bm.release(refs, b)
    assert len(bm.free_list(refs)) == g["free_after_finish_B"]
    assert bm.free_list(refs) == g["free_list_after_finish_B"]


def test_allocator_refcount_and_exhaustion():
    refs = bm.make_pool(2)
    t = bm.admit(refs, 8, 4)
    assert t == [0, 1]
    assert bm.add_token(refs, t, 8, 4) == (-1, 8)   # page full, pool empty: fails
    assert t == [0, 1]
    assert bm.admit(refs, 1, 4) is None
    bm.share_block(refs, 0)                          # a second holder of block 0
    bm.release(refs, t)
    assert bm.free_list(refs) == [1]                 # block 0 still referenced once
    bm.drop_reference(refs, 0)
    assert bm.free_list(refs) == [0, 1]
    bm.drop_reference(refs, 0)                       # a free id stays free
    assert refs == [0, 0]
    with pytest.raises(ValueError):
        bm.share_block(refs, 1)                      # a free id cannot be shared


def test_admit_gives_back_a_partial_allocation():
    refs = bm.make_pool(5, free_ids=[1, 3, 4])
    assert bm.admit(refs, 4 * 16, 16) is None       # needs 4 of 3 free
    assert bm.free_list(refs) == [1, 3, 4]
    assert bm.admit(refs, 33, 16) == [1, 3, 4]


def test_allocator_against_brute_force_lowest_free():
    """Random takes, shares and drops against a recount from scratch: the
    free list is exactly the ids whose count is 0, and every take returns
    the minimum of that set."""
    rng = np.random.default_rng(3)
    for _ in range(30):
        nb = int(rng.integers(1, 40))
        refs = bm.make_pool(nb)
        held = []
        for _ in range(300):
            op = int(rng.integers(0, 3))
            if op == 0:
                free_before = [b for b in range(nb) if refs[b] == 0]
                b = bm.take_block(refs)
                if free_before:
                    assert b == min(free_before) and refs[b] == 1
                    held.append(b)
                else:
                    assert b is None
            elif op == 1 and held:
                b = held.pop(int(rng.integers(len(held))))
                bm.drop_reference(refs, b)
            elif op == 2 and held:
                b = held[int(rng.integers(len(held)))]
                bm.share_block(refs, b)
                held.append(b)
            counts = [held.count(b) for b in range(nb)]
            assert refs == counts
            assert bm.free_list(refs) == [b for b in range(nb) if counts[b] == 0]


def test_append_slots_page_boundary():
    tables = [[7], [3, 9], []]
    lens = [16, 17, 0]
    new_tables, new_lens, slots, free_after = append_slots(tables, lens, 16, [0, 1, 2, 4], 10)
    # seq 0: page full -> lowest free id 0, token 16 at row 0 of block 0;
    # seq 1: row 1 of block 9; seq 2: empty -> opens block 1, row 0
    assert new_tables == [[7, 0], [3, 9], [1]]
    assert slots == [0 * 16 + 0, 9 * 16 + 1, 1 * 16 + 0]
    assert new_lens == [17, 18, 1]
    assert free_after == [2, 4]


def test_copy_on_write_fork_walkthrough():
    """[LAYOUT] section 四.2: a parent (blocks 0, 1; 20 tokens, so block 1 is
    partly filled) is shared by two forked children.  Each child's first
    append lands in the shared block 1 and gets a private copy (lowest free
    ids 2, then 3); once the parent is the last holder it writes in place."""
    from oracle.block_manager import append_slots_cow
    tables = [[0, 1], [0, 1], [0, 1]]          # children 0, 1 and the parent
    refs = [3, 3] + [0] * 6
    new_tables, lens, slots, pairs, free_after, refs_after = append_slots_cow(
        tables, [20, 20, 20], 16, list(range(2, 8)), 8, refs)
    assert pairs == [(1, 2), (1, 3)]
    assert new_tables == [[0, 2], [0, 3], [0, 1]]
    assert slots == [2 * 16 + 4, 3 * 16 + 4, 1 * 16 + 4]
    assert lens == [21, 21, 21]
    assert refs_after[:4] == [3, 1, 1, 1] and free_after == [4, 5, 6, 7]
    # a full page never copies: it opens a new block
    t2, _, s2, p2, _, _ = append_slots_cow([[0, 1], [0, 1]], [32, 32], 16, [2, 3], 4,
                                           [2, 2, 0, 0])
    assert p2 == [] and t2 == [[0, 1, 2], [0, 1, 3]] and s2 == [32, 48]


def test_defrag_plan_hand_example():
    """Used blocks 0, 2, 4, 5 (4 in use): 4 and 5 move into the holes 1 and 3."""
    from oracle.block_manager import apply_defrag, defrag_plan
    refs = [1, 0, 2, 0, 1, 1]
    pairs = defrag_plan(refs)
    assert pairs == [(4, 1), (5, 3)]
    tables, new_refs = apply_defrag([[0, 4], [2, 5], [2]], refs, pairs)
    assert tables == [[0, 1], [2, 3], [2]]
    assert new_refs == [1, 1, 2, 1, 0, 0]
    assert defrag_plan([1, 1, 0, 0]) == []          # already compact


# ------------------------------------------------- several query tokens

def test_multi_query_one_token_is_decode():
    case = wl.make_case(3, S=5, lens=("uniform", 1, 90), share_blocks=2)
    q, qs = wl.multi_query_inputs(case, ("const", 1))
    got = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    ref = orc.decode_two_pass(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens,
                              case.scale)
    assert np.array_equal(got, ref)


def test_multi_query_rows_are_decodes_of_their_prefix():
    """Row i of a sequence attends exactly to the keys up to its position."""
    case = wl.make_case(2, S=3, lens=("uniform", 5, 60), H=4, Hk=2, D=32)
    q, qs = wl.multi_query_inputs(case, ("uniform", 1, 9))
    got = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    for s in range(case.S):
        n = int(case.context_lens[s])
        ql = int(qs[s + 1] - qs[s])
        for i in range(ql):
            row = int(qs[s]) + i
            lens = case.context_lens.clone()
            lens[s] = n - ql + i + 1
            qq = case.q.clone()
            qq[s] = q[row]
            ref = orc.decode_two_pass(qq, case.k_pool, case.v_pool, case.block_tables, lens,
                                      case.scale, seq_ids=[s])
            assert np.array_equal(got[row], ref[0])


def test_multi_query_matches_torch_sdpa_causal():
    S, H, Hk, D, B = 2, 4, 2, 16, 4
    lens = [11, 7]
    q_lens = [4, 7]
    q, k, v, bt, cl, mb = _contiguous_case(S, H, Hk, D, B, lens, seed=21)
    g = torch.Generator().manual_seed(3)
    qs = torch.tensor([0, 4, 11], dtype=torch.int32)
    qm = torch.randn(11, H, D, generator=g, dtype=torch.float64)
    got = orc.multi_query(qm, k, v, bt, cl, qs, 0.25)
    K = _logical(k, S, mb, B, Hk, D)
    V = _logical(v, S, mb, B, Hk, D)
    for s in range(S):
        n, ql = lens[s], q_lens[s]
        Ks = K[s, :n].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)    # [H, n, D]
        Vs = V[s, :n].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)
        Qs = qm[int(qs[s]):int(qs[s + 1])].permute(1, 0, 2)                 # [H, ql, D]
        pos = torch.arange(n - ql, n).unsqueeze(1)
        mask = torch.arange(n).unsqueeze(0) <= pos                           # [ql, n]
        ref = torch.nn.functional.scaled_dot_product_attention(Qs, Ks, Vs, attn_mask=mask,
                                                               scale=0.25)
        np.testing.assert_allclose(got[int(qs[s]):int(qs[s + 1])], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-13)


# ------------------------------------------------- threaded oracle driver

@pytest.mark.parametrize("threads", [1, 3, 16])
@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 2)])
def test_threaded_oracle_equals_one_call(threads, H, Hk):
    """The thread-pool driver (whole sequences, or sequences cut into kv-head
    ranges over compact pools) gives the single call's result exactly,
    empty contexts and NaN padding included."""
    from oracle import parallel
    case = wl.make_case(3, S=5, lens_override=[0, 70, 1, 33, 200], H=H, Hk=Hk, D=64,
                        share_blocks=2, poison=True, seed=H + Hk + threads)
    ref = orc.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                              case.context_lens, case.scale)
    got = parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale, threads=threads)
    assert np.array_equal(got, ref)
    sub = parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables,
                                   case.context_lens, case.scale, seq_ids=[4, 1],
                                   threads=threads)
    assert np.array_equal(sub, ref[[4, 1]])
