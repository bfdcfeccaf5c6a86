"""The library's native block manager against the oracle's restatement of the
pages' allocator rules: the walkthrough, random operation sequences, and the
per-step append bookkeeping, all bit-exact.  CPU only (host code)."""
import numpy as np
import pytest
import torch

from oracle import block_manager as obm
from oracle.block_manager import append_slots
from paged_kv_decode_26_gb300 import workloads as wl


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_decode_26_gb300 import build
    build.build()
    import paged_kv_decode_26_gb300 as m
    return m


def test_walkthrough(pkv, golden):
    g = golden("allocator_walkthrough.json")
    bm = pkv.BlockManager(g["num_blocks"], g["block_size"])
    S, mb = 2, 8
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    lens = torch.zeros(S, dtype=torch.int32)
    # register: ceil(prompt / B) blocks each
    for s, key in enumerate(("req_A", "req_B")):
        n = g[key]["prompt_len"]
        for j in range((n + g["block_size"] - 1) // g["block_size"]):
            bt[s, j] = bm.allocate()
        lens[s] = n
        assert bt[s][bt[s] >= 0].tolist() == g[key]["blocks"]
    assert bm.free_count() == g["free_after_register"]
    slots = torch.zeros(1, dtype=torch.int64)
    opened = None
    for i in range(g["appends_A"]):
        before = int((bt[0] >= 0).sum())
        st = bm.append_slots(bt[0:1], lens[0:1], slots)
        assert st == 0
        if int((bt[0] >= 0).sum()) > before:
            opened = i + 1
    assert opened == g["new_block_on_append_number"]
    assert bt[0][bt[0] >= 0].tolist() == g["A_blocks_after_appends"]
    assert int(lens[0]) == g["A_tokens_after_appends"]
    assert bm.free_count() == g["free_after_appends"]
    for b in g["req_B"]["blocks"]:
        bm.free(b)
    assert bm.free_count() == g["free_after_finish_B"]
    assert bm.free_ids() == g["free_list_after_finish_B"]


def test_random_operation_sequences_match_oracle(pkv):
    rng = np.random.default_rng(17)
    for trial in range(20):
        nb = int(rng.integers(1, 200))
        refs = obm.make_pool(nb)
        bm = pkv.BlockManager(nb, 16)
        held = []
        for _ in range(400):
            op = rng.integers(0, 3)
            if op == 0:
                a = obm.take_block(refs)
                if a is None:
                    with pytest.raises(pkv.PagedKVError):
                        bm.allocate()
                else:
                    assert bm.allocate() == a
                    held.append(a)
            elif op == 1 and held:
                b = held.pop(int(rng.integers(len(held))))
                obm.drop_reference(refs, b)
                bm.free(b)
            elif op == 2 and held:
                b = held[int(rng.integers(len(held)))]
                obm.share_block(refs, b)
                bm.add_reference(b)
                held.append(b)
            assert bm.free_count() == len(obm.free_list(refs))
        assert bm.free_ids() == obm.free_list(refs)
        for b in range(nb):
            assert bm.ref_count(b) == refs[b]


def test_add_reference_of_free_block_is_rejected(pkv):
    bm = pkv.BlockManager(4, 16)
    with pytest.raises(pkv.PagedKVError):
        bm.add_reference(2)
    with pytest.raises(pkv.PagedKVError):
        bm.free(9)


@pytest.mark.parametrize("S,nb_extra", [(64, 40), (256, 300)])
def test_append_step_matches_oracle(pkv, S, nb_extra):
    case = wl.make_case(5, S=S, lens=("pareto", 1.5, 16, 300), d2d_pairs=8, h2d_pairs=8,
                        host_pool_blocks=16)
    tables = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    new_tables, new_lens, slots, free_after = append_slots(
        tables, case.context_lens.tolist(), case.B, case.free_ids, case.num_blocks)
    bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
    bt = case.block_tables.clone()
    lens = case.context_lens.clone()
    got_slots = torch.empty(S, dtype=torch.int64)
    assert bm.append_slots(bt, lens, got_slots) == 0
    assert got_slots.tolist() == slots
    assert lens.tolist() == new_lens
    for s in range(S):
        assert bt[s][bt[s] >= 0].tolist() == new_tables[s]
    assert bm.free_ids() == free_after


def test_append_with_exhausted_pool(pkv):
    bm = pkv.BlockManager(1, 16)
    bt = torch.full((2, 2), -1, dtype=torch.int32)
    lens = torch.zeros(2, dtype=torch.int32)
    slots = torch.empty(2, dtype=torch.int64)
    assert bm.append_slots(bt, lens, slots) == 5  # PKV_ERR_NO_BLOCKS
    assert slots.tolist() == [0, -1]
    assert lens.tolist() == [1, 0]
    assert bt[0, 0] == 0 and bt[1, 0] == -1
    tables, new_lens, ref_slots, _ = append_slots([[], []], [0, 0], 16, [0], 1)
    assert ref_slots == [0, -1] and new_lens == [1, 0]


def _fork_state(rng, nb, B, n_parents, n_children):
    """Random parents with private blocks, then children sharing a parent's
    whole table (references added), as (tables, lens, refs, free_ids)."""
    perm = rng.permutation(nb).tolist()
    tables, lens = [], []
    for _ in range(n_parents):
        n = int(rng.integers(1, 5 * B))
        k = (n + B - 1) // B
        tables.append([perm.pop() for _ in range(k)])
        lens.append(n)
    for _ in range(n_children):
        p = int(rng.integers(n_parents))
        tables.append(list(tables[p]))
        lens.append(lens[p])
    refs = [0] * nb
    for t in tables:
        for b in t:
            refs[b] += 1
    free_ids = sorted(b for b in range(nb) if refs[b] == 0)
    return tables, lens, refs, free_ids


def test_copy_on_write_matches_oracle(pkv):
    from oracle.block_manager import append_slots_cow
    rng = np.random.default_rng(5)
    B = 16
    for trial in range(30):
        nb = 200
        tables, lens, refs, free_ids = _fork_state(rng, nb, B, 6, int(rng.integers(0, 8)))
        S = len(tables)
        ref = append_slots_cow(tables, lens, B, free_ids, nb, refs)
        bm = pkv.BlockManager(nb, B, free_ids=free_ids)
        for b in range(nb):
            for _ in range(refs[b] - 1):
                bm.add_reference(b)
        mb = 8
        bt = torch.full((S, mb), -1, dtype=torch.int32)
        for s, t in enumerate(tables):
            bt[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
        lt = torch.tensor(lens, dtype=torch.int32)
        slots = torch.empty(S, dtype=torch.int64)
        st, pairs = bm.append_slots_cow(bt, lt, slots)
        assert st == 0
        new_tables, new_lens, ref_slots, ref_pairs, free_after, refs_after = ref
        assert slots.tolist() == ref_slots
        assert [tuple(x) for x in pairs.tolist()] == ref_pairs
        assert lt.tolist() == new_lens
        for s in range(S):
            assert bt[s][bt[s] >= 0].tolist() == new_tables[s]
        assert bm.free_ids() == free_after
        assert [bm.ref_count(b) for b in range(nb)] == refs_after


def test_defrag_matches_oracle(pkv):
    from oracle.block_manager import apply_defrag, defrag_plan
    rng = np.random.default_rng(8)
    for trial in range(25):
        nb, B = int(rng.integers(10, 300)), 16
        tables, lens, refs, free_ids = _fork_state(rng, nb * 2, B, 3, int(rng.integers(0, 4)))
        # shrink to ids < nb by taking a random used subset mapping
        tables = [[b % nb for b in t] for t in tables]
        refs = [0] * nb
        for t in tables:
            for b in t:
                refs[b] += 1
        free_ids = [b for b in range(nb) if refs[b] == 0]
        pairs_ref = defrag_plan(refs)
        tables_ref, refs_ref = apply_defrag(tables, refs, pairs_ref)
        bm = pkv.BlockManager(nb, B, free_ids=free_ids)
        for b in range(nb):
            for _ in range(refs[b] - 1):
                bm.add_reference(b)
        mb = max(len(t) for t in tables) + 1
        bt = torch.full((len(tables), mb), -1, dtype=torch.int32)
        for s, t in enumerate(tables):
            bt[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
        pairs = bm.defrag(bt)
        assert [tuple(p) for p in pairs.tolist()] == pairs_ref
        for s, t in enumerate(tables_ref):
            assert bt[s][bt[s] >= 0].tolist() == t
        assert [bm.ref_count(b) for b in range(nb)] == refs_ref
        n_used = sum(1 for r in refs if r > 0)
        assert bm.free_ids() == list(range(n_used, nb))
