"""The block manager on the GPU against the oracle's allocator rules (and,
as a second check, against the library's host manager): random decode steps
(appends at and between page boundaries), frees and shared blocks, compared
bit-exactly after every step -- tables, lengths, slots, reference counts and
the sorted free list."""
import numpy as np
import pytest
import torch

from oracle import block_manager as obm

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


@pytest.mark.parametrize("S,nb,B", [(5, 40, 16), (300, 2000, 16), (1500, 3000, 32), (64, 70, 16)])
def test_device_manager_matches_host_manager(pkv, S, nb, B):
    """Second check: the device manager and the host manager side by side."""
    rng = np.random.default_rng(S + nb)
    mb = 24
    host = pkv.BlockManager(nb, B)
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    lens = torch.zeros(S, dtype=torch.int32)
    # start: each sequence holds a few blocks
    for s in range(S):
        n = int(rng.integers(0, 3 * B))
        for j in range((n + B - 1) // B):
            try:
                bt[s, j] = host.allocate()
            except pkv.PagedKVError:
                n = j * B
                break
        lens[s] = n
    dev = pkv.DeviceBlockManager([host.ref_count(b) for b in range(nb)], B)
    assert dev.free_list() == host.free_ids()
    dbt, dlens = bt.cuda(), lens.cuda()
    dslots = torch.empty(S, dtype=torch.int64, device="cuda")
    hslots = torch.empty(S, dtype=torch.int64)
    for step in range(12):
        if step % 4 == 3:
            # finish a few random sequences on both sides
            done = rng.choice(S, size=max(1, S // 10), replace=False)
            ids = []
            for s in done:
                ids += [int(x) for x in bt[s] if x >= 0]
                bt[s] = -1
                lens[s] = 0
            for b in ids:
                host.free(b)
            dev.free(torch.tensor(ids, dtype=torch.int32, device="cuda"))
            dbt.copy_(bt)
            dlens.copy_(lens)
        st = host.append_slots(bt, lens, hslots)
        dev.append_slots(dbt, dlens, dslots)
        torch.cuda.synchronize()
        assert torch.equal(dslots.cpu(), hslots)
        assert torch.equal(dlens.cpu(), lens)
        assert torch.equal(dbt.cpu(), bt)
        assert dev.free_list() == host.free_ids()
        assert dev.ref_counts.cpu().tolist() == [host.ref_count(b) for b in range(nb)]
        assert dev.failed_last_append() == int((hslots < 0).sum())
        assert (st == 0) == (dev.failed_last_append() == 0)
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("S,nb,B,shared", [(5, 40, 16, 0), (300, 2000, 16, 40),
                                            (1500, 3000, 32, 100), (64, 70, 16, 8)])
def test_device_manager_matches_oracle(pkv, S, nb, B, shared):
    """Every step of the device manager equals the oracle's rules applied in
    sequence order (add_token per sequence, release of finished tables),
    starting from tables that share some blocks (reference counts > 1)."""
    rng = np.random.default_rng(7 * S + nb)
    mb = 24
    refs = obm.make_pool(nb)
    tables, lens = [], []
    for s in range(S):
        n = int(rng.integers(0, 3 * B))
        t = obm.admit(refs, n, B)
        if t is None:
            t, n = [], 0
        tables.append(t)
        lens.append(n)
    # some sequences share another's first block (a common prefix page)
    for _ in range(shared):
        a, b = (int(x) for x in rng.integers(0, S, size=2))
        if a != b and tables[a] and tables[b] and tables[b][0] != tables[a][0]:
            obm.drop_reference(refs, tables[b][0])
            obm.share_block(refs, tables[a][0])
            tables[b][0] = tables[a][0]
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    for s, t in enumerate(tables):
        if t:
            bt[s, :len(t)] = torch.tensor(t, dtype=torch.int32)
    dev = pkv.DeviceBlockManager(list(refs), B)
    assert dev.free_list() == obm.free_list(refs)
    dbt = bt.cuda()
    dlens = torch.tensor(lens, dtype=torch.int32).cuda()
    dslots = torch.empty(S, dtype=torch.int64, device="cuda")
    for step in range(12):
        if step % 4 == 3:
            done = rng.choice(S, size=max(1, S // 10), replace=False)
            ids = []
            for s in done:
                ids += tables[s]
                obm.release(refs, tables[s])
                tables[s], lens[s] = [], 0
            dev.free(torch.tensor(ids, dtype=torch.int32, device="cuda"))
            dbt[torch.as_tensor(done, device="cuda")] = -1
            dlens[torch.as_tensor(done, device="cuda")] = 0
        slots = []
        for s in range(S):
            slot, lens[s] = obm.add_token(refs, tables[s], lens[s], B)
            slots.append(slot)
        dev.append_slots(dbt, dlens, dslots)
        torch.cuda.synchronize()
        assert dslots.cpu().tolist() == slots
        assert dlens.cpu().tolist() == lens
        got_bt = dbt.cpu()
        for s in range(S):
            assert got_bt[s][got_bt[s] >= 0].tolist() == tables[s]
        assert dev.ref_counts.cpu().tolist() == refs
        assert dev.free_list() == obm.free_list(refs)
        assert dev.failed_last_append() == sum(1 for x in slots if x < 0)
    assert pkv.device_errors() == 0


def test_device_manager_exhaustion_and_bad_ids(pkv):
    dev = pkv.DeviceBlockManager([0, 0, 0], 16)
    bt = torch.full((5, 2), -1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(5, dtype=torch.int32, device="cuda")
    slots = torch.empty(5, dtype=torch.int64, device="cuda")
    dev.append_slots(bt, lens, slots)
    assert slots.tolist() == [0, 16, 32, -1, -1]
    assert dev.failed_last_append() == 2 and dev.free_list() == []
    dev.free(torch.tensor([1, 7], dtype=torch.int32, device="cuda"))   # 7 is outside the pool
    assert pkv.device_errors() & 0x8
    assert dev.free_list() == [1]
