"""The block manager on the GPU against the host manager (which is itself
checked against the oracle's restatement of the pages' allocator): random
decode steps (appends at and between page boundaries) and frees, compared
bit-exactly after every step -- tables, lengths, slots, reference counts and
the sorted free list."""
import numpy as np
import pytest
import torch

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
