"""Batched decode (pkv_decode_batched_plan + paged_attn_decode_batched):
independent problems with their own pools, tables and lengths in one
launch give, problem by problem, exactly what paged_attn_decode /
paged_attn_decode_append give (same launch shape: bit for bit), and match
the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_decode_26_gb300 import workloads as wl
from tests.parity import assert_attention_close

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


def _problems(config, sizes, H, Hk, seed):
    cases = []
    for i, S in enumerate(sizes):
        if S == 0:
            cases.append(None)
            continue
        cases.append(wl.make_case(config, S=S, lens=("uniform", 1, 300), H=H, Hk=Hk, D=128,
                                  poison=True, seed=seed + i))
    return cases


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("H,Hk,split", [(8, 8, 64), (8, 8, 512), (16, 4, 64), (16, 4, 0)])
def test_batched_equals_single_calls(pkv, tuning, H, Hk, split):
    tuning(decode_hpc="2", decode_wpt="1")  # one launch shape for both ways
    sizes = [3, 0, 5, 1, 4]
    cases = _problems(2, sizes, H, Hk, seed=H + split)
    max_ctx = max(int(c.context_lens.max()) for c in cases if c is not None)
    split_used = split or pkv.decode_split_tokens(sum(sizes), H, Hk, 128, 16, max_ctx)
    problems, singles = [], []
    for c in cases:
        if c is None:
            e = torch.empty(0, H, 128, dtype=torch.bfloat16, device="cuda")
            problems.append(dict(out=e, q=e, k_pool=torch.zeros(1, 16, Hk, 128, dtype=torch.bfloat16,
                                                                device="cuda"),
                                 v_pool=torch.zeros(1, 16, Hk, 128, dtype=torch.bfloat16,
                                                    device="cuda"),
                                 block_tables=torch.zeros(0, 1, dtype=torch.int32, device="cuda"),
                                 context_lens=torch.zeros(0, dtype=torch.int32, device="cuda")))
            singles.append(None)
            continue
        d = {k: getattr(c, k).cuda() for k in ("q", "k_pool", "v_pool", "block_tables",
                                              "context_lens")}
        out = torch.full((c.S, H, 128), float("nan"), dtype=c.out_dtype, device="cuda")
        problems.append(dict(out=out, **d))
        ref = torch.empty_like(out)
        pkv.paged_attn_decode(ref, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                              d["context_lens"], c.scale, max_ctx, split_tokens=split_used)
        singles.append(ref)
    batch = pkv.DecodeBatch(problems, cases[0].scale, max_ctx, split_tokens=split_used)
    batch.run()
    torch.cuda.synchronize()
    assert pkv.device_errors(clear=True) == 0
    for c, pr, ref in zip(cases, problems, singles):
        if c is None:
            continue
        assert torch.equal(_bits(pr["out"]), _bits(ref))
        oracle = orc.decode_two_pass(c.q, c.k_pool, c.v_pool, c.block_tables, c.context_lens,
                                     c.scale)
        assert_attention_close(pr["out"], oracle, c.out_dtype)


def test_batched_append_and_rerun(pkv, tuning):
    """Problems with a fused append and problems without in one batch; a
    second run reads the buffers' new contents (queries changed)."""
    tuning(decode_hpc="2")
    H, Hk, D = 16, 4, 128
    cases = [wl.make_case(2, S=S, lens=("uniform", 20, 200), H=H, Hk=Hk, D=D, seed=70 + i)
             for i, S in enumerate([4, 6, 2])]
    problems, pools_ref = [], []
    gen = torch.Generator().manual_seed(5)
    for i, c in enumerate(cases):
        bm = pkv.BlockManager(c.num_blocks, c.B, free_ids=c.free_ids)
        bt = c.block_tables.clone()
        need = int(((c.context_lens + 1 + c.B - 1) // c.B).max())
        if need > bt.shape[1]:
            bt = torch.cat([bt, torch.full((c.S, need - bt.shape[1]), -1, dtype=torch.int32)], 1)
        lens = c.context_lens.clone()
        pr = dict(out=torch.empty(c.S, H, D, dtype=c.out_dtype, device="cuda"), q=c.q.cuda(),
                  k_pool=c.k_pool.cuda(), v_pool=c.v_pool.cuda(), block_tables=bt.cuda(),
                  context_lens=lens.cuda())
        k, v = c.k_pool.clone(), c.v_pool.clone()
        if i != 1:                                   # problem 1 appends nothing
            slots = torch.empty(c.S, dtype=torch.int64)
            bm.append_slots(bt, lens, slots)
            kn = torch.randn(c.S, Hk, D, generator=gen).to(c.dtype)
            vn = torch.randn(c.S, Hk, D, generator=gen).to(c.dtype)
            pr.update(block_tables=bt.cuda(), context_lens=lens.cuda(), k_new=kn.cuda(),
                      v_new=vn.cuda(), slot_mapping=slots.cuda())
            orc.kv_append(k, v, kn, vn, slots)
        pools_ref.append((k, v, bt, lens))
        problems.append(pr)
    max_ctx = max(int(p_["context_lens"].max()) for p_ in problems)
    batch = pkv.DecodeBatch(problems, cases[0].scale, max_ctx)
    for run in range(2):
        if run == 1:
            for pr in problems:
                pr["q"].mul_(-1.0)                    # new contents, same storage
        batch.run()
        torch.cuda.synchronize()
        assert pkv.device_errors(clear=True) == 0
        for c, pr, (k, v, bt, lens) in zip(cases, problems, pools_ref):
            assert torch.equal(pr["k_pool"].cpu().view(torch.int16), k.view(torch.int16))
            assert torch.equal(pr["v_pool"].cpu().view(torch.int16), v.view(torch.int16))
            ref = orc.decode_two_pass(pr["q"].cpu(), k, v, bt, lens, c.scale)
            assert_attention_close(pr["out"], ref, c.out_dtype, f"run {run}")
