"""The serving loop of the pages end to end through the public API: a
prefill chunk's K/V rows are written into pages and attended causally
(kv_append + paged_attn_multi_query), then decode steps append one token
each and attend (paged_attn_decode_append), the host allocator handing out
slots throughout ([SWAP] "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析":
prefill computes attention and writes KV into pages, then decode; [LAYOUT]
section 三: the block manager's append).  Pools are compared with the
oracle's appends bit for bit, outputs with the oracle's attention."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle.block_manager import append_slots as orc_append_slots
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


@pytest.mark.parametrize("H,Hk,chunk", [(8, 2, 24), (8, 8, 40)])
def test_prefill_chunk_then_decode(pkv, H, Hk, chunk):
    case = wl.make_case(3, S=4, lens=("uniform", 20, 150), H=H, Hk=Hk, D=128, poison=True,
                        seed=H + chunk, pool_extra=0.6)
    S, B, D = case.S, case.B, case.D
    gen = torch.Generator().manual_seed(chunk)
    bm = pkv.BlockManager(case.num_blocks, B, free_ids=case.free_ids)
    tables_o = [[int(x) for x in row if x >= 0] for row in case.block_tables]
    lens_o = case.context_lens.tolist()
    free_o = list(case.free_ids)
    max_cols = case.block_tables.shape[1] + (chunk + 2) // B + 2
    bt = torch.full((S, max_cols), -1, dtype=torch.int32)
    bt[:, :case.block_tables.shape[1]] = case.block_tables
    lens = case.context_lens.clone()
    k_pool, v_pool = case.k_pool.cuda(), case.v_pool.cuda()
    k_ref, v_ref = case.k_pool.clone(), case.v_pool.clone()

    # ---- prefill: `chunk` new tokens per sequence, slots one token at a time
    slot_rows = []
    for _ in range(chunk):
        slots = torch.empty(S, dtype=torch.int64)
        assert bm.append_slots(bt, lens, slots) == 0
        tables_o, lens_o, ref_slots, free_o = orc_append_slots(tables_o, lens_o, B, free_o,
                                                              case.num_blocks)
        assert slots.tolist() == ref_slots
        slot_rows.append(slots)
    slots_chunk = torch.stack(slot_rows, 1).reshape(-1)        # sequence-major rows
    k_new = torch.randn(S * chunk, Hk, D, generator=gen).to(case.dtype)
    v_new = torch.randn(S * chunk, Hk, D, generator=gen).to(case.dtype)
    pkv.kv_append(k_pool, v_pool, k_new.cuda(), v_new.cuda(), slots_chunk.cuda())
    orc.kv_append(k_ref, v_ref, k_new, v_new, slots_chunk)
    q = torch.randn(S * chunk, H, D, generator=gen).to(case.dtype)
    qs = torch.arange(0, S * chunk + 1, chunk, dtype=torch.int32)
    out = torch.empty(S * chunk, H, D, dtype=case.out_dtype, device="cuda")
    pkv.paged_attn_multi_query(out, q.cuda(), qs.cuda(), k_pool, v_pool, bt.cuda(), lens.cuda(),
                               case.scale, chunk, int(lens.max()))
    torch.cuda.synchronize()
    assert pkv.device_errors(clear=True) == 0
    assert torch.equal(k_pool.cpu().view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(v_pool.cpu().view(torch.int16), v_ref.view(torch.int16))
    ref = orc.multi_query(q, k_ref, v_ref, bt, lens, qs, case.scale)
    assert_attention_close(out, ref, case.out_dtype, "prefill chunk")

    # ---- two decode steps: append one token each and attend, in one call
    for step in range(2):
        slots = torch.empty(S, dtype=torch.int64)
        assert bm.append_slots(bt, lens, slots) == 0
        kn = torch.randn(S, Hk, D, generator=gen).to(case.dtype)
        vn = torch.randn(S, Hk, D, generator=gen).to(case.dtype)
        qd = torch.randn(S, H, D, generator=gen).to(case.dtype)
        od = torch.empty(S, H, D, dtype=case.out_dtype, device="cuda")
        pkv.paged_attn_decode_append(od, qd.cuda(), k_pool, v_pool, bt.cuda(), lens.cuda(),
                                     case.scale, int(lens.max()), kn.cuda(), vn.cuda(),
                                     slots.cuda())
        torch.cuda.synchronize()
        assert pkv.device_errors(clear=True) == 0
        orc.kv_append(k_ref, v_ref, kn, vn, slots)
        assert torch.equal(k_pool.cpu().view(torch.int16), k_ref.view(torch.int16))
        assert torch.equal(v_pool.cpu().view(torch.int16), v_ref.view(torch.int16))
        refd = orc.decode_two_pass(qd, k_ref, v_ref, bt, lens, case.scale)
        assert_attention_close(od, refd, case.out_dtype, f"decode step {step}")
