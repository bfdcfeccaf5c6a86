"""Parity of paged_attn_multi_query (through the C ABI) with the fp64 oracle:
causal attention of each sequence's last q_len tokens over its paged
context, for query-head groups 1-8, head dims 64/128, block sizes 16/32,
fp16/bf16 inputs, speculative-sized and prefill-sized chunks, ragged pages
and NaN padding."""
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


def _run(pkv, case, q, qs, out_dtype=None):
    od = out_dtype or case.out_dtype
    out = torch.zeros(q.shape[0], case.H, case.D, dtype=od, device="cuda")
    max_q = int((qs[1:] - qs[:-1]).max()) if case.S else 0
    pkv.paged_attn_multi_query(out, q.cuda(), qs.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                               case.block_tables.cuda(), case.context_lens.cuda(), case.scale,
                               max_q, case.max_context_len)
    return out


@pytest.mark.parametrize("D,B", [(128, 16), (64, 16), (128, 32), (64, 32)])
@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("q_len", [("const", 1), ("uniform", 1, 7), ("uniform", 20, 90)])
def test_matches_oracle(pkv, D, B, H, Hk, q_len):
    case = wl.make_case(3, S=5, lens=("uniform", 1, 300), H=H, Hk=Hk, D=D, B=B, share_blocks=2,
                        poison=True, seed=D + B + H + Hk)
    q, qs = wl.multi_query_inputs(case, q_len, seed=H + D)
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    assert_attention_close(got, ref, case.out_dtype, f"{D} {B} {H}/{Hk} {q_len}")
    assert pkv.device_errors(clear=True) == 0


@pytest.mark.parametrize("dtype,out_dtype", [(torch.float16, torch.float32),
                                             (torch.float16, torch.float16),
                                             (torch.bfloat16, torch.float32)])
def test_dtypes(pkv, dtype, out_dtype):
    case = wl.make_case(2, S=4, lens=("uniform", 30, 200), H=8, Hk=2, D=128, dtype=dtype,
                        out_dtype=out_dtype, poison=True)
    q, qs = wl.multi_query_inputs(case, ("uniform", 1, 40))
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    assert_attention_close(got, ref, out_dtype)


def test_whole_context_prefill_and_one_token_rows(pkv):
    """q_len = context (a prefill from scratch: row 0 sees one key, so its
    output is exactly V_0) and q_len = 1 (equals paged_attn_decode)."""
    case = wl.make_case(2, S=3, lens_override=[70, 16, 33], H=4, Hk=4, D=128,
                        out_dtype=torch.float32)
    q, qs = wl.multi_query_inputs(case, ("const", 10 ** 6))
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    assert_attention_close(got, ref, torch.float32)
    for s in range(case.S):
        p0 = int(case.block_tables[s, 0])
        assert torch.equal(got[int(qs[s])].cpu(), case.v_pool[p0, 0].float())
    q1, qs1 = wl.multi_query_inputs(case, ("const", 1))
    got1 = _run(pkv, case, q1, qs1)
    dec = torch.empty(case.S, case.H, case.D, dtype=torch.float32, device="cuda")
    pkv.paged_attn_decode(dec, q1.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                          case.block_tables.cuda(), case.context_lens.cuda(), case.scale,
                          case.max_context_len)
    assert torch.allclose(got1, dec, rtol=1e-5, atol=2e-6)


def test_bad_q_start_is_flagged(pkv):
    case = wl.make_case(2, S=2, lens_override=[10, 20], H=2, Hk=2, D=64)
    q, qs = wl.multi_query_inputs(case, ("const", 4))
    bad = qs.clone()
    bad[1] = 30       # sequence 0 would own 30 rows of a 10-token context
    out = torch.zeros(q.shape[0], case.H, case.D, dtype=case.out_dtype, device="cuda")
    pkv.paged_attn_multi_query(out, q.cuda(), bad.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                               case.block_tables.cuda(), case.context_lens.cuda(), case.scale, 40,
                               20)
    assert pkv.device_errors(clear=True) & 0x2
