"""Parity of paged_attn_multi_query (through the C ABI) with the fp64 oracle:
causal attention of each sequence's last q_len tokens over its paged
context, for query-head groups 1-8, head dims 64/128, block sizes 16/32,
fp16/bf16 inputs, speculative-sized and prefill-sized chunks, ragged pages
and NaN padding.  Both kernels are covered: the mma.sync kernel (16 rows
per warp) and the tcgen05 kernel (128 rows per CTA), selected through
the library's mq_tc tuning knob."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle import parallel
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


def _abs_v(case, q, qs):
    """sum_t w_t |V_t| per output element (the oracle's attention with |V|),
    for the weight-rounding term of the parity bound."""
    return lambda: orc.multi_query(q, case.k_pool, case.v_pool.abs(), case.block_tables,
                                   case.context_lens, qs, case.scale)


def _close(got, ref, case, q, qs, out_dtype=None, what=""):
    assert_attention_close(got, ref, out_dtype or case.out_dtype, what,
                           abs_weighted=_abs_v(case, q, qs), kv_dtype=case.dtype)


@pytest.fixture(params=["mma", "tc"])
def path(request, tuning):
    """Forces one multi-query kernel (the tcgen05 one needs at least 128/G
    query rows in the call; smaller calls take the mma.sync kernel)."""
    tuning(mq_tc="1" if request.param == "tc" else "0")
    return request.param


@pytest.mark.parametrize("D,B", [(128, 16), (64, 16), (128, 32), (64, 32)])
@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("q_len", [("const", 1), ("uniform", 1, 7), ("uniform", 20, 90)])
def test_matches_oracle(pkv, path, D, B, H, Hk, q_len):
    case = wl.make_case(3, S=5, lens=("uniform", 1, 300), H=H, Hk=Hk, D=D, B=B, share_blocks=2,
                        poison=True, seed=D + B + H + Hk)
    q, qs = wl.multi_query_inputs(case, q_len, seed=H + D)
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    _close(got, ref, case, q, qs, what=f"{D} {B} {H}/{Hk} {q_len}")
    assert pkv.device_errors(clear=True) == 0


@pytest.mark.parametrize("dtype,out_dtype", [(torch.float16, torch.float32),
                                             (torch.float16, torch.float16),
                                             (torch.bfloat16, torch.float32)])
def test_dtypes(pkv, path, dtype, out_dtype):
    case = wl.make_case(2, S=4, lens=("uniform", 30, 200), H=8, Hk=2, D=128, dtype=dtype,
                        out_dtype=out_dtype, poison=True)
    q, qs = wl.multi_query_inputs(case, ("uniform", 1, 40))
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    _close(got, ref, case, q, qs, out_dtype)


def test_whole_context_prefill_and_one_token_rows(pkv, path):
    """q_len = context (a prefill from scratch: row 0 sees one key, so its
    output is exactly V_0) and q_len = 1 (equals paged_attn_decode)."""
    case = wl.make_case(2, S=3, lens_override=[70, 16, 33], H=4, Hk=4, D=128,
                        out_dtype=torch.float32)
    q, qs = wl.multi_query_inputs(case, ("const", 10 ** 6))
    got = _run(pkv, case, q, qs)
    ref = orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                          case.scale)
    _close(got, ref, case, q, qs, torch.float32)
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


# ------------------------------------------------- tcgen05 kernel specifics

def _oracle(case, q, qs):
    return orc.multi_query(q, case.k_pool, case.v_pool, case.block_tables, case.context_lens, qs,
                           case.scale)


@pytest.mark.parametrize("D,B", [(128, 16), (64, 32), (128, 32), (64, 16)])
@pytest.mark.parametrize("H,Hk", [(8, 8), (8, 4), (32, 4), (16, 8)])
def test_tc_several_tiles_ragged(pkv, tuning, D, B, H, Hk):
    """Chunks of 100-400 tokens: several 128-row tiles per (sequence, kv
    head) with a ragged last tile, contexts of many 64-key tiles with a
    ragged last tile, shared pages and NaN in every row outside a context."""
    tuning(mq_tc="1")
    case = wl.make_case(2, S=4, lens=("uniform", 150, 700), H=H, Hk=Hk, D=D, B=B, share_blocks=3,
                        poison=True, seed=D * B + H)
    q, qs = wl.multi_query_inputs(case, ("uniform", 100, 400), seed=H * Hk)
    got = _run(pkv, case, q, qs)
    _close(got, _oracle(case, q, qs), case, q, qs, what=f"{D} {B} {H}/{Hk}")
    assert pkv.device_errors(clear=True) == 0


@pytest.mark.parametrize("gain", [8.0, 40.0])
def test_tc_rescale_of_wide_scores(pkv, tuning, gain):
    """Queries scaled up so that scores spread over tens of binary orders:
    the running maximum of a row grows by more than 2^8 from one key tile to
    the next, which takes the kernel's O-rescaling branch."""
    tuning(mq_tc="1")
    case = wl.make_case(2, S=3, lens=("uniform", 300, 600), H=8, Hk=2, D=128,
                        out_dtype=torch.float32, poison=True, seed=5)
    q, qs = wl.multi_query_inputs(case, ("uniform", 150, 300), seed=6)
    q = (q.float() * gain).to(case.dtype)
    got = _run(pkv, case, q, qs)
    _close(got, _oracle(case, q, qs), case, q, qs, torch.float32, f"gain {gain}")
    assert pkv.device_errors(clear=True) == 0


def test_tc_increasing_scores(pkv, tuning):
    """Key t scores t * c against every query, so each new key tile raises
    every row's maximum (rescale on every tile once the growth passes 2^8)."""
    tuning(mq_tc="1")
    case = wl.make_case(2, S=2, lens_override=[640, 517], H=4, Hk=1, D=64,
                        out_dtype=torch.float32, poison=True, seed=9)
    k = case.k_pool.float()
    for s in range(case.S):
        for t in range(int(case.context_lens[s])):
            blk = int(case.block_tables[s, t // case.B])
            k[blk, t % case.B, 0, :] = 0.05 * t
    case.k_pool = k.to(case.dtype)
    q, qs = wl.multi_query_inputs(case, ("const", 256), seed=3)
    q = q.float().abs().to(case.dtype)
    got = _run(pkv, case, q, qs)
    _close(got, _oracle(case, q, qs), case, q, qs, torch.float32)
    assert pkv.device_errors(clear=True) == 0


def test_tc_missing_pages_are_skipped(pkv, tuning):
    """A block id of -1 inside a context (a page the table does not hold)
    is skipped like in the mma.sync kernel, and flagged."""
    case = wl.make_case(2, S=3, lens_override=[400, 300, 260], H=8, Hk=4, D=128,
                        out_dtype=torch.float32, seed=12)
    q, qs = wl.multi_query_inputs(case, ("const", 200), seed=13)
    bt = case.block_tables.clone()
    bt[0, 3] = -1
    bt[1, 0] = -1
    case.block_tables = bt
    outs = {}
    for mode in ("0", "1"):
        tuning(mq_tc=mode)
        outs[mode] = _run(pkv, case, q, qs)
        assert pkv.device_errors(clear=True) & 0x1
    ref = _oracle_skip_missing(case, q, qs)
    for mode, got in outs.items():
        assert_attention_close(got, ref, torch.float32, f"mq_tc={mode}",
                               abs_weighted=lambda: _oracle_skip_missing(case, q, qs, True),
                               kv_dtype=case.dtype)


def _oracle_skip_missing(case, q, qs, abs_v=False):
    """Attention over the keys whose page the table holds (fp64, plain
    softmax): the kernels skip an out-of-range block id, so its keys drop out
    of both the scores and the sum.  abs_v: attention of |V| instead."""
    out = torch.zeros(q.shape[0], case.H, case.D, dtype=torch.float64)
    bt, G = case.block_tables, case.H // case.Hk
    for s in range(case.S):
        n = int(case.context_lens[s])
        a, b = int(qs[s]), int(qs[s + 1])
        keep = torch.tensor([t for t in range(n) if int(bt[s, t // case.B]) >= 0])
        blk = torch.tensor([int(bt[s, int(t) // case.B]) for t in keep])
        K = case.k_pool[blk, keep % case.B].double()          # [n_keep, Hk, D]
        V = case.v_pool[blk, keep % case.B].double()
        if abs_v:
            V = V.abs()
        pos = torch.arange(n - (b - a), n)                    # positions of the rows
        visible = keep[None, :] <= pos[:, None]               # [rows, n_keep]
        for h in range(case.H):
            sc = (q[a:b, h].double() @ K[:, h // G].T) * case.scale
            sc = sc.masked_fill(~visible, float("-inf"))
            out[a:b, h] = torch.softmax(sc, 1) @ V[:, h // G]
    return out.numpy()


# ------------------------------------------------- full sizes (sampled)

def _oracle_rows(case, q, qs, s, a, b):
    """Oracle rows a..b-1 of sequence s's chunk.  Causal attention of a row
    only depends on the keys up to its position, so rows a..b-1 of a q_len
    chunk over n keys are the whole (b - a)-row chunk over the first
    n - q_len + b keys."""
    q0, q1 = int(qs[s]), int(qs[s + 1])
    n = int(case.context_lens[s])
    sub_q = q[q0 + a:q0 + b]
    sub_qs = torch.tensor([0, b - a], dtype=torch.int32)
    sub_len = torch.tensor([n - (q1 - q0) + b], dtype=torch.int32)
    return orc.multi_query(sub_q, case.k_pool, case.v_pool, case.block_tables[s:s + 1],
                           sub_len, sub_qs, case.scale)


@pytest.mark.parametrize("config,k", [(2, 12), (3, 12), (4, 4)])
def test_full_size_sampled(pkv, config, k):
    """The stated workload at full size with a 256-token chunk per sequence,
    in the launch the multi-query benchmark times (the tcgen05 kernel),
    checked on sampled sequences (the longest, the shortest and random
    ones): the first rows, rows across the boundary between CTAs (or query
    tiles), middle rows and the last rows; every row finite and within
    max |V|.  (Every row of every sequence would take the fp64 oracle
    minutes per workload: the chunk's causal attention over contexts of up
    to 32K keys.)"""
    import concurrent.futures as cf
    case = wl.make_case(config)
    q, qs = wl.multi_query_inputs(case, ("const", 256))
    got = _run(pkv, case, q, qs)
    assert pkv.device_errors(clear=True) == 0
    G = case.H // case.Hk
    edge = 128 if G == 1 else 2 * (128 // G)       # first token of the second CTA or tile
    seqs = wl.sampled_seqs(case, k)
    jobs = []
    for s in seqs:
        ql = int(qs[s + 1] - qs[s])
        mid = ql // 2
        for a, b in ((0, 16), (max(0, edge - 8), min(ql, edge + 8)), (max(0, mid - 8), mid + 8),
                     (max(0, ql - 16), ql)):
            if b > a:
                jobs.append((s, a, b))
    with cf.ThreadPoolExecutor(max_workers=parallel.host_threads()) as ex:
        refs = list(ex.map(lambda j: _oracle_rows(case, q, qs, *j), jobs))
    for (s, a, b), ref in zip(jobs, refs):
        q0 = int(qs[s])
        assert_attention_close(got[q0 + a:q0 + b], ref, case.out_dtype,
                               f"config {config} seq {s} rows {a}..{b}")
    g = got.float()
    assert torch.isfinite(g).all()
    assert g.abs().max() <= case.v_pool[torch.isfinite(case.v_pool.float())].float().abs().max() + 1e-2


@pytest.mark.parametrize("H,Hk", [(8, 8), (16, 4)])
def test_tc_tile_boundaries(pkv, tuning, H, Hk):
    """Chunk lengths around the 128-row query tile and the 256-row CTA span
    (one token short, exact, one over), contexts shorter than one 64-key
    tile and contexts ending at, just before and just after a key-tile
    boundary; the whole-context prefill among them."""
    tuning(mq_tc="1")
    G = H // Hk
    qt = 128 // G                                   # tokens per query tile
    q_lens = [1, qt - 1, qt, qt + 1, 2 * qt - 1, 2 * qt, 2 * qt + 1, 3 * qt + 5]
    lens = [max(q, n) for q, n in zip(q_lens, [63, 64, 65, 127, 128, 129, 300, 512])]
    lens = [min(n, 1000) for n in lens]
    case = wl.make_case(2, S=len(lens), lens_override=lens, H=H, Hk=Hk, D=128, poison=True,
                        seed=G)
    rng = np.random.default_rng(G)
    ql = np.minimum(np.array(q_lens), np.array(lens))
    qs = torch.zeros(len(lens) + 1, dtype=torch.int32)
    qs[1:] = torch.from_numpy(np.cumsum(ql).astype(np.int32))
    q = torch.from_numpy(rng.standard_normal((int(qs[-1]), H, 128))).to(case.dtype)
    got = _run(pkv, case, q, qs)
    _close(got, _oracle(case, q, qs), case, q, qs, what=f"{H}/{Hk}")
    assert pkv.device_errors(clear=True) == 0


def test_tc_bad_q_start_is_flagged(pkv, tuning):
    """The tcgen05 kernel skips and flags a sequence whose chunk is longer
    than its context, and still answers the others."""
    tuning(mq_tc="1")
    case = wl.make_case(2, S=3, lens_override=[40, 90, 70], H=16, Hk=2, D=128,
                        out_dtype=torch.float32)
    q, qs = wl.multi_query_inputs(case, ("const", 24))     # 72 rows >= 16 tokens per tile
    bad = qs.clone()
    bad[1] = 50                        # sequence 0 would own 50 rows of a 40-token context
    out = torch.zeros(q.shape[0], case.H, case.D, dtype=torch.float32, device="cuda")
    pkv.paged_attn_multi_query(out, q.cuda(), bad.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                               case.block_tables.cuda(), case.context_lens.cuda(), case.scale,
                               50, 90)
    assert pkv.device_errors(clear=True) & 0x2
    # sequence 2 (rows 50..71 of the bad layout are sequence 1's; sequence 2 keeps its rows)
    ref = _oracle(case, q, qs)
    s2 = slice(int(qs[2]), int(qs[3]))
    assert_attention_close(out[s2], ref[s2], torch.float32, "sequence 2")
