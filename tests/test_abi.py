"""The C-ABI library loads, exports every symbol include/pagedkv.h declares,
and rejects invalid calls on the host before touching a GPU.  CPU only."""
import ctypes as C
import os
import re

import pytest
import torch

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def L():
    from paged_kv_decode_26_gb300 import build
    build.build()
    from paged_kv_decode_26_gb300._lib import lib
    return lib()


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^PKV_API\s+[^(]*?(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_entry_points():
    names = _declared_symbols()
    for n in ("paged_attn_decode", "kv_append", "swap_blocks", "pkv_decode_workspace_bytes",
              "pkv_status_string", "pkv_device_errors"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_symbols():
        assert hasattr(L, name), name


def test_binding_covers_every_declared_symbol():
    from paged_kv_decode_26_gb300._lib import SIGNATURES
    assert sorted(SIGNATURES) == _declared_symbols()


def test_exports_nothing_else():
    """Only the declared C symbols are visible (built with -fvisibility=hidden)."""
    import subprocess
    from paged_kv_decode_26_gb300._lib import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set()
    for line in out.splitlines():
        parts = line.split()
        if len(parts) == 3 and parts[1] in ("T", "W"):
            exported.add(parts[2])
    ours = {s for s in exported if s.startswith(("pkv_", "paged_", "kv_", "swap_"))}
    assert ours == set(_declared_symbols())


def test_status_strings(L):
    assert L.pkv_status_string(0) == b"PKV_OK"
    assert L.pkv_status_string(1) == b"PKV_ERR_INVALID"
    assert L.pkv_status_string(5) == b"PKV_ERR_NO_BLOCKS"
    assert L.pkv_version() >= 100


NULL = C.c_void_p(0)
FAKE = C.c_void_p(4096)  # never dereferenced: every call below fails validation first


def _decode(L, **kw):
    a = dict(out=FAKE, out_dtype=1, q=FAKE, k=FAKE, v=FAKE, kv_dtype=1, bt=FAKE, mb=4, cl=FAKE,
             S=2, H=8, Hk=8, D=128, B=16, nb=10, scale=0.1, maxc=64, split=0, ws=NULL, wsb=0,
             stream=NULL)
    a.update(kw)
    return L.paged_attn_decode(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["kv_dtype"],
                               a["bt"], a["mb"], a["cl"], a["S"], a["H"], a["Hk"], a["D"], a["B"],
                               a["nb"], a["scale"], a["maxc"], a["split"], a["ws"], a["wsb"],
                               a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(S=-1), 1),
    (dict(H=6, Hk=4), 1),
    (dict(Hk=0), 1),
    (dict(D=96), 2),
    (dict(B=8), 2),
    (dict(H=48, Hk=4), 2),
    (dict(kv_dtype=2), 2),
    (dict(out_dtype=7), 1),
    (dict(nb=-1), 1),
    (dict(nb=3, k=NULL), 1),
    (dict(mb=0), 1),
    (dict(maxc=-5), 1),
    (dict(scale=float("nan")), 1),
    (dict(q=NULL), 1),
    (dict(bt=NULL), 1),
    (dict(out=C.c_void_p(4104)), 1),   # 8-byte aligned only
    (dict(mb=1 << 27, B=32), 2),       # 2^32 tokens per table row: beyond int32 tokens
])
def test_decode_rejects_invalid_arguments(L, kw, code):
    assert _decode(L, **kw) == code
    assert L.pkv_last_error_detail()


def test_decode_zero_sequences_is_a_no_op(L):
    assert _decode(L, S=0, q=NULL, out=NULL) == 0


def test_append_rejects_invalid_arguments(L):
    assert L.kv_append(FAKE, FAKE, FAKE, FAKE, 1, FAKE, -1, 8, 128, 16, 4, NULL) == 1
    assert L.kv_append(FAKE, FAKE, FAKE, FAKE, 9, FAKE, 1, 8, 128, 16, 4, NULL) == 1
    assert L.kv_append(FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, 1, 4, 16, 4, NULL) == 2  # 8-byte rows
    assert L.kv_append(FAKE, NULL, FAKE, FAKE, 1, FAKE, 1, 8, 128, 16, 4, NULL) == 1
    assert L.kv_append(FAKE, FAKE, FAKE, FAKE, 1, FAKE, 0, 8, 128, 16, 4, NULL) == 0


def test_host_step_refuses_bad_copies_before_issuing_any(L):
    """paged_attn_decode_append_host checks its copy arguments before it
    issues anything (no device is touched: the addresses are never used)."""
    from paged_kv_decode_26_gb300.api import _Copy
    dec = (FAKE, 1, FAKE, FAKE, FAKE, 1, FAKE, 4, FAKE, 2, 8, 8, 128, 16, 10, 0.1, 64, 0, NULL, 0,
           FAKE, FAKE, FAKE, NULL)
    one = (_Copy * 1)()
    one[0].host, one[0].device, one[0].bytes = 4096, 0, 64           # no device address
    assert L.paged_attn_decode_append_host(one, 1, FAKE, 0, 0, *dec) == 1
    assert L.paged_attn_decode_append_host(None, 1, FAKE, 0, 0, *dec) == 1    # no list
    assert L.paged_attn_decode_append_host(one, -1, FAKE, 0, 0, *dec) == 1
    ok = (_Copy * 1)()
    ok[0].host, ok[0].device, ok[0].bytes = 4096, 8192, 0            # empty copy: skipped
    assert L.paged_attn_decode_append_host(ok, 1, NULL, 16, 0, *dec) == 1     # no out_host
    # more bytes back than the output holds (2 x 8 x 128 bf16 = 4096 bytes)
    assert L.paged_attn_decode_append_host(ok, 1, FAKE, 4098, 0, *dec) == 1
    assert L.pkv_last_error_detail()


def test_swap_rejects_invalid_arguments(L):
    assert L.swap_blocks(FAKE, FAKE, 24, FAKE, 1, 4, 4, NULL) == 1      # not a multiple of 16
    assert L.swap_blocks(FAKE, FAKE, 0, FAKE, 1, 4, 4, NULL) == 1
    assert L.swap_blocks(FAKE, FAKE, 32, FAKE, -1, 4, 4, NULL) == 1
    assert L.swap_blocks(NULL, FAKE, 32, FAKE, 1, 4, 4, NULL) == 1
    assert L.swap_blocks(C.c_void_p(4100), FAKE, 32, FAKE, 1, 4, 4, NULL) == 1
    assert L.swap_blocks(FAKE, FAKE, 32, FAKE, 0, 4, 4, NULL) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import paged_kv_decode_26_gb300._lib as lb
    monkeypatch.setattr(lb, "_lib", None)
    monkeypatch.setattr(lb, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lb.lib()


def test_binding_requires_cuda_tensors():
    import paged_kv_decode_26_gb300 as pkv
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.paged_attn_decode(q.clone(), q, torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16),
                              torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16),
                              torch.zeros(1, 2, dtype=torch.int32),
                              torch.ones(1, dtype=torch.int32), 0.1, 16)


def test_device_allocator_rejects_invalid_arguments(L):
    assert L.pkv_device_append_slots(FAKE, FAKE, FAKE, FAKE, 4, FAKE, -1, 16, 8, FAKE, NULL) == 1
    assert L.pkv_device_append_slots(NULL, FAKE, FAKE, FAKE, 4, FAKE, 2, 16, 8, FAKE, NULL) == 1
    assert L.pkv_device_append_slots(FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 0, 8, FAKE, NULL) == 1
    assert L.pkv_device_append_slots(FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 16, 8,
                                     C.c_void_p(4100), NULL) == 1   # slots not 8-byte aligned
    assert L.pkv_device_rebuild_free_list(FAKE, NULL, FAKE, 8, NULL) == 1
    assert L.pkv_device_free_blocks(FAKE, FAKE, FAKE, NULL, 3, 8, NULL) == 1
    assert L.pkv_device_append_slots(FAKE, FAKE, FAKE, FAKE, 4, FAKE, 0, 16, 8, FAKE, NULL) == 0


def test_multi_query_rejects_invalid_arguments(L):
    def mq(**kw):
        a = dict(out=FAKE, od=1, q=FAKE, qs=FAKE, T=8, mq=4, k=FAKE, v=FAKE, kd=1, bt=FAKE, mb=4,
                 cl=FAKE, S=2, H=8, Hk=2, D=128, B=16, nb=10, scale=0.1, mc=64, st=NULL)
        a.update(kw)
        return L.paged_attn_multi_query(a["out"], a["od"], a["q"], a["qs"], a["T"], a["mq"],
                                        a["k"], a["v"], a["kd"], a["bt"], a["mb"], a["cl"],
                                        a["S"], a["H"], a["Hk"], a["D"], a["B"], a["nb"],
                                        a["scale"], a["mc"], a["st"])
    assert mq(S=-1) == 1
    assert mq(H=6, Hk=4) == 1
    assert mq(D=96) == 2
    assert mq(qs=NULL) == 1
    assert mq(mc=1000) == 1          # beyond the block table (4 blocks of 16)
    assert mq(out=C.c_void_p(4104)) == 1
    assert mq(T=0) == 0 and mq(S=0) == 0


def test_tuning_knobs_are_explicit_and_not_read_from_the_environment(L):
    """Launch shapes change only through pkv_set_tuning: an environment
    variable of the old tuning names has no effect; a knob set and reset
    round-trips; an unknown knob is refused."""
    import paged_kv_decode_26_gb300 as pkv
    from paged_kv_decode_26_gb300 import _lib
    pkv.reset_tuning()
    base = pkv.decode_split_tokens(1, 8, 8, 128, 16, 4097)
    assert base == 512
    old = os.environ.get("PKV_DECODE_SPLIT")
    os.environ["PKV_DECODE_SPLIT"] = "2048"
    try:
        assert pkv.decode_split_tokens(1, 8, 8, 128, 16, 4097) == base
    finally:
        if old is None:
            del os.environ["PKV_DECODE_SPLIT"]
        else:
            os.environ["PKV_DECODE_SPLIT"] = old
    try:
        pkv.set_tuning(decode_split=2048)
        assert pkv.get_tuning("decode_split") == 2048
        assert pkv.decode_split_tokens(1, 8, 8, 128, 16, 4097) == 2048
    finally:
        pkv.reset_tuning()
    assert pkv.get_tuning("decode_split") is None
    assert pkv.decode_split_tokens(1, 8, 8, 128, 16, 4097) == base
    assert L.pkv_set_tuning(len(_lib.TUNE_KNOBS), 3) == 1         # PKV_ERR_INVALID
    assert L.pkv_set_tuning(-1, 3) == 1
    assert L.pkv_get_tuning(99) == _lib.TUNE_AUTO
    with pytest.raises(ValueError):
        pkv.set_tuning(no_such_knob=1)


def test_tuning_knob_names_match_the_header():
    from paged_kv_decode_26_gb300 import _lib
    text = open(HEADER).read()
    enum = dict((m.group(1).lower(), int(m.group(2)))
                for m in re.finditer(r"PKV_TUNE_(\w+)\s*=\s*(\d+)", text))
    count = enum.pop("count")
    assert enum == _lib.TUNE_KNOBS and count == len(enum)


def test_binding_rejects_host_tensors_by_name():
    """The decode bindings check every tensor before any call into the
    library; a host tensor is named in the error (no GPU needed)."""
    import torch
    import paged_kv_decode_26_gb300 as pkv
    S, H, Hk, D, B, nb = 2, 8, 2, 64, 16, 4
    t = dict(out=torch.zeros(S, H, D), q=torch.zeros(S, H, D, dtype=torch.float16),
             k_pool=torch.zeros(nb, B, Hk, D, dtype=torch.float16),
             v_pool=torch.zeros(nb, B, Hk, D, dtype=torch.float16),
             block_tables=torch.zeros(S, 2, dtype=torch.int32),
             context_lens=torch.ones(S, dtype=torch.int32))
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        pkv.paged_attn_decode(t["out"], t["q"], t["k_pool"], t["v_pool"], t["block_tables"],
                              t["context_lens"], 0.125, 1)
    new = dict(k_new=torch.zeros(S, Hk, D, dtype=torch.float16),
               v_new=torch.zeros(S, Hk, D, dtype=torch.float16),
               slot_mapping=torch.zeros(S, dtype=torch.int64))
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        pkv.paged_attn_decode_append(t["out"], t["q"], t["k_pool"], t["v_pool"],
                                     t["block_tables"], t["context_lens"], 0.125, 1,
                                     new["k_new"], new["v_new"], new["slot_mapping"])
    for step in (pkv.paged_attn_decode_append_host, pkv.HostStep):
        with pytest.raises(ValueError, match="out must be a CUDA tensor"):
            step([], torch.zeros(S, H, D), t["out"], t["q"], t["k_pool"], t["v_pool"],
                 t["block_tables"], t["context_lens"], 0.125, 1, new["k_new"], new["v_new"],
                 new["slot_mapping"])
