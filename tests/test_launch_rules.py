"""The automatic decode launch shape, by host arithmetic only
(pkv_decode_launch_shape with GB300's device facts: 152 SMs, 227 KB of
shared memory a block, 228 KB an SM): which kernel a problem gets, its
split length, kv heads per CTA, ring depth and warps per kv head.  No GPU
is needed; the GPU tests check that every one of these shapes computes the
oracle's result."""
import pytest

import paged_kv_decode_26_gb300 as pkv

# (num_seqs, n_heads, n_kv_heads, head_dim, block_size, max_context_len)
LLAMA7B = (64, 32, 32, 128, 16, 4097)
TINY = (4, 8, 8, 64, 16, 201)
CONTINUOUS = (256, 32, 8, 128, 16, 1235)
GQA_PREFIX = (128, 32, 8, 128, 16, 32075)
LONG_CONTEXT = (16, 32, 32, 128, 32, 32769)


def shape(*args, **kw):
    return pkv.decode_launch_shape(*args, **kw)


@pytest.fixture
def knobs():
    yield pkv.set_tuning
    pkv.reset_tuning()


def test_bench_workloads():
    s = shape(*LLAMA7B)
    assert (s["kernel"], s["split_tokens"], s["heads_per_cta"], s["stages"],
            s["warps_per_token"]) == ("cuda_core", 512, 4, 3, 1)
    s = shape(*GQA_PREFIX)
    assert (s["kernel"], s["split_tokens"], s["max_splits"]) == ("tensor_core", 1024, 32)
    s = shape(*LONG_CONTEXT)
    assert (s["kernel"], s["split_tokens"], s["heads_per_cta"]) == ("cuda_core", 1024, 2)
    s = shape(*CONTINUOUS)
    assert (s["kernel"], s["split_tokens"], s["stages"], s["stream_ctas"]) == \
        ("streaming", 1248, 2, 304)


def test_one_wave_grids_take_two_warps_per_head_and_a_deeper_ring():
    # 4 sequences x 4 head groups, one split: 16 CTAs, far below one wave
    s = shape(*TINY)
    assert (s["heads_per_cta"], s["warps_per_token"], s["stages"]) == (2, 2, 8)
    assert s["threads"] == 32 * (1 + 2 * 2)
    # 4 MHA sequences of up to 2000 tokens: 256 CTAs, one wave only at two
    # CTAs per SM, so the deepest ring that keeps two (six pages, not eight)
    s = shape(4, 32, 32, 128, 16, 2000)
    assert (s["warps_per_token"], s["stages"], s["max_splits"]) == (2, 6, 4)
    assert 2 * (s["smem_bytes"] + 1024) <= 233472
    # 64 sequences: many waves, the plain shape
    assert shape(*LLAMA7B)["warps_per_token"] == 1


def test_streaming_decode_selection():
    # grouped heads, 2 to 2048 sequences, contexts up to 4096 tokens
    assert shape(128, 32, 8, 128, 16, 4096)["kernel"] == "streaming"
    assert shape(128, 32, 8, 128, 16, 4104)["kernel"] == "tensor_core"
    assert shape(2, 32, 8, 128, 16, 4096)["kernel"] == "streaming"
    assert shape(1, 32, 8, 128, 16, 4096)["kernel"] == "tensor_core"
    # from 256 sequences every group size and context length streams
    assert shape(256, 32, 8, 128, 16, 20000)["kernel"] == "streaming"
    assert shape(256, 32, 32, 128, 16, 4096)["kernel"] == "streaming"
    assert shape(255, 32, 32, 128, 16, 4096)["kernel"] == "cuda_core"
    assert shape(300, 16, 8, 128, 16, 600)["kernel"] == "streaming"     # groups of 2
    # the sequence lengths live in shared memory: at most 2048 sequences
    assert shape(2048, 32, 32, 128, 16, 4096)["kernel"] == "streaming"
    assert shape(2049, 32, 32, 128, 16, 4096)["kernel"] == "cuda_core"
    # an explicit split length selects the per-unit kernel
    s = shape(*CONTINUOUS, split_tokens=64)
    assert (s["kernel"], s["split_tokens"]) == ("tensor_core", 64)


def test_streaming_ring_takes_a_third_page_only_when_free():
    # MHA query rows are small: three pages still fit two CTAs per SM
    s = shape(256, 32, 32, 128, 16, 4096)
    assert s["stages"] == 3 and 2 * (s["smem_bytes"] + 2048) <= 233472
    # 2048 lengths in shared memory, or a group of 4's query rows, would
    # cost the second CTA: two pages
    assert shape(2048, 32, 32, 128, 16, 4096)["stages"] == 2
    assert shape(*CONTINUOUS)["stages"] == 2
    # head_dim 64: three pages would take a resident CTA of five
    assert shape(256, 32, 32, 64, 16, 4096)["stages"] == 2


def test_knobs_override_the_choice(knobs):
    knobs(decode_stream=0)
    assert shape(*CONTINUOUS)["kernel"] == "tensor_core"
    knobs(decode_stream=None, decode_wpt=1)
    s = shape(*TINY)
    assert (s["warps_per_token"], s["stages"]) == (1, 3)
    knobs(decode_wpt=None, decode_mma=1, decode_stream=1)
    assert shape(*TINY)["kernel"] == "streaming"          # MHA on the tensor-core consumer


def test_refusals():
    with pytest.raises(pkv.PagedKVError) as e:
        shape(*LLAMA7B, sm_count=0)
    assert e.value.status == 1
    with pytest.raises(pkv.PagedKVError) as e:
        shape(64, 32, 32, 96, 16, 4096)
    assert e.value.status == 2
    with pytest.raises(pkv.PagedKVError) as e:
        shape(64, 30, 8, 128, 16, 4096)
    assert e.value.status == 1
    with pytest.raises(pkv.PagedKVError) as e:
        shape(*CONTINUOUS, split_tokens=24)              # not a multiple of the block size
    assert e.value.status == 1
