"""The per-stream scratch: gqa_release_stream frees what the library keeps
for a stream, and the next call on that stream allocates it again and gives
the same bits; releasing a stream the library never used is a no-op."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_contract, oracle_full, to_device

pytestmark = pytest.mark.gpu


def test_release_then_reuse_stream(oracle_mod):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)
    # units split over blocks, so the call needs the split-combine scratch
    w = Workload("release", 2, 64, 8, 128, 2500, "bf16",
                 lens=("list", 2500, 1900), seed=97)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    dev = to_device(inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    a = gq.decode_inputs(dev, stream=s).clone()
    assert gq.gqa_device_errors(s) == 0
    gq.gqa_release_stream(s)
    b = gq.decode_inputs(dev, stream=s).clone()
    assert gq.gqa_device_errors(s) == 0
    torch.cuda.synchronize()
    assert_contract(a, ref, "before release")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    gq.gqa_release_stream(s)
    torch.cuda.synchronize()


def test_release_of_an_unused_stream_is_a_no_op():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    s = torch.cuda.Stream()
    gq.gqa_release_stream(s)
    gq.gqa_release_stream(s)
    assert gq.gqa_device_errors(s) == 0
