"""gqa_decode captured in a CUDA graph: replays give the eager call's bits.

A captured launch keeps the launch generation it was given, so every replay
counts its split-combine arrivals under the same tag; the block that
combines a unit leaves its counter at zero, which is what lets the next
replay start clean.  Captured after one eager call on the stream, so the
stream's scratch exists and the capture allocates nothing."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_contract, oracle_full, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # units split over several blocks: split combines and their counters
    Workload("graph_g8_split", 2, 64, 8, 128, 3000, "bf16",
             lens=("list", 3000, 1700), seed=601),
    # tensor-core kernel, cluster launch and distributed-shared-memory merge
    Workload("graph_mqa_clusters", 8, 64, 1, 128, 512, "bf16",
             lens=("uniform",), seed=602),
    # ragged 8-bit cache on the narrow-row path
    Workload("graph_fp8_ragged", 6, 32, 8, 128, 2000, "bf16", kv="e4m3",
             lens=("ragged", 1, 2000), seed=603),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_graph_replays_match_the_eager_call(oracle_mod, w):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)
    inp = make_inputs(w, pad="nan")
    dev = to_device(inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    eager = gq.decode_inputs(dev, stream=s).clone()
    assert gq.gqa_device_errors(s) == 0
    assert_contract(eager, oracle_full(oracle_mod, inp), w.name)

    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gq.decode_inputs(dev, out=out, stream=s)
    for i in range(6):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16)), i
    assert gq.gqa_device_errors(s) == 0
