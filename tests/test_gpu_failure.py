"""Failure detection on the GPU without a GPU fault: every pipeline wait in the
decode kernels has a time limit, after which the kernel records the give-up
(bit 0 of gqa_device_errors), stops waiting and finishes.  A test-only limit of
zero makes the first wait that is not already complete give up, so a wait runs
out without withholding any work, nothing faults and nothing hangs.

After such a call the stream's split-combine counters may hold arrivals that
never completed; the next call on the same stream must still be correct (each
launch tags its counts with a generation of its own)."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_contract, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _limits():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)
    gq.gqa_set_wait_limit_ns(-1)
    yield
    gq.gqa_set_wait_limit_ns(-1)
    gq.gqa_set_num_ctas(0)


# Units split over several blocks (split combines and their counters), a
# ragged 8-bit batch on the narrow-row path, and the tensor-core kernel.
CASES = [
    Workload("giveup_bf16_split", 2, 64, 8, 128, 3000, "bf16",
             lens=("list", 3000, 1700), seed=91),
    Workload("giveup_fp8_ragged", 6, 32, 8, 128, 2000, "bf16", kv="e4m3",
             lens=("ragged", 1, 2000), seed=92),
    # the tensor-core kernel (64 rows per KV head): units split over a
    # cluster's four blocks and merged through distributed shared memory
    # (every thread still reaches the cluster barriers after a give-up), and
    # ragged units split over plain blocks (global split combine)
    Workload("giveup_mqa_clusters", 8, 64, 1, 128, 512, "bf16",
             lens=("uniform",), seed=93),
    Workload("giveup_mqa_split", 2, 64, 1, 128, 1500, "bf16",
             lens=("list", 1500, 777), seed=94),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_wait_give_up_is_reported_and_the_stream_recovers(oracle_mod, w):
    inp = make_inputs(w, pad="nan")
    dev = to_device(inp)
    ref = oracle_full(oracle_mod, inp)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    # a normal call first: the stream's scratch exists and is in use
    out0 = gq.decode_inputs(dev, stream=stream)
    assert gq.gqa_device_errors(stream) == 0
    assert_contract(out0, ref, w.name + " before")

    gq.gqa_set_wait_limit_ns(0)
    gq.decode_inputs(dev, out=torch.empty_like(out0), stream=stream)
    gq.gqa_set_wait_limit_ns(-1)
    # the next call on the same stream, with no query in between: it must not
    # pick up the counts the given-up call left behind
    out1 = gq.decode_inputs(dev, out=torch.empty_like(out0), stream=stream)
    flags = gq.gqa_device_errors(stream)
    assert flags & 1, f"no wait gave up (flags {flags:#x})"
    assert_contract(out1, ref, w.name + " after a give-up")
    # the query cleared the flag; later calls are clean
    out2 = gq.decode_inputs(dev, out=torch.empty_like(out0), stream=stream)
    assert gq.gqa_device_errors(stream) == 0
    assert torch.equal(out2.view(torch.int16), out0.view(torch.int16))


def test_give_up_on_every_call_of_a_loop_finishes():
    """Many given-up calls in a row (each one with every wait giving up at
    once) all return; the stream is usable afterwards."""
    w = CASES[0]
    dev = to_device(make_inputs(w, pad="zero"))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    gq.gqa_set_wait_limit_ns(0)
    for _ in range(20):
        gq.decode_inputs(dev, stream=stream)
    gq.gqa_set_wait_limit_ns(-1)
    assert gq.gqa_device_errors(stream) & 1
    assert gq.gqa_device_errors(stream) == 0
