"""GPU parity under the tuning hook: every design choice that gqa_set_tuning
can turn off (L2 warm-up before the dependent-launch wait, cluster launches
of the tensor-core kernel, narrow rows for 8-bit caches) gives the oracle's
output within the stated tolerance either way, and the choice is visible
where it should be (bitwise-equal results where it only moves prefetches)."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_close, assert_contract, oracle_full, run_cuda

pytestmark = pytest.mark.gpu

ALL = (gq.GQA_TUNE_NO_L2_WARMUP | gq.GQA_TUNE_NO_CLUSTER |
       gq.GQA_TUNE_NO_NARROW_ROWS)


@pytest.fixture(autouse=True)
def _reset():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_tuning(0)
    gq.gqa_set_num_ctas(0)
    gq.gqa_set_kernel_path(0)
    yield
    gq.gqa_set_tuning(0)


CASES = [
    # name, B, Hq, Hkv, D, Smax, dtype, kv, lens
    ("g8_uniform", 4, 64, 8, 128, 640, "bf16", "same", ("uniform",)),
    # 8 units of four 128-token tiles: one tile a block, clusters of 4
    ("mqa_uniform_clusters", 8, 64, 1, 128, 512, "bf16", "same",
     ("uniform",)),
    ("fp8_g4_ragged", 6, 32, 8, 128, 900, "bf16", "e4m3", ("ragged", 1, 900)),
    ("e5m2_g8_ragged", 3, 64, 8, 64, 700, "f16", "e5m2", ("ragged", 50, 700)),
]


@pytest.mark.parametrize("flags", [0, gq.GQA_TUNE_NO_L2_WARMUP,
                                   gq.GQA_TUNE_NO_CLUSTER,
                                   gq.GQA_TUNE_NO_NARROW_ROWS, ALL])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_with_choice_turned_off(oracle_mod, case, flags):
    name, B, Hq, Hkv, D, Smax, dt, kv, lens = case
    w = Workload(name, B, Hq, Hkv, D, Smax, dt, kv=kv, lens=lens,
                 seed=7000 + CASES.index(case))
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    gq.gqa_set_tuning(flags)
    out = run_cuda(inp)
    if lens[0] == "uniform":
        assert_contract(out, ref, f"{name} tune={flags}")
    else:
        assert_close(out, ref, f"{name} tune={flags}")


def test_l2_warmup_changes_no_bit():
    """The warm-up only prefetches into L2: same plan, same bits."""
    w = Workload("warm", 4, 64, 8, 128, 900, "bf16", lens=("uniform",),
                 seed=7100)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in make_inputs(w, pad="nan").items()}
    a = gq.decode_inputs(dev).clone()
    gq.gqa_set_tuning(gq.GQA_TUNE_NO_L2_WARMUP)
    b = gq.decode_inputs(dev).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
