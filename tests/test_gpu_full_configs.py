"""GPU parity at the full sizes of the named workloads, in the launch
configuration the benchmark times (default grid): every output element of the
CUDA path is compared with the fp64 oracle's, under the contract tolerance
(max-abs <= 1e-2, mean-abs <= 1e-3) and the relative-L2 gate.  Cache padding
is NaN, so a read past a sequence's valid prefix would poison its row.

The group-size sweep (64 query heads over 64, 8 or 1 KV heads) is also run as
multi-head attention over the cache expanded to 64 heads (KV head j copied to
query heads jG .. jG+G-1, the repeat_kv layout of "Grouped Query Attention:
Why 8 KV Heads Decide Your Batch Size", The repeat_kv trap) at the sweep's own
B and S, and checked against the same oracle output ("Grouped Query Attention
(GQA): Efficient Multi-Head Attention", Two extremes)."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import WORKLOADS, make_inputs

from gpu_util import assert_contract, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_every_element(oracle_mod, name):
    assert torch.cuda.is_available()
    gq.gqa_set_num_ctas(0)
    w = WORKLOADS[name]
    inp = make_inputs(w, pad="nan")
    dev = to_device(inp)
    out = gq.decode_inputs(dev)
    assert gq.gqa_device_errors() == 0
    ref = oracle_full(oracle_mod, inp)
    assert_contract(out, ref, name)

    if name.startswith("gsweep_"):
        G = w.Hq // w.Hkv
        expanded = dict(dev, k=dev["k"].repeat_interleave(G, dim=1),
                        v=dev["v"].repeat_interleave(G, dim=1))
        assert expanded["k"].shape[1] == w.Hq
        mha = gq.decode_inputs(expanded)
        assert gq.gqa_device_errors() == 0
        assert_contract(mha, ref, name + " on the expanded cache")
        del expanded, mha
    del dev, out
    torch.cuda.empty_cache()
