"""GPU parity at the full sizes of the named workloads, in the launch
configuration the benchmark times (default grid): the oracle computes a sample
of output rows one by one; every output element must be finite and no kernel
may report a fault.  The contract tolerance applies unchanged."""
import numpy as np
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import WORKLOADS, make_inputs

from gpu_util import assert_contract, to_device

pytestmark = pytest.mark.gpu


def sample_rows(w, seq_lens, n_target=96, seed=0):
    """(b, h) pairs: first/last sequence, shortest/longest sequence, every
    KV-group boundary head of those, plus a seeded random spread."""
    rng = np.random.default_rng(seed)
    n_target = min(n_target, w.B * w.Hq)
    lens = seq_lens.numpy()
    bs = {0, w.B - 1, int(lens.argmin()), int(lens.argmax())}
    pairs = set()
    for b in bs:
        for j in {0, w.Hkv - 1, w.Hkv // 2}:
            pairs.add((b, j * w.G))
            pairs.add((b, j * w.G + w.G - 1))
    while len(pairs) < n_target:
        pairs.add((int(rng.integers(w.B)), int(rng.integers(w.Hq))))
    return sorted(pairs)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_sampled_rows(oracle_mod, name):
    assert torch.cuda.is_available()
    gq.gqa_set_num_ctas(0)
    w = WORKLOADS[name]
    inp = make_inputs(w, pad="zero")
    dev = to_device(inp)
    out = gq.decode_inputs(dev)
    assert gq.gqa_device_errors() == 0
    assert torch.isfinite(out).all()
    if w.T > 1:
        # multi-token chunk: the oracle on the first and last sequences
        sel = torch.tensor([0, w.B - 1])
        ref = oracle_mod.gqa_decode_chunk(inp["q"][sel], inp["k"][sel],
                                          inp["v"][sel], inp["seq_lens"][sel],
                                          inp["scale"])
        assert_contract(out[sel.cuda()].cpu(), ref, name)
        return
    pairs = sample_rows(w, inp["seq_lens"], seed=w.seed)
    k = inp.get("k_contig", inp["k"])   # a paged cache, gathered
    v = inp.get("v_contig", inp["v"])
    ref = oracle_mod.gqa_decode_rows(inp["q"], k, v,
                                     inp["seq_lens"], inp["scale"], pairs,
                                     k_scale=inp["k_scale"],
                                     v_scale=inp["v_scale"])
    idx = torch.tensor(pairs)
    got = out[idx[:, 0].cuda(), idx[:, 1].cuda()].cpu()
    assert_contract(got, ref, name)
    del dev, out
    torch.cuda.empty_cache()
