"""GPU parity of the cache-append step (gqa_append_kv) with the oracle:
bit-exact codes, scales and lengths (every code is decided in fp32 on both
sides), then the decode step over the appended cache."""
import numpy as np
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_contract, oracle_full

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "f16": torch.float16,
       "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _case(kind, in_dt, seed, B, Hkv, Smax, D, lens, scale_mul):
    g = torch.Generator().manual_seed(seed)
    kn = torch.randn((B, Hkv, D), generator=g).to(_DT[in_dt])
    vn = (3.0 * torch.randn((B, Hkv, D), generator=g)).to(_DT[in_dt])
    seq = torch.tensor(lens, dtype=torch.int32)
    if kind in ("bf16", "f16"):
        kc = torch.randn((B, Hkv, Smax, D), generator=g).to(_DT[kind])
        vc = torch.randn((B, Hkv, Smax, D), generator=g).to(_DT[kind])
        return kn, vn, kc, vc, seq, None, None
    kc = torch.randn((B, Hkv, Smax, D), generator=g).mul(50).to(_DT[kind])
    vc = torch.randn((B, Hkv, Smax, D), generator=g).mul(50).to(_DT[kind])
    ks = torch.rand((B, Hkv), generator=g).add(0.5).mul(scale_mul).float()
    vs = torch.rand((B, Hkv), generator=g).add(0.5).mul(scale_mul).float()
    if scale_mul == 0.0:
        ks[0, 0] = -1.0                # an unset scale is any value <= 0
    return kn, vn, kc, vc, seq, ks, vs


CASES = [
    # kind, in dtype, B, Hkv, Smax, D, lens, scale multiplier
    ("bf16", "bf16", 3, 2, 40, 64, (5, 0, 39), None),
    ("f16", "f16", 2, 8, 100, 128, (99, 17), None),
    ("e4m3", "bf16", 3, 2, 40, 64, (5, 0, 39), 10.0),
    ("e4m3", "bf16", 3, 2, 40, 64, (5, 0, 39), 1e-5),
    ("e4m3", "f16", 3, 2, 40, 128, (5, 0, 39), 0.0),
    ("e5m2", "bf16", 3, 2, 40, 64, (5, 0, 39), 1e-5),
    ("e5m2", "f16", 2, 4, 70, 128, (3, 66), 10.0),
    ("e4m3", "bf16", 8, 8, 2048, 128, (2047, 0, 1, 1000, 2000, 64, 65, 512),
     1e-6),
]


@pytest.mark.parametrize("case", CASES,
                         ids=[f"{c[0]}_{c[1]}_{c[7]}_{c[2]}x{c[4]}"
                              for c in CASES])
def test_append_matches_oracle_bitwise(oracle_mod, case):
    kind, in_dt, B, Hkv, Smax, D, lens, sm = case
    kn, vn, kc, vc, seq, ks, vs = _case(kind, in_dt, 50 + CASES.index(case),
                                        B, Hkv, Smax, D, lens, sm)
    k2, v2, ks2, vs2, lens2, flags = oracle_mod.append_kv(
        kn, vn, kc, vc, seq, k_scale=ks, v_scale=vs)
    assert flags == 0
    d = {n: t.cuda() for n, t in (("kn", kn), ("vn", vn), ("kc", kc),
                                  ("vc", vc), ("seq", seq))}
    dks = ks.cuda() if ks is not None else None
    dvs = vs.cuda() if vs is not None else None
    gq.gqa_append_kv(d["kn"], d["vn"], d["kc"], d["vc"], d["seq"],
                     k_scale=dks, v_scale=dvs)
    assert gq.gqa_last_launch_count() == 1
    assert gq.gqa_device_errors() == 0
    raw = torch.uint8 if kind in ("e4m3", "e5m2") else torch.int16
    np_raw = np.uint8 if raw == torch.uint8 else np.int16
    assert np.array_equal(d["kc"].cpu().view(raw).numpy(), k2.view(np_raw))
    assert np.array_equal(d["vc"].cpu().view(raw).numpy(), v2.view(np_raw))
    assert np.array_equal(d["seq"].cpu().numpy(), lens2)
    if ks is not None:
        assert np.array_equal(dks.cpu().numpy(), ks2)
        assert np.array_equal(dvs.cpu().numpy(), vs2)


def test_append_full_cache_sets_the_error_bit():
    kn, vn, kc, vc, seq, _, _ = _case("bf16", "bf16", 77, 3, 2, 40, 64,
                                      (40, 2, -3), None)
    d = {n: t.cuda() for n, t in (("kn", kn), ("vn", vn), ("kc", kc),
                                  ("vc", vc), ("seq", seq))}
    gq.gqa_append_kv(d["kn"], d["vn"], d["kc"], d["vc"], d["seq"])
    assert gq.gqa_device_errors() & 4
    assert d["seq"].cpu().tolist() == [40, 3, 1]
    assert torch.equal(d["kc"][0].cpu(), kc[0])


def test_append_then_decode(oracle_mod):
    """A decode step after the append sees the new token: the GPU result on
    the GPU-appended FP8 cache matches the oracle on the oracle-appended
    one."""
    w = Workload("app", 4, 32, 8, 128, 600, "bf16", kv="e4m3",
                 lens=("list", 599, 0, 300, 450), seed=78)
    inp = make_inputs(w, pad="zero")
    g = torch.Generator().manual_seed(79)
    kn = (4 * torch.randn((4, 8, 128), generator=g)).to(torch.bfloat16)
    vn = torch.randn((4, 8, 128), generator=g).to(torch.bfloat16)
    k2, v2, ks2, vs2, lens2, _ = oracle_mod.append_kv(
        kn, vn, inp["k"], inp["v"], inp["seq_lens"], k_scale=inp["k_scale"],
        v_scale=inp["v_scale"])
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t)
         for n, t in inp.items()}
    gq.gqa_append_kv(kn.cuda(), vn.cuda(), d["k"], d["v"], d["seq_lens"],
                     k_scale=d["k_scale"], v_scale=d["v_scale"])
    out = gq.decode_inputs(d)
    assert gq.gqa_device_errors() == 0
    ref_inp = dict(inp, k=torch.from_numpy(k2).view(torch.float8_e4m3fn),
                   v=torch.from_numpy(v2).view(torch.float8_e4m3fn),
                   k_scale=torch.from_numpy(ks2), v_scale=torch.from_numpy(vs2),
                   seq_lens=torch.from_numpy(lens2))
    assert_contract(out, oracle_full(oracle_mod, ref_inp), "append+decode")
