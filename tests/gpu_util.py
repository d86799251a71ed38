"""Shared helpers of the GPU parity tests: run the CUDA path on host inputs
and compare with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import grouped_query_attention_11_b300 as gq

# Contract tolerance for fp16/bf16 I/O with fp32 accumulation, N(0,1) inputs:
# max-abs and mean-abs error against the fp64 oracle.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
# Internal gate: relative L2 error.
REL_L2 = 1e-2
# Half an ulp of the output dtype, relative: the rounding of the final store
# alone.  Edge cases with short sequences have |out| up to ~5, where half an
# ulp of bf16 exceeds 1e-2; their bound adds this term.
HALF_ULP = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def to_device(inp: dict) -> dict:
    d = {}
    for k, v in inp.items():
        d[k] = v.cuda() if isinstance(v, torch.Tensor) else v
    return d


def run_cuda(inp_host: dict, out=None) -> torch.Tensor:
    dev = to_device(inp_host)
    res = gq.decode_inputs(dev, out=out)
    assert gq.gqa_last_launch_count() >= 1
    flags = gq.gqa_device_errors()
    assert flags == 0, f"kernel fault flags {flags:#x}"
    return res


def oracle_full(oracle_mod, inp: dict) -> np.ndarray:
    if inp["q"].dim() == 4:
        return oracle_mod.gqa_decode_chunk(inp["q"], inp["k"], inp["v"],
                                           inp["seq_lens"], inp["scale"],
                                           k_scale=inp["k_scale"],
                                           v_scale=inp["v_scale"])
    if inp.get("block_table") is not None:
        return oracle_mod.gqa_decode_paged(inp["q"], inp["k"], inp["v"],
                                           inp["block_table"], inp["seq_lens"],
                                           inp["scale"])
    return oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"], k_scale=inp["k_scale"],
                                 v_scale=inp["v_scale"])


def errors(gpu: np.ndarray, ref: np.ndarray) -> dict:
    err = np.abs(gpu - ref)
    nref = np.linalg.norm(ref)
    return {"max_abs": float(err.max()) if err.size else 0.0,
            "mean_abs": float(err.mean()) if err.size else 0.0,
            "rel_l2": float(np.linalg.norm(gpu - ref) / nref) if nref > 0
            else float(np.linalg.norm(gpu - ref))}


def assert_contract(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    """The stated tolerance, exactly: max-abs <= 1e-2, mean-abs <= 1e-3, plus
    the internal relative-L2 gate."""
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    e = errors(g, ref)
    assert e["max_abs"] <= MAX_ABS, (what, e)
    assert e["mean_abs"] <= MEAN_ABS, (what, e)
    assert e["rel_l2"] <= REL_L2, (what, e)
    return e


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    """Edge-case bound: the contract's 1e-2 plus the output dtype's half-ulp
    rounding of |ref| per element; mean and relative-L2 gates likewise."""
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    hu = HALF_ULP[gpu.dtype]
    err = np.abs(g - ref)
    bound = MAX_ABS + hu * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (what, float(err.max()), np.argwhere(bad)[:5])
    e = errors(g, ref)
    assert e["mean_abs"] <= MEAN_ABS + hu * float(np.abs(ref).mean()), (what, e)
    assert e["rel_l2"] <= REL_L2, (what, e)
    return e
