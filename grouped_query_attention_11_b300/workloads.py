"""Seeded synthetic inputs for the GQA decode step.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the fp64 oracle are fed from it.

Shapes follow the model shapes the pages discuss:

* Llama-3-8B: 32 query heads, 8 KV heads, head_dim 128 ("Grouped Query
  Attention: Why 8 KV Heads Decide Your Batch Size", What is grouped query
  attention, exactly? and the model table); 16 sequences of about 2,300 tokens
  ("Grouped-Query Attention: How Sharing KV Heads Shrinks Inference Memory",
  Decode is a bandwidth problem).
* Llama-2/3-70B: 64 query heads, 8 KV heads, head_dim 128 ("Llama-2 70B uses 64
  query heads ...", The numbers and what they mean), 8k context.
* Group-size sweep at 64 query heads: MHA (64 KV heads), GQA-8, MQA (1 KV head)
  ("Grouped Query Attention (GQA): Efficient Multi-Head Attention", Two
  extremes).
* Ragged lengths from 500-token chats to 30,000-token retrieval prompts with an
  FP8 E4M3 cache and one scale per (sequence, KV head) ("... Shrinks Inference
  Memory", Decode is a bandwidth problem and FP8 KV cache).

Recipe (all on the host, torch CPU generator seeded per workload):

1. ``seq_lens``: the uniform length, or ``randint(lo, hi + 1)`` per sequence.
2. ``q``: N(0, 1) fp32 -> q dtype (round to nearest even).
3. per sequence b, K then V for the valid tokens of all KV heads:
   N(0, 1) fp32 -> cache dtype; for the E4M3 cache, one scale per
   (sequence, KV head) and tensor = absmax over the valid tokens / 448
   (1 when the absmax is 0), then ``(x / scale)`` cast to float8_e4m3fn.
4. cache positions t >= seq_lens[b] are filled with ``pad``: NaN (so that a
   kernel that reads past the valid prefix poisons its output) or zero.

The same recipe can run on a CUDA device (``device=``), with torch's CUDA
generator seeded the same way: same shapes and distributions, different
draws.  The benchmark uses it to set up large workloads quickly; the parity
tests draw on the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0
# 8-bit cache kinds: torch dtype, largest finite value, NaN byte used as pad
_FP8 = {"e4m3": (torch.float8_e4m3fn, E4M3_MAX, 0x7F),
        "e5m2": (torch.float8_e5m2, E5M2_MAX, 0x7F)}

_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One decode-step problem: shapes, dtypes, length mix and seed."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Smax: int
    dtype: str = "bf16"          # q / out dtype: "f16" | "bf16"
    kv: str = "same"             # "same" (cache in ``dtype``) | "e4m3" | "e5m2"
    lens: tuple = ("uniform",)   # ("uniform",) -> every seq_len = Smax,
                                 # ("fixed", L), ("ragged", lo, hi),
                                 # ("list", l0, l1, ...)
    seed: int = 1000
    page_size: int = 0           # > 0: paged cache with pages of this size
    T: int = 1                   # new tokens per sequence (> 1: q [B,Hq,T,D])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv in _FP8 else 2

    def algorithmic_bytes(self, seq_lens) -> int:
        """K+V bytes of the valid tokens + q + out (+ FP8 scales)."""
        total_tokens = int(sum(int(x) for x in seq_lens))
        kv = 2 * self.Hkv * self.D * self.kv_elem_bytes * total_tokens
        qo = 2 * self.B * self.Hq * self.T * self.D * 2
        sc = 2 * self.B * self.Hkv * 4 if self.kv in _FP8 else 0
        return kv + qo + sc

    def algorithmic_flops(self, seq_lens) -> int:
        """2*D for q.k and 2*D for p*v per (query head, valid token)."""
        total_tokens = int(sum(int(x) for x in seq_lens))
        return 4 * self.G * self.Hkv * self.D * total_tokens


# The five workload families named for this path, by what they are.
WORKLOADS = {
    "tiny_b1_h8_kv2_d64_s128_f16":
        Workload("tiny_b1_h8_kv2_d64_s128_f16", 1, 8, 2, 64, 128, "f16",
                 seed=1001),
    "llama3_8b_b16_s2300_bf16":
        Workload("llama3_8b_b16_s2300_bf16", 16, 32, 8, 128, 2300, "bf16",
                 seed=1002),
    "llama70b_b8_s8192_bf16":
        Workload("llama70b_b8_s8192_bf16", 8, 64, 8, 128, 8192, "bf16",
                 seed=1003),
    "gsweep_mha_b32_h64_kv64_s4096_bf16":
        Workload("gsweep_mha_b32_h64_kv64_s4096_bf16", 32, 64, 64, 128, 4096,
                 "bf16", seed=1004),
    "gsweep_gqa8_b32_h64_kv8_s4096_bf16":
        Workload("gsweep_gqa8_b32_h64_kv8_s4096_bf16", 32, 64, 8, 128, 4096,
                 "bf16", seed=1005),
    "gsweep_mqa_b32_h64_kv1_s4096_bf16":
        Workload("gsweep_mqa_b32_h64_kv1_s4096_bf16", 32, 64, 1, 128, 4096,
                 "bf16", seed=1006),
    "ragged_fp8_b64_h32_kv8_l500_30000":
        Workload("ragged_fp8_b64_h32_kv8_l500_30000", 64, 32, 8, 128, 30000,
                 "bf16", kv="e4m3", lens=("ragged", 500, 30000), seed=1007),
    # the 70B-shaped decode over a paged cache of 64-token pages (one page per
    # tile: every tile's page comes from the block table)
    "llama70b_paged64_b8_s8192_bf16":
        Workload("llama70b_paged64_b8_s8192_bf16", 8, 64, 8, 128, 8192,
                 "bf16", seed=1003, page_size=64),
    # the 70B-shaped step with 4 new tokens per sequence, causal within the
    # chunk (speculative decoding with 4 draft tokens)
    "llama70b_chunk4_b8_s8192_bf16":
        Workload("llama70b_chunk4_b8_s8192_bf16", 8, 64, 8, 128, 8192,
                 "bf16", seed=1003, T=4),
    # the same ragged batch with the other 8-bit cache format the pages name
    "ragged_e5m2_b64_h32_kv8_l500_30000":
        Workload("ragged_e5m2_b64_h32_kv8_l500_30000", 64, 32, 8, 128, 30000,
                 "bf16", kv="e5m2", lens=("ragged", 500, 30000), seed=1007),
}

HEADLINE = "llama70b_b8_s8192_bf16"


def draw_seq_lens(w: Workload, gen: torch.Generator) -> torch.Tensor:
    """seq_lens [B] int32, on the generator's device."""
    kind = w.lens[0]
    dev = gen.device
    if kind == "uniform":
        return torch.full((w.B,), w.Smax, dtype=torch.int32, device=dev)
    if kind == "fixed":
        return torch.full((w.B,), int(w.lens[1]), dtype=torch.int32,
                          device=dev)
    if kind == "ragged":
        lo, hi = int(w.lens[1]), int(w.lens[2])
        return torch.randint(lo, hi + 1, (w.B,), generator=gen,
                             dtype=torch.int64, device=dev).to(torch.int32)
    if kind == "list":
        vals = [int(x) for x in w.lens[1:]]
        if len(vals) != w.B:
            raise ValueError("('list', ...) needs one length per sequence")
        return torch.tensor(vals, dtype=torch.int32, device=dev)
    raise ValueError(f"unknown length mix {w.lens!r}")


def _pad_value(dtype: torch.dtype, pad: str):
    if pad == "zero":
        return 0.0
    if pad == "nan":
        return float("nan")
    raise ValueError(pad)


def make_inputs(w: Workload, *, pad: str = "nan",
                seed: Optional[int] = None, device=None) -> dict:
    """Tensors for one decode step of workload ``w``, on the host (default)
    or drawn directly on ``device``.

    Returns a dict with ``q`` [B,Hq,D], ``k``/``v`` [B,Hkv,Smax,D] (q dtype, or
    float8_e4m3fn for the FP8 cache), ``k_scale``/``v_scale`` [B,Hkv] float32
    (FP8 only, else None), ``seq_lens`` [B] int32 and ``scale`` (1/sqrt(D)).
    """
    dev = torch.device(device) if device is not None else torch.device("cpu")
    gen = torch.Generator(device=dev).manual_seed(
        w.seed if seed is None else seed)
    seq_lens = draw_seq_lens(w, gen)
    if w.B > 0 and int(seq_lens.max()) > w.Smax:
        raise ValueError("a sequence is longer than the cache")
    qdt = _DT[w.dtype]
    qshape = (w.B, w.Hq, w.D) if w.T == 1 else (w.B, w.Hq, w.T, w.D)
    q = torch.randn(qshape, generator=gen, device=dev).to(qdt)

    fp8 = w.kv in _FP8
    if fp8:
        cdt, code_max, nan_code = _FP8[w.kv]
    else:
        cdt = qdt
    shape = (w.B, w.Hkv, w.Smax, w.D)
    if fp8:
        k = torch.empty(shape, dtype=torch.uint8, device=dev)
        v = torch.empty(shape, dtype=torch.uint8, device=dev)
        k_scale = torch.ones((w.B, w.Hkv), dtype=torch.float32, device=dev)
        v_scale = torch.ones((w.B, w.Hkv), dtype=torch.float32, device=dev)
        k.fill_(nan_code if pad == "nan" else 0)
        v.fill_(nan_code if pad == "nan" else 0)
    else:
        k = torch.full(shape, _pad_value(qdt, pad), dtype=cdt, device=dev)
        v = torch.full(shape, _pad_value(qdt, pad), dtype=cdt, device=dev)
        k_scale = v_scale = None

    lens_host = seq_lens.cpu()
    for b in range(w.B):
        L = int(lens_host[b])
        for name, dst, sc in (("k", k, k_scale), ("v", v, v_scale)):
            x = torch.randn((w.Hkv, L, w.D), generator=gen, device=dev)
            if L == 0:
                continue
            if fp8:
                amax = x.abs().amax(dim=(1, 2))                 # [Hkv]
                s = torch.where(amax > 0, amax / code_max,
                                torch.ones_like(amax)).to(torch.float32)
                sc[b] = s
                codes = (x / s[:, None, None]).to(cdt)
                dst[b, :, :L, :] = codes.view(torch.uint8)
            else:
                dst[b, :, :L, :] = x.to(cdt)
    if fp8:
        k = k.view(cdt)
        v = v.view(cdt)
    out = {"q": q, "k": k, "v": v, "k_scale": k_scale, "v_scale": v_scale,
           "seq_lens": seq_lens, "scale": w.scale}
    if w.page_size > 0:
        out.update(to_pages(k, v, seq_lens, w.page_size, gen, pad))
    return out


def to_pages(k, v, seq_lens, page_size: int, gen: torch.Generator,
             pad: str = "nan") -> dict:
    """Scatter contiguous caches [B, Hkv, Smax, D] into a shuffled page pool
    [num_pages, Hkv, page_size, D] with a block table [B, max_pages] (int32,
    -1 where a sequence has no page).  A few spare pages hold the pad value."""
    B, Hkv, Smax, D = k.shape
    dev = k.device
    max_pages = -(-Smax // page_size)
    num_pages = B * max_pages + max(2, B)
    perm = torch.randperm(num_pages, generator=gen,
                          device=gen.device)[:B * max_pages]
    perm = perm.view(B, max_pages).to(torch.int32).cpu()
    fill = _pad_value(k.dtype, pad) if k.dtype.itemsize == 2 else None
    shape = (num_pages, Hkv, page_size, D)
    if fill is None:   # 8-bit codes: fill through a byte view
        kp = torch.zeros(shape, dtype=torch.uint8, device=dev)
        vp = torch.zeros(shape, dtype=torch.uint8, device=dev)
        kp.fill_(0x7F if pad == "nan" else 0)
        vp.fill_(0x7F if pad == "nan" else 0)
        kp, vp = kp.view(k.dtype), vp.view(k.dtype)
    else:
        kp = torch.full(shape, fill, dtype=k.dtype, device=dev)
        vp = torch.full(shape, fill, dtype=k.dtype, device=dev)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    lens_host = seq_lens.cpu()
    for b in range(B):
        n = -(-int(lens_host[b]) // page_size)
        for i in range(n):
            pg = int(perm[b, i])
            lo, hi = i * page_size, min((i + 1) * page_size, Smax)
            kp[pg, :, :hi - lo] = k[b, :, lo:hi]
            vp[pg, :, :hi - lo] = v[b, :, lo:hi]
            table[b, i] = pg
    return {"k": kp, "v": vp, "block_table": table.to(dev), "k_contig": k,
            "v_contig": v}


def small_variant(w: Workload, *, B: Optional[int] = None,
                  Smax: Optional[int] = None, lens=None,
                  seed: Optional[int] = None) -> Workload:
    """Same heads / dtypes as ``w`` at a size the oracle finishes quickly."""
    kw = {}
    if B is not None:
        kw["B"] = B
    if Smax is not None:
        kw["Smax"] = Smax
    if lens is not None:
        kw["lens"] = lens
    if seed is not None:
        kw["seed"] = seed
    return replace(w, name=w.name + "_small", **kw)
