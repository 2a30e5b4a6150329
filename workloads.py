"""Seeded synthetic inputs for exact ring attention.

This module is shared by the tests, the benchmark and the smoke check.  It
holds the workload shapes and the random draws only -- none of the method's
arithmetic -- so the CUDA path and the CPU oracle can be fed the same bytes
without sharing any code with each other.

Recipe (the pages print no generator, so this is the plain reading):
  * ``torch.Generator('cpu').manual_seed(seed)``; fp32 draws in the order
    q, k, v, then dO, each shaped [B, H, S, d];
  * N(0, 1) via ``randn``; U(-1, 1) via ``rand * 2 - 1``;
  * the peaked-softmax workload multiplies key rows with position
    c % 64 == 0 by 8 (in fp32, before rounding);
  * finally every tensor is rounded to bf16 (round-to-nearest-even).
The oracle receives the bf16 values widened to float64, so both sides see
identical inputs.

Grouped-query workloads draw k and v with H_kv heads.

Shapes follow the pages' worked example ("Context Parallelism" guide,
section 2, "Worked Example": 32 heads, d_k = 128, S = 128K, CP = 4) and the
smaller and peaked variants around it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    P: int
    causal: bool
    seed: int
    peaked_keys: bool = False   # key rows c % 64 == 0 scaled x8
    v_uniform: bool = False     # V ~ U(-1, 1) instead of N(0, 1)
    backward: bool = False      # also draw dO
    H_kv: int = 0               # key/value heads (grouped-query); 0 means H
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def chunk(self) -> int:
        return self.S // self.P


# The five workloads: a tiny oracle check, three forward shapes and one
# forward + backward shape.
TINY_F32 = Workload("fwd_tiny_h2_s1024_d64_p4", 1, 2, 1024, 64, 4, False, 0,
                    note="fp32 draws; GPU side takes their bf16 rounding")
FWD_CAUSAL_32K = Workload("fwd_causal_h32_s32768_d128_p4", 1, 32, 32768, 128, 4, True, 1)
FWD_CAUSAL_128K = Workload("fwd_causal_h32_s131072_d128_p4", 1, 32, 131072, 128, 4, True, 2,
                           note="the 7B MHA / 128K / CP=4 worked-example shape")
FWD_PEAKED_64K = Workload("fwd_peaked_b2_h16_s65536_d128_p8", 2, 16, 65536, 128, 8, False, 3,
                          peaked_keys=True, v_uniform=True)
FWDBWD_CAUSAL_128K = Workload("fwdbwd_causal_h32_s131072_d128_p4", 1, 32, 131072, 128, 4, True, 4,
                              backward=True)
# Grouped-query variant of the 128K shape: 32 query heads over 8 key/value
# heads (the pages' example of a model with 8 KV heads, "Ring Attention vs.
# DeepSpeed Ulysses").
FWDBWD_GQA_128K = Workload("fwdbwd_gqa_h32_kv8_s131072_d128_p4", 1, 32, 131072, 128, 4, True, 5,
                           backward=True, H_kv=8)

ALL = [TINY_F32, FWD_CAUSAL_32K, FWD_CAUSAL_128K, FWD_PEAKED_64K, FWDBWD_CAUSAL_128K,
       FWDBWD_GQA_128K]


def make(w: Workload, *, B=None, H=None, S=None, d=None, P=None, causal=None,
         seed=None, backward=None, device="cpu", keep_fp32=True, H_kv=None):
    """Draw the inputs of workload ``w`` (optionally with overridden sizes).

    Returns a dict with fp32 tensors ``q32, k32, v32`` (and ``do32``) exactly
    as drawn, and their bf16 roundings ``q, k, v`` (and ``do``), contiguous
    [B, H, S, d], plus the resolved shape fields.  With ``device="cuda"`` the
    same recipe runs with a generator on that device (a different random
    stream from the CPU one; used where only throughput is measured) and
    ``keep_fp32=False`` drops the fp32 copies.
    """
    h_given = H
    B = w.B if B is None else B
    H = w.H if H is None else H
    S = w.S if S is None else S
    d = w.d if d is None else d
    P = w.P if P is None else P
    causal = w.causal if causal is None else causal
    seed = w.seed if seed is None else seed
    backward = w.backward if backward is None else backward
    if H_kv is None:
        # the workload's own grouping, unless the query heads were overridden
        H_kv = (w.H_kv or w.H) if h_given is None else H
    g = torch.Generator(device).manual_seed(seed)
    shape = (B, H, S, d)
    kv_shape = (B, H_kv, S, d)
    out = dict(B=B, H=H, H_kv=H_kv, S=S, d=d, P=P, causal=causal, scale=1.0 / math.sqrt(d))

    def draw(name, uniform=False, peaked=False, kv=False):
        shp = kv_shape if kv else shape
        if uniform:
            x = torch.rand(shp, generator=g, dtype=torch.float32, device=device) * 2 - 1
        else:
            x = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if peaked:
            x[:, :, 0::64, :] *= 8.0
        out[name] = x.to(torch.bfloat16)
        if keep_fp32:
            out[name + "32"] = x

    draw("q")
    draw("k", peaked=w.peaked_keys, kv=True)
    draw("v", uniform=w.v_uniform, kv=True)
    if backward:
        draw("do")
    return out


def sample_rows(B: int, H: int, S: int, P: int, n_random: int = 256, seed: int = 1234,
                heads=None):
    """Flat row indices (bh * S + r) to check at sizes where whole tensors are
    too slow for the oracle: row 0, the first and last row of every chunk,
    their neighbours across each chunk boundary, and ``n_random`` rows drawn
    uniformly (seeded), for every (b, h) in ``heads`` (default: all)."""
    C = S // P
    fixed = {0, S - 1}
    for i in range(P):
        for r in (i * C, i * C + 1, (i + 1) * C - 1, (i + 1) * C - 2):
            if 0 <= r < S:
                fixed.add(r)
    g = torch.Generator("cpu").manual_seed(seed)
    rnd = torch.randint(0, S, (n_random,), generator=g).tolist()
    local = sorted(fixed | set(rnd))
    if heads is None:
        heads = range(B * H)
    rows = [bh * S + r for bh in heads for r in local]
    return torch.tensor(rows, dtype=torch.int64)
