"""Seeded synthetic inputs for GQA decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through the tests and the bench) and
the CPU oracle receive the tensors made here, so that the two are compared on
identical inputs.

Recipe (stand-in for decode-time K/V caches of the GQA paper's workloads,
whose datasets and checkpoints are not used):
  * ``torch.Generator().manual_seed(1000 + index)`` draws, in this order, q
    as one ``randn(B, H, d)``, then the K cache one batch row at a time
    (``randn(G, Nmax, d)`` for b = 0..B-1), then the V cache the same way,
    then ``k_new`` and ``v_new`` (``randn(B, G, d)`` each).  All are N(0, 1)
    in fp32, then rounded to the config's dtype (bf16: round to nearest even).
  * ``torch.Generator().manual_seed(2000 + index)`` draws the ragged lengths
    with ``torch.randint(lo, hi + 1, (B,))``; fixed-length configs use L = N.
  * Cache rows at positions >= L_b are overwritten with NaN, so that any read
    of a position outside the sequence shows up in the output.

Config indices: the five listed workloads are 0..4 (the group-count sweep
points use 500 + G and the long-context case 599).

Several query tokens per sequence (``tokens`` = T > 1, the scoring pass of
speculative sampling): q is drawn as one ``randn(B, T, H, d)`` in place of
``randn(B, H, d)``, the rest as above.  The T tokens' K/V rows are the last
T cached rows, so these workloads need L_b >= T only where every token
should see something; shorter rows are the edge case of tokens that see
nothing.  Indices 604 (gqa8_t4) and 614 (mha_t4).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "sweep_names", "multi_names", "make_qkv_inputs",
           "PROJECTIONS", "make_fp8_cache"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    G: int
    d: int
    Nmax: int
    dtype: str            # "bf16" or "f32"
    lens: Tuple           # ("fixed", L) or ("uniform", lo, hi) inclusive
    index: int            # seed index
    description: str = ""
    tokens: int = 1       # query tokens per sequence

    @property
    def n_rep(self) -> int:
        return self.H // self.G

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elt(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


SWEEP_G = (1, 2, 4, 8, 16, 32, 64)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 8, 2, 64, 128, "f32", ("fixed", 128), 0,
                     "tiny GQA decode, B=1 H=8 G=2 d=64 N=128 fp32"),
    "mha": Workload("mha", 8, 32, 32, 128, 4096, "bf16", ("fixed", 4096), 1,
                    "MHA decode (G=H, 7B-like) B=8 H=G=32 d=128 N=4096 bf16"),
    "gqa8": Workload("gqa8", 16, 64, 8, 128, 8192, "bf16", ("uniform", 1, 8192), 2,
                     "GQA-8 decode (70B-like) B=16 H=64 G=8 d=128 Nmax=8192 L~U[1,8192] bf16"),
    "mqa": Workload("mqa", 64, 32, 1, 128, 2048, "bf16", ("uniform", 256, 2048), 3,
                    "MQA decode B=64 H=32 G=1 d=128 Nmax=2048 L~U[256,2048] bf16"),
    "long": Workload("long", 1, 64, 8, 128, 131072, "bf16", ("fixed", 131072), 599,
                     "long context B=1 H=64 G=8 d=128 N=131072 bf16"),
}
for _g in SWEEP_G:
    WORKLOADS[f"sweep_g{_g}"] = Workload(
        f"sweep_g{_g}", 32, 64, _g, 128, 4096, "bf16", ("fixed", 4096), 500 + _g,
        f"group-count sweep B=32 H=64 G={_g} d=128 N=4096 bf16")


WORKLOADS["gqa8_t4"] = dataclasses.replace(
    WORKLOADS["gqa8"], name="gqa8_t4", index=604, tokens=4,
    description="GQA-8 decode, 4 query tokens per sequence: B=16 T=4 H=64 G=8 d=128 Nmax=8192 "
                "L~U[1,8192] bf16")
WORKLOADS["mha_t4"] = dataclasses.replace(
    WORKLOADS["mha"], name="mha_t4", index=614, tokens=4,
    description="MHA decode, 4 query tokens per sequence: B=8 T=4 H=G=32 d=128 N=4096 bf16")


def multi_names():
    return ["gqa8_t4", "mha_t4"]


def sweep_names():
    return [f"sweep_g{g}" for g in SWEEP_G]


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def make_seq_lens(w: Workload) -> torch.Tensor:
    """Lengths L_b (int32, CPU) drawn as the recipe states."""
    if w.lens[0] == "fixed":
        return torch.full((w.B,), int(w.lens[1]), dtype=torch.int32)
    lo, hi = int(w.lens[1]), int(w.lens[2])
    g = torch.Generator().manual_seed(2000 + w.index)
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_inputs(w: Workload, seq_lens: Optional[torch.Tensor] = None,
                poison: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one decode step, on the CPU, in the workload's dtype.

    Returns q [B,H,d] ([B,T,H,d] with T = w.tokens > 1), k_cache / v_cache
    [B,G,Nmax,d], k_new / v_new [B,G,d] and seq_lens [B] (int32).  With
    ``poison`` the cache rows at positions >= L_b hold NaN.
    """
    dt = w.torch_dtype
    g = torch.Generator().manual_seed(1000 + w.index)
    qshape = (w.B, w.H, w.d) if w.tokens == 1 else (w.B, w.tokens, w.H, w.d)
    q = torch.randn(*qshape, generator=g).to(dt)
    k = torch.empty(w.B, w.G, w.Nmax, w.d, dtype=dt)
    v = torch.empty(w.B, w.G, w.Nmax, w.d, dtype=dt)
    for b in range(w.B):
        k[b] = torch.randn(w.G, w.Nmax, w.d, generator=g).to(dt)
    for b in range(w.B):
        v[b] = torch.randn(w.G, w.Nmax, w.d, generator=g).to(dt)
    k_new = torch.randn(w.B, w.G, w.d, generator=g).to(dt)
    v_new = torch.randn(w.B, w.G, w.d, generator=g).to(dt)
    if seq_lens is None:
        seq_lens = make_seq_lens(w)
    seq_lens = seq_lens.to(torch.int32).contiguous()
    if poison:
        for b in range(w.B):
            L = int(seq_lens[b])
            if 0 <= L < w.Nmax:
                k[b, :, L:, :] = float("nan")
                v[b, :, L:, :] = float("nan")
    return {"q": q, "k_cache": k, "v_cache": v, "k_new": k_new, "v_new": v_new,
            "seq_lens": seq_lens}


def make_projection(H: int, d: int, D: int, seed: int, dtype: torch.dtype) -> torch.Tensor:
    """Random per-head projection weights [H, d, D] ~ N(0, 1) for the
    mean-pool conversion, from ``manual_seed(seed)``."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(H, d, D, generator=g).to(dtype)


# Q/K/V projection layers (the step before the cache append): model width A =
# H*d as in the blog's `a = hd`, batch B rows of the decode token.
PROJECTIONS = {
    "proj_7b": dict(B=8, A=4096, H=32, G=32, d=128, seed=701),
    "proj_70b": dict(B=16, A=8192, H=64, G=8, d=128, seed=702),
}


def make_qkv_inputs(B: int, A: int, H: int, G: int, d: int, seed: int,
                    dtype: torch.dtype = torch.bfloat16) -> Dict[str, torch.Tensor]:
    """x [B,A] ~ N(0,1) and projection weights w_q [H,A,d], w_k / w_v [G,A,d]
    ~ N(0, 1/A) (so that the outputs are of unit scale), drawn in that order
    from ``manual_seed(seed)`` in fp32, then rounded to `dtype`."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, A, generator=g)
    s = A ** -0.5
    wq = torch.randn(H, A, d, generator=g) * s
    wk = torch.randn(G, A, d, generator=g) * s
    wv = torch.randn(G, A, d, generator=g) * s
    return {"x": x.to(dtype), "w_q": wq.to(dtype), "w_k": wk.to(dtype), "w_v": wv.to(dtype)}


def make_fp8_cache(w: Workload, seq_lens: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """An FP8 E4M3 cache for workload `w`: raw codes drawn uniformly over the
    254 finite codes (no value arithmetic: the bytes themselves are random),
    per-KV-head scales 2^-7 * (1 + u), u ~ U[0,1), q ~ N(0,1) bf16 [B,H,d], and
    new rows k_new / v_new ~ N(0,1) bf16.  Rows at positions >= L_b hold the
    NaN code 0x7F.  Draws from manual_seed(3000 + index) in the order q, K
    codes, V codes, k_scale, v_scale, k_new, v_new."""
    g = torch.Generator().manual_seed(3000 + w.index)
    q = torch.randn(w.B, w.H, w.d, generator=g).to(torch.bfloat16)
    def codes():
        c = torch.randint(0, 254, (w.B, w.G, w.Nmax, w.d), generator=g, dtype=torch.int32)
        c = c + (c >= 0x7F).to(torch.int32)      # skip 0x7F (NaN); 0xFF is out of the drawn range
        return c.to(torch.uint8)
    k = codes()
    v = codes()
    k_scale = (1.0 + torch.rand(w.G, generator=g)) / 128
    v_scale = (1.0 + torch.rand(w.G, generator=g)) / 128
    k_new = torch.randn(w.B, w.G, w.d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(w.B, w.G, w.d, generator=g).to(torch.bfloat16)
    if seq_lens is None:
        seq_lens = make_seq_lens(w)
    seq_lens = seq_lens.to(torch.int32).contiguous()
    for b in range(w.B):
        L = int(seq_lens[b])
        if 0 <= L < w.Nmax:
            k[b, :, L:] = 0x7F
            v[b, :, L:] = 0x7F
    return {"q": q, "k_cache": k, "v_cache": v, "k_scale": k_scale.float(), "v_scale": v_scale.float(),
            "k_new": k_new, "v_new": v_new, "seq_lens": seq_lens}
