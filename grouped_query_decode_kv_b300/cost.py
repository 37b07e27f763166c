"""Byte and flop counts of one GQA decode step (host-side arithmetic only).

The memory/arithmetic accounting follows fogdragon's CSDN blog on MQA/GQA,
section "MQA 的推导": per decode step the cache term of the memory traffic is
b*h*n*d for MHA, is divided by h when K/V are shared by all heads (MQA), and
scales with the number of KV groups g for GQA, while the arithmetic
(q.K and weights.V, b*h*n*d multiply-adds each) does not change.  The GQA
paper, section 2.2, states the same: going from H KV heads to one cuts the
cache, and the data loaded per step, by a factor H.
"""
from __future__ import annotations

from typing import Iterable

__all__ = ["kv_cache_bytes", "kv_bytes_per_token", "decode_attention_bytes",
           "decode_attention_flops", "kv_append_bytes", "cache_ratio", "qkv_project_bytes", "qkv_project_flops"]


def kv_cache_bytes(B: int, G: int, N: int, d: int, elt: int, layers: int = 1) -> int:
    """Bytes held by the K and V caches of ``layers`` attention layers:
    2 * layers * B * G * N * d * elt."""
    return 2 * layers * B * G * N * d * elt


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elt: int) -> int:
    """Cache bytes one timestep adds across a whole model."""
    return kv_cache_bytes(1, kv_heads, 1, head_dim, elt, layers=layers)


def cache_ratio(H: int, G: int) -> int:
    """How many times smaller the GQA-G cache is than the MHA one (H / G)."""
    if H % G:
        raise ValueError("H must be a multiple of G")
    return H // G


def decode_attention_bytes(seq_lens: Iterable[int], H: int, G: int, d: int, elt: int, tokens: int = 1) -> int:
    """Algorithmic HBM bytes of one decode-attention call: every cached K and V
    row of every sequence read once, q read once and out written once (with
    ``tokens`` query tokens per sequence, q and out hold tokens * H rows per
    sequence; the cache is still read once)."""
    lens = [int(x) for x in seq_lens]
    B = len(lens)
    return 2 * G * sum(lens) * d * elt + 2 * B * tokens * H * d * elt


def decode_attention_flops(seq_lens: Iterable[int], H: int, d: int, tokens: int = 1) -> int:
    """Flops of one decode-attention call: q.K and weights.V, 2*d flops per
    (head, visible position) each.  With several tokens, token t of a run of
    T sees min(L, L - T + 1 + t) positions."""
    vis = 0
    for x in seq_lens:
        L = int(x)
        vis += sum(max(0, min(L, L - tokens + 1 + t)) for t in range(tokens))
    return 4 * H * d * vis


def kv_append_bytes(B: int, G: int, d: int, elt: int) -> int:
    """Algorithmic bytes of one cache append: the new K and V rows read, then
    written into the caches."""
    return 2 * 2 * B * G * d * elt


def qkv_project_bytes(B: int, A: int, H: int, G: int, d: int, elt: int = 2) -> int:
    """Algorithmic bytes of the Q/K/V projections of one decode step (the
    blog's per-line M terms 'had+ba' for Q and, with G KV heads, 'gad+ba' for
    K and V): the weights read once, x read, q/k/v written."""
    return (H + 2 * G) * A * d * elt + B * A * elt + B * (H + 2 * G) * d * elt


def qkv_project_flops(B: int, A: int, H: int, G: int, d: int) -> int:
    """2 flops per multiply-add: 2*B*A*(H + 2G)*d."""
    return 2 * B * A * (H + 2 * G) * d
