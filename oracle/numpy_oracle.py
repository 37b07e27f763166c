"""Second, independent fp64 oracle for GQA decode attention, in NumPy.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  It is written without the
n_rep repeat used by the C oracle: the H query heads are reshaped into G
groups of n_rep contiguous heads (GQA paper, section 2.2; 2kiu.com explainer,
section 3.1) and each group attends to its own KV head through a grouped
einsum.  It serves only to cross-check the C oracle on small shapes.
"""
from __future__ import annotations

import numpy as np


def decode_attention_grouped(q, k, v, seq_lens, scale):
    """q [B,H,d], k/v [B,G,N,d] float64, seq_lens [B] -> out [B,H,d] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, d = q.shape
    G, N = k.shape[1], k.shape[2]
    assert H % G == 0
    n_rep = H // G
    qg = q.reshape(B, G, n_rep, d)
    out = np.zeros((B, G, n_rep, d), dtype=np.float64)
    for b in range(B):
        L = int(min(max(int(seq_lens[b]), 0), N))
        if L == 0:
            continue
        logits = np.einsum("grd,gnd->grn", qg[b], k[b, :, :L, :]) * scale
        logits -= logits.max(axis=-1, keepdims=True)
        w = np.exp(logits)
        w /= w.sum(axis=-1, keepdims=True)
        out[b] = np.einsum("grn,gnd->grd", w, v[b, :, :L, :])
    return out.reshape(B, H, d)
