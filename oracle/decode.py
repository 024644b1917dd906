"""CPU fp64 oracle for decode attention: one new token per sequence over a key/value cache,
with grouped key/value heads.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this
module: only the tests and the benchmark's ``cpu_baseline`` leg use it.  It shares no code
with the CUDA path and imports nothing from the package.

What it computes.  The course page ("Week 13. GPU and FlashAttention", step 1, the bullet
on attention in decode) sets decode apart from training: every sequence has its own
cache, so the batch does not raise the arithmetic intensity, which stays near
(query heads) / (key-value heads) FLOP per byte of cache; that is the second reason for
grouped key/value heads (a smaller cache, read to more use).  The step is the plain
attention definition of ``attention.py`` with one query row:

    query head h of sequence b reads key/value head g = h // G, G = Hq / Hkv;
    keys j < cache_len[b] are visible (the rest of the cache rows are ignored);
    o[b, h] = softmax(scale * q[b, h] K[b, g]^T) V[b, g],
    lse[b, h] = logsumexp(scale * q[b, h] K[b, g]^T)   (natural log).

The reading of "which K/V head serves query head h" is the contiguous grouping
g = h // G (query heads g*G ... g*G + G - 1 share K/V head g).

Pins (CPU tests): the token at position t with a cache of t + 1 keys equals row t of the
causal full-sequence forward; grouped heads equal the same decode with the key/value heads
repeated per query head; a cache of identical keys gives the mean of V; a one-key cache
gives o = v_0 and lse = scale q.k_0; lse against scipy's logsumexp.
"""
from __future__ import annotations

import numpy as np

from .attention import forward_head


def decode(q, k, v, scale: float, cache_len=None, pairs=None):
    """q [B, Hq, d]; k, v [B, Hkv, Lmax, d]; cache_len [B] or None (all Lmax).

    Returns (o [B, Hq, dv], lse [B, Hq]) in float64.  ``pairs`` optionally restricts the
    work to a list of (b, h); other entries are NaN.
    """
    q = np.asarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of key/value heads")
    G = Hq // Hkv
    o = np.full((B, Hq, v.shape[-1]), np.nan)
    lse = np.full((B, Hq), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        L = Lmax if cache_len is None else max(0, min(int(cache_len[b]), Lmax))
        g = h // G
        # Only the first L rows of the cache belong to the sequence: attend over those
        # alone, so nothing the rest of the buffer holds (even NaN) reaches the result.
        if L == 0:  # no visible key: O = 0 and lse = -inf, as for a fully masked row
            o[b, h], lse[b, h] = 0.0, -np.inf
            continue
        keep = np.ones((1, L), dtype=bool)
        ob, lb, _ = forward_head(q[b, h][None, :], k[b, g, :L], v[b, g, :L], scale, keep)
        o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse
