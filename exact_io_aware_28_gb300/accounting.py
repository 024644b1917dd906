"""FLOP and byte accounting for the attention hot path (host logic only).

FLOP convention: 4*N^2*d per head for the forward (two N x N x d matrix
products) and 10*N^2*d per head for the backward (five products, the score
recomputation included), halved for causal attention.  For a block-sparse
mask only the kept 128 x 128 blocks count.

Byte figures are the algorithmic minimum: every input read once and every
output written once.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

BLOCK = 128


def kept_pairs(N: int, causal: bool, blockmask: Optional[np.ndarray]) -> float:
    """Number of (query, key) pairs that count toward the FLOP convention, per head.

    Dense: N^2 (N^2 / 2 for causal).  Block-sparse: the sum over kept blocks of
    their row count times column count (exact for a ragged last block).
    """
    if blockmask is None:
        return N * N / 2.0 if causal else float(N * N)
    bm = np.asarray(blockmask).astype(bool)
    nb = bm.shape[0]
    sizes = np.array([min(BLOCK, N - b * BLOCK) for b in range(nb)], dtype=np.float64)
    pairs = float((bm * np.outer(sizes, sizes)).sum())
    return pairs / 2.0 if causal else pairs


def flops(B: int, H: int, N: int, d: int, causal: bool = False,
          blockmask: Optional[np.ndarray] = None) -> dict:
    pairs = kept_pairs(N, causal, blockmask)
    fwd = 4.0 * pairs * d * B * H
    bwd = 10.0 * pairs * d * B * H
    return {"fwd": fwd, "bwd": bwd, "fwd_bwd": fwd + bwd}


def dense_equivalent_flops(B: int, H: int, N: int, d: int) -> dict:
    return flops(B, H, N, d, False, None)


def score_matrix_bytes(n: int, heads: int = 1, bytes_per_element: int = 2) -> int:
    """Bytes of the materialised n x n score matrix over ``heads`` heads."""
    return n * n * heads * bytes_per_element


def memory_saving_ratio(n: int, d: int) -> float:
    """Size of the n x n score matrix over the size of the n x d output."""
    return (n * n) / float(n * d)


def ridge_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """Arithmetic intensity (FLOP/byte) at which compute and memory time are equal."""
    return peak_flops / bandwidth_bytes


def intensity(flop_count: float, byte_count: float) -> float:
    return flop_count / byte_count


def preprocess_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> int:
    """D = rowsum(dO o O) and zeroing of the fp32 dQ accumulator.

    Reads O and dO, writes D (fp32 per row) and the fp32 accumulator.
    """
    rows = B * H * N
    return rows * d * elem * 2 + rows * 4 + rows * d * 4


def dq_convert_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> int:
    """dQ = bf16(scale * dQacc): reads the fp32 accumulator, writes dQ."""
    rows = B * H * N
    return rows * d * 4 + rows * d * elem


def fwd_min_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> int:
    """Q, K, V read once; O and lse written once."""
    rows = B * H * N
    return rows * d * elem * 4 + rows * 4


def bwd_min_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> int:
    """Q, K, V, O, dO, lse read once; dQ, dK, dV written once."""
    rows = B * H * N
    return rows * d * elem * 8 + rows * 4


def decode_flops(Hq: int, d: int, cache_len) -> float:
    """Decode FLOPs: per query head and visible key, a length-d dot product for the score
    and a length-d multiply-add into the output (2*d + 2*d)."""
    return 4.0 * d * Hq * float(np.asarray(cache_len, dtype=np.float64).sum())


def decode_bytes(Hq: int, Hkv: int, d: int, cache_len, elem: int = 2) -> float:
    """Algorithmic bytes of one decode step: the visible K and V rows read once, q read,
    o (elem bytes) and lse (4 bytes) written."""
    L = float(np.asarray(cache_len, dtype=np.float64).sum())
    B = len(np.asarray(cache_len))
    return 2.0 * L * Hkv * d * elem + B * Hq * (d * elem + d * elem + 4)


def fp8_encode_bytes(B: int, H: int, N: int, d: int) -> float:
    """Algorithmic bytes of encoding Q, K and V to e4m3: each bf16 element read once, each
    code written once (V^T padded to a multiple of 128 keys), plus the fp32 scales."""
    nb = (N + BLOCK - 1) // BLOCK
    rows = B * H * N * d
    return 3.0 * rows * 2 + 2.0 * rows + B * H * d * nb * BLOCK + 4.0 * B * H * (2 * nb + 1)
