"""CPU fp64 oracle for attention with dropout on the probabilities: the counter-based
generator of the keep mask, and the forward and backward that use it.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this
module: only the tests, the package's ``smoke()`` check and the benchmark's CPU legs use it.
It shares no code with the CUDA path and imports nothing from the package.

What it computes.  The reading guide (arXiv 2205.14135), "Key ideas", kernel-fusion bullet,
lists dropout among the steps fused into the one attention kernel and says nothing more.
The plainest reading, taken here, is inverted dropout on the normalised probabilities:

    O = (P o Z) V / (1 - p),   Z_ij in {0, 1},   Pr(Z_ij = 1) = 1 - p,

with P the softmax of the masked, scaled scores of ``attention.py``; the saved logsumexp
is that softmax's and does not depend on Z.  The backward does not read a stored mask: it
regenerates Z from the same counters, in the spirit of the recomputation of S and P
(answer page "How FlashAttention works for training", section 3.1).  For the loss
L = sum(dO o O), by the chain rule, with G = (dO V^T) o Z / (1 - p):

    dV = (P o Z)^T dO / (1 - p),   D_i = sum_j P_ij G_ij = sum_c dO_ic O_ic,
    dS = P o (G - D),   dQ = scale dS K,   dK = scale dS^T Q.

(D is still the row dot product of dO with the output, now the dropped output.)

The drop probability is an 8-bit threshold t, 0 <= t <= 255: p = t / 256 and Z_ij = 0
exactly when the generator's byte u_ij for that element is below t.

Generator.  Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As
Easy as 1, 2, 3", SC 2011): a 128-bit counter (x0, x1, x2, x3) and a 64-bit key (k0, k1);
ten rounds, each taking the two 64-bit products M0 x0 and M1 x2 and forming
(hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)), the key advanced by the
Weyl constants (W0, W1) between rounds.  The round structure is written once
(``_philox``) for a word width given with its constants; the tests check the 64-bit
instance against numpy's Philox bit generator and the 32-bit instance against the
published known-answer vectors.

Element to byte (the one choice of this build the pages cannot fix).  For head bh = b H + h,
query row i and key j:

    key     = (seed mod 2^32, seed div 2^32)
    counter = (kappa, rho, bh, offset)
    rho     = 8 (i >> 4) + (i & 7)          rows i and i + 8 of each 16-row block
    kappa   = 4 (j >> 5) + ((j >> 1) & 3)   keys 32a + 2c + {0, 1} + {0, 8, 16, 24}
    u_ij    = byte 2 ((i >> 3) & 1) + (j & 1) of output word (j >> 3) & 3

so one generator call yields the 16 bytes of two rows x eight keys, and u_ij depends on
(seed, offset, bh, i, j) alone, never on N or on any tiling.
"""
from __future__ import annotations

import numpy as np

from .attention import keep_mask as attention_keep_mask
from .attention import scores, softmax_rows

PHILOX32_M = (0xD2511F53, 0xCD9E8D57)
PHILOX32_W = (0x9E3779B9, 0xBB67AE85)
PHILOX64_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
PHILOX64_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)


def _mulhilo32(a, b):
    """(hi, lo) 32-bit halves of the 64-bit products of uint32-valued arrays."""
    p = np.asarray(a, np.uint64) * np.uint64(b)
    return p >> np.uint64(32), p & np.uint64(0xFFFFFFFF)


def _mulhilo64(a, b):
    """(hi, lo) 64-bit halves of the 128-bit product of Python integers."""
    p = int(a) * int(b)
    return p >> 64, p & ((1 << 64) - 1)


def _philox(ctr, key, mulhilo, mults, weyl, wmask, rounds=10):
    """Philox4xW-R on counter words ctr = (x0, x1, x2, x3) and key (k0, k1)."""
    x0, x1, x2, x3 = ctr
    k0, k1 = key
    for r in range(rounds):
        if r > 0:  # the key advances by the Weyl constants between rounds
            k0 = (k0 + weyl[0]) & wmask
            k1 = (k1 + weyl[1]) & wmask
        hi0, lo0 = mulhilo(x0, mults[0])
        hi1, lo1 = mulhilo(x2, mults[1])
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def philox4x32(ctr, key, rounds=10):
    """Philox4x32-R; counter words are uint32-valued arrays (broadcast), key two ints.
    Returns four uint64 arrays holding 32-bit words."""
    c = tuple(np.asarray(x, np.uint64) for x in ctr)
    k = (np.uint64(int(key[0]) & 0xFFFFFFFF), np.uint64(int(key[1]) & 0xFFFFFFFF))
    return _philox(c, k, _mulhilo32, PHILOX32_M,
                   (np.uint64(PHILOX32_W[0]), np.uint64(PHILOX32_W[1])),
                   np.uint64(0xFFFFFFFF), rounds)


def philox4x64(ctr, key, rounds=10):
    """Philox4x64-R on Python integers (scalar): used to pin the round structure."""
    return _philox(tuple(int(x) for x in ctr), (int(key[0]), int(key[1])), _mulhilo64,
                   PHILOX64_M, PHILOX64_W, (1 << 64) - 1, rounds)


def random_bytes(seed: int, offset: int, bh: int, n_q: int, n_k: int) -> np.ndarray:
    """The generator's byte u_ij for every query row i < n_q and key j < n_k of head bh
    (uint8 [n_q, n_k])."""
    i = np.arange(n_q, dtype=np.int64)
    j = np.arange(n_k, dtype=np.int64)
    rho = 8 * (i >> 4) + (i & 7)
    kappa = 4 * (j >> 5) + ((j >> 1) & 3)
    # One call per distinct (rho, kappa): rho indexes rows of the grid, kappa its columns.
    n_rho, n_kappa = int(rho.max()) + 1 if n_q else 0, int(kappa.max()) + 1 if n_k else 0
    R = np.arange(n_rho, dtype=np.uint64)[:, None]
    Kp = np.arange(n_kappa, dtype=np.uint64)[None, :]
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    words = philox4x32((Kp, R, np.uint64(bh), np.uint64(offset)), key)
    words = np.stack([np.broadcast_to(w, (n_rho, n_kappa)) for w in words], axis=-1)
    word = (j >> 3) & 3                              # [n_k]
    byte = 2 * ((i >> 3) & 1)[:, None] + (j & 1)[None, :]   # [n_q, n_k]
    w = words[rho[:, None], kappa[None, :], word[None, :]]
    return ((w >> (8 * byte).astype(np.uint64)) & np.uint64(0xFF)).astype(np.uint8)


def keep_drop_mask(seed: int, offset: int, bh: int, n: int, threshold: int) -> np.ndarray:
    """Z for one head (bool [n, n]): True where the element is kept."""
    if not 0 <= threshold <= 255:
        raise ValueError("threshold must be in [0, 255]")
    return random_bytes(seed, offset, bh, n, n) >= threshold


def keep_scale(threshold: int) -> float:
    """1 / (1 - p) for p = threshold / 256."""
    return 256.0 / (256.0 - threshold)


def forward_head(q, k, v, scale: float, keep: np.ndarray, z: np.ndarray, threshold: int):
    """One head: returns (O [n, dv], lse [n], P [n, n]) with O = (P o Z) V / (1 - p)."""
    s = scores(q, k, scale, keep)
    p, lse = softmax_rows(s)
    o = ((p * z) @ np.asarray(v, np.float64)) * keep_scale(threshold)
    return o, lse, p


def backward_head(q, k, v, do, scale: float, keep: np.ndarray, z: np.ndarray,
                  threshold: int):
    """One head: (dQ, dK, dV, D) of L = sum(dO o O) for the dropped forward."""
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    _, _, p = forward_head(q, k, v, scale, keep, z, threshold)
    ks = keep_scale(threshold)
    dv = (p * z).T @ do * ks
    g = (do @ v.T) * z * ks
    D = (p * g).sum(axis=1)
    ds = p * (g - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, D


def _pairs(B, H, heads):
    return heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]


def forward(q, k, v, scale: float, threshold: int, seed: int, offset: int = 0,
            causal: bool = False, blockmask=None, kv_len=None, heads=None):
    """All heads of [B, H, N, d] inputs: (O, lse) in float64 (NaN outside ``heads``)."""
    q = np.asarray(q, np.float64)
    B, H, N, _ = q.shape
    o = np.full((B, H, N, v.shape[-1]), np.nan)
    lse = np.full((B, H, N), np.nan)
    for b, h in _pairs(B, H, heads):
        keep = attention_keep_mask(N, causal, blockmask, None if kv_len is None else kv_len[b])
        z = keep_drop_mask(seed, offset, b * H + h, N, threshold)
        o[b, h], lse[b, h], _ = forward_head(q[b, h], k[b, h], v[b, h], scale, keep, z,
                                             threshold)
    return o, lse


def backward(q, k, v, do, scale: float, threshold: int, seed: int, offset: int = 0,
             causal: bool = False, blockmask=None, kv_len=None, heads=None):
    """All heads: (dQ, dK, dV, D) in float64 (NaN outside ``heads``)."""
    q = np.asarray(q, np.float64)
    B, H, N, _ = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(q.shape, np.nan)
    dv = np.full((B, H, N, v.shape[-1]), np.nan)
    D = np.full((B, H, N), np.nan)
    for b, h in _pairs(B, H, heads):
        keep = attention_keep_mask(N, causal, blockmask, None if kv_len is None else kv_len[b])
        z = keep_drop_mask(seed, offset, b * H + h, N, threshold)
        dq[b, h], dk[b, h], dv[b, h], D[b, h] = backward_head(
            q[b, h], k[b, h], v[b, h], do[b, h], scale, keep, z, threshold)
    return dq, dk, dv, D
