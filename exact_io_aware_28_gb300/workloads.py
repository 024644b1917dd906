"""Seeded synthetic workloads for the attention hot path.

This module only draws random numbers and lays them out.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any of the method.

The five workloads follow the shapes the FlashAttention pages talk about:
a tiny fp32 correctness case, a GPT-2-shaped causal case, a BERT-large-shaped
case with key padding (FlashAttention reading guide, "Results": BERT-large at
sequence length 512, GPT-2 at 1K), a long-context causal case, and a
block-sparse case with a 128x128 block mask ("Extension: block-sparse
FlashAttention", mask M in {0,1}^{N/B_r x N/B_c}).  The datasets behind those
results are not used: i.i.d. N(0,1) inputs of the same shapes stand in.

Draw order for a seed: Q, K, V, dO (each ``randn(B, H, N, d)`` in fp32 from one
``torch.Generator('cpu')``), then the per-sequence key lengths or the block
mask.  bf16 workloads round the fp32 draws to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

BLOCK = 128  # block-mask granularity (rows and columns of one mask entry)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "fp32" or "bf16"
    causal: bool = False
    padded: bool = False        # per-sequence key lengths in [128, N]
    block_sparse: bool = False  # 128x128 block mask, diagonal kept, rest Bernoulli(p)
    keep_prob: float = 0.25
    q_head0_mult: float = 1.0   # multiply head 0 of Q (power of two: exact in bf16)
    drop_threshold: int = 0     # dropout on P with probability drop_threshold / 256
    drop_seed: int = 0          # the generator's 64-bit seed (an input, like the data)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def describe(self) -> str:
        extra = []
        if self.causal:
            extra.append("causal")
        if self.padded:
            extra.append("key-padding")
        if self.block_sparse:
            extra.append(f"block-sparse p={self.keep_prob}")
        if self.drop_threshold:
            extra.append(f"dropout {self.drop_threshold}/256")
        return (f"{self.name}: B={self.B} H={self.H} N={self.N} d={self.d} "
                f"{self.dtype}" + (" " + " ".join(extra) if extra else ""))


# The five workloads: tiny fp32 correctness case, GPT-2 shape, BERT-large shape,
# long context, block-sparse.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 128, 64, "fp32"),
    "gpt2_causal": Workload("gpt2_causal", 4, 12, 1024, 64, "bf16", causal=True,
                            q_head0_mult=4.0),
    "bert_padded": Workload("bert_padded", 16, 16, 512, 64, "bf16", padded=True),
    "long_causal": Workload("long_causal", 1, 32, 16384, 128, "bf16", causal=True),
    "block_sparse": Workload("block_sparse", 2, 8, 8192, 64, "bf16", block_sparse=True),
}
ORDER = ["tiny_fp32", "gpt2_causal", "bert_padded", "long_causal", "block_sparse"]

# The FP8 forward on the long-context shape: bf16 inputs, encoded to e4m3 on the device,
# then the e4m3 forward (same draw as long_causal).
# Training-time attention dropout on the long-context shape: p = 26/256 (~0.1, the usual
# attention-dropout rate), the same Q, K, V, dO draw as long_causal.
DROPOUT_WORKLOADS = {
    "long_causal_dropout": Workload("long_causal_dropout", 1, 32, 16384, 128, "bf16",
                                    causal=True, drop_threshold=26,
                                    drop_seed=0x5DEECE66D2B7E151),
}

FP8_WORKLOADS = {
    "long_causal_fp8": Workload("long_causal_fp8", 1, 32, 16384, 128, "bf16", causal=True),
}


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    kv_len: Optional[torch.Tensor]     # int32 [B] or None
    blockmask: Optional[torch.Tensor]  # uint8 [nb, nb] or None
    causal: bool
    scale: float


def custom(name: str, B: int, H: int, N: int, d: int, dtype: str = "bf16", **kw) -> Workload:
    """A workload of arbitrary shape with the same recipe (used for edge cases)."""
    return Workload(name, B, H, N, d, dtype, **kw)


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu") -> Inputs:
    """Draw the inputs of workload ``w`` from ``seed`` (CPU generator, fixed order)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    kv_len = None
    blockmask = None
    if w.padded:
        lo = min(BLOCK, w.N)
        kv_len = torch.randint(lo, w.N + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
    if w.block_sparse:
        nb = (w.N + BLOCK - 1) // BLOCK
        blockmask = (torch.rand((nb, nb), generator=g) < w.keep_prob).to(torch.uint8)
        blockmask.fill_diagonal_(1)
    if w.q_head0_mult != 1.0:
        q[:, 0] *= w.q_head0_mult
    dt = w.torch_dtype
    q, k, v, do = (t.to(dt).contiguous() for t in (q, k, v, do))
    if device != "cpu":
        q, k, v, do = (t.to(device) for t in (q, k, v, do))
        if kv_len is not None:
            kv_len = kv_len.to(device)
        if blockmask is not None:
            blockmask = blockmask.to(device)
    return Inputs(q, k, v, do, kv_len, blockmask, w.causal, w.scale)


# ------------------------------------------------------------------ decode

@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One new query token per sequence over a key/value cache of up to ``L`` rows.

    ``Hq`` query heads share ``Hkv`` key/value heads in contiguous groups of Hq / Hkv.
    ``ragged``: per-sequence cache lengths drawn in [max(1, L / 2), L]; otherwise all L.
    """
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    d: int
    ragged: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} L={self.L} d={self.d} bf16"
                + (" ragged cache lengths" if self.ragged else ""))


# The decode shape the course page uses as its example: Llama-3-8B (32 query heads, 8
# key/value heads, head size 128) at an 8k context, 64 sequences decoding together.
DECODE_WORKLOADS = {
    "decode_llama8b": DecodeWorkload("decode_llama8b", 64, 32, 8, 8192, 128),
}


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, Hq, d] bf16
    k: torch.Tensor          # [B, Hkv, L, d] bf16
    v: torch.Tensor          # [B, Hkv, L, d] bf16
    cache_len: torch.Tensor  # int32 [B]
    scale: float


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, device: str = "cpu") -> DecodeInputs:
    """Draw q, k, v (``randn`` in fp32 from one CPU generator, in that order, rounded to
    bf16), then the cache lengths."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((w.B, w.Hq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.L, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.L, w.d), generator=g, dtype=torch.float32)
    if w.ragged:
        lo = max(1, w.L // 2)
        cache_len = torch.randint(lo, w.L + 1, (w.B,), generator=g, dtype=torch.int64)
    else:
        cache_len = torch.full((w.B,), w.L, dtype=torch.int64)
    cache_len = cache_len.to(torch.int32)
    q, k, v = (t.to(torch.bfloat16).contiguous() for t in (q, k, v))
    if device != "cpu":
        q, k, v, cache_len = (t.to(device) for t in (q, k, v, cache_len))
    return DecodeInputs(q, k, v, cache_len, w.scale)
