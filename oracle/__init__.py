"""CPU fp64 oracle for exact attention (forward, logsumexp, backward, decode, FP8 forward,
dropout, key/value shards and their merge).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's ``smoke()``
check and by the benchmark's ``cpu_baseline`` leg, never by the product path.
"""
from .attention import (keep_mask, scores, softmax_rows, forward_head, backward_head,
                        row_dot, forward, backward)
from .online_softmax import tiled_forward_head
from .decode import decode
from . import fp8
from . import dropout
from . import seqshard

__all__ = ["keep_mask", "scores", "softmax_rows", "forward_head", "backward_head",
           "row_dot", "forward", "backward", "tiled_forward_head", "decode", "fp8", "dropout",
           "seqshard"]
