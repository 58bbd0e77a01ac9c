"""The ring all-reduce byte model of the pages, used for context lines only.

"Tensor parallelism" guide, section "Walking through a transformer block":
bytes moved per rank by a ring all-reduce of H elements of B bytes over T
ranks are about 2 (T - 1) / T * H * B.  On one GPU no such exchange happens
(the sum is done in device memory); the figure says what the same step
would move between T GPUs.
"""
from __future__ import annotations


def ring_allreduce_bytes(H: int, T: int, B: int) -> float:
    """Bytes each rank sends for a ring all-reduce of H elements of B bytes."""
    if T < 1 or H < 0 or B < 0:
        raise ValueError("T >= 1, H >= 0, B >= 0")
    return 2.0 * (T - 1) / T * H * B


def decode_bytes_per_token(H: int, T: int, B: int, layers: int, collectives_per_layer: int = 2) -> float:
    """Ring all-reduce bytes per rank per generated token (one step of H per
    collective, two collectives per transformer layer)."""
    return layers * collectives_per_layer * ring_allreduce_bytes(H, T, B)
