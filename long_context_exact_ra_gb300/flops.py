"""Work accounting for the attention workloads (FLOPs and algorithmic bytes).

Convention (the evaluation metric): forward FLOPs = 4 * b * h * s_q * s_k * d,
halved when causal; backward = 2.5 x forward (five matmuls against two).
`visible_pairs` counts the (query, key) pairs the method must actually
combine, for the honest roofline when segments mask most of the square.
"""
from __future__ import annotations

import numpy as np


def fwd_flops_nominal(B, S, H, D, causal: bool) -> float:
    f = 4.0 * B * H * S * S * D
    return f / 2 if causal else f


def bwd_flops_nominal(B, S, H, D, causal: bool) -> float:
    return 2.5 * fwd_flops_nominal(B, S, H, D, causal)


def visible_pairs(S: int, causal_block_size: int, seg_row=None) -> int:
    """Number of visible (i, j) pairs of one batch row (all heads alike)."""
    c = causal_block_size
    if seg_row is None:
        if c == 0:
            return S * S
        # row i sees keys j with j // c <= i // c: ((i // c) + 1) * c keys, capped at S
        i = np.arange(S, dtype=np.int64)
        return int(np.minimum((i // c + 1) * c, S).sum())
    seg_row = np.asarray(seg_row)
    total = 0
    # documents are runs of equal ids only for packed ids; count generally per id
    for sid in np.unique(seg_row):
        pos = np.nonzero(seg_row == sid)[0]
        if c == 0:
            total += len(pos) * len(pos)
        else:
            blk = pos // c
            # for each query position count keys of the same id with block <= its block
            sb = np.sort(blk)
            total += int(np.searchsorted(sb, blk, side="right").sum())
    return total


def fwd_flops_visible(B, S, H, D, causal_block_size, segment_ids=None) -> float:
    if segment_ids is None:
        pairs = B * visible_pairs(S, causal_block_size)
    else:
        pairs = sum(visible_pairs(S, causal_block_size, segment_ids[b]) for b in range(B))
    return 4.0 * H * D * pairs


def fwd_bytes(B, S, H, D, elem=2) -> float:
    """Algorithmic HBM bytes of the forward: Q, K, V read once, O written, lse written."""
    return 4.0 * B * S * H * D * elem + 4.0 * B * H * S
