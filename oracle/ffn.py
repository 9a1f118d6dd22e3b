"""CPU oracle for the blockwise feed-forward network (float64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the bench's CPU
baseline leg use it.  It shares no code with the CUDA library.

Sources (cited by page title and section):

* "Ring Attention with Blockwise Transformers for Near-Infinite Context"
  (paper review page): the position-wise feed-forward network
  FFN(x) = max(0, x W1 + b1) W2 + b2, applied to every row of the sequence.
* "Blockwise Feedforward网络详解RingAttention如何实现内存高效的前向传播"
  (blockwise feed-forward page), §核心技术原理 and §分块重组机制: the
  (batch, sequence, hidden) input is cut into fixed-size chunks of rows, the
  feed-forward runs on one chunk at a time (only that chunk's hidden
  activation exists at once), and the chunk results are put back in order.

Readings where the pages leave the point open:

* Weights are stored the way a linear layer stores them: w1 is [F, Dm] (W1
  transposed) and w2 is [Dm, F] (W2 transposed), so x W1 = x @ w1.T.  Biases
  b1 [F] and b2 [Dm] are float32.
* Chunks are consecutive rows of the flattened (batch * sequence) axis; the
  last chunk may be shorter.  The FFN acts on each row independently, so the
  chunked result equals the unchunked one (pinned).
* The bf16 path rounds the hidden activation to bf16 before the second
  product (it is stored in that type between the two products); the oracle
  can emulate that rounding (`round_hidden_bf16=True`) or keep it exact.
"""
from __future__ import annotations

import numpy as np


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest even, through float32) and return them as float64."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def ffn_rows(x, w1, b1, w2, b2, round_hidden_bf16: bool = False):
    """FFN(x) = max(0, x W1 + b1) W2 + b2 for a [rows, Dm] block (paper review page)."""
    x = np.asarray(x, dtype=np.float64)
    h = x @ np.asarray(w1, dtype=np.float64).T + np.asarray(b1, dtype=np.float64)
    h = np.maximum(h, 0.0)
    if round_hidden_bf16:
        h = _bf16_round(h)
    return h @ np.asarray(w2, dtype=np.float64).T + np.asarray(b2, dtype=np.float64)


def ref_blockwise_ffn(x, w1, b1, w2, b2, chunk_size: int, round_hidden_bf16: bool = False):
    """Blockwise FFN over x [B, L, Dm]: rows of the flattened (B*L) axis in chunks of
    chunk_size, each chunk through the FFN, results reassembled in order
    (blockwise feed-forward page, §核心技术原理)."""
    x = np.asarray(x, dtype=np.float64)
    B, L, Dm = x.shape
    flat = x.reshape(B * L, Dm)
    out = np.empty((B * L, np.asarray(w2).shape[0]))
    for lo in range(0, B * L, chunk_size):
        hi = min(B * L, lo + chunk_size)
        out[lo:hi] = ffn_rows(flat[lo:hi], w1, b1, w2, b2, round_hidden_bf16)
    return out.reshape(B, L, -1)
