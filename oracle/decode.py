"""CPU oracle for decoding against a sharded KV cache (float64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the bench's CPU
baseline leg use it.  It shares no code with the CUDA library.

Sources (cited by page title and section):

* "RingAttention与传统注意力机制对比为什么它是大语言模型的终极解决方案"
  (comparison page): §关键参数配置 lists ``cache_idx`` (the inference cache
  index) among the attention's parameters, and §推理成本显著降低 states that
  the blockwise computation makes incremental decoding with a KV cache
  efficient.  The same page lists an inference-optimised module among the
  implementation's files.
* "Ring Attention with Blockwise Transformers for Near-Infinite Context"
  (paper review page), 分块注意力 / 环形注意力算法: the sequence (here: the
  cache) is split into N contiguous blocks and a query block combines the
  key/value blocks in ring order k = (j - i) mod N; 排列不变性: the combined
  result does not depend on that order.
* "从论文到代码：深入理解RingAttention的块注意力计算逻辑" (code walk-through
  page), §2 数值稳定的注意力计算: the lazy-softmax running max / numerator /
  denominator update that merges the per-block results.

Readings where the pages are silent (the plainest reading that the rest of
the pages supports):

* ``cache_idx[b]`` is the number of cache entries of batch row b that precede
  the new tokens: new token t sits at position ``cache_idx[b] + t``, and its
  key/value have already been written into the cache at that position.  The
  cache holds ``L_b = clamp(cache_idx[b] + T, 0, S)`` filled entries; entries
  at ``j >= L_b`` are not keys.
* Key j is visible to new token t iff ``j < L_b`` and the forward's masks
  hold: causal block size c > 0 requires ``pos // c >= j // c``; segment ids
  (one per new token, one per cache entry) must be equal.
* Ring: the cache is cut into N contiguous shards of S / N entries; the token
  at ``pos`` belongs to shard ``j = clamp(pos, 0, S - 1) // (S / N)`` and
  combines the shards k = (j - i) mod N, i = 0..N-1, each shard's key chunks
  in ascending order.
* A token with no visible key gets out = 0 and lse = -inf; lse is the natural
  log-sum-exp of the scaled scores.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import NEG_INF, _head_softmax, visible


def filled_lengths(cache_idx, new_tokens: int, cache_len: int) -> np.ndarray:
    """L_b = clamp(cache_idx[b] + T, 0, S): the number of filled cache entries."""
    c = np.asarray(cache_idx, dtype=np.int64)
    return np.clip(c + int(new_tokens), 0, int(cache_len))


def decode_visible(cache_idx_b: int, new_tokens: int, cache_len: int, causal_block_size: int,
                   q_seg=None, kv_seg=None) -> np.ndarray:
    """Boolean [T, S]: may new token t of one batch row attend to cache entry j?"""
    pos = int(cache_idx_b) + np.arange(new_tokens)
    kpos = np.arange(cache_len)
    vis = visible(pos, kpos, causal_block_size, q_seg, kv_seg)
    L = int(filled_lengths([cache_idx_b], new_tokens, cache_len)[0])
    vis &= (kpos < L)[None, :]
    return vis


def ref_decode(q, k_cache, v_cache, cache_idx, causal_block_size: int = 1,
               q_segment_ids=None, kv_segment_ids=None):
    """Exact attention of T new tokens against the cache (the plain definition).

    q: [B, T, H, D]; k_cache, v_cache: [B, S, H, D]; cache_idx: [B] ints.
    q_segment_ids: [B, T] / kv_segment_ids: [B, S] ints, both or neither.
    Returns out [B, T, H, D] and lse [B, H, T] (float64, natural log).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_cache, dtype=np.float64)
    v = np.asarray(v_cache, dtype=np.float64)
    B, T, H, D = q.shape
    S = k.shape[1]
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, T, H, D))
    lse = np.full((B, H, T), NEG_INF)
    for b in range(B):
        qs = None if q_segment_ids is None else np.asarray(q_segment_ids)[b]
        ks = None if kv_segment_ids is None else np.asarray(kv_segment_ids)[b]
        vis = decode_visible(int(np.asarray(cache_idx)[b]), T, S, causal_block_size, qs, ks)
        for h in range(H):
            p, l = _head_softmax((q[b, :, h, :] @ k[b, :, h, :].T) * scale, vis)
            out[b, :, h, :] = p @ v[b, :, h, :]
            lse[b, h, :] = l
    return out, lse


def ref_decode_rows(q, k_cache, v_cache, cache_idx, rows, causal_block_size: int = 1,
                    q_segment_ids=None, kv_segment_ids=None):
    """ref_decode on selected (b, h, t) rows only: returns out [n, D], lse [n]."""
    rows = np.asarray(rows, dtype=np.int64)
    D = q.shape[3]
    S = k_cache.shape[1]
    T = q.shape[1]
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((len(rows), D))
    lse = np.full(len(rows), NEG_INF)
    for n, (b, h, t) in enumerate(rows):
        qs = None if q_segment_ids is None else np.asarray(q_segment_ids)[b]
        ks = None if kv_segment_ids is None else np.asarray(kv_segment_ids)[b]
        vis = decode_visible(int(np.asarray(cache_idx)[b]), T, S, causal_block_size, qs, ks)[t:t + 1]
        K = np.asarray(k_cache[b, :, h, :], dtype=np.float64)
        V = np.asarray(v_cache[b, :, h, :], dtype=np.float64)
        Q = np.asarray(q[b, t:t + 1, h, :], dtype=np.float64)
        p, l = _head_softmax((Q @ K.T) * scale, vis)
        out[n] = (p @ V)[0]
        lse[n] = l[0]
    return out, lse


def ref_ring_decode(q, k_cache, v_cache, cache_idx, causal_block_size: int = 1,
                    q_segment_ids=None, kv_segment_ids=None, num_shards: int = 1,
                    key_chunk_size: int | None = None, shard_order=None):
    """Decode the Ring Attention way: per-shard blockwise passes merged in ring order.

    For each new token (position pos, home shard j) the shards k = (j - i) mod N
    are visited for i = 0..N-1 (paper review page, 环形注意力算法); inside a
    shard the key chunks go in ascending order, and every chunk updates the
    running max, numerator and denominator with the lazy-softmax rule (code
    walk-through page, §2).  shard_order: optional callable (j, i) -> k that
    replaces the ring order (permutation-invariance checks).
    Returns out [B, T, H, D], lse [B, H, T] (float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_cache, dtype=np.float64)
    v = np.asarray(v_cache, dtype=np.float64)
    B, T, H, D = q.shape
    S = k.shape[1]
    N = num_shards
    assert S % N == 0
    Ssh = S // N
    Ck = key_chunk_size or Ssh
    assert Ssh % Ck == 0
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, T, H, D))
    lse = np.full((B, H, T), NEG_INF)
    for b in range(B):
        qs = None if q_segment_ids is None else np.asarray(q_segment_ids)[b]
        ks = None if kv_segment_ids is None else np.asarray(kv_segment_ids)[b]
        vis_all = decode_visible(int(np.asarray(cache_idx)[b]), T, S, causal_block_size, qs, ks)
        for t in range(T):
            pos = int(np.asarray(cache_idx)[b]) + t
            j = min(max(pos, 0), S - 1) // Ssh
            for h in range(H):
                m = NEG_INF
                num = np.zeros(D)
                den = 0.0
                for i in range(N):
                    kk = (j - i) % N if shard_order is None else shard_order(j, i)
                    for c0 in range(kk * Ssh, (kk + 1) * Ssh, Ck):
                        vis = vis_all[t, c0:c0 + Ck]
                        if not vis.any():
                            continue
                        s = np.where(vis, (k[b, c0:c0 + Ck, h, :] @ q[b, t, h, :]) * scale, NEG_INF)
                        m_new = max(m, float(s.max()))
                        corr = math.exp(m - m_new) if m != NEG_INF else 1.0
                        w = np.exp(s - m_new)
                        num = num * corr + w @ v[b, c0:c0 + Ck, h, :]
                        den = den * corr + float(w.sum())
                        m = m_new
                if den > 0:
                    out[b, t, h, :] = num / den
                    lse[b, h, t] = m + math.log(den)
    return out, lse
