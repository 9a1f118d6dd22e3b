"""CPU oracle for Ring Attention's blockwise exact attention (float64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the bench's CPU
baseline leg use it.  It shares no code with the CUDA library.

Sources (web pages on Ring Attention; cited by page title and section):

* [RA-review] "Ring Attention with Blockwise Transformers for Near-Infinite
  Context" (paper review page):
    - §三 技术架构, 核心公式/自注意力: Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V,
      Q,K,V in R^{s x d}.  (The fraction and square root were lost in the
      page's text extraction; the reading is division by sqrt(d).)
    - 分块注意力: the sequence is split into N blocks, device i holds Q_i,K_i,V_i.
    - 环形注意力算法: at outer step i, device j uses K_k, V_k with
      k = (j - i) mod N, then passes them on to device j+1.
    - 排列不变性: the result does not depend on the order of the KV blocks,
      the per-block results being combined with lazy softmax.
    - 四、核心创新, 精确算法: the method is exact (no approximation).
* [RA-code] "从论文到代码：深入理解RingAttention的块注意力计算逻辑" (code
  walk-through page):
    - 环形计算模式: numerator [b,q,h,d] and denominator [b,h,q] start at zero,
      a scan over the ring size, one blockwise step per KV block, then K/V move
      to the next device.
    - 1. 分块处理机制: q is cut into q_len // query_chunk_size chunks and k, v
      into kv_len // key_chunk_size chunks.
    - 2. 数值稳定的注意力计算: running max = max(previous max, chunk row max);
      weights exp(s - max); numerator = numerator * exp(prev_max - max) +
      weights @ v; denominator likewise with the row sums of the weights.
    - 3. 因果注意力掩码支持: a chunk pair runs only when below_or_on_diag(
      q_chunk_idx_start + q_chunk_idx, query_chunk_size,
      k_chunk_idx_start + k_chunk_idx, key_chunk_size, causal_block_size).

Readings where the pages are silent (the plainest reading that the rest of
the pages supports):

* visible(i, j) = (c == 0 or i // c >= j // c) and (no segments or
  seg[i] == seg[j]), c = causal_block_size.  The body of below_or_on_diag is
  not printed; the reading used is "the chunk pair holds at least one visible
  causal element", i.e. the last query position's causal block is >= the first
  key position's causal block.  Skipping under this reading never changes the
  result.
* Sharding is contiguous: global position = shard * (S / N) + local position.
* The running max starts at -inf; when it is still -inf the correction is 1
  and the weights are 0 (no NaN).
* out = numerator / denominator; a row with no visible key gets out = 0 and
  lse = -inf.
* lse (log-sum-exp, natural log) is not on the pages; it is the saved
  statistic from which the backward recomputes P.
* Backward: the plain softmax-attention gradient (P = exp(S - lse),
  Delta = rowsum(dO * out), dS = P * (dO V^T - Delta)).

Parity pins: every public function here is pinned in
tests/test_oracle_pins.py against closed forms, invariants, brute force,
finite differences or an independent library routine.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# Visibility (causal block mask AND segment mask)
# ---------------------------------------------------------------------------

def visible(qpos: np.ndarray, kpos: np.ndarray, causal_block_size: int,
            qseg: np.ndarray | None = None, kseg: np.ndarray | None = None) -> np.ndarray:
    """Boolean [len(qpos), len(kpos)]: may query position i attend to key position j?

    Causal with block size c (RA-code §3): i // c >= j // c.  c = 0 means no
    causal mask.  Segment ids: attend only within the same id.
    """
    qpos = np.asarray(qpos)[:, None]
    kpos = np.asarray(kpos)[None, :]
    vis = np.ones((qpos.shape[0], kpos.shape[1]), dtype=bool)
    c = int(causal_block_size)
    if c > 0:
        vis &= (qpos // c) >= (kpos // c)
    if qseg is not None:
        vis &= np.asarray(qseg)[:, None] == np.asarray(kseg)[None, :]
    return vis


# ---------------------------------------------------------------------------
# Direct definition: softmax(Q K^T / sqrt(d)) V with explicit masks
# ---------------------------------------------------------------------------

def _head_softmax(s: np.ndarray, vis: np.ndarray):
    """Row softmax of scores s under mask vis.  Returns (P, lse); empty rows -> 0, -inf."""
    s = np.where(vis, s, NEG_INF)
    m = s.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])  # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(has[:, None], e / np.where(has, l, 1.0)[:, None], 0.0)
        lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), NEG_INF)
    return p, lse


def ref_fwd(q, k, v, segment_ids=None, causal_block_size: int = 0):
    """Exact attention forward (RA-review §核心公式).

    q, k, v: [B, S, H, D] (any real dtype; computed in float64).
    segment_ids: [B, S] int or None.  Returns out [B,S,H,D] float64 and
    lse [B,H,S] float64 (natural log).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    out = np.zeros((B, S, H, D))
    lse = np.full((B, H, S), NEG_INF)
    pos = np.arange(S)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        seg = None if segment_ids is None else np.asarray(segment_ids)[b]
        vis = visible(pos, pos, causal_block_size, seg, seg)
        for h in range(H):
            s = (q[b, :, h, :] @ k[b, :, h, :].T) * scale
            p, lse_bh = _head_softmax(s, vis)
            out[b, :, h, :] = p @ v[b, :, h, :]
            lse[b, h, :] = lse_bh
    return out, lse


def ref_probs(q, k, segment_ids=None, causal_block_size: int = 0):
    """The attention matrix P [B,H,S,S] of the definition (for invariant checks)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, S, H, D = q.shape
    P = np.zeros((B, H, S, S))
    pos = np.arange(S)
    for b in range(B):
        seg = None if segment_ids is None else np.asarray(segment_ids)[b]
        vis = visible(pos, pos, causal_block_size, seg, seg)
        for h in range(H):
            s = (q[b, :, h, :] @ k[b, :, h, :].T) / math.sqrt(D)
            P[b, h], _ = _head_softmax(s, vis)
    return P


def ref_fwd_rows(q, k, v, rows, segment_ids=None, causal_block_size: int = 0):
    """Definition evaluated on selected query rows only.

    rows: int array [n, 3] of (b, h, i).  Returns out [n, D] and lse [n].
    q, k, v may be float32/float64/any real array of shape [B,S,H,D].
    """
    rows = np.asarray(rows, dtype=np.int64)
    B, S, H, D = q.shape
    out = np.zeros((len(rows), D))
    lse = np.full(len(rows), NEG_INF)
    scale = 1.0 / math.sqrt(D)
    pos = np.arange(S)
    order = np.lexsort((rows[:, 1], rows[:, 0]))
    start = 0
    while start < len(order):
        b, h = rows[order[start], 0], rows[order[start], 1]
        end = start
        while end < len(order) and rows[order[end], 0] == b and rows[order[end], 1] == h:
            end += 1
        idx = order[start:end]
        qi = rows[idx, 2]
        K = np.asarray(k[b, :, h, :], dtype=np.float64)
        V = np.asarray(v[b, :, h, :], dtype=np.float64)
        Q = np.asarray(q[b, qi, h, :], dtype=np.float64)
        seg = None if segment_ids is None else np.asarray(segment_ids)[b]
        vis = visible(qi, pos, causal_block_size,
                      None if seg is None else seg[qi], seg)
        s = (Q @ K.T) * scale
        p, l = _head_softmax(s, vis)
        out[idx] = p @ V
        lse[idx] = l
        start = end
    return out, lse


# ---------------------------------------------------------------------------
# Backward of the definition
# ---------------------------------------------------------------------------

def ref_bwd(q, k, v, dout, segment_ids=None, causal_block_size: int = 0):
    """Gradients dq, dk, dv [B,S,H,D] float64 of the exact attention.

    For each (b, h): P = softmax(S) under the mask, out = P V,
    Delta_i = sum_d dO_id out_id, dV = P^T dO, dP = dO V^T,
    dS = P * (dP - Delta), dQ = dS K / sqrt(D), dK = dS^T Q / sqrt(D).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, S, H, D = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    scale = 1.0 / math.sqrt(D)
    pos = np.arange(S)
    for b in range(B):
        seg = None if segment_ids is None else np.asarray(segment_ids)[b]
        vis = visible(pos, pos, causal_block_size, seg, seg)
        for h in range(H):
            Q, K, V, dO = q[b, :, h], k[b, :, h], v[b, :, h], dout[b, :, h]
            P, _ = _head_softmax((Q @ K.T) * scale, vis)
            O = P @ V
            delta = (dO * O).sum(axis=1)
            dV = P.T @ dO
            dP = dO @ V.T
            dS = P * (dP - delta[:, None])
            dq[b, :, h] = (dS @ K) * scale
            dk[b, :, h] = (dS.T @ Q) * scale
            dv[b, :, h] = dV
    return dq, dk, dv


def ref_bwd_head_blocked(Q, K, V, dO, seg, causal_block_size, q_rows, k_rows, block=4096):
    """Gradients of one (b, h) head on selected rows, without an S x S matrix.

    Q, K, V, dO: [S, D] arrays of one head.  seg: [S] ints or None.
    Returns dq [len(q_rows), D], dk [len(k_rows), D], dv [len(k_rows), D].
    Same formulas as ref_bwd; the only difference is that the softmax
    statistics (lse, out, Delta) of every query are computed in row blocks.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    S, D = Q.shape
    scale = 1.0 / math.sqrt(D)
    pos = np.arange(S)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    lse = np.empty(S)
    delta = np.empty(S)
    for lo in range(0, S, block):
        hi = min(S, lo + block)
        qi = pos[lo:hi]
        vis = visible(qi, pos, causal_block_size,
                      None if seg is None else seg[qi], seg)
        p, l = _head_softmax((Q[lo:hi] @ K.T) * scale, vis)
        lse[lo:hi] = l
        delta[lo:hi] = (dO[lo:hi] * (p @ V)).sum(axis=1)
    # dq on the selected query rows
    vis = visible(q_rows, pos, causal_block_size,
                  None if seg is None else seg[q_rows], seg)
    s = (Q[q_rows] @ K.T) * scale
    with np.errstate(invalid="ignore"):
        P = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse[q_rows][:, None]), 0.0)
    dS = P * ((dO[q_rows] @ V.T) - delta[q_rows][:, None])
    dq = (dS @ K) * scale
    # dk, dv on the selected key rows: columns of P and dS
    vis = visible(pos, k_rows, causal_block_size,
                  seg, None if seg is None else seg[k_rows])
    s = (Q @ K[k_rows].T) * scale
    with np.errstate(invalid="ignore"):
        P = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse[:, None]), 0.0)
    dv = P.T @ dO
    dS = P * ((dO @ V[k_rows].T) - delta[:, None])
    dk = (dS.T @ Q) * scale
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Literal restatement of the ring algorithm (pins the readings above)
# ---------------------------------------------------------------------------

def below_or_on_diag(q_chunk_idx: int, query_chunk_size: int,
                     k_chunk_idx: int, key_chunk_size: int,
                     causal_block_size: int) -> bool:
    """Reading of RA-code §3: does the chunk pair contain any causally visible element?

    Chunk indices are global (chunk_idx_start + local index).  The pair is run
    iff the causal block of its last query position is >= the causal block of
    its first key position.
    """
    c = causal_block_size
    last_q = (q_chunk_idx + 1) * query_chunk_size - 1
    first_k = k_chunk_idx * key_chunk_size
    return last_q // c >= first_k // c


def ref_ring_fwd(q, k, v, segment_ids=None, causal_block_size: int = 0,
                 num_shards: int = 1, query_chunk_size: int | None = None,
                 key_chunk_size: int | None = None, shard_order=None):
    """Ring Attention forward, step by step as the pages describe it.

    For each device j (query shard j), for each ring step i the device holds
    K/V shard k = (j - i) mod N (RA-review 环形注意力算法).  Within a step, the
    blockwise pass (RA-code §1) walks query chunks, and for each query chunk the
    key chunks in ascending order; a chunk pair runs only if below_or_on_diag
    (RA-code §3).  The lazy-softmax update (RA-code §2) carries the running
    max, numerator and denominator across key chunks and ring steps.

    shard_order: optional callable (j, i) -> k overriding the ring order (used
    to check that the result does not depend on the KV block order).
    Returns out [B,S,H,D], lse [B,H,S] (float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    N = num_shards
    assert S % N == 0
    Ssh = S // N
    Cq = query_chunk_size or Ssh
    Ck = key_chunk_size or Ssh
    assert Ssh % Cq == 0 and Ssh % Ck == 0
    scale = 1.0 / math.sqrt(D)
    seg = None if segment_ids is None else np.asarray(segment_ids)
    out = np.zeros((B, S, H, D))
    lse = np.full((B, H, S), NEG_INF)
    for j in range(N):  # every device of the ring (in parallel on the pages)
        qsl = slice(j * Ssh, (j + 1) * Ssh)
        # carry: running max [b,h,q], numerator [b,q,h,d], denominator [b,h,q]
        prev_max = np.full((B, H, Ssh), NEG_INF)
        numerator = np.zeros((B, Ssh, H, D))
        denominator = np.zeros((B, H, Ssh))
        for i in range(N):
            kk = (j - i) % N if shard_order is None else shard_order(j, i)
            ksl = slice(kk * Ssh, (kk + 1) * Ssh)
            q_chunk_idx_start = j * Ssh // Cq
            k_chunk_idx_start = kk * Ssh // Ck
            for qc in range(Ssh // Cq):
                for kc in range(Ssh // Ck):
                    if causal_block_size > 0 and not below_or_on_diag(
                            q_chunk_idx_start + qc, Cq, k_chunk_idx_start + kc, Ck,
                            causal_block_size):
                        continue
                    ql = slice(qc * Cq, (qc + 1) * Cq)
                    kl = slice(kc * Ck, (kc + 1) * Ck)
                    qpos = np.arange(j * Ssh + qc * Cq, j * Ssh + (qc + 1) * Cq)
                    kpos = np.arange(kk * Ssh + kc * Ck, kk * Ssh + (kc + 1) * Ck)
                    for b in range(B):
                        vis = visible(qpos, kpos, causal_block_size,
                                      None if seg is None else seg[b, qpos],
                                      None if seg is None else seg[b, kpos])
                        for h in range(H):
                            qch = q[b, qsl, h][ql]
                            kch = k[b, ksl, h][kl]
                            vch = v[b, ksl, h][kl]
                            w = np.where(vis, (qch @ kch.T) * scale, NEG_INF)
                            pm = prev_max[b, h, ql]
                            mx = np.maximum(pm, w.max(axis=1))
                            mx_safe = np.where(np.isfinite(mx), mx, 0.0)
                            corr = np.where(np.isfinite(mx), np.exp(pm - mx_safe), 1.0)
                            ew = np.exp(w - mx_safe[:, None])
                            numerator[b, ql, h] = numerator[b, ql, h] * corr[:, None] + ew @ vch
                            denominator[b, h, ql] = denominator[b, h, ql] * corr + ew.sum(axis=1)
                            prev_max[b, h, ql] = mx
        has = denominator > 0
        with np.errstate(divide="ignore", invalid="ignore"):
            o = np.where(has.transpose(0, 2, 1)[..., None],
                         numerator / np.where(has, denominator, 1.0).transpose(0, 2, 1)[..., None],
                         0.0)
            l = np.where(has, prev_max + np.log(np.where(has, denominator, 1.0)), NEG_INF)
        out[:, qsl] = o
        lse[:, :, qsl] = l
    return out, lse

