"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through its tests and the bench) and
the CPU oracle consume the arrays it returns, so that the two sides see exactly
the same values.

Recipe
------
* Values are drawn with ``numpy.random.Generator(PCG64)``.  Large tensors are
  filled in fixed-size chunks, each chunk from its own child seed
  (``SeedSequence(seed).spawn``), so the result does not depend on how many
  host threads do the filling.
* Tensors are ``[batch, seq, heads, head_dim]`` row-major, drawn i.i.d.
  ``scale * N(0, 1)`` in float32 and, for bf16 workloads, rounded to bf16 with
  round-to-nearest-even (the rounding is done here, on the host, so both sides
  start from the same bf16 values).
* Packed-document segment ids: per batch row, document lengths are drawn
  uniformly from the closed interval [256, 8192] and ids 0, 1, 2, ... are laid
  end to end until the row is full; the last document is cut at ``seq``.

The five named workloads follow the long-context Ring Attention evaluation
shapes: a tiny fp32 case, causal bf16 at 8K, packed documents at 32K, the
7B-shaped 128K case, and a forward+backward case at 64K.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22  # elements per independently seeded chunk


@dataclass(frozen=True)
class Workload:
    """Shape and masking of one attention problem (self-attention, [B,S,H,D])."""

    name: str
    batch: int
    seq: int
    heads: int
    head_dim: int
    dtype: str  # "f32" or "bf16"
    causal_block_size: int  # 0 = non-causal
    num_shards: int
    query_chunk_size: int
    key_chunk_size: int
    scale: float = 1.0  # standard deviation of q, k, v (and dO)
    segments: bool = False  # packed-document segment ids
    backward: bool = False
    seed: int = 0
    doc_len_range: tuple = field(default=(256, 8192))

    @property
    def shape(self):
        return (self.batch, self.seq, self.heads, self.head_dim)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five evaluation workloads (seed = 1000 + index).
WORKLOADS = {
    1: Workload("tiny fp32 non-causal B1 S512 H2 D64, 4 virtual shards",
                1, 512, 2, 64, "f32", 0, 4, 64, 64, seed=1001),
    2: Workload("causal bf16 fwd B2 S8192 H16 D128, 8 virtual shards",
                2, 8192, 16, 128, "bf16", 1, 8, 512, 512, seed=1002),
    3: Workload("packed-document bf16 fwd B4 S32768 H8 D64, 8 virtual shards",
                4, 32768, 8, 64, "bf16", 1, 8, 512, 512, scale=0.5,
                segments=True, seed=1003),
    4: Workload("7B-shaped causal bf16 fwd B1 S131072 H32 D128, 16 virtual shards",
                1, 131072, 32, 128, "bf16", 1, 16, 2048, 2048, seed=1004),
    5: Workload("causal bf16 fwd+bwd B1 S65536 H32 D128, 8 virtual shards",
                1, 65536, 32, 128, "bf16", 1, 8, 512, 512, backward=True,
                seed=1005),
}


def _fill_normal(seed_seq: np.random.SeedSequence, n: int, scale: float,
                 threads: int | None = None) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    children = seed_seq.spawn(nchunks)

    def work(i):
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if threads is None:
        threads = max(1, min(16, len(os.sched_getaffinity(0))))
    if nchunks <= 1 or threads <= 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))
    if scale != 1.0:
        out *= np.float32(scale)
    return out


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); return the bf16 bit patterns (uint16)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # NaN never occurs for normal draws; keep the plain RNE bit trick.
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def tensor(seed: int, stream: int, shape, scale: float, dtype: str) -> np.ndarray:
    """One seeded tensor.  f32 -> float32 array; bf16 -> uint16 bit patterns."""
    ss = np.random.SeedSequence([seed, stream])
    n = int(np.prod(shape))
    x = _fill_normal(ss, n, scale).reshape(shape)
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def packed_segment_ids(seed: int, batch: int, seq: int,
                       lo: int = 256, hi: int = 8192) -> np.ndarray:
    """[batch, seq] int32 document ids, documents of length U[lo, hi] laid end to end."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))
    seg = np.empty((batch, seq), dtype=np.int32)
    for b in range(batch):
        pos, doc = 0, 0
        while pos < seq:
            length = int(g.integers(lo, hi, endpoint=True))
            seg[b, pos:pos + length] = doc
            pos += length
            doc += 1
    return seg


@dataclass
class Inputs:
    """Host arrays for one workload.  bf16 tensors are uint16 bit patterns."""

    w: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dout: np.ndarray | None
    segment_ids: np.ndarray | None

    def as_f64(self, name: str) -> np.ndarray:
        """A tensor as float64 values (exact: bf16 and f32 both embed in f64)."""
        x = getattr(self, name)
        if x is None:
            return None
        if self.w.dtype == "bf16":
            return bf16_bits_to_f32(x).astype(np.float64)
        return x.astype(np.float64)


def make_inputs(w: Workload, with_dout: bool | None = None) -> Inputs:
    shape = w.shape
    q = tensor(w.seed, 0, shape, w.scale, w.dtype)
    k = tensor(w.seed, 1, shape, w.scale, w.dtype)
    v = tensor(w.seed, 2, shape, w.scale, w.dtype)
    if with_dout is None:
        with_dout = w.backward
    dout = tensor(w.seed, 3, shape, w.scale, w.dtype) if with_dout else None
    seg = None
    if w.segments:
        lo, hi = w.doc_len_range
        seg = packed_segment_ids(w.seed, w.batch, w.seq, lo, hi)
    return Inputs(w, q, k, v, dout, seg)


def random_segment_ids(seed: int, batch: int, seq: int, max_doc: int) -> np.ndarray:
    """Small-case segment ids: documents of length U[1, max_doc], laid end to end."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    seg = np.empty((batch, seq), dtype=np.int32)
    for b in range(batch):
        pos, doc = 0, 0
        while pos < seq:
            length = int(g.integers(1, max_doc, endpoint=True))
            seg[b, pos:pos + length] = doc
            pos += length
            doc += 1
    return seg


def sample_rows(seed: int, w: Workload, n: int) -> np.ndarray:
    """(b, h, i) query rows for sampled checks: uniform draws plus forced edges.

    Forced rows: i in {0, 1, S-1} and every virtual-shard and 128-row tile
    boundary +-1, each on a drawn (b, h).  Returns an int64 array [n_total, 3].
    """
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 55])))
    S = w.seq
    forced = {0, 1, S - 1}
    sh = S // w.num_shards
    for j in range(w.num_shards + 1):
        for d in (-1, 0, 1):
            forced.add(j * sh + d)
    for t in range(0, S + 1, 128):
        for d in (-1, 0):
            forced.add(t + d)
    forced = sorted(i for i in forced if 0 <= i < S)
    rows = []
    for i in forced:
        rows.append((int(g.integers(w.batch)), int(g.integers(w.heads)), i))
    m = max(0, n - len(rows))
    bs = g.integers(w.batch, size=m)
    hs = g.integers(w.heads, size=m)
    is_ = g.integers(S, size=m)
    rows.extend(zip(bs.tolist(), hs.tolist(), is_.tolist()))
    return np.array(rows, dtype=np.int64)


# ---------------------------------------------------------------------------
# Decoding against a KV cache
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class DecodeWorkload:
    """T new tokens per batch row against a [B, S, H, D] key/value cache."""

    name: str
    batch: int
    new_tokens: int
    cache_len: int
    heads: int
    head_dim: int
    dtype: str
    causal_block_size: int
    num_shards: int
    scale: float = 1.0
    segments: bool = False
    fill: str = "full"  # "full": cache_idx = S - T for every row; "random": seeded draws
    seed: int = 0
    doc_len_range: tuple = field(default=(256, 8192))

    def with_(self, **kw) -> "DecodeWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return DecodeWorkload(**d)


# Long-context decode with the 7B shape: the cache is the 131072-token K/V of
# the 7B-shaped forward workload (same seed, same streams: identical values).
DECODE_WORKLOADS = {
    "7b": DecodeWorkload("7B-shaped decode B1 T1 S131072 H32 D128 bf16, 16 virtual shards, full cache",
                         1, 1, 131072, 32, 128, "bf16", 1, 16, seed=1004),
}


@dataclass
class DecodeInputs:
    """Host arrays for one decode problem.  bf16 tensors are uint16 bit patterns."""

    w: DecodeWorkload
    q: np.ndarray            # [B, T, H, D]
    k_cache: np.ndarray      # [B, S, H, D]
    v_cache: np.ndarray      # [B, S, H, D]
    cache_idx: np.ndarray    # [B] int32
    q_segment_ids: np.ndarray | None   # [B, T] int32
    kv_segment_ids: np.ndarray | None  # [B, S] int32

    def as_f64(self, name: str) -> np.ndarray:
        x = getattr(self, name)
        if self.w.dtype == "bf16":
            return bf16_bits_to_f32(x).astype(np.float64)
        return x.astype(np.float64)


def decode_cache_idx(seed: int, batch: int, new_tokens: int, cache_len: int, fill: str) -> np.ndarray:
    """[B] int32 cache indices: "full" -> S - T; "random" -> U[0, S - T] per row
    with row 0 forced to S - T and row 1 (if any) to 0."""
    top = max(0, cache_len - new_tokens)
    if fill == "full":
        return np.full(batch, top, dtype=np.int32)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 31])))
    idx = g.integers(0, top, size=batch, endpoint=True).astype(np.int32)
    idx[0] = top
    if batch > 1:
        idx[1] = 0
    return idx


def make_decode_inputs(w: DecodeWorkload, cache_idx=None) -> DecodeInputs:
    cshape = (w.batch, w.cache_len, w.heads, w.head_dim)
    k = tensor(w.seed, 1, cshape, w.scale, w.dtype)
    v = tensor(w.seed, 2, cshape, w.scale, w.dtype)
    q = tensor(w.seed, 4, (w.batch, w.new_tokens, w.heads, w.head_dim), w.scale, w.dtype)
    if cache_idx is None:
        cache_idx = decode_cache_idx(w.seed, w.batch, w.new_tokens, w.cache_len, w.fill)
    cache_idx = np.asarray(cache_idx, dtype=np.int32)
    qseg = kseg = None
    if w.segments:
        lo, hi = w.doc_len_range
        kseg = packed_segment_ids(w.seed, w.batch, w.cache_len, lo, hi)
        qseg = np.zeros((w.batch, w.new_tokens), dtype=np.int32)
        for b in range(w.batch):  # a new token belongs to the document of its cache position
            for t in range(w.new_tokens):
                j = int(cache_idx[b]) + t
                qseg[b, t] = kseg[b, min(max(j, 0), w.cache_len - 1)] if w.cache_len > 0 else 0
    return DecodeInputs(w, q, k, v, cache_idx, qseg, kseg)


# ---------------------------------------------------------------------------
# Blockwise feed-forward
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class FfnWorkload:
    """x [B, L, Dm] through max(0, x w1^T + b1) w2^T + b2 in chunks of rows."""

    name: str
    batch: int
    seq: int
    model_dim: int
    ffn_dim: int
    chunk_size: int
    seed: int = 0
    bias: bool = True

    def with_(self, **kw) -> "FfnWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return FfnWorkload(**d)


# The 7B shape (hidden 4096, feed-forward width 11008) on 16384 rows in two chunks.
FFN_WORKLOADS = {
    "7b": FfnWorkload("7B-shaped blockwise feed-forward B1 L16384 Dm4096 F11008 bf16, chunks of 8192 rows",
                      1, 16384, 4096, 11008, 8192, seed=1007),
}


@dataclass
class FfnInputs:
    w: FfnWorkload
    x: np.ndarray          # [B, L, Dm] bf16 bits
    w1: np.ndarray         # [F, Dm] bf16 bits
    b1: np.ndarray | None  # [F] float32
    w2: np.ndarray         # [Dm, F] bf16 bits
    b2: np.ndarray | None  # [Dm] float32

    def as_f64(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a is None:
            return None
        return bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def make_ffn_inputs(w: FfnWorkload) -> FfnInputs:
    """x ~ N(0, 1); w1 ~ N(0, 1/Dm) and w2 ~ N(0, 1/F) (unit-variance pre-activations);
    biases ~ 0.1 N(0, 1) in float32."""
    x = tensor(w.seed, 0, (w.batch, w.seq, w.model_dim), 1.0, "bf16")
    w1 = tensor(w.seed, 1, (w.ffn_dim, w.model_dim), 1.0 / np.sqrt(w.model_dim), "bf16")
    w2 = tensor(w.seed, 2, (w.model_dim, w.ffn_dim), 1.0 / np.sqrt(w.ffn_dim), "bf16")
    b1 = tensor(w.seed, 3, (w.ffn_dim,), 0.1, "f32") if w.bias else None
    b2 = tensor(w.seed, 4, (w.model_dim,), 0.1, "f32") if w.bias else None
    return FfnInputs(w, x, w1, b1, w2, b2)
