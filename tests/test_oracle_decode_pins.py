"""Pins for the decode oracle (oracle/decode.py), checked against things other than itself.

* Incremental decoding reproduces the full forward: with the cache holding the
  sequence's K/V, the new tokens p..p+T-1 decoded at cache_idx = p must give
  rows p..p+T-1 of the (separately pinned) causal forward definition.
* An independent library routine: torch CPU float64 scaled_dot_product_attention
  given the decode mask derived from the forward's visibility (rows of the
  prefill mask restricted to the filled cache).
* Closed forms: a single visible key returns its V row and q.k/sqrt(d) as lse;
  equal scores return the mean of the visible V rows and ln(count); no visible
  key gives 0 and -inf.
* The ring restatement equals the definition for any shard count, chunking and
  shard visiting order (permutation invariance).
* Brute force with explicit Python loops on a tiny case.
* Planted mistakes: mutated copies of the oracle must fail these pins.
"""
import math
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import decode as odec
from long_context_exact_ra_gb300.inputs import random_segment_ids


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _seq(seed, B, S, H, D, scale=1.0):
    g = _rng(seed)
    return tuple(g.standard_normal((B, S, H, D)) * scale for _ in range(3))


PREFILL_CASES = [
    # B, S, H, D, c, maxdoc, p, T
    (2, 64, 2, 16, 1, None, 0, 1),
    (2, 64, 2, 16, 1, None, 37, 1),
    (2, 64, 2, 16, 1, None, 63, 1),
    (1, 48, 3, 8, 1, None, 20, 5),
    (2, 64, 2, 16, 1, 9, 30, 4),
    (1, 60, 2, 8, 4, None, 36, 4),   # c = 4: the filled end 40 is a block boundary
    (1, 40, 2, 8, 0, None, 32, 8),   # non-causal: the new tokens fill the cache
]


@pytest.mark.parametrize("B,S,H,D,c,maxdoc,p,T", PREFILL_CASES)
def test_decode_reproduces_prefill_rows(B, S, H, D, c, maxdoc, p, T):
    q, k, v = _seq(11, B, S, H, D)
    seg = None if maxdoc is None else random_segment_ids(11, B, S, maxdoc)
    full_out, full_lse = oracle.ref_fwd(q, k, v, seg, c)
    idx = np.full(B, p)
    out, lse = odec.ref_decode(q[:, p:p + T], k, v, idx, c,
                               None if seg is None else seg[:, p:p + T], seg)
    assert np.allclose(out, full_out[:, p:p + T], rtol=0, atol=1e-12)
    assert np.allclose(lse, full_lse[:, :, p:p + T], rtol=0, atol=1e-12)


@pytest.mark.parametrize("c,maxdoc", [(0, None), (1, None), (3, None), (4, 7), (0, 5)])
def test_decode_equals_forward_over_the_filled_prefix(c, maxdoc):
    """For any mask: decoding p..p+T-1 against a larger cache = the forward over positions 0..p+T-1."""
    B, S, H, D = 2, 64, 2, 8
    q, k, v = _seq(31, B, S, H, D)
    seg = None if maxdoc is None else random_segment_ids(31, B, S, maxdoc)
    for p, T in ((0, 1), (21, 3), (40, 5), (63, 1)):
        L = p + T
        pre_out, pre_lse = oracle.ref_fwd(q[:, :L], k[:, :L], v[:, :L], None if seg is None else seg[:, :L], c)
        out, lse = odec.ref_decode(q[:, p:L], k, v, np.full(B, p), c,
                                   None if seg is None else seg[:, p:L], seg)
        assert np.allclose(out, pre_out[:, p:L], rtol=0, atol=1e-12)
        assert np.allclose(lse, pre_lse[:, :, p:L], rtol=0, atol=1e-12)


def _torch_decode(q, k, v, idx, c, qseg, kseg):
    """torch float64 SDPA; the mask is the forward's mask (plain loops) cut to the filled cache."""
    B, T, H, D = q.shape
    S = k.shape[1]
    mask = np.zeros((B, T, S), dtype=bool)
    for b in range(B):
        filled = max(0, min(S, int(idx[b]) + T))
        for t in range(T):
            i = int(idx[b]) + t
            for j in range(filled):
                ok = c == 0 or i // c >= j // c
                if qseg is not None and qseg[b, t] != kseg[b, j]:
                    ok = False
                mask[b, t, j] = ok
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask)[:, None])
    return o.permute(0, 2, 1, 3).numpy(), mask


SDPA_CASES = [
    # B, T, S, H, D, c, maxdoc, idx
    (3, 1, 96, 2, 16, 1, None, [0, 50, 95]),
    (2, 4, 64, 2, 8, 1, 7, [10, 60]),
    (2, 3, 64, 1, 8, 3, None, [5, 31]),
    (2, 2, 32, 2, 8, 0, None, [7, 30]),
]


@pytest.mark.parametrize("B,T,S,H,D,c,maxdoc,idx", SDPA_CASES)
def test_decode_matches_torch_sdpa(B, T, S, H, D, c, maxdoc, idx):
    g = _rng(5)
    q = g.standard_normal((B, T, H, D))
    k = g.standard_normal((B, S, H, D))
    v = g.standard_normal((B, S, H, D))
    kseg = None if maxdoc is None else random_segment_ids(5, B, S, maxdoc)
    qseg = None
    if kseg is not None:  # the new tokens carry the ids of their own cache positions
        qseg = np.stack([kseg[b, idx[b]:idx[b] + T] for b in range(B)])
    ref, mask = _torch_decode(q, k, v, idx, c, qseg, kseg)
    out, _ = odec.ref_decode(q, k, v, np.array(idx), c, qseg, kseg)
    has = mask.any(axis=2)  # torch gives NaN for empty rows; all rows here see a key
    assert has.all()
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    rows = np.array([(b, h, t) for b in range(B) for h in range(H) for t in range(T)])
    o_r, l_r = odec.ref_decode_rows(q, k, v, np.array(idx), rows, c, qseg, kseg)
    full, lse = odec.ref_decode(q, k, v, np.array(idx), c, qseg, kseg)
    assert np.allclose(o_r, full[rows[:, 0], rows[:, 2], rows[:, 1]], rtol=0, atol=1e-13)
    assert np.allclose(l_r, lse[rows[:, 0], rows[:, 1], rows[:, 2]], rtol=0, atol=1e-13)


def test_single_visible_key():
    g = _rng(6)
    q = g.standard_normal((1, 1, 2, 8))
    k = g.standard_normal((1, 16, 2, 8))
    v = g.standard_normal((1, 16, 2, 8))
    out, lse = odec.ref_decode(q, k, v, np.array([0]), 1)
    for h in range(2):
        assert np.allclose(out[0, 0, h], v[0, 0, h], atol=1e-14)
        assert abs(lse[0, h, 0] - np.dot(q[0, 0, h], k[0, 0, h]) / math.sqrt(8)) < 1e-13


def test_equal_scores_give_mean_of_visible_rows():
    g = _rng(7)
    T, S = 3, 40
    q = np.zeros((1, T, 1, 8))
    k = g.standard_normal((1, S, 1, 8))
    v = g.standard_normal((1, S, 1, 8))
    idx = 17
    out, lse = odec.ref_decode(q, k, v, np.array([idx]), 1)
    for t in range(T):
        n = idx + t + 1
        assert np.allclose(out[0, t, 0], v[0, :n, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, t] - math.log(n)) < 1e-13


def test_no_visible_key_gives_zero_and_minus_inf():
    g = _rng(8)
    q = g.standard_normal((1, 2, 1, 4))
    k = g.standard_normal((1, 8, 1, 4))
    v = g.standard_normal((1, 8, 1, 4))
    out, lse = odec.ref_decode(q, k, v, np.array([-2]), 1)  # nothing filled yet
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    kseg = np.zeros((1, 8), dtype=np.int32)
    out, lse = odec.ref_decode(q, k, v, np.array([3]), 1, np.array([[5, 5]]), kseg)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("N,Ck,c,maxdoc", [(1, None, 1, None), (2, 8, 1, None), (4, 4, 1, 6),
                                           (8, 8, 3, None), (4, 16, 0, None)])
def test_ring_restatement_equals_definition(N, Ck, c, maxdoc):
    g = _rng(9)
    B, T, S, H, D = 2, 3, 64, 2, 8
    q = g.standard_normal((B, T, H, D)) * 2.0
    k = g.standard_normal((B, S, H, D)) * 2.0
    v = g.standard_normal((B, S, H, D))
    idx = np.array([13, 61])
    kseg = None if maxdoc is None else random_segment_ids(9, B, S, maxdoc)
    qseg = None if kseg is None else np.stack([kseg[b, min(idx[b], S - T):min(idx[b], S - T) + T] for b in range(B)])
    ref, rlse = odec.ref_decode(q, k, v, idx, c, qseg, kseg)
    out, lse = odec.ref_ring_decode(q, k, v, idx, c, qseg, kseg, N, Ck)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=0, atol=1e-12)
    perm = _rng(10 + N).permutation(N)
    out2, _ = odec.ref_ring_decode(q, k, v, idx, c, qseg, kseg, N, Ck,
                                   shard_order=lambda j, i: int(perm[i]))
    assert np.allclose(out2, ref, rtol=0, atol=1e-12)


def test_brute_force_loops():
    g = _rng(12)
    B, T, S, H, D = 1, 2, 7, 1, 3
    q = g.standard_normal((B, T, H, D))
    k = g.standard_normal((B, S, H, D))
    v = g.standard_normal((B, S, H, D))
    idx = 3
    out, lse = odec.ref_decode(q, k, v, np.array([idx]), 1)
    for t in range(T):
        pos = idx + t
        ws = []
        for j in range(S):
            if j <= pos and j < idx + T:
                s = sum(q[0, t, 0, d] * k[0, j, 0, d] for d in range(D)) / math.sqrt(D)
                ws.append((j, s))
        mx = max(s for _, s in ws)
        z = sum(math.exp(s - mx) for _, s in ws)
        for d in range(D):
            o = sum(math.exp(s - mx) * v[0, j, 0, d] for j, s in ws) / z
            assert abs(out[0, t, 0, d] - o) < 1e-13
        assert abs(lse[0, 0, t] - (mx + math.log(z))) < 1e-13


def _mutant(old, new):
    src = open(odec.__file__).read()
    assert old in src, old
    src = src.replace(old, new, 1).replace("from .attention import", "from oracle.attention import")
    mod = types.ModuleType("decode_mutant")
    exec(compile(src, "decode_mutant", "exec"), mod.__dict__)
    return mod


DEC_MUTATIONS = [
    ("filled length one short", "np.clip(c + int(new_tokens), 0, int(cache_len))",
     "np.clip(c + int(new_tokens) - 1, 0, int(cache_len))"),
    ("position offset by one", "pos = int(cache_idx_b) + np.arange(new_tokens)",
     "pos = int(cache_idx_b) + 1 + np.arange(new_tokens)"),
    ("unfilled entries visible", "vis &= (kpos < L)[None, :]", "vis &= (kpos <= L)[None, :]"),
    ("v replaced by k", "out[b, :, h, :] = p @ v[b, :, h, :]", "out[b, :, h, :] = p @ k[b, :, h, :]"),
]


@pytest.mark.parametrize("label,old,new", DEC_MUTATIONS)
def test_planted_decode_mistakes_are_caught(label, old, new):
    mod = _mutant(old, new)
    B, S, H, D = 2, 48, 2, 8
    q, k, v = _seq(21, B, S, H, D)
    caught = False
    for c in (1, 0):
        for p, T in ((0, 1), (20, 3), (44, 3)):
            L = p + T
            pre_out, _ = oracle.ref_fwd(q[:, :L], k[:, :L], v[:, :L], None, c)
            out, _ = mod.ref_decode(q[:, p:L], k, v, np.full(B, p), c)
            caught |= not np.allclose(out, pre_out[:, p:L], rtol=0, atol=1e-9)
    assert caught, label


def test_planted_ring_decode_mistake_is_caught():
    mod = _mutant("num = num * corr + w @ v[b, c0:c0 + Ck, h, :]", "num = num + w @ v[b, c0:c0 + Ck, h, :]")
    g = _rng(13)
    q = g.standard_normal((1, 1, 1, 8)) * 3
    k = g.standard_normal((1, 64, 1, 8)) * 3
    v = g.standard_normal((1, 64, 1, 8))
    ref, _ = odec.ref_decode(q, k, v, np.array([63]), 1)
    out, _ = mod.ref_ring_decode(q, k, v, np.array([63]), 1, None, None, 4, 8)
    assert not np.allclose(out, ref, atol=1e-9)
