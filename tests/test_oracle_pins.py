"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-derived closed forms (tests/golden/closed_forms.json),
* an independent library routine (torch CPU float64 scaled_dot_product_attention
  with an explicit boolean mask, and torch autograd for the gradients),
* invariants the pages state: the result does not depend on the order in which
  KV blocks are visited (permutation invariance), a single visible key returns
  its V row, equal scores return the mean of the visible V rows, and the
  attention rows sum to one,
* central finite differences for the backward,
* brute force (explicit double loops) on tiny inputs,
* planted mistakes: mutated copies of the oracle must fail these pins.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt
from long_context_exact_ra_gb300.inputs import random_segment_ids

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _qkv(seed, B, S, H, D, scale=1.0):
    g = _rng(seed)
    return tuple(g.standard_normal((B, S, H, D)) * scale for _ in range(3))


def _torch_sdpa(q, k, v, seg, c):
    """torch float64 SDPA with an explicit boolean mask built by plain loops."""
    B, S, H, D = q.shape
    mask = np.zeros((B, S, S), dtype=bool)
    for b in range(B):
        for i in range(S):
            for j in range(S):
                ok = True
                if c > 0 and not (i // c >= j // c):
                    ok = False
                if seg is not None and seg[b, i] != seg[b, j]:
                    ok = False
                mask[b, i, j] = ok
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3)
    tm = torch.from_numpy(mask)[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=tm)
    return o.permute(0, 2, 1, 3).numpy(), mask


CASES = [
    # B, S, H, D, c, seg_max_doc
    (1, 17, 2, 8, 0, None),
    (2, 33, 3, 16, 1, None),
    (1, 40, 2, 8, 3, None),
    (2, 48, 2, 8, 1, 9),
    (1, 31, 1, 4, 0, 5),
    (1, 64, 2, 32, 7, 20),
]


# --------------------------------------------------------------------------
# Closed forms (golden file)
# --------------------------------------------------------------------------

def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "log": math.log}))


def test_golden_closed_forms():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 5
    for cs in cases:
        q = np.array(cs["q"], dtype=np.float64)[None, :, None, :]
        k = np.array(cs["k"], dtype=np.float64)[None, :, None, :]
        v = np.array(cs["v"], dtype=np.float64)[None, :, None, :]
        seg = None if cs["segment_ids"] is None else np.array([cs["segment_ids"]])
        out, lse = oracle.ref_fwd(q, k, v, seg, cs["causal_block_size"])
        exp_out = np.array([[_eval(x) for x in row] for row in cs["out"]])
        exp_lse = np.array([_eval(x) for x in cs["lse"]])
        np.testing.assert_allclose(out[0, :, 0, :], exp_out, rtol=0, atol=1e-13, err_msg=cs["name"])
        np.testing.assert_allclose(lse[0, 0], exp_lse, rtol=0, atol=1e-13, err_msg=cs["name"])
        # the ring restatement must give the same closed forms
        out_r, lse_r = oracle.ref_ring_fwd(q, k, v, seg, cs["causal_block_size"], 1)
        np.testing.assert_allclose(out_r[0, :, 0, :], exp_out, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse_r[0, 0], exp_lse, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Independent library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B,S,H,D,c,maxdoc", CASES)
def test_fwd_matches_torch_sdpa(B, S, H, D, c, maxdoc):
    q, k, v = _qkv(100 + S, B, S, H, D)
    seg = None if maxdoc is None else random_segment_ids(S, B, S, maxdoc)
    out, lse = oracle.ref_fwd(q, k, v, seg, c)
    ref, mask = _torch_sdpa(q, k, v, seg, c)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse by brute force: explicit loops, math.exp / math.log
    for b in range(B):
        for h in range(H):
            for i in range(0, S, 5):
                terms = [math.exp(sum(q[b, i, h, d] * k[b, j, h, d] for d in range(D)) / math.sqrt(D))
                         for j in range(S) if mask[b, i, j]]
                assert abs(lse[b, h, i] - math.log(sum(terms))) < 1e-12


@pytest.mark.parametrize("B,S,H,D,c,maxdoc", CASES)
def test_fwd_rows_matches_torch_sdpa(B, S, H, D, c, maxdoc):
    q, k, v = _qkv(200 + S, B, S, H, D)
    seg = None if maxdoc is None else random_segment_ids(S + 1, B, S, maxdoc)
    ref, _ = _torch_sdpa(q, k, v, seg, c)
    g = _rng(S)
    rows = np.stack([g.integers(B, size=25), g.integers(H, size=25), g.integers(S, size=25)], 1)
    rows = np.concatenate([rows, [[0, 0, 0], [B - 1, H - 1, S - 1]]])
    o, l = oracle.ref_fwd_rows(q, k, v, rows, seg, c)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(o[n], ref[b, i, h], rtol=0, atol=1e-12)
    full_out, full_lse = oracle.ref_fwd(q, k, v, seg, c)
    np.testing.assert_allclose(l, full_lse[rows[:, 0], rows[:, 1], rows[:, 2]], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants stated on the pages
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("c,maxdoc", [(0, None), (1, None), (3, None), (64, None), (1, 11), (0, 13)])
def test_ring_restatement_equals_definition(N, c, maxdoc):
    B, S, H, D = 1, 128, 2, 8
    q, k, v = _qkv(7 + N, B, S, H, D)
    seg = None if maxdoc is None else random_segment_ids(N, B, S, maxdoc)
    out, lse = oracle.ref_fwd(q, k, v, seg, c)
    Ssh = S // N
    for ch in {min(16, Ssh), Ssh}:
        o2, l2 = oracle.ref_ring_fwd(q, k, v, seg, c, N, ch, ch)
        np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_permutation_invariance(seed):
    """Any order of KV blocks gives the same output (paper review §排列不变性)."""
    B, S, H, D, N = 1, 96, 2, 8, 6
    q, k, v = _qkv(seed, B, S, H, D)
    seg = random_segment_ids(seed, B, S, 30)
    g = _rng(seed)
    perms = {j: g.permutation(N) for j in range(N)}
    base = oracle.ref_ring_fwd(q, k, v, seg, 1, N, 8, 16)
    shuf = oracle.ref_ring_fwd(q, k, v, seg, 1, N, 8, 16, shard_order=lambda j, i: int(perms[j][i]))
    np.testing.assert_allclose(shuf[0], base[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(shuf[1], base[1], rtol=0, atol=1e-12)


def test_single_visible_key_returns_its_v_row():
    B, S, H, D = 2, 40, 3, 16
    q, k, v = _qkv(5, B, S, H, D, scale=3.0)
    seg = random_segment_ids(5, B, S, 7)
    out, lse = oracle.ref_fwd(q, k, v, seg, 1)
    for b in range(B):
        firsts = [0] + [i for i in range(1, S) if seg[b, i] != seg[b, i - 1]]
        for i in firsts:  # causal: only key i is visible (start of a document)
            np.testing.assert_array_equal(out[b, i], v[b, i])
            for h in range(H):
                assert abs(lse[b, h, i] - np.dot(q[b, i, h], k[b, i, h]) / math.sqrt(D)) < 1e-12


def test_equal_scores_return_mean_of_visible_rows():
    B, S, H, D = 2, 50, 2, 8
    _, k, v = _qkv(9, B, S, H, D)
    q = np.zeros((B, S, H, D))
    seg = random_segment_ids(9, B, S, 12)
    for c in (1, 4):
        out, lse = oracle.ref_fwd(q, k, v, seg, c)
        for b in range(B):
            for i in range(S):
                js = [j for j in range(S) if (j // c) <= (i // c) and seg[b, j] == seg[b, i]]
                np.testing.assert_allclose(out[b, i], v[b, js].mean(axis=0), rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[b, :, i], math.log(len(js)), rtol=0, atol=1e-13)


def test_rows_sum_to_one_and_masked_entries_are_zero():
    B, S, H, D = 2, 45, 2, 8
    q, k, _ = _qkv(11, B, S, H, D)
    seg = random_segment_ids(11, B, S, 15)
    P = oracle.ref_probs(q, k, seg, 2)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-13)
    for b in range(B):
        for i in range(S):
            for j in range(S):
                if not ((i // 2) >= (j // 2) and seg[b, i] == seg[b, j]):
                    assert np.all(P[b, :, i, j] == 0.0)
    assert np.all(P >= 0)


def test_constant_v_rows_give_that_row():
    B, S, H, D = 1, 30, 2, 8
    q, k, _ = _qkv(12, B, S, H, D, scale=4.0)
    row = np.linspace(-2, 3, D)
    v = np.broadcast_to(row, (B, S, H, D)).copy()
    out, _ = oracle.ref_fwd(q, k, v, None, 1)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-13)


def test_no_visible_key_gives_zero_and_minus_inf():
    # segment mask and causal mask together can leave a row empty only with
    # non-monotone ids: row 1 has an id that appears only after it.
    q, k, v = _qkv(13, 1, 4, 1, 4)
    seg = np.array([[0, 1, 0, 1]])
    # row 1 sees key 1 (itself); build an empty row with c=1 and a query whose id never precedes it
    seg2 = np.array([[0, 2, 0, 0]])
    out, lse = oracle.ref_fwd(q, k, v, seg2, 1)
    assert np.isfinite(lse).sum() == 4  # every row sees itself
    out, lse = oracle.ref_fwd_rows(q, k, v, np.array([[0, 0, 1]]), seg, 1)
    assert np.isfinite(lse[0])
    # an empty row: query with an id that no key <= i has, by using the row API
    # with segment ids that differ between query and every earlier key
    vis = oatt.visible(np.array([1]), np.arange(4), 1, np.array([5]), seg[0])
    assert not vis.any()
    p, l = oatt._head_softmax(np.zeros((1, 4)), vis)
    assert np.all(p == 0) and l[0] == -np.inf


# --------------------------------------------------------------------------
# Backward
# --------------------------------------------------------------------------

def _loss(q, k, v, dout, seg, c):
    out, _ = oracle.ref_fwd(q, k, v, seg, c)
    return float((out * dout).sum())


@pytest.mark.parametrize("c,maxdoc", [(0, None), (1, None), (2, 3)])
def test_bwd_central_finite_differences(c, maxdoc):
    B, S, H, D = 1, 6, 2, 4
    q, k, v = _qkv(21 + c, B, S, H, D)
    dout = _rng(99).standard_normal((B, S, H, D))
    seg = None if maxdoc is None else random_segment_ids(3, B, S, maxdoc)
    dq, dk, dv = oracle.ref_bwd(q, k, v, dout, seg, c)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], dout, seg, c)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], dout, seg, c)) / (2 * eps)
        err = np.abs(num - g).max() / max(1.0, np.abs(g).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("B,S,H,D,c,maxdoc", CASES[:4])
def test_bwd_matches_torch_autograd(B, S, H, D, c, maxdoc):
    q, k, v = _qkv(300 + S, B, S, H, D)
    dout = _rng(301).standard_normal((B, S, H, D))
    seg = None if maxdoc is None else random_segment_ids(S + 2, B, S, maxdoc)
    dq, dk, dv = oracle.ref_bwd(q, k, v, dout, seg, c)
    _, mask = _torch_sdpa(q, k, v, seg, c)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask)[:, None])
    o.backward(torch.from_numpy(dout).permute(0, 2, 1, 3))
    np.testing.assert_allclose(dq, tq.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)


def test_bwd_invariants():
    """sum_j dK_j = 0 (rows of dS sum to zero) and sum_j dV_j = sum_i dO_i (rows of P sum to one)."""
    B, S, H, D = 2, 64, 2, 16
    q, k, v = _qkv(31, B, S, H, D)
    dout = _rng(32).standard_normal((B, S, H, D))
    seg = random_segment_ids(31, B, S, 20)
    dq, dk, dv = oracle.ref_bwd(q, k, v, dout, seg, 1)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), dout.sum(axis=1), rtol=0, atol=1e-12)


def test_bwd_head_blocked_matches_torch_autograd():
    B, S, H, D = 1, 70, 1, 8
    q, k, v = _qkv(41, B, S, H, D)
    dout = _rng(42).standard_normal((B, S, H, D))
    seg = random_segment_ids(41, B, S, 25)
    _, mask = _torch_sdpa(q, k, v, seg, 1)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask)[:, None])
    o.backward(torch.from_numpy(dout).permute(0, 2, 1, 3))
    rows = np.array([0, 1, 13, 37, 69])
    dq, dk, dv = oracle.ref_bwd_head_blocked(q[0, :, 0], k[0, :, 0], v[0, :, 0], dout[0, :, 0],
                                             seg[0], 1, rows, rows, block=16)
    np.testing.assert_allclose(dq, tq.grad[0, 0].numpy()[rows], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad[0, 0].numpy()[rows], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad[0, 0].numpy()[rows], rtol=0, atol=1e-11)


# --------------------------------------------------------------------------
# Chunk-skip reading
# --------------------------------------------------------------------------

def test_below_or_on_diag_brute_force():
    """The chunk test is true exactly when the chunk pair holds a visible causal element."""
    for c in (1, 2, 3, 8, 64):
        for Cq in (1, 4, 16):
            for Ck in (1, 4, 8):
                for qi in range(12):
                    for ki in range(12):
                        anyvis = any((i // c) >= (j // c)
                                     for i in range(qi * Cq, (qi + 1) * Cq)
                                     for j in range(ki * Ck, (ki + 1) * Ck))
                        assert oracle.below_or_on_diag(qi, Cq, ki, Ck, c) == anyvis


# --------------------------------------------------------------------------
# Planted mistakes: mutated copies of the oracle must fail the pins
# --------------------------------------------------------------------------

def _mutant(old, new):
    src = open(oatt.__file__).read()
    assert old in src, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    ("dropped scale", "    scale = 1.0 / math.sqrt(D)\n    for b in range(B):\n        seg = None if segment_ids is None else np.asarray(segment_ids)[b]\n        vis = visible(pos, pos, causal_block_size, seg, seg)\n        for h in range(H):\n            s = (q[b, :, h, :] @ k[b, :, h, :].T) * scale\n            p, lse_bh",
     "    scale = 1.0\n    for b in range(B):\n        seg = None if segment_ids is None else np.asarray(segment_ids)[b]\n        vis = visible(pos, pos, causal_block_size, seg, seg)\n        for h in range(H):\n            s = (q[b, :, h, :] @ k[b, :, h, :].T) * scale\n            p, lse_bh"),
    ("causal direction flipped", "vis &= (qpos // c) >= (kpos // c)", "vis &= (qpos // c) <= (kpos // c)"),
    ("k transposed for v", "out[b, :, h, :] = p @ v[b, :, h, :]", "out[b, :, h, :] = p @ k[b, :, h, :]"),
    ("lse missing max", "lse = np.where(has, m_safe + np.log(", "lse = np.where(has, 0.0 + np.log("),
    ("segment mask ignored", "vis &= np.asarray(qseg)[:, None] == np.asarray(kseg)[None, :]", "pass"),
]


@pytest.mark.parametrize("label,old,new", MUTATIONS)
def test_planted_forward_mistakes_are_caught(label, old, new):
    mod = _mutant(old, new)
    B, S, H, D, c, maxdoc = 2, 48, 2, 8, 1, 9
    q, k, v = _qkv(77, B, S, H, D)
    seg = random_segment_ids(77, B, S, maxdoc)
    out, lse = mod.ref_fwd(q, k, v, seg, c)
    ref, _ = _torch_sdpa(q, k, v, seg, c)
    caught = not np.allclose(out, ref, rtol=0, atol=1e-9)
    if not caught:  # the lse-only mutation: caught by the single-visible-key pin
        i = 0
        caught = any(abs(lse[0, h, i] - np.dot(q[0, i, h], k[0, i, h]) / math.sqrt(D)) > 1e-9
                     for h in range(H))
    assert caught, label


BWD_MUTATIONS = [
    ("delta sign", "dS = P * (dP - delta[:, None])\n            dq[b", "dS = P * (dP + delta[:, None])\n            dq[b"),
    ("dk missing scale", "dk[b, :, h] = (dS.T @ Q) * scale", "dk[b, :, h] = (dS.T @ Q)"),
    ("dv transposed", "dV = P.T @ dO", "dV = P @ dO"),
]


@pytest.mark.parametrize("label,old,new", BWD_MUTATIONS)
def test_planted_backward_mistakes_are_caught(label, old, new):
    mod = _mutant(old, new)
    B, S, H, D = 1, 20, 1, 4
    q, k, v = _qkv(88, B, S, H, D)
    dout = _rng(89).standard_normal((B, S, H, D))
    dq, dk, dv = mod.ref_bwd(q, k, v, dout, None, 1)
    _, mask = _torch_sdpa(q, k, v, None, 1)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask)[:, None])
    o.backward(torch.from_numpy(dout).permute(0, 2, 1, 3))
    ok = (np.allclose(dq, tq.grad.permute(0, 2, 1, 3).numpy(), atol=1e-9)
          and np.allclose(dk, tk.grad.permute(0, 2, 1, 3).numpy(), atol=1e-9)
          and np.allclose(dv, tv.grad.permute(0, 2, 1, 3).numpy(), atol=1e-9))
    assert not ok, label


def test_planted_ring_mistake_is_caught():
    """Dropping the lazy-softmax correction breaks agreement with the definition."""
    mod = _mutant("numerator[b, ql, h] = numerator[b, ql, h] * corr[:, None] + ew @ vch",
                  "numerator[b, ql, h] = numerator[b, ql, h] + ew @ vch")
    q, k, v = _qkv(3, 1, 64, 1, 8, scale=2.0)
    out, _ = oracle.ref_fwd(q, k, v, None, 1)
    o2, _ = mod.ref_ring_fwd(q, k, v, None, 1, 4, 8, 8)
    assert not np.allclose(o2, out, atol=1e-9)
