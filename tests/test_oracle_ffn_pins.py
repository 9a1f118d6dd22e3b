"""Pins for the blockwise feed-forward oracle (oracle/ffn.py).

* An independent library routine: torch CPU float64 linear / relu.
* Chunking does not change the result (rows are independent), for chunk sizes
  that divide the rows, leave a ragged tail, or exceed the rows.
* Closed forms: W1 = 0 gives relu(b1) W2 + b2 on every row; pre-activations
  that are all negative give b2; the identity-like case with one hidden unit.
* Brute force with explicit Python loops on a tiny case.
* The bf16 rounding of the hidden activation is the round-to-nearest-even of the
  exact value (checked against torch's bf16 cast).
* Planted mistakes: mutated copies of the oracle must fail these pins.
"""
import types

import numpy as np
import pytest
import torch

from oracle import ffn as offn


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _params(seed, Dm, F):
    g = _rng(seed)
    w1 = g.standard_normal((F, Dm)) / np.sqrt(Dm)
    b1 = g.standard_normal(F) * 0.1
    w2 = g.standard_normal((Dm, F)) / np.sqrt(F)
    b2 = g.standard_normal(Dm) * 0.1
    return w1, b1, w2, b2


@pytest.mark.parametrize("B,L,Dm,F,chunk", [(2, 48, 16, 40, 16), (1, 100, 32, 64, 33), (3, 7, 8, 24, 64)])
def test_matches_torch_linear_relu(B, L, Dm, F, chunk):
    x = _rng(1).standard_normal((B, L, Dm))
    w1, b1, w2, b2 = _params(2, Dm, F)
    out = offn.ref_blockwise_ffn(x, w1, b1, w2, b2, chunk)
    t = torch.nn.functional
    ref = t.linear(t.relu(t.linear(torch.from_numpy(x), torch.from_numpy(w1), torch.from_numpy(b1))),
                   torch.from_numpy(w2), torch.from_numpy(b2)).numpy()
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_chunk_size_does_not_change_the_result():
    x = _rng(3).standard_normal((2, 90, 16))
    w1, b1, w2, b2 = _params(4, 16, 48)
    ref = offn.ref_blockwise_ffn(x, w1, b1, w2, b2, 180)
    for c in (1, 7, 30, 64, 179, 1000):  # equal up to the summation order of the matrix products
        assert np.allclose(offn.ref_blockwise_ffn(x, w1, b1, w2, b2, c), ref, rtol=0, atol=1e-12)


def test_closed_forms():
    g = _rng(5)
    x = g.standard_normal((1, 10, 8))
    _, b1, w2, b2 = _params(6, 8, 12)
    out = offn.ref_blockwise_ffn(x, np.zeros((12, 8)), b1, w2, b2, 4)
    assert np.allclose(out, np.maximum(b1, 0) @ w2.T + b2, atol=1e-14)
    # all pre-activations negative: the hidden layer is 0 and the output is b2
    x = np.abs(g.standard_normal((1, 6, 8)))
    w1 = -np.abs(g.standard_normal((12, 8)))
    out = offn.ref_blockwise_ffn(x, w1, -np.ones(12), w2, b2, 5)
    assert np.allclose(out, np.broadcast_to(b2, out.shape), atol=1e-14)
    # one hidden unit that copies input 0 (when positive) to output 1
    w1 = np.zeros((1, 4)); w1[0, 0] = 1.0
    w2 = np.zeros((4, 1)); w2[1, 0] = 1.0
    x = np.array([[[2.0, 5, 5, 5], [-3.0, 1, 1, 1]]])
    out = offn.ref_blockwise_ffn(x, w1, np.zeros(1), w2, np.zeros(4), 1)
    assert np.array_equal(out, np.array([[[0, 2.0, 0, 0], [0, 0, 0, 0]]]))


def test_brute_force_loops():
    g = _rng(7)
    x = g.standard_normal((1, 3, 4))
    w1, b1, w2, b2 = _params(8, 4, 5)
    out = offn.ref_blockwise_ffn(x, w1, b1, w2, b2, 2)
    for i in range(3):
        h = [max(0.0, sum(x[0, i, d] * w1[f, d] for d in range(4)) + b1[f]) for f in range(5)]
        for o in range(4):
            y = sum(h[f] * w2[o, f] for f in range(5)) + b2[o]
            assert abs(out[0, i, o] - y) < 1e-13


def test_hidden_bf16_rounding_is_round_to_nearest_even():
    v = _rng(9).standard_normal(20000) * 10
    got = offn._bf16_round(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, ref)


def _mutant(old, new):
    src = open(offn.__file__).read()
    assert old in src, old
    mod = types.ModuleType("ffn_mutant")
    exec(compile(src.replace(old, new, 1), "ffn_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    ("relu dropped", "h = np.maximum(h, 0.0)", "h = h"),
    ("first bias dropped", "h = x @ np.asarray(w1, dtype=np.float64).T + np.asarray(b1, dtype=np.float64)",
     "h = x @ np.asarray(w1, dtype=np.float64).T"),
    ("w2 not transposed", "return h @ np.asarray(w2, dtype=np.float64).T +", "return h @ np.asarray(w2, dtype=np.float64) +"),
    ("chunk rows shifted", "out[lo:hi] = ffn_rows(flat[lo:hi]", "out[lo:hi] = ffn_rows(flat[max(0, lo - 1):hi - 1]"),
]


@pytest.mark.parametrize("label,old,new", MUTATIONS)
def test_planted_mistakes_are_caught(label, old, new):
    mod = _mutant(old, new)
    x = _rng(10).standard_normal((2, 24, 16))
    w1, b1, w2, b2 = _params(11, 16, 16)
    t = torch.nn.functional
    ref = t.linear(t.relu(t.linear(torch.from_numpy(x), torch.from_numpy(w1), torch.from_numpy(b1))),
                   torch.from_numpy(w2), torch.from_numpy(b2)).numpy()
    try:
        out = mod.ref_blockwise_ffn(x, w1, b1, w2, b2, 8)
        caught = out.shape != ref.shape or not np.allclose(out, ref, atol=1e-9)
    except Exception:
        caught = True
    assert caught, label
