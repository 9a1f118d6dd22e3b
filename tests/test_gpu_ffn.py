"""GPU parity of the blockwise feed-forward (ra_blockwise_ffn, through the C ABI)
against the CPU float64 oracle (oracle/ffn.py)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_exact_ra_gb300 import ops
from long_context_exact_ra_gb300.inputs import FFN_WORKLOADS, FfnWorkload, make_ffn_inputs
from tests.gpu_util import host_f64

pytestmark = pytest.mark.gpu

# Two oracles.  The exact one is the definition FFN(x) = max(0, x W1 + b1) W2 + b2
# in float64 (paper review page; blockwise feed-forward page, §核心技术原理).
# bf16 keeps 8 significant bits: rounding moves a value by at most 2^-8 of itself,
# by about 2^-9 of itself in rms.  The kernel rounds twice:
#   * the output, at most 2^-8 |y|;
#   * the hidden activation, which it stores in bf16 between the two products.
#     Through w2 ~ N(0, 1/F) that moves an output by a sum of F small terms of
#     random sign, sigma ~ 2^-9 x rms(hidden) ~ 1.4e-3 (the hidden rms is ~0.7).
# Bound against the exact definition: 2^-8 + 8 sigma ~ 1.5e-2 relative to
# max(1, |y|); the mean stays near 1.3e-3 (a float64 model of the two roundings
# gives max 0.009 and mean 0.0013 on these shapes).  The emulating oracle rounds
# the hidden activation as the kernel stores it, which leaves the output's own
# rounding (2^-8) and fp32 accumulation order: a bound of 5e-3.
FFN_MAX_REL = 1.5e-2   # max |err| / max(1, |ref|), against the exact definition
FFN_MEAN_ABS = 2e-3
FFN_EMU_MAX_REL = 5e-3  # against the oracle that rounds the hidden activation as the kernel stores it


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def _dev(xi):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    f32 = lambda a: None if a is None else torch.from_numpy(a).cuda()  # noqa: E731
    return bf(xi.x), bf(xi.w1), f32(xi.b1), bf(xi.w2), f32(xi.b2)


def run(xi, chunk=None):
    x, w1, b1, w2, b2 = _dev(xi)
    before = ops.kernel_launches()
    out = ops.blockwise_ffn(x, w1, b1, w2, b2, chunk or xi.w.chunk_size)
    ops.sync_check()
    return out, ops.kernel_launches() - before


def check(got, ref, max_rel=FFN_MAX_REL, what="exact"):
    err = np.abs(got - ref)
    rel = (err / np.maximum(1.0, np.abs(ref))).max()
    assert rel <= max_rel, f"{what}: max rel err {rel:.3e}"
    assert err.mean() <= FFN_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"


SMALL = [
    # B, L, Dm, F, chunk, bias
    (2, 300, 256, 512, 128, True),    # ragged last chunk
    (1, 128, 64, 136, 1000, True),    # one chunk; F not a multiple of 64 (K tail) nor of 256 (N tail)
    (1, 520, 200, 264, 256, True),    # Dm and F both ragged against the 64 / 256 tiles
    (3, 77, 128, 1024, 50, True),     # chunks of 50 rows: every M tile ragged
    (2, 256, 512, 1536, 256, False),  # no biases
]


@pytest.mark.parametrize("B,L,Dm,F,chunk,bias", SMALL)
def test_ffn_small_full(B, L, Dm, F, chunk, bias):
    xi = make_ffn_inputs(FfnWorkload("ffn small", B, L, Dm, F, chunk, seed=L + F, bias=bias))
    out, launches = run(xi)
    assert launches == 2 * ((B * L + chunk - 1) // chunk)
    args = (xi.as_f64("x"), xi.as_f64("w1"), xi.as_f64("b1") if bias else np.zeros(F),
            xi.as_f64("w2"), xi.as_f64("b2") if bias else np.zeros(Dm), chunk)
    got = host_f64(out)
    check(got, oracle.ref_blockwise_ffn(*args, round_hidden_bf16=False))
    check(got, oracle.ref_blockwise_ffn(*args, round_hidden_bf16=True), FFN_EMU_MAX_REL, "emulated")


def test_ffn_chunk_size_does_not_change_the_result():
    """Rows are independent and every output element accumulates its K blocks in the
    same order whatever the chunking, so the results are bit-identical."""
    xi = make_ffn_inputs(FfnWorkload("ffn chunks", 1, 1000, 256, 768, 1000, seed=9))
    a, _ = run(xi, 1000)
    b, _ = run(xi, 300)
    c, _ = run(xi, 128)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_ffn_7b_sampled_rows():
    """The 7B shape (Dm 4096, F 11008) on 16384 rows in chunks of 8192: chunk edges and drawn rows."""
    w = FFN_WORKLOADS["7b"]
    xi = make_ffn_inputs(w)
    out, _ = run(xi)
    g = np.random.Generator(np.random.PCG64(55))
    rows = sorted({0, 1, 127, 128, w.chunk_size - 1, w.chunk_size, w.chunk_size + 1, w.seq - 1}
                  | set(g.integers(w.seq, size=40).tolist()))
    x = xi.as_f64("x")[0, rows]
    args = (x, xi.as_f64("w1"), xi.as_f64("b1"), xi.as_f64("w2"), xi.as_f64("b2"))
    got = host_f64(out)[0, rows]
    check(got, oracle.ffn_rows(*args, round_hidden_bf16=False))
    check(got, oracle.ffn_rows(*args, round_hidden_bf16=True), FFN_EMU_MAX_REL, "emulated")
