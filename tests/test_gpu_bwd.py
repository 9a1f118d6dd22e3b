"""GPU parity of the backward (through the C ABI) against the CPU float64 oracle.

The gradients are those of L = sum(dO * out); the GPU backward takes the
GPU forward's own out and lse (as a caller would), the oracle computes the
exact gradients from q, k, v, dO.  Bound (no target is stated for gradients,
derived from bf16 rounding of P, dS and the outputs):
max |err| / max(1, |ref|) <= 2e-2 and mean |err| <= 2e-3; the fp32 path is
held to 1e-5 in the same relative form.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_exact_ra_gb300 import ops
from long_context_exact_ra_gb300.inputs import WORKLOADS, Workload, make_inputs, random_segment_ids
from tests.gpu_util import as_f64, check_grad, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def run_fwd_bwd(x, w, seg):
    q, k, v, do = (to_dev(getattr(x, n), w.dtype) for n in ("q", "k", "v", "dout"))
    sg = to_dev(seg, "i32") if seg is not None else None
    cargs = (sg, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    out, lse = ops.fwd(q, k, v, *cargs)
    dq, dk, dv = ops.bwd(q, k, v, out, lse, do, *cargs)
    ops.sync_check()
    return dq, dk, dv


def full_bwd_check(w, seg=None):
    x = make_inputs(w, with_dout=True)
    if seg is None and w.segments:
        seg = x.segment_ids
    dq, dk, dv = run_fwd_bwd(x, w, seg)
    rq, rk, rv = oracle.ref_bwd(*(as_f64(getattr(x, n), w.dtype) for n in ("q", "k", "v", "dout")),
                                seg, w.causal_block_size)
    out = {}
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        got = host_f64(g)
        if w.dtype == "f32":
            rel = (np.abs(got - r) / np.maximum(1.0, np.abs(r))).max()
            assert rel <= 1e-5, f"{name}: max rel err {rel:.3e}"
        else:
            out[name] = check_grad(got, r, name)
    return out


@pytest.mark.parametrize("S,N,c,D,maxdoc", [(128, 4, 1, 64, None), (200, 4, 0, 32, 17), (256, 2, 3, 128, 40)])
def test_fp32_backward(S, N, c, D, maxdoc):
    w = Workload("fp32 bwd", 2, S, 2, D, "f32", c, N, S // N, S // N, seed=S + c)
    seg = None if maxdoc is None else random_segment_ids(S, 2, S, maxdoc)
    full_bwd_check(w, seg)


def test_config1_shape_fp32_backward():
    full_bwd_check(WORKLOADS[1])


SMALL_BF16 = [
    # S, N, causal c, D, chunk, seg max doc
    (512, 4, 1, 128, 64, None),
    (512, 4, 1, 64, 64, None),
    (1024, 2, 0, 128, 256, None),
    (768, 4, 0, 64, 64, None),
    (1200, 4, 1, 128, 100, None),   # ragged tiles in every shard
    (1200, 3, 1, 64, 80, None),
    (768, 3, 3, 128, 128, None),    # causal block size 3
    (640, 5, 100, 64, 128, None),   # causal block 100
    (1024, 4, 1, 128, 256, 300),    # packed documents + causal
    (1024, 4, 0, 64, 256, 200),     # segments, non-causal
    (384, 1, 1, 128, 384, None),
]


@pytest.mark.parametrize("S,N,c,D,ch,maxdoc", SMALL_BF16)
def test_bf16_backward_small(S, N, c, D, ch, maxdoc):
    w = Workload("bf16 bwd", 2, S, 3, D, "bf16", c, N, ch, ch, seed=S * 5 + D + c)
    seg = None if maxdoc is None else random_segment_ids(S + 3, 2, S, maxdoc)
    full_bwd_check(w, seg)


def test_config5_full_on_seq1024_slice():
    """The fwd+bwd evaluation shape (32 heads, D 128, 8 shards, causal) at seq 1024, compared in full."""
    w5 = WORKLOADS[5]
    w = w5.with_(name="cfg5 shape at seq 1024", seq=1024, query_chunk_size=128, key_chunk_size=128)
    full_bwd_check(w)


def test_backward_launches_three_kernels():
    w = Workload("cnt", 1, 512, 2, 64, "bf16", 1, 4, 128, 128, backward=True, seed=1)
    x = make_inputs(w)
    q, k, v, do = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout"))
    out, lse = ops.fwd(q, k, v, None, 1, 4, 128, 128)
    n0 = ops.kernel_launches()
    ops.bwd(q, k, v, out, lse, do, None, 1, 4, 128, 128)
    ops.sync_check()
    assert ops.kernel_launches() - n0 == 3


@pytest.mark.slow
def test_config5_sampled_rows_and_invariants():
    """Full evaluation shape (B1 S65536 H32 D128, 8 shards): gradients of one head on
    sampled query and key rows against the float64 oracle, and sum_j dV_j = sum_i dO_i
    (rows of P sum to one) on every head."""
    w = WORKLOADS[5]
    x = make_inputs(w, with_dout=True)
    dq, dk, dv = run_fwd_bwd(x, w, None)
    g = np.random.Generator(np.random.PCG64(5))
    h = int(g.integers(w.heads))
    S = w.seq
    rows = np.unique(np.concatenate([[0, 1, S // 2, S - 2, S - 1], g.integers(S, size=59)]))
    Q, K, V, dO = (as_f64(getattr(x, n)[0, :, h], "bf16") for n in ("q", "k", "v", "dout"))
    rq, rk, rv = oracle.ref_bwd_head_blocked(Q, K, V, dO, None, w.causal_block_size, rows, rows, block=2048)
    idx = torch.from_numpy(rows).cuda()
    check_grad(host_f64(dq[0, idx, h]), rq, "dq rows")
    check_grad(host_f64(dk[0, idx, h]), rk, "dk rows")
    check_grad(host_f64(dv[0, idx, h]), rv, "dv rows")
    # invariant on every head: columns of P sum ... rows of P sum to one => sum_j dV_j = sum_i dO_i
    dv_sum = dv.double().sum(dim=1).cpu().numpy()[0]           # [H, D]
    do_sum = as_f64(x.dout, "bf16").sum(axis=1)[0]            # [H, D]
    dv_rms = np.sqrt((dv.double() ** 2).sum(dim=1).cpu().numpy()[0])
    tol = 8 * 2.0 ** -9 * dv_rms + 1e-2
    assert np.all(np.abs(dv_sum - do_sum) <= tol), np.abs(dv_sum - do_sum).max()
