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


def _rows_with_edges(g, S, n_shards, n_total):
    """Rows 0, 1, S - 1, every shard boundary +-1 and every 128-row tile boundary
    (last row of a tile, first of the next), then uniform draws up to n_total."""
    forced = {0, 1, S - 1}
    sh = S // n_shards
    for j in range(n_shards + 1):
        forced.update((j * sh - 1, j * sh, j * sh + 1))
    for t in range(0, S + 1, 128):
        forced.update((t - 1, t))
    forced = np.array(sorted(i for i in forced if 0 <= i < S))
    extra = np.setdiff1d(np.arange(S), forced)
    pick = g.choice(extra, size=max(0, n_total - len(forced)), replace=False)
    return np.sort(np.concatenate([forced, pick]))


@pytest.mark.slow
def test_config5_sampled_rows_and_invariants():
    """The fwd+bwd evaluation shape at full size (B1 S65536 H32 D128, 8 shards, causal).

    * forward: out and lse on 4096 sampled (b, h, i) rows (shard and tile edges
      forced) against the float64 definition, and row 0 = v_0 exactly;
    * gradients on two drawn heads: dQ on 2048 query rows and dK, dV on 2048 key
      rows per head (4096 of each in all, shard and tile edges forced), against
      the float64 oracle with each head's full lse and Delta;
    * on every head: sum_j dV_j = sum_i dO_i (rows of P sum to one) and
      sum_j dK_j = 0 (every row of dS sums to zero: sum_j P_ij (dP_ij - Delta_i)
      = <dO_i, out_i> - Delta_i = 0).  The GPU meets both up to rounding: P, dS
      and the outputs are rounded to bf16 (8 significant bits: at most 2^-8
      relative, about 2^-9 in rms), and Delta comes from the bf16 out.  Three
      roundings (dS, the dK output, the out in Delta) each leave a sum of random
      sign over the 65536 rows of about 2^-9 times the column norm
      sqrt(sum_j g_j^2) of the gradient g, together about 2^-8 times it; the
      bound allows 8 times that plus 1e-2 absolute (over the 4096 (head, dim)
      columns the largest Gaussian deviation is about 4 of those units).  A wrong
      Delta, scale or mask makes the sums of the order of the column norm.
    """
    from concurrent.futures import ThreadPoolExecutor

    w = WORKLOADS[5]
    x = make_inputs(w, with_dout=True)
    q, k, v, do = (to_dev(getattr(x, n), w.dtype) for n in ("q", "k", "v", "dout"))
    cargs = (None, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    out, lse = ops.fwd(q, k, v, *cargs)
    dq, dk, dv = ops.bwd(q, k, v, out, lse, do, *cargs)
    ops.sync_check()
    S = w.seq
    # forward rows
    from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32, sample_rows
    from tests.gpu_util import check_lse, check_out
    rows = sample_rows(w.seed, w, 4096)
    qf, kf, vf = (bf16_bits_to_f32(getattr(x, n)) for n in ("q", "k", "v"))
    ref_o, ref_l = oracle.ref_fwd_rows(qf, kf, vf, rows, None, w.causal_block_size)
    ib, ih, ii = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    check_out(host_f64(out[ib, ii, ih]), ref_o, "bf16", what="out rows")
    check_lse(lse[ib, ih, ii].cpu().numpy().astype(np.float64), ref_l, "bf16")
    v0 = torch.from_numpy(x.v[:, 0].view(np.int16)).view(torch.bfloat16)
    assert torch.equal(out[:, 0].cpu(), v0), "row 0 must equal v[0] exactly"
    # gradients on two heads
    g = np.random.Generator(np.random.PCG64(5))
    heads = [int(h) for h in g.choice(w.heads, size=2, replace=False)]
    q_rows = [_rows_with_edges(g, S, w.num_shards, 2048) for _ in heads]
    k_rows = [_rows_with_edges(g, S, w.num_shards, 2048) for _ in heads]

    def head_ref(n):
        h = heads[n]
        Q, K, V, dO = (as_f64(getattr(x, a)[0, :, h], "bf16") for a in ("q", "k", "v", "dout"))
        return oracle.ref_bwd_head_blocked(Q, K, V, dO, None, w.causal_block_size, q_rows[n], k_rows[n], block=2048)

    with ThreadPoolExecutor(2) as ex:  # numpy releases the GIL in its array loops
        refs = list(ex.map(head_ref, range(2)))
    for n, h in enumerate(heads):
        rq, rk, rv = refs[n]
        iq, ik = torch.from_numpy(q_rows[n]).cuda(), torch.from_numpy(k_rows[n]).cuda()
        check_grad(host_f64(dq[0, iq, h]), rq, f"dq rows, head {h}")
        check_grad(host_f64(dk[0, ik, h]), rk, f"dk rows, head {h}")
        check_grad(host_f64(dv[0, ik, h]), rv, f"dv rows, head {h}")
    # invariants on every head
    do_sum = as_f64(x.dout, "bf16").sum(axis=1)[0]            # [H, D]
    for name, grad, target in (("dv", dv, do_sum), ("dk", dk, np.zeros_like(do_sum))):
        gd = grad.double()
        gsum = gd.sum(dim=1).cpu().numpy()[0]                  # [H, D]
        gnorm = torch.sqrt((gd ** 2).sum(dim=1)).cpu().numpy()[0]
        tol = 8 * 2.0 ** -8 * gnorm + 1e-2
        dev_ = np.abs(gsum - target)
        assert np.all(dev_ <= tol), f"sum of {name} rows: worst {dev_.max():.3e} (bound there {tol.flat[dev_.argmax()]:.3e})"


@pytest.mark.parametrize("D", [128, 64])
def test_backward_workspace_contents_do_not_matter(D):
    """ra_bwd_workspace_size's contents on entry do not matter: a workspace full of
    NaN bit patterns (0xFF bytes) gives the same gradients as a zeroed one.  The
    shape has a ragged last tile, whose columns past the sequence end read the
    unwritten tail of the (lse, Delta) rows; the masked tiles must give them P = 0
    and dS = 0 without multiplying by those entries."""
    w = Workload("ws contents", 1, 1200, 2, D, "bf16", 1, 4, 100, 100, backward=True, seed=99 + D)
    x = make_inputs(w, with_dout=True)
    q, k, v, do = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout"))
    cargs = (None, 1, 4, 100, 100)
    out, lse = ops.fwd(q, k, v, *cargs)
    need = ops.bwd_workspace_size(1, 1200, 2, D, torch.bfloat16)
    grads = []
    for fill in (0, 255):
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        grads.append(ops.bwd(q, k, v, out, lse, do, *cargs, workspace=ws))
    ops.sync_check()
    rq, rk, rv = oracle.ref_bwd(*(as_f64(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout")), None, 1)
    for g in grads:
        for name, t, r in zip(("dq", "dk", "dv"), g, (rq, rk, rv)):
            got = host_f64(t)
            assert np.isfinite(got).all(), name
            check_grad(got, r, name)
