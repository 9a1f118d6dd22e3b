"""GPU parity of the forward (through the C ABI) against the CPU float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_exact_ra_gb300 import ops
from long_context_exact_ra_gb300.inputs import (WORKLOADS, Workload, make_inputs, random_segment_ids,
                                                sample_rows)
from tests.gpu_util import as_f64, check_lse, check_out, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def run_fwd(x, w, seg=None):
    q, k, v = (to_dev(getattr(x, n), w.dtype) for n in ("q", "k", "v"))
    sg = to_dev(seg, "i32") if seg is not None else None
    out, lse = ops.fwd(q, k, v, sg, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    ops.sync_check()
    return out, lse


def full_check(w, seg=None):
    x = make_inputs(w)
    if seg is None and w.segments:
        seg = x.segment_ids
    out, lse = run_fwd(x, w, seg)
    ref_out, ref_lse = oracle.ref_fwd(as_f64(x.q, w.dtype), as_f64(x.k, w.dtype), as_f64(x.v, w.dtype),
                                      seg, w.causal_block_size)
    e = check_out(host_f64(out), ref_out, w.dtype, scale=w.scale)
    le = check_lse(lse.cpu().numpy().astype(np.float64), ref_lse, w.dtype)
    return e, le


# ---------------------------------------------------------------- fp32 path
def test_config1_tiny_fp32_full():
    full_check(WORKLOADS[1])


@pytest.mark.parametrize("S,N,c,D,maxdoc", [(96, 3, 1, 32, None), (200, 4, 0, 128, 17), (256, 2, 5, 100, 40)])
def test_fp32_small_cases(S, N, c, D, maxdoc):
    w = Workload("fp32 small", 2, S, 3, D, "f32", c, N, S // N, S // N, seed=S + D)
    seg = None if maxdoc is None else random_segment_ids(S, 2, S, maxdoc)
    full_check(w, seg)


# ---------------------------------------------------------------- bf16 tensor-core path
SMALL_BF16 = [
    # S, N, causal c, D, chunk, seg max doc, scale
    (512, 4, 1, 128, 64, None, 1.0),
    (512, 4, 1, 64, 64, None, 1.0),
    (1024, 2, 0, 128, 256, None, 1.0),
    (1024, 8, 0, 64, 32, None, 1.0),
    (1200, 4, 1, 128, 100, None, 1.0),    # shard 300: ragged tiles inside every shard
    (1200, 3, 1, 64, 80, None, 1.0),      # shard 400, odd tile count -> absent second Q tile
    (768, 3, 3, 128, 128, None, 1.0),     # causal block size 3
    (640, 5, 100, 64, 128, None, 1.0),    # causal block 100: diagonal blocks cross tiles
    (1024, 4, 1, 128, 256, 300, 0.5),     # packed documents + causal
    (1024, 4, 0, 64, 256, 200, 1.0),      # segments, non-causal
    (896, 7, 1, 64, 128, 90, 3.0),        # large scores: exercises the deferred rescale
    (1200, 4, 1, 64, 100, 150, 1.0),      # segments with ragged shards (partial key tiles in the summary)
    (384, 1, 1, 128, 384, None, 1.0),     # one shard (plain blockwise attention)
]


@pytest.mark.parametrize("S,N,c,D,ch,maxdoc,scale", SMALL_BF16)
def test_bf16_small_full(S, N, c, D, ch, maxdoc, scale):
    w = Workload("bf16 small", 2, S, 3, D, "bf16", c, N, ch, ch, scale=scale, seed=S * 7 + D + c)
    seg = None if maxdoc is None else random_segment_ids(S + 1, 2, S, maxdoc)
    full_check(w, seg)


def test_bf16_deterministic():
    w = Workload("det", 1, 2048, 4, 128, "bf16", 1, 4, 512, 512, seed=3)
    x = make_inputs(w)
    o1, l1 = run_fwd(x, w)
    o2, l2 = run_fwd(x, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_sequence_is_a_noop():
    q = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out, lse = ops.fwd(q, q, q, None, 1, 1, 1, 1)
    assert out.shape == q.shape and lse.shape == (1, 2, 0)


def test_invalid_arguments_raise():
    q = torch.zeros((1, 100, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.RAError) as e:
        ops.fwd(q, q, q, None, 1, 3, 1, 1)  # 100 % 3
    assert e.value.status == ops.RA_ERR_INVALID_ARG
    q96 = torch.zeros((1, 128, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.RAError) as e:
        ops.fwd(q96, q96, q96, None, 1, 1, 1, 1)
    assert e.value.status == ops.RA_ERR_UNSUPPORTED


def test_bounded_wait_timeout_is_reported_and_context_survives():
    ops.selftest_timeout(2_000_000)  # 2 ms
    with pytest.raises(ops.RAError) as e:
        ops.sync_check()
    assert e.value.status == ops.RA_ERR_TIMEOUT
    ops.sync_check()  # cleared
    test_bf16_small_full(512, 4, 1, 64, 64, None, 1.0)  # the context still works


def test_kernel_launch_count():
    w = Workload("cnt", 1, 512, 2, 64, "bf16", 1, 4, 128, 128, seed=1)
    x = make_inputs(w)
    n0 = ops.kernel_launches()
    run_fwd(x, w)
    assert ops.kernel_launches() - n0 == 1


# ---------------------------------------------------------------- evaluation configs (sampled rows)
def sampled_check(w, nrows=4096):
    x = make_inputs(w)
    out, lse = run_fwd(x, w, x.segment_ids)
    rows = sample_rows(w.seed, w, nrows)
    qf, kf, vf = (as_f64(getattr(x, n), w.dtype) if w.seq <= 32768 else None for n in ("q", "k", "v"))
    if qf is None:  # very long: keep float32 views, the oracle upcasts per head
        from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32
        qf, kf, vf = (bf16_bits_to_f32(getattr(x, n)) for n in ("q", "k", "v"))
    ref_o, ref_l = oracle.ref_fwd_rows(qf, kf, vf, rows, x.segment_ids, w.causal_block_size)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    idx_b = torch.from_numpy(b).cuda()
    idx_h = torch.from_numpy(h).cuda()
    idx_i = torch.from_numpy(i).cuda()
    got_o = host_f64(out[idx_b, idx_i, idx_h])
    got_l = lse[idx_b, idx_h, idx_i].cpu().numpy().astype(np.float64)
    check_out(got_o, ref_o, w.dtype)
    check_lse(got_l, ref_l, w.dtype)
    return x, out, lse


def closed_form_checks(w, x, out, lse):
    """Full-size pins that need no oracle: causal row 0 sees only key 0."""
    if w.causal_block_size != 1:
        return
    v0 = torch.from_numpy(x.v[:, 0].view(np.int16)).view(torch.bfloat16)
    assert torch.equal(out[:, 0].cpu(), v0), "row 0 must equal v[0] exactly"
    q0 = as_f64(x.q[:, 0], w.dtype)
    k0 = as_f64(x.k[:, 0], w.dtype)
    expect = (q0 * k0).sum(-1) / math.sqrt(w.head_dim)  # [B, H]
    np.testing.assert_allclose(lse[:, :, 0].cpu().numpy(), expect, rtol=0, atol=1e-3)


@pytest.mark.parametrize("cfg", [2, 3])
def test_config_sampled_rows(cfg):
    w = WORKLOADS[cfg]
    x, out, lse = sampled_check(w)
    closed_form_checks(w, x, out, lse)


def test_packed_documents_with_more_key_tiles_than_the_segment_summary():
    """D = 64 with 9 x 32 shards x 16 tiles = 4,608 key tiles, more than the 4,096 entries of the
    kernel's shared-memory segment summary: the producer then reads each tile's ids itself."""
    w = Workload("packed documents B9 S65536 H1 D64, 32 shards", 9, 65536, 1, 64, "bf16", 1, 32, 2048, 2048,
                 scale=0.5, segments=True, seed=4242)
    sampled_check(w, nrows=2048)


@pytest.mark.slow
def test_config4_7b_long_context_sampled_rows():
    w = WORKLOADS[4]
    x, out, lse = sampled_check(w)
    closed_form_checks(w, x, out, lse)


def test_equal_scores_give_prefix_means_at_scale():
    """Q = 0: every visible score is equal, out_i = mean(v_0..v_i), lse_i = ln(i+1)."""
    w = Workload("q=0", 1, 16384, 4, 128, "bf16", 1, 8, 512, 512, seed=11)
    x = make_inputs(w)
    x.q[...] = 0
    out, lse = run_fwd(x, w)
    v = as_f64(x.v, "bf16")
    ref = np.cumsum(v, axis=1) / np.arange(1, w.seq + 1)[None, :, None, None]
    check_out(host_f64(out), ref, "bf16")
    np.testing.assert_allclose(lse.cpu().numpy()[0], np.log(np.arange(1, w.seq + 1))[None, :].repeat(4, 0),
                               rtol=0, atol=1e-3)
