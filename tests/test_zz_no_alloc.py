"""ra_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (fixed memory arenas, runtimes that forbid allocation after
start-up, code that must not synchronize the device) cannot provide ra_bwd's
workspace; ra_bwd_noalloc uses a scratch array built into the library instead.
This file is collected last so that a run stopping at the first failure has
already run every other test.  It checks, through the C ABI, that two calls in
a row give the same gradients as ra_bwd (within the gradient tolerance used by
the other backward tests), and that too-large problems are refused.
"""
import ctypes

import numpy as np
import pytest
import torch

from long_context_exact_ra_gb300 import ops
from long_context_exact_ra_gb300.inputs import Workload, make_inputs, random_segment_ids
from tests.gpu_util import check_grad, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def _raw_noalloc(q, k, v, out, lse, do, seg, w, dq, dk, dv):
    """Call the C entry point directly (ctypes), as a C caller would."""
    L = ops.lib()
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    B, S, H, D = q.shape
    st = L.ra_bwd_noalloc(P(q), P(k), P(v), P(out), P(lse), P(do), P(seg), w.causal_block_size, w.num_shards,
                          w.query_chunk_size, w.key_chunk_size, B, S, H, D,
                          ops.RA_BF16 if q.dtype == torch.bfloat16 else ops.RA_F32,
                          P(dq), P(dk), P(dv), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ops.RA_OK, L.ra_last_error()


@pytest.mark.parametrize("S,N,c,D,ch,maxdoc", [(1024, 4, 1, 128, 256, None), (768, 3, 0, 64, 128, 100)])
def test_noalloc_backward_matches_ra_bwd_twice(S, N, c, D, ch, maxdoc):
    w = Workload("no-alloc bwd", 2, S, 4, D, "bf16", c, N, ch, ch, backward=True, seed=S + D)
    x = make_inputs(w, with_dout=True)
    seg_np = None if maxdoc is None else random_segment_ids(S, 2, S, maxdoc)
    q, k, v, do = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout"))
    seg = None if seg_np is None else to_dev(seg_np, "i32")
    args = (seg, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    out, lse = ops.fwd(q, k, v, *args)
    rq, rk, rv = ops.bwd(q, k, v, out, lse, do, *args)
    ops.sync_check()
    ref = [host_f64(t) for t in (rq, rk, rv)]
    for call in range(2):  # the shared scratch keeps the previous call's contents
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        _raw_noalloc(q, k, v, out, lse, do, seg, w, dq, dk, dv)
        ops.sync_check()
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            got = host_f64(g)
            assert np.isfinite(got).all(), f"call {call}: {name} not written"
            check_grad(got, r, f"call {call}: {name}")


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    L = ops.lib()
    cap = L.ra_bwd_noalloc_max_scratch()
    assert cap == 64 << 20
    # B1 S8192 H32 D128 needs 128 MiB of dQ accumulator: refused before any GPU work
    B, S, H, D = 1, 8192, 32, 128
    assert L.ra_bwd_workspace_size(B, S, H, D, ops.RA_BF16) > cap
    P = ctypes.c_void_p(256)
    st = L.ra_bwd_noalloc(P, P, P, P, P, P, None, 1, 8, 1024, 1024, B, S, H, D, ops.RA_BF16, P, P, P, None)
    assert st == ops.RA_ERR_INVALID_ARG
    assert b"scratch" in L.ra_last_error()


def test_noalloc_fp32_path_through_the_binding_matches_ra_bwd_twice():
    """The fp32 path (the scratch holds only Delta there) through ops.bwd_noalloc."""
    w = Workload("no-alloc fp32", 1, 512, 2, 64, "f32", 0, 4, 128, 128, backward=True, seed=17)
    x = make_inputs(w, with_dout=True)
    q, k, v, do = (to_dev(getattr(x, n), "f32") for n in ("q", "k", "v", "dout"))
    args = (None, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    out, lse = ops.fwd(q, k, v, *args)
    ref = [host_f64(t) for t in ops.bwd(q, k, v, out, lse, do, *args)]
    ops.sync_check()
    for call in range(2):
        got = ops.bwd_noalloc(q, k, v, out, lse, do, *args)
        ops.sync_check()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            rel = (np.abs(host_f64(g) - r) / np.maximum(1.0, np.abs(r))).max()
            assert rel <= 1e-5, f"call {call}: {name}: max rel err {rel:.3e}"
