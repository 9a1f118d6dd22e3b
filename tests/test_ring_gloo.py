"""The ring driver on CPU ranks (gloo, world sizes 2 and 4): every rank holds one
block of the sequence, the key/value blocks (and in the backward their dK, dV)
travel around the ring with real send/receive, and the device work of each step
is the float64 stand-in of tests/ring_fake.py.  The gathered result must equal
the CPU oracle's attention (and gradients) of the whole sequence, for
contiguous and striped blocks, causal or not, with and without segment ids:
the ring order, the exchange and the position bookkeeping are then right
(paper review page of Ring Attention, 环形通信 / 环形注意力算法; the result does
not depend on the block order, 排列不变性)."""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CASES = [
    # world, layout, causal block size, segments
    (2, "contiguous", 1, False),
    (4, "contiguous", 1, True),
    (4, "contiguous", 3, False),
    (2, "striped", 1, False),
    (4, "striped", 1, True),
    (4, "striped", 0, False),
    (2, "contiguous", 0, True),
]


def _inputs(seed, B=2, S=48, H=2, D=8, segments=False):
    g = np.random.default_rng(seed)
    q, k, v, do = (g.standard_normal((B, S, H, D)) for _ in range(4))
    seg = None
    if segments:
        seg = np.cumsum(g.random((B, S)) < 0.15, axis=1).astype(np.int32)
    return q, k, v, do, seg


def _worker(rank, ws, port, layout, c, segments, q_out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=datetime.timedelta(seconds=120))
    from long_context_exact_ra_gb300 import ring
    from tests.ring_fake import Float64RingKernels
    q, k, v, do, seg = (None if a is None else torch.from_numpy(a) for a in _inputs(ws * 10 + c, segments=segments))
    blk = lambda x: None if x is None else ring.shard(x, layout, ws, rank)  # noqa: E731
    kern = Float64RingKernels()
    tr = ring.ProcessGroupTransport()
    out, lse = ring.ring_forward(blk(q), blk(k), blk(v), blk(seg), c, layout, tr, kern)
    dq, dk, dv = ring.ring_backward(blk(q), blk(k), blk(v), out, lse, blk(do), blk(seg), c, layout, tr, kern)
    q_out.put((rank, out.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,c,segments", CASES)
def test_ring_driver_on_gloo_ranks_matches_the_oracle(world, layout, c, segments):
    import oracle
    from long_context_exact_ra_gb300 import ring
    port = _free_port()
    ctx = mp.get_context("spawn")
    qq = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, layout, c, segments, qq), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((qq.get(timeout=120) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, do, seg = _inputs(world * 10 + c, segments=segments)
    ref_o, ref_l = oracle.ref_fwd(q, k, v, seg, c)
    ref_g = oracle.ref_bwd(q, k, v, do, seg, c)
    T = lambda i: [torch.from_numpy(r[i]) for r in res]  # noqa: E731
    out = ring.unshard(T(1), layout).numpy()
    lse = ring.unshard_lse(T(2), layout).numpy()
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-10)
    for i, r in zip((3, 4, 5), ref_g):
        np.testing.assert_allclose(ring.unshard(T(i), layout).numpy(), r, rtol=0, atol=1e-10)


def test_layouts_round_trip_and_positions():
    from long_context_exact_ra_gb300 import ring
    x = torch.arange(2 * 12 * 3).reshape(2, 12, 3)
    for layout in ring.LAYOUTS:
        blocks = [ring.shard(x, layout, 4, r) for r in range(4)]
        assert torch.equal(ring.unshard(blocks, layout), x)
        for r in range(4):
            p0, st = ring.block_positions(layout, r, 4, 3)
            pos = p0 + st * torch.arange(3)
            assert torch.equal(blocks[r][0, :, 0] // 3, pos)  # element value // 3 = its position


def test_unsupported_layouts_are_rejected_before_any_transfer():
    from long_context_exact_ra_gb300 import ring
    x = torch.zeros(1, 8, 1, 4)
    with pytest.raises(ValueError):
        ring.ring_forward_local(x, x, x, None, 3, 2, "striped")
    with pytest.raises(ValueError):
        ring.ring_backward(x, x, x, x, x, x, None, 2, "striped", transport=object(), kernels=object())
    with pytest.raises(ValueError):
        ring.ring_forward(x, x, x, None, 1, "diagonal", transport=object(), kernels=object())
