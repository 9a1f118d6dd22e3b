"""GPU parity of the ring steps across devices (ra_ring_fwd_step, ra_ring_bwd_*,
ra_ring_finish) against the CPU float64 oracle of the whole sequence.

A ring of N ranks is run on one GPU: `ring_forward_local` runs every rank's
steps in turn and hands each key/value block to the next rank between steps,
exactly the order of the paper review page's ring algorithm (环形注意力算法),
with the sequence cut into contiguous or striped blocks.  A second test runs
two real ranks (two processes on the one GPU, gloo with blocks staged through
host memory) through `ring_forward` / `ring_backward`.  The kernels of the two
processes never wait on each other: every exchange happens on the host between
launches.  Tolerances are those of the single-launch path.
"""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch

import oracle
from long_context_exact_ra_gb300 import ops, ring
from long_context_exact_ra_gb300.inputs import Workload, make_inputs, random_segment_ids
from tests.gpu_util import as_f64, check_grad, check_lse, check_out, host_f64, to_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


CASES = [
    # S, world, layout, causal c, D, max doc length (segments)
    (1024, 4, "contiguous", 1, 128, None),
    (1024, 4, "striped", 1, 128, None),
    (1200, 4, "contiguous", 1, 64, None),    # blocks of 300: ragged tiles
    (1200, 4, "striped", 1, 64, None),
    (768, 2, "contiguous", 3, 128, None),    # causal block size 3
    (768, 3, "striped", 0, 64, None),        # non-causal
    (1024, 4, "contiguous", 1, 128, 150),    # packed documents
    (1024, 2, "striped", 1, 64, 90),
    (512, 1, "contiguous", 1, 128, None),    # a ring of one: a single block
]


def _case(S, world, c, D, maxdoc, seed):
    w = Workload("ring", 2, S, 3, D, "bf16", c, world, S // world, S // world, backward=True, seed=seed)
    x = make_inputs(w, with_dout=True)
    seg = None if maxdoc is None else random_segment_ids(seed, 2, S, maxdoc)
    return w, x, seg


@pytest.mark.parametrize("S,world,layout,c,D,maxdoc", CASES)
def test_ring_local_matches_oracle(S, world, layout, c, D, maxdoc):
    w, x, seg = _case(S, world, c, D, maxdoc, seed=S + world * 7 + c + D)
    q, k, v, do = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout"))
    sg = None if seg is None else to_dev(seg, "i32")
    out, lse = ring.ring_forward_local(q, k, v, sg, c, world, layout)
    dq, dk, dv = ring.ring_backward_local(q, k, v, out, lse, do, sg, c, world, layout)
    ops.sync_check()
    f = [as_f64(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout")]
    ref_o, ref_l = oracle.ref_fwd(*f[:3], seg, c)
    check_out(host_f64(out), ref_o, "bf16")
    check_lse(lse.cpu().numpy().astype(np.float64), ref_l, "bf16")
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.ref_bwd(*f, seg, c)):
        check_grad(host_f64(g), r, name)


def test_ring_forward_equals_single_launch_forward_closely():
    """The same attention through the ring (4 contiguous blocks) and through one
    launch over 4 virtual shards: both are within bf16 rounding of each other."""
    w, x, _ = _case(2048, 4, 1, 128, None, seed=77)
    q, k, v = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v"))
    o1, l1 = ops.fwd(q, k, v, None, 1, 4, 512, 512)
    o2, l2 = ring.ring_forward_local(q, k, v, None, 1, 4, "contiguous")
    ops.sync_check()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * 2.0 ** -8
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_ring_step_rejects_strided_causal_blocks():
    q = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((1, 128, 1, 64), dtype=torch.float32, device="cuda")
    lse = torch.full((1, 1, 128), float("-inf"), device="cuda")
    with pytest.raises(ops.RAError) as e:
        ops.ring_fwd_step(q, q, q, None, None, 3, 0, 1, 4, o, lse)
    assert e.value.status == ops.RA_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------- two processes
def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _two_rank_worker(rank, world, port, layout, result_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=120))
    torch.cuda.set_device(0)
    from long_context_exact_ra_gb300 import ring as rg

    class HostStaged(rg.ProcessGroupTransport):
        """gloo moves CPU tensors: stage each block through pinned host memory."""

        def start(self, tensors):
            torch.cuda.current_stream().synchronize()
            p = super().start([t.cpu() for t in tensors])
            dev = tensors[0].device

            class _P:
                def wait(self_inner):
                    return [t.to(dev) for t in p.wait()]
            return _P()

    w, x, seg = _case(1024, world, 1, 128, 200, seed=31)
    dv_ = lambda a, kind="bf16": None if a is None else to_dev(a, kind)  # noqa: E731
    full = {n: dv_(getattr(x, n)) for n in ("q", "k", "v", "dout")}
    sg = dv_(seg, "i32")
    blk = {n: rg.shard(t, layout, world, rank) for n, t in full.items()}
    sb = rg.shard(sg, layout, world, rank)
    tr = HostStaged()
    out, lse = rg.ring_forward(blk["q"], blk["k"], blk["v"], sb, 1, layout, tr)
    dq, dk, dv = rg.ring_backward(blk["q"], blk["k"], blk["v"], out, lse, blk["dout"], sb, 1, layout, tr)
    from long_context_exact_ra_gb300 import ops as o
    o.sync_check()
    result_q.put((rank, *(t.float().cpu().numpy() for t in (out, lse, dq, dk, dv))))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_two_ranks_on_one_gpu_host_staged(layout):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    qq = ctx.Queue()
    procs = [ctx.Process(target=_two_rank_worker, args=(r, world, port, layout, qq), daemon=True) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((qq.get(timeout=300) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w, x, seg = _case(1024, world, 1, 128, 200, seed=31)
    T = lambda i: [torch.from_numpy(r[i]) for r in res]  # noqa: E731
    f = [as_f64(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout")]
    ref_o, ref_l = oracle.ref_fwd(*f[:3], seg, 1)
    check_out(ring.unshard(T(1), layout).numpy().astype(np.float64), ref_o, "bf16")
    check_lse(ring.unshard_lse(T(2), layout).numpy().astype(np.float64), ref_l, "bf16")
    for i, name, r in zip((3, 4, 5), ("dq", "dk", "dv"), oracle.ref_bwd(*f, seg, 1)):
        check_grad(ring.unshard(T(i), layout).numpy().astype(np.float64), r, name)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_of_eight_at_s16384_sampled_rows(layout):
    """A ring of 8 ranks over B1 S16384 H4 D128 (causal), forward and backward,
    against the float64 oracle on sampled rows: 512 forward rows (shard and tile
    edges forced), and dQ, dK, dV on 256 query and 256 key rows of one head with
    that head's full lse and Delta."""
    w = Workload("ring s16384", 1, 16384, 4, 128, "bf16", 1, 8, 2048, 2048, backward=True, seed=4242)
    x = make_inputs(w, with_dout=True)
    q, k, v, do = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v", "dout"))
    out, lse = ring.ring_forward_local(q, k, v, None, 1, 8, layout)
    dq, dk, dv = ring.ring_backward_local(q, k, v, out, lse, do, None, 1, 8, layout)
    ops.sync_check()
    from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32, sample_rows
    rows = sample_rows(w.seed, w, 512)
    qf, kf, vf = (bf16_bits_to_f32(getattr(x, n)) for n in ("q", "k", "v"))
    ref_o, ref_l = oracle.ref_fwd_rows(qf, kf, vf, rows, None, 1)
    ib, ih, ii = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    check_out(host_f64(out[ib, ii, ih]), ref_o, "bf16")
    check_lse(lse[ib, ih, ii].cpu().numpy().astype(np.float64), ref_l, "bf16")
    g = np.random.Generator(np.random.PCG64(17))
    h = int(g.integers(w.heads))
    qr = np.unique(np.concatenate([[0, 1, w.seq - 1], g.integers(w.seq, size=253)]))
    kr = np.unique(np.concatenate([[0, 2047, 2048, w.seq - 1], g.integers(w.seq, size=252)]))
    Q, K, V, dO = (as_f64(getattr(x, n)[0, :, h], "bf16") for n in ("q", "k", "v", "dout"))
    rq, rk, rv = oracle.ref_bwd_head_blocked(Q, K, V, dO, None, 1, qr, kr, block=2048)
    iq, ik = torch.from_numpy(qr).cuda(), torch.from_numpy(kr).cuda()
    check_grad(host_f64(dq[0, iq, h]), rq, "dq rows")
    check_grad(host_f64(dk[0, ik, h]), rk, "dk rows")
    check_grad(host_f64(dv[0, ik, h]), rv, "dv rows")
