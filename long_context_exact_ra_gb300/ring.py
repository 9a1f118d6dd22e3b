"""Ring Attention across devices: the host driver of the ring steps.

Each device (rank r of N) holds one block of the sequence: its query block and,
at ring step i, the key/value block k = (r - i) mod N that has travelled i hops
around the ring ("Ring Attention with Blockwise Transformers for Near-Infinite
Context", paper review page, 环形通信 and 环形注意力算法).  Every step the device
combines its queries with the block it holds (ra_ring_fwd_step, the lazy-softmax
merge of the code walk-through page "从论文到代码：深入理解RingAttention的块注意力计算逻辑",
环形计算模式 and §2), while the block is passed on to rank r + 1 and the next one
arrives from rank r - 1, so that the transfer hides behind the block's compute
(the paper review page's condition: block compute time > block transfer time).
The backward sends the key/value blocks around again, each with float32 dK, dV
accumulators that every rank adds its share to; after N hops they are home.

Two ways of cutting the sequence into blocks:
  * contiguous: rank r holds positions r*L .. r*L + L - 1 (L = S / N);
  * striped: rank r holds positions r, r + N, r + 2N, ... (Striped Attention,
    named on the paper review page, 相关工作 / 局限性, as the fix for the causal
    imbalance of contiguous blocks: every rank then has about the same number of
    visible pairs at every step).

The device work is the C ABI of libra.so (`ops.ring_*`); this module only
orders the calls and moves blocks.  `ring_forward` / `ring_backward` run one
rank of a torch.distributed group; `ring_forward_local` / `ring_backward_local`
run all N ranks of a ring in one process (the blocks are handed from rank to
rank in place of the send/receive), which is how a ring is exercised on one GPU.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

LAYOUTS = ("contiguous", "striped")


# ----------------------------------------------------------------------------- layout
def block_positions(layout: str, rank: int, world: int, block_len: int):
    """(first position, stride) of the block held by `rank`."""
    if layout == "contiguous":
        return rank * block_len, 1
    if layout == "striped":
        return rank, world
    raise ValueError(f"unknown layout {layout!r} (one of {LAYOUTS})")


def shard(x: torch.Tensor, layout: str, world: int, rank: int) -> torch.Tensor:
    """Block `rank` of x along the sequence axis (axis 1 of [B, S, ...])."""
    S = x.shape[1]
    if S % world != 0:
        raise ValueError(f"seq {S} is not divisible by the ring size {world}")
    L = S // world
    if layout == "contiguous":
        return x[:, rank * L:(rank + 1) * L].contiguous()
    if layout == "striped":
        return x[:, rank::world].contiguous()
    raise ValueError(f"unknown layout {layout!r}")


def unshard(blocks, layout: str) -> torch.Tensor:
    """Inverse of `shard` over all ranks' blocks (axis 1)."""
    world = len(blocks)
    if layout == "contiguous":
        return torch.cat(blocks, dim=1)
    if layout == "striped":
        b0 = blocks[0]
        out = b0.new_empty((b0.shape[0], b0.shape[1] * world) + tuple(b0.shape[2:]))
        for r, b in enumerate(blocks):
            out[:, r::world] = b
        return out
    raise ValueError(f"unknown layout {layout!r}")


def shard_lse(lse: torch.Tensor, layout: str, world: int, rank: int) -> torch.Tensor:
    """Block `rank` of a [B, H, S] tensor (sequence on axis 2)."""
    return shard(lse.transpose(1, 2), layout, world, rank).transpose(1, 2).contiguous()


def unshard_lse(blocks, layout: str) -> torch.Tensor:
    return unshard([b.transpose(1, 2) for b in blocks], layout).transpose(1, 2).contiguous()


def check_layout(layout: str, causal_block_size: int) -> None:
    """Reject what the ring-step calls do not support, before any block moves (a rank
    that failed inside the ring would leave its neighbours waiting on a transfer)."""
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout!r} (one of {LAYOUTS})")
    if causal_block_size < 0:
        raise ValueError("causal_block_size must be >= 0")
    if layout == "striped" and causal_block_size > 1:
        raise ValueError("striped blocks support causal_block_size 0 or 1")


def block_sees_nothing(layout: str, c: int, q0: int, k0: int, L: int) -> bool:
    """True when no key of the k/v block is visible to any query of the block (the
    step can be skipped; the kernels would skip every tile of it anyway)."""
    if c <= 0 or layout != "contiguous":
        return False
    return (q0 + L - 1) // c < k0 // c


# ----------------------------------------------------------------------------- device calls
class CudaRingKernels:
    """The device work of one ring step, through the C ABI (libra.so)."""

    def __init__(self):
        from . import ops  # loads the library; raises when it is missing
        self.ops = ops

    def fwd_carry(self, q):
        B, L, H, D = q.shape
        o = torch.zeros((B, L, H, D), dtype=torch.float32, device=q.device)
        lse = torch.full((B, H, L), float("-inf"), dtype=torch.float32, device=q.device)
        return o, lse

    def fwd_step(self, q, k, v, qseg, kseg, c, q0, k0, stride, o, lse):
        self.ops.ring_fwd_step(q, k, v, qseg, kseg, c, q0, k0, stride, o, lse)

    def fwd_finish(self, o, like):
        out = torch.empty_like(like)
        self.ops.ring_finish(o, out)
        return out

    def bwd_begin(self, out, lse, dout):
        B, L, H, D = out.shape
        ws = torch.empty(max(16, self.ops.ring_bwd_workspace_size(B, L, H, D)), dtype=torch.uint8, device=out.device)
        self.ops.ring_bwd_begin(out, lse, dout, ws)
        return ws

    def grad_carry(self, k):
        return torch.zeros(k.shape, dtype=torch.float32, device=k.device)

    def bwd_step(self, q, k, v, dout, qseg, kseg, c, q0, k0, stride, dk, dv, ws):
        self.ops.ring_bwd_step(q, k, v, dout, qseg, kseg, c, q0, k0, stride, dk, dv, ws)

    def bwd_end(self, ws, like):
        dq = torch.empty_like(like)
        self.ops.ring_bwd_end(ws, dq)
        return dq

    def grad_finish(self, g, like):
        out = torch.empty_like(like)
        self.ops.ring_finish(g, out)
        return out


# ----------------------------------------------------------------------------- transport
class ProcessGroupTransport:
    """Send to rank + 1 and receive from rank - 1 over a torch.distributed group
    (NCCL for CUDA tensors, gloo for CPU tensors).  `start` posts the exchange and
    returns a handle whose `wait()` gives the received tensors, so the caller can
    compute while the transfer is in flight."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _peer(self, r):
        r %= self.world
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def start(self, tensors):
        recv = [torch.empty_like(t) for t in tensors]
        ops = [self.dist.P2POp(self.dist.isend, t, self._peer(self.rank + 1), self.group) for t in tensors]
        ops += [self.dist.P2POp(self.dist.irecv, t, self._peer(self.rank - 1), self.group) for t in recv]
        reqs = self.dist.batch_isend_irecv(ops)
        return _Pending(reqs, recv)


@dataclass
class _Pending:
    reqs: list
    recv: list

    def wait(self):
        for r in self.reqs:
            r.wait()
        return self.recv


# ----------------------------------------------------------------------------- one ring step
def _fwd_step(kern, layout, c, rank, world, L, q, qseg, kv, o, lse, step):
    """Ring step `step` of rank `rank`: its queries against the k/v block it holds,
    which is block (rank - step) mod world."""
    kb = (rank - step) % world
    q0, stride = block_positions(layout, rank, world, L)
    k0, _ = block_positions(layout, kb, world, L)
    k, v, kseg = kv
    if not block_sees_nothing(layout, c, q0, k0, L):
        kern.fwd_step(q, k, v, qseg, kseg, c, q0, k0, stride, o, lse)


def _bwd_step(kern, layout, c, rank, world, L, q, dout, qseg, kvg, ws, step):
    kb = (rank - step) % world
    q0, stride = block_positions(layout, rank, world, L)
    k0, _ = block_positions(layout, kb, world, L)
    k, v, kseg, dk, dv = kvg
    if not block_sees_nothing(layout, c, q0, k0, L):
        kern.bwd_step(q, k, v, dout, qseg, kseg, c, q0, k0, stride, dk, dv, ws)


def _with_seg(tensors, seg):
    return list(tensors) + ([seg] if seg is not None else [])


def _split_seg(tensors, n, has_seg):
    return tuple(tensors[:n]) + ((tensors[n] if has_seg else None),)


# ----------------------------------------------------------------------------- distributed driver
def ring_forward(q, k, v, segment_ids=None, causal_block_size=0, layout="contiguous", transport=None,
                 kernels=None):
    """Forward of this rank's block: q, k, v [B, L, H, D] and segment_ids [B, L] are
    the block the rank holds under `layout`.  Returns (out [B, L, H, D] like q,
    lse [B, H, L] float32) for the rank's queries."""
    check_layout(layout, causal_block_size)
    tr = transport or ProcessGroupTransport()
    kern = kernels or CudaRingKernels()
    rank, world = tr.rank, tr.world
    L = q.shape[1]
    o, lse = kern.fwd_carry(q)
    has_seg = segment_ids is not None
    kv = (k, v, segment_ids)
    for step in range(world):
        pending = tr.start(_with_seg(kv[:2], kv[2])) if step + 1 < world else None
        _fwd_step(kern, layout, causal_block_size, rank, world, L, q, segment_ids, kv, o, lse, step)
        if pending is not None:
            kv = _split_seg(pending.wait(), 2, has_seg)
    return kern.fwd_finish(o, q), lse


def ring_backward(q, k, v, out, lse, dout, segment_ids=None, causal_block_size=0, layout="contiguous",
                  transport=None, kernels=None):
    """Backward of this rank's block (out, lse from ring_forward).  The k/v blocks
    travel around the ring again, each with its float32 dK, dV; the next block is
    posted before the current one's gradients are computed, and the gradients
    follow once they are.  Returns (dq, dk, dv) for the rank's own block."""
    check_layout(layout, causal_block_size)
    tr = transport or ProcessGroupTransport()
    kern = kernels or CudaRingKernels()
    rank, world = tr.rank, tr.world
    L = q.shape[1]
    has_seg = segment_ids is not None
    ws = kern.bwd_begin(out, lse, dout)
    k_cur, v_cur, s_cur = k, v, segment_ids
    dk, dv = kern.grad_carry(k), kern.grad_carry(v)
    for step in range(world):
        pend_kv = tr.start(_with_seg((k_cur, v_cur), s_cur)) if step + 1 < world else None
        _bwd_step(kern, layout, causal_block_size, rank, world, L, q, dout, segment_ids,
                  (k_cur, v_cur, s_cur, dk, dv), ws, step)
        # after the last step this hop brings every block's gradients home
        pend_g = tr.start([dk, dv]) if world > 1 else None
        if pend_kv is not None:
            k_cur, v_cur, s_cur = _split_seg(pend_kv.wait(), 2, has_seg)
        if pend_g is not None:
            dk, dv = pend_g.wait()
    return kern.bwd_end(ws, q), kern.grad_finish(dk, k), kern.grad_finish(dv, v)


# ----------------------------------------------------------------------------- one-process ring
def ring_forward_local(q, k, v, segment_ids=None, causal_block_size=0, world=2, layout="contiguous",
                       kernels=None):
    """All `world` ranks of a ring in one process, on full [B, S, H, D] tensors:
    the sequence is cut into blocks under `layout`, every rank's step runs in
    turn, and the blocks move to the next rank between steps.  Returns the full
    (out, lse) in sequence order."""
    check_layout(layout, causal_block_size)
    kern = kernels or CudaRingKernels()
    L = q.shape[1] // world
    qs = [shard(q, layout, world, r) for r in range(world)]
    segs = [None if segment_ids is None else shard(segment_ids, layout, world, r) for r in range(world)]
    held = [(shard(k, layout, world, r), shard(v, layout, world, r), segs[r]) for r in range(world)]
    carries = [kern.fwd_carry(qs[r]) for r in range(world)]
    for step in range(world):
        for r in range(world):
            _fwd_step(kern, layout, causal_block_size, r, world, L, qs[r], segs[r], held[r], *carries[r], step)
        held = [held[(r - 1) % world] for r in range(world)]  # rank r receives from rank r - 1
    outs = [kern.fwd_finish(carries[r][0], qs[r]) for r in range(world)]
    return unshard(outs, layout), unshard_lse([c[1] for c in carries], layout)


def ring_backward_local(q, k, v, out, lse, dout, segment_ids=None, causal_block_size=0, world=2,
                        layout="contiguous", kernels=None):
    """Backward of `ring_forward_local` (full tensors in, full dq, dk, dv out)."""
    check_layout(layout, causal_block_size)
    kern = kernels or CudaRingKernels()
    L = q.shape[1] // world
    sh = lambda x, r: shard(x, layout, world, r)  # noqa: E731
    qs, dos = [sh(q, r) for r in range(world)], [sh(dout, r) for r in range(world)]
    segs = [None if segment_ids is None else sh(segment_ids, r) for r in range(world)]
    wss = [kern.bwd_begin(sh(out, r), shard_lse(lse, layout, world, r), dos[r]) for r in range(world)]
    held = []
    for r in range(world):
        kb, vb = sh(k, r), sh(v, r)
        held.append((kb, vb, segs[r], kern.grad_carry(kb), kern.grad_carry(vb)))
    for step in range(world):
        for r in range(world):
            _bwd_step(kern, layout, causal_block_size, r, world, L, qs[r], dos[r], segs[r], held[r], wss[r], step)
        held = [held[(r - 1) % world] for r in range(world)]
    dq = unshard([kern.bwd_end(wss[r], qs[r]) for r in range(world)], layout)
    dk = unshard([kern.grad_finish(held[r][3], qs[r]) for r in range(world)], layout)
    dv = unshard([kern.grad_finish(held[r][4], qs[r]) for r in range(world)], layout)
    return dq, dk, dv
