"""The kernels' own record of the tiles they visit (ra_debug_visitlog) against
the ring order of the paper review page of Ring Attention (环形注意力算法):

* forward: the unit of query tiles in shard j visits key shards
  k = (j - i) mod N at steps i = 0, 1, ..., and within a shard its key tiles in
  ascending order;
* backward: the unit of a key tile in shard k visits query shards (k + i) mod N
  (the devices the key block passes through), query tiles ascending;
* the visited tiles are exactly the tiles holding a visible element (the causal
  skip of the code walk-through page, §3; no segment ids here, where the tile
  test is exact).

The attention result cannot show any of this: it does not depend on the visit
order beyond rounding (排列不变性)."""
from collections import defaultdict

import numpy as np
import pytest
import torch

from long_context_exact_ra_gb300 import ops, ring
from long_context_exact_ra_gb300.inputs import Workload, make_inputs
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu
T = 128  # rows per tile


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def _read_log(buf):
    words = buf.cpu().numpy()
    n = int(words[0])
    cap = (len(words) - ops.VISITLOG_HEADER_WORDS) // ops.VISITLOG_ENTRY_WORDS
    assert 0 < n <= cap, f"{n} entries claimed, {cap} held"
    e = words[ops.VISITLOG_HEADER_WORDS:ops.VISITLOG_HEADER_WORDS + n * 8].reshape(n, 8)
    return e


def _units(entries):
    """unit key (kind, b, h, home shard, home tile) -> [(step, vshard, vtile), ...] in claim order"""
    u = defaultdict(list)
    for row in entries:
        kind = int(row[0]) & 0xFF
        u[(kind, int(row[1]), int(row[2]), int(row[3]), int(row[4]))].append((int(row[5]), int(row[6]), int(row[7])))
    return u


def _tiles(L):
    return (L + T - 1) // T


def expected_fwd(S, N, c, j, pr):
    L = S // N
    q0 = j * L + 2 * pr * T
    qtiles = [(q0 + w * T, min(q0 + (w + 1) * T, (j + 1) * L) - 1) for w in range(2) if q0 + w * T < (j + 1) * L]
    out = []
    for i in range(N):
        ks = (j - i) % N
        for t in range(_tiles(L)):
            ka = ks * L + t * T
            if any(c == 0 or ql // c >= ka // c for _, ql in qtiles):
                out.append((i, ks, t))
    return out


def expected_bwd(S, N, c, k, t):
    L = S // N
    k0 = k * L + t * T
    out = []
    for i in range(N):
        js = (k + i) % N
        for tt in range(_tiles(L)):
            ql = min(js * L + (tt + 1) * T, (js + 1) * L) - 1
            if c == 0 or ql // c >= k0 // c:
                out.append((i, js, tt))
    return out


CASES = [(N, c, L) for N in (3, 4, 8) for c in (0, 1, 100) for L in (384, 300)]


def _run(S, N, c, backward):
    w = Workload("visit log", 1, S, 2, 64, "bf16", c, N, S // N, S // N, backward=backward, seed=S + N + c)
    x = make_inputs(w, with_dout=backward)
    q, k, v = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v"))
    args = (None, c, N, S // N, S // N)
    buf = torch.zeros(8 + 8 * 20000, dtype=torch.int32, device="cuda")
    if not backward:
        ops.debug_visitlog(buf)
        try:
            out = ops.fwd(q, k, v, *args)
        finally:
            ops.debug_visitlog(None)
        ops.sync_check()
        return buf, out
    out, lse = ops.fwd(q, k, v, *args)
    do = to_dev(x.dout, "bf16")
    ops.debug_visitlog(buf)
    try:
        g = ops.bwd(q, k, v, out, lse, do, *args)
    finally:
        ops.debug_visitlog(None)
    ops.sync_check()
    return buf, g


@pytest.mark.parametrize("N,c,L", CASES)
def test_forward_visits_key_shards_in_ring_order(N, c, L):
    S = N * L
    buf, _ = _run(S, N, c, backward=False)
    units = _units(_read_log(buf))
    pairs = (_tiles(L) + 1) // 2
    for b in range(1):
        for h in range(2):
            for j in range(N):
                for pr in range(pairs):
                    got = units.pop((0, b, h, j, pr), [])
                    assert got == expected_fwd(S, N, c, j, pr), (b, h, j, pr)
    assert not units, f"unexpected units {list(units)[:4]}"


@pytest.mark.parametrize("N,c,L", CASES)
def test_backward_visits_query_shards_in_ring_order(N, c, L):
    S = N * L
    buf, _ = _run(S, N, c, backward=True)
    units = _units(_read_log(buf))
    for h in range(2):
        for k in range(N):
            for t in range(_tiles(L)):
                got = units.pop((1, 0, h, k, t), [])
                assert got == expected_bwd(S, N, c, k, t), (h, k, t)
    assert not units


def test_log_is_off_by_default_and_results_do_not_change():
    S, N, c = 1024, 4, 1
    w = Workload("visit log off", 1, S, 2, 128, "bf16", c, N, 256, 256, seed=5)
    x = make_inputs(w)
    q, k, v = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v"))
    buf = torch.zeros(8 + 8 * 4096, dtype=torch.int32, device="cuda")
    ops.debug_visitlog(buf)
    o1, l1 = ops.fwd(q, k, v, None, c, N, 256, 256)
    ops.debug_visitlog(None)
    n1 = int(buf[0].item())
    o2, l2 = ops.fwd(q, k, v, None, c, N, 256, 256)
    ops.sync_check()
    assert n1 > 0 and int(buf[0].item()) == n1
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_overflow_is_counted_not_written_past_the_buffer():
    S, N = 2048, 4
    w = Workload("visit log overflow", 1, S, 2, 64, "bf16", 0, N, 512, 512, seed=6)
    x = make_inputs(w)
    q, k, v = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v"))
    buf = torch.full((8 + 8 * 16 + 64,), -7, dtype=torch.int32, device="cuda")
    buf[0] = 0
    ops.debug_visitlog(buf[:8 + 8 * 16])
    ops.fwd(q, k, v, None, 0, N, 512, 512)
    ops.debug_visitlog(None)
    ops.sync_check()
    # units: 2 heads x 4 shards x 2 query tile pairs (shards of 4 tiles), each
    # visiting all 16 key tiles (non-causal): 256 entries claimed, 16 written
    assert int(buf[0].item()) == 2 * N * 2 * 16
    assert (buf[8 + 8 * 16:] == -7).all()


def test_striped_ring_balances_causal_work_across_ranks():
    """Per-rank visited tiles (from the kernels' log) of a causal ring of 8 ranks:
    with contiguous blocks rank r sees r whole blocks plus the diagonal one, so
    the last rank does about 13 times the work of the first; striped blocks give
    every rank the same work (Striped Attention, paper review page,
    相关工作 / 局限性), at the price of a partial diagonal in every block pair."""
    S, N = 16384, 8
    w = Workload("balance", 1, S, 1, 128, "bf16", 1, N, S // N, S // N, seed=9)
    x = make_inputs(w)
    q, k, v = (to_dev(getattr(x, n), "bf16") for n in ("q", "k", "v"))
    per_rank = {}
    for layout in ring.LAYOUTS:
        counts = []
        L = S // N
        for r in range(N):
            qb = ring.shard(q, layout, N, r)
            n = 0
            for step in range(N):
                kb = (r - step) % N
                q0, st = ring.block_positions(layout, r, N, L)
                k0, _ = ring.block_positions(layout, kb, N, L)
                if ring.block_sees_nothing(layout, 1, q0, k0, L):
                    continue
                buf = torch.zeros(8 + 8 * 8192, dtype=torch.int32, device="cuda")
                o = torch.zeros(qb.shape, dtype=torch.float32, device="cuda")
                lse = torch.full((1, 1, L), float("-inf"), device="cuda")
                ops.debug_visitlog(buf)
                ops.ring_fwd_step(qb, ring.shard(k, layout, N, kb), ring.shard(v, layout, N, kb), None, None, 1,
                                  q0, k0, st, o, lse)
                ops.debug_visitlog(None)
                n += int(buf[0].item())
            counts.append(n)
        per_rank[layout] = counts
    ops.sync_check()
    print("visited key tiles per rank (forward, causal, 8 ranks, S16384):", per_rank)
    c, s = per_rank["contiguous"], per_rank["striped"]
    # contiguous: rank r visits r * (8 pairs x 16 key tiles) + 72 tiles of its diagonal block
    assert c == [128 * r + 72 for r in range(N)]
    assert max(s) / min(s) < 1.05
