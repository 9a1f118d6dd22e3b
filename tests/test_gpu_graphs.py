"""The library's calls are stream-ordered with no host synchronisation inside, so
they can be captured into a CUDA graph and replayed.  Checks: forward + backward
captured once and replayed on new input values give the eager results, and a
captured decode step follows a cache index that changes in device memory
between replays (the decode loop needs no host round trip).

The bf16 forward draws its units from a per-call counter when called eagerly
and uses a fixed schedule under capture: both must give bit-identical results
(packed documents, several L2 head groups with a short last one, ragged
shards), and calls in flight on two streams at once must not share a counter."""
import numpy as np
import pytest
import torch

from long_context_exact_ra_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def _fill(t, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    t.copy_(torch.randn(t.shape, generator=g, device="cuda", dtype=torch.float32).to(t.dtype))


def test_fwd_bwd_graph_replay_matches_eager():
    B, S, H, D, N = 1, 1024, 4, 128, 4
    q, k, v, do = (torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    out, lse = torch.empty_like(q), torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(ops.bwd_workspace_size(B, S, H, D, torch.bfloat16), dtype=torch.uint8, device="cuda")
    args = (None, 1, N, 256, 256)

    def step():
        ops.fwd(q, k, v, *args, out=out, lse=lse)
        ops.bwd(q, k, v, out, lse, do, *args, dq=dq, dk=dk, dv=dv, workspace=ws)

    for i, t in enumerate((q, k, v, do)):
        _fill(t, i)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first call outside capture (one-time device set-up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for rep in range(2):
        for i, t in enumerate((q, k, v, do)):
            _fill(t, 100 * rep + i)
        graph.replay()
        torch.cuda.synchronize()
        ops.sync_check()
        got = [x.clone() for x in (out, lse, dq, dk, dv)]
        step()  # eager on the same inputs
        ops.sync_check()
        assert torch.equal(got[0], out) and torch.equal(got[1], lse)  # the forward is deterministic
        for g_, e_ in zip(got[2:], (dq, dk, dv)):  # dQ adds partials with atomics: order may differ
            assert (g_.float() - e_.float()).abs().max().item() <= 1e-2


def test_decode_graph_follows_the_device_cache_index():
    B, T, S, H, D, N = 2, 1, 2048, 4, 128, 4
    q = torch.empty(B, T, H, D, dtype=torch.bfloat16, device="cuda")
    kc, vc = (torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(2))
    for i, t in enumerate((q, kc, vc)):
        _fill(t, 50 + i)
    idx = torch.tensor([10, 700], dtype=torch.int32, device="cuda")
    out, lse = torch.empty_like(q), torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    ws = torch.empty(ops.decode_workspace_size(B, T, S, H, D, N, torch.bfloat16), dtype=torch.uint8, device="cuda")

    def step():
        ops.decode(q, kc, vc, idx, None, None, 1, N, out=out, lse=lse, workspace=ws)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for new in ([11, 701], [500, 2047], [0, 1]):
        idx.copy_(torch.tensor(new, dtype=torch.int32))  # device memory the graph reads
        graph.replay()
        torch.cuda.synchronize()
        got = (out.clone(), lse.clone())
        step()
        torch.cuda.synchronize()
        assert torch.equal(got[0], out) and torch.equal(got[1], lse), new
    # the last indices leave one and two visible keys: every token still sees a key
    assert np.isfinite(lse.cpu().numpy()).all()


def _fwd_static_and_dynamic(q, k, v, seg, c, N):
    """The forward captured in a graph (fixed unit schedule) and called eagerly
    (units drawn from a per-call counter)."""
    B, S, H, D = q.shape
    out_g, lse_g = torch.empty_like(q), torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.fwd(q, k, v, seg, c, N, out=out_g, lse=lse_g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.fwd(q, k, v, seg, c, N, out=out_g, lse=lse_g)
    graph.replay()
    torch.cuda.synchronize()
    out_e, lse_e = ops.fwd(q, k, v, seg, c, N)
    ops.sync_check()
    return (out_g, lse_g), (out_e, lse_e)


@pytest.mark.parametrize("B,S,H,D,N,c,docs", [
    (3, 1536, 5, 64, 3, 1, True),      # packed documents, one head group, units of uneven cost
    (1, 40960, 3, 128, 4, 1, False),   # 20 MB of K/V per head (48 MB groups): 2 heads, then a short group of 1
    (2, 8192, 20, 128, 4, 1, False),   # 4 MB of K/V per head (128 MB groups): 32 heads, then a short group of 8
    (1, 1000, 3, 128, 2, 0, False),    # ragged shards, non-causal
])
def test_forward_unit_schedule_does_not_change_results(B, S, H, D, N, c, docs):
    q, k, v = (torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    for i, t in enumerate((q, k, v)):
        _fill(t, 300 + i)
    seg = None
    if docs:
        g = np.random.Generator(np.random.PCG64(7))
        ids = np.zeros((B, S), dtype=np.int32)
        for b in range(B):
            pos, doc = 0, 0
            while pos < S:
                n = int(g.integers(1, 400))
                ids[b, pos:pos + n] = doc
                pos, doc = pos + n, doc + 1
        seg = torch.from_numpy(ids).cuda()
    (og, lg), (oe, le) = _fwd_static_and_dynamic(q, k, v, seg, c, N)
    assert torch.equal(og, oe) and torch.equal(lg, le)


def test_concurrent_forward_calls_use_separate_counters():
    B, S, H, D, N = 2, 4096, 4, 128, 4
    inputs = []
    for j in range(2):
        t = [torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        for i, x in enumerate(t):
            _fill(x, 500 + 10 * j + i)
        inputs.append(t)
    ref = [ops.fwd(*t, None, 1, N) for t in inputs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    got = [[None, None] for _ in range(2)]
    for rep in range(3):  # several rounds of two calls in flight on two streams
        for j, s in enumerate(streams):
            with torch.cuda.stream(s):
                got[j] = ops.fwd(*inputs[j], None, 1, N, stream=s)
    torch.cuda.synchronize()
    ops.sync_check()
    for (o, l), (ro, rl) in zip(got, ref):
        assert torch.equal(o, ro) and torch.equal(l, rl)
