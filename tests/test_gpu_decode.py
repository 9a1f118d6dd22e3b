"""GPU parity of decoding against a sharded KV cache (ra_decode, through the C ABI)
against the CPU float64 oracle (oracle/decode.py)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_exact_ra_gb300 import ops
from long_context_exact_ra_gb300.inputs import DECODE_WORKLOADS, DecodeWorkload, make_decode_inputs
from tests.gpu_util import check_lse, check_out, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ops.lib()


def run_decode(x):
    w = x.w
    q = to_dev(x.q, w.dtype)
    k = to_dev(x.k_cache, w.dtype)
    v = to_dev(x.v_cache, w.dtype)
    idx = torch.from_numpy(x.cache_idx).cuda()
    qs = None if x.q_segment_ids is None else torch.from_numpy(x.q_segment_ids).cuda()
    ks = None if x.kv_segment_ids is None else torch.from_numpy(x.kv_segment_ids).cuda()
    before = ops.kernel_launches()
    out, lse = ops.decode(q, k, v, idx, qs, ks, w.causal_block_size, w.num_shards)
    ops.sync_check()
    launches = ops.kernel_launches() - before
    return host_f64(out), lse.cpu().numpy().astype(np.float64), launches


def full_check(x):
    w = x.w
    out, lse, launches = run_decode(x)
    assert launches == (2 if w.cache_len > 0 else 1)
    ref_out, ref_lse = oracle.ref_decode(x.as_f64("q"), x.as_f64("k_cache"), x.as_f64("v_cache"), x.cache_idx,
                                         w.causal_block_size, x.q_segment_ids, x.kv_segment_ids)
    check_out(out, ref_out, w.dtype, scale=w.scale)
    check_lse(lse, ref_lse, w.dtype)
    return out, lse


SMALL = [
    # B, T, S, H, D, dtype, c, N, segments, fill
    (3, 1, 1024, 4, 128, "bf16", 1, 4, False, "random"),
    (3, 1, 1024, 4, 64, "bf16", 1, 8, False, "random"),
    (2, 3, 768, 2, 128, "bf16", 1, 3, False, "random"),
    (2, 5, 1000, 3, 64, "bf16", 1, 5, False, "random"),     # shard 200: ragged 32-key tiles
    (2, 8, 640, 2, 128, "bf16", 3, 2, False, "random"),     # causal block 3, 8 tokens
    (2, 13, 512, 2, 128, "bf16", 1, 4, False, "random"),    # two token groups
    (2, 4, 1024, 2, 128, "bf16", 0, 4, False, "random"),    # non-causal: the filled cache
    (3, 2, 2048, 2, 128, "bf16", 1, 8, True, "random"),     # packed documents
    (2, 1, 4096, 2, 128, "bf16", 1, 16, False, "full"),
    (2, 1, 512, 2, 64, "f32", 1, 4, False, "random"),
    (2, 6, 384, 3, 128, "f32", 2, 3, True, "random"),
    (1, 1, 256, 1, 128, "bf16", 1, 1, False, "full"),       # one shard
]


@pytest.mark.parametrize("B,T,S,H,D,dtype,c,N,seg,fill", SMALL)
def test_decode_small_full(B, T, S, H, D, dtype, c, N, seg, fill):
    w = DecodeWorkload("decode small", B, T, S, H, D, dtype, c, N, segments=seg, fill=fill,
                       seed=S + 3 * T + D + c, doc_len_range=(20, 300))
    full_check(make_decode_inputs(w))


@pytest.mark.parametrize("idx_of", ["edges", "outside"])
def test_decode_cache_index_edges(idx_of):
    """Shard and tile boundaries +-1, the first and last slot, and indices that put
    new tokens before the cache start or past its end (defined by the clamp)."""
    S, N, T = 1024, 4, 2
    if idx_of == "edges":
        idx = [0, 1, 255, 256, 257, 511, 512, 31, 32, 33, S - T, S - T - 1]
    else:
        idx = [-T, -1, S - 1, S + 5]
    w = DecodeWorkload("decode edges", len(idx), T, S, 2, 128, "bf16", 1, N, seed=77)
    full_check(make_decode_inputs(w, cache_idx=np.array(idx, dtype=np.int32)))


def test_decode_empty_cache_and_no_tokens():
    w = DecodeWorkload("decode empty", 2, 3, 0, 2, 64, "bf16", 1, 1, seed=5)
    x = make_decode_inputs(w, cache_idx=np.array([0, 0], dtype=np.int32))
    out, lse, launches = run_decode(x)
    assert launches == 1 and np.all(out == 0) and np.all(np.isneginf(lse))
    q = torch.zeros((1, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 64, 2, 64), dtype=torch.bfloat16, device="cuda")
    before = ops.kernel_launches()
    ops.decode(q, k, k, torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert ops.kernel_launches() == before


def test_decode_7b_full_cache_all_rows():
    """The 131072-token 7B-shaped cache (16 shards), every (head, token) row against the oracle."""
    x = make_decode_inputs(DECODE_WORKLOADS["7b"])
    out, lse, _ = run_decode(x)
    w = x.w
    rows = np.array([(0, h, 0) for h in range(w.heads)])
    ro, rl = oracle.ref_decode_rows(x.as_f64("q"), _F64View(x.k_cache), _F64View(x.v_cache), x.cache_idx, rows,
                                    w.causal_block_size)
    got = out[0, 0]  # [H, D]
    check_out(got, ro, w.dtype)
    check_lse(lse[0, :, 0], rl, w.dtype)


def test_decode_7b_eight_tokens_sampled_rows():
    """Eight new tokens at a random fill of the 7B-shaped cache; all (head, token) rows checked."""
    w = DECODE_WORKLOADS["7b"].with_(new_tokens=8, fill="random", seed=1004)
    x = make_decode_inputs(w, cache_idx=np.array([70001], dtype=np.int32))
    out, lse, _ = run_decode(x)
    rows = np.array([(0, h, t) for h in range(0, w.heads, 4) for t in range(8)])
    ro, rl = oracle.ref_decode_rows(x.as_f64("q"), _F64View(x.k_cache), _F64View(x.v_cache), x.cache_idx, rows,
                                    w.causal_block_size)
    got = out[rows[:, 0], rows[:, 2], rows[:, 1]]
    check_out(got, ro, w.dtype)
    check_lse(lse[rows[:, 0], rows[:, 1], rows[:, 2]], rl, w.dtype)


class _F64View:
    """Index a bf16-bit-pattern array and get float64 values (avoids a full-size float64 copy)."""

    def __init__(self, bits):
        self.bits = bits
        self.shape = bits.shape

    def __getitem__(self, key):
        from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32
        return bf16_bits_to_f32(self.bits[key]).astype(np.float64)
