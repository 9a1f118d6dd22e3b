"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/ra.h declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

from long_context_exact_ra_gb300 import ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ra.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(ops.LIB_PATH):
        from long_context_exact_ra_gb300 import build
        build.build()
    return ops.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(ops.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    # and nothing else with C linkage under the ra_ prefix
    out = os.popen(f"nm -D --defined-only {ops.LIB_PATH}").read()
    exported = sorted(set(re.findall(r" T (ra_\w+)", out)))
    assert exported == declared_functions()


def _fwd(L, q=16, k=16, v=16, out=16, lse=16, seg=None, c=0, N=1, qc=1, kc=1, B=1, S=128, H=1, D=64, dt=1):
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ra_fwd(P(q), P(k), P(v), P(seg), c, N, qc, kc, B, S, H, D, dt, P(out), P(lse), None)


def test_validation_rejects_bad_arguments(L):
    assert _fwd(L, q=None) == ops.RA_ERR_INVALID_ARG
    assert b"q is NULL" in L.ra_last_error()
    assert _fwd(L, lse=None) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, v=24) == ops.RA_ERR_INVALID_ARG  # misaligned
    assert b"16-byte" in L.ra_last_error()
    assert _fwd(L, seg=20) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, S=130, N=4) == ops.RA_ERR_INVALID_ARG  # seq % num_shards
    assert _fwd(L, S=128, N=4, qc=3) == ops.RA_ERR_INVALID_ARG  # shard % chunk
    assert _fwd(L, S=128, N=4, kc=64) == ops.RA_ERR_INVALID_ARG  # 32 % 64
    assert _fwd(L, c=-1) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, N=0) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, B=0) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, qc=0) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, dt=7) == ops.RA_ERR_INVALID_ARG
    assert _fwd(L, B=1 << 10, S=1 << 12, H=1 << 6, D=128) == ops.RA_ERR_INVALID_ARG  # 2^31 elements
    assert _fwd(L, D=96) == ops.RA_ERR_UNSUPPORTED  # bf16 only 64 / 128
    assert _fwd(L, D=256, dt=0) == ops.RA_ERR_UNSUPPORTED
    # an empty problem succeeds without touching the GPU
    assert _fwd(L, S=0) == ops.RA_OK
    assert L.ra_last_error() == b""


def test_bwd_validation_and_workspace(L):
    ws = L.ra_bwd_workspace_size(2, 1000, 3, 128, 1)
    assert ws >= 2 * 1000 * 3 * 128 * 4 + 2 * 3 * 1000 * 4
    assert ws % 256 == 0
    assert L.ra_bwd_workspace_size(2, 1000, 3, 64, 0) >= 2 * 3 * 1000 * 4
    assert L.ra_bwd_workspace_size(0, 10, 1, 64, 1) == 0
    P = ctypes.c_void_p
    args = [P(16)] * 6 + [None, 1, 1, 1, 1, 1, 128, 1, 64, 1, P(16), P(16), P(16), P(16)]
    st = L.ra_bwd(*args, ctypes.c_size_t(16), None)  # workspace too small
    assert st == ops.RA_ERR_INVALID_ARG and b"workspace" in L.ra_last_error()


def test_selftest_limit_is_validated(L):
    assert L.ra_selftest_timeout(0, None) == ops.RA_ERR_INVALID_ARG
    assert L.ra_selftest_timeout(2_000_000_000, None) == ops.RA_ERR_INVALID_ARG


def _dec(L, q=16, k=16, v=16, idx=16, qseg=None, kseg=None, c=1, N=1, B=1, T=1, S=128, H=1, D=128, dt=1,
         out=16, lse=16, ws=16, wsb=1 << 30):
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ra_decode(P(q), P(k), P(v), P(idx), P(qseg), P(kseg), c, N, B, T, S, H, D, dt, P(out), P(lse),
                       P(ws), ctypes.c_size_t(wsb), None)


def test_decode_validation_and_workspace(L):
    assert _dec(L, q=None) == ops.RA_ERR_INVALID_ARG and b"q is NULL" in L.ra_last_error()
    assert _dec(L, idx=None) == ops.RA_ERR_INVALID_ARG and b"cache_idx" in L.ra_last_error()
    assert _dec(L, idx=18) == ops.RA_ERR_INVALID_ARG  # int32 array not 4-byte aligned
    assert _dec(L, k=24) == ops.RA_ERR_INVALID_ARG and b"16-byte" in L.ra_last_error()
    assert _dec(L, qseg=16) == ops.RA_ERR_INVALID_ARG  # segment ids must come in pairs
    assert _dec(L, S=130, N=4) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, c=-1) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, N=0) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, B=0) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, B=70000) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, dt=5) == ops.RA_ERR_INVALID_ARG
    assert _dec(L, D=96) == ops.RA_ERR_UNSUPPORTED
    assert _dec(L, T=65) == ops.RA_ERR_UNSUPPORTED
    assert _dec(L, wsb=8) == ops.RA_ERR_INVALID_ARG and b"workspace" in L.ra_last_error()
    # no new token: nothing to do, no GPU touched
    assert _dec(L, T=0) == ops.RA_OK and L.ra_last_error() == b""
    # the workspace is a function of the shape: partial (m, l, o) per (b, h, token, work item)
    ws1 = L.ra_decode_workspace_size(1, 1, 131072, 32, 128, 16, 1)
    ws2 = L.ra_decode_workspace_size(1, 2, 131072, 32, 128, 16, 1)
    assert ws1 > 0 and ws2 >= 2 * ws1 - 512 and ws1 % 256 == 0
    assert L.ra_decode_workspace_size(1, 1, 0, 1, 64, 1, 1) == 0
    assert L.ra_decode_workspace_size(0, 1, 128, 1, 64, 1, 1) == 0


def _ffn(L, x=16, w1=16, b1=None, w2=16, b2=None, B=1, S=256, Dm=64, F=128, chunk=128, dt=1, out=16, ws=16,
         wsb=1 << 30):
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    return L.ra_blockwise_ffn(P(x), P(w1), P(b1), P(w2), P(b2), B, S, Dm, F, chunk, dt, P(out), P(ws),
                              ctypes.c_size_t(wsb), None)


def test_ffn_validation_and_workspace(L):
    assert _ffn(L, x=None) == ops.RA_ERR_INVALID_ARG and b"x is NULL" in L.ra_last_error()
    assert _ffn(L, w2=24) == ops.RA_ERR_INVALID_ARG and b"16-byte" in L.ra_last_error()
    assert _ffn(L, b1=20) == ops.RA_ERR_INVALID_ARG
    assert _ffn(L, Dm=60) == ops.RA_ERR_INVALID_ARG  # not a multiple of 8
    assert _ffn(L, F=100) == ops.RA_ERR_INVALID_ARG
    assert _ffn(L, chunk=0) == ops.RA_ERR_INVALID_ARG
    assert _ffn(L, B=0) == ops.RA_ERR_INVALID_ARG
    assert _ffn(L, dt=0) == ops.RA_ERR_UNSUPPORTED
    assert _ffn(L, wsb=100) == ops.RA_ERR_INVALID_ARG and b"workspace" in L.ra_last_error()
    assert _ffn(L, S=0) == ops.RA_OK and L.ra_last_error() == b""
    # one chunk of hidden activations: min(rows, chunk) x F bf16
    assert L.ra_ffn_workspace_size(2, 1000, 128, 512) == 512 * 128 * 2
    assert L.ra_ffn_workspace_size(1, 100, 128, 512) == 100 * 128 * 2
    assert L.ra_ffn_workspace_size(0, 100, 128, 512) == 0


def test_ring_step_and_visit_log_validation(L):
    """Rejections that happen before any CUDA call."""
    P = ctypes.c_void_p
    a = P(256)

    def fwd_step(c=1, q0=0, k0=0, stride=1, dt=ops.RA_BF16, qseg=None, kseg=None, S=128, D=64, o=a):
        return L.ra_ring_fwd_step(a, a, a, qseg, kseg, c, q0, k0, stride, 1, S, 1, D, dt, o, a, None)

    assert fwd_step(c=3, q0=1, k0=0, stride=4) == ops.RA_ERR_UNSUPPORTED       # strided + block causal
    assert b"strided" in L.ra_last_error()
    assert fwd_step(q0=-1) == ops.RA_ERR_INVALID_ARG
    assert fwd_step(stride=0) == ops.RA_ERR_INVALID_ARG
    assert fwd_step(k0=1 << 30) == ops.RA_ERR_INVALID_ARG                       # positions below 2^30
    assert fwd_step(dt=ops.RA_F32) == ops.RA_ERR_UNSUPPORTED                    # bf16 only
    assert fwd_step(qseg=P(512)) == ops.RA_ERR_INVALID_ARG                      # both ids or neither
    assert fwd_step(o=None) == ops.RA_ERR_INVALID_ARG
    assert fwd_step(D=96) == ops.RA_ERR_UNSUPPORTED
    assert L.ra_ring_bwd_step(a, a, a, a, None, None, 1, 0, 0, 1, 1, 128, 1, 64, ops.RA_BF16, a, a, a, 16,
                              None) == ops.RA_ERR_INVALID_ARG                    # workspace too small
    assert b"workspace" in L.ra_last_error()
    assert L.ra_ring_bwd_workspace_size(1, 128, 1, 64, ops.RA_BF16) == L.ra_bwd_workspace_size(1, 128, 1, 64,
                                                                                               ops.RA_BF16)
    assert L.ra_ring_finish(a, a, 6, ops.RA_BF16, None) == ops.RA_ERR_INVALID_ARG  # count % 4
    assert L.ra_ring_finish(a, a, 8, ops.RA_F32, None) == ops.RA_ERR_UNSUPPORTED
    assert L.ra_ring_finish(a, a, 0, ops.RA_BF16, None) == ops.RA_OK              # nothing to do
    # visit log: alignment and size rules; NULL turns it off
    assert L.ra_debug_visitlog(P(260), 64) == ops.RA_ERR_INVALID_ARG
    assert L.ra_debug_visitlog(a, 15) == ops.RA_ERR_INVALID_ARG
    assert L.ra_debug_visitlog(None, 0) == ops.RA_OK
