"""Thin Python binding of libra.so (include/ra.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors ([batch, seq, heads, head_dim],
contiguous); torch provides device memory and the current stream.  If the
library is missing or fails to load, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT = 0, 1, 2, 3, 4
RA_F32, RA_BF16 = 0, 1
_STATUS = {1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device wait timed out"}

EXPORTS = ("ra_fwd", "ra_bwd", "ra_bwd_workspace_size", "ra_sync_check", "ra_last_error",
           "ra_kernel_launches", "ra_selftest_timeout", "ra_bwd_noalloc", "ra_bwd_noalloc_max_scratch",
           "ra_decode", "ra_decode_workspace_size", "ra_blockwise_ffn", "ra_ffn_workspace_size",
           "ra_debug_visitlog", "ra_ring_fwd_step", "ra_ring_bwd_workspace_size", "ra_ring_bwd_begin",
           "ra_ring_bwd_step", "ra_ring_bwd_end", "ra_ring_finish")


class RAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libra.so once (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with long_context_exact_ra_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.ra_fwd.restype = i32
    L.ra_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.ra_bwd.restype = i32
    L.ra_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                         vp, vp, vp, vp, sz, vp]
    L.ra_bwd_workspace_size.restype = sz
    L.ra_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.ra_sync_check.restype = i32
    L.ra_sync_check.argtypes = [vp]
    L.ra_last_error.restype = ctypes.c_char_p
    L.ra_last_error.argtypes = []
    L.ra_kernel_launches.restype = ctypes.c_uint64
    L.ra_kernel_launches.argtypes = []
    L.ra_selftest_timeout.restype = i32
    L.ra_selftest_timeout.argtypes = [ctypes.c_int64, vp]
    L.ra_bwd_noalloc.restype = i32
    L.ra_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                 vp, vp, vp, vp]
    L.ra_bwd_noalloc_max_scratch.restype = sz
    L.ra_bwd_noalloc_max_scratch.argtypes = []
    L.ra_decode_workspace_size.restype = sz
    L.ra_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.ra_decode.restype = i32
    L.ra_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.ra_ffn_workspace_size.restype = sz
    L.ra_ffn_workspace_size.argtypes = [i32, i32, i32, i32]
    L.ra_blockwise_ffn.restype = i32
    L.ra_blockwise_ffn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, sz, vp]
    i64 = ctypes.c_longlong
    L.ra_debug_visitlog.restype = i32
    L.ra_debug_visitlog.argtypes = [vp, sz]
    L.ra_ring_fwd_step.restype = i32
    L.ra_ring_fwd_step.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.ra_ring_bwd_workspace_size.restype = sz
    L.ra_ring_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.ra_ring_bwd_begin.restype = i32
    L.ra_ring_bwd_begin.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, sz, vp]
    L.ra_ring_bwd_step.restype = i32
    L.ra_ring_bwd_step.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32, i32, i32, i32, vp, vp,
                                   vp, sz, vp]
    L.ra_ring_bwd_end.restype = i32
    L.ra_ring_bwd_end.argtypes = [vp, sz, i32, i32, i32, i32, i32, vp, vp]
    L.ra_ring_finish.restype = i32
    L.ra_ring_finish.argtypes = [vp, vp, sz, i32, vp]
    _lib = L
    return L


def _check(status: int):
    if status != RA_OK:
        raise RAError(status, lib().ra_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return RA_F32
    if t.dtype == torch.bfloat16:
        return RA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(name, t, like=None, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype):
        raise ValueError(f"{name} must match q in shape and dtype")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def _check_segment_ids(segment_ids, B, S):
    if segment_ids is not None:
        _check_tensor("segment_ids", segment_ids, dtype=torch.int32)
        if tuple(segment_ids.shape) != (B, S):
            raise ValueError("segment_ids must be [batch, seq]")


def _chunks(S, num_shards, query_chunk_size, key_chunk_size):
    ssh = S // num_shards if num_shards > 0 else 0
    qc = query_chunk_size if query_chunk_size is not None else max(ssh, 1)
    kc = key_chunk_size if key_chunk_size is not None else max(ssh, 1)
    return qc, kc


def fwd(q, k, v, segment_ids=None, causal_block_size=0, num_shards=1,
        query_chunk_size=None, key_chunk_size=None, out=None, lse=None, stream=None):
    """ra_fwd: returns (out [B,S,H,D] like q, lse [B,H,S] float32)."""
    _check_tensor("q", q)
    _check_tensor("k", k, q)
    _check_tensor("v", v, q)
    B, S, H, D = q.shape
    _check_segment_ids(segment_ids, B, S)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    _check_tensor("out", out, q)
    _check_tensor("lse", lse, dtype=torch.float32)
    qc, kc = _chunks(S, num_shards, query_chunk_size, key_chunk_size)
    _check(lib().ra_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(segment_ids), int(causal_block_size),
                        int(num_shards), int(qc), int(kc), B, S, H, D, _dtype_code(q),
                        _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def bwd_workspace_size(B, S, H, D, dtype) -> int:
    code = RA_BF16 if dtype == torch.bfloat16 else RA_F32
    return int(lib().ra_bwd_workspace_size(B, S, H, D, code))


def bwd(q, k, v, out, lse, dout, segment_ids=None, causal_block_size=0, num_shards=1,
        query_chunk_size=None, key_chunk_size=None, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """ra_bwd: returns (dq, dk, dv), each like q."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_tensor(name, t, q)
    _check_tensor("lse", lse, dtype=torch.float32)
    B, S, H, D = q.shape
    _check_segment_ids(segment_ids, B, S)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    need = bwd_workspace_size(B, S, H, D, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    qc, kc = _chunks(S, num_shards, query_chunk_size, key_chunk_size)
    _check(lib().ra_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(segment_ids),
                        int(causal_block_size), int(num_shards), int(qc), int(kc), B, S, H, D,
                        _dtype_code(q), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def bwd_noalloc(q, k, v, out, lse, dout, segment_ids=None, causal_block_size=0, num_shards=1,
                query_chunk_size=None, key_chunk_size=None, dq=None, dk=None, dv=None, stream=None):
    """ra_bwd_noalloc: the backward with the library's built-in scratch (for callers
    that cannot allocate device memory).  Returns (dq, dk, dv)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_tensor(name, t, q)
    _check_tensor("lse", lse, dtype=torch.float32)
    B, S, H, D = q.shape
    _check_segment_ids(segment_ids, B, S)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    qc, kc = _chunks(S, num_shards, query_chunk_size, key_chunk_size)
    _check(lib().ra_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(segment_ids),
                                int(causal_block_size), int(num_shards), int(qc), int(kc), B, S, H, D,
                                _dtype_code(q), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))
    return dq, dk, dv


def decode_workspace_size(B, T, S, H, D, num_shards, dtype) -> int:
    code = RA_BF16 if dtype == torch.bfloat16 else RA_F32
    return int(lib().ra_decode_workspace_size(B, T, S, H, D, num_shards, code))


def decode(q, k_cache, v_cache, cache_idx, q_segment_ids=None, kv_segment_ids=None,
           causal_block_size=1, num_shards=1, out=None, lse=None, workspace=None, stream=None):
    """ra_decode: T new tokens q [B,T,H,D] against the cache [B,S,H,D] at cache_idx [B] (int32).

    Returns (out [B,T,H,D] like q, lse [B,H,T] float32)."""
    _check_tensor("q", q)
    B, T, H, D = q.shape
    _check_tensor("k_cache", k_cache)
    _check_tensor("v_cache", v_cache, k_cache)
    if k_cache.dtype != q.dtype or k_cache.shape[0] != B or k_cache.shape[2] != H or k_cache.shape[3] != D:
        raise ValueError("k_cache must be [B, S, H, D] with q's dtype, batch, heads and head_dim")
    S = k_cache.shape[1]
    _check_tensor("cache_idx", cache_idx, dtype=torch.int32)
    if tuple(cache_idx.shape) != (B,):
        raise ValueError("cache_idx must be [batch]")
    if (q_segment_ids is None) != (kv_segment_ids is None):
        raise ValueError("q_segment_ids and kv_segment_ids must be given together")
    if q_segment_ids is not None:
        _check_tensor("q_segment_ids", q_segment_ids, dtype=torch.int32)
        _check_tensor("kv_segment_ids", kv_segment_ids, dtype=torch.int32)
        if tuple(q_segment_ids.shape) != (B, T) or tuple(kv_segment_ids.shape) != (B, S):
            raise ValueError("segment ids must be [batch, new_tokens] and [batch, cache_len]")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _check_tensor("out", out, q)
    _check_tensor("lse", lse, dtype=torch.float32)
    need = decode_workspace_size(B, T, S, H, D, num_shards, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib().ra_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_idx), _ptr(q_segment_ids),
                           _ptr(kv_segment_ids), int(causal_block_size), int(num_shards), B, T, S, H, D,
                           _dtype_code(q), _ptr(out), _ptr(lse), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def ffn_workspace_size(B, L, F, chunk_size) -> int:
    return int(lib().ra_ffn_workspace_size(B, L, F, chunk_size))


def blockwise_ffn(x, w1, b1, w2, b2, chunk_size, out=None, workspace=None, stream=None):
    """ra_blockwise_ffn: max(0, x w1^T + b1) w2^T + b2 over x [B, L, Dm] bf16 in chunks of rows.

    w1 [F, Dm] and w2 [Dm, F] bf16 (linear-layer layout); b1 [F], b2 [Dm] float32 or None."""
    _check_tensor("x", x, dtype=torch.bfloat16)
    B, L, Dm = x.shape
    _check_tensor("w1", w1, dtype=torch.bfloat16)
    _check_tensor("w2", w2, dtype=torch.bfloat16)
    F = w1.shape[0]
    if tuple(w1.shape) != (F, Dm) or tuple(w2.shape) != (Dm, F):
        raise ValueError("w1 must be [F, Dm] and w2 [Dm, F]")
    for name, t, n in (("b1", b1, F), ("b2", b2, Dm)):
        if t is not None:
            _check_tensor(name, t, dtype=torch.float32)
            if tuple(t.shape) != (n,):
                raise ValueError(f"{name} must have {n} entries")
    if out is None:
        out = torch.empty_like(x)
    _check_tensor("out", out, x)
    need = ffn_workspace_size(B, L, F, chunk_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(lib().ra_blockwise_ffn(_ptr(x), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), B, L, Dm, F, int(chunk_size),
                                  RA_BF16, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))
    return out


def sync_check(stream=None):
    """Synchronize and raise RAError if a kernel reported a timed-out wait."""
    _check(lib().ra_sync_check(_stream(stream)))


def kernel_launches() -> int:
    return int(lib().ra_kernel_launches())


def selftest_timeout(limit_ns: int, stream=None):
    _check(lib().ra_selftest_timeout(int(limit_ns), _stream(stream)))


# ----------------------------------------------------------------------------- debug visit log
VISITLOG_HEADER_WORDS = 8
VISITLOG_ENTRY_WORDS = 8


def debug_visitlog(buf):
    """ra_debug_visitlog: make the calling thread's next bf16 attention calls record
    the tiles their kernels visit into `buf` (int32 CUDA tensor; word 0 counts the
    entries, which start at word 8, 8 words each), or stop recording (buf=None)."""
    if buf is not None:
        _check_tensor("visit log", buf, dtype=torch.int32)
    _check(lib().ra_debug_visitlog(_ptr(buf), 0 if buf is None else buf.numel()))


# ----------------------------------------------------------------------------- ring steps
def _ring_seg(q_segment_ids, kv_segment_ids, B, S):
    if (q_segment_ids is None) != (kv_segment_ids is None):
        raise ValueError("q_segment_ids and kv_segment_ids must be given together")
    _check_segment_ids(q_segment_ids, B, S)
    _check_segment_ids(kv_segment_ids, B, S)


def ring_fwd_step(q, k, v, q_segment_ids, kv_segment_ids, causal_block_size, q_pos0, k_pos0, pos_stride,
                  o_carry, lse_carry, stream=None):
    """ra_ring_fwd_step: merge attention(q block, k/v block) into (o_carry fp32 [B,S,H,D], lse_carry [B,H,S])."""
    _check_tensor("q", q)
    _check_tensor("k", k, q)
    _check_tensor("v", v, q)
    B, S, H, D = q.shape
    _ring_seg(q_segment_ids, kv_segment_ids, B, S)
    _check_tensor("o_carry", o_carry, dtype=torch.float32)
    _check_tensor("lse_carry", lse_carry, dtype=torch.float32)
    if tuple(o_carry.shape) != (B, S, H, D) or tuple(lse_carry.shape) != (B, H, S):
        raise ValueError("o_carry must be [B, S, H, D] and lse_carry [B, H, S]")
    _check(lib().ra_ring_fwd_step(_ptr(q), _ptr(k), _ptr(v), _ptr(q_segment_ids), _ptr(kv_segment_ids),
                                  int(causal_block_size), int(q_pos0), int(k_pos0), int(pos_stride), B, S, H, D,
                                  _dtype_code(q), _ptr(o_carry), _ptr(lse_carry), _stream(stream)))


def ring_bwd_workspace_size(B, S, H, D) -> int:
    return int(lib().ra_ring_bwd_workspace_size(B, S, H, D, RA_BF16))


def ring_bwd_begin(out, lse, dout, workspace, stream=None):
    """ra_ring_bwd_begin: Delta and the zeroed dQ accumulator of this query block, in `workspace`."""
    _check_tensor("out", out)
    _check_tensor("dout", dout, out)
    _check_tensor("lse", lse, dtype=torch.float32)
    B, S, H, D = out.shape
    _check(lib().ra_ring_bwd_begin(_ptr(out), _ptr(lse), _ptr(dout), B, S, H, D, _dtype_code(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def ring_bwd_step(q, k, v, dout, q_segment_ids, kv_segment_ids, causal_block_size, q_pos0, k_pos0, pos_stride,
                  dk_carry, dv_carry, workspace, stream=None):
    """ra_ring_bwd_step: add this (query block, key/value block) pair's gradients: dQ into the
    workspace accumulator, dK and dV into the fp32 carries of the key/value block."""
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _check_tensor(name, t, q)
    B, S, H, D = q.shape
    _ring_seg(q_segment_ids, kv_segment_ids, B, S)
    for name, t in (("dk_carry", dk_carry), ("dv_carry", dv_carry)):
        _check_tensor(name, t, dtype=torch.float32)
        if tuple(t.shape) != (B, S, H, D):
            raise ValueError(f"{name} must be [B, S, H, D]")
    _check(lib().ra_ring_bwd_step(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(q_segment_ids), _ptr(kv_segment_ids),
                                  int(causal_block_size), int(q_pos0), int(k_pos0), int(pos_stride), B, S, H, D,
                                  _dtype_code(q), _ptr(dk_carry), _ptr(dv_carry), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def ring_bwd_end(workspace, dq, stream=None):
    """ra_ring_bwd_end: dq (like q) from the workspace's dQ accumulator."""
    _check_tensor("dq", dq)
    B, S, H, D = dq.shape
    _check(lib().ra_ring_bwd_end(_ptr(workspace), workspace.numel() * workspace.element_size(), B, S, H, D,
                                 _dtype_code(dq), _ptr(dq), _stream(stream)))


def ring_finish(src, dst, stream=None):
    """ra_ring_finish: dst (bf16) = src (fp32), element by element."""
    _check_tensor("src", src, dtype=torch.float32)
    _check_tensor("dst", dst, dtype=torch.bfloat16)
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same number of elements")
    _check(lib().ra_ring_finish(_ptr(src), _ptr(dst), src.numel(), RA_BF16, _stream(stream)))
