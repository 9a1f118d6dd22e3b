"""A float64 CPU stand-in for the device work of one ring step.

The ring driver (long_context_exact_ra_gb300/ring.py) only orders the ring-step
calls and moves blocks between ranks; these fakes let its exchange and position
bookkeeping run on CPU ranks (gloo) without a GPU.  Each fake does in float64
what the corresponding C-ABI call does on the device, from the oracle's
visibility rule:
  fwd_step : attention of the query block against one key/value block at the
             given global positions, merged into the running (out, lse) carry
             with the lazy-softmax update at block granularity;
  bwd_*    : P = exp(S - lse) under the mask, dV += P^T dO,
             dS = P * (dO V^T - Delta), dK += dS^T Q / sqrt(D), dQ += dS K / sqrt(D).
"""
import math

import numpy as np
import torch

import oracle


def _positions(p0, stride, n):
    return p0 + stride * np.arange(n)


def _mask(b, qseg, kseg, c, q0, k0, stride, L):
    qs = None if qseg is None else qseg[b].numpy()
    ks = None if kseg is None else kseg[b].numpy()
    return torch.from_numpy(oracle.visible(_positions(q0, stride, L), _positions(k0, stride, L), c, qs, ks))


class Float64RingKernels:
    def fwd_carry(self, q):
        B, L, H, D = q.shape
        return (torch.zeros((B, L, H, D), dtype=torch.float64),
                torch.full((B, H, L), -math.inf, dtype=torch.float64))

    def fwd_step(self, q, k, v, qseg, kseg, c, q0, k0, stride, o, lse):
        B, L, H, D = q.shape
        for b in range(B):
            vis = _mask(b, qseg, kseg, c, q0, k0, stride, L)
            for h in range(H):
                s = (q[b, :, h] @ k[b, :, h].T) / math.sqrt(D)
                s = torch.where(vis, s, torch.tensor(-math.inf, dtype=torch.float64))
                lb = torch.logsumexp(s, dim=1)  # -inf for a row with no visible key
                seen = torch.isfinite(lb)
                p = torch.where(seen[:, None], torch.exp(s - torch.where(seen, lb, 0.0)[:, None]), 0.0)
                ob = p @ v[b, :, h]
                lo = lse[b, h]
                ln = torch.logaddexp(lo, lb)
                wo = torch.where(torch.isfinite(lo), torch.exp(lo - ln), 0.0)
                wn = torch.where(seen, torch.exp(lb - ln), 0.0)
                upd = seen
                o[b, :, h] = torch.where(upd[:, None], o[b, :, h] * wo[:, None] + ob * wn[:, None], o[b, :, h])
                lse[b, h] = torch.where(upd, ln, lo)

    def fwd_finish(self, o, like):
        return o.clone()

    def bwd_begin(self, out, lse, dout):
        delta = (out * dout).sum(-1).permute(0, 2, 1).contiguous()  # [B, H, L]
        return {"lse": lse.clone(), "delta": delta, "dq": torch.zeros_like(out)}

    def grad_carry(self, k):
        return torch.zeros(k.shape, dtype=torch.float64)

    def bwd_step(self, q, k, v, dout, qseg, kseg, c, q0, k0, stride, dk, dv, ws):
        B, L, H, D = q.shape
        sc = 1.0 / math.sqrt(D)
        for b in range(B):
            vis = _mask(b, qseg, kseg, c, q0, k0, stride, L)
            for h in range(H):
                s = (q[b, :, h] @ k[b, :, h].T) * sc
                P = torch.where(vis, torch.exp(torch.where(vis, s, 0.0) - ws["lse"][b, h][:, None]), 0.0)
                dv[b, :, h] += P.T @ dout[b, :, h]
                dS = P * (dout[b, :, h] @ v[b, :, h].T - ws["delta"][b, h][:, None])
                dk[b, :, h] += (dS.T @ q[b, :, h]) * sc
                ws["dq"][b, :, h] += (dS @ k[b, :, h]) * sc

    def bwd_end(self, ws, like):
        return ws["dq"]

    def grad_finish(self, g, like):
        return g.clone()
