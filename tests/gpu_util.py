"""Helpers for the GPU parity tests: device copies, guarded outputs, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import mla_workloads as W
from mla_latent_kv_79_b300 import MLAConfig, PagedCache

# Tolerances: relative max-abs error on outputs, absolute on log-sum-exp.
TOL_OUT_BF16 = 2e-2
TOL_LSE_BF16 = 1e-3
# fp32 path: fp32 accumulation over at most a few thousand terms.
TOL_OUT_F32 = 1e-4
TOL_LSE_F32 = 1e-4
BF16_U = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits, round to nearest)


def lse_rounding_bound(q, keys, appended=(), scale=1.0):
    """Rigorous first-order bound on |lse' - lse| when the query q and the cache rows listed
    in `appended` are rounded to bf16 before attention (every other row is already bf16).

    lse is 1-Lipschitz in the max-norm of the scores, and a score q.k moves by at most
    scale * sum_c (u |q_c||k_c|  +  [k rounded] (u + u^2) |q_c||k_c|).
    q [n_h, W], keys [L, W] (float64 oracle values).  Returns [n_h]."""
    a = np.abs(q) @ np.abs(keys).T                     # [n_h, L]
    per = np.full(keys.shape[0], BF16_U)
    for t in appended:
        per[t] += BF16_U + BF16_U * BF16_U
    return scale * np.max(a * per[None, :], axis=1)


def rel(g, r) -> float:
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.max(np.abs(g - r)) / max(float(np.max(np.abs(r))), 1e-30))


def dev(a, dtype="bf16"):
    return W.to_device(a, dtype)


def host(t):
    return W.from_device(t)


def cfg_of(shape, dtype) -> MLAConfig:
    return MLAConfig.from_shape(shape, dtype)


def cache_of(case) -> PagedCache:
    return PagedCache(dev(case["pool"], case["dtype"]), torch.from_numpy(case["page_table"]).cuda(),
                      torch.from_numpy(case["seq_lens"]).cuda())


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class Guarded:
    """An output buffer with canary elements on both sides, checked after the call."""

    PAD = 64

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * self.PAD, dtype=dtype, device="cuda")
        self.buf.fill_(-12345.0 if dtype != torch.int32 else -7)
        if fill is not None:
            self.buf[self.PAD:self.PAD + n].fill_(fill)
        self.canary = self.buf.clone()
        self.t = self.buf[self.PAD:self.PAD + n].view(*shape)

    def check(self):
        n = self.t.numel()
        assert torch.equal(self.buf[:self.PAD], self.canary[:self.PAD]), "write before the buffer"
        assert torch.equal(self.buf[self.PAD + n:], self.canary[self.PAD + n:]), "write past the buffer"
