"""Helpers for the GPU parity tests: device copies, guarded outputs, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import mla_workloads as W
from mla_latent_kv_79_b300 import MLAConfig, PagedCache

# Tolerances (the benchmark spec): relative max-abs error on outputs, absolute on log-sum-exp.
TOL_OUT_BF16 = 2e-2
TOL_LSE_BF16 = 1e-3
# fp32 path: fp32 accumulation over at most a few thousand terms.
TOL_OUT_F32 = 1e-4
TOL_LSE_F32 = 1e-4
# Chains that round an intermediate (q_cat) to bf16 before the attention kernel: the score
# error of a bf16-rounded query is ~ scale * 2^-8/sqrt(3) * ||q . k||_2 ~ 1.1e-3 per score at
# the DeepSeek-V2 shapes, so lse may move by a few of those when one token dominates.
TOL_LSE_BF16_CHAIN = 5e-3


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
