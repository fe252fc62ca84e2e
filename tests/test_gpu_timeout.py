"""GPU test of the bounded-wait timeout path, without a fault, a trap or an endless wait.

With the wait limit set to one microsecond, the decode kernel's ordinary waits (for queries and
pages still in flight, for the other CTA of the pair) run out.  Every CTA then leaves its waits,
lets the copies it issued land, lets its issued MMAs complete, frees its tensor memory and
returns; the call reports MLA_ERR_DEVICE_TIMEOUT through the device error word.  The next call
with the default limit must give the oracle's results: the context and the library stay usable.
"""
import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M
from mla_latent_kv_79_b300 import _lib

from tests.gpu_util import TOL_LSE_BF16, TOL_OUT_BF16, cache_of, cfg_of, dev, host, rel

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2
MLA_ERR_DEVICE_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _ready():
    from mla_latent_kv_79_b300 import build
    build.build()
    M.lib()
    yield


def test_decode_timeout_reports_and_recovers():
    lens = [4096] * 8 + [1000, 64, 1, 3000]
    case = W.make_decode_case(DS, "bf16", lens, seed=95)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    q = dev(case["q_cat"])
    old_simt = M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 0)
    assert M.mla_get_device_error() == 0
    old = M.mla_set_tuning(_lib.MLA_TUNE_WAIT_LIMIT_US, 1)
    try:
        M.mla_decode(cfg, cache, q)
        torch.cuda.synchronize()
        status = M.mla_get_device_error()
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_WAIT_LIMIT_US, old)
        M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, old_simt)
    assert M.mla_last_attention_path() == 2, "the tcgen05 kernel must be the one that timed out"
    assert status == MLA_ERR_DEVICE_TIMEOUT, _lib.STATUS_NAMES.get(status, status)
    assert M.mla_get_device_error() == 0, "the error word is cleared by the read"

    # the same call with the default limit: correct results, no error
    o, lse = M.mla_decode(cfg, cache, q)
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    go, gl = host(o), host(lse)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    pool = W.to_f64(case["pool"], "bf16")
    qc = W.to_f64(case["q_cat"], "bf16")
    for b in (0, 7, 8, 9, 10, 11):
        rows = O.sequence_rows(pool, case["page_table"][b], lens[b])
        ro, rl = O.attention_latent(qc[b], rows, DS.d_latent, sc)
        assert rel(go[b], ro) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b
