"""GPU tests of mla_decode_static, the decode entry point that allocates nothing (its split
partials live in a fixed device array of the library).  Through the C ABI it must give
mla_decode's results on the same inputs (and the oracle's), on two calls in a row, without the device's free
memory moving after the first call's set-up, and must reject a configuration whose scratch exceeds the array.

The file is named to be collected last: it has to pass both after every other GPU test and
run alone in a fresh process (where its own calls do the one-time address look-up)."""
import ctypes

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
# split over many units, a single token, ragged tails, an empty sequence
LENS = [4096, 1, 777, 0, 2050, 64]


def _compare(o, lse, o_ref, lse_ref):
    go, gl, ro, rl = host(o), host(lse), host(o_ref), host(lse_ref)
    for b in range(len(LENS)):
        if LENS[b] == 0:
            assert np.all(go[b] == 0) and np.all(np.isneginf(gl[b])), b
            continue
        assert rel(go[b], ro[b]) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl[b])) <= TOL_LSE_BF16, b


def _compare_oracle(case, o, lse):
    """The static entry point's outputs against the CPU oracle itself."""
    go, gl = host(o), host(lse)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    pool = W.to_f64(case["pool"], "bf16")
    q = W.to_f64(case["q_cat"], "bf16")
    for b, L in enumerate(LENS):
        if L == 0:
            continue
        ro, rl = O.attention_latent(q[b], O.sequence_rows(pool, case["page_table"][b], L), DS.d_latent, sc)
        assert rel(go[b], ro) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b


@pytest.mark.parametrize("path", ["auto", "simt"])
def test_static_decode_matches_decode_twice(path):
    case = W.make_decode_case(DS, "bf16", LENS, seed=91, spare_pages=3)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    q = dev(case["q_cat"])
    B = len(LENS)
    old = M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 1 if path == "simt" else 0)
    try:
        o_ref, lse_ref = M.mla_decode(cfg, cache, q)
        o = torch.empty((B, DS.n_heads, DS.d_latent), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, DS.n_heads), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        # the first call of the process on this device does the one-time set-up (address
        # look-up; the driver may place the array then); the two calls after it allocate nothing
        for i in range(3):
            o.fill_(float("nan"))
            lse.fill_(float("nan"))
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            st = M.lib().mla_decode_static(ctypes.byref(cfg.c()), ctypes.byref(cache.c()),
                                           ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                           ctypes.c_void_p(lse.data_ptr()), None)
            assert st == 0, _lib.STATUS_NAMES.get(st, st)
            torch.cuda.synchronize()
            if i > 0:
                assert torch.cuda.mem_get_info()[0] == free_before, f"call {i} moved free memory"
            assert M.mla_get_device_error() == 0
            _compare(o, lse, o_ref, lse_ref)
            if i == 2:
                _compare_oracle(case, o, lse)
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, old)


def test_static_decode_python_wrapper():
    case = W.make_decode_case(DS, "bf16", [300, 5000], seed=92)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    q = dev(case["q_cat"])
    o_ref, lse_ref = M.mla_decode(cfg, cache, q)
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    M.mla_decode_static(cfg, cache, q, o, lse)
    torch.cuda.synchronize()
    assert rel(host(o), host(o_ref)) <= TOL_OUT_BF16
    assert np.max(np.abs(host(lse) - host(lse_ref))) <= TOL_LSE_BF16


def test_static_decode_rejects_scratch_beyond_limit():
    # 960 latent columns: 2 x SMs x 128 x 961 x 4 bytes, far above 80 MiB on any B300
    cfg = _lib.MlaConfig(n_heads=128, d_nope=128, d_rope=64, d_latent=960, d_model=5120, page_size=64,
                         rope_base=10000.0, softmax_scale=0.0, dtype=_lib.MLA_BF16)
    need = ctypes.c_size_t(0)
    assert M.lib().mla_workspace_size(ctypes.byref(cfg), ctypes.byref(need)) == 0
    assert need.value > _lib.MLA_STATIC_SCRATCH_BYTES
    st = M.lib().mla_decode_static(ctypes.byref(cfg), None, None, None, None, None)
    assert st == _lib.MLA_ERR_SCRATCH_LIMIT
    assert b"no-allocation" in M.lib().mla_status_string(st)
