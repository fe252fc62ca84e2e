"""GPU parity of the compressed query side of the operator notes (section 4): c_q = x W_DQ,
Q = c_q W_UQ, the RoPE query from c_q, and the absorbed query with W_UQ folded into W_UK."""
import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M
from mla_latent_kv_79_b300 import _lib

from tests.gpu_util import TOL_LSE_BF16, TOL_OUT_BF16, cfg_of, dev, host, i32, rel

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2
D_CQ = DS.d_latent  # the page gives the query latent the latent's width


@pytest.fixture(scope="module", autouse=True)
def _ready():
    from mla_latent_kv_79_b300 import build
    build.build()
    M.lib()
    yield


@pytest.fixture(params=["tcgen05", "simt"])
def path(request):
    old = M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 1 if request.param == "simt" else 0)
    yield request.param
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, old)
    assert M.mla_get_device_error() == 0


def weights(seed, n):
    rng = np.random.default_rng(seed)
    return dict(
        x=W.quantise(W.normal(rng, (n, DS.d_model)), "bf16"),
        w_dq=W.weight(rng, DS.d_model, D_CQ, "bf16"),
        w_uq=W.weight(rng, D_CQ, DS.n_heads * DS.d_nope, "bf16"),
        w_qr=W.weight(rng, D_CQ, DS.n_heads * DS.d_rope, "bf16"),
        w_uk=W.weight(rng, DS.d_latent, DS.n_heads * DS.d_nope, "bf16"),
        pos=rng.integers(0, 100000, size=n).astype(np.int32),
    )


def f64(a):
    return W.to_f64(a, "bf16")


@pytest.mark.parametrize("n", [37, 300])
def test_compressed_query_chain_matches_oracle(path, n):
    """c_q, q_nope, q_rope, the folded weight and both ways to q_cat against the oracle."""
    w = weights(90 + n, n)
    cfg = cfg_of(DS, "bf16")
    c_q = M.mla_query_latent(cfg, dev(w["x"]), dev(w["w_dq"]))
    q_nope, q_rope = M.mla_query_up(cfg, c_q, dev(w["w_uq"]), dev(w["w_qr"]))
    q_cat_a = M.mla_absorb_q(cfg, q_nope, q_rope, i32(w["pos"]), dev(w["w_uk"]))
    w_uqk = M.mla_fold_uq_uk(cfg, dev(w["w_uq"]), dev(w["w_uk"]))
    _, q_rope_only = M.mla_query_up(cfg, c_q, None, dev(w["w_qr"]))
    q_cat_c = M.mla_absorb_q_compressed(cfg, c_q, q_rope_only, i32(w["pos"]), w_uqk)
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0

    cq_ref = O.query_latent(f64(w["x"]), f64(w["w_dq"]))
    assert rel(host(c_q), cq_ref) <= TOL_OUT_BF16
    qn_ref, qr_ref = O.query_projection_compressed(f64(w["x"]), f64(w["w_dq"]), f64(w["w_uq"]), f64(w["w_qr"]),
                                                   w["pos"], DS.n_heads, DS.rope_base)
    assert rel(host(q_nope), qn_ref) <= TOL_OUT_BF16
    # q_rope is returned unrotated; the oracle's is rotated at the token's position
    qr_unrot = O.query_projection_compressed(f64(w["x"]), f64(w["w_dq"]), f64(w["w_uq"]), f64(w["w_qr"]),
                                             np.zeros(n), DS.n_heads, DS.rope_base)[1]
    assert rel(host(q_rope), qr_unrot) <= TOL_OUT_BF16
    assert np.array_equal(host(q_rope_only), host(q_rope))
    wuqk_ref = O.absorb_uq_uk(f64(w["w_uq"]), f64(w["w_uk"]), DS.n_heads)
    assert rel(host(w_uqk), wuqk_ref) <= TOL_OUT_BF16
    qcat_ref = O.absorb_query(qn_ref, O.query_projection_compressed(f64(w["x"]), f64(w["w_dq"]), f64(w["w_uq"]),
                                                                    f64(w["w_qr"]), np.zeros(n), DS.n_heads,
                                                                    DS.rope_base)[1],
                              w["pos"], f64(w["w_uk"]), DS.rope_base)
    for got in (host(q_cat_a), host(q_cat_c)):
        assert rel(got[..., :DS.d_latent], qcat_ref[..., :DS.d_latent]) <= TOL_OUT_BF16
        assert rel(got[..., DS.d_latent:], qcat_ref[..., DS.d_latent:]) <= TOL_OUT_BF16


def test_compressed_query_decode_chain():
    """x -> c_q -> q_cat (folded weight) -> decode -> out, against the un-absorbed oracle with the
    compressed query; lse at 1e-3 against the oracle on the device's q_cat and cache rows."""
    lens = [700, 64, 1, 2049]
    case = W.make_decode_case(DS, "bf16", lens, seed=93)
    B = len(lens)
    w = weights(94, B)
    cfg = cfg_of(DS, "bf16")
    cache = M.PagedCache(dev(case["pool"]), i32(case["page_table"]), i32(case["seq_lens"]))
    pos = case["pos"]
    c_q = M.mla_query_latent(cfg, dev(w["x"]), dev(w["w_dq"]))
    _, q_rope = M.mla_query_up(cfg, c_q, None, dev(w["w_qr"]))
    w_uqk = M.mla_fold_uq_uk(cfg, dev(w["w_uq"]), dev(case["w_uk"]))
    q_cat = M.mla_absorb_q_compressed(cfg, c_q, q_rope, i32(pos), w_uqk)
    o_lat, lse = M.mla_decode(cfg, cache, q_cat)
    o = M.mla_out(cfg, o_lat, dev(case["w_uv"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    qn, qr = O.query_projection_compressed(f64(w["x"]), f64(w["w_dq"]), f64(w["w_uq"]), f64(w["w_qr"]), pos,
                                           DS.n_heads, DS.rope_base)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    pool = f64(case["pool"])
    go, gl, gq = host(o), host(lse), host(q_cat)
    for b in range(B):
        rows = O.sequence_rows(pool, case["page_table"][b], lens[b])
        ro, _, _, _ = O.attention_unabsorbed(qn[b], qr[b], rows[:, :DS.d_latent], rows[:, DS.d_latent:],
                                             f64(case["w_uk"]), f64(case["w_uv"]), sc)
        assert rel(go[b], ro.reshape(-1)) <= TOL_OUT_BF16, b
        _, rl = O.attention_latent(gq[b], rows, DS.d_latent, sc)
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b
