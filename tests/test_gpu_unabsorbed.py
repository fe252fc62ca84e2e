"""GPU parity of the un-absorbed causal prefill (restore K and V from the cached latent, then
192-wide causal attention), against the oracle's un-absorbed chain of the operator-notes page.

o is compared with the oracle run on the cache rows the device holds (2e-2 relative per query
row).  lse is compared at 1e-3 with the oracle's attention on the same bf16 intermediates the
device computes with (the rotated query part, K and V rounded to bf16 by the storage cast of
the input generator), and against the plain oracle with the first-order rounding bound."""
import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M

from tests.gpu_util import TOL_LSE_BF16, TOL_OUT_BF16, cfg_of, dev, host, i32, rel

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2
SC = O.default_scale(DS.d_nope, DS.d_rope)
DH, DC = DS.d_nope, DS.d_latent


@pytest.fixture(scope="module", autouse=True)
def _ready():
    from mla_latent_kv_79_b300 import build
    build.build()
    M.lib()
    yield


def f64(a):
    return W.to_f64(a, "bf16")


def to_bf16(a):
    return W.to_f64(W.quantise(np.asarray(a, dtype=np.float32), "bf16"), "bf16")


def built_cache(T, seed):
    """A sequence of T tokens whose cache rows are appended on the device from x."""
    case = W.make_prefill_case(DS, "bf16", T, seed)
    cfg = cfg_of(DS, "bf16")
    cache = M.PagedCache(dev(case["pool"]), i32(case["page_table"]), i32(case["seq_lens"]))
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]), i32(case["append_seq"]),
                       i32(case["append_pos"]))
    return case, cfg, cache


def device_rows(cache, case, T):
    ps = DS.page_size
    pages = torch.from_numpy(np.asarray(case["page_table"][0][:W.pages_for(T, ps)], dtype=np.int64)).cuda()
    bits = cache.pool.view(torch.int16).index_select(0, pages).cpu().numpy().view(np.uint16)
    return f64(bits.reshape(-1, DS.width)[:T])


def cols(w, heads):
    return np.concatenate([w[:, h * DH:(h + 1) * DH] for h in heads], axis=1)


def lse_on_intermediates(q_nope_h, q_r_h, K_h, k_rope, V_h):
    """The oracle's attention for one head when K_h and V_h are given: the latent is [K_h | V_h]
    and the up-projections select its halves (exact in float64)."""
    eye, zero = np.eye(DH), np.zeros((DH, DH))
    o, _, lse, _ = O.attention_unabsorbed(q_nope_h[None], q_r_h[None], np.concatenate([K_h, V_h], axis=1), k_rope,
                                          np.vstack([eye, zero]), np.vstack([zero, eye]), SC)
    return o[0], lse[0]


@pytest.mark.parametrize("q_start,n_q", [(0, 300), (300, 120), (5, 131)])
def test_unabsorbed_prefill_matches_oracle(q_start, n_q):
    """Every query row against the oracle's causal un-absorbed prefill; query tiles that start
    mid-tile (q_start not a multiple of 128) and a ragged last tile."""
    T = q_start + n_q
    case, cfg, cache = built_cache(T, seed=60 + q_start)
    qn, qr = case["q_nope"][q_start:], case["q_rope"][q_start:]
    o, lse = M.mla_prefill_unabsorbed(cfg, cache, 0, q_start, dev(qn), dev(qr), dev(case["w_uk"]), dev(case["w_uv"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    assert M.mla_last_attention_path() == 3
    go, gl = host(o), host(lse)
    rows = device_rows(cache, case, T)
    q_r = O.rope_rotate(f64(case["q_rope"]), np.arange(T)[:, None], DS.rope_base)
    ro, _, rl = O.causal_prefill_unabsorbed(f64(case["q_nope"]), q_r, rows[:, :DC], rows[:, DC:], f64(case["w_uk"]),
                                            f64(case["w_uv"]), SC)
    for i in range(n_q):
        assert rel(go[i], ro[q_start + i].reshape(-1)) <= TOL_OUT_BF16, i
    # lse: 1e-3 against the oracle on the device's bf16 intermediates, sampled rows x heads
    heads = [0, 1, 37, 64, 127]
    K, V = O.restore_kv(rows[:, :DC], cols(f64(case["w_uk"]), heads), cols(f64(case["w_uv"]), heads), len(heads))
    Kb, Vb = to_bf16(K), to_bf16(V)
    q_rb = to_bf16(q_r)
    for i in sorted({0, 1, n_q // 2, n_q - 1}):
        t = q_start + i
        for j, h in enumerate(heads):
            oo, ll = lse_on_intermediates(f64(case["q_nope"])[t, h], q_rb[t, h], Kb[:t + 1, j], rows[:t + 1, DC:],
                                          Vb[:t + 1, j])
            assert abs(gl[i, h] - ll) <= TOL_LSE_BF16, (i, h, gl[i, h] - ll)
            assert rel(go[i, h * DH:(h + 1) * DH], oo) <= TOL_OUT_BF16, (i, h)


def test_unabsorbed_equals_absorbed_prefill():
    """The two forms of the same prefill (the glossary's absorption is exact by associativity):
    mla_prefill + mla_out and mla_prefill_unabsorbed agree within the rounding of both."""
    T = 400
    case, cfg, cache = built_cache(T, seed=77)
    q_cat = M.mla_absorb_q(cfg, dev(case["q_nope"]), dev(case["q_rope"]), i32(case["append_pos"]), dev(case["w_uk"]))
    o_lat, lse_a = M.mla_prefill(cfg, cache, 0, 0, q_cat)
    o_a = M.mla_out(cfg, o_lat, dev(case["w_uv"]))
    o_u, lse_u = M.mla_prefill_unabsorbed(cfg, cache, 0, 0, dev(case["q_nope"]), dev(case["q_rope"]),
                                          dev(case["w_uk"]), dev(case["w_uv"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    assert rel(host(o_u), host(o_a)) <= TOL_OUT_BF16
    assert np.max(np.abs(host(lse_u) - host(lse_a))) <= 2e-2  # both round their query to bf16


def test_unabsorbed_prefill_t8192_sampled():
    """The full-size prefill workload (8192 tokens, 128 heads): sampled query rows x 16 heads."""
    T = 8192
    case = W.make_workload("prefill_t8192")
    cfg = cfg_of(DS, "bf16")
    cache = M.PagedCache(dev(case["pool"]), i32(case["page_table"]), i32(case["seq_lens"]))
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]), i32(case["append_seq"]),
                       i32(case["append_pos"]))
    o, lse = M.mla_prefill_unabsorbed(cfg, cache, 0, 0, dev(case["q_nope"]), dev(case["q_rope"]), dev(case["w_uk"]),
                                      dev(case["w_uv"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    rng = np.random.default_rng(8)
    tok = sorted(set([0, 1, 63, 64, 127, 128, 4095, 4096, T - 2, T - 1] + list(rng.integers(0, T, 6))))
    heads = sorted(set([0, 127] + list(rng.choice(DS.n_heads, 14, replace=False))))
    idx = torch.tensor(tok, dtype=torch.int64, device="cuda")
    go, gl = host(o.index_select(0, idx)), host(lse.index_select(0, idx))
    rows = device_rows(cache, case, T)
    K, V = O.restore_kv(rows[:, :DC], cols(f64(case["w_uk"]), heads), cols(f64(case["w_uv"]), heads), len(heads))
    q_r = O.rope_rotate(f64(case["q_rope"])[tok], np.asarray(tok)[:, None], DS.rope_base)
    qn = f64(case["q_nope"])[tok]
    Kb, Vb, q_rb = to_bf16(K), to_bf16(V), to_bf16(q_r)
    for a, t in enumerate(tok):
        for j, h in enumerate(heads):
            ro, rl = lse_on_intermediates(qn[a, h], q_r[a, h], K[:t + 1, j], rows[:t + 1, DC:], V[:t + 1, j])
            assert rel(go[a, h * DH:(h + 1) * DH], ro) <= TOL_OUT_BF16, (t, h)
            _, lb = lse_on_intermediates(qn[a, h], q_rb[a, h], Kb[:t + 1, j], rows[:t + 1, DC:], Vb[:t + 1, j])
            assert abs(gl[a, h] - lb) <= TOL_LSE_BF16, (t, h, gl[a, h] - lb)
