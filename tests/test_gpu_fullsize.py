"""GPU parity at the full sizes of the four DeepSeek-V2-shaped workloads, in the launch
configuration the benchmark times (default tuning: tcgen05 kernels, automatic split units).

Outputs are compared with the CPU oracle on every output the oracle can afford (all heads of
all sequences where that is cheap, sampled sequences or query tokens otherwise); the cache
append is compared row by row with the oracle's down-projection and checked to leave every
other row bit-identical.  Tolerances: relative max-abs 2e-2 on outputs, 1e-3 on lse."""
import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M

from tests.gpu_util import TOL_LSE_BF16, TOL_OUT_BF16, cache_of, cfg_of, dev, host, i32, rel

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2
SC = O.default_scale(DS.d_nope, DS.d_rope)


def rows_f64(pool_bits, pt_row, length):
    return W.to_f64(W.gather_rows(pool_bits, pt_row, length), "bf16")


def device_rows(pool_t, pt_row, length):
    """Rows [0, length) of one sequence read back from the device pool (bf16 bits)."""
    ps = DS.page_size
    pages = torch.from_numpy(np.asarray(pt_row[:W.pages_for(length, ps)], dtype=np.int64)).to(pool_t.device)
    bits = pool_t.view(torch.int16).index_select(0, pages).cpu().numpy().view(np.uint16)
    return bits.reshape(-1, DS.width)[:length]


def check_attention(go, gl, q_cat_f64, rows, what):
    ro, rl = O.attention_latent(q_cat_f64, rows, DS.d_latent, SC)
    assert rel(go, ro) <= TOL_OUT_BF16, what
    assert np.max(np.abs(gl - rl)) <= TOL_LSE_BF16, what


def test_decode_b16_l4096_all_outputs():
    case = W.make_workload("decode_b16_l4096")
    cfg = cfg_of(DS, "bf16")
    o, lse = M.mla_decode(cfg, cache_of(case), dev(case["q_cat"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    go, gl = host(o), host(lse)
    qc = W.to_f64(case["q_cat"], "bf16")
    for b in range(16):
        check_attention(go[b], gl[b], qc[b], rows_f64(case["pool"], case["page_table"][b], int(case["seq_lens"][b])), b)


def test_decode_long_b4_all_outputs():
    case = W.make_workload("decode_long_b4")
    assert list(case["seq_lens"]) == [32768, 65536, 98304, 131072]
    cfg = cfg_of(DS, "bf16")
    o, lse = M.mla_decode(cfg, cache_of(case), dev(case["q_cat"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    go, gl = host(o), host(lse)
    qc = W.to_f64(case["q_cat"], "bf16")
    for b in range(4):
        check_attention(go[b], gl[b], qc[b], rows_f64(case["pool"], case["page_table"][b], int(case["seq_lens"][b])), b)


def test_decode_ragged_b256_with_append():
    case = W.make_workload("decode_ragged_b256")
    B = 256
    lens0 = case["append_pos"]           # lengths before the append
    assert case["seq_lens"].shape == (B,) and np.all(case["seq_lens"] == lens0 + 1)
    assert lens0.min() >= 256 and lens0.max() <= 8192
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]),
                       i32(case["append_seq"]), i32(case["append_pos"]))
    o, lse = M.mla_decode(cfg, cache, dev(case["q_cat"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    go, gl = host(o), host(lse)

    # the appended rows: [c_kv | RoPE(k)] of the oracle, rounded once to bf16 by the path
    c_ref, k_ref = O.latent_kv(W.to_f64(case["x"], "bf16"), W.to_f64(case["w_dkv"], "bf16"),
                               W.to_f64(case["w_kr"], "bf16"), case["append_pos"], DS.rope_base)
    ref_rows = np.concatenate([c_ref, k_ref], axis=1)
    qc = W.to_f64(case["q_cat"], "bf16")
    sample = sorted(set(list(range(0, B, 8)) + [int(np.argmin(lens0)), int(np.argmax(lens0)), B - 1]))
    for b in sample:
        L = int(case["seq_lens"][b])
        got_bits = device_rows(cache.pool, case["page_table"][b], L)
        # every row before the appended one is untouched, bit for bit
        assert np.array_equal(got_bits[:L - 1], W.gather_rows(case["pool"], case["page_table"][b], L - 1)), b
        new = W.to_f64(got_bits[L - 1], "bf16")
        assert rel(new[:DS.d_latent], ref_rows[b, :DS.d_latent]) <= TOL_OUT_BF16, b
        assert rel(new[DS.d_latent:], ref_rows[b, DS.d_latent:]) <= TOL_OUT_BF16, b
        # attention over the cache as the device holds it
        check_attention(go[b], gl[b], qc[b], W.to_f64(got_bits, "bf16"), b)


def test_prefill_t8192_cache_build_absorb_and_causal_attention():
    case = W.make_workload("prefill_t8192")
    T = 8192
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]),
                       i32(case["append_seq"]), i32(case["append_pos"]))
    q_cat = M.mla_absorb_q(cfg, dev(case["q_nope"]), dev(case["q_rope"]), i32(case["append_pos"]),
                           dev(case["w_uk"]))
    o, lse = M.mla_prefill(cfg, cache, 0, 0, q_cat)
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0

    rng = np.random.default_rng(5)
    tok = sorted(set([0, 1, 63, 64, 65, 127, 4095, 4096, T - 2, T - 1] + list(rng.integers(0, T, 6))))
    idx = torch.tensor(tok, dtype=torch.int64, device="cuda")
    go, gl = host(o.index_select(0, idx)), host(lse.index_select(0, idx))
    gq = host(q_cat.index_select(0, idx))
    pool_bits = device_rows(cache.pool, case["page_table"][0], T)

    # cache build: sampled rows against the oracle's down-projection
    xs = W.to_f64(case["x"], "bf16")[tok]
    c_ref, k_ref = O.latent_kv(xs, W.to_f64(case["w_dkv"], "bf16"), W.to_f64(case["w_kr"], "bf16"),
                               np.asarray(tok), DS.rope_base)
    got = W.to_f64(pool_bits[tok], "bf16")
    assert rel(got[:, :DS.d_latent], c_ref) <= TOL_OUT_BF16
    assert rel(got[:, DS.d_latent:], k_ref) <= TOL_OUT_BF16
    # absorbed queries of the sampled tokens
    q_ref = O.absorb_query(W.to_f64(case["q_nope"], "bf16")[tok], W.to_f64(case["q_rope"], "bf16")[tok],
                           np.asarray(tok), W.to_f64(case["w_uk"], "bf16"), DS.rope_base)
    assert rel(gq, q_ref) <= TOL_OUT_BF16
    # causal attention of the sampled queries over the cache and queries as the device holds them
    rows = W.to_f64(pool_bits, "bf16")
    for j, i in enumerate(tok):
        check_attention(go[j], gl[j], gq[j], rows[:i + 1], i)
