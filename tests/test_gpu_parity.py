"""GPU parity: every entry point of the C ABI against the CPU oracle on seeded inputs.

Sizes span several 64-token pages and ragged tails; each test runs on the SIMT kernels and
on the default dispatch (tcgen05 where the shape takes it)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M
from mla_latent_kv_79_b300 import _lib
from tests.gpu_util import (TOL_LSE_BF16, TOL_LSE_F32, TOL_OUT_BF16, TOL_OUT_F32, Guarded,
                            cache_of, cfg_of, dev, host, i32, lse_rounding_bound, rel)

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_79_b300 import build
    build.build()
    M.lib()
    yield
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 0)
    M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, 0)


@pytest.fixture(params=["simt", "auto"])
def path(request):
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 1 if request.param == "simt" else 0)
    yield request.param
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 0)


def f64(a, dtype="bf16"):
    return W.to_f64(a, dtype)


def tol(dtype):
    return (TOL_OUT_BF16, TOL_LSE_BF16) if dtype == "bf16" else (TOL_OUT_F32, TOL_LSE_F32)


def oracle_decode(case, b, heads=None, q_cat=None):
    """Oracle o_lat, lse of sequence b from the stored q_cat and cache rows."""
    s = case["shape"]
    L = int(case["seq_lens"][b])
    rows = O.sequence_rows(f64(case["pool"], case["dtype"]), case["page_table"][b], L)
    qc = f64(case["q_cat"], case["dtype"])[b] if q_cat is None else q_cat[b]
    if heads is not None:
        qc = qc[heads]
    return O.attention_latent(qc, rows, s.d_latent, O.default_scale(s.d_nope, s.d_rope))


def assert_no_device_error():
    assert M.mla_get_device_error() == 0


# ----------------------------------------------------------------------------------- append

@pytest.mark.parametrize("dtype,shape", [("bf16", DS), ("f32", W.TINY)])
def test_append_matches_oracle_and_touches_only_its_rows(path, dtype, shape):
    lens = [0, 10, 63, 70]
    case = W.make_decode_case(shape, dtype, [l for l in lens], seed=31, spare_pages=3)
    r = np.random.default_rng(32)
    # 100 new tokens spread over the sequences at fresh positions beyond their lengths
    seq = np.concatenate([np.full(25, b, np.int32) for b in range(4)])
    pos = np.concatenate([np.arange(25, dtype=np.int32) + l for l in lens])
    pt_alloc, n_pages = W.make_page_table(r, [l + 25 for l in lens], shape.page_size, 2, True)
    pool0 = W.empty_pool(n_pages, shape, dtype)
    x = W.quantise(W.normal(r, (100, shape.d_model)), dtype)
    wd = W.weight(r, shape.d_model, shape.d_latent, dtype)
    wk = W.weight(r, shape.d_model, shape.d_rope, dtype)
    cfg = cfg_of(shape, dtype)
    cache = M.PagedCache(dev(pool0, dtype), i32(pt_alloc), i32(np.array(lens) + 25))
    M.mla_cache_append(cfg, cache, dev(x, dtype), dev(wd, dtype), dev(wk, dtype), i32(seq), i32(pos))
    torch.cuda.synchronize()
    assert_no_device_error()
    got = host(cache.pool)
    c_ref, k_ref = O.latent_kv(f64(x, dtype), f64(wd, dtype), f64(wk, dtype), pos, shape.rope_base)
    ps = shape.page_size
    written = np.zeros(got.shape[:2], bool)
    g_c = np.empty_like(c_ref)
    g_k = np.empty_like(k_ref)
    for n in range(100):
        page = pt_alloc[seq[n], pos[n] // ps]
        written[page, pos[n] % ps] = True
        g_c[n] = got[page, pos[n] % ps, :shape.d_latent]
        g_k[n] = got[page, pos[n] % ps, shape.d_latent:]
    t_out = tol(dtype)[0]
    assert rel(g_c, c_ref) <= t_out and rel(g_k, k_ref) <= t_out
    # every other slot is bit-for-bit the sentinel it held before
    before = f64(pool0, dtype)
    assert np.array_equal(got[~written], before[~written])


def test_append_integer_inputs_are_bit_exact(path):
    """Small-integer x and power-of-two weights at position 0: fp32 accumulation is exact,
    so the stored bf16 row equals the oracle's exact value bit for bit."""
    s = W.replace_shape(DS, d_model=256)
    r = np.random.default_rng(33)
    # three nonzero activations (+-1, +-2) per token and weights +-2^-k (k <= 3): every dot
    # product is a multiple of 2^-3 below 8 in magnitude, exact in fp32 and in bf16
    x = np.zeros((16, s.d_model), np.float32)
    for n in range(16):
        idx = r.choice(s.d_model, size=3, replace=False)
        x[n, idx] = r.choice([-2.0, -1.0, 1.0, 2.0], size=3)
    wd = (2.0 ** -r.integers(0, 4, size=(s.d_model, s.d_latent)) * r.choice([-1, 1], size=(s.d_model, s.d_latent))).astype(np.float32)
    wk = (2.0 ** -r.integers(0, 4, size=(s.d_model, s.d_rope)) * r.choice([-1, 1], size=(s.d_model, s.d_rope))).astype(np.float32)
    pt = np.arange(16, dtype=np.int32).reshape(16, 1)
    pool0 = W.empty_pool(16, s, "bf16")
    cfg = cfg_of(s, "bf16")
    cache = M.PagedCache(dev(pool0), i32(pt), i32(np.ones(16)))
    M.mla_cache_append(cfg, cache, dev(W.quantise(x, "bf16")), dev(W.quantise(wd, "bf16")),
                       dev(W.quantise(wk, "bf16")), i32(np.arange(16)), i32(np.zeros(16)))
    got = host(cache.pool)[:, 0, :]
    c_ref, k_ref = O.latent_kv(x.astype(np.float64), wd.astype(np.float64), wk.astype(np.float64),
                               np.zeros(16), s.rope_base)
    ref = np.concatenate([c_ref, k_ref], axis=1)
    ref_b = W.bf16_bits_to_f32(W.to_bf16_bits(ref.astype(np.float32)))
    assert np.array_equal(ref_b, ref.astype(np.float32)), "fixture not exactly representable"
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------------------------- absorb / out

@pytest.mark.parametrize("dtype,shape,n", [("bf16", DS, 37), ("bf16", DS, 200), ("f32", W.TINY, 5)])
def test_absorb_q_matches_oracle(path, dtype, shape, n):
    case = W.make_decode_case(shape, dtype, [1] * n, seed=41)
    pos = np.random.default_rng(42).integers(0, 100000, size=n).astype(np.int32)
    cfg = cfg_of(shape, dtype)
    out = Guarded((n, shape.n_heads, shape.width), cfg.torch_dtype)
    M.mla_absorb_q(cfg, dev(case["q_nope"], dtype), dev(case["q_rope"], dtype), i32(pos),
                   dev(case["w_uk"], dtype), q_cat=out.t)
    torch.cuda.synchronize()
    out.check()
    ref = O.absorb_query(f64(case["q_nope"], dtype), f64(case["q_rope"], dtype), pos,
                         f64(case["w_uk"], dtype), shape.rope_base)
    got = host(out.t)
    t_out = tol(dtype)[0]
    assert rel(got[..., :shape.d_latent], ref[..., :shape.d_latent]) <= t_out
    assert rel(got[..., shape.d_latent:], ref[..., shape.d_latent:]) <= t_out


@pytest.mark.parametrize("dtype,shape,n", [("bf16", DS, 37), ("bf16", DS, 200), ("f32", W.TINY, 5)])
def test_out_matches_oracle(path, dtype, shape, n):
    r = np.random.default_rng(43)
    o_lat = W.quantise(W.normal(r, (n, shape.n_heads, shape.d_latent)), dtype)
    w_uv = W.weight(r, shape.d_latent, shape.n_heads * shape.d_nope, dtype)
    cfg = cfg_of(shape, dtype)
    out = Guarded((n, shape.n_heads * shape.d_nope), cfg.torch_dtype)
    M.mla_out(cfg, dev(o_lat, dtype), dev(w_uv, dtype), o=out.t)
    torch.cuda.synchronize()
    out.check()
    ref = O.up_project_output(f64(o_lat, dtype), f64(w_uv, dtype))
    assert rel(host(out.t), ref) <= tol(dtype)[0]


@pytest.mark.parametrize("dtype,shape,n", [("bf16", DS, 37), ("f32", W.TINY, 5)])
def test_query_proj_then_absorb_matches_oracle(path, dtype, shape, n):
    """The query side, q_nope = x . W_Q and q_rope = x . W_QR (unrotated), then mla_absorb_q,
    against the oracle's query projection (which rotates q_rope itself)."""
    r = np.random.default_rng(45)
    x = W.quantise(W.normal(r, (n, shape.d_model)), dtype)
    w_q = W.weight(r, shape.d_model, shape.n_heads * shape.d_nope, dtype)
    w_qr = W.weight(r, shape.d_model, shape.n_heads * shape.d_rope, dtype)
    w_uk = W.weight(r, shape.d_latent, shape.n_heads * shape.d_nope, dtype)
    pos = r.integers(0, 5000, size=n).astype(np.int32)
    cfg = cfg_of(shape, dtype)
    qn = Guarded((n, shape.n_heads, shape.d_nope), cfg.torch_dtype)
    qr = Guarded((n, shape.n_heads, shape.d_rope), cfg.torch_dtype)
    M.mla_query_proj(cfg, dev(x, dtype), dev(w_q, dtype), dev(w_qr, dtype), q_nope=qn.t, q_rope=qr.t)
    q_cat = M.mla_absorb_q(cfg, qn.t, qr.t, i32(pos), dev(w_uk, dtype))
    torch.cuda.synchronize()
    assert_no_device_error()
    qn.check()
    qr.check()
    ref_qn, ref_qr = O.query_projection(f64(x, dtype), f64(w_q, dtype), f64(w_qr, dtype), pos, shape.n_heads,
                                        shape.rope_base)
    t_out = tol(dtype)[0]
    assert rel(host(qn.t), ref_qn) <= t_out
    # the RoPE half of q_cat is the oracle's rotated RoPE query (mla_absorb_q applies the rotation)
    assert rel(host(q_cat)[..., shape.d_latent:], ref_qr) <= t_out


@pytest.mark.parametrize("dtype,shape,n", [("bf16", DS, 37), ("bf16", DS, 200), ("f32", W.TINY, 5)])
def test_out_proj_matches_oracle(path, dtype, shape, n):
    """The final projection over the concatenated heads, out = o . W_O, against the oracle's."""
    r = np.random.default_rng(44)
    o = W.quantise(W.normal(r, (n, shape.n_heads * shape.d_nope)), dtype)
    w_o = W.weight(r, shape.n_heads * shape.d_nope, shape.d_model, dtype)
    cfg = cfg_of(shape, dtype)
    out = Guarded((n, shape.d_model), cfg.torch_dtype)
    M.mla_out_proj(cfg, dev(o, dtype), dev(w_o, dtype), out=out.t)
    torch.cuda.synchronize()
    assert_no_device_error()
    out.check()
    assert rel(host(out.t), O.output_projection(f64(o, dtype), f64(w_o, dtype))) <= tol(dtype)[0]


@pytest.mark.parametrize("ksplit,stages", [(1, 0), (2, 0), (3, 0), (8, 2)])
def test_gemm_k_split_matches_oracle(ksplit, stages):
    """The tcgen05 GEMMs with K split over a cluster forced to uneven splits (W_UV's 8 K chunks
    in 3 parts, d_model's 80 and W_O's 256 in 3 or 8), and with the split turned off (1) for a
    decode-sized append and output projection: every mode's result is the oracle's whatever the
    split."""
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 0)
    old_k = M.mla_set_tuning(_lib.MLA_TUNE_GEMM_KSPLIT, ksplit)
    old_s = M.mla_set_tuning(_lib.MLA_TUNE_GEMM_STAGES, stages)
    try:
        r = np.random.default_rng(47)
        cfg = cfg_of(DS, "bf16")
        n = 45
        # absorb
        case = W.make_decode_case(DS, "bf16", [1] * n, seed=48)
        pos = r.integers(0, 100000, size=n).astype(np.int32)
        q_cat = Guarded((n, DS.n_heads, DS.width), cfg.torch_dtype)
        M.mla_absorb_q(cfg, dev(case["q_nope"]), dev(case["q_rope"]), i32(pos), dev(case["w_uk"]), q_cat=q_cat.t)
        # out
        o_lat = W.quantise(W.normal(r, (n, DS.n_heads, DS.d_latent)), "bf16")
        w_uv = W.weight(r, DS.d_latent, DS.n_heads * DS.d_nope, "bf16")
        o = Guarded((n, DS.n_heads * DS.d_nope), cfg.torch_dtype)
        M.mla_out(cfg, dev(o_lat), dev(w_uv), o=o.t)
        # output projection over the heads
        o_in = W.quantise(W.normal(r, (n, DS.n_heads * DS.d_nope)), "bf16")
        w_o = W.weight(r, DS.n_heads * DS.d_nope, DS.d_model, "bf16")
        op = Guarded((n, DS.d_model), cfg.torch_dtype)
        M.mla_out_proj(cfg, dev(o_in), dev(w_o), out=op.t)
        # append: one token per sequence at ragged positions
        lens = r.integers(1, 200, size=n)
        pt, n_pages = W.make_page_table(r, [int(l) + 1 for l in lens], DS.page_size, 2, True)
        pool0 = W.empty_pool(n_pages, DS, "bf16")
        cache = M.PagedCache(dev(pool0), i32(pt), i32(lens + 1))
        x = W.quantise(W.normal(r, (n, DS.d_model)), "bf16")
        wd = W.weight(r, DS.d_model, DS.d_latent, "bf16")
        wk = W.weight(r, DS.d_model, DS.d_rope, "bf16")
        M.mla_cache_append(cfg, cache, dev(x), dev(wd), dev(wk), i32(np.arange(n)), i32(lens))
        torch.cuda.synchronize()
        assert_no_device_error()
        q_cat.check()
        o.check()
        op.check()
        assert rel(host(op.t), O.output_projection(f64(o_in), f64(w_o))) <= TOL_OUT_BF16
        ref = O.absorb_query(f64(case["q_nope"]), f64(case["q_rope"]), pos, f64(case["w_uk"]), DS.rope_base)
        got = host(q_cat.t)
        assert rel(got[..., :DS.d_latent], ref[..., :DS.d_latent]) <= TOL_OUT_BF16
        assert rel(got[..., DS.d_latent:], ref[..., DS.d_latent:]) <= TOL_OUT_BF16
        assert rel(host(o.t), O.up_project_output(f64(o_lat), f64(w_uv))) <= TOL_OUT_BF16
        got_pool = host(cache.pool)
        c_ref, k_ref = O.latent_kv(f64(x), f64(wd), f64(wk), lens, DS.rope_base)
        written = np.zeros(got_pool.shape[:2], bool)
        for b in range(n):
            page, slot = pt[b, lens[b] // DS.page_size], lens[b] % DS.page_size
            written[page, slot] = True
            assert rel(got_pool[page, slot, :DS.d_latent], c_ref[b]) <= TOL_OUT_BF16, b
            assert rel(got_pool[page, slot, DS.d_latent:], k_ref[b]) <= TOL_OUT_BF16, b
        assert np.array_equal(got_pool[~written], f64(pool0)[~written])
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_GEMM_KSPLIT, old_k)
        M.mla_set_tuning(_lib.MLA_TUNE_GEMM_STAGES, old_s)


# ----------------------------------------------------------------------------------- decode

DECODE_LENS = [1, 63, 64, 65, 300, 1000, 2049, 130]


@pytest.mark.parametrize("units", [0, 1, 3, 7])
def test_decode_matches_oracle(path, units):
    case = W.make_decode_case(DS, "bf16", DECODE_LENS, seed=51, spare_pages=5)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    B = len(DECODE_LENS)
    o = Guarded((B, DS.n_heads, DS.d_latent), torch.bfloat16)
    lse = Guarded((B, DS.n_heads), torch.float32)
    old = M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, units)
    try:
        M.mla_decode(cfg, cache, dev(case["q_cat"]), o_lat=o.t, lse=lse.t)
        torch.cuda.synchronize()
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old)
    o.check(); lse.check()
    assert_no_device_error()
    go, gl = host(o.t), host(lse.t)
    for b in range(B):
        ro, rl = oracle_decode(case, b)
        assert rel(go[b], ro) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b


def test_decode_f32_tiny_shapes(path):
    case = W.make_decode_case(W.TINY, "f32", [1, 64, 65, 200], seed=52)
    cfg = cfg_of(W.TINY, "f32")
    o, lse = M.mla_decode(cfg, cache_of(case), dev(case["q_cat"], "f32"))
    go, gl = host(o), host(lse)
    for b in range(4):
        ro, rl = oracle_decode(case, b)
        assert rel(go[b], ro) <= TOL_OUT_F32 and np.max(np.abs(gl[b] - rl)) <= TOL_LSE_F32


def test_decode_split_counts_agree(path):
    case = W.make_decode_case(DS, "bf16", [3000, 70, 1], seed=53)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    q = dev(case["q_cat"])
    outs = []
    for units in (1, 2, 7, 64, 10000):
        old = M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, units)
        try:
            o, l = M.mla_decode(cfg, cache, q)
        finally:
            M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old)
        outs.append((host(o), host(l)))
    for o, l in outs[1:]:
        assert rel(o, outs[0][0]) <= TOL_OUT_BF16
        assert np.max(np.abs(l - outs[0][1])) <= TOL_LSE_BF16


@pytest.mark.parametrize("lens,units", [([3000, 70, 1], 2), ([2944, 70], 2), ([1600, 70, 1], 2),
                                        ([3000, 70, 1], 3), ([70, 3000, 1], 2)])
def test_decode_split_then_multipage_segment(path, lens, units):
    """A unit whose split segment (fp32 partial, slow drain) is followed by a multi-page
    segment: the next segment's P buffers fill during the drain."""
    case = W.make_decode_case(DS, "bf16", lens, seed=53)
    old = M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, units)
    try:
        o, l = M.mla_decode(cfg_of(DS, "bf16"), cache_of(case), dev(case["q_cat"]))
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old)
    go, gl = host(o), host(l)
    for b in range(len(lens)):
        ro, rl = oracle_decode(case, b)
        assert rel(go[b], ro) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b
    assert_no_device_error()


@pytest.mark.parametrize("units", [1, 3])
def test_decode_running_max_jumps(path, units):
    """Later cache rows scaled by 4 and then 16 (exact in bf16): the scores jump by far more
    than the lazy-rescale threshold, so O and l are rescaled mid-segment."""
    lens = [1000, 2049]
    case = W.make_decode_case(DS, "bf16", lens, seed=59)
    pool = case["pool"].copy()
    for b, L in enumerate(lens):
        rows = W.bf16_bits_to_f32(W.gather_rows(pool, case["page_table"][b], L)).copy()
        rows[128:] *= 4.0
        rows[640:] *= 4.0
        W.scatter_rows(pool, case["page_table"][b], W.quantise(rows, "bf16"))
    case = dict(case, pool=pool)
    old = M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, units)
    try:
        o, l = M.mla_decode(cfg_of(DS, "bf16"), cache_of(case), dev(case["q_cat"]))
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old)
    go, gl = host(o), host(l)
    for b in range(len(lens)):
        ro, rl = oracle_decode(case, b)
        assert rel(go[b], ro) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, b
    assert_no_device_error()


def test_decode_page_table_is_bit_exact(path):
    """A shuffled page table gives bit-identical results to the identity table over the
    same token data (paging is pure indexing)."""
    lens = [200, 64, 1000]
    case = W.make_decode_case(DS, "bf16", lens, seed=54, spare_pages=0, shuffled=True)
    pool_id = np.empty_like(case["pool"])
    pt_id = np.full_like(case["page_table"], -1)
    nxt = 0
    for b, L in enumerate(lens):
        for p in range(W.pages_for(L, 64)):
            pool_id[nxt] = case["pool"][case["page_table"][b, p]]
            pt_id[b, p] = nxt
            nxt += 1
    cfg = cfg_of(DS, "bf16")
    q = dev(case["q_cat"])
    o1, l1 = M.mla_decode(cfg, cache_of(case), q)
    case2 = dict(case, pool=pool_id[:nxt], page_table=pt_id)
    o2, l2 = M.mla_decode(cfg, cache_of(case2), q)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_empty_sequence(path):
    case = W.make_decode_case(DS, "bf16", [0, 100], seed=55)
    cfg = cfg_of(DS, "bf16")
    o, l = M.mla_decode(cfg, cache_of(case), dev(case["q_cat"]))
    go, gl = host(o), host(l)
    assert np.all(go[0] == 0) and np.all(np.isneginf(gl[0]))
    ro, rl = oracle_decode(case, 1)
    assert rel(go[1], ro) <= TOL_OUT_BF16 and np.max(np.abs(gl[1] - rl)) <= TOL_LSE_BF16
    assert_no_device_error()


@pytest.mark.parametrize("lens", [[0, 300, 2049, 64], [0, 0], [0, 1, 0]])
def test_two_steps_share_buffers_with_empty_sequence(path, lens):
    """Two decode steps back to back on one stream and one set of buffers, as a serving loop
    runs them: step 1's mla_out reads o_lat while step 2's decode (which writes o_lat, and for
    the empty sequence stores zeros without any attention work) may already be starting under
    programmatic launch.  Both steps' outputs must be the oracle's."""
    case = W.make_decode_case(DS, "bf16", lens, seed=81, spare_pages=2)
    r = np.random.default_rng(82)
    q2 = W.normal(r, case["q_cat"].shape)
    q2[..., :DS.d_latent] *= np.float32(np.sqrt(DS.d_nope / DS.d_latent))
    q2 = W.quantise(q2, "bf16")
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    B = len(lens)
    w_uv = dev(case["w_uv"])
    o_lat = torch.empty((B, DS.n_heads, DS.d_latent), dtype=torch.bfloat16, device="cuda")
    lse1 = torch.empty((B, DS.n_heads), dtype=torch.float32, device="cuda")
    lse2 = torch.empty_like(lse1)
    o1 = torch.empty((B, DS.n_heads * DS.d_nope), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    o_lat.fill_(float("nan"))
    q1d, q2d = dev(case["q_cat"]), dev(q2)
    torch.cuda.synchronize()
    M.mla_decode(cfg, cache, q1d, o_lat=o_lat, lse=lse1)
    M.mla_out(cfg, o_lat, w_uv, o=o1)
    M.mla_decode(cfg, cache, q2d, o_lat=o_lat, lse=lse2)
    M.mla_out(cfg, o_lat, w_uv, o=o2)
    torch.cuda.synchronize()
    assert_no_device_error()
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    pool = f64(case["pool"])
    for q, o, l in ((f64(case["q_cat"]), host(o1), host(lse1)), (f64(q2), host(o2), host(lse2))):
        for b, L in enumerate(lens):
            if L == 0:
                assert np.all(o[b] == 0) and np.all(np.isneginf(l[b])), b
                continue
            rows = O.sequence_rows(pool, case["page_table"][b], L)
            ro_lat, rl = O.attention_latent(q[b], rows, DS.d_latent, sc)
            ro = O.up_project_output(ro_lat[None], f64(case["w_uv"]))[0]
            assert rel(o[b], ro) <= TOL_OUT_BF16, b
            assert np.max(np.abs(l[b] - rl)) <= TOL_LSE_BF16, b


def test_decode_bad_page_id_reports_bounds_error(path):
    case = W.make_decode_case(DS, "bf16", [100, 100], seed=56)
    pt = case["page_table"].copy()
    pt[1, 1] = case["num_pages"] + 5          # outside the pool: the kernel checks and skips it
    case = dict(case, page_table=pt)
    cfg = cfg_of(DS, "bf16")
    o, l = M.mla_decode(cfg, cache_of(case), dev(case["q_cat"]))
    assert M.mla_get_device_error() == 6   # MLA_ERR_DEVICE_BOUNDS
    assert M.mla_get_device_error() == 0   # cleared by the previous read
    # sequence 0 is unaffected
    ro, rl = oracle_decode(case, 0)
    assert rel(host(o)[0], ro) <= TOL_OUT_BF16


def test_device_error_word_reports_and_clears(path):
    case = W.make_decode_case(DS, "bf16", [100], seed=57)
    pt = case["page_table"].copy()
    pt[0, 0] = -3
    M.mla_decode(cfg_of(DS, "bf16"), cache_of(dict(case, page_table=pt)), dev(case["q_cat"]))
    assert M.mla_get_device_error() == 6   # MLA_ERR_DEVICE_BOUNDS
    assert M.mla_get_device_error() == 0


def test_workspace_too_small_is_rejected(path):
    case = W.make_decode_case(DS, "bf16", [10], seed=58)
    cfg = cfg_of(DS, "bf16")
    ws = torch.empty(M.mla_workspace_size(cfg) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MLAError) as e:
        M.mla_decode(cfg, cache_of(case), dev(case["q_cat"]), workspace=ws)
    assert e.value.status == 4


# ----------------------------------------------------------------------------------- prefill

@pytest.mark.parametrize("q_start,n_q", [(0, 300), (200, 100), (63, 2)])
def test_prefill_matches_oracle(path, q_start, n_q):
    T = q_start + n_q
    case = W.make_decode_case(DS, "bf16", [T], seed=61, spare_pages=4)
    r = np.random.default_rng(62)
    qc = W.normal(r, (n_q, DS.n_heads, DS.width))
    qc[..., :DS.d_latent] *= np.float32(np.sqrt(DS.d_nope / DS.d_latent))
    qc = W.quantise(qc, "bf16")
    cfg = cfg_of(DS, "bf16")
    o = Guarded((n_q, DS.n_heads, DS.d_latent), torch.bfloat16)
    lse = Guarded((n_q, DS.n_heads), torch.float32)
    M.mla_prefill(cfg, cache_of(case), 0, q_start, dev(qc), o_lat=o.t, lse=lse.t)
    torch.cuda.synchronize()
    o.check(); lse.check()
    go, gl = host(o.t), host(lse.t)
    rows = O.sequence_rows(f64(case["pool"]), case["page_table"][0], T)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    for i in sorted(set([0, 1, n_q - 1, n_q // 2] + list(range(0, n_q, 37)))):
        ro, rl = O.attention_latent(f64(qc)[i], rows[:q_start + i + 1], DS.d_latent, sc)
        assert rel(go[i], ro) <= TOL_OUT_BF16, i
        assert np.max(np.abs(gl[i] - rl)) <= TOL_LSE_BF16, i
    assert_no_device_error()


# ----------------------------------------------------------------------------------- chains

def test_tiny_f32_chain_matches_unabsorbed_oracle(path):
    """Tiny fp32 problem end to end: build the cache from x, absorb, decode, up-project;
    the oracle restores K and V and runs plain attention, then W_O."""
    case = W.make_tiny_case()
    s = case["shape"]
    cfg = cfg_of(s, "f32")
    cache = cache_of(case)
    M.mla_cache_append(cfg, cache, dev(case["x"], "f32"), dev(case["w_dkv"], "f32"),
                       dev(case["w_kr"], "f32"), i32(case["append_seq"]), i32(case["append_pos"]))
    x = case["x"].astype(np.float64)
    q_nope, q_rope = O.query_projection(x[-1:], case["w_q"], case["w_qr"], case["pos"], s.n_heads,
                                        s.rope_base)
    # the kernel receives the query projections (unrotated RoPE part) as inputs
    q_rope_raw = (x[-1:] @ case["w_qr"].astype(np.float64)).reshape(1, s.n_heads, s.d_rope)
    q_cat = M.mla_absorb_q(cfg, dev(q_nope.astype(np.float32), "f32"),
                           dev(q_rope_raw.astype(np.float32), "f32"), i32(case["pos"]),
                           dev(case["w_uk"], "f32"))
    o_lat, lse = M.mla_decode(cfg, cache, q_cat)
    o = M.mla_out(cfg, o_lat, dev(case["w_uv"], "f32"))
    torch.cuda.synchronize()
    c_kv, k_r = O.latent_kv(x, case["w_dkv"], case["w_kr"], case["append_pos"], s.rope_base)
    ro, rol, rl, _ = O.attention_unabsorbed(q_nope[0], q_rope[0], c_kv, k_r, case["w_uk"],
                                            case["w_uv"], O.default_scale(s.d_nope, s.d_rope))
    assert rel(host(o_lat)[0], rol) <= TOL_OUT_F32
    assert rel(host(o)[0], ro.reshape(-1)) <= TOL_OUT_F32
    assert np.max(np.abs(host(lse)[0] - rl)) <= TOL_LSE_F32
    out = O.output_projection(host(o).reshape(1, s.n_heads, s.d_nope), case["w_o"])
    ref_out = O.output_projection(ro[None], case["w_o"])
    assert rel(out, ref_out) <= TOL_OUT_F32


def test_bf16_chain_append_absorb_decode_out_proj(path):
    lens = [100, 64, 1, 700]
    case = W.make_decode_case(DS, "bf16", lens, seed=71, append=True)
    cfg = cfg_of(DS, "bf16")
    cache = cache_of(case)
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]),
                       i32(case["append_seq"]), i32(case["append_pos"]))
    q_cat = M.mla_absorb_q(cfg, dev(case["q_nope"]), dev(case["q_rope"]), i32(case["pos"]),
                           dev(case["w_uk"]))
    o_lat, lse = M.mla_decode(cfg, cache, q_cat)
    o = M.mla_out(cfg, o_lat, dev(case["w_uv"]))
    out = M.mla_out_proj(cfg, o, dev(case["w_o"]))
    torch.cuda.synchronize()
    assert_no_device_error()
    go, gl, gol, gout = host(o), host(lse), host(o_lat), host(out)
    gq, gpool = host(q_cat), host(cache.pool)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    x = f64(case["x"])
    c_new, k_new = O.latent_kv(x, f64(case["w_dkv"]), f64(case["w_kr"]), case["append_pos"], DS.rope_base)
    pool = f64(case["pool"])
    for b, L0 in enumerate(lens):
        rows = O.sequence_rows(pool, case["page_table"][b], L0)
        c_kv = np.concatenate([rows[:, :DS.d_latent], c_new[b:b + 1]])
        k_r = np.concatenate([rows[:, DS.d_latent:], k_new[b:b + 1]])
        q_r = O.rope_rotate(f64(case["q_rope"])[b], case["pos"][b], DS.rope_base)
        ro, rol, rl, _ = O.attention_unabsorbed(f64(case["q_nope"])[b], q_r, c_kv, k_r,
                                                f64(case["w_uk"]), f64(case["w_uv"]), sc)
        assert rel(gol[b], rol) <= TOL_OUT_BF16, b
        assert rel(go[b], ro.reshape(-1)) <= TOL_OUT_BF16, b
        # the whole layer output, the un-absorbed chain through W_O
        assert rel(gout[b], O.output_projection(ro.reshape(1, -1), f64(case["w_o"]))[0]) <= TOL_OUT_BF16, b
        # q_cat against the oracle's absorption, then attention checked at the stated tolerances
        # against the oracle evaluated on the device's own bf16 q_cat and cache rows (the path
        # stores both in bf16 before attention reads them)
        q_ref = O.absorb_query(f64(case["q_nope"])[b:b + 1], f64(case["q_rope"])[b:b + 1],
                               case["pos"][b:b + 1], f64(case["w_uk"]), DS.rope_base)[0]
        assert rel(gq[b], q_ref) <= TOL_OUT_BF16, b
        rows_dev = O.sequence_rows(gpool, case["page_table"][b], L0 + 1)
        ro_dev, rl_dev = O.attention_latent(gq[b], rows_dev, DS.d_latent, sc)
        assert rel(gol[b], ro_dev) <= TOL_OUT_BF16, b
        assert np.max(np.abs(gl[b] - rl_dev)) <= TOL_LSE_BF16, b
        # against the un-absorbed chain the lse may move by the first-order effect of those two
        # bf16 roundings (a diagnostic bound, looser than the tolerance above)
        keys = np.concatenate([c_kv, k_r], axis=1)
        bound = lse_rounding_bound(q_ref, keys, appended=[L0], scale=sc)
        assert np.all(np.abs(gl[b] - rl) <= TOL_LSE_BF16 + bound), b
