"""GPU parity of the MX-encoded latent cache (MXFP8 / MXFP4 blocks of 32 with E8M0 scales).

Decode over an MX cache is compared with the oracle's attention on the dequantised rows (the
oracle's MX decoder, pinned in the CPU suite); the append's encoding is compared with the
oracle's MX encoder, bit for bit where the fp32 row is exact, and by the rounding bound where
the two sides' fp32 sums of the row may differ in the last place.
"""
import numpy as np
import pytest
import torch

import mla_workloads as W
import oracle.mla_oracle as O
import mla_latent_kv_79_b300 as M
from mla_latent_kv_79_b300 import _lib

from tests.gpu_util import TOL_LSE_BF16, TOL_OUT_BF16, Guarded, cfg_of, dev, host, i32, rel

pytestmark = pytest.mark.gpu

DS = W.DEEPSEEK_V2
ELEM = {"mxfp8": "e4m3", "mxfp4": "e2m1"}
FMT = {"mxfp8": _lib.MLA_KV_MXFP8, "mxfp4": _lib.MLA_KV_MXFP4}


@pytest.fixture(scope="module", autouse=True)
def _ready():
    from mla_latent_kv_79_b300 import build
    build.build()
    M.lib()
    yield


@pytest.fixture(params=["tcgen05", "simt"])
def path(request):
    old = M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, 1 if request.param == "simt" else 0)
    assert M.mla_get_device_error() == 0
    yield request.param
    M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, old)
    assert M.mla_get_device_error() == 0


def mx_cache(case):
    return M.PagedCache(torch.from_numpy(case["codes"]).cuda(), i32(case["page_table"]), i32(case["seq_lens"]),
                        FMT[case["kv"]], torch.from_numpy(case["scales"]).cuda())


def dequant_rows(codes_pool, scales_pool, pt_row, length, kv):
    """Dequantised rows [length, W] of one sequence (the oracle's MX decoder)."""
    codes = O.sequence_rows(codes_pool, pt_row, length).astype(np.int64)
    sc = O.sequence_rows(scales_pool, pt_row, length).astype(np.int64)
    if kv == "mxfp4":
        codes = O.mx_unpack_e2m1(codes)
    return O.mx_decode_rows(codes, sc, ELEM[kv])


def check_decode(case, o, lse, seqs=None):
    go, gl = host(o), host(lse)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    qc = W.to_f64(case["q_cat"], "bf16")
    for b in (range(len(case["seq_lens"])) if seqs is None else seqs):
        L = int(case["seq_lens"][b])
        if L == 0:
            assert np.all(go[b] == 0) and np.all(np.isneginf(gl[b])), b
            continue
        rows = dequant_rows(case["codes"], case["scales"], case["page_table"][b], L, case["kv"])
        ro, rl = O.attention_latent(qc[b], rows, DS.d_latent, sc)
        assert np.all(np.isfinite(go[b])), b
        assert rel(go[b], ro) <= TOL_OUT_BF16, (b, rel(go[b], ro))
        assert np.max(np.abs(gl[b] - rl)) <= TOL_LSE_BF16, (b, np.max(np.abs(gl[b] - rl)))


# ----------------------------------------------------------------------------------- decode

@pytest.mark.parametrize("kv", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("units", [0, 1, 3])
def test_mx_decode_matches_oracle(path, kv, units):
    """Ragged lengths (one token, page edges, several pages, an empty sequence) over a shuffled
    page table; every slot no token owns holds NaN codes and NaN scale bytes."""
    lens = [1, 63, 64, 65, 300, 1000, 2049, 130, 0]
    case = W.make_mx_decode_case(DS, kv, lens, seed=70 + units)
    cfg = cfg_of(DS, "bf16")
    old = M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, units)
    try:
        o = Guarded((len(lens), DS.n_heads, DS.d_latent), torch.bfloat16)
        lse = Guarded((len(lens), DS.n_heads), torch.float32)
        M.mla_decode(cfg, mx_cache(case), dev(case["q_cat"]), o_lat=o.t, lse=lse.t)
        torch.cuda.synchronize()
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old)
    assert M.mla_get_device_error() == 0
    assert M.mla_last_attention_path() == (2 if path == "tcgen05" else 1)
    o.check()
    lse.check()
    check_decode(case, o.t, lse.t)


@pytest.mark.parametrize("kv", ["mxfp8", "mxfp4"])
def test_mx_decode_tcgen05_equals_simt(kv):
    """The two kernels read the same dequantised values: their outputs agree far inside the
    oracle tolerance (bf16 output rounding and summation order only)."""
    case = W.make_mx_decode_case(DS, kv, [777, 4096, 5], seed=79)
    cfg = cfg_of(DS, "bf16")
    outs = []
    for simt in (0, 1):
        old = M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, simt)
        try:
            o, lse = M.mla_decode(cfg, mx_cache(case), dev(case["q_cat"]))
            torch.cuda.synchronize()
        finally:
            M.mla_set_tuning(_lib.MLA_TUNE_FORCE_SIMT, old)
        outs.append((host(o), host(lse)))
    assert rel(outs[0][0], outs[1][0]) <= 1e-2
    assert np.max(np.abs(outs[0][1] - outs[1][1])) <= 2e-4


@pytest.mark.parametrize("kv", ["mxfp8", "mxfp4"])
def test_mx_prefill_matches_oracle(path, kv):
    """Causal queries over an MX cache: query i at position q_start + i sees t <= q_start + i."""
    T, q0, nq = 700, 500, 200
    case = W.make_mx_decode_case(DS, kv, [T], seed=81)
    cfg = cfg_of(DS, "bf16")
    q = W.normal(np.random.default_rng(82), (nq, DS.n_heads, DS.width))
    q[..., :DS.d_latent] *= np.float32(np.sqrt(DS.d_nope / DS.d_latent))
    qb = W.quantise(q, "bf16")
    o, lse = M.mla_prefill(cfg, mx_cache(case), 0, q0, dev(qb))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    go, gl = host(o), host(lse)
    rows = dequant_rows(case["codes"], case["scales"], case["page_table"][0], T, kv)
    sc = O.default_scale(DS.d_nope, DS.d_rope)
    qf = W.to_f64(qb, "bf16")
    for i in (0, 1, 13, 99, 100, 199):
        ro, rl = O.attention_latent(qf[i], rows[:q0 + i + 1], DS.d_latent, sc)
        assert rel(go[i], ro) <= TOL_OUT_BF16, i
        assert np.max(np.abs(gl[i] - rl)) <= TOL_LSE_BF16, i


# ----------------------------------------------------------------------------------- append

def _empty_mx(num_pages, kv):
    row_bytes = DS.width if kv == "mxfp8" else DS.width // 2
    codes = np.full((num_pages, DS.page_size, row_bytes), 0xA5, np.uint8)
    scales = np.full((num_pages, DS.page_size, DS.width // 32), 0x5A, np.uint8)
    return codes, scales


def _zero_sign_free(codes, kv):
    c = np.asarray(codes, dtype=np.int64)
    if kv == "mxfp8":
        return np.where(c == 0x80, 0, c)
    lo, hi = c & 0xF, c >> 4
    return np.where(lo == 8, 0, lo) | (np.where(hi == 8, 0, hi) << 4)


def _encode_oracle(rows, kv):
    codes, sc = O.mx_encode_rows(rows, ELEM[kv])
    if kv == "mxfp4":
        codes = O.mx_pack_e2m1(codes.reshape(-1)).reshape(rows.shape[0], -1)
    return codes.astype(np.uint8), sc.astype(np.uint8)


@pytest.mark.parametrize("kv", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("ksplit", [0, 1])
def test_mx_append_integer_inputs_are_bit_exact(kv, ksplit):
    """Small-integer x and power-of-two weights at position 0 make every fp32 sum exact, so the
    stored codes and scale bytes equal the oracle's encoding of the exact row bit for bit.
    ksplit 0 lets 48 tokens split K over a cluster (the decode-step path); 1 forces one CTA per
    tile (the many-token path)."""
    s = W.replace_shape(DS, d_model=256)
    r = np.random.default_rng(34)
    n = 48
    x = np.zeros((n, s.d_model), np.float32)
    for t in range(n):
        idx = r.choice(s.d_model, size=3, replace=False)
        x[t, idx] = r.choice([-2.0, -1.0, 1.0, 2.0], size=3)
    wd = (2.0 ** -r.integers(0, 4, size=(s.d_model, s.d_latent)) * r.choice([-1, 1], size=(s.d_model, s.d_latent))).astype(np.float32)
    wk = (2.0 ** -r.integers(0, 4, size=(s.d_model, s.d_rope)) * r.choice([-1, 1], size=(s.d_model, s.d_rope))).astype(np.float32)
    pt = np.arange(n, dtype=np.int32).reshape(n, 1)
    codes0, scales0 = _empty_mx(n, kv)
    cache = M.PagedCache(torch.from_numpy(codes0).cuda(), i32(pt), i32(np.ones(n)), FMT[kv],
                         torch.from_numpy(scales0).cuda())
    old = M.mla_set_tuning(_lib.MLA_TUNE_GEMM_KSPLIT, ksplit)
    try:
        M.mla_cache_append(cfg_of(s, "bf16"), cache, dev(W.quantise(x, "bf16")), dev(W.quantise(wd, "bf16")),
                           dev(W.quantise(wk, "bf16")), i32(np.arange(n)), i32(np.zeros(n)))
        torch.cuda.synchronize()
    finally:
        M.mla_set_tuning(_lib.MLA_TUNE_GEMM_KSPLIT, old)
    assert M.mla_get_device_error() == 0
    c_ref, k_ref = O.latent_kv(x.astype(np.float64), wd.astype(np.float64), wk.astype(np.float64),
                               np.zeros(n), s.rope_base)
    rows = np.concatenate([c_ref, k_ref], axis=1)
    assert np.array_equal(rows.astype(np.float32).astype(np.float64), rows), "fixture not exact in fp32"
    want_c, want_s = _encode_oracle(rows, kv)
    got_c, got_s = cache.pool.cpu().numpy(), cache.kv_scales.cpu().numpy()
    assert np.array_equal(got_s[:, 0], want_s)
    # an exact zero may carry either sign bit (the order of an exact cancellation is the
    # kernel's): compare codes with negative zero read as zero
    assert np.array_equal(_zero_sign_free(got_c[:, 0], kv), _zero_sign_free(want_c, kv))
    # every other slot of every page is untouched
    assert np.array_equal(got_c[:, 1:], codes0[:, 1:]) and np.array_equal(got_s[:, 1:], scales0[:, 1:])


@pytest.mark.parametrize("kv", ["mxfp8", "mxfp4"])
def test_mx_append_then_decode_matches_oracle(kv):
    """One new token per sequence appended into an MX cache (random bf16 x and weights, long
    positions), then decode.  The stored blocks agree with the oracle's encoding of its own
    row wherever the row's fp32 value is away from a rounding boundary, and always lie within
    the format's rounding bound of it; the decode matches the oracle on the stored rows."""
    lens = [5, 64, 1000, 4095, 0, 130]
    case = W.make_mx_decode_case(DS, kv, lens, seed=91, append=True)
    cfg = cfg_of(DS, "bf16")
    cache = mx_cache(case)
    codes_before, scales_before = case["codes"].copy(), case["scales"].copy()
    M.mla_cache_append(cfg, cache, dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"]), i32(case["append_seq"]),
                       i32(case["append_pos"]))
    o, lse = M.mla_decode(cfg, cache, dev(case["q_cat"]))
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0
    got_c, got_s = cache.pool.cpu().numpy(), cache.kv_scales.cpu().numpy()
    pt = case["page_table"]
    B = len(lens)
    rows_at = [(int(pt[b, lens[b] // 64]), lens[b] % 64) for b in range(B)]
    # only the appended slots changed
    mask = np.zeros(got_c.shape[:2], bool)
    for p, sl in rows_at:
        mask[p, sl] = True
    assert np.array_equal(got_c[~mask], codes_before[~mask]) and np.array_equal(got_s[~mask], scales_before[~mask])
    # the encoding of each appended row against the oracle's row
    c_ref, k_ref = O.latent_kv(W.to_f64(case["x"], "bf16"), W.to_f64(case["w_dkv"], "bf16"),
                               W.to_f64(case["w_kr"], "bf16"), case["append_pos"], DS.rope_base)
    ref = np.concatenate([c_ref, k_ref], axis=1)
    gc = np.stack([got_c[p, sl] for p, sl in rows_at]).astype(np.int64)
    gs = np.stack([got_s[p, sl] for p, sl in rows_at]).astype(np.int64)
    codes_u = O.mx_unpack_e2m1(gc) if kv == "mxfp4" else gc
    deq = O.mx_decode_rows(codes_u, gs, ELEM[kv])
    f = O.MX_FORMATS[ELEM[kv]]
    e = np.repeat(gs - 127, 32, axis=-1)
    a = np.abs(np.ldexp(ref, -e))
    half_step = np.ldexp(2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** (1 - f["bias"])))) - f["mbits"] - 1), e)
    # slack: the two sides' fp32 / f64 sums of a 5120-term row differ by ~1e-7 of its scale
    slack = 1e-5 * np.max(np.abs(ref), axis=1, keepdims=True)
    assert np.all(np.abs(deq - ref) <= half_step + slack)
    want_c, want_s = O.mx_encode_rows(ref.astype(np.float32).astype(np.float64), ELEM[kv])
    assert np.mean(gs == want_s) >= 0.99
    assert np.mean(codes_u == want_c) >= 0.99
    # decode over the stored cache
    final = dict(case, codes=got_c, scales=got_s)
    check_decode(final, o, lse)
