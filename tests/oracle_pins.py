"""Pins for the CPU oracle: checks against facts fixed by the pages or by mathematics.

Every pin takes the oracle namespace `O` as an argument so the mutation tests can run the
same pins against copies of the oracle with one planted mistake each.  A pin raises
AssertionError when it fails.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _rand_problem(seed, n_h=3, d_h=5, d_c=7, d_r=4, L=6):
    r = np.random.default_rng(seed)
    return dict(
        q_nope=r.standard_normal((n_h, d_h)), q_rope_raw=r.standard_normal((n_h, d_r)),
        c_kv=r.standard_normal((L, d_c)), k_rope=r.standard_normal((L, d_r)),
        w_uk=r.standard_normal((d_c, n_h * d_h)) / math.sqrt(d_c),
        w_uv=r.standard_normal((d_c, n_h * d_h)) / math.sqrt(d_c),
        n_h=n_h, d_h=d_h, d_c=d_c, d_r=d_r, L=L)


# ------------------------------------------------------------------------------ pages' integers

def pin_cache_sizes_from_pages(O):
    """The operator-notes page's cache table: 32768 numbers/token for MHA at n_h=d_h=128,
    512 for MLA at d_c=512, ~32.77 B vs ~0.51 B numbers at 1M context, about 1/64 (~98.4 %)."""
    g = json.load(open(os.path.join(GOLDEN, "cache_sizes.json")))
    mha = O.mha_numbers_per_token(g["mha"]["n_h"], g["mha"]["d_h"])
    mla = O.mla_numbers_per_token(g["mla"]["d_c"])
    assert mha == g["mha"]["numbers_per_token"]
    assert mla == g["mla"]["numbers_per_token"]
    assert round(1_000_000 * mha / 1e9, 2) == g["mha"]["context_1m_billion"]
    assert round(1_000_000 * mla / 1e9, 2) == g["mla"]["context_1m_billion"]
    assert mha // mla == g["ratio_denominator"] and mha % mla == 0
    assert round(100.0 * (1.0 - mla / mha), 1) == g["reduction_percent"]
    # with the decoupled RoPE key of width 64 the cached row is 576 numbers
    assert O.mla_numbers_per_token(512, 64) == 576


# ------------------------------------------------------------------------------ RoPE

def pin_rope_closed_form(O):
    """Textbook 2x2 rotation: pair i turns by pos * base^(-2i/d)."""
    # d=2: theta_0 = 1, so position p is a rotation by p radians.
    for p in (0, 1, 2.5, 7):
        got = O.rope_rotate(np.array([1.0, 0.0]), p, 10000.0)
        assert np.allclose(got, [math.cos(p), math.sin(p)], atol=1e-15)
        got = O.rope_rotate(np.array([0.0, 1.0]), p, 10000.0)
        assert np.allclose(got, [-math.sin(p), math.cos(p)], atol=1e-15)
    # d=4, base 100: theta_1 = 100^(-1/2) = 0.1; only pair 1 is populated.
    got = O.rope_rotate(np.array([0.0, 0.0, 1.0, 0.0]), 3, 100.0)
    assert np.allclose(got, [0, 0, math.cos(0.3), math.sin(0.3)], atol=1e-15)
    # interleaved pairs: the odd element of pair 0 only mixes with element 0
    got = O.rope_rotate(np.array([0.0, 1.0, 0.0, 0.0]), 1, 100.0)
    assert np.allclose(got, [-math.sin(1.0), math.cos(1.0), 0, 0], atol=1e-15)


def pin_rope_invariants(O):
    r = np.random.default_rng(11)
    v = r.standard_normal((5, 64))
    assert np.array_equal(O.rope_rotate(v, 0, 10000.0), v)           # position 0 = identity
    pos = r.integers(0, 200000, size=5)
    w = O.rope_rotate(v, pos, 10000.0)
    assert np.allclose(np.linalg.norm(w, axis=1), np.linalg.norm(v, axis=1), rtol=1e-12)
    # composition R(a) R(b) = R(a + b)
    assert np.allclose(O.rope_rotate(O.rope_rotate(v, 17, 10000.0), 40, 10000.0),
                       O.rope_rotate(v, 57, 10000.0), atol=1e-11)
    # relative position: <R_m q, R_n k> depends on m - n only
    q, k = r.standard_normal(64), r.standard_normal(64)
    a = O.rope_rotate(q, 1000, 10000.0) @ O.rope_rotate(k, 990, 10000.0)
    b = O.rope_rotate(q, 10, 10000.0) @ k
    assert abs(a - b) < 1e-10


# ------------------------------------------------------------------------------ projections

def pin_latent_kv_bruteforce(O):
    """c_kv = x W_DKV (nothing rotated) and k_rope = RoPE(x W_KR) by explicit loops; with
    d_rope = 2 the rotation angle is the position itself."""
    r = np.random.default_rng(12)
    N, dm, dc = 3, 5, 4
    x, wd, wk = r.standard_normal((N, dm)), r.standard_normal((dm, dc)), r.standard_normal((dm, 2))
    pos = np.array([0, 3, 11])
    c, k = O.latent_kv(x, wd, wk, pos, 10000.0)
    for n in range(N):
        for j in range(dc):
            assert abs(c[n, j] - sum(x[n, i] * wd[i, j] for i in range(dm))) < 1e-12
        a = sum(x[n, i] * wk[i, 0] for i in range(dm))
        b = sum(x[n, i] * wk[i, 1] for i in range(dm))
        cs, sn = math.cos(pos[n]), math.sin(pos[n])
        assert abs(k[n, 0] - (a * cs - b * sn)) < 1e-12
        assert abs(k[n, 1] - (a * sn + b * cs)) < 1e-12


def pin_integer_append_exact(O):
    """Small-integer x and power-of-two weights at position 0: every product and sum is
    exact, so the result equals the integer arithmetic exactly."""
    x = np.array([[1.0, -2.0, 3.0, 0.0]])
    wd = np.array([[0.5, 1.0], [0.25, -1.0], [2.0, 0.0], [8.0, 4.0]])
    wk = np.array([[1.0, 0.0], [0.0, 1.0], [0.5, 0.5], [0.0, 0.0]])
    c, k = O.latent_kv(x, wd, wk, np.array([0]), 10000.0)
    assert np.array_equal(c, [[0.5 - 0.5 + 6.0, 1.0 + 2.0 + 0.0]])
    assert np.array_equal(k, [[1.0 + 1.5, -2.0 + 1.5]])


def pin_query_projection_bruteforce(O):
    r = np.random.default_rng(13)
    n_h, dh, dm = 2, 3, 4
    x = r.standard_normal((2, dm))
    wq, wqr = r.standard_normal((dm, n_h * dh)), r.standard_normal((dm, n_h * 2))
    qn, qr = O.query_projection(x, wq, wqr, np.array([0, 2]), n_h, 10000.0)
    for n, p in enumerate((0, 2)):
        for h in range(n_h):
            for j in range(dh):
                assert abs(qn[n, h, j] - sum(x[n, i] * wq[i, h * dh + j] for i in range(dm))) < 1e-12
            a = sum(x[n, i] * wqr[i, h * 2] for i in range(dm))
            b = sum(x[n, i] * wqr[i, h * 2 + 1] for i in range(dm))
            assert abs(qr[n, h, 0] - (a * math.cos(p) - b * math.sin(p))) < 1e-12
            assert abs(qr[n, h, 1] - (a * math.sin(p) + b * math.cos(p))) < 1e-12


def pin_compressed_query(O):
    """c_q = x W_DQ by brute force; the compressed query equals the direct one with
    W_Q = W_DQ W_UQ and W_QR = W_DQ W_QR' (associativity); with W_DQ = I it is the direct one."""
    r = np.random.default_rng(17)
    n_h, dh, dr, dm, dcq = 2, 3, 2, 5, 4
    x = r.standard_normal((3, dm))
    wdq = r.standard_normal((dm, dcq))
    wuq, wqr = r.standard_normal((dcq, n_h * dh)), r.standard_normal((dcq, n_h * dr))
    cq = O.query_latent(x, wdq)
    for n in range(3):
        for k in range(dcq):
            assert abs(cq[n, k] - sum(x[n, i] * wdq[i, k] for i in range(dm))) < 1e-12
    pos = np.array([0, 5, 1000])
    qn, qr = O.query_projection_compressed(x, wdq, wuq, wqr, pos, n_h, 10000.0)
    qn2, qr2 = O.query_projection(x, wdq @ wuq, wdq @ wqr, pos, n_h, 10000.0)
    assert np.max(np.abs(qn - qn2)) < 1e-12 and np.max(np.abs(qr - qr2)) < 1e-12
    qn3, qr3 = O.query_projection_compressed(cq, np.eye(dcq), wuq, wqr, pos, n_h, 10000.0)
    assert np.max(np.abs(qn3 - qn)) < 1e-12 and np.max(np.abs(qr3 - qr)) < 1e-12
    # the RoPE query comes from c_q (not from x): W_QR has d_cq rows
    assert qr.shape == (3, n_h, dr)


def pin_absorb_uq_uk(O):
    """Brute-force entries of W_UQ_h W_UK_h^T, and c_q (W_UQ_h W_UK_h^T) == (c_q W_UQ_h) W_UK_h^T,
    the absorbed query's latent part (associativity, to 1e-10)."""
    r = np.random.default_rng(19)
    n_h, dh, dc, dcq = 3, 4, 5, 6
    wuq, wuk = r.standard_normal((dcq, n_h * dh)), r.standard_normal((dc, n_h * dh))
    w = O.absorb_uq_uk(wuq, wuk, n_h)
    assert w.shape == (dcq, n_h * dc)
    for h in range(n_h):
        for k in range(dcq):
            for c in range(dc):
                ref = sum(wuq[k, h * dh + j] * wuk[c, h * dh + j] for j in range(dh))
                assert abs(w[k, h * dc + c] - ref) < 1e-12
    cq = r.standard_normal((2, dcq))
    qn = (cq @ wuq).reshape(2, n_h, dh)
    qcat = O.absorb_query(qn, np.zeros((2, n_h, 2)), np.zeros(2), wuk, 10000.0)
    assert np.max(np.abs((cq @ w).reshape(2, n_h, dc) - qcat[..., :dc])) < 1e-10


# ------------------------------------------------------------------------------ attention

def pin_attention_bruteforce(O):
    """Un-absorbed attention with explicit loops over heads, tokens and dims (math.exp)."""
    P = _rand_problem(14, n_h=2, d_h=2, d_c=3, d_r=2, L=3)
    n_h, d_h, d_c, d_r, L = P["n_h"], P["d_h"], P["d_c"], P["d_r"], P["L"]
    scale = 1.0 / math.sqrt(d_h + d_r)
    qn, qr, c, kr, wuk, wuv = (P["q_nope"], P["q_rope_raw"], P["c_kv"], P["k_rope"],
                               P["w_uk"], P["w_uv"])
    o, o_lat, lse, _ = O.attention_unabsorbed(qn, qr, c, kr, wuk, wuv, scale)
    for h in range(n_h):
        s = []
        for t in range(L):
            dot = 0.0
            for j in range(d_h):
                k = sum(c[t, cc] * wuk[cc, h * d_h + j] for cc in range(d_c))
                dot += qn[h, j] * k
            dot += sum(qr[h, i] * kr[t, i] for i in range(d_r))
            s.append(dot * scale)
        z = sum(math.exp(v) for v in s)
        assert abs(lse[h] - math.log(z)) < 1e-12
        p = [math.exp(v) / z for v in s]
        for j in range(d_h):
            ref = sum(p[t] * sum(c[t, cc] * wuv[cc, h * d_h + j] for cc in range(d_c))
                      for t in range(L))
            assert abs(o[h, j] - ref) < 1e-12
        for cc in range(d_c):
            assert abs(o_lat[h, cc] - sum(p[t] * c[t, cc] for t in range(L))) < 1e-12


def pin_attention_closed_forms(O):
    P = _rand_problem(15)
    n_h, d_h, d_c, d_r, L = P["n_h"], P["d_h"], P["d_c"], P["d_r"], P["L"]
    scale = 1.0 / math.sqrt(d_h + d_r)
    wuk, wuv = P["w_uk"], P["w_uv"]
    # one token: p = 1, o = V[0], o_lat = c_kv[0]
    o, o_lat, lse, _ = O.attention_unabsorbed(P["q_nope"], P["q_rope_raw"], P["c_kv"][:1],
                                              P["k_rope"][:1], wuk, wuv, scale)
    V0 = (P["c_kv"][:1] @ wuv).reshape(n_h, d_h)
    assert _rel(o, V0) < 1e-13 and _rel(o_lat, np.repeat(P["c_kv"][:1], n_h, 0)) < 1e-13
    # zero query: uniform weights, lse = ln L, o_lat = mean of the latents
    o, o_lat, lse, _ = O.attention_unabsorbed(np.zeros((n_h, d_h)), np.zeros((n_h, d_r)),
                                              P["c_kv"], P["k_rope"], wuk, wuv, scale)
    assert np.allclose(lse, math.log(L), atol=1e-14)
    assert _rel(o_lat, np.repeat(P["c_kv"].mean(0, keepdims=True), n_h, 0)) < 1e-13
    # all rows equal with a known score: c_kv = e0, k_rope = e0, W_UK[0, h*d_h] = a,
    # q_nope[h] = b e0, q_rope[h] = g e0  ->  s = (a b + g) * scale, lse = s + ln L
    a, b, g = 1.5, -0.75, 2.0
    c = np.zeros((L, d_c)); c[:, 0] = 1.0
    kr = np.zeros((L, d_r)); kr[:, 0] = 1.0
    wk = np.zeros((d_c, n_h * d_h)); wk[0, ::d_h] = a
    qn = np.zeros((n_h, d_h)); qn[:, 0] = b
    qr = np.zeros((n_h, d_r)); qr[:, 0] = g
    _, o_lat, lse, _ = O.attention_unabsorbed(qn, qr, c, kr, wk, wuv, scale)
    assert np.allclose(lse, (a * b + g) * scale + math.log(L), atol=1e-14)
    assert np.allclose(o_lat, np.repeat(c[:1], n_h, 0), atol=1e-15)
    # two tokens with scores differing by d: p0 = 1 / (1 + e^{-d})
    c2 = np.zeros((2, d_c)); c2[0, 0] = 1.0; c2[1, 1] = 1.0
    kr2 = np.zeros((2, d_r))
    wk2 = np.zeros((d_c, n_h * d_h)); wk2[0, ::d_h] = 1.0
    qn2 = np.zeros((n_h, d_h)); qn2[:, 0] = 3.0 / scale
    _, o_lat, lse, _ = O.attention_unabsorbed(qn2, np.zeros((n_h, d_r)), c2, kr2, wk2, wuv, scale)
    p0 = 1.0 / (1.0 + math.exp(-3.0))
    assert np.allclose(o_lat[:, 0], p0, atol=1e-14) and np.allclose(o_lat[:, 1], 1 - p0, atol=1e-14)
    assert np.allclose(lse, math.log(math.exp(3.0) + 1.0), atol=1e-14)


def pin_default_scale(O):
    """The score scale 1/sqrt(d_h + d_r): the score is a dot product over the d_h nope and the
    d_r RoPE dimensions (the decoupled key of the glossary), so the operator notes' division
    by sqrt(d) of the dot product's width takes d = d_h + d_r."""
    assert abs(O.default_scale(128, 64) - 1.0 / math.sqrt(192.0)) < 1e-17
    assert abs(O.default_scale(16, 8) - 1.0 / math.sqrt(24.0)) < 1e-17
    # tiny case: raw dot products 3*sqrt(d_h + d_r) and 0 are scaled to scores 3 and 0, so the
    # first token's weight is 1 / (1 + e^-3) and lse = ln(e^3 + 1)
    d_h, d_r, d_c = 16, 8, 4
    rows = np.zeros((2, d_c + d_r))
    rows[0, 0] = 1.0
    rows[1, 1] = 1.0
    q = np.zeros((1, d_c + d_r))
    q[0, 0] = 3.0 * math.sqrt(d_h + d_r)
    o_lat, lse = O.attention_latent(q, rows, d_c, O.default_scale(d_h, d_r))
    p0 = 1.0 / (1.0 + math.exp(-3.0))
    assert abs(o_lat[0, 0] - p0) < 1e-14 and abs(o_lat[0, 1] - (1.0 - p0)) < 1e-14
    assert abs(lse[0] - math.log(math.exp(3.0) + 1.0)) < 1e-14


def pin_softmax_properties(O):
    r = np.random.default_rng(16)
    s = r.standard_normal((4, 9)) * 5
    p, lse = O.softmax_lse(s)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)
    p2, lse2 = O.softmax_lse(s + 123.0)
    assert np.allclose(p2, p, atol=1e-14) and np.allclose(lse2, lse + 123.0, atol=1e-12)
    s[:, 3] = -np.inf
    p3, _ = O.softmax_lse(s)
    assert np.all(p3[:, 3] == 0.0)
    assert np.allclose(np.log(np.exp(s[0, np.isfinite(s[0])]).sum()), O.softmax_lse(s)[1][0])


def pin_absorbed_equals_unabsorbed(O):
    """Associativity (rmj dispatch; glossary absorption paragraph): folding W_UK into the
    query and W_UV into the output gives the same attention as restoring K and V."""
    for seed, kw in ((21, {}), (22, dict(n_h=4, d_h=8, d_c=16, d_r=4, L=37)),
                     (23, dict(n_h=1, d_h=3, d_c=2, d_r=2, L=1))):
        P = _rand_problem(seed, **kw)
        d_h, d_c, d_r = P["d_h"], P["d_c"], P["d_r"]
        scale = 1.0 / math.sqrt(d_h + d_r)
        pos = 5
        qr_rot = O.rope_rotate(P["q_rope_raw"], pos, 10000.0)
        o, o_lat, lse, _ = O.attention_unabsorbed(P["q_nope"], qr_rot, P["c_kv"], P["k_rope"],
                                                  P["w_uk"], P["w_uv"], scale)
        q_cat = O.absorb_query(P["q_nope"][None], P["q_rope_raw"][None], np.array([pos]),
                               P["w_uk"], 10000.0)[0]
        rows = np.concatenate([P["c_kv"], P["k_rope"]], axis=1)
        o_lat2, lse2 = O.attention_latent(q_cat, rows, d_c, scale)
        o2 = O.up_project_output(o_lat2[None], P["w_uv"])[0]
        assert _rel(o_lat2, o_lat) < 1e-10
        assert np.max(np.abs(lse2 - lse)) < 1e-10
        assert _rel(o2, o.reshape(-1)) < 1e-10


def pin_causal_prefill(O):
    """Row i of the masked [T, T] prefill equals single-query attention over tokens 0..i."""
    r = np.random.default_rng(24)
    T, n_h, d_h, d_c, d_r = 7, 2, 3, 5, 4
    qn, qr = r.standard_normal((T, n_h, d_h)), r.standard_normal((T, n_h, d_r))
    c, kr = r.standard_normal((T, d_c)), r.standard_normal((T, d_r))
    wuk, wuv = r.standard_normal((d_c, n_h * d_h)), r.standard_normal((d_c, n_h * d_h))
    scale = 1.0 / math.sqrt(d_h + d_r)
    o, o_lat, lse = O.causal_prefill_unabsorbed(qn, qr, c, kr, wuk, wuv, scale)
    for i in range(T):
        oi, oli, lsei, _ = O.attention_unabsorbed(qn[i], qr[i], c[:i + 1], kr[:i + 1], wuk, wuv,
                                                  scale)
        assert _rel(o[i], oi) < 1e-12 and _rel(o_lat[i], oli) < 1e-12
        assert np.max(np.abs(lse[i] - lsei)) < 1e-12
    # query 0 sees only token 0: o_lat = c_kv[0]
    assert _rel(o_lat[0], np.repeat(c[:1], n_h, 0)) < 1e-13


def pin_output_projection_bruteforce(O):
    r = np.random.default_rng(25)
    o = r.standard_normal((2, 3, 2))          # [N, n_h, d_h]
    wo = r.standard_normal((6, 4))
    out = O.output_projection(o, wo)
    for n in range(2):
        for j in range(4):
            ref = sum(o[n, h, d] * wo[h * 2 + d, j] for h in range(3) for d in range(2))
            assert abs(out[n, j] - ref) < 1e-12
    # head slice: o_lat @ W_UV_h by loops
    ol = r.standard_normal((1, 2, 3))
    wuv = r.standard_normal((3, 2 * 4))
    up = O.up_project_output(ol, wuv)
    for h in range(2):
        for j in range(4):
            assert abs(up[0, h * 4 + j] - sum(ol[0, h, c] * wuv[c, h * 4 + j] for c in range(3))) < 1e-12


def pin_paged_gather(O):
    """Token t of a sequence lives in page table[t // page_size], slot t % page_size."""
    pool = np.arange(5 * 4 * 2, dtype=np.float64).reshape(5, 4, 2)
    rows = O.sequence_rows(pool, np.array([3, 0, 4]), 10)
    for t in range(10):
        assert np.array_equal(rows[t], pool[[3, 0, 4][t // 4], t % 4])


# ------------------------------------------------------------------------------ MX cache formats

def pin_e4m3_table(O):
    """Every E4M3 code decodes as torch's float8_e4m3fn does (a library routine), and the
    OCP 8-bit format's landmarks hold: 448 largest, 2^-6 smallest normal, 2^-9 smallest
    subnormal, S.1111.111 NaN."""
    import torch
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.asarray([O.fp_element_value(c, "e4m3") for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and int(np.isnan(got).sum()) == 2
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert O.fp_element_value(0x7E, "e4m3") == 448.0 and O.fp_element_value(0x08, "e4m3") == 2.0 ** -6
    assert O.fp_element_value(0x01, "e4m3") == 2.0 ** -9 and O.fp_element_value(0x38, "e4m3") == 1.0
    assert O.fp_element_value(0xB8, "e4m3") == -1.0


def pin_e2m1_table(O):
    """The sixteen E2M1 values of the OCP MX specification's FP4 element table."""
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = [O.fp_element_value(c, "e2m1") for c in range(16)]
    assert got[:8] == want and got[8:] == [-v for v in want]


def pin_element_rounding(O):
    """Round to nearest, ties to the even code, saturating: E4M3 against torch's
    float32 -> float8_e4m3fn conversion (RNE) inside the finite range, hand-worked E2M1
    ties, and the array form equal to the scalar definition."""
    import torch
    r = np.random.default_rng(7)
    v = np.concatenate([r.standard_normal(400) * 60.0, r.standard_normal(200) * 2.0 ** -7,
                        (O.element_table("e4m3")[:-1] + O.element_table("e4m3")[1:]) / 2])
    v = np.concatenate([v, -v]).astype(np.float32).astype(np.float64)
    v = v[np.abs(v) < 448.0]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.asarray([O.fp_element_encode(x, "e4m3") for x in v])
    assert np.array_equal(got, ref.astype(np.int64))
    assert O.fp_element_encode(1000.0, "e4m3") == 0x7E and O.fp_element_encode(-500.0, "e4m3") == 0xFE
    # E2M1: midpoints go to the even code; beyond 6 saturates; -0.1 keeps its sign bit
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7, 100.0: 7,
             0.26: 1, 2.49: 4, 2.51: 5, -0.1: 8, -3.4: 13, -5.1: 15}
    for x, c in cases.items():
        assert O.fp_element_encode(x, "e2m1") == c, (x, c)
    for fmt in ("e4m3", "e2m1"):
        w = np.concatenate([v / (1.0 if fmt == "e4m3" else 70.0), [0.0, -0.0]])
        assert np.array_equal(O.fp_elements_encode(w, fmt), [O.fp_element_encode(x, fmt) for x in w])


def pin_mx_block_exponent(O):
    """The block exponent is the smallest e with max|v| <= max_elem * 2^e (hand-worked
    cases), -127 for a zero block, and scales with the block: 2^k * block -> e + k."""
    assert O.mx_block_exponent([1.0, -0.5], "e4m3") == -8      # 1 * 2^8 = 256 <= 448
    assert O.mx_block_exponent([1.75], "e4m3") == -8           # 448 exactly
    assert O.mx_block_exponent([-1.76], "e4m3") == -7          # 450.56 > 448
    assert O.mx_block_exponent([1.5], "e2m1") == -2            # 6 exactly
    assert O.mx_block_exponent([1.6], "e2m1") == -1
    assert O.mx_block_exponent([0.0, -0.0], "e4m3") == -127
    r = np.random.default_rng(3)
    for fmt in ("e4m3", "e2m1"):
        blk = r.standard_normal(32)
        for k in (-20, -3, 5, 40):
            assert O.mx_block_exponent(np.ldexp(blk, k), fmt) == O.mx_block_exponent(blk, fmt) + k
        rows = r.standard_normal((2, 64))
        c0, s0 = O.mx_encode_rows(rows, fmt)
        c1, s1 = O.mx_encode_rows(np.ldexp(rows, 9), fmt)
        assert np.array_equal(c0, c1) and np.array_equal(s1, s0 + 9)


def pin_mx_round_trip_and_bound(O):
    """Dequantised values re-encode to themselves exactly; encoding a real row errs by at
    most half the element grid's spacing at the scaled magnitude; blocks are 32 wide."""
    r = np.random.default_rng(11)
    for fmt, top in (("e4m3", 0x7E), ("e2m1", 7)):
        f = O.MX_FORMATS[fmt]
        sign = 0x80 if fmt == "e4m3" else 0x8
        codes = r.integers(0, top + 1, size=(3, 96)) | (r.integers(0, 2, size=(3, 96)) * sign)
        scales = r.integers(100, 150, size=(3, 3))
        vals = O.mx_decode_rows(codes, scales, fmt)
        for b in range(3):   # block b of every row uses scales[:, b] and nothing else
            blk = vals[:, 32 * b:32 * b + 32]
            assert np.array_equal(blk, np.ldexp(np.vectorize(lambda c: O.fp_element_value(c, fmt))(
                codes[:, 32 * b:32 * b + 32]), scales[:, b:b + 1] - 127))
        c2, s2 = O.mx_encode_rows(vals, fmt)
        assert np.array_equal(O.mx_decode_rows(c2, s2, fmt), vals)
        x = r.standard_normal((4, 64)) * np.exp(r.standard_normal((4, 1)) * 3)
        c, s = O.mx_encode_rows(x, fmt)
        e = np.repeat(s - 127, 32, axis=-1)
        a = np.abs(np.ldexp(x, -e))
        assert np.all(a <= f["max"])
        min_normal = 2.0 ** (1 - f["bias"])
        binade = np.floor(np.log2(np.maximum(a, min_normal)))
        half_step = np.ldexp(2.0 ** (binade - f["mbits"] - 1), e)
        assert np.all(np.abs(O.mx_decode_rows(c, s, fmt) - x) <= half_step)


def pin_e2m1_packing(O):
    """Two E2M1 codes per byte, element 2i in the low nibble: codes (2, 4), i.e. 1.0 then
    2.0, pack to 0x42."""
    assert list(O.mx_pack_e2m1([2, 4, 15, 0])) == [0x42, 0x0F]
    assert list(O.mx_unpack_e2m1(np.asarray([0x42, 0x0F]))) == [2, 4, 15, 0]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
