"""CPU oracle for Multi-head Latent Attention over a latent KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute this
module: only the tests, the smoke check and the benchmark's CPU-baseline / reference leg
use it.  It shares no code with the CUDA library and imports nothing from it.

Everything is float64 numpy.  Inputs arrive as float64 arrays (bf16 or f32 storage values
already widened).  Citations name the page and its section:

  [OPN]  "Operator Notes (1): MLA - Multi-head Latent Attention at the Operator Level"
         (naphjohn LLM blog), section 2 "Line-by-Line Operator Pseudocode" (weight shapes
         and the prefill chain), section 3 "How Much the Cache Shrinks" (cache table),
         section 4 (query compression).
  [GLO]  "multi-head latent attention" (chipfoundryservices glossary): the paragraphs on
         the decoupled RoPE key and on absorbing the up-projections into the query and
         output projections; the MHA/GQA/MLA comparison table.
  [RMJ]  "Multi-Head Latent Attention and the Compression of the KV Cache" (rmj-insight
         dispatch): associativity lets the up-projection be absorbed into the query.
  [IPM]  "Multi-Head Latent Attention (MLA) Explained: What DeepSeek's Architecture Means
         for AI Inference Costs" (institutepm knowledge hub), section "Which Models Use MLA
         and What Is Next": MXFP4 quantisation of the KV cache.

Readings taken where the pages are silent (each is listed with its reason in the design
notes of the repository):
  * score scale 1/sqrt(d_h + d_rope): the dot product spans the nope and the rope parts;
  * RoPE on interleaved pairs (2i, 2i+1), angle pos * base^(-2i/d_rope), base 10000;
  * one RoPE key of width d_rope per token, shared by all heads; one RoPE query per head;
  * per-head weight slices are column block h of W_UK / W_UV / W_Q / W_QR (row-major,
    head-major reading of the [d_c, n_h*d_h] shapes) and row block h of W_O;
  * 0-based positions; causal prefill lets query i see tokens t <= i.

Pins for every function live in tests/test_oracle.py (closed forms, brute-force loops on
tiny inputs, the pages' cache-size integers, associativity between the two forms).
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ------------------------------------------------------------------------------------------
# cache accounting  ([OPN] section 1 and the section 3 table)
# ------------------------------------------------------------------------------------------

def mha_numbers_per_token(n_h: int, d_h: int) -> int:
    """MHA caches K and V for every head: 2 * n_h * d_h numbers per token ([OPN] s.1)."""
    return 2 * n_h * d_h


def mla_numbers_per_token(d_c: int, d_rope: int = 0) -> int:
    """MLA caches only the latent c_kv ([OPN] s.3) plus the decoupled RoPE key ([GLO])."""
    return d_c + d_rope


# ------------------------------------------------------------------------------------------
# rotary position embedding  ([GLO] decoupled RoPE key paragraph; convention is a reading)
# ------------------------------------------------------------------------------------------

def rope_angles(pos, d_rope: int, base: float) -> np.ndarray:
    """Angle pos * base^(-2i/d_rope) for pair i; shape pos.shape + (d_rope/2,)."""
    i = np.arange(d_rope // 2, dtype=F64)
    theta = np.power(F64(base), -2.0 * i / d_rope)
    return np.asarray(pos, dtype=F64)[..., None] * theta


def rope_rotate(v, pos, base: float) -> np.ndarray:
    """Rotate each interleaved pair (v[2i], v[2i+1]) of the last axis by its angle.

    `pos` broadcasts against v.shape[:-1].
    """
    v = np.asarray(v, dtype=F64)
    ang = rope_angles(np.broadcast_to(np.asarray(pos), v.shape[:-1]), v.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    even, odd = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = even * c - odd * s
    out[..., 1::2] = even * s + odd * c
    return out


# ------------------------------------------------------------------------------------------
# projections
# ------------------------------------------------------------------------------------------

def head_cols(w, h: int, width: int) -> np.ndarray:
    """Column block h of a [rows, n_h*width] weight: the slice that belongs to head h."""
    return np.asarray(w, dtype=F64)[:, h * width:(h + 1) * width]


def latent_kv(x, w_dkv, w_kr, pos, base: float):
    """Down-projection that fills the cache ([OPN] s.2 'c_kv = x @ W_DKV', the only KV state
    cached) and the decoupled RoPE key ([GLO]): k_rope = RoPE(x @ W_KR, pos).

    x [N, d_model], w_dkv [d_model, d_c], w_kr [d_model, d_rope], pos [N].
    Returns c_kv [N, d_c], k_rope [N, d_rope].
    """
    x = np.asarray(x, dtype=F64)
    c_kv = x @ np.asarray(w_dkv, dtype=F64)
    k_rope = rope_rotate(x @ np.asarray(w_kr, dtype=F64), pos, base)
    return c_kv, k_rope


def query_projection(x, w_q, w_qr, pos, n_h: int, base: float):
    """Simplest query side ([OPN] s.2 'Q = x @ W_Q') plus a per-head RoPE query.

    x [N, d_model], w_q [d_model, n_h*d_h], w_qr [d_model, n_h*d_rope], pos [N].
    Returns q_nope [N, n_h, d_h], q_rope [N, n_h, d_rope] (rotated).
    """
    x = np.asarray(x, dtype=F64)
    N = x.shape[0]
    q = (x @ np.asarray(w_q, dtype=F64)).reshape(N, n_h, -1)
    qr = (x @ np.asarray(w_qr, dtype=F64)).reshape(N, n_h, -1)
    return q, rope_rotate(qr, np.asarray(pos)[:, None], base)


def query_latent(x, w_dq):
    """Compressed query ([OPN] s.4 'c_q = x @ W_DQ'): x [N, d_model], w_dq [d_model, d_cq]."""
    return np.asarray(x, dtype=F64) @ np.asarray(w_dq, dtype=F64)


def query_projection_compressed(x, w_dq, w_uq, w_qr, pos, n_h: int, base: float):
    """The query side with compression ([OPN] s.4): c_q = x @ W_DQ, then Q = c_q @ W_UQ, and
    the per-head RoPE query from the same latent, RoPE(c_q @ W_QR) (reading: with compression
    the decoupled RoPE query is projected from c_q, as the uncompressed one is from x).

    x [N, d_model], w_dq [d_model, d_cq], w_uq [d_cq, n_h*d_h], w_qr [d_cq, n_h*d_rope], pos [N].
    Returns q_nope [N, n_h, d_h], q_rope [N, n_h, d_rope] (rotated).
    """
    return query_projection(query_latent(x, w_dq), w_uq, w_qr, pos, n_h, base)


def absorb_uq_uk(w_uq, w_uk, n_h: int):
    """W_UQ folded into W_UK ([GLO] absorption, [RMJ] associativity): per head the
    [d_cq, d_c] product W_UQ_h @ W_UK_h^T, so that c_q @ (W_UQ_h @ W_UK_h^T) is the absorbed
    query's latent part.  w_uq [d_cq, n_h*d_h], w_uk [d_c, n_h*d_h].  Returns [d_cq, n_h*d_c]
    with head h in column block h."""
    w_uq = np.asarray(w_uq, dtype=F64)
    w_uk = np.asarray(w_uk, dtype=F64)
    d_h = w_uq.shape[1] // n_h
    return np.concatenate([head_cols(w_uq, h, d_h) @ head_cols(w_uk, h, d_h).T for h in range(n_h)], axis=1)


def restore_kv(c_kv, w_uk, w_uv, n_h: int):
    """Up-projections that restore per-head K and V from the latent ([OPN] s.2
    'K = c_kv @ W_UK', 'V = c_kv @ W_UV').  Returns K, V as [L, n_h, d_h]."""
    c_kv = np.asarray(c_kv, dtype=F64)
    L = c_kv.shape[0]
    K = (c_kv @ np.asarray(w_uk, dtype=F64)).reshape(L, n_h, -1)
    V = (c_kv @ np.asarray(w_uv, dtype=F64)).reshape(L, n_h, -1)
    return K, V


# ------------------------------------------------------------------------------------------
# softmax attention
# ------------------------------------------------------------------------------------------

def softmax_lse(scores):
    """Row softmax over the last axis: returns (p, lse) with lse = log sum exp(scores).

    Entries equal to -inf are masked out.
    """
    s = np.asarray(scores, dtype=F64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    lse = (m + np.log(z))[..., 0]
    return e / z, lse


def attention_unabsorbed(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale: float):
    """One query token attending to L cached tokens, un-absorbed ([OPN] s.2 chain).

    K and V are restored per head from the latent; the score of head h and token t is
    (q_nope[h] . K[t, h] + q_rope[h] . k_rope[t]) * scale; softmax over t; o[h] = p @ V[:, h].
    The latent-space output o_lat[h] = p @ c_kv is returned as well (it is what the absorbed
    kernel produces before the W_UV up-projection).

    q_nope [n_h, d_h], q_rope [n_h, d_rope] (rotated), c_kv [L, d_c], k_rope [L, d_rope]
    (rotated).  Returns o [n_h, d_h], o_lat [n_h, d_c], lse [n_h], p [n_h, L].
    """
    q_nope = np.asarray(q_nope, dtype=F64)
    q_rope = np.asarray(q_rope, dtype=F64)
    c_kv = np.asarray(c_kv, dtype=F64)
    k_rope = np.asarray(k_rope, dtype=F64)
    n_h = q_nope.shape[0]
    K, V = restore_kv(c_kv, w_uk, w_uv, n_h)
    scores = (np.einsum("hd,thd->ht", q_nope, K) + q_rope @ k_rope.T) * scale
    p, lse = softmax_lse(scores)
    o = np.einsum("ht,thd->hd", p, V)
    o_lat = p @ c_kv
    return o, o_lat, lse, p


def causal_prefill_unabsorbed(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale: float):
    """T queries of one sequence against its own T cached tokens with a causal mask
    ([OPN] s.2 'scores = Q @ K^T / sqrt(d)' as a [n_h, T, T] matrix; query i sees t <= i).

    q_nope [T, n_h, d_h], q_rope [T, n_h, d_rope] (rotated), c_kv [T, d_c], k_rope [T, d_rope].
    Returns o [T, n_h, d_h], o_lat [T, n_h, d_c], lse [T, n_h].
    """
    q_nope = np.asarray(q_nope, dtype=F64)
    q_rope = np.asarray(q_rope, dtype=F64)
    c_kv = np.asarray(c_kv, dtype=F64)
    T, n_h, _ = q_nope.shape
    K, V = restore_kv(c_kv, w_uk, w_uv, n_h)
    scores = (np.einsum("ihd,thd->hit", q_nope, K)
              + np.einsum("ihr,tr->hit", q_rope, np.asarray(k_rope, dtype=F64))) * scale
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    scores = np.where(mask[None], -np.inf, scores)
    p, lse = softmax_lse(scores)                    # p [n_h, T, T], lse [n_h, T]
    o = np.einsum("hit,thd->ihd", p, V)
    o_lat = np.einsum("hit,tc->ihc", p, c_kv)
    return o, o_lat, lse.T


def output_projection(o, w_o):
    """Final projection over the concatenated heads ([OPN] s.2 'out = O @ W_O')."""
    o = np.asarray(o, dtype=F64)
    return o.reshape(o.shape[0], -1) @ np.asarray(w_o, dtype=F64)


# ------------------------------------------------------------------------------------------
# absorbed form ([GLO] absorption paragraph, [RMJ] associativity)
# ------------------------------------------------------------------------------------------

def absorb_query(q_nope, q_rope, pos, w_uk, base: float):
    """Fold W_UK into the query: q_lat[n, h] = W_UK_h @ q_nope[n, h] (a d_c vector), and
    append the rotated RoPE query.  Returns q_cat [N, n_h, d_c + d_rope].

    q_nope [N, n_h, d_h], q_rope [N, n_h, d_rope] (NOT yet rotated), pos [N].
    """
    q_nope = np.asarray(q_nope, dtype=F64)
    N, n_h, d_h = q_nope.shape
    w_uk = np.asarray(w_uk, dtype=F64)
    q_lat = np.stack([q_nope[:, h, :] @ head_cols(w_uk, h, d_h).T for h in range(n_h)], axis=1)
    q_r = rope_rotate(q_rope, np.asarray(pos)[:, None], base)
    return np.concatenate([q_lat, q_r], axis=-1)


def attention_latent(q_cat, cache_rows, d_c: int, scale: float):
    """Softmax attention computed directly on the latent cache rows.

    Keys are the whole cached row [c_kv | k_rope], values its first d_c entries; this is
    the absorbed form whose equality with `attention_unabsorbed` is pinned in the tests.

    q_cat [n_h, d_c + d_rope], cache_rows [L, d_c + d_rope].  Returns o_lat [n_h, d_c],
    lse [n_h].
    """
    q_cat = np.asarray(q_cat, dtype=F64)
    rows = np.asarray(cache_rows, dtype=F64)
    p, lse = softmax_lse((q_cat @ rows.T) * scale)
    return p @ rows[:, :d_c], lse


def up_project_output(o_lat, w_uv):
    """Absorbed output side: o[n, h] = o_lat[n, h] @ W_UV_h.  Returns [N, n_h*d_h]."""
    o_lat = np.asarray(o_lat, dtype=F64)
    N, n_h, _ = o_lat.shape
    w_uv = np.asarray(w_uv, dtype=F64)
    d_h = w_uv.shape[1] // n_h
    return np.concatenate([o_lat[:, h, :] @ head_cols(w_uv, h, d_h) for h in range(n_h)], axis=1)


# ------------------------------------------------------------------------------------------
# paged cache access (the cache layout is a data structure of the method: [GLO] pairs MLA
# with PagedAttention)
# ------------------------------------------------------------------------------------------

def sequence_rows(pool, page_table_row, length: int):
    """Cached rows of positions [0, length) of one sequence, widened to float64.

    pool [num_pages, page_size, width] float64; token t lives in page
    page_table_row[t // page_size], slot t % page_size.
    """
    pool = np.asarray(pool)
    ps = pool.shape[1]
    rows = [pool[int(page_table_row[t // ps]), t % ps] for t in range(length)]
    return np.asarray(rows, dtype=F64).reshape(length, pool.shape[2])


def default_scale(d_nope: int, d_rope: int) -> float:
    return 1.0 / np.sqrt(F64(d_nope + d_rope))


# ------------------------------------------------------------------------------------------
# low-precision latent cache  ([IPM] "Which Models Use MLA and What Is Next": MXFP4
# quantisation of the KV cache data type; the formats themselves are those of the OCP
# Microscaling Formats (MX) specification v1.0, which the pages do not restate)
#
#   [IPM]  "Multi-Head Latent Attention (MLA) Explained: What DeepSeek's Architecture Means
#          for AI Inference Costs" (institutepm knowledge hub).
#
# A cached row of W numbers is cut into blocks of 32 consecutive elements.  Each block keeps
# one shared scale 2^e (an E8M0 byte, e + 127) and 32 element codes: E4M3 bytes (MXFP8) or
# E2M1 nibbles (MXFP4).  The dequantised value of element i of a block is 2^e * elem(code_i).
# Readings (the pages name the format family only): the elements of a row are quantised in
# the order [c_kv | rotated k_rope]; the block exponent is the smallest e with
# max |v| <= max_elem * 2^e, i.e. the specification's floor(log2(max |v|)) - emax_elem,
# raised by one when the block's largest element would otherwise saturate (so no element is
# clipped), clamped to the E8M0 range [-127, 127] (a zero block gets e = -127); element codes
# round to nearest, ties to the even code, and saturate at the largest finite magnitude (only
# reachable at the clamp); a negative value that rounds to zero keeps its sign bit.
# ------------------------------------------------------------------------------------------

MX_BLOCK = 32

# element formats: exponent bits, mantissa bits, exponent bias, emax (exponent of the
# largest normal binade) and the largest finite magnitude
MX_FORMATS = {
    "e4m3": dict(ebits=4, mbits=3, bias=7, emax=8, max=448.0),
    "e2m1": dict(ebits=2, mbits=1, bias=1, emax=2, max=6.0),
}


def fp_element_value(code: int, fmt: str) -> float:
    """Value of one element code.  E4M3 (byte): S.EEEE.MMM, bias 7, no infinities,
    S.1111.111 is NaN.  E2M1 (nibble): S.EE.M, bias 1, every code finite.  Exponent field 0
    encodes subnormals 2^(1-bias) * M / 2^mbits."""
    f = MX_FORMATS[fmt]
    nbits = 1 + f["ebits"] + f["mbits"]
    code = int(code) & ((1 << nbits) - 1)
    sign = -1.0 if code >> (nbits - 1) else 1.0
    E = (code >> f["mbits"]) & ((1 << f["ebits"]) - 1)
    M = code & ((1 << f["mbits"]) - 1)
    if fmt == "e4m3" and E == 15 and M == 7:
        return float("nan")
    if E == 0:
        return sign * 2.0 ** (1 - f["bias"]) * M / 2 ** f["mbits"]
    return sign * 2.0 ** (E - f["bias"]) * (1.0 + M / 2 ** f["mbits"])


def fp_element_encode(v: float, fmt: str) -> int:
    """Code of the representable value nearest to v (ties to the even code), saturating at
    +/- max.  Walks the non-negative finite codes, which increase with their value."""
    f = MX_FORMATS[fmt]
    nbits = 1 + f["ebits"] + f["mbits"]
    sign_bit = 1 << (nbits - 1)
    v = float(v)
    neg = v < 0 or (v == 0 and math.copysign(1.0, v) < 0)
    a = abs(v)
    n_finite = sign_bit - 1 if fmt == "e4m3" else sign_bit  # e4m3 drops S.1111.111 (NaN)
    if a >= f["max"]:
        mag = n_finite - 1
    else:
        mag = 0
        while fp_element_value(mag + 1, fmt) <= a:
            mag += 1
        lo, hi = fp_element_value(mag, fmt), fp_element_value(mag + 1, fmt)
        if a - lo > hi - a or (a - lo == hi - a and mag % 2 == 1):
            mag += 1
    return (sign_bit if neg else 0) | mag


def mx_block_exponent(block, fmt: str) -> int:
    """Shared exponent of a block: the smallest e with max |v| <= max_elem * 2^e, clamped to
    [-127, 127].  With e0 = floor(log2(max |v|)) - emax the scaled maximum lies in
    [2^emax, 2^(emax+1)), so e is e0, or e0 + 1 when that scaled maximum exceeds max_elem."""
    f = MX_FORMATS[fmt]
    amax = float(np.max(np.abs(np.asarray(block, dtype=F64))))
    if amax == 0.0:
        return -127
    _, ex = math.frexp(amax)  # amax = m * 2^ex with 0.5 <= m < 1, so floor(log2 amax) = ex - 1
    e = ex - 1 - f["emax"]
    if math.ldexp(amax, -e) > f["max"]:
        e += 1
    return int(min(127, max(-127, e)))


def element_table(fmt: str) -> np.ndarray:
    """Values of the non-negative finite codes 0, 1, 2, ... (increasing with the code)."""
    f = MX_FORMATS[fmt]
    n = (1 << (f["ebits"] + f["mbits"])) - (1 if fmt == "e4m3" else 0)
    return np.asarray([fp_element_value(c, fmt) for c in range(n)], dtype=F64)


def fp_elements_encode(values, fmt: str) -> np.ndarray:
    """fp_element_encode over an array: the same nearest-even, saturating choice, found by a
    search of the increasing table instead of a walk."""
    f = MX_FORMATS[fmt]
    nbits = 1 + f["ebits"] + f["mbits"]
    tab = element_table(fmt)
    v = np.asarray(values, dtype=F64)
    a = np.abs(v)
    lo = np.clip(np.searchsorted(tab, a, side="right") - 1, 0, len(tab) - 1)
    hi = np.minimum(lo + 1, len(tab) - 1)
    dlo, dhi = a - tab[lo], tab[hi] - a
    up = (hi > lo) & ((dlo > dhi) | ((dlo == dhi) & (lo % 2 == 1)))
    mag = np.where(a >= f["max"], len(tab) - 1, np.where(up, hi, lo))
    neg = np.signbit(v)
    return np.where(neg, (1 << (nbits - 1)) | mag, mag).astype(np.int64)


def mx_encode_rows(rows, fmt: str):
    """Encode rows [..., W] (W a multiple of 32).  Returns (codes [..., W] ints, scale bytes
    [..., W/32] ints); the scale byte of a block is its exponent e + 127."""
    rows = np.asarray(rows, dtype=F64)
    W = rows.shape[-1]
    assert W % MX_BLOCK == 0
    blocks = rows.reshape(-1, W // MX_BLOCK, MX_BLOCK)
    e = np.empty(blocks.shape[:2], dtype=np.int64)
    for i in range(blocks.shape[0]):
        for b in range(blocks.shape[1]):
            e[i, b] = mx_block_exponent(blocks[i, b], fmt)
    scaled = np.ldexp(blocks, -e[..., None])
    codes = fp_elements_encode(scaled, fmt).reshape(rows.shape)
    return codes, (e + 127).reshape(rows.shape[:-1] + (W // MX_BLOCK,))


def mx_decode_rows(codes, scale_bytes, fmt: str) -> np.ndarray:
    """Dequantise rows: element i of block b is 2^(scale_bytes[b] - 127) * elem(codes[i])."""
    codes = np.asarray(codes, dtype=np.int64)
    f = MX_FORMATS[fmt]
    nbits = 1 + f["ebits"] + f["mbits"]
    value_of = np.asarray([fp_element_value(c, fmt) for c in range(1 << nbits)], dtype=F64)
    e = np.asarray(scale_bytes, dtype=np.int64) - 127
    return np.ldexp(value_of[codes], np.repeat(e, MX_BLOCK, axis=-1))


def mx_pack_e2m1(codes) -> np.ndarray:
    """Two E2M1 codes per byte: element 2i in the low nibble of byte i, 2i+1 in the high."""
    c = np.asarray(codes, dtype=np.int64)
    return ((c[0::2] & 0xF) | ((c[1::2] & 0xF) << 4)).astype(np.uint8)


def mx_unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.int64)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = (p >> 4) & 0xF
    return out
