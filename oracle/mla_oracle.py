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
