"""CPU tests of the oracle against its pins, plus planted-mistake (mutation) checks."""
from __future__ import annotations

import math
import types

import numpy as np
import pytest

import oracle.mla_oracle as OR
from tests import oracle_pins as PINS


def _namespace(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(OR, k) for k in dir(OR) if not k.startswith("__")})
    for k, v in overrides.items():
        setattr(ns, k, v)
    return ns


@pytest.mark.parametrize("pin", PINS.ALL_PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    pin(_namespace())


# ---------------------------------------------------------------------------- planted mistakes

def _rope_sign_flip(v, pos, base):
    v = np.asarray(v, dtype=np.float64)
    ang = OR.rope_angles(np.broadcast_to(np.asarray(pos), v.shape[:-1]), v.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(v)
    out[..., 0::2] = v[..., 0::2] * c + v[..., 1::2] * s
    out[..., 1::2] = -v[..., 0::2] * s + v[..., 1::2] * c
    return out


def _rope_half_split(v, pos, base):
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    ang = OR.rope_angles(np.broadcast_to(np.asarray(pos), v.shape[:-1]), d, base)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., : d // 2], v[..., d // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _rope_wrong_freq(v, pos, base):
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.asarray(np.broadcast_to(np.asarray(pos), v.shape[:-1]), dtype=np.float64)[..., None] \
        * np.power(base, -i / d)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(v)
    out[..., 0::2] = v[..., 0::2] * c - v[..., 1::2] * s
    out[..., 1::2] = v[..., 0::2] * s + v[..., 1::2] * c
    return out


def _attn_no_rope(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale):
    return OR.attention_unabsorbed(q_nope, np.zeros_like(np.asarray(q_rope, float)), c_kv,
                                   k_rope, w_uk, w_uv, scale)


def _attn_wrong_scale(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale):
    d_h = np.asarray(q_nope).shape[-1]
    d_r = np.asarray(q_rope).shape[-1]
    return OR.attention_unabsorbed(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv,
                                   scale * math.sqrt(d_h + d_r) / math.sqrt(d_h))


def _attn_head_swap(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale):
    q = np.asarray(q_nope, dtype=np.float64)
    n_h, d_h = q.shape
    w = np.asarray(w_uk, dtype=np.float64)
    w = np.concatenate([w[:, h * d_h:(h + 1) * d_h] for h in reversed(range(n_h))], axis=1)
    return OR.attention_unabsorbed(q_nope, q_rope, c_kv, k_rope, w, w_uv, scale)


def _absorb_transposed(q_nope, q_rope, pos, w_uk, base):
    # restores head slices as rows-major blocks of the flattened weight (a transposed reading)
    q_nope = np.asarray(q_nope, dtype=np.float64)
    N, n_h, d_h = q_nope.shape
    w = np.asarray(w_uk, dtype=np.float64)
    d_c = w.shape[0]
    wt = w.reshape(n_h, d_h, d_c)  # wrong: treats [d_c, n_h*d_h] as head-major rows
    q_lat = np.einsum("nhd,hdc->nhc", q_nope, wt)
    q_r = OR.rope_rotate(q_rope, np.asarray(pos)[:, None], base)
    return np.concatenate([q_lat, q_r], axis=-1)


def _latent_rotated(x, w_dkv, w_kr, pos, base):
    c, k = OR.latent_kv(x, w_dkv, w_kr, pos, base)
    return OR.rope_rotate(c, pos, base), k


def _prefill_mask_off_by_one(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale):
    # lets query i also see token i + 1
    T = np.asarray(q_nope).shape[0]
    o, o_lat, lse = [], [], []
    for i in range(T):
        j = min(T, i + 2)
        a, b, c, _ = OR.attention_unabsorbed(q_nope[i], q_rope[i], c_kv[:j], k_rope[:j], w_uk,
                                             w_uv, scale)
        o.append(a); o_lat.append(b); lse.append(c)
    return np.stack(o), np.stack(o_lat), np.stack(lse)


def _lse_missing_max(scores):
    s = np.asarray(scores, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(-1, keepdims=True)
    return e / z, np.log(z)[..., 0]


def _up_wrong_head(o_lat, w_uv):
    o_lat = np.asarray(o_lat, dtype=np.float64)
    N, n_h, _ = o_lat.shape
    return OR.up_project_output(o_lat[:, ::-1, :], w_uv)


def _out_proj_transposed(o, w_o):
    o = np.asarray(o, dtype=np.float64)
    N, n_h, d_h = o.shape
    return o.transpose(0, 2, 1).reshape(N, -1) @ np.asarray(w_o, dtype=np.float64)


def _mha_numbers_single(n_h, d_h):
    return n_h * d_h


def _scale_sqrt_dh(d_nope, d_rope):
    return 1.0 / math.sqrt(d_nope)


def _gather_wrong_slot(pool, pt_row, length):
    pool = np.asarray(pool)
    ps = pool.shape[1]
    return np.asarray([pool[int(pt_row[t // ps]), (t + 1) % ps] for t in range(length)],
                      dtype=np.float64)


def _mx_exponent_floor_only(block, fmt):
    # the specification's floor rule without the raise: large elements saturate
    a = float(np.max(np.abs(np.asarray(block, dtype=np.float64))))
    if a == 0.0:
        return -127
    return int(max(-127, min(127, math.frexp(a)[1] - 1 - OR.MX_FORMATS[fmt]["emax"])))


def _encode_ties_away(v, fmt):
    c = OR.fp_element_encode(v, fmt)
    lo = OR.fp_element_value(c, fmt)
    nxt = c + 1
    if abs(abs(v) - abs(lo)) > 0 and (c & 1) == 0:
        hi = OR.fp_element_value(nxt, fmt) if not math.isnan(OR.fp_element_value(nxt, fmt)) else lo
        if abs(abs(v) - abs(lo)) == abs(abs(hi) - abs(v)):
            return nxt
    return c


def _e4m3_bias8(code, fmt):
    v = OR.fp_element_value(code, fmt)
    return v / 2.0 if fmt == "e4m3" else v


def _pack_swapped(codes):
    c = np.asarray(codes, dtype=np.int64)
    return ((c[1::2] & 0xF) | ((c[0::2] & 0xF) << 4)).astype(np.uint8)


def _decode_blocks_of_16(codes, scale_bytes, fmt):
    codes = np.asarray(codes, dtype=np.int64)
    vals = np.vectorize(lambda c: OR.fp_element_value(c, fmt))(codes).astype(np.float64)
    e = np.asarray(scale_bytes, dtype=np.int64) - 127
    e = np.repeat(e, 16, axis=-1)
    e = np.concatenate([e, np.repeat(e[..., -1:], codes.shape[-1] - e.shape[-1], axis=-1)], axis=-1)
    return np.ldexp(vals, e[..., :codes.shape[-1]])


def _uq_uk_transposed(w_uq, w_uk, n_h):
    w_uq = np.asarray(w_uq, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    d_h = w_uq.shape[1] // n_h
    return np.concatenate([w_uq[:, h * d_h:(h + 1) * d_h] @ w_uk[:, ((n_h - 1 - h) * d_h):((n_h - h) * d_h)].T
                           for h in range(n_h)], axis=1)


def _compressed_rope_from_x(x, w_dq, w_uq, w_qr, pos, n_h, base):
    # rope query taken from the first d_cq columns of x instead of from c_q
    c_q = OR.query_latent(x, w_dq)
    q, _ = OR.query_projection(c_q, w_uq, w_qr, pos, n_h, base)
    xs = np.asarray(x, dtype=np.float64)[:, :np.asarray(w_qr).shape[0]]
    _, qr = OR.query_projection(xs, w_uq, w_qr, pos, n_h, base)
    return q, qr


MUTANTS = {
    "rope_sign_flip": dict(rope_rotate=_rope_sign_flip),
    "rope_half_split": dict(rope_rotate=_rope_half_split),
    "rope_wrong_freq": dict(rope_rotate=_rope_wrong_freq),
    "attention_drops_rope_term": dict(attention_unabsorbed=_attn_no_rope),
    "attention_scale_sqrt_dh": dict(attention_unabsorbed=_attn_wrong_scale),
    "attention_head_swap": dict(attention_unabsorbed=_attn_head_swap),
    "absorb_transposed_weight": dict(absorb_query=_absorb_transposed),
    "latent_rotated": dict(latent_kv=_latent_rotated),
    "prefill_mask_off_by_one": dict(causal_prefill_unabsorbed=_prefill_mask_off_by_one),
    "lse_missing_max": dict(softmax_lse=_lse_missing_max),
    "up_projection_wrong_head": dict(up_project_output=_up_wrong_head),
    "out_projection_transposed": dict(output_projection=_out_proj_transposed),
    "mha_count_drops_v": dict(mha_numbers_per_token=_mha_numbers_single),
    "paged_gather_wrong_slot": dict(sequence_rows=_gather_wrong_slot),
    "default_scale_sqrt_dh": dict(default_scale=_scale_sqrt_dh),
    "mx_exponent_floor_only": dict(mx_block_exponent=_mx_exponent_floor_only),
    "mx_ties_away_from_zero": dict(fp_element_encode=_encode_ties_away),
    "e4m3_bias_8": dict(fp_element_value=_e4m3_bias8),
    "e2m1_nibbles_swapped": dict(mx_pack_e2m1=_pack_swapped),
    "mx_decode_blocks_of_16": dict(mx_decode_rows=_decode_blocks_of_16),
    "uq_uk_wrong_head": dict(absorb_uq_uk=_uq_uk_transposed),
    "compressed_rope_from_x": dict(query_projection_compressed=_compressed_rope_from_x),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    ns = _namespace(**MUTANTS[name])
    failures = []
    for pin in PINS.ALL_PINS:
        try:
            pin(ns)
        except (AssertionError, ValueError, IndexError):
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
