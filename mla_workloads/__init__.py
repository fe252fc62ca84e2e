"""Seeded synthetic inputs for the MLA latent-KV hot path.

This module only draws random numbers, quantises them to the storage type and lays them
out (paged cache pool, page table, lengths).  It holds none of the attention arithmetic:
no projection, rotation, softmax or reduction.  Both the CUDA path (through the tests and
the benchmark) and the CPU oracle receive exactly the arrays produced here.

Shapes follow the DeepSeek-V2 reading of the pages (n_h=128, d_h=128, d_rope=64,
d_c=512, d_model=5120, page size 64); value distributions are N(0, 1) for latents,
activations and queries, and N(0, 1/fan_in) for weights.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

SENTINEL = 16384.0  # finite, exactly representable in bf16; fills every slot no token owns


@dataclass(frozen=True)
class Shape:
    n_heads: int
    d_nope: int
    d_rope: int
    d_latent: int
    d_model: int
    page_size: int = 64
    rope_base: float = 10000.0

    @property
    def width(self) -> int:
        """Numbers cached per token: the latent plus the decoupled RoPE key."""
        return self.d_latent + self.d_rope


DEEPSEEK_V2 = Shape(n_heads=128, d_nope=128, d_rope=64, d_latent=512, d_model=5120)
TINY = Shape(n_heads=4, d_nope=16, d_rope=8, d_latent=32, d_model=64)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    dtype: str            # storage / operand type: "f32" or "bf16"
    mode: str             # "tiny_decode" | "decode" | "append_decode" | "prefill"
    seed: int
    batch: int
    lens: tuple = ()      # fixed cached lengths per sequence (decode)
    len_range: tuple = () # (lo, hi) inclusive integer-uniform lengths (ragged decode)
    tokens: int = 0       # query tokens (prefill / tiny)
    spare_pages: int = 64
    shuffled: bool = True
    kv: str = ""          # "" plain cache rows of `dtype`; "mxfp8" / "mxfp4" an MX cache
    form: str = ""        # prefill: "" absorbed (the latent path), "unabsorbed" (restore K and V)

    def describe(self) -> str:
        s = self.shape
        return (f"{self.name}: B={self.batch} n_h={s.n_heads} d_h={s.d_nope} d_rope={s.d_rope} "
                f"d_c={s.d_latent} d_model={s.d_model} dtype={self.dtype} mode={self.mode}")


WORKLOADS = {
    # Tiny fp32 decode: one query token (the last of 64) against 64 cached tokens.
    "tiny_f32": Workload("tiny_f32", TINY, "f32", "tiny_decode", seed=0, batch=1, tokens=64,
                         spare_pages=0, shuffled=False),
    # DeepSeek-V2-shaped decode, B=16, 4096 cached tokens each.
    "decode_b16_l4096": Workload("decode_b16_l4096", DEEPSEEK_V2, "bf16", "decode", seed=1,
                                 batch=16, lens=(4096,) * 16),
    # Long-context decode, B=4.
    "decode_long_b4": Workload("decode_long_b4", DEEPSEEK_V2, "bf16", "decode", seed=2, batch=4,
                               lens=(32768, 65536, 98304, 131072)),
    # Ragged high-concurrency decode with one appended token per sequence.
    "decode_ragged_b256": Workload("decode_ragged_b256", DEEPSEEK_V2, "bf16", "append_decode",
                                   seed=3, batch=256, len_range=(256, 8192)),
    # The B=16 x 4096 decode over MX-encoded caches (E4M3 and E2M1 elements, 32-element blocks).
    "decode_b16_l4096_mxfp8": Workload("decode_b16_l4096_mxfp8", DEEPSEEK_V2, "bf16", "decode", seed=5,
                                       batch=16, lens=(4096,) * 16, kv="mxfp8"),
    "decode_b16_l4096_mxfp4": Workload("decode_b16_l4096_mxfp4", DEEPSEEK_V2, "bf16", "decode", seed=6,
                                       batch=16, lens=(4096,) * 16, kv="mxfp4"),
    # Causal prefill of 8192 tokens that also builds the cache.
    "prefill_t8192": Workload("prefill_t8192", DEEPSEEK_V2, "bf16", "prefill", seed=4, batch=1,
                              tokens=8192),
    # The same prefill in the un-absorbed form of the operator notes (restore K and V per head).
    "prefill_t8192_unabsorbed": Workload("prefill_t8192_unabsorbed", DEEPSEEK_V2, "bf16", "prefill", seed=4,
                                         batch=1, tokens=8192, form="unabsorbed"),
}


# --------------------------------------------------------------------------------------
# storage-type helpers (quantisation of synthetic data; no method arithmetic)
# --------------------------------------------------------------------------------------

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even) and return the raw bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a stored array (bf16 bits or float32) to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def quantise(a: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(a) if dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def weight(rng, fan_in: int, fan_out: int, dtype: str) -> np.ndarray:
    """[fan_in, fan_out] weight drawn N(0, 1/fan_in), stored in `dtype`."""
    return quantise(normal(rng, (fan_in, fan_out), 1.0 / np.sqrt(fan_in)), dtype)


def sentinel_rows(n: int, width: int, dtype: str) -> np.ndarray:
    """Rows of +/-SENTINEL (alternating by column): finite, loud if ever attended."""
    row = np.where(np.arange(width) % 2 == 0, SENTINEL, -SENTINEL).astype(np.float32)
    return quantise(np.broadcast_to(row, (n, width)).copy(), dtype)


# --------------------------------------------------------------------------------------
# paged cache layout
# --------------------------------------------------------------------------------------

def pages_for(length: int, page_size: int) -> int:
    return -(-int(length) // page_size)


def make_page_table(rng, lens_alloc, page_size: int, spare_pages: int, shuffled: bool):
    """Physical page ids for every sequence, enough for `lens_alloc[b]` tokens.

    Returns (page_table [B, max_pages] int32 with -1 past each sequence's pages,
    num_pages).  Physical ids are a seeded permutation when `shuffled`.
    """
    need = [pages_for(l, page_size) for l in lens_alloc]
    total = int(sum(need)) + int(spare_pages)
    ids = rng.permutation(total).astype(np.int32) if shuffled else np.arange(total, dtype=np.int32)
    max_pages = max(1, max(need) if need else 1)
    pt = np.full((len(need), max_pages), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(need):
        pt[b, :n] = ids[cur:cur + n]
        cur += n
    return pt, total


def empty_pool(num_pages: int, shape: Shape, dtype: str) -> np.ndarray:
    rows = sentinel_rows(1, shape.width, dtype)[0]
    pool = np.empty((num_pages, shape.page_size, shape.width),
                    dtype=np.uint16 if dtype == "bf16" else np.float32)
    pool[...] = rows
    return pool


def scatter_rows(pool: np.ndarray, pt_row: np.ndarray, rows: np.ndarray, start: int = 0):
    """Place `rows` (token order, starting at position `start`) into the pages of one sequence."""
    ps = pool.shape[1]
    t = start
    i = 0
    n = rows.shape[0]
    while i < n:
        page = int(pt_row[t // ps])
        off = t % ps
        k = min(ps - off, n - i)
        pool[page, off:off + k] = rows[i:i + k]
        i += k
        t += k


def gather_rows(pool: np.ndarray, pt_row: np.ndarray, length: int) -> np.ndarray:
    """Rows of positions [0, length) of one sequence, in token order (a copy)."""
    ps = pool.shape[1]
    out = np.empty((length, pool.shape[2]), dtype=pool.dtype)
    for p in range(pages_for(length, ps)):
        lo = p * ps
        hi = min(length, lo + ps)
        out[lo:hi] = pool[int(pt_row[p]), :hi - lo]
    return out


# --------------------------------------------------------------------------------------
# per-workload generators
# --------------------------------------------------------------------------------------

def draw_lens(w: Workload, rng) -> np.ndarray:
    if w.lens:
        return np.asarray(w.lens, dtype=np.int32)
    lo, hi = w.len_range
    return rng.integers(lo, hi, size=w.batch, endpoint=True).astype(np.int32)


def make_decode_case(shape: Shape, dtype: str, lens, seed: int, *, spare_pages: int = 8,
                     shuffled: bool = True, append: bool = False) -> dict:
    """A decode problem over a paged latent cache.

    Draw order (PCG64, `seed`): page table, cache rows per sequence, q_nope, q_rope,
    W_UK, W_UV, W_O, q_cat, then (append only) x, W_DKV, W_KR.

    With `append`, `lens` are the lengths BEFORE the append; one new token per sequence
    goes to position lens[b]; the returned `seq_lens` already include it.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = int(lens.shape[0])
    final = lens + (1 if append else 0)
    pt, num_pages = make_page_table(rng, final, shape.page_size, spare_pages, shuffled)
    pool = empty_pool(num_pages, shape, dtype)
    for b in range(B):
        rows = quantise(normal(rng, (int(lens[b]), shape.width)), dtype)
        scatter_rows(pool, pt[b], rows)
    H, dh, dr, dc = shape.n_heads, shape.d_nope, shape.d_rope, shape.d_latent
    case = dict(
        shape=shape, dtype=dtype, pool=pool, page_table=pt, num_pages=num_pages,
        seq_lens=final.astype(np.int32), pos=(final - 1).astype(np.int32),
        q_nope=quantise(normal(rng, (B, H, dh)), dtype),
        q_rope=quantise(normal(rng, (B, H, dr)), dtype),
        w_uk=weight(rng, dc, H * dh, dtype),
        w_uv=weight(rng, dc, H * dh, dtype),
        w_o=weight(rng, H * dh, shape.d_model, dtype),
    )
    # synthetic absorbed queries for checking the attention kernel on its own: latent part
    # N(0, d_h/d_c) (the spread of q_nope @ W_UK^T), RoPE part N(0, 1)
    qc = normal(rng, (B, H, shape.width))
    qc[..., :dc] *= np.float32(np.sqrt(dh / dc))
    case["q_cat"] = quantise(qc, dtype)
    if append:
        case.update(
            x=quantise(normal(rng, (B, shape.d_model)), dtype),
            w_dkv=weight(rng, shape.d_model, dc, dtype),
            w_kr=weight(rng, shape.d_model, dr, dtype),
            append_seq=np.arange(B, dtype=np.int32),
            append_pos=lens.astype(np.int32),
        )
    return case


# MX caches (low-precision latent cache): synthetic codes and scale bytes, drawn directly.
# E4M3 codes come from torch's float32 -> float8_e4m3fn cast of N(0,1) * 128 clipped to the
# format's range (a storage cast, like the bf16 rounding above); E2M1 codes are uniform
# nibbles; block scale bytes are uniform over a narrow band, so that the dequantised rows have
# the spread of N(0,1) latents.  Slots that no token owns hold NaN codes (E4M3) or 0xFF bytes
# and NaN scale bytes: an MX cache reader must never let them reach a result.
MX_FMTS = {"mxfp8": 1, "mxfp4": 2}


def mx_codes(rng, n_rows: int, width: int, fmt: str) -> np.ndarray:
    if fmt == "mxfp8":
        import torch
        v = np.clip(normal(rng, (n_rows, width)) * np.float32(128.0), -448.0, 448.0).astype(np.float32)
        return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return rng.integers(0, 256, size=(n_rows, width // 2), dtype=np.uint8)


def mx_scale_bytes(rng, n_rows: int, width: int, fmt: str) -> np.ndarray:
    lo, hi = (119, 121) if fmt == "mxfp8" else (125, 127)
    return rng.integers(lo, hi, size=(n_rows, width // 32), endpoint=True).astype(np.uint8)


def make_mx_decode_case(shape: Shape, fmt: str, lens, seed: int, *, spare_pages: int = 8,
                        shuffled: bool = True, append: bool = False) -> dict:
    """A decode problem over an MX-encoded paged cache (fmt "mxfp8" or "mxfp4").

    Draw order (PCG64, `seed`): page table, then per sequence its codes and scale bytes, then
    q_cat, q_nope, q_rope, W_UK, W_UV, W_O, then (append only) x, W_DKV, W_KR.  Queries and
    weights are bf16 bits.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = int(lens.shape[0])
    final = lens + (1 if append else 0)
    pt, num_pages = make_page_table(rng, final, shape.page_size, spare_pages, shuffled)
    W, ps = shape.width, shape.page_size
    row_bytes = W if fmt == "mxfp8" else W // 2
    codes = np.full((num_pages, ps, row_bytes), 0x7F if fmt == "mxfp8" else 0xFF, dtype=np.uint8)
    scales = np.full((num_pages, ps, W // 32), 0xFF, dtype=np.uint8)
    for b in range(B):
        n = int(lens[b])
        scatter_rows(codes, pt[b], mx_codes(rng, n, W, fmt))
        scatter_rows(scales, pt[b], mx_scale_bytes(rng, n, W, fmt))
    H, dc = shape.n_heads, shape.d_latent
    qc = normal(rng, (B, H, W))
    qc[..., :dc] *= np.float32(np.sqrt(shape.d_nope / dc))
    case = dict(shape=shape, dtype="bf16", kv=fmt, codes=codes, scales=scales, page_table=pt,
                num_pages=num_pages, seq_lens=final.astype(np.int32), pos=(final - 1).astype(np.int32),
                q_cat=quantise(qc, "bf16"))
    case.update(
        q_nope=quantise(normal(rng, (B, H, shape.d_nope)), "bf16"),
        q_rope=quantise(normal(rng, (B, H, shape.d_rope)), "bf16"),
        w_uk=weight(rng, dc, H * shape.d_nope, "bf16"),
        w_uv=weight(rng, dc, H * shape.d_nope, "bf16"),
        w_o=weight(rng, H * shape.d_nope, shape.d_model, "bf16"),
    )
    if append:
        case.update(
            x=quantise(normal(rng, (B, shape.d_model)), "bf16"),
            w_dkv=weight(rng, shape.d_model, dc, "bf16"),
            w_kr=weight(rng, shape.d_model, shape.d_rope, "bf16"),
            append_seq=np.arange(B, dtype=np.int32),
            append_pos=lens.astype(np.int32),
        )
    return case


def make_prefill_case(shape: Shape, dtype: str, T: int, seed: int, *, spare_pages: int = 8,
                      shuffled: bool = True) -> dict:
    """Causal prefill of one sequence of T tokens that first builds its cache from x.

    Draw order: page table, x, W_DKV, W_KR, q_nope, q_rope, W_UK, W_UV, W_O.
    """
    rng = np.random.default_rng(seed)
    pt, num_pages = make_page_table(rng, [T], shape.page_size, spare_pages, shuffled)
    H, dh, dr, dc = shape.n_heads, shape.d_nope, shape.d_rope, shape.d_latent
    return dict(
        shape=shape, dtype=dtype, pool=empty_pool(num_pages, shape, dtype), page_table=pt,
        num_pages=num_pages, T=T,
        x=quantise(normal(rng, (T, shape.d_model)), dtype),
        w_dkv=weight(rng, shape.d_model, dc, dtype),
        w_kr=weight(rng, shape.d_model, dr, dtype),
        q_nope=quantise(normal(rng, (T, H, dh)), dtype),
        q_rope=quantise(normal(rng, (T, H, dr)), dtype),
        w_uk=weight(rng, dc, H * dh, dtype),
        w_uv=weight(rng, dc, H * dh, dtype),
        w_o=weight(rng, H * dh, shape.d_model, dtype),
        append_seq=np.zeros(T, dtype=np.int32),
        append_pos=np.arange(T, dtype=np.int32),
        seq_lens=np.array([T], dtype=np.int32),
    )


def make_tiny_case(shape: Shape = TINY, T: int = 64, seed: int = 0) -> dict:
    """Tiny fp32 problem: the cache is built from x[0..T) and the query is token T-1.

    Draw order: x, W_DKV, W_KR, W_Q, W_QR, W_UK, W_UV, W_O.  Contiguous pages.
    """
    rng = np.random.default_rng(seed)
    H, dh, dr, dc, dm = shape.n_heads, shape.d_nope, shape.d_rope, shape.d_latent, shape.d_model
    pt, num_pages = make_page_table(rng, [T], shape.page_size, 0, False)
    return dict(
        shape=shape, dtype="f32", pool=empty_pool(num_pages, shape, "f32"), page_table=pt,
        num_pages=num_pages, T=T,
        x=quantise(normal(rng, (T, dm)), "f32"),
        w_dkv=weight(rng, dm, dc, "f32"),
        w_kr=weight(rng, dm, dr, "f32"),
        w_q=weight(rng, dm, H * dh, "f32"),
        w_qr=weight(rng, dm, H * dr, "f32"),
        w_uk=weight(rng, dc, H * dh, "f32"),
        w_uv=weight(rng, dc, H * dh, "f32"),
        w_o=weight(rng, H * dh, dm, "f32"),
        append_seq=np.zeros(T, dtype=np.int32),
        append_pos=np.arange(T, dtype=np.int32),
        seq_lens=np.array([T], dtype=np.int32),
        pos=np.array([T - 1], dtype=np.int32),
    )


def make_workload(name: str) -> dict:
    """Full-size inputs of one named workload."""
    w = WORKLOADS[name]
    if w.mode == "tiny_decode":
        return make_tiny_case(w.shape, w.tokens, w.seed)
    if w.mode == "prefill":
        return make_prefill_case(w.shape, w.dtype, w.tokens, w.seed, spare_pages=w.spare_pages,
                                 shuffled=w.shuffled)
    rng = np.random.default_rng(w.seed)
    lens = draw_lens(w, rng)
    if w.kv:
        return make_mx_decode_case(w.shape, w.kv, lens, w.seed + 1000, spare_pages=w.spare_pages,
                                   shuffled=w.shuffled, append=(w.mode == "append_decode"))
    return make_decode_case(w.shape, w.dtype, lens, w.seed + 1000, spare_pages=w.spare_pages,
                            shuffled=w.shuffled, append=(w.mode == "append_decode"))


def replace_shape(shape: Shape, **kw) -> Shape:
    return dataclasses.replace(shape, **kw)


def to_device(a: np.ndarray, dtype: str, device="cuda"):
    """Copy a stored array to a torch device tensor of the storage type (bf16 bits -> bfloat16)."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_device(t) -> np.ndarray:
    """Device tensor -> numpy float64 (bf16 widened exactly)."""
    import torch
    return t.detach().to("cpu", torch.float64).numpy()
