"""MLA latent-KV hot path on B300: torch-facing binding of libmla.so.

Each function marshals torch tensors into the C ABI of include/mla.h and calls the
entry point of the same name; every step of the computation runs in libmla's CUDA kernels.
PyTorch provides device memory and streams only.  Outputs that the caller does not pass are
allocated here with torch (the library itself never allocates).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import MLAError, MLA_F32, MLA_BF16, MLA_KV_PLAIN, MLA_KV_MXFP8, MLA_KV_MXFP4  # noqa: F401

__all__ = ["MLAConfig", "PagedCache", "mla_cache_append", "mla_absorb_q", "mla_workspace_size",
           "mla_decode", "mla_decode_static", "mla_prefill", "mla_prefill_unabsorbed", "mla_out", "mla_out_proj",
           "mla_query_proj", "mla_query_latent", "mla_query_up", "mla_fold_uq_uk", "mla_absorb_q_compressed",
           "mla_get_device_error",
           "mla_set_tuning",
           "mla_last_attention_path", "MLAError", "lib"]


def lib():
    return _lib.load()


_TORCH_DTYPE = {MLA_F32: torch.float32, MLA_BF16: torch.bfloat16}


@dataclass
class MLAConfig:
    n_heads: int
    d_nope: int
    d_rope: int
    d_latent: int
    d_model: int
    page_size: int = 64
    rope_base: float = 10000.0
    softmax_scale: float = 0.0
    dtype: int = MLA_BF16

    @property
    def width(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def torch_dtype(self):
        return _TORCH_DTYPE[self.dtype]

    def c(self) -> _lib.MlaConfig:
        return _lib.MlaConfig(self.n_heads, self.d_nope, self.d_rope, self.d_latent, self.d_model,
                              self.page_size, self.rope_base, self.softmax_scale, self.dtype)

    @staticmethod
    def from_shape(shape, dtype: str) -> "MLAConfig":
        return MLAConfig(shape.n_heads, shape.d_nope, shape.d_rope, shape.d_latent, shape.d_model,
                         shape.page_size, shape.rope_base, 0.0, MLA_BF16 if dtype == "bf16" else MLA_F32)


@dataclass
class PagedCache:
    """Caller-owned paged latent cache: pool [num_pages, P, W], page_table [B, max_pages]
    int32, seq_lens [B] int32 (all device tensors).  An MX cache (kv_format MLA_KV_MXFP8 or
    MLA_KV_MXFP4) holds uint8 codes in `pool` ([num_pages, P, W] or [num_pages, P, W/2]) and
    the block scale bytes in `kv_scales` ([num_pages, P, W/32] uint8)."""
    pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    kv_format: int = MLA_KV_PLAIN
    kv_scales: torch.Tensor = None

    def c(self) -> _lib.MlaCache:
        return _lib.MlaCache(self.pool.data_ptr(), self.pool.shape[0], self.page_table.data_ptr(),
                             self.page_table.shape[1], self.page_table.shape[0],
                             self.seq_lens.data_ptr(), self.kv_format, _ptr(self.kv_scales))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def mla_cache_append(cfg: MLAConfig, cache: PagedCache, x, w_dkv, w_kr, seq_idx, pos, stream=None):
    n = x.shape[0]
    st = lib().mla_cache_append(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(x), _ptr(w_dkv),
                                _ptr(w_kr), _ptr(seq_idx), _ptr(pos), n, _stream(stream))
    _lib.check(st, "mla_cache_append")


def mla_absorb_q(cfg: MLAConfig, q_nope, q_rope, pos, w_uk, q_cat=None, stream=None):
    n = q_nope.shape[0]
    if q_cat is None:
        q_cat = torch.empty((n, cfg.n_heads, cfg.width), dtype=cfg.torch_dtype, device=q_nope.device)
    st = lib().mla_absorb_q(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(pos), _ptr(w_uk),
                            _ptr(q_cat), n, _stream(stream))
    _lib.check(st, "mla_absorb_q")
    return q_cat


def mla_workspace_size(cfg: MLAConfig) -> int:
    b = ctypes.c_size_t(0)
    _lib.check(lib().mla_workspace_size(ctypes.byref(cfg.c()), ctypes.byref(b)), "mla_workspace_size")
    return int(b.value)


def alloc_workspace(cfg: MLAConfig, device="cuda") -> torch.Tensor:
    return torch.empty(mla_workspace_size(cfg), dtype=torch.uint8, device=device)


def mla_decode(cfg: MLAConfig, cache: PagedCache, q_cat, o_lat=None, lse=None, workspace=None,
               stream=None):
    B = cache.page_table.shape[0]
    dev = q_cat.device
    if o_lat is None:
        o_lat = torch.empty((B, cfg.n_heads, cfg.d_latent), dtype=cfg.torch_dtype, device=dev)
    if lse is None:
        lse = torch.empty((B, cfg.n_heads), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(cfg, dev)
    st = lib().mla_decode(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(q_cat), _ptr(o_lat),
                          _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "mla_decode")
    return o_lat, lse


def mla_decode_static(cfg: MLAConfig, cache: PagedCache, q_cat, o_lat, lse, stream=None):
    """mla_decode without a workspace: the library keeps the split partials in a fixed device
    array of MLA_STATIC_SCRATCH_BYTES, so nothing is allocated here or in the call; the
    outputs are the caller's.  Calls that overlap in time race on that array."""
    st = lib().mla_decode_static(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(q_cat),
                                 _ptr(o_lat), _ptr(lse), _stream(stream))
    _lib.check(st, "mla_decode_static")
    return o_lat, lse


def mla_prefill(cfg: MLAConfig, cache: PagedCache, seq: int, q_start: int, q_cat, o_lat=None,
                lse=None, workspace=None, stream=None):
    T = q_cat.shape[0]
    dev = q_cat.device
    if o_lat is None:
        o_lat = torch.empty((T, cfg.n_heads, cfg.d_latent), dtype=cfg.torch_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(cfg, dev)
    st = lib().mla_prefill(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), seq, q_start, T,
                           _ptr(q_cat), _ptr(o_lat), _ptr(lse), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _lib.check(st, "mla_prefill")
    return o_lat, lse


def mla_prefill_unabsorbed(cfg: MLAConfig, cache: PagedCache, seq: int, q_start: int, q_nope, q_rope, w_uk, w_uv,
                           o=None, lse=None, workspace=None, stream=None):
    """Causal prefill in the un-absorbed form (restore K and V, 192-wide scores); returns (o, lse)
    with o [T, n_h * d_h], the output mla_prefill + mla_out would give."""
    T = q_nope.shape[0]
    dev = q_nope.device
    if o is None:
        o = torch.empty((T, cfg.n_heads * cfg.d_nope), dtype=cfg.torch_dtype, device=dev)
    if lse is None:
        lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=dev)
    if workspace is None:
        b = ctypes.c_size_t(0)
        _lib.check(lib().mla_prefill_unabsorbed_workspace_size(ctypes.byref(cfg.c()), q_start, T, ctypes.byref(b)),
                   "mla_prefill_unabsorbed_workspace_size")
        workspace = torch.empty(int(b.value), dtype=torch.uint8, device=dev)
    st = lib().mla_prefill_unabsorbed(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), seq, q_start, T, _ptr(q_nope),
                                      _ptr(q_rope), _ptr(w_uk), _ptr(w_uv), _ptr(o), _ptr(lse), _ptr(workspace),
                                      workspace.numel(), _stream(stream))
    _lib.check(st, "mla_prefill_unabsorbed")
    return o, lse


def mla_out(cfg: MLAConfig, o_lat, w_uv, o=None, stream=None):
    n = o_lat.shape[0]
    if o is None:
        o = torch.empty((n, cfg.n_heads * cfg.d_nope), dtype=cfg.torch_dtype, device=o_lat.device)
    st = lib().mla_out(ctypes.byref(cfg.c()), _ptr(o_lat), _ptr(w_uv), _ptr(o), n, _stream(stream))
    _lib.check(st, "mla_out")
    return o


def mla_query_proj(cfg: MLAConfig, x, w_q, w_qr, q_nope=None, q_rope=None, stream=None):
    n = x.shape[0]
    if q_nope is None:
        q_nope = torch.empty((n, cfg.n_heads, cfg.d_nope), dtype=cfg.torch_dtype, device=x.device)
    if q_rope is None:
        q_rope = torch.empty((n, cfg.n_heads, cfg.d_rope), dtype=cfg.torch_dtype, device=x.device)
    st = lib().mla_query_proj(ctypes.byref(cfg.c()), _ptr(x), _ptr(w_q), _ptr(w_qr), _ptr(q_nope), _ptr(q_rope), n,
                              _stream(stream))
    _lib.check(st, "mla_query_proj")
    return q_nope, q_rope


def mla_query_latent(cfg: MLAConfig, x, w_dq, c_q=None, stream=None):
    """c_q = x . W_DQ; d_cq is W_DQ's column count."""
    n, d_cq = x.shape[0], w_dq.shape[1]
    if c_q is None:
        c_q = torch.empty((n, d_cq), dtype=cfg.torch_dtype, device=x.device)
    _lib.check(lib().mla_query_latent(ctypes.byref(cfg.c()), d_cq, _ptr(x), _ptr(w_dq), _ptr(c_q), n, _stream(stream)),
               "mla_query_latent")
    return c_q


def mla_query_up(cfg: MLAConfig, c_q, w_uq=None, w_qr=None, q_nope=None, q_rope=None, stream=None):
    """q_nope = c_q . W_UQ (when w_uq is given) and q_rope = c_q . W_QR (when w_qr is given)."""
    n, d_cq = c_q.shape
    if w_uq is not None and q_nope is None:
        q_nope = torch.empty((n, cfg.n_heads, cfg.d_nope), dtype=cfg.torch_dtype, device=c_q.device)
    if w_qr is not None and q_rope is None:
        q_rope = torch.empty((n, cfg.n_heads, cfg.d_rope), dtype=cfg.torch_dtype, device=c_q.device)
    st = lib().mla_query_up(ctypes.byref(cfg.c()), d_cq, _ptr(c_q), _ptr(w_uq), _ptr(w_qr),
                            _ptr(q_nope) if w_uq is not None else 0, _ptr(q_rope) if w_qr is not None else 0, n,
                            _stream(stream))
    _lib.check(st, "mla_query_up")
    return q_nope, q_rope


def mla_fold_uq_uk(cfg: MLAConfig, w_uq, w_uk, w_uqk=None, stream=None):
    """W_UQ folded into W_UK: [d_cq, n_h * d_c], head h in column block h."""
    d_cq = w_uq.shape[0]
    if w_uqk is None:
        w_uqk = torch.empty((d_cq, cfg.n_heads * cfg.d_latent), dtype=cfg.torch_dtype, device=w_uq.device)
    _lib.check(lib().mla_fold_uq_uk(ctypes.byref(cfg.c()), d_cq, _ptr(w_uq), _ptr(w_uk), _ptr(w_uqk), _stream(stream)),
               "mla_fold_uq_uk")
    return w_uqk


def mla_absorb_q_compressed(cfg: MLAConfig, c_q, q_rope, pos, w_uqk, q_cat=None, stream=None):
    n, d_cq = c_q.shape
    if q_cat is None:
        q_cat = torch.empty((n, cfg.n_heads, cfg.width), dtype=cfg.torch_dtype, device=c_q.device)
    st = lib().mla_absorb_q_compressed(ctypes.byref(cfg.c()), d_cq, _ptr(c_q), _ptr(q_rope), _ptr(pos), _ptr(w_uqk),
                                       _ptr(q_cat), n, _stream(stream))
    _lib.check(st, "mla_absorb_q_compressed")
    return q_cat


def mla_out_proj(cfg: MLAConfig, o, w_o, out=None, stream=None):
    n = o.shape[0]
    if out is None:
        out = torch.empty((n, cfg.d_model), dtype=cfg.torch_dtype, device=o.device)
    st = lib().mla_out_proj(ctypes.byref(cfg.c()), _ptr(o), _ptr(w_o), _ptr(out), n, _stream(stream))
    _lib.check(st, "mla_out_proj")
    return out


def mla_get_device_error(stream=None) -> int:
    return int(lib().mla_get_device_error(_stream(stream)))


def mla_set_tuning(key: int, value: int) -> int:
    return int(lib().mla_set_tuning(key, value))


def mla_last_attention_path() -> int:
    return int(lib().mla_last_attention_path())
