"""CPU tests of the C-ABI boundary: libmla.so loads, exports every entry point that
include/mla.h declares, and its host-side checks reject bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from mla_latent_kv_79_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_79_b300 import build
    build.build()
    return _lib.load()


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for name in ("mla_cache_append", "mla_absorb_q", "mla_decode", "mla_prefill", "mla_out",
                 "mla_out_proj", "mla_query_proj", "mla_workspace_size", "mla_get_device_error",
                 "mla_status_string"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(_lib.SIGNATURES), "binding and header disagree"


def test_nothing_else_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("mla_")}
    assert exported == set(declared_symbols())


def test_version_and_strings(lib):
    assert lib.mla_abi_version() == 2
    for code in range(8):
        assert lib.mla_status_string(code)
    assert lib.mla_status_string(99) == b"unknown status"


def test_tuning_knobs_roundtrip(lib):
    old = lib.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, 7)
    assert lib.mla_set_tuning(_lib.MLA_TUNE_ATTN_UNITS, old) == 7
    assert lib.mla_set_tuning(99, 1) == -1


def _cfg(**kw):
    base = dict(n_heads=128, d_nope=128, d_rope=64, d_latent=512, d_model=5120, page_size=64,
                rope_base=10000.0, softmax_scale=0.0, dtype=_lib.MLA_BF16)
    base.update(kw)
    return _lib.MlaConfig(**base)


@pytest.mark.parametrize("bad", [dict(n_heads=0), dict(d_rope=63), dict(d_latent=-2),
                                 dict(page_size=0), dict(dtype=7), dict(rope_base=0.0),
                                 dict(softmax_scale=-1.0)])
def test_bad_config_rejected_on_host(lib, bad):
    cfg = _cfg(**bad)
    st = lib.mla_absorb_q(ctypes.byref(cfg), 16, 16, 16, 16, 16, 1, None)
    assert st == 1  # MLA_ERR_INVALID_ARG


def test_unsupported_row_width(lib):
    # bf16 rows of 600 + 6 = 606 numbers are not 16-byte multiples
    cfg = _cfg(d_latent=600, d_rope=6)
    assert lib.mla_absorb_q(ctypes.byref(cfg), 16, 16, 16, 16, 16, 1, None) == 2


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = _cfg()
    assert lib.mla_absorb_q(ctypes.byref(cfg), None, 16, 16, 16, 16, 1, None) == 1
    assert lib.mla_absorb_q(ctypes.byref(cfg), 18, 16, 16, 16, 16, 1, None) == 1
    assert lib.mla_out(ctypes.byref(cfg), 16, 16, 8, 1, None) == 1
    cache = _lib.MlaCache(0, 10, 16, 4, 2, 16)
    assert lib.mla_cache_append(ctypes.byref(cfg), ctypes.byref(cache), 16, 16, 16, 16, 16, 1, None) == 1
    cache = _lib.MlaCache(16, 10, 16, 4, 2, 16)
    assert lib.mla_prefill(ctypes.byref(cfg), ctypes.byref(cache), 5, 0, 1, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mla_prefill(ctypes.byref(cfg), ctypes.byref(cache), 0, 250, 10, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mla_decode(ctypes.byref(cfg), None, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mla_out_proj(ctypes.byref(cfg), None, 16, 16, 1, None) == 1
    assert lib.mla_out_proj(ctypes.byref(cfg), 16, 24, 16, 1, None) == 1
    assert lib.mla_query_proj(ctypes.byref(cfg), 16, 16, None, 16, 16, 1, None) == 1
    assert lib.mla_query_proj(ctypes.byref(cfg), 16, 16, 16, 16, 40, 1, None) == 1
    assert lib.mla_out_proj(ctypes.byref(cfg), 16, 16, 16, -1, None) == 1


def test_mx_cache_checked_on_host(lib):
    """An MX cache needs a known format, a 16-byte aligned scale array and rows of whole
    32-element blocks; each failure is reported before anything touches a GPU."""
    cfg = _cfg()
    args = (5, 0, 1, 16, 16, 16, 16, 1 << 30, None)   # seq 5 >= batch 2: rejected last
    ok = _lib.MlaCache(16, 10, 16, 4, 2, 16, _lib.MLA_KV_MXFP8, 32)
    assert lib.mla_prefill(ctypes.byref(cfg), ctypes.byref(ok), *args) == 1
    for fmt, scales, want in ((7, 32, 1), (_lib.MLA_KV_MXFP4, 0, 1), (_lib.MLA_KV_MXFP8, 40, 1)):
        cache = _lib.MlaCache(16, 10, 16, 4, 2, 16, fmt, scales)
        assert lib.mla_prefill(ctypes.byref(cfg), ctypes.byref(cache), 0, 0, 1, 16, 16, 16, 16, 1 << 30,
                               None) == want
    # W = 512 + 48 = 560 is not a multiple of 32
    cfg = _cfg(d_rope=48)
    assert lib.mla_prefill(ctypes.byref(cfg), ctypes.byref(ok), 0, 0, 1, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mla_cache_append(ctypes.byref(cfg), ctypes.byref(ok), 16, 16, 16, 16, 16, 1, None) == 2
    # a plain cache ignores kv_scales
    plain = _lib.MlaCache(16, 10, 16, 4, 2, 16, _lib.MLA_KV_PLAIN, 0)
    assert lib.mla_prefill(ctypes.byref(_cfg()), ctypes.byref(plain), *args) == 1


def test_unabsorbed_prefill_checked_on_host(lib):
    """Workspace size is the sum of its 256-byte-aligned parts; bad shapes, positions, pointers and
    workspaces are rejected before anything touches a GPU."""
    cfg = _cfg()
    b = ctypes.c_size_t(0)
    assert lib.mla_prefill_unabsorbed_workspace_size(ctypes.byref(cfg), 100, 28, ctypes.byref(b)) == 0
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    L, T = 128, 28
    assert b.value == al(L * 576 * 2) + 2 * al(L * 128 * 128 * 2) + al(T * 128 * 192 * 2)
    assert lib.mla_prefill_unabsorbed_workspace_size(ctypes.byref(cfg), -1, 28, ctypes.byref(b)) == 1
    cache = _lib.MlaCache(16, 10, 16, 4, 2, 16, 0, 0)
    args = lambda seq, q0, n: (ctypes.byref(cfg), ctypes.byref(cache), seq, q0, n, 16, 16, 16, 16, 16, 16,  # noqa: E731
                               256, 1 << 30, None)
    assert lib.mla_prefill_unabsorbed(*args(2, 0, 1)) == 1       # seq outside the batch
    assert lib.mla_prefill_unabsorbed(*args(0, 250, 10)) == 1    # past the page table (4 pages of 64)
    assert lib.mla_prefill_unabsorbed(*args(0, 0, 0)) == 0       # no queries: a no-op
    bad = (ctypes.byref(cfg), ctypes.byref(cache), 0, 0, 1, 16, 16, 16, 24, 16, 16, 256, 1 << 30, None)
    assert lib.mla_prefill_unabsorbed(*bad) == 1                 # misaligned w_uv


def test_zero_tokens_is_a_noop(lib):
    cfg = _cfg()
    assert lib.mla_absorb_q(ctypes.byref(cfg), None, None, None, None, None, 0, None) == 0
    assert lib.mla_out(ctypes.byref(cfg), None, None, None, 0, None) == 0
    assert lib.mla_out_proj(ctypes.byref(cfg), None, None, None, 0, None) == 0
    assert lib.mla_query_proj(ctypes.byref(cfg), None, None, None, None, None, 0, None) == 0


def test_projection_rows_must_be_16_byte_multiples(lib):
    # bf16 rows of d_model = 36 elements are 72 bytes: not a multiple of 16
    cfg = _cfg(d_model=36)
    assert lib.mla_out_proj(ctypes.byref(cfg), 16, 16, 16, 1, None) == 2
    assert lib.mla_query_proj(ctypes.byref(cfg), 16, 16, 16, 16, 16, 1, None) == 2


def test_binding_fails_loudly_without_library(tmp_path):
    saved = _lib._lib
    try:
        _lib._lib = None
        with pytest.raises(RuntimeError):
            _lib.load(str(tmp_path / "missing.so"))
    finally:
        _lib._lib = saved
