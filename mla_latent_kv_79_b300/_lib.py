"""ctypes view of libmla.so (include/mla.h).  Loading never falls back to anything else:
a missing or unloadable library raises."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla.so")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
                4: "MLA_ERR_WORKSPACE", 5: "MLA_ERR_DEVICE_TIMEOUT", 6: "MLA_ERR_DEVICE_BOUNDS",
                7: "MLA_ERR_SCRATCH_LIMIT"}
MLA_ERR_SCRATCH_LIMIT = 7
MLA_STATIC_SCRATCH_BYTES = 80 << 20
MLA_F32, MLA_BF16 = 0, 1
MLA_TUNE_ATTN_UNITS, MLA_TUNE_FORCE_SIMT, MLA_TUNE_WAIT_LIMIT_US = 0, 1, 2
MLA_TUNE_GEMM_HEADS, MLA_TUNE_GEMM_STAGES, MLA_TUNE_NO_PDL, MLA_TUNE_SCHEDULE = 3, 4, 5, 6
MLA_TUNE_GEMM_KSPLIT = 7
MLA_KV_PLAIN, MLA_KV_MXFP8, MLA_KV_MXFP4 = 0, 1, 2


class MlaConfig(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("d_nope", ctypes.c_int32), ("d_rope", ctypes.c_int32),
                ("d_latent", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class MlaCache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("seq_lens", ctypes.c_void_p),
                ("kv_format", ctypes.c_int32), ("kv_scales", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_CFG = ctypes.POINTER(MlaConfig)
_CACHE = ctypes.POINTER(MlaCache)

# name -> (restype, argtypes); every entry point declared in include/mla.h
SIGNATURES = {
    "mla_abi_version": (_I, []),
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_cache_append": (_I, [_CFG, _CACHE, _P, _P, _P, _P, _P, _I, _P]),
    "mla_absorb_q": (_I, [_CFG, _P, _P, _P, _P, _P, _I, _P]),
    "mla_workspace_size": (_I, [_CFG, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_decode": (_I, [_CFG, _CACHE, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_decode_static": (_I, [_CFG, _CACHE, _P, _P, _P, _P]),
    "mla_prefill": (_I, [_CFG, _CACHE, _I, _I, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_prefill_unabsorbed_workspace_size": (_I, [_CFG, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_prefill_unabsorbed": (_I, [_CFG, _CACHE, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "mla_query_latent": (_I, [_CFG, _I, _P, _P, _P, _I, _P]),
    "mla_query_up": (_I, [_CFG, _I, _P, _P, _P, _P, _P, _I, _P]),
    "mla_fold_uq_uk": (_I, [_CFG, _I, _P, _P, _P, _P]),
    "mla_absorb_q_compressed": (_I, [_CFG, _I, _P, _P, _P, _P, _P, _I, _P]),
    "mla_out": (_I, [_CFG, _P, _P, _P, _I, _P]),
    "mla_out_proj": (_I, [_CFG, _P, _P, _P, _I, _P]),
    "mla_query_proj": (_I, [_CFG, _P, _P, _P, _P, _P, _I, _P]),
    "mla_get_device_error": (_I, [_P]),
    "mla_set_tuning": (_I, [_I, _I]),
    "mla_last_attention_path": (_I, []),
    "mla_set_attention_events": (None, [_P, _P]),
    "mla_kernel_launches": (ctypes.c_uint64, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmla.so once; raise if it is absent (build it with mla_latent_kv_79_b300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmla.so not built at {path}; run `python -m mla_latent_kv_79_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def check(status: int, what: str):
    if status != MLA_OK:
        raise MLAError(status, what)
