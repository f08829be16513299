"""ctypes loader for libmsa_gb300.so (the C ABI declared in include/msa.h).

The library is built in-tree by ``build.py``. Loading fails loudly when it is missing:
there is no fallback implementation of any step.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

MSA_OK = 0
ERRORS = {-1: "MSA_ERR_ARG", -2: "MSA_ERR_SHAPE", -3: "MSA_ERR_UNSUPPORTED",
          -4: "MSA_ERR_WORKSPACE", -5: "MSA_ERR_CUDA", -6: "MSA_ERR_DEVICE"}

# (name, restype, argtypes) for every entry point of include/msa.h
P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = [
    ("msa_index_score_topk_workspace_size", SZ, [I32, I32, I32, I32]),
    ("msa_index_score_topk", ctypes.c_int,
     [P, P, P, P, I32, I32, I32, I32, I32, I64, I32, P, P, P, SZ, P]),
    ("msa_index_score_topk_page_table", ctypes.c_int,
     [P, P, P, P, I32, I32, I32, I32, I32, I64, I32, P, P, P, P, P, SZ, P]),
    ("msa_index_score_topk_noalloc", ctypes.c_int,
     [P, P, P, P, I32, I32, I32, I32, I32, I64, I32, P, P, P]),
    ("msa_build_sparse_page_table", ctypes.c_int, [P, P, P, I32, I32, I32, I32, I32, I64, P, P, P]),
    ("msa_stage_selected_kv", ctypes.c_int, [P, P, I64, P, I32, I32, I32, I32, P, P, P, P]),
    ("msa_paged_sparse_decode_workspace_size", SZ, [I32, I32, I32, I32]),
    ("msa_paged_sparse_decode", ctypes.c_int,
     [P, P, P, P, P, I32, I32, I32, I32, I32, I64, P, P, P, SZ, P]),
    ("msa_sparse_prefill_workspace_size", SZ, [I32, I64, I32, I32, I32]),
    ("msa_sparse_prefill", ctypes.c_int, [P, P, P, P, I32, I64, I32, I32, I32, I32, P, P, P, SZ, P]),
    ("msa_sparse_prefill_paged", ctypes.c_int,
     [P, P, P, P, I64, P, I32, I64, I32, I32, I32, I32, P, P, P, SZ, P]),
    ("msa_prefill_bucket_workspace_size", SZ, [I32, I32, I32, I32]),
    ("msa_prefill_bucket", ctypes.c_int, [P, I32, I32, I32, I32, P, P, P, SZ, P]),
    ("msa_lse_merge", ctypes.c_int, [P, I32, P, I64, I32, I32, I32, P, P, P]),
    ("msa_last_error", ctypes.c_char_p, []),
    ("msa_device_error", ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    ("msa_version", ctypes.c_char_p, []),
]


class MSAError(RuntimeError):
    def __init__(self, name: str, code: int, msg: str):
        super().__init__(f"{name} failed with {ERRORS.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the C ABI library (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and (not os.path.exists(path) or _build.is_stale()):
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"MSA CUDA library not built ({path} missing); run "
                    "`python -m block_sparse_attention_msa_gb300.build` -- there is no fallback")
            lib = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(name: str, rc: int):
    if rc != MSA_OK:
        msg = load().msa_last_error().decode(errors="replace")
        raise MSAError(name, rc, msg)
