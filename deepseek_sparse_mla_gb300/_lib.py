"""ctypes loader for libdsa.so and the C structs of include/dsa.h.

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA = 0, -1, -2, -3, -4
DSA_ERR_DEVICE_CHECK = -5
STATUS_NAMES = {0: "DSA_OK", -1: "DSA_ERR_INVALID_ARG", -2: "DSA_ERR_UNSUPPORTED", -3: "DSA_ERR_WORKSPACE",
                -4: "DSA_ERR_CUDA", -5: "DSA_ERR_DEVICE_CHECK"}
# device status bits (dsa_read_status)
DEVICE_TMA_TIMEOUT, DEVICE_MMA_TIMEOUT, DEVICE_BAD_PAGE, DEVICE_CONFIG = 0x1, 0x2, 0x4, 0x8
KEY_BF16, KEY_FP8_E4M3, KEY_INT8 = 0, 1, 2
LATENT_BF16, LATENT_E4M3 = 0, 1

# every entry point include/dsa.h declares
EXPORTS = ("dsa_abi_version", "dsa_last_error", "dsa_kernel_launches", "dsa_cache_bytes", "dsa_indexer_workspace_bytes",
           "dsa_mla_workspace_bytes", "dsa_kv_append", "dsa_indexer_scores_topk", "dsa_indexer_scores_topk_static",
           "dsa_indexer_page_workspace_bytes", "dsa_indexer_page_topk", "dsa_sparse_mla_decode", "dsa_sparse_mla_prefill",
           "dsa_dcp_candidates", "dsa_dcp_select", "dsa_dcp_merge", "dsa_sparse_mla_decode_ragged",
           "dsa_kv_append_layers", "dsa_read_status", "dsa_check_device_status", "dsa_sparse_mla_decode_layers")


class DsaCache(ctypes.Structure):
    _fields_ = [("latent", ctypes.c_void_p), ("index_keys", ctypes.c_void_p), ("index_scales", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("key_format", ctypes.c_int32),
                ("latent_format", ctypes.c_int32), ("latent_scales", ctypes.c_void_p)]


class DsaBatch(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("query_start_loc", ctypes.c_void_p), ("num_requests", ctypes.c_int32),
                ("num_rows", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("block_table_stride", ctypes.c_int32)]


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libdsa.so is not built ({path}); run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.dsa_abi_version.restype = I32
    lib.dsa_abi_version.argtypes = []
    lib.dsa_last_error.restype = ctypes.c_char_p
    lib.dsa_last_error.argtypes = []
    lib.dsa_kernel_launches.restype = ctypes.c_uint64
    lib.dsa_kernel_launches.argtypes = []
    lib.dsa_read_status.restype = I32
    lib.dsa_read_status.argtypes = [P, P, P]
    lib.dsa_check_device_status.restype = I32
    lib.dsa_check_device_status.argtypes = [ctypes.c_uint32]
    lib.dsa_cache_bytes.restype = SZ
    lib.dsa_cache_bytes.argtypes = [I32, I32, I32, I32, I32]
    lib.dsa_indexer_workspace_bytes.restype = SZ
    lib.dsa_indexer_workspace_bytes.argtypes = [I32, I32, I32]
    lib.dsa_mla_workspace_bytes.restype = SZ
    lib.dsa_mla_workspace_bytes.argtypes = [I32, I32]
    lib.dsa_kv_append.restype = I32
    lib.dsa_kv_append.argtypes = [ctypes.POINTER(DsaCache), P, P, P, I32, P, P, I32, P]
    lib.dsa_indexer_scores_topk.restype = I32
    lib.dsa_indexer_scores_topk.argtypes = [ctypes.POINTER(DsaCache), ctypes.POINTER(DsaBatch), P, P, I32, P, P, P,
                                            SZ, P]
    lib.dsa_indexer_scores_topk_static.restype = I32
    lib.dsa_indexer_scores_topk_static.argtypes = [ctypes.POINTER(DsaCache), ctypes.POINTER(DsaBatch), P, P, I32, P,
                                                   P, P]
    lib.dsa_indexer_page_workspace_bytes.restype = SZ
    lib.dsa_indexer_page_workspace_bytes.argtypes = [I32, I32, I32, I32]
    lib.dsa_indexer_page_topk.restype = I32
    lib.dsa_indexer_page_topk.argtypes = [ctypes.POINTER(DsaCache), ctypes.POINTER(DsaBatch), P, P, I32, P, P, P, P,
                                          SZ, P]
    for name in ("dsa_sparse_mla_decode", "dsa_sparse_mla_prefill"):
        fn = getattr(lib, name)
        fn.restype = I32
        fn.argtypes = [ctypes.POINTER(DsaCache), ctypes.POINTER(DsaBatch), P, P, I32, ctypes.c_float, P, P, P, SZ, P]
    lib.dsa_sparse_mla_decode_layers.restype = I32
    lib.dsa_sparse_mla_decode_layers.argtypes = [ctypes.POINTER(DsaCache), I32, ctypes.POINTER(DsaBatch), P, P, I32,
                                                 ctypes.c_float, P, P, P, SZ, P]
    lib.dsa_kv_append_layers.restype = I32
    lib.dsa_kv_append_layers.argtypes = [ctypes.POINTER(DsaCache), I32, P, P, P, I32, P, P, I32, P]
    lib.dsa_dcp_candidates.restype = I32
    lib.dsa_dcp_candidates.argtypes = [P, ctypes.c_int64, P, I32, I32, I32, I32, P, P, P]
    lib.dsa_dcp_select.restype = I32
    lib.dsa_dcp_select.argtypes = [P, P, I32, I32, I32, I32, P, P, P, P]
    lib.dsa_sparse_mla_decode_ragged.restype = I32
    lib.dsa_sparse_mla_decode_ragged.argtypes = [ctypes.POINTER(DsaCache), ctypes.POINTER(DsaBatch), P, P, I32, P,
                                                 ctypes.c_float, P, P, P, SZ, P]
    lib.dsa_dcp_merge.restype = I32
    lib.dsa_dcp_merge.argtypes = [P, P, I32, I32, P, P, P]
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != DSA_OK:
        raise DsaError(status, load().dsa_last_error().decode())
