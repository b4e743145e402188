"""The C ABI on the host: the library loads, exports every declared entry point, and rejects
bad arguments before any launch (no GPU needed; no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")

INVALID, UNSUPPORTED, WORKSPACE = -1, -2, -3
A = 1 << 20          # a fake, 256-byte aligned "device" address: never dereferenced on these paths


def declared():
    text = open(HEADER).read()
    return re.findall(r"^DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared()
    for n in ("dsa_kv_append", "dsa_indexer_scores_topk", "dsa_sparse_mla_decode", "dsa_sparse_mla_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from deepseek_sparse_mla_gb300 import _lib
    for n in declared():
        assert hasattr(lib, n), n
    assert set(declared()) == set(_lib.EXPORTS)
    assert lib.dsa_abi_version() == 4


def test_missing_library_fails_loudly(tmp_path):
    from deepseek_sparse_mla_gb300 import _lib
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(ImportError):
            _lib.load(str(tmp_path / "libdsa.so"))
    finally:
        _lib._lib = saved


def _cache(latent=A, keys=A, scales=A, pages=16, P=64, fmt=1):
    from deepseek_sparse_mla_gb300._lib import DsaCache
    return DsaCache(latent, keys, scales, pages, P, fmt)


def _batch(B=2, rows=2, L=300, qsl=0, bt=A, sl=A):
    from deepseek_sparse_mla_gb300._lib import DsaBatch
    return DsaBatch(bt, sl, qsl, B, rows, L, 8)


def _err(lib):
    return lib.dsa_last_error().decode()


def test_cache_bytes_counts_index_keys_and_scales(lib):
    pages, P = 1000, 64
    latent = pages * P * 576 * 2
    assert lib.dsa_cache_bytes(pages, P, 1, 1, 0) == latent + pages * P * (128 + 4)
    assert lib.dsa_cache_bytes(pages, P, 0, 1, 0) == latent + pages * P * 256
    assert lib.dsa_cache_bytes(pages, P, 1, 0, 0) == latent
    assert lib.dsa_cache_bytes(0, P, 1, 1, 0) == 0 and lib.dsa_cache_bytes(pages, P, 7, 1, 0) == 0
    # packed 8-bit latent: 512 codes + 128 bytes of k_R + a 4-byte scale per slot
    assert lib.dsa_cache_bytes(pages, P, 1, 0, 1) == pages * P * (512 + 128 + 4)
    assert lib.dsa_cache_bytes(pages, P, 1, 1, 1) == pages * P * (512 + 128 + 4 + 128 + 4)
    assert lib.dsa_cache_bytes(pages, P, 1, 1, 5) == 0
    # int8 index keys: 128 codes + a 2-byte binary16 scale per slot
    assert lib.dsa_cache_bytes(pages, P, 2, 1, 0) == latent + pages * P * (128 + 2)


def test_workspace_sizes_depend_only_on_shape(lib):
    a = lib.dsa_indexer_workspace_bytes(64, 131072, 2048)
    assert a == lib.dsa_indexer_workspace_bytes(64, 131072, 2048) and a >= 64 * 131072 * 4
    big = lib.dsa_indexer_workspace_bytes(4096, 65536, 2048)
    # score block and top-k candidate lists (a quarter of it here) are bounded, not R x L
    assert big <= (256 << 20) + (64 << 20) + 65536 * 4 + 4096 * 16
    # attention: a timeout word and two partial slots per persistent CTA, independent of the row count
    # beyond one CTA per SM
    slot = 64 * (512 + 2) * 4
    assert lib.dsa_mla_workspace_bytes(64, 2048) == 256 + 768 + 2 * 152 * slot      # 152 words: 608 -> 768 bytes
    assert lib.dsa_mla_workspace_bytes(4096, 2048) == lib.dsa_mla_workspace_bytes(100000, 2048)
    assert lib.dsa_mla_workspace_bytes(2, 128) == 256 + 256 + 2 * 4 * slot    # 2 rows x 2 tiles -> 4 CTAs
    assert lib.dsa_indexer_workspace_bytes(1, 0, 2048) == 0


def test_append_rejects_bad_arguments(lib):
    T, P = 4, ctypes.c_void_p
    assert lib.dsa_kv_append(None, P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    c = _cache(P=48)
    assert lib.dsa_kv_append(ctypes.byref(c), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    assert "power of two" in _err(lib)
    c = _cache(latent=A + 8)
    assert lib.dsa_kv_append(ctypes.byref(c), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    c = _cache()
    assert lib.dsa_kv_append(ctypes.byref(c), P(A), P(A), None, 0, None, P(A), T, None) == INVALID
    assert "k_idx is required" in _err(lib)
    shared = _cache(keys=0, scales=0)
    assert lib.dsa_kv_append(ctypes.byref(shared), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    bf16_cache = _cache(scales=0, fmt=0)
    assert lib.dsa_kv_append(ctypes.byref(bf16_cache), P(A), P(A), P(A), 1, P(A), P(A), T, None) == INVALID
    c = _cache()
    assert lib.dsa_kv_append(ctypes.byref(c), P(A), P(A), P(A), 1, None, P(A), T, None) == INVALID   # no scales
    bad_layout = _cache(fmt=0)                                          # bf16 keys with a scale array
    assert lib.dsa_kv_append(ctypes.byref(bad_layout), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    assert "not interchangeable" in _err(lib)
    assert lib.dsa_kv_append(ctypes.byref(c), P(A), P(A), P(A), 0, None, P(A), 0, None) == 0   # empty: no-op


def test_int8_keys_are_checked(lib):
    T, P = 4, ctypes.c_void_p
    int8_cache = _cache(fmt=2)
    assert lib.dsa_kv_append(ctypes.byref(int8_cache), P(A), P(A), P(A), 0, None, P(A), 0, None) == 0
    no_scales = _cache(scales=0, fmt=2)                                 # int8 keys need their half scales
    assert lib.dsa_kv_append(ctypes.byref(no_scales), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID
    assert "int8 index keys need" in _err(lib)
    # pre-quantised codes only go into a cache of their own format, with their scales
    assert lib.dsa_kv_append(ctypes.byref(int8_cache), P(A), P(A), P(A), 1, P(A), P(A), T, None) == INVALID
    fp8_cache = _cache(fmt=1)
    assert lib.dsa_kv_append(ctypes.byref(fp8_cache), P(A), P(A), P(A), 2, P(A), P(A), T, None) == INVALID
    assert lib.dsa_kv_append(ctypes.byref(int8_cache), P(A), P(A), P(A), 2, None, P(A), T, None) == INVALID
    assert lib.dsa_kv_append(ctypes.byref(int8_cache), P(A), P(A), P(A), 2, P(A + 1), P(A), T, None) == INVALID
    assert lib.dsa_kv_append(ctypes.byref(_cache(fmt=3)), P(A), P(A), P(A), 0, None, P(A), T, None) == INVALID


def test_indexer_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    ws = lib.dsa_indexer_workspace_bytes(2, 300, 128)
    shared = _cache(keys=0, scales=0)
    b = _batch()
    args = lambda k, wsb: (P(A), P(A), k, P(A), None, P(A), wsb, None)   # noqa: E731
    assert lib.dsa_indexer_scores_topk(ctypes.byref(shared), ctypes.byref(b), *args(128, ws)) == INVALID
    assert "shared layer" in _err(lib)
    c = _cache()
    assert lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(b), *args(0, ws)) == INVALID
    assert lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(b), *args(9000, ws)) == INVALID
    assert lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(b), *args(128, ws - 1)) == WORKSPACE
    multi = _batch(B=2, rows=5)                                         # several rows per request need query_start_loc
    assert lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(multi), *args(128, ws)) == INVALID
    nometa = _batch(bt=0)
    assert lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(nometa), *args(128, ws)) == INVALID


def test_sparse_mla_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    c = _cache(keys=0, scales=0)                     # attention reads only latent pages
    b = _batch()
    ws = lib.dsa_mla_workspace_bytes(2, 128)
    call = lib.dsa_sparse_mla_decode
    assert call(ctypes.byref(c), ctypes.byref(b), P(A), None, 128, 0.0625, P(A), None, P(A), ws, None) == INVALID
    assert "owner layer's index buffer" in _err(lib)
    assert call(ctypes.byref(c), ctypes.byref(b), P(A), P(A), 128, -1.0, P(A), None, P(A), ws, None) == INVALID
    assert call(ctypes.byref(c), ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws - 1, None) == WORKSPACE
    multi = _batch(B=2, rows=6, qsl=A)
    assert call(ctypes.byref(c), ctypes.byref(multi), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws, None) == INVALID
    # prefill needs query_start_loc
    assert lib.dsa_sparse_mla_prefill(ctypes.byref(c), ctypes.byref(_batch(rows=2)), P(A), P(A), 128, 0.0625, P(A),
                                      None, P(A), ws, None) == INVALID


def test_page_topk_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    b = _batch()
    ws = lib.dsa_indexer_page_workspace_bytes(2, 300, 64, 4)
    args = lambda kp, tok, wsb: (P(A), P(A), kp, P(A), tok, None, P(A), wsb, None)   # noqa: E731
    c = _cache()
    assert lib.dsa_indexer_page_topk(ctypes.byref(c), ctypes.byref(b), *args(0, P(A), ws)) == INVALID
    assert lib.dsa_indexer_page_topk(ctypes.byref(c), ctypes.byref(b), *args(200, P(A), ws)) == INVALID
    assert "DSA_MAX_TOPK" in _err(lib)                       # 200 pages x 64 positions > 8192
    assert lib.dsa_indexer_page_topk(ctypes.byref(c), ctypes.byref(b), *args(4, P(A), ws - 1)) == WORKSPACE
    big = _cache(P=256)
    assert lib.dsa_indexer_page_topk(ctypes.byref(big), ctypes.byref(b), *args(4, P(A), ws)) == UNSUPPORTED
    shared = _cache(keys=0, scales=0)
    assert lib.dsa_indexer_page_topk(ctypes.byref(shared), ctypes.byref(b), *args(4, P(A), ws)) == INVALID
    assert lib.dsa_indexer_page_topk(ctypes.byref(c), ctypes.byref(b), P(A), P(A), 4, None, None, None, P(A), ws,
                                     None) == INVALID                          # page_idx is required


def test_page_workspace_holds_page_scores_not_token_scores(lib):
    # 64 rows of 131,072 keys: token scores need 32 MiB; 64-key pages need 32-key unit maxima (1 MiB)
    # and the page scores pooled from them (0.5 MiB); 32-key pages only their page scores
    tok = lib.dsa_indexer_workspace_bytes(64, 131072, 2048)
    page = lib.dsa_indexer_page_workspace_bytes(64, 131072, 64, 32)
    assert tok >= 64 * 131072 * 4 and page < 64 * (4096 + 2048) * 4 + (1 << 16)
    assert lib.dsa_indexer_page_workspace_bytes(64, 131072, 32, 64) < 64 * 4096 * 4 + (1 << 16)
    assert lib.dsa_indexer_page_workspace_bytes(0, 100, 64, 4) > 0 and lib.dsa_indexer_page_workspace_bytes(4, 0, 64, 4) == 0


def test_dcp_entry_points_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    # dsa_dcp_candidates(scores, stride, local_idx, topk, rows, rank, world, cand_scores, cand_pos, stream)
    assert lib.dsa_dcp_candidates(P(A), 4096, P(A), 2048, 4, 0, 9, P(A), P(A), None) == UNSUPPORTED   # world > 8
    assert lib.dsa_dcp_candidates(P(A), 4096, P(A), 2048, 4, 0, 0, P(A), P(A), None) == UNSUPPORTED   # world 0
    assert lib.dsa_dcp_candidates(P(A), 4096, P(A), 2048, 4, 2, 2, P(A), P(A), None) == INVALID       # rank >= world
    assert lib.dsa_dcp_candidates(P(A), 4096, P(A), 4096, 4, 0, 8, P(A), P(A), None) == UNSUPPORTED   # 8 x 4096 > 16384
    assert lib.dsa_dcp_candidates(P(A), 4096, P(A), 9000, 4, 0, 1, P(A), P(A), None) == INVALID       # topk > 8192
    assert lib.dsa_dcp_candidates(None, 4096, P(A), 2048, 4, 0, 2, P(A), P(A), None) == INVALID
    assert lib.dsa_dcp_candidates(P(A), 0, P(A), 2048, 4, 0, 2, P(A), P(A), None) == INVALID
    assert lib.dsa_dcp_candidates(P(A), 1 << 30, P(A), 2048, 4, 0, 4, P(A), P(A), None) == UNSUPPORTED  # int32 positions
    assert lib.dsa_dcp_candidates(None, 4096, None, 2048, 0, 0, 2, None, None, None) == 0             # no rows: no-op
    # dsa_dcp_select(cand_scores, cand_pos, world, rows, topk, rank, global_idx, local_idx, local_count, stream)
    assert lib.dsa_dcp_select(P(A), P(A), 8, 4, 2049, 0, P(A), P(A), None, None) == UNSUPPORTED
    assert lib.dsa_dcp_select(P(A), None, 2, 4, 2048, 0, P(A), P(A), None, None) == INVALID
    assert lib.dsa_dcp_select(P(A), P(A), 2, -1, 2048, 0, P(A), P(A), None, None) == INVALID
    # the ragged attention call needs its row counts
    b = _batch(B=2, rows=2, L=300)
    c = _cache(fmt=0)
    assert lib.dsa_sparse_mla_decode_ragged(ctypes.byref(c), ctypes.byref(b), P(A), P(A), 128, None, 0.0625, P(A),
                                            None, P(A), 1 << 30, None) == INVALID
    # dsa_dcp_merge(outs, lses, world, rows, out, lse, stream)
    assert lib.dsa_dcp_merge(P(A), P(A), 9, 4, P(A), None, None) == UNSUPPORTED
    assert lib.dsa_dcp_merge(P(A + 8), P(A), 2, 4, P(A), None, None) == INVALID                        # unaligned outs
    assert lib.dsa_dcp_merge(P(A), None, 2, 4, P(A), None, None) == INVALID
    assert lib.dsa_dcp_merge(None, None, 2, 0, None, None, None) == 0


def test_latent_format_is_checked(lib):
    from deepseek_sparse_mla_gb300._lib import DsaCache
    P = ctypes.c_void_p
    b = _batch(B=2, rows=2, L=300)
    ws = lib.dsa_mla_workspace_bytes(2, 128)

    def call(cache):
        return lib.dsa_sparse_mla_decode(ctypes.byref(cache), ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None,
                                         P(A), ws, None)

    assert call(DsaCache(A, 0, 0, 16, 64, 0, 1, 0)) == INVALID          # e4m3 latent without its scales
    assert "latent_scales" in _err(lib)
    assert call(DsaCache(A, 0, 0, 16, 64, 0, 0, A)) == INVALID          # scales on a bf16 latent
    assert call(DsaCache(A, 0, 0, 16, 64, 0, 3, A)) == INVALID          # not a latent format
    assert call(DsaCache(A, 0, 0, 16, 64, 0, 1, A + 4)) == INVALID      # unaligned scales


def test_multi_layer_append_rejects_bad_arguments(lib):
    from deepseek_sparse_mla_gb300._lib import DsaCache
    P = ctypes.c_void_p
    two = (DsaCache * 2)(DsaCache(A, A, A, 16, 64, 1, 0, 0), DsaCache(A, 0, 0, 16, 64, 0, 0, 0))
    arr = lambda *v: (ctypes.c_void_p * len(v))(*v)       # noqa: E731
    ok_args = (arr(A, A), arr(A, A), arr(A, None), 0, None, P(A), 0, None)
    assert lib.dsa_kv_append_layers(two, 2, *ok_args) == 0                       # no tokens: a no-op
    assert lib.dsa_kv_append_layers(two, 0, *ok_args) == UNSUPPORTED
    assert lib.dsa_kv_append_layers(two, 17, *ok_args) == UNSUPPORTED
    assert lib.dsa_kv_append_layers(None, 2, *ok_args) == INVALID
    # the owner layer without its keys, and keys for the shared layer: rejected before any launch
    assert lib.dsa_kv_append_layers(two, 2, arr(A, A), arr(A, A), arr(None, None), 0, None, P(A), 8, None) == INVALID
    assert "layer 0" in _err(lib)
    assert lib.dsa_kv_append_layers(two, 2, arr(A, A), arr(A, A), arr(A, A), 0, None, P(A), 8, None) == INVALID
    assert "layer 1" in _err(lib)
    assert lib.dsa_kv_append_layers(two, 2, arr(A, A), arr(A, A + 8), arr(A, None), 0, None, P(A), 8, None) == INVALID


def test_layer_group_attention_rejects_bad_arguments(lib):
    """dsa_sparse_mla_decode_layers: the layers' caches must agree in page size, page count and latent
    format, 1 to 4 layers, a workspace for every layer's rows; all checked before any launch."""
    from deepseek_sparse_mla_gb300._lib import DsaCache
    P = ctypes.c_void_p
    layer = lambda pages=16, size=64, fmt=0, scales=0: DsaCache(A, 0, 0, pages, size, 0, fmt, scales)   # noqa: E731
    b = _batch()
    call = lib.dsa_sparse_mla_decode_layers
    ws4 = lib.dsa_mla_workspace_bytes(8, 128)
    four = (DsaCache * 5)(*[layer() for _ in range(5)])
    assert call(None, 2, ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws4, None) == INVALID
    assert call(four, 0, ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws4, None) == UNSUPPORTED
    assert call(four, 5, ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws4, None) == UNSUPPORTED
    for other in (layer(pages=32), layer(size=128), layer(fmt=1, scales=A)):
        pair = (DsaCache * 2)(layer(), other)
        assert call(pair, 2, ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), ws4, None) == INVALID
        assert "layer 1" in _err(lib)
    # the workspace covers every layer's rows: one sized for a single layer's rows is too small here
    small = lib.dsa_mla_workspace_bytes(2, 128)
    assert small < ws4
    assert call(four, 4, ctypes.byref(b), P(A), P(A), 128, 0.0625, P(A), None, P(A), small, None) == WORKSPACE
    # a shared index buffer is required, as for the one-layer call
    assert call(four, 4, ctypes.byref(b), P(A), None, 128, 0.0625, P(A), None, P(A), ws4, None) == INVALID
    assert "owner layer's index buffer" in _err(lib)


def test_device_status_helpers(lib):
    """dsa_check_device_status names the bits; dsa_read_status validates its arguments before any launch."""
    assert lib.dsa_check_device_status(0) == 0
    assert lib.dsa_check_device_status(0x4) == -5
    assert "DSA_DEVICE_BAD_PAGE" in _err(lib)
    assert lib.dsa_check_device_status(0x3) == -5
    msg = _err(lib)
    assert "DSA_DEVICE_TMA_TIMEOUT" in msg and "DSA_DEVICE_MMA_TIMEOUT" in msg
    assert lib.dsa_check_device_status(0x30) == -5 and "0x30" in _err(lib)
    P = ctypes.c_void_p
    assert lib.dsa_read_status(P(A), None, None) == INVALID
    assert lib.dsa_read_status(P(A), P(A + 2), None) == INVALID           # misaligned output word
    assert lib.dsa_read_status(P(A + 16), P(A), None) == INVALID          # workspace not 256-byte aligned
