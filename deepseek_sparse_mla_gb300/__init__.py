"""GLM-5.2 DeepSeek Sparse Attention (DSA) step on GB300 (sm_103a) behind a C ABI.

The step of one decoder layer over a paged KV cache: append the step's tokens,
score every visible cached position with the lightning indexer, select the
top-k positions into a shared index buffer, and run absorbed sparse MLA over
the selected positions (IndexShare layers reuse the owner's buffer).

This module is a thin binding over ``libdsa.so`` (``include/dsa.h``): it checks
tensor dtypes and shapes, passes raw device pointers and the current CUDA
stream, and raises on a non-OK status.  Every step of the computation runs in
the library's CUDA kernels; there is no other implementation to fall back to.
PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import DsaError, KEY_BF16, KEY_FP8_E4M3, KEY_INT8  # noqa: F401
from ._lib import DEVICE_BAD_PAGE, DEVICE_CONFIG, DEVICE_MMA_TIMEOUT, DEVICE_TMA_TIMEOUT  # noqa: F401

INDEX_HEADS, INDEX_DIM, HEADS, LATENT_DIM, ROPE_DIM, ROW_DIM = 32, 128, 64, 512, 64, 576
DEFAULT_SCALE = 1.0 / 16.0     # 1/sqrt(192 + 64)
_FORMATS = {"bf16": KEY_BF16, "fp8": KEY_FP8_E4M3, "int8": KEY_INT8, None: KEY_BF16}
_LATENT_FORMATS = {"bf16": _lib.LATENT_BF16, "fp8": _lib.LATENT_E4M3}

__all__ = ["LayerCache", "Batch", "kv_append", "kv_append_layers", "indexer_scores_topk", "indexer_page_topk", "sparse_mla_decode", "sparse_mla_decode_layers", "sparse_mla_prefill",
           "cache_bytes", "indexer_workspace_bytes", "mla_workspace_bytes", "DsaError", "DEFAULT_SCALE",
           "dcp_candidates", "dcp_select", "dcp_merge", "read_status"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


class LayerCache:
    """One layer's paged caches (device tensors owned by this object).

    latent [num_pages, page_size, 576] bf16 (or, with latent_format "fp8", packed 8-bit rows
    [num_pages, page_size, 640] uint8 = 512 e4m3 codes of c_KV + k_R as 64 bf16, with latent_scales
    [num_pages, page_size] fp32); for an indexer-owning layer also
    index_keys [num_pages, page_size, 128] (bf16, uint8 e4m3 codes, or int8 codes) and
    index_scales [num_pages, page_size] (fp32 for e4m3, float16 for int8).  key_format None
    makes an IndexShare layer that holds only latent pages."""

    def __init__(self, num_pages: int, page_size: int, key_format: str | None = None, device="cuda",
                 latent_format: str = "bf16"):
        self.num_pages, self.page_size, self.key_format = int(num_pages), int(page_size), key_format
        self.latent_format = latent_format
        self.latent_scales = None
        if latent_format == "bf16":
            self.latent = torch.zeros((num_pages, page_size, ROW_DIM), dtype=torch.bfloat16, device=device)
        elif latent_format == "fp8":
            # packed 8-bit rows: [512 e4m3 codes of c_KV | k_R as 64 bf16] = 640 bytes, a scale per slot
            self.latent = torch.zeros((num_pages, page_size, LATENT_DIM + 2 * ROPE_DIM), dtype=torch.uint8,
                                      device=device)
            self.latent_scales = torch.zeros((num_pages, page_size), dtype=torch.float32, device=device)
        else:
            raise ValueError(f"latent_format {latent_format!r}")
        self.index_keys = self.index_scales = None
        if key_format == "bf16":
            self.index_keys = torch.zeros((num_pages, page_size, INDEX_DIM), dtype=torch.bfloat16, device=device)
        elif key_format == "fp8":
            self.index_keys = torch.zeros((num_pages, page_size, INDEX_DIM), dtype=torch.uint8, device=device)
            self.index_scales = torch.zeros((num_pages, page_size), dtype=torch.float32, device=device)
        elif key_format == "int8":
            self.index_keys = torch.zeros((num_pages, page_size, INDEX_DIM), dtype=torch.int8, device=device)
            self.index_scales = torch.zeros((num_pages, page_size), dtype=torch.float16, device=device)
        elif key_format is not None:
            raise ValueError(f"key_format {key_format!r}")

    def struct(self) -> _lib.DsaCache:
        return _lib.DsaCache(self.latent.data_ptr(), 0 if self.index_keys is None else self.index_keys.data_ptr(),
                             0 if self.index_scales is None else self.index_scales.data_ptr(), self.num_pages,
                             self.page_size, _FORMATS[self.key_format], _LATENT_FORMATS[self.latent_format],
                             0 if self.latent_scales is None else self.latent_scales.data_ptr())


class Batch:
    """Batch metadata on the device: block_table [B, stride] int32, seq_lens [B] int32 (KV length
    after this step's append), query_start_loc [B+1] int32 or None (decode: one row per request)."""

    def __init__(self, block_table, seq_lens, query_start_loc=None, num_rows: int | None = None,
                 max_seq_len: int | None = None):
        self.block_table = block_table.to(torch.int32).contiguous()
        self.seq_lens = seq_lens.to(torch.int32).contiguous()
        self.query_start_loc = None if query_start_loc is None else query_start_loc.to(torch.int32).contiguous()
        self.num_requests = int(self.seq_lens.shape[0])
        if num_rows is None:
            num_rows = self.num_requests if query_start_loc is None else int(self.query_start_loc[-1].item())
        if max_seq_len is None:
            max_seq_len = int(self.seq_lens.max().item())
        self.num_rows, self.max_seq_len = int(num_rows), int(max_seq_len)

    def struct(self) -> _lib.DsaBatch:
        return _lib.DsaBatch(self.block_table.data_ptr(), self.seq_lens.data_ptr(),
                             0 if self.query_start_loc is None else self.query_start_loc.data_ptr(),
                             self.num_requests, self.num_rows, self.max_seq_len, int(self.block_table.shape[1]))


def cache_bytes(num_pages: int, page_size: int, key_format: str | None, owner: bool, latent_format: str = "bf16") -> int:
    return int(_lib.load().dsa_cache_bytes(num_pages, page_size, _FORMATS[key_format], int(owner),
                                           _LATENT_FORMATS[latent_format]))


def indexer_workspace_bytes(num_rows: int, max_seq_len: int, topk: int) -> int:
    return int(_lib.load().dsa_indexer_workspace_bytes(num_rows, max_seq_len, topk))


def indexer_page_workspace_bytes(num_rows: int, max_seq_len: int, page_size: int, page_budget: int) -> int:
    return int(_lib.load().dsa_indexer_page_workspace_bytes(num_rows, max_seq_len, page_size, page_budget))


def mla_workspace_bytes(num_rows: int, topk: int) -> int:
    return int(_lib.load().dsa_mla_workspace_bytes(num_rows, topk))


def _workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def read_status(workspace=None, stream=None, device=None) -> int:
    """The DSA_DEVICE_* bits of the last call that used `workspace` (None: the static scratch of
    dsa_indexer_scores_topk_static on the current device); 0 means no device-side problem.
    Synchronises the stream to read the value."""
    dev = workspace.device if workspace is not None else (device or torch.device("cuda", torch.cuda.current_device()))
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    _lib.check(_lib.load().dsa_read_status(_ptr(workspace), _ptr(out), _stream(stream)))
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return int(out.item()) & 0xFFFFFFFF


def _check_device(workspace, stream):
    """Raise DsaError(DSA_ERR_DEVICE_CHECK) when the call that used `workspace` set device status bits."""
    bits = read_status(workspace, stream)
    if bits:
        lib = _lib.load()
        raise DsaError(lib.dsa_check_device_status(bits), lib.dsa_last_error().decode())


def kv_append(cache: LayerCache, c_kv, k_rope, slot_mapping, k_idx=None, k_idx_scales=None, stream=None):
    """Scatter T new tokens into the layer's pages (bf16 keys are quantised for an fp8 or int8 cache;
    pre-quantised keys are uint8 e4m3 codes with float32 scales, or int8 codes with float16 scales)."""
    T = int(slot_mapping.shape[0])
    _need(c_kv, torch.bfloat16, (T, LATENT_DIM), "c_kv")
    _need(k_rope, torch.bfloat16, (T, ROPE_DIM), "k_rope")
    _need(slot_mapping, torch.int64, (T,), "slot_mapping")
    fmt = KEY_BF16
    if k_idx is not None:
        if k_idx.dtype == torch.uint8:
            fmt = KEY_FP8_E4M3
            _need(k_idx, torch.uint8, (T, INDEX_DIM), "k_idx")
            _need(k_idx_scales, torch.float32, (T,), "k_idx_scales")
        elif k_idx.dtype == torch.int8:
            fmt = KEY_INT8
            _need(k_idx, torch.int8, (T, INDEX_DIM), "k_idx")
            _need(k_idx_scales, torch.float16, (T,), "k_idx_scales")
        else:
            _need(k_idx, torch.bfloat16, (T, INDEX_DIM), "k_idx")
    c = cache.struct()
    _lib.check(_lib.load().dsa_kv_append(ctypes.byref(c), _ptr(c_kv), _ptr(k_rope), _ptr(k_idx), fmt,
                                         _ptr(k_idx_scales), _ptr(slot_mapping), T, _stream(stream)))


def kv_append_layers(caches, c_kv, k_rope, slot_mapping, k_idx=None, stream=None):
    """kv_append for several layers in one launch: the same T tokens and slots in every layer,
    c_kv[l] / k_rope[l] per layer, k_idx[l] (bf16) on the layers that own index keys, else None."""
    n = len(caches)
    T = int(slot_mapping.shape[0])
    _need(slot_mapping, torch.int64, (T,), "slot_mapping")
    k_idx = [None] * n if k_idx is None else list(k_idx)
    if not (len(c_kv) == len(k_rope) == len(k_idx) == n):
        raise ValueError("one c_kv, k_rope and k_idx entry per layer")
    for l in range(n):
        _need(c_kv[l], torch.bfloat16, (T, LATENT_DIM), f"c_kv[{l}]")
        _need(k_rope[l], torch.bfloat16, (T, ROPE_DIM), f"k_rope[{l}]")
        if k_idx[l] is not None:
            _need(k_idx[l], torch.bfloat16, (T, INDEX_DIM), f"k_idx[{l}]")
    structs = (_lib.DsaCache * n)(*[c.struct() for c in caches])
    ptrs = lambda ts: (ctypes.c_void_p * n)(*[None if t is None else t.data_ptr() for t in ts])   # noqa: E731
    _lib.check(_lib.load().dsa_kv_append_layers(structs, n, ptrs(c_kv), ptrs(k_rope), ptrs(k_idx), KEY_BF16, None,
                                                _ptr(slot_mapping), T, _stream(stream)))


def indexer_scores_topk(owner: LayerCache, batch: Batch, q_idx, w, topk: int, topk_idx=None, scores_out=None,
                        workspace=None, stream=None, check=False):
    """Lightning-indexer scores and top-k selection; returns the index buffer [R, topk] int32.
    check=True reads the call's device status afterwards (synchronising) and raises DsaError on a
    non-zero status."""
    R = batch.num_rows
    _need(q_idx, torch.bfloat16, (R, INDEX_HEADS, INDEX_DIM), "q_idx")
    _need(w, torch.float32, (R, INDEX_HEADS), "w")
    if topk_idx is None:
        topk_idx = torch.empty((R, topk), dtype=torch.int32, device=q_idx.device)
    _need(topk_idx, torch.int32, (R, topk), "topk_idx")
    if scores_out is not None:
        _need(scores_out, torch.float32, (R, batch.max_seq_len), "scores_out")
    need = indexer_workspace_bytes(R, batch.max_seq_len, topk)
    if workspace is None:
        workspace = _workspace(need, q_idx.device)
    c, b = owner.struct(), batch.struct()
    _lib.check(_lib.load().dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(b), _ptr(q_idx), _ptr(w), topk,
                                                   _ptr(topk_idx), _ptr(scores_out), _ptr(workspace),
                                                   workspace.numel() * workspace.element_size(), _stream(stream)))
    if check:
        _check_device(workspace, stream)
    return topk_idx


def indexer_page_topk(owner: LayerCache, batch: Batch, q_idx, w, page_budget: int, page_idx=None, token_idx=None,
                      expand=True, page_scores_out=None, workspace=None, stream=None, check=False):
    """Page-granular selection: page scores (max over visible tokens), the page budget, and (unless
    expand is False) the selected pages' positions.  Returns (page_idx [R, page_budget],
    token_idx [R, page_budget * page_size] or None)."""
    R, P = batch.num_rows, owner.page_size
    _need(q_idx, torch.bfloat16, (R, INDEX_HEADS, INDEX_DIM), "q_idx")
    _need(w, torch.float32, (R, INDEX_HEADS), "w")
    if page_idx is None:
        page_idx = torch.empty((R, page_budget), dtype=torch.int32, device=q_idx.device)
    _need(page_idx, torch.int32, (R, page_budget), "page_idx")
    if expand and token_idx is None:
        token_idx = torch.empty((R, page_budget * P), dtype=torch.int32, device=q_idx.device)
    if token_idx is not None:
        _need(token_idx, torch.int32, (R, page_budget * P), "token_idx")
    if page_scores_out is not None:
        _need(page_scores_out, torch.float32, (R, -(-batch.max_seq_len // P)), "page_scores_out")
    if workspace is None:
        workspace = _workspace(indexer_page_workspace_bytes(R, batch.max_seq_len, P, page_budget), q_idx.device)
    c, b = owner.struct(), batch.struct()
    _lib.check(_lib.load().dsa_indexer_page_topk(ctypes.byref(c), ctypes.byref(b), _ptr(q_idx), _ptr(w), page_budget,
                                                 _ptr(page_idx), _ptr(token_idx), _ptr(page_scores_out),
                                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                 _stream(stream)))
    if check:
        _check_device(workspace, stream)
    return page_idx, token_idx


def _sparse_mla(fn, layer, batch, q, topk_idx, scale, out, lse, workspace, stream, row_counts=None, check=False):
    R = batch.num_rows
    _need(q, torch.bfloat16, (R, HEADS, ROW_DIM), "q")
    if topk_idx is None:
        raise ValueError("topk_idx is required: a shared layer reuses the owner layer's index buffer")
    topk = int(topk_idx.shape[1])
    _need(topk_idx, torch.int32, (R, topk), "topk_idx")
    if out is None:
        out = torch.empty((R, HEADS, LATENT_DIM), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, (R, HEADS, LATENT_DIM), "out")
    if lse is not None:
        _need(lse, torch.float32, (R, HEADS), "lse")
    if workspace is None:
        workspace = _workspace(mla_workspace_bytes(R, topk), q.device)
    c, b = layer.struct(), batch.struct()
    if row_counts is None:
        _lib.check(fn(ctypes.byref(c), ctypes.byref(b), _ptr(q), _ptr(topk_idx), topk, float(scale), _ptr(out),
                      _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    else:
        _need(row_counts, torch.int32, (R,), "row_counts")
        _lib.check(_lib.load().dsa_sparse_mla_decode_ragged(
            ctypes.byref(c), ctypes.byref(b), _ptr(q), _ptr(topk_idx), topk, _ptr(row_counts), float(scale), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    if check:
        _check_device(workspace, stream)
    return out, lse


def sparse_mla_decode(layer: LayerCache, batch: Batch, q, topk_idx, scale: float = DEFAULT_SCALE, out=None, lse=None,
                      workspace=None, stream=None, row_counts=None, check=False):
    """Sparse absorbed MLA for decode rows (one per request); returns (out [R,64,512] bf16, lse).
    row_counts (optional int32 [R]): row r's valid entries lead its buffer and entries from
    row_counts[r] on are -1; the call then spends time only on those leading entries.
    check=True reads the call's device status afterwards and raises DsaError on a non-zero one."""
    return _sparse_mla(_lib.load().dsa_sparse_mla_decode, layer, batch, q, topk_idx, scale, out, lse, workspace, stream,
                       row_counts, check)


def sparse_mla_decode_layers(layers, batch: Batch, q, topk_idx, scale: float = DEFAULT_SCALE, out=None, lse=None,
                             workspace=None, stream=None, check=False):
    """sparse_mla_decode for the layers of an IndexShare group in one call (they share topk_idx):
    q [L, R, 64, 576] bf16 with layer l's queries at [l]; returns (out [L, R, 64, 512] bf16, lse
    [L, R, 64] fp32 or None).  The layers' caches agree in page size, page count and latent format."""
    L, R = len(layers), batch.num_rows
    _need(q, torch.bfloat16, (L, R, HEADS, ROW_DIM), "q")
    if topk_idx is None:
        raise ValueError("topk_idx is required: the shared layers reuse the owner layer's index buffer")
    topk = int(topk_idx.shape[1])
    _need(topk_idx, torch.int32, (R, topk), "topk_idx")
    if out is None:
        out = torch.empty((L, R, HEADS, LATENT_DIM), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, (L, R, HEADS, LATENT_DIM), "out")
    if lse is not None:
        _need(lse, torch.float32, (L, R, HEADS), "lse")
    if workspace is None:
        workspace = _workspace(mla_workspace_bytes(L * R, topk), q.device)
    structs = (_lib.DsaCache * L)(*[c.struct() for c in layers])
    b = batch.struct()
    _lib.check(_lib.load().dsa_sparse_mla_decode_layers(
        structs, L, ctypes.byref(b), _ptr(q), _ptr(topk_idx), topk, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    if check:
        _check_device(workspace, stream)
    return out, lse


def sparse_mla_prefill(layer: LayerCache, batch: Batch, q, topk_idx, scale: float = DEFAULT_SCALE, out=None, lse=None,
                       workspace=None, stream=None, check=False):
    """Sparse absorbed MLA for extend/prefill/verify rows (causal per row); returns (out, lse)."""
    return _sparse_mla(_lib.load().dsa_sparse_mla_prefill, layer, batch, q, topk_idx, scale, out, lse, workspace, stream,
                       check=check)


def dcp_candidates(local_scores, local_idx, rank: int, world: int, cand_scores=None, cand_pos=None, stream=None):
    """Decode context parallelism, step 1: this rank's local top-k as (score, global position)
    candidates.  local_scores [R, S] fp32 (the indexer's scores_out), local_idx [R, topk] int32.
    Returns (cand_scores [R, topk] fp32, cand_pos [R, topk] int32)."""
    R, topk = local_idx.shape
    _need(local_idx, torch.int32, (R, topk), "local_idx")
    _need(local_scores, torch.float32, (R, local_scores.shape[1]), "local_scores")
    if cand_scores is None:
        cand_scores = torch.empty((R, topk), dtype=torch.float32, device=local_idx.device)
    if cand_pos is None:
        cand_pos = torch.empty((R, topk), dtype=torch.int32, device=local_idx.device)
    _need(cand_scores, torch.float32, (R, topk), "cand_scores")
    _need(cand_pos, torch.int32, (R, topk), "cand_pos")
    _lib.check(_lib.load().dsa_dcp_candidates(_ptr(local_scores), int(local_scores.shape[1]), _ptr(local_idx), topk, R,
                                              rank, world, _ptr(cand_scores), _ptr(cand_pos), _stream(stream)))
    return cand_scores, cand_pos


def dcp_select(all_scores, all_pos, rank: int, global_idx=None, local_idx=None, local_count=None, stream=None):
    """Step 2, after the candidate all-gather: all_scores / all_pos [world, R, topk].  Returns
    (global_idx [R, topk], local_idx [R, topk], local_count [R]): the row's top-k as global positions
    (ascending), this rank's share of it as local positions (ascending, compacted to the front of
    the row, -1 after), and the share's size; local_idx and local_count feed sparse_mla_decode."""
    world, R, topk = all_scores.shape
    _need(all_scores, torch.float32, (world, R, topk), "all_scores")
    _need(all_pos, torch.int32, (world, R, topk), "all_pos")
    dev = all_pos.device
    global_idx = torch.empty((R, topk), dtype=torch.int32, device=dev) if global_idx is None else global_idx
    local_idx = torch.empty((R, topk), dtype=torch.int32, device=dev) if local_idx is None else local_idx
    local_count = torch.empty((R,), dtype=torch.int32, device=dev) if local_count is None else local_count
    _need(global_idx, torch.int32, (R, topk), "global_idx")
    _need(local_idx, torch.int32, (R, topk), "local_idx")
    _need(local_count, torch.int32, (R,), "local_count")
    _lib.check(_lib.load().dsa_dcp_select(_ptr(all_scores), _ptr(all_pos), world, R, topk, rank, _ptr(global_idx),
                                          _ptr(local_idx), _ptr(local_count), _stream(stream)))
    return global_idx, local_idx, local_count


def dcp_merge(outs, lses, out=None, lse=None, stream=None):
    """Step 3, after the out/lse all-gather: outs [world, R, 64, 512] bf16, lses [world, R, 64]
    fp32.  Returns (out [R, 64, 512] bf16, lse [R, 64] fp32): the LSE merge of the ranks' parts."""
    world, R = outs.shape[0], outs.shape[1]
    _need(outs, torch.bfloat16, (world, R, HEADS, LATENT_DIM), "outs")
    _need(lses, torch.float32, (world, R, HEADS), "lses")
    if out is None:
        out = torch.empty((R, HEADS, LATENT_DIM), dtype=torch.bfloat16, device=outs.device)
    if lse is None:
        lse = torch.empty((R, HEADS), dtype=torch.float32, device=outs.device)
    _need(out, torch.bfloat16, (R, HEADS, LATENT_DIM), "out")
    _need(lse, torch.float32, (R, HEADS), "lse")
    _lib.check(_lib.load().dsa_dcp_merge(_ptr(outs), _ptr(lses), world, R, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse
