"""Device status at the C boundary: dsa_read_status after every entry point that has a workspace.

A call that runs as specified leaves 0.  A visible position whose block-table page id is outside the
pool is reported as DSA_DEVICE_BAD_PAGE by the indexer and by the attention kernel ("GLM-5.2 on vLLM
Ascend: Request-to-Backend Inference Path", "Failure and Correctness Boundaries": wrong metadata must
surface).  The out-of-range id is never dereferenced: every kernel checks a page id against the pool
before it forms an address, so these cases read no memory outside the caches.
"""
import ctypes

import numpy as np
import pytest

import workloads as wlm
from parity import GpuProblem, HostProblem

pytestmark = pytest.mark.gpu


def _status(lib, ws):
    import torch
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = lib.dsa_read_status(ctypes.c_void_p(ws.data_ptr() if ws is not None else 0), ctypes.c_void_p(out.data_ptr()),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    return int(out.item()) & 0xFFFFFFFF


@pytest.mark.parametrize("name", ["decode_b64_fp8_indexshare", "prefill_chunk_4096", "verify_b8x4_240k"])
def test_status_is_clear_after_every_entry_point(lib, name):
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = wlm.reduced(name)
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    R, k = wl.num_rows, wl.topk
    # stale bytes in the workspaces must not leak into the status
    ws_i = torch.full((dsa.indexer_workspace_bytes(R, wl.max_seq_len, k),), 0xFF, dtype=torch.uint8, device="cuda")
    idx = dsa.indexer_scores_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, k, workspace=ws_i)
    assert _status(lib, ws_i) == 0
    ws_a = torch.full((dsa.mla_workspace_bytes(R, k),), 0xFF, dtype=torch.uint8, device="cuda")
    fn = dsa.sparse_mla_decode if wl.is_decode else dsa.sparse_mla_prefill
    for layer in range(wl.layers):
        fn(gp.caches[layer], gp.batch, gp.q[layer], idx, wl.scale, workspace=ws_a)
        assert _status(lib, ws_a) == 0
    if wl.is_decode:
        counts = (idx >= 0).sum(dim=1).to(torch.int32)
        dsa.sparse_mla_decode(gp.caches[1], gp.batch, gp.q[1], idx, wl.scale, workspace=ws_a, row_counts=counts)
        assert _status(lib, ws_a) == 0
    if wl.page_size <= 128 and k % wl.page_size == 0:
        budget = k // wl.page_size
        ws_p = torch.full((dsa.indexer_page_workspace_bytes(R, wl.max_seq_len, wl.page_size, budget),), 0xFF,
                          dtype=torch.uint8, device="cuda")
        dsa.indexer_page_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, budget, workspace=ws_p)
        assert _status(lib, ws_p) == 0
    # the binding's checked path raises nothing on a clean call
    dsa.indexer_scores_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, k, workspace=ws_i, check=True)
    fn(gp.caches[-1], gp.batch, gp.q[-1], idx, wl.scale, workspace=ws_a, check=True)


def test_static_scratch_status_is_clear(lib):
    import torch
    wl = wlm.reduced("decode_b32_8k")
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    idx = torch.empty((wl.num_rows, wl.topk), dtype=torch.int32, device="cuda")
    c, b = gp.caches[0].struct(), gp.batch.struct()
    P = ctypes.c_void_p
    st = lib.dsa_indexer_scores_topk_static(ctypes.byref(c), ctypes.byref(b), P(gp.q_idx.data_ptr()),
                                            P(gp.w.data_ptr()), wl.topk, P(idx.data_ptr()), None,
                                            P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert _status(lib, None) == 0


def _bad_page_problem():
    """A decode problem whose request 0 has one visible page id replaced by an id beyond the pool."""
    import torch
    wl = wlm.reduced("decode_b64_fp8_indexshare")
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    lp = 1                                              # logical page 1 of request 0 (visible: L_0 > 2 pages)
    assert wl.seq_lens[0] > 2 * wl.page_size
    bt = gp.batch.block_table.clone()
    bt[0, lp] = wl.num_pages + 7
    import deepseek_sparse_mla_gb300 as dsa
    bad = dsa.Batch(bt, gp.batch.seq_lens, None, num_rows=wl.num_rows, max_seq_len=wl.max_seq_len)
    return wl, gp, bad, lp


def test_out_of_range_page_is_reported_by_the_indexer(lib):
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl, gp, bad, _ = _bad_page_problem()
    ws = torch.empty((dsa.indexer_workspace_bytes(wl.num_rows, wl.max_seq_len, wl.topk),), dtype=torch.uint8,
                     device="cuda")
    dsa.indexer_scores_topk(gp.caches[0], bad, gp.q_idx, gp.w, wl.topk, workspace=ws)
    assert _status(lib, ws) & dsa.DEVICE_BAD_PAGE
    with pytest.raises(dsa.DsaError) as e:
        dsa.indexer_scores_topk(gp.caches[0], bad, gp.q_idx, gp.w, wl.topk, workspace=ws, check=True)
    assert e.value.status == -5 and "DSA_DEVICE_BAD_PAGE" in str(e.value)
    # the next clean call on the same workspace clears it
    dsa.indexer_scores_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, wl.topk, workspace=ws)
    assert _status(lib, ws) == 0


def test_out_of_range_page_is_reported_and_skipped_by_attention(lib):
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    from parity import bf16_tensor_to_f64
    from oracle import dsa_oracle as o
    wl, gp, bad, lp = _bad_page_problem()
    idx, _ = gp.indexer()
    # row 0 selects every position of the bad page, plus its own selection elsewhere
    sel = idx.clone()
    P = wl.page_size
    sel[0, :P] = torch.arange(lp * P, lp * P + P, dtype=torch.int32, device="cuda")
    ws = torch.empty((dsa.mla_workspace_bytes(wl.num_rows, wl.topk),), dtype=torch.uint8, device="cuda")
    out, _ = dsa.sparse_mla_decode(gp.caches[1], bad, gp.q[1], sel, wl.scale, workspace=ws)
    assert _status(lib, ws) & dsa.DEVICE_BAD_PAGE
    # the bad page's entries are skipped: row 0 equals the oracle over the selection without them
    keep = sel.cpu().numpy().copy()
    row = keep[0]
    row[(row >= 0) & (row // P == lp)] = -1                # every entry in the bad page, wherever it sits
    o_out, _ = o.sparse_mla(gp.hp.caches[1], wl.block_table, wl.seq_lens, wl.query_start_loc, gp.hp.q[1], keep, wl.scale,
                            rows=[0])
    err = np.abs(bf16_tensor_to_f64(out[:1]) - o_out[:1])
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    with pytest.raises(dsa.DsaError):
        dsa.sparse_mla_decode(gp.caches[1], bad, gp.q[1], sel, wl.scale, workspace=ws, check=True)
