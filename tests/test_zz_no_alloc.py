"""The allocation-free indexer entry point against the workspace one, through the C ABI.

dsa_indexer_scores_topk_static runs the indexer and top-k on a fixed scratch array inside the
library.  Two calls in a row must agree with dsa_indexer_scores_topk (caller workspace) on the
same inputs: scores within the parity score tolerance and index sets within the swap tolerance
at the k-th score.  This file sorts last so the check also runs after every other GPU test has
used the library in the same process; it passes on its own too.
"""
import ctypes

import numpy as np
import pytest

import workloads as wlm
from parity import GpuProblem, HostProblem, check_scores, check_topk

pytestmark = pytest.mark.gpu

OK, WORKSPACE = 0, -3


def _call_workspace(lib, gp, k, idx, scores, ws):
    import torch
    c, b = gp.caches[0].struct(), gp.batch.struct()
    P = ctypes.c_void_p
    return lib.dsa_indexer_scores_topk(ctypes.byref(c), ctypes.byref(b), P(gp.q_idx.data_ptr()), P(gp.w.data_ptr()), k,
                                       P(idx.data_ptr()), P(scores.data_ptr()), P(ws.data_ptr()), ws.numel(),
                                       P(torch.cuda.current_stream().cuda_stream))


def _call_static(lib, gp, k, idx, scores):
    import torch
    c, b = gp.caches[0].struct(), gp.batch.struct()
    P = ctypes.c_void_p
    return lib.dsa_indexer_scores_topk_static(ctypes.byref(c), ctypes.byref(b), P(gp.q_idx.data_ptr()),
                                              P(gp.w.data_ptr()), k, P(idx.data_ptr()),
                                              P(scores.data_ptr()) if scores is not None else None,
                                              P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["decode_b32_8k", "decode_b64_fp8_indexshare", "prefill_chunk_4096"])
def test_static_scratch_matches_workspace_entry_point(lib, name):
    import torch
    wl = wlm.reduced(name)
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    R, L, k = wl.num_rows, wl.max_seq_len, wl.topk
    assert lib.dsa_indexer_workspace_bytes(R, L, k) <= 16 << 20
    ws = torch.empty(lib.dsa_indexer_workspace_bytes(R, L, k), dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty((R, k), dtype=torch.int32, device="cuda")
    ref_sc = torch.empty((R, L), dtype=torch.float32, device="cuda")
    assert _call_workspace(lib, gp, k, ref_idx, ref_sc, ws) == OK, lib.dsa_last_error()
    torch.cuda.synchronize()
    ref_i, ref_s = ref_idx.cpu().numpy(), ref_sc.cpu().numpy().astype(np.float64)
    _, pos = wl.row_request(), wl.row_position()
    for call in range(2):                                  # two calls in a row on the same scratch
        idx = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((R, L), np.nan, dtype=torch.float32, device="cuda")
        assert _call_static(lib, gp, k, idx, sc) == OK, lib.dsa_last_error()
        torch.cuda.synchronize()
        g_i, g_s = idx.cpu().numpy(), sc.cpu().numpy()
        for r in range(R):
            p = int(pos[r])
            check_scores(g_s[r], ref_s[r, :p + 1], p, L)
            check_topk(g_i[r], ref_i[r], ref_s[r, :p + 1], p, k)
    # the index buffer alone (no score output) is the benchmark's form of the call
    idx = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    assert _call_static(lib, gp, k, idx, None) == OK, lib.dsa_last_error()
    torch.cuda.synchronize()
    for r in range(R):
        p = int(pos[r])
        check_topk(idx[r].cpu().numpy(), ref_i[r], ref_s[r, :p + 1], p, k)


def test_static_scratch_rejects_shapes_beyond_its_size(lib):
    import torch
    wl = wlm.reduced("decode_b32_8k")
    gp = GpuProblem(HostProblem(wl))
    from deepseek_sparse_mla_gb300._lib import DsaBatch
    b = gp.batch.struct()
    big = DsaBatch(b.block_table, b.seq_lens, b.query_start_loc, b.num_requests, 64, 131072, b.block_table_stride)
    assert lib.dsa_indexer_workspace_bytes(64, 131072, 2048) > 16 << 20
    idx = torch.empty((64, 2048), dtype=torch.int32, device="cuda")
    c = gp.caches[0].struct()
    P = ctypes.c_void_p
    st = lib.dsa_indexer_scores_topk_static(ctypes.byref(c), ctypes.byref(big), P(gp.q_idx.data_ptr()),
                                            P(gp.w.data_ptr()), 2048, P(idx.data_ptr()), None,
                                            P(torch.cuda.current_stream().cuda_stream))
    assert st == WORKSPACE
    assert "static array" in lib.dsa_last_error().decode()
