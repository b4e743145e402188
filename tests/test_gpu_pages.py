"""GPU parity of page-granular selection against the float64 oracle, through the C ABI.

dsa_indexer_page_topk pools the indexer scores into page scores (the maximum over a page's
visible tokens), keeps the page budget and expands it to positions.  Checked per row: page scores
within the score tolerance, the page set within the swap tolerance at the budget's score, the
expansion bit-exact for the pages the GPU chose, and attention over the expanded positions against
the oracle.  Pages of 1, 16, 64 and 128 keys cover the in-warp, cross-warp and whole-tile poolings.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from parity import (GpuProblem, HostProblem, bf16_tensor_to_f64, check_attention, check_scores, check_topk)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def run_page_case(wl, budget, attend=True):
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    P = wl.page_size
    n_pages = -(-wl.max_seq_len // P)
    pscores = torch.empty((wl.num_rows, n_pages), dtype=torch.float32, device="cuda")
    page_idx, token_idx = dsa.indexer_page_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, budget,
                                                page_scores_out=pscores)
    torch.cuda.synchronize()
    g_pages, g_tok, g_ps = page_idx.cpu().numpy(), token_idx.cpu().numpy(), pscores.cpu().numpy()
    o_pages, o_tok, o_ps, _ = o.page_indexer_topk(hp.caches[0], wl.block_table, wl.seq_lens, wl.query_start_loc,
                                                  hp.q_idx, hp.w, budget)
    _, pos = o.row_positions(wl.seq_lens, wl.query_start_loc)
    for r in range(wl.num_rows):
        p = int(pos[r])
        check_scores(g_ps[r], o_ps[r], p // P, n_pages)
        check_topk(g_pages[r], o_pages[r], o_ps[r], p // P, budget)
        assert np.array_equal(g_tok[r], o.pages_to_positions(g_pages[r], P, p)), f"row {r}: expansion differs"
    if attend:
        for layer in range(wl.layers):
            out, lse = gp.attention(layer, token_idx)
            o_out, o_lse = hp.oracle_attention(layer, g_tok)
            check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)
    return g_pages, o_pages


@pytest.mark.parametrize("name,P,fmt,budget", [
    ("page64_fp8", 64, "fp8", 8),
    ("page64_bf16", 64, "bf16", 5),
    ("page16_fp8", 16, "fp8", 12),
    ("page128_bf16", 128, "bf16", 3),
    ("page1_fp8", 1, "fp8", 40),
])
def test_page_selection_parity(name, P, fmt, budget):
    wl = wlm.Workload(name, [2500, 900, 3001, 130], [1] * 4, P, fmt, 2048, 2, 3100 + P)
    run_page_case(wl, budget)


def test_page_selection_with_multi_row_requests():
    """Extend rows of one request share keys but see different prefixes: each row pools only its
    visible tokens, so the rows' last pages differ."""
    wl = wlm.Workload("page_extend", [1500, 700], [5, 3], 64, "fp8", 512, 1, 3120)
    run_page_case(wl, 6)


def test_budget_of_every_page_selects_every_visible_position():
    wl = wlm.Workload("page_all", [333, 1024], [1, 1], 64, "bf16", 128, 1, 3121)
    g_pages, _ = run_page_case(wl, 16, attend=False)
    assert list(g_pages[0][:6]) == list(range(6)) and np.all(g_pages[0][6:] == -1)
    assert list(g_pages[1]) == list(range(16))


def test_invisible_keys_do_not_promote_their_page():
    """Huge keys written just past each row's position, inside its last page, must not win that page
    the budget: masks precede the page maximum."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = wlm.Workload("page_mask", [1000, 1300], [1, 1], 64, "bf16", 128, 1, 3122)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    q = o.bf16_to_f64(hp.q_idx)
    for b, L in enumerate(wl.seq_lens):
        tail = np.arange(L, -(-L // 64) * 64)                 # invisible positions of the last page
        w = hp.w[b].astype(np.float64)
        direction = (q[b] * (w > 0)[:, None]).sum(axis=0)
        big = wlm.bf16_bits(np.tile(np.sign(direction) * 40.0, (len(tail), 1)).astype(np.float32))
        slots = torch.from_numpy(wl.slots(b, tail).astype(np.int64)).cuda()
        z = torch.zeros((len(tail), 512), dtype=torch.bfloat16, device="cuda")
        dsa.kv_append(gp.caches[0], z, torch.zeros((len(tail), 64), dtype=torch.bfloat16, device="cuda"), slots,
                      k_idx=wlm.bits_to_torch(big, "cuda"))
    page_idx, _ = dsa.indexer_page_topk(gp.caches[0], gp.batch, gp.q_idx, gp.w, 1, expand=False)
    torch.cuda.synchronize()
    o_pages, _, o_ps, _ = o.page_indexer_topk(hp.caches[0], wl.block_table, wl.seq_lens, wl.query_start_loc,
                                              hp.q_idx, hp.w, 1)
    _, pos = o.row_positions(wl.seq_lens, wl.query_start_loc)
    for r in range(wl.num_rows):
        check_topk(page_idx[r].cpu().numpy(), o_pages[r], o_ps[r], int(pos[r]) // 64, 1)
