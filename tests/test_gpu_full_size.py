"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark times.

Each workload is set up exactly as ``bench.py`` sets it up (every request's prefix resident in
the paged caches, the step's new tokens appended, the same workspaces and the same calls), so
the kernels run with the full grid, full score blocks and full split-k partition.  A few sampled
requests are then re-drawn with the host generators and written over their slots, so that the
float64 oracle can recompute their rows one by one from the same values: indexer scores over
every visible position, the top-k set (swap tolerance at the k-th score), the page-granular
selection (page scores, the page set, its expansion), and the attention output and LSE on the
oracle's own index set.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from parity import check_attention, check_scores, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def sampled_rows(wl: wlm.Workload):
    """Rows checked against the oracle: the shortest and longest contexts, first and last rows,
    and one seeded draw, so that ragged and maximal sizes are both covered."""
    req, pos = o.row_positions(wl.seq_lens, wl.query_start_loc)
    R = wl.num_rows
    rng = np.random.default_rng(wl.seed + 77)
    rows = {0, R - 1, int(np.argmin(pos)), int(np.argmax(pos)), int(rng.integers(0, R))}
    return sorted(rows), req, pos


def key_values(bits: np.ndarray, key_format: str) -> np.ndarray:
    if key_format == "fp8":
        codes, scales = o.quantize_index_keys(bits)
        return o.e4m3_to_f64(codes) * scales.astype(np.float64)[:, None]
    return o.bf16_to_f64(bits)


def latent_values(bits: np.ndarray, latent_format: str) -> np.ndarray:
    """Cached rows as attention sees them: bf16, or the packed 8-bit c_KV (code * scale) with bf16 k_R."""
    rows = o.bf16_to_f64(bits)
    if latent_format == "fp8":
        codes, scales = o.quantize_latent(bits[:, :512])
        rows[:, :512] = o.e4m3_to_f64(codes) * scales.astype(np.float64)[:, None]
    return rows


@pytest.mark.parametrize("name,latent", [("decode_b32_8k", "bf16"), ("decode_b64_fp8_indexshare", "bf16"),
                                         ("prefill_chunk_4096", "bf16"), ("verify_b8x4_240k", "bf16"),
                                         ("decode_b64_fp8_indexshare", "fp8")])
def test_full_size_sampled_rows(name, latent):
    import dataclasses
    import torch
    import bench
    import deepseek_sparse_mla_gb300 as dsa
    wl = dataclasses.replace(wlm.FULL[name](), latent_format=latent)
    prob = bench.DeviceProblem(wl)
    # the step's append of the new tokens, as the benchmark step does it
    for layer in range(wl.layers):
        dsa.kv_append(prob.caches[layer], prob.new_c[layer], prob.new_r[layer], prob.slots,
                      k_idx=prob.new_k if layer == 0 else None)
    rows, req, pos = sampled_rows(wl)
    host_lat, host_keys = {}, {}
    for b in sorted({int(req[r]) for r in rows}):
        L = int(wl.seq_lens[b])
        slots = torch.from_numpy(wl.slots(b, np.arange(L)).astype(np.int64)).cuda()
        host_keys[b] = wlm.request_index_keys(wl, b)
        for layer in range(wl.layers):
            lat = wlm.request_latent(wl, b, layer)
            host_lat[(b, layer)] = lat
            dsa.kv_append(prob.caches[layer], wlm.bits_to_torch(lat[:, :512], "cuda"),
                          wlm.bits_to_torch(lat[:, 512:], "cuda"), slots,
                          k_idx=wlm.bits_to_torch(host_keys[b], "cuda") if layer == 0 else None)
    torch.cuda.synchronize()

    # indexer + top-k as timed (score block in the workspace), then once more writing the scores out
    idx = dsa.indexer_scores_topk(prob.caches[0], prob.batch, prob.q_idx, prob.w, wl.topk,
                                  topk_idx=prob.topk_idx, workspace=prob.ws_idx).clone()
    scores = torch.empty((wl.num_rows, wl.max_seq_len), dtype=torch.float32, device="cuda")
    idx2 = dsa.indexer_scores_topk(prob.caches[0], prob.batch, prob.q_idx, prob.w, wl.topk, scores_out=scores,
                                   workspace=prob.ws_idx)
    assert torch.equal(idx, idx2), "the selection depends on where the scores are written"
    g_idx = idx.cpu().numpy()
    q_idx, w = wlm.indexer_queries(wl)
    oracle_idx = {}
    for r in rows:
        b, p = int(req[r]), int(pos[r])
        keys = key_values(host_keys[b][:p + 1], wl.key_format)
        o_scores = o.index_scores(o.bf16_to_f64(q_idx[r]), w[r], keys)
        check_scores(scores[r].cpu().numpy(), o_scores, p, wl.max_seq_len)
        oracle_idx[r] = o.topk_select(o_scores, wl.topk)
        check_topk(g_idx[r], oracle_idx[r], o_scores, p, wl.topk)
    del scores

    # page-granular selection with a budget of topk / page_size pages, on the same rows
    P = wl.page_size
    budget = wl.topk // P
    n_pages = -(-wl.max_seq_len // P)
    pscores = torch.empty((wl.num_rows, n_pages), dtype=torch.float32, device="cuda")
    page_idx, token_idx = dsa.indexer_page_topk(prob.caches[0], prob.batch, prob.q_idx, prob.w, budget,
                                                page_scores_out=pscores)
    g_pages, g_tok, g_ps = page_idx.cpu().numpy(), token_idx.cpu().numpy(), pscores.cpu().numpy()
    for r in rows:
        p = int(pos[r])
        keys = key_values(host_keys[int(req[r])][:p + 1], wl.key_format)
        o_ps = o.page_scores(o.index_scores(o.bf16_to_f64(q_idx[r]), w[r], keys), P)
        check_scores(g_ps[r], o_ps, p // P, n_pages)
        check_topk(g_pages[r], o.page_topk_select(o_ps, budget), o_ps, p // P, budget)
        assert np.array_equal(g_tok[r], o.pages_to_positions(g_pages[r], P, p))
    del pscores

    # attention on the oracle's index sets for the sampled rows, every layer of the group
    idx_att = idx.clone()
    for r in rows:
        idx_att[r] = torch.from_numpy(oracle_idx[r]).cuda()
    mla = dsa.sparse_mla_decode if wl.is_decode else dsa.sparse_mla_prefill
    if prob.group_attention:
        # as the benchmark step runs it: every layer of the group in one call
        dsa.sparse_mla_decode_layers(prob.caches, prob.batch, bench.stacked(prob.q), idx_att, wl.scale,
                                     out=bench.stacked(prob.out), lse=bench.stacked(prob.lse), workspace=prob.ws_mla,
                                     check=True)
    for layer in range(wl.layers):
        if not prob.group_attention:
            mla(prob.caches[layer], prob.batch, prob.q[layer], idx_att, wl.scale, out=prob.out[layer],
                lse=prob.lse[layer], workspace=prob.ws_mla, check=True)
        torch.cuda.synchronize()
        q = wlm.mla_queries(wl, layer)
        out_bits = wlm.torch_to_bits(prob.out[layer][rows])
        lse = prob.lse[layer][rows].cpu().numpy()
        for n, r in enumerate(rows):
            b, p = int(req[r]), int(pos[r])
            sel = o.valid_selection(oracle_idx[r], p)
            o_out, o_lse = o.attend(o.bf16_to_f64(q[r]), latent_values(host_lat[(b, layer)][sel], latent), wl.scale)
            check_attention(o.bf16_to_f64(out_bits[n]), lse[n], o_out, o_lse)
