"""GPU parity of decode context parallelism ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs",
"Reaching 240K context with DCP"), through the C ABI.

The ranks are emulated on one GPU, one after the other: each rank holds its interleaved share of
every request (token s at local position s // world of rank s mod world) in a cache of its own, and
the exchanges are torch.stack of the ranks' tensors.  No kernel waits on another rank.

Checked per row: the sharded indexer scores equal the unsharded ones bit for bit (a key's score
does not depend on where it is cached), so the global selection equals the single-device GPU
top-k exactly and the oracle's within the swap tolerance; every rank's local index buffer names
exactly its share (compacted, with its size); each rank's attention over its share with the sizes
(the ragged entry point) matches the attention without them; and the merged attention matches the
oracle's attention over the selection.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from parity import (GpuProblem, HostProblem, bf16_tensor_to_f64, check_attention, check_topk)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def shard(hp, world, rank):
    """This rank's cache and decode batch: its tokens of every request, in local order."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = hp.wl
    lens = [len(o.dcp_local_positions(L, rank, world)) for L in wl.seq_lens]
    lw = wlm.Workload(f"{wl.name}_r{rank}", lens, [1] * len(lens), wl.page_size, wl.key_format, wl.topk, 1,
                      wl.seed + 17 * (rank + 1))
    cache = dsa.LayerCache(lw.num_pages, lw.page_size, wl.key_format, "cuda")
    for b, L in enumerate(wl.seq_lens):
        g = o.dcp_local_positions(L, rank, world)
        lat = hp.latent[0][b][g]
        slots = torch.from_numpy(lw.slots(b, np.arange(len(g))).astype(np.int64)).cuda()
        dsa.kv_append(cache, wlm.bits_to_torch(np.ascontiguousarray(lat[:, :512]), "cuda"),
                      wlm.bits_to_torch(np.ascontiguousarray(lat[:, 512:]), "cuda"), slots,
                      k_idx=wlm.bits_to_torch(np.ascontiguousarray(hp.keys[b][g]), "cuda"))
    batch = dsa.Batch(torch.from_numpy(lw.block_table).cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda"),
                      None, num_rows=lw.num_rows, max_seq_len=lw.max_seq_len)
    return cache, batch, lens


def run_dcp(wl, world):
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    full_idx, full_scores = gp.indexer()
    ranks = [shard(hp, world, r) for r in range(world)]
    k, R = wl.topk, wl.num_rows
    # rank-local indexer and candidates
    cands, local_scores = [], []
    for r, (cache, batch, lens) in enumerate(ranks):
        sc = torch.empty((R, batch.max_seq_len), dtype=torch.float32, device="cuda")
        top = dsa.indexer_scores_topk(cache, batch, gp.q_idx, gp.w, k, scores_out=sc)
        cands.append(dsa.dcp_candidates(sc, top, r, world))
        local_scores.append(sc)
    all_s = torch.stack([c[0] for c in cands])
    all_p = torch.stack([c[1] for c in cands])
    sels = [dsa.dcp_select(all_s, all_p, r) for r in range(world)]
    parts, plain = [], []
    for r, (cache, batch, lens) in enumerate(ranks):
        lse = torch.empty((R, 64), dtype=torch.float32, device="cuda")
        out, _ = dsa.sparse_mla_decode(cache, batch, gp.q[0], sels[r][1], wl.scale, lse=lse, row_counts=sels[r][2])
        parts.append((out, lse))
        plain.append(dsa.sparse_mla_decode(cache, batch, gp.q[0], sels[r][1], wl.scale,
                                           lse=torch.empty((R, 64), dtype=torch.float32, device="cuda")))
    out, lse = dsa.dcp_merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
    torch.cuda.synchronize()

    fs, fi = full_scores.cpu().numpy(), full_idx.cpu().numpy()
    for r in range(world):
        ls = local_scores[r].cpu().numpy()
        for b, L in enumerate(wl.seq_lens):
            g = o.dcp_local_positions(L, r, world)
            assert np.array_equal(ls[b, :len(g)].view(np.uint32), fs[b, g].view(np.uint32)), \
                f"rank {r} row {b}: sharded scores differ from the unsharded ones"
    g0 = sels[0][0].cpu().numpy()
    o_idx, o_scores = hp.oracle_topk()
    for r in range(world):
        gi, li, cnt = (t.cpu().numpy() for t in sels[r])
        assert np.array_equal(gi, g0), f"rank {r} selected differently from rank 0"
        for b in range(R):
            mine = gi[b][(gi[b] >= 0) & (gi[b] % world == r)] // world
            assert cnt[b] == len(mine), f"rank {r} row {b}: share size"
            assert np.array_equal(li[b][:len(mine)], mine) and np.all(li[b][len(mine):] == -1), f"rank {r}: local buffer"
        # the sizes only shorten the work: same result as the attention over the whole buffer
        g_o, g_l = bf16_tensor_to_f64(parts[r][0]), parts[r][1].cpu().numpy()
        p_o, p_l = bf16_tensor_to_f64(plain[r][0]), plain[r][1].cpu().numpy()
        assert np.abs(g_o - p_o).max() <= 2e-2, f"rank {r}: ragged attention differs from the full-width call"
        fin = np.isfinite(p_l)
        assert np.array_equal(fin, np.isfinite(g_l)) and np.all(np.abs(g_l[fin] - p_l[fin]) <= 1e-4 * np.maximum(1, np.abs(p_l[fin])))
    for b, L in enumerate(wl.seq_lens):
        assert np.array_equal(g0[b], fi[b]), f"row {b}: DCP selection differs from the single-device top-k"
        check_topk(g0[b], o_idx[b], o_scores[b], L - 1, k)
    o_out, o_lse = hp.oracle_attention(0, g0)
    check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)
    return g0, [p[1].cpu().numpy() for p in parts]


@pytest.mark.parametrize("world,fmt,topk", [(2, "fp8", 2048), (3, "bf16", 512), (4, "fp8", 64), (8, "fp8", 2048)])
def test_dcp_decode_parity(world, fmt, topk):
    wl = wlm.Workload(f"dcp{world}", [6000, 2100, 9001, 500], [1] * 4, 64, fmt, topk, 1, 4100 + world)
    run_dcp(wl, world)


def test_dcp_world_one_is_the_single_device_step():
    wl = wlm.Workload("dcp1", [3000, 700], [1, 1], 64, "bf16", 256, 1, 4109)
    run_dcp(wl, 1)


def test_dcp_rank_without_selected_positions():
    """With world 8 and a budget of 4, at least four ranks hold none of a row's selected positions:
    their local attention runs over an all -1 buffer, gives lse = -inf, and drops out of the merge."""
    wl = wlm.Workload("dcp_short", [9, 16, 12], [1] * 3, 16, "bf16", 4, 1, 4110)
    g0, lses = run_dcp(wl, 8)
    for r in range(8):
        for b in range(3):
            if not np.any((g0[b] >= 0) & (g0[b] % 8 == r)):
                assert np.all(np.isneginf(lses[r][b])), f"rank {r} row {b}: nothing selected but lse finite"


@pytest.mark.parametrize("topk", [2048, 512])
def test_ragged_attention_matches_the_oracle(topk):
    """Row counts of 0, 1, a tile, a tile and one, a ragged middle and the whole buffer, over index
    buffers whose first count entries are the oracle's selection (ascending) and -1 after."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    lens = [9000, 700, 5000, 3000, 12000, 2500, 800, 4096]
    wl = wlm.Workload("ragged", lens, [1] * len(lens), 64, "bf16", topk, 1, 4120 + topk)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    o_idx, _ = hp.oracle_topk()
    counts = [0, 1, 64, 65, topk // 3 + 7, topk, 129, topk - 1]
    buf = np.full((wl.num_rows, topk), -1, dtype=np.int32)
    for r, c in enumerate(counts):
        sel = o_idx[r][o_idx[r] >= 0]
        c = min(c, len(sel))
        counts[r] = c
        buf[r, :c] = sel[:c]
    idx = torch.from_numpy(buf).cuda()
    lse = torch.empty((wl.num_rows, 64), dtype=torch.float32, device="cuda")
    out, _ = dsa.sparse_mla_decode(gp.caches[0], gp.batch, gp.q[0], idx, wl.scale, lse=lse,
                                   row_counts=torch.tensor(counts, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    o_out, o_lse = hp.oracle_attention(0, buf)
    check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)


def test_dcp_merge_against_the_oracle():
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    rng = np.random.default_rng(4111)
    world, R = 5, 3
    outs = wlm.bf16_bits(rng.standard_normal((world, R, 64, 512)).astype(np.float32))
    lses = (rng.standard_normal((world, R, 64)) * 4).astype(np.float32)
    lses[1, 0, :] = -np.inf                               # a rank with nothing selected in row 0
    lses[:, 2, 7] = -np.inf                               # a head with nothing selected anywhere
    out, lse = dsa.dcp_merge(wlm.bits_to_torch(outs, "cuda"), torch.from_numpy(lses).cuda())
    torch.cuda.synchronize()
    g_out, g_lse = bf16_tensor_to_f64(out), lse.cpu().numpy()
    of = o.bf16_to_f64(outs)
    for r in range(R):
        parts = [(of[w, r], lses[w, r].astype(np.float64)) for w in range(world)]
        want_out, want_lse = o.lse_merge(parts)
        dead = np.isneginf(lses[:, r, :]).all(axis=0)
        want_out[dead], want_lse[dead] = 0.0, -np.inf
        check_attention(g_out[r], g_lse[r], want_out, want_lse)


@pytest.mark.parametrize("L,world,k,ties", [(9000, 2, 2048, False), (9000, 8, 2048, True), (600000, 2, 2048, True),
                                            (300000, 8, 2048, False), (1000, 3, 2048, False), (70000, 4, 64, True)])
def test_dcp_select_against_the_oracle(L, world, k, ties):
    """dsa_dcp_select alone on candidates built from a score vector as each rank's local top-k:
    rows whose positions fit the bitmap ordering (below 262,144) and rows that take the sort, with
    heavy ties across ranks, rows shorter than k and a budget below one tile."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    rng = np.random.default_rng(L + world + k)
    R = 3
    lens = [L, max(1, L // 3), min(L, 5)]
    all_s = np.full((world, R, k), -np.inf, dtype=np.float32)
    all_p = np.full((world, R, k), -1, dtype=np.int32)
    rows = []
    for r, n in enumerate(lens):
        sc = rng.standard_normal(n).astype(np.float32)
        if ties:
            sc[rng.integers(0, n, n // 2)] = np.float32(1.5)          # a tie that straddles the k-th score
        rows.append(sc)
        for w in range(world):
            share = o.dcp_local_positions(n, w, world)
            loc = o.topk_select(sc[share].astype(np.float64), k)
            m = loc >= 0
            all_s[w, r, :m.sum()] = sc[share][loc[m]]
            all_p[w, r, :m.sum()] = share[loc[m]]
    for rank in sorted({0, world - 1}):
        g, li, cnt = dsa.dcp_select(torch.from_numpy(all_s).cuda(), torch.from_numpy(all_p).cuda(), rank)
        torch.cuda.synchronize()
        g, li, cnt = g.cpu().numpy(), li.cpu().numpy(), cnt.cpu().numpy()
        for r, sc in enumerate(rows):
            want = o.topk_select(sc.astype(np.float64), k)
            assert np.array_equal(g[r], want), f"rank {rank} row {r}: global selection"
            mine = want[(want >= 0) & (want % world == rank)] // world
            assert cnt[r] == len(mine) and np.array_equal(li[r][:len(mine)], mine) and np.all(li[r][len(mine):] == -1)
