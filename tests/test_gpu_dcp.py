"""GPU parity of decode context parallelism ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs",
"Reaching 240K context with DCP"), through the C ABI.

The ranks are emulated on one GPU, one after the other: each rank holds its interleaved share of
every request (token s at local position s // world of rank s mod world) in a cache of its own, and
the exchanges are torch.stack of the ranks' tensors.  No kernel waits on another rank.

Checked per row: the sharded indexer scores equal the unsharded ones bit for bit (a key's score
does not depend on where it is cached), so the global selection equals the single-device GPU
top-k exactly and the oracle's within the swap tolerance; every rank's local index buffer names
exactly its share; and the merged attention matches the oracle's attention over the selection.
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
    parts = []
    for r, (cache, batch, lens) in enumerate(ranks):
        lse = torch.empty((R, 64), dtype=torch.float32, device="cuda")
        out, _ = dsa.sparse_mla_decode(cache, batch, gp.q[0], sels[r][1], wl.scale, lse=lse)
        parts.append((out, lse))
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
        gi, li = sels[r][0].cpu().numpy(), sels[r][1].cpu().numpy()
        assert np.array_equal(gi, g0), f"rank {r} selected differently from rank 0"
        mine = (gi >= 0) & (gi % world == r)
        assert np.array_equal(li[mine], gi[mine] // world) and np.all(li[~mine] == -1), f"rank {r}: local buffer"
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
