"""Host logic of decode context parallelism on CPU: two and three gloo ranks, no GPU.

DcpDecode runs its two exchanges through torch.distributed (all_gather_into_tensor) and takes its
device steps from an injected namespace.  Here those steps are float64 stand-ins built on the
oracle, so the test checks what the host side owns: the interleaved sharding, the rank-major
gathers, that every rank gets the same global selection (the single-device top-k of the whole row)
and its own share of it, and that the merged attention is the single-device attention.
"""
import os
import socket
from types import SimpleNamespace

import numpy as np
import pytest

from oracle import dsa_oracle as o

L_ROWS = [50, 23, 7]          # per request: the row's whole length
TOPK, H, DL, DR, SCALE = 6, 3, 5, 2, 0.4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    rng = np.random.default_rng(77)
    scores = [rng.standard_normal(L) for L in L_ROWS]
    for s in scores:
        s[::5] = 0.5                                         # ties across ranks
    rows = [rng.standard_normal((L, DL + DR)) for L in L_ROWS]
    q = rng.standard_normal((len(L_ROWS), H, DL + DR))
    return scores, rows, q


def _fake_ops(rank, world):
    """Stand-ins for the device steps: the 'cache' of a rank is its share of the scores and rows."""
    import torch

    def indexer_scores_topk(owner, batch, q_idx, w, topk, scores_out=None):
        scores_out.fill_(-float("inf"))
        top = torch.full((batch.num_rows, topk), -1, dtype=torch.int32)
        for b, s in enumerate(owner["scores"]):
            scores_out[b, :len(s)] = torch.from_numpy(s)
            top[b] = torch.from_numpy(o.topk_select(s, topk).astype(np.int32))
        return top

    def dcp_candidates(scores, top, rank_, world_):
        assert (rank_, world_) == (rank, world)
        valid = top >= 0
        sc = torch.where(valid, scores.gather(1, top.clamp(min=0).long()), torch.tensor(-float("inf"), dtype=scores.dtype))
        pos = torch.where(valid, top * world + rank, torch.tensor(-1, dtype=torch.int32))
        return sc, pos.to(torch.int32)

    def dcp_select(all_s, all_p, rank_):
        assert all_s.shape[0] == world and rank_ == rank
        k = all_s.shape[2]
        g = torch.full((all_s.shape[1], k), -1, dtype=torch.int32)
        for r in range(all_s.shape[1]):
            cand = sorted((-float(s), int(p)) for s, p in zip(all_s[:, r].flatten(), all_p[:, r].flatten()) if p >= 0)
            chosen = sorted(p for _, p in cand[:k])
            g[r, :len(chosen)] = torch.tensor(chosen, dtype=torch.int32)
        li = torch.full_like(g, -1)
        cnt = torch.zeros(g.shape[0], dtype=torch.int32)
        for r in range(g.shape[0]):
            mine = [int(p) // world for p in g[r] if p >= 0 and p % world == rank]
            li[r, :len(mine)] = torch.tensor(mine, dtype=torch.int32)
            cnt[r] = len(mine)
        return g, li, cnt

    def sparse_mla_decode(layer, batch, q, local_idx, scale, lse=None, row_counts=None):
        assert row_counts is not None and bool(torch.all(local_idx[torch.arange(local_idx.shape[1]) >= row_counts[:, None]] == -1))
        outs, lses = [], []
        for b in range(batch.num_rows):
            sel = local_idx[b][local_idx[b] >= 0].numpy()
            out, l_ = o.attend(q[b].numpy(), layer["rows"][b][sel], scale, DL)
            outs.append(out)
            lses.append(l_)
        return torch.from_numpy(np.stack(outs)), torch.from_numpy(np.stack(lses))

    def dcp_merge(outs, lses):
        merged = [o.lse_merge([(outs[w, b].numpy(), lses[w, b].numpy()) for w in range(world)])
                  for b in range(outs.shape[1])]
        return (torch.from_numpy(np.stack([m[0] for m in merged])), torch.from_numpy(np.stack([m[1] for m in merged])))

    return SimpleNamespace(indexer_scores_topk=indexer_scores_topk, dcp_candidates=dcp_candidates,
                           dcp_select=dcp_select, sparse_mla_decode=sparse_mla_decode, dcp_merge=dcp_merge)


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import torch
    import torch.distributed as dist
    from deepseek_sparse_mla_gb300 import dcp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    scores, rows, q = _problem()
    share = [np.asarray(list(dcp.local_positions(L, rank, world)), dtype=np.int64) for L in L_ROWS]
    assert [len(s) for s in share] == [dcp.local_len(L, rank, world) for L in L_ROWS]
    cache = {"scores": [s[p] for s, p in zip(scores, share)], "rows": [r[p] for r, p in zip(rows, share)]}
    batch = SimpleNamespace(num_rows=len(L_ROWS), max_seq_len=max(len(p) for p in share))
    step = dcp.DcpDecode(rank, world, ops=_fake_ops(rank, world))
    g, li, cnt = step.select(cache, batch, torch.zeros(1), None, TOPK)
    out, lse = step.attend(cache, batch, torch.from_numpy(q), li, cnt, SCALE)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), g=g.numpy(), li=li.numpy(), out=out.numpy(), lse=lse.numpy())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dcp_decode_on_gloo_ranks(tmp_path, world):
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    scores, rows, q = _problem()
    for b, L in enumerate(L_ROWS):
        want = o.topk_select(scores[b], TOPK)
        sel = want[want >= 0]
        want_out, want_lse = o.attend(q[b], rows[b][sel], SCALE, DL)
        for r, x in enumerate(res):
            assert np.array_equal(x["g"][b], want), f"rank {r} row {b}: selection"
            mine = want[(want >= 0) & (want % world == r)] // world
            assert np.array_equal(x["li"][b][:len(mine)], mine) and np.all(x["li"][b][len(mine):] == -1)
            assert np.allclose(x["out"][b], want_out, atol=1e-12) and np.allclose(x["lse"][b], want_lse, atol=1e-12)


def test_dcp_decode_rejects_bad_ranks():
    from deepseek_sparse_mla_gb300 import dcp
    with pytest.raises(ValueError):
        dcp.DcpDecode(2, 2, gather=lambda t: t, ops=SimpleNamespace())
    with pytest.raises(ValueError):
        dcp.DcpDecode(0, 9, gather=lambda t: t, ops=SimpleNamespace())
    step = dcp.DcpDecode(0, 4, gather=lambda t: t, ops=SimpleNamespace())
    with pytest.raises(ValueError):
        step.select(None, SimpleNamespace(num_rows=1, max_seq_len=1), None, None, 8192)


def test_local_lengths_partition_the_row():
    from deepseek_sparse_mla_gb300 import dcp
    for L in (1, 7, 64, 1001):
        for world in (1, 2, 3, 8):
            assert sum(dcp.local_len(L, r, world) for r in range(world)) == L
            assert sorted(p for r in range(world) for p in dcp.local_positions(L, r, world)) == list(range(L))
