"""Decode context parallelism over torch.distributed: one rank per GPU, the KV of every request
sharded along the sequence.

("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Reaching 240K context with DCP": sharding the
KV along the sequence lets each rank score only its share of the keys.)  Token s of a request
lives on rank s mod world at local position s // world (``local_positions``), so every rank
holds a near-equal share of every request and each rank's cache is an ordinary paged cache over
its local positions.  A decode step on one rank is:

  1. ``indexer_scores_topk`` over the local cache (its local top-k and scores);
  2. ``dcp_candidates`` -> all-gather -> ``dcp_select``: the top-k of the union of every rank's
     local top-k, which holds the whole row's top-k, so the selection equals the single-device one;
  3. ``sparse_mla_decode`` over the local cache with this rank's share of that selection (a
     compacted buffer with its per-row sizes, so the rank's attention covers only its share);
  4. all-gather of out / lse -> ``dcp_merge`` (LSE merge): the single-device attention.

The two all-gathers are the only exchanges.  ``gather`` is any callable that maps this rank's
tensor to the stacked tensor of every rank's ([world, *shape], rank-major):
``all_gather_stack`` does it with ``torch.distributed.all_gather_into_tensor``.  The device steps
are taken from ``ops`` (the library's functions by default) so that the host logic can run
against stand-ins.
"""
from __future__ import annotations

from types import SimpleNamespace

import torch

from . import DEFAULT_SCALE, HEADS


def local_positions(seq_len: int, rank: int, world: int) -> range:
    """Global positions of a request's tokens that rank holds, in local order (local position j
    holds global position j * world + rank)."""
    return range(rank, seq_len, world)


def local_len(seq_len: int, rank: int, world: int) -> int:
    """Number of a request's tokens that rank holds."""
    return max(0, (seq_len - rank + world - 1) // world)


def all_gather_stack(t: torch.Tensor, group=None) -> torch.Tensor:
    """[world, *t.shape] of every rank's t, rank-major (torch.distributed.all_gather_into_tensor)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    flat = t.contiguous().reshape(-1)
    out = torch.empty(world * flat.numel(), dtype=t.dtype, device=t.device)
    dist.all_gather_into_tensor(out, flat, group=group)
    return out.view((world,) + tuple(t.shape))


def _library_ops():
    from . import dcp_candidates, dcp_merge, dcp_select, indexer_scores_topk, sparse_mla_decode
    return SimpleNamespace(indexer_scores_topk=indexer_scores_topk, dcp_candidates=dcp_candidates,
                           dcp_select=dcp_select, sparse_mla_decode=sparse_mla_decode, dcp_merge=dcp_merge)


class DcpDecode:
    """One rank's side of a decode step under context parallelism.

    rank, world  this rank and the number of ranks (1..8, world * topk <= 16384);
    gather       callable: tensor -> [world, *shape] of every rank's (default: all_gather_stack);
    ops          the device steps (default: this package's C-ABI wrappers)."""

    def __init__(self, rank: int, world: int, gather=None, ops=None):
        if not 1 <= world <= 8 or not 0 <= rank < world:
            raise ValueError(f"rank {rank} / world {world}: world must be 1..8 and 0 <= rank < world")
        self.rank, self.world = int(rank), int(world)
        self.gather = gather if gather is not None else all_gather_stack
        self.ops = ops if ops is not None else _library_ops()

    def select(self, owner, batch, q_idx, w, topk: int):
        """Indexer over the local cache, candidate exchange, global top-k.  batch describes the
        local cache (decode rows: seq_lens are the local lengths, max_seq_len their bound).
        Returns (global_idx [R, topk], local_idx [R, topk], local_count [R]), int32."""
        if self.world * topk > 16384:
            raise ValueError(f"world * topk = {self.world * topk} exceeds 16384")
        R = batch.num_rows
        scores = torch.empty((R, batch.max_seq_len), dtype=torch.float32, device=q_idx.device)
        local_top = self.ops.indexer_scores_topk(owner, batch, q_idx, w, topk, scores_out=scores)
        cand_s, cand_p = self.ops.dcp_candidates(scores, local_top, self.rank, self.world)
        return self.ops.dcp_select(self.gather(cand_s), self.gather(cand_p), self.rank)

    def attend(self, layer, batch, q, local_idx, local_count=None, scale: float = DEFAULT_SCALE):
        """Local sparse MLA over this rank's share of the selection, out/lse exchange, LSE merge.
        Returns (out [R, 64, 512] bf16, lse [R, 64] fp32), identical on every rank."""
        R = batch.num_rows
        lse = torch.empty((R, HEADS), dtype=torch.float32, device=q.device)
        out, lse = self.ops.sparse_mla_decode(layer, batch, q, local_idx, scale, lse=lse, row_counts=local_count)
        return self.ops.dcp_merge(self.gather(out), self.gather(lse))
