#!/usr/bin/env python3
"""Throughput of the GLM-5.2 DSA decode step on GB300.

One step = one IndexShare group of the decode workload "decode batch 64,
contexts U[16K, 128K], page size 64, fp8 index keys, 1 owner + 3 shared layers":
append the step's 64 new tokens to 4 layers, score + top-k on the owner layer,
and absorbed sparse MLA on all 4 layers with the owner's index buffer.  The
metric is layer-steps/s (4 per group step).

Default run: N=1.  Under torchrun every rank runs its own replica (requests are
independent; no collective on the data path) and the JSON line reports the
aggregate over ranks ("scaling": "weak").

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wlm  # noqa: E402

METRIC = "sparse-DSA decode layer-steps/s (indexer+top-k+MLA) @128K ctx; % of HBM roofline"
UNIT = "layer-steps/s"
DEFAULT_WORKLOAD = "decode_b64_fp8_indexshare"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# the workload resident on the device
# ---------------------------------------------------------------------------
class DeviceProblem:
    """A full-size workload resident in HBM: every layer's paged cache holds each request's
    prefix (drawn on the device with torch's seeded generator and appended through the
    library), and the step's inputs (new tokens, queries, metadata) are on the device."""

    def __init__(self, wl: wlm.Workload, device="cuda", selection="token", locality_noise=0.17):
        import torch
        import deepseek_sparse_mla_gb300 as dsa
        self.wl, self.dev, self.selection = wl, device, selection
        B, R, layers = wl.num_requests, wl.num_rows, wl.layers
        self.caches = [dsa.LayerCache(wl.num_pages, wl.page_size, wl.key_format if l == 0 else None, device,
                                      latent_format=wl.latent_format)
                       for l in range(layers)]
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        self.seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=device)
        self.qsl = None if wl.is_decode else torch.from_numpy(wl.query_start_loc).to(device)
        self.batch = dsa.Batch(self.block_table, self.seq_lens, self.qsl, num_rows=R, max_seq_len=wl.max_seq_len)
        new_c, new_r, new_k = [[] for _ in range(layers)], [[] for _ in range(layers)], []
        for b in range(B):
            L, q = wl.seq_lens[b], wl.q_lens[b]
            pre = torch.from_numpy(wl.slots(b, np.arange(L - q))).to(device)
            for l in range(layers):
                x = wlm.request_latent_device(wl, b, l, device)
                k = wlm.request_index_keys_device(wl, b, device) if l == 0 else None
                if L - q > 0:
                    dsa.kv_append(self.caches[l], x[:L - q, :512].contiguous(), x[:L - q, 512:].contiguous(), pre,
                                  k_idx=None if k is None else k[:L - q].contiguous())
                new_c[l].append(x[L - q:, :512])
                new_r[l].append(x[L - q:, 512:])
                if l == 0:
                    new_k.append(k[L - q:])
            torch.cuda.synchronize()
        self.new_c = [torch.cat(v).contiguous() for v in new_c]
        self.new_r = [torch.cat(v).contiguous() for v in new_r]
        self.new_k = torch.cat(new_k).contiguous()
        self.slots = torch.from_numpy(wl.new_token_slots()).to(device)
        q_idx, w = wlm.indexer_queries(wl)
        self.q_idx = wlm.bits_to_torch(q_idx, device)
        self.w = torch.from_numpy(w).to(device)
        # the layers' queries and outputs lie back to back ([layers, R, ...]), so a layer group's attention
        # can run as one call over the stacked tensors
        self.q = list(torch.stack([wlm.bits_to_torch(wlm.mla_queries(wl, l), device) for l in range(layers)]).unbind(0))
        self.topk_idx = torch.empty((R, wl.topk), dtype=torch.int32, device=device)
        self.out = list(torch.empty((layers, R, 64, 512), dtype=torch.bfloat16, device=device).unbind(0))
        self.lse = list(torch.empty((layers, R, 64), dtype=torch.float32, device=device).unbind(0))
        # decode layer groups (one index buffer for every layer): one attention call for all layers
        self.group_attention = wl.is_decode and layers > 1
        self.ws_idx = torch.empty(dsa.indexer_workspace_bytes(R, wl.max_seq_len, wl.topk), dtype=torch.uint8,
                                  device=device)
        self.ws_mla = torch.empty(dsa.mla_workspace_bytes(layers * R, wl.topk), dtype=torch.uint8, device=device)
        self.loc_idx = None
        if selection == "locality":
            self.loc_idx = torch.from_numpy(locality_selection(wl, locality_noise)).to(device)
        if selection == "page":
            # page-granular selection: topk / page_size pages, expanded into the same-size index buffer
            self.page_budget = wl.topk // wl.page_size
            assert self.page_budget * wl.page_size == wl.topk, "the token budget must be whole pages"
            self.page_idx = torch.empty((R, self.page_budget), dtype=torch.int32, device=device)
            self.ws_page = torch.empty(dsa.indexer_page_workspace_bytes(R, wl.max_seq_len, wl.page_size,
                                                                        self.page_budget),
                                       dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def step(self, marks=None, io=None, calls=None):
        """One DSA step of the layer group on the current stream.  io: the set of per-step inputs
        and outputs to use (this object's own by default, or one made by io_set()).  calls: issue only
        the step's first `calls` library calls (append, indexer, then one attention call per layer)."""
        import deepseek_sparse_mla_gb300 as dsa
        wl = self.wl
        io = self if io is None else io
        n_calls = self.num_calls() if calls is None else calls
        mla = dsa.sparse_mla_decode if wl.is_decode else dsa.sparse_mla_prefill
        if marks is not None:
            marks.mark("append")
        dsa.kv_append_layers(self.caches, io.new_c, io.new_r, io.slots,
                             k_idx=[io.new_k] + [None] * (wl.layers - 1))
        if n_calls < 2:
            return
        if marks is not None:
            marks.mark("indexer")
        if self.selection == "page":
            dsa.indexer_page_topk(self.caches[0], io.batch, io.q_idx, io.w, self.page_budget, page_idx=self.page_idx,
                                  token_idx=self.topk_idx, workspace=self.ws_page)
        else:
            dsa.indexer_scores_topk(self.caches[0], io.batch, io.q_idx, io.w, wl.topk, topk_idx=self.topk_idx,
                                    workspace=self.ws_idx)
        idx = self.topk_idx if self.loc_idx is None else self.loc_idx
        if self.group_attention and n_calls > 2:
            if marks is not None:
                marks.mark("attention")
            dsa.sparse_mla_decode_layers(self.caches, io.batch, stacked(io.q), idx, wl.scale, out=stacked(io.out),
                                         lse=stacked(io.lse), workspace=self.ws_mla)
            if marks is not None:
                marks.mark(None)
            return
        for l in range(min(wl.layers, n_calls - 2)):
            if marks is not None:
                marks.mark("attention")
            mla(self.caches[l], io.batch, io.q[l], idx, wl.scale, out=io.out[l], lse=io.lse[l],
                workspace=self.ws_mla)
        if marks is not None:
            marks.mark(None)

    def num_calls(self):
        """Library calls in a step: append, indexer, then the attention (one call per layer, or one for
        the layer group)."""
        return 3 if self.group_attention else 2 + self.wl.layers

    def io_set(self):
        """A second set of the step's device inputs and outputs (same values), so that the copies of
        one step can overlap the kernels of another."""
        import types
        import deepseek_sparse_mla_gb300 as dsa
        c = lambda t: None if t is None else t.clone()   # noqa: E731
        io = types.SimpleNamespace(new_c=[c(t) for t in self.new_c], new_r=[c(t) for t in self.new_r],
                                   new_k=c(self.new_k), slots=c(self.slots), q_idx=c(self.q_idx), w=c(self.w),
                                   q=list(c(stacked(self.q)).unbind(0)), block_table=c(self.block_table),
                                   seq_lens=c(self.seq_lens), qsl=c(self.qsl),
                                   out=list(torch_empty_like(stacked(self.out)).unbind(0)),
                                   lse=list(torch_empty_like(stacked(self.lse)).unbind(0)))
        io.batch = dsa.Batch(io.block_table, io.seq_lens, io.qsl, num_rows=self.wl.num_rows,
                             max_seq_len=self.wl.max_seq_len)
        return io

    # per-step host<->device traffic of the end-to-end measurement
    def step_inputs(self, io=None):
        io = self if io is None else io
        return (io.new_c + io.new_r + [io.new_k, io.slots, io.q_idx, io.w] + io.q +
                [io.block_table, io.seq_lens] + ([io.qsl] if io.qsl is not None else []))

    def step_outputs(self, io=None):
        io = self if io is None else io
        return io.out + io.lse

    def assign_io(self, io, ins, outs):
        """Point io's step inputs and outputs at `ins` / `outs` (in step_inputs / step_outputs order)."""
        import deepseek_sparse_mla_gb300 as dsa
        L = self.wl.layers
        io.new_c, io.new_r = list(ins[:L]), list(ins[L:2 * L])
        io.new_k, io.slots, io.q_idx, io.w = ins[2 * L:2 * L + 4]
        io.q = list(ins[2 * L + 4:3 * L + 4])
        io.block_table, io.seq_lens = ins[3 * L + 4:3 * L + 6]
        io.qsl = ins[3 * L + 6] if len(ins) > 3 * L + 6 else None
        io.out, io.lse = list(outs[:L]), list(outs[L:])
        io.batch = dsa.Batch(io.block_table, io.seq_lens, io.qsl, num_rows=self.wl.num_rows,
                             max_seq_len=self.wl.max_seq_len)


def capture_step(prob, lib, io=None, calls=None):
    """The step (or its first `calls` library calls) captured once into a CUDA graph (the library's
    calls allocate nothing and never synchronise, so they capture as they are, programmatic launch
    edges included).  Returns the graph and the number of the library's kernels one replay runs."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prob.step(io=io, calls=calls)                    # a first run outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = lib.dsa_kernel_launches()
    with torch.cuda.graph(g):
        prob.step(io=io, calls=calls)
    torch.cuda.synchronize()
    return g, int(lib.dsa_kernel_launches() - n0)


def replay_ms(graph, reps=30, warm=5):
    """Mean device time of one replay of `graph` (CUDA events on the current stream, back to back)."""
    import torch
    for _ in range(warm):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def locality_selection(wl: wlm.Workload, noise: float) -> np.ndarray:
    """Index buffer [R, topk] of locality-shaped page selections: the rows of a request, in blocks of up
    to 64, rank its pages by one shared N(0, 1) score per page plus N(0, noise^2) per row
    (workloads.locality_page_scores), and each row keeps the topk / page_size best pages among those it
    can see, expanded to their visible positions (ascending, -1 padded).  A small noise makes the rows
    of a block select nearly the same pages ("Making GLM-5.2 Sparse on TPUs", "Reuse pages across
    queries"); a large one, independent uniformly random pages."""
    P, k = wl.page_size, wl.topk
    budget = max(1, k // P)
    out = np.full((wl.num_rows, k), -1, dtype=np.int32)
    pos = wl.row_position()
    r0 = 0
    for b, (L, q) in enumerate(zip(wl.seq_lens, wl.q_lens)):
        pages = -(-L // P)
        for blk in range(0, q, 64):
            rows = range(r0 + blk, r0 + min(q, blk + 64))
            sc = wlm.locality_page_scores(len(rows), pages, noise, wl.seed * 1000 + b * 64 + blk // 64)
            for i, r in enumerate(rows):
                vis = int(pos[r]) // P + 1                       # pages holding a visible position
                keep = np.sort(np.argsort(-sc[i, :vis], kind="stable")[:budget])
                toks = (keep[:, None] * P + np.arange(P)).ravel()
                toks = toks[toks <= pos[r]][:k]
                out[r, :toks.size] = toks
        r0 += q
    return out


def torch_empty_like(t):
    import torch
    return torch.empty_like(t)


def stacked(ts):
    """[len(ts), ...] view of equally shaped contiguous tensors that lie back to back in memory."""
    import torch
    t0 = ts[0]
    step = t0.numel()
    for i, t in enumerate(ts):
        if not t.is_contiguous() or t.shape != t0.shape or t.data_ptr() != t0.data_ptr() + i * step * t0.element_size():
            raise ValueError("the layers' tensors do not lie back to back")
    return torch.as_strided(t0, (len(ts),) + tuple(t0.shape), (step,) + tuple(t0.stride()))


def pack_views(tensors, device):
    """One flat device buffer holding copies of `tensors` (each at a 256-byte aligned offset) and views
    of it with their shapes and dtypes, so that a step's inputs (or outputs) move in one copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    flat = torch.empty(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        v = flat[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return flat, views


class Marks:
    """CUDA events between the library calls of a step (same stream as the launches)."""

    def __init__(self):
        self.spans = {}
        self._open = []

    def mark(self, name):
        import torch
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        if self._open:
            self._open[-1][2] = e
        if name is not None:
            self._open.append([name, e, None])

    def collect(self):
        for name, a, b in self._open:
            self.spans.setdefault(name, []).append(a.elapsed_time(b))
        self._open = []


# ---------------------------------------------------------------------------
# algorithmic bytes (what the step must move; scores/partials are overhead)
# ---------------------------------------------------------------------------
def algorithmic_bytes(wl: wlm.Workload) -> dict:
    pos = wl.row_position()
    R, k = wl.num_rows, wl.topk
    selected = np.minimum(k, pos + 1).sum()
    keys = sum(wl.seq_lens) * wl.key_bytes_per_token()
    indexer = keys + R * 32 * 128 * 2 + R * 32 * 4 + R * k * 4
    # one cached latent row: 1152 bytes of bf16, or a packed 8-bit row of 640 bytes and its 4-byte scale
    row = 1152 if wl.latent_format == "bf16" else 640 + 4
    attention = selected * row + R * 64 * 576 * 2 + R * 64 * 512 * 2 + R * 64 * 4 + R * k * 4
    key_in = 256
    key_out = wl.key_bytes_per_token()
    append_owner = R * (1152 + row + key_in + key_out)
    append_shared = R * (1152 + row)
    # useful flops: a (row, visible key) costs 32 heads x 128 multiply-adds in the indexer; a (row, selected
    # entry) costs 64 heads x (576 + 512) multiply-adds in attention (QK over [c_KV | k_R], PV over c_KV)
    indexer_flops = float((pos + 1).sum()) * 2 * 32 * 128
    attention_flops = float(selected) * 2 * 64 * (576 + 512)
    return {"indexer": float(indexer), "attention": float(attention), "append_owner": float(append_owner),
            "indexer_flops": indexer_flops, "attention_flops": attention_flops,
            "append_shared": float(append_shared), "index_key_bytes": float(keys),
            "gather_bytes_per_layer": float(selected * row),
            "step": float(indexer + wl.layers * attention + append_owner + (wl.layers - 1) * append_shared)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Dense bf16 TFLOP/s: the burst figure (each call is timed alone, not over a seconds-long loop)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def source_digest(files) -> str:
    """First 16 hex digits of the sha256 of the named csrc files, concatenated in order."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "deepseek_sparse_mla_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_traffic(call: str, files, workload: str):
    """DRAM bytes per call from profiles/traffic.json, if it was captured (or scaled) for this workload
    on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            doc = json.load(f)
        ent = doc[call]
        if doc.get("workload") != workload or ent.get("source_sha256_16") != source_digest(files):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 200 ms; started before warm-up so its start-up never overlaps the
    timed region, and only the samples taken inside [t_begin, t_end] are kept."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.t_begin = None
        self.t_end = None

    def mark_begin(self):
        self.t_begin = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def start(self):
        import torch
        ident = None
        try:
            ident = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            if not ident.startswith("GPU-"):
                ident = "GPU-" + ident
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")
            ident = vis[torch.cuda.current_device()] if vis and vis[0] else "0"
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_begin is not None and self.t_begin - 0.25 <= r[0] <= (self.t_end or 1e30) + 0.25]
        use = inside if inside else rows[-3:]
        reasons = set()
        for r in use:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in use]
        mx = [r[2] for r in use]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if inside else "last samples before stop (timed region shorter than 200 ms)"}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no collective on the data path)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus, backend="nccl", device="cuda"):
    """(rank, world) from the launcher's environment; joins the process group when world > 1.

    Ranks never exchange data on the DSA path: each serves its own replica (its own requests and
    caches).  The group only carries the barriers and the max-over-ranks of the timings."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    if device == "cuda":
        torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend == "nccl":
            dist.init_process_group(backend, device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(name: str, rank: int) -> wlm.Workload:
    """Rank r's replica: the named workload's shape and recipe, drawn from its own seed (rank 0 is
    the canonical workload), so ranks serve disjoint request sets of the same size."""
    wl = (wlm.FULL[name] if name in wlm.FULL else wlm.PROFILE[name])()
    if rank == 0:
        return wl
    return wlm.Workload(f"{wl.name}_replica{rank}", list(wl.seq_lens), list(wl.q_lens), wl.page_size, wl.key_format,
                        wl.topk, wl.layers, wl.seed + 100000 * rank)


def aggregate_rate(elapsed_ms_max: float, world: int, layers: int, steps: int) -> float:
    """Whole-job layer-steps/s: every rank ran `steps` group steps of `layers` layers; the job
    took as long as its slowest rank."""
    return world * layers * steps / (elapsed_ms_max / 1e3)


# ---------------------------------------------------------------------------
# the oracle as a CPU baseline (bounded sample)
# ---------------------------------------------------------------------------
def oracle_request_problem(wl, b, device):
    """One request of the workload as a stand-alone oracle problem (its own pages, identity page table).

    Data come from the same seeded device generator the GPU problem was built from."""
    from oracle import dsa_oracle as o
    L, q = wl.seq_lens[b], wl.q_lens[b]
    P = wl.page_size
    pages = -(-L // P)
    bt = np.arange(pages, dtype=np.int32)[None, :]
    slots = np.arange(L, dtype=np.int64)
    caches = []
    for l in range(wl.layers):
        lat = wlm.torch_to_bits(wlm.request_latent_device(wl, b, l, device))
        keys = wlm.torch_to_bits(wlm.request_index_keys_device(wl, b, device)) if l == 0 else None
        c = o.PagedCache(pages, P, wl.key_format if l == 0 else None,
                         latent_format="e4m3" if wl.latent_format == "fp8" else "bf16")
        c.append(lat[:L - q, :512], lat[:L - q, 512:], slots[:L - q],
                 k_idx_bits=None if keys is None else keys[:L - q])
        caches.append((c, lat[L - q:], None if keys is None else keys[L - q:]))
    return caches, bt


def time_oracle_request(wl, b, caches, bt, q_idx, w, qs):
    """Seconds the oracle takes for request b's share of one step (append, indexer, top-k, all layers)."""
    from oracle import dsa_oracle as o
    L, q = wl.seq_lens[b], wl.q_lens[b]
    r0 = int(wl.query_start_loc[b])
    qsl = np.array([0, q], dtype=np.int32)
    t0 = time.perf_counter()
    for l, (c, new_lat, new_keys) in enumerate(caches):
        c.append(new_lat[:, :512], new_lat[:, 512:], np.arange(L - q, L), k_idx_bits=new_keys)
    idx, _ = o.indexer_topk(caches[0][0], bt, [L], qsl, q_idx[r0:r0 + q], w[r0:r0 + q], wl.topk)
    for l, (c, _, _) in enumerate(caches):
        o.sparse_mla(c, bt, [L], qsl, qs[l][r0:r0 + q], idx, wl.scale)
    return time.perf_counter() - t0


def stratified_requests(wl, n):
    order = np.argsort(wl.seq_lens, kind="stable")
    pick = order[np.unique(np.linspace(0, len(order) - 1, n).round().astype(int))]
    return [int(b) for b in pick]


def cpu_baseline(wl, device, n_req=64):
    q_idx, w = wlm.indexer_queries(wl)
    qs = [wlm.mla_queries(wl, l) for l in range(wl.layers)]
    total = 0.0
    picked = stratified_requests(wl, n_req)
    for b in picked:
        caches, bt = oracle_request_problem(wl, b, device)
        total += time_oracle_request(wl, b, caches, bt, q_idx, w, qs)
    step_s = total * wl.num_requests / len(picked)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": wl.layers / step_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"float64 numpy oracle on {len(picked)} of {wl.num_requests} requests (stratified by "
                       f"context length: {[wl.seq_lens[b] for b in picked]}), append + indexer + top-k + "
                       f"{wl.layers} attention layers, {total:.2f} s, scaled by request count"),
            "seconds": total}


# ---------------------------------------------------------------------------
# main arms
# ---------------------------------------------------------------------------
def reference_main(args):
    """The oracle on the host cores, timed as it stands.  Every step (warm-up and timed alike) runs the
    same stratified sample of the workload's requests (spread over the context lengths) through append,
    indexer, top-k and every attention layer; the rate counts the layer-steps that sample makes up
    (a layer-step is one layer's work for the whole batch), so it is not extrapolated from one
    request.  ms_per_step is the time the sample step took."""
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import torch
    wl = rank_workload(args.workload, 0)
    device = "cuda" if torch.cuda.is_available() else "cpu"
    q_idx, w = wlm.indexer_queries(wl)
    qs = [wlm.mla_queries(wl, l) for l in range(wl.layers)]
    picked = stratified_requests(wl, min(wl.num_requests, args.reference_requests))
    probs = [oracle_request_problem(wl, b, device) for b in picked]
    times = []
    for i in range(args.warmup + args.steps):
        t = sum(time_oracle_request(wl, b, caches, bt, q_idx, w, qs) for b, (caches, bt) in zip(picked, probs))
        if i >= args.warmup:
            times.append(t)
    step_s = float(np.mean(times))
    frac = len(picked) / wl.num_requests                       # share of a full group step one step covers
    value = wl.layers * frac / step_s
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"each step: the float64 numpy oracle on the same {len(picked)} of {wl.num_requests} requests "
              f"(stratified by context length: {[wl.seq_lens[b] for b in picked]}), append + indexer + top-k + "
              f"{wl.layers} attention layers; the rate counts the {wl.layers * frac:.3f} layer-steps that "
              f"sample makes up")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, **{k: v for k, v in wl.summary().items() if k != "workload"}},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "full_group_step_ms_estimate": step_s * 1e3 / frac}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# decode context parallelism: one rank's device work
# ---------------------------------------------------------------------------
def dcp_main(args):
    """One rank's side of the decode step under context parallelism over `world` ranks, on one GPU.

    Rank 0 holds every request's interleaved share (ceil(L / world) tokens) in its own caches and
    runs: append, the indexer and top-k over its keys, dcp_candidates, dcp_select, and per layer the
    sparse MLA over its share plus dcp_merge.  The two all-gathers cross GPUs in a deployment; here
    their results are prepared once before the timed region, as if the exchange had delivered them:
    every rank's slot holds this rank's tensor, candidate positions relabelled to that rank's
    interleave and scores scaled by 1 + r 2^-20 so that they do not tie (a copy would tie every score
    world ways) while each rank still holds about 1/world of the selection.  The timed step is the
    rank's kernels only, replayed from a CUDA graph.  Every request's new token is appended on this
    rank (the worst case)."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    from deepseek_sparse_mla_gb300 import _lib
    W = args.dcp
    full = rank_workload(args.workload, 0)
    lens = [-(-L // W) for L in full.seq_lens]
    wl = wlm.Workload(f"{full.name}_dcp{W}_rank0", lens, [1] * len(lens), full.page_size, full.key_format, full.topk,
                      full.layers, full.seed + 7000 + W)
    prob = DeviceProblem(wl)
    R, k = wl.num_rows, wl.topk
    dev = "cuda"
    scores = torch.empty((R, wl.max_seq_len), dtype=torch.float32, device=dev)
    cs = torch.empty((R, k), dtype=torch.float32, device=dev)
    cp = torch.empty((R, k), dtype=torch.int32, device=dev)
    gidx = torch.empty((R, k), dtype=torch.int32, device=dev)
    lidx = torch.empty((R, k), dtype=torch.int32, device=dev)
    lcnt = torch.empty((R,), dtype=torch.int32, device=dev)
    merged = [torch.empty((R, 64, 512), dtype=torch.bfloat16, device=dev) for _ in range(wl.layers)]
    merged_lse = [torch.empty((R, 64), dtype=torch.float32, device=dev) for _ in range(wl.layers)]
    ex = {}

    def step():
        dsa.kv_append_layers(prob.caches, prob.new_c, prob.new_r, prob.slots,
                             k_idx=[prob.new_k] + [None] * (wl.layers - 1))
        dsa.indexer_scores_topk(prob.caches[0], prob.batch, prob.q_idx, prob.w, k, topk_idx=prob.topk_idx,
                                scores_out=scores, workspace=prob.ws_idx)
        dsa.dcp_candidates(scores, prob.topk_idx, 0, W, cand_scores=cs, cand_pos=cp)
        dsa.dcp_select(ex["s"], ex["p"], 0, global_idx=gidx, local_idx=lidx, local_count=lcnt)
        for l in range(wl.layers):
            dsa.sparse_mla_decode(prob.caches[l], prob.batch, prob.q[l], lidx, wl.scale, out=prob.out[l],
                                  lse=prob.lse[l], workspace=prob.ws_mla, row_counts=lcnt)
            dsa.dcp_merge(ex["o"][l], ex["l"][l], out=merged[l], lse=merged_lse[l])

    # the exchanged tensors, from one pass of the rank's own steps
    dsa.indexer_scores_topk(prob.caches[0], prob.batch, prob.q_idx, prob.w, k, topk_idx=prob.topk_idx,
                            scores_out=scores, workspace=prob.ws_idx)
    dsa.dcp_candidates(scores, prob.topk_idx, 0, W, cand_scores=cs, cand_pos=cp)
    rel = torch.arange(W, dtype=torch.int32, device=dev).view(W, 1, 1)
    relf = 1.0 + torch.arange(W, dtype=torch.float32, device=dev).view(W, 1, 1) * 2.0 ** -20
    ex["s"] = (cs.unsqueeze(0) * relf).contiguous()
    ex["p"] = torch.where(cp.unsqueeze(0) >= 0, cp.unsqueeze(0) + rel, cp.unsqueeze(0)).contiguous()
    dsa.dcp_select(ex["s"], ex["p"], 0, global_idx=gidx, local_idx=lidx, local_count=lcnt)
    ex["o"], ex["l"] = [], []
    for l in range(wl.layers):
        dsa.sparse_mla_decode(prob.caches[l], prob.batch, prob.q[l], lidx, wl.scale, out=prob.out[l],
                              lse=prob.lse[l], workspace=prob.ws_mla, row_counts=lcnt)
        ex["o"].append(prob.out[l].unsqueeze(0).expand(W, R, 64, 512).contiguous())
        ex["l"].append(prob.lse[l].unsqueeze(0).expand(W, R, 64).contiguous())
    torch.cuda.synchronize()

    lib = _lib.load()
    graph, per_step = None, 0
    if not args.eager:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            n0 = lib.dsa_kernel_launches()
            with torch.cuda.graph(graph):
                step()
            per_step = int(lib.dsa_kernel_launches() - n0)
        except Exception as e:
            print(f"graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graph = None
    run_step = graph.replay if graph is not None else step
    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    launches0 = lib.dsa_kernel_launches()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        run_step()
    t1.record()
    torch.cuda.synchronize()
    launches = per_step * args.steps if graph is not None else int(lib.dsa_kernel_launches() - launches0)
    ms = t0.elapsed_time(t1) / args.steps
    line = {"metric": f"DCP rank decode layer-steps/s (world {W}, the rank's kernels; exchanges excluded)",
            "value": wl.layers / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": full.name, "world": W, "rank_share": wl.summary(),
                       "launch": "CUDA graph replay" if graph is not None else "eager"},
            "gpu_launches": launches}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wlm.FULL) + sorted(wlm.PROFILE))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--selection", choices=["token", "page", "locality"], default="token",
                    help="token top-k (the method's selection), page-granular selection of topk / page_size "
                         "pages, or attention over locality-shaped page selections (to measure L2 reuse; the "
                         "indexer still runs)")
    ap.add_argument("--locality-noise", type=float, default=0.17,
                    help="--selection locality: per-row noise on the shared page scores (large: uniform pages)")
    ap.add_argument("--reference-requests", type=int, default=8,
                    help="--impl reference: requests per oracle step (a fixed stratified sample)")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the sustained replay measurement after the timed region")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="for profilers: set up, run this many steps (replayed from the step's graph unless "
                         "--eager) and exit without timing")
    ap.add_argument("--cpu-sample-requests", type=int, default=64)
    ap.add_argument("--eager", action="store_true",
                    help="launch the step call by call instead of replaying it from a CUDA graph")
    ap.add_argument("--latent", choices=["bf16", "fp8"], default="bf16",
                    help="latent cache format: bf16, or packed 8-bit (e4m3 c_KV with a scale per token, bf16 k_R)")
    ap.add_argument("--keys", choices=["default", "bf16", "fp8", "int8"], default="default",
                    help="index-key format of the owner layer (default: the workload's own; int8 keys carry a "
                         "binary16 scale per token)")
    ap.add_argument("--dcp", type=int, default=0,
                    help="time one rank's device work of decode context parallelism over this many ranks")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return reference_main(args)
    if args.dcp:
        return dcp_main(args)

    import torch
    import deepseek_sparse_mla_gb300 as dsa
    from deepseek_sparse_mla_gb300 import _lib
    rank, world = dist_setup(args.gpus)
    wl = rank_workload(args.workload, rank)
    if args.latent != "bf16":
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_latent_{args.latent}", latent_format=args.latent)
    if args.keys not in ("default", wl.key_format):
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_keys_{args.keys}", key_format=args.keys)
    prob = DeviceProblem(wl, selection=args.selection, locality_noise=args.locality_noise)
    page_mode = args.selection == "page"
    lib = _lib.load()

    # ---- device-resident timing --------------------------------------------------------
    # The step is replayed from a CUDA graph (one host call per step instead of one per library call;
    # small batches are otherwise bound by the host's launch rate), or launched call by call (--eager).
    graph, per_step = None, 0
    if not args.eager:
        try:
            graph, per_step = capture_step(prob, lib)
        except Exception as e:                           # capture unavailable: launch call by call
            print(f"graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graph = None
    run_step = graph.replay if graph is not None else prob.step
    if args.profile_steps > 0:
        for _ in range(args.profile_steps):
            run_step()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"profile_steps": args.profile_steps, "workload": wl.name, "kernels_per_step": per_step}),
                  flush=True)
        return
    clocks = ClockSampler()
    clocks.start()
    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    time.sleep(0.5)                      # nvidia-smi is up and sampling before the timed region
    barrier(world)
    torch.cuda.synchronize()
    launches0 = lib.dsa_kernel_launches()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_begin()
    t0.record()
    for _ in range(args.steps):
        run_step()
    t1.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop()
    # a replay launches the captured kernels without a host call into the library
    launches = per_step * args.steps if graph is not None else int(lib.dsa_kernel_launches() - launches0)
    barrier(world)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms_per_step = elapsed_ms / args.steps
    value = aggregate_rate(elapsed_ms, world, wl.layers, args.steps)

    # ---- sustained: the same replays for a few seconds, clocks sampled throughout -------------
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustained_seconds * 1e3 / ms_per_step)))
        clocks_s = ClockSampler()
        clocks_s.start()
        for _ in range(args.warmup):
            run_step()
        torch.cuda.synchronize()
        time.sleep(0.5)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks_s.mark_begin()
        s0.record()
        for _ in range(n_sus):
            run_step()
        s1.record()
        torch.cuda.synchronize()
        clocks_s.mark_end()
        sus_ms = max_over_ranks(s0.elapsed_time(s1), world)
        sustained = {"value": aggregate_rate(sus_ms, world, wl.layers, n_sus), "unit": UNIT, "steps": n_sus,
                     "ms_per_step": sus_ms / n_sus, "seconds": sus_ms / 1e3, "clocks": clocks_s.stop()}

    # ---- per-call breakdown ----------------------------------------------------------------
    # With graph replay: the step's first j library calls captured as graphs of their own; a call's
    # time is what it adds to the replayed prefix (programmatic-launch overlap with the call before
    # it included), so the calls' times add up to the replayed step.  Eager: events between calls.
    per_call = None
    if graph is not None:
        try:
            n_calls = prob.num_calls()
            pre = [0.0] + [replay_ms(capture_step(prob, lib, calls=j)[0]) for j in range(1, n_calls + 1)]
            marg = [pre[j] - pre[j - 1] for j in range(1, n_calls + 1)]
            per_call = {"append": marg[0] / wl.layers, "indexer": marg[1], "attention": float(np.mean(marg[2:]))}
            breakdown = "marginal times of the replayed step's call prefixes (CUDA graphs)"
        except Exception as e:
            print(f"prefix capture failed ({e}); per-call times from eager calls", file=sys.stderr)
    if per_call is None:
        marks = Marks()
        for _ in range(max(3, min(args.steps, 20))):
            prob.step(marks)
            torch.cuda.synchronize()
            marks.collect()
        per_call = {k: float(np.mean(v)) for k, v in marks.spans.items()}     # ms per call
        per_call["append"] /= wl.layers                                         # one span covers every layer's append
        breakdown = "CUDA events between eager library calls"
    # a layer group's attention runs as one call over every layer (its bytes and flops are the layers')
    att_layers = wl.layers if prob.group_attention else 1
    calls = {"append": wl.layers, "indexer": 1, "attention": wl.layers // att_layers}
    share = {k: per_call[k] * calls[k] for k in per_call}
    tot = sum(share.values())
    alg = algorithmic_bytes(wl)
    peak, peak_kind = load_peaks()
    bytes_of = {"indexer": alg["indexer"], "attention": alg["attention"] * att_layers,
                "append": (alg["append_owner"] + (wl.layers - 1) * alg["append_shared"]) / wl.layers}
    # each timed call, the kernels it launches and the sources they come from
    files = {"indexer": (("indexer.cu", "topk.cu"),
                         "indexer_page_topk: indexer_groups_kernel + indexer_tc_kernel (page scores) + topk_kernel + "
                         "page_expand_kernel" if page_mode else
                         "indexer_scores_topk: indexer_groups_kernel + indexer_tc_kernel + topk_chunk_kernel + topk_kernel"),
             "attention": (("sparse_mla.cu",),
                           f"sparse_mla_decode_layers: sparse_mla_tc_kernel over the {wl.layers} layers' (layer, row, tile) "
                           "units on every SM + mla_merge_kernel for rows cut between CTAs" if prob.group_attention else
                           "sparse_mla_decode: sparse_mla_tc_kernel (clusters merge in shared memory; "
                           "mla_merge_kernel when rows are cut between CTAs)"),
             "append": (("kv_append.cu",), "kv_append_layers: kv_append_kernel (every layer in one launch)")}
    dom = max(share, key=share.get)
    # the dominant call's bound: its useful flops per algorithmic byte against the ridge (measured bf16
    # rate / measured HBM rate); above it the call is a dense contraction, rated in TFLOP/s
    tpeak, tpeak_kind = load_tensor_peak()
    flops_of = {"indexer": alg["indexer_flops"], "attention": alg["attention_flops"] * att_layers}
    ridge = tpeak * 1e12 / (peak * 1e9)
    intensity = flops_of.get(dom, 0.0) / bytes_of[dom]
    traffic = kernel_traffic(dom, files[dom][0], wl.name + (" (page selection)" if page_mode else ""))
    if intensity > ridge:
        achieved = flops_of[dom] / (per_call[dom] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": files[dom][1], "achieved": achieved, "peak": tpeak,
                    "unit": "TFLOP/s", "frac": achieved / tpeak, "peak_kind": tpeak_kind, "traffic": traffic,
                    "algorithmic_flops_per_launch": flops_of[dom], "algorithmic_bytes_per_launch": bytes_of[dom],
                    "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    else:
        achieved = bytes_of[dom] / (per_call[dom] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": files[dom][1], "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                    "algorithmic_bytes_per_launch": bytes_of[dom], "intensity_flop_per_byte": intensity,
                    "ridge_flop_per_byte": ridge}
    kernels = {k: {"ms_per_call": per_call[k], "calls_per_step": calls[k], "share": share[k] / tot,
                   "algorithmic_GBps": bytes_of[k] / (per_call[k] * 1e-3) / 1e9,
                   "frac_of_peak": bytes_of[k] / (per_call[k] * 1e-3) / 1e9 / peak} for k in per_call}
    for k in flops_of:
        if k in kernels:
            kernels[k]["algorithmic_TFLOPs"] = flops_of[k] / (per_call[k] * 1e-3) / 1e12
            kernels[k]["frac_of_tensor_peak"] = kernels[k]["algorithmic_TFLOPs"] / tpeak
    step_gbps = alg["step"] / (ms_per_step * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers ---------------------------
    # Every step copies its inputs from pinned host memory and its outputs back.  Two sets of device
    # inputs/outputs let a copy stream move step i+1's inputs and step i-1's outputs while step i's
    # kernels run (the usual double buffering of a serving loop); a step starts only after its own
    # inputs have landed, and a set is refilled only after the step that used it and its read-back.
    # Each set's inputs and outputs live in one flat device buffer (views of it are what the calls get),
    # so a step's inputs arrive in one host-to-device copy and its outputs leave in one.
    ios = [prob, prob.io_set()]
    flats = []
    for io in ios:
        f_in, v_in = pack_views(prob.step_inputs(io), "cuda")
        f_out, v_out = pack_views(prob.step_outputs(io), "cuda")
        prob.assign_io(io, v_in, v_out)
        flats.append((f_in, f_out))
    torch.cuda.synchronize()
    h_in = flats[0][0].cpu().pin_memory()
    h_out = torch.empty(flats[0][1].shape, dtype=torch.uint8, pin_memory=True)
    h2d, d2h = int(h_in.numel()), int(h_out.numel())
    comp, copy = torch.cuda.current_stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    e2e_graphs = None
    if graph is not None:
        try:
            e2e_graphs = [capture_step(prob, lib, io)[0] for io in ios]
        except Exception as e:
            print(f"graph capture failed ({e}); end-to-end steps launch eagerly", file=sys.stderr)

    def e2e_run(n):
        copy.wait_stream(comp)
        with torch.cuda.stream(copy):
            flats[0][0].copy_(h_in, non_blocking=True)
            ready[0].record(copy)
        for i in range(n):
            s = i & 1
            comp.wait_event(ready[s])
            if e2e_graphs is not None:
                e2e_graphs[s].replay()
            else:
                prob.step(io=ios[s])
            done[s].record(comp)
            with torch.cuda.stream(copy):
                if i + 1 < n:
                    if i >= 1:
                        copy.wait_event(done[s ^ 1])          # step i-1 is done with the other set
                    flats[s ^ 1][0].copy_(h_in, non_blocking=True)
                    ready[s ^ 1].record(copy)
                copy.wait_event(done[s])
                h_out.copy_(flats[s][1], non_blocking=True)
        comp.wait_stream(copy)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_run(args.steps)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e = {"value": aggregate_rate(e2e_ms, world, wl.layers, args.steps), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, "cuda", args.cpu_sample_requests)

    if rank == 0:
        summary = wl.summary()
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": wl.name, **{k: v for k, v in summary.items() if k != "workload"},
                           "selection": ("page budget: %d pages of %d positions" % (prob.page_budget, wl.page_size)
                                         if page_mode else
                                         ("attention over locality-shaped page selections (noise %g; the indexer "
                                          "still runs)" % args.locality_noise if args.selection == "locality"
                                          else "token top-k")),
                           "l2": "no flush: each step reads %.0f MB (> 129 MB L2)" % (alg["step"] / 1e6),
                           "launch": ("the step captured once in a CUDA graph and replayed (%d kernels a step)" % per_step
                                      if graph is not None else "eager: one host call per library call"),
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk, "sustained": sustained, "kernels": kernels, "kernels_from": breakdown,
                "step_algorithmic_GBps": step_gbps, "step_frac_of_peak": step_gbps / peak,
                "step_frac_of_8TBps": step_gbps / 8000.0}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
