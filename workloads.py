"""Seeded synthetic workloads for the DSA step (decode, chunked prefill, speculative verify).

This module is shared by the tests, the benchmark and the smoke check.  It only
draws random numbers, rounds them to the storage formats (bf16 by
round-to-nearest-even from float32), and lays out the paged-cache metadata
(page tables over a seeded random permutation of physical pages, slot
mappings, query_start_loc).  It holds none of the step's arithmetic: no
scoring, selection, fp8 quantisation, softmax or attention.  Both the CUDA
path and the float64 oracle consume what it produces, each with its own code.

Shapes follow GLM-5.2's DSA layer as described in "vLLM Inference Path:
GLM-5.2 as an Example" (Model Shape table): 64 MLA heads, KV latent rank 512
plus a 64-wide RoPE key, and an indexer with 32 heads of width 128.

Recipe (every workload):
  * cached tokens: c_KV, k_R ~ N(0,1) rounded to bf16; indexer keys ~ N(0,1)
    rounded to bf16 (an fp8 cache stores them after per-token quantisation,
    done by each side's own append);
  * per-row queries: q_idx, q ~ N(0,1) in bf16; head weights w ~ N(0,1)/sqrt(32)
    in float32;
  * pages: each request holds ceil(L/P) pages drawn from a seeded permutation
    of a pool with 1 % spare pages, so that logical neighbours are physically
    scattered;
  * the step's new tokens are the last q_len positions of each request: they
    are appended by the step, the prefix before them is appended at set-up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

H_I, D_I = 32, 128           # indexer heads and head width
H, D_L, D_R = 64, 512, 64    # MLA heads, latent width, RoPE width
D = D_L + D_R                # cached latent row width (576)
SOFTMAX_SCALE = 1.0 / math.sqrt(192 + 64)   # 1/16: tied to the unabsorbed q/k width

# stream tags keep every random draw independent and individually reproducible
_TAG_LATENT, _TAG_IKEY, _TAG_Q, _TAG_QIDX, _TAG_W, _TAG_LENS, _TAG_PAGES = range(7)


@dataclass
class Workload:
    name: str
    seq_lens: list            # L_b: KV length of request b after this step's append
    q_lens: list              # query rows of request b (1 = decode)
    page_size: int
    key_format: str           # "bf16" | "fp8" | "int8"
    topk: int
    layers: int               # attention calls per step: 1 owner + (layers-1) IndexShare layers
    seed: int
    scale: float = SOFTMAX_SCALE
    spare_frac: float = 0.01
    block_table: np.ndarray = field(default=None, repr=False)
    num_pages: int = 0
    latent_format: str = "bf16"   # "bf16", or "fp8": packed 8-bit latent (e4m3 c_KV + scale, bf16 k_R)

    def __post_init__(self):
        self.seq_lens = [int(x) for x in self.seq_lens]
        self.q_lens = [int(x) for x in self.q_lens]
        assert len(self.seq_lens) == len(self.q_lens)
        assert all(1 <= q <= L for q, L in zip(self.q_lens, self.seq_lens))
        if self.block_table is None:
            self.block_table, self.num_pages = make_page_table(
                self.seq_lens, self.page_size, self.seed, self.spare_frac)

    # ---- batch metadata -------------------------------------------------
    @property
    def num_requests(self) -> int:
        return len(self.seq_lens)

    @property
    def num_rows(self) -> int:
        return int(sum(self.q_lens))

    @property
    def max_seq_len(self) -> int:
        return int(max(self.seq_lens))

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def is_decode(self) -> bool:
        return all(q == 1 for q in self.q_lens)

    def row_request(self) -> np.ndarray:
        return np.repeat(np.arange(self.num_requests), self.q_lens).astype(np.int32)

    def row_position(self) -> np.ndarray:
        """Absolute position of each query row: L_b - q_len_b + i."""
        out = []
        for L, q in zip(self.seq_lens, self.q_lens):
            out.extend(range(L - q, L))
        return np.asarray(out, dtype=np.int64)

    def slots(self, b: int, positions) -> np.ndarray:
        """Physical slot (page id * page_size + offset) of logical positions of request b."""
        positions = np.asarray(positions, dtype=np.int64)
        pages = self.block_table[b, positions // self.page_size].astype(np.int64)
        return pages * self.page_size + positions % self.page_size

    def new_token_slots(self) -> np.ndarray:
        """slot_mapping of the step's appended tokens, in row order."""
        return np.concatenate([self.slots(b, np.arange(L - q, L))
                               for b, (L, q) in enumerate(zip(self.seq_lens, self.q_lens))])

    # ---- algorithmic sizes (bytes the step must move) -----------------------
    def key_bytes_per_token(self) -> int:
        return {"bf16": D_I * 2, "fp8": D_I + 4, "int8": D_I + 2}[self.key_format]

    def summary(self) -> dict:
        return {"workload": self.name, "requests": self.num_requests, "rows": self.num_rows,
                "seq_lens": f"{min(self.seq_lens)}..{max(self.seq_lens)} (sum {sum(self.seq_lens)})",
                "page_size": self.page_size, "index_keys": self.key_format, "topk": self.topk,
                "layers": self.layers, "latent": self.latent_format}


def make_page_table(seq_lens, page_size, seed, spare_frac=0.01):
    """Page table over a seeded random permutation of a pool with spare pages.

    Unused entries are -1.  Returns (block_table [B, max_pages] int32, num_pages).
    """
    need = [-(-int(L) // page_size) for L in seq_lens]
    total = int(sum(need))
    num_pages = total + max(1, math.ceil(total * spare_frac))
    rng = np.random.default_rng([seed, _TAG_PAGES])
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(seq_lens), max(need)), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[at:at + n]
        at += n
    return bt, num_pages


# ---------------------------------------------------------------------------
# storage-format rounding of random draws
# ---------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _rng(*tags):
    return np.random.default_rng([int(t) for t in tags])


def _normal_bf16(rng, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


# ---------------------------------------------------------------------------
# host (numpy) generation: every array a pure function of (seed, tags)
# ---------------------------------------------------------------------------
def request_latent(wl: Workload, b: int, layer: int) -> np.ndarray:
    """All L_b cached rows [c_KV(512) | k_R(64)] of request b for one layer, bf16 bits [L_b, 576]."""
    return _normal_bf16(_rng(wl.seed, _TAG_LATENT, b, layer), (wl.seq_lens[b], D))


def request_index_keys(wl: Workload, b: int) -> np.ndarray:
    """All L_b indexer keys of request b before any quantisation, bf16 bits [L_b, 128]."""
    return _normal_bf16(_rng(wl.seed, _TAG_IKEY, b), (wl.seq_lens[b], D_I))


def mla_queries(wl: Workload, layer: int) -> np.ndarray:
    """Absorbed MLA queries [q_latent(512) | q_rope(64)] per head, bf16 bits [R, 64, 576]."""
    return _normal_bf16(_rng(wl.seed, _TAG_Q, layer), (wl.num_rows, H, D))


def indexer_queries(wl: Workload):
    """(q_idx bf16 bits [R, 32, 128], w float32 [R, 32] ~ N(0,1)/sqrt(32))."""
    q_idx = _normal_bf16(_rng(wl.seed, _TAG_QIDX), (wl.num_rows, H_I, D_I))
    w = (_rng(wl.seed, _TAG_W).standard_normal((wl.num_rows, H_I)) / math.sqrt(H_I)).astype(np.float32)
    return q_idx, w


# ---------------------------------------------------------------------------
# device (torch) generation for full-size workloads: same recipe, torch's
# seeded CUDA generator, per (request, layer) so any request can be re-drawn
# ---------------------------------------------------------------------------
def _torch_seed(*tags) -> int:
    h = 1469598103934665603
    for t in tags:
        h = ((h ^ (int(t) & 0xFFFFFFFF)) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def request_latent_device(wl: Workload, b: int, layer: int, device, lo: int = 0, hi: int | None = None):
    """bf16 tensor [L_b, 576] on `device` (rows lo..hi of it if given), drawn with torch's generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(wl.seed, _TAG_LATENT, b, layer))
    x = torch.randn((wl.seq_lens[b], D), generator=g, device=device, dtype=torch.float32)
    return x[lo:hi].to(torch.bfloat16)


def request_index_keys_device(wl: Workload, b: int, device, lo: int = 0, hi: int | None = None):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(wl.seed, _TAG_IKEY, b))
    x = torch.randn((wl.seq_lens[b], D_I), generator=g, device=device, dtype=torch.float32)
    return x[lo:hi].to(torch.bfloat16)


def locality_page_scores(qb: int, num_pages: int, noise: float, seed: int) -> np.ndarray:
    """[qb, num_pages] float64 page scores of qb nearby query rows whose preferences mostly agree: one
    shared N(0, 1) score per page plus N(0, noise^2) per row.  The locality-shaped selection regime of
    the query-blocking microbenchmark ("Making GLM-5.2 Sparse on TPUs", "Reuse pages across queries"),
    for which the pages print no data: noise 0 gives every row the same pages, and large noise tends to
    uniformly random selections.  At 64 rows, 32 pages per row and 880 pages, noise 0.17 gives a union
    of about 69 pages, the page's figure."""
    rng = _rng(seed, _TAG_PAGES, qb, num_pages)
    shared = rng.standard_normal(num_pages)
    return shared[None, :] + noise * rng.standard_normal((qb, num_pages))


def torch_to_bits(t) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (host copy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_torch(bits: np.ndarray, device=None):
    """numpy uint16 bf16 bit patterns -> bf16 torch tensor."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


# ---------------------------------------------------------------------------
# the five workloads of the DSA step, and reduced forms for quick parity runs
# ---------------------------------------------------------------------------
def tiny_decode() -> Workload:
    return Workload("tiny_decode_b2_ctx300_512", [300, 512], [1, 1], 64, "bf16", 128, 1, 1001)


def decode_b32_8k() -> Workload:
    return Workload("decode_b32_ctx8192_bf16", [8192] * 32, [1] * 32, 64, "bf16", 2048, 1, 1002)


def decode_b64_fp8_indexshare() -> Workload:
    lens = _rng(1003, _TAG_LENS).integers(16384, 131072 + 1, 64)
    return Workload("decode_b64_ctx16k-128k_fp8_indexshare4", lens, [1] * 64, 64, "fp8", 2048, 4, 1003)


def prefill_chunk_4096() -> Workload:
    return Workload("prefill_4096_after_61440_bf16", [65536], [4096], 128, "bf16", 2048, 1, 1004)


def verify_b8x4_240k() -> Workload:
    return Workload("verify_b8x4_ctx240000_fp8", [240000] * 8, [4] * 8, 64, "fp8", 2048, 1, 1005)


FULL = {
    "tiny_decode": tiny_decode,
    "decode_b32_8k": decode_b32_8k,
    "decode_b64_fp8_indexshare": decode_b64_fp8_indexshare,
    "prefill_chunk_4096": prefill_chunk_4096,
    "verify_b8x4_240k": verify_b8x4_240k,
}


def profile_decode_b64_ctx16k_32k() -> Workload:
    """The headline decode shape (64 rows, fp8 keys, top-k 2048) at 16K-32K contexts and one layer:
    about 2 GB resident, small enough for a many-pass profiler capture of one launch."""
    lens = _rng(4001, _TAG_LENS).integers(16384, 32768 + 1, 64)
    return Workload("profile_decode_b64_ctx16k-32k_fp8", lens, [1] * 64, 64, "fp8", 2048, 1, 4001)


def profile_decode_b24_ctx48k_96k() -> Workload:
    """Long decode rows (24 rows of 48K-96K positions, fp8 keys, top-k 2048, one layer): the rows are
    split into 2-3 top-k chunks, as in the headline shape; about 2.3 GB resident."""
    lens = _rng(4002, _TAG_LENS).integers(49152, 98304 + 1, 24)
    return Workload("profile_decode_b24_ctx48k-96k_fp8", lens, [1] * 24, 64, "fp8", 2048, 1, 4002)


# workloads that exist for profiler captures only (not parity or benchmark configurations)
def profile_decode_b64_ctx8k_12k_layers4() -> Workload:
    """The headline's layer group (64 rows x 4 layers sharing one top-2048 index buffer) at 8K-12K
    contexts: about 3 GB resident, for a capture of the one-call attention over the four layers (whose
    cost depends on the selected rows, not on the context length)."""
    lens = _rng(4003, _TAG_LENS).integers(8192, 12288 + 1, 64)
    return Workload("profile_decode_b64_ctx8k-12k_fp8_layers4", lens, [1] * 64, 64, "fp8", 2048, 4, 4003)


PROFILE = {"profile_decode_b64_ctx16k_32k": profile_decode_b64_ctx16k_32k,
           "profile_decode_b24_ctx48k_96k": profile_decode_b24_ctx48k_96k,
           "profile_decode_b64_ctx8k_12k_layers4": profile_decode_b64_ctx8k_12k_layers4}


def reduced(name: str) -> Workload:
    """Same structure as the named workload at sizes a float64 oracle finishes in seconds.

    Every reduced case keeps a ragged tail (lengths not a multiple of the page
    size or of 128) and contexts longer than top-k, so selection is exercised.
    """
    if name == "tiny_decode":
        return tiny_decode()
    if name == "decode_b32_8k":
        return Workload("decode_b4_ctx2500_bf16", [2500, 2500, 3001, 2049], [1] * 4, 64, "bf16", 2048, 1, 2002)
    if name == "decode_b64_fp8_indexshare":
        lens = _rng(2003, _TAG_LENS).integers(2100, 5000, 6)
        return Workload("decode_b6_ctx2k-5k_fp8_indexshare4", lens, [1] * 6, 64, "fp8", 2048, 4, 2003)
    if name == "prefill_chunk_4096":
        return Workload("prefill_300_after_1900_bf16", [2200], [300], 128, "bf16", 2048, 1, 2004)
    if name == "verify_b8x4_240k":
        return Workload("verify_b2x4_ctx3000_fp8", [3000, 2777], [4, 4], 64, "fp8", 2048, 1, 2005)
    raise KeyError(name)
