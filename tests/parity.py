"""Parity harness: run the CUDA path and the float64 oracle on the same seeded inputs and compare.

Tolerances (stated by the task's parity contract for this step):
  * index keys / latent rows after append: bit-exact;
  * indexer scores: |gpu - oracle| <= 1e-2 * max(|oracle|, rms of the row's oracle scores);
  * top-k sets: same size, no duplicates, only visible positions, sorted ascending, and any
    position in exactly one of the two sets has an oracle score within 1e-3 relative of the
    oracle's k-th score (relative to max(|k-th score|, row rms));
  * attention (run on the oracle's index set): max-abs <= 2e-2 and mean-abs <= 2e-3 over the
    bf16 outputs; lse within 1e-3 * max(1, |lse|).
"""
from __future__ import annotations

import numpy as np

import workloads as wlm
from oracle import dsa_oracle as o

SCORE_RTOL = 1e-2
SWAP_RTOL = 1e-3
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3
LSE_TOL = 1e-3


# ---------------------------------------------------------------------------
# host problem: seeded inputs + oracle caches
# ---------------------------------------------------------------------------
class HostProblem:
    def __init__(self, wl: wlm.Workload):
        self.wl = wl
        L = wl.seq_lens
        self.latent = [[wlm.request_latent(wl, b, layer) for b in range(wl.num_requests)] for layer in range(wl.layers)]
        self.keys = [wlm.request_index_keys(wl, b) for b in range(wl.num_requests)]
        self.q_idx, self.w = wlm.indexer_queries(wl)
        self.q = [wlm.mla_queries(wl, layer) for layer in range(wl.layers)]
        self.qsl = wl.query_start_loc
        self.caches = []
        for layer in range(wl.layers):
            c = o.PagedCache(wl.num_pages, wl.page_size, wl.key_format if layer == 0 else None,
                             latent_format="e4m3" if wl.latent_format == "fp8" else "bf16")
            for b in range(wl.num_requests):
                c.append(self.latent[layer][b][:, :512], self.latent[layer][b][:, 512:], wl.slots(b, np.arange(L[b])),
                         k_idx_bits=self.keys[b] if layer == 0 else None)
            self.caches.append(c)

    def oracle_topk(self, rows=None):
        wl = self.wl
        return o.indexer_topk(self.caches[0], wl.block_table, wl.seq_lens, self.qsl, self.q_idx, self.w, wl.topk,
                              rows=rows)

    def oracle_attention(self, layer, idx, rows=None):
        wl = self.wl
        return o.sparse_mla(self.caches[layer], wl.block_table, wl.seq_lens, self.qsl, self.q[layer], idx, wl.scale,
                            rows=rows)

    # split every request's tokens into the prefix (appended at set-up) and the step's new tokens
    def token_split(self, layer):
        wl = self.wl
        pre_c, pre_r, pre_k, pre_s, new_c, new_r, new_k, new_s = ([] for _ in range(8))
        for b, (L, q) in enumerate(zip(wl.seq_lens, wl.q_lens)):
            lat = self.latent[layer][b]
            pre_c.append(lat[:L - q, :512]); pre_r.append(lat[:L - q, 512:])
            new_c.append(lat[L - q:, :512]); new_r.append(lat[L - q:, 512:])
            pre_k.append(self.keys[b][:L - q]); new_k.append(self.keys[b][L - q:])
            pre_s.append(wl.slots(b, np.arange(L - q))); new_s.append(wl.slots(b, np.arange(L - q, L)))
        cat = np.concatenate
        return ((cat(pre_c), cat(pre_r), cat(pre_k), cat(pre_s)), (cat(new_c), cat(new_r), cat(new_k), cat(new_s)))


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
class GpuProblem:
    """The same problem on the device, driven through the library's Python binding."""

    def __init__(self, hp: HostProblem, device="cuda"):
        import torch
        import deepseek_sparse_mla_gb300 as dsa
        self.hp, self.wl, self.dev = hp, hp.wl, device
        wl = self.wl
        self.caches = [dsa.LayerCache(wl.num_pages, wl.page_size, wl.key_format if layer == 0 else None, device,
                                      latent_format=wl.latent_format)
                       for layer in range(wl.layers)]
        decode = wl.is_decode
        self.batch = dsa.Batch(torch.from_numpy(wl.block_table).to(device),
                               torch.tensor(wl.seq_lens, dtype=torch.int32, device=device),
                               None if decode else torch.from_numpy(wl.query_start_loc).to(device),
                               num_rows=wl.num_rows, max_seq_len=wl.max_seq_len)
        self.q_idx = wlm.bits_to_torch(hp.q_idx, device)
        self.w = torch.from_numpy(hp.w).to(device)
        self.q = [wlm.bits_to_torch(x, device) for x in hp.q]
        self.new = []
        for layer in range(wl.layers):
            pre, new = hp.token_split(layer)
            self._append(layer, *pre)                       # set-up: the cached prefix
            self.new.append([self._dev(x) for x in new])    # the step's tokens, appended by step()

    def _dev(self, x):
        import torch
        if x.dtype == np.uint16:
            return wlm.bits_to_torch(x, self.dev)
        return torch.from_numpy(np.ascontiguousarray(x)).to(self.dev)

    def _append(self, layer, c, r, k, s):
        import deepseek_sparse_mla_gb300 as dsa
        if len(s) == 0:
            return
        dsa.kv_append(self.caches[layer], self._dev(c), self._dev(r), self._dev(s.astype(np.int64)),
                      k_idx=self._dev(k) if layer == 0 else None)

    def append_step(self):
        import deepseek_sparse_mla_gb300 as dsa
        for layer in range(self.wl.layers):
            c, r, k, s = self.new[layer]
            dsa.kv_append(self.caches[layer], c, r, s, k_idx=k if layer == 0 else None)

    def indexer(self, with_scores=True):
        import torch
        import deepseek_sparse_mla_gb300 as dsa
        scores = None
        if with_scores:
            scores = torch.empty((self.wl.num_rows, self.wl.max_seq_len), dtype=torch.float32, device=self.dev)
        idx = dsa.indexer_scores_topk(self.caches[0], self.batch, self.q_idx, self.w, self.wl.topk, scores_out=scores)
        return idx, scores

    def attention(self, layer, idx):
        import torch
        import deepseek_sparse_mla_gb300 as dsa
        lse = torch.empty((self.wl.num_rows, 64), dtype=torch.float32, device=self.dev)
        fn = dsa.sparse_mla_decode if self.wl.is_decode else dsa.sparse_mla_prefill
        out, _ = fn(self.caches[layer], self.batch, self.q[layer], idx, self.wl.scale, lse=lse)
        return out, lse


# ---------------------------------------------------------------------------
# comparisons
# ---------------------------------------------------------------------------
def bf16_tensor_to_f64(t) -> np.ndarray:
    return o.bf16_to_f64(wlm.torch_to_bits(t))


def check_cache_bytes(gp: GpuProblem, hp: HostProblem):
    import torch
    for layer in range(hp.wl.layers):
        g, h = gp.caches[layer], hp.caches[layer]
        if h.latent_format == "e4m3":
            lat = g.latent.cpu().numpy()                                  # [N, P, 640] bytes
            assert np.array_equal(lat[..., :512], h.latent_codes), f"latent codes differ (layer {layer})"
            assert np.array_equal(lat[..., 512:].copy().view(np.uint16), h.latent[..., 512:]), f"k_R differs (layer {layer})"
            assert np.array_equal(g.latent_scales.cpu().numpy().view(np.uint32), h.latent_scales.view(np.uint32)), \
                f"latent scales differ (layer {layer})"
        else:
            assert np.array_equal(wlm.torch_to_bits(g.latent), h.latent), f"latent pages differ (layer {layer})"
        if h.index_keys is not None:
            gk = (g.index_keys.cpu().numpy() if g.index_keys.dtype in (torch.uint8, torch.int8)
                  else wlm.torch_to_bits(g.index_keys))
            assert np.array_equal(gk, h.index_keys), "index-key pages differ"
            if h.index_scales is not None:          # fp32 scales (e4m3 keys) or binary16 bits (int8 keys)
                bits = np.uint16 if h.index_scales.dtype == np.uint16 else np.uint32
                assert np.array_equal(g.index_scales.cpu().numpy().view(bits), h.index_scales.view(bits)), \
                    "index scales differ"


def check_scores(g_row: np.ndarray, o_row: np.ndarray, pos: int, max_seq_len: int):
    n = pos + 1
    assert len(o_row) == n
    rms = float(np.sqrt(np.mean(o_row ** 2))) if n else 0.0
    err = np.abs(g_row[:n].astype(np.float64) - o_row)
    bound = SCORE_RTOL * np.maximum(np.abs(o_row), rms)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"score mismatch at positions {bad[:5]}: gpu {g_row[bad[:5]]} oracle {o_row[bad[:5]]}"
    assert np.all(np.isneginf(g_row[n:max_seq_len])), "positions beyond the row are not masked to -inf"


def check_topk(g_row: np.ndarray, o_row: np.ndarray, o_scores: np.ndarray, pos: int, k: int):
    g = g_row[g_row >= 0]
    o_sel = o_row[o_row >= 0]
    assert np.all(g_row[len(g):] == -1) and np.all(g_row[:len(g)] >= 0), "padding is not a -1 tail"
    assert len(g) == len(o_sel) == min(k, pos + 1), (len(g), len(o_sel))
    assert np.all(np.diff(g) > 0), "indices not strictly ascending (duplicates or unsorted)"
    assert g.min(initial=0) >= 0 and g.max(initial=0) <= pos, "an index names an invisible position"
    diff = np.setxor1d(g, o_sel)
    if diff.size:
        srt = np.sort(o_scores)[::-1]
        theta = srt[k - 1]
        rms = float(np.sqrt(np.mean(o_scores ** 2)))
        tol = SWAP_RTOL * max(abs(theta), rms)
        far = diff[np.abs(o_scores[diff] - theta) > tol]
        assert far.size == 0, f"swapped positions {far[:5]} are not near-ties of the k-th score {theta}"
    return int(diff.size)


def check_attention(g_out: np.ndarray, g_lse: np.ndarray, o_out: np.ndarray, o_lse: np.ndarray):
    err = np.abs(g_out - o_out)
    assert err.max() <= ATT_MAX_ABS, f"attention max-abs error {err.max():.3e}"
    assert err.mean() <= ATT_MEAN_ABS, f"attention mean-abs error {err.mean():.3e}"
    fin = np.isfinite(o_lse)
    assert np.array_equal(fin, np.isfinite(g_lse)), "lse -inf pattern differs"
    lerr = np.abs(g_lse[fin] - o_lse[fin])
    assert np.all(lerr <= LSE_TOL * np.maximum(1.0, np.abs(o_lse[fin]))), f"lse error {lerr.max():.3e}"
    return float(err.max()), float(err.mean())
