import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdsa")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if it is missing or stale."""
    from deepseek_sparse_mla_gb300 import build as dsa_build
    dsa_build.build_library(quiet=True)
    from deepseek_sparse_mla_gb300 import _lib
    return _lib.load()


# ---------------------------------------------------------------------------
# tiny cases with small, discriminating widths for the brute-force pins
# ---------------------------------------------------------------------------
class TinyCase:
    """Random tiny DSA problem with its own widths; builds an oracle cache."""

    def __init__(self, seed, seq_lens, q_lens, page_size, key_format="bf16",
                 n_idx_heads=2, d_index=4, n_heads=2, d_latent=6, d_rope=3, spare=3, latent_format="bf16"):
        import workloads as wlm
        from oracle import dsa_oracle as o
        rng = np.random.default_rng(seed)
        self.seq_lens = list(seq_lens)
        self.q_lens = list(q_lens)
        self.P = page_size
        self.key_format = key_format
        self.d_latent, self.d_rope, self.d_index = d_latent, d_rope, d_index
        self.qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        need = [-(-L // page_size) for L in seq_lens]
        self.num_pages = sum(need) + spare
        perm = rng.permutation(self.num_pages)
        self.block_table = np.full((len(seq_lens), max(need)), -1, dtype=np.int32)
        at = 0
        for b, n in enumerate(need):
            self.block_table[b, :n] = perm[at:at + n]
            at += n
        self.latent = [wlm.bf16_bits(rng.standard_normal((L, d_latent + d_rope)).astype(np.float32))
                       for L in seq_lens]
        self.keys = [wlm.bf16_bits(rng.standard_normal((L, d_index)).astype(np.float32)) for L in seq_lens]
        R = int(sum(q_lens))
        self.q_idx = wlm.bf16_bits(rng.standard_normal((R, n_idx_heads, d_index)).astype(np.float32))
        self.w = (rng.standard_normal((R, n_idx_heads)) / np.sqrt(n_idx_heads)).astype(np.float32)
        self.q = wlm.bf16_bits(rng.standard_normal((R, n_heads, d_latent + d_rope)).astype(np.float32))
        self.cache = o.PagedCache(self.num_pages, page_size, key_format, d_latent, d_rope, d_index,
                                  latent_format=latent_format)
        for b, L in enumerate(seq_lens):
            slots = self.slots(b, np.arange(L))
            self.cache.append(self.latent[b][:, :d_latent], self.latent[b][:, d_latent:], slots,
                              k_idx_bits=self.keys[b])

    def slots(self, b, positions):
        positions = np.asarray(positions)
        return self.block_table[b, positions // self.P].astype(np.int64) * self.P + positions % self.P

    def rows(self):
        """(request, position) of each query row."""
        out = []
        for b, (L, q) in enumerate(zip(self.seq_lens, self.q_lens)):
            out.extend((b, L - q + i) for i in range(q))
        return out


@pytest.fixture
def tiny_case():
    return TinyCase
