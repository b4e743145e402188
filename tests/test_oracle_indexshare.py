"""IndexShare: the layer schedule and the reuse of an owner's index buffer."""
import os

import numpy as np

from oracle import dsa_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "index_topk_pattern.txt")


def _golden():
    d = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            d[k.strip()] = v.strip()
    return d


def test_pattern_from_indexer_types_matches_printed_string():
    g = _golden()
    owners = [int(x) for x in g["owners"].split()]
    n = int(g["layers"])
    types = ["full" if i in owners else "shared" for i in range(n)]
    pattern = o.indexshare_pattern(types)
    assert pattern == g["pattern"]
    assert pattern.count("F") == int(g["full"]) and pattern.count("S") == int(g["shared"])


def test_every_shared_layer_reuses_the_nearest_preceding_owner():
    g = _golden()
    owners = o.owner_of_layer(g["pattern"])
    full = [int(x) for x in g["owners"].split()]
    for layer, owner in enumerate(owners):
        assert owner == max(f for f in full if f <= layer)
    # the decode-benchmark group: layers 6..9 are one owner and three shared layers
    assert owners[6:10] == [6, 6, 6, 6]


def test_shared_layers_attend_with_the_owner_indices(tiny_case):
    """Shared layers run attention on their own latent pages with the owner's index set."""
    owner = tiny_case(31, [29, 18], [1, 2], 4, "bf16")
    shared = tiny_case(32, [29, 18], [1, 2], 4, None)                  # other latents, no index keys
    shared.block_table = owner.block_table
    shared.cache = o.PagedCache(owner.num_pages, 4, None, shared.d_latent, shared.d_rope, shared.d_index)
    for b, L in enumerate(shared.seq_lens):
        shared.cache.append(shared.latent[b][:, :6], shared.latent[b][:, 6:], owner.slots(b, np.arange(L)))
    idx, _ = o.indexer_topk(owner.cache, owner.block_table, owner.seq_lens, owner.qsl, owner.q_idx, owner.w, 7)
    out_s, lse_s = o.sparse_mla(shared.cache, owner.block_table, owner.seq_lens, owner.qsl, shared.q, idx, 0.3)
    # reference: the shared layer's own rows at the owner's positions
    for r, (b, pos) in enumerate(owner.rows()):
        sel = [int(s) for s in idx[r] if s >= 0]
        rows = o.bf16_to_f64(shared.latent[b][sel])
        ref = o.attend(o.bf16_to_f64(shared.q[r]), rows, 0.3, 6)
        np.testing.assert_allclose(out_s[r], ref[0], rtol=1e-13)
        np.testing.assert_allclose(lse_s[r], ref[1], rtol=1e-13)
