"""The one-launch append over several layers (dsa_kv_append_layers) against per-layer appends, byte
for byte: an owner layer with e4m3 index keys, a shared bf16 layer and a shared packed 8-bit layer,
with skipped slots (negative and beyond the pool)."""
import numpy as np
import pytest

import workloads as wlm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def test_fused_append_equals_per_layer_appends():
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    rng = np.random.default_rng(6100)
    pages, P, T = 40, 16, 300
    spec = [("fp8", "bf16"), (None, "bf16"), (None, "fp8")]          # (key format, latent format)
    c_kv = [wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 512)).astype(np.float32)), "cuda") for _ in spec]
    k_rope = [wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 64)).astype(np.float32)), "cuda") for _ in spec]
    k_idx = wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 128)).astype(np.float32)), "cuda")
    slots = rng.permutation(pages * P)[:T].astype(np.int64)
    slots[5], slots[77] = -1, pages * P + 3                          # skipped
    slots = torch.from_numpy(slots).cuda()

    def caches():
        out = []
        for kf, lf in spec:
            c = dsa.LayerCache(pages, P, kf, "cuda", latent_format=lf)
            c.latent.view(torch.uint8).fill_(0xA5)                   # canaries: untouched slots keep them
            out.append(c)
        return out

    one, each = caches(), caches()
    dsa.kv_append_layers(one, c_kv, k_rope, slots, k_idx=[k_idx, None, None])
    for l, c in enumerate(each):
        dsa.kv_append(c, c_kv[l], k_rope[l], slots, k_idx=k_idx if l == 0 else None)
    torch.cuda.synchronize()
    for a, b in zip(one, each):
        assert torch.equal(a.latent.view(torch.uint8), b.latent.view(torch.uint8))
        for x, y in ((a.index_keys, b.index_keys), (a.index_scales, b.index_scales), (a.latent_scales, b.latent_scales)):
            assert (x is None) == (y is None)
            if x is not None:
                assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
