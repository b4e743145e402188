"""GPU parity of the packed 8-bit latent cache (SFA C8: "GLM-5.2 on vLLM Ascend", "Quantization and
Hardware Branches") against the float64 oracle, through the C ABI.

dsa_kv_append writes each token's c_KV as 512 e4m3 codes with an fp32 scale and its k_R as bf16:
codes, k_R and scales must equal the oracle's bit for bit.  Attention over such a cache gathers the
640-byte rows, expands them to fp16 in shared memory and runs fp16 MMAs; it is checked against the
oracle's attention over code * scale with the usual attention tolerance, in the cluster split
(decode) and the unit split (more than 76 rows), with short rows, -1 padding, out-of-range entries
and rows with nothing selected.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from parity import GpuProblem, HostProblem, bf16_tensor_to_f64, check_attention, check_cache_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def _run(wl, idx_fn=None):
    import torch
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    torch.cuda.synchronize()
    check_cache_bytes(gp, hp)
    if idx_fn is None:
        o_idx, _ = hp.oracle_topk()
    else:
        o_idx = idx_fn(wl)
    idx = torch.from_numpy(np.ascontiguousarray(o_idx)).cuda()
    for layer in range(wl.layers):
        out, lse = gp.attention(layer, idx)
        torch.cuda.synchronize()
        o_out, o_lse = hp.oracle_attention(layer, o_idx)
        check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)


@pytest.mark.parametrize("name,seq_lens,q_lens,P,topk", [
    ("c8_decode", [3000, 900, 4100, 257], [1] * 4, 64, 2048),          # cluster split
    ("c8_decode_short", [40, 300, 1], [1] * 3, 16, 128),               # rows shorter than k
    ("c8_verify", [5000, 2600], [4, 4], 64, 512),                      # multi-row requests
])
def test_c8_attention_parity(name, seq_lens, q_lens, P, topk):
    wl = wlm.Workload(name, seq_lens, q_lens, P, "fp8", topk, 2, 5100 + sum(seq_lens) % 97, latent_format="fp8")
    _run(wl)


def test_c8_unit_split_with_many_rows():
    """More than 76 rows: the (row, tile) units are split over the persistent CTAs and rows cut
    between CTAs are finished by the merge kernel."""
    lens = [700 + 37 * i for i in range(80)]
    wl = wlm.Workload("c8_many", lens, [1] * 80, 64, "bf16", 256, 1, 5200, latent_format="fp8")
    _run(wl)


def test_c8_padding_out_of_range_and_empty_rows():
    wl = wlm.Workload("c8_edges", [500, 800, 64], [1] * 3, 32, "bf16", 192, 1, 5300, latent_format="fp8")

    def idx(w):
        o_idx, _ = HostProblem(w).oracle_topk()
        o_idx = o_idx.copy()
        o_idx[0, 100:] = -1                      # -1 padding
        o_idx[1, :5] = [900, 5000, 801, 800, 10000]   # beyond the row's position: skipped
        o_idx[2, :] = -1                         # nothing selected: out 0, lse -inf
        return o_idx
    _run(wl, idx)


def test_c8_exactly_representable_rows_match_the_bf16_cache():
    """Rows whose c_KV values are e4m3 values / 512 with amax 0.875 (= 448 / 512) quantise exactly
    (scale 1/512): the packed cache holds the same values as the bf16 cache, and attention over
    either matches the oracle's."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    from oracle.dsa_oracle import PagedCache
    rng = np.random.default_rng(5400)
    L, R = 2048, 2
    codes = rng.integers(0, 0x7E, size=(R * L, 512)).astype(np.uint8) | (rng.integers(0, 2, (R * L, 512)) << 7).astype(np.uint8)
    vals = o.e4m3_to_f64(codes) / 512.0
    vals[:, 0] = 0.875
    c_bits = wlm.bf16_bits(vals.astype(np.float32))
    assert np.array_equal(o.bf16_to_f64(c_bits), vals)
    r_bits = wlm.bf16_bits(rng.standard_normal((R * L, 64)).astype(np.float32))
    P, pages = 64, R * L // 64
    bt_np = np.arange(pages, dtype=np.int32).reshape(R, L // P)
    bt = torch.from_numpy(bt_np).cuda()
    batch = dsa.Batch(bt, torch.tensor([L] * R, dtype=torch.int32, device="cuda"), None, num_rows=R, max_seq_len=L)
    q_bits = wlm.bf16_bits(rng.standard_normal((R, 64, 576)).astype(np.float32))
    q = wlm.bits_to_torch(q_bits, "cuda")
    idx_np = np.stack([np.sort(rng.choice(L, 1024, replace=False)) for _ in range(R)]).astype(np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    host = PagedCache(pages, P, None)
    host.append(c_bits, r_bits, np.arange(R * L))
    o_out, o_lse = o.sparse_mla(host, bt_np, [L] * R, np.arange(R + 1, dtype=np.int32), q_bits, idx_np, dsa.DEFAULT_SCALE)
    for fmt in ("bf16", "fp8"):
        c = dsa.LayerCache(pages, P, None, "cuda", latent_format=fmt)
        dsa.kv_append(c, wlm.bits_to_torch(c_bits, "cuda"), wlm.bits_to_torch(r_bits, "cuda"),
                      torch.arange(R * L, dtype=torch.int64, device="cuda"))
        lse = torch.empty((R, 64), dtype=torch.float32, device="cuda")
        out, _ = dsa.sparse_mla_decode(c, batch, q, idx, dsa.DEFAULT_SCALE, lse=lse)
        torch.cuda.synchronize()
        if fmt == "fp8":
            assert np.all(c.latent_scales.cpu().numpy() == np.float32(1 / 512))
        check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)


def test_c8_attention_with_row_counts():
    """The packed latent with a compacted buffer and row counts (a DCP rank's share): the same
    result as the oracle over the leading entries."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = wlm.Workload("c8_ragged", [4000, 2500, 900, 3100], [1] * 4, 64, "bf16", 1024, 1, 5500, latent_format="fp8")
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    o_idx, _ = hp.oracle_topk()
    counts = [0, 65, 1024, 300]
    buf = np.full_like(o_idx, -1)
    for r, c in enumerate(counts):
        sel = o_idx[r][o_idx[r] >= 0]
        counts[r] = min(c, len(sel))
        buf[r, :counts[r]] = sel[:counts[r]]
    lse = torch.empty((wl.num_rows, 64), dtype=torch.float32, device="cuda")
    out, _ = dsa.sparse_mla_decode(gp.caches[0], gp.batch, gp.q[0], torch.from_numpy(buf).cuda(), wl.scale, lse=lse,
                                   row_counts=torch.tensor(counts, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    o_out, o_lse = hp.oracle_attention(0, buf)
    check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)
