"""GPU parity: the CUDA path against the float64 oracle on the same seeded inputs.

Reduced forms of the five workloads (several tiles, ragged tails, contexts longer than top-k)
are compared element by element; edge cases cover short contexts, k = 1, page sizes 1 and
1024, empty and out-of-range selections, page/request permutation and append canaries.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from parity import (GpuProblem, HostProblem, bf16_tensor_to_f64, check_attention, check_cache_bytes, check_scores,
                    check_topk)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


def run_and_check(wl, check_selection=True):
    import torch
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    torch.cuda.synchronize()
    check_cache_bytes(gp, hp)
    idx_g, scores_g = gp.indexer()
    o_idx, o_scores = hp.oracle_topk()
    g_idx, g_sc = idx_g.cpu().numpy(), scores_g.cpu().numpy()
    _, pos = o.row_positions(wl.seq_lens, wl.query_start_loc)
    swaps = 0
    for r in range(wl.num_rows):
        check_scores(g_sc[r], o_scores[r], int(pos[r]), wl.max_seq_len)
        if check_selection:
            swaps += check_topk(g_idx[r], o_idx[r], o_scores[r], int(pos[r]), wl.topk)
    oracle_idx = torch.from_numpy(o_idx).to("cuda")
    errs = []
    for layer in range(wl.layers):
        out, lse = gp.attention(layer, oracle_idx)
        o_out, o_lse = hp.oracle_attention(layer, o_idx)
        errs.append(check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse))
        # the product path on its own selection runs too and stays finite
        out2, lse2 = gp.attention(layer, idx_g)
        assert torch.isfinite(out2.float()).all()
    return hp, gp, swaps, errs


@pytest.mark.parametrize("name", list(wlm.FULL))
def test_reduced_workload_parity(name):
    run_and_check(wlm.reduced(name))


def test_short_contexts_select_every_position():
    wl = wlm.Workload("short", [1, 2, 127, 128, 129, 300], [1] * 6, 16, "bf16", 128, 1, 3001)
    run_and_check(wl)


def test_topk_one_and_page_size_one():
    wl = wlm.Workload("k1_p1", [50, 333], [1, 1], 1, "fp8", 1, 2, 3002)
    run_and_check(wl)


def test_large_pages_and_multi_row_requests():
    wl = wlm.Workload("p1024_extend", [1500, 2600, 700], [3, 5, 1], 1024, "bf16", 512, 2, 3003)
    run_and_check(wl)


def test_prefill_rows_on_both_sides_of_topk():
    """Extend rows whose visible count crosses k inside the chunk: the first rows keep every position."""
    wl = wlm.Workload("extend_cross_k", [600], [200], 64, "fp8", 512, 1, 3004)
    run_and_check(wl)


def test_empty_and_out_of_range_selections():
    import torch
    wl = wlm.Workload("sel_edge", [90, 200], [1, 1], 16, "bf16", 32, 1, 3005)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    idx = np.full((2, 32), -1, dtype=np.int32)
    idx[1, :6] = [0, 5, 199, 250, -7, 100]          # 250 > pos, -7 invalid: both skipped
    out, lse = gp.attention(0, torch.from_numpy(idx).cuda())
    o_out, o_lse = hp.oracle_attention(0, idx)
    g_out, g_lse = bf16_tensor_to_f64(out), lse.cpu().numpy()
    assert not g_out[0].any() and np.all(np.isneginf(g_lse[0]))
    check_attention(g_out, g_lse, o_out, o_lse)


def test_unit_split_rows_with_empty_pieces():
    """80 rows x 2 tiles (160 units on 152 CTAs): rows 9, 19, ..., 79 are whole in one CTA and written there, the
    other 72 are cut between two CTAs and finished by the merge kernel.  Selections cycle through empty, full and
    one valid tile only (the other piece, or the other half of a whole row, holds no valid entry), each pattern on
    whole and on cut rows: an empty row must come out as zeros with lse = -inf, and an empty piece adds nothing."""
    import torch
    rng = np.random.default_rng(3011)
    seq_lens = rng.integers(150, 400, size=80)
    wl = wlm.Workload("unit_split_edge", seq_lens, [1] * 80, 16, "bf16", 128, 1, 3011)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    idx = np.full((80, 128), -1, dtype=np.int32)
    pattern = (np.arange(80) // 10 + np.arange(80) % 10) % 4
    for r, L in enumerate(seq_lens):
        sel = rng.choice(int(L), size=128, replace=False).astype(np.int32)
        if pattern[r] == 1:
            idx[r] = sel
        elif pattern[r] == 2:
            idx[r, 64:] = sel[64:]                   # only the second tile has valid entries
        elif pattern[r] == 3:
            idx[r, :64] = sel[:64]                   # only the first tile has valid entries
    out, lse = gp.attention(0, torch.from_numpy(idx).cuda())
    o_out, o_lse = hp.oracle_attention(0, idx)
    g_out, g_lse = bf16_tensor_to_f64(out), lse.cpu().numpy()
    empty = pattern == 0
    assert not g_out[empty].any() and np.all(np.isneginf(g_lse[empty]))
    assert np.all(np.isfinite(g_lse[~empty]))
    check_attention(g_out, g_lse, o_out, o_lse)


def test_page_permutation_gives_identical_results():
    """Same logical tokens under two physical page layouts: bitwise identical outputs."""
    import torch
    a = wlm.Workload("perm_a", [777, 1300], [1, 1], 64, "fp8", 256, 1, 3006)
    b = wlm.Workload("perm_a", [777, 1300], [1, 1], 64, "fp8", 256, 1, 3006)
    perm = np.random.default_rng(5).permutation(b.num_pages).astype(np.int32)
    b.block_table = np.where(a.block_table >= 0, perm[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    res = []
    for wl in (a, b):
        gp = GpuProblem(HostProblem(wl))
        gp.append_step()
        idx, sc = gp.indexer()
        out, lse = gp.attention(0, idx)
        torch.cuda.synchronize()
        res.append((idx.cpu().numpy(), sc.cpu().numpy(), wlm.torch_to_bits(out), lse.cpu().numpy()))
    for x, y in zip(*res):
        assert np.array_equal(x, y)


def test_request_isolation_under_batch_permutation():
    """A request's rows give the same result alone and inside a permuted batch."""
    import torch
    wl = wlm.Workload("iso", [900, 2100, 1500], [1, 1, 1], 64, "bf16", 256, 1, 3007)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    idx, _ = gp.indexer()
    out, lse = gp.attention(0, idx)
    import deepseek_sparse_mla_gb300 as dsa
    order = [2, 0, 1]
    bt = torch.from_numpy(wl.block_table[order]).cuda()
    sl = torch.tensor([wl.seq_lens[i] for i in order], dtype=torch.int32, device="cuda")
    batch = dsa.Batch(bt, sl, None, num_rows=3, max_seq_len=wl.max_seq_len)
    idx_p = dsa.indexer_scores_topk(gp.caches[0], batch, gp.q_idx[order].contiguous(), gp.w[order].contiguous(), 256)
    out_p, _ = dsa.sparse_mla_decode(gp.caches[0], batch, gp.q[0][order].contiguous(), idx_p)
    assert torch.equal(idx_p, idx[order])
    assert torch.equal(out_p, out[order])


def test_append_leaves_other_slots_untouched():
    """Canary: after append only the addressed slots change, in both caches."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    c = dsa.LayerCache(8, 16, "fp8")
    c.latent.view(torch.int16).fill_(0x5A5A)
    c.index_keys.fill_(0xA5)
    c.index_scales.fill_(-3.0)
    slots = torch.tensor([3, 17, 127, -1, 128 * 4], dtype=torch.int64, device="cuda")   # -1 and out-of-range skipped
    T = 5
    rng = np.random.default_rng(1)
    ckv = wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 512), dtype=np.float32)), "cuda")
    kr = wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 64), dtype=np.float32)), "cuda")
    ki = wlm.bits_to_torch(wlm.bf16_bits(rng.standard_normal((T, 128), dtype=np.float32)), "cuda")
    dsa.kv_append(c, ckv, kr, slots, k_idx=ki)
    torch.cuda.synchronize()
    lat = c.latent.view(-1, 576).view(torch.int16).cpu().numpy()
    keys = c.index_keys.view(-1, 128).cpu().numpy()
    sc = c.index_scales.view(-1).cpu().numpy()
    written = [3, 17, 127]
    others = np.setdiff1d(np.arange(128), written)
    assert np.all(lat[others] == 0x5A5A) and np.all(keys[others] == 0xA5) and np.all(sc[others] == -3.0)
    host = o.PagedCache(8, 16, "fp8")
    host.append(wlm.torch_to_bits(ckv)[:3], wlm.torch_to_bits(kr)[:3], np.array(written), k_idx_bits=wlm.torch_to_bits(ki)[:3])
    assert np.array_equal(lat[written].view(np.uint16), host.latent.reshape(-1, 576)[written])
    assert np.array_equal(keys[written], host.index_keys.reshape(-1, 128)[written])
    assert np.array_equal(sc[written], host.index_scales.reshape(-1)[written])


def test_prequantised_keys_are_copied():
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    c = dsa.LayerCache(4, 8, "fp8")
    rng = np.random.default_rng(2)
    codes = torch.from_numpy(rng.integers(0, 0x7E, (3, 128), dtype=np.uint8)).cuda()
    scales = torch.tensor([0.5, 2.0, 1e-3], dtype=torch.float32, device="cuda")
    z = torch.zeros((3, 512), dtype=torch.bfloat16, device="cuda")
    dsa.kv_append(c, z, torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda"),
                  torch.tensor([0, 9, 31], dtype=torch.int64, device="cuda"), k_idx=codes, k_idx_scales=scales)
    keys = c.index_keys.view(-1, 128)
    assert torch.equal(keys[[0, 9, 31]], codes)
    assert torch.equal(c.index_scales.view(-1)[[0, 9, 31]], scales)


def test_selection_order_does_not_matter_and_forces_rescales():
    """The index buffer is a set: entries sorted by ascending score make every later tile raise the
    running maximum (so the accumulator is rescaled several times) and must give the oracle's result."""
    import torch
    wl = wlm.Workload("rescale", [5000, 4100], [1, 1], 64, "bf16", 2048, 1, 3008)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    o_idx, _ = hp.oracle_topk()
    q = o.bf16_to_f64(hp.q[0])
    ordered = o_idx.copy()
    for r in range(wl.num_rows):
        sel = o_idx[r]
        rows = hp.caches[0].latent_rows(wl.block_table[r], sel)
        z0 = rows @ q[r, 0]                                   # head 0's logits
        ordered[r] = sel[np.argsort(z0)]
    out, lse = gp.attention(0, torch.from_numpy(ordered).cuda())
    o_out, o_lse = hp.oracle_attention(0, o_idx)
    check_attention(bf16_tensor_to_f64(out), lse.cpu().numpy(), o_out, o_lse)


def test_device_status_word_is_clear_after_calls():
    """Kernels record bounded-wait timeouts in the first word of the workspace; a normal call leaves 0."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = wlm.reduced("decode_b64_fp8_indexshare")
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    idx, _ = gp.indexer()
    ws = torch.full((dsa.mla_workspace_bytes(wl.num_rows, wl.topk),), 0xFF, dtype=torch.uint8, device="cuda")
    dsa.sparse_mla_decode(gp.caches[1], gp.batch, gp.q[1], idx, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_results_are_deterministic_across_calls():
    import torch
    wl = wlm.reduced("decode_b64_fp8_indexshare")
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    a = gp.indexer()
    b = gp.indexer()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    oa = gp.attention(1, a[0])
    ob = gp.attention(1, a[0])
    assert torch.equal(oa[0], ob[0]) and torch.equal(oa[1], ob[1])


def test_long_rows_split_into_chunks():
    """Rows longer than the top-k chunk (32,768 positions) are scanned by several CTAs whose candidate
    lists are merged: rows just below, at and just above the boundary, and one spanning three chunks."""
    wl = wlm.Workload("long_chunks", [70001, 32768, 32769, 40000], [1] * 4, 64, "fp8", 256, 1, 3010)
    run_and_check(wl)


def test_all_equal_scores_keep_the_first_positions():
    """A zero indexer query gives every position the score 0: the tie rule (smaller position first)
    fixes the selection exactly, and every candidate list overflows, so the full-row select runs."""
    import torch
    wl = wlm.Workload("ties", [5000, 40000, 300], [1] * 3, 64, "bf16", 2048, 1, 3011)
    gp = GpuProblem(HostProblem(wl))
    gp.append_step()
    gp.q_idx.zero_()
    idx, sc = gp.indexer()
    torch.cuda.synchronize()
    g_idx, g_sc = idx.cpu().numpy(), sc.cpu().numpy()
    for r, L in enumerate(wl.seq_lens):
        assert np.all(g_sc[r, :L] == 0.0)
        want = np.arange(wl.topk, dtype=np.int32) if L > wl.topk else np.r_[np.arange(L), np.full(wl.topk - L, -1)]
        assert np.array_equal(g_idx[r], want)


def test_e4m3_scales_of_small_pages():
    """Pages of 16 and 32 keys put 8 or 4 pages' scales into each 128-key tile (two or one gathers of
    four page rows), with ragged lengths that leave part of the last group without a page."""
    run_and_check(wlm.Workload("fp8_p16", [700, 1500, 333], [1, 1, 1], 16, "fp8", 256, 1, 3012))
    run_and_check(wlm.Workload("fp8_p32", [1111, 2050], [1, 1], 32, "fp8", 512, 1, 3013))


def _sampled_positions(n):
    """Positions the top-k sample threshold reads in a row of n >= 4096 scores: 512 runs of 8
    consecutive scores, run j starting at the multiple of 8 at or below j n / 512."""
    j = np.arange(512, dtype=np.int64)
    return ((((j * n) >> 9) & ~7)[:, None] + np.arange(8)).ravel()


def _order_key(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


@pytest.mark.parametrize("seq_lens", [[20000, 9000], [100000, 70001]])
def test_planted_sample_pushes_threshold_above_kth_score(seq_lens):
    """High scores planted exactly on the positions the sample threshold reads put that threshold far
    above the row's true k-th score, so fewer than k positions clear it and the full-row select runs
    (rows scanned by one CTA, and rows split into chunks).  Every query head is the unit vector e_0 and
    the head weights are positive, so a position's score is ReLU(key[0]): a descending ramp on the
    sampled positions (shuffled over them), -1 elsewhere."""
    wl = wlm.Workload("planted_sample", list(seq_lens), [1] * len(seq_lens), 64, "bf16", 2048, 1, 3020)
    hp = HostProblem(wl)
    rng = np.random.default_rng(3021)
    for b, L in enumerate(wl.seq_lens):
        keys = o.bf16_to_f64(hp.keys[b]).astype(np.float32)
        keys[:, 0] = -1.0
        sp = _sampled_positions(L)
        keys[sp, 0] = rng.permutation(np.linspace(1.0, 1000.0, sp.size)).astype(np.float32)
        hp.keys[b] = wlm.bf16_bits(keys)
    q = np.zeros((wl.num_rows, 32, 128), dtype=np.float32)
    q[:, :, 0] = 1.0
    hp.q_idx = wlm.bf16_bits(q)
    hp.w = np.full((wl.num_rows, 32), 1.0 / 32, dtype=np.float32)
    hp.caches[0] = o.PagedCache(wl.num_pages, wl.page_size, wl.key_format)
    for b, L in enumerate(wl.seq_lens):
        hp.caches[0].append(hp.latent[0][b][:, :512], hp.latent[0][b][:, 512:], wl.slots(b, np.arange(L)),
                            k_idx_bits=hp.keys[b])
    o_idx, o_sc = hp.oracle_topk()
    # the construction does what it is for: fewer than k positions reach the sample threshold's bin
    k = wl.topk
    for r, L in enumerate(wl.seq_lens):
        samp = np.sort(_order_key(o_sc[r][_sampled_positions(L)]))[::-1]
        rank = k * 4096 // L
        margin = 3 * int(np.sqrt(rank + 1.0)) + 8
        edge = (samp[rank + margin] >> 20) << 20
        assert np.count_nonzero(_order_key(o_sc[r][:L]) >= edge) < k
    gp = GpuProblem(hp)
    gp.append_step()
    idx, sc = gp.indexer()
    import torch
    torch.cuda.synchronize()
    g_idx, g_sc = idx.cpu().numpy(), sc.cpu().numpy()
    for r, L in enumerate(wl.seq_lens):
        check_scores(g_sc[r], o_sc[r], L - 1, wl.max_seq_len)
        check_topk(g_idx[r], o_idx[r], o_sc[r], L - 1, k)


def _layer_group_workload(kind):
    if kind == "clusters":
        return wlm.reduced("decode_b64_fp8_indexshare")          # 6 rows x 4 layers: clusters of 4 CTAs
    lens = np.random.default_rng(2203).integers(1500, 3200, 20).tolist()
    if kind == "unit_split":                                       # 80 stacked rows: rows cut between CTAs
        return wlm.Workload("decode_b20_ctx1500-3200_fp8_layers4", lens, [1] * 20, 64, "fp8", 512, 4, 2203)
    return wlm.Workload("decode_b3_ctx1500-3200_c8_layers2", lens[:3], [1] * 3, 64, "fp8", 512, 2, 2204,
                        latent_format="fp8")


@pytest.mark.parametrize("kind", ["clusters", "unit_split", "packed_latent"])
def test_layer_group_attention_in_one_call(kind):
    """dsa_sparse_mla_decode_layers: an IndexShare group's layers attend with the owner's buffer in
    one call (stacked q / out / lse), each layer against the oracle on the oracle's selection and
    against the one-layer call."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = _layer_group_workload(kind)
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    gp.append_step()
    o_idx, _ = hp.oracle_topk()
    idx = torch.from_numpy(o_idx).to("cuda")
    q = torch.stack(gp.q).contiguous()
    lse = torch.empty((wl.layers, wl.num_rows, 64), dtype=torch.float32, device="cuda")
    out, _ = dsa.sparse_mla_decode_layers(gp.caches, gp.batch, q, idx, wl.scale, lse=lse, check=True)
    torch.cuda.synchronize()
    for layer in range(wl.layers):
        o_out, o_lse = hp.oracle_attention(layer, o_idx)
        check_attention(bf16_tensor_to_f64(out[layer]), lse[layer].cpu().numpy(), o_out, o_lse)
        one, one_lse = gp.attention(layer, idx)
        assert (out[layer].float() - one.float()).abs().max().item() <= 2e-2
        fin = torch.isfinite(one_lse)
        assert torch.equal(fin, torch.isfinite(lse[layer]))
        assert (lse[layer][fin] - one_lse[fin]).abs().max().item() <= 1e-4


def test_layer_group_call_rejects_mismatched_layers():
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    wl = wlm.reduced("decode_b64_fp8_indexshare")
    hp = HostProblem(wl)
    gp = GpuProblem(hp)
    other = dsa.LayerCache(wl.num_pages * 2, wl.page_size, None, "cuda")
    idx = torch.zeros((wl.num_rows, wl.topk), dtype=torch.int32, device="cuda")
    q = torch.zeros((2, wl.num_rows, 64, 576), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError):
        dsa.sparse_mla_decode_layers([gp.caches[0], other], gp.batch, q, idx, wl.scale)
    with pytest.raises(dsa.DsaError):
        dsa.sparse_mla_decode_layers([gp.caches[0]] * 5, gp.batch,
                                     torch.zeros((5, wl.num_rows, 64, 576), dtype=torch.bfloat16, device="cuda"),
                                     idx, wl.scale)
