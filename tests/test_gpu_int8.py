"""GPU parity of int8 index keys with binary16 scales ("GLM-5.2 on vLLM Ascend", section 7 and
"Quantization and Hardware Branches": INT8 indexer keys with FP16 scales).

The append quantises bf16 keys into int8 codes and half scales bit for bit as the oracle does; the
indexer splits each landed key tile into two exact e4m3 terms on chip and must give the oracle's
scores and top-k within the parity tolerances.  Cases: decode rows over several tiles with ragged
tails, pages of 4 keys (scales through registers), 16, 64 and 128 keys (bulk scale copies), extend
rows in groups of two with an odd tail, two IndexShare layers, and pre-quantised keys copied as given.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import dsa_oracle as o
from test_gpu_parity import run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    return lib


CASES = [
    # name, seq_lens, q_lens, page size, top-k, layers, seed
    ("int8_decode_p64", [300, 512, 1000, 4097], [1, 1, 1, 1], 64, 256, 1, 3101),
    ("int8_decode_p4", [333, 700], [1, 1], 4, 128, 1, 3102),
    ("int8_decode_p16", [700, 1500, 129], [1, 1, 1], 16, 256, 1, 3103),
    ("int8_extend_p64", [600, 900, 77], [5, 3, 1], 64, 256, 2, 3104),
    ("int8_decode_p128_long", [20000, 9000], [1, 1], 128, 2048, 1, 3105),
]


@pytest.mark.parametrize("name,seq_lens,q_lens,P,topk,layers,seed", CASES, ids=[c[0] for c in CASES])
def test_int8_keys_match_the_oracle(name, seq_lens, q_lens, P, topk, layers, seed):
    run_and_check(wlm.Workload(name, seq_lens, q_lens, P, "int8", topk, layers, seed))


def test_prequantised_int8_keys_are_copied():
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    c = dsa.LayerCache(4, 8, "int8")
    rng = np.random.default_rng(3)
    codes = torch.from_numpy(rng.integers(-127, 128, (3, 128), dtype=np.int8)).cuda()
    scales = torch.tensor([0.5, 2.0, 1e-3], dtype=torch.float16, device="cuda")
    z = torch.zeros((3, 512), dtype=torch.bfloat16, device="cuda")
    dsa.kv_append(c, z, torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda"),
                  torch.tensor([0, 9, 31], dtype=torch.int64, device="cuda"), k_idx=codes, k_idx_scales=scales)
    keys = c.index_keys.view(-1, 128)
    assert torch.equal(keys[[0, 9, 31]], codes)
    assert torch.equal(c.index_scales.view(-1)[[0, 9, 31]], scales)


def test_int8_append_edge_rows_match_the_oracle_bit_for_bit():
    """amax 0, a scale below half's range, a constant row, a scale held at 65504, a subnormal half scale."""
    import torch
    import deepseek_sparse_mla_gb300 as dsa
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 128)).astype(np.float32)
    x[0] = 0.0
    x[1] *= np.float32(2.0 ** -30)
    x[2, :] = np.float32(-0.75)
    x[3] *= np.float32(2.0 ** 24)
    x[4] *= np.float32(2.0 ** -17)
    bits = wlm.bf16_bits(x)
    want_codes, want_scales = o.quantize_index_keys_int8(bits)
    c = dsa.LayerCache(1, 8, "int8")
    z = torch.zeros((6, 512), dtype=torch.bfloat16, device="cuda")
    dsa.kv_append(c, z, torch.zeros((6, 64), dtype=torch.bfloat16, device="cuda"),
                  torch.arange(6, dtype=torch.int64, device="cuda"), k_idx=wlm.bits_to_torch(bits, "cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(c.index_keys.view(-1, 128)[:6].cpu().numpy(), want_codes)
    assert np.array_equal(c.index_scales.view(-1)[:6].cpu().numpy().view(np.uint16), want_scales)
