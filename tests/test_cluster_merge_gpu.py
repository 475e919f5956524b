"""Parity of the in-cluster merge (attn_set_cluster_merge: every 256-row
query block split into 2, 4 or 8 equal key-range pieces that run as one
thread-block cluster and merge their partials over distributed shared
memory) with the fp64 oracle, through the C ABI.

Reference: the oracle's attention (page S23-J17 §3: the exact softmax
attention the tiled method reproduces; the merge is its r = exp(m_s - M)
rescaling across pieces, §3.1).  Bars as in test_parity_gpu: max |O - O_ref|
<= 1e-2, max |lse - lse_ref| <= 1e-3.  Covers ragged lengths, causal blocks
whose pieces are unequal or empty, both head dims and both 16-bit types, and
agreement with the default merge (a combine pass).
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import Workload, generate, sample_rows

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    attn.set_pair_forward(False)
    yield attn_lib
    attn.set_cluster_merge(0)


CASES = [
    # B, Hq, Hkv, L, d, dtype, causal, cluster size
    (1, 1, 1, 2048, 128, "bf16", False, 4),
    (1, 2, 1, 1000, 64, "fp16", False, 2),    # ragged: the last block has 232 rows, the last key tile 104 keys
    (2, 4, 2, 700, 128, "bf16", True, 2),     # causal: pieces of unequal length
    (1, 2, 2, 300, 128, "bf16", True, 8),     # most pieces of the first block are empty
    (1, 4, 4, 1536, 64, "bf16", False, 8),
    (1, 1, 1, 8192, 128, "bf16", False, 8),   # sampled rows
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_cluster_merge_matches_oracle(case):
    B, Hq, Hkv, L, d, dtype, causal, cs = case
    wl = Workload("cm", B=B, Hq=Hq, Hkv=Hkv, Lq=L, Lk=L, d=d, dtype=dtype, causal=causal, seed=L + cs)
    inp = generate(wl)
    dev = torch.device("cuda", 0)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    attn.set_cluster_merge(cs)
    assert attn.cluster_merge() == cs
    o, lse = attn.attn_fwd(q, k, v, causal=causal)
    assert attn.get_error() == attn.ATTN_OK
    o, lse = o.float().cpu().double().numpy(), lse.cpu().double().numpy()
    if L <= 2048:
        o_ref, lse_ref = oracle.attention(inp.q, inp.k, inp.v, causal=causal, scale=wl.softmax_scale)
    else:
        rows = sample_rows(wl, 128)
        o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=causal, scale=wl.softmax_scale)
        idx = np.array(rows)
        o, lse = o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]]
    fin = ~np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), ~fin)
    assert float(np.abs(o - o_ref).max()) <= O_TOL
    assert float(np.abs(lse[fin] - lse_ref[fin]).max()) <= LSE_TOL


def test_cluster_merge_agrees_with_the_combine_pass():
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, 3000, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(2, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(2, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    attn.set_cluster_merge(0)
    o0, l0 = attn.attn_fwd(q, k, v, causal=False)
    for cs in (2, 4, 8):
        attn.set_cluster_merge(cs)
        o1, l1 = attn.attn_fwd(q, k, v, causal=False)
        assert attn.get_error() == attn.ATTN_OK
        assert float((o1.float() - o0.float()).abs().max()) <= O_TOL
        assert float((l1 - l0).abs().max()) <= LSE_TOL


def test_cluster_merge_ignores_other_sizes():
    attn.set_cluster_merge(4)
    attn.set_cluster_merge(3)
    assert attn.cluster_merge() == 4
    attn.set_cluster_merge(16)
    assert attn.cluster_merge() == 4
