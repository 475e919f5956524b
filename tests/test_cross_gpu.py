"""Parity of the packed forward with separate query and key offsets
(attn_fwd_varlen: cross-attention, queries extending a key/value cache)
against the oracle's per-sequence dense runs; every element compared.
Bar: max |O - O_ref| <= 1e-2, max |lse - lse_ref| <= 1e-3; rows with no key
give O = 0 and lse = -inf on both sides."""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def cu_of(lengths):
    return torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32)


def run_case(lq, lk, Hq, Hkv, d, causal, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(sum(lq), Hq, d, generator=g).to(dtype)
    k = torch.randn(max(sum(lk), 1), Hkv, d, generator=g).to(dtype)
    v = torch.randn(max(sum(lk), 1), Hkv, d, generator=g).to(dtype)
    dev = torch.device("cuda", 0)
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, cu_seqlens=cu_of(lq).to(dev),
                           cu_seqlens_k=cu_of(lk).to(dev))
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.varlen_cross_attention(q, k, v, lq, lk, causal=causal, scale=d ** -0.5)
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), inf)
    assert float(np.abs(o - o_ref).max()) <= O_TOL
    if (~inf).any():
        assert float(np.abs(lse[~inf] - lse_ref[~inf]).max()) <= LSE_TOL
    assert np.all(o[inf.T] == 0.0)


CASES = [
    # query lengths, key lengths, Hq, Hkv, d, causal, dtype
    ([37, 300, 1, 129], [500, 77, 256, 129], 4, 2, 64, False, torch.bfloat16),      # cross-attention
    ([64, 200, 5, 256], [64 + 700, 200 + 33, 5 + 1000, 256], 4, 4, 128, True, torch.bfloat16),   # cache + queries
    ([300, 20, 130], [100, 0, 130], 2, 1, 64, True, torch.float16),                   # keys < queries, no keys
    ([0, 17, 0], [50, 3, 0], 2, 2, 128, False, torch.bfloat16),                       # empty sequences
    ([1, 1, 1, 1], [900, 1, 2000, 33], 8, 2, 128, True, torch.bfloat16),              # one new token per sequence
    # grouped heads sharing a tile (group 2..32: 64..4 queries x group heads per 128 rows)
    ([1, 2, 17, 16, 33, 0], [1, 700, 17, 300, 4000, 9], 16, 2, 128, True, torch.bfloat16),   # group 8
    ([5, 8, 9, 0, 70], [300, 8, 1, 40, 70], 32, 2, 64, False, torch.float16),           # group 16, d 64
    ([1, 3, 4, 5, 130], [2000, 3, 500, 129, 130], 32, 1, 128, True, torch.bfloat16),    # group 32 (one kv head)
    ([64, 65, 200, 1], [64, 1000, 200, 257], 8, 2, 128, True, torch.bfloat16),         # group 4 over several blocks
    ([1, 7, 40], [1000, 7, 300], 6, 2, 128, True, torch.bfloat16),                     # group 3: one head per tile
    # queries that fill one 128-row sub-tile over several key tiles, where the
    # first rows see only the first key tile (causal, short cache)
    ([100, 30, 3], [200, 140, 700], 2, 2, 128, True, torch.bfloat16),
    ([100, 30, 3], [200, 140, 700], 2, 2, 64, True, torch.float16),
]

# Up to 32 sequences are placed in order of their key counts (ties by index);
# more keep their order.  32 and 33 sequences with repeated lengths and empty
# ones, and a kv-cache-like mix.
_rng = np.random.default_rng(123)
_lq32 = _rng.integers(0, 300, 32).tolist()
_lq32[5] = 0
_lk32 = [a + int(c) for a, c in zip(_lq32, _rng.choice([0, 64, 500, 1500], 32))]
_lq33 = _rng.integers(1, 200, 33).tolist()
CASES += [
    (_lq32, _lk32, 8, 2, 128, True, torch.bfloat16),
    (_lq32, _lq32, 4, 4, 64, False, torch.bfloat16),
    (_lq33, [a + 100 for a in _lq33], 8, 2, 128, True, torch.bfloat16),
    ([300] * 12, [300, 800, 300, 2000, 300, 800, 300, 2000, 300, 800, 300, 2000], 2, 2, 64, True, torch.float16),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_cross_varlen(case):
    lq, lk, Hq, Hkv, d, causal, dtype = case
    run_case(lq, lk, Hq, Hkv, d, causal, dtype, seed=sum(lq) + sum(lk))


def test_cross_needs_both_offsets_and_matching_counts():
    dev = torch.device("cuda", 0)
    q = torch.randn(10, 2, 64, device=dev, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q, cu_seqlens_k=cu)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q, cu_seqlens=cu, cu_seqlens_k=torch.tensor([0, 5, 10], dtype=torch.int32, device=dev))


def test_cross_varlen_maximum_sequence_count():
    # 4096 sequences (the most one call takes): the kernel's prefix table of
    # units per sequence is full; short sequences, some empty on either side.
    # fp16: with a handful of keys per row O is not averaged down, and bf16's
    # rounding of P and O alone can pass 1e-2 where |O| approaches 4
    rng = np.random.default_rng(4096)
    lq = rng.integers(0, 9, 4096).tolist()
    lk = [a + int(c) for a, c in zip(lq, rng.integers(0, 6, 4096))]
    run_case(lq, lk, 4, 2, 64, True, torch.float16, seed=4096)
