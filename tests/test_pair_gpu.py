"""Parity of the CTA-pair forward (dense, head_dim 128) with the fp64 oracle,
through the C ABI.

The pair kernel runs one tcgen05 .cta_group::2 MMA over two SMs (256 query
rows against 256 keys) and merges split key ranges inside the kernel; it must
compute the same function as the definition.  Bars as in test_parity_gpu:
max |O - O_ref| <= 1e-2, max |lse - lse_ref| <= 1e-3 on unit-normal inputs,
rows without keys O = 0 and lse = -inf.  Shapes cover one tile, ragged tails
of both the query block (a CTA of the pair with no valid row) and the key
tile, GQA, causal with Lq != Lk (including blocks that see no key), fp16,
split pieces merged in the kernel, and the single-CTA kernel on the same
inputs for comparison.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import WORKLOADS, Workload, generate, sample_rows

from .test_parity_gpu import check, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    attn.set_pair_forward(True)
    assert attn.pair_forward_used(128, False)
    yield attn_lib
    attn.set_pair_forward(False)


SHAPES = [
    # B, Hq, Hkv, Lq, Lk, dtype, causal
    (1, 1, 1, 256, 256, "bf16", False),      # one unit, one tile
    (1, 1, 1, 128, 256, "bf16", False),      # the second CTA of the pair has no row
    (1, 2, 2, 300, 300, "bf16", True),       # ragged query block and key tile
    (2, 4, 2, 513, 513, "bf16", True),       # GQA, ragged
    (1, 2, 1, 200, 1000, "fp16", False),     # Lq != Lk
    (1, 2, 2, 100, 600, "bf16", True),       # causal bottom-right, Lq < Lk
    (1, 2, 2, 700, 100, "bf16", True),       # causal, Lq > Lk: rows and whole blocks without keys
    (1, 1, 1, 1, 1, "bf16", False),
    (3, 8, 8, 77, 77, "fp16", True),
    (1, 8, 2, 512, 1024, "bf16", False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_pair_small_shapes_full(shape):
    B, Hq, Hkv, Lq, Lk, dt, causal = shape
    wl = Workload("pair", B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=128, dtype=dt, causal=causal, seed=13)
    inp = generate(wl)
    o, lse = run(inp, causal)
    o_ref, lse_ref = oracle.attention(inp.q, inp.k, inp.v, causal=causal, scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, str(shape))


@pytest.mark.parametrize("L", [2048, 4096])
def test_pair_split_merge(L):
    """A long causal single head: the schedule splits key ranges and the
    kernel merges the pieces (each piece merges one row slice of its block
    once every piece has written its partial)."""
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert attn.fwd_splits(1, 1, 1, L, L, 128, True, n_sms)
    wl = Workload("pair_split", B=1, Hq=1, Hkv=1, Lq=L, Lk=L, d=128, dtype="bf16", causal=True, seed=17)
    inp = generate(wl)
    o, lse = run(inp, True)
    o_ref, lse_ref = oracle.attention(inp.q, inp.k, inp.v, causal=True, scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, f"split L{L}")


def test_pair_headline_sampled_and_repeatable():
    wl = WORKLOADS["single_head_l8192_d128_causal"]
    inp = generate(wl)
    o, lse = run(inp, True)
    rows = sample_rows(wl, 256)
    o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=True, scale=wl.softmax_scale)
    idx = np.array(rows)
    check(o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref, wl.name)
    # causal row 0 sees only key 0
    assert np.array_equal(o[0, 0, 0], inp.v[0, 0, 0].double().numpy())
    o2, lse2 = run(inp, True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_pair_matches_single_cta_kernel():
    """Both kernels on the same inputs (GQA, causal, a split schedule)."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, 3000, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(1, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(1, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    o1, l1 = attn.attn_fwd(q, k, v, causal=True)
    attn.set_pair_forward(False)
    try:
        o2, l2 = attn.attn_fwd(q, k, v, causal=True)
    finally:
        attn.set_pair_forward(True)
    assert attn.get_error() == attn.ATTN_OK
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
    assert float((l1 - l2).abs().max()) <= 1e-3
