"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bar (stated for this method): max |O_gpu - O_ref| <= 1e-2 with bf16/fp16
output and fp32 accumulation on unit-normal inputs, and max |lse_gpu -
lse_ref| <= 1e-3; rows that see no key must give O = 0 and lse = -inf on both
sides.  Small shapes are compared element by element; the full-size
workloads, run exactly as the benchmark runs them, are compared on sampled
rows the oracle evaluates one by one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import WORKLOADS, Workload, generate, sample_rows

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


def run(inp, causal, scale=None):
    dev = torch.device("cuda", 0)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cu = inp.cu_seqlens.to(dev) if inp.cu_seqlens is not None else None
    o, lse = attn.attn_fwd(q, k, v, causal=causal, scale=scale, cu_seqlens=cu)
    assert attn.get_error() == attn.ATTN_OK
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(o, lse, o_ref, lse_ref, what="", o_tol=O_TOL):
    """Element-wise comparison.  A failure message reports the max-abs error
    and, separately, how many violating elements have |O_ref| >= 4: there a
    bf16 output's half-ulp (2^-6) already exceeds the 1e-2 bar, so even a
    correctly rounded result can miss it.  The bar itself is not relaxed."""
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), inf_ref), f"{what}: -inf rows differ"
    dev = np.abs(o - o_ref)
    err_o = np.max(dev) if o.size else 0.0
    fin = ~inf_ref
    err_l = np.max(np.abs(lse[fin] - lse_ref[fin])) if fin.any() else 0.0
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    bar = o_tol if np.isscalar(o_tol) else o_tol
    bad = dev > bar
    if np.any(bad):
        big = bad & (np.abs(o_ref) >= 4.0)
        raise AssertionError(f"{what}: max |dO| = {err_o:.3e}; {int(bad.sum())} elements over the bar, "
                             f"{int(big.sum())} of them with |O_ref| >= 4 (bf16 half-ulp > 1e-2 there)")
    assert err_l <= LSE_TOL, f"{what}: max |dlse| = {err_l:.3e}"
    return err_o, err_l


# ---------------------------------------------------------------------------
# the worked example: scores [0, ln 2], values [1, 3] -> 7/3
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_worked_example(dtype):
    d = 64
    q = torch.zeros(1, 1, 1, d)
    q[0, 0, 0, 0] = 1.0
    k = torch.zeros(1, 2, 1, d)
    k[0, 1, 0, 0] = 1.0
    v = torch.zeros(1, 2, 1, d)
    v[0, 0, 0, 0] = 1.0
    v[0, 1, 0, 0] = 3.0
    dev = torch.device("cuda", 0)
    o, lse = attn.attn_fwd(q.to(dev, dtype), k.to(dev, dtype), v.to(dev, dtype), scale=math.log(2.0))
    assert attn.get_error() == attn.ATTN_OK
    assert abs(float(o[0, 0, 0, 0]) - 7.0 / 3.0) < O_TOL
    assert torch.all(o[0, 0, 0, 1:] == 0)
    assert abs(float(lse[0, 0, 0]) - math.log(3.0)) < LSE_TOL


# ---------------------------------------------------------------------------
# small shapes, every element
# ---------------------------------------------------------------------------

SMALL = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal
    (1, 2, 2, 256, 256, 64, "bf16", False),
    (1, 2, 2, 256, 256, 64, "bf16", True),
    (2, 4, 2, 300, 300, 128, "bf16", True),     # ragged tail, GQA
    (2, 4, 2, 300, 300, 128, "fp16", False),
    (1, 3, 1, 129, 700, 128, "bf16", False),    # Lq != Lk
    (1, 2, 1, 100, 333, 64, "bf16", True),      # causal, bottom-right, Lq < Lk
    (1, 2, 2, 300, 100, 64, "fp16", True),      # causal, Lq > Lk: rows without keys
    (2, 2, 2, 1, 1, 64, "bf16", False),
    (1, 1, 1, 1, 5, 128, "bf16", True),
    (1, 2, 2, 640, 640, 64, "fp16", True),
    (3, 8, 8, 77, 77, 128, "bf16", True),
    (1, 8, 2, 512, 1024, 128, "bf16", False),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "-".join(map(str, s)))
def test_small_shapes_full(shape):
    B, Hq, Hkv, Lq, Lk, d, dt, causal = shape
    wl = Workload("small", B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=d, dtype=dt, causal=causal, seed=11)
    inp = generate(wl)
    o, lse = run(inp, causal)
    o_ref, lse_ref = oracle.attention(inp.q, inp.k, inp.v, causal=causal, scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, str(shape))


def test_config_mha_l256_d64_full():
    wl = WORKLOADS["mha_l256_d64"]
    inp = generate(wl)
    o, lse = run(inp, wl.causal)
    o_ref, lse_ref = oracle.attention(inp.q, inp.k, inp.v, causal=wl.causal, scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, wl.name)


def test_config_varlen_full():
    wl = WORKLOADS["varlen_b16_h12_d64"]
    inp = generate(wl)
    o, lse = run(inp, wl.causal)
    o_ref, lse_ref = oracle.varlen_attention(inp.q, inp.k, inp.v, inp.lengths, causal=wl.causal,
                                             scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, wl.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lengths", [[0, 1, 255, 256, 257, 600, 3], [513], [1, 1, 1], [700, 0, 0, 129]])
def test_varlen_edges_full(lengths, causal):
    wl = Workload("varlen_edges", B=len(lengths), Hq=4, Hkv=2, Lq=0, Lk=0, d=128, dtype="bf16",
                  causal=causal, seed=5, varlen=True)
    inp = generate(wl, lengths=lengths)
    o, lse = run(inp, causal)
    o_ref, lse_ref = oracle.varlen_attention(inp.q, inp.k, inp.v, inp.lengths, causal=causal,
                                             scale=wl.softmax_scale)
    check(o, lse, o_ref, lse_ref, f"varlen {lengths}")


def test_split_kv_small():
    # a long causal single head is split along the key range by the schedule
    B, H, L, d = 1, 1, 4096, 64
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, n_part = attn.plan(B, H, H, L, L, d, True, n_sms)
    assert n_part > 0
    wl = Workload("split", B=B, Hq=H, Hkv=H, Lq=L, Lk=L, d=d, dtype="bf16", causal=True, seed=3)
    inp = generate(wl)
    o, lse = run(inp, True)
    rows = sample_rows(wl, 160)
    o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=True, scale=wl.softmax_scale)
    idx = np.array(rows)
    check(o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref, "split")


@pytest.fixture
def single_cta():
    """Dense head_dim-128 forwards on the single-CTA kernel for one test."""
    attn.set_pair_forward(False)
    yield


def test_split_kv_more_than_one_merge_batch(single_cta):
    # a query block split into more than eight pieces: the combine pass reads
    # pieces in batches and rescales across batches (single head, causal,
    # d 128, single-CTA kernel; L = 12288 gives 10-12 pieces for SM counts
    # from 132 to 160)
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = next((x for x in (12288, 14336, 16384) if attn.plan(1, 1, 1, x, x, 128, True, n_sms)[0][:, 5].max() > 8),
             None)
    assert L is not None, "no candidate length splits a block into more than 8 pieces"
    wl = Workload("split9", B=1, Hq=1, Hkv=1, Lq=L, Lk=L, d=128, dtype="bf16", causal=True, seed=11)
    inp = generate(wl)
    o, lse = run(inp, True)
    rows = sample_rows(wl, 192)
    o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=True, scale=wl.softmax_scale)
    idx = np.array(rows)
    check(o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref, "split > 8")


# ---------------------------------------------------------------------------
# the full-size workloads, sampled rows
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["single_head_l8192_d128_causal", "mha_b2_h16_l2048_d64_fp16_causal",
                                  "gqa_b2_hq32_hkv8_l4096_d128_causal"])
def test_full_size_sampled(name):
    wl = WORKLOADS[name]
    inp = generate(wl)
    o, lse = run(inp, wl.causal)
    rows = sample_rows(wl, 256)
    o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=wl.causal, scale=wl.softmax_scale)
    idx = np.array(rows)
    check(o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref, name)
    if wl.causal:
        # causal row 0 sees only key 0: O equals V[0] exactly
        g = np.arange(wl.Hq) // (wl.Hq // wl.Hkv)
        v0 = inp.v[:, 0].double().numpy()[:, g]
        assert np.array_equal(o[:, 0], v0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


# ---------------------------------------------------------------------------
# value magnitude: the split-KV path must be as exact as the unsplit one
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("pair", [True, False], ids=["pair", "single"])
@pytest.mark.parametrize("vscale", [1e5, 1e-6])
@pytest.mark.parametrize("L,split", [(4096, True), (512, False)])
def test_value_magnitude_split_and_unsplit(L, split, vscale, pair):
    """bf16 values scaled by 1e5 or 1e-6 (single head, causal, d 128).  A
    split schedule stores each piece's partial output and merges the pieces;
    the result must stay finite and as accurate as without splitting.  Bar:
    the 1e-2 bar of unit-normal values scaled with the values, plus the bf16
    rounding of O itself (half an ulp, 2^-8 relative); lse does not depend on
    the values (1e-3)."""
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    attn.set_pair_forward(pair)
    try:
        _magnitude_case(L, split, vscale, n_sms)
    finally:
        attn.set_pair_forward(False)


def _magnitude_case(L, split, vscale, n_sms):
    assert attn.fwd_splits(1, 1, 1, L, L, 128, True, n_sms) == split
    wl = Workload("vmag", B=1, Hq=1, Hkv=1, Lq=L, Lk=L, d=128, dtype="bf16", causal=True, seed=21)
    inp = generate(wl)
    g = torch.Generator().manual_seed(22)
    inp.v = (torch.randn(inp.v.shape, generator=g) * vscale).to(torch.bfloat16)
    o, lse = run(inp, True)
    rows = sample_rows(wl, 256)
    o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=True, scale=wl.softmax_scale)
    idx = np.array(rows)
    o_s = o[idx[:, 0], idx[:, 2], idx[:, 1]]
    tol = 1e-2 * vscale + 2.0 ** -8 * np.abs(o_ref)
    check(o_s, lse[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref, f"L{L} v x {vscale:g}", o_tol=tol)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


# ---------------------------------------------------------------------------
# properties and degenerate cases
# ---------------------------------------------------------------------------

def test_zero_scale_is_mean_of_values():
    wl = Workload("zs", B=1, Hq=2, Hkv=2, Lq=200, Lk=200, d=64, dtype="bf16", causal=True, seed=8)
    inp = generate(wl)
    o, lse = run(inp, True, scale=0.0)
    v = inp.v.double().numpy()
    ref = np.cumsum(v, axis=1) / np.arange(1, 201)[None, :, None, None]
    assert np.max(np.abs(o - ref)) <= O_TOL
    assert np.max(np.abs(lse - np.log(np.arange(1, 201))[None, None, :])) <= LSE_TOL


def test_repeat_is_bitwise_identical():
    wl = WORKLOADS["single_head_l8192_d128_causal"]
    inp = generate(wl)
    dev = torch.device("cuda", 0)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    o1, l1 = attn.attn_fwd(q, k, v, causal=True)
    o2, l2 = attn.attn_fwd(q, k, v, causal=True)
    assert attn.get_error() == attn.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_wait_timeout_is_reported_and_context_survives():
    attn.set_wait_timeout_ns(1_000_000)   # 1 ms
    try:
        assert attn.selftest_wait_timeout() == attn.ATTN_OK
        assert attn.get_error() == attn.ATTN_EDEVICE
        assert attn.last_device_error() & 0xF00 == attn.ATTN_DEVERR_WAIT_TIMEOUT
    finally:
        attn.set_wait_timeout_ns(2_000_000_000)
    assert attn.get_error() == attn.ATTN_OK
    test_worked_example(torch.bfloat16)


def test_malformed_cu_seqlens_reported():
    dev = torch.device("cuda", 0)
    q = torch.randn(300, 2, 64, device=dev, dtype=torch.bfloat16)
    for bad in ([0, 200, 100, 300], [5, 100, 300], [0, 100, 301]):
        cu = torch.tensor(bad, dtype=torch.int32, device=dev)
        attn.attn_fwd(q, q, q, cu_seqlens=cu)
        assert attn.get_error() == attn.ATTN_EDEVICE
        assert attn.last_device_error() == attn.ATTN_DEVERR_BAD_SEQLENS
    assert attn.get_error() == attn.ATTN_OK


def test_forward_is_bitwise_reproducible():
    """The schedule is fixed per problem shape and split pieces merge in a
    fixed order, so repeated calls give identical bits (split-KV headline
    shape scaled down, GQA, causal)."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(31)
    q = torch.randn(1, 3000, 8, 128, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(1, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(1, 3000, 2, 128, generator=g).to(torch.bfloat16).to(dev)
    o1, l1 = attn.attn_fwd(q, k, v, causal=True)
    o2, l2 = attn.attn_fwd(q, k, v, causal=True)
    assert attn.get_error() == attn.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_output_alignment_16_and_32_bytes_agree(d):
    """The epilogue stores whole 32-byte pieces where the output pointer is
    32-byte aligned and 16-byte pieces otherwise; both give the same bits,
    and both match the oracle (dense and packed varlen)."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(40 + d)
    q = torch.randn(1, 300, 4, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 300, 2, d, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 300, 2, d, generator=g).to(torch.bfloat16)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = attn.attn_fwd(qd, kd, vd, causal=True)
    buf = torch.zeros(o1.numel() + 8, dtype=o1.dtype, device=dev)   # 8 elements = 16 bytes off
    o2 = buf[8:].view_as(o1)
    assert o2.data_ptr() % 32 == 16
    l2 = torch.empty_like(l1)
    attn.attn_fwd(qd, kd, vd, causal=True, out=o2, lse=l2)
    assert attn.get_error() == attn.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, scale=d ** -0.5)
    assert np.max(np.abs(o1.float().cpu().double().numpy() - o_ref)) <= O_TOL
    # packed varlen, two sequences
    cu = torch.tensor([0, 130, 300], dtype=torch.int32, device=dev)
    o3, l3 = attn.attn_fwd(qd[0], kd[0], vd[0], causal=True, cu_seqlens=cu)
    buf = torch.zeros(o3.numel() + 8, dtype=o3.dtype, device=dev)
    o4 = buf[8:].view_as(o3)
    l4 = torch.empty_like(l3)
    attn.attn_fwd(qd[0], kd[0], vd[0], causal=True, cu_seqlens=cu, out=o4, lse=l4)
    assert attn.get_error() == attn.ATTN_OK
    assert torch.equal(o3, o4) and torch.equal(l3, l4)
