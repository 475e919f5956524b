"""Parity of attn_decode (one new query per sequence against a packed
key/value cache) with the oracle's per-sequence dense attention, every
element compared, and with attn_fwd_varlen on the same inputs, on both of
its routes: the transposed tensor-core decode kernel (caches cut into
pieces of key tiles whose partials a second launch merges; at head_dim 64
steps of two key tiles, and the packed forward's decode mode above 3143
sequences) and the CUDA-core chunk kernels.  Bar: max |O - O_ref| <= 1e-2, max |lse - lse_ref|
<= 1e-3; a sequence with no key gives O = 0 and lse = -inf on both sides."""

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


@pytest.fixture(params=[True, False], ids=["tensor_cores", "cuda_cores"], autouse=True)
def path(request):
    attn.set_decode_path(request.param)
    assert attn.decode_path() == request.param
    yield request.param
    attn.set_decode_path(True)


def cu_of(lengths):
    return torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int32)


def make(lk, Hq, Hkv, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(len(lk), Hq, d, generator=g).to(dtype)
    k = torch.randn(sum(lk), Hkv, d, generator=g).to(dtype)
    v = torch.randn(sum(lk), Hkv, d, generator=g).to(dtype)
    return q, k, v


def check(o, lse, o_ref, lse_ref):
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), inf)
    assert np.all(np.isfinite(o))
    assert float(np.abs(o - o_ref).max()) <= O_TOL
    if (~inf).any():
        assert float(np.abs(lse[~inf] - lse_ref[~inf]).max()) <= LSE_TOL
    assert np.all(o[inf.T] == 0.0)


CASES = [
    # cache lengths, Hq, Hkv, d, dtype
    ([4097, 4097, 4097], 32, 8, 128, torch.bfloat16),            # the decode shape, fewer sequences
    ([0, 1, 255, 256, 257, 1000], 8, 2, 128, torch.bfloat16),   # chunk edges and an empty sequence
    ([5, 700, 0, 3000], 8, 8, 64, torch.float16),               # one query head per key/value head
    ([300, 513, 1], 4, 2, 64, torch.bfloat16),                  # group 2
    ([2000, 17], 16, 2, 128, torch.float16),                    # group 8
    ([20000, 3], 8, 2, 128, torch.bfloat16),                    # a long cache: 157 chunks to merge
    ([131072], 32, 8, 128, torch.bfloat16),                     # one sequence, the long decode shape
    ([5000, 1, 0, 12345, 777, 128, 129], 8, 2, 64, torch.bfloat16),   # pieces, tile edges, an empty cache
    ([640] * 40, 32, 4, 128, torch.float16),                    # group 8 over many sequences
    # head_dim 64: steps of two key tiles, a last step of one tile (128, 257),
    # pieces of whole steps merged
    ([128, 257, 256, 1, 384], 16, 4, 64, torch.bfloat16),
    ([20000, 3], 8, 2, 64, torch.float16),
    ([131072], 32, 8, 64, torch.bfloat16),                      # the long decode shape at d 64
    ([640] * 40, 32, 4, 64, torch.float16),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_decode_matches_oracle(case):
    lk, Hq, Hkv, d, dtype = case
    q, k, v = make(lk, Hq, Hkv, d, dtype, seed=sum(lk) + Hq)
    dev = torch.device("cuda", 0)
    scale = d ** -0.5
    o, lse = attn.attn_decode(q.to(dev), k.to(dev), v.to(dev), cu_of(lk).to(dev), scale=scale)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.varlen_cross_attention(q, k, v, [1] * len(lk), lk, causal=False, scale=scale)
    check(o, lse, o_ref, lse_ref)


def test_decode_agrees_with_the_packed_forward():
    lk = [4097, 33, 0, 1500]
    Hq, Hkv, d = 16, 4, 128
    q, k, v = make(lk, Hq, Hkv, d, torch.bfloat16, seed=5)
    dev = torch.device("cuda", 0)
    qd, kd, vd, cu_k = q.to(dev), k.to(dev), v.to(dev), cu_of(lk).to(dev)
    o1, l1 = attn.attn_decode(qd, kd, vd, cu_k)
    cu_q = torch.arange(len(lk) + 1, dtype=torch.int32, device=dev)
    o2, l2 = attn.attn_fwd(qd, kd, vd, causal=True, cu_seqlens=cu_q, cu_seqlens_k=cu_k)
    assert attn.get_error() == attn.ATTN_OK
    assert float((o1.float() - o2.float()).abs().max()) <= 2 * O_TOL
    fin = torch.isfinite(l2)
    assert torch.equal(torch.isfinite(l1), fin)
    assert float((l1[fin] - l2[fin]).abs().max()) <= 2 * LSE_TOL


def test_decode_no_keys_at_all():
    dev = torch.device("cuda", 0)
    q = torch.randn(3, 4, 64, device=dev, dtype=torch.bfloat16)
    k = torch.empty(0, 2, 64, device=dev, dtype=torch.bfloat16)
    o, lse = attn.attn_decode(q, k, k, torch.zeros(4, dtype=torch.int32, device=dev))
    assert attn.get_error() == attn.ATTN_OK
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_every_cache_empty_with_keys_present(d):
    # valid offsets that give every sequence zero keys while k and v hold rows
    dev = torch.device("cuda", 0)
    q = torch.randn(3, 8, d, device=dev, dtype=torch.bfloat16)
    k = torch.randn(300, 2, d, device=dev, dtype=torch.bfloat16)
    o, lse = attn.attn_decode(q, k, k, torch.zeros(4, dtype=torch.int32, device=dev))
    assert attn.get_error() == attn.ATTN_OK
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_malformed_offsets_reported():
    dev = torch.device("cuda", 0)
    q = torch.randn(3, 4, 64, device=dev, dtype=torch.bfloat16)
    k = torch.randn(300, 2, 64, device=dev, dtype=torch.bfloat16)
    for bad in ([0, 200, 100, 300], [5, 100, 200, 300], [0, 100, 200, 301]):
        o, lse = attn.attn_decode(q, k, k, torch.tensor(bad, dtype=torch.int32, device=dev))
        assert attn.get_error() == attn.ATTN_EDEVICE
        assert attn.last_device_error() == attn.ATTN_DEVERR_BAD_SEQLENS
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert attn.get_error() == attn.ATTN_OK


def test_decode_unsupported_group_raises():
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 6, 64, device=dev, dtype=torch.bfloat16)
    k = torch.randn(10, 2, 64, device=dev, dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError):
        attn.attn_decode(q, k, k, torch.tensor([0, 10], dtype=torch.int32, device=dev))


@pytest.mark.parametrize("B,d", [(4096, 128), (4096, 64), (3143, 64), (3144, 64)])
def test_decode_maximum_sequence_count(path, B, d):
    # up to 4096 sequences, one new query each, caches of 1 to 40 keys (fp16:
    # with so few keys per row O is not averaged down, and bf16's rounding of
    # P and O alone can pass 1e-2 where |O| approaches 4).  At head_dim 64 the
    # transposed kernel's prefix table holds 3143 sequences; more take the
    # packed forward's decode mode.
    rng = np.random.default_rng(7)
    lk = rng.integers(1, 41, B).tolist()
    q, k, v = make(lk, 8, 2, d, torch.float16, seed=7)
    dev = torch.device("cuda", 0)
    scale = d ** -0.5
    o, lse = attn.attn_decode(q.to(dev), k.to(dev), v.to(dev), cu_of(lk).to(dev), scale=scale)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.varlen_cross_attention(q, k, v, [1] * len(lk), lk, causal=False, scale=scale)
    check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_merge_of_more_than_32_pieces(d):
    # one key/value head with eight query heads: one (sequence, head group)
    # unit, so the cache is cut into as many pieces as there are SMs and the
    # merge takes them in chunks of 32
    lk = [65536]
    q, k, v = make(lk, 8, 1, d, torch.bfloat16, seed=31 + d)
    dev = torch.device("cuda", 0)
    scale = d ** -0.5
    o, lse = attn.attn_decode(q.to(dev), k.to(dev), v.to(dev), cu_of(lk).to(dev), scale=scale)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.varlen_cross_attention(q, k, v, [1], lk, causal=False, scale=scale)
    check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("vscale", [1e5, 1e-6])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_value_magnitude_through_pieces(d, vscale):
    # bf16 values scaled by 1e5 or 1e-6 on caches that are cut into pieces
    # (fp32 partials, then the merge): the result stays finite and as accurate
    # as unit-normal values, the bar scaled with the values plus half a bf16
    # ulp of O; lse does not depend on the values
    lk = [20000, 3, 9000]
    q, k, v = make(lk, 8, 2, d, torch.bfloat16, seed=41)
    g = torch.Generator().manual_seed(42)
    v = (torch.randn(v.shape, generator=g) * vscale).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    scale = d ** -0.5
    o, lse = attn.attn_decode(q.to(dev), k.to(dev), v.to(dev), cu_of(lk).to(dev), scale=scale)
    assert attn.get_error() == attn.ATTN_OK
    o_ref, lse_ref = oracle.varlen_cross_attention(q, k, v, [1] * len(lk), lk, causal=False, scale=scale)
    on = o.float().cpu().double().numpy()
    assert np.all(np.isfinite(on)) and np.all(np.isfinite(lse.cpu().numpy()))
    tol = 1e-2 * vscale + 2.0 ** -8 * np.abs(o_ref)
    assert np.all(np.abs(on - o_ref) <= tol)
    assert float(np.abs(lse.cpu().double().numpy() - lse_ref).max()) <= LSE_TOL
