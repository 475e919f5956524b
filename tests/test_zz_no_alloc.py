"""attn_fwd_noalloc, the allocation-free entry point.

Some callers cannot allocate device memory during a call: their memory is
owned by a pool or caching allocator that has already reserved it (a
surprise cudaMalloc may fail), or they cannot afford the device-wide
synchronisation that cudaFree implies.  For them attn_fwd_noalloc runs the
same kernels as attn_fwd with its scratch (schedule and split-KV partials) in
a static device array.  These tests call it through the C ABI and check it
against attn_fwd, on two calls in a row with different inputs (the array
keeps the previous call's contents), across a change of problem shape, and
that a problem too large for the array is refused without a launch.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import WORKLOADS, Workload, generate

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return attn_lib


def noalloc(q, k, v, causal, scale, cu=None):
    """Calls attn_fwd_noalloc through the C ABI; returns (O, lse, return code)."""
    L = attn.lib()
    o = torch.empty_like(q)
    if cu is None:
        B, Lq, Hq, d = q.shape
        _, Lk, Hkv, _ = k.shape
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    else:
        Lq, Hq, d = q.shape
        Lk, Hkv, _ = k.shape
        B = cu.numel() - 1
        lse = torch.empty((Hq, Lq), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = L.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, Hq, Hkv, Lq, Lk, d, int(causal), ctypes.c_float(scale),
                            cu.data_ptr() if cu is not None else None, stream)
    return o, lse, rc


def assert_close(o, lse, o_ref, lse_ref):
    assert torch.isfinite(o).all()
    assert float((o.float() - o_ref.float()).abs().max()) <= O_TOL
    inf = torch.isneginf(lse_ref)
    assert torch.equal(torch.isneginf(lse), inf)
    if (~inf).any():
        assert float((lse[~inf] - lse_ref[~inf]).abs().max()) <= LSE_TOL


def test_noalloc_matches_attn_fwd_two_calls_in_a_row():
    wl = WORKLOADS["single_head_l8192_d128_causal"]
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, n_part = attn.plan(wl.B, wl.Hq, wl.Hkv, wl.Lq, wl.Lk, wl.d, wl.causal, n_sms)
    assert n_part > 0, "this shape must use split-KV partials, i.e. the scratch array"
    dev = torch.device("cuda", 0)
    for seed in (21, 22):
        inp = generate(wl, seed=seed)
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=True, scale=wl.softmax_scale)
        o, lse, rc = noalloc(q, k, v, True, wl.softmax_scale)
        assert rc == attn.ATTN_OK
        assert attn.get_error() == attn.ATTN_OK
        assert_close(o, lse, o_ref, lse_ref)


def test_noalloc_shape_change_and_varlen():
    dev = torch.device("cuda", 0)
    for shape in [(2, 8, 2, 700, 700, 64, True), (1, 2, 2, 300, 900, 128, False), (2, 8, 2, 700, 700, 64, True)]:
        B, Hq, Hkv, Lq, Lk, d, causal = shape
        wl = Workload("na", B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=d, dtype="bf16", causal=causal, seed=4)
        inp = generate(wl)
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=causal)
        o, lse, rc = noalloc(q, k, v, causal, wl.softmax_scale)
        assert rc == attn.ATTN_OK
        assert attn.get_error() == attn.ATTN_OK
        assert_close(o, lse, o_ref, lse_ref)
    wl = WORKLOADS["varlen_b16_h12_d64"]
    inp = generate(wl)
    q, k, v, cu = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens.to(dev)
    o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=False, cu_seqlens=cu)
    o, lse, rc = noalloc(q, k, v, False, wl.softmax_scale, cu=cu)
    assert rc == attn.ATTN_OK and attn.get_error() == attn.ATTN_OK
    assert_close(o, lse, o_ref, lse_ref)


def test_noalloc_allocates_nothing():
    """A call with a shape the entry point has not seen before changes neither
    the device's free memory nor torch's allocation count.  A first call of
    another shape that runs the same kernels comes before the measurement,
    so that loading the library's kernels (which reserves memory for their
    code) is not counted."""
    dev = torch.device("cuda", 0)
    shapes = [(1, 1, 1, 8192, 8192), (1, 2, 1, 6144, 6144)]   # both split, schedules in the array
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    ins = []
    for (B, Hq, Hkv, Lq, Lk) in shapes:
        assert attn.plan(B, Hq, Hkv, Lq, Lk, 128, True, n_sms)[2] > 0
        wl = Workload("na0", B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, d=128, dtype="bf16", causal=True, seed=9)
        inp = generate(wl)
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev)
        ins.append((q, k, v, o, lse, wl))
    L = attn.lib()
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call(q, k, v, o, lse, wl):
        return L.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  wl.B, wl.Hq, wl.Hkv, wl.Lq, wl.Lk, wl.d, 1, ctypes.c_float(wl.softmax_scale),
                                  None, stream)

    assert call(*ins[0]) == attn.ATTN_OK
    torch.cuda.synchronize(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    assert call(*ins[1]) == attn.ATTN_OK
    torch.cuda.synchronize(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert free1 == free0
    assert attn.get_error() == attn.ATTN_OK
    q, k, v, o, lse, wl = ins[1]
    o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=True)
    assert_close(o, lse, o_ref, lse_ref)


def test_noalloc_varlen_grouped_heads():
    """Packed sequences with four query heads per key/value head: attn_fwd
    lets the group share a tile, the allocation-free entry point does not;
    both must give the same result."""
    dev = torch.device("cuda", 0)
    wl = Workload("na_gqa", B=6, Hq=8, Hkv=2, Lq=0, Lk=0, d=64, dtype="bf16", causal=True, seed=12, varlen=True,
                  len_lo=1, len_hi=700)
    inp = generate(wl)
    q, k, v, cu = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens.to(dev)
    for causal in (True, False):
        o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=causal, cu_seqlens=cu)
        o, lse, rc = noalloc(q, k, v, causal, wl.softmax_scale, cu=cu)
        assert rc == attn.ATTN_OK and attn.get_error() == attn.ATTN_OK
        assert_close(o, lse, o_ref, lse_ref)


def test_noalloc_refuses_problems_beyond_its_array():
    # 133120 one-block units (B 1040, 128 query heads on one KV head, L 256,
    # d 64): the schedule (32 bytes per unit) exceeds the array's 4 MiB
    # schedule region.  The tensors are allocated at full size (uninitialised)
    # so that even a launch by mistake would stay inside them.
    B, Hq, Hkv, L, d = 1040, 128, 1, 256, 64
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    units, _, _ = attn.plan(B, Hq, Hkv, L, L, d, False, n_sms)
    assert units.shape[0] * 8 * 4 > (4 << 20)
    dev = torch.device("cuda", 0)
    q = torch.empty(B, L, Hq, d, device=dev, dtype=torch.bfloat16)
    kv = torch.empty(B, L, Hkv, d, device=dev, dtype=torch.bfloat16)
    before = attn.launch_count()
    o, lse, rc = noalloc(q, kv, kv, False, d ** -0.5)
    assert rc == attn.ATTN_ETOOLARGE
    assert attn.launch_count() == before
    assert "static buffer" in attn.strerror(rc)
