"""The boundary's stream and memory behaviour on a GPU, through the C ABI.

attn_fwd allocates nothing per call beyond its cached schedules and
workspaces, and never synchronises: the first call of a problem shape writes
its schedule with a kernel on the call's stream.  Such a first call can
therefore be captured into a CUDA graph, and the graph replayed on new
values of the same buffers.  The schedule cache is bounded: after more
shapes than it holds, the evicted schedules' device copies are released and
device memory stays flat.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_attn_gb300 import attn
from tiled_attention_attn_gb300.inputs import Workload, generate, sample_rows

from .test_parity_gpu import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(attn_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.set_wait_timeout_ns(2_000_000_000)
    return attn_lib


# first-of-shape calls: a schedule too large for the launch parameters
# (576 units), and a split schedule (its workspace is grown during capture)
CAPTURE_SHAPES = [(4, 16, 8, 2304, 2304, 64, True), (1, 1, 1, 7936, 7936, 128, True)]


@pytest.mark.parametrize("shape", CAPTURE_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_first_call_of_a_shape_inside_graph_capture(shape):
    B, Hq, Hkv, L, _, d, causal = shape
    dev = torch.device("cuda", 0)
    wl = Workload("cap", B=B, Hq=Hq, Hkv=Hkv, Lq=L, Lk=L, d=d, dtype="bf16", causal=causal, seed=23)
    inp = generate(wl)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, L, dtype=torch.float32, device=dev)
    before, _ = attn.cache_stats()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.attn_fwd(q, k, v, causal=causal, scale=wl.softmax_scale, out=o, lse=lse)
    plans, pinned = attn.cache_stats()
    assert pinned >= 1 and plans >= before
    for rep in range(2):
        if rep == 1:
            # new values in the captured buffers
            inp2 = generate(wl, seed=24)
            q.copy_(inp2.q.to(dev))
            k.copy_(inp2.k.to(dev))
            v.copy_(inp2.v.to(dev))
            inp = inp2
        g.replay()
        torch.cuda.synchronize(dev)
        assert attn.get_error() == attn.ATTN_OK
        rows = sample_rows(wl, 96)
        o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rows, causal=causal, scale=wl.softmax_scale)
        idx = np.array(rows)
        on = o.float().cpu().double().numpy()
        ln = lse.cpu().double().numpy()
        check(on[idx[:, 0], idx[:, 2], idx[:, 1]], ln[idx[:, 0], idx[:, 1], idx[:, 2]], o_ref, lse_ref,
              f"graph replay {rep}")
    # an eager call of the same shape after the capture agrees with the replay
    o2, lse2 = attn.attn_fwd(q, k, v, causal=causal, scale=wl.softmax_scale)
    assert attn.get_error() == attn.ATTN_OK
    assert torch.equal(o2, o) and torch.equal(lse2, lse)


def test_schedule_cache_is_bounded_and_releases_memory():
    """300 dense shapes whose schedules need device copies (256 heads x one
    256-row block each): the cache keeps at most 256 per kernel, and device
    memory after the evictions stays within a small margin of where it began."""
    dev = torch.device("cuda", 0)
    Hq, d = 256, 64
    q = torch.randn(1, 320, Hq, d, device=dev, dtype=torch.bfloat16)
    # warm-up: kernels loaded, pools created
    q1 = q[:, :1].contiguous()
    attn.attn_fwd(q1, q1, q1)
    torch.cuda.synchronize(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    for L in range(2, 302):
        qs = q[:, :L].contiguous()
        attn.attn_fwd(qs, qs, qs, out=torch.empty_like(qs), lse=torch.empty(1, Hq, L, dtype=torch.float32, device=dev))
    torch.cuda.synchronize(dev)
    assert attn.get_error() == attn.ATTN_OK
    plans, pinned = attn.cache_stats()
    assert plans - pinned <= 2 * 256
    torch.cuda.empty_cache()
    torch.cuda.synchronize(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free0 - free1 < 64 * 1024 * 1024
