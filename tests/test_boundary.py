"""The C ABI library loads, exports every symbol include/attn.h declares and
rejects bad arguments on the host, before anything reaches CUDA."""

import ctypes

import pytest

from tiled_attention_attn_gb300 import attn


def test_header_declares_the_entry_points():
    names = attn.declared_functions()
    for n in ("attn_fwd", "attn_fwd_fp16", "attn_get_error", "attn_strerror", "attn_plan",
              "attn_set_wait_timeout_ns", "attn_selftest_wait_timeout", "attn_last_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(attn_lib):
    for name in attn.declared_functions():
        assert hasattr(attn_lib, name), name


def test_strerror(attn_lib):
    assert attn.strerror(attn.ATTN_OK) == "ok"
    assert "invalid" in attn.strerror(attn.ATTN_EINVAL)
    assert "unsupported" in attn.strerror(attn.ATTN_EUNSUPPORTED)
    assert attn.strerror(12345) == "unknown error"


def _call(L, q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=1, Lq=8, Lk=8, d=64, causal=0,
          scale=0.125, cu=None, fn="attn_fwd"):
    f = getattr(L, fn)
    return f(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, d, causal, ctypes.c_float(scale), cu, None)


@pytest.mark.parametrize("fn", ["attn_fwd", "attn_fwd_fp16"])
@pytest.mark.parametrize("bad", [
    dict(q=None), dict(k=None), dict(v=None), dict(o=None), dict(lse=None),
    dict(q=8), dict(o=24), dict(lse=2),                      # misaligned pointers
    dict(B=0), dict(Hq=0), dict(Hkv=0), dict(Lq=-1), dict(Lk=-1),
    dict(Hq=3, Hkv=2),                                       # Hq % Hkv != 0
    dict(causal=2), dict(scale=float("nan")), dict(scale=float("inf")), dict(scale=-1.0),
    dict(cu=16, Lq=8, Lk=9),                                 # varlen is self-attention
    dict(cu=16, B=5000),                                     # too many sequences
    dict(B=1 << 20, Lq=1 << 12, Hq=1 << 10, Hkv=1 << 10),    # rows overflow 32-bit coordinates
])
def test_bad_arguments_rejected_on_host(attn_lib, fn, bad):
    assert _call(attn_lib, fn=fn, **bad) == attn.ATTN_EINVAL


@pytest.mark.parametrize("d", [32, 80, 96, 256])
def test_unsupported_head_dim(attn_lib, d):
    assert _call(attn_lib, d=d) == attn.ATTN_EUNSUPPORTED


def test_empty_query_is_a_no_op(attn_lib):
    # Lq = 0: nothing to compute, nothing enqueued, no CUDA call
    assert _call(attn_lib, Lq=0) == attn.ATTN_OK


def test_timeout_setter_accepts_values(attn_lib):
    attn.set_wait_timeout_ns(10)
    attn.set_wait_timeout_ns(2_000_000_000)


def _call_bwd(L, q=16, k=16, v=16, o=16, lse=16, dout=16, dq=16, dk=16, dv=16, B=1, Hq=2, Hkv=1, Lq=8, Lk=8,
              d=64, causal=0, scale=0.125, fp16=0):
    return L.attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Lq, Lk, d, causal, ctypes.c_float(scale),
                      fp16, None)


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(k=None), dict(v=None), dict(o=None), dict(lse=None), dict(dout=None),
    dict(dq=None), dict(dk=None), dict(dv=None), dict(q=None, Lk=0), dict(k=None, Lq=0),
    dict(q=8), dict(dout=24), dict(dk=40), dict(lse=2),       # misaligned pointers
    dict(B=0), dict(Hq=0), dict(Hkv=0), dict(Lq=-1), dict(Lk=-1),
    dict(Hq=3, Hkv=2), dict(causal=2), dict(fp16=2),
    dict(scale=float("nan")), dict(scale=-1.0),
    dict(B=1 << 20, Lq=1 << 12, Hq=1 << 10, Hkv=1 << 10),
])
def test_backward_bad_arguments_rejected_on_host(attn_lib, bad):
    assert _call_bwd(attn_lib, **bad) == attn.ATTN_EINVAL


def test_backward_empty_side_accepts_null_pointers(attn_lib):
    # Lq = 0 and Lk = 0 together: nothing to zero, no CUDA call
    assert _call_bwd(attn_lib, q=None, o=None, lse=None, dout=None, dq=None, k=None, v=None, dk=None, dv=None,
                     Lq=0, Lk=0) == attn.ATTN_OK


@pytest.mark.parametrize("d", [32, 96, 256])
def test_backward_unsupported_head_dim(attn_lib, d):
    assert _call_bwd(attn_lib, d=d) == attn.ATTN_EUNSUPPORTED


@pytest.mark.parametrize("bad", [dict(h_rot=0), dict(h_rot=4, h_total=3), dict(h_total=0), dict(rot=7),
                                 dict(x=None), dict(fp16=2)])
def test_rotary_packed_bad_arguments(attn_lib, bad):
    a = dict(x=16, y=16, B=1, L=4, h_total=3, h_rot=2, d=64, rot=64, fp16=0)
    a.update(bad)
    assert attn_lib.attn_rotary_packed(a["x"], a["y"], a["B"], a["L"], a["h_total"], a["h_rot"], a["d"], a["rot"],
                                       ctypes.c_float(10000.0), 0, None, 0, None, a["fp16"], None) == attn.ATTN_EINVAL


def test_backward_varlen_needs_both_offsets(attn_lib):
    args = [16] * 9 + [1, 2, 1, 8, 8, 64, 0, ctypes.c_float(0.125)]
    assert attn_lib.attn_bwd_varlen(*args, None, 16, 0, None) == attn.ATTN_EINVAL
    assert attn_lib.attn_bwd_varlen(*args, 16, None, 0, None) == attn.ATTN_EINVAL
    assert attn_lib.attn_bwd_varlen(*args, 16, 16, 2, None) == attn.ATTN_EINVAL


def test_missing_library_fails_loudly(tmp_path):
    # no CPU or library fallback: without the built library the binding raises
    with pytest.raises(RuntimeError, match="missing"):
        attn.lib(str(tmp_path / "libattn_absent.so"))


def _call_decode(L, q=16, k=16, v=16, o=16, lse=16, B=2, Hq=4, Hkv=2, total_k=8, d=64, scale=0.125, cu=16,
                 fp16=0):
    return L.attn_decode(q, k, v, o, lse, B, Hq, Hkv, total_k, d, ctypes.c_float(scale), cu, fp16, None)


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(o=None), dict(lse=None), dict(cu=None), dict(k=None), dict(v=None),
    dict(q=8), dict(k=24), dict(v=40), dict(o=40), dict(lse=2),      # misaligned pointers
    dict(B=0), dict(Hq=0), dict(Hkv=0), dict(total_k=-1), dict(Hq=3, Hkv=2), dict(fp16=2),
    dict(scale=float("nan")), dict(scale=-1.0),
    dict(B=1 << 22, Hq=1 << 10, Hkv=1 << 10),
])
def test_decode_bad_arguments_rejected_on_host(attn_lib, bad):
    assert _call_decode(attn_lib, **bad) == attn.ATTN_EINVAL


@pytest.mark.parametrize("shape", [dict(d=32), dict(d=96), dict(d=256), dict(Hq=6, Hkv=2), dict(Hq=16, Hkv=1)])
def test_decode_unsupported_shapes(attn_lib, shape):
    assert _call_decode(attn_lib, **shape) == attn.ATTN_EUNSUPPORTED


def test_schedule_cache_eviction_policy(attn_lib):
    """The schedule cache's policy on host-side entries: it never holds more
    unpinned entries than its capacity, evicts the excess, and keeps pinned
    (captured) entries."""
    live, released = attn.selftest_plan_cache(300, 256)
    assert live == 256 and released == 300 - 256
    live, released = attn.selftest_plan_cache(1000, 256, pin_every=10)
    assert live <= 256 + 1000 // 10
    assert released > 0
    live, released = attn.selftest_plan_cache(100, 256)
    assert live == 100 and released == 0
