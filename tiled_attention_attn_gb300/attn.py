"""ctypes binding of libattn.so (include/attn.h), argument marshalling only.

Every step of the forward pass runs in the library's CUDA kernels; this module
checks tensor shapes, allocates outputs with torch, passes raw device pointers
and the current stream, and turns return codes into exceptions.  There is no
other implementation behind it: if the library is missing, calls fail.
"""

from __future__ import annotations

import ctypes
import math
import os
import re
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

ATTN_OK = 0
ATTN_EINVAL = -1
ATTN_EUNSUPPORTED = -2
ATTN_ELAUNCH = -3
ATTN_ENOMEM = -4
ATTN_EDEVICE = -5
ATTN_ETOOLARGE = -6
ATTN_DEVERR_WAIT_TIMEOUT = 0x100
ATTN_DEVERR_BAD_SEQLENS = 0x200

HEADER = os.path.join(_build.ROOT, "include", "attn.h")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code) if _lib is not None else code} (code {code})")
        self.code = code


def declared_functions() -> list:
    """Names of the functions include/attn.h declares."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(attn_\w+)\s*\(", text)


def lib(path: Optional[str] = None):
    """Load libattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("TILED_ATTN_LIB") or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with tiled_attention_attn_gb300.build.build()")
        L = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp]
        for name in ("attn_fwd", "attn_fwd_fp16", "attn_fwd_noalloc"):
            fn = getattr(L, name)
            fn.argtypes = fwd_args
            fn.restype = i
        L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp, i, vp]
        L.attn_fwd_varlen.restype = i
        L.attn_get_error.argtypes = [vp]
        L.attn_get_error.restype = i
        L.attn_last_device_error.argtypes = []
        L.attn_last_device_error.restype = i
        L.attn_strerror.argtypes = [i]
        L.attn_strerror.restype = ctypes.c_char_p
        L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        L.attn_set_wait_timeout_ns.restype = None
        L.attn_selftest_wait_timeout.argtypes = [vp]
        L.attn_selftest_wait_timeout.restype = i
        L.attn_launch_count.argtypes = []
        L.attn_launch_count.restype = ctypes.c_ulonglong
        L.attn_profile_enable.argtypes = [i]
        L.attn_profile_enable.restype = i
        L.attn_profile_disable.argtypes = []
        L.attn_profile_disable.restype = None
        fp = ctypes.POINTER(ctypes.c_float)
        L.attn_profile_read.argtypes = [fp, fp, i, ctypes.POINTER(ctypes.c_int)]
        L.attn_profile_read.restype = i
        L.attn_trace_enable.argtypes = [vp, i]
        L.attn_trace_enable.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        L.attn_plan.argtypes = [i, i, i, i, i, i, i, i, ip, i, ip, ip, ip]
        L.attn_plan.restype = i
        L.attn_rotary.argtypes = [vp, vp, i, i, i, i, i, f, i, vp, i, vp, i, vp]
        L.attn_rotary.restype = i
        L.attn_unpad_index.argtypes = [vp, i, i, vp, vp, vp]
        L.attn_unpad_index.restype = i
        L.attn_gather_rows.argtypes = [vp, i, vp, i, vp, i, vp, vp]
        L.attn_gather_rows.restype = i
        L.attn_scatter_rows.argtypes = [vp, vp, i, vp, i, vp, i, vp]
        L.attn_scatter_rows.restype = i
        L.attn_scatter_lse.argtypes = [vp, vp, i, vp, i, i, i, vp, vp]
        L.attn_scatter_lse.restype = i
        L.attn_rotary_packed.argtypes = [vp, vp, i, i, i, i, i, i, f, i, vp, i, vp, i, vp]
        L.attn_rotary_packed.restype = i
        L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
        L.attn_bwd.restype = i
        L.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp, i, vp]
        L.attn_bwd_varlen.restype = i
        L.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, i, vp]
        L.attn_decode.restype = i
        L.attn_set_pair_forward.argtypes = [i]
        L.attn_set_pair_forward.restype = None
        L.attn_set_cluster_merge.argtypes = [i]
        L.attn_set_cluster_merge.restype = None
        L.attn_cluster_merge.argtypes = []
        L.attn_cluster_merge.restype = i
        L.attn_fwd_rope.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, f, i, i, i, vp]
        L.attn_fwd_rope.restype = i
        L.attn_set_decode_path.argtypes = [i]
        L.attn_set_decode_path.restype = None
        L.attn_decode_path.argtypes = []
        L.attn_decode_path.restype = i
        L.attn_pair_forward_used.argtypes = [i, i]
        L.attn_pair_forward_used.restype = i
        L.attn_plan_pair.argtypes = [i, i, i, i, i, i, i, ip, i, ip, ip, ip]
        L.attn_plan_pair.restype = i
        L.attn_cache_stats.argtypes = [ip, ip]
        L.attn_cache_stats.restype = i
        L.attn_selftest_plan_cache.argtypes = [i, i, i, ip, ip]
        L.attn_selftest_plan_cache.restype = i
        if path is None:
            _lib = L
        return L


def strerror(code: int) -> str:
    return lib().attn_strerror(int(code)).decode()


def _stream_handle(device: torch.device, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: Optional[float] = None, cu_seqlens: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None,
             cu_seqlens_k: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O = softmax(scale * Q K^T [+ causal mask]) V and the row log-sum-exp.

    Dense: q (B, Lq, Hq, d), k and v (B, Lk, Hkv, d); returns O like q and
    lse (B, Hq, Lq) float32.  Varlen (``cu_seqlens`` given, int32 on the
    device, B+1 entries): q, k, v packed (total, H, d); lse is (Hq, total).
    With ``cu_seqlens_k`` as well, the keys have their own offsets (k, v
    packed as (total_k, Hkv, d)): cross-attention or a key/value cache, causal
    aligned bottom-right per sequence.  ``scale`` defaults to 1/sqrt(d).
    """
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q, k, v must be bfloat16 or float16")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k and v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k and v must be contiguous")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if cu_seqlens_k is not None and cu_seqlens is None:
        raise ValueError("cu_seqlens_k needs cu_seqlens")
    if cu_seqlens is not None:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("varlen q, k, v are (total, H, d)")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        if cu_seqlens_k is not None and (cu_seqlens_k.dtype != torch.int32 or not cu_seqlens_k.is_cuda
                                         or cu_seqlens_k.numel() != cu_seqlens.numel()):
            raise ValueError("cu_seqlens_k must be an int32 CUDA tensor with as many entries as cu_seqlens")
        B = cu_seqlens.numel() - 1
        Lq, Hq, _ = q.shape
        Lk, Hkv, _ = k.shape
        lse_shape = (Hq, Lq)
        cu_ptr = cu_seqlens.data_ptr()
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense q is (B, Lq, Hq, d) and k, v are (B, Lk, Hkv, d)")
        B, Lq, Hq, _ = q.shape
        _, Lk, Hkv, _ = k.shape
        lse_shape = (B, Hq, Lq)
        cu_ptr = None
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if tuple(lse.shape) != lse_shape or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous float32 tensor of shape {lse_shape}")
    L = lib()
    with torch.cuda.device(q.device):
        if cu_seqlens_k is not None:
            rc = L.attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   int(B), int(Hq), int(Hkv), int(Lq), int(Lk), int(d), int(bool(causal)),
                                   ctypes.c_float(float(scale)), cu_ptr, cu_seqlens_k.data_ptr(),
                                   int(q.dtype == torch.float16), _stream_handle(q.device, stream))
        else:
            fn = L.attn_fwd if q.dtype == torch.bfloat16 else L.attn_fwd_fp16
            rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    int(B), int(Hq), int(Hkv), int(Lq), int(Lk), int(d), int(bool(causal)),
                    ctypes.c_float(float(scale)), cu_ptr, _stream_handle(q.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_rope(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                  scale: Optional[float] = None, rot_dim: Optional[int] = None, base: float = 10000.0,
                  interleaved: bool = False, q_offset: int = 0, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """attn_fwd of rotary-embedded q and k (dense (B, L, H, d) layouts): query
    i at position q_offset + i, key j at position j, rotation as ``rotary``;
    the rotation of q happens inside the forward kernel.  q and k are not
    modified."""
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q, k, v must be bfloat16 or float16")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    for t in (q, k, v):
        _check_cuda(t)
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("dense q is (B, Lq, Hq, d) and k, v are (B, Lk, Hkv, d)")
    B, Lq, Hq, d = q.shape
    _, Lk, Hkv, _ = k.shape
    rot = d if rot_dim is None else int(rot_dim)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if tuple(lse.shape) != (B, Hq, Lq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous float32 tensor of shape {(B, Hq, Lq)}")
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), int(B),
                                 int(Hq), int(Hkv), int(Lq), int(Lk), int(d), int(bool(causal)),
                                 ctypes.c_float(float(scale)), rot, ctypes.c_float(float(base)),
                                 int(bool(interleaved)), int(q_offset), int(q.dtype == torch.float16),
                                 _stream_handle(q.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_rope")
    return out, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
             dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None, cu_seqlens: Optional[torch.Tensor] = None,
             cu_seqlens_k: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Gradients (dq, dk, dv) of sum(dout * O) for the forward.

    Dense: q, out, dout (B, Lq, Hq, d); k, v (B, Lk, Hkv, d); lse (B, Hq, Lq)
    float32, with out and lse as attn_fwd returned them for the same q, k, v,
    causal and scale.  Varlen (``cu_seqlens`` given, and ``cu_seqlens_k`` for
    separate key offsets): q, out, dout (total_q, Hq, d), k, v (total_k, Hkv,
    d), lse (Hq, total_q).  dq is shaped like q, dk and dv like k.
    """
    ts = (q, k, v, out, dout)
    if q.dtype not in (torch.bfloat16, torch.float16) or any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, out and dout must share one 16-bit dtype")
    if any(not t.is_cuda or not t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("tensors must be contiguous CUDA tensors")
    if cu_seqlens_k is not None and cu_seqlens is None:
        raise ValueError("cu_seqlens_k needs cu_seqlens")
    varlen = cu_seqlens is not None
    nd = 3 if varlen else 4
    if q.dim() != nd or k.dim() != nd or k.shape != v.shape or out.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q, out, dout are (B, Lq, Hq, d) and k, v are (B, Lk, Hkv, d); packed without B")
    if varlen:
        cu_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
        for c in (cu_seqlens, cu_k):
            if c.dtype != torch.int32 or not c.is_cuda or c.numel() != cu_seqlens.numel():
                raise ValueError("cu_seqlens (and cu_seqlens_k) must be int32 CUDA tensors of B+1 entries")
        B = cu_seqlens.numel() - 1
        Lq, Hq, d = q.shape
        Lk, Hkv, _ = k.shape
        lse_shape = (Hq, Lq)
    else:
        B, Lq, Hq, d = q.shape
        _, Lk, Hkv, _ = k.shape
        lse_shape = (B, Hq, Lq)
    if tuple(lse.shape) != lse_shape or lse.dtype != torch.float32:
        raise ValueError(f"lse must be a float32 tensor of shape {lse_shape}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for g, ref in ((dq, q), (dk, k), (dv, v)):
        if g.shape != ref.shape or g.dtype != ref.dtype or not g.is_contiguous() or not g.is_cuda:
            raise ValueError("dq, dk, dv must be contiguous CUDA tensors shaped like q, k, v")
    with torch.cuda.device(q.device):
        if varlen:
            rc = lib().attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), int(B), int(Hq),
                                       int(Hkv), int(Lq), int(Lk), int(d), int(bool(causal)),
                                       ctypes.c_float(float(scale)), cu_seqlens.data_ptr(), cu_k.data_ptr(),
                                       int(q.dtype == torch.float16), _stream_handle(q.device, stream))
        else:
            rc = lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), int(B), int(Hq),
                                int(Hkv), int(Lq), int(Lk), int(d), int(bool(causal)), ctypes.c_float(float(scale)),
                                int(q.dtype == torch.float16), _stream_handle(q.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_k: torch.Tensor,
                scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One decoding step: q (B, Hq, d) holds one new query per sequence, k
    and v (total_k, Hkv, d) the packed caches with offsets ``cu_seqlens_k``
    (int32 on the device, B+1 entries).  Returns O (B, Hq, d) and lse
    (Hq, B) float32, equal to attn_fwd with cu_seqlens = [0, 1, ..., B] and
    these key offsets.  Hq / Hkv must be 1, 2, 4 or 8."""
    if q.dtype not in (torch.bfloat16, torch.float16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one 16-bit dtype")
    if not (q.is_cuda and k.is_cuda and v.is_cuda) or not (q.is_contiguous() and k.is_contiguous()
                                                            and v.is_contiguous()):
        raise ValueError("q, k and v must be contiguous CUDA tensors")
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or k.shape[2] != q.shape[2]:
        raise ValueError("q is (B, Hq, d) and k, v are (total_k, Hkv, d)")
    B, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    if cu_seqlens_k.dtype != torch.int32 or not cu_seqlens_k.is_cuda or cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_k must be an int32 CUDA tensor of B+1 entries")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, B), dtype=torch.float32, device=q.device) if lse is None else lse
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if tuple(lse.shape) != (Hq, B) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous float32 tensor of shape {(Hq, B)}")
    with torch.cuda.device(q.device):
        rc = lib().attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), int(B),
                               int(Hq), int(Hkv), int(total_k), int(d), ctypes.c_float(float(scale)),
                               cu_seqlens_k.data_ptr(), int(q.dtype == torch.float16),
                               _stream_handle(q.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode")
    return out, lse


# ---------------------------------------------------------------------------
# padded batches around the varlen forward (include/attn.h, attn_unpad_index
# and the row gather / scatter kernels)
# ---------------------------------------------------------------------------

class _AttnFunction(torch.autograd.Function):
    """attn_fwd in the forward, attn_bwd in the backward (the lse the forward
    returns is what the backward recomputes the weights from)."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, cu_seqlens, cu_seqlens_k):
        o, lse = attn_fwd(q, k, v, causal=causal, scale=scale, cu_seqlens=cu_seqlens, cu_seqlens_k=cu_seqlens_k)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.cu, ctx.cu_k = causal, scale, cu_seqlens, cu_seqlens_k
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, o, lse, do.contiguous(), causal=ctx.causal, scale=ctx.scale,
                              cu_seqlens=ctx.cu, cu_seqlens_k=ctx.cu_k)
        return dq, dk, dv, None, None, None, None


def attn_func(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: Optional[float] = None, cu_seqlens: Optional[torch.Tensor] = None,
              cu_seqlens_k: Optional[torch.Tensor] = None, return_lse: bool = False):
    """Differentiable attention: O = softmax(scale Q K^T [+ causal]) V with
    gradients for q, k and v through attn_bwd.  Shapes and arguments as
    attn_fwd (dense or varlen); returns O, or (O, lse) with ``return_lse``
    (lse carries no gradient)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = _AttnFunction.apply(q, k, v, bool(causal), float(scale), cu_seqlens, cu_seqlens_k)
    return (o, lse) if return_lse else o


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def unpad_index(key_padding_mask: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """(cu_seqlens (B+1,), indices (B*L,)) int32 on the mask's device for a
    (B, L) key-padding mask (True / nonzero = keep); indices[cu[B]:] are
    unspecified.  No host synchronisation."""
    if key_padding_mask.dim() != 2:
        raise ValueError("key_padding_mask is (B, L)")
    m = key_padding_mask.contiguous()
    if m.dtype == torch.bool:
        m = m.view(torch.uint8)
    if m.dtype != torch.uint8:
        raise TypeError("key_padding_mask must be bool or uint8")
    _check_cuda(m)
    B, L = m.shape
    cu = torch.empty(B + 1, dtype=torch.int32, device=m.device)
    idx = torch.empty(B * L, dtype=torch.int32, device=m.device)
    with torch.cuda.device(m.device):
        rc = lib().attn_unpad_index(m.data_ptr(), int(B), int(L), cu.data_ptr(), idx.data_ptr(),
                                    _stream_handle(m.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_unpad_index")
    return cu, idx


def gather_rows(src: torch.Tensor, indices: torch.Tensor, n_dev: torch.Tensor, n_max: int,
                out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[r] = src[indices[r]] for r < min(n_max, n_dev[0]) along the first axis."""
    _check_cuda(src, indices, n_dev)
    if out is None:
        out = torch.empty((n_max,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    _check_cuda(out)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 0
    with torch.cuda.device(src.device):
        rc = lib().attn_gather_rows(src.data_ptr(), int(src.shape[0]), indices.data_ptr(), int(n_max),
                                    n_dev.data_ptr(), int(row_bytes), out.data_ptr(),
                                    _stream_handle(src.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_gather_rows")
    return out


def scatter_rows(src: torch.Tensor, indices: torch.Tensor, n_dev: torch.Tensor, out: torch.Tensor,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[indices[r]] = src[r] for r < min(src rows, n_dev[0]); other rows of out untouched."""
    _check_cuda(src, indices, n_dev, out)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 0
    with torch.cuda.device(src.device):
        rc = lib().attn_scatter_rows(src.data_ptr(), indices.data_ptr(), int(src.shape[0]), n_dev.data_ptr(),
                                     int(row_bytes), out.data_ptr(), int(out.shape[0]),
                                     _stream_handle(src.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_scatter_rows")
    return out


def scatter_lse(src: torch.Tensor, indices: torch.Tensor, n_dev: torch.Tensor, out: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Varlen lse (Hq, n_max) into the padded out (B, Hq, L); other entries untouched."""
    _check_cuda(src, indices, n_dev, out)
    Hq, n_max = src.shape
    B, _, L = out.shape
    with torch.cuda.device(src.device):
        rc = lib().attn_scatter_lse(src.data_ptr(), indices.data_ptr(), int(n_max), n_dev.data_ptr(), int(Hq),
                                    int(B), int(L), out.data_ptr(), _stream_handle(src.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_scatter_lse")
    return out


def attn_fwd_padded(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, key_padding_mask: torch.Tensor,
                    causal: bool = False, scale: Optional[float] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Self-attention of a padded batch (B, L, H, d) with its key-padding mask
    (B, L), True = keep: the kept tokens are gathered into the packed layout,
    the varlen forward runs on them, and O (zero at padded positions) and lse
    (B, Hq, L; -inf at padded positions) are scattered back.  The packed
    buffers are sized B*L rows, so no step waits for the host."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, L, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be (B, L, Hkv, d) like q")
    if tuple(key_padding_mask.shape) != (B, L):
        raise ValueError("key_padding_mask must be (B, L)")
    cu, idx = unpad_index(key_padding_mask, stream)
    n_dev = cu[B:]
    N = B * L
    qp = gather_rows(q.view(N, Hq, d), idx, n_dev, N, stream=stream)
    kp = gather_rows(k.view(N, Hkv, d), idx, n_dev, N, stream=stream)
    vp = gather_rows(v.view(N, Hkv, d), idx, n_dev, N, stream=stream)
    op, lsep = attn_fwd(qp, kp, vp, causal=causal, scale=scale, cu_seqlens=cu, stream=stream)
    o = torch.zeros_like(q)
    scatter_rows(op, idx, n_dev, o.view(N, Hq, d), stream=stream)
    lse = torch.full((B, Hq, L), float("-inf"), dtype=torch.float32, device=q.device)
    scatter_lse(lsep, idx, n_dev, lse, stream=stream)
    return o, lse


class _PaddedAttnFunction(torch.autograd.Function):
    """The padded module's path with gradients (training page §2.5): gather
    the kept tokens, the varlen forward, scatter O back; the backward
    gathers dO, runs the varlen backward and scatters dq, dk, dv (zero at
    padded positions)."""

    @staticmethod
    def forward(ctx, q, k, v, key_padding_mask, causal, scale):
        B, L, Hq, d = q.shape
        Hkv = k.shape[2]
        cu, idx = unpad_index(key_padding_mask)
        n_dev = cu[B:]
        N = B * L
        qp = gather_rows(q.view(N, Hq, d), idx, n_dev, N)
        kp = gather_rows(k.view(N, Hkv, d), idx, n_dev, N)
        vp = gather_rows(v.view(N, Hkv, d), idx, n_dev, N)
        op, lsep = attn_fwd(qp, kp, vp, causal=causal, scale=scale, cu_seqlens=cu)
        o = torch.zeros_like(q)
        scatter_rows(op, idx, n_dev, o.view(N, Hq, d))
        lse = torch.full((B, Hq, L), float("-inf"), dtype=torch.float32, device=q.device)
        scatter_lse(lsep, idx, n_dev, lse)
        ctx.save_for_backward(qp, kp, vp, op, lsep, cu, idx)
        ctx.causal, ctx.scale, ctx.shape = causal, scale, (B, L, Hq, Hkv, d)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        qp, kp, vp, op, lsep, cu, idx = ctx.saved_tensors
        B, L, Hq, Hkv, d = ctx.shape
        N, n_dev = B * L, cu[B:]
        dop = gather_rows(do.contiguous().view(N, Hq, d), idx, n_dev, N)
        dqp, dkp, dvp = attn_bwd(qp, kp, vp, op, lsep, dop, causal=ctx.causal, scale=ctx.scale, cu_seqlens=cu)
        grads = []
        for gp, H in ((dqp, Hq), (dkp, Hkv), (dvp, Hkv)):
            g = torch.zeros((B, L, H, d), dtype=gp.dtype, device=gp.device)
            scatter_rows(gp, idx, n_dev, g.view(N, H, d))
            grads.append(g)
        return grads[0], grads[1], grads[2], None, None, None


def attn_func_padded(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, key_padding_mask: torch.Tensor,
                     causal: bool = False, scale: Optional[float] = None, return_lse: bool = False):
    """attn_fwd_padded with gradients for q, k and v: q (B, L, Hq, d), k, v
    (B, L, Hkv, d), key_padding_mask (B, L) with True = keep.  Padded
    positions get O = 0 and no gradient."""
    B, L, Hq, d = q.shape
    if k.shape != (B, L, k.shape[2], d) or v.shape != k.shape or tuple(key_padding_mask.shape) != (B, L):
        raise ValueError("q (B, L, Hq, d), k and v (B, L, Hkv, d), key_padding_mask (B, L)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o, lse = _PaddedAttnFunction.apply(q, k, v, key_padding_mask, bool(causal), float(scale))
    return (o, lse) if return_lse else o


def rotary(x: torch.Tensor, rot_dim: Optional[int] = None, base: float = 10000.0, interleaved: bool = False,
           cu_seqlens: Optional[torch.Tensor] = None, offsets: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Rotary position embedding of x: (B, L, H, d), or packed (total, H, d)
    with ``cu_seqlens``.  Token i of sequence b is at position i + offsets[b]
    (``offsets``: int32 CUDA tensor of B, e.g. cache lengths).  ``out`` may be
    x itself (in place); default a new tensor."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("x must be bfloat16 or float16")
    _check_cuda(x)
    d = x.shape[-1]
    rot = d if rot_dim is None else int(rot_dim)
    if cu_seqlens is not None:
        if x.dim() != 3:
            raise ValueError("packed x is (total, H, d)")
        _check_cuda(cu_seqlens)
        B, L, H, total = cu_seqlens.numel() - 1, 0, x.shape[1], x.shape[0]
    else:
        if x.dim() != 4:
            raise ValueError("dense x is (B, L, H, d)")
        B, L, H = x.shape[0], x.shape[1], x.shape[2]
        total = 0
    if offsets is not None:
        _check_cuda(offsets)
        if offsets.dtype != torch.int32 or offsets.numel() != B:
            raise ValueError("offsets must be int32 with one entry per sequence")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("out must be shaped like x")
    _check_cuda(out)
    with torch.cuda.device(x.device):
        rc = lib().attn_rotary(x.data_ptr(), out.data_ptr(), int(B), int(L), int(H), int(d), rot,
                               ctypes.c_float(float(base)), int(bool(interleaved)),
                               cu_seqlens.data_ptr() if cu_seqlens is not None else None, int(total),
                               offsets.data_ptr() if offsets is not None else None,
                               int(x.dtype == torch.float16), _stream_handle(x.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_rotary")
    return out


def rotary_packed(x: torch.Tensor, rot_dim: Optional[int] = None, base: float = 10000.0, interleaved: bool = False,
                  cu_seqlens: Optional[torch.Tensor] = None, offsets: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Rotary embedding of a packed qkv (B, L, 3, H, d) (Q and K rotated) or
    kv (B, L, 2, H, d) (K rotated) tensor, V untouched; with ``cu_seqlens``
    the leading (B, L) is packed as (total,).  ``out`` may be x (in place, as
    the training page's module works); default a new tensor with V copied."""
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("x must be bfloat16 or float16")
    _check_cuda(x)
    lead = 1 if cu_seqlens is not None else 2
    if x.dim() != lead + 3 or x.shape[lead] not in (2, 3):
        raise ValueError("x is (B, L, 3, H, d) / (B, L, 2, H, d), or (total, 3 | 2, H, d) with cu_seqlens")
    parts, H, d = x.shape[lead], x.shape[lead + 1], x.shape[lead + 2]
    rot = d if rot_dim is None else int(rot_dim)
    if cu_seqlens is not None:
        _check_cuda(cu_seqlens)
        B, L, total = cu_seqlens.numel() - 1, 0, x.shape[0]
    else:
        B, L, total = x.shape[0], x.shape[1], 0
    if offsets is not None:
        _check_cuda(offsets)
        if offsets.dtype != torch.int32 or offsets.numel() != B:
            raise ValueError("offsets must be int32 with one entry per sequence")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("out must be shaped like x")
    _check_cuda(out)
    h_rot = (parts - 1) * H   # qkv: Q and K; kv: K
    with torch.cuda.device(x.device):
        rc = lib().attn_rotary_packed(x.data_ptr(), out.data_ptr(), int(B), int(L), int(parts * H), int(h_rot),
                                      int(d), rot, ctypes.c_float(float(base)), int(bool(interleaved)),
                                      cu_seqlens.data_ptr() if cu_seqlens is not None else None, int(total),
                                      offsets.data_ptr() if offsets is not None else None,
                                      int(x.dtype == torch.float16), _stream_handle(x.device, stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_rotary_packed")
    return out


def get_error(stream: Optional[torch.cuda.Stream] = None, device=None) -> int:
    """Synchronise the stream and return (and clear) the library's device error status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().attn_get_error(_stream_handle(dev, stream)))


def last_device_error() -> int:
    return int(lib().attn_last_device_error())


def set_wait_timeout_ns(ns: int) -> None:
    lib().attn_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(stream: Optional[torch.cuda.Stream] = None, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().attn_selftest_wait_timeout(_stream_handle(dev, stream)))


def plan(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, d: int, causal: bool, num_sms: int):
    """The persistent-kernel schedule for a dense problem (host only).

    Returns (units, n_ctas, n_partials) with units an (n, 8) int tensor of
    (b*Hq+h, m_block, kv_begin, kv_end, split, n_split, slot, cta)."""
    L = lib()
    n_units, n_ctas, n_part = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = L.attn_plan(B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), num_sms, None, 0,
                     ctypes.byref(n_units), ctypes.byref(n_ctas), ctypes.byref(n_part))
    if rc not in (ATTN_OK, ATTN_ENOMEM):
        raise AttnError(rc, "attn_plan")
    buf = (ctypes.c_int * (8 * max(n_units.value, 1)))()
    rc = L.attn_plan(B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), num_sms, buf, n_units.value,
                     ctypes.byref(n_units), ctypes.byref(n_ctas), ctypes.byref(n_part))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_plan")
    units = torch.tensor(list(buf)[: 8 * n_units.value], dtype=torch.int64).reshape(-1, 8)
    return units, n_ctas.value, n_part.value


def plan_pair(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, causal: bool, num_pairs: int):
    """The CTA-pair kernel's schedule for a dense problem (host only).

    Returns (units, n_pairs, n_partials); units is an (n, 8) int tensor of
    (b*Hq+h, 256-row block, kv_begin, kv_end, split, n_split, slot, pair)
    with [kv_begin, kv_end) counted in 256-key tiles."""
    L = lib()
    n_units, n_pairs, n_part = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = L.attn_plan_pair(B, Hq, Hkv, Lq, Lk, int(bool(causal)), num_pairs, None, 0,
                          ctypes.byref(n_units), ctypes.byref(n_pairs), ctypes.byref(n_part))
    if rc not in (ATTN_OK, ATTN_ENOMEM):
        raise AttnError(rc, "attn_plan_pair")
    buf = (ctypes.c_int * (8 * max(n_units.value, 1)))()
    rc = L.attn_plan_pair(B, Hq, Hkv, Lq, Lk, int(bool(causal)), num_pairs, buf, n_units.value,
                          ctypes.byref(n_units), ctypes.byref(n_pairs), ctypes.byref(n_part))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_plan_pair")
    units = torch.tensor(list(buf)[: 8 * n_units.value], dtype=torch.int64).reshape(-1, 8)
    return units, n_pairs.value, n_part.value


def set_pair_forward(enable: bool) -> None:
    """Dense head_dim-128 forwards on CTA pairs (True) or on the single-CTA
    kernel (False, the default)."""
    lib().attn_set_pair_forward(int(bool(enable)))


def set_cluster_merge(cluster_size: int) -> None:
    """attn_set_cluster_merge: 0 merges split key ranges in a combine pass,
    2, 4 or 8 splits every query block into that many pieces that run as one
    cluster and merge over distributed shared memory."""
    lib().attn_set_cluster_merge(int(cluster_size))


def cluster_merge() -> int:
    """attn_cluster_merge: the current setting."""
    return int(lib().attn_cluster_merge())


def pair_forward_used(d: int, varlen: bool) -> bool:
    """Whether attn_fwd runs such a problem on the CTA-pair kernel."""
    return bool(lib().attn_pair_forward_used(int(d), int(bool(varlen))))


def set_decode_path(tensor_cores: bool) -> None:
    """attn_decode on the packed forward's tensor-core tiles (True, the
    default) or on the CUDA-core chunk kernels (False)."""
    lib().attn_set_decode_path(int(bool(tensor_cores)))


def decode_path() -> bool:
    """True when attn_decode takes the tensor-core route."""
    return bool(lib().attn_decode_path())


def fwd_splits(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, d: int, causal: bool, num_sms: int) -> bool:
    """Whether the schedule attn_fwd uses for this dense shape splits key ranges."""
    if pair_forward_used(d, False):
        return plan_pair(B, Hq, Hkv, Lq, Lk, causal, num_sms // 2)[2] > 0
    return plan(B, Hq, Hkv, Lq, Lk, d, causal, num_sms)[2] > 0


def cache_stats() -> Tuple[int, int]:
    """(cached schedules, of which pinned by a stream capture) on the current device."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().attn_cache_stats(ctypes.byref(a), ctypes.byref(b))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_cache_stats")
    return a.value, b.value


def selftest_plan_cache(n_keys: int, capacity: int, pin_every: int = 0) -> Tuple[int, int]:
    """Runs the schedule cache's eviction policy on host-side entries:
    (largest number of live entries, entries released)."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().attn_selftest_plan_cache(int(n_keys), int(capacity), int(pin_every), ctypes.byref(a), ctypes.byref(b))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_selftest_plan_cache")
    return a.value, b.value


def launch_count() -> int:
    """Kernels this library has launched in this process."""
    return int(lib().attn_launch_count())


def profile_enable(n: int) -> None:
    rc = lib().attn_profile_enable(int(n))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_profile_enable")


def profile_disable() -> None:
    lib().attn_profile_disable()


def profile_read(max_calls: int):
    """(main-kernel ms, whole-call ms) of the profiled calls, as two lists."""
    main = (ctypes.c_float * max(max_calls, 1))()
    call = (ctypes.c_float * max(max_calls, 1))()
    n = ctypes.c_int(0)
    rc = lib().attn_profile_read(main, call, int(max_calls), ctypes.byref(n))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_profile_read")
    k = min(n.value, max_calls)
    return list(main)[:k], list(call)[:k]


def trace_enable(buf: Optional[torch.Tensor], events_per_stream: int = 0) -> None:
    """Record the forward kernel's phase trace into ``buf`` (a CUDA tensor of at
    least n_sms * 4 * events_per_stream * 16 bytes); ``None`` turns it off.
    Needs the traced build (libattn_trace.so, selected with TILED_ATTN_LIB)."""
    if buf is None:
        rc = lib().attn_trace_enable(None, 0)
    else:
        rc = lib().attn_trace_enable(buf.data_ptr(), int(events_per_stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_trace_enable")
