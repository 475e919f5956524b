"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library's compute path never does, and nothing here
imports the library.

``oracle.c`` holds the arithmetic (see its header for the definition it
follows); this module compiles it with gcc, loads it with ctypes, widens the
rounded bf16/fp16 inputs to float64 exactly and marshals arrays.  It also
holds the oracle's own conversion of a packed variable-length batch into the
padded batch plus key_padding_mask that the pages' MHA module takes
(lei6393.com training-integration page, §2.5): the oracle evaluates the padded
form, an independent route to the packed result the CUDA path produces.  The
unpad / pad steps of that section (index of the kept tokens, row gather and
scatter) are written out here too, as plain definitions.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile ``src`` into the shared library ``out`` (gcc, OpenMP if present)."""
    if not force and out == LIB and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", out, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def _load(path: str = LIB):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    ip = ctypes.POINTER(ctypes.c_int)
    I, D = ctypes.c_int, ctypes.c_double
    lib.oracle_attention.argtypes = [dp, dp, dp, u8p, dp, dp, dp, I, I, I, I, I, I, I, D]
    lib.oracle_attention.restype = I
    lib.oracle_attention_rows.argtypes = [dp, dp, dp, u8p, ip, I, dp, dp, I, I, I, I, I, I, I, D]
    lib.oracle_attention_rows.restype = I
    lib.oracle_online_rows.argtypes = [dp, dp, dp, u8p, ip, I, dp, dp, I, I, I, I, I, I, I, D, I, I, dp]
    lib.oracle_online_rows.restype = I
    lib.oracle_attention_backward.argtypes = [dp, dp, dp, dp, u8p, dp, dp, dp, I, I, I, I, I, I, I, D]
    lib.oracle_attention_backward.restype = I
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    return lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _load()
    return _lib


def load_variant(path: str):
    """Load another build of the oracle source (used to plant mistakes)."""
    return _load(path)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# --------------------------------------------------------------------------
# marshalling
# --------------------------------------------------------------------------

def f64(x) -> np.ndarray:
    """Widen a tensor or array to a contiguous float64 numpy array.  bf16 and
    fp16 values are exactly representable in float64."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _u8(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc}")


def _dims(q: np.ndarray, k: np.ndarray):
    B, Lq, Hq, d = q.shape
    Bk, Lk, Hkv, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("q and k disagree on batch or head_dim")
    return B, Hq, Hkv, Lq, Lk, d


def attention(q, k, v, causal: bool = False, scale: Optional[float] = None,
              key_padding_mask=None, with_probs: bool = False, _lib=None):
    """O (B,Lq,Hq,d) and lse (B,Hq,Lq) in float64 (and P (B,Hq,Lq,Lk) if asked)."""
    L = _lib or lib()
    q, k, v = f64(q), f64(k), f64(v)
    B, Hq, Hkv, Lq, Lk, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kpm = None if key_padding_mask is None else np.ascontiguousarray(np.asarray(key_padding_mask, dtype=np.uint8))
    o = np.empty((B, Lq, Hq, d), np.float64)
    lse = np.empty((B, Hq, Lq), np.float64)
    p = np.empty((B, Hq, Lq, Lk), np.float64) if with_probs else None
    rc = L.oracle_attention(_dp(q), _dp(k), _dp(v), _u8(kpm), _dp(o), _dp(lse), _dp(p),
                            B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), float(scale))
    _check(rc, "oracle_attention")
    return (o, lse, p) if with_probs else (o, lse)


def attention_backward(q, k, v, dout, causal: bool = False, scale: Optional[float] = None,
                       key_padding_mask=None, _lib=None):
    """Gradients (dq, dk, dv) in float64 of sum(dout * O) for the attention
    above (training page §5.3 recomputes the weights in the backward; the
    formulas are the chain rule through the definition, see oracle.c).
    dout is shaped like q; dq like q, dk and dv like k."""
    L = _lib or lib()
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    B, Hq, Hkv, Lq, Lk, d = _dims(q, k)
    if dout.shape != q.shape or v.shape != k.shape:
        raise ValueError("dout must be shaped like q and v like k")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kpm = None if key_padding_mask is None else np.ascontiguousarray(np.asarray(key_padding_mask, dtype=np.uint8))
    dq = np.empty(q.shape, np.float64)
    dk = np.empty(k.shape, np.float64)
    dv = np.empty(k.shape, np.float64)
    rc = L.oracle_attention_backward(_dp(q), _dp(k), _dp(v), _dp(dout), _u8(kpm), _dp(dq), _dp(dk), _dp(dv),
                                     B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), float(scale))
    _check(rc, "oracle_attention_backward")
    return dq, dk, dv


def attention_rows(q, k, v, rows: Sequence[Tuple[int, int, int]], causal: bool = False,
                   scale: Optional[float] = None, key_padding_mask=None, _lib=None):
    """O and lse of the selected (b, h, i) rows only: (n, d) and (n,)."""
    L = _lib or lib()
    q, k, v = f64(q), f64(k), f64(v)
    B, Hq, Hkv, Lq, Lk, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kpm = None if key_padding_mask is None else np.ascontiguousarray(np.asarray(key_padding_mask, dtype=np.uint8))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = L.oracle_attention_rows(_dp(q), _dp(k), _dp(v), _u8(kpm),
                                 r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n,
                                 _dp(o), _dp(lse), B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), float(scale))
    _check(rc, "oracle_attention_rows")
    return o, lse


def online_rows(q, k, v, rows: Sequence[Tuple[int, int, int]], beta: int, form: int = 0,
                causal: bool = False, scale: Optional[float] = None, key_padding_mask=None,
                trace: bool = False, _lib=None):
    """The blocked online-softmax recurrence over key blocks of size ``beta``.

    form 0: (m, l, u, r) recurrence; form 1: normalised-o recurrence.  With
    ``trace`` it also returns the (m, l, u[0]) state after every block for the
    first row (o[0] in place of u[0] for form 1)."""
    L = _lib or lib()
    q, k, v = f64(q), f64(k), f64(v)
    B, Hq, Hkv, Lq, Lk, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kpm = None if key_padding_mask is None else np.ascontiguousarray(np.asarray(key_padding_mask, dtype=np.uint8))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    nblk = (Lk + beta - 1) // beta
    tr = np.full((max(nblk, 1), 3), np.nan, np.float64) if trace else None
    rc = L.oracle_online_rows(_dp(q), _dp(k), _dp(v), _u8(kpm),
                              r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n,
                              _dp(o), _dp(lse), B, Hq, Hkv, Lq, Lk, d, int(bool(causal)), float(scale),
                              int(beta), int(form), _dp(tr))
    _check(rc, "oracle_online_rows")
    return (o, lse, tr) if trace else (o, lse)


# --------------------------------------------------------------------------
# packed variable-length batches, evaluated through the padded form
# --------------------------------------------------------------------------

def pad_packed(packed, lengths: Sequence[int], max_len: Optional[int] = None):
    """Packed (total, H, d) -> padded (B, max_len, H, d) float64 plus the
    key_padding_mask (B, max_len) with True = keep and the padding at the end
    of each row (lei6393.com training page, §2.5)."""
    x = f64(packed)
    B = len(lengths)
    T = max_len if max_len is not None else (max(lengths) if B else 0)
    out = np.zeros((B, T) + x.shape[1:], np.float64)
    mask = np.zeros((B, T), np.uint8)
    off = 0
    for b, n in enumerate(lengths):
        out[b, :n] = x[off:off + n]
        mask[b, :n] = 1
        off += n
    return out, mask


def varlen_attention(q, k, v, lengths: Sequence[int], causal: bool = False,
                     scale: Optional[float] = None):
    """Packed varlen attention via the padded batch + key_padding_mask.

    Returns O packed as (total, Hq, d) and lse as (Hq, total)."""
    lengths = [int(n) for n in lengths]
    qp, mask = pad_packed(q, lengths)
    kp, _ = pad_packed(k, lengths)
    vp, _ = pad_packed(v, lengths)
    o, lse = attention(qp, kp, vp, causal=causal, scale=scale, key_padding_mask=mask)
    total = sum(lengths)
    Hq, d = o.shape[2], o.shape[3]
    o_packed = np.empty((total, Hq, d), np.float64)
    lse_packed = np.empty((Hq, total), np.float64)
    off = 0
    for b, n in enumerate(lengths):
        o_packed[off:off + n] = o[b, :n]
        lse_packed[:, off:off + n] = lse[b, :, :n]
        off += n
    return o_packed, lse_packed


def varlen_cross_attention(q, k, v, lengths_q: Sequence[int], lengths_k: Sequence[int], causal: bool = False,
                           scale: Optional[float] = None):
    """Packed varlen attention with separate query and key lengths
    (cross-attention, or queries extending a key/value cache: training page
    §2.4, §4), one dense call per sequence.  q packed (total_q, Hq, d); k, v
    packed (total_k, Hkv, d).  Causal aligns each sequence bottom-right (its
    queries are the last Lq_b of Lk_b positions).  Returns O (total_q, Hq, d)
    and lse (Hq, total_q); a query with no key gives O = 0, lse = -inf."""
    q, k, v = f64(q), f64(k), f64(v)
    Hq, d = q.shape[1], q.shape[2]
    o = np.zeros((q.shape[0], Hq, d), np.float64)
    lse = np.full((Hq, q.shape[0]), -np.inf, np.float64)
    oq = ok = 0
    for nq, nk in zip(lengths_q, lengths_k):
        nq, nk = int(nq), int(nk)
        if nq > 0 and nk > 0:
            ob, lb = attention(q[None, oq:oq + nq], k[None, ok:ok + nk], v[None, ok:ok + nk], causal=causal,
                               scale=scale)
            o[oq:oq + nq] = ob[0]
            lse[:, oq:oq + nq] = lb[0]
        oq += nq
        ok += nk
    return o, lse


def varlen_attention_backward(q, k, v, dout, lengths_q: Sequence[int], lengths_k: Sequence[int],
                              causal: bool = False, scale: Optional[float] = None):
    """Gradients of a packed batch with per-sequence query and key lengths, one
    dense backward per sequence (the same composition as
    varlen_cross_attention).  q, dout (total_q, Hq, d); k, v (total_k, Hkv, d).
    Returns dq (total_q, Hq, d), dk, dv (total_k, Hkv, d); rows of empty
    pairings are zero."""
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(k.shape, np.float64)
    oq = ok = 0
    for nq, nk in zip(lengths_q, lengths_k):
        nq, nk = int(nq), int(nk)
        if nq > 0 and nk > 0:
            a, b_, c = attention_backward(q[None, oq:oq + nq], k[None, ok:ok + nk], v[None, ok:ok + nk],
                                          dout[None, oq:oq + nq], causal=causal, scale=scale)
            dq[oq:oq + nq] = a[0]
            dk[ok:ok + nk] = b_[0]
            dv[ok:ok + nk] = c[0]
        oq += nq
        ok += nk
    return dq, dk, dv


# --------------------------------------------------------------------------
# padded <-> packed: the unpad / pad steps around the variable-length call
# (lei6393.com training-integration page, §2.5).  Plain definitions.
# --------------------------------------------------------------------------

def unpad_index(mask):
    """Kept tokens of a key-padding mask (B, L), nonzero = keep.

    Returns (cu_seqlens, indices): indices lists b*L + i for every kept
    position, row by row and in order within a row; cu_seqlens (B+1) holds
    the running count of kept tokens before each row (cu[0] = 0)."""
    m = np.asarray(mask) != 0
    B, L = m.shape
    cu = [0]
    idx = []
    for b in range(B):
        kept = np.nonzero(m[b])[0]
        idx.extend(int(b * L + i) for i in kept)
        cu.append(cu[-1] + len(kept))
    return np.asarray(cu, np.int64), np.asarray(idx, np.int64)


def gather_rows(src, indices):
    """Rows indices[0], indices[1], ... of src (first axis), stacked."""
    src = np.asarray(src)
    out = np.empty((len(indices),) + src.shape[1:], src.dtype)
    for r, i in enumerate(indices):
        out[r] = src[int(i)]
    return out


def scatter_rows(src, indices, n_rows: int, fill=0):
    """An array of n_rows rows of ``fill`` with row indices[r] = src[r]."""
    src = np.asarray(src)
    out = np.full((n_rows,) + src.shape[1:], fill, src.dtype)
    for r, i in enumerate(indices):
        out[int(i)] = src[r]
    return out


def padded_attention(q, k, v, mask, causal: bool = False, scale: Optional[float] = None):
    """Attention of a padded self-attention batch (B, L, H, d) with its
    key-padding mask, as the padded module returns it: kept query rows
    attend to the kept keys (causal: to those at or before them); padded
    query positions give O = 0 and lse = -inf (the padded output is filled
    with zeros around the kept rows)."""
    m = np.asarray(mask) != 0
    o, lse = attention(q, k, v, causal=causal, scale=scale, key_padding_mask=m.astype(np.uint8))
    o[~m] = 0.0
    lse = np.where(m[:, None, :], lse, -np.inf)
    return o, lse


def rotary(x, positions, rot_dim: int, base: float = 10000.0, interleaved: bool = False):
    """Rotary position embedding in float64 (training page §4): x (N, H, d)
    with one position per row N.  Pair p < rot_dim/2 is (p, p + rot_dim/2)
    (GPT-NeoX) or (2p, 2p+1) (GPT-J); with a = position * base^(-2p/rot_dim)
    it becomes (x1 cos a - x2 sin a, x1 sin a + x2 cos a).  Features from
    rot_dim on are unchanged."""
    x = f64(x)
    pos = np.asarray(positions, np.float64)
    out = x.copy()
    half = rot_dim // 2
    for p in range(half):
        a = pos * base ** (-2.0 * p / rot_dim)
        c, s = np.cos(a)[:, None], np.sin(a)[:, None]
        i1, i2 = (2 * p, 2 * p + 1) if interleaved else (p, p + half)
        x1, x2 = x[:, :, i1], x[:, :, i2]
        out[:, :, i1] = x1 * c - x2 * s
        out[:, :, i2] = x1 * s + x2 * c
    return out


def standard_attention_traffic_bytes(L: int, d: int, io_bytes: int = 2, score_bytes: int = 4) -> dict:
    """Byte count of the materialising (standard) attention for one head, as
    the clxhxhhr.top S23-J17 §3 table accounts it: Q, K, V read and O written
    once in the I/O dtype; S and P (L x L in fp32) each written once and read
    once."""
    qkvo = 4 * L * d * io_bytes
    s = L * L * score_bytes
    p = L * L * score_bytes
    return {"q_each": L * d * io_bytes, "s": s, "p": p, "qkvo": qkvo,
            "intermediate": 2 * s + 2 * p, "total": qkvo + 2 * s + 2 * p}
