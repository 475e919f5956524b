"""Planted mistakes: each plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand) must make at least one pin fail.

Each case copies the oracle source to a temporary directory, applies one
textual change, compiles it with gcc and runs the pin battery below against
that build.  The real oracle is never modified.
"""

import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.golden_fixtures import load

MUTATIONS = {
    "drop_scale": ("s[j] = scale * acc;", "s[j] = acc;", 1),
    "exp_sign": ("p[j] = exp(s[j] - m);", "p[j] = exp(m - s[j]);", 1),
    "no_normalise": ("p[j] /= denom;", "p[j] /= 1.0;", 1),
    "gqa_interleaved": ("const int g = h / group;", "const int g = h % Hkv;", 1),
    "causal_strict": ("if (causal && j > i + (Lk - Lq))", "if (causal && j >= i + (Lk - Lq))", 1),
    "causal_offset_sign": ("if (causal && j > i + (Lk - Lq))", "if (causal && j > i - (Lk - Lq))", 1),
    "values_from_keys": ("acc += p[j] * v[kidx(b, j, g, c, Lk, Hkv, d)];",
                         "acc += p[j] * k[kidx(b, j, g, c, Lk, Hkv, d)];", 1),
    "lse_without_max": ("*lse_out = m + log(denom);", "*lse_out = log(denom);", 1),
    "transposed_k": ("acc += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, g, c, Lk, Hkv, d)];",
                     "acc += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, c % Lk, g, j % d, Lk, Hkv, d)];", 1),
    "mask_ignored": ("if (kmask_b && !kmask_b[j])", "if (0 && kmask_b && !kmask_b[j])", 1),
    "query_head_for_kv": ("acc += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, g, c, Lk, Hkv, d)];",
                          "acc += q[qidx(b, i, h, c, Lq, Hq, d)] * k[kidx(b, j, h % Hkv, c, Lk, Hkv, d)];", 1),
}


def _battery(L):
    """Run the pins against oracle build ``L``; return the names that fail."""
    failed = []
    rng = np.random.default_rng(5)

    def check(name, cond):
        if not cond:
            failed.append(name)

    # worked example
    g = load("online_softmax_example_5_6.txt")
    q = np.zeros((1, 1, 1, 4)); q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 2, 1, 4)); k[0, 1, 0, 0] = 1.0
    v = np.zeros((1, 2, 1, 4)); v[0, 0, 0, 0] = g["value_0"]; v[0, 1, 0, 0] = g["value_1"]
    o, lse = oracle.attention(q, k, v, scale=g["score_1"], _lib=L)
    check("worked_example", abs(o[0, 0, 0, 0] - g["result"]) < 1e-14 and abs(lse[0, 0, 0] - math.log(3)) < 1e-14)

    # torch fp64 SDPA, GQA, causal, rectangular
    for (B, Hq, Hkv, Lq, Lk, d, causal) in [(2, 4, 2, 9, 9, 8, True), (1, 4, 1, 5, 11, 8, True),
                                            (1, 2, 2, 7, 7, 4, False), (1, 4, 2, 6, 6, 8, False)]:
        q, k, v = rng.standard_normal((B, Lq, Hq, d)), rng.standard_normal((B, Lk, Hkv, d)), \
            rng.standard_normal((B, Lk, Hkv, d))
        sc = 1.0 / math.sqrt(d)
        o, lse = oracle.attention(q, k, v, causal=causal, scale=sc, _lib=L)
        qt = torch.from_numpy(q).permute(0, 2, 1, 3)
        kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, 1)
        vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, 1)
        mask = None
        if causal:
            mask = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq)
        ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=sc)
        s = (qt @ kt.transpose(-1, -2)) * sc
        if mask is not None:
            s = s.masked_fill(~mask, float("-inf"))
        lt = torch.logsumexp(s, -1)
        check(f"sdpa{(B, Hq, Hkv, Lq, Lk, d, causal)}",
              np.max(np.abs(o - ot.permute(0, 2, 1, 3).numpy())) < 1e-12 and
              np.max(np.abs(lse - lt.numpy())) < 1e-12)

    # causal row 0 is V[0]
    q, k, v = rng.standard_normal((1, 6, 2, 4)), rng.standard_normal((1, 6, 2, 4)), rng.standard_normal((1, 6, 2, 4))
    o, lse = oracle.attention(q, k, v, causal=True, _lib=L)
    check("causal_row0", np.array_equal(o[0, 0], v[0, 0]))

    # padded + mask == per-sequence runs
    lengths = [4, 2, 6]
    H, d = 2, 4
    tot = sum(lengths)
    q, k, v = rng.standard_normal((tot, H, d)), rng.standard_normal((tot, H, d)), rng.standard_normal((tot, H, d))
    qp, mask = oracle.pad_packed(q, lengths)
    kp, _ = oracle.pad_packed(k, lengths)
    vp, _ = oracle.pad_packed(v, lengths)
    op, _ = oracle.attention(qp, kp, vp, key_padding_mask=mask, _lib=L)
    ok = True
    off = 0
    for b, n in enumerate(lengths):
        o1, _ = oracle.attention(q[None, off:off + n], k[None, off:off + n], v[None, off:off + n], _lib=L)
        ok &= bool(np.max(np.abs(op[b, :n] - o1[0])) < 1e-13)
        off += n
    check("padded_vs_runs", ok)

    # zero scale: the mean of the values
    q, k, v = rng.standard_normal((1, 5, 1, 3)), rng.standard_normal((1, 5, 1, 3)), rng.standard_normal((1, 5, 1, 3))
    o, lse = oracle.attention(q, k, v, scale=0.0, _lib=L)
    check("zero_scale", np.max(np.abs(o[0, :, 0] - v[0, :, 0].mean(0))) < 1e-13 and
          np.max(np.abs(lse - math.log(5))) < 1e-13)
    return failed


@pytest.fixture(scope="module")
def tmpdir_mod(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mut")


def test_battery_passes_on_real_oracle():
    assert _battery(oracle.lib()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmpdir_mod):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new, count = MUTATIONS[name]
    src = open(oracle.SRC, encoding="utf-8").read()
    assert src.count(old) >= count, f"mutation site for {name} no longer in the oracle source"
    mutated = src.replace(old, new, count)
    d = os.path.join(str(tmpdir_mod), name)
    os.makedirs(d, exist_ok=True)
    path_c = os.path.join(d, "oracle_mut.c")
    with open(path_c, "w", encoding="utf-8") as f:
        f.write(mutated)
    path_so = os.path.join(d, "liboracle_mut.so")
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-o", path_so, path_c, "-lm"],
                   check=True, capture_output=True)
    failed = _battery(oracle.load_variant(path_so))
    assert failed, f"planted mistake {name} passed every pin"
