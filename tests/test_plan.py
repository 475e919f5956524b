"""Host logic of the persistent schedule (no GPU): every query block is covered
exactly once, only key tiles with at least one allowed key are scheduled,
split pieces tile the key range, workspace slots are consistent and the
placement is balanced."""

import math
from collections import defaultdict

import pytest

from tiled_attention_attn_gb300 import attn

SHAPES = [
    # B, Hq, Hkv, Lq, Lk, d, causal
    (1, 2, 2, 256, 256, 64, False),
    (1, 1, 1, 8192, 8192, 128, True),
    (2, 16, 16, 2048, 2048, 64, True),
    (2, 32, 8, 4096, 4096, 128, True),
    (3, 4, 2, 300, 300, 128, True),
    (1, 2, 1, 100, 300, 64, True),      # Lq < Lk, bottom-right causal
    (1, 2, 1, 300, 100, 64, True),      # Lq > Lk: early rows see no key
    (2, 3, 3, 1, 1, 64, False),
    (1, 1, 1, 129, 700, 128, False),
    (1, 4, 4, 4096, 4096, 64, True),
]


def allowed_tiles(Lq, Lk, causal, mb):
    """Key tiles holding at least one allowed key for some valid row of 256-row block mb."""
    rows = range(mb * 256, min(mb * 256 + 256, Lq))
    tiles = set()
    for j in range((Lk + 127) // 128):
        keys = range(j * 128, min(j * 128 + 128, Lk))
        if not causal:
            if len(rows) and len(keys):
                tiles.add(j)
            continue
        # some row i and key k with k <= i + (Lk - Lq)
        if len(rows) and len(keys) and keys[0] <= rows[-1] + (Lk - Lq):
            tiles.add(j)
    return tiles


@pytest.mark.parametrize("num_sms", [152, 7, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_plan_covers_every_block_once(attn_lib, shape, num_sms):
    B, Hq, Hkv, Lq, Lk, d, causal = shape
    units, n_ctas, n_part = attn.plan(B, Hq, Hkv, Lq, Lk, d, causal, num_sms)
    assert 1 <= n_ctas <= num_sms
    n_mb = (Lq + 255) // 256
    pieces = defaultdict(list)
    ctas = units[:, 7].tolist()
    assert ctas == sorted(ctas), "units must be grouped by CTA"
    assert set(ctas) == set(range(n_ctas)), "every CTA gets work"
    for u in units.tolist():
        bh, mb, a, e, split, ns, slot, cta = u
        assert 0 <= bh < B * Hq and 0 <= mb < n_mb
        pieces[(bh, mb)].append((a, e, split, ns, slot))
    assert len(pieces) == B * Hq * n_mb
    slots = []
    for (bh, mb), ps in pieces.items():
        ps.sort(key=lambda x: x[2])
        ns = ps[0][3]
        assert len(ps) == ns and [p[2] for p in ps] == list(range(ns))
        covered = []
        for a, e, split, n, slot in ps:
            assert n == ns
            covered.extend(range(a, e))
            if ns > 1:
                assert slot >= 0
                slots.append(slot)
                assert e > a
            else:
                assert slot == -1
        expect = allowed_tiles(Lq, Lk, causal, mb)
        # the union of pieces is exactly the block's allowed tiles, without overlap
        assert len(covered) == len(set(covered))
        assert set(covered) == set(range(max(expect) + 1)) if expect else covered == []
        assert set(covered) == expect
        if ns > 1:
            bases = [p[4] - p[2] for p in ps]
            assert len(set(bases)) == 1
    assert sorted(slots) == list(range(n_part))


def test_headline_plan_is_balanced(attn_lib):
    # single head, L = 8192, d = 128, causal: 2080 query/key tile pairs over 152 CTAs
    units, n_ctas, n_part = attn.plan(1, 1, 1, 8192, 8192, 128, True, 152)
    load = defaultdict(int)
    for bh, mb, a, e, split, ns, slot, cta in units.tolist():
        rows0 = min(2 * mb, 63)
        for j in range(a, e):
            load[cta] += (j <= 2 * mb) + (j <= 2 * mb + 1)
    total = sum(load.values())
    assert total == 2080
    assert n_ctas <= 152
    # pieces are whole key tiles (two tile pairs): the busiest CTA carries at
    # most one tile more than the mean load rounded up to whole tiles
    assert max(load.values()) <= 2 * math.ceil(total / 152 / 2) + 2
    assert n_part > 0   # the longest rows are split along the key range


def test_plan_rejects_bad_shapes(attn_lib):
    with pytest.raises(attn.AttnError):
        attn.plan(1, 3, 2, 128, 128, 64, False, 152)
    with pytest.raises(attn.AttnError):
        attn.plan(1, 2, 2, 128, 128, 96, False, 152)


@pytest.mark.parametrize("shape", [(1, 1, 1, 8192, 8192, True), (2, 32, 8, 4096, 4096, True),
                                   (1, 8, 2, 3000, 3000, True), (3, 4, 4, 700, 900, False),
                                   (1, 2, 2, 1000, 300, True), (1, 1, 1, 16384, 16384, True)])
@pytest.mark.parametrize("pairs", [76, 66])
def test_pair_plan_covers_each_tile_once(attn_lib, shape, pairs):
    """The CTA-pair schedule: every 256-key tile a 256-row block needs is run
    by exactly one piece; a pair runs at most one split piece, as its first
    unit (split pieces wait for each other before merging); split slots of a
    group are consecutive."""
    B, Hq, Hkv, Lq, Lk, causal = shape
    units, n_pairs, n_part = attn.plan_pair(B, Hq, Hkv, Lq, Lk, causal, pairs)
    assert n_pairs <= pairs
    n_kt = (Lk + 255) // 256
    need = {}
    for bh in range(B * Hq):
        for mb in range((Lq + 255) // 256):
            nt = n_kt
            if causal:
                last_row = min(mb * 256 + 255, Lq - 1)
                mk = last_row + (Lk - Lq)
                nt = 0 if mk < 0 else min(n_kt, mk // 256 + 1)
            need[(bh, mb)] = nt
    covered = {}
    per_pair = {}
    for u in units.tolist():
        bh, mb, a, e, split, n_split, slot, p = u
        for t in range(a, e):
            assert (bh, mb, t) not in covered
            covered[(bh, mb, t)] = True
        per_pair.setdefault(p, []).append(u)
        if n_split > 1:
            assert 0 <= slot < n_part
    for (bh, mb), nt in need.items():
        for t in range(nt):
            assert (bh, mb, t) in covered
    assert len(covered) == sum(need.values())
    for p, us in per_pair.items():
        split = [i for i, u in enumerate(us) if u[5] > 1]
        assert len(split) <= 1 and (not split or split[0] == 0)
