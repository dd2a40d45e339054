"""The split schedule (host replica of the device walk) on the CPU.

Checks, for random ragged batches and every split count: each token of each
(sequence, KV head) pair is covered by exactly one CTA, in whole positions of
the kernel's seg_unit tokens (only a pair's last may be short); each CTA's
tokens lie in its run of a line on which a non-empty pair occupies seg_cost
start-up positions and then one position per seg_unit tokens, with runs
balanced to one position and filled exactly; every pair has exactly one owner
record; partial slots are unique and inside the workspace; and the CTAs
contributing partials to a split pair form the contiguous range the owner
records.
"""
from collections import defaultdict

import numpy as np
import pytest

import kv_cache_decode_gb300 as kvd


@pytest.fixture(scope="module", autouse=True)
def lib():
    from kv_cache_decode_gb300 import _build
    _build.build()
    return kvd.load()


def _check(lens, Hq, Hkv, D, n_split, s_max=None, max_len=None):
    lens = np.asarray(lens, dtype=np.int32)
    s_max = s_max or max(1, int(lens.max(initial=1)))
    max_len = s_max if max_len is None else max_len
    rows, eff = kvd.schedule_describe(lens, s_max, max_len, Hq, Hkv, D, n_split)
    B = len(lens)
    P = B * Hkv
    info = kvd.kernel_info(Hq, Hkv, D)
    X, U = info["seg_cost"], info["seg_unit"]
    assert U in (1, info["tile_tokens"])
    Lc = np.clip(lens, 0, min(s_max, max_len))
    ext = np.where(Lc > 0, -(-Lc // U) + X, 0).astype(np.int64)
    total = int(ext.sum()) * Hkv
    assert eff == (1 if total == 0 else min(n_split, total))
    # independent restatement of the runs: CTA c covers positions
    # [c*total//eff, (c+1)*total//eff); tokens [i*U, (i+1)*U) of pair p sit at
    # position start_p + X + i
    bounds = [c * total // eff for c in range(eff + 1)]
    pstart = np.concatenate([[0], np.cumsum(np.repeat(ext, Hkv))])

    covered = defaultdict(list)
    owner = defaultdict(list)
    per_cta = defaultdict(int)
    slots = set()
    contributors = defaultdict(set)
    for c, b, h, lo, hi, kind, slot, c_last in rows.tolist():
        assert 0 <= c < eff and 0 <= b < B and 0 <= h < Hkv
        p = b * Hkv + h
        if kind == 3:
            assert Lc[b] == 0 and lo == hi == 0
            owner[p].append((c, kind, c))
            continue
        assert 0 <= lo < hi <= Lc[b]
        assert lo % U == 0 and (hi % U == 0 or hi == Lc[b]), "segments are whole positions"
        v0 = pstart[p] + X
        assert bounds[c] <= v0 + lo // U and v0 + -(-hi // U) <= bounds[c + 1], \
            "segment outside the CTA's run"
        covered[p].append((lo, hi))
        per_cta[c] += hi - lo
        if kind in (0, 1):
            owner[p].append((c, kind, c_last))
        if kind in (1, 2):
            assert slot == c + p and slot not in slots and 0 <= slot < n_split + P - 1
            slots.add(slot)
            contributors[p].add(c)

    for p in range(P):
        b = p // Hkv
        assert len(owner[p]) == 1, (p, owner[p])
        iv = sorted(covered[p])
        pos = 0
        for lo, hi in iv:
            assert lo == pos
            pos = hi
        assert pos == Lc[b]
        c0, kind, c_last = owner[p][0]
        # the owner's run holds the pair's first tile (its position, if empty)
        at = pstart[p] + X if Lc[b] > 0 else pstart[p]
        if at == total:
            assert c0 == eff - 1
        else:
            assert bounds[c0] <= at < bounds[c0 + 1]
        if kind == 1:
            assert contributors[p] == set(range(c0, c_last + 1))
        elif kind == 0:
            assert len(iv) == 1 and not contributors[p]
    if total:
        assert sum(per_cta.values()) == int(Lc.sum()) * Hkv
        runs = np.diff(bounds)
        assert runs.max() - runs.min() <= 1 and runs.min() >= 1
        # a CTA's positions plus the prefixes inside its run fill the run exactly
        tiles = defaultdict(int)
        for c, b, h, lo, hi, kind, slot, c_last in rows.tolist():
            if kind != 3:
                tiles[c] += -(-hi // U) - lo // U
        pre = defaultdict(int)
        for p in range(P):
            if Lc[p // Hkv] > 0:
                for v in range(pstart[p], pstart[p] + X):
                    pre[int(np.searchsorted(bounds, v, side="right")) - 1] += 1
        assert all(tiles[c] + pre[c] == runs[c] for c in range(eff))
    return rows, eff


@pytest.mark.parametrize("seed", range(12))
def test_random_ragged(seed):
    r = np.random.default_rng(seed)
    B = int(r.integers(1, 40))
    Hkv = int(r.choice([1, 2, 4, 8]))
    G = int(r.choice([1, 4, 8, 48]))
    lens = r.integers(0, 300, B)
    lens[r.random(B) < 0.2] = 0
    for n_split in (1, 2, 3, 7, 64, 152, 1000, 100000):
        _check(lens, G * Hkv, Hkv, 128, n_split, s_max=300)


def test_configs_shapes():
    _check([2048] * 64, 48, 1, 256, 152)
    _check([256], 8, 1, 128, 4)
    r = np.random.default_rng(3)
    _check(r.integers(512, 4097, 32), 40, 40, 128, 152, s_max=4096)
    _check(r.integers(1024, 8193, 128), 32, 8, 128, 152, s_max=8192)
    _check([65536] * 4, 48, 1, 256, 152, s_max=65536)


def test_edge_cases():
    _check([0, 0, 0], 8, 2, 64, 5, s_max=16)          # no work at all: one CTA owns every pair
    _check([0, 5, 0, 0, 7, 0], 8, 2, 64, 3, s_max=16)  # empties before, between and after
    _check([1], 8, 1, 64, 50, s_max=16)               # more CTAs than tokens
    _check([16, 16], 4, 4, 128, 32, s_max=16)         # one token per CTA
    _check([5, 100, 3], 8, 1, 128, 2, s_max=200, max_len=50)  # clamped to max_seq_len
    _check([-3, 20], 8, 1, 128, 3, s_max=16)          # negative and too-long lengths clamp


def test_long_trials_shape():
    import workloads
    for i in (0, 7, 15):
        w = workloads.long_trial(i)
        _check(workloads.seq_lens(w), w.Hq, w.Hkv, w.D, 152, s_max=w.S_max)
