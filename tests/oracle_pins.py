"""Checks that pin the CPU oracle to facts fixed outside it.

Each check takes the oracle's ctypes library (so that the mutation tests can
run the same checks against deliberately broken builds of the oracle) and
raises AssertionError when the oracle disagrees with the fact it tests.

None of these re-types the oracle's formula: each compares it with a closed
form, an invariant, torch's float64 attention routine, or an exact 50-digit
decimal evaluation.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def _random_case(seed, B, Hq, Hkv, D, S_max, lens, scale=None, spread=1.0):
    r = np.random.default_rng(seed)
    q = _bits(r.standard_normal((B, Hq, D)) * spread)
    k = _bits(r.standard_normal((B, S_max, Hkv, D)) * spread)
    v = _bits(r.standard_normal((B, S_max, Hkv, D)))
    lens = np.asarray(lens, dtype=np.int32)
    if scale is None:
        scale = float(np.float32(1.0 / math.sqrt(D)))
    return q, k, v, lens, scale


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def check_identical_keys_give_mean_of_v(lib):
    """All scores equal -> uniform weights -> the mean of the valid V rows."""
    B, Hq, Hkv, D, S = 2, 6, 2, 16, 9
    q, k, v, lens, scale = _random_case(11, B, Hq, Hkv, D, S, [7, 4])
    for b in range(B):
        for g in range(Hkv):
            k[b, :, g, :] = k[b, 0, g, :]
    out, _ = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    vf = _f64(v)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            expect = vf[b, :lens[b], h // G, :].mean(axis=0)
            assert np.max(np.abs(out[b, h] - expect)) < 1e-14, (b, h)


def check_dominant_score_returns_that_row(lib):
    """One score 1000+ above the rest -> that V row (others weigh < e^-1000)."""
    B, Hq, Hkv, D, S = 1, 4, 2, 8, 6
    r = np.random.default_rng(5)
    qf = np.zeros((B, Hq, D), np.float32)
    qf[..., 0] = 1.0
    kf = (r.standard_normal((B, S, Hkv, D)) * 0.5).astype(np.float32)
    star = {0: 3, 1: 1}
    for g, t in star.items():
        kf[0, t, g, 0] = 1024.0
    q, k = _bits(qf), _bits(kf)
    v = _bits(r.standard_normal((B, S, Hkv, D)))
    lens = np.array([S], np.int32)
    out, lse = oracle.decode_attention(q, k, v, lens, 1.0, lib=lib)
    vf = _f64(v)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        assert np.array_equal(out[0, h], vf[0, star[g], g]), h
        assert abs(lse[0, h] - 1024.0) < 1e-9
        w = oracle.attention_weights(q, k, lens, 1.0, 0, h, lib=lib)
        onehot = np.zeros(S)
        onehot[star[g]] = 1.0
        assert np.array_equal(w, onehot), h


def check_single_token_returns_v0(lib):
    """L = 1 -> weight exactly 1 -> v_0 exactly, whatever q and k are."""
    q, k, v, _, scale = _random_case(3, 3, 8, 2, 32, 4, [1, 1, 1], spread=3.0)
    lens = np.array([1, 1, 1], np.int32)
    out, _ = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    vf = _f64(v)
    for b in range(3):
        for h in range(8):
            assert np.array_equal(out[b, h], vf[b, 0, h // 4]), (b, h)


def check_empty_sequence(lib):
    """L = 0 -> zero output and a -inf normaliser (the documented reading)."""
    q, k, v, _, scale = _random_case(4, 2, 2, 1, 8, 4, [0, 3])
    lens = np.array([0, 3], np.int32)
    out, lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def check_weights_sum_to_one(lib):
    q, k, v, lens, scale = _random_case(6, 2, 4, 1, 64, 300, [300, 17], spread=2.0)
    for b in range(2):
        for h in range(4):
            w = oracle.attention_weights(q, k, lens, scale, b, h, lib=lib)
            assert w.shape == (lens[b],)
            assert np.all(w >= 0.0)
            assert abs(math.fsum(w) - 1.0) < 1e-14, (b, h)


def check_token_permutation_invariance(lib):
    """Attention is a set function of the (key, value) pairs it attends to."""
    B, Hq, Hkv, D, S = 2, 8, 2, 32, 40
    q, k, v, lens, scale = _random_case(7, B, Hq, Hkv, D, S, [40, 25])
    out, lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    r = np.random.default_rng(8)
    k2, v2 = k.copy(), v.copy()
    for b in range(B):
        perm = r.permutation(lens[b])
        k2[b, :lens[b]] = k[b, perm]
        v2[b, :lens[b]] = v[b, perm]
    out2, lse2 = oracle.decode_attention(q, k2, v2, lens, scale, lib=lib)
    assert np.max(np.abs(out - out2)) < 1e-13
    assert np.max(np.abs(lse - lse2)) < 1e-12


def check_padding_never_read(lib):
    """Rows past seq_lens[b] (NaN here) never reach the output."""
    q, k, v, lens, scale = _random_case(9, 2, 4, 2, 16, 12, [5, 12])
    k[0, 5:] = 0x7FC0
    v[0, 5:] = 0x7FC0
    out, lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def check_chunked_equals_direct(lib):
    """Split-and-merge equals unsplit for every chunk count, empty chunks included."""
    B, Hq, Hkv, D, S = 3, 8, 2, 32, 70
    q, k, v, lens, scale = _random_case(10, B, Hq, Hkv, D, S, [70, 1, 33], spread=2.0)
    ref, ref_lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    for n in (1, 2, 3, 7, 33, 70, 75, 200):
        out, lse = oracle.decode_attention_chunked(q, k, v, lens, scale, n, lib=lib)
        assert np.max(np.abs(out - ref)) < 1e-12, n
        assert np.max(np.abs(lse - ref_lse)) < 1e-12, n


# ---------------------------------------------------------------------------
# Library routine: torch float64 scaled_dot_product_attention
# ---------------------------------------------------------------------------

def check_against_torch_sdpa(lib):
    import torch
    import torch.nn.functional as F
    cases = [  # (seed, B, Hq, Hkv, D, S_max, lens)
        (20, 2, 8, 1, 64, 50, [50, 13]),      # multiquery
        (21, 3, 8, 2, 16, 33, [33, 1, 20]),   # grouped
        (22, 2, 4, 4, 8, 9, [9, 4]),          # multi-head
        (23, 1, 12, 3, 32, 64, [64]),
    ]
    for seed, B, Hq, Hkv, D, S, lens in cases:
        q, k, v, lens, scale = _random_case(seed, B, Hq, Hkv, D, S, lens, spread=1.5)
        out, lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
        qf, kf, vf = (torch.from_numpy(_f64(x)) for x in (q, k, v))
        G = Hq // Hkv
        for b in range(B):
            L = int(lens[b])
            kk = kf[b, :L].permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
            vv = vf[b, :L].permute(1, 0, 2).repeat_interleave(G, dim=0)
            qq = qf[b].unsqueeze(1)                                      # [Hq, 1, D]
            ref = F.scaled_dot_product_attention(qq, kk, vv, scale=scale)[:, 0, :]
            assert np.max(np.abs(out[b] - ref.numpy())) < 1e-12, (seed, b)
            s = torch.einsum("hd,hld->hl", qf[b], kk) * scale
            ref_lse = torch.logsumexp(s, dim=-1)
            assert np.max(np.abs(lse[b] - ref_lse.numpy())) < 1e-12, (seed, b)


# ---------------------------------------------------------------------------
# Exact evaluation: 50-digit decimal arithmetic on tiny inputs
# ---------------------------------------------------------------------------

def _decimal_attention(qf, kf, vf, L, G, scale):
    getcontext().prec = 50
    B, Hq, D = qf.shape
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    sc = Decimal(float(scale))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = [sc * sum(Decimal(float(qf[b, h, d])) * Decimal(float(kf[b, t, g, d]))
                          for d in range(D)) for t in range(L[b])]
            e = [x.exp() for x in s]
            z = sum(e)
            for d in range(D):
                out[b, h, d] = float(sum(e[t] * Decimal(float(vf[b, t, g, d]))
                                         for t in range(L[b])) / z)
            lse[b, h] = float(z.ln())
    return out, lse


def check_decimal_brute_force(lib):
    for seed, B, Hq, Hkv, D, S, lens in [(30, 2, 4, 2, 8, 5, [5, 3]),
                                         (31, 1, 3, 1, 4, 4, [4]),
                                         (32, 2, 2, 2, 6, 5, [2, 5])]:
        q, k, v, lens, scale = _random_case(seed, B, Hq, Hkv, D, S, lens, spread=2.0)
        out, lse = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
        ref, ref_lse = _decimal_attention(_f64(q), _f64(k), _f64(v), lens, Hq // Hkv, scale)
        assert np.max(np.abs(out - ref)) < 1e-14, seed
        assert np.max(np.abs(lse - ref_lse)) < 1e-13, seed


# ---------------------------------------------------------------------------
# Cached decoding equals full recomputation (toy one-layer model)
# ---------------------------------------------------------------------------

def check_cached_decode_equals_recompute(lib):
    """Generating with a KV cache (append, then attend) gives, at every step,
    the same attention output as recomputing causal attention over the whole
    prefix: a token only attends to earlier tokens, so earlier keys and values
    never change (All About Transformer Inference, "Transformer inference basics")."""
    import torch
    import torch.nn.functional as F
    r = np.random.default_rng(40)
    T, E, Hq, Hkv, D = 12, 16, 4, 2, 8
    G = Hq // Hkv
    x = r.standard_normal((T, E))
    Wq = r.standard_normal((E, Hq, D)) / math.sqrt(E)
    Wk = r.standard_normal((E, Hkv, D)) / math.sqrt(E)
    Wv = r.standard_normal((E, Hkv, D)) / math.sqrt(E)
    qb = _bits(np.einsum("te,ehd->thd", x, Wq))
    kb = _bits(np.einsum("te,ehd->thd", x, Wk))
    vb = _bits(np.einsum("te,ehd->thd", x, Wv))
    scale = float(np.float32(1.0 / math.sqrt(D)))

    # Full recomputation with a causal mask over all T tokens at once.
    qf, kf, vf = (torch.from_numpy(_f64(a)) for a in (qb, kb, vb))
    full = F.scaled_dot_product_attention(
        qf.permute(1, 0, 2), kf.permute(1, 0, 2).repeat_interleave(G, 0),
        vf.permute(1, 0, 2).repeat_interleave(G, 0), is_causal=True, scale=scale,
    ).permute(1, 0, 2).numpy()  # [T, Hq, D]

    # Step by step: append token t's key/value, then decode with L = t + 1.
    kc = np.full((1, T, Hkv, D), 0x7FC0, np.uint16)
    vc = np.full((1, T, Hkv, D), 0x7FC0, np.uint16)
    for t in range(T):
        kc, vc, skipped = oracle.kv_append(kc, vc, kb[t][None], vb[t][None],
                                           np.array([t], np.int32), lib=lib)
        assert skipped == 0
        out, _ = oracle.decode_attention(qb[t][None], kc, vc, np.array([t + 1], np.int32),
                                         scale, lib=lib)
        assert np.max(np.abs(out[0] - full[t])) < 1e-12, t


def check_append_is_a_byte_copy(lib):
    r = np.random.default_rng(50)
    B, S, Hkv, D = 3, 6, 2, 8
    kc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    vc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    kn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    vn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    pos = np.array([0, 5, 6], np.int32)  # the last one is out of range
    k2, v2, skipped = oracle.kv_append(kc, vc, kn, vn, pos, lib=lib)
    ek, ev = kc.copy(), vc.copy()
    ek[0, 0], ev[0, 0] = kn[0], vn[0]
    ek[1, 5], ev[1, 5] = kn[1], vn[1]
    assert skipped == 1
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


def _page_table(seed, B, S, P, lens, spare=3):
    """A shuffled placement of each sequence's blocks in a pool of pages.

    Block j of sequence b goes to page perm[b * nb + j]; entries past a
    sequence's blocks are -1. Returns (table, num_pages).
    """
    r = np.random.default_rng(seed)
    nb = S // P
    num_pages = B * nb + spare
    perm = r.permutation(num_pages)[:B * nb]
    table = np.full((B, nb), -1, np.int32)
    for b in range(B):
        for j in range(-(-int(lens[b]) // P)):
            table[b, j] = perm[b * nb + j]
    return table, num_pages


def _fill_pool(cache, table, num_pages, seed):
    """Pages of random bits, then block j of sequence b copied in as one slice."""
    B, S, Hkv, D = cache.shape
    P = S // table.shape[1]
    pool = np.random.default_rng(seed).integers(0, 2**16, (num_pages, P, Hkv, D), dtype=np.uint16)
    for b in range(B):
        for j in range(table.shape[1]):
            if table[b, j] >= 0:
                pool[table[b, j]] = cache[b, j * P:(j + 1) * P]
    return pool


def check_paged_identity_pool_is_the_cache(lib):
    # A pool that is the contiguous cache reshaped page by page, with the
    # table naming page b * nb + j for block j of sequence b.
    r = np.random.default_rng(60)
    B, S, Hkv, D, P = 3, 12, 2, 4, 4
    cache = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    pool = cache.reshape(B * S // P, P, Hkv, D)
    table = np.arange(B * S // P, dtype=np.int32).reshape(B, S // P)
    lens = np.array([12, 5, 0], np.int32)
    got, zeroed = oracle.paged_gather(pool, table, lens, lib=lib)
    assert zeroed == 0
    for b in range(B):
        assert np.array_equal(got[b, :lens[b]], cache[b, :lens[b]]), b


def check_paged_shuffled_pool(lib):
    B, S, Hkv, D, P = 4, 16, 2, 8, 4
    lens = np.array([16, 1, 7, 9], np.int32)
    table, num_pages = _page_table(61, B, S, P, lens)
    r = np.random.default_rng(62)
    kc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    got, zeroed = oracle.paged_gather(_fill_pool(kc, table, num_pages, 63), table, lens, lib=lib)
    assert zeroed == 0
    for b in range(B):
        assert np.array_equal(got[b, :lens[b]], kc[b, :lens[b]]), b
    # attention over the pools equals attention over the contiguous caches
    q = _bits(r.standard_normal((B, 4, D)))
    kc = _bits(r.standard_normal((B, S, Hkv, D)))
    vc = _bits(r.standard_normal((B, S, Hkv, D)))
    kpool, vpool = _fill_pool(kc, table, num_pages, 64), _fill_pool(vc, table, num_pages, 65)
    direct, lse_d = oracle.decode_attention(q, kc, vc, lens, 0.25, lib=lib)
    paged, lse_p = oracle.decode_attention_paged(q, kpool, vpool, table, lens, 0.25, lib=lib)
    assert np.array_equal(direct, paged) and np.array_equal(lse_d, lse_p)


def check_paged_tiny_hand_example(lib):
    # P = 2, one sequence of 3 tokens: block 0 is page 2, block 1 is page 0, so
    # tokens 0, 1 are rows 0, 1 of page 2 and token 2 is row 0 of page 0.
    P = 2
    kp = np.zeros((3, P, 1, 2), np.float32)
    vp = np.zeros((3, P, 1, 2), np.float32)
    kp[2, 0, 0], kp[2, 1, 0], kp[0, 0, 0] = [0, 0], [1, 0], [2, 0]
    vp[2, 0, 0], vp[2, 1, 0], vp[0, 0, 0] = [1, 0], [0, 1], [1, 1]
    kp[0, 1, 0] = kp[1, :, 0] = [9, 9]  # never attended
    vp[0, 1, 0] = vp[1, :, 0] = [-5, 7]
    table = np.array([[2, 0]], np.int32)
    q = _bits(np.array([[[1.0, 0.0]]]))
    out, lse = oracle.decode_attention_paged(q, _bits(kp), _bits(vp), table, np.array([3], np.int32),
                                             1.0, lib=lib)
    e = [math.exp(0.0), math.exp(1.0), math.exp(2.0)]
    z = sum(e)
    want = [(e[0] + e[2]) / z, (e[1] + e[2]) / z]
    assert abs(out[0, 0, 0] - want[0]) < 1e-15 and abs(out[0, 0, 1] - want[1]) < 1e-15, out
    assert abs(lse[0, 0] - math.log(z)) < 1e-15


def check_paged_invalid_entry_reads_zero_rows(lib):
    B, S, Hkv, D, P = 2, 12, 1, 4, 4
    lens = np.array([10, 12], np.int32)
    table, num_pages = _page_table(66, B, S, P, lens)
    kc = np.random.default_rng(67).integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    kpool = _fill_pool(kc, table, num_pages, 68)
    table[1, 1] = num_pages  # not a page of the pool: tokens 4..7 of sequence 1
    table[0, 2] = -7         # tokens 8, 9 of sequence 0
    got, zeroed = oracle.paged_gather(kpool, table, lens, lib=lib)
    assert zeroed == 4 + 2
    want = kc.copy()
    want[1, 4:8] = 0
    want[0, 8:10] = 0
    for b in range(B):
        assert np.array_equal(got[b, :lens[b]], want[b, :lens[b]]), b


def check_paged_append(lib):
    B, S, Hkv, D, P = 5, 16, 2, 4, 8
    lens = np.array([16, 9, 8, 1, 16], np.int32)
    table, num_pages = _page_table(69, B, S, P, lens)
    r = np.random.default_rng(70)
    kpool = r.integers(0, 2**16, (num_pages, P, Hkv, D), dtype=np.uint16)
    vpool = r.integers(0, 2**16, (num_pages, P, Hkv, D), dtype=np.uint16)
    kn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    vn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    table[4, 1] = -1                              # sequence 4's second block is unassigned
    pos = np.array([15, 8, 7, 0, 9], np.int32)    # page ends and starts; sequence 4 hits -1
    k2, v2, skipped, bad = oracle.kv_append_paged(kpool, vpool, kn, vn, table, pos, lib=lib)
    assert skipped == 1 and bad == 1
    # exactly the named rows changed
    ek, ev = kpool.copy(), vpool.copy()
    ek[table[0, 1], 7], ev[table[0, 1], 7] = kn[0], vn[0]
    ek[table[1, 1], 0], ev[table[1, 1], 0] = kn[1], vn[1]
    ek[table[2, 0], 7], ev[table[2, 0], 7] = kn[2], vn[2]
    ek[table[3, 0], 0], ev[table[3, 0], 0] = kn[3], vn[3]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    # pos outside [0, capacity) is skipped without a bad-page count
    _, _, skipped, bad = oracle.kv_append_paged(kpool, vpool, kn, vn, table,
                                                np.array([16, -1, 0, 0, 0], np.int32), lib=lib)
    assert skipped == 2 and bad == 0
    # an entry one past the pool's pages: skipped and counted (the arrays hold
    # one page more than the pool size passed, so a wrong write stays in memory)
    import ctypes
    kx, vx = kpool.copy(), vpool.copy()
    t2 = table.copy()
    t2[0, 1] = num_pages - 1
    badc = ctypes.c_int(0)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    skipped = lib.kvo_kv_append_paged(ptr(kx), ptr(vx), ptr(kn), ptr(vn), ptr(t2), ptr(pos), B,
                                      t2.shape[1], P, num_pages - 1, Hkv, D, ctypes.byref(badc))
    assert skipped == 2 and badc.value == 2
    assert np.array_equal(kx[num_pages - 1], kpool[num_pages - 1])


def check_q8_closed_forms(lib):
    # max |x| = 127 gives scale 1, so codes are x rounded half to even and the
    # extreme elements map to +-127; an all-zero row gives scale 0 and codes 0.
    x = _bits(np.array([[127.0, 2.5, 3.5, -2.5, -127.0, 0.5, 1.5, 0.0],
                        [0.0] * 8,
                        [-6.0, 3.0, 1.5, 0.0, 0.75, -0.25, 6.0, 2.0]], np.float32))
    codes, scales = oracle.quantize_q8(x, lib=lib)
    assert scales[0] == 1.0 and scales[1] == 0.0
    assert list(codes[0]) == [127, 2, 4, -2, -127, 0, 2, 0], codes[0]
    assert list(codes[1]) == [0] * 8
    # third row: a = 6, scale = 6/127 in float32; the extremes are exactly +-127
    assert scales[2] == np.float32(6.0) / np.float32(127.0)
    assert codes[2][0] == -127 and codes[2][6] == 127 and codes[2][3] == 0
    back = oracle.dequantize_q8(codes, scales, lib=lib)
    assert back[0][0] == 127.0 and back[0][1] == 2.0 and back[2][6] == float(scales[2]) * 127


def check_q8_error_bound(lib):
    # Every element reads back within half a step (the scale) of its value,
    # the largest element of each row reads back as +-127 steps, and signs
    # are kept.
    r = np.random.default_rng(71)
    mags = np.exp(r.uniform(-6, 6, size=(400, 1)))
    xf = (r.standard_normal((400, 96)) * mags).astype(np.float32)
    x = _bits(xf)
    xv = _f64(x)
    codes, scales = oracle.quantize_q8(x, lib=lib)
    back = oracle.dequantize_q8(codes, scales, lib=lib)
    err = np.abs(back - xv)
    assert np.all(err <= scales[:, None].astype(np.float64) * (0.5 + 1e-5)), float(np.max(err / scales[:, None]))
    amax = np.abs(xv).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(400), amax]) == 127)
    assert np.all(np.sign(codes) == np.where(np.abs(xv) < scales[:, None] / 2, 0, np.sign(xv)))


def check_f64kv_attention_is_the_bf16_attention(lib):
    # The double-cache attention on caches holding exactly the bf16 values is
    # the bf16-cache attention, bit for bit.
    q, k, v, lens, scale = _random_case(72, 3, 8, 2, 16, 10, [10, 3, 0])
    out_a, lse_a = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    out_b, lse_b = oracle.decode_attention_f64kv(q, _f64(k), _f64(v), lens, scale, lib=lib)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def check_q8_attention_close_to_bf16(lib):
    # Attention over the int8 rows stays within the quantization error of the
    # bf16 attention: each row moves by at most half a step, and the output is
    # a convex combination of value rows.
    q, k, v, lens, scale = _random_case(73, 2, 4, 1, 64, 40, [40, 17])
    kc, ks = oracle.quantize_q8(k, lib=lib)
    vc, vs = oracle.quantize_q8(v, lib=lib)
    out_q, _ = oracle.decode_attention_q8(q, kc, vc, ks, vs, lens, scale, lib=lib)
    out_b, _ = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    assert np.max(np.abs(out_q - out_b)) < 0.05
    assert np.max(np.abs(out_q - out_b)) > 0.0


def check_q8_append(lib):
    r = np.random.default_rng(74)
    B, S, Hkv, D = 3, 6, 2, 8
    kc = r.integers(-127, 128, (B, S, Hkv, D), dtype=np.int8)
    vc = r.integers(-127, 128, (B, S, Hkv, D), dtype=np.int8)
    ks = r.random((B, S, Hkv)).astype(np.float32)
    vs = r.random((B, S, Hkv)).astype(np.float32)
    kn = _bits(r.standard_normal((B, Hkv, D)))
    vn = _bits(r.standard_normal((B, Hkv, D)))
    pos = np.array([0, 5, 6], np.int32)  # the last one is out of range
    k2, v2, ks2, vs2, skipped = oracle.kv_append_q8(kc, vc, ks, vs, kn, vn, pos, lib=lib)
    assert skipped == 1
    ek, eks = oracle.quantize_q8(kn, lib=lib)
    ev, evs = oracle.quantize_q8(vn, lib=lib)
    want_k, want_ks = kc.copy(), ks.copy()
    want_k[0, 0], want_k[1, 5], want_ks[0, 0], want_ks[1, 5] = ek[0], ek[1], eks[0], eks[1]
    assert np.array_equal(k2, want_k) and np.array_equal(ks2, want_ks)
    want_v, want_vs = vc.copy(), vs.copy()
    want_v[0, 0], want_v[1, 5], want_vs[0, 0], want_vs[1, 5] = ev[0], ev[1], evs[0], evs[1]
    assert np.array_equal(v2, want_v) and np.array_equal(vs2, want_vs)


def check_multi_token_one_is_single(lib):
    q, k, v, lens, scale = _random_case(80, 3, 8, 2, 16, 12, [12, 5, 0])
    a, la = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    b, lb = oracle.decode_attention_multi(q[:, None], k, v, lens, scale, lib=lib)
    assert np.array_equal(a, b[:, 0]) and np.array_equal(la, lb[:, 0])


def check_multi_token_against_torch_causal(lib):
    # The last T positions of a causal self-attention (torch float64, explicit
    # causal mask over the whole sequence) are the multi-token decode.
    torch = __import__("pytest").importorskip("torch")
    B, T, Hq, Hkv, D, S = 2, 3, 4, 2, 8, 9
    q, k, v, _, scale = _random_case(81, B, Hq, Hkv, D, S, [S, S])
    r = np.random.default_rng(82)
    qm = _bits(r.standard_normal((B, T, Hq, D)))
    lens = np.array([9, 6], np.int32)
    out, _ = oracle.decode_attention_multi(qm, k, v, lens, scale, lib=lib)
    G = Hq // Hkv
    for b in range(B):
        L = int(lens[b])
        kk = torch.from_numpy(_f64(k[b, :L])).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        vv = torch.from_numpy(_f64(v[b, :L])).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qq = torch.from_numpy(_f64(qm[b])).permute(1, 0, 2)                                    # [Hq, T, D]
        pos_q = torch.arange(L - T, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos_q                                               # [T, L]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        assert np.max(np.abs(ref.permute(1, 0, 2).numpy() - out[b])) < 1e-12, b


def check_multi_token_append(lib):
    r = np.random.default_rng(83)
    B, S, Hkv, D, T = 3, 8, 2, 4, 3
    kc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    vc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    kn = r.integers(0, 2**16, (B, T, Hkv, D), dtype=np.uint16)
    vn = r.integers(0, 2**16, (B, T, Hkv, D), dtype=np.uint16)
    pos = np.array([0, 5, 7], np.int32)  # the last sequence has room for one of its three rows
    k2, v2, skipped = oracle.kv_append_multi(kc, vc, kn, vn, pos, lib=lib)
    assert skipped == 2
    ek, ev = kc.copy(), vc.copy()
    for b, p0 in enumerate(pos):
        for i in range(T):
            if p0 + i < S:
                ek[b, p0 + i], ev[b, p0 + i] = kn[b, i], vn[b, i]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)


def _q8_pool(cache_codes, cache_scales, table, num_pages, seed):
    """int8 page pools: pages of random codes and scales, then block j of
    sequence b copied in as one slice (as _fill_pool does for bf16)."""
    B, S, Hkv, D = cache_codes.shape
    P = S // table.shape[1]
    r = np.random.default_rng(seed)
    cp = r.integers(-128, 128, (num_pages, P, Hkv, D), dtype=np.int8)
    sp = r.standard_normal((num_pages, P, Hkv)).astype(np.float32)
    for b in range(B):
        for j in range(table.shape[1]):
            if table[b, j] >= 0:
                cp[table[b, j]] = cache_codes[b, j * P:(j + 1) * P]
                sp[table[b, j]] = cache_scales[b, j * P:(j + 1) * P]
    return cp, sp


def check_paged_q8_pools_are_the_cache(lib):
    # Shuffled int8 pools gather back to the contiguous codes and scales
    # exactly, and attention over them equals the contiguous int8 attention.
    B, S, Hkv, D, P = 4, 16, 2, 8, 4
    lens = np.array([16, 1, 7, 0], np.int32)
    table, num_pages = _page_table(80, B, S, P, lens)
    r = np.random.default_rng(81)
    kc, ks = oracle.quantize_q8(_bits(r.standard_normal((B, S, Hkv, D))), lib=lib)
    vc, vs = oracle.quantize_q8(_bits(r.standard_normal((B, S, Hkv, D))), lib=lib)
    kcp, ksp = _q8_pool(kc, ks, table, num_pages, 82)
    vcp, vsp = _q8_pool(vc, vs, table, num_pages, 83)
    gc, gs, zeroed = oracle.paged_gather_q8(kcp, ksp, table, lens, lib=lib)
    assert zeroed == 0 and gc.dtype == np.int8 and gs.dtype == np.float32
    for b in range(B):
        assert np.array_equal(gc[b, :lens[b]], kc[b, :lens[b]]), b
        assert np.array_equal(gs[b, :lens[b]].view(np.uint32), ks[b, :lens[b]].view(np.uint32)), b
    q = _bits(r.standard_normal((B, 4, D)))
    direct, lse_d = oracle.decode_attention_q8(q, kc, vc, ks, vs, lens, 0.5, lib=lib)
    paged, lse_p = oracle.decode_attention_q8_paged(q, kcp, vcp, ksp, vsp, table, lens, 0.5, lib=lib)
    assert np.array_equal(direct, paged) and np.array_equal(lse_d, lse_p)
    # an entry that names no page reads zero codes and a zero scale
    table[0, 1] = -2
    gc, gs, zeroed = oracle.paged_gather_q8(kcp, ksp, table, lens, lib=lib)
    assert zeroed == P and not gc[0, P:2 * P].any() and not gs[0, P:2 * P].any()
    assert np.array_equal(gc[0, :P], kc[0, :P]) and np.array_equal(gc[0, 2 * P:], kc[0, 2 * P:])


def check_paged_q8_append(lib):
    # The paged int8 append writes the rows the contiguous int8 append writes,
    # at the table's pages; a position past the capacity or an entry that
    # names no page is skipped.
    B, S, Hkv, D, P = 5, 16, 2, 8, 8
    lens = np.array([16, 9, 8, 1, 16], np.int32)
    table, num_pages = _page_table(84, B, S, P, lens)
    r = np.random.default_rng(85)
    kc, ks = oracle.quantize_q8(_bits(r.standard_normal((B, S, Hkv, D))), lib=lib)
    vc, vs = oracle.quantize_q8(_bits(r.standard_normal((B, S, Hkv, D))), lib=lib)
    kcp, ksp = _q8_pool(kc, ks, table, num_pages, 86)
    vcp, vsp = _q8_pool(vc, vs, table, num_pages, 87)
    kn = _bits(r.standard_normal((B, Hkv, D)))
    vn = _bits(r.standard_normal((B, Hkv, D)))
    pos = np.array([15, 8, 7, 0, 16], np.int32)  # page ends and starts; sequence 4 past the capacity
    table[2, 0] = num_pages                      # sequence 2's row names no page
    got = oracle.kv_append_q8_paged(kcp, vcp, ksp, vsp, kn, vn, table, pos, lib=lib)
    assert got[4] == 2 and got[5] == 1
    want = oracle.kv_append_q8(kc, vc, ks, vs, kn, vn, np.where(np.arange(B) == 2, -1, pos), lib=lib)
    for b, t in ((0, 15), (1, 8), (3, 0)):
        page, row = table[b, t // P], t % P
        for g, w in zip(got[:4], want[:4]):
            assert np.array_equal(np.asarray(g[page, row]).view(np.uint8), np.asarray(w[b, t]).view(np.uint8)), (b, t)
    # nothing else changed
    changed = np.zeros((num_pages, P), bool)
    for b, t in ((0, 15), (1, 8), (3, 0)):
        changed[table[b, t // P], t % P] = True
    assert np.array_equal(got[0][~changed], kcp[~changed]) and np.array_equal(got[3][~changed].view(np.uint32),
                                                                               vsp[~changed].view(np.uint32))


def check_unified_max_equals_definition(lib):
    # Scores within the window: every chunking gives the softmax itself (out
    # and lse), with no row falling back.
    r = np.random.default_rng(90)
    B, S, Hq, Hkv, D = 3, 40, 4, 2, 8
    q = _bits(r.standard_normal((B, Hq, D)))
    k = _bits(r.standard_normal((B, S, Hkv, D)))
    v = _bits(r.standard_normal((B, S, Hkv, D)))
    lens = np.array([40, 17, 1], np.int32)
    want, want_lse = oracle.decode_attention(q, k, v, lens, 0.3, lib=lib)
    for phi in (0.0, 1.5, -2.0):
        for n_chunks in (1, 3, 40):
            out, lse, fb = oracle.decode_attention_unified_max(q, k, v, lens, 0.3, phi, n_chunks, lib=lib)
            assert not fb.any()
            assert np.max(np.abs(out - want)) < 1e-13 and np.max(np.abs(lse - want_lse)) < 1e-13, (phi, n_chunks)


def check_unified_max_closed_form(lib):
    # Identical keys with phi equal to their score: every weight is exp(0) = 1,
    # so the output is the plain mean of the value rows and lse = phi + ln L.
    D, L = 4, 6
    q = _bits(np.array([[[1.0, 2.0, 0.0, 0.0]]]))
    k = _bits(np.tile(np.array([0.5, 0.25, 3.0, -1.0]), (1, L, 1, 1)))
    vals = np.arange(L * D, dtype=np.float64).reshape(1, L, 1, D)
    v = _bits(vals)
    phi = 0.5 * (0.5 + 0.5)  # scale * q . k with scale 0.5
    out, lse, fb = oracle.decode_attention_unified_max(q, k, v, np.array([L], np.int32), 0.5, phi, 4, lib=lib)
    assert not fb.any()
    assert np.array_equal(out[0, 0], vals[0, :, 0, :].mean(axis=0))
    assert abs(lse[0, 0] - (phi + math.log(L))) < 1e-15


def check_unified_max_window_edges(lib):
    # One token per row, scores 0: phi = -8 ln 2 puts the score on the upper
    # edge (kept), a little lower phi outside (recomputed); likewise the lower
    # edge at phi = 64 ln 2. Recomputed rows equal the definition.
    q = _bits(np.zeros((1, 1, 2)))
    k = _bits(np.ones((1, 1, 1, 2)))
    v = _bits(np.array([[[[3.0, -1.0]]]]))
    lens = np.array([1], np.int32)
    lo, hi = oracle.UMAX_WINDOW
    for phi, falls in ((-hi, False), (-hi - 1e-9, True), (-lo, False), (-lo + 1e-9, True)):
        out, lse, fb = oracle.decode_attention_unified_max(q, k, v, lens, 1.0, phi, 1, lib=lib)
        assert bool(fb[0, 0]) == falls, phi
        assert np.max(np.abs(out[0, 0] - [3.0, -1.0])) < 1e-14 and abs(lse[0, 0]) < 1e-12


def check_e4m3_format_values(lib):
    # Values the E4M3 definition fixes: bias 7, 3 mantissa bits, subnormals
    # m/8 * 2^-6, largest finite 1.75 * 2^8.
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875,
             0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    for code, want in fixed.items():
        assert oracle.e4m3_value(code, lib=lib) == want, hex(code)


def check_e4m3_rounding(lib):
    # Every finite value encodes to its own code (+-0 to +0); midpoints between
    # neighbours go to the code with the even low bit; past 448 saturates.
    for c in list(range(1, 0x7F)) + list(range(0x81, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_value(c, lib=lib), lib=lib) == c, hex(c)
    assert oracle.e4m3_encode(-0.0, lib=lib) == 0 and oracle.e4m3_encode(-1e-9, lib=lib) == 0
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_value(c, lib=lib), oracle.e4m3_value(c + 1, lib=lib)
        mid = np.float32((lo + hi) / 2)
        if float(mid) != (lo + hi) / 2:
            continue  # not a float32 value
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid), lib=lib) == (want if want else 0), hex(c)
    for y in (448.0, 449.0, 464.0, 500.0, 1e30):
        assert oracle.e4m3_encode(y, lib=lib) == 0x7E and oracle.e4m3_encode(-y, lib=lib) == 0xFE


def check_e4m3_against_torch(lib):
    # torch's float8_e4m3fn conversion (round to nearest even) agrees on every
    # value inside the finite range, subnormals included (torch keeps the sign
    # of a zero result; the scheme here stores +0).
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(73)
    ys = np.concatenate([r.uniform(-448, 448, 3000), r.uniform(-0.02, 0.02, 3000),
                         np.exp(r.uniform(-12, 6, 3000)) * r.choice([-1, 1], 3000)]).astype(np.float32)
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)
    got = np.array([oracle.e4m3_encode(float(y), lib=lib) for y in ys])
    assert np.array_equal(got, ref), ys[got != ref][:5]


def check_fp8_quantizer(lib):
    # The largest element of each row reads back as +-448 steps of its scale
    # and every element within half an E4M3 spacing of its value.
    r = np.random.default_rng(74)
    mags = np.exp(r.uniform(-6, 6, size=(300, 1)))
    x = _bits((r.standard_normal((300, 64)) * mags).astype(np.float32))
    xv = _f64(x)
    codes, scales = oracle.quantize_fp8(x, lib=lib)
    assert codes.dtype == np.uint8
    back = oracle.dequantize_fp8(codes, scales, lib=lib)
    amax = np.abs(xv).argmax(axis=1)
    assert np.all((codes[np.arange(300), amax] & 0x7F) == 0x7E)
    y = np.abs(xv) / scales[:, None]
    spacing = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3))
    assert np.all(np.abs(back - xv) <= scales[:, None] * spacing * (0.5 + 1e-3))
    # int8 and fp8 paged caches gather back to their contiguous rows byte for byte
    B, S, Hkv, D, P = 2, 8, 1, 64, 4
    lens = np.array([8, 5], np.int32)
    table = np.array([[3, 0], [1, 2]], np.int32)
    cc, cs = codes[:B * S].reshape(B, S, Hkv, D), scales[:B * S].reshape(B, S, Hkv)
    pool_c = np.zeros((4, P, Hkv, D), np.uint8)
    pool_s = np.zeros((4, P, Hkv), np.float32)
    for b in range(B):
        for j in range(2):
            pool_c[table[b, j]], pool_s[table[b, j]] = cc[b, j * P:(j + 1) * P], cs[b, j * P:(j + 1) * P]
    gc, gs, _ = oracle.paged_gather_q8(pool_c, pool_s, table, lens, lib=lib, fmt="fp8")
    for b in range(B):
        assert np.array_equal(gc[b, :lens[b]], cc[b, :lens[b]]) and np.array_equal(gs[b, :lens[b]], cs[b, :lens[b]])


def check_fp8_attention_close_to_bf16(lib):
    # Attention over the fp8 rows of N(0, 1) caches stays near the bf16
    # attention (E4M3 keeps 3 mantissa bits: about 3 % per element).
    q, k, v, lens, scale = _random_case(75, 3, 8, 2, 32, 40, [40, 9, 1])
    kc, ks = oracle.quantize_fp8(k, lib=lib)
    vc, vs = oracle.quantize_fp8(v, lib=lib)
    ref, _ = oracle.decode_attention(q, k, v, lens, scale, lib=lib)
    got, _ = oracle.decode_attention_q8(q, kc, vc, ks, vs, lens, scale, lib=lib, fmt="fp8")
    assert np.max(np.abs(got - ref)) < 0.1


def check_merge_attention_of_shards(lib):
    # Attention over a sequence's tokens split into disjoint shards, each
    # attended alone, merges back to the attention over all of them; a shard
    # with no tokens adds nothing, and a row with none anywhere stays empty.
    r = np.random.default_rng(91)
    B, S, Hq, Hkv, D = 3, 30, 4, 2, 8
    q = _bits(r.standard_normal((B, Hq, D)))
    k = _bits(r.standard_normal((B, S, Hkv, D)))
    v = _bits(r.standard_normal((B, S, Hkv, D)))
    lens = np.array([30, 11, 0], np.int32)
    want, want_lse = oracle.decode_attention(q, k, v, lens, 0.4, lib=lib)
    cuts = [0, 7, 7, 19, 30]  # shard 1 holds no tokens
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = np.clip(lens - a, 0, b - a).astype(np.int32)
        o, l = oracle.decode_attention(q, np.ascontiguousarray(k[:, a:b]) if b > a else k[:, :1] * 0,
                                       np.ascontiguousarray(v[:, a:b]) if b > a else v[:, :1] * 0,
                                       sl if b > a else np.zeros(B, np.int32), 0.4, lib=lib)
        outs.append(o)
        lses.append(l)
    out, lse = oracle.merge_attention(outs, lses)
    assert np.max(np.abs(out - want)) < 1e-13
    live = np.isfinite(want_lse)
    assert np.max(np.abs(lse[live] - want_lse[live])) < 1e-13 and np.all(np.isneginf(lse[~live]))
    assert np.all(out[2] == 0)
    # one shard alone is itself
    o1, l1 = oracle.merge_attention(outs[:1], lses[:1])
    assert np.array_equal(o1[:2], outs[0][:2])


ALL_CHECKS = [
    check_identical_keys_give_mean_of_v,
    check_dominant_score_returns_that_row,
    check_single_token_returns_v0,
    check_empty_sequence,
    check_weights_sum_to_one,
    check_token_permutation_invariance,
    check_padding_never_read,
    check_chunked_equals_direct,
    check_against_torch_sdpa,
    check_decimal_brute_force,
    check_cached_decode_equals_recompute,
    check_append_is_a_byte_copy,
    check_paged_identity_pool_is_the_cache,
    check_paged_shuffled_pool,
    check_paged_tiny_hand_example,
    check_paged_invalid_entry_reads_zero_rows,
    check_paged_append,
    check_q8_closed_forms,
    check_q8_error_bound,
    check_f64kv_attention_is_the_bf16_attention,
    check_q8_attention_close_to_bf16,
    check_q8_append,
    check_paged_q8_pools_are_the_cache,
    check_paged_q8_append,
    check_unified_max_equals_definition,
    check_unified_max_closed_form,
    check_unified_max_window_edges,
    check_e4m3_format_values,
    check_e4m3_rounding,
    check_e4m3_against_torch,
    check_fp8_quantizer,
    check_fp8_attention_close_to_bf16,
    check_merge_attention_of_shards,
    check_multi_token_one_is_single,
    check_multi_token_against_torch_causal,
    check_multi_token_append,
]
