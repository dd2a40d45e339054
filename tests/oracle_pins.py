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
]
