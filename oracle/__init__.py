"""CPU float64 oracle for single-token decode attention over a KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import this package. The CUDA
path never imports it, and it imports nothing from the CUDA path.

The arithmetic lives in ``kvd_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use and wraps it with ctypes. Inputs are
bf16 bit patterns (uint16 numpy arrays) from the ``workloads`` generators.

Functions and the passages they follow (page title, section):

* ``decode_attention``: softmax over the cached sequence of q . k, times V, per
  query head, with query head n using KV head n // (Hq / Hkv). All About
  Transformer Inference, "Sharding the KV cache" (attention algorithm:
  Reshape, O = Q *_H K, Softmax_S, O *_S V); Efficiently Scaling Transformer
  Inference, section 3.3 (multiquery attention).
* ``decode_attention_chunked``: the same result assembled from per-chunk
  partial softmax states merged by log-sum-exp. All About Transformer
  Inference, "Sharding the KV cache", sequence-sharding bullet (the pages name
  the accumulation but print no formula; the textbook identity is used).
* ``attention_weights``: the softmax weights themselves, for invariant checks.
* ``kv_append``: byte copy of the new token's key/value rows into the cache.
  All About Transformer Inference, "Transformer inference basics" (Generation)
  and "Implementation: JetStream" (generate).
* ``paged_gather``, ``kv_append_paged``, ``decode_attention_paged``: the same
  over a paged cache (a pool of pages of P tokens and a block table: token t
  of sequence b is row t mod P of page table[b, t // P]). All About
  Transformer Inference, "Tricks for improving generation throughput and
  latency", the ragged HBM reads and Paged Attention bullet; the layout is
  this library's reading (the pages give none). Attention over a paged cache
  is attention over the gathered contiguous cache.
* ``quantize_q8``, ``dequantize_q8``, ``kv_append_q8``, ``decode_attention_q8``:
  an int8 cache with one float32 scale per (token, KV head) row, symmetric
  absmax (scale = max|x| / 127, codes = round-half-even(x / scale) in
  float32). All About Transformer Inference, "Tricks for improving
  generation throughput and latency", the quantization bullet names int8 KV
  caches; the scheme is this library's reading. Attention over it is the
  attention above over the rows read back (scale * code), in double.
* ``quantize_fp8``, ``dequantize_fp8``, ``e4m3_encode``, ``e4m3_value``: the
  fp8 cache, the same per-row scheme with the OCP E4M3 format in place of
  int8 (scale = max|x| / 448, code = E4M3(x / scale), round to nearest even,
  saturating, +0 for values that round to zero); the same page names fp8 KV
  caches beside int8. The encoder searches the format's finite values, so it
  follows from the format's definition alone. The 8-bit functions below take
  ``fmt="fp8"`` for it.
* ``paged_gather_q8``, ``kv_append_q8_paged``, ``decode_attention_q8_paged``:
  an int8 cache in page pools (codes [num_pages, P, Hkv, D], scales
  [num_pages, P, Hkv]), the two readings above combined: the page gather and
  paged append move the codes' and scales' bytes exactly as they move bf16
  rows (the same C routines over the bytes), and attention is the int8
  attention over the gathered cache.
* ``decode_attention_unified_max``: FlashDecoding++'s asynchronized softmax
  with a unified maximum (FlashDecoding++ summary page, solution 1: the
  partial softmax results of the splits share one maximum phi and need no
  synchronised update). Each of n_chunks chunks sums exp(s - phi) and
  exp(s - phi) v with no maximum of its own and the chunks are added up; the
  page leaves the out-of-range case open, and here a row with a score outside
  [phi - 64 ln 2, phi + 8 ln 2] is recomputed by ``decode_attention`` and
  reported. Plain numpy, float64.
* ``merge_attention``: attention results of disjoint shards of each
  sequence's tokens (each normalised, with its natural-log normaliser lse)
  combined into the attention over all of them: with L = ln sum_j exp(lse_j),
  out = sum_j exp(lse_j - L) out_j and lse = L (shards with lse = -inf hold
  no token and add nothing). All About Transformer Inference, "Sharding the
  KV cache": sequence-sharded partial results are accumulated as in Flash
  Attention; the identity is the textbook one. Plain numpy, float64.
* ``kv_append_multi``, ``decode_attention_multi``: T new tokens per sequence
  (a speculative-decoding check step): their rows are appended at pos[b] ..
  pos[b] + T - 1, and query token i attends to the cached tokens and the new
  tokens up to itself, i.e. to the first L_b - T + 1 + i tokens (causal).
  All About Transformer Inference, appendix "Speculative Sampling" (the large
  model scores all drafted tokens in one pass over the shared KV cache) and
  "Transformer inference basics" (a token attends to itself and earlier
  tokens). Built on ``decode_attention`` once per query token.

Pins (tests/test_oracle_pins.py): closed forms (identical keys give the mean of
V; a dominant score returns that V row; one token returns it exactly), the
invariants (weights sum to one, token-permutation invariance, chunked equals
direct for every chunk count), cached decoding equal to full causal
recomputation on a toy model, torch's float64 scaled_dot_product_attention on
small shapes, and a 50-digit decimal brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", out, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    return out


def _load(path: Optional[str] = None):
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    Dbl = ctypes.c_double
    lib.kvo_decode_attention.argtypes = [P, P, P, P, I, I, I, I, I, Dbl, P, P, I]
    lib.kvo_decode_attention.restype = I
    lib.kvo_decode_attention_chunked.argtypes = [P, P, P, P, I, I, I, I, I, Dbl, I, P, P]
    lib.kvo_decode_attention_chunked.restype = I
    lib.kvo_attention_weights.argtypes = [P, P, P, I, I, I, I, I, Dbl, I, I, P]
    lib.kvo_attention_weights.restype = I
    lib.kvo_kv_append.argtypes = [P, P, P, P, P, I, I, I, I]
    lib.kvo_kv_append.restype = I
    lib.kvo_paged_gather.argtypes = [P, P, P, I, I, I, I, I, I, P]
    lib.kvo_paged_gather.restype = I
    lib.kvo_kv_append_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
    lib.kvo_kv_append_paged.restype = I
    L = ctypes.c_long
    lib.kvo_quantize_q8.argtypes = [P, L, I, P, P]
    lib.kvo_quantize_q8.restype = I
    lib.kvo_dequantize_q8.argtypes = [P, P, L, I, P]
    lib.kvo_dequantize_q8.restype = I
    lib.kvo_decode_attention_f64kv.argtypes = [P, P, P, P, I, I, I, I, I, Dbl, P, P, I]
    lib.kvo_decode_attention_f64kv.restype = I
    lib.kvo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.kvo_e4m3_encode.restype = I
    lib.kvo_e4m3_value.argtypes = [I]
    lib.kvo_e4m3_value.restype = Dbl
    lib.kvo_quantize_fp8.argtypes = [P, L, I, P, P]
    lib.kvo_quantize_fp8.restype = I
    lib.kvo_dequantize_fp8.argtypes = [P, P, L, I, P]
    lib.kvo_dequantize_fp8.restype = I
    lib.kvo_max_threads.argtypes = []
    lib.kvo_max_threads.restype = I
    return lib


def _u16(a):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _shapes(q, k):
    B, Hq, D = q.shape
    Bk, S_max, Hkv, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q [B,Hq,D] and cache [B,S_max,Hkv,D] disagree")
    return B, S_max, Hq, Hkv, D


def decode_attention(q, k_cache, v_cache, seq_lens, scale, n_threads: int = 0, lib=None):
    """Float64 attention output [B, Hq, D] and natural-log normaliser [B, Hq]."""
    lib = lib or _load()
    B, S_max, Hq, Hkv, D = _shapes(q, k_cache)
    q, qp = _u16(q)
    k_cache, kp = _u16(k_cache)
    v_cache, vp = _u16(v_cache)
    seq_lens, lp = _i32(seq_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = lib.kvo_decode_attention(qp, kp, vp, lp, B, S_max, Hq, Hkv, D, float(scale),
                                  out.ctypes.data_as(ctypes.c_void_p),
                                  lse.ctypes.data_as(ctypes.c_void_p), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle decode_attention failed ({rc})")
    return out, lse


def decode_attention_chunked(q, k_cache, v_cache, seq_lens, scale, n_chunks: int, lib=None):
    """Float64 attention assembled from n_chunks partial softmax states."""
    lib = lib or _load()
    B, S_max, Hq, Hkv, D = _shapes(q, k_cache)
    q, qp = _u16(q)
    k_cache, kp = _u16(k_cache)
    v_cache, vp = _u16(v_cache)
    seq_lens, lp = _i32(seq_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = lib.kvo_decode_attention_chunked(qp, kp, vp, lp, B, S_max, Hq, Hkv, D, float(scale),
                                          int(n_chunks), out.ctypes.data_as(ctypes.c_void_p),
                                          lse.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle decode_attention_chunked failed ({rc})")
    return out, lse


UMAX_WINDOW = (-64.0 * math.log(2.0), 8.0 * math.log(2.0))  # s - phi, natural-log units


def _bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_attention_unified_max(q, k_cache, v_cache, seq_lens, scale, phi, n_chunks: int, lib=None):
    """Unified-maximum attention: (out [B, Hq, D], lse [B, Hq], fell_back [B, Hq]).

    Per (b, h), the L_b scores s_t = scale * q . k_t go to n_chunks contiguous
    chunks of ceil(L_b / n_chunks) tokens; chunk j holds l_j = sum exp(s_t - phi)
    and o_j = sum exp(s_t - phi) v_t, and the row is (sum_j o_j) / (sum_j l_j),
    lse = phi + ln(sum_j l_j). A row with any s_t - phi outside UMAX_WINDOW is
    taken from decode_attention instead and flagged. Empty rows: zeros, -inf.
    """
    B, S_max, Hq, Hkv, D = _shapes(q, k_cache)
    G = Hq // Hkv
    qf, kf, vf = _bf16_f64(q), _bf16_f64(k_cache), _bf16_f64(v_cache)
    lens = np.asarray(seq_lens, dtype=np.int64)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf)
    fell_back = np.zeros((B, Hq), dtype=bool)
    lo, hi = UMAX_WINDOW
    for b in range(B):
        L = int(max(0, min(lens[b], S_max)))
        if L == 0:
            continue
        c = -(-L // n_chunks)
        for h in range(Hq):
            g = h // G
            s = scale * (kf[b, :L, g, :] @ qf[b, h])
            if np.any(s - phi < lo) or np.any(s - phi > hi):
                fell_back[b, h] = True
                continue
            l_sum, o_sum = 0.0, np.zeros(D)
            for j0 in range(0, L, c):
                j1 = min(j0 + c, L)
                w = np.exp(s[j0:j1] - phi)
                l_sum += w.sum()
                o_sum += w @ vf[b, j0:j1, g, :]
            out[b, h] = o_sum / l_sum
            lse[b, h] = phi + math.log(l_sum)
    if fell_back.any():
        ref, ref_lse = decode_attention(q, k_cache, v_cache, seq_lens, scale, lib=lib)
        out[fell_back], lse[fell_back] = ref[fell_back], ref_lse[fell_back]
    return out, lse, fell_back


def merge_attention(outs, lses):
    """(out [..., D], lse [...]) from shard results outs [n, ..., D] and lses [n, ...]."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    if outs.shape[:-1] != lses.shape:
        raise ValueError("outs [n, ..., D] and lses [n, ...] disagree")
    top = np.max(lses, axis=0)
    live = np.isfinite(top)
    shifted = np.where(live, top, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - shifted), 0.0)  # exp(lse_j - max)
    total = w.sum(axis=0)
    out = np.where(live[..., None], np.einsum("n...,n...d->...d", w, outs) / np.where(live, total, 1.0)[..., None],
                   0.0)
    lse = np.where(live, shifted + np.log(np.where(live, total, 1.0)), -np.inf)
    return out, lse


def attention_weights(q, k_cache, seq_lens, scale, b: int, h: int, lib=None):
    """Softmax weights [seq_lens[b]] of query head h of sequence b."""
    lib = lib or _load()
    B, S_max, Hq, Hkv, D = _shapes(q, k_cache)
    q, qp = _u16(q)
    k_cache, kp = _u16(k_cache)
    seq_lens, lp = _i32(seq_lens)
    w = np.zeros(max(int(seq_lens[b]), 1), dtype=np.float64)
    rc = lib.kvo_attention_weights(qp, kp, lp, B, S_max, Hq, Hkv, D, float(scale), int(b), int(h),
                                   w.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle attention_weights failed ({rc})")
    return w[:int(seq_lens[b])]


def kv_append(k_cache, v_cache, k_new, v_new, pos, lib=None):
    """Copies of the caches with each sequence's new row written at pos[b].

    Returns (k_cache', v_cache', n_skipped) where n_skipped counts sequences
    whose pos lay outside [0, S_max) and were left unchanged.
    """
    lib = lib or _load()
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    B, S_max, Hkv, D = kc.shape
    k_new, knp = _u16(k_new)
    v_new, vnp = _u16(v_new)
    pos, pp = _i32(pos)
    rc = lib.kvo_kv_append(kc.ctypes.data_as(ctypes.c_void_p), vc.ctypes.data_as(ctypes.c_void_p),
                           knp, vnp, pp, B, S_max, Hkv, D)
    if rc < 0:
        raise ValueError(f"oracle kv_append failed ({rc})")
    return kc, vc, rc


def paged_gather(pages, block_table, seq_lens, lib=None):
    """Contiguous cache [B, max_blocks * P, Hkv, D] from a pool [num_pages, P, Hkv, D].

    Rows t < seq_lens[b] come from row t % P of page block_table[b, t // P]
    (zero rows where that entry is not a page of the pool); the other rows are
    bf16 NaN. Returns (cache, number of tokens that read zero rows).
    """
    lib = lib or _load()
    pages, pp = _u16(pages)
    num_pages, P, Hkv, D = pages.shape
    block_table, tp = _i32(block_table)
    B, max_blocks = block_table.shape
    seq_lens, lp = _i32(seq_lens)
    out = np.full((B, max_blocks * P, Hkv, D), 0x7FC0, dtype=np.uint16)
    rc = lib.kvo_paged_gather(pp, tp, lp, B, max_blocks, P, num_pages, Hkv, D,
                              out.ctypes.data_as(ctypes.c_void_p))
    if rc < 0:
        raise ValueError(f"oracle paged_gather failed ({rc})")
    return out, rc


def kv_append_paged(k_pages, v_pages, k_new, v_new, block_table, pos, lib=None):
    """Copies of the page pools with each sequence's new row written at pos[b].

    Returns (k_pages', v_pages', n_skipped, n_bad_page): sequences whose pos
    lies outside [0, max_blocks * P) or whose block-table entry is not a page
    of the pool are left out (the latter also counted in n_bad_page).
    """
    lib = lib or _load()
    kp = np.array(k_pages, dtype=np.uint16, copy=True, order="C")
    vp = np.array(v_pages, dtype=np.uint16, copy=True, order="C")
    num_pages, P, Hkv, D = kp.shape
    block_table, tp = _i32(block_table)
    B, max_blocks = block_table.shape
    k_new, knp = _u16(k_new)
    v_new, vnp = _u16(v_new)
    pos, pp = _i32(pos)
    bad = ctypes.c_int(0)
    rc = lib.kvo_kv_append_paged(kp.ctypes.data_as(ctypes.c_void_p), vp.ctypes.data_as(ctypes.c_void_p),
                                 knp, vnp, tp, pp, B, max_blocks, P, num_pages, Hkv, D,
                                 ctypes.byref(bad))
    if rc < 0:
        raise ValueError(f"oracle kv_append_paged failed ({rc})")
    return kp, vp, rc, bad.value


def decode_attention_paged(q, k_pages, v_pages, block_table, seq_lens, scale, n_threads: int = 0,
                           lib=None):
    """decode_attention over the caches gathered from the page pools."""
    kc, _ = paged_gather(k_pages, block_table, seq_lens, lib=lib)
    vc, _ = paged_gather(v_pages, block_table, seq_lens, lib=lib)
    return decode_attention(q, kc, vc, seq_lens, scale, n_threads=n_threads, lib=lib)


def quantize_q8(x, lib=None):
    """int8 codes (same shape) and float32 scales (shape[:-1]) of bf16 rows x[..., D]."""
    lib = lib or _load()
    x, xp = _u16(x)
    D = x.shape[-1]
    rows = x.size // D
    codes = np.zeros(x.shape, dtype=np.int8)
    scales = np.zeros(x.shape[:-1], dtype=np.float32)
    rc = lib.kvo_quantize_q8(xp, rows, D, codes.ctypes.data_as(ctypes.c_void_p),
                             scales.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle quantize_q8 failed ({rc})")
    return codes, scales


def dequantize_q8(codes, scales, lib=None):
    """Rows read back from int8: scales[..., None] * codes, as float64."""
    lib = lib or _load()
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    D = codes.shape[-1]
    if scales.shape != codes.shape[:-1]:
        raise ValueError("scales must have the codes' shape without the last axis")
    out = np.zeros(codes.shape, dtype=np.float64)
    rc = lib.kvo_dequantize_q8(codes.ctypes.data_as(ctypes.c_void_p), scales.ctypes.data_as(ctypes.c_void_p),
                               codes.size // D, D, out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle dequantize_q8 failed ({rc})")
    return out


def quantize_fp8(x, lib=None):
    """fp8 E4M3 codes (uint8, same shape) and float32 scales (shape[:-1]) of bf16
    rows x[..., D]: scale = max|x| / 448, code = E4M3(x / scale) (kvo_e4m3_encode)."""
    lib = lib or _load()
    x, xp = _u16(x)
    D = x.shape[-1]
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[:-1], dtype=np.float32)
    rc = lib.kvo_quantize_fp8(xp, x.size // D, D, codes.ctypes.data_as(ctypes.c_void_p),
                              scales.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle quantize_fp8 failed ({rc})")
    return codes, scales


def dequantize_fp8(codes, scales, lib=None):
    """Rows read back from fp8: scales[..., None] * E4M3 value of codes, as float64."""
    lib = lib or _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    D = codes.shape[-1]
    if scales.shape != codes.shape[:-1]:
        raise ValueError("scales must have the codes' shape without the last axis")
    out = np.zeros(codes.shape, dtype=np.float64)
    rc = lib.kvo_dequantize_fp8(codes.ctypes.data_as(ctypes.c_void_p), scales.ctypes.data_as(ctypes.c_void_p),
                                codes.size // D, D, out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle dequantize_fp8 failed ({rc})")
    return out


def e4m3_encode(y: float, lib=None) -> int:
    """The E4M3 code of one float32 value (round to nearest even, saturating, +0 for zero)."""
    return int((lib or _load()).kvo_e4m3_encode(float(y)))


def e4m3_value(code: int, lib=None) -> float:
    """The value an E4M3 code stands for."""
    return float((lib or _load()).kvo_e4m3_value(int(code)))


# The 8-bit cache formats: code dtype, quantizer, reader.
_FORMATS = {"int8": (np.int8, "quantize_q8", "dequantize_q8"),
            "fp8": (np.uint8, "quantize_fp8", "dequantize_fp8")}


def _fmt(fmt):
    if fmt not in _FORMATS:
        raise ValueError(f"unknown 8-bit cache format {fmt!r}")
    dt, qn, dn = _FORMATS[fmt]
    return dt, globals()[qn], globals()[dn]


def decode_attention_f64kv(q, k_cache, v_cache, seq_lens, scale, n_threads: int = 0, lib=None):
    """decode_attention with float64 caches [B, S_max, Hkv, D] (e.g. rows read back from int8)."""
    lib = lib or _load()
    q, qp = _u16(q)
    k = np.ascontiguousarray(k_cache, dtype=np.float64)
    v = np.ascontiguousarray(v_cache, dtype=np.float64)
    B, Hq, D = q.shape
    Bk, S_max, Hkv, Dk = k.shape
    if Bk != B or Dk != D or v.shape != k.shape:
        raise ValueError("q [B,Hq,D] and caches [B,S_max,Hkv,D] disagree")
    seq_lens, lp = _i32(seq_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = lib.kvo_decode_attention_f64kv(qp, k.ctypes.data_as(ctypes.c_void_p), v.ctypes.data_as(ctypes.c_void_p),
                                        lp, B, S_max, Hq, Hkv, D, float(scale),
                                        out.ctypes.data_as(ctypes.c_void_p),
                                        lse.ctypes.data_as(ctypes.c_void_p), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle decode_attention_f64kv failed ({rc})")
    return out, lse


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, lib=None, fmt="int8"):
    """Copies of an 8-bit cache (codes [B, S_max, Hkv, D], int8 or, fmt "fp8",
    E4M3 as uint8; scales [B, S_max, Hkv]) with each sequence's new bf16 rows
    quantized and written at pos[b]; rows with pos outside [0, S_max) are
    skipped. Returns (kc, vc, ks, vs, n_skipped)."""
    dt, quant, _ = _fmt(fmt)
    kc, vc = np.array(k_codes, dtype=dt, copy=True), np.array(v_codes, dtype=dt, copy=True)
    ks, vs = np.array(k_scales, dtype=np.float32, copy=True), np.array(v_scales, dtype=np.float32, copy=True)
    S_max = kc.shape[1]
    nk, nks = quant(k_new, lib=lib)
    nv, nvs = quant(v_new, lib=lib)
    skipped = 0
    for b, t in enumerate(np.asarray(pos, dtype=np.int64)):
        if t < 0 or t >= S_max:
            skipped += 1
            continue
        kc[b, t], vc[b, t], ks[b, t], vs[b, t] = nk[b], nv[b], nks[b], nvs[b]
    return kc, vc, ks, vs, skipped


def _u16_rows(a, dtype):
    """A C-contiguous array of dtype viewed as rows of 16-bit words (the last
    axis's bytes; a scale array gets a last axis of its one float)."""
    a = np.ascontiguousarray(a, dtype=dtype)
    if dtype == np.float32:
        a = a[..., None]
    return a.view(np.uint16)


def paged_gather_q8(code_pool, scale_pool, block_table, seq_lens, lib=None, fmt="int8"):
    """Contiguous int8 cache (codes [B, max_blocks * P, Hkv, D], scales
    [B, max_blocks * P, Hkv]) from page pools, gathered as paged_gather moves
    bf16 rows: rows t < seq_lens[b] from row t % P of page block_table[b, t // P],
    zero codes and a zero scale where the entry names no page; rows past the
    length are not defined. Returns (codes, scales, tokens that read zero rows)."""
    dt = _fmt(fmt)[0]
    codes, zeroed = paged_gather(_u16_rows(code_pool, dt), block_table, seq_lens, lib=lib)
    scales, _ = paged_gather(_u16_rows(scale_pool, np.float32), block_table, seq_lens, lib=lib)
    return codes.view(dt), scales.view(np.float32)[..., 0], zeroed


def kv_append_q8_paged(k_code_pool, v_code_pool, k_scale_pool, v_scale_pool, k_new, v_new, block_table, pos,
                       lib=None, fmt="int8"):
    """Copies of int8 page pools with each sequence's new bf16 rows quantized
    (quantize_q8) and written at pos[b], as kv_append_paged writes bf16 rows.
    Returns (kc, vc, ks, vs, n_skipped, n_bad_page)."""
    dt, quant, _ = _fmt(fmt)
    nk, nks = quant(k_new, lib=lib)
    nv, nvs = quant(v_new, lib=lib)
    kc, vc, skipped, bad = kv_append_paged(_u16_rows(k_code_pool, dt), _u16_rows(v_code_pool, dt),
                                           _u16_rows(nk, dt), _u16_rows(nv, dt), block_table, pos, lib=lib)
    ks, vs, _, _ = kv_append_paged(_u16_rows(k_scale_pool, np.float32), _u16_rows(v_scale_pool, np.float32),
                                   _u16_rows(nks, np.float32), _u16_rows(nvs, np.float32), block_table, pos,
                                   lib=lib)
    return (kc.view(dt), vc.view(dt), ks.view(np.float32)[..., 0], vs.view(np.float32)[..., 0],
            skipped, bad)


def decode_attention_q8_paged(q, k_code_pool, v_code_pool, k_scale_pool, v_scale_pool, block_table, seq_lens,
                              scale, n_threads: int = 0, lib=None, fmt="int8"):
    """decode_attention_q8 over the 8-bit cache gathered from the page pools."""
    kc, ks, _ = paged_gather_q8(k_code_pool, k_scale_pool, block_table, seq_lens, lib=lib, fmt=fmt)
    vc, vs, _ = paged_gather_q8(v_code_pool, v_scale_pool, block_table, seq_lens, lib=lib, fmt=fmt)
    return decode_attention_q8(q, kc, vc, ks, vs, seq_lens, scale, n_threads=n_threads, lib=lib, fmt=fmt)


def decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, seq_lens, scale, n_threads: int = 0,
                        lib=None, fmt="int8"):
    """Attention over an 8-bit cache (int8, or fmt "fp8": E4M3): the rows read
    back, then decode_attention_f64kv."""
    deq = _fmt(fmt)[2]
    k = deq(k_codes, k_scales, lib=lib)
    v = deq(v_codes, v_scales, lib=lib)
    return decode_attention_f64kv(q, k, v, seq_lens, scale, n_threads=n_threads, lib=lib)


def kv_append_multi(k_cache, v_cache, k_new, v_new, pos, lib=None):
    """Copies of the caches with T new rows per sequence (k_new [B, T, Hkv, D])
    written at pos[b] + i; rows outside [0, S_max) are skipped and counted."""
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    T = k_new.shape[1]
    skipped = 0
    for i in range(T):
        kc, vc, n = kv_append(kc, vc, k_new[:, i], v_new[:, i], np.asarray(pos, np.int64) + i, lib=lib)
        skipped += n
    return kc, vc, skipped


def decode_attention_multi(q, k_cache, v_cache, seq_lens, scale, n_threads: int = 0, lib=None):
    """q [B, T, Hq, D]; query token i of sequence b attends to its first
    max(0, L_b - T + 1 + i) cached tokens. Returns out [B, T, Hq, D], lse [B, T, Hq]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, T, Hq, D = q.shape
    L = np.asarray(seq_lens, dtype=np.int64)
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    lse = np.zeros((B, T, Hq), dtype=np.float64)
    for i in range(T):
        Li = np.clip(L - T + 1 + i, 0, None).astype(np.int32)
        out[:, i], lse[:, i] = decode_attention(q[:, i], k_cache, v_cache, Li, scale, n_threads=n_threads, lib=lib)
    return out, lse


def max_threads(lib=None) -> int:
    lib = lib or _load()
    return int(lib.kvo_max_threads())
