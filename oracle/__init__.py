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

Pins (tests/test_oracle_pins.py): closed forms (identical keys give the mean of
V; a dominant score returns that V row; one token returns it exactly), the
invariants (weights sum to one, token-permutation invariance, chunked equals
direct for every chunk count), cached decoding equal to full causal
recomputation on a toy model, torch's float64 scaled_dot_product_attention on
small shapes, and a 50-digit decimal brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
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


def max_threads(lib=None) -> int:
    lib = lib or _load()
    return int(lib.kvo_max_threads())
