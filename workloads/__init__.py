"""Seeded synthetic workloads for single-token decode attention over a KV cache.

This module only draws and lays out numbers: it holds none of the attention
arithmetic. The CUDA path and the CPU oracle both take their inputs from here,
and nothing else is shared between them.

Shapes follow the pages' workloads:

* ``palm``: PaLM-540B-style multiquery decode step, one layer. 48 query heads
  share one KV head of width 256 (Efficiently Scaling Transformer Inference,
  Table D.1), batch 64, context 2048 (same paper, abstract and Table 2).
* ``mha``: LLaMA-2-13B-style multi-head decode step, 40 query heads and 40 KV
  heads of width 128 (How to Parallelize a Transformer for Training, section
  "Some Problems to Work", hyper-parameter table), ragged contexts.
* ``gqa``: grouped-query decode step, 32 query heads over 8 KV heads (All About
  Transformer Inference, "Tricks for improving generation throughput and
  latency", the LLaMA-3 8B example), ragged contexts, with 1 % of key rows
  scaled by 8 so that the softmax is peaked.
* ``long``: multiquery decode with a 32x longer context (Efficiently Scaling
  Transformer Inference, Table 1), plus 16 trials of ragged lengths.
* ``tiny``: one sequence, 8 query heads over one KV head, context 256.

Recipe
------
Every tensor value is a float32 draw from numpy's PCG64 standard normal,
rounded to bfloat16 with round-to-nearest-even. Each tensor of each sequence
has its own stream, keyed by ``(seed, tag, sequence index)``, so any subset of
a batch can be regenerated alone, bit for bit. Context lengths are drawn from
``integers(lo, hi, endpoint=True)`` on a stream keyed by ``(seed, tag)``.

"Context L" is the attended length *after* the new token is appended: the
cache holds ``L - 1`` prefilled tokens, the new token's key and value go to
slot ``L - 1``, and attention then covers ``L`` tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Iterable, List, Optional

import numpy as np

# Stream tags.
_TAG_LEN, _TAG_Q, _TAG_K, _TAG_V, _TAG_KMASK, _TAG_QM = 0, 1, 2, 3, 4, 5

#: bf16 quiet NaN. Cache slots past a sequence's length are filled with it in
#: tests, so that any read beyond the valid length poisons the result.
BF16_NAN = 0x7FC0


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    S_max: int
    len_lo: int  # attended context length (after append), inclusive bounds
    len_hi: int
    seed: int
    peaked_frac: float = 0.0  # fraction of key rows multiplied by peaked_mult
    peaked_mult: float = 8.0
    description: str = ""

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D), as the float32 value the kernels receive."""
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def with_batch(self, B: int) -> "Workload":
        return replace(self, B=B)


def _w(name, B, Hq, Hkv, D, S_max, lo, hi, seed, **kw) -> Workload:
    return Workload(name, B, Hq, Hkv, D, S_max, lo, hi, seed, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": _w("tiny", 1, 8, 1, 128, 256, 256, 256, 1,
               description="tiny MQA decode: B 1, 8 q heads / 1 kv head, D 128, L 256"),
    "palm": _w("palm", 64, 48, 1, 256, 2048, 2048, 2048, 2,
               description="PaLM-540B-style MQA decode, one layer: B 64, 48q/1kv, D 256, L 2048"),
    "mha": _w("mha", 32, 40, 40, 128, 4096, 512, 4096, 3,
              description="LLaMA-2-13B-style MHA decode, one layer: B 32, 40q/40kv, D 128, L~U[512,4096]"),
    "gqa": _w("gqa", 128, 32, 8, 128, 8192, 1024, 8192, 4, peaked_frac=0.01,
              description="GQA decode, one layer: B 128, 32q/8kv, D 128, L~U[1024,8192], 1% keys x8"),
    "long": _w("long", 4, 48, 1, 256, 65536, 65536, 65536, 5,
               description="long-context MQA decode: B 4, 48q/1kv, D 256, L 65536"),
}


def long_trial(i: int) -> Workload:
    """One of the 16 ragged long-context trials: lengths U[1, 131072]."""
    if not 0 <= i < 16:
        raise ValueError("trial index must be in [0, 16)")
    return _w(f"long_trial{i}", 4, 48, 1, 256, 131072, 1, 131072, 500 + i,
              description=f"long-context MQA trial {i}: B 4, 48q/1kv, D 256, L~U[1,131072]")


def get(name: str) -> Workload:
    if name.startswith("long_trial"):
        return long_trial(int(name[len("long_trial"):]))
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
# bf16 <-> f32 bit conversion (data preparation only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the bf16 bit patterns as uint16. Inputs here are finite normals, so
    no NaN/Inf special case is needed; it is still handled for safety.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # No finite value (nor infinity) overflows 32 bits here: |x| <= 0x7F800000.
    r = (u >> 16) & np.uint32(1)
    r += u
    r += np.uint32(0x7FFF)
    r >>= 16
    rounded = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded[nan] = BF16_NAN
    return rounded


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Streams
# ---------------------------------------------------------------------------

def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def seq_lens(w: Workload) -> np.ndarray:
    """Attended context length of every sequence (int32[B])."""
    if w.len_lo == w.len_hi:
        return np.full(w.B, w.len_lo, dtype=np.int32)
    r = _rng(w.seed, _TAG_LEN)
    return r.integers(w.len_lo, w.len_hi, size=w.B, endpoint=True).astype(np.int32)


def query(w: Workload, b: int) -> np.ndarray:
    """bf16 bits of sequence b's query, [Hq, D]."""
    r = _rng(w.seed, _TAG_Q, b)
    return f32_to_bf16_bits(r.standard_normal((w.Hq, w.D), dtype=np.float32))


def kv_rows(w: Workload, b: int, L: int):
    """bf16 bits of sequence b's first L key and value rows, each [L, Hkv, D].

    Row L-1 is the token appended by this decode step; rows 0..L-2 are the
    prefilled cache. For peaked workloads a Bernoulli(peaked_frac) draw per
    (token, kv head) multiplies that whole key row by peaked_mult before
    rounding (a power of two, so exact in bf16).
    """
    rk = _rng(w.seed, _TAG_K, b)
    rv = _rng(w.seed, _TAG_V, b)
    k = rk.standard_normal((L, w.Hkv, w.D), dtype=np.float32)
    v = rv.standard_normal((L, w.Hkv, w.D), dtype=np.float32)
    if w.peaked_frac > 0.0:
        rm = _rng(w.seed, _TAG_KMASK, b)
        mask = rm.random((L, w.Hkv)) < w.peaked_frac
        k[mask] *= np.float32(w.peaked_mult)
    return f32_to_bf16_bits(k), f32_to_bf16_bits(v)


@dataclass
class StepInputs:
    """Host arrays for one decode step (bf16 tensors as uint16 bit patterns).

    ``k_cache``/``v_cache`` hold the cache *before* the append: slots
    ``t < seq_lens[b] - 1`` are data, the rest are ``pad_bits``. The new token's
    key/value (``k_new``/``v_new``) go to slot ``pos[b] = seq_lens[b] - 1``.
    """
    workload: Workload
    batch_index: np.ndarray  # which sequences of the workload these rows are
    q: np.ndarray            # u16 [B, Hq, D]
    k_cache: np.ndarray      # u16 [B, S_max, Hkv, D]
    v_cache: np.ndarray
    k_new: np.ndarray        # u16 [B, Hkv, D]
    v_new: np.ndarray
    pos: np.ndarray          # i32 [B]
    seq_lens: np.ndarray     # i32 [B] attended length after append
    extra: dict = field(default_factory=dict)


def step_inputs(w: Workload, batch_index: Optional[Iterable[int]] = None,
                pad_bits: int = BF16_NAN, lens: Optional[np.ndarray] = None,
                S_max: Optional[int] = None) -> StepInputs:
    """Build the host-side inputs of one decode step.

    ``batch_index`` selects a subset of the workload's sequences (default: all).
    ``lens`` overrides the drawn context lengths (used by edge-case tests).
    """
    all_lens = seq_lens(w) if lens is None else np.asarray(lens, dtype=np.int32)
    idx = np.arange(w.B) if batch_index is None else np.asarray(list(batch_index), dtype=np.int64)
    S = w.S_max if S_max is None else S_max
    B = len(idx)
    L = all_lens[idx].astype(np.int32)
    if (L < 0).any() or (L > S).any():
        raise ValueError("context lengths must lie in [0, S_max]")
    q = np.empty((B, w.Hq, w.D), dtype=np.uint16)
    kc = np.full((B, S, w.Hkv, w.D), pad_bits, dtype=np.uint16)
    vc = np.full((B, S, w.Hkv, w.D), pad_bits, dtype=np.uint16)
    kn = np.zeros((B, w.Hkv, w.D), dtype=np.uint16)
    vn = np.zeros((B, w.Hkv, w.D), dtype=np.uint16)
    for i, b in enumerate(idx):
        q[i] = query(w, int(b))
        Lb = int(L[i])
        if Lb == 0:
            continue
        k, v = kv_rows(w, int(b), Lb)
        kc[i, :Lb - 1] = k[:Lb - 1]
        vc[i, :Lb - 1] = v[:Lb - 1]
        kn[i] = k[Lb - 1]
        vn[i] = v[Lb - 1]
    pos = np.maximum(L - 1, 0).astype(np.int32)
    return StepInputs(w, idx, q, kc, vc, kn, vn, pos, L)


def random_small(seed: int, B: int, Hq: int, Hkv: int, D: int, S_max: int,
                 lens: List[int], peaked_frac: float = 0.0) -> StepInputs:
    """A small ad-hoc workload with explicit lengths (brute-force and edge cases)."""
    w = Workload(f"small{seed}", B, Hq, Hkv, D, S_max, 0, S_max, seed,
                 peaked_frac=peaked_frac)
    return step_inputs(w, lens=np.asarray(lens, dtype=np.int32))


@dataclass
class PagedStepInputs:
    """One decode step over a paged cache (bf16 tensors as uint16 bit patterns).

    ``k_pages``/``v_pages`` are pools of ``page_size``-token pages laid out like
    a cache of that capacity; ``block_table[b, j]`` names the page holding
    tokens ``[j * page_size, (j + 1) * page_size)`` of sequence b, or -1 where
    the sequence has no such block. ``step`` holds the same step in contiguous
    form (its q, new rows, pos and lengths apply unchanged).
    """
    step: StepInputs
    page_size: int
    k_pages: np.ndarray      # u16 [num_pages, page_size, Hkv, D]
    v_pages: np.ndarray
    block_table: np.ndarray  # i32 [B, max_blocks]


def paged_step_inputs(inp: StepInputs, page_size: int, seed: int = 0, spare: int = 3,
                      pad_bits: int = BF16_NAN, shuffle: bool = True) -> PagedStepInputs:
    """Spread a step's cache over a shuffled pool of pages.

    Each sequence gets the ceil(L_b / page_size) blocks its attended length
    needs (the appended token's slot included; one block for an empty
    sequence, whose placeholder new row goes to slot 0), placed on pages drawn in a
    random order from a pool with ``spare`` extra pages; unused pages and the
    rows past each sequence's cached tokens hold ``pad_bits``. With
    ``shuffle=False`` the pages are taken in order (each sequence's pages
    consecutive in the pool). A layout only: page j of sequence b receives
    rows [j * P, (j + 1) * P) of its cache.
    """
    P = int(page_size)
    B, S, Hkv, D = inp.k_cache.shape
    max_blocks = -(-S // P)
    nblk = [max(1, -(-int(L) // P)) for L in inp.seq_lens]
    num_pages = sum(nblk) + spare
    order = np.random.default_rng((seed, P, B)).permutation(num_pages) if shuffle else np.arange(num_pages)
    kp = np.full((num_pages, P, Hkv, D), pad_bits, dtype=np.uint16)
    vp = np.full((num_pages, P, Hkv, D), pad_bits, dtype=np.uint16)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for j in range(nblk[b]):
            page = int(order[nxt])
            nxt += 1
            table[b, j] = page
            rows = inp.k_cache[b, j * P:(j + 1) * P]
            kp[page, :rows.shape[0]] = rows
            vp[page, :rows.shape[0]] = inp.v_cache[b, j * P:(j + 1) * P]
    return PagedStepInputs(inp, P, kp, vp, table)


@dataclass
class MultiStepInputs:
    """One multi-token step: T new tokens per sequence (bf16 bits).

    The cache holds the first ``seq_lens[b] - T`` rows; the T new rows
    (``k_new``/``v_new`` [B, T, Hkv, D]) go to ``pos[b] = seq_lens[b] - T``
    onward, and ``q`` [B, T, Hq, D] holds the T queries.
    """
    workload: Workload
    T: int
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    pos: np.ndarray
    seq_lens: np.ndarray


def multi_step_inputs(w: Workload, T: int, lens: Optional[np.ndarray] = None,
                      pad_bits: int = BF16_NAN) -> MultiStepInputs:
    """A step with T new tokens per sequence: lengths drawn as for the
    workload (or ``lens``), each at least T; the last T rows of each sequence's
    key/value draw are the new tokens, and its T queries come from a stream of
    their own."""
    L = (seq_lens(w) if lens is None else np.asarray(lens, dtype=np.int32)).astype(np.int32)
    if (L < T).any() or (L > w.S_max).any():
        raise ValueError("lengths must lie in [T, S_max]")
    B = w.B
    q = np.empty((B, T, w.Hq, w.D), dtype=np.uint16)
    kc = np.full((B, w.S_max, w.Hkv, w.D), pad_bits, dtype=np.uint16)
    vc = np.full((B, w.S_max, w.Hkv, w.D), pad_bits, dtype=np.uint16)
    kn = np.zeros((B, T, w.Hkv, w.D), dtype=np.uint16)
    vn = np.zeros((B, T, w.Hkv, w.D), dtype=np.uint16)
    for b in range(B):
        r = _rng(w.seed, _TAG_QM, b)
        q[b] = f32_to_bf16_bits(r.standard_normal((T, w.Hq, w.D), dtype=np.float32))
        Lb = int(L[b])
        k, v = kv_rows(w, b, Lb)
        kc[b, :Lb - T], vc[b, :Lb - T] = k[:Lb - T], v[:Lb - T]
        kn[b], vn[b] = k[Lb - T:], v[Lb - T:]
    return MultiStepInputs(w, T, q, kc, vc, kn, vn, (L - T).astype(np.int32), L)
