"""Byte and FLOP model of the decode step, used for the roofline numbers.

Pure host arithmetic (no GPU, no torch). Pinned by tests against the worked
numbers the pages print.

* KV-cache bytes per token: 2 (key and value) x layers x KV heads x head dim x
  bytes per element (All About Transformer Inference, "What about memory?";
  the worked answer in "Worked problems", question 1, gives 262,144 bytes for
  64 layers, 8 KV heads, head dim 256 in int8).
* Decode attention is bound by HBM bandwidth: each generated token reads the
  whole valid KV cache once while doing a constant, small number of FLOPs per
  byte (All About Transformer Inference, "What about attention?";
  Efficiently Scaling Transformer Inference, section 2, "Memory costs").
"""
from __future__ import annotations

from typing import Iterable

import numpy as np


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """Bytes of key plus value cache one token occupies across all layers."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def kv_cache_bytes(tokens: int, n_layers: int, n_kv_heads: int, head_dim: int,
                   bytes_per_elem: float) -> float:
    return tokens * kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_elem)


def max_context(memory_bytes: float, batch: int, per_token_bytes: float) -> int:
    """Longest context whose KV cache for `batch` sequences fits in memory_bytes."""
    return int(memory_bytes // (batch * per_token_bytes))


def attention_kv_bytes(seq_lens: Iterable[int], n_heads_kv: int, head_dim: int,
                       bytes_per_elem: int = 2) -> int:
    """Bytes of K and V one decode step must read: sum_b L_b * Hkv * D * 2 * elem."""
    total_tokens = int(np.sum(np.asarray(list(seq_lens), dtype=np.int64)))
    return total_tokens * n_heads_kv * head_dim * 2 * bytes_per_elem


def attention_step_bytes(seq_lens: Iterable[int], n_heads_q: int, n_heads_kv: int,
                         head_dim: int, bytes_per_elem: int = 2) -> int:
    """Algorithmic bytes of one decode-attention launch: the valid K/V rows,
    plus reading q and writing the output (each [B, Hq, D] in bf16).
    Workspace traffic for split partials is overhead and not counted."""
    lens = np.asarray(list(seq_lens), dtype=np.int64)
    B = int(lens.size)
    return (attention_kv_bytes(lens, n_heads_kv, head_dim, bytes_per_elem)
            + 2 * B * n_heads_q * head_dim * bytes_per_elem)


def attention_step_bytes_q8(seq_lens: Iterable[int], n_heads_q: int, n_heads_kv: int, head_dim: int) -> int:
    """attention_step_bytes for an int8 cache: each valid K and V row is head_dim
    one-byte codes plus one float32 scale; q in and the output out stay bf16."""
    lens = np.asarray(list(seq_lens), dtype=np.int64)
    B = int(lens.size)
    return int(lens.sum()) * n_heads_kv * (head_dim + 4) * 2 + 2 * B * n_heads_q * head_dim * 2


def append_bytes(batch: int, n_heads_kv: int, head_dim: int, bytes_per_elem: int = 2) -> int:
    """Algorithmic bytes of one append: read k_new and v_new, write two cache rows."""
    return 4 * batch * n_heads_kv * head_dim * bytes_per_elem


def attention_step_flops(seq_lens: Iterable[int], n_heads_q: int, head_dim: int) -> int:
    """2*D FLOPs for q.k plus 2*D for p*v, per query head and attended token."""
    total_tokens = int(np.sum(np.asarray(list(seq_lens), dtype=np.int64)))
    return 4 * n_heads_q * head_dim * total_tokens
