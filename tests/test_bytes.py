"""The byte model against the worked KV-cache sizes printed on the pages."""
import os

import pytest

from kv_cache_decode_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizes.txt")
TPU_V4_HBM = 32 * 2**30          # Efficiently Scaling Transformer Inference, section 4 setup
KV_FRACTION = 0.30               # Table 1 caption: 30 % of memory reserved for the KV cache
PALM_LAYERS = 118                # Table D.1


def _cases():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, fn, args, expected, tol = (x.strip() for x in line.split("|"))
        kw = {k: float(v) for k, v in (a.split("=") for a in args.split(","))}
        out.append((name, fn, kw, float(expected), float(tol)))
    return out


def _eval(fn, kw):
    if fn == "kv_bytes_per_token":
        return roofline.kv_bytes_per_token(int(kw["n_layers"]), int(kw["n_kv_heads"]),
                                           int(kw["head_dim"]), kw["bytes_per_elem"])
    if fn == "kv_cache_bytes":
        return roofline.kv_cache_bytes(int(kw["tokens"]), int(kw["n_layers"]),
                                       int(kw["n_kv_heads"]), int(kw["head_dim"]),
                                       kw["bytes_per_elem"])
    if fn == "max_context_esti":
        mem = kw["chips"] * TPU_V4_HBM * KV_FRACTION
        per_tok = roofline.kv_bytes_per_token(PALM_LAYERS, int(kw["kv_heads"]),
                                              int(kw["head_dim"]), 2)
        return roofline.max_context(mem, int(kw["batch"]), per_tok)
    raise KeyError(fn)


@pytest.mark.parametrize("name,fn,kw,expected,tol", _cases(), ids=[c[0] for c in _cases()])
def test_worked_sizes(name, fn, kw, expected, tol):
    got = _eval(fn, kw)
    if tol == 0:
        assert got == expected
    else:
        assert abs(got - expected) <= tol * expected, (got, expected)


def test_llama2_13b_four_sequences_exceed_params():
    """All About Transformer Inference, "What about memory?": for LLaMA-2-13B in
    bf16 a single 8192-token sequence's KV cache is so large that four of them
    outweigh the 26 GB of bf16 parameters (40 layers, 40 KV heads of 128:
    How to Parallelize a Transformer for Training, "Some Problems to Work")."""
    per_seq = roofline.kv_cache_bytes(8192, 40, 40, 128, 2)
    assert 3 * per_seq < 26e9 < 4 * per_seq
    assert abs(per_seq - 6.71e9) < 0.01e9


def test_step_bytes_and_flops():
    lens = [3, 0, 5]
    # 8 tokens * Hkv 2 * D 4 * (K and V) * 2 bytes = 256, plus q and out: 2*3*4*4*2 = 192
    assert roofline.attention_kv_bytes(lens, 2, 4) == 256
    assert roofline.attention_step_bytes(lens, 4, 2, 4) == 256 + 192
    assert roofline.attention_step_flops(lens, 4, 4) == 4 * 4 * 4 * 8
    assert roofline.append_bytes(3, 2, 4) == 4 * 3 * 2 * 4 * 2


def test_step_bytes_int8():
    # Two sequences of 3 and 5 tokens, 2 KV heads of width 64, 8 query heads:
    # 8 tokens x 2 heads x (64 codes + 4 scale bytes) x 2 (K, V), plus q and out in bf16.
    got = roofline.attention_step_bytes_q8([3, 5], 8, 2, 64)
    assert got == 8 * 2 * 68 * 2 + 2 * 2 * 8 * 64 * 2
    # against the bf16 count: the cache part shrinks to (D + 4) / (2 D)
    bf = roofline.attention_kv_bytes([3, 5], 2, 64)
    assert got - 2 * 2 * 8 * 64 * 2 == bf * (64 + 4) // (2 * 64)
