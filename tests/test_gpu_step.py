"""kvd_decode_step (append + attention in one call) against the two calls it
stands for, kvd_kv_append then kvd_decode_attention, and against the oracle.

The step starts its attention launch while the append runs and only its
cache loads wait for the append, so these tests check that the new token's
row is always seen: the outputs must be bit-identical to the two-call
sequence (same kernels, same schedule), the caches identical, and both within
the usual tolerance of the oracle. Shapes cover both engines (tcgen05 for the
wide MQA group, mma.sync for GQA), split and unsplit pairs, ragged and empty
sequences, and the new row at the end of a sequence, in its middle and past
the attended range.
"""
import numpy as np
import pytest

import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, oracle_step, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu


def _run(inp, dev, out_dtype, n_split, fused, pos=None, lens=None):
    import torch
    import kv_cache_decode_gb300 as kvd
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_cache, inp.v_cache, inp.k_new, inp.v_new))
    pos_t = torch.from_numpy(inp.pos if pos is None else pos).to(dev)
    lens_t = torch.from_numpy(inp.seq_lens if lens is None else lens).to(dev)
    S = inp.k_cache.shape[1]
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    ws = kvd.alloc_workspace(q, kc, S, n_split, out_dtype)
    scale = inp.workload.scale
    if fused:
        kvd.decode_step(q, kc, vc, kn, vn, pos_t, lens_t, S, scale, out, workspace=ws, n_split=n_split, lse=lse)
    else:
        kvd.kv_append(kc, vc, kn, vn, pos_t)
        kvd.decode_attention(q, kc, vc, lens_t, S, scale, out, workspace=ws, n_split=n_split, lse=lse)
    torch.cuda.synchronize()
    o = bf16_tensor_bits(out) if out_dtype == "bf16" else out.cpu().numpy()
    return o, lse.cpu().numpy(), bf16_tensor_bits(kc), bf16_tensor_bits(vc)


CASES = [
    # name, B, Hq, Hkv, D, S, lengths lo..hi, seed
    ("mqa48", 8, 48, 1, 256, 1024, 1024, 1024, 21),   # tcgen05, split pairs
    ("mqa48r", 9, 48, 1, 256, 700, 1, 700, 22),       # tcgen05, ragged
    ("gqa4", 16, 32, 8, 128, 1500, 1, 1500, 23),      # mma.sync, ragged
    ("mha", 6, 8, 8, 64, 300, 1, 300, 24),            # mma.sync, head_dim 64
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_split", [0, 1, 7])
def test_step_matches_two_calls(case, out_dtype, n_split):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    w = workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed)
    inp = workloads.step_inputs(w)
    ref = _run(inp, dev, out_dtype, n_split, fused=False)
    got = _run(inp, dev, out_dtype, n_split, fused=True)
    for a, b, what in zip(got, ref, ("out", "lse", "k_cache", "v_cache")):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), f"{name} {what}"
    o = got[0]
    o64 = bf16_bits_to_f32(o).astype(np.float64) if out_dtype == "bf16" else o.astype(np.float64)
    assert_close(o64, oracle_step(inp)[0], out_dtype, f"{name} step vs oracle")


def test_step_new_row_anywhere():
    """pos inside the attended range (middle of the sequence), at its end, and
    past it (written to the cache but not attended)."""
    dev = cuda_or_skip()
    w = workloads.Workload("mqa_pos", 6, 48, 1, 256, 512, 300, 300, 31)
    inp = workloads.step_inputs(w)
    pos = np.array([5, 299, 100, 350, 0, 511], dtype=np.int32)
    for engine_case in (inp,):
        ref = _run(engine_case, dev, "f32", 5, fused=False, pos=pos)
        got = _run(engine_case, dev, "f32", 5, fused=True, pos=pos)
        for a, b, what in zip(got, ref, ("out", "lse", "k_cache", "v_cache")):
            assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), what
    w2 = workloads.Workload("gqa_pos", 6, 16, 4, 128, 512, 300, 300, 32)
    inp2 = workloads.step_inputs(w2)
    ref = _run(inp2, dev, "f32", 5, fused=False, pos=pos)
    got = _run(inp2, dev, "f32", 5, fused=True, pos=pos)
    for a, b, what in zip(got, ref, ("out", "lse", "k_cache", "v_cache")):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), what


def test_step_empty_batch_members():
    dev = cuda_or_skip()
    w = workloads.Workload("mqa_empty", 5, 48, 1, 256, 256, 0, 256, 33)
    inp = workloads.step_inputs(w)
    lens = np.array([0, 256, 0, 17, 0], dtype=np.int32)
    ref = _run(inp, dev, "bf16", 0, fused=False, lens=lens)
    got = _run(inp, dev, "bf16", 0, fused=True, lens=lens)
    for a, b, what in zip(got, ref, ("out", "lse", "k_cache", "v_cache")):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), what
