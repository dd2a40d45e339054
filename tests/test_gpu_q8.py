"""int8 KV cache on the GPU, through the C ABI: bulk quantization and the
quantizing append against the oracle's quantizer (bit for bit: every code and
scale), and attention over the int8 cache against the oracle's attention over
the rows read back (the usual tolerances). Shapes cover the head dimensions
and groups from MHA to MQA (above 16 query heads per KV head on the tensor-core
kernel's converting variant, or in several mma.sync CTAs of 16 per token run),
ragged and empty sequences; rows past each
sequence's end hold an invalid code and NaN scales, so any over-read fails.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, Hq, Hkv, D, S, lengths lo..hi, seed
    ("gqa4", 9, 32, 8, 128, 900, 0, 900, 51),
    ("mha64", 5, 6, 6, 64, 400, 1, 400, 52),
    ("g8d256", 4, 16, 2, 256, 300, 1, 300, 53),
    ("g16", 3, 16, 1, 128, 1100, 1, 1100, 54),
    # groups above 16: the tensor-core kernel's converting variant at head_dim
    # 128 and 256 (Q blocks of 48 and, for g64d128, 64 rows); at head_dim 64,
    # and for groups above 48 at 256, several mma.sync CTAs of 16 query heads
    # per token run
    ("mqa48", 4, 48, 1, 256, 700, 1, 700, 56),
    ("g32d128", 5, 64, 2, 128, 600, 0, 600, 57),
    ("g20d64", 3, 20, 1, 64, 520, 1, 520, 58),
    ("g64d128", 3, 64, 1, 128, 500, 1, 500, 59),
    ("g56d256", 2, 56, 1, 256, 300, 1, 300, 60),
    # groups that are not a multiple of 8 (padded Q rows), several KV heads
    ("g20d256", 3, 20, 1, 256, 300, 1, 300, 61),
    ("g24d128kv3", 3, 72, 3, 128, 400, 0, 400, 62),
]


def _oracle_cache(inp):
    """Oracle codes/scales of the cached rows (t < L_b - 1), other rows 0 / NaN."""
    B, S, Hkv, D = inp.k_cache.shape
    out = []
    for c in (inp.k_cache, inp.v_cache):
        codes = np.zeros((B, S, Hkv, D), np.int8)
        scales = np.full((B, S, Hkv), np.nan, np.float32)
        for b in range(B):
            n = max(int(inp.seq_lens[b]) - 1, 0)
            if n:
                codes[b, :n], scales[b, :n] = oracle.quantize_q8(c[b, :n])
        out += [codes, scales]
    return out  # kc, ks, vc, vs


def _gpu_cache(inp, dev):
    """The same, quantized on the GPU from the bf16 cache."""
    import torch
    import kv_cache_decode_gb300 as kvd
    B, S, Hkv, D = inp.k_cache.shape
    cached = torch.from_numpy(np.maximum(inp.seq_lens - 1, 0).astype(np.int32)).to(dev)
    res = []
    for c in (inp.k_cache, inp.v_cache):
        codes = torch.full((B, S, Hkv, D), -128, dtype=torch.int8, device=dev)
        scales = torch.full((B, S, Hkv), float("nan"), dtype=torch.float32, device=dev)
        kvd.kv_quantize_q8(to_dev_bf16(c, dev), codes, scales, cached, S)
        res += [codes, scales]
    return res


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_quantize_matches_oracle(case):
    import torch
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    kc, ks, vc, vs = _gpu_cache(inp, dev)
    torch.cuda.synchronize()
    okc, oks, ovc, ovs = _oracle_cache(inp)
    for b in range(B):
        n = max(int(inp.seq_lens[b]) - 1, 0)
        assert np.array_equal(kc[b, :n].cpu().numpy(), okc[b, :n]) and np.array_equal(vc[b, :n].cpu().numpy(), ovc[b, :n])
        assert np.array_equal(ks[b, :n].cpu().numpy().view(np.uint32), oks[b, :n].view(np.uint32))
        assert np.array_equal(vs[b, :n].cpu().numpy().view(np.uint32), ovs[b, :n].view(np.uint32))
        # rows past the cached ones are untouched
        assert (kc[b, n:].cpu().numpy() == -128).all() and np.isnan(ks[b, n:].cpu().numpy()).all()


def _run(inp, dev, out_dtype, n_split, fused=True):
    import torch
    import kv_cache_decode_gb300 as kvd
    kc, ks, vc, vs = _gpu_cache(inp, dev)
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    S = inp.k_cache.shape[1]
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = kvd.alloc_workspace(q, inp.k_cache, S, n_split, out_dtype)
    if fused:
        kvd.decode_step_q8(q, kc, vc, ks, vs, kn, vn, pos, lens, S, inp.workload.scale, out, workspace=ws,
                           n_split=n_split, lse=lse, status=status)
    else:
        kvd.kv_append_q8(kc, vc, ks, vs, kn, vn, pos, status=status)
        kvd.decode_attention_q8(q, kc, vc, ks, vs, lens, S, inp.workload.scale, out, workspace=ws,
                                n_split=n_split, lse=lse, status=status)
    torch.cuda.synchronize()
    o = bf16_tensor_bits(out) if out_dtype == "bf16" else out.cpu().numpy()
    return (o, lse.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy(),
            int(status.item()))


def _oracle_step(inp):
    kc, ks, vc, vs = _oracle_cache(inp)
    kc, vc, ks, vs, _ = oracle.kv_append_q8(kc, vc, ks, vs, inp.k_new, inp.v_new, inp.pos)
    out, lse = oracle.decode_attention_q8(inp.q, kc, vc, ks, vs, inp.seq_lens, inp.workload.scale)
    return out, lse, kc, vc, ks, vs


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_q8_step_matches_oracle(case, out_dtype):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    want, want_lse, okc, ovc, oks, ovs = _oracle_step(inp)
    for n_split in (0, 7):
        o, l, kc, vc, ks, vs, status = _run(inp, dev, out_dtype, n_split)
        assert status == 0
        for b in range(B):
            n = int(inp.seq_lens[b])
            assert np.array_equal(kc[b, :n], okc[b, :n]) and np.array_equal(vc[b, :n], ovc[b, :n]), "appended codes"
            assert np.array_equal(ks[b, :n].view(np.uint32), oks[b, :n].view(np.uint32)), "appended scales"
        o64 = bf16_bits_to_f32(o).astype(np.float64) if out_dtype == "bf16" else o.astype(np.float64)
        assert_close(o64, want, out_dtype, f"{name} q8 n_split {n_split}")
        finite = np.isfinite(want_lse)
        assert np.max(np.abs(l[finite] - want_lse[finite]), initial=0.0) < (4e-3 if out_dtype == "bf16" else 1e-4)
        assert np.all(np.isneginf(l[~finite]))


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]], ids=["d128", "d256", "mqa48"])
def test_q8_step_equals_two_calls(case):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    a = _run(inp, dev, "f32", 5, fused=True)
    b = _run(inp, dev, "f32", 5, fused=False)
    for x, y, what in zip(a[:6], b[:6], ("out", "lse", "k", "v", "ks", "vs")):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), what
    assert a[6] == b[6] == 0


def test_q8_append_out_of_range():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    inp = workloads.step_inputs(workloads.Workload("app8", 3, 8, 2, 128, 64, 1, 64, 55))
    kc, ks, vc, vs = _gpu_cache(inp, dev)
    pos = inp.pos.copy()
    pos[1] = 64  # past the cache
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kn, vn = to_dev_bf16(inp.k_new, dev), to_dev_bf16(inp.v_new, dev)
    kvd.kv_append_q8(kc, vc, ks, vs, kn, vn, torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    okc, oks, ovc, ovs = _oracle_cache(inp)
    okc, ovc, oks, ovs, skipped = oracle.kv_append_q8(okc, ovc, oks, ovs, inp.k_new, inp.v_new, pos)
    assert skipped == 1 and int(status.item()) == 0x2
    assert np.array_equal(kc.cpu().numpy()[np.isfinite(oks)], okc[np.isfinite(oks)])
    assert np.array_equal(ks.cpu().numpy()[np.isfinite(oks)].view(np.uint32), oks[np.isfinite(oks)].view(np.uint32))
