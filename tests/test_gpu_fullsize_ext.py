"""The paged, 8-bit (int8 and fp8) and multi-token paths at the workloads' full sizes, in the
launch configuration the benchmark uses (heuristic split): paged steps
bit-identical to the contiguous steps (which the full-size tests hold to the
oracle), int8 and multi-token steps against the oracle on a sample of whole
sequences."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu


def _step(dev, inp, paged=None):
    import torch
    import kv_cache_decode_gb300 as kvd
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    S = inp.k_cache.shape[1]
    out = torch.full(inp.q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = kvd.alloc_workspace(q, inp.k_cache, S)
    if paged is None:
        kc, vc = to_dev_bf16(inp.k_cache, dev), to_dev_bf16(inp.v_cache, dev)
        kvd.decode_step(q, kc, vc, kn, vn, pos, lens, S, inp.workload.scale, out, workspace=ws, status=status)
    else:
        kp, vp = to_dev_bf16(paged.k_pages, dev), to_dev_bf16(paged.v_pages, dev)
        bt = torch.from_numpy(paged.block_table).to(dev)
        kvd.decode_step_paged(q, kp, vp, kn, vn, pos, bt, lens, S, inp.workload.scale, out, workspace=ws,
                              status=status)
    torch.cuda.synchronize()
    return bf16_tensor_bits(out), int(status.item())


@pytest.mark.parametrize("name,page", [("palm", 64), ("palm", 16), ("long", 64), ("gqa", 16), ("mha", 64)])
def test_paged_full_size_equals_contiguous(name, page):
    dev = cuda_or_skip()
    inp = workloads.step_inputs(workloads.get(name))
    ref, st0 = _step(dev, inp)
    got, st1 = _step(dev, inp, workloads.paged_step_inputs(inp, page, seed=page))
    assert st0 == st1 == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name", ["gqa", "palm"])
@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_8bit_full_size(name, fmt):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.get(name)
    inp = workloads.step_inputs(w)
    B, S, Hkv, D = inp.k_cache.shape
    fp8 = fmt == "fp8"
    cached = torch.from_numpy(np.maximum(inp.seq_lens - 1, 0).astype(np.int32)).to(dev)
    dev_q8 = []
    for c in (inp.k_cache, inp.v_cache):
        codes = torch.full((B, S, Hkv, D), 0x7F if fp8 else -128, dtype=torch.uint8 if fp8 else torch.int8,
                           device=dev)
        scales = torch.full((B, S, Hkv), float("nan"), dtype=torch.float32, device=dev)
        (kvd.kv_quantize_fp8 if fp8 else kvd.kv_quantize_q8)(to_dev_bf16(c, dev), codes, scales, cached, S)
        dev_q8 += [codes, scales]
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    out = torch.full(inp.q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = kvd.alloc_workspace(q, inp.k_cache, S)
    kvd.decode_ex(q, dev_q8[0], dev_q8[2], torch.from_numpy(inp.seq_lens).to(dev), S, w.scale, out,
                  k_scales=dev_q8[1], v_scales=dev_q8[3], k_new=kn, v_new=vn, pos=torch.from_numpy(inp.pos).to(dev),
                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = bf16_bits_to_f32(bf16_tensor_bits(out)).astype(np.float64)
    L = inp.seq_lens
    quant = oracle.quantize_fp8 if fp8 else oracle.quantize_q8
    cdt = np.uint8 if fp8 else np.int8
    rows = sorted({int(np.argmin(L)), int(np.argmax(L)), 17, B - 1})
    for b in rows:
        n = int(L[b]) - 1
        kc = np.zeros((1, S, Hkv, D), cdt)
        vc = np.zeros((1, S, Hkv, D), cdt)
        ks = np.zeros((1, S, Hkv), np.float32)
        vs = np.zeros((1, S, Hkv), np.float32)
        kc[0, :n], ks[0, :n] = quant(inp.k_cache[b, :n])
        vc[0, :n], vs[0, :n] = quant(inp.v_cache[b, :n])
        kc, vc, ks, vs, _ = oracle.kv_append_q8(kc, vc, ks, vs, inp.k_new[b:b + 1], inp.v_new[b:b + 1],
                                                inp.pos[b:b + 1], fmt=fmt)
        want, _ = oracle.decode_attention_q8(inp.q[b:b + 1], kc, vc, ks, vs, L[b:b + 1], w.scale, fmt=fmt)
        assert_close(got[b:b + 1], want, "bf16", f"{name} {fmt} row {b}")


@pytest.mark.parametrize("name,T", [("gqa", 4), ("mha", 16), ("gqa", 8), ("palm", 2)])
def test_multi_token_full_size(name, T):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.get(name)
    mi = workloads.multi_step_inputs(w, T)
    B, _, Hq, D = mi.q.shape
    S, Hkv = mi.k_cache.shape[1], mi.k_cache.shape[2]
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_cache, mi.v_cache, mi.k_new, mi.v_new))
    out = torch.full(mi.q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    kvd.decode_step_multi(q, kc, vc, kn, vn, torch.from_numpy(mi.pos).to(dev), torch.from_numpy(mi.seq_lens).to(dev),
                          S, w.scale, out, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = bf16_bits_to_f32(bf16_tensor_bits(out)).astype(np.float64)
    L = mi.seq_lens
    rows = sorted({int(np.argmin(L)), int(np.argmax(L)), 3})
    for b in rows:
        kcb, vcb, _ = oracle.kv_append_multi(mi.k_cache[b:b + 1], mi.v_cache[b:b + 1], mi.k_new[b:b + 1],
                                             mi.v_new[b:b + 1], mi.pos[b:b + 1])
        want, _ = oracle.decode_attention_multi(mi.q[b:b + 1], kcb, vcb, L[b:b + 1], w.scale)
        assert_close(got[b:b + 1].reshape(1, T * Hq, D), want.reshape(1, T * Hq, D), "bf16", f"{name} T{T} row {b}")
