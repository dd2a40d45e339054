"""kvd_decode_ex, the one entry point for feature combinations: each form it
shares with a dedicated call is bit-identical to that call, and the
combinations with no dedicated call (paged multi-token, int8 multi-token) are
checked against the contiguous multi-token call (bit for bit) or the oracle."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16

pytestmark = pytest.mark.gpu


def _ws(kvd, torch, B, T, Hq, Hkv, D, S, dev, out_dtype="bf16"):
    _, n = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, 0, out_dtype)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("page,Hq,Hkv,D,T", [(16, 32, 8, 128, 4), (64, 32, 8, 128, 4), (32, 48, 1, 256, 2)],
                         ids=["p16_g4t4", "p64_g4t4", "p32_mqa48t2"])
def test_paged_multi_equals_contiguous_multi(page, Hq, Hkv, D, T):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("pm", 6, Hq, Hkv, D, 700, T, 700, 71)
    mi = workloads.multi_step_inputs(w, T)
    B, _, Hq, D = mi.q.shape
    S, Hkv = mi.k_cache.shape[1], mi.k_cache.shape[2]
    q, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_new, mi.v_new))
    pos = torch.from_numpy(mi.pos).to(dev)
    lens = torch.from_numpy(mi.seq_lens).to(dev)
    # contiguous reference
    kc, vc = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
    ref = torch.empty(mi.q.shape, dtype=torch.bfloat16, device=dev)
    kvd.decode_step_multi(q, kc, vc, kn, vn, pos, lens, S, w.scale, ref, workspace=_ws(kvd, torch, B, T, Hq, Hkv, D, S, dev))
    # paged: the same rows on shuffled pages (the step inputs' lengths give each sequence its blocks)
    pin = workloads.paged_step_inputs(workloads.StepInputs(w, np.arange(B), mi.q[:, 0], mi.k_cache, mi.v_cache,
                                                           mi.k_new[:, 0], mi.v_new[:, 0], mi.pos, mi.seq_lens),
                                      page, seed=page)
    kp, vp = to_dev_bf16(pin.k_pages, dev), to_dev_bf16(pin.v_pages, dev)
    bt = torch.from_numpy(pin.block_table).to(dev)
    got = torch.empty(mi.q.shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.decode_ex(q, kp, vp, lens, S, w.scale, got, block_table=bt, k_new=kn, v_new=vn, pos=pos,
                  workspace=_ws(kvd, torch, B, T, Hq, Hkv, D, S, dev), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bf16_tensor_bits(got), bf16_tensor_bits(ref))


@pytest.mark.parametrize("Hq,Hkv,D,T", [(16, 4, 128, 3), (48, 1, 256, 2)], ids=["g4t3", "mqa48t2"])
def test_int8_multi_matches_oracle(Hq, Hkv, D, T):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("qm", 5, Hq, Hkv, D, 600, T, 600, 72)
    mi = workloads.multi_step_inputs(w, T)
    B, _, Hq, D = mi.q.shape
    S, Hkv = mi.k_cache.shape[1], mi.k_cache.shape[2]
    cached = np.maximum(mi.seq_lens - T, 0).astype(np.int32)
    codes, scales = [], []
    for c in (mi.k_cache, mi.v_cache):
        cd = torch.full((B, S, Hkv, D), -128, dtype=torch.int8, device=dev)
        sc = torch.full((B, S, Hkv), float("nan"), dtype=torch.float32, device=dev)
        kvd.kv_quantize_q8(to_dev_bf16(c, dev), cd, sc, torch.from_numpy(cached).to(dev), S)
        codes.append(cd)
        scales.append(sc)
    q, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_new, mi.v_new))
    out = torch.full(mi.q.shape, float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.decode_ex(q, codes[0], codes[1], torch.from_numpy(mi.seq_lens).to(dev), S, w.scale, out,
                  k_scales=scales[0], v_scales=scales[1], k_new=kn, v_new=vn, pos=torch.from_numpy(mi.pos).to(dev),
                  workspace=_ws(kvd, torch, B, T, Hq, Hkv, D, S, dev, "f32"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: quantize the cached rows, append the T new rows quantized, attend token by token
    kc = np.zeros((B, S, Hkv, D), np.int8)
    vc = np.zeros((B, S, Hkv, D), np.int8)
    ks = np.full((B, S, Hkv), np.nan, np.float32)
    vs = np.full((B, S, Hkv), np.nan, np.float32)
    for b in range(B):
        n = int(cached[b])
        if n:
            kc[b, :n], ks[b, :n] = oracle.quantize_q8(mi.k_cache[b, :n])
            vc[b, :n], vs[b, :n] = oracle.quantize_q8(mi.v_cache[b, :n])
    for i in range(T):
        kc, vc, ks, vs, _ = oracle.kv_append_q8(kc, vc, ks, vs, mi.k_new[:, i], mi.v_new[:, i], mi.pos + i)
    assert np.array_equal(codes[0].cpu().numpy()[np.isfinite(ks)], kc[np.isfinite(ks)])
    kd, vd = oracle.dequantize_q8(np.where(np.isfinite(ks)[..., None], kc, 0), np.nan_to_num(ks)), \
        oracle.dequantize_q8(np.where(np.isfinite(vs)[..., None], vc, 0), np.nan_to_num(vs))
    got = out.cpu().numpy().astype(np.float64)
    for i in range(T):
        Li = np.clip(mi.seq_lens - T + 1 + i, 0, None).astype(np.int32)
        want, _ = oracle.decode_attention_f64kv(mi.q[:, i], kd, vd, Li, w.scale)
        assert_close(got[:, i], want, "f32", f"int8 multi token {i}")


def test_ex_single_forms_equal_dedicated_calls():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("ex1", 5, 32, 8, 128, 500, 1, 500, 73)
    inp = workloads.step_inputs(w)
    B, Hq, D = inp.q.shape
    S, Hkv = inp.k_cache.shape[1], inp.k_cache.shape[2]
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    ws = _ws(kvd, torch, B, 1, Hq, Hkv, D, S, dev)
    # contiguous bf16 step
    kc1, vc1 = to_dev_bf16(inp.k_cache, dev), to_dev_bf16(inp.v_cache, dev)
    kc2, vc2 = to_dev_bf16(inp.k_cache, dev), to_dev_bf16(inp.v_cache, dev)
    a = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
    b = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=dev)
    kvd.decode_step(q, kc1, vc1, kn, vn, pos, lens, S, w.scale, a, workspace=ws)
    kvd.decode_ex(q, kc2, vc2, lens, S, w.scale, b, k_new=kn, v_new=vn, pos=pos, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_bits(a), bf16_tensor_bits(b))
    # attention only, no append
    kvd.decode_attention(q, kc1, vc1, lens, S, w.scale, a, workspace=ws)
    kvd.decode_ex(q, kc1, vc1, lens, S, w.scale, b, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_bits(a), bf16_tensor_bits(b))
