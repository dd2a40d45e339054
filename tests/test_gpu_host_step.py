"""kvd_decode_step_host: the step from host inputs to a host result equals the
device-input step bit for bit (output copied back, caches after the append),
for one and several query tokens on both engines, and a bound HostStep
re-reads its host inputs on every call."""
import numpy as np
import pytest

import workloads
from gpu_helpers import bf16_tensor_bits, cuda_or_skip, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,D,T", [(32, 8, 128, 1), (48, 1, 256, 1), (32, 8, 128, 3), (48, 1, 256, 2)],
                         ids=["mma_t1", "tcgen05_t1", "mma_t3", "tcgen05_t2"])
def test_host_step_equals_device_step(Hq, Hkv, D, T):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("hs", 7, Hq, Hkv, D, 600, T, 600, 111)
    mi = workloads.multi_step_inputs(w, T)
    B, S = mi.q.shape[0], mi.k_cache.shape[1]
    squeeze = (lambda a: a[:, 0]) if T == 1 else (lambda a: a)
    q_np, kn_np, vn_np = squeeze(mi.q), squeeze(mi.k_new), squeeze(mi.v_new)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, 0, "bf16")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    # device-input step
    kc1, vc1 = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
    ref = torch.empty(q_np.shape, dtype=torch.bfloat16, device=dev)
    kvd.decode_step_multi(to_dev_bf16(mi.q, dev), kc1, vc1, to_dev_bf16(mi.k_new, dev), to_dev_bf16(mi.v_new, dev),
                          torch.from_numpy(mi.pos).to(dev), torch.from_numpy(mi.seq_lens).to(dev), S, w.scale,
                          ref.view(mi.q.shape), workspace=ws)
    torch.cuda.synchronize()
    # host-input step
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    q_h, kn_h, vn_h = (pin(a.view(np.int16)).view(torch.bfloat16) for a in (q_np, kn_np, vn_np))
    pos_h, lens_h = pin(mi.pos), pin(mi.seq_lens)
    kc2, vc2 = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
    out = torch.empty(q_np.shape, dtype=torch.bfloat16, device=dev)
    out_h = torch.full(q_np.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    staging = torch.empty(kvd.step_staging_bytes(B, T, Hq, Hkv, D), dtype=torch.uint8, device=dev)
    step = kvd.HostStep(q_h, kn_h, vn_h, pos_h, lens_h, kc2, vc2, staging, S, w.scale, out, out_h, workspace=ws)
    step()
    torch.cuda.synchronize()
    assert np.array_equal(out_h.view(torch.int16).numpy().view(np.uint16), bf16_tensor_bits(ref))
    assert np.array_equal(bf16_tensor_bits(kc2), bf16_tensor_bits(kc1))
    assert np.array_equal(bf16_tensor_bits(vc2), bf16_tensor_bits(vc1))
    # the bound step reads the host inputs again: zero queries give the plain mean of V
    q_h.zero_()
    step()
    torch.cuda.synchronize()
    got = out_h.float().numpy()
    assert np.all(np.isfinite(got)) and not np.array_equal(out_h.view(torch.int16).numpy().view(np.uint16),
                                                           bf16_tensor_bits(ref))


@pytest.mark.parametrize("T", [1, 2])
def test_packed_host_inputs_equal_separate(T):
    """Inputs in one pinned packet laid out like the staging buffer (one copy
    in) give the same step as separate host tensors (five copies)."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    Hq, Hkv, D = 16, 4, 128
    w = workloads.Workload("hp", 5, Hq, Hkv, D, 500, T, 500, 112)
    mi = workloads.multi_step_inputs(w, T)
    B, S = mi.q.shape[0], mi.k_cache.shape[1]
    squeeze = (lambda a: a[:, 0]) if T == 1 else (lambda a: a)
    q_np, kn_np, vn_np = squeeze(mi.q), squeeze(mi.k_new), squeeze(mi.v_new)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, 0, "bf16")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    staging = torch.empty(kvd.step_staging_bytes(B, T, Hq, Hkv, D), dtype=torch.uint8, device=dev)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    sep = [pin(a.view(np.int16)).view(torch.bfloat16) for a in (q_np, kn_np, vn_np)] + [pin(mi.pos), pin(mi.seq_lens)]
    packet, *views = kvd.alloc_host_packet(B, T, Hq, Hkv, D)
    for dst, src in zip(views, sep):
        dst.copy_(src)
    outs = []
    for inputs in (sep, views):
        kc, vc = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
        out = torch.empty(q_np.shape, dtype=torch.bfloat16, device=dev)
        out_h = torch.full(q_np.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
        kvd.decode_step_host(*inputs, kc, vc, staging, S, w.scale, out, out_h, workspace=ws)
        torch.cuda.synchronize()
        outs.append((out_h.view(torch.int16).numpy().copy(), bf16_tensor_bits(kc)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert not np.isnan((outs[1][0].view(np.uint16).astype(np.uint32) << 16).view(np.float32)).any()


@pytest.mark.parametrize("T", [1, 2])
def test_direct_host_output_equals_copy(T):
    """out=None: the kernels write the result straight into pinned host memory;
    the same bits as the device output copied back."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    Hq, Hkv, D = 48, 1, 256
    w = workloads.Workload("hd", 6, Hq, Hkv, D, 500, T, 500, 114)
    mi = workloads.multi_step_inputs(w, T)
    B, S = mi.q.shape[0], mi.k_cache.shape[1]
    squeeze = (lambda a: a[:, 0]) if T == 1 else (lambda a: a)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, 0, "bf16")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    staging = torch.empty(kvd.step_staging_bytes(B, T, Hq, Hkv, D), dtype=torch.uint8, device=dev)
    packet, *views = kvd.alloc_host_packet(B, T, Hq, Hkv, D)
    for dst, src in zip(views, (squeeze(mi.q), squeeze(mi.k_new), squeeze(mi.v_new), mi.pos, mi.seq_lens)):
        dst.copy_(torch.from_numpy(np.ascontiguousarray(src.view(np.int16) if src.dtype == np.uint16 else src))
                  .view(dst.dtype))
    outs = []
    for direct in (False, True):
        kc, vc = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
        out = None if direct else torch.empty(views[0].shape, dtype=torch.bfloat16, device=dev)
        out_h = torch.full(views[0].shape, float("nan"), dtype=torch.bfloat16).pin_memory()
        kvd.decode_step_host(*views, kc, vc, staging, S, w.scale, out, out_h, workspace=ws)
        torch.cuda.synchronize()
        outs.append(out_h.view(torch.int16).numpy().copy())
    assert np.array_equal(outs[0], outs[1])
    assert not np.isnan((outs[1].view(np.uint16).astype(np.uint32) << 16).view(np.float32)).any()
