"""The no-allocation entry point, kvd_decode_attention_static.

It serves callers that may not allocate device memory while decoding (a
serving loop with a frozen memory budget, a plugin handed only its tensors, a
path that must not risk the synchronisation cudaMalloc can cause): it uses a
scratch array compiled into the library instead of a caller workspace.

Checked through the C ABI against kvd_decode_attention and against the CPU
oracle (same tolerances as the other parity tests), on two calls in a row,
since the shared array keeps the previous call's contents. Kept in a file of
its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, oracle_step, spread_step, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu


def _host(out, out_dtype):
    if out_dtype == "bf16":
        return bf16_bits_to_f32(bf16_tensor_bits(out)).astype(np.float64)
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case,out_dtype", [
    (("mqa", 8, 48, 1, 256, 2048, None), "bf16"),   # tensor-core path, split pairs
    (("gqa", 16, 32, 8, 128, 1500, 1), "f32"),      # mma path, ragged lengths
])
def test_static_entry_point_matches_workspace_entry_point(case, out_dtype):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, seed = case
    if seed is None:
        w = workloads.Workload(name, B, Hq, Hkv, D, S, S, S, 11)
    else:
        w = workloads.Workload(name, B, Hq, Hkv, D, S, 1, S, seed, peaked_frac=0.01)
    inp = workloads.step_inputs(w)
    q, kc, vc = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_cache, inp.v_cache))
    kvd.kv_append(kc, vc, to_dev_bf16(inp.k_new, dev), to_dev_bf16(inp.v_new, dev),
                  torch.from_numpy(inp.pos).to(dev))
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32

    ref = torch.empty(inp.q.shape, dtype=tdt, device=dev)
    ws = kvd.alloc_workspace(q, kc, S, 0, out_dtype)
    kvd.decode_attention(q, kc, vc, lens, S, w.scale, ref, workspace=ws)
    torch.cuda.synchronize()
    ref_h = _host(ref, out_dtype)

    want, _ = oracle_step(inp)
    lib = kvd.load()
    code = kvd.OUT_BF16 if out_dtype == "bf16" else kvd.OUT_F32
    for call in range(2):
        out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        rc = lib.kvd_decode_attention_static(
            q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(), B, S, S, Hq, Hkv, D,
            ctypes.c_float(w.scale), 0, out.data_ptr(), code, None, status.data_ptr(),
            torch.cuda.current_stream().cuda_stream or None)
        assert rc == kvd.OK, kvd.status_string(rc)
        torch.cuda.synchronize()
        assert status.item() == 0
        got = _host(out, out_dtype)
        assert_close(got, ref_h, out_dtype, f"{name} static call {call}")
        assert_close(got, want, out_dtype, f"{name} static call {call} vs oracle", spread=spread_step(inp))


def test_static_entry_point_rejects_oversized_workspace():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    B, Hq, Hkv, D, S = 2, 48, 1, 256, 4096
    n_split = 5000  # (n_split + pairs - 1) * 48 * 256 * 4 bytes is far above the static array
    _, need = kvd.decode_plan(B, Hq, Hkv, D, S, 0, n_split)
    assert need > kvd.STATIC_WORKSPACE_BYTES
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((B, S, Hkv, D), dtype=torch.bfloat16, device=dev)
    lens = torch.full((B,), S, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    rc = kvd.load().kvd_decode_attention_static(
        q.data_ptr(), kc.data_ptr(), kc.data_ptr(), lens.data_ptr(), B, S, S, Hq, Hkv, D,
        ctypes.c_float(0.0625), n_split, out.data_ptr(), kvd.OUT_BF16, None, None, None)
    assert rc == kvd.ERR_WORKSPACE_TOO_SMALL
