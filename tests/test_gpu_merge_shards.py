"""kvd_merge_attention: attention over each sequence's tokens split into
disjoint shards (each attended alone by kvd_decode_attention, its out and lse
kept) merges back to the attention over all of them, against the oracle;
empty shards and empty sequences included; both engines, bf16 and fp32."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (48, 1, 256), (6, 6, 64)], ids=["gqa", "mqa", "mha"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_shards_merge_to_the_whole(Hq, Hkv, D, dt):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("shards", 6, Hq, Hkv, D, 600, 0, 600, 131)
    inp = workloads.step_inputs(w)
    B, S = inp.q.shape[0], inp.k_cache.shape[1]
    kc, vc, _ = oracle.kv_append(inp.k_cache, inp.v_cache, inp.k_new, inp.v_new, inp.pos)
    want, want_lse = oracle.decode_attention(inp.q, kc, vc, inp.seq_lens, w.scale)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    q = to_dev_bf16(inp.q, dev)
    cuts = [0, 100, 100, 357, S]  # the second shard holds no tokens
    outs = torch.empty((len(cuts) - 1,) + inp.q.shape, dtype=tdt, device=dev)
    lses = torch.empty((len(cuts) - 1, B, Hq), dtype=torch.float32, device=dev)
    for j, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        n = max(b - a, 1)
        ks = to_dev_bf16(np.ascontiguousarray(kc[:, a:a + n]), dev)
        vs = to_dev_bf16(np.ascontiguousarray(vc[:, a:a + n]), dev)
        lens = torch.from_numpy(np.clip(inp.seq_lens - a, 0, b - a).astype(np.int32)).to(dev)
        ws = kvd.alloc_workspace(q, ks, n, 0, dt)
        kvd.decode_attention(q, ks, vs, lens, n, w.scale, outs[j], workspace=ws, lse=lses[j])
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    kvd.merge_attention(outs, lses, out, lse=lse)
    torch.cuda.synchronize()
    got = bf16_bits_to_f32(bf16_tensor_bits(out)).astype(np.float64) if dt == "bf16" else out.cpu().numpy().astype(
        np.float64)
    # bf16 shards carry one more rounding each: hold them to the bf16 tolerance as well
    assert_close(got, want, dt, f"merged shards {dt}")
    l = lse.cpu().numpy()
    live = np.isfinite(want_lse)
    assert np.max(np.abs(l[live] - want_lse[live]), initial=0.0) < (4e-3 if dt == "bf16" else 1e-4)
    assert np.all(np.isneginf(l[~live]))
    # the GPU merge is the oracle's merge of the GPU shards (float32 arithmetic)
    so = (bf16_bits_to_f32(bf16_tensor_bits(outs)) if dt == "bf16" else outs.cpu().numpy()).astype(np.float64)
    mo, _ = oracle.merge_attention(so, lses.cpu().numpy())
    assert np.max(np.abs(got - mo)) < (1e-2 if dt == "bf16" else 1e-5)


@pytest.mark.parametrize("bad", [float("nan"), float("inf")], ids=["nan", "inf"])
def test_invalid_shard_normaliser_gives_nan_row(bad):
    """A shard whose normaliser is NaN or +inf is no valid result: its row comes
    out NaN (every column and lse) instead of a mix of the other shards; the
    other rows are untouched by it."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    n, rows, D = 3, 5, 128
    g = torch.Generator().manual_seed(7)
    outs = torch.randn((n, rows, D), generator=g).to(dev)
    lses = torch.randn((n, rows), generator=g).to(dev)
    lses[1, 2] = bad
    out = torch.zeros((rows, D), dtype=torch.float32, device=dev)
    lse = torch.zeros((rows,), dtype=torch.float32, device=dev)
    kvd.merge_attention(outs, lses, out, lse=lse)
    torch.cuda.synchronize()
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.all(np.isnan(o[2])) and np.isnan(l[2])
    good = [r for r in range(rows) if r != 2]
    want, want_lse = oracle.merge_attention(outs.cpu().numpy().astype(np.float64)[:, good],
                                            lses.cpu().numpy().astype(np.float64)[:, good])
    assert np.max(np.abs(o[good] - want)) < 1e-5
    assert np.max(np.abs(l[good] - want_lse)) < 1e-5
