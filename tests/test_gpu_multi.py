"""Multi-token decode on the GPU (T drafted tokens per sequence, causal among
them), through the C ABI, against the oracle; T = 1 against the single-token
calls bit for bit. Shapes cover the head dimensions, groups from MHA to MQA,
pairs of one block of 16 rows (T * G <= 16) and of several (the last one
partly filled), ragged lengths down to T, and split and unsplit pairs."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, Hq, Hkv, D, S, lengths lo..hi, seed, T
    ("g4t4", 6, 32, 8, 128, 700, 4, 700, 61, 4),
    ("mha_t8", 5, 6, 6, 64, 400, 8, 400, 62, 8),
    ("g2t3d256", 4, 8, 4, 256, 300, 3, 300, 63, 3),
    ("g8t2", 7, 16, 2, 128, 900, 2, 900, 64, 2),
    ("g1t16", 3, 4, 4, 128, 500, 16, 500, 65, 16),
    # several blocks of 16 rows per pair
    ("g4t8", 5, 32, 8, 128, 600, 8, 600, 66, 8),          # 32 rows: 2 blocks
    ("mqa48t2", 4, 48, 1, 256, 500, 2, 500, 67, 2),       # 96 rows: 6 blocks, MQA
    ("g20t3d64", 3, 20, 1, 64, 400, 3, 400, 68, 3),       # 60 rows: 4 blocks, the last of 12
    ("g16t5", 3, 32, 2, 128, 450, 5, 450, 69, 5),         # 80 rows: 5 blocks
    # the tcgen05 kernel's 128-row tile with the tokens stacked: two KV heads
    # (each token's query rows a separate box), and a group of 20 padded to 24
    ("g24t4kv2", 5, 48, 2, 128, 500, 4, 500, 70, 4),      # 4 x 24 = 96 rows in one tile
]


def _run(mi, dev, out_dtype, n_split, fused=True):
    import torch
    import kv_cache_decode_gb300 as kvd
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_cache, mi.v_cache, mi.k_new, mi.v_new))
    pos = torch.from_numpy(mi.pos).to(dev)
    lens = torch.from_numpy(mi.seq_lens).to(dev)
    B, T, Hq, D = mi.q.shape
    S, Hkv = mi.k_cache.shape[1], mi.k_cache.shape[2]
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = torch.full((B, T, Hq, D), float("nan"), dtype=tdt, device=dev)
    lse = torch.full((B, T, Hq), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, n_split, out_dtype)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    if fused:
        kvd.decode_step_multi(q, kc, vc, kn, vn, pos, lens, S, mi.workload.scale, out, workspace=ws,
                              n_split=n_split, lse=lse, status=status)
    else:
        kvd.kv_append_multi(kc, vc, kn, vn, pos, status=status)
        kvd.decode_attention_multi(q, kc, vc, lens, S, mi.workload.scale, out, workspace=ws, n_split=n_split,
                                   lse=lse, status=status)
    torch.cuda.synchronize()
    o = bf16_tensor_bits(out) if out_dtype == "bf16" else out.cpu().numpy()
    return o, lse.cpu().numpy(), bf16_tensor_bits(kc), bf16_tensor_bits(vc), int(status.item())


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_multi_step_matches_oracle(case, out_dtype):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed, T = case
    mi = workloads.multi_step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed), T)
    kc, vc, skipped = oracle.kv_append_multi(mi.k_cache, mi.v_cache, mi.k_new, mi.v_new, mi.pos)
    assert skipped == 0
    want, want_lse = oracle.decode_attention_multi(mi.q, kc, vc, mi.seq_lens, mi.workload.scale)
    for n_split in (0, 7):
        o, l, gk, gv, status = _run(mi, dev, out_dtype, n_split)
        assert status == 0
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc), "caches after the append"
        o64 = bf16_bits_to_f32(o).astype(np.float64) if out_dtype == "bf16" else o.astype(np.float64)
        assert_close(o64.reshape(B, T * Hq, D), want.reshape(B, T * Hq, D), out_dtype, f"{name} n_split {n_split}")
        tol = 4e-3 if out_dtype == "bf16" else 1e-4
        assert np.max(np.abs(l - want_lse)) < tol


@pytest.mark.parametrize("case", [CASES[0], CASES[4], CASES[6]], ids=["g4t4", "g1t16", "mqa48t2"])
def test_multi_step_equals_two_calls(case):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed, T = case
    mi = workloads.multi_step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed), T)
    a = _run(mi, dev, "f32", 5, fused=True)
    b = _run(mi, dev, "f32", 5, fused=False)
    for x, y, what in zip(a[:4], b[:4], ("out", "lse", "k", "v")):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), what
    assert a[4] == b[4] == 0


def test_multi_one_token_is_the_single_token_call():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("one", 5, 32, 8, 128, 600, 1, 600, 66)
    mi = workloads.multi_step_inputs(w, 1)
    a = _run(mi, dev, "bf16", 7)
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q[:, 0], mi.k_cache, mi.v_cache, mi.k_new[:, 0], mi.v_new[:, 0]))
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    ws = kvd.alloc_workspace(q, kc, w.S_max, 7)
    kvd.decode_step(q, kc, vc, kn, vn, torch.from_numpy(mi.pos).to(dev), torch.from_numpy(mi.seq_lens).to(dev),
                    w.S_max, w.scale, out, workspace=ws, n_split=7, lse=lse)
    torch.cuda.synchronize()
    assert np.array_equal(a[0][:, 0], bf16_tensor_bits(out))
    assert np.array_equal(a[1][:, 0].view(np.uint32), lse.cpu().numpy().view(np.uint32))


def test_multi_rows_past_capacity_are_skipped():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    w = workloads.Workload("cap", 3, 8, 2, 128, 64, 4, 64, 67)
    mi = workloads.multi_step_inputs(w, 4, lens=np.array([64, 10, 4], np.int32))
    pos = mi.pos.copy()
    pos[1] = 62  # rows 62, 63 fit, 64 and 65 do not
    kc, vc = to_dev_bf16(mi.k_cache, dev), to_dev_bf16(mi.v_cache, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append_multi(kc, vc, to_dev_bf16(mi.k_new, dev), to_dev_bf16(mi.v_new, dev),
                        torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    ek, ev, skipped = oracle.kv_append_multi(mi.k_cache, mi.v_cache, mi.k_new, mi.v_new, pos)
    assert skipped == 2 and int(status.item()) == 0x2
    assert np.array_equal(bf16_tensor_bits(kc), ek) and np.array_equal(bf16_tensor_bits(vc), ev)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (48, 1, 256), (32, 1, 128)],
                         ids=["one_block", "twelve_blocks", "one_tile_of_128"])
def test_multi_short_sequences_give_empty_rows(Hq, Hkv, D):
    """A sequence shorter than T: its first query tokens see no token (zero rows,
    lse -inf), the rest see what exists; rows appended before position 0 are
    skipped."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    T = 4
    w = workloads.Workload("short_mt", 3, Hq, Hkv, D, 64, 4, 64, 68)
    mi = workloads.multi_step_inputs(w, T, lens=np.array([4, 9, 6], np.int32))
    lens = np.array([2, 9, 0], np.int32)  # sequence 0 holds 2 tokens after the step, sequence 2 none
    pos = lens - T                        # -2, 5, -4: rows before position 0 are skipped
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_cache, mi.v_cache, mi.k_new, mi.v_new))
    out = torch.full(mi.q.shape, float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full(mi.q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B, _, Hq, D = mi.q.shape
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, 64, 0, 3, "f32")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    kvd.decode_step_multi(q, kc, vc, kn, vn, torch.from_numpy(pos.astype(np.int32)).to(dev),
                          torch.from_numpy(lens).to(dev), 64, w.scale, out, workspace=ws, n_split=3, lse=lse,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0x2
    ekc, evc, skipped = oracle.kv_append_multi(mi.k_cache, mi.v_cache, mi.k_new, mi.v_new, pos)
    assert skipped == 2 + 4
    want, want_lse = oracle.decode_attention_multi(mi.q, ekc, evc, lens, w.scale)
    got = out.cpu().numpy().astype(np.float64)
    assert_close(got.reshape(B, T * Hq, D), want.reshape(B, T * Hq, D), "f32", "short multi")
    l = lse.cpu().numpy()
    assert np.all(np.isneginf(l[0, :2])) and np.all(np.isneginf(l[2])) and np.all(got[0, :2] == 0)
    assert np.max(np.abs(l[np.isfinite(want_lse)] - want_lse[np.isfinite(want_lse)])) < 1e-4


@pytest.mark.parametrize("Hq,Hkv,D", [(64, 1, 64), (16, 1, 64)], ids=["tcgen05_g64", "mma_g16"])
def test_multi_token_maximum_sizes(Hq, Hkv, D):
    """T = KVD_MAX_TOKENS (64) with the widest group of each engine: 64 virtual
    sequences per sequence on the tcgen05 engine (group 64), 64 blocks of 16
    rows per pair on the mma.sync engine (group 16)."""
    dev = cuda_or_skip()
    T = 64
    w = workloads.Workload("maxT", 2, Hq, Hkv, D, 200, T, 200, 113)
    mi = workloads.multi_step_inputs(w, T)
    kc, vc, skipped = oracle.kv_append_multi(mi.k_cache, mi.v_cache, mi.k_new, mi.v_new, mi.pos)
    assert skipped == 0
    want, want_lse = oracle.decode_attention_multi(mi.q, kc, vc, mi.seq_lens, mi.workload.scale)
    B = mi.q.shape[0]
    for n_split in (0, 5):
        o, l, gk, gv, status = _run(mi, dev, "f32", n_split)
        assert status == 0
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
        assert_close(o.astype(np.float64).reshape(B, T * Hq, D), want.reshape(B, T * Hq, D), "f32",
                     f"max T n_split {n_split}")
        assert np.max(np.abs(l - want_lse)) < 1e-4
