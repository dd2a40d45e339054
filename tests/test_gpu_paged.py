"""Paged KV cache on the GPU, through the C ABI: append, attention and the
one-call step over a shuffled pool of pages, against the oracle (which
gathers the pages on the host) and against the contiguous calls.

The paged calls run the same kernels and schedule as the contiguous ones with
only the row addresses changed, so their outputs must be bit-identical to the
contiguous calls on the same rows; both are also checked against the oracle.
Shapes cover both engines (tcgen05 for groups above 16, mma.sync below), all
supported page sizes up to one above the tile, ragged and empty sequences, and
the edge cases of the table: new rows at page boundaries, and entries that
name no page of the pool.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

BAD_PAGE = 0x8

CASES = [
    # name, B, Hq, Hkv, D, S, lengths lo..hi, seed
    ("mqa48", 6, 48, 1, 256, 700, 1, 700, 41),    # tcgen05, D 256
    ("gqa32", 5, 64, 2, 128, 600, 1, 600, 42),    # tcgen05, D 128, group 32
    ("g20d64", 4, 20, 1, 64, 520, 1, 520, 43),    # tcgen05, D 64, group 20
    ("gqa4", 9, 32, 8, 128, 900, 1, 900, 44),     # mma.sync, D 128
    ("mha64", 5, 6, 6, 64, 400, 1, 400, 45),      # mma.sync, D 64
    ("g8d256", 4, 16, 2, 256, 300, 1, 300, 46),   # mma.sync, D 256
]


def _out(dev, shape, out_dtype):
    import torch
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    return torch.full(shape, float("nan"), dtype=tdt, device=dev)


def _host(out, out_dtype):
    return bf16_tensor_bits(out) if out_dtype == "bf16" else out.cpu().numpy()


def _as_f64(o, out_dtype):
    return bf16_bits_to_f32(o).astype(np.float64) if out_dtype == "bf16" else o.astype(np.float64)


def _contiguous(inp, dev, out_dtype, n_split):
    import torch
    import kv_cache_decode_gb300 as kvd
    q, kc, vc, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_cache, inp.v_cache, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    S = inp.k_cache.shape[1]
    out = _out(dev, inp.q.shape, out_dtype)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    ws = kvd.alloc_workspace(q, kc, S, n_split, out_dtype)
    kvd.decode_step(q, kc, vc, kn, vn, pos, lens, S, inp.workload.scale, out, workspace=ws,
                    n_split=n_split, lse=lse)
    torch.cuda.synchronize()
    return _host(out, out_dtype), lse.cpu().numpy()


def _paged(pin, dev, out_dtype, n_split, fused=True, table=None, lens=None):
    import torch
    import kv_cache_decode_gb300 as kvd
    inp = pin.step
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    kp, vp = to_dev_bf16(pin.k_pages, dev), to_dev_bf16(pin.v_pages, dev)
    bt = torch.from_numpy(pin.block_table if table is None else table).to(dev)
    pos = torch.from_numpy(inp.pos).to(dev)
    lens_np = inp.seq_lens if lens is None else lens
    lens_t = torch.from_numpy(lens_np).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mx = inp.k_cache.shape[1]  # as the contiguous call, so that both plan the same split
    out = _out(dev, inp.q.shape, out_dtype)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    ws = kvd.alloc_workspace(q, kp, mx, n_split, out_dtype)
    if fused:
        kvd.decode_step_paged(q, kp, vp, kn, vn, pos, bt, lens_t, mx, inp.workload.scale, out,
                              workspace=ws, n_split=n_split, lse=lse, status=status)
    else:
        kvd.kv_append_paged(kp, vp, kn, vn, bt, pos, status=status)
        kvd.decode_attention_paged(q, kp, vp, bt, lens_t, mx, inp.workload.scale, out, workspace=ws,
                                   n_split=n_split, lse=lse, status=status)
    torch.cuda.synchronize()
    return (_host(out, out_dtype), lse.cpu().numpy(), bf16_tensor_bits(kp), bf16_tensor_bits(vp),
            int(status.item()))


def _oracle_paged(pin, table=None, lens=None):
    inp = pin.step
    t = pin.block_table if table is None else table
    kp, vp, _, _ = oracle.kv_append_paged(pin.k_pages, pin.v_pages, inp.k_new, inp.v_new, t, inp.pos)
    L = inp.seq_lens if lens is None else lens
    out, lse = oracle.decode_attention_paged(inp.q, kp, vp, t, L, inp.workload.scale)
    return out, lse, kp, vp


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("page", [16, 32, 64, 128])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_paged_step_matches_contiguous_and_oracle(case, page, out_dtype):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    w = workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed)
    inp = workloads.step_inputs(w)
    pin = workloads.paged_step_inputs(inp, page, seed=seed)
    for n_split in (0, 7):
        ref_o, ref_l = _contiguous(inp, dev, out_dtype, n_split)
        o, l, kp, vp, status = _paged(pin, dev, out_dtype, n_split)
        assert status == 0
        assert np.array_equal(np.asarray(o).view(np.uint8), np.asarray(ref_o).view(np.uint8)), f"{name} P{page} out"
        assert np.array_equal(l.view(np.uint8), ref_l.view(np.uint8)), f"{name} P{page} lse"
    want, want_lse, okp, ovp = _oracle_paged(pin)
    assert np.array_equal(kp, okp) and np.array_equal(vp, ovp), "pools after the append"
    assert_close(_as_f64(o, out_dtype), want, out_dtype, f"{name} P{page} vs oracle")
    finite = np.isfinite(want_lse)
    assert np.max(np.abs(l[finite] - want_lse[finite])) < 1e-3
    assert np.all(np.isneginf(l[~finite]))


@pytest.mark.parametrize("case", [CASES[0], CASES[3]], ids=["tcgen05", "mma"])
def test_paged_step_equals_two_calls(case):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    w = workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed)
    pin = workloads.paged_step_inputs(workloads.step_inputs(w), 32, seed=seed + 1)
    a = _paged(pin, dev, "f32", 5, fused=True)
    b = _paged(pin, dev, "f32", 5, fused=False)
    for x, y, what in zip(a[:4], b[:4], ("out", "lse", "k_pages", "v_pages")):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), what
    assert a[4] == b[4] == 0


def test_paged_append_edges():
    """New rows at the first and last row of a page, past the capacity, and
    into a block whose entry names no page."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    P = 16
    w = workloads.Workload("app", 6, 8, 2, 128, 64, 1, 64, 47)
    inp = workloads.step_inputs(w, lens=np.array([16, 17, 32, 1, 64, 40], np.int32))
    pin = workloads.paged_step_inputs(inp, P, seed=3)
    table = pin.block_table.copy()
    pos = inp.pos.copy()            # 15, 16, 31, 0, 63, 39
    pos[4] = 64                     # past the capacity of 4 pages
    table[5, 39 // P] = pin.k_pages.shape[0] + 5  # names no page
    kp, vp = to_dev_bf16(pin.k_pages, dev), to_dev_bf16(pin.v_pages, dev)
    kn, vn = to_dev_bf16(inp.k_new, dev), to_dev_bf16(inp.v_new, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append_paged(kp, vp, kn, vn, torch.from_numpy(table).to(dev), torch.from_numpy(pos).to(dev),
                        status=status)
    torch.cuda.synchronize()
    ek, ev, skipped, bad = oracle.kv_append_paged(pin.k_pages, pin.v_pages, inp.k_new, inp.v_new, table, pos)
    assert skipped == 2 and bad == 1
    assert np.array_equal(bf16_tensor_bits(kp), ek) and np.array_equal(bf16_tensor_bits(vp), ev)
    assert int(status.item()) == (0x2 | BAD_PAGE)


@pytest.mark.parametrize("case", [CASES[0], CASES[3]], ids=["tcgen05", "mma"])
@pytest.mark.parametrize("page", [16, 64])
def test_paged_bad_entry_reads_zero_rows(case, page):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    w = workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed)
    inp = workloads.step_inputs(w)
    pin = workloads.paged_step_inputs(inp, page, seed=seed + 2)
    table = pin.block_table.copy()
    # a middle block of the longest sequence names no page; its tokens read zeros
    b = int(np.argmax(inp.seq_lens))
    nb = -(-int(inp.seq_lens[b]) // page)
    assert nb >= 3
    table[b, nb // 2] = -3
    o, l, _, _, status = _paged(pin, dev, "f32", 0, table=table)
    assert status & BAD_PAGE
    want, _, _, _ = _oracle_paged(pin, table=table)
    assert_close(o.astype(np.float64), want, "f32", f"{name} P{page} bad entry")


def test_paged_empty_and_short_sequences():
    dev = cuda_or_skip()
    w = workloads.Workload("short", 7, 48, 1, 256, 300, 0, 300, 48)
    lens = np.array([0, 1, 16, 17, 0, 64, 65], np.int32)
    inp = workloads.step_inputs(w, lens=lens)
    for page in (16, 128):
        pin = workloads.paged_step_inputs(inp, page, seed=page)
        ref_o, _ = _contiguous(inp, dev, "bf16", 0)
        o, _, _, _, status = _paged(pin, dev, "bf16", 0)
        assert status == 0
        assert np.array_equal(o, ref_o)
        want, _, _, _ = _oracle_paged(pin)
        assert_close(_as_f64(o, "bf16"), want, "bf16", f"short P{page}")
