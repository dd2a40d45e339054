"""Paged int8 KV cache on the GPU, through the C ABI (kvd_kv_append_q8_paged
and kvd_decode_ex with scale pools and a block table): the same kernels as
the contiguous int8 calls with only the row addresses changed, so the outputs
must be bit-identical to the contiguous int8 step on the same rows; the pools
after the append must equal the oracle's paged int8 append byte for byte, and
the outputs the oracle's attention over the gathered cache. Shapes cover
MHA, GQA and MQA (several CTAs of 16 query heads per token run), page sizes
below and above the 64-token tile, and table entries that name no page."""
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
    ("gqa4", 9, 32, 8, 128, 900, 0, 900, 91),
    ("mqa48", 4, 48, 1, 256, 700, 1, 700, 92),
    ("mha64", 5, 6, 6, 64, 400, 1, 400, 93),
    ("g8d256", 4, 16, 2, 256, 300, 1, 300, 94),  # mma.sync, 16 consecutive rows a thread
]


def _to_pool(rows, table, P, num_pages, fill):
    """Pool [num_pages, P, ...] holding block j of sequence b of a contiguous
    array [B, S, ...] on page table[b, j] (a layout only)."""
    pool = np.full((num_pages, P) + rows.shape[2:], fill, dtype=rows.dtype)
    for b in range(table.shape[0]):
        for j in range(table.shape[1]):
            if table[b, j] >= 0:
                blk = rows[b, j * P:(j + 1) * P]
                pool[table[b, j], :blk.shape[0]] = blk
    return pool


def _contiguous_q8(inp, dev):
    """Codes and scales of the cached rows (t < L_b - 1) from the GPU quantizer;
    other rows hold code -128 and NaN scales."""
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
    return res  # kc, ks, vc, vs


def _host(out, out_dtype):
    return bf16_tensor_bits(out) if out_dtype == "bf16" else out.cpu().numpy()


def _run_pair(inp, pin, dev, out_dtype, n_split, table=None):
    """The contiguous int8 step and the paged int8 step on the same rows.
    Returns (contiguous (out, lse), paged (out, lse, kc, vc, ks, vs pools),
    status of the paged step, host pools before the step)."""
    import torch
    import kv_cache_decode_gb300 as kvd
    kc, ks, vc, vs = _contiguous_q8(inp, dev)
    P = pin.page_size
    t = pin.block_table if table is None else table
    num_pages = pin.k_pages.shape[0]
    host = [_to_pool(x.cpu().numpy(), pin.block_table, P, num_pages, f)
            for x, f in ((kc, -128), (vc, -128), (ks, np.nan), (vs, np.nan))]
    pools = [torch.from_numpy(h.copy()).to(dev) for h in host]
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    S = inp.k_cache.shape[1]
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    res = []
    ws = kvd.alloc_workspace(q, inp.k_cache, S, n_split, out_dtype)
    # contiguous int8 step
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    kvd.decode_step_q8(q, kc, vc, ks, vs, kn, vn, pos, lens, S, inp.workload.scale, out, workspace=ws,
                       n_split=n_split, lse=lse)
    torch.cuda.synchronize()
    res.append((_host(out, out_dtype), lse.cpu().numpy()))
    # paged int8 step, planned with the same max_seq_len
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.decode_ex(q, pools[0], pools[1], lens, S, inp.workload.scale, out, k_scales=pools[2], v_scales=pools[3],
                  block_table=torch.from_numpy(t).to(dev), k_new=kn, v_new=vn, pos=pos, workspace=ws,
                  n_split=n_split, lse=lse, status=status)
    torch.cuda.synchronize()
    res.append((_host(out, out_dtype), lse.cpu().numpy()) + tuple(x.cpu().numpy() for x in pools))
    return res[0], res[1], int(status.item()), host


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("page", [16, 128])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_paged_q8_step_matches_contiguous_and_oracle(case, page, out_dtype):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    pin = workloads.paged_step_inputs(inp, page, seed=seed)
    for n_split in (0, 7):
        (co, cl), paged, status, host = _run_pair(inp, pin, dev, out_dtype, n_split)
        po, pl = paged[:2]
        assert status == 0
        assert np.array_equal(np.asarray(po).view(np.uint8), np.asarray(co).view(np.uint8)), f"{name} P{page} out"
        assert np.array_equal(pl.view(np.uint8), cl.view(np.uint8)), f"{name} P{page} lse"
    # pools after the append: the oracle's paged int8 append, byte for byte
    okc, ovc, oks, ovs, skipped, bad = oracle.kv_append_q8_paged(host[0], host[1], host[2], host[3], inp.k_new,
                                                                 inp.v_new, pin.block_table, inp.pos)
    assert skipped == 0 and bad == 0
    for g, w, what in zip(paged[2:], (okc, ovc, oks, ovs), ("k codes", "v codes", "k scales", "v scales")):
        assert np.array_equal(g.view(np.uint8), w.view(np.uint8)), what
    want, want_lse = oracle.decode_attention_q8_paged(inp.q, okc, ovc, oks, ovs, pin.block_table, inp.seq_lens,
                                                      inp.workload.scale)
    got = bf16_bits_to_f32(po).astype(np.float64) if out_dtype == "bf16" else po.astype(np.float64)
    assert_close(got, want, out_dtype, f"{name} P{page} vs oracle")
    finite = np.isfinite(want_lse)
    assert np.max(np.abs(pl[finite] - want_lse[finite]), initial=0.0) < (4e-3 if out_dtype == "bf16" else 1e-4)
    assert np.all(np.isneginf(pl[~finite]))


@pytest.mark.parametrize("case", [CASES[0], CASES[1]], ids=["gqa4", "mqa48"])
def test_paged_q8_bad_entry_reads_zero_rows(case):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    page = 32
    pin = workloads.paged_step_inputs(inp, page, seed=seed + 1)
    table = pin.block_table.copy()
    b = int(np.argmax(inp.seq_lens))
    nb = -(-int(inp.seq_lens[b]) // page)
    assert nb >= 3
    table[b, nb // 2] = -3  # a middle block names no page: its tokens read zero rows
    _, paged, status, host = _run_pair(inp, pin, dev, "f32", 0, table=table)
    assert status & BAD_PAGE
    okc, ovc, oks, ovs, _, _ = oracle.kv_append_q8_paged(host[0], host[1], host[2], host[3], inp.k_new,
                                                         inp.v_new, table, inp.pos)
    want, _ = oracle.decode_attention_q8_paged(inp.q, okc, ovc, oks, ovs, table, inp.seq_lens, inp.workload.scale)
    assert_close(paged[0].astype(np.float64), want, "f32", f"{name} bad entry")


def test_paged_q8_append_edges():
    """New rows at the first and last row of a page, past the capacity, and
    into a block whose entry names no page (kvd_kv_append_q8_paged alone)."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    P = 16
    w = workloads.Workload("app8p", 6, 8, 2, 128, 64, 1, 64, 94)
    inp = workloads.step_inputs(w, lens=np.array([16, 17, 32, 1, 64, 40], np.int32))
    pin = workloads.paged_step_inputs(inp, P, seed=5)
    table = pin.block_table.copy()
    pos = inp.pos.copy()            # 15, 16, 31, 0, 63, 39
    pos[4] = 64                     # past the capacity of 4 pages
    table[5, 39 // P] = pin.k_pages.shape[0] + 5  # names no page
    num_pages = pin.k_pages.shape[0]
    r = np.random.default_rng(95)
    host = [r.integers(-127, 128, (num_pages, P, 2, 128), dtype=np.int8) for _ in range(2)]
    host += [r.random((num_pages, P, 2), dtype=np.float32) for _ in range(2)]
    pools = [torch.from_numpy(h.copy()).to(dev) for h in host]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append_q8_paged(pools[0], pools[1], pools[2], pools[3], to_dev_bf16(inp.k_new, dev),
                           to_dev_bf16(inp.v_new, dev), torch.from_numpy(table).to(dev),
                           torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    want = oracle.kv_append_q8_paged(host[0], host[1], host[2], host[3], inp.k_new, inp.v_new, table, pos)
    assert want[4] == 2 and want[5] == 1
    for g, x, what in zip(pools, want[:4], ("k codes", "v codes", "k scales", "v scales")):
        assert np.array_equal(g.cpu().numpy().view(np.uint8), x.view(np.uint8)), what
    assert int(status.item()) == (0x2 | BAD_PAGE)
